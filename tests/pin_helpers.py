"""Test-side helpers for the oracle pins: contiguous K/V scattered into a
paged pool by the test itself (independent of the oracle's gather), and the
independent references the pins compare against."""
from __future__ import annotations

import numpy as np
import torch

NAN = {"bf16": 0x7FC0, "fp16": 0x7E00}
TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def bits_to_torch64(bits: np.ndarray, dtype: str) -> torch.Tensor:
    """Library conversion of raw 16-bit patterns to float64 (torch, not the oracle)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy())
    return t.view(TORCH_DT[dtype]).to(torch.float64)


def random_bits(rng: np.random.Generator, shape, dtype: str, scale: float = 1.0) -> np.ndarray:
    x = torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32))
    return x.to(TORCH_DT[dtype]).view(torch.int16).numpy().view(np.uint16)


def paged_case(rng, lens, hq, hkv, bs, d=128, dtype="bf16", pool_slack=5, poison=True, perm=None):
    """Contiguous per-sequence K/V of the given lengths, scattered into a shuffled pool.

    Returns dict with q [B,Hq,D], k_cache/v_cache [nb,Hkv,bs,D] (uint16 bits),
    block_tables, context_lens, and the contiguous per-sequence K/V bits.
    """
    B = len(lens)
    nblk = [(L + bs - 1) // bs for L in lens]
    nb = sum(nblk) + pool_slack
    if perm is None:
        perm = rng.permutation(nb)
    kc = random_bits(rng, (nb, hkv, bs, d), dtype)
    vc = random_bits(rng, (nb, hkv, bs, d), dtype)
    if poison:
        kc[:] = NAN[dtype]
        vc[:] = NAN[dtype]
    maxb = max(1, max(nblk))
    bt = np.full((B, maxb), -1, dtype=np.int32)
    Ks, Vs = [], []
    nxt = 0
    for s, L in enumerate(lens):
        K = random_bits(rng, (hkv, L, d), dtype)
        V = random_bits(rng, (hkv, L, d), dtype)
        Ks.append(K)
        Vs.append(V)
        for j in range(nblk[s]):
            pb = int(perm[nxt])
            nxt += 1
            bt[s, j] = pb
            n = min(bs, L - j * bs)
            kc[pb, :, :n, :] = K[:, j * bs:j * bs + n, :]
            vc[pb, :, :n, :] = V[:, j * bs:j * bs + n, :]
    q = random_bits(rng, (B, hq, d), dtype)
    return dict(q=q, k_cache=kc, v_cache=vc, block_tables=bt, context_lens=np.asarray(lens, dtype=np.int32),
                K=Ks, V=Vs, num_blocks=nb, dtype=dtype, hq=hq, hkv=hkv, bs=bs, d=d)


def sdpa_reference(case, scale: float) -> np.ndarray:
    """torch scaled_dot_product_attention in float64 over the contiguous tensors."""
    B, hq, d = case["q"].shape
    hkv = case["hkv"]
    G = hq // hkv
    out = np.zeros((B, hq, d))
    for s, L in enumerate(case["context_lens"]):
        if L == 0:
            continue
        q = bits_to_torch64(case["q"][s], case["dtype"]).reshape(1, hq, 1, d)
        K = bits_to_torch64(case["K"][s], case["dtype"]).repeat_interleave(G, dim=0).reshape(1, hq, L, d)
        V = bits_to_torch64(case["V"][s], case["dtype"]).repeat_interleave(G, dim=0).reshape(1, hq, L, d)
        o = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=scale)
        out[s] = o.reshape(hq, d).numpy()
    return out
