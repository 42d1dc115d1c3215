"""Randomised GPU parity sweep and out-of-bounds guard checks.

Each sweep case draws a configuration (element type, block size, KV heads,
GQA group, batch, length mix with edge values, partition size, output type,
fused or separate block write) from a fixed seed, NaN-poisons every unused
pool slot and compares the whole step with the fp64 oracle.  The guard test
surrounds the output, the workspace and the pools with canary bytes and
checks that no kernel writes outside its buffers.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_11_gb300 as pkv
from paged_kv_cache_11_gb300 import workload as W
from tests.step_helpers import case_seeds, gpu_step, max_abs_err, oracle_step, single_token_step, to_bits, to_dev

pytestmark = pytest.mark.gpu
TOL = 5e-3
EDGE = (1, 2, 15, 16, 17, 31, 32, 33, 511, 512, 513)


def _case(seed):
    rng = np.random.default_rng(seed)
    dtype = ["bf16", "fp16"][rng.integers(2)]
    bs = [16, 32][rng.integers(2)]
    hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([1, 2, 3, 4, 5, 8, 9, 12, 16, 20]))
    B = int(rng.integers(1, 13))
    lens = []
    for _ in range(B):
        r = rng.random()
        lens.append(int(rng.choice(EDGE)) if r < 0.35 else (0 if r < 0.42 else int(rng.integers(1, 3000))))
    P = int(rng.choice([0, 0, 16, 32, 64, 256, 512, 1024])) // bs * bs if rng.random() < 0.6 else 0
    out_dtype = [torch.float32, torch.float32, torch.bfloat16, torch.float16][rng.integers(4)]
    fused = bool(rng.integers(2))
    return dict(dtype=dtype, bs=bs, hkv=hkv, hq=hkv * group, lens=tuple(lens), P=P, out_dtype=out_dtype,
                fused=fused)


@pytest.mark.parametrize("seed", case_seeds(40))
def test_random_configuration(gpu, seed):
    c = _case(1000 + seed)
    wl = W.make_workload("tiny", seed=seed, num_seqs=len(c["lens"]), lens=("fixed", c["lens"]),
                         num_q_heads=c["hq"], num_kv_heads=c["hkv"], block_size=c["bs"], dtype=c["dtype"],
                         pool_blocks=0)
    wl.poison()
    fused = c["fused"] and single_token_step(wl)
    kc, vc, out = gpu_step(wl, gpu, partition_size=c["P"], out_dtype=c["out_dtype"], fused=fused)
    okc, ovc, ref = oracle_step(wl)
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc), c
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all(), c
    ulp_half = {torch.float32: 0.0, torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}[c["out_dtype"]]
    err = np.abs(o - ref)
    assert (err <= TOL + ulp_half * np.abs(ref)).all(), (c, float(err.max()))
    assert pkv.check_device_error() == 0


def _guarded(n_elems, dtype, dev, guard=4096):
    """A buffer of n_elems between two guard bands of canary bytes; returns (full, view, band)."""
    elt = torch.tensor([], dtype=dtype).element_size()
    g = guard // elt
    full = torch.empty(n_elems + 2 * g, dtype=dtype, device=dev)
    full.view(torch.uint8).fill_(0xA5)
    return full, full[g:g + n_elems], g


def _guards_intact(full, g):
    b = full.view(torch.uint8)
    elt = full.element_size()
    return bool((b[:g * elt] == 0xA5).all()) and bool((b[-g * elt:] == 0xA5).all())


@pytest.mark.parametrize("P", [0, 64, 16])
def test_no_write_outside_buffers(gpu, P):
    dev = gpu
    wl = W.make_workload("llama8b", num_seqs=5, lens=("uniform", 100, 1400), seed=31)
    nb, hkv, bs, d = wl.k_cache.shape
    kfull, kc, kg = _guarded(wl.k_cache.size, torch.bfloat16, dev)
    vfull, vc, vg = _guarded(wl.v_cache.size, torch.bfloat16, dev)
    kc, vc = kc.view(nb, hkv, bs, d), vc.view(nb, hkv, bs, d)
    kc.copy_(to_dev(wl.k_cache, "bf16", dev))
    vc.copy_(to_dev(wl.v_cache, "bf16", dev))
    ofull, out, og = _guarded(wl.num_seqs * wl.num_q_heads * d, torch.float32, dev)
    out = out.view(wl.num_seqs, wl.num_q_heads, d)
    need = pkv.paged_attention_workspace_bytes(wl.num_seqs, wl.num_q_heads, d, wl.max_context_len, P)
    wfull, ws, wg = _guarded(max(need, 256), torch.uint8, dev)
    q = to_dev(wl.q, "bf16", dev)
    bt, cl = torch.from_numpy(wl.block_tables).to(dev), torch.from_numpy(wl.context_lens).to(dev)
    pkv.paged_attention_append_decode(q, to_dev(wl.new_k, "bf16", dev), to_dev(wl.new_v, "bf16", dev),
                                      torch.from_numpy(wl.slot_mapping).to(dev), kc, vc, bt, cl, wl.scale, out=out,
                                      max_context_len=wl.max_context_len, partition_size=P, workspace=ws)
    free = sorted(set(range(nb)) - set(wl.block_tables[wl.block_tables >= 0].tolist()))
    pairs = np.array([[wl.block_tables[0, 0], free[0]], [wl.block_tables[1, 0], free[1]]], dtype=np.int64)
    pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).to(dev))
    i = np.arange(40)
    src = wl.block_tables[2, i // bs].astype(np.int64) * bs + i % bs
    dst = np.asarray(free[2:2 + (40 + bs - 1) // bs], dtype=np.int64)[i // bs] * bs + i % bs
    pkv.compact_tokens(torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev), kc, vc)
    torch.cuda.synchronize()
    assert pkv.check_device_error() == 0
    for full, g in ((kfull, kg), (vfull, vg), (ofull, og), (wfull, wg)):
        assert _guards_intact(full, g)
    okc, ovc, ref = oracle_step(wl)
    assert oracle.copy_blocks(okc, ovc, pairs) == 0
    assert oracle.compact(okc, ovc, src, dst) == 0
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    assert max_abs_err(out, ref) <= TOL
