"""Run one decode step of a workload through the C ABI (GPU) and through the
oracle (CPU), on the same seeded inputs.

A step is: copy_blocks of the workload's copy-on-write pairs, then
paged_kv_append of the step's new tokens, then paged_attention_decode.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle

TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def case_seeds(n: int) -> range:
    """Seeds of a randomised sweep: n, or n times PKV_SOAK for a longer soak
    run (the first n cases are always the same)."""
    return range(n * max(1, int(os.environ.get("PKV_SOAK", "1"))))


def to_dev(bits: np.ndarray, dtype: str, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(TORCH_DT[dtype])


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def single_token_step(wl) -> bool:
    """True when the step appends exactly one token per sequence, at its last position."""
    return len(wl.cow_pairs) == 0 and np.array_equal(wl.append_seq, np.arange(wl.num_seqs))


def gpu_step(wl, device, partition_size: int = 0, out_dtype=torch.float32, max_context_len=None, fused=False):
    import paged_kv_cache_11_gb300 as pkv
    dt = wl.dtype
    kc = to_dev(wl.k_cache, dt, device)
    vc = to_dev(wl.v_cache, dt, device)
    q = to_dev(wl.q, dt, device)
    bt = torch.from_numpy(wl.block_tables).to(device)
    cl = torch.from_numpy(wl.context_lens).to(device)
    mcl = wl.max_context_len if max_context_len is None else max_context_len
    if fused:
        assert single_token_step(wl)
        out = pkv.paged_attention_append_decode(q, to_dev(wl.new_k, dt, device), to_dev(wl.new_v, dt, device),
                                                torch.from_numpy(wl.slot_mapping).to(device), kc, vc, bt, cl,
                                                wl.scale, max_context_len=mcl, partition_size=partition_size,
                                                out_dtype=out_dtype)
        torch.cuda.synchronize()
        return kc, vc, out
    if len(wl.cow_pairs):
        pkv.copy_blocks(kc, vc, torch.from_numpy(wl.cow_pairs).to(device))
    if len(wl.slot_mapping):
        pkv.paged_kv_append(to_dev(wl.new_k, dt, device), to_dev(wl.new_v, dt, device),
                            torch.from_numpy(wl.slot_mapping).to(device), kc, vc)
    out = pkv.paged_attention_decode(q, kc, vc, bt, cl, wl.scale, max_context_len=mcl,
                                     partition_size=partition_size, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return kc, vc, out


def oracle_step(wl, select=None, threads: int = 8, in_place: bool = False):
    """Apply copy + append to (copies of) the host pools, then decode."""
    kc = wl.k_cache if in_place else wl.k_cache.copy()
    vc = wl.v_cache if in_place else wl.v_cache.copy()
    if len(wl.cow_pairs):
        assert oracle.copy_blocks(kc, vc, wl.cow_pairs) == 0
    if len(wl.slot_mapping):
        assert oracle.append(wl.new_k, wl.new_v, wl.slot_mapping, kc, vc) == 0
    out, status = oracle.decode(wl.q, kc, vc, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                                select=select, threads=threads)
    assert not status.any()
    return kc, vc, out


def max_abs_err(got: torch.Tensor, ref: np.ndarray, select=None) -> float:
    g = got.float().cpu().numpy().astype(np.float64)
    if select is not None:
        idx = tuple(np.asarray(select).T)
        return float(np.abs(g[idx] - ref[idx]).max())
    return float(np.abs(g - ref).max())
