"""paged_attention_decode_static: the decode entry point for callers that
cannot allocate device memory (their device memory is all owned by another
allocator, or they must not call cudaMalloc in a latency-critical loop).

It is called here through the C ABI, twice in a row, and compared with
paged_attention_decode given a caller-allocated workspace, within the
attention tolerance the parity tests use.  The file sorts last so that a
failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_11_gb300 import binding
from paged_kv_cache_11_gb300 import workload as W
from tests.step_helpers import to_dev

pytestmark = pytest.mark.gpu
TOL = 5e-3


def _static_fn():
    lib = binding._lib()
    fn = lib.paged_attention_decode_static
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, ctypes.c_float, vp, i32, ctypes.POINTER(binding.CacheDesc),
                   i32, vp]
    fn.restype = ctypes.c_int
    return fn


def test_static_workspace_decode_matches_workspace_decode(gpu):
    wl = W.make_workload("llama8b", num_seqs=6, lens=("uniform", 600, 3000), seed=5)
    dev = gpu
    kc, vc, q = to_dev(wl.k_cache, "bf16", dev), to_dev(wl.v_cache, "bf16", dev), to_dev(wl.q, "bf16", dev)
    bt = torch.from_numpy(wl.block_tables).to(dev)
    cl = torch.from_numpy(wl.context_lens).to(dev)
    mcl = wl.max_context_len
    P = 512  # several partitions per sequence: the partials go through the workspace
    assert binding.paged_attention_workspace_bytes(wl.num_seqs, wl.num_q_heads, 128, mcl, P) > 0
    ref = binding.paged_attention_decode(q, kc, vc, bt, cl, wl.scale, max_context_len=mcl, partition_size=P)
    fn = _static_fn()
    desc = binding.cache_desc(kc)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # two calls in a row share the static array
        out = torch.full_like(ref, float("nan"))
        st = fn(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.shape[1], cl.data_ptr(), wl.num_seqs,
                wl.num_q_heads, mcl, wl.scale, out.data_ptr(), binding.PKV_FP32, ctypes.byref(desc), P, stream)
        assert st == binding.PKV_OK, binding.status_string(st)
        torch.cuda.synchronize()
        assert binding.check_device_error() == 0
        assert (out - ref).abs().max().item() <= TOL


def test_static_workspace_rejects_oversized_calls(gpu):
    fn = _static_fn()
    desc = binding.CacheDesc(32768, 8, 32, 128, binding.PKV_BF16)
    # 64 sequences x 64 heads x 256 partitions of partials: far beyond the 16 MiB array
    st = fn(256, 256, 256, 256, 4096, 256, 64, 64, 131072, 0.1, 256, binding.PKV_FP32, ctypes.byref(desc), 512, None)
    assert st == binding.PKV_ERR_WORKSPACE
