"""paged_attention_decode_static: the decode entry point for callers that
cannot allocate device memory (their device memory is all owned by another
allocator, or they must not call cudaMalloc in a latency-critical loop).

It is called here through the C ABI, twice in a row per case, and must give
the same bits as paged_attention_decode given a caller-allocated workspace at
the same partition size (the same kernels run; only where the partials live
differs), and match the fp64 oracle within the attention tolerance the parity
tests use.  The cases take the three ways partials are merged: inside the
decode kernel (a few partitions), with the automatic partition choice, and by
the separate merge kernel (more than 16 partitions).  The device's free
memory must not change across the calls.  The file sorts last so that a
failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_11_gb300 import binding
from paged_kv_cache_11_gb300 import workload as W
from tests.step_helpers import max_abs_err, to_dev

pytestmark = pytest.mark.gpu
TOL = 5e-3
STATIC_BYTES = 16 << 20  # the library's fixed array

CASES = [
    # (workload overrides, partition size)
    (dict(num_seqs=6, lens=("uniform", 600, 3000), seed=5), 512),    # <= 16 partitions: merged in the kernel
    (dict(num_seqs=6, lens=("uniform", 600, 3000), seed=5), 0),      # automatic partition
    (dict(num_seqs=2, lens=("fixed", (8192, 5000)), seed=6), 256),   # 32 partitions: the merge kernel
]


def _static_fn():
    lib = binding._lib()
    fn = lib.paged_attention_decode_static
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, ctypes.c_float, vp, i32, ctypes.POINTER(binding.CacheDesc),
                   i32, vp]
    fn.restype = ctypes.c_int
    return fn


def test_static_workspace_decode_matches_workspace_decode(gpu):
    dev = gpu
    fn = _static_fn()
    stream = torch.cuda.current_stream().cuda_stream
    runs = []
    for kw, P in CASES:
        wl = W.make_workload("llama8b", **kw)
        kc, vc, q = to_dev(wl.k_cache, "bf16", dev), to_dev(wl.v_cache, "bf16", dev), to_dev(wl.q, "bf16", dev)
        bt = torch.from_numpy(wl.block_tables).to(dev)
        cl = torch.from_numpy(wl.context_lens).to(dev)
        mcl = wl.max_context_len
        need = binding.paged_attention_workspace_bytes(wl.num_seqs, wl.num_q_heads, 128, mcl, P)
        assert 0 < need <= STATIC_BYTES  # the partials go through the workspace, and fit the array
        ref = binding.paged_attention_decode(q, kc, vc, bt, cl, wl.scale, max_context_len=mcl, partition_size=P)
        outs = [torch.full_like(ref, float("nan")) for _ in range(3)]
        desc = binding.cache_desc(kc)

        def call(out, wl=wl, kc=kc, vc=vc, q=q, bt=bt, cl=cl, mcl=mcl, P=P, desc=desc):
            st = fn(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.shape[1], cl.data_ptr(),
                    wl.num_seqs, wl.num_q_heads, mcl, wl.scale, out.data_ptr(), binding.PKV_FP32, ctypes.byref(desc),
                    P, stream)
            assert st == binding.PKV_OK, binding.status_string(st)

        call(outs[0])  # warm-up: the first call on the device finds the array; kernels load on first use
        torch.cuda.synchronize()
        assert binding.check_device_error() == 0
        runs.append((wl, ref, outs, call))

    free0 = torch.cuda.mem_get_info(dev)[0]
    alloc0 = torch.cuda.memory_allocated(dev)
    for wl, ref, outs, call in runs:
        for out in outs[1:]:  # two calls in a row share the static array
            call(out)
            torch.cuda.synchronize()
            assert binding.check_device_error() == 0
            assert torch.equal(out, ref)
    assert torch.cuda.mem_get_info(dev)[0] == free0, "the static entry point allocated device memory"
    assert torch.cuda.memory_allocated(dev) == alloc0

    for wl, ref, outs, _ in runs:
        want, status = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale,
                                     wl.dtype, threads=8)
        assert not status.any()
        assert max_abs_err(outs[-1], want) <= TOL


def test_static_workspace_rejects_oversized_calls(gpu):
    # 64 sequences x 64 heads x 256 partitions of partials: far beyond the 16 MiB array
    assert binding.paged_attention_workspace_bytes(64, 64, 128, 131072, 512) > STATIC_BYTES
    fn = _static_fn()
    desc = binding.CacheDesc(32768, 8, 32, 128, binding.PKV_BF16)
    # q and out are null: if the size check ever stopped rejecting this call,
    # the argument checks after it would, before anything is launched
    st = fn(None, 256, 256, 256, 4096, 256, 64, 64, 131072, 0.1, None, binding.PKV_FP32, ctypes.byref(desc), 512,
            None)
    assert st == binding.PKV_ERR_WORKSPACE
