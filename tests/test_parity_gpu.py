"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.

Bar: bit-exact for append and copy_blocks (the whole pool is compared,
unused slots NaN-poisoned); max-abs error <= 5e-3 for attention outputs
stored as fp32 (fp32 accumulation of bf16/fp16 products), plus half an ulp of
the storage type when the output is stored as bf16/fp16.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_11_gb300 as pkv
from paged_kv_cache_11_gb300 import workload as W
from tests.step_helpers import gpu_step, max_abs_err, oracle_step, single_token_step, to_bits, to_dev

pytestmark = pytest.mark.gpu
TOL = 5e-3


def _check(wl, device, **kw):
    if not getattr(wl, "_poisoned", False):
        wl.poison()
        wl._poisoned = True
    kc, vc, out = gpu_step(wl, device, **kw)
    okc, ovc, ref = oracle_step(wl)
    assert np.array_equal(to_bits(kc), okc), "K pool differs after copy_blocks + append"
    assert np.array_equal(to_bits(vc), ovc), "V pool differs after copy_blocks + append"
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    err = max_abs_err(out, ref)
    assert err <= TOL, err
    return out, ref, err


# ------------------------------------------------------------------ workloads, reduced
def test_tiny_workload(gpu):
    _check(W.make_workload("tiny"), gpu)


@pytest.mark.parametrize("P", [0, 16, 64, 4096])
def test_llama8b_small(gpu, P):
    wl = W.make_workload("llama8b", num_seqs=6, lens=("uniform", 512, 2100))
    _check(wl, gpu, partition_size=P)


def test_opt13b_small(gpu):
    wl = W.make_workload("opt13b", num_seqs=8, lens=("uniform", 1, 700))
    _check(wl, gpu)


def test_shared_prefix_small(gpu):
    wl = W.make_workload("shared_prefix", groups=2, per_group=4, prefix=64, suffix=(32, 100))
    assert len(wl.cow_pairs) == 6
    _check(wl, gpu)


def test_long_context_small(gpu):
    wl = W.make_workload("llama70b_long", num_seqs=2, lens=("fixed", (3000, 1537)))
    _check(wl, gpu)


@pytest.mark.parametrize("fused", [False, True])
def test_many_short_sequences(gpu, fused):
    """6000 sequences of 0-70 tokens: a grid with thousands of sequence rows,
    mostly one or two blocks each, through the separate and the fused step."""
    wl = W.make_workload("llama8b", num_seqs=6000, lens=("uniform", 0, 70), seed=31)
    assert (wl.context_lens == 0).any() and wl.max_context_len <= 70
    if fused:
        assert single_token_step(wl) is False  # empty sequences append nothing
        live = wl.context_lens > 0
        slots = np.full(wl.num_seqs, -1, dtype=np.int64)
        slots[wl.append_seq] = wl.slot_mapping
        nk = np.zeros((wl.num_seqs,) + wl.new_k.shape[1:], dtype=wl.new_k.dtype)
        nv = np.zeros_like(nk)
        nk[wl.append_seq], nv[wl.append_seq] = wl.new_k, wl.new_v
        assert live.sum() == len(wl.slot_mapping)
        wl.slot_mapping, wl.new_k, wl.new_v = slots, nk, nv
        wl.append_seq = np.arange(wl.num_seqs, dtype=np.int32)
    _check(wl, gpu, fused=fused)


@pytest.mark.parametrize("fused", [False, True])
def test_maximum_batch(gpu, fused):
    """65535 sequences, the most one call takes (one grid row each), of 1-16
    tokens with 4 query heads on one KV head, through the separate and the
    fused step."""
    wl = W.make_workload("tiny", num_seqs=65535, lens=("uniform", 1, 16), num_q_heads=4, num_kv_heads=1,
                         pool_blocks=0, seed=37)
    assert single_token_step(wl) and wl.max_context_len == 16
    _check(wl, gpu, fused=fused)


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("lens", [(0, 1, 16, 17), (1,), (32, 31, 33, 2)])
@pytest.mark.parametrize("bs", [16, 32])
def test_short_and_boundary_lengths(gpu, lens, bs):
    wl = W.make_workload("tiny", num_seqs=len(lens), lens=("fixed", lens), block_size=bs)
    _check(wl, gpu)


@pytest.mark.parametrize("hq,hkv", [(16, 1), (32, 1), (24, 3), (8, 8), (12, 2)])
def test_gqa_groups(gpu, hq, hkv):
    wl = W.make_workload("tiny", num_seqs=3, lens=("fixed", (40, 700, 5)), num_q_heads=hq, num_kv_heads=hkv,
                         pool_blocks=0)
    _check(wl, gpu)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_low_precision_output(gpu, out_dtype):
    wl = W.make_workload("llama8b", num_seqs=4, lens=("uniform", 1, 1500))
    wl.poison()
    _, _, out = gpu_step(wl, gpu, out_dtype=out_dtype)
    _, _, ref = oracle_step(wl)
    ulp_half = 2.0 ** -8 if out_dtype == torch.bfloat16 else 2.0 ** -11
    err = np.abs(out.float().cpu().numpy() - ref)
    assert (err <= TOL + ulp_half * np.abs(ref)).all(), err.max()


def test_length_one_returns_v_bitwise(gpu):
    wl = W.make_workload("tiny", num_seqs=4, lens=("fixed", (1, 1, 1, 1)))
    _, vc, out = gpu_step(wl, gpu)
    for s in range(4):
        slot = int(wl.slot_mapping[s])
        v = vc[slot // 16, 0, slot % 16].float()
        for h in range(4):
            assert torch.equal(out[s, h], v)


def test_identical_keys_give_mean_of_v(gpu):
    wl = W.make_workload("tiny", num_seqs=2, lens=("fixed", (37, 300)), pool_blocks=0)
    wl.k_cache[:] = wl.k_cache[0, 0, 0]
    wl.new_k[:] = wl.k_cache[0, 0, 0]
    _, vc, out = gpu_step(wl, gpu)
    vbits = to_bits(vc)
    for s in range(2):
        L = int(wl.context_lens[s])
        rows = [vbits[wl.block_tables[s, t // 16], 0, t % 16] for t in range(L)]
        mean = oracle.to_f64(np.stack(rows), "bf16").mean(axis=0)
        assert np.abs(out[s].float().cpu().numpy() - mean).max() <= TOL


def test_physical_permutation_is_bitwise_invisible(gpu):
    a = W.make_workload("llama8b", num_seqs=5, lens=("uniform", 100, 1300), seed=77)
    b = W.make_workload("llama8b", num_seqs=5, lens=("uniform", 100, 1300), seed=77)
    perm = np.random.default_rng(0).permutation(b.num_blocks)
    # same logical contents, different physical placement
    b.k_cache = np.empty_like(a.k_cache)
    b.v_cache = np.empty_like(a.v_cache)
    b.k_cache[perm] = a.k_cache
    b.v_cache[perm] = a.v_cache
    b.block_tables = np.where(a.block_tables >= 0, perm[np.maximum(a.block_tables, 0)], -1).astype(np.int32)
    bs = 16
    b.slot_mapping = perm[a.slot_mapping // bs] * bs + a.slot_mapping % bs
    _, _, oa = gpu_step(a, gpu)
    _, _, ob = gpu_step(b, gpu)
    assert torch.equal(oa, ob)
    _, _, oa = gpu_step(a, gpu, partition_size=32)
    _, _, ob = gpu_step(b, gpu, partition_size=32)
    assert torch.equal(oa, ob)


def test_more_partitions_than_one_grid_dimension(gpu):
    """65600 one-block partitions, more than one grid dimension holds.  The
    sequence's block table repeats the same 64 blocks 1025 times, and a
    softmax over tokens that each appear n times is the softmax over one copy,
    so the 1,049,600-token result is the oracle's over the first 1024 tokens."""
    wl = W.make_workload("tiny", num_seqs=1, lens=("fixed", (1024,)), pool_blocks=64, seed=21)
    reps = 1025
    L = 1024 * reps
    bt = np.tile(wl.block_tables[:, :64], (1, reps)).astype(np.int32)
    ref, status = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, wl.dtype)
    assert not status.any()
    kc, vc, q = to_dev(wl.k_cache, wl.dtype, gpu), to_dev(wl.v_cache, wl.dtype, gpu), to_dev(wl.q, wl.dtype, gpu)
    out = pkv.paged_attention_decode(q, kc, vc, torch.from_numpy(bt).to(gpu),
                                     torch.tensor([L], dtype=torch.int32, device=gpu), wl.scale,
                                     max_context_len=L, partition_size=16)
    assert pkv.check_device_error() == 0
    assert max_abs_err(out, ref) <= TOL


def test_split_k_matches_single_pass(gpu):
    wl = W.make_workload("llama70b_long", num_seqs=2, lens=("fixed", (5000, 2600)))
    _, _, single = gpu_step(wl, gpu, partition_size=5024)
    for P in (32, 512, 1024):
        _, _, split = gpu_step(wl, gpu, partition_size=P)
        assert (split - single).abs().max().item() <= 1e-5


@pytest.mark.parametrize("P", [0, 64])  # fused merge / separate merge kernel
def test_workspace_reuse_and_garbage(gpu, P):
    """One workspace reused across calls and pre-filled with garbage gives the same bits."""
    import paged_kv_cache_11_gb300 as pkv
    wl = W.make_workload("llama8b", num_seqs=7, lens=("uniform", 300, 2500), seed=3)
    dev = gpu
    kc, vc, q = to_dev(wl.k_cache, "bf16", dev), to_dev(wl.v_cache, "bf16", dev), to_dev(wl.q, "bf16", dev)
    bt, cl = torch.from_numpy(wl.block_tables).to(dev), torch.from_numpy(wl.context_lens).to(dev)
    mcl = wl.max_context_len
    need = pkv.paged_attention_workspace_bytes(wl.num_seqs, wl.num_q_heads, 128, mcl, P)
    assert need > 0
    outs = []
    for fill in (0x00, 0xFF, 0x5A, None, None):
        ws = torch.empty(need, dtype=torch.uint8, device=dev) if fill is not None or not outs else ws
        if fill is not None:
            ws.fill_(fill)
        outs.append(pkv.paged_attention_decode(q, kc, vc, bt, cl, wl.scale, max_context_len=mcl, partition_size=P,
                                               workspace=ws).clone())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    ref, _ = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, "bf16",
                           threads=8)
    assert max_abs_err(outs[0], ref) <= TOL


def test_shared_blocks_equal_copied_blocks(gpu):
    """Sequences mapping the group's shared prefix == the same sequences with private copies."""
    wl = W.make_workload("shared_prefix", groups=1, per_group=3, prefix=64, suffix=(32, 60), pool_blocks=64)
    _, _, shared = gpu_step(wl, gpu)
    # give sequences 1 and 2 private copies of the 4 shared prefix blocks
    free = sorted(set(range(wl.num_blocks)) - set(wl.block_tables[wl.block_tables >= 0].tolist()))
    assert len(free) >= 8
    bt = wl.block_tables.copy()
    k, v = wl.k_cache.copy(), wl.v_cache.copy()
    for s in (1, 2):
        for j in range(4):
            dst = free.pop()
            k[dst], v[dst] = k[bt[s, j]], v[bt[s, j]]
            bt[s, j] = dst
    wl.block_tables, wl.k_cache, wl.v_cache = bt, k, v
    _, _, copied = gpu_step(wl, gpu)
    assert torch.equal(shared, copied)


# ------------------------------------------------------------------ fused block write + decode
@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("llama8b", dict(num_seqs=6, lens=("uniform", 512, 2100))),
    ("opt13b", dict(num_seqs=9, lens=("uniform", 1, 700))),
    ("llama70b_long", dict(num_seqs=2, lens=("fixed", (3000, 1537)))),
    ("tiny", dict(num_seqs=5, lens=("fixed", (1, 16, 17, 32, 33)), num_q_heads=32, num_kv_heads=2, pool_blocks=0)),
])
@pytest.mark.parametrize("P", [0, 64])
def test_fused_append_decode(gpu, name, kw, P):
    wl = W.make_workload(name, **kw)
    assert single_token_step(wl)
    _check(wl, gpu, fused=True, partition_size=P)
    # bit-identical to the separate block write + decode
    kc1, vc1, o1 = gpu_step(wl, gpu, partition_size=P)
    kc2, vc2, o2 = gpu_step(wl, gpu, partition_size=P, fused=True)
    assert torch.equal(o1, o2)
    # the pools hold NaN poison, so compare bit patterns
    assert np.array_equal(to_bits(kc1), to_bits(kc2)) and np.array_equal(to_bits(vc1), to_bits(vc2))


def test_fused_append_rejects_a_slot_that_is_not_the_last_position(gpu):
    import paged_kv_cache_11_gb300 as pkv
    pkv.check_device_error()
    wl = W.make_workload("llama8b", num_seqs=3, lens=("fixed", (40, 300, 17)))
    wl.slot_mapping = wl.slot_mapping.copy()
    wl.slot_mapping[1] -= 1                      # the position before the last one
    kc, vc, _ = gpu_step(wl, gpu, fused=True)
    assert pkv.check_device_error() == 1
    kbits = to_bits(kc)
    wrong = int(wl.slot_mapping[1])
    assert np.array_equal(kbits[wrong // 16, :, wrong % 16], wl.k_cache[wrong // 16, :, wrong % 16])  # untouched


# ------------------------------------------------------------------ errors
def test_bad_metadata_is_reported_and_zeroed(gpu):
    import paged_kv_cache_11_gb300 as pkv
    pkv.check_device_error()
    wl = W.make_workload("llama8b", num_seqs=3, lens=("fixed", (300, 900, 100)))
    dev = gpu
    kc, vc = to_dev(wl.k_cache, "bf16", dev), to_dev(wl.v_cache, "bf16", dev)
    q = to_dev(wl.q, "bf16", dev)
    bt = wl.block_tables.copy()
    bt[1, 3] = wl.num_blocks + 5
    cl = torch.from_numpy(wl.context_lens).to(dev)
    for P in (0, 64):
        out = pkv.paged_attention_decode(q, kc, vc, torch.from_numpy(bt).to(dev), cl, wl.scale,
                                         max_context_len=wl.max_context_len, partition_size=P)
        assert pkv.check_device_error() == 4
        assert not out[1].any() and out[0].any() and out[2].any()
    bad_len = wl.context_lens.copy()
    bad_len[2] = wl.max_context_len + 1
    out = pkv.paged_attention_decode(q, kc, vc, torch.from_numpy(wl.block_tables).to(dev),
                                     torch.from_numpy(bad_len).to(dev), wl.scale, max_context_len=wl.max_context_len)
    assert pkv.check_device_error() == 3
    assert not out[2].any() and out[0].any()
    assert pkv.check_device_error() == 0  # cleared
    # append with a slot outside the pool
    slots = torch.tensor([0, wl.num_blocks * 16], dtype=torch.int64, device=dev)
    kv = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device=dev)
    pkv.paged_kv_append(kv, kv, slots, kc, vc)
    assert pkv.check_device_error() == 1
    pkv.copy_blocks(kc, vc, torch.tensor([[0, wl.num_blocks]], dtype=torch.int64, device=dev))
    assert pkv.check_device_error() == 2


def test_host_checks(gpu):
    import paged_kv_cache_11_gb300 as pkv
    from paged_kv_cache_11_gb300.binding import (PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE,
                                                 PagedKVError)
    wl = W.make_workload("tiny")
    dev = gpu
    kc, vc = to_dev(wl.k_cache, "bf16", dev), to_dev(wl.v_cache, "bf16", dev)
    q = to_dev(wl.q, "bf16", dev)
    bt, cl = torch.from_numpy(wl.block_tables).to(dev), torch.from_numpy(wl.context_lens).to(dev)
    ws = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(PagedKVError) as e:
        pkv.paged_attention_decode(q, kc, vc, bt, cl, wl.scale, max_context_len=100, partition_size=32, workspace=ws)
    assert e.value.status == PKV_ERR_WORKSPACE
    with pytest.raises(PagedKVError) as e:
        pkv.paged_attention_decode(q[:, :, :64].contiguous(), kc[..., :64].contiguous(), vc[..., :64].contiguous(),
                                   bt, cl, wl.scale)
    assert e.value.status == PKV_ERR_UNSUPPORTED
    # zero sequences: a no-op
    pkv.paged_attention_decode(q[:0], kc, vc, bt[:0], cl[:0], wl.scale)
    assert pkv.check_device_error() == 0
    # more sequences than one call takes: refused before any launch (only the
    # shapes are read, so the tensors are never touched)
    n = 65536
    qn = torch.empty((n, wl.num_q_heads, 128), dtype=torch.bfloat16, device=dev)
    btn = torch.zeros((n, wl.block_tables.shape[1]), dtype=torch.int32, device=dev)
    cln = torch.zeros(n, dtype=torch.int32, device=dev)
    launches = pkv.launch_count()
    with pytest.raises(PagedKVError) as e:
        pkv.paged_attention_decode(qn, kc, vc, btn, cln, wl.scale, max_context_len=100)
    assert e.value.status == PKV_ERR_INVALID_ARG and pkv.launch_count() == launches


# ------------------------------------------------------------------ full sizes, sampled outputs
def _sample(wl, n, seed=0):
    rng = np.random.default_rng(seed)
    s = rng.integers(0, wl.num_seqs, n)
    h = rng.integers(0, wl.num_q_heads, n)
    pairs = sorted(set(zip(s.tolist(), h.tolist())))
    # always include the longest and the shortest sequence
    for s0 in (int(np.argmax(wl.context_lens)), int(np.argmin(wl.context_lens))):
        pairs.append((s0, 0))
        pairs.append((s0, wl.num_q_heads - 1))
    return sorted(set(pairs))


@pytest.mark.slow
@pytest.mark.parametrize("name,nsample,fused", [
    ("llama8b", 48, False), ("llama8b", 48, True), ("opt13b", 48, False), ("opt13b", 48, True),
    ("shared_prefix", 48, False), ("shared_prefix_prefill", 48, False),
    ("llama70b_long", 6, False), ("llama70b_long", 6, True)])
def test_full_size_sampled(gpu, name, nsample, fused):
    """The full-size workloads with the automatic partition; fused: the single
    block-write + decode launch the benchmark times for one-token steps."""
    wl = W.make_workload(name)
    if fused:
        # the benchmark's partition choice for these shapes on one GB300
        want = {"llama8b": 1024, "opt13b": 4096, "llama70b_long": 4096}[name]
        if torch.cuda.get_device_properties(gpu).multi_processor_count == 152:
            assert pkv.paged_attention_partition_size(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads,
                                                      wl.max_context_len) == want
    kc, vc, out = gpu_step(wl, gpu, fused=fused)
    sel = _sample(wl, nsample)
    okc, ovc, ref = oracle_step(wl, select=sel, in_place=True)
    # the step's writes, bit-exact; the rest of the pool untouched
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    err = max_abs_err(out, ref, select=sel)
    assert err <= TOL, err
    o = out.float()
    assert torch.isfinite(o).all()


@pytest.mark.slow
def test_llama70b_long_at_512_token_partitions(gpu):
    """llama70b_long at the split named for that workload, 512-token
    partitions (256 per row, merged by the merge kernel), through the fused
    step; the automatic choice above takes 4096."""
    wl = W.make_workload("llama70b_long")
    assert pkv.paged_attention_plan(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.block_size,
                                    wl.max_context_len, 512) == "split+reduce"
    kc, vc, out = gpu_step(wl, gpu, fused=True, partition_size=512)
    sel = _sample(wl, 6, seed=1)
    okc, ovc, ref = oracle_step(wl, select=sel, in_place=True)
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    err = max_abs_err(out, ref, select=sel)
    assert err <= TOL, err
    assert torch.isfinite(out).all()


# ------------------------------------------------------------------ graph capture
@pytest.mark.parametrize("P", [0, 64])  # merge in the decode kernel / merge kernel
def test_decode_step_captured_in_a_cuda_graph(gpu, P):
    """A fused decode step captured once and replayed: each replay gives the direct call's bits
    (the split-K arrival counters are reset by their last arrival, so a replayed epoch starts clean)."""
    import paged_kv_cache_11_gb300 as pkv
    wl = W.make_workload("llama8b", num_seqs=16, lens=("uniform", 300, 2000), seed=12)
    dev = gpu
    kc, vc, q = to_dev(wl.k_cache, "bf16", dev), to_dev(wl.v_cache, "bf16", dev), to_dev(wl.q, "bf16", dev)
    nk, nv = to_dev(wl.new_k, "bf16", dev), to_dev(wl.new_v, "bf16", dev)
    sm = torch.from_numpy(wl.slot_mapping).to(dev)
    bt, cl = torch.from_numpy(wl.block_tables).to(dev), torch.from_numpy(wl.context_lens).to(dev)
    mcl = wl.max_context_len
    need = pkv.paged_attention_workspace_bytes(wl.num_seqs, wl.num_q_heads, 128, mcl, P)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((wl.num_seqs, wl.num_q_heads, 128), device=dev)
    step = lambda: pkv.paged_attention_append_decode(q, nk, nv, sm, kc, vc, bt, cl, wl.scale, out=out,
                                                     max_context_len=mcl, partition_size=P, workspace=ws)
    step()
    torch.cuda.synchronize()
    ref = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm the stream before capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(5):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert pkv.check_device_error() == 0
