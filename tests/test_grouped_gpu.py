"""Grouped decode (paged_attention_decode_grouped) against the fp64 oracle.

Sequences forked from one prompt share its blocks; grouped decode reads the
shared blocks once per (group, KV head) for all members and merges with each
member's own tokens.  Its result must be plain decode's: the oracle (which
knows nothing of groups) is the reference, pools must be untouched, and the
plain GPU kernel must agree to within accumulation-order differences.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_11_gb300 as pkv
from paged_kv_cache_11_gb300 import workload as W
from tests.step_helpers import case_seeds, max_abs_err, oracle_step, to_bits, to_dev

pytestmark = pytest.mark.gpu
TOL = 5e-3
PREFIX_LEN, GROUP = 6, 7  # PKV_DEVERR_PREFIX_LEN, PKV_DEVERR_GROUP


def _dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_grouped(wl, gs, pl, mg, dev, kc=None, vc=None, partition_size=0, out_dtype=torch.float32, workspace=None,
                max_prefix_len=None, out=None):
    dt = wl.dtype
    kc = to_dev(wl.k_cache, dt, dev) if kc is None else kc
    vc = to_dev(wl.v_cache, dt, dev) if vc is None else vc
    mpl = int(pl.max()) if max_prefix_len is None and len(pl) else (max_prefix_len or 0)
    out = pkv.paged_attention_decode_grouped(
        to_dev(wl.q, dt, dev), kc, vc, _dev(wl.block_tables, dev), _dev(wl.context_lens, dev), _dev(gs, dev),
        _dev(pl, dev), wl.scale, max_group_size=mg, max_prefix_len=mpl, max_context_len=wl.max_context_len,
        partition_size=partition_size, out_dtype=out_dtype, workspace=workspace, out=out)
    torch.cuda.synchronize()
    return kc, vc, out


def oracle_out(wl):
    out, status = oracle.decode(wl.q, wl.k_cache, wl.v_cache, wl.block_tables, wl.context_lens, wl.scale, wl.dtype,
                                threads=8)
    assert not status.any()
    return out


def _tol(out_dtype, ref):
    half_ulp = {torch.float32: 0.0, torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}[out_dtype]
    return TOL + half_ulp * np.abs(ref)


# ------------------------------------------------------------------ the shared-prefix decode step
@pytest.mark.parametrize("bs,step", [(16, "decode"), (16, "continuation"), (32, "decode"), (32, "continuation")])
def test_shared_prefix_step(gpu, bs, step):
    """Forked samples of 4 prompts: CoW copy + append (one token per sample, or
    each sample's whole continuation), then grouped decode."""
    wl = W.make_workload("shared_prefix", groups=4, per_group=16, prefix=512, suffix=(32, 300), seed=21,
                         block_size=bs, step=step)
    wl.poison()
    dev, dt = gpu, wl.dtype
    kc, vc = to_dev(wl.k_cache, dt, dev), to_dev(wl.v_cache, dt, dev)
    pkv.copy_blocks(kc, vc, _dev(wl.cow_pairs, dev))
    pkv.paged_kv_append(to_dev(wl.new_k, dt, dev), to_dev(wl.new_v, dt, dev), _dev(wl.slot_mapping, dev), kc, vc)
    gs, pl, mg = W.prefix_groups(wl)
    assert (pl[:] == 512).all() and mg == 16
    _, _, out = run_grouped(wl, gs, pl, mg, dev, kc=kc, vc=vc)
    okc, ovc, ref = oracle_step(wl)
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    assert max_abs_err(out, ref) <= TOL
    plain = pkv.paged_attention_decode(to_dev(wl.q, dt, dev), kc, vc, _dev(wl.block_tables, dev),
                                       _dev(wl.context_lens, dev), wl.scale, max_context_len=wl.max_context_len)
    torch.cuda.synchronize()
    assert float((plain - out).abs().max()) <= 2e-5
    assert pkv.check_device_error() == 0


def _grouped_step(wl, gs, pl, mg, dev, fused):
    """copy_blocks of the step's copy-on-write pairs, then either the grouped
    call with the block write inside it, or paged_kv_append + the grouped call."""
    dt = wl.dtype
    kc, vc = to_dev(wl.k_cache, dt, dev), to_dev(wl.v_cache, dt, dev)
    if len(wl.cow_pairs):
        pkv.copy_blocks(kc, vc, _dev(wl.cow_pairs, dev))
    nk, nv, sm = to_dev(wl.new_k, dt, dev), to_dev(wl.new_v, dt, dev), _dev(wl.slot_mapping, dev)
    if fused:
        out = pkv.paged_attention_append_decode_grouped(
            to_dev(wl.q, dt, dev), nk, nv, sm, kc, vc, _dev(wl.block_tables, dev), _dev(wl.context_lens, dev),
            _dev(gs, dev), _dev(pl, dev), wl.scale, max_group_size=mg, max_prefix_len=int(pl.max()),
            max_context_len=wl.max_context_len)
        torch.cuda.synchronize()
    else:
        pkv.paged_kv_append(nk, nv, sm, kc, vc)
        _, _, out = run_grouped(wl, gs, pl, mg, dev, kc=kc, vc=vc)
    return kc, vc, out


@pytest.mark.parametrize("bs", [16, 32])
def test_fused_grouped_step(gpu, bs):
    """The decode step of forked samples in two calls: the copy-on-write
    copies, then the grouped call with each sample's new-token write inside
    it.  Pools bit-exact against the oracle's copy + append, outputs within
    the tolerance, and the same bits as copy + append + grouped call."""
    wl = W.make_workload("shared_prefix", groups=4, per_group=16, prefix=512, suffix=(32, 300), seed=22,
                         block_size=bs)
    wl.poison()
    gs, pl, mg = W.prefix_groups(wl)
    kc, vc, out = _grouped_step(wl, gs, pl, mg, gpu, fused=True)
    assert pkv.check_device_error() == 0
    okc, ovc, ref = oracle_step(wl)
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    assert max_abs_err(out, ref) <= TOL
    _, _, sep = _grouped_step(wl, gs, pl, mg, gpu, fused=False)
    assert torch.equal(out, sep)
    assert pkv.check_device_error() == 0


def test_fused_grouped_rejects_a_slot_that_is_not_the_last_position(gpu):
    pkv.check_device_error()
    wl = W.make_workload("shared_prefix", groups=2, per_group=4, prefix=64, suffix=(32, 100), seed=23)
    s = next(i for i, L in enumerate(wl.context_lens) if (int(L) - 1) % 16 != 0)
    wl.slot_mapping = wl.slot_mapping.copy()
    wl.slot_mapping[s] -= 1  # the position before the last one, in the same block
    gs, pl, mg = W.prefix_groups(wl)
    kc, _, _ = _grouped_step(wl, gs, pl, mg, gpu, fused=True)
    assert pkv.check_device_error() == 1  # PKV_DEVERR_SLOT
    wrong = int(wl.slot_mapping[s])
    okc = wl.k_cache.copy()
    oracle.copy_blocks(okc, wl.v_cache.copy(), wl.cow_pairs)
    kbits = to_bits(kc)
    assert np.array_equal(kbits[wrong // 16, :, wrong % 16], okc[wrong // 16, :, wrong % 16])  # untouched


@pytest.mark.slow
@pytest.mark.parametrize("name,fused", [("shared_prefix", True), ("shared_prefix", False),
                                        ("shared_prefix_prefill", False)])
def test_full_size_step_sampled(gpu, name, fused):
    """The shared-prefix steps the benchmark times, at full size (16 groups x
    16 members, 1024-token prompt, 256 sequences): the 240 copy-on-write
    copies, the append (256 tokens, or the 68k-token continuation), then the
    grouped call with its automatic partitions.  The pools are compared bit
    for bit; outputs are sampled against the oracle (every group's first and
    last member, plus random rows)."""
    wl = W.make_workload(name)
    gs, pl, mg = W.prefix_groups(wl)
    assert len(gs) - 1 == 16 and mg == 16 and (pl >= 1024).all()
    kc, vc, out = _grouped_step(wl, gs, pl, mg, gpu, fused=fused)
    rng = np.random.default_rng(5)
    sel = {(int(s), int(h)) for s, h in zip(rng.integers(0, wl.num_seqs, 64), rng.integers(0, wl.num_q_heads, 64))}
    for g in range(len(gs) - 1):
        sel |= {(int(gs[g]), 0), (int(gs[g + 1]) - 1, wl.num_q_heads - 1)}
    sel = sorted(sel)
    okc, ovc, ref = oracle_step(wl, select=sel, in_place=True)
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    assert max_abs_err(out, ref, select=sel) <= TOL
    assert torch.isfinite(out).all()
    assert pkv.check_device_error() == 0


@pytest.mark.parametrize("bs,dtype", [(16, "bf16"), (32, "fp16")])
def test_prefix_running_max_raised(gpu, bs, dtype):
    """Scores that jump far above the running max in later 64-token chunks of
    the shared prefix: the prefix kernel raises its max and rescales the
    output accumulator in tensor memory twice, then accumulates a score just
    below the new max without a raise.  Every query is a multiple of one
    direction u; the shared K rows at prefix tokens 40, 170, 300 and 460 are
    multiples of u whose scores are about 16, 26, 36 and 37 in log2 units."""
    members = [[(512, 600), (512, 530), (512, 512), (256, 700)]]
    wl, gs, pl, mg = W.make_grouped_workload(21, members, 8, 2, bs, dtype)  # G = 4
    D = 128
    u = np.where(np.arange(D) % 3 == 0, 1.0, -1.0).astype(np.float32)
    lead = 0  # the group's first member holds the shared blocks in its table
    for t, c in ((40, 1.0), (170, 1.6), (300, 2.2), (460, 2.25)):
        pb = int(wl.block_tables[lead][t // bs])
        for kvh in range(wl.k_cache.shape[1]):
            wl.k_cache[pb, kvh, t % bs] = W.round_f32(c * u, dtype)
    wl.q[:] = W.round_f32(np.broadcast_to(u, wl.q.shape), dtype)
    wl.poison()
    kc, vc, out = run_grouped(wl, gs, pl, mg, gpu)
    ref = oracle_out(wl)
    assert max_abs_err(out, ref) <= TOL
    # the decode kernel's warp core raises its max the same way (plain decode)
    plain = pkv.paged_attention_decode(to_dev(wl.q, wl.dtype, gpu), kc, vc, _dev(wl.block_tables, gpu),
                                       _dev(wl.context_lens, gpu), wl.scale, max_context_len=wl.max_context_len)
    torch.cuda.synchronize()
    assert max_abs_err(plain, ref) <= TOL
    assert pkv.check_device_error() == 0


@pytest.mark.parametrize("groups", [16, 32])
def test_long_prefix_partitions(gpu, groups):
    """Enough groups for the call to take longer prefix partitions (on one
    GB300: 512 tokens for 16 groups of a 1024-token prompt over 8 KV heads,
    1024 tokens for 32 groups)."""
    wl = W.make_workload("shared_prefix", groups=groups, per_group=2, prefix=1024, suffix=(32, 200), seed=40 + groups)
    wl.poison()
    dev, dt = gpu, wl.dtype
    kc, vc = to_dev(wl.k_cache, dt, dev), to_dev(wl.v_cache, dt, dev)
    pkv.copy_blocks(kc, vc, _dev(wl.cow_pairs, dev))
    pkv.paged_kv_append(to_dev(wl.new_k, dt, dev), to_dev(wl.new_v, dt, dev), _dev(wl.slot_mapping, dev), kc, vc)
    gs, pl, mg = W.prefix_groups(wl)
    assert (pl[:] == 1024).all()
    _, _, out = run_grouped(wl, gs, pl, mg, dev, kc=kc, vc=vc)
    okc, ovc, ref = oracle_step(wl)
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    assert max_abs_err(out, ref) <= TOL
    plain = pkv.paged_attention_decode(to_dev(wl.q, dt, dev), kc, vc, _dev(wl.block_tables, dev),
                                       _dev(wl.context_lens, dev), wl.scale, max_context_len=wl.max_context_len)
    torch.cuda.synchronize()
    assert float((plain - out).abs().max()) <= 2e-5
    assert pkv.check_device_error() == 0


# ------------------------------------------------------------------ randomised groups
def _case(seed):
    rng = np.random.default_rng(seed)
    dtype = ["bf16", "fp16"][rng.integers(2)]
    bs = [16, 32][rng.integers(2)]
    hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 20, 32, 64]))
    if hkv * G > 256:
        hkv = max(1, 256 // G)
    members, total = [], 0
    for _ in range(int(rng.integers(1, 6))):
        n = int(rng.integers(1, 21))
        if total + n > 40:
            break
        top = bs * int(rng.integers(0, 2200 // bs))
        lead_L = top + (int(rng.integers(0, 700)) if rng.random() < 0.85 else 0)
        mem = [(top, lead_L)]
        for _ in range(n - 1):
            r = rng.random()
            p = top if r < 0.7 else bs * int(rng.integers(0, top // bs + 1))
            L = p + (int(rng.integers(0, 700)) if rng.random() < 0.85 else 0)
            mem.append((p, L))
        members.append(mem)
        total += n
    if rng.random() < 0.3:
        members.append([(0, 0)])                   # an empty sequence of its own
    P = [0, 0, 0, 16, 64, 512][rng.integers(6)] // bs * bs
    out_dtype = [torch.float32, torch.float32, torch.bfloat16, torch.float16][rng.integers(4)]
    return dict(dtype=dtype, bs=bs, hkv=hkv, G=G, members=members, P=P, out_dtype=out_dtype)


@pytest.mark.parametrize("seed", case_seeds(24))
def test_random_groups(gpu, seed):
    c = _case(500 + seed)
    wl, gs, pl, mg = W.make_grouped_workload(seed, c["members"], c["hkv"] * c["G"], c["hkv"], c["bs"], c["dtype"])
    wl.poison()
    kc, vc, out = run_grouped(wl, gs, pl, mg, gpu, partition_size=c["P"], out_dtype=c["out_dtype"])
    assert np.array_equal(to_bits(kc), wl.k_cache) and np.array_equal(to_bits(vc), wl.v_cache)
    ref = oracle_out(wl)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all(), c
    err = np.abs(o - ref)
    assert (err <= _tol(c["out_dtype"], ref)).all(), (c, float(err.max()))
    assert pkv.check_device_error() == 0
    if c["out_dtype"] == torch.float32:
        plain = pkv.paged_attention_decode(to_dev(wl.q, wl.dtype, gpu), kc, vc, _dev(wl.block_tables, gpu),
                                           _dev(wl.context_lens, gpu), wl.scale, max_context_len=wl.max_context_len)
        torch.cuda.synchronize()
        assert float((plain - out).abs().max()) <= 2e-5


@pytest.mark.parametrize("seed", case_seeds(12))
def test_random_groups_fused_write(gpu, seed):
    """The random group layouts as a decode step: every sequence whose last
    position lies past its shared prefix writes its new token there inside
    the grouped call (the others have no new token this step)."""
    c = _case(700 + seed)
    wl, gs, pl, mg = W.make_grouped_workload(seed, c["members"], c["hkv"] * c["G"], c["hkv"], c["bs"], c["dtype"])
    bs = c["bs"]
    slots = np.full(wl.num_seqs, -1, dtype=np.int64)
    for s in range(wl.num_seqs):
        L = int(wl.context_lens[s])
        if L > int(pl[s]):
            slots[s] = int(wl.block_tables[s, (L - 1) // bs]) * bs + (L - 1) % bs
    wl.slot_mapping = slots
    wl.append_seq = np.arange(wl.num_seqs, dtype=np.int32)
    wl.new_k = W.normal(seed, W.S_NEW_K, (wl.num_seqs, c["hkv"], 128), c["dtype"])
    wl.new_v = W.normal(seed, W.S_NEW_V, (wl.num_seqs, c["hkv"], 128), c["dtype"])
    wl.poison()
    dev, dt = gpu, wl.dtype
    kc, vc = to_dev(wl.k_cache, dt, dev), to_dev(wl.v_cache, dt, dev)
    out = pkv.paged_attention_append_decode_grouped(
        to_dev(wl.q, dt, dev), to_dev(wl.new_k, dt, dev), to_dev(wl.new_v, dt, dev), _dev(slots, dev), kc, vc,
        _dev(wl.block_tables, dev), _dev(wl.context_lens, dev), _dev(gs, dev), _dev(pl, dev), wl.scale,
        max_group_size=mg, max_prefix_len=int(pl.max()), max_context_len=wl.max_context_len,
        partition_size=c["P"], out_dtype=c["out_dtype"])
    torch.cuda.synchronize()
    assert pkv.check_device_error() == 0
    okc, ovc, ref = oracle_step(wl)
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all(), c
    err = np.abs(o - ref)
    assert (err <= _tol(c["out_dtype"], ref)).all(), (c, float(err.max()))


def test_many_prefix_partitions_use_the_merge_kernel(gpu):
    """17 prefix partitions + the own tokens: more than the in-kernel merge takes."""
    wl, gs, pl, mg = W.make_grouped_workload(7, [[(4352, 4400), (4352, 4500), (4096, 4097)], [(0, 900)]], 16, 4, 16,
                                             "bf16")
    wl.poison()
    _, _, out = run_grouped(wl, gs, pl, mg, gpu)
    assert max_abs_err(out, oracle_out(wl)) <= TOL
    assert pkv.check_device_error() == 0


@pytest.mark.parametrize("G,members", [
    (64, [[(256, 300), (256, 256), (128, 600)]]),           # one member per row tile
    (3, [[(512, 700)] + [(512, 520 + 7 * i) for i in range(24)]]),  # 21 members per tile, two tiles
    (4, [[(256, 256), (256, 256)], [(512, 512)]]),         # no own tokens at all
    (8, [[(0, 40), (0, 50)], [(16, 16)]]),                 # prefix 0 in a group; a group of one
])
def test_group_shapes(gpu, G, members):
    wl, gs, pl, mg = W.make_grouped_workload(11, members, G * 2, 2, 16, "fp16")
    wl.poison()
    _, _, out = run_grouped(wl, gs, pl, mg, gpu)
    assert max_abs_err(out, oracle_out(wl)) <= TOL
    assert pkv.check_device_error() == 0


# ------------------------------------------------------------------ bad metadata
MEMBERS = [[(64, 100), (64, 80), (32, 90)], [(32, 70), (32, 40)], [(16, 50)]]


def _bad_case(gpu, gs=None, pl_edit=None, mg=None, G=4, hkv=2):
    wl, gs0, pl, mg0 = W.make_grouped_workload(3, MEMBERS, G * hkv, hkv, 16, "bf16")
    wl.poison()
    ref = oracle_out(wl)
    pl = pl.copy()
    if pl_edit:
        for s, v in pl_edit.items():
            pl[s] = v
    _, _, out = run_grouped(wl, gs0 if gs is None else np.asarray(gs, dtype=np.int32), pl,
                            mg0 if mg is None else mg, gpu, max_prefix_len=96)
    return out.float().cpu().numpy(), ref, pkv.check_device_error()


@pytest.mark.parametrize("edit", [{1: 40}, {2: 112}, {4: -16}, {0: 128}, {5: 96}])
def test_bad_prefix_len_zeroes_that_sequence(gpu, edit):
    """Not a multiple of the block size, beyond the context, negative: error 6, that output zero."""
    out, ref, err = _bad_case(gpu, pl_edit=edit)
    bad = next(iter(edit))
    assert err == PREFIX_LEN
    for t in range(out.shape[0]):
        if t == bad:
            assert (out[t] == 0).all()
        else:  # including the members of a group whose first member is the bad one
            assert np.abs(out[t] - ref[t]).max() <= TOL, t


def test_sequence_outside_every_group_is_zeroed(gpu):
    out, ref, err = _bad_case(gpu, gs=[0, 3, 5])   # sequence 5 (prefix 16) in no group
    assert err == GROUP
    assert (out[5] == 0).all()
    assert np.abs(out[:5] - ref[:5]).max() <= TOL


def test_members_beyond_the_row_tiles_are_zeroed(gpu):
    """G = 64: one member per prefix CTA; max_group_size 2 leaves the third member of group 0 out."""
    out, ref, err = _bad_case(gpu, mg=2, G=64, hkv=1)
    assert err == GROUP
    assert (out[2] == 0).all()
    keep = [0, 1, 3, 4, 5]
    assert np.abs(out[keep] - ref[keep]).max() <= TOL


def test_out_of_order_group_starts_are_reported(gpu):
    out, _, err = _bad_case(gpu, gs=[0, 3, 1, 6])
    assert err == GROUP
    assert np.isfinite(out).all()


# ------------------------------------------------------------------ workspace and replay
def test_workspace_contents_do_not_matter(gpu):
    wl, gs, pl, mg = W.make_grouped_workload(4, MEMBERS * 3, 8, 2, 16, "bf16")
    ref = oracle_out(wl)
    need = pkv.paged_attention_grouped_workspace_bytes(wl.num_seqs, 8, 128, wl.max_context_len, int(pl.max()))
    ws = torch.empty(need, dtype=torch.uint8, device=gpu)
    for fill in (0xFF, 0x00, 0x7F, None):
        if fill is None:
            ws.copy_(torch.randint(0, 256, (need,), dtype=torch.uint8))
        else:
            ws.fill_(fill)
        for _ in range(2):  # and reuse
            _, _, out = run_grouped(wl, gs, pl, mg, gpu, workspace=ws)
            assert max_abs_err(out, ref) <= TOL
    assert pkv.check_device_error() == 0


def test_grouped_decode_in_a_cuda_graph(gpu):
    """Captured once, replayed with the group metadata changed in place between replays."""
    dev = gpu
    wl, gs, pl, mg = W.make_grouped_workload(9, MEMBERS * 2, 8, 2, 16, "bf16")
    ref = oracle_out(wl)
    dt = wl.dtype
    q, kc, vc = to_dev(wl.q, dt, dev), to_dev(wl.k_cache, dt, dev), to_dev(wl.v_cache, dt, dev)
    bt, cl = _dev(wl.block_tables, dev), _dev(wl.context_lens, dev)
    gs_d, pl_d = _dev(gs, dev), _dev(pl, dev)
    mpl = int(pl.max())
    need = pkv.paged_attention_grouped_workspace_bytes(wl.num_seqs, 8, 128, wl.max_context_len, mpl)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out = torch.empty((wl.num_seqs, 8, 128), dtype=torch.float32, device=dev)

    def call():
        pkv.paged_attention_decode_grouped(q, kc, vc, bt, cl, gs_d, pl_d, wl.scale, max_group_size=mg,
                                           max_prefix_len=mpl, max_context_len=wl.max_context_len, out=out,
                                           workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert max_abs_err(out, ref) <= TOL
    assert pkv.check_device_error() == 0
    # sequence 11 (a group of one with a 16-token prefix) leaves every group
    gs_d.copy_(_dev(np.asarray(list(gs[:-2]) + [gs[-2]] * 2, dtype=np.int32), dev))
    g.replay()
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert (o[11] == 0).all() and np.abs(o[:11] - ref[:11]).max() <= TOL
    assert pkv.check_device_error() == GROUP
    gs_d.copy_(_dev(gs, dev))
    g.replay()
    torch.cuda.synchronize()
    assert max_abs_err(out, ref) <= TOL
    assert pkv.check_device_error() == 0


# ------------------------------------------------------------------ host-side checks
def test_host_checks(gpu):
    wl, gs, pl, mg = W.make_grouped_workload(2, MEMBERS, 8, 2, 16, "bf16")
    with pytest.raises(pkv.PagedKVError) as e:   # max_prefix_len above max_context_len
        run_grouped(wl, gs, pl, mg, gpu, max_prefix_len=wl.max_context_len + 16)
    assert e.value.status == 1
    with pytest.raises(pkv.PagedKVError) as e:   # workspace too small
        run_grouped(wl, gs, pl, mg, gpu, workspace=torch.empty(256, dtype=torch.uint8, device=gpu))
    assert e.value.status == 3
    wl65, gs65, pl65, mg65 = W.make_grouped_workload(2, MEMBERS, 65, 1, 16, "bf16")
    with pytest.raises(pkv.PagedKVError) as e:   # more than 64 query heads per KV head
        run_grouped(wl65, gs65, pl65, mg65, gpu)
    assert e.value.status == 2
