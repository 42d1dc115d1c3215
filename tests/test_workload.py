"""Host-side logic: the seeded input generator, the block manager's
fork/append/free bookkeeping, the workload table and the byte accounting."""
import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

from paged_kv_cache_11_gb300 import workload as W
from paged_kv_cache_11_gb300.block_manager import BlockManager, OutOfBlocks

GOLDEN = Path(__file__).parent / "golden"


# ---------------------------------------------------------------- generator
def test_generator_is_counter_based_and_seeded():
    a = W.normal(7, 3, (5000,), "fp32")
    assert np.array_equal(a, W.normal(7, 3, (5000,), "fp32", threads=1))
    assert np.array_equal(a[1001:3001], W.normal(7, 3, (2000,), "fp32", offset=1001))
    assert not np.array_equal(a, W.normal(8, 3, (5000,), "fp32"))
    assert not np.array_equal(a, W.normal(7, 4, (5000,), "fp32"))


def test_generator_moments():
    x = W.normal(1, 1, (1_000_000,), "fp32").astype(np.float64)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    assert abs((x ** 4).mean() - 3) < 0.05  # normal kurtosis


def test_generator_rounding_matches_library_conversions():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200_000).astype(np.float32),
                        (rng.standard_normal(20_000) * 1e-5).astype(np.float32),   # fp16 subnormals
                        np.array([0.0, -0.0, 65504.0, 65520.0, 1e9, 6.1035156e-05, 5.96e-08, 2.98e-08],
                                 dtype=np.float32)])
    bf = W.round_f32(x, "bf16")
    ref_bf = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf, ref_bf)
    hf = W.round_f32(x, "fp16")
    with np.errstate(over="ignore"):  # 65520 and 1e9 round to inf on purpose
        ref_hf = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(hf, ref_hf)


def test_generator_dtype_paths_agree_with_rounding():
    f = W.normal(9, 2, (4096,), "fp32")
    assert np.array_equal(W.normal(9, 2, (4096,), "bf16"), W.round_f32(f, "bf16"))
    assert np.array_equal(W.normal(9, 2, (4096,), "fp16"), W.round_f32(f, "fp16"))


def test_permutation_and_uniform_ints():
    p = W.permutation(3, 7, 1000)
    assert sorted(p.tolist()) == list(range(1000)) and not np.array_equal(p, np.arange(1000))
    u = W.uniform_ints(3, 6, 10000, 512, 4096)
    assert u.min() >= 512 and u.max() <= 4096 and abs(u.mean() - 2304) < 40


# ---------------------------------------------------------------- byte accounting
def test_kv_bytes_per_token_reproduces_the_pages():
    for e in json.loads((GOLDEN / "kv_bytes_per_token.json").read_text())["entries"]:
        b = W.kv_bytes_per_token(e["layers"], e["kv_heads"], e["head_dim"], e["elt_bytes"])
        assert b == e["exact_formula_bytes"], e["model"]
        # the printed, rounded figures agree to the precision they are printed with
        assert abs(b - e["printed_bytes_per_token"]) / b < 0.06, e["model"]
        ctx = b * e["printed_context_tokens"]
        assert abs(ctx - e["printed_context_bytes"]) / ctx < 0.07, e["model"]


# ---------------------------------------------------------------- block manager
def test_sixty_tokens_occupy_four_blocks():
    """A 60-token request holds only the blocks for 60 tokens; waste <= one block."""
    bm = BlockManager(10, 16)
    bm.add_sequence(0)
    bm.append_tokens(0, 60)
    assert len(bm.block_table(0)) == math.ceil(60 / 16) == 4
    assert bm.num_free == 6
    assert 4 * 16 - 60 < 16


def test_fresh_block_exactly_when_last_is_full():
    bm = BlockManager(64, 16, W.permutation(1, 1, 64))
    bm.add_sequence(0)
    for p in range(100):
        before = len(bm.block_table(0))
        slot, cow = bm.append_token(0)
        assert cow is None
        assert len(bm.block_table(0)) == before + (1 if p % 16 == 0 else 0)
        t = bm.block_table(0)
        assert slot == t[p // 16] * 16 + p % 16 == bm.slot(0, p)


def test_fork_shares_and_copy_on_write_copies_only_the_last_shared_block():
    bm = BlockManager(32, 16)
    bm.add_sequence(0)
    bm.append_tokens(0, 40)                         # blocks: 2 full + 1 holding 8 tokens
    bm.fork(0, 1)
    t0 = bm.block_table(0)
    assert bm.block_table(1) == t0 and all(bm.refcount[b] == 2 for b in t0)
    slot, cow = bm.append_token(1)                  # write into the shared last block
    assert cow is not None and cow[0] == t0[2]
    t1 = bm.block_table(1)
    assert t1[:2] == t0[:2] and t1[2] == cow[1] != t0[2]   # only the last block changed
    assert slot == cow[1] * 16 + 8
    assert bm.refcount[t0[2]] == 1 and bm.refcount[cow[1]] == 1
    slot0, cow0 = bm.append_token(0)                # the last holder writes in place
    assert cow0 is None and slot0 == t0[2] * 16 + 8
    bm.free(1)
    assert bm.refcount[cow[1]] == 0 and all(bm.refcount[b] == 1 for b in t0)
    bm.free(0)
    assert bm.num_free == 32


def test_out_of_blocks():
    bm = BlockManager(2, 16)
    bm.add_sequence(0)
    bm.append_tokens(0, 32)
    with pytest.raises(OutOfBlocks):
        bm.append_token(0)


# ---------------------------------------------------------------- workloads
def _check_slots(wl):
    bs = wl.block_size
    pos = {}
    for t, s in enumerate(wl.append_seq):
        L = int(wl.context_lens[s])
        p = pos.get(s, None)
        if p is None:  # the first appended token of s: position L - (number appended to s)
            p = L - int((wl.append_seq == s).sum())
        assert wl.slot_mapping[t] == wl.block_tables[s, p // bs] * bs + p % bs
        pos[s] = p + 1


def test_tiny_workload():
    wl = W.make_workload("tiny")
    assert wl.context_lens.tolist() == [1, 17, 33, 100]
    assert wl.num_blocks == 64 and wl.block_tables.shape == (4, 7)
    used = np.concatenate([wl.block_tables[s, :(L + 15) // 16] for s, L in enumerate(wl.context_lens)])
    assert len(set(used.tolist())) == len(used) == 13
    assert len(wl.slot_mapping) == 4 and len(wl.cow_pairs) == 0
    _check_slots(wl)
    assert wl.q.shape == (4, 4, 128) and wl.k_cache.shape == (64, 1, 16, 128)


@pytest.mark.parametrize("name", ["llama8b", "opt13b"])
def test_decode_workload_metadata(name):
    wl = W.make_workload(name, with_data=False)
    spec = W.SPECS[name]
    lo, hi = spec.lens[1], spec.lens[2]
    assert wl.num_seqs == spec.num_seqs and lo <= wl.context_lens.min() and wl.context_lens.max() <= hi
    needed = int(sum((int(L) + 15) // 16 for L in wl.context_lens))
    assert wl.num_blocks == math.ceil(1.25 * needed)
    _check_slots(wl)
    # one appended token per sequence, at position L - 1; a fresh block when (L - 1) % 16 == 0
    assert len(wl.slot_mapping) == wl.num_seqs
    fresh = [(int(L) - 1) % 16 == 0 for L in wl.context_lens]
    assert any(fresh) or name == "llama8b"


def test_shared_prefix_workload():
    wl = W.make_workload("shared_prefix", with_data=False)
    G, M = 16, 16
    assert wl.num_seqs == G * M and len(wl.cow_pairs) == G * (M - 1) == 240
    for g in range(G):
        rows = wl.block_tables[g * M:(g + 1) * M]
        assert (rows[:, :64] == rows[0, :64]).all()       # the 1024-token prefix is shared
        last = {int(r[64]) for r in rows}                  # the partly filled prompt block: 16 distinct after CoW
        assert len(last) == M
        srcs = set(wl.cow_pairs[g * (M - 1):(g + 1) * (M - 1), 0].tolist())
        assert len(srcs) == 1 and srcs.pop() in last       # all copies read the group's original block
        suf = wl.context_lens[g * M:(g + 1) * M] - 1024
        assert (suf >= 1 + 32).all() and (suf <= 15 + 512).all()
    assert len(set(wl.cow_pairs[:, 1].tolist())) == 240
    assert not set(wl.cow_pairs[:, 1].tolist()) & set(wl.cow_pairs[:, 0].tolist())
    _check_slots(wl)
    assert wl.unique_kv_bytes() < wl.kv_bytes()
    # the decode step: one new token per sample, at its last position, in a
    # block of its own (never a shared one and never a copy destination)
    assert len(wl.slot_mapping) == 256 and np.array_equal(wl.append_seq, np.arange(256))
    for s in range(wl.num_seqs):
        L = int(wl.context_lens[s])
        blk = int(wl.block_tables[s, (L - 1) // 16])
        assert wl.slot_mapping[s] == blk * 16 + (L - 1) % 16
        others = np.delete(wl.block_tables, s, axis=0)
        assert blk not in others and blk not in wl.cow_pairs[:, 1]


def test_shared_prefix_prefill_workload():
    """The same batch, with each sample's whole continuation written by the step."""
    a = W.make_workload("shared_prefix", with_data=False)
    b = W.make_workload("shared_prefix_prefill", with_data=False)
    assert np.array_equal(a.context_lens, b.context_lens) and np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(a.cow_pairs, b.cow_pairs)
    # every token past the prompt (1024 + t_g tokens per group) is appended
    tails = np.repeat(W.uniform_ints(b.seed, W.S_GROUP, 16, 1, 15), 16)
    assert len(b.slot_mapping) == int((b.context_lens - 1024 - tails).sum()) > 60000
    # the decode step's slots are the continuation's last slots
    last = {int(s): int(sl) for s, sl in zip(b.append_seq, b.slot_mapping)}
    assert all(last[s] == a.slot_mapping[s] for s in range(256))
    _check_slots(b)


def test_long_context_workload_metadata():
    wl = W.make_workload("llama70b_long", with_data=False)
    assert wl.num_blocks == 8 * 4096 and wl.block_tables.shape == (8, 4096)
    assert sorted(wl.block_tables.ravel().tolist()) == list(range(32768))
    assert wl.kv_bytes() == 4 * 2 ** 30
    _check_slots(wl)


def test_poison_touches_only_unused_slots_and_step_targets():
    wl = W.make_workload("tiny")
    k0 = wl.k_cache.copy()
    wl.poison()
    valid = wl.valid_slot_mask()
    targets = np.zeros_like(valid)
    targets[wl.slot_mapping // 16, wl.slot_mapping % 16] = True
    keep = valid & ~targets
    kt, k0t = wl.k_cache.transpose(0, 2, 1, 3), k0.transpose(0, 2, 1, 3)
    assert np.array_equal(kt[keep], k0t[keep])
    assert (kt[~keep] == W.NAN_BITS["bf16"]).all()


# ---------------------------------------------------------------- swap / compaction bookkeeping
def test_swap_out_and_in_round_trip():
    from paged_kv_cache_11_gb300.block_manager import swap_in, swap_out
    gpu, cpu = BlockManager(16, 16, W.permutation(2, 2, 16)), BlockManager(8, 16)
    gpu.add_sequence(0)
    gpu.append_tokens(0, 50)                         # 4 blocks
    t = gpu.block_table(0)
    out_pairs = swap_out(gpu, cpu, 0)
    assert [a for a, _ in out_pairs] == t and gpu.num_free == 16 and cpu.num_free == 4
    assert cpu.num_tokens(0) == 50 and [b for _, b in out_pairs] == cpu.block_table(0)
    in_pairs = swap_in(cpu, gpu, 0)
    assert [a for a, _ in in_pairs] == [b for _, b in out_pairs] and cpu.num_free == 8
    assert gpu.num_tokens(0) == 50 and len(gpu.block_table(0)) == 4
    slot, cow = gpu.append_token(0)                  # the sequence continues where it stopped
    assert cow is None and slot == gpu.block_table(0)[3] * 16 + 50 % 16


def test_compaction_trigger_and_targets_leave_shared_blocks_intact():
    bm = BlockManager(32, 16)
    bm.add_sequence(0)
    bm.append_tokens(0, 64)                          # 4 full blocks
    bm.fork(0, 1)                                    # shared prompt
    shared = bm.block_table(0)
    bm.append_tokens(1, 16)                          # sequence 1: 5 blocks, last one full
    assert bm.needs_compaction(1, 5) and not bm.needs_compaction(1, 6) and not bm.needs_compaction(0, 5)
    keep = list(range(0, 80, 3))                     # 27 tokens -> 2 target blocks (<= N_max - 1)
    src, dst = bm.compact(1, keep)
    t = bm.block_table(1)
    assert len(t) == 2 and bm.num_tokens(1) == 27 and not set(t) & set(shared)
    assert src[0] == shared[0] * 16 and dst == [t[i // 16] * 16 + i % 16 for i in range(27)]
    assert bm.block_table(0) == shared and all(bm.refcount[b] == 1 for b in shared)


def test_deferred_free_keeps_compaction_sources_out_of_later_targets():
    bm = BlockManager(12, 16)
    for s in range(2):
        bm.add_sequence(s)
        bm.append_tokens(s, 48)                     # 3 blocks each
    old = set(bm.block_table(0)) | set(bm.block_table(1))
    src0, dst0 = bm.compact(0, range(0, 48, 2), defer_free=True)
    src1, dst1 = bm.compact(1, range(0, 48, 2), defer_free=True)
    assert not (set(d // 16 for d in dst0 + dst1) & old)
    assert bm.release_deferred() == 6 and bm.num_free == 12 - 4


def test_grouped_workload_shares_exactly_the_requested_blocks():
    members = [[(64, 100), (32, 40), (64, 64), (0, 17)], [(0, 33)], [(16, 16), (16, 50)]]
    wl, gs, pl, mg = W.make_grouped_workload(5, members, 8, 2, 16, "bf16")
    assert gs.tolist() == [0, 4, 5, 7] and mg == 4
    assert pl.tolist() == [64, 32, 64, 0, 0, 16, 16]
    assert wl.context_lens.tolist() == [100, 40, 64, 17, 33, 16, 50]
    bt = wl.block_tables
    for s, p in ((1, 32), (2, 64), (3, 0), (6, 16)):
        lead = 0 if s < 4 else 5
        n = p // 16
        assert (bt[s, :n] == bt[lead, :n]).all()
        own = bt[s, n:(wl.context_lens[s] + 15) // 16]
        assert not set(own.tolist()) & set(bt[lead, :(wl.context_lens[lead] + 15) // 16].tolist())


def test_prefix_groups_of_the_shared_prefix_workload():
    """16 groups of 16 forked samples: 1024 prompt tokens in 64 shared blocks each."""
    wl = W.make_workload("shared_prefix", with_data=False)
    gs, pl, mg = W.prefix_groups(wl)
    assert gs.tolist() == list(range(0, 257, 16)) and mg == 16
    assert (pl == 1024).all()
    # plain decode workloads: every sequence on its own, nothing shared
    wl = W.make_workload("llama8b", num_seqs=5, with_data=False)
    gs, pl, mg = W.prefix_groups(wl)
    assert gs.tolist() == [0, 1, 2, 3, 4, 5] and (pl == 0).all() and mg == 1
