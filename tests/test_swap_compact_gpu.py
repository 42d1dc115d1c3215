"""GPU parity of the swap (GPU pool <-> page-locked host pool) and compaction
kernels against the oracle, bit-exact, plus the decode invariants that follow
from them."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_11_gb300 as pkv
from paged_kv_cache_11_gb300 import workload as W
from paged_kv_cache_11_gb300.block_manager import BlockManager, swap_in, swap_out
from tests.step_helpers import max_abs_err, to_bits, to_dev

pytestmark = pytest.mark.gpu
TOL = 5e-3


def _host_pool(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view({"bf16": torch.bfloat16,
                                                                         "fp16": torch.float16}[dtype])
    return t.pin_memory()


@pytest.mark.parametrize("layers", [1, 3])
def test_swap_out_and_in_bit_exact(gpu, layers):
    rng = np.random.default_rng(layers)
    hkv, bs, d = 8, 16, 128
    g_bits = [W.normal(layers, 10 + l, (40, hkv, bs, d), "bf16") for l in range(2 * layers)]
    h_bits = [W.normal(layers, 30 + l, (24, hkv, bs, d), "bf16") for l in range(2 * layers)]
    gk = [to_dev(g_bits[2 * l], "bf16", gpu) for l in range(layers)]
    gv = [to_dev(g_bits[2 * l + 1], "bf16", gpu) for l in range(layers)]
    hk = [_host_pool(h_bits[2 * l], "bf16") for l in range(layers)]
    hv = [_host_pool(h_bits[2 * l + 1], "bf16") for l in range(layers)]
    out_pairs = np.stack([rng.permutation(40)[:17], rng.permutation(24)[:17]], axis=1).astype(np.int64)
    pkv.swap_blocks(gk, gv, hk, hv, torch.from_numpy(out_pairs).to(gpu))
    torch.cuda.synchronize()
    for l in range(layers):
        ek, ev = h_bits[2 * l].copy(), h_bits[2 * l + 1].copy()
        assert oracle.swap_blocks(g_bits[2 * l], g_bits[2 * l + 1], ek, ev, out_pairs) == 0
        assert np.array_equal(to_bits(hk[l]), ek) and np.array_equal(to_bits(hv[l]), ev)
    # and back in, to other GPU blocks; the pair list may live in pinned host memory
    in_pairs = np.stack([out_pairs[:, 1], rng.permutation(40)[:17]], axis=1).astype(np.int64)
    pkv.swap_blocks(hk, hv, gk, gv, torch.from_numpy(in_pairs).pin_memory())
    torch.cuda.synchronize()
    for l in range(layers):
        got = to_bits(gk[l])
        for a, b in out_pairs:
            dst = in_pairs[in_pairs[:, 0] == b, 1][0]
            assert np.array_equal(got[dst], g_bits[2 * l][a])
    assert pkv.check_device_error() == 0


@pytest.mark.parametrize("layers", [3, 33])
def test_copy_blocks_every_layer_bit_exact(gpu, layers):
    """Batched copy-on-write copy over several layers' pools in one call (33
    layers: more than one launch's 32).  Every layer's K and V pools must equal
    the oracle's copy of that layer, byte for byte; blocks outside the pairs
    keep their bytes."""
    rng = np.random.default_rng(100 + layers)
    nb, hkv, bs, d = 40, 8, 16, 128
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:9], perm[9:18]], axis=1).astype(np.int64)  # distinct dsts, none of them a src
    bits = [W.normal(layers, 50 + l, (nb, hkv, bs, d), "bf16") for l in range(2 * layers)]
    ks = [to_dev(bits[2 * l], "bf16", gpu) for l in range(layers)]
    vs = [to_dev(bits[2 * l + 1], "bf16", gpu) for l in range(layers)]
    pkv.copy_blocks(ks, vs, torch.from_numpy(pairs).to(gpu))
    torch.cuda.synchronize()
    assert pkv.check_device_error() == 0
    for l in range(layers):
        ek, ev = bits[2 * l].copy(), bits[2 * l + 1].copy()
        assert oracle.copy_blocks(ek, ev, pairs) == 0
        assert np.array_equal(to_bits(ks[l]), ek) and np.array_equal(to_bits(vs[l]), ev), f"layer {l}"


def test_swapped_sequence_decodes_the_same(gpu):
    """Swap a workload's sequences out to host memory and back into other blocks: same output bits."""
    wl = W.make_workload("llama8b", num_seqs=4, lens=("uniform", 300, 1500), seed=9)
    kc, vc, q = to_dev(wl.k_cache, "bf16", gpu), to_dev(wl.v_cache, "bf16", gpu), to_dev(wl.q, "bf16", gpu)
    bt, cl = torch.from_numpy(wl.block_tables).to(gpu), torch.from_numpy(wl.context_lens).to(gpu)
    before = pkv.paged_attention_decode(q, kc, vc, bt, cl, wl.scale, max_context_len=wl.max_context_len)
    # rebuild the manager state: every sequence maps its table; swap all out, then back in
    gpu_bm = BlockManager(wl.num_blocks, 16, W.permutation(1, 1, wl.num_blocks))
    for s in range(wl.num_seqs):
        gpu_bm.add_sequence(s)
        gpu_bm.append_tokens(s, int(wl.context_lens[s]))
    old_tables = {s: gpu_bm.block_table(s) for s in range(wl.num_seqs)}
    # the device pool holds the workload's data at the workload's tables: copy it to the manager's blocks
    src = np.concatenate([wl.block_tables[s, :len(old_tables[s])] for s in range(wl.num_seqs)])
    dst = np.concatenate([old_tables[s] for s in range(wl.num_seqs)])
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    pkv.swap_blocks(kc, vc, kc2, vc2, torch.from_numpy(np.stack([src, dst], 1).astype(np.int64)).to(gpu))
    cpu_bm = BlockManager(sum(len(t) for t in old_tables.values()), 16)
    hk = torch.empty((cpu_bm.num_blocks, 8, 16, 128), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    out_pairs = sum((swap_out(gpu_bm, cpu_bm, s) for s in range(wl.num_seqs)), [])
    pkv.swap_blocks(kc2, vc2, hk, hv, torch.tensor(out_pairs, dtype=torch.int64, device=gpu))
    kc2.fill_(float("nan"))
    vc2.fill_(float("nan"))
    # other sequences would now reuse the freed GPU blocks; bring ours back in reverse order
    in_pairs = sum((swap_in(cpu_bm, gpu_bm, s) for s in reversed(range(wl.num_seqs))), [])
    pkv.swap_blocks(hk, hv, kc2, vc2, torch.tensor(in_pairs, dtype=torch.int64, device=gpu))
    bt2 = np.full_like(wl.block_tables, -1)
    for s in range(wl.num_seqs):
        t = gpu_bm.block_table(s)
        bt2[s, :len(t)] = t
    after = pkv.paged_attention_decode(q, kc2, vc2, torch.from_numpy(bt2).to(gpu), cl, wl.scale,
                                       max_context_len=wl.max_context_len)
    assert torch.equal(before, after)
    assert pkv.check_device_error() == 0


def test_compaction_bit_exact_and_decode_over_kept_tokens(gpu):
    wl = W.make_workload("llama8b", num_seqs=3, lens=("fixed", (400, 700, 257)), seed=11, pool_factor=2.0)
    bm = BlockManager(wl.num_blocks, 16, W.permutation(4, 4, wl.num_blocks))
    # a manager whose tables equal the workload's: replay the allocation order
    for s in range(wl.num_seqs):
        bm.add_sequence(s)
        bm.append_tokens(s, int(wl.context_lens[s]))
    tables = {s: bm.block_table(s) for s in range(wl.num_seqs)}
    bt = np.full((wl.num_seqs, wl.block_tables.shape[1]), -1, np.int32)
    for s, t in tables.items():
        bt[s, :len(t)] = t
    rng = np.random.default_rng(0)
    n_max = 8                                           # at most 8 blocks: keep <= 7 * 16 tokens
    srcs, dsts, kept = [], [], {}
    for s in range(wl.num_seqs):
        L = int(wl.context_lens[s])
        keep = np.unique(np.concatenate([rng.choice(L - 1, 100, replace=False), [L - 1]]))
        a, b = bm.compact(s, keep, defer_free=True)  # one launch for all: no target may be a source
        srcs += a
        dsts += b
        kept[s] = keep
    assert not set(srcs) & set(dsts)
    bm.release_deferred()
    kc, vc = to_dev(wl.k_cache, "bf16", gpu), to_dev(wl.v_cache, "bf16", gpu)
    pkv.compact_tokens(torch.tensor(srcs, dtype=torch.int64, device=gpu),
                       torch.tensor(dsts, dtype=torch.int64, device=gpu), kc, vc)
    okc, ovc = wl.k_cache.copy(), wl.v_cache.copy()
    assert oracle.compact(okc, ovc, srcs, dsts) == 0
    assert np.array_equal(to_bits(kc), okc) and np.array_equal(to_bits(vc), ovc)
    new_lens = np.array([len(kept[s]) for s in range(wl.num_seqs)], np.int32)
    nbt = np.full((wl.num_seqs, n_max), -1, np.int32)
    for s in range(wl.num_seqs):
        t = bm.block_table(s)
        assert len(t) <= n_max - 1
        nbt[s, :len(t)] = t
    q = to_dev(wl.q, "bf16", gpu)
    out = pkv.paged_attention_decode(q, kc, vc, torch.from_numpy(nbt).to(gpu), torch.from_numpy(new_lens).to(gpu),
                                     wl.scale, max_context_len=int(new_lens.max()))
    ref, st = oracle.decode(wl.q, okc, ovc, nbt, new_lens, wl.scale, "bf16", threads=8)
    assert not st.any()
    assert max_abs_err(out, ref) <= TOL
    assert pkv.check_device_error() == 0
