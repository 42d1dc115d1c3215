"""Pins of the oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value:
  * library routines (torch scaled_dot_product_attention in float64; numpy and
    torch element conversions) on the contiguous tensors the test scattered;
  * invariants the pages state (paging changes no output: techtrendfeed "KV
    Cache Administration", "Why this modified LLM serving"; aitalk.it
    "PagedAttention e RadixAttention"; blocks need not be adjacent: tonho.wtf
    "vllm", "como funciona"; a shared block and its copy give the same
    result, and a write copies only the last shared block: same section);
  * closed forms (L = 1, identical keys, L = 2 sigmoid form);
  * brute force on tiny inputs (append / copy byte moves).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.pin_helpers import NAN, bits_to_torch64, paged_case, random_bits, sdpa_reference

SCALE = 1.0 / math.sqrt(128)


# ---------------------------------------------------------------- element decode
def test_bf16_decode_exhaustive_matches_torch():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.to_f64(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_fp16_decode_exhaustive_matches_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.to_f64(bits, "fp16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- attention
CASES = [
    # (lens, hq, hkv, bs, dtype)
    ([1, 17, 33, 100], 4, 1, 16, "bf16"),      # the tiny workload's lengths
    ([16, 15, 32, 31, 1], 8, 8, 16, "fp16"),   # MHA, block boundaries
    ([64, 97, 5], 32, 8, 16, "bf16"),          # GQA 4
    ([200, 33, 1, 64], 16, 2, 32, "bf16"),     # GQA 8, block 32
    ([77, 300], 40, 40, 16, "fp16"),           # OPT-13B-like heads
]


@pytest.mark.parametrize("lens,hq,hkv,bs,dtype", CASES)
def test_decode_equals_contiguous_sdpa(lens, hq, hkv, bs, dtype):
    rng = np.random.default_rng(sum(lens) + hq)
    case = paged_case(rng, lens, hq, hkv, bs, dtype=dtype)
    out, status = oracle.decode(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                case["context_lens"], SCALE, dtype)
    assert not status.any()
    ref = sdpa_reference(case, SCALE)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_decode_equals_numpy_softmax_two_ways():
    """A second, hand-written reference: explicit exp / sum in numpy float64."""
    rng = np.random.default_rng(7)
    case = paged_case(rng, [50, 3], 8, 2, 16, dtype="bf16")
    out, _ = oracle.decode(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                           case["context_lens"], 0.37, "bf16")
    G = 4
    for s in range(2):
        for h in range(8):
            q = bits_to_torch64(case["q"][s, h], "bf16").numpy()
            K = bits_to_torch64(case["K"][s][h // G], "bf16").numpy()
            V = bits_to_torch64(case["V"][s][h // G], "bf16").numpy()
            z = 0.37 * (K @ q)
            w = np.exp(z - z.max())
            np.testing.assert_allclose(out[s, h], (w / w.sum()) @ V, rtol=0, atol=1e-12)


def test_permutation_of_physical_ids_changes_nothing():
    rng = np.random.default_rng(11)
    lens = [40, 1, 129, 16]
    nb = sum((L + 15) // 16 for L in lens) + 9
    a = paged_case(np.random.default_rng(3), lens, 8, 2, 16, pool_slack=9, perm=np.arange(nb))
    b = paged_case(np.random.default_rng(3), lens, 8, 2, 16, pool_slack=9, perm=rng.permutation(nb))
    assert not np.array_equal(a["block_tables"], b["block_tables"])
    oa, _ = oracle.decode(a["q"], a["k_cache"], a["v_cache"], a["block_tables"], a["context_lens"], SCALE, "bf16")
    ob, _ = oracle.decode(b["q"], b["k_cache"], b["v_cache"], b["block_tables"], b["context_lens"], SCALE, "bf16")
    assert np.array_equal(oa, ob)


def test_shared_blocks_equal_copied_blocks():
    """Two sequences mapping the same prefix blocks == the same sequences holding copies."""
    rng = np.random.default_rng(5)
    bs, hkv, d, hq = 16, 2, 128, 8
    nb = 20
    kc = random_bits(rng, (nb, hkv, bs, d), "bf16")
    vc = random_bits(rng, (nb, hkv, bs, d), "bf16")
    q = random_bits(rng, (2, hq, d), "bf16")
    lens = np.array([50, 61], dtype=np.int32)
    shared = np.array([[0, 1, 2, 3], [0, 1, 2, 4]], dtype=np.int32)  # blocks 0-2 shared
    o1, _ = oracle.decode(q, kc, vc, shared, lens, SCALE, "bf16")
    kc2, vc2 = kc.copy(), vc.copy()
    for src, dst in ((0, 10), (1, 11), (2, 12)):
        kc2[dst], vc2[dst] = kc2[src], vc2[src]
    copied = np.array([[0, 1, 2, 3], [10, 11, 12, 4]], dtype=np.int32)
    o2, _ = oracle.decode(q, kc2, vc2, copied, lens, SCALE, "bf16")
    assert np.array_equal(o1, o2)


def test_context_length_one_returns_v_exactly():
    rng = np.random.default_rng(9)
    case = paged_case(rng, [1, 1, 1], 8, 2, 16, dtype="fp16")
    out, _ = oracle.decode(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                           case["context_lens"], SCALE, "fp16")
    for s in range(3):
        for h in range(8):
            assert np.array_equal(out[s, h], bits_to_torch64(case["V"][s][h // 4][0], "fp16").numpy())


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(10)
    case = paged_case(rng, [37, 100], 4, 1, 16, dtype="bf16")
    key_row = random_bits(rng, (128,), "bf16")
    for s, L in enumerate(case["context_lens"]):
        for j in range((L + 15) // 16):
            n = min(16, L - 16 * j)
            case["k_cache"][case["block_tables"][s, j], :, :n, :] = key_row
    out, _ = oracle.decode(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                           case["context_lens"], SCALE, "bf16")
    for s in range(2):
        mean_v = bits_to_torch64(case["V"][s][0], "bf16").numpy().mean(axis=0)
        for h in range(4):
            np.testing.assert_allclose(out[s, h], mean_v, rtol=0, atol=1e-12)


def test_two_token_closed_form():
    """L = 2: out = sigmoid(z1 - z0) V1 + sigmoid(z0 - z1) V0."""
    rng = np.random.default_rng(12)
    case = paged_case(rng, [2], 2, 1, 16, dtype="bf16")
    out, _ = oracle.decode(case["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                           case["context_lens"], 0.5, "bf16")
    K = bits_to_torch64(case["K"][0][0], "bf16").numpy()
    V = bits_to_torch64(case["V"][0][0], "bf16").numpy()
    for h in range(2):
        q = bits_to_torch64(case["q"][0, h], "bf16").numpy()
        z0, z1 = 0.5 * float(K[0] @ q), 0.5 * float(K[1] @ q)
        sig = lambda x: 1.0 / (1.0 + math.exp(-x))
        np.testing.assert_allclose(out[0, h], sig(z1 - z0) * V[1] + sig(z0 - z1) * V[0], rtol=0, atol=1e-13)


def test_poisoned_unused_slots_do_not_leak():
    rng = np.random.default_rng(13)
    a = paged_case(np.random.default_rng(1), [5, 18, 40], 8, 2, 16, pool_slack=6, poison=True, perm=np.arange(12))
    b = paged_case(np.random.default_rng(1), [5, 18, 40], 8, 2, 16, pool_slack=6, poison=False, perm=np.arange(12))
    oa, _ = oracle.decode(a["q"], a["k_cache"], a["v_cache"], a["block_tables"], a["context_lens"], SCALE, "bf16")
    ob, _ = oracle.decode(b["q"], b["k_cache"], b["v_cache"], b["block_tables"], b["context_lens"], SCALE, "bf16")
    assert np.isfinite(oa).all()
    assert np.array_equal(oa, ob)
    del rng


@pytest.mark.parametrize("P", [16, 32, 48, 512])
def test_partitioned_form_equals_plain(P):
    rng = np.random.default_rng(P)
    case = paged_case(rng, [1, 16, 17, 100, 513, 1100], 8, 2, 16, dtype="bf16")
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"], SCALE, "bf16")
    plain, _ = oracle.decode(*args)
    split, _ = oracle.decode(*args, partition_size=P)
    np.testing.assert_allclose(split, plain, rtol=0, atol=1e-12)
    np.testing.assert_allclose(split, sdpa_reference(case, SCALE), rtol=0, atol=1e-12)


def test_zero_length_gives_zeros_and_select_subset():
    rng = np.random.default_rng(14)
    case = paged_case(rng, [0, 20, 35], 4, 2, 16, dtype="bf16")
    args = (case["q"], case["k_cache"], case["v_cache"], case["block_tables"], case["context_lens"], SCALE, "bf16")
    full, status = oracle.decode(*args, threads=3)
    assert not status.any()
    assert np.array_equal(full[0], np.zeros((4, 128)))
    part, _ = oracle.decode(*args, select=[(1, 3), (2, 0)])
    assert np.array_equal(part[1, 3], full[1, 3]) and np.array_equal(part[2, 0], full[2, 0])
    assert not part[1, :3].any() and not part[2, 1:].any()


def test_bad_metadata_flags_sequence_and_zeroes_it():
    rng = np.random.default_rng(15)
    case = paged_case(rng, [20, 20, 20], 4, 1, 16, dtype="bf16", pool_slack=0)
    bt = case["block_tables"].copy()
    bt[1, 1] = case["num_blocks"]          # outside the pool
    cl = case["context_lens"].copy()
    cl[2] = 16 * bt.shape[1] + 1           # longer than the table
    out, status = oracle.decode(case["q"], case["k_cache"], case["v_cache"], bt, cl, SCALE, "bf16")
    assert list(status) == [0, 1, 1]
    assert not out[1:].any()
    assert np.isfinite(out[0]).all() and out[0].any()


# ---------------------------------------------------------------- append / copy
def test_append_writes_rows_to_their_slots_and_nothing_else():
    rng = np.random.default_rng(16)
    nb, hkv, bs, d = 6, 3, 16, 128
    kc = random_bits(rng, (nb, hkv, bs, d), "bf16")
    vc = random_bits(rng, (nb, hkv, bs, d), "bf16")
    k0, v0 = kc.copy(), vc.copy()
    slots = np.array([0, 17, -1, 95, 96, 40], dtype=np.int64)   # -1: padding, 96: outside the pool
    k = random_bits(rng, (6, hkv, d), "bf16")
    v = random_bits(rng, (6, hkv, d), "bf16")
    bad = oracle.append(k, v, slots, kc, vc)
    assert bad == 1
    ek, ev = k0.copy(), v0.copy()
    for t, s in enumerate(slots):
        if 0 <= s < nb * bs:
            ek[s // bs, :, s % bs, :] = k[t]
            ev[s // bs, :, s % bs, :] = v[t]
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_copy_blocks_copies_only_the_listed_blocks():
    rng = np.random.default_rng(17)
    nb, hkv, bs, d = 8, 2, 16, 128
    kc = random_bits(rng, (nb, hkv, bs, d), "fp16")
    vc = random_bits(rng, (nb, hkv, bs, d), "fp16")
    k0, v0 = kc.copy(), vc.copy()
    bad = oracle.copy_blocks(kc, vc, np.array([[1, 5], [2, 6], [3, 99]]))
    assert bad == 1
    for c, c0 in ((kc, k0), (vc, v0)):
        assert np.array_equal(c[5], c0[1]) and np.array_equal(c[6], c0[2])
        keep = [0, 1, 2, 3, 4, 7]
        assert np.array_equal(c[keep], c0[keep])


def test_nan_bits_are_what_the_helpers_use():
    assert np.isnan(oracle.to_f64(np.array([NAN["bf16"]], np.uint16), "bf16")[0])
    assert np.isnan(oracle.to_f64(np.array([NAN["fp16"]], np.uint16), "fp16")[0])


# ---------------------------------------------------------------- swap / compaction
def test_swap_blocks_moves_exactly_the_listed_blocks_between_pools():
    rng = np.random.default_rng(18)
    hkv, bs, d = 2, 16, 128
    gk, gv = random_bits(rng, (9, hkv, bs, d), "bf16"), random_bits(rng, (9, hkv, bs, d), "bf16")
    hk, hv = random_bits(rng, (5, hkv, bs, d), "bf16"), random_bits(rng, (5, hkv, bs, d), "bf16")
    h0k, h0v = hk.copy(), hv.copy()
    bad = oracle.swap_blocks(gk, gv, hk, hv, np.array([[7, 0], [2, 3], [9, 1], [1, 5]]))
    assert bad == 2                                  # src 9 (GPU pool of 9) and dst 5 (host pool of 5)
    assert np.array_equal(hk[0], gk[7]) and np.array_equal(hk[3], gk[2])
    assert np.array_equal(hv[0], gv[7]) and np.array_equal(hv[3], gv[2])
    assert np.array_equal(hk[[1, 2, 4]], h0k[[1, 2, 4]]) and np.array_equal(hv[[1, 2, 4]], h0v[[1, 2, 4]])


def test_compaction_moves_rows_and_attention_sees_only_the_kept_tokens():
    """Decode over the compacted table equals attention restricted to the kept positions
    (gist.science "Zipage": kept tokens are rewritten into fresh target blocks)."""
    rng = np.random.default_rng(19)
    case = paged_case(rng, [70], 8, 2, 16, dtype="bf16", pool_slack=6)
    L = 70
    keep = np.sort(rng.choice(L, 29, replace=False))
    keep[-1] = L - 1                                   # the newest token is always kept
    keep = np.unique(keep)
    free = sorted(set(range(case["num_blocks"])) - set(case["block_tables"][0].tolist()))
    targets = free[:(len(keep) + 15) // 16]
    src = [int(case["block_tables"][0, p // 16]) * 16 + int(p) % 16 for p in keep]
    dst = [targets[i // 16] * 16 + i % 16 for i in range(len(keep))]
    kc, vc = case["k_cache"].copy(), case["v_cache"].copy()
    assert oracle.compact(kc, vc, src, dst) == 0
    for a, b in zip(src, dst):
        assert np.array_equal(kc[b // 16, :, b % 16], case["k_cache"][a // 16, :, a % 16])
        assert np.array_equal(vc[b // 16, :, b % 16], case["v_cache"][a // 16, :, a % 16])
    bt = np.full((1, len(targets)), -1, np.int32)
    bt[0] = targets
    out, _ = oracle.decode(case["q"], kc, vc, bt, np.array([len(keep)], np.int32), SCALE, "bf16")
    kept = dict(case)
    kept["K"] = [case["K"][0][:, keep, :]]
    kept["V"] = [case["V"][0][:, keep, :]]
    kept["context_lens"] = np.array([len(keep)], np.int32)
    np.testing.assert_allclose(out, sdpa_reference(kept, SCALE), rtol=0, atol=1e-12)
