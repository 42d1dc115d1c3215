"""Seeded synthetic workloads: the input generator shared by the tests, the
benchmark and the oracle's callers.

It holds no attention arithmetic.  Numbers come from ``libpkvgen.so``
(counter-based SplitMix64, Box-Muller N(0,1), IEEE round-to-nearest-even into
bf16/fp16); block tables, slot mappings and copy-on-write pairs come from the
host block manager run over a seeded permutation of the pool.

The five workloads mirror the shapes the pages size (page, section):

* ``tiny`` -- 4 sequences of {1, 17, 33, 100} tokens, 4 query / 1 KV head, a
  64-block pool; parity only.
* ``llama8b`` -- Llama-3-8B-class layer (briefia.fr "L'ampleur du cache KV":
  32 layers, 8 KV heads, head dim 128, 2 bytes): 32 query / 8 KV heads, bf16,
  block 16, 64 sequences with contexts uniform in [512, 4096].
* ``opt13b`` -- OPT-13B-class MHA layer (tonho.wtf "vllm", "o problema": 800 KB
  per token = 2 x 5120 x 40 layers x 2 B, hidden 5120 = 40 heads x 128): 40/40
  heads, fp16, block 16, 128 sequences, contexts uniform in [1, 2048]; each
  step appends one token per sequence (a fresh block when the last is full).
* ``shared_prefix`` -- parallel sampling (tonho.wtf "vllm", "como funciona"):
  16 groups of 16 sequences; each group's prompt of 1024 + t_g tokens
  (t_g uniform in [1, 15]) is mapped by all 16 samples (reference count 16),
  so its last block is shared and partly filled; each sample holds its own
  32-512 token continuation, whose first write into the shared block copied
  it (15 copies per group; the 16th sample wrote in place).  The step is a
  decode step: the 240 copy-on-write pairs of the shared partial blocks,
  then one new token per sample (256 tokens), then attention.  The copies
  are repeated every step; each rewrites the same bytes (the prompt's
  partial block, whose slots past the prompt are then the first
  continuation tokens of the copying samples).
* ``shared_prefix_prefill`` -- the same batch, with each sample's whole
  continuation written by the step (about 68k tokens appended) before the
  attention.
* ``llama70b_long`` -- Llama-3.1-70B-class long context (aitalk.it
  "PagedAttention e RadixAttention", opening: 0.31 MB per token, 128k tokens
  ~ 40 GB): 64 query / 8 KV heads, bf16, block 32, 8 sequences of 131072
  tokens; 4 GiB of K+V per layer.

Stated sizes and distributions are from the workload table; where the pages
print no distribution (the value of K, V and q) the entries are N(0, 1).
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass, field, replace
from pathlib import Path

import numpy as np

from .block_manager import BlockManager

GEN_PATH = Path(__file__).resolve().parent / "_lib" / "libpkvgen.so"

# stream ids of the generator
S_K_POOL, S_V_POOL, S_Q, S_NEW_K, S_NEW_V, S_LENS, S_PERM, S_GROUP = 1, 2, 3, 4, 5, 6, 7, 8
DTYPE_CODE = {"bf16": 0, "fp16": 1}
NAN_BITS = {"bf16": 0x7FC0, "fp16": 0x7E00}

_GEN = None


def _gen():
    global _GEN
    if _GEN is None:
        if not GEN_PATH.exists():
            raise RuntimeError(f"{GEN_PATH} is not built; run `python -m paged_kv_cache_11_gb300._build`")
        lib = ctypes.CDLL(str(GEN_PATH))
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.pkvgen_normal.argtypes = [u64, u64, u64, i64, ctypes.c_int, vp, ctypes.c_int]
        lib.pkvgen_normal.restype = ctypes.c_int
        lib.pkvgen_u64_fill.argtypes = [u64, u64, u64, i64, vp]
        lib.pkvgen_u64_fill.restype = None
        lib.pkvgen_round_f32.argtypes = [vp, i64, ctypes.c_int, vp]
        lib.pkvgen_round_f32.restype = None
        _GEN = lib
    return _GEN


def default_threads() -> int:
    import os
    return max(1, min(64, os.cpu_count() or 1))


def normal(seed: int, stream: int, shape, dtype: str, offset: int = 0, threads: int | None = None) -> np.ndarray:
    """N(0,1) samples of the (seed, stream) sequence, as raw 16-bit patterns (bf16/fp16) or float32."""
    n = int(np.prod(shape))
    code = {"bf16": 0, "fp16": 1, "fp32": 2}[dtype]
    out = np.empty(n, dtype=np.float32 if dtype == "fp32" else np.uint16)
    rc = _gen().pkvgen_normal(seed, stream, offset, n, code, out.ctypes.data, threads or default_threads())
    if rc != 0:
        raise RuntimeError("pkvgen_normal failed")
    return out.reshape(shape)


def u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _gen().pkvgen_u64_fill(seed, stream, offset, n, out.ctypes.data)
    return out


def round_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """The generator's fp32 -> bf16/fp16 rounding (exposed for its tests)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _gen().pkvgen_round_f32(x.ctypes.data, x.size, DTYPE_CODE[dtype], out.ctypes.data)
    return out


def uniform_ints(seed: int, stream: int, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    """n integers uniform in [lo, hi] (modulo reduction of 64-bit draws)."""
    r = u64(seed, stream, n, offset)
    return (lo + (r % np.uint64(hi - lo + 1))).astype(np.int64)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of range(n) driven by the (seed, stream) sequence."""
    r = u64(seed, stream, max(n - 1, 0))
    a = np.arange(n, dtype=np.int64)
    for k, i in enumerate(range(n - 1, 0, -1)):
        j = int(r[k] % np.uint64(i + 1))
        a[i], a[j] = a[j], a[i]
    return a


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, elt_bytes: int) -> int:
    """K and V bytes one token occupies: 2 x layers x KV heads x head_dim x bytes per value
    (briefia.fr "L'ampleur du cache KV"; tonho.wtf "vllm", "o problema")."""
    return 2 * num_layers * num_kv_heads * head_dim * elt_bytes


@dataclass(frozen=True)
class Spec:
    name: str
    index: int
    num_q_heads: int
    num_kv_heads: int
    block_size: int
    dtype: str
    num_seqs: int = 0
    lens: tuple = ()              # ("fixed", [...]) or ("uniform", lo, hi)
    pool_factor: float = 1.25
    pool_blocks: int = 0          # fixed pool size (0: pool_factor x blocks needed)
    head_dim: int = 128
    # shared-prefix workloads
    groups: int = 0
    per_group: int = 0
    prefix: int = 0
    tail: tuple = (1, 15)
    suffix: tuple = (32, 512)
    # "decode": the step appends each sample's last token; "continuation": its
    # whole continuation
    step: str = "decode"

    @property
    def kind(self) -> str:
        return "shared_prefix" if self.groups else "decode"


SPECS = {
    "tiny": Spec("tiny", 0, 4, 1, 16, "bf16", num_seqs=4, lens=("fixed", (1, 17, 33, 100)), pool_blocks=64),
    "llama8b": Spec("llama8b", 1, 32, 8, 16, "bf16", num_seqs=64, lens=("uniform", 512, 4096)),
    "opt13b": Spec("opt13b", 2, 40, 40, 16, "fp16", num_seqs=128, lens=("uniform", 1, 2048)),
    "shared_prefix": Spec("shared_prefix", 3, 32, 8, 16, "bf16", groups=16, per_group=16, prefix=1024),
    "shared_prefix_prefill": Spec("shared_prefix_prefill", 3, 32, 8, 16, "bf16", groups=16, per_group=16,
                                  prefix=1024, step="continuation"),
    "llama70b_long": Spec("llama70b_long", 4, 64, 8, 32, "bf16", num_seqs=8, lens=("fixed", (131072,) * 8),
                          pool_factor=1.0),
}


def default_seed(spec: Spec) -> int:
    return 0x9E3779B9 ^ spec.index


@dataclass
class Workload:
    spec: Spec
    seed: int
    num_blocks: int
    context_lens: np.ndarray      # int32 [B], tokens attended (including this step's)
    block_tables: np.ndarray      # int32 [B, max_blocks]; -1 past the sequence's blocks
    slot_mapping: np.ndarray      # int64 [T], slots written by this step's append
    append_seq: np.ndarray        # int32 [T], the sequence of each appended token
    cow_pairs: np.ndarray         # int64 [n, 2], copied before the append
    k_cache: np.ndarray | None = None   # uint16 [nb, Hkv, bs, D] pool before the step
    v_cache: np.ndarray | None = None
    q: np.ndarray | None = None         # uint16 [B, Hq, D]
    new_k: np.ndarray | None = None     # uint16 [T, Hkv, D]
    new_v: np.ndarray | None = None
    groups: np.ndarray | None = None    # int32 [B], group of each sequence (shared_prefix)
    meta: dict = field(default_factory=dict)

    # -- shape helpers ---------------------------------------------------
    @property
    def dtype(self) -> str:
        return self.spec.dtype

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_q_heads(self) -> int:
        return self.spec.num_q_heads

    @property
    def num_kv_heads(self) -> int:
        return self.spec.num_kv_heads

    @property
    def head_dim(self) -> int:
        return self.spec.head_dim

    @property
    def block_size(self) -> int:
        return self.spec.block_size

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.head_dim)

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def elt_bytes(self) -> int:
        return 2

    def kv_bytes(self) -> int:
        """K+V bytes of the attended contexts (logical: shared blocks counted once per sequence)."""
        return int(self.context_lens.astype(np.int64).sum()) * kv_bytes_per_token(
            1, self.num_kv_heads, self.head_dim, self.elt_bytes)

    def unique_kv_bytes(self) -> int:
        """K+V bytes of the distinct physical slots the decode reads."""
        slots = set()
        bs = self.block_size
        for s in range(self.num_seqs):
            L = int(self.context_lens[s])
            for j in range((L + bs - 1) // bs):
                n = min(bs, L - j * bs)
                slots.update((int(self.block_tables[s, j]), o) for o in range(n))
        return len(slots) * kv_bytes_per_token(1, self.num_kv_heads, self.head_dim, self.elt_bytes)

    def valid_slot_mask(self) -> np.ndarray:
        """bool [num_blocks, block_size]: slots holding a token of some context after the step."""
        bs = self.block_size
        mask = np.zeros((self.num_blocks, bs), dtype=bool)
        for s in range(self.num_seqs):
            L = int(self.context_lens[s])
            nb = (L + bs - 1) // bs
            ids = self.block_tables[s, :nb].astype(np.int64)
            if nb:
                mask[ids[:-1], :] = True
                mask[ids[-1], : L - (nb - 1) * bs] = True
        return mask

    def poison(self) -> None:
        """Write NaN into every pool slot that no context reads after the step, into the
        slots this step's append writes, and into every copy-on-write destination block,
        so that a missed mask, append or copy shows up in the result."""
        nan = NAN_BITS[self.dtype]
        bad = ~self.valid_slot_mask()
        good = self.slot_mapping[self.slot_mapping >= 0]
        bad[good // self.block_size, good % self.block_size] = True
        if len(self.cow_pairs):
            bad[self.cow_pairs[:, 1], :] = True
        for cache in (self.k_cache, self.v_cache):
            cache.transpose(0, 2, 1, 3)[bad] = nan


def _lengths(spec: Spec, seed: int, num_seqs: int, lens) -> np.ndarray:
    kind = lens[0]
    if kind == "fixed":
        vals = np.asarray(lens[1], dtype=np.int64)
        if len(vals) != num_seqs:
            vals = np.resize(vals, num_seqs)
        return vals
    lo, hi = lens[1], lens[2]
    return uniform_ints(seed, S_LENS, num_seqs, lo, hi)


def make_workload(name: str, seed: int | None = None, with_data: bool = True, threads: int | None = None,
                  **overrides) -> Workload:
    """Build a workload.  ``overrides`` replace fields of the spec (e.g. num_seqs,
    lens=("uniform", lo, hi), groups, per_group, prefix, suffix, pool_blocks)."""
    spec = replace(SPECS[name], **overrides) if overrides else SPECS[name]
    if seed is None:
        seed = default_seed(spec)
    bs = spec.block_size

    def run(bm: BlockManager):
        slots, app_seq, cows, lens, groups = [], [], [], [], []
        if spec.kind == "decode":
            L = _lengths(spec, seed, spec.num_seqs, spec.lens)
            for s in range(spec.num_seqs):
                bm.add_sequence(s)
                if L[s] == 0:
                    lens.append(0)
                    continue
                bm.append_tokens(s, int(L[s]) - 1)          # the context already in the cache
                slot, cow = bm.append_token(s)               # this step's token
                slots.append(slot)
                app_seq.append(s)
                if cow:
                    cows.append(cow)
                lens.append(int(L[s]))
                groups.append(s)
        else:
            G, M = spec.groups, spec.per_group
            tails = uniform_ints(seed, S_GROUP, G, spec.tail[0], spec.tail[1])
            sufs = uniform_ints(seed, S_LENS, G * M, spec.suffix[0], spec.suffix[1])
            parent = G * M
            for g in range(G):
                bm.add_sequence(parent + g)
                bm.append_tokens(parent + g, spec.prefix + int(tails[g]))
                for i in range(M):
                    bm.fork(parent + g, g * M + i)
                bm.free(parent + g)                          # the samples hold the prompt blocks
            whole = spec.step == "continuation"
            for g in range(G):
                for i in range(M):
                    s = g * M + i
                    n = int(sufs[s])
                    # decode step: the continuation but its last token is in
                    # the cache already (its copy-on-write pair is repeated
                    # by the step); the last token is this step's
                    sl, cw = bm.append_tokens(s, n if whole else n - 1)
                    if not whole:
                        slot, c1 = bm.append_token(s)
                        sl = [slot]
                        cw += [c1] if c1 else []
                    slots += sl
                    app_seq += [s] * len(sl)
                    cows += cw
                    lens.append(bm.num_tokens(s))
                    groups.append(g)
        return slots, app_seq, cows, lens, groups

    # first pass on an unbounded pool to size the real one
    probe = BlockManager(1 << 22, bs) if spec.pool_blocks == 0 else None
    if probe is not None:
        run(probe)
        needed = (1 << 22) - probe.num_free
        num_blocks = max(1, math.ceil(spec.pool_factor * needed))
    else:
        num_blocks = spec.pool_blocks
    bm = BlockManager(num_blocks, bs, permutation(seed, S_PERM, num_blocks))
    slots, app_seq, cows, lens, groups = run(bm)
    B = len(lens)
    tables = [bm.block_table(s) for s in range(B)]
    maxb = max(1, max(len(t) for t in tables))
    bt = np.full((B, maxb), -1, dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, : len(t)] = t
    wl = Workload(
        spec=spec, seed=seed, num_blocks=num_blocks,
        context_lens=np.asarray(lens, dtype=np.int32),
        block_tables=bt,
        slot_mapping=np.asarray(slots, dtype=np.int64),
        append_seq=np.asarray(app_seq, dtype=np.int32),
        cow_pairs=np.asarray(cows, dtype=np.int64).reshape(-1, 2),
        groups=np.asarray(groups, dtype=np.int32),
    )
    if with_data:
        fill_data(wl, threads=threads)
    return wl


def fill_data(wl: Workload, threads: int | None = None) -> None:
    spec, seed = wl.spec, wl.seed
    D, hkv, bs = spec.head_dim, spec.num_kv_heads, spec.block_size
    T = len(wl.slot_mapping)
    wl.k_cache = normal(seed, S_K_POOL, (wl.num_blocks, hkv, bs, D), spec.dtype, threads=threads)
    wl.v_cache = normal(seed, S_V_POOL, (wl.num_blocks, hkv, bs, D), spec.dtype, threads=threads)
    wl.q = normal(seed, S_Q, (wl.num_seqs, spec.num_q_heads, D), spec.dtype, threads=threads)
    wl.new_k = normal(seed, S_NEW_K, (T, hkv, D), spec.dtype, threads=threads)
    wl.new_v = normal(seed, S_NEW_V, (T, hkv, D), spec.dtype, threads=threads)


def prefix_groups(wl: Workload) -> tuple[np.ndarray, np.ndarray, int]:
    """Shared-prefix groups of a workload, as grouped decode takes them.

    A group is a run of consecutive sequences with the same ``groups`` id (a
    workload without one per sequence makes every sequence its own group).
    A member's prefix length is the whole blocks its block table shares with
    the group's first member, within both contexts; every member of a group
    gets the smallest of these, and a group of one shares nothing.

    Returns (group_starts int32 [num_groups + 1], prefix_lens int32 [B],
    largest group size).
    """
    B, bs = wl.num_seqs, wl.block_size
    ids = wl.groups if wl.groups is not None and len(wl.groups) == B else np.arange(B)
    starts = [0] + [s for s in range(1, B) if ids[s] != ids[s - 1]] + [B]
    plen = np.zeros(B, dtype=np.int32)
    for a, b in zip(starts[:-1], starts[1:]):
        if b - a < 2:
            continue
        common = None
        for s in range(a + 1, b):
            n = min(int(wl.context_lens[a]), int(wl.context_lens[s])) // bs
            same = wl.block_tables[s, :n] == wl.block_tables[a, :n]
            k = n if same.all() else int(np.argmin(same))
            common = k if common is None else min(common, k)
        plen[a:b] = common * bs
    sizes = np.diff(starts)
    return np.asarray(starts, dtype=np.int32), plen, int(sizes.max()) if len(sizes) else 1


def make_grouped_workload(seed: int, members: list[list[tuple[int, int]]], num_q_heads: int, num_kv_heads: int,
                          block_size: int, dtype: str, pool_factor: float = 1.25,
                          threads: int | None = None) -> tuple[Workload, np.ndarray, np.ndarray, int]:
    """A decode batch of forked groups for grouped decode, without a decode step's append.

    ``members[g]`` lists (prefix_len, context_len) per member of group g, in
    order; prefix lengths are multiples of ``block_size``.  The group's first
    member is the parent: it holds the longest prefix, and each other member
    is forked from it when the parent's context reaches that member's prefix
    length, so the member shares exactly those blocks; every member then
    writes its own tokens up to its context length.  A group of one with
    prefix 0 is a plain sequence.

    Returns (workload, group_starts, prefix_lens, largest group size).
    """
    bs = block_size
    spec = Spec("grouped", 9, num_q_heads, num_kv_heads, bs, dtype, pool_factor=pool_factor)

    def run(bm: BlockManager):
        seq, lens, gid, plens, starts = 0, [], [], [], [0]
        for g, mem in enumerate(members):
            lead = seq
            order = sorted(range(1, len(mem)), key=lambda i: mem[i][0])
            top = max(p for p, _ in mem)
            assert all(p % bs == 0 for p, _ in mem) and top <= mem[0][1] and all(p <= L for p, L in mem)
            bm.add_sequence(lead)
            for i in order:                          # parent grows; fork each member at its prefix
                bm.append_tokens(lead, mem[i][0] - bm.num_tokens(lead))
                bm.fork(lead, lead + i)
            bm.append_tokens(lead, mem[0][1] - bm.num_tokens(lead))
            for i in range(1, len(mem)):
                bm.append_tokens(lead + i, mem[i][1] - bm.num_tokens(lead + i))
            for i, (p, L) in enumerate(mem):
                lens.append(L)
                gid.append(g)
                plens.append(p if i else (top if len(mem) > 1 else p))
            seq += len(mem)
            starts.append(seq)
        return lens, gid, plens, starts

    probe = BlockManager(1 << 22, bs)
    run(probe)
    num_blocks = max(1, math.ceil(pool_factor * ((1 << 22) - probe.num_free)))
    bm = BlockManager(num_blocks, bs, permutation(seed, S_PERM, num_blocks))
    lens, gid, plens, starts = run(bm)
    B = len(lens)
    tables = [bm.block_table(s) for s in range(B)]
    maxb = max(1, max(len(t) for t in tables))
    bt = np.full((B, maxb), -1, dtype=np.int32)
    for s, t in enumerate(tables):
        bt[s, : len(t)] = t
    wl = Workload(spec=spec, seed=seed, num_blocks=num_blocks, context_lens=np.asarray(lens, dtype=np.int32),
                  block_tables=bt, slot_mapping=np.zeros(0, dtype=np.int64), append_seq=np.zeros(0, dtype=np.int32),
                  cow_pairs=np.zeros((0, 2), dtype=np.int64), groups=np.asarray(gid, dtype=np.int32))
    fill_data(wl, threads=threads)
    sizes = [len(m) for m in members]
    return wl, np.asarray(starts, dtype=np.int32), np.asarray(plens, dtype=np.int32), max(sizes) if sizes else 1
