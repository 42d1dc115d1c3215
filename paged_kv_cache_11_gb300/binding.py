"""ctypes binding of ``libpagedkv.so`` (``include/pagedkv.h``).

Argument marshalling only: tensors become device pointers, the cache tensor's
shape becomes a ``pkv_cache_desc``, and the current PyTorch stream becomes the
``stream`` argument.  Every step of the path runs in the library's kernels.
The library must have been built (``paged_kv_cache_11_gb300._build``); there is
no fallback of any kind.
"""
from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Sequence

import torch

LIB_PATH = Path(__file__).resolve().parent / "_lib" / "libpagedkv.so"

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA, PKV_ERR_DEVICE_METADATA = range(6)
PKV_BF16, PKV_FP16, PKV_FP32 = 0, 1, 2
DEVERR_NAMES = {0: "none", 1: "slot", 2: "copy_id", 3: "context_len", 4: "block_id", 5: "timeout",
                6: "prefix_len", 7: "group"}

_DTYPE_CODE = {torch.bfloat16: PKV_BF16, torch.float16: PKV_FP16, torch.float32: PKV_FP32}


class CacheDesc(ctypes.Structure):
    _fields_ = [
        ("num_blocks", ctypes.c_int64),
        ("num_kv_heads", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


class PagedKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_LIB: ctypes.CDLL | None = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is not None:
        return _LIB
    if not LIB_PATH.exists():
        raise RuntimeError(
            f"{LIB_PATH} is not built; run `python -m paged_kv_cache_11_gb300._build` "
            "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(str(LIB_PATH))
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    desc_p = ctypes.POINTER(CacheDesc)
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_version.argtypes = []
    lib.pkv_version.restype = ctypes.c_int
    lib.pkv_launch_count.argtypes = []
    lib.pkv_launch_count.restype = ctypes.c_uint64
    lib.paged_kv_append.argtypes = [vp, vp, vp, i64, vp, vp, desc_p, vp]
    lib.paged_kv_append.restype = ctypes.c_int
    lib.paged_attention_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.paged_attention_workspace_bytes.restype = sz
    lib.paged_attention_plan.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.paged_attention_plan.restype = i32
    lib.paged_attention_partition_size.argtypes = [i32, i32, i32, i32, i32]
    lib.paged_attention_partition_size.restype = i32
    lib.paged_attention_decode.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, ctypes.c_float, vp, i32,
                                           desc_p, i32, vp, sz, vp]
    lib.paged_attention_decode.restype = ctypes.c_int
    lib.paged_attention_append_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                                  ctypes.c_float, vp, i32, desc_p, i32, vp, sz, vp]
    lib.paged_attention_append_decode.restype = ctypes.c_int
    lib.paged_attention_decode_static.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, ctypes.c_float, vp,
                                                  i32, desc_p, i32, vp]
    lib.paged_attention_decode_static.restype = ctypes.c_int
    lib.paged_attention_decode_grouped.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, vp, i32, i32, vp, i32,
                                                   ctypes.c_float, vp, i32, desc_p, i32, vp, sz, vp]
    lib.paged_attention_decode_grouped.restype = ctypes.c_int
    lib.paged_attention_append_decode_grouped.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, vp, i32,
                                                          i32, vp, i32, ctypes.c_float, vp, i32, desc_p, i32, vp, sz,
                                                          vp]
    lib.paged_attention_append_decode_grouped.restype = ctypes.c_int
    lib.paged_attention_grouped_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.paged_attention_grouped_workspace_bytes.restype = sz
    lib.copy_blocks.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i32, vp, i32, desc_p, vp]
    lib.copy_blocks.restype = ctypes.c_int
    lib.swap_blocks.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i64, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                i64, i32, vp, i32, desc_p, vp]
    lib.swap_blocks.restype = ctypes.c_int
    lib.compact_tokens.argtypes = [vp, vp, i64, vp, vp, desc_p, vp]
    lib.compact_tokens.restype = ctypes.c_int
    lib.pkv_check_device_error.argtypes = [vp, ctypes.POINTER(i32)]
    lib.pkv_check_device_error.restype = ctypes.c_int
    lib.pkv_wait_selftest.argtypes = [i32, vp]
    lib.pkv_wait_selftest.restype = ctypes.c_int
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    return _lib().pkv_status_string(int(status)).decode()


def version() -> int:
    return int(_lib().pkv_version())


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(_lib().pkv_launch_count())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    """Descriptor of a cache tensor shaped [num_blocks, num_kv_heads, block_size, head_dim]."""
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = k_cache.shape
    return CacheDesc(nb, hkv, bs, d, _DTYPE_CODE.get(k_cache.dtype, -1))


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PagedKVError(status, what)


def paged_kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                    v_cache: torch.Tensor, stream=None) -> None:
    """Block write: k_cache[slot // bs, h, slot % bs] = k[t, h] for every token t (same for v)."""
    for t in (k, v, slot_mapping, k_cache, v_cache):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    _require(slot_mapping.dtype == torch.int64, "slot_mapping must be int64")
    desc = cache_desc(k_cache)
    _check(_lib().paged_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), slot_mapping.numel(), _ptr(k_cache),
                                  _ptr(v_cache), ctypes.byref(desc), _stream(stream)), "paged_kv_append")


def paged_attention_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_context_len: int,
                                    partition_size: int = 0) -> int:
    return int(_lib().paged_attention_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                                                      partition_size))


PLAN_NAMES = {0: "single", 1: "split", 2: "split+reduce"}


def paged_attention_plan(num_seqs: int, num_q_heads: int, num_kv_heads: int, block_size: int, max_context_len: int,
                         partition_size: int = 0) -> str:
    """Decomposition a decode call with these sizes uses on the current device."""
    k = int(_lib().paged_attention_plan(num_seqs, num_q_heads, num_kv_heads, block_size, max_context_len,
                                        partition_size))
    return PLAN_NAMES.get(k, "invalid")


def paged_attention_partition_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, max_context_len: int,
                                   partition_size: int = 0) -> int:
    """Split-K partition (tokens) a decode call with these sizes uses on the current device."""
    return int(_lib().paged_attention_partition_size(num_seqs, num_q_heads, num_kv_heads, max_context_len,
                                                     partition_size))


def paged_attention_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                           out: torch.Tensor | None = None, max_context_len: int | None = None,
                           partition_size: int = 0, workspace: torch.Tensor | None = None,
                           out_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """Paged decode attention; returns ``out`` [num_seqs, num_q_heads, head_dim].

    ``max_context_len`` bounds ``context_lens`` (default: the block tables'
    capacity).  A workspace is allocated with torch when one is needed and
    none is given.
    """
    for t in (q, k_cache, v_cache, block_tables, context_lens):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    _require(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32,
             "block_tables and context_lens must be int32")
    _require(q.dim() == 3 and block_tables.dim() == 2, "q is [num_seqs, num_q_heads, head_dim]")
    desc = cache_desc(k_cache)
    num_seqs, hq, d = q.shape
    max_blocks = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = max_blocks * desc.block_size
    if out is None:
        out = torch.empty((num_seqs, hq, d), dtype=out_dtype, device=q.device)
    _require(out.is_cuda and out.is_contiguous(), "out must be a contiguous CUDA tensor")
    need = paged_attention_workspace_bytes(num_seqs, hq, d, max_context_len, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().paged_attention_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks, _ptr(context_lens), num_seqs, hq,
        int(max_context_len), float(scale), _ptr(out), _DTYPE_CODE.get(out.dtype, -1), ctypes.byref(desc),
        int(partition_size), _ptr(workspace), ws_bytes, _stream(stream)), "paged_attention_decode")
    return out


def paged_attention_append_decode(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                  slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                  out: torch.Tensor | None = None, max_context_len: int | None = None,
                                  partition_size: int = 0, workspace: torch.Tensor | None = None,
                                  out_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """One decode step in one launch: write sequence s's new token (k_new[s], v_new[s]) to
    slot_mapping[s] -- the slot of its last context position -- then attend."""
    for t in (q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, context_lens):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == q.shape[0],
             "slot_mapping: int64, one slot per sequence")
    desc = cache_desc(k_cache)
    num_seqs, hq, d = q.shape
    max_blocks = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = max_blocks * desc.block_size
    if out is None:
        out = torch.empty((num_seqs, hq, d), dtype=out_dtype, device=q.device)
    need = paged_attention_workspace_bytes(num_seqs, hq, d, max_context_len, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().paged_attention_append_decode(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        max_blocks, _ptr(context_lens), num_seqs, hq, int(max_context_len), float(scale), _ptr(out),
        _DTYPE_CODE.get(out.dtype, -1), ctypes.byref(desc), int(partition_size), _ptr(workspace), ws_bytes,
        _stream(stream)), "paged_attention_append_decode")
    return out


def paged_attention_grouped_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int, max_context_len: int,
                                            max_prefix_len: int, partition_size: int = 0) -> int:
    return int(_lib().paged_attention_grouped_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                                                              max_prefix_len, partition_size))


def paged_attention_decode_grouped(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                   block_tables: torch.Tensor, context_lens: torch.Tensor, group_starts: torch.Tensor,
                                   prefix_lens: torch.Tensor, scale: float, max_group_size: int,
                                   max_prefix_len: int, out: torch.Tensor | None = None,
                                   max_context_len: int | None = None, partition_size: int = 0,
                                   workspace: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float32,
                                   stream=None) -> torch.Tensor:
    """paged_attention_decode where the sequences group_starts[g] .. group_starts[g+1]-1
    share the blocks of their first prefix_lens[s] tokens with the group's first member;
    shared blocks are read once per (group, KV head)."""
    for t in (q, k_cache, v_cache, block_tables, context_lens, group_starts, prefix_lens):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    for t in (block_tables, context_lens, group_starts, prefix_lens):
        _require(t.dtype == torch.int32, "block_tables, context_lens, group_starts, prefix_lens must be int32")
    _require(q.dim() == 3 and block_tables.dim() == 2 and group_starts.dim() == 1, "bad shapes")
    desc = cache_desc(k_cache)
    num_seqs, hq, d = q.shape
    max_blocks = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = max_blocks * desc.block_size
    if out is None:
        out = torch.empty((num_seqs, hq, d), dtype=out_dtype, device=q.device)
    _require(out.is_cuda and out.is_contiguous(), "out must be a contiguous CUDA tensor")
    need = paged_attention_grouped_workspace_bytes(num_seqs, hq, d, max_context_len, max_prefix_len, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().paged_attention_decode_grouped(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks, _ptr(context_lens), num_seqs, hq,
        int(max_context_len), _ptr(group_starts), group_starts.numel() - 1, int(max_group_size), _ptr(prefix_lens),
        int(max_prefix_len), float(scale), _ptr(out), _DTYPE_CODE.get(out.dtype, -1), ctypes.byref(desc),
        int(partition_size), _ptr(workspace), ws_bytes, _stream(stream)), "paged_attention_decode_grouped")
    return out


def paged_attention_append_decode_grouped(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                                          slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                          block_tables: torch.Tensor, context_lens: torch.Tensor,
                                          group_starts: torch.Tensor, prefix_lens: torch.Tensor, scale: float,
                                          max_group_size: int, max_prefix_len: int, out: torch.Tensor | None = None,
                                          max_context_len: int | None = None, partition_size: int = 0,
                                          workspace: torch.Tensor | None = None,
                                          out_dtype: torch.dtype = torch.float32, stream=None) -> torch.Tensor:
    """One grouped decode step in one call: write sequence s's new token (k_new[s], v_new[s]) to
    slot_mapping[s] -- the slot of its last context position, past its shared prefix -- then
    paged_attention_decode_grouped."""
    for t in (q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, context_lens, group_starts, prefix_lens):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    for t in (block_tables, context_lens, group_starts, prefix_lens):
        _require(t.dtype == torch.int32, "block_tables, context_lens, group_starts, prefix_lens must be int32")
    _require(slot_mapping.dtype == torch.int64 and slot_mapping.numel() == q.shape[0],
             "slot_mapping: int64, one slot per sequence")
    _require(q.dim() == 3 and block_tables.dim() == 2 and group_starts.dim() == 1, "bad shapes")
    desc = cache_desc(k_cache)
    num_seqs, hq, d = q.shape
    max_blocks = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = max_blocks * desc.block_size
    if out is None:
        out = torch.empty((num_seqs, hq, d), dtype=out_dtype, device=q.device)
    _require(out.is_cuda and out.is_contiguous(), "out must be a contiguous CUDA tensor")
    need = paged_attention_grouped_workspace_bytes(num_seqs, hq, d, max_context_len, max_prefix_len, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().paged_attention_append_decode_grouped(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        max_blocks, _ptr(context_lens), num_seqs, hq, int(max_context_len), _ptr(group_starts),
        group_starts.numel() - 1, int(max_group_size), _ptr(prefix_lens), int(max_prefix_len), float(scale),
        _ptr(out), _DTYPE_CODE.get(out.dtype, -1), ctypes.byref(desc), int(partition_size), _ptr(workspace),
        ws_bytes, _stream(stream)), "paged_attention_append_decode_grouped")
    return out


def paged_attention_decode_static(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                                  out: torch.Tensor, max_context_len: int, partition_size: int = 0,
                                  stream=None) -> torch.Tensor:
    """paged_attention_decode for callers that cannot allocate device memory: no
    workspace argument, the split-K partials go to the library's fixed 16 MiB
    device array (calls needing more raise PagedKVError(PKV_ERR_WORKSPACE))."""
    for t in (q, k_cache, v_cache, block_tables, context_lens, out):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    desc = cache_desc(k_cache)
    num_seqs, hq, _ = q.shape
    _check(_lib().paged_attention_decode_static(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
        num_seqs, hq, int(max_context_len), float(scale), _ptr(out), _DTYPE_CODE.get(out.dtype, -1),
        ctypes.byref(desc), int(partition_size), _stream(stream)), "paged_attention_decode_static")
    return out


def copy_blocks(k_caches: torch.Tensor | Sequence[torch.Tensor], v_caches: torch.Tensor | Sequence[torch.Tensor],
                src_dst_pairs: torch.Tensor, stream=None) -> None:
    """Copy-on-write block copy: for each (src, dst) pair, block dst := block src in every layer, K and V."""
    if isinstance(k_caches, torch.Tensor):
        k_caches = [k_caches]
    if isinstance(v_caches, torch.Tensor):
        v_caches = [v_caches]
    _require(len(k_caches) == len(v_caches) and len(k_caches) > 0, "need one K and one V cache per layer")
    for t in (*k_caches, *v_caches, src_dst_pairs):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    _require(src_dst_pairs.dtype == torch.int64 and (src_dst_pairs.numel() % 2 == 0),
             "src_dst_pairs must be int64 [n, 2]")
    desc = cache_desc(k_caches[0])
    n = len(k_caches)
    karr = (ctypes.c_void_p * n)(*[t.data_ptr() for t in k_caches])
    varr = (ctypes.c_void_p * n)(*[t.data_ptr() for t in v_caches])
    _check(_lib().copy_blocks(karr, varr, n, _ptr(src_dst_pairs), src_dst_pairs.numel() // 2, ctypes.byref(desc),
                              _stream(stream)), "copy_blocks")


def _ptr_array(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def swap_blocks(src_k: torch.Tensor | Sequence[torch.Tensor], src_v: torch.Tensor | Sequence[torch.Tensor],
                dst_k: torch.Tensor | Sequence[torch.Tensor], dst_v: torch.Tensor | Sequence[torch.Tensor],
                src_dst_pairs: torch.Tensor, stream=None) -> None:
    """Move whole blocks src -> dst between two pools (GPU or pinned host memory), every layer, K and V."""
    src_k, src_v, dst_k, dst_v = ([t] if isinstance(t, torch.Tensor) else list(t) for t in (src_k, src_v, dst_k, dst_v))
    _require(len(src_k) == len(src_v) == len(dst_k) == len(dst_v) > 0, "one K and one V pool per layer on each side")
    for t in (*src_k, *src_v, *dst_k, *dst_v):
        _require(t.is_contiguous() and (t.is_cuda or t.is_pinned()), "pools must be contiguous, on the GPU or pinned")
    _require(src_dst_pairs.dtype == torch.int64 and src_dst_pairs.numel() % 2 == 0, "src_dst_pairs: int64 [n, 2]")
    _require(src_dst_pairs.is_cuda or src_dst_pairs.is_pinned(), "src_dst_pairs must be GPU-addressable")
    desc = cache_desc(src_k[0])
    _check(_lib().swap_blocks(_ptr_array(src_k), _ptr_array(src_v), src_k[0].shape[0], _ptr_array(dst_k),
                              _ptr_array(dst_v), dst_k[0].shape[0], len(src_k), _ptr(src_dst_pairs),
                              src_dst_pairs.numel() // 2, ctypes.byref(desc), _stream(stream)), "swap_blocks")


def compact_tokens(src_slots: torch.Tensor, dst_slots: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   stream=None) -> None:
    """Move the K/V rows of every head from slot src_slots[i] to slot dst_slots[i]."""
    for t in (src_slots, dst_slots, k_cache, v_cache):
        _require(t.is_cuda and t.is_contiguous(), "tensors must be contiguous CUDA tensors")
    _require(src_slots.dtype == torch.int64 and dst_slots.dtype == torch.int64 and
             src_slots.numel() == dst_slots.numel(), "src_slots/dst_slots: int64 of equal length")
    desc = cache_desc(k_cache)
    _check(_lib().compact_tokens(_ptr(src_slots), _ptr(dst_slots), src_slots.numel(), _ptr(k_cache), _ptr(v_cache),
                                 ctypes.byref(desc), _stream(stream)), "compact_tokens")


def wait_selftest(limit_us: int = 50_000, stream=None) -> None:
    """pkv_wait_selftest: one CTA's bounded wait on a phase nothing completes
    runs out after limit_us and records PKV_DEVERR_TIMEOUT (read it with
    check_device_error)."""
    _check(_lib().pkv_wait_selftest(int(limit_us), _stream(stream)), "pkv_wait_selftest")


def check_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the first device-side error code (0: none)."""
    code = ctypes.c_int32(0)
    st = _lib().pkv_check_device_error(_stream(stream), ctypes.byref(code))
    if st not in (PKV_OK, PKV_ERR_DEVICE_METADATA):
        raise PagedKVError(st, "pkv_check_device_error")
    return int(code.value)
