"""The oracle -- TEST INFRASTRUCTURE, not part of the product path.

A plain, slow fp64 CPU statement of what the paged KV cache decode path
computes (``pkv_oracle.c``), loaded through ctypes.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs
may import it.  It shares no code with ``paged_kv_cache_11_gb300`` and imports
nothing from it; it takes raw 16-bit element patterns in numpy arrays.

Functions (sources cited in ``pkv_oracle.c``):

* ``append``      -- block write of new K/V rows into their slots
* ``copy_blocks`` -- whole-block copy of (src, dst) pairs
* ``swap_blocks`` -- whole-block moves between two pools (swap out / in)
* ``compact``     -- token-row moves into fresh target blocks (Zipage)
* ``decode``      -- softmax(scale * q . K) V over each sequence's context,
                     gathered through its block table; optional partitioned
                     (split-K) form and optional subset of (seq, head) outputs
* ``to_f64``      -- exact decode of bf16 / fp16 bit patterns

Parity of every function is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "pkv_oracle.c"
LIB = HERE / "_build" / "libpkv_oracle.so"
DTYPES = {"bf16": 0, "fp16": 1}

_LIB = None


def build(force: bool = False) -> Path:
    """Compile the oracle (gcc, -O2, no fast-math)."""
    LIB.parent.mkdir(exist_ok=True)
    if force or not LIB.exists() or LIB.stat().st_mtime < SRC.stat().st_mtime:
        tmp = LIB.with_suffix(".so.tmp")
        r = subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread", str(SRC), "-o",
                            str(tmp), "-lm"], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


def _lib():
    global _LIB
    if _LIB is None:
        build()
        lib = ctypes.CDLL(str(LIB))
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_elem_to_f64.argtypes = [ctypes.c_uint16, i32]
        lib.oracle_elem_to_f64.restype = ctypes.c_double
        lib.oracle_to_f64.argtypes = [vp, i64, i32, vp]
        lib.oracle_to_f64.restype = None
        lib.oracle_append.argtypes = [vp, vp, vp, i64, vp, vp, i64, i32, i32, i32]
        lib.oracle_append.restype = i64
        lib.oracle_copy_blocks.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32]
        lib.oracle_copy_blocks.restype = i64
        lib.oracle_swap_blocks.argtypes = [vp, vp, i64, vp, vp, i64, vp, i64, i32, i32, i32]
        lib.oracle_swap_blocks.restype = i64
        lib.oracle_compact.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32]
        lib.oracle_compact.restype = i64
        lib.oracle_decode.argtypes = [i32, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i64, ctypes.c_double,
                                      i32, vp, vp, i64, vp, i32]
        lib.oracle_decode.restype = i64
        _LIB = lib
    return _LIB


def _u16(a: np.ndarray, name: str) -> np.ndarray:
    if a.dtype != np.uint16 or not a.flags.c_contiguous:
        raise TypeError(f"{name} must be a C-contiguous uint16 array of raw element bits")
    return a


def to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _lib().oracle_to_f64(bits.ctypes.data, bits.size, DTYPES[dtype], out.ctypes.data)
    return out


def append(k, v, slot_mapping, k_cache, v_cache) -> int:
    """In place on the host caches [nb, Hkv, bs, D]; returns the count of out-of-pool slots."""
    k, v, kc, vc = (_u16(a, n) for a, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")))
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, hkv, bs, d = kc.shape
    return int(_lib().oracle_append(k.ctypes.data, v.ctypes.data, sm.ctypes.data, sm.size, kc.ctypes.data,
                                    vc.ctypes.data, nb, hkv, bs, d))


def copy_blocks(k_cache, v_cache, pairs) -> int:
    kc, vc = _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    nb, hkv, bs, d = kc.shape
    return int(_lib().oracle_copy_blocks(kc.ctypes.data, vc.ctypes.data, pr.ctypes.data, pr.shape[0], nb, hkv, bs, d))


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs) -> int:
    """Whole blocks src (of the source pool) -> dst (of the destination pool), in place on dst."""
    sk, sv, dk, dv = (_u16(a, n) for a, n in ((src_k, "src_k"), (src_v, "src_v"), (dst_k, "dst_k"), (dst_v, "dst_v")))
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    _, hkv, bs, d = sk.shape
    return int(_lib().oracle_swap_blocks(sk.ctypes.data, sv.ctypes.data, sk.shape[0], dk.ctypes.data, dv.ctypes.data,
                                         dk.shape[0], pr.ctypes.data, pr.shape[0], hkv, bs, d))


def compact(k_cache, v_cache, src_slots, dst_slots) -> int:
    """Token rows src slot -> dst slot (every head, K and V), in place."""
    kc, vc = _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    a = np.ascontiguousarray(src_slots, dtype=np.int64)
    b = np.ascontiguousarray(dst_slots, dtype=np.int64)
    nb, hkv, bs, d = kc.shape
    return int(_lib().oracle_compact(kc.ctypes.data, vc.ctypes.data, a.ctypes.data, b.ctypes.data, a.size, nb, hkv,
                                     bs, d))


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: str, partition_size: int = 0,
           select=None, threads: int = 1):
    """Returns (out float64 [B, Hq, D], status int32 [B]); status 1 marks bad metadata (zero output).

    ``select``: optional iterable of (seq, q_head) pairs; other outputs stay 0.
    """
    q, kc, vc = _u16(q, "q"), _u16(k_cache, "k_cache"), _u16(v_cache, "v_cache")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = kc.shape
    if d2 != d or vc.shape != kc.shape or bt.shape[0] != B or cl.shape[0] != B:
        raise ValueError("shape mismatch")
    out = np.zeros((B, hq, d), dtype=np.float64)
    status = np.zeros(B, dtype=np.int32)
    sel = None
    nsel = 0
    if select is not None:
        sel = np.ascontiguousarray(np.asarray(list(select), dtype=np.int32).reshape(-1, 2))
        nsel = sel.shape[0]
    rc = _lib().oracle_decode(DTYPES[dtype], q.ctypes.data, kc.ctypes.data, vc.ctypes.data, bt.ctypes.data,
                              bt.shape[1], cl.ctypes.data, B, hq, hkv, bs, d, nb, float(scale), int(partition_size),
                              out.ctypes.data, None if sel is None else sel.ctypes.data, nsel, status.ctypes.data,
                              int(threads))
    if rc < 0:
        raise ValueError("oracle_decode rejected its arguments")
    return out, status
