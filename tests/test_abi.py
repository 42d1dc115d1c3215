"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/pagedkv.h declares, and rejects bad arguments on the
host before touching CUDA."""
import ctypes
import re
from pathlib import Path

import pytest

from paged_kv_cache_11_gb300 import _build, binding

HEADER = Path(__file__).resolve().parent.parent / "include" / "pagedkv.h"


@pytest.fixture(scope="module")
def lib():
    _build.build_library()
    return binding._lib()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return re.findall(r"^(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"paged_kv_append", "paged_attention_decode", "copy_blocks", "paged_attention_workspace_bytes",
            "pkv_check_device_error", "pkv_status_string", "pkv_launch_count", "pkv_version",
            "paged_attention_partition_size", "paged_attention_plan", "paged_attention_append_decode",
            "swap_blocks", "compact_tokens", "paged_attention_decode_grouped", "paged_attention_append_decode_grouped",
            "paged_attention_grouped_workspace_bytes", "paged_attention_decode_static", "pkv_wait_selftest"} <= names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_header_compiles_and_links_as_c(lib, tmp_path):
    """The boundary is a C ABI: a C99 program includes the header, links every
    entry point from the library and runs the calls that need no GPU."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("gcc not found")
    exe = tmp_path / "abi_c_program"
    src = Path(__file__).resolve().parent / "abi_c_program.c"
    libdir = binding.LIB_PATH.parent
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", str(HEADER.parent), str(src), "-o",
                        str(exe), "-L", str(libdir), "-lpagedkv", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "c abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)


def test_built_for_sm_103a_only():
    src = (Path(_build.__file__)).read_text()
    assert "arch=compute_103a,code=sm_103a" in src


def test_status_strings(lib):
    assert binding.status_string(0) == "ok"
    assert binding.status_string(3).startswith("workspace")
    assert binding.status_string(99) == "unknown status"
    assert binding.version() >= 100


def _desc(**kw):
    d = dict(num_blocks=64, num_kv_heads=1, block_size=16, head_dim=128, dtype=binding.PKV_BF16)
    d.update(kw)
    return binding.CacheDesc(**d)


def _decode(lib, desc, num_seqs=1, hq=4, max_ctx=16, out_dtype=binding.PKV_FP32, P=0, ws=None, ws_bytes=0,
            maxb=4, ptr=16):
    return lib.paged_attention_decode(ptr, ptr, ptr, ptr, maxb, ptr, num_seqs, hq, max_ctx, 0.1, ptr, out_dtype,
                                      ctypes.byref(desc), P, ws, ws_bytes, None)


def test_decode_host_validation(lib):
    d = _desc()
    assert _decode(lib, d, num_seqs=0) == binding.PKV_OK                     # no-op
    assert _decode(lib, _desc(head_dim=64)) == binding.PKV_ERR_UNSUPPORTED
    assert _decode(lib, _desc(block_size=8)) == binding.PKV_ERR_UNSUPPORTED
    assert _decode(lib, _desc(dtype=binding.PKV_FP32)) == binding.PKV_ERR_UNSUPPORTED
    assert _decode(lib, _desc(num_kv_heads=2), hq=3) == binding.PKV_ERR_INVALID_ARG
    assert _decode(lib, d, max_ctx=65) == binding.PKV_ERR_INVALID_ARG         # above 4 blocks x 16
    assert _decode(lib, d, P=24) == binding.PKV_ERR_INVALID_ARG               # not a multiple of 16
    assert _decode(lib, d, out_dtype=7) == binding.PKV_ERR_INVALID_ARG
    assert _decode(lib, d, ptr=18) == binding.PKV_ERR_INVALID_ARG             # misaligned pointers
    assert _decode(lib, d, max_ctx=64, P=16) == binding.PKV_ERR_WORKSPACE     # split needs a workspace
    assert _decode(lib, d, num_seqs=70000) == binding.PKV_ERR_INVALID_ARG


def test_plan_query(lib):
    assert binding.paged_attention_plan(8, 64, 8, 32, 131072, 0) == "split+reduce"   # long contexts
    assert binding.paged_attention_plan(4, 4, 1, 16, 100, 0) == "single"             # few rows, short
    assert binding.paged_attention_plan(64, 32, 8, 16, 4096, 0) == "split"
    assert binding.paged_attention_plan(64, 32, 8, 16, 4096, 4096) == "single"       # explicit partition
    assert binding.paged_attention_plan(8, 64, 7, 16, 100, 0) == "invalid"


def test_partition_size_query(lib):
    assert binding.paged_attention_partition_size(8, 64, 8, 131072, 256) == 256   # explicit: as given
    assert binding.paged_attention_partition_size(8, 64, 7, 131072, 0) == 0       # 64 % 7 != 0
    assert binding.paged_attention_partition_size(8, 64, 8, 131072, 0) in (512, 1024, 2048, 4096)


def test_partition_choice_for_the_benchmark_shapes(lib):
    """The automatic split-K partition: the largest of 512..4096 tokens that still
    gives two waves of work units.  Without a GPU the library assumes 148 SMs;
    these choices are the same with the GB300's 152."""
    f = binding.paged_attention_partition_size
    assert f(64, 32, 8, 4096, 0) == 1024      # llama8b: 512 rows x 4 partitions
    assert f(8, 64, 8, 131072, 0) == 4096     # llama70b_long: 64 rows x 32 partitions
    assert f(128, 40, 40, 2048, 0) == 4096    # opt13b: one partition per row either way
    assert f(4, 4, 1, 100, 0) == 512          # too little work for longer partitions


def test_workspace_bytes(lib):
    assert binding.paged_attention_workspace_bytes(8, 64, 128, 512, 0) == 0          # one partition
    n = binding.paged_attention_workspace_bytes(8, 64, 128, 131072, 0)
    rows = 8 * 64 * 256
    assert n >= rows * 128 * 4 + rows * 4 and n % 256 == 0
    assert binding.paged_attention_workspace_bytes(-1, 64, 128, 10, 0) == 0


def _grouped(lib, desc, hq=4, max_ctx=64, num_groups=1, max_group=4, max_prefix=32, gs=16, pl=16, ws=None,
             ws_bytes=0, P=0):
    ptr = 16
    return lib.paged_attention_decode_grouped(ptr, ptr, ptr, ptr, 4, ptr, 2, hq, max_ctx, gs, num_groups, max_group,
                                              pl, max_prefix, 0.1, ptr, binding.PKV_FP32, ctypes.byref(desc), P, ws,
                                              ws_bytes, None)


def test_grouped_host_validation(lib):
    d = _desc()
    assert _grouped(lib, d, hq=65) == binding.PKV_ERR_UNSUPPORTED               # > 64 query heads per KV head
    assert _grouped(lib, d, max_prefix=80) == binding.PKV_ERR_INVALID_ARG       # above max_context_len
    assert _grouped(lib, d, max_prefix=-16) == binding.PKV_ERR_INVALID_ARG
    assert _grouped(lib, d, num_groups=-1) == binding.PKV_ERR_INVALID_ARG
    assert _grouped(lib, d, max_group=0) == binding.PKV_ERR_INVALID_ARG
    assert _grouped(lib, d, pl=None) == binding.PKV_ERR_INVALID_ARG              # prefix_lens missing
    assert _grouped(lib, d, gs=None) == binding.PKV_ERR_INVALID_ARG              # group_starts missing
    assert _grouped(lib, d, pl=18) == binding.PKV_ERR_INVALID_ARG                # misaligned
    assert _grouped(lib, d) == binding.PKV_ERR_WORKSPACE                         # always needs one
    assert _grouped(lib, d, ws=256, ws_bytes=1024) == binding.PKV_ERR_WORKSPACE  # too small


def test_grouped_workspace_bytes(lib):
    f = binding.paged_attention_grouped_workspace_bytes
    # partials for ceil(1024 / 256) prefix + ceil(1551 / 512) own partitions per row, plus a group word per sequence
    rows = 256 * 32 * (4 + 4)
    n = f(256, 32, 128, 1551, 1024, 0)
    assert n >= rows * 128 * 4 + rows * 4 + 256 * 4 and n % 256 == 0
    assert f(256, 32, 128, 1551, 0, 0) > 0                   # needed even without a prefix
    assert f(256, 32, 128, 100, 200, 0) == 0                 # prefix above the context bound
    assert f(-1, 32, 128, 100, 0, 0) == 0


def test_append_and_copy_host_validation(lib):
    d = _desc()
    assert lib.paged_kv_append(16, 16, 16, 0, 16, 16, ctypes.byref(d), None) == binding.PKV_OK   # no tokens
    assert lib.paged_kv_append(16, 16, 16, -1, 16, 16, ctypes.byref(d), None) == binding.PKV_ERR_INVALID_ARG
    assert lib.paged_kv_append(None, 16, 16, 4, 16, 16, ctypes.byref(d), None) == binding.PKV_ERR_INVALID_ARG
    assert lib.paged_kv_append(24, 16, 16, 4, 16, 16, ctypes.byref(d), None) == binding.PKV_ERR_INVALID_ARG
    assert lib.paged_kv_append(16, 16, 16, 4, 16, 16, None, None) == binding.PKV_ERR_INVALID_ARG
    arr = (ctypes.c_void_p * 1)(16)
    assert lib.copy_blocks(arr, arr, 1, 16, 0, ctypes.byref(d), None) == binding.PKV_OK             # no pairs
    bad = (ctypes.c_void_p * 1)(20)
    assert lib.copy_blocks(bad, arr, 1, 16, 3, ctypes.byref(d), None) == binding.PKV_ERR_INVALID_ARG
    assert lib.copy_blocks(arr, arr, -1, 16, 3, ctypes.byref(d), None) == binding.PKV_ERR_INVALID_ARG
