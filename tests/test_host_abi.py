"""CPU-only checks of the C ABI: the library builds, loads, exports every symbol
that include/gbscan.h declares, and rejects bad arguments before any CUDA call.
No compute call reaches a GPU here."""
import ctypes
import os
import re
import subprocess

import pytest

import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbscan.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gb.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gb_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_api():
    names = declared_functions()
    for need in ("gb_scan_inclusive", "gb_scan_exclusive", "gb_scan_batched", "gb_compact",
                 "gb_partition", "gb_scan_segmented", "gb_pack_by_counts", "gb_scan_reduce_then_scan",
                 "gb_scan_then_fan", "gb_temp_storage_bytes", "gb_device_error", "gb_last_device_error",
                 "gb_status_string"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(gb_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, "declared but not exported: %s" % missing
    assert set(declared_functions()) == set(gb.SIGNATURES), "binding and header disagree"


def test_c_translation_unit_compiles_against_header(tmp_path):
    """The header is plain C: a C program that calls every entry point compiles and links."""
    c = tmp_path / "use.c"
    c.write_text('#include "gbscan.h"\nint main(void){\n'
                 ' size_t t = gb_temp_storage_bytes(GB_KIND_SCAN, GB_F32, 1, 100, 0);\n'
                 ' (void)gb_scan_inclusive; (void)gb_scan_exclusive; (void)gb_scan_batched;\n'
                 ' (void)gb_compact; (void)gb_pack_by_counts; (void)gb_scan_reduce_then_scan;\n'
                 ' (void)gb_partition; (void)gb_scan_segmented; (void)gb_scan_then_fan;\n'
                 ' (void)gb_device_error; (void)gb_last_device_error; (void)gb_last_cuda_error;\n'
                 ' (void)gb_set_profile_events;\n'
                 ' (void)gb_set_wait_limit_ns; (void)gb_set_stalled_tile;\n'
                 ' return t > 0 && gb_version() > 0 ? 0 : 1; }\n')
    exe = tmp_path / "use"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(c),
                           "-o", str(exe), _build.LIB, "-Wl,-rpath," + os.path.dirname(_build.LIB)])
    assert subprocess.run([str(exe)]).returncode == 0


def test_status_strings(lib):
    for code in range(8):
        assert lib.gb_status_string(code).startswith(b"GB_")
    assert lib.gb_version() == 10000


def test_temp_sizes(lib):
    # Row kernel: 4096 fp32 (2048 fp64) per tile, 8-byte packed status for 4-byte types,
    # a flag plus two value slots for 8-byte types; 256-byte header.
    n = 100_000_000
    tiles = (n + 4095) // 4096
    assert lib.gb_temp_storage_bytes(gb.KIND_SCAN, gb.F32, 1, n, 0) == 256 + ((tiles * 8 + 255) // 256) * 256
    t64 = (10_000_000 + 2047) // 2048
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert lib.gb_temp_storage_bytes(gb.KIND_SCAN, gb.F64, 1, 10_000_000, 0) == 256 + r(t64 * 4) + 2 * r(t64 * 8)
    for kind in range(8):
        assert lib.gb_temp_storage_bytes(kind, gb.F32, 1, 12345, 17) > 0
    assert lib.gb_temp_storage_bytes(99, gb.F32, 1, 10, 10) == 0
    assert lib.gb_temp_storage_bytes(gb.KIND_SCAN, 17, 1, 10, 10) == 0
    assert lib.gb_temp_storage_bytes(gb.KIND_SCAN, gb.F32, 0, 10, 10) == 0


def test_argument_checks_before_cuda(lib):
    p = ctypes.c_void_p(256)
    assert lib.gb_scan_inclusive(gb.F32, 1, gb.ADD, p, p, -1, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive(7, 1, gb.ADD, p, p, 10, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive(gb.F32, 1, 5, p, p, 10, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive(gb.F32, 0, gb.ADD, p, p, 10, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive(gb.F32, 1, gb.ADD, None, p, 10, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive(gb.F32, 1, gb.ADD, p, p, 0, None, 0, None) == gb.OK
    assert lib.gb_scan_exclusive(gb.F32, 1, gb.MAX, p, p, 10, None, None, 0, None) == gb.ERR_NO_IDENTITY
    assert lib.gb_scan_exclusive(gb.I32, 1, gb.MIN, p, p, 10, None, None, 0, None) == gb.ERR_NO_IDENTITY
    assert lib.gb_scan_batched(gb.F32, 1, gb.ADD, 1, p, p, 10, 10, 2, None, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_batched(gb.F32, 1, gb.ADD, 1, p, p, 0, 10, 0, None, None, 0, None) == gb.OK
    assert lib.gb_scan_batched(gb.F32, 1, gb.ADD, 1, p, p, 10, 0, 0, None, None, 0, None) == gb.OK
    t = ctypes.c_float(0.5)
    assert lib.gb_compact(gb.F32, p, 1 << 31, gb.LT, ctypes.byref(t), p, p, None, 0, None) == gb.ERR_RANGE
    assert lib.gb_compact(gb.F32, p, 10, 9, ctypes.byref(t), p, p, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_compact(gb.F32, p, 10, gb.LT, None, p, p, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_pack_by_counts(p, -1, None, p, 10, p, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_pack_by_counts(p, 10, None, None, 10, p, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_pack_by_counts(p, 10, None, p, 10, None, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_reduce_then_scan(gb.F32, gb.MAX, 0, p, p, 10, None, None, 0, None) == gb.ERR_NO_IDENTITY
    assert lib.gb_scan_then_fan(gb.F32, gb.MIN, 0, p, p, 10, None, None, 0, None) == gb.ERR_NO_IDENTITY
    assert lib.gb_scan_then_fan(gb.F32, 9, 1, p, p, 10, None, None, 0, None) == gb.ERR_INVALID
    # partition: predicates, the bit split on integers only, bit index range, sizes
    assert lib.gb_partition(gb.F32, p, 1 << 31, gb.LT, ctypes.byref(t), p, None, p, None, 0, None) == gb.ERR_RANGE
    assert lib.gb_partition(gb.F32, p, 10, 7, ctypes.byref(t), p, None, p, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_partition(gb.F32, p, 10, gb.BIT_CLEAR, ctypes.byref(t), p, None, p, None, 0, None) == \
        gb.ERR_UNSUPPORTED
    b32 = ctypes.c_int32(32)
    assert lib.gb_partition(gb.I32, p, 10, gb.BIT_CLEAR, ctypes.byref(b32), p, None, p, None, 0, None) == \
        gb.ERR_INVALID
    assert lib.gb_partition(gb.F32, p, 10, gb.LT, ctypes.byref(t), None, None, p, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_partition(gb.F32, p, 10, gb.LT, ctypes.byref(t), p, None, None, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_partition(gb.F32, ctypes.c_void_p(258), 10, gb.LT, ctypes.byref(t), p, None, p, None, 0, None) == \
        gb.ERR_INVALID  # elements must be naturally aligned
    # segmented: identity rules as for the exclusive scans, flags required
    assert lib.gb_scan_segmented(gb.F32, gb.MAX, 0, p, p, p, 10, None, None, 0, None) == gb.ERR_NO_IDENTITY
    assert lib.gb_scan_segmented(gb.F32, gb.ADD, 1, p, None, p, 10, None, None, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_segmented(gb.F32, gb.ADD, 1, p, p, p, 0, None, None, 0, None) == gb.OK
    # the no-allocation scan: the same checks as gb_scan_inclusive, before any CUDA call
    assert lib.gb_scan_inclusive_noalloc(gb.F32, gb.ADD, p, p, -1, None) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive_noalloc(9, gb.ADD, p, p, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive_noalloc(gb.F32, 5, p, p, 0, None) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive_noalloc(gb.F32, gb.ADD, p, p, 0, None) == gb.OK
    assert lib.gb_scan_inclusive_noalloc(gb.F32, gb.ADD, p, p, 1 << 40, None) == gb.ERR_RANGE
    # the per-call status needs the call's scratch (256-byte aligned)
    assert lib.gb_last_device_error(None, None) == gb.ERR_INVALID
    assert lib.gb_last_device_error(ctypes.c_void_p(258), None) == gb.ERR_INVALID


def test_valid_call_without_gpu_fails_loudly(lib):
    """With no usable GPU a valid call reports GB_ERR_CUDA: there is no CPU fallback."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = ctypes.c_void_p(256)
    assert lib.gb_scan_inclusive(gb.F32, 1, gb.ADD, p, p, 10, None, 0, None) == gb.ERR_CUDA
    assert lib.gb_last_cuda_error() != 0
    with pytest.raises((RuntimeError, ValueError)):
        gb.scan_inclusive(torch.zeros(10))


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(gb, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        gb.load(str(tmp_path / "missing.so"))
