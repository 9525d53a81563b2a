"""The inclusive scan that allocates nothing (gb_scan_inclusive_noalloc).

It serves callers that cannot call cudaMalloc or cudaMallocAsync, such as code
running under an allocator it does not own, or code that must not grow device
memory after start-up: its scratch is a static device array inside the library.
These tests call it through the C ABI and compare it with the ordinary entry point
(gb_scan_inclusive with caller-supplied scratch), with the float tolerance the other
parity tests use, on two calls in a row, so a second call that inherits the first
call's scratch contents is checked too.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 1 << 20  # the array's size, as documented in include/gbscan.h


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _reference(x, op):
    """The same scan through the ordinary entry point, scratch from torch."""
    code = gb.dtype_code(x.dtype)
    out = torch.empty_like(x)
    nbytes = gb.load().gb_temp_storage_bytes(gb.KIND_SCAN, code, 1, x.numel(), 0)
    temp = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    rc = gb.load().gb_scan_inclusive(code, 1, gb.OPS[op], _ptr(x), _ptr(out), x.numel(), _ptr(temp), nbytes,
                                     _stream())
    assert rc == gb.OK
    return out


def _no_alloc(x, op):
    out = torch.empty_like(x)
    rc = gb.load().gb_scan_inclusive_noalloc(gb.dtype_code(x.dtype), gb.OPS[op], _ptr(x), _ptr(out),
                                             x.numel(), _stream())
    assert rc == gb.OK, gb.load().gb_status_string(rc)
    return out


def _close(got, want, x):
    if got.dtype.is_floating_point:
        bound = 1e-5 * torch.cumsum(x.double().abs(), 0) + 1e-6
        return bool(((got.double() - want.double()).abs() <= bound).all())
    return bool(torch.equal(got, want))


@pytest.mark.parametrize("dtype,op,n", [(torch.float32, "add", 3 * 4096 + 77), (torch.float32, "add", 2_000_003),
                                        (torch.int32, "add", 1_000_000), (torch.float64, "max", 500_001),
                                        (torch.int64, "min", 40_000)])
def test_no_alloc_matches_ordinary_entry_point_twice(dtype, op, n):
    assert torch.cuda.is_available()
    gb.load()
    if dtype.is_floating_point:
        x = torch.from_numpy(workloads.normal(n, np.dtype(str(dtype).split(".")[1]), 21)).cuda()
    else:
        x = torch.from_numpy(workloads.small_ints(n, 21, -1000, 1000, dtype=np.dtype(str(dtype).split(".")[1]))).cuda()
    want = _reference(x, op)
    first = _no_alloc(x, op)
    # A different input in between, then the same input again: the scratch array
    # keeps the previous call's contents and must be cleared by the call.
    other = _no_alloc(torch.flip(x, [0]).contiguous(), op)
    second = _no_alloc(x, op)
    torch.cuda.synchronize()
    assert _close(first, want, x)
    assert _close(second, want, x)
    assert _close(other, _reference(torch.flip(x, [0]).contiguous(), op), torch.flip(x, [0]))
    assert gb.device_error() == gb.OK


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    lib = gb.load()
    x = torch.zeros(16, dtype=torch.float32, device="cuda")
    too_big = (SCRATCH_BYTES - 256) // 8 * 4096 + 1   # one tile more than the status words fit
    assert lib.gb_temp_storage_bytes(gb.KIND_SCAN, gb.F32, 1, too_big, 0) > SCRATCH_BYTES
    rc = lib.gb_scan_inclusive_noalloc(gb.F32, gb.ADD, _ptr(x), _ptr(x), too_big, _stream())
    assert rc == gb.ERR_RANGE
    fits = too_big - 1
    assert lib.gb_temp_storage_bytes(gb.KIND_SCAN, gb.F32, 1, fits, 0) <= SCRATCH_BYTES
    assert lib.gb_scan_inclusive_noalloc(gb.F32, gb.ADD, _ptr(x), _ptr(x), -1, _stream()) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive_noalloc(gb.F32, gb.ADD, _ptr(x), _ptr(x), 0, _stream()) == gb.OK
