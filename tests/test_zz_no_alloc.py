"""The inclusive scan that allocates nothing (gb_scan_inclusive_noalloc).

It serves callers that cannot call cudaMalloc or cudaMallocAsync, such as code
running under an allocator it does not own, or code that must not grow device
memory after start-up: its scratch is a static device array inside the library.
These tests call it through the C ABI and check it against the CPU oracle (bit for
bit for integers, within the float tolerance the other parity tests use) and against
the ordinary entry point, on two calls in a row with a different input between them,
so a call that inherits the previous call's scratch contents is checked too.  The
cases reach every kernel the entry point can run on the array: the segment kernel
(aligned rows up to 96 MiB), the L2-resident look-back kernel (aligned rows past
96 MiB, up to the 1e8 size of the benchmark's headline) and the row kernel (views
that are not 16-byte aligned).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads
from parity import as3, assert_scan_matches

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 1 << 20  # the array's size, as documented in include/gbscan.h


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ordinary(x, op):
    """The same scan through the ordinary entry point, scratch from torch."""
    code = gb.dtype_code(x.dtype)
    out = torch.empty_like(x)
    nbytes = gb.load().gb_temp_storage_bytes(gb.KIND_SCAN, code, 1, x.numel(), 0)
    temp = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    rc = gb.load().gb_scan_inclusive(code, 1, gb.OPS[op], _ptr(x), _ptr(out), x.numel(), _ptr(temp), nbytes,
                                     _stream())
    assert rc == gb.OK
    torch.cuda.synchronize()
    return out


def _no_alloc(x, op, out):
    rc = gb.load().gb_scan_inclusive_noalloc(gb.dtype_code(x.dtype), gb.OPS[op], _ptr(x), _ptr(out),
                                             x.numel(), _stream())
    assert rc == gb.OK, gb.load().gb_status_string(rc)
    return out


def _view(x_host, off):
    """x on the device, `off` elements past a 256-byte aligned allocation (off > 0
    leaves the view without 16-byte alignment), and an output view like it."""
    base = torch.empty(x_host.size + off, dtype=torch.from_numpy(x_host[:1]).dtype, device="cuda")
    base[off:].copy_(torch.from_numpy(x_host))
    out = torch.empty_like(base)
    return base[off:], out[off:]


def _check(got, x_host, op, what):
    if x_host.dtype.kind == "f":
        assert_scan_matches(got.cpu().numpy(), as3(x_host, 1, x_host.size, 1), op, True, what=what)
    else:
        want = torch.from_numpy(oracle.scan(x_host, op)).cuda()
        assert torch.equal(got, want), what


def _close(a, b, x_host):
    """Two GPU results agree: bit for bit for integers, within twice the float bound."""
    if not a.dtype.is_floating_point:
        return bool(torch.equal(a, b))
    xd = torch.from_numpy(x_host).cuda().double()
    bound = 2e-5 * torch.cumsum(xd.abs(), 0) + 2e-6
    return bool(((a.double() - b.double()).abs() <= bound).all())


CASES = [
    (np.float32, "add", 3 * 4096 + 77, 0),
    (np.float32, "add", 2_000_003, 0),
    (np.int32, "add", 1_000_000, 0),
    (np.float64, "max", 500_001, 0),
    (np.int64, "min", 40_000, 0),
    (np.float32, "add", 30_000_001, 0),     # past 96 MiB: the L2-resident look-back kernel
    (np.int32, "add", 100_000_000, 0),      # the headline's size, exact integer sums
    (np.float32, "add", 1_000_003, 1),      # not 16-byte aligned: the row kernel
    (np.int64, "add", 700_001, 1),
    (np.int32, "max", 5_000_001, 3),
]


@pytest.mark.parametrize("dtype,op,n,off", CASES)
def test_no_alloc_matches_oracle_twice(dtype, op, n, off):
    assert torch.cuda.is_available()
    gb.load()
    if np.dtype(dtype).kind == "f":
        x = workloads.normal(n, dtype, 21)
    else:
        x = workloads.small_ints(n, 21, -1000, 1000, dtype=dtype)
    xd, out = _view(x, off)
    rev = np.ascontiguousarray(x[::-1])
    rd, rout = _view(rev, off)
    first = _no_alloc(xd, op, out).clone()
    # A different input in between, then the same input again: the scratch array
    # keeps the previous call's contents and must be cleared by the call.
    other = _no_alloc(rd, op, rout)
    second = _no_alloc(xd, op, out)
    torch.cuda.synchronize()
    what = "%s %s n=%d off=%d" % (np.dtype(dtype).name, op, n, off)
    _check(first, x, op, what + " first call")
    _check(second, x, op, what + " second call")
    _check(other, rev, op, what + " reversed input")
    assert _close(second, _ordinary(xd, op), x), what + ": differs from gb_scan_inclusive"
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
    # the type and operator are checked even when there is nothing to scan
    assert lib.gb_scan_inclusive_noalloc(9, gb.ADD, _ptr(x), _ptr(x), 0, _stream()) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive_noalloc(gb.F32, 7, _ptr(x), _ptr(x), 0, _stream()) == gb.ERR_INVALID
