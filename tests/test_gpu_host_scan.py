"""GPU parity of the host-buffer scan (gb_scan_inclusive_host): chunks copied in,
scanned with the running total of the chunks before them, and copied out, with the
copies overlapping the scans; compared with the oracle element by element."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import stream_compaction_decoupled_gb300 as gb
from stream_compaction_decoupled_gb300 import workloads
from parity import as3, assert_scan_matches

pytestmark = pytest.mark.gpu

NP = {"i32": np.int32, "f32": np.float32, "f64": np.float64, "i64": np.int64, "u32": np.uint32}


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()


def make(dt, n, seed):
    if dt.startswith("f"):
        return workloads.normal(n, NP[dt], seed)
    if dt.startswith("u"):  # the whole range: max/min must compare as unsigned
        return workloads.full_range_uints(n, seed, NP[dt])
    return workloads.small_ints(n, seed, -1000, 1000, dtype=NP[dt])


def host(x, pinned=True):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.pin_memory() if pinned else t


def run(x, op, chunk, pinned=True):
    xh = host(x, pinned)
    out = gb.scan_inclusive_host(xh, op, chunk_elems=chunk)
    torch.cuda.current_stream().synchronize()
    return out.numpy()


@pytest.mark.parametrize("dt", ["i32", "u32", "f32", "i64", "f64"])
@pytest.mark.parametrize("op", ["add", "max", "min"])
@pytest.mark.parametrize("n,chunk", [(1, 0), (4096, 4096), (10_000, 4096), (100_003, 16_384), (1_000_001, 65_536),
                                     (257, 16)])
def test_host_scan_chunks(dt, op, n, chunk):
    if dt == "u32" and not hasattr(torch, "uint32"):
        pytest.skip("no torch uint32")
    x = make(dt, n, n % 977 + chunk % 13)
    got = run(x, op, chunk)
    assert_scan_matches(got, as3(x, 1, n, 1), op, True, what="host %s %s n=%d chunk=%d" % (dt, op, n, chunk))
    assert gb.device_error() == gb.OK


def test_host_scan_default_chunks_large():
    """120 MB of fp32 in the default 48 MiB chunks (three chunks, the last ragged)."""
    x = workloads.normal(30_000_001, np.float32, 3)
    got = run(x, "add", 0)
    assert_scan_matches(got, as3(x, 1, x.size, 1), "add", True, what="host fp32 3e7")
    xi = workloads.small_ints(30_000_001, 4, -5, 6)
    assert np.array_equal(run(xi, "add", 0), oracle.scan(xi))


def test_host_scan_in_place_pageable_and_work_buffer():
    x = workloads.small_ints(500_000, 8, -9, 10)
    want = oracle.scan(x)
    xh = host(x)
    gb.scan_inclusive_host(xh, out=xh, chunk_elems=65_536)  # in place
    torch.cuda.current_stream().synchronize()
    assert np.array_equal(xh.numpy(), want)
    assert np.array_equal(run(x, "add", 100_000, pinned=False), want)  # pageable
    nb = gb.host_scan_work_bytes(torch.int32, x.size, 100_000)
    work = torch.empty(nb, dtype=torch.uint8, device="cuda")
    out = gb.scan_inclusive_host(host(x), chunk_elems=100_000, work=work)
    torch.cuda.current_stream().synchronize()
    assert np.array_equal(out.numpy(), want)


def test_host_scan_back_to_back_calls():
    """Calls queued one after another share the library's copy streams and events."""
    xs = [workloads.small_ints(300_007, 20 + i, -50, 51) for i in range(4)]
    outs = [gb.scan_inclusive_host(host(x), chunk_elems=32_768) for x in xs]
    torch.cuda.current_stream().synchronize()
    for x, o in zip(xs, outs):
        assert np.array_equal(o.numpy(), oracle.scan(x))


def test_host_scan_argument_errors():
    lib = gb.load()
    x = host(np.zeros(16, dtype=np.float32))
    p = ctypes.c_void_p(x.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.gb_scan_inclusive_host(gb.F32, gb.ADD, None, p, 16, 0, None, 0, s) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive_host(9, gb.ADD, p, p, 16, 0, None, 0, s) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive_host(gb.F32, gb.ADD, p, p, -1, 0, None, 0, s) == gb.ERR_INVALID
    assert lib.gb_scan_inclusive_host(gb.F32, gb.ADD, p, p, 0, 0, None, 0, s) == gb.OK
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    assert lib.gb_scan_inclusive_host(gb.F32, gb.ADD, p, p, 16, 0, ctypes.c_void_p(small.data_ptr()), 64,
                                      s) == gb.ERR_TEMP
    assert lib.gb_host_scan_work_bytes(gb.F32, 0, 0) == 0
