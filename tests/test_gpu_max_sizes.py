"""GPU checks at the largest sizes the API accepts, against closed forms computed on
the device (the arrays are too large to carry to the host oracle): scans past 2^31
elements (64-bit positions), compaction and partition at n = 2^31 - 1 (their 32-bit
index limit).  Inputs are built with torch on the device; the expected values are the
closed forms, never the library's own output.
"""
import pytest
import torch

import stream_compaction_decoupled_gb300 as gb

pytestmark = pytest.mark.gpu

BIG = 2**31 + 4099


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gb.load()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_int32_ones_past_2_31():
    """Inclusive add of ones: out[i] = i + 1 modulo 2^32 (two's complement); the
    exclusive scan is the same shifted by one."""
    x = torch.ones(BIG, dtype=torch.int32, device="cuda")
    y = gb.scan_inclusive(x)
    want = torch.arange(1, BIG + 1, dtype=torch.int64, device="cuda")
    want = ((want + 2**31) % 2**32 - 2**31).to(torch.int32)
    assert torch.equal(y, want)
    del y
    e = gb.scan_exclusive(x)
    assert int(e[0].item()) == 0 and torch.equal(e[1:], want[:-1])
    assert gb.device_error() == gb.OK


def test_int64_max_scan_past_2_31():
    """Max-scan of an ascending sequence is the sequence itself; a single late spike
    then holds to the end."""
    x = torch.arange(BIG, dtype=torch.int64, device="cuda")
    x[BIG - 10] = 2**40
    y = gb.scan_inclusive(x, "max")
    assert torch.equal(y[: BIG - 10], x[: BIG - 10])
    assert bool((y[BIG - 10:] == 2**40).all())
    assert gb.device_error() == gb.OK


def test_compact_and_partition_at_the_index_limit():
    """n = 2^31 - 1 alternating 0, 1, 0, ...: x < 0.5 selects exactly the even indices."""
    n = 2**31 - 1
    x = (torch.arange(n, dtype=torch.int32, device="cuda") & 1).to(torch.float32)
    evens = torch.arange(0, n, 2, dtype=torch.int32, device="cuda")
    odds = torch.arange(1, n, 2, dtype=torch.int32, device="cuda")
    idx, cnt = gb.compact(x, "lt", 0.5)
    m = int(cnt.item())
    assert m == evens.numel() and torch.equal(idx[:m], evens)
    del idx
    out, pidx, pcnt = gb.partition(x, "lt", 0.5)
    assert int(pcnt.item()) == m
    assert torch.equal(pidx[:m], evens) and torch.equal(pidx[m:n], odds)
    assert bool((out[:m] == 0).all()) and bool((out[m:n] == 1).all())
    assert gb.device_error() == gb.OK
