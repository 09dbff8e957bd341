"""bsgemv_run_noalloc: the GEMV for callers that cannot allocate device memory (runtimes that own
all device memory up front, code inside another framework's memory pool).  It uses a fixed
scratch area compiled into the library instead of a plan's cudaMalloc'd workspace, and the
geometry of a plan sized for 16 rows whatever the call's M.  So its output must be bit-identical
to the planned entry point's (bsgemv_plan with max_M = 16 + bsgemv_run), within the bound of the
oracle used by every parity test, and the same for a row at every M -- on two calls in a row (the
second reuses the scratch area left by the first).  Its error word is read with
bsgemv_device_status(NULL, stream).

This file is collected last so that a run stopping at the first failure has run every other
test before it.
"""
import numpy as np
import pytest

import oracle
from block_scaled_bit_gb300 import bsgemv, synth

pytestmark = pytest.mark.gpu

CASES = [
    ("int8", "f16", 128, True, 4096, 2048, 1),     # tiles split over several CTAs
    ("int4", "bf16", 32, False, 3000, 4096, 5),    # ragged N
    ("nvfp4", "f16", 16, False, 2048, 2048, 4),
    ("fp8", "f16", 128, False, 512, 2048, 9),      # two n8 tiles
    ("int4", "f16", 32, True, 151936, 4096, 1),    # a large N, most tiles inside one CTA
]


def sample_rows(N):
    return np.unique(np.concatenate([np.arange(min(N, 200)), np.arange(max(0, N - 200), N),
                                     np.random.default_rng(N).integers(0, N, 200)]))


@pytest.mark.parametrize("fmt,act,bs,zp,N,K,M", CASES)
def test_noalloc_matches_planned_entry_point(fmt, act, bs, zp, N, K, M):
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    case = synth.make_case(fmt, act, bs, zp, N, K, M, 4242 + N)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan(fmt, act, bs, zp, N, K, 16) as plan:
        plan.run(d.A, d.W, d.scales, d.zp, d.y, M=M)
        torch.cuda.synchronize()
        assert plan.device_status() == bsgemv.OK
    ref = bsgemv.y_bits(d.y)
    rows = sample_rows(N)
    bad, worst, _ = oracle.tolerance_violations(case, ref[:, rows], rows=rows)
    assert bad == 0, f"planned call: {bad} outputs outside the bound (worst {worst:.3g})"
    for call in range(2):
        y = torch.full_like(d.y, -1)
        status = bsgemv.run_noalloc_status(fmt, act, bs, zp, N, K, d.A, d.W, d.scales, d.zp, y, M=M)
        assert status == bsgemv.OK, bsgemv.status_string(status)
        assert bsgemv.noalloc_device_status() == bsgemv.OK
        got = bsgemv.y_bits(y)
        assert np.array_equal(got, ref), f"call {call}: differs from the planned entry point"
        b2, w2, _ = oracle.tolerance_violations(case, got[:, rows], rows=rows)
        assert b2 == 0, f"call {call}: {b2} outputs outside the bound (worst {w2:.3g})"


def test_noalloc_rows_are_the_same_for_every_M():
    """A row computed in a 1-row call and in a 9-row call (one and two n8 tiles) is bit-identical:
    the call's geometry does not depend on M."""
    import torch
    torch.cuda.set_device(0)
    case = synth.make_case("int4", "f16", 32, True, 12288, 4096, 16, 99)
    d = bsgemv.upload(case, "cuda")
    outs = {}
    for M in (1, 8, 9, 16):
        y = torch.full((M, case.N), -1, dtype=torch.int16, device="cuda")
        status = bsgemv.run_noalloc_status("int4", "f16", 32, True, case.N, case.K, d.A[:M], d.W,
                                           d.scales, d.zp, y, M=M)
        assert status == bsgemv.OK
        torch.cuda.synchronize()
        outs[M] = bsgemv.y_bits(y)
    for M in (1, 8, 9):
        assert np.array_equal(outs[M], outs[16][:M]), f"M={M}"


def test_noalloc_rejects_problems_beyond_its_scratch_area():
    import torch
    torch.cuda.set_device(0)
    dummy = torch.zeros(64, dtype=torch.int16, device="cuda")
    # 8193 tiles of 64 output columns: one more than the scratch area holds
    status = bsgemv.run_noalloc_status("int8", "f16", 128, False, 8193 * 64, 128, dummy, dummy,
                                       dummy, None, dummy, M=1)
    assert status == bsgemv.ERR_SCRATCH_LIMIT
    assert "scratch" in bsgemv.status_string(status)
    assert bsgemv.noalloc_device_status() == bsgemv.OK
