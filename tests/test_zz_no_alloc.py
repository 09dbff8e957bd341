"""bsgemv_run_noalloc: the GEMV for callers that cannot allocate device memory (runtimes that own
all device memory up front, code inside another framework's memory pool).  It uses a fixed
scratch area compiled into the library instead of a plan's cudaMalloc'd workspace; its output
must match the planned entry point's (bsgemv_plan + bsgemv_run) within the tolerance used by
every parity test, on two calls in a row (the second call reuses the scratch area left by the
first).

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


@pytest.mark.parametrize("fmt,act,bs,zp,N,K,M", CASES)
def test_noalloc_matches_planned_entry_point(fmt, act, bs, zp, N, K, M):
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    case = synth.make_case(fmt, act, bs, zp, N, K, M, 4242 + N)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan(fmt, act, bs, zp, N, K, M) as plan:
        plan.run(d.A, d.W, d.scales, d.zp, d.y, M=M)
        torch.cuda.synchronize()
    ref = oracle.act_values(bsgemv.y_bits(d.y), act)
    rows = np.unique(np.concatenate([np.arange(min(N, 200)), np.arange(max(0, N - 200), N),
                                     np.random.default_rng(N).integers(0, N, 200)]))
    _, _, absdot = oracle.gemv(case, rows=rows)
    bound = oracle.ulp(ref[:, rows], act) + 1e-3 * absdot
    for call in range(2):
        y = torch.full_like(d.y, -1)
        status = bsgemv.run_noalloc_status(fmt, act, bs, zp, N, K, d.A, d.W, d.scales, d.zp, y, M=M)
        assert status == bsgemv.OK, bsgemv.status_string(status)
        torch.cuda.synchronize()
        got = oracle.act_values(bsgemv.y_bits(y), act)
        assert np.all(np.abs(got[:, rows] - ref[:, rows]) <= bound), f"call {call}"
        assert np.all(np.isfinite(got))


def test_noalloc_rejects_problems_beyond_its_scratch_area():
    import torch
    torch.cuda.set_device(0)
    dummy = torch.zeros(64, dtype=torch.int16, device="cuda")
    # 8193 tiles of 64 output columns: one more than the scratch area holds
    status = bsgemv.run_noalloc_status("int8", "f16", 128, False, 8193 * 64, 128, dummy, dummy,
                                       dummy, None, dummy, M=1)
    assert status == bsgemv.ERR_SCRATCH_LIMIT
    assert "scratch" in bsgemv.status_string(status)
