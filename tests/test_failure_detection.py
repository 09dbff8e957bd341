"""Failure detection on the GPU without a fault: a bounded wait made to run out.

The test hook bsgemv_plan_set_test_fault makes CTA 0's copy warp leave out one stage of its
range (nothing is copied for it, nothing arrives on its barrier) and lowers every wait's limit to
1 ms.  The consumer warps' wait on that stage then runs out: the kernel must record it, stop
reading its ring, let its copy warp drain what it issued, finish its partial sums and return --
no hang, no fault, the context usable.  bsgemv_device_status then reports
BSGEMV_ERR_DEVICE_TIMEOUT, and the plan's next normal calls give the bits of a call made before
the fault (its arrival counters were left at zero).
"""
import numpy as np
import pytest

from block_scaled_bit_gb300 import bsgemv, synth

pytestmark = pytest.mark.gpu

WAIT_NS = 1_000_000  # 1 ms


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    torch.cuda.set_device(0)
    bsgemv.lib()
    return torch


def cta0_range(g):
    """Stages in CTA 0's range: stream-K floor(T / G), cluster split floor(spt / C)."""
    if g["cluster"] > 0:
        return g["stages_per_tile"] // g["cluster"]
    return g["total_stages"] // g["ctas"]


@pytest.mark.parametrize("fmt,act,bs,zp,N,K,M,split,max_M", [
    ("int8", "f16", 128, True, 2048, 4096, 4, "stream_k", 16),   # tiles shared by several CTAs
    ("int4", "bf16", 32, False, 40000, 2048, 1, "auto", 16),     # long ranges, 128-row tiles
    ("int4", "f16", 32, True, 40000, 2048, 3, "auto", 16),
    ("fp8", "f16", 128, False, 512, 2048, 9, "cluster", 16),     # cluster split, two n8 tiles
    ("nvfp4", "bf16", 16, False, 2048, 2048, 2, "auto", 16),
    ("int4", "f16", 32, False, 12288, 4096, 2, "auto", 8),       # 128-row tiles in 4-CTA clusters
])
@pytest.mark.parametrize("where", ["first", "last"])
def test_a_wait_that_runs_out_is_reported_and_the_plan_recovers(torch_cuda, fmt, act, bs, zp, N,
                                                                 K, M, split, max_M, where):
    torch = torch_cuda
    case = synth.make_case(fmt, act, bs, zp, N, K, M, 31 + N)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan(fmt, act, bs, zp, N, K, max_M) as plan:
        if split == "stream_k":
            assert plan.set_override(ctas=37) == bsgemv.OK
        elif split == "cluster":
            assert plan.set_split("cluster", 4) == bsgemv.OK
        g = plan.describe()
        n0 = cta0_range(g)
        assert n0 >= 2
        # the first stage (copied before the dependency wait) or the last (a ring slot reused)
        skip = 0 if where == "first" else n0 - 1
        plan.run(d.A, d.W, d.scales, d.zp, d.y, M=M)
        torch.cuda.synchronize()
        assert plan.device_status() == bsgemv.OK
        ref = bsgemv.y_bits(d.y)

        assert plan.set_test_fault(skip, WAIT_NS) == bsgemv.OK
        bad = torch.empty_like(d.y)
        plan.run(d.A, d.W, d.scales, d.zp, bad, M=M)
        assert plan.device_status() == bsgemv.ERR_DEVICE_TIMEOUT
        assert plan.device_status() == bsgemv.OK  # read and cleared

        assert plan.set_test_fault(-1, 0) == bsgemv.OK
        for _ in range(2):
            y = torch.full_like(d.y, -1)
            plan.run(d.A, d.W, d.scales, d.zp, y, M=M)
            torch.cuda.synchronize()
            assert plan.device_status() == bsgemv.OK
            assert np.array_equal(bsgemv.y_bits(y), ref)
        assert plan.describe() == g


def test_a_lowered_limit_alone_changes_nothing(torch_cuda):
    """A short limit without a missing stage: every wait still completes in time."""
    torch = torch_cuda
    case = synth.make_case("int4", "f16", 32, True, 12288, 4096, 4, 7)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan("int4", "f16", 32, True, case.N, case.K, 8) as plan:
        plan.run(d.A, d.W, d.scales, d.zp, d.y)
        torch.cuda.synchronize()
        ref = bsgemv.y_bits(d.y)
        assert plan.set_test_fault(-1, 50 * WAIT_NS) == bsgemv.OK
        y = torch.empty_like(d.y)
        plan.run(d.A, d.W, d.scales, d.zp, y)
        assert plan.device_status() == bsgemv.OK
        assert np.array_equal(bsgemv.y_bits(y), ref)


def test_test_hook_arguments(torch_cuda):
    with bsgemv.Plan("int8", "f16", 32, True, 256, 512, 1) as plan:
        assert plan.set_test_fault(-2, 0) == bsgemv.ERR_INVALID_ARG
        assert plan.set_test_fault(0, -1) == bsgemv.ERR_INVALID_ARG
        assert plan.set_test_fault(-1, 0) == bsgemv.OK
