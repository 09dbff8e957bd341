"""Seeded random problems on the GPU: format, block size, zero points, activation type, N, K,
max_M, the call's M, the tile height (automatic, 64 or 128 rows where allowed) and the K split
(automatic, a stream-K CTA count, or a cluster size) drawn together, so that combinations no
hand-written case names are exercised.  Each must match the oracle within its bound on sampled
output columns (all of them when N is small), give the same row bits at a second M of the same
plan, and leave the device status clear."""
import numpy as np
import pytest

import conftest
import oracle
from block_scaled_bit_gb300 import bsgemv, synth

pytestmark = pytest.mark.gpu

FORMATS = [("int4", (16, 32, 64, 128, 256), True), ("int8", (16, 32, 64, 128, 256), True),
           ("fp8", (128,), False), ("nvfp4", (16,), False)]


def draw(i):
    r = np.random.default_rng(20261202 + i)
    fmt, sizes, zp_ok = FORMATS[r.integers(len(FORMATS))]
    bs = int(r.choice(sizes))
    zp = bool(zp_ok and r.integers(2))
    act = ("f16", "bf16")[int(r.integers(2))]
    N = int(r.choice([r.integers(1, 200), r.integers(200, 3000), r.integers(3000, 40000)]))
    unit = max(64, bs)
    K = unit * int(r.integers(1, max(2, 6144 // unit)))
    max_M = int(r.choice([1, 4, 8, 12, 16, 20, 24, 32]))
    M = int(r.integers(1, max_M + 1))
    M2 = int(r.integers(1, max_M + 1))
    rows = int(r.choice([0, 64, 128]))
    split = str(r.choice(["auto", "auto", "stream_k", "cluster"]))
    arg = int(r.integers(1, 700)) if split == "stream_k" else int(r.choice([2, 3, 4, 8]))
    return fmt, bs, zp, act, N, K, max_M, M, M2, rows, split, arg


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    torch.cuda.set_device(0)
    bsgemv.lib()
    return torch


@pytest.mark.parametrize("i", range(48))
def test_random_problem_matches_the_oracle(torch_cuda, i):
    torch = torch_cuda
    fmt, bs, zp, act, N, K, max_M, M, M2, rows, split, arg = draw(i)
    case = synth.make_case(fmt, act, bs, zp, N, K, max(M, M2), 900 + i)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan(fmt, act, bs, zp, N, K, max_M) as plan:
        if rows and plan.set_override(rows_per_tile=rows) != bsgemv.OK:
            assert rows == 128 and max_M > 16  # the only refusal: 128-row tiles above 16 rows
        if split == "stream_k":
            assert plan.set_override(ctas=arg) == bsgemv.OK
        elif split == "cluster":
            plan.set_split("cluster", arg)  # (a size that does not fit leaves the plan as it was)
        outs = {}
        for m in (M, M2):
            y = torch.full((m, N), -1, dtype=torch.int16, device="cuda")
            plan.run(d.A[:m], d.W, d.scales, d.zp, y, M=m)
            torch.cuda.synchronize()
            assert plan.device_status() == bsgemv.OK
            outs[m] = bsgemv.y_bits(y)
        g = plan.describe()
    m = min(M, M2)
    assert np.array_equal(outs[M][:m], outs[M2][:m]), "row bits differ between two M of a plan"
    cols = np.arange(N) if N <= 600 else np.unique(np.concatenate(
        [np.arange(150), np.arange(N - 150, N), np.random.default_rng(i).integers(0, N, 300)]))
    big = max(M, M2)
    bad, worst, _ = oracle.tolerance_violations(case, outs[big][:, cols], rows=cols)
    conftest.record_worst(f"random {i}: {fmt} {act} bs{bs} zp{int(zp)} N{N} K{K} M{big} "
                          f"rows{g['rows_per_tile']} cluster{g['cluster']} ctas{g['ctas']}", worst)
    assert bad == 0, f"{bad} outputs outside the bound (worst {worst:.3g}); geometry {g}"
