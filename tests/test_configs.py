"""Every synthetic workload configuration at its full size, in the launch configuration the
benchmark times (plan max_M = the configuration's largest M, default geometry), checked against the oracle on sampled
output columns: the first and last two tiles (ragged tail included) and a seeded random
sample in between, for every M of the configuration."""
import numpy as np
import pytest

import conftest
import oracle
from block_scaled_bit_gb300 import bsgemv, synth

pytestmark = pytest.mark.gpu

SHAPES = synth.all_shapes()


def sample_rows(N, seed, k=96):
    rng = np.random.default_rng(seed)
    edge = list(range(min(N, 128))) + list(range(max(0, N - 128), N))
    mid = rng.integers(0, N, size=k).tolist()
    return np.unique(np.array(edge + mid, dtype=np.int64))


@pytest.mark.parametrize("shape", SHAPES, ids=[s.name for s in SHAPES])
def test_full_size_config(shape):
    import torch
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    case = shape.case(max(shape.Ms))
    d = bsgemv.upload(case, "cuda")
    rows = sample_rows(case.N, shape.seed)
    with bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp, case.N, case.K,
                     max(shape.Ms)) as plan:
        outs = {}
        for M in shape.Ms:
            y = torch.empty((M, case.N), dtype=torch.int16, device="cuda")
            plan.run(d.A[:M], d.W, d.scales, d.zp, y, M=M)
            torch.cuda.synchronize()
            outs[M] = bsgemv.y_bits(y)
        assert plan.device_status() == bsgemv.OK
    top = outs[max(shape.Ms)]
    bad, worst, _ = oracle.tolerance_violations(case, top[:, rows], rows=rows)
    conftest.record_worst(f"full-size {shape.name} M={max(shape.Ms)}", worst)
    assert bad == 0, f"{bad} sampled outputs outside the bound (worst {worst:.3g})"
    for M, y in outs.items():
        # each smaller M is bit-identical to the first M rows of the largest
        assert np.array_equal(y, top[:M]), f"M={M} differs from rows of M={max(shape.Ms)}"
    # properties that hold at any size: no NaN/inf for these finite, in-range inputs
    vals = oracle.act_values(top, case.act)
    assert np.all(np.isfinite(vals))
