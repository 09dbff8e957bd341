"""Both tile heights on every format: 64-row tiles (one weight box per stage and k-box) and
128-row tiles (two 64-row halves, each consumer warp owning a 16-row group of both), forced
through bsgemv_plan_set_override's rows_per_tile on shapes that choose the other height on their
own.  Each must match the oracle within its bound at every M of the plan, keep every row
bit-identical across M, and repeat bit for bit; N ragged against both tile heights, K ragged
against the stage ("[CUDA] Block-scaled MatMul decode GEMV: tensor cores, packed FP4 decode and
M-tiling", description, row-tiling paragraph: rows per block as a tuning choice; the results do
not depend on it beyond the summation order)."""
import numpy as np
import pytest

import conftest
import oracle
from block_scaled_bit_gb300 import bsgemv, synth

pytestmark = pytest.mark.gpu

CASES = [
    ("int4", "f16", 32, True, 1000, 2112),     # N = 7 x 128 + 104, K = 8 x 256 + 64
    ("int4", "bf16", 16, False, 4500, 1024),
    ("int8", "f16", 128, True, 3000, 2304),    # K = 9 x 256 (one-half stages), 18 x 128 (two)
    ("int8", "bf16", 32, False, 700, 1088),
    ("fp8", "f16", 128, False, 2200, 1920),
    ("fp8", "bf16", 128, False, 333, 4096),
    ("nvfp4", "f16", 16, False, 5000, 2048),
    ("nvfp4", "bf16", 16, False, 130, 512),
]


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    torch.cuda.set_device(0)
    bsgemv.lib()
    return torch


@pytest.mark.parametrize("rows_per_tile", [64, 128])
@pytest.mark.parametrize("split", ["auto", "stream_k", "cluster"])
@pytest.mark.parametrize("fmt,act,bs,zp,N,K", CASES)
def test_both_tile_heights_match_the_oracle(torch_cuda, fmt, act, bs, zp, N, K, split,
                                            rows_per_tile):
    torch = torch_cuda
    case = synth.make_case(fmt, act, bs, zp, N, K, 16, 700 + N)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan(fmt, act, bs, zp, N, K, 16) as plan:
        assert plan.set_override(rows_per_tile=rows_per_tile) == bsgemv.OK
        if split == "stream_k":
            assert plan.set_override(ctas=61) == bsgemv.OK
        elif split == "cluster" and plan.set_split("cluster", 2) != bsgemv.OK:
            pytest.skip("a 2-CTA cluster split does not fit this shape")
        g = plan.describe()
        assert g["rows_per_tile"] == rows_per_tile
        assert g["tiles"] == -(-N // rows_per_tile)
        outs = {}
        for M in (16, 1, 9, 16):
            y = torch.full((M, N), -1, dtype=torch.int16, device="cuda")
            plan.run(d.A[:M], d.W, d.scales, d.zp, y, M=M)
            torch.cuda.synchronize()
            assert plan.device_status() == bsgemv.OK
            got = bsgemv.y_bits(y)
            if M in outs:
                assert np.array_equal(got, outs[M]), "a repeated call differs"
            outs[M] = got
        bad, worst, _ = oracle.tolerance_violations(case, outs[16])
        conftest.record_worst(f"tile_rows {rows_per_tile} {split} {fmt} {act} bs{bs} N{N} K{K}",
                              worst)
        assert bad == 0, f"{bad} outputs outside the bound (worst {worst:.3g})"
        for M in (1, 9):
            assert np.array_equal(outs[M], outs[16][:M]), f"row bits differ at M={M}"


def test_tile_height_override_rules(torch_cuda):
    with bsgemv.Plan("int4", "f16", 32, False, 4096, 4096, 16) as plan:
        assert plan.set_override(rows_per_tile=96) == bsgemv.ERR_INVALID_ARG
        assert plan.set_override(rows_per_tile=128) == bsgemv.OK
        assert plan.describe()["rows_per_tile"] == 128
        assert plan.set_override(rows_per_tile=64) == bsgemv.OK
        assert plan.describe()["rows_per_tile"] == 64
    # 128-row tiles exist for kernels of up to 16 rows, and not for the CUDA-core variant
    with bsgemv.Plan("int4", "f16", 32, False, 4096, 4096, 17) as plan:
        g = plan.describe()
        assert plan.set_override(rows_per_tile=128) == bsgemv.ERR_UNSUPPORTED
        assert plan.describe() == g
    with bsgemv.Plan("int4", "f16", 32, False, 4096, 4096, 8) as plan:
        assert plan.set_override(variant=bsgemv.VARIANTS["cuda_core"]) == bsgemv.OK
        assert plan.set_override(rows_per_tile=128) == bsgemv.ERR_UNSUPPORTED
        assert plan.describe()["rows_per_tile"] == 64
