"""GPU pins without a tolerance: the CUDA library (through the C ABI) against the CPU oracle where
the result has exactly one right answer.

1. Every code of every format through the GEMV's own register decoders (bsgemv_debug_dequant),
   bit-exact to the oracle's dequantised weight (rounded once to fp32; NaN where the oracle has
   NaN): all 256 E4M3 codes as FP8 weights and as NVFP4 block scales (0x00, subnormals, 0x7E = 448,
   the NaN codes 0x7F / 0xFF), all 16 E2M1 codes under every block-scale code, every (q, zp) pair
   of int4 and int8.  The decode-GEMV page ("[CUDA] Block-scaled MatMul decode GEMV: tensor cores,
   packed FP4 decode and M-tiling", description, FP8 and NVFP4 tensor-core paragraphs) states the
   exactness the decoders rely on (E4M3 lossless in f16 / bf16, the E2M1 x E4M3 fold exact), and its
   prmt-decode paragraph sweeps every byte the same way.
2. NaN codes through bsgemv_run: NaN in exactly the outputs where the oracle has NaN.
3. Inputs on which every fp32 partial sum is exact (small-integer activations, power-of-two block
   scales, coarse weight grids; see synth.exact_case): the GEMV output must be the oracle's bits,
   whatever the summation order -- so a dropped, doubled or misplaced scale block fails here even
   at K = 2048, where the 1e-3 * sum|a w| bound could not see it.  Every format and block size,
   both activation types, every K split (stream-K, cluster, the CUDA-core variant), M = 1 / 9 / 16
   / 32.
4. One-hot activations (row m = e_{k_m}): y[m, n] = round(deq[n, k_m]) exactly -- the lane
   ownership probe of the decode-GEMV page's review (a row / column swap fails instead of
   cancelling).
"""
import numpy as np
import pytest

import conftest
import oracle
from block_scaled_bit_gb300 import bsgemv, synth

pytestmark = pytest.mark.gpu

ACTS = ("f16", "bf16")
INT_BS = (16, 32, 64, 128, 256)
FMTS = ([("int4", bs, z) for bs in INT_BS for z in (True, False)]
        + [("int8", bs, z) for bs in INT_BS for z in (True, False)]
        + [("fp8", 128, False), ("nvfp4", 16, False)])
# grid of every partial sum of synth.exact_case (NVFP4 after its 2^-6 global scale): the sum is
# exact in fp32 while sum_k |a_k w_k| < 2^24 grid steps
EXACT_GRID = {"int4": 2.0 ** -2, "int8": 2.0 ** -2, "fp8": 2.0 ** -6, "nvfp4": 2.0 ** -9}


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    torch.cuda.set_device(0)
    bsgemv.lib()
    return torch


def same_values(a_bits, b_bits, act):
    """Elementwise: the same value, or both NaN.  For fp16 / bf16 this is bit identity except
    for the sign of a zero (a sum of zero terms is +0 under round-to-nearest, the zero weight
    itself may be -0) and the payload of a NaN, neither of which is part of the result."""
    a = oracle.act_values(a_bits, act)
    b = oracle.act_values(b_bits, act)
    return (a == b) | (np.isnan(a) & np.isnan(b))


def run_plan(plan, case, M=None):
    import torch
    M = case.M if M is None else M
    d = bsgemv.upload(case, "cuda")
    plan.run(d.A, d.W, d.scales, d.zp, d.y, M=M)
    torch.cuda.synchronize()
    assert plan.device_status() == bsgemv.OK
    return bsgemv.y_bits(d.y)


def configure(plan, how):
    """Force the K split / variant under test; False if this plan cannot take it."""
    if how == "stream_k":
        return plan.set_override(ctas=37) == bsgemv.OK
    if how == "cluster":
        return plan.set_split("cluster", 4) == bsgemv.OK
    if how == "cuda_core":
        return plan.set_override(variant=bsgemv.VARIANTS["cuda_core"]) == bsgemv.OK
    return True


# ---------------------------------------------------------------------------- 1. every code
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("fmt,bs,zp", FMTS)
def test_every_code_decodes_bit_exact(torch_cuda, fmt, bs, zp, act):
    torch = torch_cuda
    N = 70  # four full 16-row groups and a ragged one
    case = synth.all_codes_case(fmt, act, bs, zp, N, 1, 31 + bs)
    d = bsgemv.upload(case, "cuda")
    out = torch.full((case.N, case.K), 7.0, dtype=torch.float32, device="cuda")
    with bsgemv.Plan(fmt, act, bs, zp, case.N, case.K, 1) as plan:
        plan.debug_dequant(d.W, d.scales, d.zp, out)
        torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = oracle.dequant(case).astype(np.float32)  # exact value, rounded once to fp32
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    bad = np.argwhere(~same)
    assert bad.size == 0, (f"{len(bad)} dequantised values differ, first at (n, k) = "
                           f"{tuple(bad[0])}: {got[tuple(bad[0])]!r} vs {want[tuple(bad[0])]!r}")
    if fmt in ("fp8", "nvfp4"):  # the NaN codes are in every row: NaN must be there
        assert np.isnan(got).any(axis=1).all()


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("fmt,bs,zp", [f for f in FMTS if f[0] in ("int4", "int8")])
@pytest.mark.parametrize("M", [1, 9])
def test_every_int_code_through_the_gemv(torch_cuda, fmt, bs, zp, act, M):
    """The all-codes weights (every (q, zp) pair, extreme q - zp = +-255) through bsgemv_run:
    within the bound of the oracle."""
    case = synth.all_codes_case(fmt, act, bs, zp, 70, M, 77 + bs)
    with bsgemv.Plan(fmt, act, bs, zp, case.N, case.K, 16) as plan:
        y = run_plan(plan, case)
    bad, worst, _ = oracle.tolerance_violations(case, y)
    conftest.record_worst(f"every_int_code {fmt} bs{bs} zp{int(zp)} {act} M{M}", worst)
    assert bad == 0, f"{bad} outputs outside the bound (worst error/bound {worst:.3g})"


# ---------------------------------------------------------------------------- 2. NaN codes
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
@pytest.mark.parametrize("how,M", [("auto", 1), ("auto", 9), ("auto", 16), ("stream_k", 4),
                                   ("cluster", 3), ("cuda_core", 1), ("cuda_core", 6)])
def test_nan_codes_reach_exactly_the_oracles_nan_outputs(torch_cuda, fmt, act, how, M):
    N, K = 357, 2048
    nan_rows = [0, 5, 63, 64, 200, 356]
    case = synth.nan_rows_case(fmt, act, N, K, M, 900 + M, nan_rows)
    with bsgemv.Plan(fmt, act, 128 if fmt == "fp8" else 16, False, N, K,
                     8 if how == "cuda_core" else 16) as plan:
        assert configure(plan, how)
        y = run_plan(plan, case)
    ref_bits, _, _ = oracle.gemv(case)
    ref_nan = np.isnan(oracle.act_values(ref_bits, act))
    assert ref_nan[:, nan_rows].all() and ref_nan.sum() == M * len(nan_rows)  # the case itself
    y_nan = np.isnan(oracle.act_values(y, act))
    assert np.array_equal(y_nan, ref_nan), f"NaN at {np.argwhere(y_nan != ref_nan)[:5].tolist()}"
    bad, worst, _ = oracle.tolerance_violations(case, y)
    conftest.record_worst(f"nan_codes {fmt} {act} {how} M{M}", worst)
    assert bad == 0, f"{bad} outputs outside the bound (worst error/bound {worst:.3g})"


# ---------------------------------------------------------------------------- 3. exact sums
@pytest.mark.parametrize("how", ["auto", "stream_k", "cluster", "cuda_core"])
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("fmt,bs,zp", FMTS)
def test_exact_inputs_give_the_oracles_bits(torch_cuda, fmt, bs, zp, act, how):
    N, K = 357, 2048
    Ms = (1, 8) if how == "cuda_core" else (1, 9, 16, 32)
    for M in Ms:
        case = synth.exact_case(fmt, act, bs, zp, N, K, M, 500 + bs)
        ref_bits, _, absdot = oracle.gemv(case)
        # the inputs keep every partial sum exact in fp32 (else the pin would not hold)
        assert absdot.max() < 2.0 ** 24 * EXACT_GRID[fmt]
        max_M = 8 if how == "cuda_core" else (32 if M > 16 else 16)
        with bsgemv.Plan(fmt, act, bs, zp, N, K, max_M) as plan:
            if not configure(plan, how):
                assert how == "cluster" and M > 16, f"{how} refused at M={M}"
                continue
            y = run_plan(plan, case)
        diff = np.argwhere(~same_values(y, ref_bits, act))
        assert diff.size == 0, (f"M={M}: {len(diff)} outputs differ from the oracle's bits, first "
                                f"(m, n) = {tuple(diff[0])}")


# ---------------------------------------------------------------------------- 4. one-hot rows
@pytest.mark.parametrize("how", ["auto", "stream_k", "cuda_core"])
@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("fmt,bs,zp", FMTS)
def test_one_hot_rows_select_one_dequantised_weight(torch_cuda, fmt, bs, zp, act, how):
    N, K = 300, 2048
    M = 8 if how == "cuda_core" else 16
    case, ks = synth.one_hot_case(fmt, act, bs, zp, N, K, M, 700 + bs)
    deq = oracle.dequant(case)                         # exact, [N, K]
    want = oracle.round_act(deq[:, ks].T, act)         # [M, N]: round(deq[n, k_m])
    ref_bits, _, _ = oracle.gemv(case)
    assert same_values(ref_bits, want, act).all()      # the oracle agrees with itself here
    with bsgemv.Plan(fmt, act, bs, zp, N, K, M) as plan:
        assert configure(plan, how)
        y = run_plan(plan, case)
    diff = np.argwhere(~same_values(y, want, act))
    assert diff.size == 0, (f"{len(diff)} outputs are not round(deq[n, k_m]), first (m, n) = "
                            f"{tuple(diff[0])}")
