"""Property tests of the launch geometry (pure host code, no GPU): for random problems and SM
counts, bsgemv_geometry_for either rejects the problem with a documented status or returns a
geometry the kernels can run -- every stage covered by exactly one CTA, a grid within one wave
of the residency it was sized for, shared memory within the per-CTA and per-SM budgets, and the
regions at the alignment the kernels rely on."""
import pytest

from block_scaled_bit_gb300 import bsgemv

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies

FORMATS = [("int4", (16, 32, 64, 128, 256), (False, True)), ("int8", (16, 32, 64, 128, 256), (False, True)),
           ("fp8", (128,), (False,)), ("nvfp4", (16,), (False,))]


@st.composite
def problems(draw):
    fmt, sizes, zps = draw(st.sampled_from(FORMATS))
    bs = draw(st.sampled_from(sizes))
    zp = draw(st.sampled_from(zps))
    k_units = draw(st.integers(1, 400))
    K = max(64, bs) * k_units if max(64, bs) % 64 == 0 else 64 * k_units
    N = draw(st.one_of(st.integers(1, 300), st.integers(300, 300_000)))
    max_M = draw(st.integers(1, 32))
    sms = draw(st.sampled_from([1, 2, 7, 66, 132, 148, 152, 160]))
    act = draw(st.sampled_from(["f16", "bf16"]))
    return fmt, act, bs, zp, N, K, max_M, sms


@hypothesis.settings(max_examples=400, deadline=None)
@hypothesis.given(problems())
def test_geometry_is_runnable(p):
    fmt, act, bs, zp, N, K, max_M, sms = p
    try:
        g = bsgemv.geometry_for(fmt, act, bs, zp, N, K, max_M, sms)
    except bsgemv.BsgemvError as e:  # only the documented rejections
        assert e.status in (bsgemv.ERR_UNSUPPORTED, bsgemv.ERR_INVALID_ARG)
        assert K % bs != 0 or K % 64 != 0
        return
    spt, tiles = g["stages_per_tile"], g["tiles"]
    rpt = g["rows_per_tile"]
    # k per stage: 256, or 128 for the 8-bit formats with 128-row tiles
    kc = 128 if rpt == 128 and fmt in ("int8", "fp8") else 256
    assert g["k_per_stage"] == kc and rpt in (64, 128) and (rpt == 64 or max_M <= 16)
    assert tiles == -(-N // rpt) and spt == -(-K // kc) and g["total_stages"] == tiles * spt
    slots = sms * g["ctas_per_sm"]
    C = g["cluster"]
    if C:
        assert g["ctas"] == tiles * C and C <= spt and C <= 8 and g["ctas"] <= slots
    else:
        assert 1 <= g["ctas"] <= min(g["total_stages"], slots)
        # stream-K ranges: every stage in exactly one CTA's [s0, s1)
        G, T = g["ctas"], g["total_stages"]
        assert all((i + 1) * T // G >= i * T // G for i in range(G)) and (G * T) // G == T
    assert g["ctas_per_sm"] in (1, 2, 3, 4)
    assert g["smem_bytes"] <= 232448
    if g["ctas_per_sm"] > 1:
        assert g["ctas_per_sm"] * (g["smem_bytes"] + 1024) <= 233472
    assert (1 if C else 2) <= g["stages"] <= 12
    assert g["smem_bytes"] % 8 == 0
    # the same problem gives the same geometry whatever the activation dtype
    other = "bf16" if act == "f16" else "f16"
    assert bsgemv.geometry_for(fmt, other, bs, zp, N, K, max_M, sms) == g


@hypothesis.settings(max_examples=200, deadline=None)
@hypothesis.given(st.sampled_from(["f16", "bf16"]), st.integers(1, 1 << 16), st.integers(1, 1 << 15),
                  st.integers(1, 8), st.sampled_from([1, 7, 132, 152]))
def test_dense_geometry_is_runnable(act, N, K, max_M, sms):
    try:
        g = bsgemv.dense_geometry_for(act, N, K, max_M, sms)
    except bsgemv.BsgemvError:
        raise AssertionError(f"dense geometry rejected {(act, N, K, max_M, sms)}")
    S = g["cluster"]
    assert 1 <= S <= min(8, g["stages_per_tile"]) and g["ctas"] == g["tiles"] * S
    assert S == 1 or g["ctas"] <= 2 * sms
    assert g["smem_bytes"] <= 232448
