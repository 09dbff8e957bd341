"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on the same seeded
inputs.

The bar: the dequantisation stage is bit-exact (bsgemv_debug_dequant runs the GEMV's own
register decoders); the GEMV output satisfies |y - y_ref| <= 1 ulp(|y_ref|) + 1e-3 sum|a*w| on
every element; every row is bit-identical for every M of a plan; repeated calls are
bit-identical.
"""
import os

import numpy as np
import pytest

import conftest
import oracle
from block_scaled_bit_gb300 import bsgemv, synth

pytestmark = pytest.mark.gpu

INT_BS = (16, 32, 64, 128, 256)
DEQ_CASES = ([("int4", a, bs, z) for a in ("f16", "bf16") for bs in INT_BS for z in (True, False)]
             + [("int8", a, bs, z) for a in ("f16", "bf16") for bs in INT_BS for z in (True, False)]
             + [("fp8", a, 128, False) for a in ("f16", "bf16")]
             + [("nvfp4", a, 16, False) for a in ("f16", "bf16")])


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    torch.cuda.set_device(0)
    bsgemv.lib()
    return torch


def run(case, plan=None, M=None, max_M=16, stream=None):
    """Upload, run through the C ABI, return output bits [M, N]."""
    import torch
    M = case.M if M is None else M
    own = plan is None
    if own:
        plan = bsgemv.Plan(case.fmt, case.act, case.block_size, case.has_zp, case.N, case.K, max_M)
    d = bsgemv.upload(case.with_M(M) if M != case.M else case, "cuda")
    plan.run(d.A, d.W, d.scales, d.zp, d.y, M=M, stream=stream)
    torch.cuda.synchronize()
    assert plan.device_status() == bsgemv.OK
    out = bsgemv.y_bits(d.y)
    if own:
        plan.close()
    return out


def assert_parity(case, ybits, rows=None):
    bad, worst, ref = oracle.tolerance_violations(case, ybits if rows is None else ybits[:, rows], rows=rows)
    conftest.record_worst(current_test(), worst)
    assert bad == 0, f"{bad} outputs outside the bound (worst error/bound {worst:.3g})"
    return worst


def current_test() -> str:
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


# ---------------------------------------------------------------------------- decode stage
@pytest.mark.parametrize("fmt,act,bs,zp", DEQ_CASES)
def test_debug_dequant_is_bit_exact(torch_cuda, fmt, act, bs, zp):
    torch = torch_cuda
    K = max(1024, 4 * bs)
    case = synth.make_case(fmt, act, bs, zp, 97, K, 1, 100 + bs)
    d = bsgemv.upload(case, "cuda")
    out = torch.full((case.N, case.K), float("nan"), dtype=torch.float32, device="cuda")
    with bsgemv.Plan(fmt, act, bs, zp, case.N, case.K, 1) as plan:
        plan.debug_dequant(d.W, d.scales, d.zp, out)
        torch.cuda.synchronize()
    got = out.cpu().numpy()
    want = oracle.dequant(case).astype(np.float32)   # exact value, rounded once to fp32
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------------------- GEMV parity
PARITY_CASES = ([("int4", a, bs, z) for a in ("f16", "bf16") for bs in (16, 32, 128) for z in (True, False)]
                + [("int8", a, bs, z) for a in ("f16", "bf16") for bs in (16, 32, 128, 256) for z in (True, False)]
                + [("fp8", a, 128, False) for a in ("f16", "bf16")]
                + [("nvfp4", a, 16, False) for a in ("f16", "bf16")])


@pytest.mark.parametrize("fmt,act,bs,zp", PARITY_CASES)
@pytest.mark.parametrize("M", [1, 5, 9, 16])
def test_gemv_parity_ragged(torch_cuda, fmt, act, bs, zp, M):
    # several tiles with a ragged last tile, several stages with a ragged last stage
    K = 1536 if bs <= 256 else 2048
    case = synth.make_case(fmt, act, bs, zp, 357, K, M, 7 * bs + M)
    assert_parity(case, run(case))


@pytest.mark.parametrize("fmt,act,bs,zp", [("int4", "f16", 32, True), ("int8", "bf16", 128, True),
                                           ("fp8", "f16", 128, False), ("nvfp4", "bf16", 16, False),
                                           ("int4", "bf16", 16, False)])
def test_rows_bit_identical_across_M(torch_cuda, fmt, act, bs, zp):
    case16 = synth.make_case(fmt, act, bs, zp, 300, 2048, 16, 55)
    with bsgemv.Plan(fmt, act, bs, zp, case16.N, case16.K, 16) as plan:
        y16 = run(case16, plan)
        for M in range(1, 16):
            yM = run(case16.with_M(M), plan)
            assert np.array_equal(yM, y16[:M]), f"M={M}"
    assert_parity(case16, y16)


def test_repeated_calls_bit_identical_and_counters_reset(torch_cuda):
    case = synth.make_case("int8", "f16", 32, True, 1000, 4096, 4, 77)
    with bsgemv.Plan("int8", "f16", 32, True, case.N, case.K, 4) as plan:
        # few CTAs for many stages: every tile is split over several CTAs
        assert plan.set_override(ctas=37) == bsgemv.OK
        first = run(case, plan)
        for _ in range(3):
            assert np.array_equal(run(case, plan), first)
    assert_parity(case, first)


@pytest.mark.parametrize("ctas", [1, 2, 3, 17, 64, 150, 10 ** 6])
def test_every_stream_k_split_is_correct(torch_cuda, ctas):
    case = synth.make_case("int4", "f16", 32, True, 777, 2048, 3, 91)
    with bsgemv.Plan("int4", "f16", 32, True, case.N, case.K, 4) as plan:
        assert plan.set_override(ctas=ctas) == bsgemv.OK
        g = plan.describe()
        assert g["ctas"] == min(ctas, g["total_stages"])
        y = run(case, plan)
    assert_parity(case, y)


@pytest.mark.parametrize("fmt,act,bs,zp,N,K", [
    ("int8", "f16", 32, True, 2048, 4096), ("int4", "bf16", 32, False, 700, 2048),
    ("nvfp4", "f16", 16, False, 300, 4096), ("fp8", "bf16", 128, False, 130, 2560),
    ("int4", "f16", 16, True, 257, 1280)])
@pytest.mark.parametrize("cluster,M", [(c, m) for c in (1, 2, 3, 5, 8, 16) for m in (1, 2)]
                         + [(2, 11), (3, 11), (4, 9)])
def test_cluster_split_is_correct(torch_cuda, fmt, act, bs, zp, N, K, cluster, M):
    """Each tile split over a thread-block cluster of `cluster` CTAs (uneven shares when the
    cluster size does not divide the tile's stages), reduced in the leader's shared memory."""
    case = synth.make_case(fmt, act, bs, zp, N, K, M, 1000 + cluster + N)
    with bsgemv.Plan(fmt, act, bs, zp, N, K, M) as plan:
        g0 = plan.describe()
        status = plan.set_split("cluster", cluster)
        if cluster > g0["stages_per_tile"] or g0["tiles"] * cluster > g0["sm_count"] * g0["ctas_per_sm"]:
            assert status == bsgemv.ERR_UNSUPPORTED  # more CTAs than stages, or than one wave
            return
        assert status == bsgemv.OK
        g = plan.describe()
        assert g["cluster"] == cluster and g["ctas"] == g["tiles"] * cluster
        y = run(case, plan, max_M=M)
        assert plan.device_status() == bsgemv.OK
    assert_parity(case, y)


def test_stream_k_and_cluster_split_agree_within_tolerance(torch_cuda):
    """Same problem, both splits: each within the bound of the oracle, and rows bit-identical
    across M inside each."""
    case16 = synth.make_case("int8", "f16", 128, True, 1000, 4096, 16, 321)
    for split in ("stream_k", "cluster"):
        with bsgemv.Plan("int8", "f16", 128, True, case16.N, case16.K, 16) as plan:
            assert plan.set_split(split) == bsgemv.OK
            assert (plan.describe()["cluster"] > 0) == (split == "cluster")
            y16 = run(case16, plan)
            for M in (1, 3, 9):
                assert np.array_equal(run(case16.with_M(M), plan), y16[:M])
        assert_parity(case16, y16)


@pytest.mark.parametrize("stages", [2, 3, 8])
def test_ring_depths(torch_cuda, stages):
    case = synth.make_case("fp8", "bf16", 128, False, 500, 2048, 8, 93)
    with bsgemv.Plan("fp8", "bf16", 128, False, case.N, case.K, 8) as plan:
        assert plan.set_override(stages=stages) == bsgemv.OK
        y = run(case, plan)
    assert_parity(case, y)


@pytest.mark.parametrize("fmt,bs,zp,N,K", [
    ("int4", 32, True, 1, 64), ("int4", 16, True, 1, 64), ("int8", 64, True, 1, 64),
    ("fp8", 128, False, 1, 128), ("nvfp4", 16, False, 1, 64), ("int4", 64, False, 65, 320),
    ("int8", 32, True, 63, 192), ("nvfp4", 16, False, 129, 448), ("int4", 256, True, 2, 768),
    ("int8", 256, True, 130, 256),
])
@pytest.mark.parametrize("M", [1, 16])
def test_edge_shapes(torch_cuda, fmt, bs, zp, N, K, M):
    case = synth.make_case(fmt, "f16", bs, zp, N, K, M, N + K)
    assert_parity(case, run(case))


@pytest.mark.parametrize("M", [2, 12])
@pytest.mark.parametrize("rows_per_tile", [64, 128])
@pytest.mark.parametrize("fmt,bs,zp", [("int8", 32, True), ("int4", 32, True), ("int4", 16, False),
                                       ("fp8", 128, False), ("nvfp4", 16, False)])
def test_side_data_fallback_matches_tma(torch_cuda, fmt, bs, zp, rows_per_tile, M):
    """Scales / zero points that cannot be TMA-tiled (misaligned base) are read from global
    memory (the kernels built for that source); the arithmetic is the same, so the output is
    bit-identical, for both tile heights and one or two n8 tiles."""
    torch = torch_cuda
    case = synth.make_case(fmt, "f16", bs, zp, 300, 2048, M, 5)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan(fmt, "f16", bs, zp, case.N, case.K, 16) as plan:
        assert plan.set_override(rows_per_tile=rows_per_tile) == bsgemv.OK
        plan.run(d.A, d.W, d.scales, d.zp, d.y, M=M)
        torch.cuda.synchronize()
        ref = bsgemv.y_bits(d.y)
        # the same bytes one element past a 16-byte boundary
        es = d.scales.element_size()
        flat = d.scales.reshape(-1)
        s2 = torch.empty(flat.numel() + 1, dtype=flat.dtype, device="cuda")[1:]
        s2.copy_(flat)
        assert s2.data_ptr() % 16 == es % 16 and s2.data_ptr() % es == 0
        z2 = d.zp
        if zp:
            z2 = torch.empty(d.zp.numel() + 3, dtype=torch.uint8, device="cuda")[3:]
            z2.copy_(d.zp.view(-1))
            assert z2.data_ptr() % 16 != 0
        y2 = torch.empty_like(d.y)
        plan.run(d.A, d.W, s2, z2, y2, M=M)
        torch.cuda.synchronize()
        assert plan.device_status() == bsgemv.OK
    assert np.array_equal(bsgemv.y_bits(y2), ref)
    assert_parity(case, ref)


@pytest.mark.parametrize("fmt,bs,zp", [("int8", 32, True), ("int4", 16, True), ("fp8", 128, False),
                                       ("nvfp4", 16, False)])
def test_side_data_fallback_cuda_core_variant(torch_cuda, fmt, bs, zp):
    """The CUDA-core variant's kernels for scales read from global memory: bit-identical to its
    side-ring kernels."""
    torch = torch_cuda
    case = synth.make_case(fmt, "bf16", bs, zp, 333, 1024, 5, 6)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan(fmt, "bf16", bs, zp, case.N, case.K, 8) as plan:
        assert plan.set_override(variant=bsgemv.VARIANTS["cuda_core"]) == bsgemv.OK
        plan.run(d.A, d.W, d.scales, d.zp, d.y, M=5)
        torch.cuda.synchronize()
        ref = bsgemv.y_bits(d.y)
        flat = d.scales.reshape(-1)
        s2 = torch.empty(flat.numel() + 1, dtype=flat.dtype, device="cuda")[1:]
        s2.copy_(flat)
        y2 = torch.empty_like(d.y)
        plan.run(d.A, d.W, s2, d.zp, y2, M=5)
        torch.cuda.synchronize()
        assert plan.device_status() == bsgemv.OK
    assert np.array_equal(bsgemv.y_bits(y2), ref)
    assert_parity(case, ref)


def test_run_host_matches_device_run(torch_cuda):
    torch = torch_cuda
    case = synth.make_case("nvfp4", "f16", 16, False, 2048, 2048, 3, 17)
    d = bsgemv.upload(case, "cuda")
    A_host = torch.from_numpy(case.A.view(np.int16)).pin_memory()
    y_host = torch.empty((3, case.N), dtype=torch.int16).pin_memory()
    with bsgemv.Plan("nvfp4", "f16", 16, False, case.N, case.K, 4) as plan:
        plan.run_host(A_host, d.W, d.scales, d.zp, y_host, M=3)
        plan.run(d.A, d.W, d.scales, d.zp, d.y)
        torch.cuda.synchronize()
    assert np.array_equal(y_host.numpy().view(np.uint16), bsgemv.y_bits(d.y))
    assert_parity(case, bsgemv.y_bits(d.y))


def test_run_host_async_steps_match_device_runs(torch_cuda):
    """Several calls enqueued through bsgemv_run_host_async on one stream and one plan (sharing
    its staging buffer), one synchronisation: every host output equals the device run's."""
    torch = torch_cuda
    case = synth.make_case("int8", "f16", 32, True, 3000, 2048, 4, 19)
    d = bsgemv.upload(case, "cuda")
    stream = torch.cuda.Stream()
    with bsgemv.Plan("int8", "f16", 32, True, case.N, case.K, 4) as plan:
        plan.run(d.A, d.W, d.scales, d.zp, d.y)
        torch.cuda.synchronize()
        ref = bsgemv.y_bits(d.y)
        outs = []
        for M in (4, 1, 3, 4):
            A_host = torch.from_numpy(np.ascontiguousarray(case.A[:M]).view(np.int16)).pin_memory()
            y_host = torch.full((M, case.N), -1, dtype=torch.int16).pin_memory()
            plan.run_host_async(A_host, d.W, d.scales, d.zp, y_host, M=M, stream=stream)
            outs.append((M, A_host, y_host))
        stream.synchronize()
    for M, _, y_host in outs:
        assert np.array_equal(y_host.numpy().view(np.uint16), ref[:M]), f"M={M}"


@pytest.mark.parametrize("memory", ["pinned", "pinned_offset", "pageable"])
def test_run_host_copies_for_every_kind_of_host_buffer(torch_cuda, memory):
    """Pinned, 16-byte aligned buffers are copied by kernels through their device mapping (a
    ragged byte count: M * N * 2 = 6006); a pinned buffer off the 16-byte grid, or pageable
    memory, by copy-engine transfers.  Every path gives the device run's bits."""
    torch = torch_cuda
    case = synth.make_case("int4", "bf16", 32, True, 1001, 1024, 3, 23)
    d = bsgemv.upload(case, "cuda")
    a = np.ascontiguousarray(case.A).view(np.int16)

    def host(shape_or_array, fill=None):
        arr = shape_or_array if fill is None else np.full(shape_or_array, fill, dtype=np.int16)
        if memory == "pageable":
            return torch.from_numpy(np.array(arr))
        if memory == "pinned":
            return torch.from_numpy(np.array(arr)).pin_memory()
        flat = torch.empty(arr.size + 1, dtype=torch.int16).pin_memory()[1:]  # 2 bytes off
        flat.copy_(torch.from_numpy(np.array(arr)).reshape(-1))
        return flat.view(arr.shape)

    A_host = host(a)
    y_host = host((3, case.N), fill=-1)
    with bsgemv.Plan("int4", "bf16", 32, True, case.N, case.K, 4) as plan:
        plan.run(d.A, d.W, d.scales, d.zp, d.y)
        torch.cuda.synchronize()
        ref = bsgemv.y_bits(d.y)
        plan.run_host(A_host, d.W, d.scales, d.zp, y_host, M=3)
        assert plan.device_status() == bsgemv.OK
    assert np.array_equal(y_host.numpy().view(np.uint16), ref)


def test_errors_on_device(torch_cuda):
    torch = torch_cuda
    case = synth.make_case("int4", "f16", 32, True, 128, 512, 4, 3)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan("int4", "f16", 32, True, case.N, case.K, 4) as plan:
        raw = torch.empty(d.A.numel() + 8, dtype=torch.int16, device="cuda")
        A_mis = raw[1:1 + d.A.numel()].view(d.A.shape)
        assert plan.run_status(A_mis, d.W, d.scales, d.zp, d.y) == bsgemv.ERR_MISALIGNED
        assert plan.run_status(d.A, d.W, d.scales, d.zp, d.y, M=5) == bsgemv.ERR_M_TOO_LARGE
        assert plan.run_status(d.A, d.W, d.scales, d.zp, d.y, M=0) == bsgemv.ERR_INVALID_ARG
        assert plan.run_status(d.A, d.W, d.scales, None, d.y) == bsgemv.ERR_INVALID_ARG
        assert plan.run_status(d.A, None, d.scales, d.zp, d.y) == bsgemv.ERR_INVALID_ARG
        assert plan.set_override(variant=7) == bsgemv.ERR_INVALID_ARG
        assert plan.device_status() == bsgemv.OK
    with bsgemv.Plan("int4", "f16", 32, True, case.N, case.K, 16) as plan:
        # the CUDA-core variant accumulates at most 8 activation rows per lane
        assert plan.set_override(variant=bsgemv.VARIANTS["cuda_core"]) == bsgemv.ERR_UNSUPPORTED
        assert plan.describe()["variant"] == bsgemv.VARIANTS["mma"]
    with bsgemv.Plan("int8", "f16", 32, False, 64, 512, 1) as plan:
        c8 = synth.make_case("int8", "f16", 32, False, 64, 512, 1, 4)
        d8 = bsgemv.upload(c8, "cuda")
        # a zero point given to a plan without zero points is an error, not ignored
        assert plan.run_status(d8.A, d8.W, d8.scales, d.zp, d8.y) == bsgemv.ERR_INVALID_ARG


def test_plan_records_device_and_geometry(torch_cuda):
    torch = torch_cuda
    with bsgemv.Plan("int4", "bf16", 32, False, 151936, 4096, 16) as plan:
        g = plan.describe()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert g["sm_count"] == sms
    assert g == bsgemv.geometry_for("int4", "bf16", 32, False, 151936, 4096, 16, sms)


# ---------------------------------------------------------------------------- int4 kernels
@pytest.mark.parametrize("act,bs,zp", [("f16", 32, False), ("f16", 16, True), ("f16", 128, True),
                                       ("bf16", 32, False), ("bf16", 64, True)])
def test_int4_long_ranges_rows_bit_identical_for_M_1_to_3(torch_cuda, act, bs, zp):
    """int4 over long CTA ranges (about 8 stages per CTA) at M = 1, 2, 3: each call's ring is
    laid out for its own M (deeper for fewer rows), the split is the plan's, so the rows must be
    bit-identical across M and within the bound of the oracle."""
    N, K = 40000, 2048  # 625 tiles x 8 stages over one wave of CTAs: about 8 stages per CTA
    case = synth.make_case("int4", act, bs, zp, N, K, 3, 4242 + bs)
    rows = np.arange(0, N, 37)
    with bsgemv.Plan("int4", act, bs, zp, N, K, 3) as plan:
        g = plan.describe()
        assert -(-g["total_stages"] // g["ctas"]) >= 5
        outs = {M: run(case, plan=plan, M=M) for M in (1, 2, 3)}
    assert_parity(case.with_M(3), outs[3], rows=rows)
    assert np.array_equal(outs[1], outs[3][:1])
    assert np.array_equal(outs[2], outs[3][:2])


# ---------------------------------------------------------------------------- CUDA-core variant
CC_CASES = ([("int4", a, bs, z) for a in ("f16", "bf16") for bs in (16, 32, 64, 128, 256) for z in (True, False)]
            + [("int8", a, bs, z) for a in ("f16", "bf16") for bs in (16, 32, 64, 128, 256) for z in (True, False)]
            + [("fp8", a, 128, False) for a in ("f16", "bf16")]
            + [("nvfp4", a, 16, False) for a in ("f16", "bf16")])


def cuda_core_plan(fmt, act, bs, zp, N, K, max_M):
    plan = bsgemv.Plan(fmt, act, bs, zp, N, K, max_M)
    assert plan.set_override(variant=bsgemv.VARIANTS["cuda_core"]) == bsgemv.OK
    assert plan.describe()["variant"] == bsgemv.VARIANTS["cuda_core"]
    return plan


@pytest.mark.parametrize("fmt,act,bs,zp", CC_CASES)
def test_cuda_core_variant_parity_and_rows_across_M(torch_cuda, fmt, act, bs, zp):
    """The CUDA-core variant (fp32 FMAs on the CUDA cores instead of mma.sync, same decoders and
    pipeline): within the bound of the oracle for M = 1 and M = 8 (its two kernels) over several
    tiles with ragged N and K tails, and every row bit-identical across M = 1..8 of one plan."""
    K = 1536 if bs <= 128 else 1792
    case8 = synth.make_case(fmt, act, bs, zp, 357, K, 8, 11 * bs + 5)
    with cuda_core_plan(fmt, act, bs, zp, case8.N, case8.K, 8) as plan:
        y8 = run(case8, plan)
        for M in (1, 2, 7):
            assert np.array_equal(run(case8.with_M(M), plan), y8[:M]), f"M={M}"
    assert_parity(case8, y8)


@pytest.mark.parametrize("split,cluster,ctas", [("stream_k", 0, 37), ("stream_k", 0, 0),
                                                ("cluster", 3, 0), ("cluster", 8, 0)])
@pytest.mark.parametrize("M", [1, 6])
def test_cuda_core_variant_under_every_split(torch_cuda, split, cluster, ctas, M):
    """Both K splits (stream-K with a last-arriver reduction, cluster split reduced in shared
    memory) take the CUDA-core variant's partial sums in the same fragment layout."""
    # int4: 8 KB stages, so that 3- and 8-CTA clusters fit next to the reduction buffer
    case = synth.make_case("int4", "bf16", 64, True, 700, 4096, M, 606 + M)
    with cuda_core_plan("int4", "bf16", 64, True, case.N, case.K, 8) as plan:
        assert plan.set_split(split, cluster) == bsgemv.OK
        if ctas:
            assert plan.set_override(ctas=ctas) == bsgemv.OK
        g = plan.describe()
        assert g["variant"] == bsgemv.VARIANTS["cuda_core"]
        assert (g["cluster"] == cluster) if split == "cluster" else g["cluster"] == 0
        y = run(case, plan)
    assert_parity(case, y)


def test_cuda_core_and_mma_variants_agree_within_tolerance(torch_cuda):
    """Same problem through both variants: different summation orders, each within the bound."""
    case = synth.make_case("nvfp4", "f16", 16, False, 2048, 2048, 4, 808)
    with bsgemv.Plan("nvfp4", "f16", 16, False, case.N, case.K, 4) as plan:
        y_mma = run(case, plan)
        assert plan.set_override(variant=bsgemv.VARIANTS["cuda_core"]) == bsgemv.OK
        y_cc = run(case, plan)
        assert plan.set_override(variant=bsgemv.VARIANTS["mma"]) == bsgemv.OK
        assert np.array_equal(run(case, plan), y_mma)
    assert_parity(case, y_mma)
    assert_parity(case, y_cc)


# ---------------------------------------------------------------------------- bias epilogue
def run_bias(case, plan, M=None):
    import torch
    M = case.M if M is None else M
    d = bsgemv.upload(case.with_M(M) if M != case.M else case, "cuda")
    plan.run(d.A, d.W, d.scales, d.zp, d.y, M=M, bias=d.bias)
    torch.cuda.synchronize()
    assert plan.device_status() == bsgemv.OK
    return bsgemv.y_bits(d.y)


BIAS_CASES = [("int4", "f16", 32, True), ("int4", "bf16", 16, False), ("int8", "f16", 128, True),
              ("int8", "bf16", 32, False), ("fp8", "f16", 128, False), ("fp8", "bf16", 128, False),
              ("nvfp4", "f16", 16, False), ("nvfp4", "bf16", 16, False)]


@pytest.mark.parametrize("fmt,act,bs,zp", BIAS_CASES)
def test_bias_epilogue_parity_and_rows_across_M(torch_cuda, fmt, act, bs, zp):
    """y = A . deq(W)^T + bias through bsgemv_run_bias: within the bound of the oracle (which adds
    the bias before its one rounding) over ragged tiles and stages, rows bit-identical across M."""
    case = synth.make_case(fmt, act, bs, zp, 357, 1536, 16, 5 * bs + 1).with_bias()
    with bsgemv.Plan(fmt, act, bs, zp, case.N, case.K, 16) as plan:
        y16 = run_bias(case, plan)
        for M in (1, 8, 9):
            assert np.array_equal(run_bias(case, plan, M), y16[:M]), f"M={M}"
    assert_parity(case, y16)


@pytest.mark.parametrize("fmt,act,bs,zp", BIAS_CASES[::2])
def test_bias_with_zero_activations_is_the_bias(torch_cuda, fmt, act, bs, zp):
    """With A = 0 every product is zero: y must equal the bias exactly."""
    import dataclasses
    case = synth.make_case(fmt, act, bs, zp, 200, 1024, 3, 41).with_bias()
    case = dataclasses.replace(case, A=np.zeros_like(case.A))
    with bsgemv.Plan(fmt, act, bs, zp, case.N, case.K, 4) as plan:
        y = run_bias(case, plan)
    want = oracle.act_values(case.bias, act)
    assert np.array_equal(oracle.act_values(y, act), np.broadcast_to(want, y.shape))


@pytest.mark.parametrize("how", ["stream_k", "cluster", "cuda_core"])
def test_bias_under_every_split_and_variant(torch_cuda, how):
    case = synth.make_case("int4", "f16", 32, True, 700, 4096, 5, 77).with_bias(sigma=10.0)
    with bsgemv.Plan("int4", "f16", 32, True, case.N, case.K, 8) as plan:
        if how == "stream_k":
            assert plan.set_override(ctas=37) == bsgemv.OK
        elif how == "cluster":
            assert plan.set_split("cluster", 4) == bsgemv.OK
        else:
            assert plan.set_override(variant=bsgemv.VARIANTS["cuda_core"]) == bsgemv.OK
        y = run_bias(case, plan)
        d = bsgemv.upload(case, "cuda")
        odd = d.bias.data_ptr() + 1  # an odd byte address: not a 16-bit element boundary
        assert plan.run_status(d.A, d.W, d.scales, d.zp, d.y, bias=odd) == bsgemv.ERR_MISALIGNED
    assert_parity(case, y)


# ---------------------------------------------------------------------------- autotune
@pytest.mark.parametrize("fmt,act,bs,zp,N,K", [("int8", "f16", 128, True, 4096, 4096),
                                               ("nvfp4", "bf16", 16, False, 2048, 2048),
                                               ("int4", "f16", 32, False, 12288, 4096),
                                               ("fp8", "f16", 128, False, 512, 2048)])
def test_autotune_keeps_a_candidate_and_stays_deterministic(torch_cuda, fmt, act, bs, zp, N, K):
    """bsgemv_plan_autotune times the candidate geometries and keeps one; the plan then gives
    results within the bound of the oracle with rows bit-identical across M."""
    case = synth.make_case(fmt, act, bs, zp, N, K, 8, 99)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan(fmt, act, bs, zp, N, K, 8) as plan:
        sms = plan.describe()["sm_count"]
        g = plan.autotune(d.A, d.W, d.scales, d.zp, d.y, M=8, reps=5)
        assert g["variant"] == bsgemv.VARIANTS["mma"]
        assert g["rows_per_tile"] in (64, 128) and 1 <= g["stages"] <= 12
        if g["cluster"] > 0:
            assert 1 <= g["cluster"] <= 8 and g["ctas"] == g["tiles"] * g["cluster"]
        else:
            # stream-K candidates run 1 .. 4 CTAs per SM, or the default grid
            assert g["ctas"] <= min(g["total_stages"], sms * max(4, g["ctas_per_sm"]))
        y8 = run(case, plan)
        for M in (1, 3):
            assert np.array_equal(run(case.with_M(M), plan), y8[:M]), f"M={M}"
        assert plan.describe() == g  # running does not change the geometry
    assert_parity(case, y8)


def test_autotune_argument_errors_leave_the_plan_unchanged(torch_cuda):
    case = synth.make_case("int8", "f16", 32, True, 1000, 2048, 2, 5)
    d = bsgemv.upload(case, "cuda")
    with bsgemv.Plan("int8", "f16", 32, True, case.N, case.K, 2) as plan:
        g0 = plan.describe()
        assert plan.autotune_status(d.A, d.W, d.scales, d.zp, d.y, M=2, reps=0) == bsgemv.ERR_INVALID_ARG
        assert plan.autotune_status(d.A, d.W, d.scales, d.zp, d.y, M=3) == bsgemv.ERR_M_TOO_LARGE
        assert plan.autotune_status(d.A, d.W, d.scales, None, d.y, M=2) == bsgemv.ERR_INVALID_ARG
        assert plan.describe() == g0


# ---------------------------------------------------------------------------- M = 17 .. 32
WIDE_CASES = [("int4", "f16", 32, True), ("int4", "bf16", 16, False), ("int4", "f16", 128, False),
              ("int8", "f16", 128, True), ("int8", "bf16", 16, True), ("int8", "f16", 256, False),
              ("fp8", "f16", 128, False), ("fp8", "bf16", 128, False),
              ("nvfp4", "f16", 16, False), ("nvfp4", "bf16", 16, False)]


@pytest.mark.parametrize("fmt,act,bs,zp", WIDE_CASES)
@pytest.mark.parametrize("M", [17, 24, 32])
def test_gemv_parity_up_to_32_rows(torch_cuda, fmt, act, bs, zp, M):
    """Plans with max_M > 16 run four n8 activation tiles (2 CTAs per SM): within the bound over
    ragged tiles and stages."""
    K = 1536 if bs <= 128 else 1792
    case = synth.make_case(fmt, act, bs, zp, 357, K, M, 3 * bs + M)
    assert_parity(case, run(case, max_M=32))


@pytest.mark.parametrize("fmt,act,bs,zp", WIDE_CASES[::3])
def test_rows_bit_identical_across_M_up_to_32(torch_cuda, fmt, act, bs, zp):
    case32 = synth.make_case(fmt, act, bs, zp, 300, 2048, 32, 56)
    with bsgemv.Plan(fmt, act, bs, zp, case32.N, case32.K, 32) as plan:
        assert plan.describe()["ctas_per_sm"] == 2
        y32 = run(case32, plan)
        for M in (1, 2, 3, 8, 9, 16, 17, 31):
            assert np.array_equal(run(case32.with_M(M), plan), y32[:M]), f"M={M}"
    assert_parity(case32, y32)


@pytest.mark.parametrize("fmt,act,bs,zp", WIDE_CASES)
def test_plans_for_24_rows_run_three_tiles(torch_cuda, fmt, act, bs, zp):
    """Plans with 17 <= max_M <= 24 are sized for three n8 tiles at 3 CTAs per SM: parity at
    M = 17 and 24, and rows bit-identical across M (one, two and three tiles)."""
    K = 1536 if bs <= 128 else 1792
    case24 = synth.make_case(fmt, act, bs, zp, 357, K, 24, 5 * bs + 24)
    with bsgemv.Plan(fmt, act, bs, zp, case24.N, case24.K, 24) as plan:
        assert plan.describe()["ctas_per_sm"] == 3
        y24 = run(case24, plan)
        for M in (1, 9, 17, 23):
            assert np.array_equal(run(case24.with_M(M), plan), y24[:M]), f"M={M}"
    assert_parity(case24, y24)
    assert_parity(case24.with_M(17), y24[:17])


def test_plans_for_24_rows_that_keep_four_tiles(torch_cuda):
    """A small shape whose 24-row plan keeps four n8 tiles at 2 CTAs per SM (for the cluster
    split): calls with 17..24 rows run four tiles, fewer rows one or two; rows bit-identical."""
    case = synth.make_case("fp8", "f16", 128, False, 4096, 2048, 24, 2424)
    with bsgemv.Plan("fp8", "f16", 128, False, case.N, case.K, 24) as plan:
        g = plan.describe()
        assert (g["ctas_per_sm"], g["cluster"]) == (2, 4)
        y24 = run(case, plan)
        for M in (1, 8, 9, 17, 20):
            assert np.array_equal(run(case.with_M(M), plan), y24[:M]), f"M={M}"
    assert_parity(case, y24)


@pytest.mark.parametrize("how", ["stream_k", "cluster", "bias"])
def test_32_rows_under_every_split_and_with_bias(torch_cuda, how):
    case = synth.make_case("int4", "bf16", 32, True, 700, 4096, 29, 2929)
    with bsgemv.Plan("int4", "bf16", 32, True, case.N, case.K, 32) as plan:
        if how == "stream_k":
            assert plan.set_override(ctas=37) == bsgemv.OK
            y = run(case, plan)
        elif how == "cluster":
            assert plan.set_split("cluster", 4) == bsgemv.OK
            y = run(case, plan)
        else:
            case = case.with_bias()
            y = run_bias(case, plan)
    assert_parity(case, y)


# ---------------------------------------------------------------------------- dense GEMV
def run_dense(act, A_bits, B_bits, plan, M=None):
    import torch
    M = A_bits.shape[0] if M is None else M
    dA = torch.from_numpy(np.ascontiguousarray(A_bits[:M]).view(np.int16)).cuda()
    dB = torch.from_numpy(np.ascontiguousarray(B_bits).view(np.int16)).cuda()
    y = torch.empty((M, B_bits.shape[1]), dtype=torch.int16, device="cuda")
    plan.run(dA, dB, y, M=M)
    torch.cuda.synchronize()
    assert plan.device_status() == bsgemv.OK
    return bsgemv.y_bits(y)


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(8, 16), (32, 2048), (1024, 2048), (1000, 1000), (72, 4104),
                                 (256, 128), (4096, 512)])
def test_dense_gemv_parity_and_rows_across_M(torch_cuda, act, N, K):
    """The dense small-N split-K GEMV: within the bound of the oracle for M = 8 (ragged N and K
    tails, every split the plan chooses), and every row bit-identical for M = 1 .. 7."""
    A, B = synth.dense_operands(act, 8, N, K, seed=N + K)
    with bsgemv.DensePlan(act, N, K, 8) as plan:
        y8 = run_dense(act, A, B, plan)
        for M in (1, 2, 5, 7):
            assert np.array_equal(run_dense(act, A, B, plan, M), y8[:M]), f"M={M}"
        for _ in range(2):  # repeated calls: nothing to reset, same bits
            assert np.array_equal(run_dense(act, A, B, plan), y8)
    bad, worst, _ = oracle.dense_tolerance_violations(A, B, act, y8)
    conftest.record_worst(current_test(), worst)
    assert bad == 0, f"{bad} outputs outside the bound (worst {worst:.3g})"


@pytest.mark.parametrize("act", ["f16", "bf16"])
@pytest.mark.parametrize("N,K", [(1, 2048), (3, 100), (7, 5000), (9, 1), (33, 777), (1001, 2048),
                                 (64, 2044), (16, 8)])
def test_dense_gemv_without_tma_pitches(torch_cuda, act, N, K):
    """N or K not a multiple of 8 (the split-K page's tests include N = 1): the CUDA-core kernel,
    within the bound of the oracle, rows bit-identical across M, repeated calls identical."""
    A, B = synth.dense_operands(act, 8, N, K, seed=3 * N + K)
    with bsgemv.DensePlan(act, N, K, 8) as plan:
        assert plan.describe()["variant"] == bsgemv.VARIANTS["cuda_core"]
        y8 = run_dense(act, A, B, plan)
        for M in (1, 3, 6):
            assert np.array_equal(run_dense(act, A, B, plan, M), y8[:M]), f"M={M}"
        assert np.array_equal(run_dense(act, A, B, plan), y8)
    bad, worst, _ = oracle.dense_tolerance_violations(A, B, act, y8)
    conftest.record_worst(current_test(), worst)
    assert bad == 0, f"{bad} outputs outside the bound (worst {worst:.3g})"


def test_dense_errors_on_device(torch_cuda):
    torch = torch_cuda
    A, B = synth.dense_operands("f16", 4, 64, 256, seed=3)
    with bsgemv.DensePlan("f16", 64, 256, 4) as plan:
        dA = torch.from_numpy(A.view(np.int16)).cuda()
        dB = torch.from_numpy(B.view(np.int16)).cuda()
        y = torch.empty((4, 64), dtype=torch.int16, device="cuda")
        assert plan.run_status(dA, dB, y, M=5) == bsgemv.ERR_M_TOO_LARGE
        assert plan.run_status(dA, dB, y, M=0) == bsgemv.ERR_INVALID_ARG
        assert plan.run_status(dA.data_ptr() + 2, dB, y, M=4) == bsgemv.ERR_MISALIGNED
        assert plan.run_status(dA, None, y, M=4) == bsgemv.ERR_INVALID_ARG
        assert plan.device_status() == bsgemv.OK


# ---------------------------------------------------------------------------- ordering
@pytest.mark.parametrize("fmt,act,bs,zp,N,K", [("int8", "f16", 128, True, 4096, 4096),
                                               ("int4", "bf16", 32, False, 12288, 4096),
                                               ("nvfp4", "f16", 16, False, 2048, 2048)])
def test_activations_written_by_the_previous_kernel_are_seen(torch_cuda, fmt, act, bs, zp, N, K):
    """Each GEMV starts while the previous kernel drains (programmatic dependent launch) and
    prefetches weights before the dependency wait, activations only after it: a kernel that
    rewrites A right before the call must be seen.  Five rounds of (overwrite A, GEMV) on one
    stream, each output equal to the same GEMV run alone on that round's activations."""
    torch = torch_cuda
    case = synth.make_case(fmt, act, bs, zp, N, K, 4, 4711)
    d = bsgemv.upload(case, "cuda")
    rounds = [torch.randn((4, K), generator=torch.Generator().manual_seed(r)).to(
        torch.float16 if act == "f16" else torch.bfloat16).view(torch.int16).cuda() for r in range(5)]
    stream = torch.cuda.Stream()
    ys = [torch.empty((4, N), dtype=torch.int16, device="cuda") for _ in rounds]
    with bsgemv.Plan(fmt, act, bs, zp, N, K, 4) as plan:
        with torch.cuda.stream(stream):
            for a, y in zip(rounds, ys):
                d.A.copy_(a)                     # a torch kernel writes A ...
                plan.run(d.A, d.W, d.scales, d.zp, y, stream=stream)   # ... the GEMV reads it
        stream.synchronize()
        for a, y in zip(rounds, ys):
            ref = torch.empty_like(y)
            plan.run(a, d.W, d.scales, d.zp, ref)
            torch.cuda.synchronize()
            assert torch.equal(ref, y)


def test_dense_activations_written_by_the_previous_kernel_are_seen(torch_cuda):
    torch = torch_cuda
    N, K = 1024, 2048
    A, B = synth.dense_operands("f16", 8, N, K, seed=9)
    dB = torch.from_numpy(B.view(np.int16)).cuda()
    dA = torch.empty((8, K), dtype=torch.int16, device="cuda")
    rounds = [torch.randn((8, K), generator=torch.Generator().manual_seed(r)).half().view(torch.int16).cuda()
              for r in range(5)]
    ys = [torch.empty((8, N), dtype=torch.int16, device="cuda") for _ in rounds]
    stream = torch.cuda.Stream()
    with bsgemv.DensePlan("f16", N, K, 8) as plan:
        with torch.cuda.stream(stream):
            for a, y in zip(rounds, ys):
                dA.copy_(a)
                plan.run(dA, dB, y, stream=stream)
        stream.synchronize()
        for a, y in zip(rounds, ys):
            ref = torch.empty_like(y)
            plan.run(a, dB, ref)
            torch.cuda.synchronize()
            assert torch.equal(ref, y)


def test_two_plans_on_two_streams_concurrently(torch_cuda):
    """Plans own separate workspaces: two of them driven from two streams at once give the same
    bits as when run alone."""
    torch = torch_cuda
    c1 = synth.make_case("int8", "f16", 32, True, 12288, 4096, 2, 71)
    c2 = synth.make_case("int4", "f16", 32, True, 4096, 12288, 3, 72)
    d1, d2 = bsgemv.upload(c1, "cuda"), bsgemv.upload(c2, "cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with bsgemv.Plan("int8", "f16", 32, True, c1.N, c1.K, 2) as p1, \
            bsgemv.Plan("int4", "f16", 32, True, c2.N, c2.K, 3) as p2:
        p1.run(d1.A, d1.W, d1.scales, d1.zp, d1.y)
        p2.run(d2.A, d2.W, d2.scales, d2.zp, d2.y)
        torch.cuda.synchronize()
        r1, r2 = d1.y.clone(), d2.y.clone()
        outs1 = [torch.empty_like(d1.y) for _ in range(10)]
        outs2 = [torch.empty_like(d2.y) for _ in range(10)]
        for o1, o2 in zip(outs1, outs2):
            p1.run(d1.A, d1.W, d1.scales, d1.zp, o1, stream=s1)
            p2.run(d2.A, d2.W, d2.scales, d2.zp, o2, stream=s2)
        torch.cuda.synchronize()
        assert p1.device_status() == bsgemv.OK and p2.device_status() == bsgemv.OK
    assert all(torch.equal(o, r1) for o in outs1)
    assert all(torch.equal(o, r2) for o in outs2)
