"""The C-ABI library without a GPU: it loads, exports every entry point include/bsgemv.h
declares, rejects bad arguments on the host, and its launch geometry (a pure host predicate) is
a deterministic function of the problem and a fixed SM count."""
import os
import re

import numpy as np
import pytest

from block_scaled_bit_gb300 import bsgemv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from block_scaled_bit_gb300 import _build
    _build.build()
    return bsgemv.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "bsgemv.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsgemv_\w+)\s*\(", text)))


def test_every_declared_function_is_exported(L):
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(L, name), name
    assert set(names) == set(bsgemv.EXPORTS)


def test_status_strings(L):
    for code in range(-8, 1):
        assert bsgemv.status_string(code) not in ("", "unknown status")
    assert bsgemv.status_string(-99) == "unknown status"
    assert L.bsgemv_version() >= 100


@pytest.mark.parametrize("args,code", [
    (("int4", "f16", 32, True, 0, 512, 1), bsgemv.ERR_INVALID_ARG),      # N = 0
    (("int4", "f16", 32, True, 64, 512, 0), bsgemv.ERR_INVALID_ARG),     # max_M = 0
    (("int4", "f16", 32, True, 64, 512, 33), bsgemv.ERR_INVALID_ARG),    # max_M > 32
    (("int4", "f16", 48, True, 64, 512, 1), bsgemv.ERR_UNSUPPORTED),     # block size
    (("int4", "f16", 32, True, 64, 544, 1), bsgemv.ERR_UNSUPPORTED),     # K % 64
    (("fp8", "f16", 64, False, 64, 512, 1), bsgemv.ERR_UNSUPPORTED),     # fp8 needs 128
    (("fp8", "f16", 128, True, 64, 512, 1), bsgemv.ERR_UNSUPPORTED),     # fp8 has no zp
    (("nvfp4", "f16", 32, False, 64, 512, 1), bsgemv.ERR_UNSUPPORTED),   # nvfp4 needs 16
])
def test_invalid_problems_rejected_on_host(L, args, code):
    fmt, act, bs, zp, N, K, mm = args
    with pytest.raises(bsgemv.BsgemvError) as e:
        bsgemv.geometry_for(fmt, act, bs, zp, N, K, mm, 152)
    assert e.value.status == code
    # bsgemv_plan validates its arguments before it touches CUDA
    with pytest.raises(bsgemv.BsgemvError) as e:
        bsgemv.Plan(fmt, act, bs, zp, N, K, mm)
    assert e.value.status == code


def test_bad_format_bits(L):
    import ctypes
    g = bsgemv.Geometry()
    assert L.bsgemv_geometry_for(0x200 | 1, 32, 0, 64, 512, 1, 152, ctypes.byref(g)) == bsgemv.ERR_INVALID_ARG
    assert L.bsgemv_geometry_for(5, 32, 0, 64, 512, 1, 152, ctypes.byref(g)) == bsgemv.ERR_INVALID_ARG
    assert L.bsgemv_run(None, None, None, None, None, None, 1, None) == bsgemv.ERR_INVALID_ARG
    assert L.bsgemv_destroy(None) == bsgemv.OK


def test_plan_without_gpu_reports_unsupported(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(bsgemv.BsgemvError) as e:
        bsgemv.Plan("int8", "f16", 128, True, 4096, 4096, 1)
    assert e.value.status in (bsgemv.ERR_UNSUPPORTED, bsgemv.ERR_CUDA)


# ---------------------------------------------------------------------------- geometry
SHAPES = [("int4", 32, False, 151936, 4096), ("int8", 128, True, 2048, 4096),
          ("int8", 32, True, 12288, 4096), ("fp8", 128, False, 512, 2048),
          ("nvfp4", 16, False, 248320, 2048), ("int4", 32, True, 1024, 512),
          ("int4", 16, True, 1, 64), ("int8", 256, False, 77, 768)]


@pytest.mark.parametrize("fmt,bs,zp,N,K", SHAPES)
@pytest.mark.parametrize("sms", [132, 148, 152])
@pytest.mark.parametrize("max_M", [1, 8, 16, 17, 32])
def test_geometry_predicates(L, fmt, bs, zp, N, K, sms, max_M):
    g = bsgemv.geometry_for(fmt, "f16", bs, zp, N, K, max_M, sms)
    four = fmt in ("int4", "nvfp4")
    # 64-row tiles, or 128 (two halves) for plans of up to 16 rows where at most 5 resident CTAs
    # share a 128-row tile on average and there are at least 2 such stages per resident CTA; a
    # stage is 256 k, or 128 k for the 8-bit formats with 128-row tiles (16 KB of weight, but
    # 8 KB for the 4-bit formats with 64-row tiles)
    rpt = g["rows_per_tile"]
    assert rpt in (64, 128) and g["consumer_warps"] == 4
    assert g["k_per_stage"] == (128 if rpt == 128 and not four else 256)
    assert g["tiles"] == -(-N // rpt)
    tall_tiles = -(-N // 128)
    tall_stages = tall_tiles * -(-K // (256 if four else 128))
    if max_M > 16:
        assert rpt == 64
    else:  # (128-row tiles run 3 CTAs per SM)
        tall_ok = tall_tiles * 5 >= sms * 3 and tall_stages >= 2 * sms * 3
        if rpt == 128:
            assert tall_ok and g["ctas_per_sm"] == 3
        elif tall_ok:  # kept at 64 rows only where those keep a cluster split 128 rows lose
            assert g["cluster"] >= 2
    assert g["stages_per_tile"] == -(-K // g["k_per_stage"])
    assert g["total_stages"] == g["tiles"] * g["stages_per_tile"]
    # persistent grid: never more CTAs than stages or than the resident slots
    slots = sms * g["ctas_per_sm"]
    assert 1 <= g["ctas"] <= min(g["total_stages"], slots)
    C, spt = g["cluster"], g["stages_per_tile"]
    stream_k_stages = -(-g["total_stages"] // min(g["total_stages"], slots))
    if C == 0:  # stream-K: one wave; a whole number of CTAs per tile when tiles are few
        if g["total_stages"] > slots and slots // g["tiles"] >= 2:
            assert g["ctas"] == g["tiles"] * (slots // g["tiles"])
        elif g["total_stages"] >= slots:
            assert g["ctas"] == slots
    else:  # cluster split: C CTAs per tile, within one stage of stream-K's work per CTA
        assert 1 <= C <= 8 and C <= spt and spt % C == 0
        assert g["ctas"] == g["tiles"] * C
        assert -(-spt // C) <= max(stream_k_stages + 1, 4)
    # shared memory fits the residency it was sized for
    assert g["smem_bytes"] <= 232448
    assert g["ctas_per_sm"] * (g["smem_bytes"] + 1024) <= 233472
    # the ring: 2..12 stages, or the CTA's whole share of a tile under the cluster split
    assert (1 if g["cluster"] else 2) <= g["stages"] <= 12
    assert g["sm_count"] == sms
    # the same inputs give the same geometry; act dtype does not change it
    assert bsgemv.geometry_for(fmt, "bf16", bs, zp, N, K, max_M, sms) == g


def test_summation_order_independent_of_max_M(L):
    """The per-row summation order is fixed by the work split (CTAs, tiles, stages).  It depends
    on max_M through the residency class -- with 64-row tiles 4 CTAs per SM for max_M <= 8, 3 for
    max_M <= 24, 2 for max_M <= 32 (more accumulator registers); with 128-row tiles (plans for up
    to 16 rows with long work per CTA) 3 for every max_M -- never on M of a call (not an
    argument), which gives row bit-identity across M within a plan."""
    keys = ("ctas", "tiles", "stages_per_tile", "k_per_stage", "rows_per_tile", "consumer_warps")

    def geo(N, K, max_M):
        return bsgemv.geometry_for("int4", "f16", 32, False, N, K, max_M, 152)

    for N, K in ((4096, 4096), (151936, 4096), (300, 2048)):
        tall = geo(N, K, 1)["rows_per_tile"] == 128
        # (plans with max_M > 16 also differ by their activation ring, 32 rows per stage, which
        # can change the cluster size that fits: the geometry is the plan's, never the call's)
        groups = ((1, 2, 5, 8, 9, 12, 16),) if tall else ((1, 2, 5, 8), (9, 12, 16))
        for group in groups:
            ref = geo(N, K, group[0])
            for max_M in group[1:]:
                g = geo(N, K, max_M)
                assert {k: g[k] for k in keys} == {k: ref[k] for k in keys}
        assert geo(N, K, 8)["ctas_per_sm"] == (3 if tall else 4)
        assert geo(N, K, 9)["ctas_per_sm"] == 3
        assert geo(N, K, 16)["rows_per_tile"] == (128 if tall else 64)
        assert geo(N, K, 17)["ctas_per_sm"] == 3 and geo(N, K, 17)["rows_per_tile"] == 64
        assert geo(N, K, 24)["ctas_per_sm"] == 3
        assert geo(N, K, 25)["ctas_per_sm"] == 2
    assert geo(151936, 4096, 1)["rows_per_tile"] == 128  # the lm_head: 1187 tiles, 456 CTAs


def test_stream_k_ranges_cover_every_stage_once():
    """Pure arithmetic of the stream-K split used by the kernel: CTA i owns stages
    [i*T//G, (i+1)*T//G); the CTA owning stage x is ceil((x+1)*G/T) - 1."""
    for T in (1, 2, 7, 32, 64, 1000, 37984):
        for G in sorted({g for g in (1, 2, 3, 304, 296, T) if g <= T}):
            owner = []
            for i in range(G):
                s0, s1 = i * T // G, (i + 1) * T // G
                assert s1 > s0
                owner += [i] * (s1 - s0)
            assert len(owner) == T
            for x in range(0, T, max(1, T // 97)):
                assert -(-((x + 1) * G) // T) - 1 == owner[x]


def test_owner_lookup_without_division():
    """The kernel finds the CTA owning stage x (the largest i with i*T < (x+1)*G) from a
    single-precision quotient corrected by exact products; it must equal the integer formula
    for every grid size up to 640 CTAs and stage counts up to 2^31."""
    import random
    f32 = np.float32

    def owner(x, T, G):
        lim = (x + 1) * G
        i = int(f32(f32(lim - 1) / f32(T)))
        while (i + 1) * T < lim:
            i += 1
        while i > 0 and i * T >= lim:
            i -= 1
        return i

    rng = random.Random(7)
    for T in (1, 2, 3, 64, 1000, 37984, 2 ** 20 + 7, 2 ** 31 - 1):
        for G in (1, 3, 152, 456, 608, 640):
            if G > T:
                continue
            for x in [0, T - 1] + [rng.randrange(T) for _ in range(300)]:
                assert owner(x, T, G) == ((x + 1) * G + T - 1) // T - 1


def test_split_choice_on_the_configuration_shapes(L):
    """Automatic K split at 152 SMs (4 CTAs per SM with 64-row tiles, 3 with 128-row tiles):
    shapes with few tiles take a cluster of CTAs
    per tile (reduced in shared memory), shapes with more tiles than resident CTAs stream-K, with
    a whole number of CTAs per tile when the tiles are fewer than the resident CTAs."""
    def split(fmt, bs, zp, N, K, max_M=1):
        g = bsgemv.geometry_for(fmt, "f16", bs, zp, N, K, max_M, 152)
        return g["cluster"], -(-g["stages_per_tile"] // max(1, g["cluster"])) if g["cluster"] else None
    assert split("int8", 32, True, 2048, 4096) == (8, 2)     # 32 tiles x 16 stages
    assert split("int8", 128, True, 4096, 12288) == (8, 6)   # 64 tiles x 48 stages
    assert split("fp8", 128, False, 5120, 6144) == (6, 4)    # 80 tiles x 24 stages
    # 128-row tiles (96 tiles x 32 stages, 3 CTAs per SM): 4-CTA clusters of 8 stages each
    assert split("int8", 128, True, 12288, 4096) == (4, 8)
    assert split("fp8", 128, False, 5120, 17408)[0] == 0     # 80 tiles x 68 stages
    assert split("int8", 128, True, 4096, 4096) == (8, 2)    # 64 tiles x 16 stages
    assert split("int8", 128, True, 5120, 2048) == (4, 2)    # 80 tiles x 8 stages
    assert split("fp8", 128, False, 512, 2048) == (8, 1)     # 8 tiles x 8 stages
    assert split("int4", 32, False, 151936, 4096)[0] == 0    # 1187 tiles of 128 rows: stream-K
    # plans for max_M = 8: 8-CTA clusters no longer fit next to the activation ring, 4 do
    assert split("fp8", 128, False, 2048, 4096, 8) == (4, 4)  # 32 tiles x 16 stages
    # plans for 16 rows (3 CTAs per SM): 8-CTA clusters exceed the 456 resident CTAs; a 6-CTA
    # cluster of 2-3 stages per CTA cuts the largest share of the even 4-CTA split by a quarter
    assert split("int4", 32, False, 4096, 4096, 16) == (6, 3)   # 64 tiles x 16 stages
    assert split("int4", 32, False, 4096, 4096, 8) == (8, 2)    # 4 CTAs per SM: 8 fit
    # a smaller cut keeps the even split (6 CTAs of 8 stages, not 7 of 7)
    assert split("int4", 32, False, 4096, 12288, 16) == (6, 8)  # 64 tiles x 48 stages
    g = bsgemv.geometry_for("fp8", "f16", 128, False, 5120, 17408, 1, 152)
    assert g["ctas"] == 560                                  # 80 tiles x 7 CTAs
    assert split("nvfp4", 16, False, 248320, 2048)[0] == 0   # 1940 tiles of 128 rows: stream-K


def test_shared_memory_layout_is_aligned_for_every_problem(L):
    """The plan's shared-memory layout keeps every region at the alignment the kernel relies on
    (weight boxes 1024, side boxes 128 as TMA destinations, activation rows and the reduction
    buffer 16, barriers 8); the host rejects a layout that does not instead of launching it.
    Every format, block size and max_M on a spread of shapes must therefore yield a geometry."""
    import itertools
    fmts = ([("int4", bs, zp) for bs in (16, 32, 64, 128, 256) for zp in (False, True)] +
            [("int8", bs, zp) for bs in (16, 32, 64, 128, 256) for zp in (False, True)] +
            [("fp8", 128, False), ("nvfp4", 16, False)])
    for (fmt, bs, zp), N, K, max_M in itertools.product(
            fmts, (1, 333, 5120, 151936), (256, 2048, 12288),
            (1, 2, 3, 5, 8, 9, 13, 16, 17, 23, 32)):
        g = bsgemv.geometry_for(fmt, "f16", bs, zp, N, K, max_M, 152)
        assert g["smem_bytes"] % 8 == 0


# ---------------------------------------------------------------------------- dense GEMV
@pytest.mark.parametrize("args,code", [
    (("f16", 0, 2048, 1), bsgemv.ERR_INVALID_ARG),        # N = 0
    (("f16", 64, 2048, 9), bsgemv.ERR_INVALID_ARG),       # max_M > 8
    (("f16", 64, 2048, 0), bsgemv.ERR_INVALID_ARG),       # max_M = 0
    (("f16", 64, 0, 1), bsgemv.ERR_INVALID_ARG),          # K = 0
])
def test_dense_invalid_problems_rejected_on_host(L, args, code):
    act, N, K, mm = args
    with pytest.raises(bsgemv.BsgemvError) as e:
        bsgemv.dense_geometry_for(act, N, K, mm, 152)
    assert e.value.status == code
    with pytest.raises(bsgemv.BsgemvError) as e:
        bsgemv.DensePlan(act, N, K, mm)
    assert e.value.status == code


@pytest.mark.parametrize("N,K", [(1, 2048), (7, 100), (1001, 4096), (64, 2044), (64, 8)])
def test_dense_geometry_without_tma_pitches(L, N, K):
    """N or K not a multiple of 8 (or K < 16): the CUDA-core kernel, 8 columns per CTA."""
    g = bsgemv.dense_geometry_for("f16", N, K, 8, 152)
    assert g["variant"] == bsgemv.VARIANTS["cuda_core"] and g["rows_per_tile"] == 8
    assert g["tiles"] == -(-N // 8) and g["stages_per_tile"] == -(-K // 256)
    S = g["cluster"]
    assert 1 <= S <= min(8, g["stages_per_tile"]) and g["ctas"] == g["tiles"] * S


@pytest.mark.parametrize("N,K", [(8, 16), (32, 2048), (256, 2048), (1024, 2048), (1000, 4096),
                                 (4096, 4096), (65536, 512)])
@pytest.mark.parametrize("sms", [132, 152])
def test_dense_geometry(L, N, K, sms):
    g = bsgemv.dense_geometry_for("f16", N, K, 8, sms)
    assert g["rows_per_tile"] == 64 and g["k_per_stage"] == 64 and g["consumer_warps"] == 4
    assert g["tiles"] == -(-N // 64) and g["stages_per_tile"] == -(-K // 64)
    S = g["cluster"]
    assert 1 <= S <= 8 and S <= g["stages_per_tile"]           # every CTA holds a stage
    assert g["ctas"] == g["tiles"] * S
    assert S == 1 or g["ctas"] <= 2 * sms                       # split only to fill the SMs
    assert 1 <= g["stages"] <= 8 and g["stages"] <= -(-g["stages_per_tile"] // S)
    assert g["smem_bytes"] <= 232448
    assert bsgemv.dense_geometry_for("bf16", N, K, 8, sms) == g


def test_residency_of_plans_for_17_to_24_rows(L):
    """Plans for 17..24 rows take three n8 tiles at 3 CTAs per SM, unless that residency loses the
    cluster split (shares of at most 4 stages) that four tiles at 2 CTAs per SM keep."""
    def geo(fmt, bs, zp, N, K, mm):
        g = bsgemv.geometry_for(fmt, "f16", bs, zp, N, K, mm, 152)
        return g["ctas_per_sm"], g["cluster"]
    assert geo("fp8", 128, False, 4096, 2048, 24) == (2, 4)       # small: the split wins
    assert geo("int8", 128, True, 2048, 4096, 20) == (2, 4)
    assert geo("int4", 32, False, 12288, 4096, 24)[0] == 3        # larger: three tiles win
    assert geo("int4", 32, False, 4096, 12288, 17)[0] == 3        # long shares (12 stages)
    assert geo("nvfp4", 16, False, 248320, 2048, 24) == (3, 0)
    for mm in (17, 20, 24):   # the same plan geometry for every max_M of the range
        assert geo("fp8", 128, False, 4096, 2048, mm) == (2, 4)


def test_header_is_c_and_the_library_links_from_c(L, tmp_path):
    """include/bsgemv.h compiles as C11 and a C program links against the library and runs its
    host-only entry points."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = bsgemv.lib_path()
    exe = tmp_path / "c_abi_check"
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi_check.c"), lib, "-o", str(exe),
                        f"-Wl,-rpath,{os.path.dirname(lib)}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr
