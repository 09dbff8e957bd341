"""Seeded synthetic inputs for the block-scaled small-M GEMV.

This module only draws random numbers and stores them in the documented storage formats.  It
holds none of the method's arithmetic (no decoding, dequantisation or dot products), so both the
CUDA path and the CPU oracle can be fed from it.  Conversions to storage types are done by
library casts: numpy's float64 -> float16 (round-to-nearest-even), torch's float32 -> bfloat16 and
float32 -> float8_e4m3fn (round-to-nearest-even).

Storage layouts (the [N, blocks, blob] layout of "[CUDA] Batched small-M GEMV for MatMulNBits
(4-bit/8-bit)", Description):
  int4   W [N, K/2] u8 (two codes per byte, low nibble = even k), scales [N, nb] fp16,
         zp [N, ceil(nb/2)] u8 (two per byte, low nibble = even block)      nb = K / block_size
  int8   W [N, K] u8, scales [N, nb] fp16, zp [N, nb] u8
  fp8    W [N, K] E4M3 codes, scales [N, K/128] fp32
  nvfp4  W [N, K/2] u8 (two E2M1 codes per byte, low nibble = even k), scales [N, K/16] E4M3 codes,
         gscale [1] fp32
  A      [M, K] fp16 or bf16 bit patterns (uint16)

Because every nibble pattern is equally likely, uniform int4 / E2M1 codes packed two per byte are
exactly uniform random bytes, and so are uniformly drawn packed int4 zero points.

Seeds follow seed = 1000 * config + 10 * shape index + block-size code; the activations of a case
come from their own stream so that row m of A is the same for every M (row m of an M-row draw is
row m of the 16-row draw).
"""
from __future__ import annotations

import dataclasses

import numpy as np

MAX_M = 32  # activation rows drawn per case; row m is the same for every M


@dataclasses.dataclass
class Case:
    fmt: str                 # "int4" | "int8" | "fp8" | "nvfp4"
    act: str                 # "f16" | "bf16"
    block_size: int
    has_zp: bool
    N: int
    K: int
    M: int
    A: np.ndarray            # uint16 [M, K]
    W: np.ndarray            # uint8 [N, row bytes]
    scales: np.ndarray       # uint16 (fp16 bits) | float32 | uint8 (E4M3 codes)  [N, nb]
    zp: np.ndarray | None    # uint8 or None
    gscale: np.ndarray | None  # float32 [1] (nvfp4) or None
    seed: int = 0
    name: str = ""
    bias: np.ndarray | None = None  # uint16 [N] activation-dtype bits, or None (no bias)

    def with_M(self, M: int) -> "Case":
        """The same weights with the first M rows of this case's 16-row activation draw."""
        A = activations(self.seed, M, self.K, self.act)
        return dataclasses.replace(self, M=M, A=A)

    def with_bias(self, sigma: float = 1.0) -> "Case":
        """The same case with a bias [N] ~ N(0, sigma^2) rounded to the activation dtype, drawn
        from its own stream (the weights and activations are unchanged)."""
        rng = np.random.Generator(np.random.PCG64([self.seed, 0xB1A5]))
        x = rng.standard_normal(self.N) * sigma
        bias = to_f16_bits(x) if self.act == "f16" else to_bf16_bits(x)
        return dataclasses.replace(self, bias=bias)

    @property
    def nb(self) -> int:
        return self.K // self.block_size

    def algorithmic_bytes(self, M: int | None = None) -> int:
        """Bytes of W + scales + zp + A + y that one call must move (the roofline numerator)."""
        M = self.M if M is None else M
        b = self.W.nbytes + self.scales.nbytes
        if self.zp is not None:
            b += self.zp.nbytes
        if self.gscale is not None:
            b += 4
        if self.bias is not None:
            b += self.bias.nbytes
        return b + 2 * M * self.K + 2 * M * self.N


# ------------------------------------------------------------------------------------ dtypes
def to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.float32)))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float -> E4M3 code by torch's round-to-nearest-even cast, after saturating to +-448."""
    import torch
    x = np.clip(np.asarray(x, dtype=np.float32), -448.0, 448.0)
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


# ------------------------------------------------------------------------------------ draws
def activations(seed: int, M: int, K: int, act: str) -> np.ndarray:
    """A ~ N(0, 1) rounded to the activation dtype; row m is independent of M."""
    if not 1 <= M <= MAX_M:
        raise ValueError(f"M must be in 1..{MAX_M}")
    rng = np.random.Generator(np.random.PCG64([seed, 0xA11CE]))
    x = rng.standard_normal((MAX_M, K))[:M]
    return to_f16_bits(x) if act == "f16" else to_bf16_bits(x)


def make_case(fmt: str, act: str, block_size: int, has_zp: bool, N: int, K: int, M: int,
              seed: int, *, scale_range=None, zp_range=None, fp8_sigma: float = 64.0,
              nvfp4_scale_codes=(0x18, 0x58), gscale: float = 1.0 / 64.0, name: str = "") -> Case:
    """Draw one seeded case.  Defaults follow the synthetic recipe of each format:
    int4: scales U[0.005, 0.02], zp uniform nibbles; int8: scales U[0.001, 0.004], zp U{120..136};
    fp8: W = E4M3(N(0,1) * 64, saturated), scales U[0.5, 2] / 448 (fp32);
    nvfp4: codes uniform, E4M3 scale codes uniform over 0x18..0x58 ([2^-4, 2^4]), gscale 1/64."""
    if K % block_size != 0:
        raise ValueError("K must be a multiple of block_size")
    rng = np.random.Generator(np.random.PCG64(seed))
    nb = K // block_size
    zp = None
    g = None
    if fmt == "int4":
        W = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
        lo, hi = scale_range or (0.005, 0.02)
        scales = to_f16_bits(rng.uniform(lo, hi, size=(N, nb)))
        if has_zp:
            if zp_range is None:
                zp = rng.integers(0, 256, size=(N, (nb + 1) // 2), dtype=np.uint8)
            else:  # a restricted nibble range, packed low nibble = even block
                z = rng.integers(zp_range[0], zp_range[1] + 1, size=(N, 2 * ((nb + 1) // 2)))
                zp = (z[:, 0::2] | (z[:, 1::2] << 4)).astype(np.uint8)
    elif fmt == "int8":
        W = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
        lo, hi = scale_range or (0.001, 0.004)
        scales = to_f16_bits(rng.uniform(lo, hi, size=(N, nb)))
        if has_zp:
            zlo, zhi = zp_range or (120, 136)
            zp = rng.integers(zlo, zhi + 1, size=(N, nb), dtype=np.uint8)
    elif fmt == "fp8":
        if block_size != 128:
            raise ValueError("fp8 uses one scale per 128 k")
        W = np.empty((N, K), dtype=np.uint8)
        step = max(1, (1 << 24) // K)
        for r0 in range(0, N, step):
            r1 = min(N, r0 + step)
            W[r0:r1] = to_e4m3_codes(rng.standard_normal((r1 - r0, K)) * fp8_sigma)
        lo, hi = scale_range or (0.5, 2.0)
        scales = (rng.uniform(lo, hi, size=(N, nb)) / 448.0).astype(np.float32)
        has_zp = False
    elif fmt == "nvfp4":
        if block_size != 16:
            raise ValueError("nvfp4 uses one E4M3 scale per 16 k")
        W = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
        c0, c1 = nvfp4_scale_codes
        scales = rng.integers(c0, c1 + 1, size=(N, nb), dtype=np.uint8)
        g = np.array([gscale], dtype=np.float32)
        has_zp = False
    else:
        raise ValueError(f"unknown format {fmt!r}")
    A = activations(seed, M, K, act)
    return Case(fmt, act, block_size, bool(has_zp), N, K, M, A, W, scales, zp, g, seed, name)


# ------------------------------------------------------------------------------------ pin inputs
# Inputs built to pin the GPU path to the oracle bit for bit (not draws of a workload).  They
# hold codes and values only; what they make exact or special is stated per function.

def _act_bits(x, act: str) -> np.ndarray:
    return to_f16_bits(x) if act == "f16" else to_bf16_bits(x)


def _pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[R, 2n] codes 0..15 -> [R, n] bytes, the even position in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _row_perms(rng, rows: int, n: int) -> np.ndarray:
    """`rows` independent permutations of 0 .. n-1."""
    return np.argsort(rng.random((rows, n)), axis=1)


ALL_CODES_K = {"int4": 16 * 16 * 16, "int8": 256 * 256, "fp8": 4 * 256, "nvfp4": 16 * 256}


def all_codes_case(fmt: str, act: str, block_size: int, has_zp: bool, N: int, M: int,
                   seed: int) -> Case:
    """Every code of the format in every row, K fixed per format (ALL_CODES_K):
    int4 / int8: the codes of each row are consecutive random permutations of 0..15 / 0..255.
      With zero points, K is cut into spans of max(levels, block_size) k; every block of span j
      has the zero point j mod levels, every span holds whole permutations, and there are at
      least `levels` spans -- so every (q, zp) pair occurs in every row.  Without zero points
      every code meets the implicit zero point;
    fp8: all 256 E4M3 codes (NaN 0x7F / 0xFF, subnormals, +-0, +-448) four times per row;
    nvfp4: all 256 E4M3 codes as block scales (one per 16-block, a random order per row), and
      every E2M1 code once in every block.
    Scales of the int formats and FP8 come from the format's usual draw; A ~ N(0, 1)."""
    rng = np.random.Generator(np.random.PCG64([seed, 0xC0DE5]))
    K = ALL_CODES_K[fmt]
    base = make_case(fmt, act, block_size, has_zp, N, K, M, seed)
    if fmt in ("int4", "int8"):
        levels = 16 if fmt == "int4" else 256
        q = np.concatenate([_row_perms(rng, N, levels) for _ in range(K // levels)], axis=1)
        W = _pack_nibbles(q) if fmt == "int4" else q.astype(np.uint8)
        zp = base.zp
        if has_zp:
            nb = K // block_size
            span = max(levels, block_size)
            zb = ((np.arange(nb) * block_size // span) % levels)[None, :].repeat(N, axis=0)
            if fmt == "int4":
                z = np.zeros((N, 2 * ((nb + 1) // 2)), dtype=np.int64)
                z[:, :nb] = zb
                zp = _pack_nibbles(z)
            else:
                zp = zb.astype(np.uint8)
        return dataclasses.replace(base, W=W, zp=zp, name=f"allcodes_{fmt}")
    if fmt == "fp8":
        W = np.concatenate([_row_perms(rng, N, 256) for _ in range(K // 256)], axis=1).astype(np.uint8)
        return dataclasses.replace(base, W=W, name="allcodes_fp8")
    # nvfp4
    e2m1 = np.concatenate([_row_perms(rng, N, 16) for _ in range(K // 16)], axis=1)
    scales = _row_perms(rng, N, 256).astype(np.uint8)
    return dataclasses.replace(base, W=_pack_nibbles(e2m1), scales=scales, name="allcodes_nvfp4")


def nan_rows_case(fmt: str, act: str, N: int, K: int, M: int, seed: int, nan_rows) -> Case:
    """FP8 or NVFP4 weights whose only NaN codes (E4M3 0x7F / 0xFF: FP8 weight codes, NVFP4
    block scales) sit in the rows `nan_rows`, one or a few per row at random k; every other
    E4M3 code is drawn uniformly from the 254 finite codes (subnormals, +-0, +-448 included)."""
    rng = np.random.Generator(np.random.PCG64([seed, 0x4A4E]))
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    if fmt == "fp8":
        base = make_case("fp8", act, 128, False, N, K, M, seed)
        W = finite[rng.integers(0, finite.size, size=(N, K))]
        for n in nan_rows:
            for _ in range(int(rng.integers(1, 4))):
                W[n, rng.integers(0, K)] = rng.choice([0x7F, 0xFF])
        return dataclasses.replace(base, W=W, name="nanrows_fp8")
    if fmt != "nvfp4":
        raise ValueError("NaN codes exist in the E4M3-coded formats only")
    base = make_case("nvfp4", act, 16, False, N, K, M, seed)
    S = finite[rng.integers(0, finite.size, size=(N, K // 16))]
    for n in nan_rows:
        for _ in range(int(rng.integers(1, 4))):
            S[n, rng.integers(0, K // 16)] = rng.choice([0x7F, 0xFF])
    return dataclasses.replace(base, scales=S, name="nanrows_nvfp4")


def exact_case(fmt: str, act: str, block_size: int, has_zp: bool, N: int, K: int, M: int,
               seed: int) -> Case:
    """Inputs whose every partial sum, in any order, is exact in fp32, so that an fp32
    accumulation reaches the exact dot product and the output rounds as the oracle's does:
    small-integer activations in [-3, 3], power-of-two block scales, weight values on a coarse
    grid, K small enough that sum_k |a_k w_k| stays below 2^24 grid steps:
      int4  scales 2^-2 .. 2^2 (fp16), q and zp uniform nibbles;
      int8  scales 2^-2 .. 2^0 (fp16), q and zp uniform bytes;
      fp8   E4M3 codes of exponent field 5..9 (|w| in [0.25, 7.5]), either sign, scales
            2^-1 .. 2^0 (fp32);
      nvfp4 E2M1 codes uniform, E4M3 block scales 2^-2 .. 2^2 (codes 0x28 .. 0x48, mantissa 0),
            global scale 2^-6.
    Row m of A is the same for every M."""
    base = make_case(fmt, act, block_size, has_zp, N, K, M, seed)
    rng = np.random.Generator(np.random.PCG64([seed, 0xE4AC7]))
    nb = K // block_size
    arng = np.random.Generator(np.random.PCG64([seed, 0xA11CE, 3]))   # row m independent of M
    A = _act_bits(arng.integers(-3, 4, size=(MAX_M, K))[:M].astype(np.float64), act)
    if fmt == "int4":
        scales = to_f16_bits(np.exp2(rng.integers(-2, 3, size=(N, nb))))
        return dataclasses.replace(base, A=A, scales=scales, name="exact_int4")
    if fmt == "int8":
        scales = to_f16_bits(np.exp2(rng.integers(-2, 1, size=(N, nb))))
        zp = rng.integers(0, 256, size=(N, nb), dtype=np.uint8) if has_zp else None
        return dataclasses.replace(base, A=A, scales=scales, zp=zp, name="exact_int8")
    if fmt == "fp8":
        e = rng.integers(5, 10, size=(N, K))
        m = rng.integers(0, 8, size=(N, K))
        s = rng.integers(0, 2, size=(N, K))
        W = ((s << 7) | (e << 3) | m).astype(np.uint8)
        scales = np.exp2(rng.integers(-1, 1, size=(N, nb))).astype(np.float32)
        return dataclasses.replace(base, A=A, W=W, scales=scales, name="exact_fp8")
    if fmt == "nvfp4":
        scales = (rng.integers(5, 10, size=(N, nb)) << 3).astype(np.uint8)
        return dataclasses.replace(base, A=A, scales=scales,
                                   gscale=np.array([2.0 ** -6], dtype=np.float32), name="exact_nvfp4")
    raise ValueError(f"unknown format {fmt!r}")


def one_hot_rows(M: int, K: int, act: str) -> tuple:
    """Activations whose row m is 1.0 at k_m and 0 elsewhere (the k_m distinct, spread over the
    blocks of K); returns (A bits [M, K], k_m [M])."""
    ks = (np.arange(M) * 613 + 17) % K
    x = np.zeros((M, K))
    x[np.arange(M), ks] = 1.0
    return _act_bits(x, act), ks


def one_hot_case(fmt: str, act: str, block_size: int, has_zp: bool, N: int, K: int, M: int,
                 seed: int) -> tuple:
    """A one-hot activation case (see one_hot_rows) over the format's usual weight draw, with
    FP8 scales drawn on the fp16 grid (U[0.5, 2] / 448 rounded to fp16, stored as fp32) so that
    every dequantised weight is exact in fp32.  Returns (case, k_m)."""
    base = make_case(fmt, act, block_size, has_zp, N, K, M, seed)
    A, ks = one_hot_rows(M, K, act)
    case = dataclasses.replace(base, A=A, name=f"onehot_{fmt}")
    if fmt == "fp8":
        s16 = np.asarray(base.scales, dtype=np.float64).astype(np.float16).astype(np.float32)
        case = dataclasses.replace(case, scales=s16)
    return case, ks


def dense_operands(act: str, M: int, N: int, K: int, seed: int):
    """Dense small-N GEMV inputs ("[CUDA] MatMul: add an opt-in split-K GEMV for small-N fp16
    shapes"): A [M, K] ~ N(0, 1) and B [K, N] ~ N(0, 1/K) (unit-variance outputs), row-major,
    rounded to the activation dtype; returned as uint16 bit patterns.  Row m of A is the same
    for every M."""
    A = activations(seed, M, K, act)
    rng = np.random.Generator(np.random.PCG64([seed, 0xDE45E]))
    x = rng.standard_normal((K, N)) / np.sqrt(K)
    B = to_f16_bits(x) if act == "f16" else to_bf16_bits(x)
    return A, B


# ------------------------------------------------------------------------------------ configs
@dataclasses.dataclass(frozen=True)
class Shape:
    config: int
    fmt: str
    act: str
    block_size: int
    has_zp: bool
    N: int
    K: int
    Ms: tuple
    shape_index: int
    label: str = ""

    @property
    def seed(self) -> int:
        return 1000 * self.config + 10 * self.shape_index + {16: 1, 32: 2, 64: 3, 128: 4, 256: 5}[self.block_size]

    @property
    def name(self) -> str:
        zp = "zp" if self.has_zp else "nozp"
        return f"c{self.config}_{self.fmt}_{self.act}_bs{self.block_size}_{zp}_N{self.N}_K{self.K}"

    def case(self, M: int | None = None) -> Case:
        return make_case(self.fmt, self.act, self.block_size, self.has_zp, self.N, self.K,
                         self.Ms[0] if M is None else M, self.seed, name=self.name)


def config_shapes(config: int) -> list:
    """The five synthetic workload configurations, enumerated shape by shape."""
    out = []
    if config == 1:   # int4 with zero points, K=512, N=1024, bs 32, M=1
        out.append(Shape(1, "int4", "f16", 32, True, 1024, 512, (1,), 0))
    elif config == 2:  # int8 with zero points, M=1, bs 128 and 32; shapes given as K x N
        kn = [(2048, 5120), (4096, 2048), (4096, 4096), (4096, 12288), (12288, 4096)]
        for bs in (128, 32):
            for i, (K, N) in enumerate(kn):
                out.append(Shape(2, "int8", "f16", bs, True, N, K, (1,), i))
    elif config == 3:  # int4, zp fixed at 8, bs 32, M sweep, fp16 and bf16; shapes K x N
        kn = [(4096, 4096), (4096, 12288), (12288, 4096), (4096, 151936)]
        for act in ("f16", "bf16"):
            for i, (K, N) in enumerate(kn):
                out.append(Shape(3, "int4", act, 32, False, N, K, (1, 2, 4, 8, 16), i))
    elif config == 4:  # FP8 E4M3, bs 128 fp32 scale; shapes N x K
        nk = [(8192, 2048), (4096, 2048), (2048, 4096), (512, 2048), (5120, 6144), (6144, 5120),
              (5120, 17408)]
        for i, (N, K) in enumerate(nk):
            out.append(Shape(4, "fp8", "f16", 128, False, N, K, (1, 4, 8), i))
    elif config == 5:  # NVFP4; shapes N x K
        nk = [(248320, 2048), (2048, 2048), (512, 2048)]
        for i, (N, K) in enumerate(nk):
            out.append(Shape(5, "nvfp4", "f16", 16, False, N, K, (1, 2, 4), i))
    else:
        raise ValueError("config must be 1..5")
    return out


def all_shapes() -> list:
    return [s for c in range(1, 6) for s in config_shapes(c)]
