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
