"""The seeded generators produce the documented storage formats and distributions."""
import numpy as np

from block_scaled_bit_gb300 import synth


def test_shapes_dtypes_and_ranges():
    c = synth.make_case("int4", "f16", 32, True, 64, 512, 3, 1)
    assert c.W.shape == (64, 256) and c.W.dtype == np.uint8
    assert c.scales.shape == (64, 16) and c.scales.dtype == np.uint16
    s = c.scales.view(np.float16).astype(np.float64)
    assert s.min() >= 0.005 * (1 - 2 ** -10) and s.max() <= 0.02 * (1 + 2 ** -10)
    assert c.zp.shape == (64, 8) and c.A.shape == (3, 512)
    c8 = synth.make_case("int8", "f16", 128, True, 32, 1024, 1, 2)
    assert c8.zp.min() >= 120 and c8.zp.max() <= 136 and c8.scales.shape == (32, 8)
    f8 = synth.make_case("fp8", "f16", 128, False, 16, 512, 1, 3)
    assert f8.scales.dtype == np.float32 and f8.W.shape == (16, 512)
    assert not np.isin(f8.W, [0x7F, 0xFF]).any(), "saturated, never NaN"
    vals = synth.to_e4m3_codes(np.array([500.0, -1e6, 448.0, 0.0]))
    assert vals.tolist() == [0x7E, 0xFE, 0x7E, 0x00], "saturates to +-448, never NaN"
    n4 = synth.make_case("nvfp4", "bf16", 16, False, 16, 256, 2, 4)
    assert n4.scales.min() >= 0x18 and n4.scales.max() <= 0x58 and n4.gscale[0] == 1 / 64
    assert n4.W.shape == (16, 128) and n4.scales.shape == (16, 16)


def test_seeded_and_rows_independent_of_M():
    a = synth.make_case("int8", "bf16", 32, True, 8, 256, 16, 9)
    b = synth.make_case("int8", "bf16", 32, True, 8, 256, 4, 9)
    assert np.array_equal(a.W, b.W) and np.array_equal(a.A[:4], b.A)
    assert np.array_equal(a.with_M(2).A, a.A[:2])


def test_config_enumeration():
    shapes = synth.all_shapes()
    assert len(synth.config_shapes(2)) == 10 and len(synth.config_shapes(3)) == 8
    # one seed per (config, shape, block size); the fp16 and bf16 variants share weights
    assert len({s.seed for s in shapes}) == len({(s.config, s.shape_index, s.block_size) for s in shapes})
    c1 = synth.config_shapes(1)[0]
    assert (c1.N, c1.K, c1.block_size, c1.has_zp) == (1024, 512, 32, True)


def test_rows_up_to_32_and_bias_draws():
    a32 = synth.make_case("int4", "f16", 32, False, 16, 256, 32, 5)
    a16 = synth.make_case("int4", "f16", 32, False, 16, 256, 16, 5)
    assert a32.A.shape == (32, 256) and np.array_equal(a32.A[:16], a16.A)
    b = a32.with_bias()
    assert b.bias.shape == (16,) and b.bias.dtype == np.uint16
    assert np.array_equal(b.with_M(3).bias, b.bias)            # the bias does not depend on M
    assert np.array_equal(b.W, a32.W) and np.array_equal(b.A, a32.A)
    assert np.array_equal(synth.make_case("int4", "f16", 32, False, 16, 256, 32, 5).with_bias().bias,
                          b.bias)                              # seeded
    assert b.algorithmic_bytes() == a32.algorithmic_bytes() + 2 * 16


def test_dense_operands():
    A, B = synth.dense_operands("f16", 8, 300, 1024, seed=1)
    assert A.shape == (8, 1024) and B.shape == (1024, 300) and A.dtype == B.dtype == np.uint16
    A2, B2 = synth.dense_operands("f16", 3, 300, 1024, seed=1)
    assert np.array_equal(A2, A[:3]) and np.array_equal(B2, B)
    var = B.view(np.float16).astype(np.float64).var()
    assert abs(var * 1024 - 1.0) < 0.05                        # B ~ N(0, 1/K)
    Ab, Bb = synth.dense_operands("bf16", 2, 8, 64, seed=2)
    assert Ab.dtype == Bb.dtype == np.uint16 and Bb.shape == (64, 8)
