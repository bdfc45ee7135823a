"""Bit-exact checks of the engine's storage-format routines against the oracle
(uint8 codes, scales, zero-points; INT4 codes and fp16 scales; E5M2 bytes)."""
import json
import os

import numpy as np
import pytest

import oracle as O
import synthetic as S
from autoregressive_decode_gb300 import kie

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_e5m2_all_fp16_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    gpu = kie.convert_fp8_e5m2(bits.view(np.float16))
    ref = O.e5m2_from_f16_bits(bits)
    f = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(f)
    np.testing.assert_array_equal(gpu[~nan], ref[~nan])
    back = O.e5m2_to_f16_bits(gpu[nan]).view(np.float16)
    assert np.all(np.isnan(back.astype(np.float32)))


@pytest.mark.parametrize("seed", range(4))
def test_u8_segments_bit_exact(seed):
    n_seg, seg = 37, 128 * 64
    x = S.outlier_f16(100 + seed, 5, (n_seg, seg))
    x[3] = np.float16(-2.5)                      # constant segment
    x[4, :] = np.float16(0.0)
    x[4, 0], x[4, 1] = np.float16(-1.2), np.float16(2.8)   # the page's worked example range
    codes, scale, zp = kie.quantize_kv_u8(x, n_seg)
    for s in range(n_seg):
        c, sc, z = O.u8_quantize(x[s].astype(np.float32))
        assert scale[s] == sc and zp[s] == z, s
        np.testing.assert_array_equal(codes[s], c)
    g = json.load(open(os.path.join(GOLD, "adaptive_range_worked_example.json")))
    assert zp[4] == g["zero_point_printed"]


@pytest.mark.parametrize("shape", [(64, 128), (33, 4096), (7, 11008)])
def test_int4_bit_exact(shape):
    w = S.normal_f16(200 + shape[0], 9, shape)
    w[0, :128] = 0                                # all-zero group
    codes, sc = kie.quantize_int4_g128(w)
    rc, rs = O.int4_quantize_g128(w)
    np.testing.assert_array_equal(sc.view(np.uint16), rs.view(np.uint16))
    np.testing.assert_array_equal(codes, rc)


@pytest.mark.parametrize("shape", [(64, 2048), (37, 8192), (9, 250)])
def test_fp8_rows_bit_exact(shape):
    """FP8 E4M3 weight codes and fp32 row scales equal the oracle's, including
    an all-zero row and a row with one large outlier."""
    w = S.normal_f16(300 + shape[0], 9, shape)
    w[0] = 0
    w[1, 3] = np.float16(40.0)
    codes, sc = kie.quantize_fp8_rows(w)
    rc, rs = O.fp8_quantize_rows(w)
    np.testing.assert_array_equal(sc.view(np.uint32), rs.view(np.uint32))
    np.testing.assert_array_equal(codes, rc)


@pytest.mark.parametrize("shape", [(64, 2048), (37, 4096 + 16)])
def test_nvfp4_quantiser_bit_exact(shape):
    """NVFP4 codes, E4M3 block scales and fp32 row scales from the GPU
    quantiser equal the oracle's, bit for bit (including an all-zero row, a
    row with negative zeros and a row of tiny values)."""
    rows, cols = shape
    w = S.normal_f16(77, 5, shape)
    w[3] = 0
    w[5, ::3] = np.float16(-0.0)
    w[7] = (w[7].astype(np.float32) * 1e-3).astype(np.float16)
    codes, bs, rs = kie.quantize_nvfp4_rows(w)
    rc, rb, rr = O.fp4_quantize_rows(w)
    np.testing.assert_array_equal(rs.view(np.uint32), rr.view(np.uint32))
    np.testing.assert_array_equal(bs, rb)
    np.testing.assert_array_equal(codes, rc)
