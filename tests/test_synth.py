"""Seeded input generator: determinism, distributions, bf16/e4m3 rounding against
their format definitions, outlier channels and the orthogonal rotation."""
import math

import numpy as np
import pytest

from exact_tiled_attention_16_gb300 import synth


def test_determinism_and_independence():
    a = synth.normal_f32((4, 64), 7, synth.STREAM_Q)
    b = synth.normal_f32((4, 64), 7, synth.STREAM_Q)
    c = synth.normal_f32((4, 64), 7, synth.STREAM_K)
    d = synth.normal_f32((4, 64), 8, synth.STREAM_Q)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_normal_moments():
    x = synth.normal_f32((1 << 20,), 3, 0).astype(np.float64)
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1) < 5e-3
    assert abs((x ** 4).mean() - 3) < 3e-2  # Gaussian kurtosis


def test_bf16_rne_against_definition():
    # exactly representable values survive; halfway cases go to the even mantissa
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)
    vals = np.array([one, one + ulp / 2, one + ulp + ulp / 2, one + ulp / 4, -3.5, 0.0, 65280.0],
                    dtype=np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(vals))
    np.testing.assert_array_equal(got, np.array([1.0, 1.0, 1.0 + 2 * ulp, 1.0, -3.5, 0.0, 65280.0],
                                                dtype=np.float32))


def test_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    x = synth.normal_f32((100000,), 1, 0) * np.float32(37.0)
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_table_against_spec():
    # OCP FP8 E4M3: max finite 448 = 1.75*2^8, min normal 2^-6, min subnormal 2^-9
    assert synth.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert synth.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6
    assert synth.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9
    assert synth.e4m3_decode(np.uint8(0x38)) == 1.0
    assert synth.e4m3_decode(np.uint8(0xB8)) == -1.0
    assert np.isnan(synth.e4m3_decode(np.uint8(0x7F)))
    assert np.isnan(synth.e4m3_decode(np.uint8(0xFF)))
    # every finite code round-trips through encode
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = synth.e4m3_decode(codes)
    back = synth.e4m3_encode_satfinite(vals)
    np.testing.assert_array_equal(back, codes)
    # a negative value that rounds to zero keeps its sign
    assert synth.e4m3_encode_satfinite(np.array(-1e-6)) == 0x80


def test_e4m3_rounding_and_saturation():
    enc = synth.e4m3_encode_satfinite
    dec = synth.e4m3_decode
    assert dec(enc(np.array(1000.0))) == 448.0
    assert dec(enc(np.array(-1e9))) == -448.0
    assert dec(enc(np.array(464.0))) == 448.0
    # tie between 1.0 (code 0x38, even) and 1.125 (0x39) -> 1.0
    assert dec(enc(np.array(1.0625))) == 1.0
    # tie between 1.125 (0x39) and 1.25 (0x3A, even) -> 1.25
    assert dec(enc(np.array(1.1875))) == 1.25
    # half of the smallest subnormal ties to zero
    assert dec(enc(np.array(2.0 ** -10))) == 0.0
    assert dec(enc(np.array(2.0 ** -10 * 1.01))) == 2.0 ** -9


def test_e4m3_matches_torch_in_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8")
    x = synth.normal_f32((200000,), 2, 0).astype(np.float64) * 40.0
    x = np.clip(x, -448, 448)
    ours = synth.e4m3_encode_satfinite(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_block_quantize_roundtrip():
    g = np.random.default_rng(0)
    x = g.standard_normal((2, 3, 300, 16)) * 5
    x[0, 1, 128:256] = 0.0  # an all-zero block gets scale 1
    codes, scales = synth.block_quantize_e4m3(x)
    assert codes.shape == x.shape and scales.shape == (2, 3, 3)
    assert scales[0, 1, 1] == 1.0
    deq = synth.block_dequantize_e4m3(codes, scales)
    # per block the largest magnitude maps to +-448 exactly (up to fp32 scale rounding)
    for t in range(3):
        blk = np.abs(x[:, :, t * 128:(t + 1) * 128]).max(axis=(2, 3))
        mx = np.abs(synth.e4m3_decode(codes[:, :, t * 128:(t + 1) * 128])).max(axis=(2, 3))
        assert np.all((mx == 448.0) | (blk == 0))
    # relative error of e4m3 is at most 2^-4 for normal values
    big = np.abs(x) > 2.0 ** -6 * np.repeat(scales, 128, axis=2)[:, :, :300, None]
    rel = np.abs(deq - x)[big] / np.abs(x)[big]
    assert rel.max() <= 2.0 ** -4 + 1e-12


def test_outlier_channels():
    ch = synth.outlier_channels(64, 0.02, 4, synth.STREAM_OUTLIER_QK)
    assert len(ch) == 2 and len(set(ch.tolist())) == 2
    assert len(synth.outlier_channels(128, 0.01, 5, 3)) == 2
    w = synth.make_bf16(1, 2, 256, 64, False, 4, qk_outlier_frac=0.02, qk_outlier_mult=20.0)
    q = synth.bf16_bits_to_f64(w.q)
    k = synth.bf16_bits_to_f64(w.k)
    ch = w.meta["qk_outlier_channels"]
    other = [c for c in range(64) if c not in ch]
    assert q[..., ch].std() > 15 and k[..., ch].std() > 15
    assert abs(q[..., other].std() - 1) < 0.05


def test_haar_orthogonal():
    r = synth.haar_orthogonal(128, 5)
    np.testing.assert_allclose(r.T @ r, np.eye(128), atol=1e-12)
    np.testing.assert_array_equal(r, synth.haar_orthogonal(128, 5))
    # rotation preserves inner products, so Q'K'^T = Q K^T before quantisation
    g = np.random.default_rng(1)
    a, b = g.standard_normal((10, 128)), g.standard_normal((12, 128))
    np.testing.assert_allclose((a @ r) @ (b @ r).T, a @ b.T, atol=1e-10)


def test_fp8_workload_shapes():
    w = synth.make_fp8(1, 2, 300, 128, False, 5)
    assert w.q.dtype == np.uint8 and w.q.shape == (1, 2, 300, 128)
    assert w.q_scale.shape == (1, 2, 3) and w.q_scale.dtype == np.float32
    q, k, v = w.head_f64(0, 1)
    assert q.shape == (300, 128) and np.isfinite(q).all()


def test_sample_rows():
    r = synth.sample_rows(16384, 256, 3, 0, 5)
    assert len(r) == 256 and len(set(r.tolist())) == 256
    for x in (0, 1, 127, 128, 16383):
        assert x in r
    np.testing.assert_array_equal(r, synth.sample_rows(16384, 256, 3, 0, 5))
    assert not np.array_equal(r, synth.sample_rows(16384, 256, 3, 0, 6))
    np.testing.assert_array_equal(synth.sample_rows(100, 256, 3, 0, 0), np.arange(100))


def test_flop_count_convention():
    w = synth.make_bf16(1, 1, 8, 4, True, 0)
    assert w.flops() == 4 * 8 * 8 * 4 / 2
    assert math.isclose(synth.make_bf16(1, 1, 8, 4, False, 0).flops(), 4 * 8 * 8 * 4)


# --------------------------------------------------------------------- MXFP4
def test_e2m1_decode_table_from_the_format():
    """Codes decode by the E2M1 definition: sign bit 3, exponent bits 2-1 (bias
    1), mantissa bit 0; exponent field 0 is subnormal (m * 0.5)."""
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
        assert synth.e2m1_decode(np.array([code]))[0] == (-mag if s else mag)


def test_e2m1_encode_rounding_and_saturation():
    vals = synth.e2m1_decode(np.arange(8))
    # every representable value encodes to itself, either sign
    np.testing.assert_array_equal(synth.e2m1_encode_satfinite(vals), np.arange(8))
    np.testing.assert_array_equal(synth.e2m1_encode_satfinite(-vals[1:]), np.arange(1, 8) | 8)
    # midpoints go to the even code; values past 6 saturate
    mids = (vals[:-1] + vals[1:]) / 2
    np.testing.assert_array_equal(synth.e2m1_encode_satfinite(mids), [0, 2, 2, 4, 4, 6, 6])
    np.testing.assert_array_equal(synth.e2m1_encode_satfinite(np.array([6.01, 1e9])), [7, 7])
    # nearest otherwise: brute force over a grid
    g = np.linspace(0, 6, 6001)
    nearest = np.abs(g[:, None] - vals[None, :]).min(axis=1)
    got = np.abs(synth.e2m1_decode(synth.e2m1_encode_satfinite(g)) - g)
    np.testing.assert_allclose(got, nearest, atol=0)


def test_mx_shared_exponent_definition():
    """E = floor(log2 amax) - 2: amax / 2^E lies in [4, 8); all-zero blocks -127."""
    a = np.exp2(np.random.default_rng(0).uniform(-60, 60, size=10000))
    e = synth.mx_shared_exponent(a)
    r = a / np.exp2(e.astype(float))
    assert (r >= 4).all() and (r < 8).all()
    assert synth.mx_shared_exponent(np.array([0.0]))[0] == -127
    assert synth.mx_shared_exponent(np.array([1.0, 4.0, 7.99]))[2] == 0


def test_mxfp4_layout_round_trip_and_error_bound():
    g = np.random.default_rng(1)
    B, H, N, d = 2, 3, 96, 8
    # representable blocks survive exactly: values e2m1 * 2^E with one element at 4 * 2^E
    e = g.integers(-10, 10, size=(B, H, d, N // 32))
    codes = g.integers(0, 16, size=(B, H, d, N))
    codes[..., ::32] = 6
    x = synth.e2m1_decode(codes) * np.repeat(np.exp2(e.astype(float)), 32, axis=3)
    v = x.transpose(0, 1, 3, 2)  # [B,H,N,d]
    packed, sc = synth.mxfp4_quantize_keys(v)
    assert packed.shape == (B, H, d, N // 2) and sc.shape == (B, H, d, N // 32)
    np.testing.assert_array_equal(synth.mxfp4_dequantize_keys(packed, sc), v)
    np.testing.assert_array_equal(sc.astype(int) - 127, e)
    # nibble order: key 2i in the low nibble of byte i
    assert (packed[0, 0, 0, 0] & 15) == (synth.e2m1_encode_satfinite(v[0, 0, 0, 0] / 2.0 ** e[0, 0, 0, 0]))
    # arbitrary data: error at most half an e2m1 step, or the saturation at 6 X
    w = g.standard_normal((B, H, N, d)) * 3
    packed, sc = synth.mxfp4_quantize_keys(w)
    back = synth.mxfp4_dequantize_keys(packed, sc)
    X = np.repeat(np.exp2(sc.astype(float) - 127), 32, axis=3).transpose(0, 1, 3, 2)
    y = np.abs(w) / X
    half_step = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
    allowed = np.where(y > 6, y - 6, half_step) * X
    assert (np.abs(back - w) <= allowed + 1e-12).all()
