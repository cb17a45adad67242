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
