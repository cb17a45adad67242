"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the tests, the benchmark and the fp64 oracle's callers.
It holds only input preparation -- random draws, bf16 rounding, outlier channels,
the random orthogonal rotation and the e4m3 block quantiser that turn a draw into
the operands a caller hands to the library -- and none of the attention
arithmetic itself (no scores, no softmax, no products with V).

Workload recipes (one per test/bench configuration) follow the shapes and value
distributions named for exact attention in the FlashAttention-2 article
("Background" and "Performance" sections) and the FlashAttention-3 notes on FP8
(block quantisation with one scale per small tile, and incoherent processing:
multiplying Q and K by a random orthogonal matrix before quantising, from the
news article "FlashAttention scaling, multi-GPU training and weight
quantisation", section 1).  The pages name no public dataset, so every input is
drawn here from a seed.

Numbers are drawn with numpy's PCG64 bit generator seeded by (seed, stream);
distinct streams give independent tensors (Q, K, V, outlier sets, rotation).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

# Streams of the PCG64 generator: one per independent draw of a workload.
STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2
STREAM_OUTLIER_QK, STREAM_OUTLIER_V = 3, 4
STREAM_ROTATION = 5
STREAM_ROWS = 6
STREAM_DO = 7

E4M3_MAX = 448.0
FP8_BLOCK = 128  # tokens per quantisation block


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def normal_f32(shape, seed: int, stream: int) -> np.ndarray:
    """I.i.d. N(0,1) draws in float32."""
    return rng(seed, stream).standard_normal(size=shape, dtype=np.float32)


# ----------------------------------------------------------------------------
# bf16 (1 sign, 8 exponent, 7 mantissa bits): the upper half of an IEEE float32.
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 with round-to-nearest-even; returns the uint16 bits.

    Inputs are finite (the generators never produce inf/NaN)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


# ----------------------------------------------------------------------------
# OCP 8-bit floating point, E4M3 ("FN" variant): 1 sign bit, 4 exponent bits with
# bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN, so the largest finite
# magnitude is 1.75 * 2^8 = 448.  Exponent field 0 encodes subnormals m/8 * 2^-6.
# ----------------------------------------------------------------------------

def _e4m3_positive_table() -> np.ndarray:
    """Magnitudes of codes 0x00..0x7E (all non-negative finite values), ascending."""
    vals = np.empty(127, dtype=np.float64)
    for code in range(127):
        e = code >> 3
        m = code & 7
        if e == 0:
            vals[code] = (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3_POS = _e4m3_positive_table()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """e4m3 byte codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8)
    mag_code = (c & np.uint8(0x7F)).astype(np.int64)
    out = np.where(mag_code == 0x7F, np.nan, _E4M3_POS[np.minimum(mag_code, 126)])
    return np.where((c & np.uint8(0x80)) != 0, -out, out)


def e4m3_encode_satfinite(x: np.ndarray) -> np.ndarray:
    """float -> e4m3 code, round-to-nearest-even, saturating to +-448.

    Ties between two neighbouring codes go to the one with an even mantissa,
    i.e. the even code.  As in IEEE arithmetic, a negative input that rounds to
    zero gives -0 (0x80).  Inputs must be finite."""
    xf = np.asarray(x, dtype=np.float64)
    a = np.abs(xf)
    a = np.minimum(a, E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, a, side="left")  # first code with value >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(_E4M3_POS[hi] == a, hi, code)
    sign = np.signbit(xf).astype(np.uint8) << np.uint8(7)  # negative values keep their sign, even at zero
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def block_quantize_e4m3(x: np.ndarray, block: int = FP8_BLOCK):
    """Per-(b, h, token-block) scaling of x [B,H,N,d] to e4m3.

    For every (b, h, block of `block` consecutive tokens) over all d channels:
    s = amax / 448 as float32 (s = 1 where the block is all zeros), and the
    codes are e4m3_RNE_satfinite(x / s).  Returns (codes uint8 [B,H,N,d],
    scales float32 [B,H,ceil(N/block)])."""
    B, H, N, d = x.shape
    T = (N + block - 1) // block
    codes = np.empty((B, H, N, d), dtype=np.uint8)
    scales = np.empty((B, H, T), dtype=np.float32)
    for t in range(T):
        sl = slice(t * block, min(N, (t + 1) * block))
        xb = x[:, :, sl, :].astype(np.float64)
        amax = np.abs(xb).max(axis=(2, 3))
        s = (amax / E4M3_MAX).astype(np.float32)
        s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
        scales[:, :, t] = s
        codes[:, :, sl, :] = e4m3_encode_satfinite(xb / s.astype(np.float64)[:, :, None, None])
    return codes, scales


def block_dequantize_e4m3(codes: np.ndarray, scales: np.ndarray, block: int = FP8_BLOCK) -> np.ndarray:
    """codes [B,H,N,d], scales [B,H,T] -> float64 x8 * s (exact in fp64)."""
    N = codes.shape[2]
    tok_scale = np.repeat(scales.astype(np.float64), block, axis=2)[:, :, :N]
    return e4m3_decode(codes) * tok_scale[..., None]


# ----------------------------------------------------------------------------
# OCP FP4 E2M1 with MX block scaling (MXFP4): element codes are 1 sign bit,
# 2 exponent bits (bias 1) and 1 mantissa bit, magnitudes {0, 0.5, 1, 1.5, 2,
# 3, 4, 6} for codes 0..7 (exponent field 0: subnormal m * 0.5); no infinities
# or NaNs.  A block of 32 elements shares one E8M0 scale (an unsigned biased
# exponent, value 2^(byte - 127), byte 255 reserved for NaN); the shared
# exponent is floor(log2(amax)) - 2, 2 being the largest element exponent.
# Two codes share a byte, the even-indexed element in the low nibble.
# ----------------------------------------------------------------------------
E2M1_MAX = 6.0
MX_BLOCK = 32
_E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """4-bit codes (0..15, one per array element) -> float64 values."""
    c = np.asarray(codes).astype(np.int64)
    mag = _E2M1_POS[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e2m1_encode_satfinite(x: np.ndarray) -> np.ndarray:
    """float -> 4-bit e2m1 code (uint8 0..15), round to nearest, ties to the
    even code, saturating to +-6; negative inputs keep the sign bit."""
    xf = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(xf), E2M1_MAX)
    hi = np.minimum(np.searchsorted(_E2M1_POS, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    dlo = a - _E2M1_POS[lo]
    dhi = _E2M1_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(_E2M1_POS[hi] == a, hi, code)
    return (code.astype(np.uint8) | (np.signbit(xf).astype(np.uint8) << np.uint8(3))).astype(np.uint8)


def mx_shared_exponent(amax: np.ndarray) -> np.ndarray:
    """E8M0 shared exponent of MXFP4 blocks: floor(log2(amax)) - 2, clamped to
    [-127, 127]; -127 for an all-zero block."""
    a = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(np.where(a > 0, a, 1.0))  # a = f * 2^e, f in [0.5, 1)
    ex = (e - 1) - 2
    return np.where(a > 0, np.clip(ex, -127, 127), -127).astype(np.int64)


def mxfp4_quantize_keys(v: np.ndarray):
    """MXFP4 quantisation of V [B,H,N,d] along the key axis, stored transposed.

    For every (b, h, channel c, block of 32 consecutive keys): X = 2^E with E =
    mx_shared_exponent(amax of the block), codes = e2m1_RNE_satfinite(v / X).
    Returns (packed codes uint8 [B,H,d,N/2] -- key 2i in the low nibble of byte
    i --, scale bytes uint8 [B,H,d,N/32] = E + 127).  N must be a multiple of 32."""
    B, H, N, d = v.shape
    assert N % MX_BLOCK == 0
    vt = np.asarray(v, dtype=np.float64).transpose(0, 1, 3, 2)  # [B,H,d,N]
    blocks = vt.reshape(B, H, d, N // MX_BLOCK, MX_BLOCK)
    e = mx_shared_exponent(np.abs(blocks).max(axis=4))
    codes = e2m1_encode_satfinite(blocks / np.ldexp(1.0, e)[..., None]).reshape(B, H, d, N)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << np.uint8(4))).astype(np.uint8)
    return np.ascontiguousarray(packed), (e + 127).astype(np.uint8)


def mxfp4_dequantize_keys(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """(packed [B,H,d,N/2], scale bytes [B,H,d,N/32]) -> V [B,H,N,d] float64."""
    B, H, d, half = packed.shape
    N = 2 * half
    codes = np.empty((B, H, d, N), dtype=np.uint8)
    codes[..., 0::2] = packed & np.uint8(15)
    codes[..., 1::2] = packed >> np.uint8(4)
    x = np.ldexp(1.0, scales.astype(np.int64) - 127)
    vals = e2m1_decode(codes).reshape(B, H, d, N // MX_BLOCK, MX_BLOCK) * x[..., None]
    return vals.reshape(B, H, d, N).transpose(0, 1, 3, 2)


# ----------------------------------------------------------------------------
# Outlier channels and the random orthogonal rotation
# ----------------------------------------------------------------------------

def outlier_channels(d: int, frac: float, seed: int, stream: int) -> np.ndarray:
    """ceil(frac * d) distinct channel indices, drawn without replacement, sorted."""
    count = int(math.ceil(frac * d - 1e-9))
    return np.sort(rng(seed, stream).choice(d, size=count, replace=False))


def haar_orthogonal(d: int, seed: int, stream: int = STREAM_ROTATION) -> np.ndarray:
    """Haar-distributed d x d orthogonal matrix (float64).

    QR of a standard Gaussian matrix, with the columns of Q multiplied by the
    signs of diag(R) so that the factorisation is unique (Mezzadri, "How to
    generate random matrices from the classical compact groups", 2007)."""
    g = rng(seed, stream).standard_normal(size=(d, d))
    qm, rm = np.linalg.qr(g)
    signs = np.sign(np.diag(rm))
    signs[signs == 0] = 1.0
    return qm * signs[None, :]


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    """One seeded attention problem in the layout the library takes.

    BF16: q, k, v are uint16 bf16 bits [B,H,N,d].
    FP8:  q, k, v are uint8 e4m3 codes [B,H,N,d] with float32 scales
          q_scale/k_scale/v_scale [B,H,ceil(N/128)].
    """
    name: str
    dtype: str  # "bf16" or "e4m3"
    B: int
    H: int
    N: int
    d: int
    causal: bool
    scale: float
    seed: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    q_scale: np.ndarray | None = None
    k_scale: np.ndarray | None = None
    v_scale: np.ndarray | None = None
    meta: dict = field(default_factory=dict)

    def flops(self) -> float:
        """Counted work: 4*B*H*Nq*N*d (Nq query rows against N keys; Nq = N unless
        the queries were cut to fewer rows), halved under the square causal mask."""
        nq = self.q.shape[2]
        f = 4.0 * self.B * self.H * nq * self.N * self.d
        return f / 2.0 if self.causal else f

    def head_f64(self, b: int, h: int):
        """(q, k, v) of one head as the exact float64 values the kernel sees."""
        if self.dtype == "bf16":
            return (bf16_bits_to_f64(self.q[b, h]), bf16_bits_to_f64(self.k[b, h]),
                    bf16_bits_to_f64(self.v[b, h]))
        if self.dtype == "e4m3_e2m1":
            return (block_dequantize_e4m3(self.q[b:b + 1, h:h + 1], self.q_scale[b:b + 1, h:h + 1])[0, 0],
                    block_dequantize_e4m3(self.k[b:b + 1, h:h + 1], self.k_scale[b:b + 1, h:h + 1])[0, 0],
                    mxfp4_dequantize_keys(self.v[b:b + 1, h:h + 1], self.v_scale[b:b + 1, h:h + 1])[0, 0])
        return (block_dequantize_e4m3(self.q[b:b + 1, h:h + 1], self.q_scale[b:b + 1, h:h + 1])[0, 0],
                block_dequantize_e4m3(self.k[b:b + 1, h:h + 1], self.k_scale[b:b + 1, h:h + 1])[0, 0],
                block_dequantize_e4m3(self.v[b:b + 1, h:h + 1], self.v_scale[b:b + 1, h:h + 1])[0, 0])


def make_bf16(B, H, N, d, causal, seed, scale=None, qk_outlier_frac=0.0, qk_outlier_mult=1.0,
              name="bf16") -> Workload:
    """Q, K, V i.i.d. N(0,1) (float32 draw, bf16 RNE).  Optionally a seeded set of
    ceil(frac*d) channels, shared by Q and K and by every (b, h), is multiplied by
    qk_outlier_mult before rounding, so that outlier products meet in Q K^T."""
    shape = (B, H, N, d)
    q = normal_f32(shape, seed, STREAM_Q)
    k = normal_f32(shape, seed, STREAM_K)
    v = normal_f32(shape, seed, STREAM_V)
    meta = {}
    if qk_outlier_frac > 0:
        ch = outlier_channels(d, qk_outlier_frac, seed, STREAM_OUTLIER_QK)
        q[..., ch] *= np.float32(qk_outlier_mult)
        k[..., ch] *= np.float32(qk_outlier_mult)
        meta["qk_outlier_channels"] = ch.tolist()
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return Workload(name, "bf16", B, H, N, d, bool(causal), float(scale), seed,
                    f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v), meta=meta)


def make_grad_out(B, H, N, d, seed) -> np.ndarray:
    """Upstream gradient dO [B,H,N,d] for the backward pass: i.i.d. N(0,1)
    (float32 draw, bf16 RNE bits), on its own stream of the workload's seed."""
    return f32_to_bf16_bits(normal_f32((B, H, N, d), seed, STREAM_DO))


def make_fp8(B, H, N, d, causal, seed, scale=None, outlier_frac=0.01, outlier_mult=10.0,
             rotate=True, name="e4m3") -> Workload:
    """Block-scaled e4m3 workload.

    Q, K, V ~ N(0,1) (float64 draw from float32 normals) with ceil(frac*d) outlier
    channels multiplied by outlier_mult (one set shared by Q and K, another for V);
    Q and K are multiplied on the right by one seeded Haar-orthogonal d x d matrix
    (V is not rotated); then each of Q', K', V is quantised per 128-token block."""
    shape = (B, H, N, d)
    q = normal_f32(shape, seed, STREAM_Q).astype(np.float64)
    k = normal_f32(shape, seed, STREAM_K).astype(np.float64)
    v = normal_f32(shape, seed, STREAM_V).astype(np.float64)
    meta = {}
    if outlier_frac > 0:
        ch_qk = outlier_channels(d, outlier_frac, seed, STREAM_OUTLIER_QK)
        ch_v = outlier_channels(d, outlier_frac, seed, STREAM_OUTLIER_V)
        q[..., ch_qk] *= outlier_mult
        k[..., ch_qk] *= outlier_mult
        v[..., ch_v] *= outlier_mult
        meta["qk_outlier_channels"] = ch_qk.tolist()
        meta["v_outlier_channels"] = ch_v.tolist()
    if rotate:
        r = haar_orthogonal(d, seed)
        q = q @ r
        k = k @ r
    q8, qs = block_quantize_e4m3(q)
    k8, ks = block_quantize_e4m3(k)
    v8, vs = block_quantize_e4m3(v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return Workload(name, "e4m3", B, H, N, d, bool(causal), float(scale), seed, q8, k8, v8,
                    qs, ks, vs, meta=meta)


def make_fp4p(B, H, N, d, causal, seed, scale=None, outlier_frac=0.01, outlier_mult=10.0,
              rotate=True, name="e4m3_e2m1") -> Workload:
    """Workload of the Direct-P FP4 path: Q and K exactly as make_fp8 draws and
    quantises them (e4m3, per-128-token scales); V from the same draw (with its
    outlier channels) quantised to MXFP4 along the keys and stored transposed:
    w.v = packed codes [B,H,d,N/2], w.v_scale = E8M0 bytes [B,H,d,N/32]."""
    w8 = make_fp8(B, H, N, d, causal, seed, scale, outlier_frac, outlier_mult, rotate, name)
    v = normal_f32((B, H, N, d), seed, STREAM_V).astype(np.float64)
    if outlier_frac > 0:
        v[..., outlier_channels(d, outlier_frac, seed, STREAM_OUTLIER_V)] *= outlier_mult
    vt, vts = mxfp4_quantize_keys(v)
    w8.dtype = "e4m3_e2m1"
    w8.v, w8.v_scale = vt, vts
    return w8


# The five workload shapes (seeded; the FlashAttention pages quote no dataset).
CONFIGS = {
    "cfg1": dict(kind="bf16", B=1, H=2, N=128, d=64, causal=False, seed=1),
    "cfg2n": dict(kind="bf16", B=4, H=16, N=2048, d=128, causal=False, seed=2),
    "cfg2c": dict(kind="bf16", B=4, H=16, N=2048, d=128, causal=True, seed=2),
    "cfg3": dict(kind="bf16", B=1, H=32, N=16384, d=128, causal=True, seed=3),
    "cfg4": dict(kind="bf16", B=16, H=16, N=4096, d=64, causal=False, seed=4,
                 qk_outlier_frac=0.02, qk_outlier_mult=20.0),
    "cfg5": dict(kind="e4m3", B=2, H=16, N=8192, d=128, causal=False, seed=5,
                 outlier_frac=0.01, outlier_mult=10.0),
    # the Direct-P FP4 path on cfg5's shape and draw: Q, K e4m3, V MXFP4
    "cfg5p": dict(kind="e4m3_e2m1", B=2, H=16, N=8192, d=128, causal=False, seed=5,
                  outlier_frac=0.01, outlier_mult=10.0),
}


def make_config(name: str) -> Workload:
    c = dict(CONFIGS[name])
    kind = c.pop("kind")
    if kind == "bf16":
        return make_bf16(name=name, **c)
    if kind == "e4m3_e2m1":
        return make_fp4p(name=name, **c)
    return make_fp8(name=name, **c)


def sample_rows(N: int, count: int, seed: int, b: int, h: int) -> np.ndarray:
    """Query rows checked for one head of a large workload: {0, 1, 127, 128, N-1}
    (those < N) plus rows drawn uniformly without replacement, sorted."""
    fixed = sorted({r for r in (0, 1, 127, 128, N - 1) if 0 <= r < N})
    if count >= N:
        return np.arange(N)
    g = np.random.Generator(np.random.PCG64([int(seed), STREAM_ROWS, int(b), int(h)]))
    pool = np.setdiff1d(np.arange(N), np.array(fixed))
    extra = g.choice(pool, size=max(0, count - len(fixed)), replace=False)
    return np.sort(np.concatenate([np.array(fixed, dtype=np.int64), extra.astype(np.int64)]))
