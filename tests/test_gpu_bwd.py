"""GPU parity of the BF16 attention backward (attn_bwd through the C ABI) against
the fp64 gradient oracle on the same seeded bf16 inputs.

The backward takes O and LSE from the library's own forward pass (what a caller
does), so the check covers the pair.

Tolerance: tests/bwd_tolerance.py derives per-element and aggregate bounds from
the bf16 roundings the kernels make, measured against the size of the summed
terms (so that gradients that vanish exactly, as with a single visible key, are
covered); tests/test_bwd_tolerance.py shows on the CPU that planted mistakes
exceed them.
"""
import numpy as np
import pytest

from exact_tiled_attention_16_gb300 import synth
from oracle.attention_bwd import attention_bwd_head, attention_bwd_key_rows, attention_bwd_query_rows
from tests.bwd_tolerance import U, bwd_bounds, check

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_16_gb300 as pkg
    pkg.load_library()


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_bwd(w, do_bits):
    """Forward then backward on the GPU; returns (dq, dk, dv) as float64 arrays."""
    import exact_tiled_attention_16_gb300 as pkg
    q, k, v = _dev(w.q), _dev(w.k), _dev(w.v)
    do = _dev(do_bits)
    o, lse = pkg.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    dq, dk, dv = pkg.attn_bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    rc, where = pkg.check_device_errors()
    assert rc == 0, f"device error word set by wait {where}"
    return _f64(dq), _f64(dk), _f64(dv)


def check_heads(w, do_bits, got, heads=None):
    dq, dk, dv = got
    heads = heads if heads is not None else [(b, h) for b in range(w.B) for h in range(w.H)]
    for b, h in heads:
        q, k, v = w.head_f64(b, h)
        do = synth.bf16_bits_to_f64(do_bits[b, h])
        ref = attention_bwd_head(q, k, v, do, w.causal, w.scale)
        bounds = bwd_bounds(q, k, v, do, w.causal, w.scale)
        tag = f"B{w.B}H{w.H}N{w.N}d{w.d} causal={w.causal} head ({b},{h})"
        for name, g, r in zip(("dq", "dk", "dv"), (dq[b, h], dk[b, h], dv[b, h]), ref):
            check(g, r, bounds[name], f"{name} {tag}")


SMALL = [
    # (B, H, N, d): one partial tile, ragged tails, several tiles
    (1, 1, 1, 64), (1, 1, 7, 128), (1, 2, 128, 64), (2, 1, 129, 128), (1, 3, 200, 64),
    (1, 1, 257, 128), (2, 2, 384, 64), (1, 2, 1000, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=[f"B{b}H{h}N{n}d{d}" for b, h, n, d in SMALL])
def test_small_full_oracle(shape, causal):
    B, H, N, d = shape
    w = synth.make_bf16(B, H, N, d, causal, seed=300 + N + d)
    do_bits = synth.make_grad_out(B, H, N, d, seed=300 + N + d)
    check_heads(w, do_bits, run_bwd(w, do_bits))


@pytest.mark.parametrize("shape,causal", [((4, 40, 512, 128), False), ((2, 40, 640, 64), True),
                                          ((3, 60, 300, 128), True)],
                         ids=["d128_nc_4rounds", "d64_c_rounds", "d128_c_ragged_rounds"])
def test_many_units_per_cta(shape, causal):
    """More units than SMs: each CTA runs several units, so TMEM accumulators,
    rings and barrier phases are reused across units."""
    B, H, N, d = shape
    w = synth.make_bf16(B, H, N, d, causal, seed=400 + N)
    do_bits = synth.make_grad_out(B, H, N, d, seed=400 + N)
    got = run_bwd(w, do_bits)
    heads = [(b, h) for b in range(B) for h in range(H)]
    pick = np.random.default_rng(7).choice(len(heads), size=6, replace=False)
    check_heads(w, do_bits, got, heads=[heads[i] for i in pick] + [heads[-1]])


def test_zigzag_order_odd_blocks():
    """Causal with many block pairs and streamed tensors beyond the L2 budget: both
    passes take the zigzag order; an odd block count (33) leaves each head's middle
    block alone in an odd iteration, which every role must skip alike."""
    B, H, N, d = 1, 64, 4224, 64
    w = synth.make_bf16(B, H, N, d, True, seed=4224)
    do_bits = synth.make_grad_out(B, H, N, d, seed=4224)
    got = run_bwd(w, do_bits)
    check_heads(w, do_bits, got, heads=[(0, 0), (0, 31), (0, 63)])


@pytest.mark.parametrize("name", ["cfg2n", "cfg2c"])
def test_cfg2_heads(name):
    w = synth.make_config(name)
    do_bits = synth.make_grad_out(w.B, w.H, w.N, w.d, seed=w.seed)
    got = run_bwd(w, do_bits)
    check_heads(w, do_bits, got, heads=[(0, 0), (1, 7), (w.B - 1, w.H - 1)])


@pytest.mark.parametrize("name", ["cfg3", "cfg4"])
def test_large_config_sampled(name):
    """Full-size inputs: sampled dq rows and dk/dv keys of one head against the
    oracle, and the sum rules of the gradients on every head."""
    w = synth.make_config(name)
    do_bits = synth.make_grad_out(w.B, w.H, w.N, w.d, seed=w.seed)
    dq, dk, dv = run_bwd(w, do_bits)
    b, h = w.B - 1, w.H // 2
    q, k, v = w.head_f64(b, h)
    do = synth.bf16_bits_to_f64(do_bits[b, h])
    rows = synth.sample_rows(w.N, 96, seed=5, b=b, h=h)
    keys = synth.sample_rows(w.N, 48, seed=6, b=b, h=h)
    bounds = bwd_bounds(q, k, v, do, w.causal, w.scale, rows=rows, keys=keys)
    check(dq[b, h][rows], attention_bwd_query_rows(q, k, v, do, w.causal, w.scale, rows), bounds["dq"],
          f"dq {name}")
    rk, rv = attention_bwd_key_rows(q, k, v, do, w.causal, w.scale, keys)
    check(dk[b, h][keys], rk, bounds["dk"], f"dk {name}")
    check(dv[b, h][keys], rv, bounds["dv"], f"dv {name}")
    # every row of dS sums to zero, so sum_j dk_j = 0; rows of P sum to one, so
    # sum_j dv_j = sum_i do_i (per head, at any size)
    do_all = synth.bf16_bits_to_f32(do_bits).astype(np.float64)
    sum_dk = dk.sum(axis=2)
    assert np.abs(sum_dk).max() <= 8 * U * np.abs(dk).sum(axis=2).max()
    sum_dv = dv.sum(axis=2)
    ref_dv = do_all.sum(axis=2)
    assert np.abs(sum_dv - ref_dv).max() <= 8 * U * np.abs(dv).sum(axis=2).max()


def test_deterministic_bitwise():
    w = synth.make_bf16(2, 4, 1500, 128, True, seed=9)
    do_bits = synth.make_grad_out(2, 4, 1500, 128, seed=9)
    import exact_tiled_attention_16_gb300 as pkg
    q, k, v, do = _dev(w.q), _dev(w.k), _dev(w.v), _dev(do_bits)
    o, lse = pkg.attn_fwd(q, k, v, causal=True, scale=w.scale)
    g1 = pkg.attn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale)
    g2 = pkg.attn_bwd(q, k, v, o, do, lse, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_zero_upstream_gradient_gives_zero():
    import exact_tiled_attention_16_gb300 as pkg
    w = synth.make_bf16(1, 3, 333, 64, True, seed=13)
    q, k, v = _dev(w.q), _dev(w.k), _dev(w.v)
    o, lse = pkg.attn_fwd(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = pkg.attn_bwd(q, k, v, o, torch.zeros_like(q), lse, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    for g in (dq, dk, dv):
        assert (g.float() == 0).all()


def test_no_writes_outside_outputs():
    """dq, dk, dv are written in place inside guard regions that must stay intact."""
    import exact_tiled_attention_16_gb300 as pkg
    B, H, N, d = 1, 2, 333, 128
    w = synth.make_bf16(B, H, N, d, False, seed=17)
    do_bits = synth.make_grad_out(B, H, N, d, seed=17)
    q, k, v, do = _dev(w.q), _dev(w.k), _dev(w.v), _dev(do_bits)
    o, lse = pkg.attn_fwd(q, k, v, scale=w.scale)
    guard, n = 4096, B * H * N * d
    bufs = [torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    views = [b[guard:guard + n].view(B, H, N, d) for b in bufs]
    nws = pkg.bwd_workspace_bytes(B, H, N) // 4
    ws = torch.full((nws + 2 * 1024,), float("nan"), dtype=torch.float32, device="cuda")
    pkg.attn_bwd(q, k, v, o, do, lse, scale=w.scale, dq=views[0], dk=views[1], dv=views[2],
                 workspace=ws[1024:1024 + nws])
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.isnan(b[:guard].float()).all() and torch.isnan(b[-guard:].float()).all()
        assert not torch.isnan(b[guard:guard + n].float()).any()
    assert torch.isnan(ws[:1024]).all() and torch.isnan(ws[-1024:]).all()
    check_heads(w, do_bits, tuple(_f64(x) for x in views))


def test_workspace_too_small_launches_nothing():
    import exact_tiled_attention_16_gb300._lib as L
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device="cuda")
    dq = torch.full_like(q, 7.0)
    ws = torch.zeros(127, dtype=torch.float32, device="cuda")
    p = q.data_ptr()
    rc = L.attn_bwd_raw(p, p, p, p, p, lse.data_ptr(), dq.data_ptr(), dq.data_ptr(), dq.data_ptr(), 1, 1, 128, 64,
                        False, 0.125, ws.data_ptr(), 127 * 4, torch.cuda.current_stream().cuda_stream)
    assert rc == L.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (dq.float() == 7.0).all()


@pytest.mark.parametrize("pin", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("shape", [(1, 3, 700, 128, True), (2, 16, 1024, 64, False), (1, 32, 512, 128, True)],
                         ids=["B1H3N700d128c", "B2H16N1024d64n", "B1H32N512d128c_8_chunks"])
def test_host_buffers_bitwise_equal_to_device_call(shape, pin):
    """attn_bwd_host: every tensor in host memory, pipelined in chunks of whole
    heads (each chunk's scratch in its workspace slot); every chunk runs attn_bwd
    on whole heads, so the gradients are bit for bit those of attn_bwd."""
    import exact_tiled_attention_16_gb300 as pkg
    B, H, N, d, causal = shape
    w = synth.make_bf16(B, H, N, d, causal, seed=1300 + N)
    do_bits = synth.make_grad_out(B, H, N, d, seed=1300 + N)
    q, k, v, do = _dev(w.q), _dev(w.k), _dev(w.v), _dev(do_bits)
    o, lse = pkg.attn_fwd(q, k, v, causal=causal, scale=w.scale)
    g_d = pkg.attn_bwd(q, k, v, o, do, lse, causal=causal, scale=w.scale)
    torch.cuda.synchronize()

    def host(t):
        t = t.cpu()
        return t.pin_memory() if pin else t
    g_h = pkg.attn_bwd_host(*(host(t) for t in (q, k, v, o, do, lse)), causal=causal, scale=w.scale)
    torch.cuda.current_stream().synchronize()
    for a, b in zip(g_h, g_d):
        assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16))
    assert pkg.check_device_errors()[0] == 0
