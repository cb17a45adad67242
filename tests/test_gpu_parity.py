"""GPU parity of the BF16 attention forward (through the C ABI) against the fp64
oracle on the same seeded inputs.

Tolerances (bf16 inputs, fp32 accumulation, bf16 P and O):
max|dO| <= 2e-2, mean|dO| <= 2e-3, max|dLSE| <= 1e-3.
"""
import math

import numpy as np
import pytest

from exact_tiled_attention_16_gb300 import synth
from tests.gpu_utils import assert_bf16_tol, compare_rows, run_bf16, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_16_gb300 as pkg
    pkg.load_library()


SMALL = [
    # (B, H, N, d): single tile, ragged tails, several tiles
    (1, 1, 1, 64), (1, 1, 7, 128), (1, 2, 128, 64), (2, 1, 129, 128), (1, 3, 200, 64),
    (1, 1, 257, 128), (2, 2, 384, 64), (1, 2, 1000, 128), (3, 5, 640, 64),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SMALL, ids=[f"B{b}H{h}N{n}d{d}" for b, h, n, d in SMALL])
def test_small_full_oracle(shape, causal):
    B, H, N, d = shape
    w = synth.make_bf16(B, H, N, d, causal, seed=100 + N + d)
    o, lse = run_bf16(w)
    assert_bf16_tol(compare_rows(w, o, lse), f"{shape} causal={causal}")


def test_cfg1_full():
    w = synth.make_config("cfg1")
    o, lse = run_bf16(w)
    assert_bf16_tol(compare_rows(w, o, lse), "cfg1")


@pytest.mark.parametrize("name", ["cfg2n", "cfg2c"])
def test_cfg2_full(name):
    w = synth.make_config(name)
    o, lse = run_bf16(w)
    assert_bf16_tol(compare_rows(w, o, lse), name)


@pytest.mark.parametrize("name", ["cfg3", "cfg4"])
def test_large_config_sampled_rows(name):
    w = synth.make_config(name)
    o, lse = run_bf16(w)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert_bf16_tol(compare_rows(w, o, lse, rows_per_head=256), name)


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_sampled(causal):
    """A single long head: many K/V blocks and, causal, the heaviest tiles."""
    w = synth.make_bf16(1, 1, 65536 + 77, 128, causal, seed=21)
    o, lse = run_bf16(w)
    assert_bf16_tol(compare_rows(w, o, lse, rows_per_head=256), "N=65613")


def test_deterministic_bitwise():
    w = synth.make_bf16(2, 4, 1500, 128, True, seed=9)
    q, k, v = to_device(w)
    import exact_tiled_attention_16_gb300 as pkg
    o1, l1 = pkg.attn_fwd(q, k, v, causal=True, scale=w.scale)
    o2, l2 = pkg.attn_fwd(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_causal_last_row_equals_noncausal():
    """The last causal row sees every key: bit for bit the non-causal row, both
    computed in one pass over the keys (the non-causal launch's split of its last
    round over CTA pairs, which merges two halves, is turned off here)."""
    import exact_tiled_attention_16_gb300 as pkg
    wc = synth.make_bf16(1, 4, 1024, 128, True, seed=31)
    wn = synth.make_bf16(1, 4, 1024, 128, False, seed=31)
    oc, lc = run_bf16(wc)
    pkg.diag_set_pair_tail(False)
    try:
        on, ln_ = run_bf16(wn)
    finally:
        pkg.diag_set_pair_tail(True)
    np.testing.assert_array_equal(oc[:, :, -1], on[:, :, -1])
    np.testing.assert_array_equal(lc[:, :, -1], ln_[:, :, -1])
    # causal row 0 is v0 (rounded to bf16 twice at most)
    v0 = synth.bf16_bits_to_f64(wc.v[:, :, 0])
    np.testing.assert_allclose(oc[:, :, 0], v0, atol=1e-2, rtol=1e-2)


def test_invariants_on_gpu():
    import exact_tiled_attention_16_gb300 as pkg
    B, H, N, d = 1, 2, 700, 64
    w = synth.make_bf16(B, H, N, d, False, seed=41)
    q, k, v = to_device(w)
    # constant V -> constant O
    vc = torch.full_like(v, 1.5)
    for causal in (False, True):
        o, _ = pkg.attn_fwd(q, k, vc, causal=causal)
        torch.cuda.synchronize()
        assert (o.float() - 1.5).abs().max().item() <= 1.5 * 1e-2
    # Q = 0 -> mean of the visible V rows, lse = ln(#visible)
    qz = torch.zeros_like(q)
    for causal in (False, True):
        o, lse = pkg.attn_fwd(qz, k, v, causal=causal, scale=0.3)
        torch.cuda.synchronize()
        vf = v.double()
        if causal:
            ref = vf.cumsum(dim=2) / torch.arange(1, N + 1, device=vf.device, dtype=vf.dtype)[None, None, :, None]
            nvis = torch.arange(1, N + 1, device=vf.device, dtype=torch.float64)
        else:
            ref = vf.mean(dim=2, keepdim=True).expand_as(vf)
            nvis = torch.full((N,), float(N), device=vf.device, dtype=torch.float64)
        assert (o.double() - ref).abs().max().item() <= 2e-2
        assert (lse.double() - nvis.log()[None, None]).abs().max().item() <= 1e-3


def test_lse_optional():
    w = synth.make_bf16(1, 2, 300, 128, True, seed=51)
    o1, l1 = run_bf16(w)
    o2, l2 = run_bf16(w, want_lse=False)
    assert l2 is None
    np.testing.assert_array_equal(o1, o2)


@pytest.mark.parametrize("causal", [True, False], ids=["causal_row_stores", "noncausal_tma_store"])
@pytest.mark.parametrize("d", [64, 128])
def test_no_writes_outside_outputs(causal, d):
    """O and LSE are written in place inside guard regions that must stay intact
    (non-causal launches store O with TMA, whose boxes are clipped at the ragged
    tail N = 333 and at every head boundary; causal ones store rows directly, 32
    bytes at a time when O is 32-byte aligned, else 16).  O is placed 32-byte
    aligned and then 16 bytes off: the two results are the same bits."""
    import exact_tiled_attention_16_gb300._lib as L
    B, H, N = 1, 3, 333
    w = synth.make_bf16(B, H, N, d, causal, seed=61)
    q, k, v = to_device(w)
    results = []
    for shift in (0, 8):  # elements: 0 and 16 bytes past a 32-byte boundary
        guard = 4096
        o_buf = torch.full((B * H * N * d + 2 * guard + shift,), float("nan"), dtype=torch.bfloat16, device="cuda")
        l_buf = torch.full((B * H * N + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
        assert o_buf.data_ptr() % 256 == 0
        o_view = o_buf[guard + shift:guard + shift + B * H * N * d]
        l_view = l_buf[guard:guard + B * H * N]
        assert (o_view.data_ptr() % 32 == 0) == (shift == 0)
        rc = L.attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_view.data_ptr(), l_view.data_ptr(),
                            B, H, N, d, causal, w.scale, torch.cuda.current_stream().cuda_stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.isnan(o_buf[:guard + shift].float()).all() and torch.isnan(o_buf[-guard:].float()).all()
        assert torch.isnan(l_buf[:guard]).all() and torch.isnan(l_buf[-guard:]).all()
        assert not torch.isnan(o_view.float()).any() and not torch.isnan(l_view).any()
        assert_bf16_tol(compare_rows(w, o_view.view(B, H, N, d).float().cpu().numpy().astype(np.float64),
                                     l_view.view(B, H, N).cpu().numpy().astype(np.float64)), f"guarded, shift {shift}")
        results.append(o_view.clone())
    assert torch.equal(results[0].view(torch.int16), results[1].view(torch.int16))


def test_invalid_arguments_launch_nothing():
    import exact_tiled_attention_16_gb300._lib as L
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 7.0)
    s = torch.cuda.current_stream().cuda_stream
    assert L.attn_fwd_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 0, 1, 1, 128, 96, 0, 0.1, s) == -3
    assert L.attn_fwd_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 0, 1, 1, 128, 64, 0, -1.0, s) == -10
    torch.cuda.synchronize()
    assert (o.float() == 7.0).all()


def test_bounded_wait_selftest():
    """A wait that nobody satisfies gives up with ATTN_ERR_TIMEOUT; the context stays usable."""
    import exact_tiled_attention_16_gb300 as pkg
    assert pkg.set_wait_timeout_ns(2_000_000) == 0  # 2 ms
    try:
        assert pkg.selftest_wait_timeout() == -8
    finally:
        assert pkg.set_wait_timeout_ns(4_000_000_000) == 0
    assert pkg.check_device_errors()[0] == 0
    w = synth.make_bf16(1, 1, 256, 64, False, seed=71)
    o, lse = run_bf16(w)
    assert_bf16_tol(compare_rows(w, o, lse), "after selftest")


def test_torch_streams():
    """The call is asynchronous on the given stream."""
    import exact_tiled_attention_16_gb300 as pkg
    w = synth.make_bf16(1, 2, 512, 128, False, seed=81)
    q, k, v = to_device(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = pkg.attn_fwd(q, k, v, scale=1 / math.sqrt(128))
    s.synchronize()
    assert_bf16_tol(compare_rows(w, o.float().cpu().numpy().astype(np.float64),
                                 lse.cpu().numpy().astype(np.float64)), "side stream")


ORDER_CASES = [(0, 0), (1, 0), (2, 1), (2, 3), (2, 0)]


@pytest.mark.parametrize("order", ORDER_CASES, ids=["heads", "zigzag", "groups1", "groups3", "groups_all"])
@pytest.mark.parametrize("shape", [(2, 76, 640, 128), (3, 50, 1024, 64), (1, 7, 2304, 128), (2, 40, 777, 64),
                                   (8, 76, 512, 128)],
                         ids=["pairs3_odd", "pairs4_d64", "few_heads_9pairs", "ragged_tail_d64", "pairs2_many_rounds"])
def test_every_unit_order_covers_every_unit(shape, order):
    """Each unit order of causal launches forced in turn (head-major, zigzag with
    heavy+light pairs combined, head groups of one, of three -- a smaller last
    group when the head count is not a multiple -- and of all heads): every row
    must be written and correct, including odd pair counts (the middle pair of a
    zigzag head alone), ragged last pairs and heads whose pairs land on different
    CTAs in different rounds."""
    import exact_tiled_attention_16_gb300 as pkg
    B, H, N, d = shape
    w = synth.make_bf16(B, H, N, d, True, seed=91 + N)
    q, k, v = to_device(w)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    pkg.diag_force_fwd_order(*order)
    try:
        info, _ = pkg.diag_fwd_schedule(B * H, N, N, True, d=d, num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
        assert info["order"] == order[0]
        pkg.attn_fwd(q, k, v, causal=True, scale=w.scale, o=o, lse=lse)
        torch.cuda.synchronize()
    finally:
        pkg.diag_force_fwd_order(-1)
    assert not torch.isnan(o.float()).any() and not torch.isnan(lse).any()
    assert_bf16_tol(compare_rows(w, o.float().cpu().numpy().astype(np.float64),
                                 lse.cpu().numpy().astype(np.float64)), f"order {order} {shape}")


@pytest.mark.parametrize("causal", [False, True])
def test_instances_past_the_unit_table(causal):
    """2560 heads of 1024 rows (10240 units, 68 rounds of 152 CTAs): more rounds
    than the unit table holds (48 beside the non-causal O staging buffers, 64
    otherwise), so the launch runs the table-less instance that computes every
    unit on each role (head-major or zigzag order); sampled rows of every head."""
    import exact_tiled_attention_16_gb300 as pkg
    B, H, N, d = 64, 40, 1024, 64
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    info, _ = pkg.diag_fwd_schedule(B * H, N, N, causal, d=d, num_sms=sms)
    if info["rounds"] <= 64:
        pytest.skip(f"{sms} SMs: every CTA's rounds fit in the table")
    assert info["table"] == 0
    w = synth.make_bf16(B, H, N, d, causal, seed=5150 + causal)
    o, lse = run_bf16(w)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert_bf16_tol(compare_rows(w, o, lse, rows_per_head=8), f"untabled causal={causal}")


@pytest.mark.parametrize("shape", [(1, 2, 4096, 128), (1, 3, 3100, 128), (1, 3, 6200, 64), (1, 2, 8192, 64),
                                   (1, 32, 4096, 128)],
                         ids=["all_split_d128", "ragged_odd_blocks_d128", "ragged_odd_blocks_d64", "all_split_d64",
                              "B1H32N4096_tail_of_56"])
def test_pair_tail_split_last_round(shape):
    """Non-causal launches whose last round is split over CTA pairs (clusters of
    two: the odd CTA sends its half's unnormalised O, max and sum through
    distributed shared memory, the even CTA merges): rows against the oracle
    (every row of the small cases, the split units' heads sampled in the large
    one), and the result against the same launch with the split turned off."""
    import exact_tiled_attention_16_gb300 as pkg
    B, H, N, d = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    info, _ = pkg.diag_fwd_schedule(B * H, N, N, False, d=d, num_sms=sms)
    if not info["pair_tail"]:
        pytest.skip(f"{sms} SMs: this shape's last round is not split")
    w = synth.make_bf16(B, H, N, d, False, seed=8800 + N + H)
    o, lse = run_bf16(w)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = None if B * H * N <= 20000 else 128
    assert_bf16_tol(compare_rows(w, o, lse, rows_per_head=rows), f"pair tail {shape}")
    pkg.diag_set_pair_tail(False)
    try:
        o2, lse2 = run_bf16(w)
    finally:
        pkg.diag_set_pair_tail(True)
    assert np.abs(o - o2).max() <= 2e-2 and np.abs(lse - lse2).max() <= 1e-3


@pytest.mark.parametrize("d,N", [(128, 3100), (64, 6200)])
def test_pair_tail_writes_nothing_outside_outputs(d, N):
    """The merging CTA of a split unit stores its rows directly: O and LSE inside
    guard regions that must stay intact (ragged N, every unit split)."""
    import exact_tiled_attention_16_gb300 as pkg
    import exact_tiled_attention_16_gb300._lib as L
    B, H = 1, 2
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if not pkg.diag_fwd_schedule(B * H, N, N, False, d=d, num_sms=sms)[0]["pair_tail"]:
        pytest.skip("no pair tail on this device")
    w = synth.make_bf16(B, H, N, d, False, seed=62)
    q, k, v = to_device(w)
    guard = 4096
    o_buf = torch.full((B * H * N * d + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * N + 2 * guard,), float("nan"), dtype=torch.float32, device="cuda")
    o_view = o_buf[guard:guard + B * H * N * d]
    l_view = l_buf[guard:guard + B * H * N]
    rc = L.attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_view.data_ptr(), l_view.data_ptr(),
                        B, H, N, d, False, w.scale, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.isnan(o_buf[:guard].float()).all() and torch.isnan(o_buf[-guard:].float()).all()
    assert torch.isnan(l_buf[:guard]).all() and torch.isnan(l_buf[-guard:]).all()
    assert not torch.isnan(o_view.float()).any() and not torch.isnan(l_view).any()
    assert_bf16_tol(compare_rows(w, o_view.view(B, H, N, d).float().cpu().numpy().astype(np.float64),
                                 l_view.view(B, H, N).cpu().numpy().astype(np.float64)), "guarded pair tail")


def _sweep_shapes():
    g = np.random.default_rng(2024)
    shapes = []
    for i in range(16):
        d = (64, 128)[i % 2]
        causal = bool((i // 2) % 2)
        N = int(g.integers(1, 1600))
        B = int(g.integers(1, 4))
        H = int(g.integers(1, 7))
        shapes.append((B, H, N, d, causal))
    return shapes


@pytest.mark.parametrize("shape", _sweep_shapes(), ids=lambda s: f"B{s[0]}H{s[1]}N{s[2]}d{s[3]}{'c' if s[4] else 'n'}")
def test_random_shape_sweep(shape):
    """Seeded random shapes (ragged N, several heads, both masks and head dims):
    every output row against the oracle, so the TMA-stored (non-causal) and
    row-stored (causal) epilogues, the ragged-tail masks and the unit orders meet
    shapes no hand-picked case covers."""
    B, H, N, d, causal = shape
    w = synth.make_bf16(B, H, N, d, causal, seed=7000 + N)
    o, lse = run_bf16(w)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert_bf16_tol(compare_rows(w, o, lse), f"sweep {shape}")
