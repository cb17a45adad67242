"""GPU parity of the partial-attention, merge and split-K/V entry points against
the fp64 oracle: partial results over one key shard (with absolute query/key
positions for the causal mask), exact LSE-weighted merges, a ring of K/V shards
merged online on one GPU, and split-K/V attention including decode-shaped
(Nq < Nk) inputs.  Tolerances as the BF16 path (partials are fp32 but built from
bf16 P)."""
import math

import numpy as np
import pytest

from exact_tiled_attention_16_gb300 import synth
from oracle.attention import attention_head
from tests.gpu_utils import BF16_MAX_ABS_LSE, BF16_MAX_ABS_O, BF16_MEAN_ABS_O

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


def _check(o_gpu, lse_gpu, o_ref, lse_ref, what):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), empty), f"{what}: empty rows differ"
    assert np.all(o_gpu[empty] == 0.0), f"{what}: empty rows must have O = 0"
    d = np.abs(o_gpu[~empty] - o_ref[~empty]) if (~empty).any() else np.zeros(1)
    dl = np.abs(lse_gpu[~empty] - lse_ref[~empty]) if (~empty).any() else np.zeros(1)
    assert d.max() <= BF16_MAX_ABS_O and d.mean() <= BF16_MEAN_ABS_O, f"{what}: max {d.max():.3g} mean {d.mean():.3g}"
    assert dl.max() <= BF16_MAX_ABS_LSE, f"{what}: lse {dl.max():.3g}"


def _oracle_rows(w, b, h, rows, key_lo, key_hi, causal):
    q, k, v = w.head_f64(b, h)
    return attention_head(q, k, v, causal, w.scale, rows=rows, key_lo=key_lo, key_hi=key_hi)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_partial_shard_matches_oracle_key_range(causal, d):
    import exact_tiled_attention_16_gb300 as pkg
    N = 700
    w = synth.make_bf16(1, 3, N, d, causal, seed=300 + d)
    for (a, b) in [(0, 700), (0, 128), (128, 333), (333, 700), (650, 700)]:
        q = _dev(w.q)
        k = _dev(w.k[:, :, a:b])
        v = _dev(w.v[:, :, a:b])
        o, lse = pkg.attn_fwd_partial(q, k, v, causal=causal, q_offset=0, k_offset=a, scale=w.scale)
        torch.cuda.synchronize()
        for h in range(3):
            ro, rl = _oracle_rows(w, 0, h, np.arange(N), a, b, causal)
            _check(o[0, h].cpu().numpy(), lse[0, h].cpu().numpy(), ro, rl, f"shard {a}:{b} h{h}")


def test_partial_query_shard_with_offsets():
    """Queries of positions c..e against keys of positions a..b (one device's
    share of a sequence-parallel layout)."""
    import exact_tiled_attention_16_gb300 as pkg
    N = 1000
    w = synth.make_bf16(2, 2, N, 128, True, seed=17)
    for (c, e, a, b) in [(500, 1000, 0, 500), (500, 1000, 500, 1000), (0, 300, 200, 900), (256, 512, 384, 640)]:
        q = _dev(w.q[:, :, c:e])
        k = _dev(w.k[:, :, a:b])
        v = _dev(w.v[:, :, a:b])
        o, lse = pkg.attn_fwd_partial(q, k, v, causal=True, q_offset=c, k_offset=a, scale=w.scale)
        torch.cuda.synchronize()
        for bb in range(2):
            for h in range(2):
                ro, rl = _oracle_rows(w, bb, h, np.arange(c, e), a, b, True)
                _check(o[bb, h].cpu().numpy(), lse[bb, h].cpu().numpy(), ro, rl, f"q{c}:{e} k{a}:{b}")


@pytest.mark.parametrize("causal", [False, True])
def test_ring_of_shards_merged_online(causal):
    """R K/V shards visited one after another, each partial merged into a running
    fp32 (O, lse) in place; equals unsharded attention."""
    import exact_tiled_attention_16_gb300 as pkg
    N, R = 1536, 4
    w = synth.make_bf16(1, 4, N, 128, causal, seed=23)
    q = _dev(w.q)
    cuts = [0, 300, 768, 1100, 1536]
    acc_o = acc_l = None
    for r in range(R):
        a, b = cuts[r], cuts[r + 1]
        o_s, l_s = pkg.attn_fwd_partial(q, _dev(w.k[:, :, a:b]), _dev(w.v[:, :, a:b]), causal=causal,
                                        k_offset=a, scale=w.scale)
        if acc_o is None:
            acc_o, acc_l = o_s, l_s
        else:
            pkg.attn_merge([(acc_o, acc_l), (o_s, l_s)], out=acc_o, lse=acc_l, out_fp32=True)
    o_bf16, lse = pkg.attn_merge([(acc_o, acc_l)])
    torch.cuda.synchronize()
    for h in range(4):
        ro, rl = _oracle_rows(w, 0, h, np.arange(N), 0, N, causal)
        _check(acc_o[0, h].cpu().numpy(), acc_l[0, h].cpu().numpy(), ro, rl, f"ring fp32 h{h}")
        _check(o_bf16[0, h].float().cpu().numpy(), lse[0, h].cpu().numpy(), ro, rl, f"ring bf16 h{h}")


def test_merge_of_all_partials_at_once_equals_attn_fwd():
    import exact_tiled_attention_16_gb300 as pkg
    N = 1024
    w = synth.make_bf16(1, 2, N, 64, True, seed=29)
    q, k, v = _dev(w.q), _dev(w.k), _dev(w.v)
    parts = [pkg.attn_fwd_partial(q, _dev(w.k[:, :, a:b]), _dev(w.v[:, :, a:b]), causal=True, k_offset=a,
                                  scale=w.scale) for a, b in [(0, 256), (256, 512), (512, 768), (768, 1024)]]
    o_m, l_m = pkg.attn_merge(parts)
    o_f, l_f = pkg.attn_fwd(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert (o_m.float() - o_f.float()).abs().max().item() <= 2e-2
    assert (l_m - l_f).abs().max().item() <= 1e-4


def test_merge_empty_partials():
    import exact_tiled_attention_16_gb300 as pkg
    o1 = torch.randn(1, 1, 40, 64, device="cuda")
    l1 = torch.full((1, 1, 40), float("-inf"), device="cuda")
    l1[0, 0, :20] = 0.5
    o1[0, 0, 20:] = 0.0
    o2 = torch.zeros(1, 1, 40, 64, device="cuda")
    l2 = torch.full((1, 1, 40), float("-inf"), device="cuda")
    o, lse = pkg.attn_merge([(o1, l1), (o2, l2)], out_fp32=True)
    torch.cuda.synchronize()
    assert torch.isneginf(lse[0, 0, 20:]).all() and (o[0, 0, 20:] == 0).all()
    assert torch.allclose(o[0, 0, :20], o1[0, 0, :20]) and torch.allclose(lse[0, 0, :20], l1[0, 0, :20])


def test_merge_weights_closed_form():
    """Two partials with lse a and b: weights sigmoid(a-b) and sigmoid(b-a)."""
    import exact_tiled_attention_16_gb300 as pkg
    g = torch.Generator(device="cuda").manual_seed(0)
    o1 = torch.randn(2, 3, 50, 128, device="cuda", generator=g)
    o2 = torch.randn(2, 3, 50, 128, device="cuda", generator=g)
    l1 = torch.randn(2, 3, 50, device="cuda", generator=g) * 3
    l2 = torch.randn(2, 3, 50, device="cuda", generator=g) * 3
    o, lse = pkg.attn_merge([(o1, l1), (o2, l2)], out_fp32=True)
    torch.cuda.synchronize()
    w1 = torch.sigmoid(l1 - l2)[..., None]
    assert torch.allclose(o, w1 * o1 + (1 - w1) * o2, atol=1e-5, rtol=1e-5)
    assert torch.allclose(lse, torch.logaddexp(l1, l2), atol=1e-5, rtol=1e-5)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16])
@pytest.mark.parametrize("causal", [False, True])
def test_splitkv_square(splits, causal):
    import exact_tiled_attention_16_gb300 as pkg
    from tests.gpu_utils import assert_bf16_tol, compare_rows
    w = synth.make_bf16(1, 3, 2000, 128, causal, seed=40 + splits)
    o, lse = pkg.attn_fwd_splitkv(_dev(w.q), _dev(w.k), _dev(w.v), splits, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert_bf16_tol(compare_rows(w, o.float().cpu().numpy().astype(np.float64),
                                 lse.cpu().numpy().astype(np.float64)), f"splitkv S={splits}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_splitkv_decode_shaped(causal, d):
    """Few queries against many keys; causal queries sit at the last positions."""
    import exact_tiled_attention_16_gb300 as pkg
    Nq, Nk = 200, 9000
    wk = synth.make_bf16(2, 2, Nk, d, causal, seed=51)
    qbits = wk.q[:, :, Nk - Nq:]  # queries = the last Nq rows of a seeded Nk-row draw
    o, lse = pkg.attn_fwd_splitkv(_dev(qbits), _dev(wk.k), _dev(wk.v), 8, causal=causal, scale=wk.scale)
    torch.cuda.synchronize()
    for b in range(2):
        for h in range(2):
            ro, rl = _oracle_rows(wk, b, h, np.arange(Nk - Nq, Nk), 0, Nk, causal)
            _check(o[b, h].float().cpu().numpy(), lse[b, h].cpu().numpy(), ro, rl, f"decode b{b}h{h}")


def test_splitkv_deterministic_and_workspace_checked():
    import exact_tiled_attention_16_gb300 as pkg
    import exact_tiled_attention_16_gb300._lib as L
    w = synth.make_bf16(1, 2, 1024, 64, False, seed=61)
    q, k, v = _dev(w.q), _dev(w.k), _dev(w.v)
    o1, l1 = pkg.attn_fwd_splitkv(q, k, v, 4)
    o2, l2 = pkg.attn_fwd_splitkv(q, k, v, 4)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    rc = L.attn_fwd_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o1.data_ptr(), 0, 1, 2, 1024, 1024, 64,
                                False, 0.125, 4, small.data_ptr(), 16, torch.cuda.current_stream().cuda_stream)
    assert rc == L.ATTN_ERR_WORKSPACE
