"""attn_fwd_host: the forward on host buffers, with transfers and kernels
pipelined in chunks of heads, gives the outputs of attn_fwd on the same inputs --
bit for bit with the split of a launch's last round over CTA pairs turned off
(each chunk then runs the same kernel on whole heads), within the BF16 tolerance
with it on -- with pinned or pageable host memory, ragged last chunks, without
LSE, and on back-to-back calls that share the workspace."""
import numpy as np
import pytest

from exact_tiled_attention_16_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_16_gb300 as pkg
    pkg.load_library()


def _host(bits, pin):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


SHAPES = [(1, 1, 200, 64, False), (2, 3, 333, 128, True), (1, 5, 1000, 64, True), (2, 16, 512, 128, False),
          (1, 7, 129, 128, True)]


@pytest.mark.parametrize("pin", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{b}H{h}N{n}d{d}{'c' if c else 'n'}" for b, h, n, d, c in SHAPES])
def test_bitwise_equal_to_device_call(shape, pin):
    import exact_tiled_attention_16_gb300 as pkg
    B, H, N, d, causal = shape
    w = synth.make_bf16(B, H, N, d, causal, seed=600 + N)
    qh, kh, vh = (_host(x, pin) for x in (w.q, w.k, w.v))
    # with the pair-tail split on: equal within the BF16 tolerance
    o_h, l_h = pkg.attn_fwd_host(qh, kh, vh, causal=causal, scale=w.scale)
    torch.cuda.current_stream().synchronize()
    o_d, l_d = pkg.attn_fwd(qh.cuda(), kh.cuda(), vh.cuda(), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert (o_h.float() - o_d.cpu().float()).abs().max().item() <= 2e-2
    assert (l_h - l_d.cpu()).abs().max().item() <= 1e-3
    # with it off: bit for bit
    pkg.diag_set_pair_tail(False)
    try:
        o_h, l_h = pkg.attn_fwd_host(qh, kh, vh, causal=causal, scale=w.scale)
        torch.cuda.current_stream().synchronize()
        o_d, l_d = pkg.attn_fwd(qh.cuda(), kh.cuda(), vh.cuda(), causal=causal, scale=w.scale)
        torch.cuda.synchronize()
    finally:
        pkg.diag_set_pair_tail(True)
    assert torch.equal(o_h.view(torch.int16), o_d.cpu().view(torch.int16))
    assert torch.equal(l_h.view(torch.int32), l_d.cpu().view(torch.int32))
    assert pkg.check_device_errors()[0] == 0


def test_without_lse_and_back_to_back_calls():
    import exact_tiled_attention_16_gb300 as pkg
    pkg.diag_set_pair_tail(False)  # bit for bit (see the module docstring)
    try:
        _back_to_back(pkg)
    finally:
        pkg.diag_set_pair_tail(True)


def _back_to_back(pkg):
    B, H, N, d = 2, 6, 700, 128
    ws = torch.empty(pkg.fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    outs = []
    ins = []
    for seed in (1, 2, 3):
        w = synth.make_bf16(B, H, N, d, seed == 2, seed=seed)
        qh, kh, vh = (_host(x, True) for x in (w.q, w.k, w.v))
        o, lse = pkg.attn_fwd_host(qh, kh, vh, causal=w.causal, scale=w.scale, want_lse=False, workspace=ws)
        assert lse is None
        outs.append(o)
        ins.append((qh, kh, vh, w))
    torch.cuda.current_stream().synchronize()
    for o, (qh, kh, vh, w) in zip(outs, ins):
        o_d, _ = pkg.attn_fwd(qh.cuda(), kh.cuda(), vh.cuda(), causal=w.causal, scale=w.scale)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_d.cpu().view(torch.int16))


def test_workspace_too_small_launches_nothing():
    import exact_tiled_attention_16_gb300._lib as L
    q = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16).pin_memory()
    o = torch.full_like(q, 7.0)
    need = L.fwd_host_workspace_bytes(1, 2, 256, 64)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = L.attn_fwd_host_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), 0, 1, 2, 256, 64, 0, 0.125,
                             ws.data_ptr(), need - 256, torch.cuda.current_stream().cuda_stream)
    assert rc == L.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (o.float() == 7.0).all()


FP8_SHAPES = [(1, 2, 1000, 128, False), (2, 9, 700, 128, True), (1, 32, 2048, 128, False)]


@pytest.mark.parametrize("pin", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("shape", FP8_SHAPES, ids=[f"B{b}H{h}N{n}{'c' if c else 'n'}" for b, h, n, d, c in FP8_SHAPES])
def test_fp8_host_bitwise_equal_to_device_call(shape, pin):
    """attn_fwd_fp8_host: the e4m3 codes and block scales in host memory, pipelined
    in chunks of whole heads; every chunk runs attn_fwd_fp8's kernel, so with the
    split of a last round over CTA pairs off (these shapes have too few key blocks
    for it anyway) the outputs are bit for bit those of attn_fwd_fp8."""
    import exact_tiled_attention_16_gb300 as pkg
    B, H, N, d, causal = shape
    w = synth.make_fp8(B, H, N, d, causal, seed=700 + N)

    def host(x):
        t = torch.from_numpy(np.ascontiguousarray(x))
        return t.pin_memory() if pin else t.clone()
    q8, k8, v8, qs, ks, vs = (host(x) for x in (w.q, w.k, w.v, w.q_scale, w.k_scale, w.v_scale))
    pkg.diag_set_pair_tail(False)
    try:
        o_h, l_h = pkg.attn_fwd_fp8_host(q8, k8, v8, qs, ks, vs, causal=causal, scale=w.scale)
        torch.cuda.current_stream().synchronize()
        o_d, l_d = pkg.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qs.cuda(), ks.cuda(), vs.cuda(),
                                    causal=causal, scale=w.scale)
        torch.cuda.synchronize()
    finally:
        pkg.diag_set_pair_tail(True)
    assert torch.equal(o_h.view(torch.int16), o_d.cpu().view(torch.int16))
    assert torch.equal(l_h.view(torch.int32), l_d.cpu().view(torch.int32))
    assert pkg.check_device_errors()[0] == 0


def test_fp8_host_with_pair_tail():
    """B1 H16 N8192: every chunk of the pipeline (two heads, 64 units) splits all its
    units over CTA pairs, the whole-tensor launch only its last round; both against
    the oracle on sampled rows, and against each other within one bf16 step of O."""
    import exact_tiled_attention_16_gb300 as pkg
    from tests.gpu_utils import assert_fp8_tol, compare_rows
    B, H, N = 1, 16, 8192
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if not pkg.diag_fwd_schedule(2, N, N, False, fp8=True, num_sms=sms)[0]["pair_tail"]:
        pytest.skip(f"{sms} SMs: a chunk's units are not split")
    w = synth.make_fp8(B, H, N, 128, False, seed=4242)
    q8, k8, v8, qs, ks, vs = (torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
                              for x in (w.q, w.k, w.v, w.q_scale, w.k_scale, w.v_scale))
    o_h, l_h = pkg.attn_fwd_fp8_host(q8, k8, v8, qs, ks, vs, causal=False, scale=w.scale)
    torch.cuda.current_stream().synchronize()
    o_d, l_d = pkg.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qs.cuda(), ks.cuda(), vs.cuda(), causal=False,
                                scale=w.scale)
    torch.cuda.synchronize()
    assert pkg.check_device_errors()[0] == 0
    o_h = o_h.float().numpy().astype(np.float64)
    o_d = o_d.float().cpu().numpy().astype(np.float64)
    l_h = l_h.numpy().astype(np.float64)
    l_d = l_d.cpu().numpy().astype(np.float64)
    assert (np.abs(o_h - o_d) <= 2e-2 + 2.0 ** -7 * np.abs(o_d)).all() and np.abs(l_h - l_d).max() <= 1e-3
    det = {}
    assert_fp8_tol(compare_rows(w, o_h, l_h, rows_per_head=64, excess=True, detail=det), "fp8 host, pair tail", det)


def test_fp8_host_workspace_too_small_launches_nothing():
    import exact_tiled_attention_16_gb300._lib as L
    B, H, N, d = 1, 2, 256, 128
    q = torch.zeros(B, H, N, d, dtype=torch.uint8).pin_memory()
    sc = torch.ones(B, H, N // 128, dtype=torch.float32).pin_memory()
    o = torch.full((B, H, N, d), 7.0, dtype=torch.bfloat16).pin_memory()
    need = L.fp8_host_workspace_bytes(B, H, N, d)
    assert need > 0 and L.fp8_host_workspace_bytes(B, H, N, 64) == 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = L.attn_fwd_fp8_host_raw(q.data_ptr(), q.data_ptr(), q.data_ptr(), sc.data_ptr(), sc.data_ptr(), sc.data_ptr(),
                                 o.data_ptr(), 0, B, H, N, d, False, 0.1, ws.data_ptr(), need - 256, 0)
    assert rc == L.ATTN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (o.float() == 7.0).all()
