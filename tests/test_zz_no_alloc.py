"""attn_fwd_splitkv_static: split-K/V attention for callers that may not allocate
device memory (their memory belongs to another allocator, or cudaMalloc's possible
device synchronisation is not acceptable on their path).  Its scratch is a fixed
array inside the library, so the caller passes only inputs and outputs.

Checked through the C ABI on two calls in a row (the second a smaller problem,
so stale partials left in the shared array by the first call would show): each
result is bitwise the workspace-taking attn_fwd_splitkv's (the same kernels on
the same inputs are deterministic, so any difference at all would be a leak
through the shared array), and each is compared with the fp64 oracle on a
seeded sample of query rows within the BF16 tolerances.  The size limit is
checked to launch nothing.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from exact_tiled_attention_16_gb300 import synth
from oracle.attention import attention_head
from tests.gpu_utils import BF16_MAX_ABS_LSE, BF16_MAX_ABS_O, BF16_MEAN_ABS_O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_16_gb300._lib as L
    so = L.load_library()
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    so.attn_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp]
    so.attn_fwd_splitkv_static.restype = ci
    so.attn_splitkv_static_scratch_bytes.argtypes = []
    so.attn_splitkv_static_scratch_bytes.restype = ctypes.c_size_t
    return so


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _static_call(lib, q, k, v, o, lse, causal, scale, splits):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    return lib.attn_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                       B, H, Nq, Nk, d, 1 if causal else 0, float(scale), splits,
                                       torch.cuda.current_stream().cuda_stream)


def test_two_calls_in_a_row_match_workspace_entry(lib):
    import exact_tiled_attention_16_gb300 as pkg
    problems = [
        # (B, H, Nq, Nk, d, causal, splits): the first fills much of the scratch,
        # the second is smaller and reads only what it wrote itself
        (2, 4, 384, 6000, 128, False, 8),
        (1, 3, 100, 2500, 64, True, 5),
    ]
    for i, (B, H, Nq, Nk, d, causal, splits) in enumerate(problems):
        w = synth.make_bf16(B, H, Nk, d, causal, seed=900 + i)
        q, k, v = _dev(w.q[:, :, Nk - Nq:]), _dev(w.k), _dev(w.v)
        o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
        assert _static_call(lib, q, k, v, o, lse, causal, w.scale, splits) == 0
        o_ws, lse_ws = pkg.attn_fwd_splitkv(q, k, v, splits, causal=causal, scale=w.scale)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o_ws.view(torch.int16)), f"call {i}: O differs from attn_fwd_splitkv"
        assert torch.equal(lse.view(torch.int32), lse_ws.view(torch.int32)), f"call {i}: LSE differs"
        # the oracle on 64 seeded query rows of every head (queries = the last Nq positions)
        o_np = o.float().cpu().numpy().astype(np.float64)
        lse_np = lse.cpu().numpy().astype(np.float64)
        for b in range(B):
            for h in range(H):
                qf, kf, vf = w.head_f64(b, h)
                sel = synth.sample_rows(Nq, 64, 900 + i, b, h)
                ro, rl = attention_head(qf, kf, vf, causal, w.scale, rows=Nk - Nq + sel)
                d_o = np.abs(o_np[b, h][sel] - ro)
                assert d_o.max() <= BF16_MAX_ABS_O and d_o.mean() <= BF16_MEAN_ABS_O, f"call {i} b{b}h{h}"
                assert np.abs(lse_np[b, h][sel] - rl).max() <= BF16_MAX_ABS_LSE, f"call {i} b{b}h{h} lse"


def test_oversized_problem_is_rejected_without_launch(lib):
    import exact_tiled_attention_16_gb300._lib as L
    limit = lib.attn_splitkv_static_scratch_bytes()
    assert limit == 32 << 20
    # 16 splits x 32 heads x 512 rows x 129 floats x 4 bytes = 135 MB > 32 MiB
    B, H, Nq, Nk, d = 2, 16, 512, 4096, 128
    q = torch.zeros((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, H, Nk, d), dtype=torch.bfloat16, device="cuda")
    o = torch.full((B, H, Nq, d), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), 5.0, dtype=torch.float32, device="cuda")
    assert _static_call(lib, q, k, k, o, lse, False, 0.1, 16) == L.ATTN_ERR_SCRATCH
    torch.cuda.synchronize()
    assert (o.float() == 3.0).all() and (lse == 5.0).all()
