"""The C-ABI library builds, loads and exports every symbol include/attn.h
declares; argument validation returns the documented codes before any CUDA
call (no GPU needed for these)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_16_gb300 import build as b
    b.build()
    import exact_tiled_attention_16_gb300._lib as L
    return L.load_library()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("attn_fwd", "attn_status_string", "attn_check_device_errors"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    nm = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True)
    exported = set(re.findall(r"\sT\s+(\w+)$", nm.stdout, flags=re.M))
    for name in declared_functions():
        assert name in exported, f"{name} declared in include/ but not exported"
        assert hasattr(lib, name)


def test_status_strings(lib):
    import exact_tiled_attention_16_gb300._lib as L
    assert L.attn_status_string(0) == "ATTN_OK"
    for code in range(-13, 0):
        assert L.attn_status_string(code).startswith("ATTN_ERR_")
    assert "unknown" in L.attn_status_string(-999)


def _call(lib, q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=128, d=64, causal=0,
          scale=0.125, dtype=0):
    import exact_tiled_attention_16_gb300._lib as L
    return L.attn_fwd_raw(q, k, v, o, lse, B, H, N, d, causal, scale, 0, dtype)


# Cases rejected by host-side validation, before any CUDA call or launch.
INVALID = [
    (dict(q=0), -1), (dict(k=0), -1), (dict(v=0), -1), (dict(o=0), -1),
    (dict(B=0), -2), (dict(H=-1), -2), (dict(N=0), -2),
    (dict(d=32), -3), (dict(d=96), -3), (dict(d=256), -3),
    (dict(scale=0.0), -10), (dict(scale=-1.0), -10), (dict(scale=float("inf")), -10),
    (dict(scale=float("nan")), -10),
    (dict(q=0x1008), -5), (dict(o=0x4004), -5), (dict(lse=0x5002), -5),
    (dict(B=1 << 16, H=1 << 16), -6),
    (dict(dtype=7), -4),
]


@pytest.mark.parametrize("kwargs,code", INVALID, ids=[str(c[0]) for c in INVALID])
def test_validation_codes(lib, kwargs, code):
    assert _call(lib, **kwargs) == code


def _call_fp8(lib, d=128, qs=0x6000, **kw):
    import exact_tiled_attention_16_gb300._lib as L
    args = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000, B=1, H=1, N=128, causal=0, scale=0.125)
    args.update(kw)
    return L.attn_fwd_fp8_raw(args["q"], args["k"], args["v"], qs, 0x7000, 0x8000, args["o"], args["lse"],
                              args["B"], args["H"], args["N"], d, args["causal"], args["scale"], 0)


def test_fp8_validation_codes(lib):
    assert _call_fp8(lib, d=64) == -3
    assert _call_fp8(lib, qs=0) == -1
    assert _call_fp8(lib, qs=0x6002) == -5
    assert _call_fp8(lib, q=0) == -1
    assert _call_fp8(lib, N=0) == -2
    assert _call_fp8(lib, scale=0.0) == -10


def test_fp4p_validation_codes(lib):
    import exact_tiled_attention_16_gb300._lib as L

    def call(d=128, N=256, vts=0x7000, qs=0x6000, q=0x1000, scale=0.1):
        return L.attn_fwd_fp4p_raw(q, 0x2000, 0x3000, qs, 0x6100, vts, 0x4000, 0x5000, 1, 2, N, d, 0, scale, 0)
    assert call(d=64) == -3
    assert call(N=200) == -2   # N must be a multiple of 128
    assert call(vts=0) == -1
    assert call(vts=0x7002) == -5
    assert call(qs=0) == -1
    assert call(q=0) == -1
    assert call(scale=0.0) == -10


def test_fwd_host_validation(lib):
    import exact_tiled_attention_16_gb300._lib as L
    need = L.fwd_host_workspace_bytes(2, 3, 100, 64)
    # six heads, one per chunk (at most eight chunks): two slots of Q, K, V, O (100 x 64
    # bf16 each) and the chunk's LSE (400 bytes) rounded up to 256 bytes
    assert need == 2 * (4 * 100 * 64 * 2 + 512)
    # 32 heads in eight chunks of four
    assert L.fwd_host_workspace_bytes(1, 32, 256, 128) == 2 * (4 * 4 * 256 * 128 * 2 + 4096)
    assert L.fwd_host_workspace_bytes(1, 1, 100, 96) == 0

    def call(ws=0x10000, nbytes=need, d=64):
        return L.attn_fwd_host_raw(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 2, 3, 100, d, 0, 0.125, ws, nbytes, 0)
    assert call(ws=0) == -1
    assert call(ws=0x10010) == -5
    assert call(nbytes=need - 1) == -13
    assert call(d=96) == -3


def test_partial_merge_splitkv_validation(lib):
    import exact_tiled_attention_16_gb300._lib as L
    P = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, lse=0x5000)
    # partial: lse_part required, offsets >= 0
    assert L.attn_fwd_partial_raw(P["q"], P["k"], P["v"], P["o"], 0, 1, 1, 128, 128, 64, 0, 0, 0, 0.1, 0) == -1
    assert L.attn_fwd_partial_raw(P["q"], P["k"], P["v"], P["o"], P["lse"], 1, 1, 128, 128, 64, 1, -1, 0, 0.1,
                                  0) == -2
    assert L.attn_fwd_partial_raw(P["q"], P["k"], P["v"], P["o"], P["lse"], 1, 1, 128, 0, 64, 0, 0, 0, 0.1, 0) == -2
    # merge: part count, alignment, head dim
    assert L.attn_merge_raw([], [], P["o"], P["lse"], True, 1, 1, 8, 64, 0) == -2
    assert L.attn_merge_raw([0x1000] * 17, [0x2000] * 17, P["o"], P["lse"], True, 1, 1, 8, 64, 0) == -2
    assert L.attn_merge_raw([0x1008], [0x2000], P["o"], P["lse"], True, 1, 1, 8, 64, 0) == -5
    assert L.attn_merge_raw([0x1000], [0x2000], P["o"], P["lse"], True, 1, 1, 8, 96, 0) == -3
    assert L.attn_merge_raw([0], [0x2000], P["o"], P["lse"], True, 1, 1, 8, 64, 0) == -1
    # split-K/V: workspace, split count, causal needs Nq <= Nk
    assert L.attn_fwd_splitkv_raw(P["q"], P["k"], P["v"], P["o"], P["lse"], 1, 1, 128, 256, 64, 0, 0.1, 2, 0,
                                  1 << 20, 0) == -1
    assert L.attn_fwd_splitkv_raw(P["q"], P["k"], P["v"], P["o"], P["lse"], 1, 1, 128, 256, 64, 0, 0.1, 0,
                                  0x6000, 1 << 20, 0) == -2
    assert L.attn_fwd_splitkv_raw(P["q"], P["k"], P["v"], P["o"], P["lse"], 1, 1, 300, 256, 64, 1, 0.1, 2,
                                  0x6000, 1 << 20, 0) == -2
    # workspace size: S * B*H*Nq * (d + 1) * 4 bytes
    assert L.splitkv_workspace_bytes(2, 3, 100, 64, 4) == 4 * 6 * 100 * 65 * 4
    assert L.splitkv_workspace_bytes(1, 1, 1, 96, 1) == 0


def test_bwd_validation(lib):
    import exact_tiled_attention_16_gb300._lib as L
    a = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, dout=0x5000, lse=0x6000, dq=0x7000, dk=0x8000, dv=0x9000,
             B=1, H=2, N=100, d=64, causal=1, scale=0.125, workspace=0xa000, workspace_bytes=2048)

    def call(**kw):
        x = dict(a)
        x.update(kw)
        return L.attn_bwd_raw(x["q"], x["k"], x["v"], x["o"], x["dout"], x["lse"], x["dq"], x["dk"], x["dv"],
                              x["B"], x["H"], x["N"], x["d"], x["causal"], x["scale"], x["workspace"],
                              x["workspace_bytes"], 0)
    for name in ("q", "o", "dout", "lse", "dq", "dk", "dv", "workspace"):
        assert call(**{name: 0}) == -1, name
    assert call(N=0) == -2
    assert call(d=96) == -3
    assert call(scale=0.0) == -10
    assert call(dout=0x5008) == -5
    assert call(dk=0x8002) == -5
    assert call(lse=0x6002) == -5
    assert call(workspace=0xa008) == -5
    # two float arrays of B*H rows of N rounded up to 128
    assert call(workspace_bytes=2047) == -13
    assert L.bwd_workspace_bytes(1, 2, 100) == 2 * 2 * 128 * 4
    assert L.bwd_workspace_bytes(2, 3, 257) == 2 * 6 * 384 * 4
    assert L.bwd_workspace_bytes(0, 2, 100) == 0


def test_wait_timeout_setter(lib):
    assert lib.attn_set_wait_timeout_ns(10) == -2
    assert lib.attn_set_wait_timeout_ns(4_000_000_000) == 0


def test_no_device_fails_loudly(lib):
    """Without a GPU the valid call reports a CUDA error: nothing falls back to the CPU."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a device is present; this checks the no-device path")
    assert _call(lib) == -11


def test_binding_raises_without_library(tmp_path, monkeypatch):
    import exact_tiled_attention_16_gb300._lib as L
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(L, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        L.load_library()
