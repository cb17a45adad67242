"""Host-side logic of bench.py (no GPU): the kernel instance it names matches the
library's instance table, the kernel hash covers every CUDA source, the oracle
row probe (the 1-thread CPU baseline) prints what the bench reads, and the
reference arm's JSON line carries the per-row figures."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_kernel_instance_follows_the_instance_table():
    text = open(os.path.join(bench.CSRC, "attn_api.cu")).read()
    assert "#define ATTN_BF16_D128 128, 2, 2, false" in text
    # D, K stages, V stages, fp8, partial, fp4, TMA store of O (non-causal BF16 only),
    # unit table (BF16 launches whose rounds fit in it), pair tail (non-causal BF16
    # table launches and FP8 launches that split their last round over CTA pairs)
    assert bench.kernel_instance("bf16", 128, causal=True) == "attn::attn_fwd_kernel<128, 2, 2, 0, 0, 0, 0, 0, 0>"
    assert (bench.kernel_instance("bf16", 128, causal=True, table=True)
            == "attn::attn_fwd_kernel<128, 2, 2, 0, 0, 0, 0, 1, 0>")
    assert bench.kernel_instance("bf16", 128, causal=False) == "attn::attn_fwd_kernel<128, 2, 2, 0, 0, 0, 1, 0, 0>"
    assert bench.kernel_instance("bf16", 64, causal=False) == "attn::attn_fwd_kernel<64, 4, 4, 0, 0, 0, 1, 0, 0>"
    assert (bench.kernel_instance("bf16", 64, causal=False, table=True)
            == "attn::attn_fwd_kernel<64, 4, 4, 0, 0, 0, 1, 1, 0>")
    assert (bench.kernel_instance("bf16", 128, causal=False, table=True, pair_tail=True)
            == "attn::attn_fwd_kernel<128, 2, 2, 0, 0, 0, 1, 1, 1>")
    assert (bench.kernel_instance("bf16", 128, causal=True, table=True, pair_tail=True)
            == "attn::attn_fwd_kernel<128, 2, 2, 0, 0, 0, 0, 1, 0>")
    assert bench.kernel_instance("bf16", 128, partial=True) == "attn::attn_fwd_kernel<128, 2, 2, 0, 1, 0, 0, 0, 0>"
    assert bench.kernel_instance("e4m3", 128) == "attn::attn_fwd_kernel<128, 3, 3, 1, 0, 0, 0, 0, 0>"
    assert bench.kernel_instance("e4m3_e2m1", 128) == "attn::attn_fwd_kernel<128, 4, 4, 1, 0, 1, 0, 0, 0>"
    assert bench.kernel_instance("e4m3", 128, causal=True, table=True) == "attn::attn_fwd_kernel<128, 3, 3, 1, 0, 0, 0, 0, 0>"
    # FP8 launches compute their units but may split their last round
    assert (bench.kernel_instance("e4m3", 128, pair_tail=True)
            == "attn::attn_fwd_kernel<128, 3, 3, 1, 0, 0, 0, 0, 1>")
    assert (bench.kernel_instance("e4m3_e2m1", 128, pair_tail=True)
            == "attn::attn_fwd_kernel<128, 4, 4, 1, 0, 1, 0, 0, 0>")


def test_custom_workloads():
    """--custom B,H,N,d,causal[,e4m3]: a seeded BF16 workload, or a block-scaled e4m3
    one with cfg5's recipe, of that shape; --all carries the FP8 shape whose last
    round is split over CTA pairs."""
    import argparse
    import numpy as np
    w = bench.make_workload(argparse.Namespace(custom="1,2,300,64,1", workload="cfg3"))
    assert (w.dtype, w.B, w.H, w.N, w.d, w.causal) == ("bf16", 1, 2, 300, 64, True)
    assert w.name == "custom_B1H2N300d64c"
    w = bench.make_workload(argparse.Namespace(custom="1,2,300,128,0,e4m3", workload="cfg3"))
    assert (w.dtype, w.B, w.H, w.N, w.d, w.causal) == ("e4m3", 1, 2, 300, 128, False)
    assert w.name == "custom_B1H2N300d128n_e4m3"
    assert w.q.dtype == np.uint8 and w.q_scale.shape == (1, 2, 3)
    with pytest.raises(SystemExit):
        bench.make_workload(argparse.Namespace(custom="1,2,300,128,0,fp16", workload="cfg3"))
    assert "custom:1,16,8192,128,0,e4m3" in bench.ALL_WORKLOADS


def test_kernel_hash_covers_every_cuda_source(tmp_path, monkeypatch):
    srcs = bench.kernel_sources()
    for must in ("attn_fwd_kernel.cuh", "attn_bwd_kernel.cuh", "ptx.cuh", "attn_api.cu", "attn_diag.cu",
                 "attn_merge.cuh", "tmem_ldst.inc"):
        assert must in srcs
    h = bench.kernel_hash()
    assert len(h) == 16 and h == bench.kernel_hash()
    # a changed source changes the hash
    for f in srcs:
        (tmp_path / f).write_bytes(open(os.path.join(bench.CSRC, f), "rb").read())
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    assert bench.kernel_hash() == h
    (tmp_path / "ptx.cuh").write_bytes((tmp_path / "ptx.cuh").read_bytes() + b"\n")
    assert bench.kernel_hash() != h


def test_traffic_is_reported_only_for_the_current_kernel():
    t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for key, e in t.items():
        if isinstance(e, dict):
            got = bench.traffic_for(key)
            assert got == (e["dram_bytes_per_launch"] if e["kernel_hash"] == bench.kernel_hash() else None)


def test_cpu_row_probe_with_one_blas_thread():
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-row-probe", "--custom",
                        "1,2,256,64,1", "--cpu-budget", "0.5", "--probe-rows", "16"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["threads"] == 1 and d["rows"] > 0 and d["ms_per_row"] > 0
    assert abs(d["ms_per_row"] - d["seconds"] * 1e3 / d["rows"]) < 1e-9


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--small",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["ms_per_row_all_cores"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
