"""The FMA-pipe exponential on the GPU (attn_eval_exp2 runs the library's own
device function exp2_poly2) against the float32 emulation of tests/test_exp2_poly.py,
the exact 2^x and the special-function unit's ex2.approx on the same inputs; and
the exponential-throughput diagnostic the benchmark uses."""
import numpy as np
import pytest

from tests.test_exp2_poly import BOUND, _grid, exp2_poly_emul

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_16_gb300 as pkg
    pkg.load_library()


def test_device_polynomial_matches_emulation_and_bound():
    import exact_tiled_attention_16_gb300 as pkg
    x = np.concatenate([_grid(), np.array([-127.0, -200.0, -np.inf, -126.5, 0.0, 8.0, 14.0], np.float32)])
    y_poly, y_sfu = pkg.eval_exp2(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    y_poly = y_poly.cpu().numpy()
    y_sfu = y_sfu.cpu().numpy()
    emu = exp2_poly_emul(x)
    # the same float32 steps: equal up to the emulation's rare double rounding
    # (one float32 step of p, i.e. at most 2^-23 relative)
    ok = np.isfinite(emu) & (emu > 0)
    ulp = np.abs(y_poly[ok].view(np.int32).astype(np.int64) - emu[ok].view(np.int32).astype(np.int64))
    assert ulp.max() <= 1, f"device and emulation differ by {ulp.max()} float32 steps"
    assert np.array_equal(y_poly[~ok].view(np.uint32), emu[~ok].view(np.uint32))
    # against the exact 2^x and against ex2.approx on [-126, 20]
    sel = (x >= -126.0) & (x <= 20.0)
    exact = np.exp2(x[sel].astype(np.float64))
    rel = np.abs(y_poly[sel].astype(np.float64) / exact - 1.0)
    assert rel.max() <= BOUND, f"max relative error {rel.max():.3e}"
    rel_sfu = np.abs(y_poly[sel].astype(np.float64) / y_sfu[sel].astype(np.float64) - 1.0)
    assert rel_sfu.max() <= BOUND + 2.0 ** -20, f"against ex2.approx {rel_sfu.max():.3e}"
    # masked scores (-inf) and anything at or below -127 give +0.0
    assert np.all(y_poly[np.isin(x, np.array([-127.0, -200.0, -np.inf], np.float32))].view(np.uint32) == 0)


def test_exp2_rates_diagnostic():
    import exact_tiled_attention_16_gb300 as pkg
    sfu, poly = pkg.measure_exp2_rates()
    print(f"[exp2 rates] ex2.approx {sfu:.2f} and polynomial {poly:.2f} exponentials per SM clock per SM")
    # at least the 16 per clock of the pre-Blackwell-Ultra special-function units,
    # and finite
    assert 16.0 <= sfu < 1024.0 and 1.0 <= poly < 1024.0
