"""The TMEM loads with a max reduction (tcgen05.ld.red .max) that give the forward
kernel its row maxima (BF16, FP8) and its 32-key block maxima (Direct-P FP4).  A
wrong maximum would not show in the attention parity tests -- the softmax does not
depend on the shift as long as nothing overflows -- so the loads are checked here
on their own, through the library's diagnostic entry point: the values they return
and the maxima, bit for bit against the host."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_tiled_attention_16_gb300 as pkg
    pkg.load_library()


def _tile(seed):
    """128 rows of 128 f32 scores: every row's maximum sits in a different column
    (row r at column r), so a reduction over part of the columns fails; rows of
    large magnitudes, all-negative rows, rows with -inf (masked keys), a row of
    -inf alone and rows whose maximum repeats."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((128, 128)) * 8.0).astype(np.float32)
    for r in range(128):
        x[r, r] = np.abs(x[r]).max() + 1.0 + r
    x[16:24] *= np.float32(1e30)
    x[24:32] = -np.abs(x[24:32]) - 1.0
    x[24:32, 24:32] = -np.float32(0.5)  # the largest of an all-negative row
    x[32:40, ::2] = -np.inf
    x[40:48, :] = -np.inf
    x[40:47, 5 * np.arange(7)] = np.arange(7, dtype=np.float32) - 3.0
    x[47] = -np.inf
    x[48:56, 100:104] = x[48:56].max(axis=1, keepdims=True)
    return x


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_load_with_max_returns_the_row_and_its_maximum(seed):
    import exact_tiled_attention_16_gb300 as pkg
    x = _tile(seed)
    vals, mx, bmx = pkg.diag_tmem_row_max(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    vals = vals.cpu().numpy()
    mx = mx.cpu().numpy()
    bmx = bmx.cpu().numpy()
    assert np.array_equal(vals.view(np.uint32), x.view(np.uint32)), "the loaded values differ from the stored ones"
    want = x.max(axis=1)
    bad = np.nonzero(mx.view(np.uint32) != want.view(np.uint32))[0]
    assert bad.size == 0, f"rows {bad[:8].tolist()}: got {mx[bad[:8]].tolist()}, want {want[bad[:8]].tolist()}"
    assert mx[47] == -np.inf
    # the four-group form (Direct-P FP4): each 32-column group's maximum
    want_b = x.reshape(128, 4, 32).max(axis=2)
    assert np.array_equal(bmx.view(np.uint32), want_b.view(np.uint32)), "a 32-column group maximum differs"


def test_rejects_bad_arguments():
    import exact_tiled_attention_16_gb300 as pkg
    with pytest.raises(ValueError):
        pkg.diag_tmem_row_max(torch.zeros(64, 128, device="cuda"))
    with pytest.raises(ValueError):
        pkg.diag_tmem_row_max(torch.zeros(128, 128))
