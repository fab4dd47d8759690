"""dspark_copy_target_rows: exactly the rows a verification reads under a schedule (T[b, j]
for j <= l_b) are fetched, from pinned host memory or from device memory, and nothing else
is written; a schedule entry outside [0, gamma] is clamped and reported."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
ds = pytest.importorskip("speculative_decoding_03_gb300")


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _expect(src, ell, fill):
    out = np.full_like(src, fill)
    for b, L in enumerate(ell):
        L = min(max(int(L), 0), src.shape[1] - 1)
        out[b, :L + 1] = src[b, :L + 1]
    return out


@pytest.mark.parametrize("where", ["pinned", "device"])
def test_copy_target_rows_fetches_exactly_the_verified_rows(where):
    _need_gpu()
    B, gamma, V = 5, 4, 9000          # two segments of a row, the second ragged
    rng = np.random.default_rng(3)
    src_np = rng.normal(size=(B, gamma + 1, V)).astype(np.float32)
    src = torch.from_numpy(src_np).pin_memory() if where == "pinned" else torch.from_numpy(src_np).cuda()
    ell = np.array([0, 4, 2, 1, 3], np.int32)
    T = torch.full((B, gamma + 1, V), -7.0, device="cuda")
    ws = ds.Workspace(B, gamma, V, 16, 0)
    ds.copy_target_rows(src, T, torch.from_numpy(ell).cuda(), ws)
    np.testing.assert_array_equal(T.cpu().numpy(), _expect(src_np, ell, -7.0))
    assert ws.status() == 0


def test_copy_target_rows_clamps_and_reports_a_bad_schedule():
    _need_gpu()
    B, gamma, V = 3, 2, 64
    src_np = np.arange(B * (gamma + 1) * V, dtype=np.float32).reshape(B, gamma + 1, V)
    src = torch.from_numpy(src_np).pin_memory()
    ell = np.array([7, -3, 1], np.int32)
    T = torch.zeros((B, gamma + 1, V), device="cuda")
    ws = ds.Workspace(B, gamma, V, 16, 0)
    ds.copy_target_rows(src, T, torch.from_numpy(ell).cuda(), ws)
    np.testing.assert_array_equal(T.cpu().numpy(), _expect(src_np, ell, 0.0))
    assert ws.status() == 5          # DSPARK_ERR_DEVICE_CHECK, read and cleared
    assert ws.status() == 0
