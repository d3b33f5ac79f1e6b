"""The allocation-free alpha search, awq_search_scale_noalloc.

Some callers cannot allocate device memory (a plug-in whose host program owns
the whole device memory pool; a loop that must avoid cudaMalloc because it
can synchronise the device).  This entry point keeps its scratch in a
library-owned device array instead of a caller workspace.  Called through the
C ABI it must give the same results as awq_search_scale with a workspace, on
two calls in a row (the array keeps the previous call's contents), and it
must refuse a problem that needs more scratch than the array holds.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import synthgen as sg

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MSE_TOL = 1e-3


@pytest.fixture(scope="module")
def wb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_bit_stats_b300 import build
    build.build()
    import weight_only_bit_stats_b300 as m
    return m


def _noalloc(wb, W, X, m, alphas, s, mse, best):
    arr = (ctypes.c_double * len(alphas))(*alphas)
    N, K = W.shape
    T = X.shape[0]
    return wb.lib().awq_search_scale_noalloc(
        W.data_ptr(), N, K, K, X.data_ptr(), T, K, m.data_ptr(), arr, len(alphas), 128,
        s.data_ptr(), mse.data_ptr(), best.data_ptr(), None,
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_search_matches_workspace_search(wb):
    alphas = wb.ALPHA_GRID
    # two calls in a row on different layers and shapes: what the first call
    # left in the shared scratch must not leak into the second
    for layer, (N, K, T) in enumerate([(1024, 1024, 512), (384, 2048, 300)]):
        W, X, _, _ = sg.layer_inputs(20 + layer, 0, N, K, T)
        Wd = torch.from_numpy(W).cuda()
        Xd = torch.from_numpy(X).cuda()
        m = wb.act_mean(wb.act_stats(Xd), T)
        s_ref, mse_ref, best_ref = wb.search_scale(Wd, Xd, m, alphas)
        s = torch.full((K,), float("nan"), dtype=torch.float32, device="cuda")
        mse = torch.full((len(alphas),), float("nan"), dtype=torch.float64, device="cuda")
        best = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = _noalloc(wb, Wd, Xd, m, alphas, s, mse, best)
        assert rc == 0, wb.lib().awq_last_error_string()
        wb.sync_status()
        assert int(best.cpu()[0]) == int(best_ref.cpu()[0])
        assert np.array_equal(s.cpu().numpy(), s_ref.cpu().numpy())
        ref = mse_ref.cpu().numpy()
        assert np.max(np.abs(mse.cpu().numpy() - ref) / ref) <= MSE_TOL


def test_noalloc_refuses_oversized_problem(wb):
    """A problem whose scratch exceeds the library's array is refused on the
    host with AWQ_ERR_WORKSPACE and a message naming the limit."""
    K = 131072
    assert wb.lib().awq_search_workspace_size(1024, K, 512, 64) > 16 << 20
    small = torch.zeros(1024, dtype=torch.float16, device="cuda")
    out = torch.zeros(16, dtype=torch.float64, device="cuda")
    arr = (ctypes.c_double * 64)(*[i / 64 for i in range(64)])
    rc = wb.lib().awq_search_scale_noalloc(small.data_ptr(), 1024, K, K, small.data_ptr(), 512, K,
                                           out.data_ptr(), arr, 64, 128, out.data_ptr(),
                                           out.data_ptr(), out.data_ptr(), None, None)
    assert rc == 5
    assert b"16 MiB" in wb.lib().awq_last_error_string()
