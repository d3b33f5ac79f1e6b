"""The alpha search through the Gram matrix (awq_gram, awq_search_scale_gram)
through the C ABI, against the fp64 oracle.

||X E^T||_F^2 = tr(E X^T X E^T): the route changes how the search objective
is evaluated, not what it is, so the bars are those of the direct search:
per-alpha MSE within 1e-3 relative of the oracle, the chosen alpha equal to
the oracle's (or an oracle near-tie within 2e-3), s bit-exact.  G/T itself is
checked element by element against the oracle's X^T X / T within its fp16
rounding and the fp32 accumulation over T tokens."""
import numpy as np
import pytest

import synthgen as sg

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MSE_TOL = 1e-3
NEAR_TIE = 2e-3


@pytest.fixture(scope="module")
def wb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_bit_stats_b300 import build
    build.build()
    import weight_only_bit_stats_b300 as m
    return m


@pytest.fixture(scope="module")
def orc(oracle_mod):
    return oracle_mod


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


@pytest.mark.parametrize("T,K", [(1, 128), (300, 384), (700, 1024), (4096, 512), (5000, 2048)])
def test_gram_matrix(wb, orc, T, K):
    _, X, _, _ = sg.layer_inputs(60, 0, 8, K, T)
    G = torch.full((K, K), float("nan"), dtype=torch.float16, device="cuda")
    wb.gram(dev(X), out=G)
    g = host(G).astype(np.float64)
    ref = orc.gram(X) / T
    d = np.sqrt(np.outer(np.diag(ref), np.diag(ref)))
    # fp16 rounding of the result (half an ulp: 2^-11 relative, 2^-25 absolute
    # below the normal range) plus the fp32 accumulation over T products,
    # each rounding at most 2^-23 of a partial sum bounded (Cauchy-Schwarz) by
    # T sqrt(G_ii G_jj); random in sign, so growing as sqrt(T): 8 sqrt(T)
    # 2^-23 sqrt(G_ii G_jj) after the division by T
    tol = 2.0 ** -11 * np.abs(ref) + 2.0 ** -25 + 8.0 * np.sqrt(T) * 2.0 ** -23 * d
    assert np.all(np.isfinite(g))
    assert np.all(np.abs(g - ref) <= tol), float(np.max(np.abs(g - ref) / tol))
    wb.sync_status()


def _gram_search_check(wb, orc, W, X):
    T = X.shape[0]
    m = orc.act_mean(orc.act_stats(X), T)
    G = wb.gram(dev(X))
    s, mse, best, cands = wb.search_scale_gram(dev(W), G, dev(m), return_candidates=True)
    s, mse, best, cands = host(s), host(mse), int(host(best)[0]), host(cands)
    ref_c = np.stack([orc.candidate_scales(m, a) for a in orc.ALPHA_GRID])
    assert np.array_equal(cands, ref_c)
    G64 = orc.gram(X)
    ref_mse = np.array([orc.search_mse_gram(W, G64, T, c) for c in ref_c])
    rel = np.abs(mse - ref_mse) / ref_mse
    assert np.max(rel) <= MSE_TOL, (rel, mse, ref_mse)
    ref_best = int(np.argmin(ref_mse))
    if best != ref_best:
        assert abs(ref_mse[best] - ref_mse[ref_best]) <= NEAR_TIE * ref_mse[ref_best]
    assert np.array_equal(s, ref_c[best])
    wb.sync_status()
    return mse, ref_mse


@pytest.mark.parametrize("N,K,T", [(128, 128, 200), (136, 384, 700), (256, 1024, 3000),
                                   (520, 640, 1500)])
def test_gram_search_parity(wb, orc, N, K, T):
    """Ragged row tiles (N % 128 != 0) and column blocks (K % 512 != 0)."""
    W, X, _, _ = sg.layer_inputs(61, 0, N, K, T)
    _gram_search_check(wb, orc, W, X)


def test_gram_search_llama7b_rows_t8192(wb, orc):
    """K = 4096 with T = 8192 calibration tokens (T > K, where the route
    pays): 512 rows of the LLaMA-7B-shaped o projection, every alpha."""
    W, X, _, _ = sg.layer_inputs(0, 1, 512, 4096, 8192)
    _gram_search_check(wb, orc, W, X)


@pytest.mark.parametrize("N,K,T", [(4096, 4096, 512), (512, 11008, 8192), (4096, 4096, 65536),
                                   (1024, 11008, 65536)])
def test_gram_search_equals_direct_search(wb, orc, N, K, T):
    """The two GPU routes of the same objective at full K and up to 65 536
    calibration tokens: per-alpha MSE within 1e-3 of each other, the same
    alpha (or a near-tie of the direct route's) and the same s."""
    W, X, _, _ = sg.layer_inputs(62, 0, N, K, T)
    Wd, Xd = dev(W), dev(X)
    m = wb.act_mean(wb.act_stats(Xd), T)
    s1, mse1, b1 = wb.search_scale(Wd, Xd, m)
    G = wb.gram(Xd)
    del Xd
    s2, mse2, b2 = wb.search_scale_gram(Wd, G, m)
    mse1, mse2 = host(mse1), host(mse2)
    b1, b2 = int(host(b1)[0]), int(host(b2)[0])
    assert np.max(np.abs(mse2 - mse1) / mse1) <= MSE_TOL
    if b1 != b2:
        assert abs(mse1[b2] - mse1[b1]) <= NEAR_TIE * mse1[b1]
    else:
        assert np.array_equal(host(s1), host(s2))
    assert mse2[b2] <= mse2[0]
    wb.sync_status()
