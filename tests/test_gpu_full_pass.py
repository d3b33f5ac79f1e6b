"""The full LLaMA-7B-shaped quantisation pass (32 decoder layers x 7 linears,
128 x 512 = 65536 calibration tokens per input, then the matmul at M in
{1, 16, 64, 256}), checked on decoder layers 0 and 31:

* statistics of each of the layer's four inputs over all 65536 tokens:
  bit-exact against the oracle;
* the alpha search over all 65536 tokens on the GPU (the fp64 oracle cannot
  afford it: its mse values are unpinned here), with mse(best) <= mse(0);
  and the same search on the first 512 tokens on both sides: per-alpha mse
  within 1e-3, same alpha (or an oracle near-tie), same s;
* the INT4 pack of every linear with the full-token s: bit-exact;
* the matmul at M = 1, 16, 64, 256: 2e-3 on sampled outputs.
"""
import numpy as np
import pytest

import synthgen as sg

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

T_FULL = 128 * 512
T_SUB = 512
MSE_TOL = 1e-3
NEAR_TIE = 2e-3
GEMM_TOL = 2e-3


@pytest.fixture(scope="module")
def wb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_bit_stats_b300 import build
    build.build()
    import weight_only_bit_stats_b300 as m
    return m


def _host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


@pytest.mark.parametrize("layer", [0, 31])
def test_llama7b_full_pass_layer(wb, oracle_mod, layer):
    orc = oracle_mod
    rng = np.random.default_rng(1000 + layer)
    means = {}
    xs_dev = {}
    for idx, (name, K) in enumerate(sg.LLAMA7B_LAYER_INPUTS):
        X = sg.layer_activations(layer, idx, T_FULL, K)
        Xd = torch.from_numpy(X).cuda()
        abs_sum = wb.act_stats(Xd)
        ref = orc.act_stats(X)
        assert np.array_equal(_host(abs_sum), ref), name
        means[idx] = (wb.act_mean(abs_sum, T_FULL), orc.act_mean(ref, T_FULL), X[:T_SUB].copy())
        xs_dev[idx] = Xd
        del X
    for j, (name, N, K) in enumerate(sg.LLAMA7B_LAYER_LINEARS):
        idx = sg.LLAMA7B_LINEAR_INPUT[j]
        m_dev, m_ref, X_sub = means[idx]
        assert np.array_equal(_host(m_dev), m_ref)
        W = sg.gen_weights(sg.layer_seed(sg.SEED_W, layer, j), N, K, 0.02)
        Wd = torch.from_numpy(W).cuda()
        # full-token search on the GPU
        s, mse, best = wb.search_scale(Wd, xs_dev[idx], m_dev)
        mse_h, b = _host(mse), int(_host(best)[0])
        assert np.all(np.isfinite(mse_h)) and mse_h[b] <= mse_h[0], name
        # the same search on 512 tokens, against the oracle
        s5, mse5, best5 = wb.search_scale(Wd, torch.from_numpy(X_sub).cuda(), m_dev)
        mse5, b5 = _host(mse5), int(_host(best5)[0])
        ref_mse = np.array([orc.search_mse(W, X_sub, orc.candidate_scales(m_ref, a))
                            for a in orc.ALPHA_GRID])
        assert np.max(np.abs(mse5 - ref_mse) / ref_mse) <= MSE_TOL, name
        rb = int(np.argmin(ref_mse))
        assert b5 == rb or abs(ref_mse[b5] - ref_mse[rb]) <= NEAR_TIE * ref_mse[rb], name
        assert np.array_equal(_host(s5), orc.candidate_scales(m_ref, orc.ALPHA_GRID[b5]))
        # pack with the full-token s
        s_h = _host(s)
        assert np.array_equal(s_h, orc.candidate_scales(m_ref, orc.ALPHA_GRID[b]))
        qw, sc, ze = wb.pack_int4(Wd, s)
        rq, rs, rz = orc.pack_int4(W, s_h)
        qw_h = _host(qw).view(np.uint32)
        sc_h = _host(sc.view(torch.int16)).view(np.uint16)
        ze_h = _host(ze.view(torch.int16)).view(np.uint16)
        assert np.array_equal(qw_h, rq) and np.array_equal(sc_h, rs)
        assert np.array_equal(ze_h, rz), name
        del W, Wd
        # the matmul at M = 1, 16, 64, 256 on sampled outputs
        _, _, Xm, _ = sg.layer_inputs(layer, j, N, K, 0, M=256)
        for M in (1, 16, 64, 256):
            y = _host(wb.w4a16_gemm(torch.from_numpy(Xm[:M]).cuda(), qw, sc, ze))
            ms = np.concatenate([np.repeat(np.arange(M), 64), rng.integers(0, M, 2048)])
            ns = np.concatenate([np.tile(rng.choice(N, 64, replace=False), M),
                                 rng.integers(0, N, 2048)])
            ref = orc.w4a16_pairs(Xm[:M], qw_h, sc_h, ze_h, ms, ns)
            err = np.max(np.abs(y[ms, ns].astype(np.float64) - ref)) / np.max(np.abs(ref))
            assert err <= GEMM_TOL, (name, M, err)
    wb.sync_status()
