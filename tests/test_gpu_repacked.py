"""The repacked decode tiles (awq_repack_int4) and the decode matmul over them
(w4a16_gemm_repacked), through the C ABI.

Bars: the repack is a byte permutation, so its output must equal, bit for
bit, the layout the header defines applied to the oracle's packed words,
scales and zero-points (built here in numpy from that definition); the
matmul must satisfy max|Y - Y_ref| / max|Y_ref| <= 2e-3 against the fp64
oracle on the identical packed weights and fp16 inputs, every output
checked; outputs are poisoned with NaN first."""
import numpy as np
import pytest

import synthgen as sg

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GEMM_TOL = 2e-3
TILE = 1088


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


def rel_err(y, ref):
    return float(np.max(np.abs(y.astype(np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))


def tiles_from_definition(qw, sc, ze):
    """The tile layout written out from its definition: tile (j, g) at byte
    (j G + g) 1088; chunk 32 h + L of 16 bytes = words 16 g + 4 (L % 4) .. +3
    of row 16 j + L / 4 + 8 h; then for r = 0..7 the scale and zero-point of
    rows 16 j + r and 16 j + r + 8; rows past N are zero."""
    N, K8 = qw.shape
    G = K8 // 16
    S = (N + 15) // 16
    q = np.zeros((S * 16, K8), dtype=np.uint32)
    s = np.zeros((S * 16, G), dtype=np.uint16)
    z = np.zeros((S * 16, G), dtype=np.uint16)
    q[:N], s[:N], z[:N] = qw, sc, ze
    q = q.reshape(S, 16, G, 16)
    s = s.reshape(S, 16, G)
    z = z.reshape(S, 16, G)
    out = np.zeros((S, G, TILE), dtype=np.uint8)
    for h in range(2):
        for L in range(32):
            r, w0 = L // 4 + 8 * h, 4 * (L % 4)
            c = 32 * h + L
            out[:, :, 16 * c:16 * c + 16] = np.ascontiguousarray(
                q[:, r, :, w0:w0 + 4]).view(np.uint8).reshape(S, G, 16)
    for r in range(8):
        sz = np.stack([s[:, r], z[:, r], s[:, r + 8], z[:, r + 8]], axis=-1)   # [S, G, 4]
        out[:, :, 1024 + 8 * r:1024 + 8 * r + 8] = sz.view(np.uint8).reshape(S, G, 8)
    return out.reshape(-1)


def _packed(orc, N, K, M, layer=50, seed=0, s=None):
    W, _, X, _ = sg.layer_inputs(layer, seed, N, K, 0, M=M)
    rq, rs, rz = orc.pack_int4(W, s)
    return X, rq, rs, rz


def _dev_packed(rq, rs, rz):
    return dev(rq.view(np.int32)), dev(rs.view(np.float16)), dev(rz.view(np.float16))


@pytest.mark.parametrize("N,K", [(8, 128), (136, 384), (520, 2304), (1024, 1024), (4096, 4096)])
def test_repack_layout_bit_exact(wb, orc, N, K):
    _, rq, rs, rz = _packed(orc, N, K, 1)
    nbytes = wb.lib().awq_repack_int4_bytes(N, K)
    assert nbytes == (N + 15) // 16 * (K // 128) * TILE
    tiles = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")   # poisoned
    wb.repack_int4(*_dev_packed(rq, rs, rz), out=tiles)
    assert np.array_equal(host(tiles), tiles_from_definition(rq, rs, rz))


def _check_repacked(wb, orc, X, rq, rs, rz, tol=GEMM_TOL):
    M, N = X.shape[0], rq.shape[0]
    tiles = wb.repack_int4(*_dev_packed(rq, rs, rz))
    Y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    wb.w4a16_gemm_repacked(dev(X), tiles, N, out=Y)
    y = host(Y)
    assert np.all(np.isfinite(y))
    err = rel_err(y, orc.w4a16_gemm(X, rq, rs, rz))
    assert err <= tol, err
    return y, tiles


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8, 9, 12, 16])
@pytest.mark.parametrize("N,K", [(8, 256), (64, 128), (136, 384), (1024, 1024), (520, 2304)])
def test_repacked_decode_parity(wb, orc, M, N, K):
    X, rq, rs, rz = _packed(orc, N, K, M)
    _check_repacked(wb, orc, X, rq, rs, rz)


def test_repacked_decode_token_columns_independent(wb, orc):
    """The work split depends on N and K only and each output column on its
    own token: token 0 of an 8-token decode equals the 1-token decode, and
    the first 9 tokens of a 16-token decode equal the 9-token decode, bit
    for bit."""
    X, rq, rs, rz = _packed(orc, 2048, 4096, 16, layer=51)
    tiles = wb.repack_int4(*_dev_packed(rq, rs, rz))
    y = {M: host(wb.w4a16_gemm_repacked(dev(X[:M]), tiles, 2048)) for M in (1, 8, 9, 16)}
    assert np.array_equal(y[8][:1].view(np.uint16), y[1].view(np.uint16))
    assert np.array_equal(y[16][:9].view(np.uint16), y[9].view(np.uint16))


@pytest.mark.parametrize("M", [1, 7, 16])
@pytest.mark.parametrize("N,K", [(2384, 256), (2400, 1152), (4752, 384), (3000, 11008)])
def test_repacked_decode_cross_cta_split(wb, orc, M, N, K):
    """149-297 slabs (just over one to two per SM), long and short K: every
    output against the oracle and repeated calls bit-identical."""
    X, rq, rs, rz = _packed(orc, N, K, M, layer=52, seed=1)
    y, tiles = _check_repacked(wb, orc, X, rq, rs, rz)
    x = dev(X)
    for _ in range(3):
        Y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        wb.w4a16_gemm_repacked(x, tiles, N, out=Y)
        assert np.array_equal(host(Y).view(np.uint16), y.view(np.uint16))
    wb.sync_status()


def test_repacked_llama7b_decode_full(wb, orc):
    """LLaMA-7B-shaped decode at M = 1 over the repacked tiles of the GPU's
    own AWQ pack (search on 512 calibration tokens): every output checked."""
    for j, (name, N, K) in enumerate(sg.LLAMA7B_DECODE_PROJ):
        W, Xc, Xm, _ = sg.layer_inputs(0, j, N, K, 512, M=1)
        m = wb.act_mean(wb.act_stats(dev(Xc)), 512)
        s, _, _ = wb.search_scale(dev(W), dev(Xc), m)
        qw, sc, ze = wb.pack_int4(dev(W), s)
        tiles = wb.repack_int4(qw, sc, ze)
        rq, rs, rz = orc.pack_int4(W, host(s))
        assert np.array_equal(host(tiles), tiles_from_definition(rq, rs, rz)), name
        Y = torch.full((1, N), float("nan"), dtype=torch.float16, device="cuda")
        wb.w4a16_gemm_repacked(dev(Xm), tiles, N, out=Y)
        assert rel_err(host(Y), orc.w4a16_gemm(Xm, rq, rs, rz)) <= GEMM_TOL, name
        wb.sync_status()


@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_repacked_llama13b_small_batch_full(wb, orc, M):
    """LLaMA-13B-shaped gate+up (27648 x 5120) and down (5120 x 13824) at
    M = 1, 4, 8, 16, every output; M = 16 on the down projection exceeds
    shared memory for staged activations and takes the L1 path."""
    for j, (name, N, K) in enumerate(sg.LLAMA13B_DECODE_PROJ):
        W, _, Xm, _ = sg.layer_inputs(1, j, N, K, 0, M=M)
        rq, rs, rz = orc.pack_int4(W)
        del W
        _check_repacked(wb, orc, Xm, rq, rs, rz)


def test_repacked_fused_input_scaling(wb, orc):
    """inv_s given: the result equals the repacked decode of the oracle's
    scaled activations fp16(fp32(X) * inv_s), bit for bit."""
    N, K = 520, 2304
    W, Xc, X, _ = sg.layer_inputs(53, 0, N, K, 64, M=16)
    m = orc.act_mean(orc.act_stats(Xc), 64)
    s = orc.candidate_scales(m, 0.45)
    inv = (np.float32(1) / s).astype(np.float32)
    rq, rs, rz = orc.pack_int4(W, s)
    tiles = wb.repack_int4(*_dev_packed(rq, rs, rz))
    for M in (1, 5, 9, 16):
        Xs = orc.scale_activations(X[:M], inv)
        y_fused = host(wb.w4a16_gemm_repacked(dev(X[:M]), tiles, N, inv_s=dev(inv)))
        y_plain = host(wb.w4a16_gemm_repacked(dev(Xs.view(np.float16)), tiles, N))
        assert np.array_equal(y_fused.view(np.uint16), y_plain.view(np.uint16))
        assert rel_err(y_fused, orc.w4a16_gemm(Xs, rq, rs, rz)) <= GEMM_TOL


def test_repacked_chain_early_weights(wb, orc):
    """Back-to-back repacked decodes with early weight fetches enabled, three
    rounds: every output against the oracle."""
    layers = []
    for j, (N, K, M) in enumerate([(1024, 1024, 1), (520, 2304, 3), (2048, 4096, 1),
                                   (4096, 11008, 8), (136, 384, 16)]):
        X, rq, rs, rz = _packed(orc, N, K, M, layer=54, seed=j)
        tiles = wb.repack_int4(*_dev_packed(rq, rs, rz))
        layers.append((dev(X), tiles, N, orc.w4a16_gemm(X, rq, rs, rz)))
    torch.cuda.synchronize()
    wb.set_weight_prefetch(True)
    try:
        for _ in range(3):
            outs = [wb.w4a16_gemm_repacked(x, t, N) for (x, t, N, _) in layers]
            for y, layer in zip(outs, layers):
                assert rel_err(host(y), layer[3]) <= GEMM_TOL
        wb.sync_status()
    finally:
        wb.set_weight_prefetch(False)


def test_repacked_empty_and_strided(wb, orc):
    X, rq, rs, rz = _packed(orc, 256, 512, 5, layer=55)
    tiles = wb.repack_int4(*_dev_packed(rq, rs, rz))
    assert wb.w4a16_gemm_repacked(dev(X[:0]), tiles, 256).shape == (0, 256)
    big = torch.zeros((5, 640), dtype=torch.float16, device="cuda")
    big[:, :512] = dev(X)
    y = host(wb.w4a16_gemm_repacked(big[:, :512], tiles, 256))
    assert rel_err(y, orc.w4a16_gemm(X, rq, rs, rz)) <= GEMM_TOL


# ------------------------------------------------------------- 3 bits ----

TILE3 = 832


def tiles3_from_definition(planes, sc, ze):
    """The 3-bit tile layout from its definition: tile (j, g) at byte
    (j G + g) 832; row r's plane words 12 g .. 12 g + 11 at 48 r; then the
    scale and zero-point block of the 4-bit tile; rows past N zero."""
    N, W3 = planes.shape
    G = W3 // 12
    S = (N + 15) // 16
    pl = np.zeros((S * 16, W3), dtype=np.uint32)
    s = np.zeros((S * 16, G), dtype=np.uint16)
    z = np.zeros((S * 16, G), dtype=np.uint16)
    pl[:N], s[:N], z[:N] = planes, sc, ze
    pl = pl.reshape(S, 16, G, 12)
    s = s.reshape(S, 16, G)
    z = z.reshape(S, 16, G)
    out = np.zeros((S, G, TILE3), dtype=np.uint8)
    out[:, :, :768] = np.ascontiguousarray(pl.transpose(0, 2, 1, 3)).view(np.uint8).reshape(S, G, 768)
    for r in range(8):
        sz = np.stack([s[:, r], z[:, r], s[:, r + 8], z[:, r + 8]], axis=-1)
        out[:, :, 768 + 8 * r:768 + 8 * r + 8] = sz.view(np.uint8).reshape(S, G, 8)
    return out.reshape(-1)


@pytest.mark.parametrize("N,K", [(8, 128), (136, 384), (520, 2304), (4096, 4096)])
def test_repack3_layout_bit_exact(wb, orc, N, K):
    W, _, _, _ = sg.layer_inputs(56, 0, N, K, 0)
    rp, rs, rz = orc.pack_int3(W)
    nbytes = wb.lib().awq_repack_int3_bytes(N, K)
    assert nbytes == (N + 15) // 16 * (K // 128) * TILE3
    tiles = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    wb.repack_int3(dev(rp.view(np.int32)), dev(rs.view(np.float16)), dev(rz.view(np.float16)),
                   out=tiles)
    assert np.array_equal(host(tiles), tiles3_from_definition(rp, rs, rz))


def _check_repacked3(wb, orc, X, rp, rs, rz):
    M, N = X.shape[0], rp.shape[0]
    tiles = wb.repack_int3(dev(rp.view(np.int32)), dev(rs.view(np.float16)),
                           dev(rz.view(np.float16)))
    Y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    wb.w3a16_gemm_repacked(dev(X), tiles, N, out=Y)
    y = host(Y)
    assert np.all(np.isfinite(y))
    err = rel_err(y, orc.w3a16_gemm(X, rp, rs, rz))
    assert err <= GEMM_TOL, err
    return y, tiles


@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 16])
@pytest.mark.parametrize("N,K", [(8, 256), (136, 384), (1024, 1024), (520, 2304), (2400, 1152)])
def test_repacked3_decode_parity(wb, orc, M, N, K):
    W, _, X, _ = sg.layer_inputs(57, 0, N, K, 0, M=M)
    rp, rs, rz = orc.pack_int3(W)
    _check_repacked3(wb, orc, X, rp, rs, rz)


def test_repacked3_llama7b_qkv_and_long_k(wb, orc):
    """The LLaMA-7B qkv projection at M = 1 over the GPU's own 3-bit pack,
    and M = 16 with K = 13824, where the activations do not fit in shared
    memory and are read through L1."""
    W, _, X, _ = sg.layer_inputs(0, 0, 12288, 4096, 0, M=1)
    pl, sc, ze = wb.pack_int3(dev(W))
    rp, rs, rz = orc.pack_int3(W)
    assert np.array_equal(host(pl).view(np.uint32), rp)
    _check_repacked3(wb, orc, X, rp, rs, rz)
    W, _, X, _ = sg.layer_inputs(58, 0, 136, 13824, 0, M=16)
    rp, rs, rz = orc.pack_int3(W)
    _check_repacked3(wb, orc, X, rp, rs, rz)
    wb.sync_status()
