"""Pins of the CPU oracle against facts fixed outside the oracle itself:
the IEEE 754 binary16 format, exact rational arithmetic, closed forms,
library routines (numpy matmul / argmin), brute force over the 16 levels,
and invariants the AWQ pages state ("AWQ: Activation-aware Weight
Quantization ...", fdeinterviews.com/papers/awq, third paragraph: scaling a
weight channel by s and its input by 1/s leaves the output unchanged;
s = average activation magnitude ** alpha).  No GPU needed."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import synthgen as sg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- fp16 ----

def test_fp16_h2d_all_patterns(oracle_mod):
    """Every finite fp16 pattern widens exactly (numpy's binary16 as the
    reference); NaN patterns give NaN."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle_mod.h2d(bits)
    ref = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_fp16_golden_constants(oracle_mod):
    """Named binary16 encodings from the IEEE 754 standard."""
    path = os.path.join(GOLDEN, "fp16_constants.txt")
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        val, bits, kind = line.split()
        v = float(Fraction(val))
        assert oracle_mod.d2h_rn(v) == int(bits, 16), line
        if kind == "exact":
            assert oracle_mod.h2d(np.array([int(bits, 16)], dtype=np.uint16))[0] == v
        n += 1
    assert n >= 10


def test_fp16_rounding_ties_and_random(oracle_mod):
    """Round-to-nearest-even at every exact midpoint between neighbouring
    finite fp16 values, just either side of it, and on random doubles over
    the whole range; numpy's float64->float16 conversion is the reference."""
    pos = np.arange(0, 0x7BFF, dtype=np.uint16)          # 0 .. below max
    lo = pos.view(np.float16).astype(np.float64)
    hi = (pos + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2                                    # exact in fp64
    cases = [mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf)]
    r = _rng(1)
    cases.append(r.standard_normal(2_000_000) * np.exp2(r.integers(-30, 17, 2_000_000)))
    cases.append(np.array([65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25, 2.0 ** -26,
                           3 * 2.0 ** -25, 2.0 ** -14 - 2.0 ** -25]))
    for c in cases:
        x = np.concatenate([c, -c])
        got = oracle_mod.d2h_array(x)
        with np.errstate(over="ignore"):        # values past 65520 round to inf
            ref = x.astype(np.float16).view(np.uint16)
        assert np.array_equal(got, ref)


def test_fp16_fp32_inputs_dense_sample(oracle_mod):
    """fp32 inputs (what the quantiser rounds) around every binary16 binade:
    all 2^16 low-mantissa patterns of 2^12 fp32 top halves."""
    r = _rng(2)
    tops = r.integers(0x3000, 0x4800, 4096, dtype=np.uint32)   # exponents near fp16 range
    lows = np.arange(1 << 16, dtype=np.uint32)
    f32 = ((tops[:, None] << 16) | lows[None, :]).ravel().view(np.float32)
    got = oracle_mod.d2h_array(f32.astype(np.float64))
    with np.errstate(over="ignore"):            # the top binades round to inf
        ref = f32.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------- step a1 stats ---

def test_act_stats_bruteforce_fractions(oracle_mod):
    """Sum of |x| is exact: compare with Fraction arithmetic on the exact
    fp16 values, including subnormals and the largest finite value."""
    r = _rng(3)
    T, K = 7, 16
    bits = r.integers(0, 0x7BFF, (T, K)).astype(np.uint16)
    bits[0, 0] = 0x0001          # least subnormal
    bits[1, 0] = 0x7BFF          # 65504
    bits[2, :] |= 0x8000         # negative values count by magnitude
    got = oracle_mod.act_stats(bits)
    vals = bits.view(np.float16).astype(np.float64)
    for k in range(K):
        exact = sum(Fraction(abs(v)) for v in vals[:, k]) * (1 << 24)
        assert exact.denominator == 1
        assert got[k] == exact.numerator
    m = oracle_mod.act_mean(got, T)
    for k in range(K):
        assert m[k] == float(Fraction(int(got[k]), (1 << 24) * T))   # correctly rounded


def test_act_stats_order_independent_and_streamed(oracle_mod):
    """Only statistics are collected (pages, seventh paragraph): permuting the
    tokens or splitting them into streamed batches changes nothing."""
    _, X, _, _ = sg.layer_inputs(0, 1, 8, 256, 300)
    a = oracle_mod.act_stats(X)
    perm = _rng(4).permutation(X.shape[0])
    assert np.array_equal(a, oracle_mod.act_stats(X[perm]))
    part = oracle_mod.act_stats(X[:123])
    assert np.array_equal(a, oracle_mod.act_stats(X[123:], part))
    # mean |x| of N(0,1) is sqrt(2/pi); outlier channels are 20x that
    m = oracle_mod.act_mean(a, X.shape[0])
    ch = sg.outlier_channels(sg.layer_seed(sg.SEED_CHANNELS, 0, 1), 256)
    rest = np.setdiff1d(np.arange(256), ch)
    assert abs(m[rest].mean() - math.sqrt(2 / math.pi)) < 0.02
    assert abs(m[ch].mean() / m[rest].mean() - 20) < 2


def test_act_stats_nonfinite_rejected(oracle_mod):
    X = np.zeros((2, 8), dtype=np.uint16)
    X[1, 3] = 0x7C00
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.act_stats(X)


# ---------------------------------------------- step a2 candidate scales ---

def test_candidate_scales_alpha_zero_is_one(oracle_mod):
    m = np.abs(_rng(5).standard_normal(1024)) + 1e-3
    s = oracle_mod.candidate_scales(m, 0.0)
    assert s.dtype == np.float32 and np.all(s == 1.0)


def test_candidate_scales_power_law_and_centre(oracle_mod):
    """s_i / s_j = (m_i / m_j)^alpha and sqrt(max s * min s) = 1, up to the
    final fp32 rounding; zero channels are floored at 1e-4."""
    r = _rng(6)
    m = np.exp(r.uniform(-3, 3, 2048))
    m[7] = 0.0
    for alpha in (0.05, 0.35, 0.5, 0.95, 1.0):
        s = oracle_mod.candidate_scales(m, alpha).astype(np.float64)
        mm = np.maximum(m, 1e-4)
        i, j = r.integers(0, 2048, 500), r.integers(0, 2048, 500)
        ratio = s[i] / s[j]
        ref = np.exp(alpha * (np.log(mm[i]) - np.log(mm[j])))
        assert np.max(np.abs(ratio / ref - 1)) < 4e-7
        assert abs(math.sqrt(s.max() * s.min()) - 1) < 2e-7
        if alpha > 0:
            order = np.argsort(mm, kind="stable")
            assert np.all(np.diff(s[order]) >= 0)       # monotone in m


def test_candidate_scales_constant_channels(oracle_mod):
    for c in (1e-6, 0.3, 7.0):
        s = oracle_mod.candidate_scales(np.full(256, c), 0.7)
        assert np.all(s == 1.0)


# ----------------------------------------------------- steps a3/a5 quant ---

def _wprime(W16, s):
    """w' = fp32(W * s): numpy's IEEE fp32 multiply (independent route)."""
    w = W16.astype(np.float32)
    return w if s is None else (w * s.astype(np.float32)).astype(np.float32)


def _check_nearest(oracle_mod, W16, s, bits=4):
    qmax = (1 << bits) - 1
    q, sc, ze = oracle_mod.quantize(W16, s, bits)
    N, K = W16.shape
    G = K // 128
    wp = _wprime(W16, s).astype(np.float64)
    scale = np.repeat(sc.view(np.float16).astype(np.float64), 128, axis=1)
    z = np.repeat(ze.view(np.float16).astype(np.float64), 128, axis=1)
    assert np.all(z == np.round(z)) and np.all((z >= 0) & (z <= qmax))
    assert int(q.max()) <= qmax
    # brute force: distance to each of the 2^bits levels
    levels = (np.arange(qmax + 1)[None, None, :] - z[..., None]) * scale[..., None]
    dist = np.abs(levels - wp[..., None])
    best = dist.min(axis=2)
    mine = np.take_along_axis(dist, q[..., None].astype(np.int64), axis=2)[..., 0]
    # q must be a nearest level; a miss is only allowed at an exact midpoint
    # whose fp32 quotient rounded across .5 (counted, expected ~0)
    miss = mine > best
    n_miss = int(miss.sum())
    assert n_miss <= max(2, q.size // 100000), n_miss
    if n_miss:
        assert np.all(mine[miss] - best[miss] <= scale[miss] * 2.0 ** -20)
    # half-step bound for unclamped, just over one step for clamped elements
    deq = (q.astype(np.float64) - z) * scale
    err = np.abs(deq - wp)
    t = np.rint(wp / scale) + z
    unclamped = (t >= 0) & (t <= qmax)
    assert np.all(err[unclamped] <= scale[unclamped] / 2 * (1 + 2.0 ** -20))
    assert np.all(err[~unclamped] <= scale[~unclamped] * (1 + 2.0 ** -10))
    return q, sc, ze


def test_quantizer_nearest_level_bruteforce(oracle_mod):
    W, _, _, _ = sg.layer_inputs(0, 2, 64, 512, 0)
    _check_nearest(oracle_mod, W, None)
    s = np.exp(_rng(7).uniform(-1.5, 1.5, 512)).astype(np.float32)
    _check_nearest(oracle_mod, W, s)


def test_quantizer_edge_groups(oracle_mod):
    """Constant, all-zero, tiny, huge, single-outlier and one-signed groups."""
    K = 128
    rows = [np.zeros(K), np.full(K, 0.25), np.full(K, -3.0),
            np.linspace(-1e-6, 1e-6, K), np.linspace(-6e4, 6e4, K),
            np.r_[np.zeros(K - 1), 5.0], np.linspace(0.5, 2.0, K),
            np.linspace(-2.0, -0.5, K)]
    W = np.stack(rows).astype(np.float16)
    q, sc, ze = oracle_mod.quantize(W)
    scale = sc.view(np.float16).astype(np.float64)[:, 0]
    z = ze.view(np.float16).astype(np.float64)[:, 0]
    assert np.all(scale >= 2.0 ** -14)
    assert scale[0] == 2.0 ** -14 and z[0] == 0 and np.all(q[0] == 0)   # zeros stay 0
    # zero-points are the integers 0..15 in fp16, +0.0 for zero (never -0.0)
    allowed = {oracle_mod.d2h_rn(float(v)) for v in range(16)}
    assert 0x0000 in allowed and 0x8000 not in allowed
    assert set(np.unique(ze).tolist()) <= allowed
    # one-signed groups: zero-point clamps, levels still ordered with w
    for r in (6, 7):
        assert np.all(np.diff(q[r].astype(int)) >= 0)
    _check_nearest(oracle_mod, W[3:6], None)


def _golden_groups():
    """Lines of the hand-derived group fixture: (bits, group weights, scale
    bits, zero-point, [(position, level), ...])."""
    out = []
    for line in open(os.path.join(GOLDEN, "quant_groups.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        head, vals, levels = line.split("|")
        bits, fill = head.split()
        vals, expect = vals.split("->")
        ws = [float(v) for v in vals.split()]
        sc_bits, zero = expect.split()
        qs = [int(v) for v in levels.split()]
        assert len(qs) == len(ws)
        g = np.full(128, float(fill))
        g[:len(ws)] = ws
        assert np.array_equal(g.astype(np.float16).astype(np.float64), g)   # exact in fp16
        out.append((int(bits), g.astype(np.float16)[None, :], int(sc_bits, 16), int(zero),
                    list(enumerate(qs))))
    return out


def test_quantizer_golden_groups(oracle_mod):
    """Stored scale, zero-point and levels of hand-derived groups
    (tests/golden/quant_groups.txt): the scale is the NEAREST fp16 to
    range/qmax (lines where truncation, or rounding up, gives another fp16,
    one of them crossing a binade), the zero-point is rint of -lo/scale (lines
    where floor, ceil, or ties away from zero give another integer), and the
    clamps of a one-signed group; at 4 and 3 bits."""
    groups = _golden_groups()
    assert len(groups) >= 8 and {b for b, *_ in groups} == {3, 4}
    for bits, w, sc_bits, zero, levels in groups:
        q, sc, ze = oracle_mod.quantize(w, None, bits=bits)
        assert int(sc[0, 0]) == sc_bits, (bits, w[0, :4], hex(int(sc[0, 0])))
        assert ze.view(np.float16)[0, 0] == zero and int(ze[0, 0]) == oracle_mod.d2h_rn(zero)
        for pos, lev in levels:
            assert int(q[0, pos]) == lev, (bits, w[0, pos], int(q[0, pos]), lev)


def test_quantizer_nonfinite_rejected(oracle_mod):
    W = np.zeros((1, 128), dtype=np.float16)
    W[0, 5] = np.inf
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.quantize(W)


def _grid_aligned(rng, N, K, bits=4):
    """Weights that lie exactly on a 2^bits-level grid spanning levels
    0..2^bits - 1, with power-of-two scales and per-channel power-of-two s:
    the quantiser must return exactly that grid."""
    qmax = (1 << bits) - 1
    G = K // 128
    q = rng.integers(0, qmax + 1, (N, K))
    q[:, ::128] = 0
    q[:, 1::128] = qmax
    z = rng.integers(0, qmax + 1, (N, G))
    scale = np.exp2(rng.integers(-9, -4, (N, G))).astype(np.float64)
    s = np.exp2(rng.integers(-2, 3, K)).astype(np.float32)
    wp = (q - np.repeat(z, 128, axis=1)) * np.repeat(scale, 128, axis=1)
    W = (wp / s.astype(np.float64)).astype(np.float16)
    assert np.array_equal(W.astype(np.float64) * s, wp)       # exact by construction
    return W, s, q, z, scale


def test_quantizer_grid_aligned_exact(oracle_mod):
    W, s, q0, z0, scale0 = _grid_aligned(_rng(8), 16, 512)
    q, sc, ze = oracle_mod.quantize(W, s)
    assert np.array_equal(q, q0)
    assert np.array_equal(ze.view(np.float16).astype(np.float64), z0)
    assert np.array_equal(sc.view(np.float16).astype(np.float64), scale0)


def test_alpha_zero_is_plain_rtn(oracle_mod):
    """alpha = 0 gives s = 1, i.e. plain round-to-nearest ("plain rounding",
    the baseline the pages compare against)."""
    W, X, _, _ = sg.layer_inputs(1, 0, 32, 256, 64)
    m = oracle_mod.act_mean(oracle_mod.act_stats(X), 64)
    s0 = oracle_mod.candidate_scales(m, 0.0)
    a = oracle_mod.quantize(W, s0)
    b = oracle_mod.quantize(W, None)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_normaliser_power_of_two_invariance(oracle_mod):
    """Dividing s by a power of two leaves levels and zero-points unchanged,
    scales the stored scale exactly, and leaves the search residual (hence
    the MSE) bit-identical: the normaliser is free."""
    W, X, _, _ = sg.layer_inputs(1, 1, 32, 256, 64)
    m = oracle_mod.act_mean(oracle_mod.act_stats(X), 64)
    s = oracle_mod.candidate_scales(m, 0.5)
    for c in (0.5, 2.0, 4.0):
        q1, sc1, ze1 = oracle_mod.quantize(W, s)
        q2, sc2, ze2 = oracle_mod.quantize(W, (s * np.float32(c)).astype(np.float32))
        assert np.array_equal(q1, q2) and np.array_equal(ze1, ze2)
        assert np.array_equal(sc1.view(np.float16).astype(np.float64) * c,
                              sc2.view(np.float16).astype(np.float64))
        e1 = oracle_mod.search_residual(W, s)
        e2 = oracle_mod.search_residual(W, (s * np.float32(c)).astype(np.float32))
        assert np.array_equal(e1, e2)


# ------------------------------------------------------------ packing -----

def test_pack_layout_golden(oracle_mod):
    """The packed-word layout fixture: element k of a row sits in word k/8,
    bits 4*(k%8)..4*(k%8)+3."""
    path = os.path.join(GOLDEN, "pack_layout.txt")
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        levels, words = line.split("->")
        q = np.array([int(v) for v in levels.split()], dtype=np.uint8)[None, :]
        w = np.array([int(v, 16) for v in words.split()], dtype=np.uint32)[None, :]
        assert np.array_equal(oracle_mod.pack_nibbles(q), w)
        assert np.array_equal(oracle_mod.unpack_nibbles(w, q.shape[1]), q)
        n += 1
    assert n >= 3


def test_pack_unpack_roundtrip(oracle_mod):
    r = _rng(9)
    q = r.integers(0, 16, (33, 256)).astype(np.uint8)
    assert np.array_equal(oracle_mod.unpack_nibbles(oracle_mod.pack_nibbles(q), 256), q)
    words = r.integers(0, 1 << 32, (17, 64), dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(oracle_mod.pack_nibbles(oracle_mod.unpack_nibbles(words, 512)), words)


def test_packed_bytes_quarter_of_fp16(oracle_mod):
    """4 bits per weight: a quarter of the fp16 bytes, plus 4 bytes of
    scale/zero per group of 128 (the pages: roughly 4x less weight memory than fp16)."""
    W, _, _, _ = sg.layer_inputs(0, 3, 64, 1024, 0)
    qw, sc, ze = oracle_mod.pack_int4(W)
    assert qw.nbytes * 4 == W.nbytes
    assert sc.nbytes + ze.nbytes == 4 * 64 * 1024 // 128


# ---------------------------------------------------------- matmul -------

def test_scaling_invariance_identity(oracle_mod):
    """(W diag(s)) (diag(s)^-1 X) = W X to fp64 rounding, before any
    quantisation (pages, third paragraph)."""
    r = _rng(10)
    W = r.standard_normal((48, 256)) * 0.02
    X = r.standard_normal((9, 256))
    s = np.exp(r.uniform(-2, 2, 256))
    y0 = oracle_mod.linear(X, W)
    y1 = oracle_mod.linear(X / s, W * s)
    assert np.max(np.abs(y1 - y0)) <= 1e-13 * np.max(np.abs(y0))


def test_gemm_routes_agree(oracle_mod):
    """The matmul step (numpy fp64 on the dequantised matrix) agrees with the
    sampled-pair route (plain C loops straight from the packed words)."""
    W, _, X, _ = sg.layer_inputs(2, 0, 96, 384, 0, M=5)
    qw, sc, ze = oracle_mod.pack_int4(W)
    Y = oracle_mod.w4a16_gemm(X, qw, sc, ze)
    mm, nn = np.meshgrid(np.arange(5), np.arange(96), indexing="ij")
    Yp = oracle_mod.w4a16_pairs(X, qw, sc, ze, mm.ravel(), nn.ravel()).reshape(5, 96)
    assert np.max(np.abs(Y - Yp)) <= 1e-12 * np.max(np.abs(Y))


def test_gemm_single_group_closed_form(oracle_mod):
    """X nonzero in one group only, every level one step above the zero-point,
    scale 2^-8: then Y[m,n] = 2^-8 * sum of that group's x, exactly."""
    K, N = 512, 8
    q = np.full((N, K), 6, dtype=np.uint8)
    qw = oracle_mod.pack_nibbles(q)
    sc = np.full((N, 4), 0x1C00, dtype=np.uint16)           # 2^-8
    ze = np.full((N, 4), oracle_mod.d2h_rn(5.0), dtype=np.uint16)
    X = np.zeros((3, K), dtype=np.float16)
    r = _rng(11)
    X[:, 256:384] = r.standard_normal((3, 128)).astype(np.float16)
    Y = oracle_mod.w4a16_gemm(X, qw, sc, ze)
    ref = X.astype(np.float64)[:, 256:384].sum(axis=1) * 2.0 ** -8
    assert np.array_equal(Y, np.repeat(ref[:, None], N, axis=1))


# ---------------------------------------------------------- search -------

def test_search_mse_equals_output_mse(oracle_mod):
    """The residual route ||X E^T||^2/(TN) equals the output MSE of
    Q(W diag(s)) diag(s)^-1 X against W X computed from the two layers'
    outputs (a different formula)."""
    W, X, _, _ = sg.layer_inputs(3, 0, 40, 256, 33)
    m = oracle_mod.act_mean(oracle_mod.act_stats(X), 33)
    s = oracle_mod.candidate_scales(m, 0.45)
    mse = oracle_mod.search_mse(W, X, s)
    q, sc, ze = oracle_mod.quantize(W, s)
    deq = oracle_mod.dequant(q, sc, ze)
    X64 = X.astype(np.float64)
    Yq = oracle_mod.linear(X64 / s.astype(np.float64), deq)     # Q(W s) (X / s)
    Yf = oracle_mod.linear(X64, W.astype(np.float64))
    ref = np.mean((Yq - Yf) ** 2)
    assert abs(mse - ref) <= 1e-12 * ref


def test_search_mse_bruteforce_exact_tiny(oracle_mod):
    """N=2, K=128, T=4: exact rational MSE by enumeration of every term."""
    W, X, _, _ = sg.layer_inputs(4, 0, 2, 128, 4)
    s = np.exp(_rng(12).uniform(-1, 1, 128)).astype(np.float32)
    q, sc, ze = oracle_mod.quantize(W, s)
    Wv = [[Fraction(float(v)) for v in row] for row in W.astype(np.float64)]
    Xv = [[Fraction(float(v)) for v in row] for row in X.astype(np.float64)]
    sv = [Fraction(float(v)) for v in s.astype(np.float64)]
    scale = [Fraction(float(v)) for v in sc.view(np.float16).astype(np.float64)[:, 0]]
    zero = [Fraction(float(v)) for v in ze.view(np.float16).astype(np.float64)[:, 0]]
    total = Fraction(0)
    for t in range(4):
        for n in range(2):
            yq = sum((int(q[n, k]) - zero[n]) * scale[n] * Xv[t][k] / sv[k] for k in range(128))
            yf = sum(Wv[n][k] * Xv[t][k] for k in range(128))
            total += (yq - yf) ** 2
    exact = float(total / 8)
    assert abs(oracle_mod.search_mse(W, X, s) - exact) <= 1e-13 * exact


def test_search_grid_aligned_zero_mse(oracle_mod):
    """Weights already on the quantisation grid of W diag(s) lose nothing:
    the residual and the MSE are exactly zero."""
    W, s, _, _, _ = _grid_aligned(_rng(13), 8, 256)
    X = sg.gen_acts(5, 16, 256)
    assert oracle_mod.search_mse(W, X, s) == 0.0


def test_search_scale_picks_argmin(oracle_mod):
    """alpha* is numpy's first argmin of the MSE vector; mse(alpha*) <=
    mse(0) = plain RTN; on outlier activations scaling helps (alpha* > 0)."""
    W, X, _, _ = sg.layer_inputs(5, 0, 128, 512, 128)
    m = oracle_mod.act_mean(oracle_mod.act_stats(X), 128)
    s_best, mse, best = oracle_mod.search_scale(W, X, m)
    assert best == int(np.argmin(mse))
    assert mse[best] <= mse[0]
    assert mse[0] == oracle_mod.search_mse(W, X, None)
    assert np.array_equal(s_best, oracle_mod.candidate_scales(m, oracle_mod.ALPHA_GRID[best]))
    assert best > 0 and mse[best] < 0.8 * mse[0]


def test_search_tie_goes_to_lowest_alpha(oracle_mod):
    """Equal MSE for every alpha (all channels alike, so s = 1 for all):
    the lowest index wins."""
    W, _, _, _ = sg.layer_inputs(6, 0, 16, 256, 0)
    X = sg.gen_acts(9, 8, 256)
    m = np.full(256, 0.8)
    _, mse, best = oracle_mod.search_scale(W, X, m, alphas=(0.3, 0.1, 0.2))
    assert mse[0] == mse[1] == mse[2] and best == 0


def test_scale_activations_independent_route(oracle_mod):
    """The matmul's input scaling fp16(fp32(x * inv_s)): numpy's IEEE float32
    multiply and float16 conversion give the same bits."""
    rng = np.random.default_rng(21)
    X = (rng.standard_normal((7, 384)) * 3).astype(np.float16)
    X[0, :5] = [0.0, -0.0, 65504.0, -6.1e-5, 1e-7]
    inv = np.exp(rng.uniform(-3, 3, 384)).astype(np.float32)
    got = oracle_mod.scale_activations(X, inv)
    with np.errstate(over="ignore"):
        ref = (X.astype(np.float32) * inv[None, :]).astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------- 3-bit variant ----
# The pages evaluate the method at 3 and 4 bits (fourth paragraph) and call
# 3 bits possible with a noticeable gap (last paragraph).  The 3-bit
# quantiser is the 4-bit one with levels 0..7; these pins hold it to the
# same facts.

def test_int3_nearest_level_bruteforce(oracle_mod):
    W, _, _, _ = sg.layer_inputs(0, 3, 64, 512, 0)
    _check_nearest(oracle_mod, W, None, bits=3)
    s = np.exp(_rng(17).uniform(-1.5, 1.5, 512)).astype(np.float32)
    _check_nearest(oracle_mod, W, s, bits=3)


def test_int3_grid_aligned_exact(oracle_mod):
    W, s, q0, z0, scale0 = _grid_aligned(_rng(18), 16, 512, bits=3)
    q, sc, ze = oracle_mod.quantize(W, s, bits=3)
    assert np.array_equal(q, q0)
    assert np.array_equal(ze.view(np.float16).astype(np.float64), z0)
    assert np.array_equal(sc.view(np.float16).astype(np.float64), scale0)


def test_int3_alpha_zero_is_plain_rtn(oracle_mod):
    W, X, _, _ = sg.layer_inputs(1, 2, 32, 256, 64)
    m = oracle_mod.act_mean(oracle_mod.act_stats(X), 64)
    a = oracle_mod.quantize(W, oracle_mod.candidate_scales(m, 0.0), bits=3)
    b = oracle_mod.quantize(W, None, bits=3)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_int3_step_is_range_over_seven(oracle_mod):
    """One group spanning [-1, 6] in steps of 1: scale 1, zero-point 1, and
    the levels are the values plus one (range / 7 = 1 exactly)."""
    w = np.tile(np.arange(-1, 7, dtype=np.float64), 16)[None, :].astype(np.float16)
    q, sc, ze = oracle_mod.quantize(w, None, bits=3)
    assert sc.view(np.float16)[0, 0] == 1.0 and ze.view(np.float16)[0, 0] == 1.0
    assert np.array_equal(q[0], (w[0].astype(np.float64) + 1).astype(np.uint8))


def test_planes3_layout_golden(oracle_mod):
    """The 3-bit bit-plane fixture: per 32 levels, word p holds bit p of
    level i at bit i."""
    cases = []
    with open(os.path.join(GOLDEN, "planes3_layout.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            cases.append(([(int(k), int(v)) for k, v in (t.split(":") for t in lhs.split())],
                          [int(h, 16) for h in rhs.split()]))
    assert len(cases) >= 5
    for pairs, words in cases:
        q = np.zeros((1, 32), dtype=np.uint8)
        for k, v in pairs:
            q[0, k] = v
        got = oracle_mod.pack_planes3(q)
        assert [int(x) for x in got[0]] == words
        assert np.array_equal(oracle_mod.unpack_planes3(got, 32), q)


def test_planes3_roundtrip(oracle_mod):
    q = _rng(19).integers(0, 8, (5, 384)).astype(np.uint8)
    w = oracle_mod.pack_planes3(q)
    assert w.shape == (5, 384 // 32 * 3)            # exactly 3 bits per level
    assert np.array_equal(oracle_mod.unpack_planes3(w, 384), q)


def test_int3_search_mse_bruteforce_exact_tiny(oracle_mod):
    """N=2, K=128, T=4 at 3 bits: exact rational MSE by enumeration."""
    W, X, _, _ = sg.layer_inputs(4, 1, 2, 128, 4)
    s = np.exp(_rng(20).uniform(-1, 1, 128)).astype(np.float32)
    q, sc, ze = oracle_mod.quantize(W, s, bits=3)
    assert int(q.max()) <= 7
    Wv = [[Fraction(float(v)) for v in row] for row in W.astype(np.float64)]
    Xv = [[Fraction(float(v)) for v in row] for row in X.astype(np.float64)]
    sv = [Fraction(float(v)) for v in s.astype(np.float64)]
    scale = [Fraction(float(v)) for v in sc.view(np.float16).astype(np.float64)[:, 0]]
    zero = [Fraction(float(v)) for v in ze.view(np.float16).astype(np.float64)[:, 0]]
    total = Fraction(0)
    for t in range(4):
        for n in range(2):
            yq = sum((int(q[n, k]) - zero[n]) * scale[n] * Xv[t][k] / sv[k] for k in range(128))
            yf = sum(Wv[n][k] * Xv[t][k] for k in range(128))
            total += (yq - yf) ** 2
    exact = float(total / 8)
    assert abs(oracle_mod.search_mse(W, X, s, bits=3) - exact) <= 1e-13 * exact


# ------------------------------------------------- Gram-matrix search -----
# NEXT row f2: the same objective through G = X^T X, which costs 2 N K^2 per
# alpha instead of 2 T N K (smaller once T > K).

def test_gram_route_equals_output_mse(oracle_mod):
    """||X E^T||_F^2 = tr(E X^T X E^T): the Gram route gives the direct
    output MSE to fp64 rounding, for every alpha and at 3 and 4 bits."""
    W, X, _, _ = sg.layer_inputs(5, 0, 24, 256, 300)
    m = oracle_mod.act_mean(oracle_mod.act_stats(X), 300)
    G = oracle_mod.gram(X)
    assert np.array_equal(G, G.T)
    for bits in (4, 3):
        for a in (0.0, 0.35, 0.95):
            s = oracle_mod.candidate_scales(m, a)
            d = oracle_mod.search_mse(W, X, s, bits=bits)
            g = oracle_mod.search_mse_gram(W, G, 300, s, bits=bits)
            assert abs(g - d) <= 1e-11 * d


def test_gram_route_exact_tiny(oracle_mod):
    """N=2, K=128, T=3: the Gram route against exact rationals."""
    W, X, _, _ = sg.layer_inputs(5, 1, 2, 128, 3)
    s = np.exp(_rng(21).uniform(-1, 1, 128)).astype(np.float32)
    E = oracle_mod.search_residual(W, s)
    Xv = [[Fraction(float(v)) for v in row] for row in X.astype(np.float64)]
    Ev = [[Fraction(float(v)) for v in row] for row in E]
    Gv = [[sum(Xv[t][i] * Xv[t][j] for t in range(3)) for j in range(128)] for i in range(128)]
    total = sum(Ev[n][i] * Gv[i][j] * Ev[n][j] for n in range(2) for i in range(128) for j in range(128))
    exact = float(total / 6)
    g = oracle_mod.search_mse_gram(W, oracle_mod.gram(X), 3, s)
    assert abs(g - exact) <= 1e-12 * exact


def test_w3a16_matches_the_nibble_route(oracle_mod):
    """Levels 0..7 stored as bit planes or as nibbles dequantise to the same
    weights: the 3-bit matmul equals the (pinned) 4-bit one on them."""
    W, _, X, _ = sg.layer_inputs(6, 0, 40, 384, 0, M=5)
    q, sc, ze = oracle_mod.quantize(W, None, bits=3)
    y3 = oracle_mod.w3a16_gemm(X, oracle_mod.pack_planes3(q), sc, ze)
    y4 = oracle_mod.w4a16_gemm(X, oracle_mod.pack_nibbles(q), sc, ze)
    assert np.array_equal(y3, y4)
