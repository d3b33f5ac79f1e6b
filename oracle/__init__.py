"""CPU oracle for the AWQ hot path.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  It never imports or calls the
CUDA library, and the CUDA library never uses it.

Layout: the bit-level steps of the method (fp16 rounding, the INT4
quantiser, packing, statistics, candidate scales) are plain C in
``awq_oracle.c`` (built with ``-ffp-contract=off``, no fast-math); the two
contractions (the dequantised matmul and the search's output MSE) use
numpy's fp64 matmul as a library step on the exact fp64 operands.

Method source: "AWQ: Activation-aware Weight Quantization for On-Device LLM
Compression and Acceleration" (fdeinterviews.com/papers/awq), third
paragraph (scaling trick, s = average activation magnitude ** alpha, alpha
by grid search on a calibration set, every weight in low bits), seventh
paragraph (only activation statistics are collected), fourth and last
paragraphs (evaluated at 3 and 4 bits; 4 bits the default).  Group size 128, asymmetric fp16 scale/zero, mean |x|, output MSE
and the 20-point alpha grid are the workload definition, not the pages'.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

GROUP = 128
ALPHA_GRID = tuple(i / 20.0 for i in range(20))  # {0, 0.05, ..., 0.95}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "awq_oracle.c")
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_LIB = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build() -> str:
    """Compile the C oracle in-tree (idempotent); returns the .so path."""
    if os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    tmp = _SO + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-ffp-contract=off", "-fno-fast-math", "-Wall",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(build())
        lib.awqo_h2d.argtypes = [ctypes.c_uint16]
        lib.awqo_h2d.restype = ctypes.c_double
        lib.awqo_d2h_rn.argtypes = [ctypes.c_double]
        lib.awqo_d2h_rn.restype = ctypes.c_uint16
        lib.awqo_act_stats.argtypes = [_ptr, _i64, _i64, _i64, ctypes.c_int, _ptr]
        lib.awqo_act_mean.argtypes = [_ptr, _i64, _i64, _ptr]
        lib.awqo_candidate_scales.argtypes = [_ptr, _i64, ctypes.c_double, _ptr]
        lib.awqo_quantize.argtypes = [_ptr, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr]
        lib.awqo_quantize_bits.argtypes = [_ptr, _i64, _i64, _i64, _ptr, ctypes.c_int, _ptr,
                                           _ptr, _ptr]
        lib.awqo_pack_planes3.argtypes = [_ptr, _i64, _i64, _ptr]
        lib.awqo_unpack_planes3.argtypes = [_ptr, _i64, _i64, _ptr]
        lib.awqo_pack_nibbles.argtypes = [_ptr, _i64, _i64, _ptr]
        lib.awqo_unpack_nibbles.argtypes = [_ptr, _i64, _i64, _ptr]
        lib.awqo_dequant.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _ptr]
        lib.awqo_search_residual.argtypes = [_ptr, _i64, _i64, _i64, _ptr, _ptr, _ptr,
                                             _ptr, _ptr]
        lib.awqo_h2d_array.argtypes = [_ptr, _i64, _ptr]
        lib.awqo_d2h_array.argtypes = [_ptr, _i64, _ptr]
        lib.awqo_w4a16_pairs.argtypes = [_ptr, _i64, _i64, _ptr, _ptr, _ptr, _i64,
                                         _ptr, _ptr, _ptr]
        lib.awqo_scale_activations.argtypes = [_ptr, _i64, _i64, _ptr, _ptr]
        _LIB = lib
    return _LIB


class OracleError(RuntimeError):
    pass


def _bits(a: np.ndarray) -> np.ndarray:
    """fp16 array (or uint16 bit patterns) -> contiguous uint16 bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected fp16 or uint16 bits, got {a.dtype}")
    return a


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


# ---- fp16 --------------------------------------------------------------

def h2d(bits: np.ndarray) -> np.ndarray:
    """Exact fp64 value of fp16 bit patterns."""
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _lib().awqo_h2d_array(_p(b), b.size, _p(out))
    return out


def d2h_rn(x: float) -> int:
    """Bits of the fp16 nearest to ``x`` (ties to even)."""
    return int(_lib().awqo_d2h_rn(float(x)))


def d2h_array(x: np.ndarray) -> np.ndarray:
    """fp16 bits nearest to each fp64 value (ties to even)."""
    xx = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(xx.shape, dtype=np.uint16)
    _lib().awqo_d2h_array(_p(xx), xx.size, _p(out))
    return out


# ---- step a1: activation statistics -----------------------------------

def act_stats(X: np.ndarray, abs_sum: np.ndarray | None = None) -> np.ndarray:
    """Exact per-channel sum of |x| in units of 2^-24 (int64 [K]).

    Passing ``abs_sum`` adds this batch to a running sum (streamed
    calibration batches)."""
    b = _bits(X)
    T, K = b.shape
    acc = np.zeros(K, dtype=np.int64) if abs_sum is None else np.array(abs_sum, dtype=np.int64)
    r = _lib().awqo_act_stats(_p(b), T, K, K, 0 if abs_sum is None else 1, _p(acc))
    if r:
        raise OracleError(f"act_stats: status {r} (non-finite activation)")
    return acc


def act_mean(abs_sum: np.ndarray, n_tokens: int) -> np.ndarray:
    """Average activation magnitude m[k] = abs_sum[k] * 2^-24 / n_tokens."""
    a = np.ascontiguousarray(abs_sum, dtype=np.int64)
    m = np.empty(a.size, dtype=np.float64)
    _lib().awqo_act_mean(_p(a), int(n_tokens), a.size, _p(m))
    return m


# ---- step a2: candidate scales -----------------------------------------

def candidate_scales(m: np.ndarray, alpha: float) -> np.ndarray:
    """s = max(m, 1e-4)**alpha / sqrt(max * min), rounded once to fp32."""
    mm = np.ascontiguousarray(m, dtype=np.float64)
    s = np.empty(mm.size, dtype=np.float32)
    _lib().awqo_candidate_scales(_p(mm), mm.size, float(alpha), _p(s))
    return s


# ---- steps a3/a5: quantiser and packing ---------------------------------

def quantize(W: np.ndarray, s: np.ndarray | None = None, bits: int = 4):
    """Levels 0..2^bits - 1 (bits 4, or 3) of W*diag(s): returns (q uint8
    [N,K], scales fp16-bits [N,K/128], zeros fp16-bits [N,K/128])."""
    if bits not in (3, 4):
        raise OracleError("bits must be 3 or 4")
    b = _bits(W)
    N, K = b.shape
    if K % GROUP:
        raise OracleError("K must be a multiple of 128")
    G = K // GROUP
    q = np.empty((N, K), dtype=np.uint8)
    sc = np.empty((N, G), dtype=np.uint16)
    ze = np.empty((N, G), dtype=np.uint16)
    sp = None
    if s is not None:
        s = np.ascontiguousarray(s, dtype=np.float32)
        assert s.size == K
        sp = _p(s)
    r = _lib().awqo_quantize_bits(_p(b), N, K, K, sp, bits, _p(q), _p(sc), _p(ze))
    if r:
        raise OracleError(f"quantize: status {r}")
    return q, sc, ze


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    w = np.empty((N, K // 8), dtype=np.uint32)
    _lib().awqo_pack_nibbles(_p(q), N, K, _p(w))
    return w


def unpack_nibbles(words: np.ndarray, K: int) -> np.ndarray:
    w = np.ascontiguousarray(words, dtype=np.uint32)
    N = w.shape[0]
    q = np.empty((N, K), dtype=np.uint8)
    _lib().awqo_unpack_nibbles(_p(w), N, K, _p(q))
    return q


def pack_planes3(q: np.ndarray) -> np.ndarray:
    """3-bit levels -> uint32 [N, K/32 * 3]: per 32 levels, bit plane p in
    word p (level i of the block at bit i)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    if K % 32:
        raise OracleError("K must be a multiple of 32")
    w = np.empty((N, K // 32 * 3), dtype=np.uint32)
    _lib().awqo_pack_planes3(_p(q), N, K, _p(w))
    return w


def unpack_planes3(words: np.ndarray, K: int) -> np.ndarray:
    w = np.ascontiguousarray(words, dtype=np.uint32)
    N = w.shape[0]
    q = np.empty((N, K), dtype=np.uint8)
    _lib().awqo_unpack_planes3(_p(w), N, K, _p(q))
    return q


def pack_int3(W: np.ndarray, s: np.ndarray | None = None):
    """(bit planes uint32 [N, 3K/32], scales, zeros) of W*diag(s) at 3 bits."""
    q, sc, ze = quantize(W, s, bits=3)
    return pack_planes3(q), sc, ze


def pack_int4(W: np.ndarray, s: np.ndarray | None = None):
    """(qweight uint32 [N,K/8], scales, zeros) of W*diag(s)."""
    q, sc, ze = quantize(W, s)
    return pack_nibbles(q), sc, ze


def dequant(q: np.ndarray, scales: np.ndarray, zeros: np.ndarray) -> np.ndarray:
    """(q - z) * scale in fp64, [N,K]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    sc, ze = _bits(scales), _bits(zeros)
    out = np.empty((N, K), dtype=np.float64)
    _lib().awqo_dequant(_p(q), _p(sc), _p(ze), N, K, _p(out))
    return out


# ---- steps a3/a4: the alpha search ---------------------------------------

def search_residual(W: np.ndarray, s: np.ndarray | None, quant=None,
                    bits: int = 4) -> np.ndarray:
    """E = Q(W diag(s)) diag(s)^-1 - W in fp64, [N,K]."""
    b = _bits(W)
    N, K = b.shape
    q, sc, ze = quant if quant is not None else quantize(b, s, bits)
    sp = None
    if s is not None:
        s = np.ascontiguousarray(s, dtype=np.float32)
        sp = _p(s)
    E = np.empty((N, K), dtype=np.float64)
    _lib().awqo_search_residual(_p(b), N, K, K, sp, _p(np.ascontiguousarray(q)),
                                _p(_bits(sc)), _p(_bits(ze)), _p(E))
    return E


def search_mse(W: np.ndarray, X: np.ndarray, s: np.ndarray | None,
               row_chunk: int = 4096, bits: int = 4) -> float:
    """Output MSE of Q(W diag(s)) diag(s)^-1 against W on activations X:
    ||X E^T||_F^2 / (T N), all in fp64 (numpy matmul as the library step)."""
    b = _bits(W)
    N, K = b.shape
    X64 = h2d(X)
    T = X64.shape[0]
    if s is not None:
        s = np.ascontiguousarray(s, dtype=np.float32)
    total = 0.0
    for n0 in range(0, N, row_chunk):
        E = search_residual(b[n0:n0 + row_chunk], s, bits=bits)
        Y = X64 @ E.T
        total += float(np.sum(Y * Y))
    return total / (T * N)


def gram(X: np.ndarray) -> np.ndarray:
    """G = X^T X in fp64 [K,K] from the exact fp64 values of the fp16 X
    (numpy matmul as the library step)."""
    X64 = h2d(X)
    return X64.T @ X64


def search_mse_gram(W: np.ndarray, G: np.ndarray, T: int, s: np.ndarray | None,
                    row_chunk: int = 4096, bits: int = 4) -> float:
    """The search objective through the Gram matrix G = X^T X of the T
    calibration tokens: ||X E^T||_F^2 = tr(E G E^T), so the MSE is
    sum((E G) * E) / (T N), in fp64.  Equal to ``search_mse`` up to fp64
    rounding; its cost does not grow with T once G exists."""
    b = _bits(W)
    N, K = b.shape
    G = np.ascontiguousarray(G, dtype=np.float64)
    assert G.shape == (K, K)
    if s is not None:
        s = np.ascontiguousarray(s, dtype=np.float32)
    total = 0.0
    for n0 in range(0, N, row_chunk):
        E = search_residual(b[n0:n0 + row_chunk], s, bits=bits)
        total += float(np.sum((E @ G) * E))
    return total / (T * N)


def search_scale(W: np.ndarray, X: np.ndarray, m: np.ndarray,
                 alphas=ALPHA_GRID, bits: int = 4):
    """Grid search over alpha: returns (s_best fp32 [K], mse fp64 [n_alpha],
    best index).  Ties go to the lowest index (ascending scan, strict <)."""
    mse = np.empty(len(alphas), dtype=np.float64)
    cands = []
    for i, a in enumerate(alphas):
        s = candidate_scales(m, a)
        cands.append(s)
        mse[i] = search_mse(W, X, s, bits=bits)
    best = 0
    for i in range(1, len(alphas)):
        if mse[i] < mse[best]:
            best = i
    return cands[best], mse, best


# ---- steps a6/a7: the dequantised matmul --------------------------------

def w3a16_gemm(X: np.ndarray, planes: np.ndarray, scales: np.ndarray,
               zeros: np.ndarray, row_chunk: int = 4096) -> np.ndarray:
    """Y = X deq(Wq)^T in fp64 over the 3-bit planes of ``pack_int3``."""
    X64 = h2d(X)
    M, K = X64.shape
    N = planes.shape[0]
    G = K // GROUP
    Y = np.empty((M, N), dtype=np.float64)
    for n0 in range(0, N, row_chunk):
        n1 = min(N, n0 + row_chunk)
        q = unpack_planes3(planes[n0:n1], K)
        D = dequant(q, _bits(scales)[n0:n1].reshape(-1, G), _bits(zeros)[n0:n1].reshape(-1, G))
        Y[:, n0:n1] = X64 @ D.T
    return Y


def w4a16_gemm(X: np.ndarray, qweight: np.ndarray, scales: np.ndarray,
               zeros: np.ndarray, row_chunk: int = 4096) -> np.ndarray:
    """Y = X deq(Wq)^T in fp64, [M, N]."""
    X64 = h2d(X)
    M, K = X64.shape
    N = qweight.shape[0]
    G = K // GROUP
    Y = np.empty((M, N), dtype=np.float64)
    for n0 in range(0, N, row_chunk):
        n1 = min(N, n0 + row_chunk)
        q = unpack_nibbles(qweight[n0:n1], K)
        D = dequant(q, _bits(scales)[n0:n1].reshape(-1, G), _bits(zeros)[n0:n1].reshape(-1, G))
        Y[:, n0:n1] = X64 @ D.T
    return Y


def w4a16_pairs(X: np.ndarray, qweight: np.ndarray, scales: np.ndarray,
                zeros: np.ndarray, ms: np.ndarray, ns: np.ndarray) -> np.ndarray:
    """Y[m_i, n_i] for listed pairs, fp64, straight from the packed words."""
    xb = _bits(X)
    K = xb.shape[1]
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms.size, dtype=np.float64)
    _lib().awqo_w4a16_pairs(_p(xb), K, K, _p(np.ascontiguousarray(qweight, dtype=np.uint32)),
                            _p(_bits(scales)), _p(_bits(zeros)), ms.size, _p(ms), _p(ns),
                            _p(out))
    return out


def scale_activations(X: np.ndarray, inv_s: np.ndarray) -> np.ndarray:
    """The matmul's input scaling: fp16(fp32(X * inv_s)) per element (bits)."""
    xb = _bits(X)
    M, K = xb.shape
    inv = np.ascontiguousarray(inv_s, dtype=np.float32)
    out = np.empty((M, K), dtype=np.uint16)
    _lib().awqo_scale_activations(_p(xb), M, K, _p(inv), _p(out))
    return out


def linear(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Plain fp64 X W^T (the unquantised layer)."""
    return np.asarray(X, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T
