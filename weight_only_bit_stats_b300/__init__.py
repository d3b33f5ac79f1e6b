"""Python binding of libawq_b300.so: the AWQ hot path on one B300 (sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors must be CUDA tensors on the current device; results are produced on
``torch.cuda.current_stream()``.  There is no CPU fallback: if the library is
missing, importing the binding's functions raises.

Steps (names follow the C ABI in ``include/awq.h``):

* ``act_stats`` / ``act_mean``  -- per-input-channel mean |x| (exact sums)
* ``candidate_scales``          -- s = mean|x|^alpha, normalised
* ``search_scale``              -- alpha grid search by output MSE
* ``gram`` / ``search_scale_gram`` -- the same search through G/T = X^T X / T
* ``pack_int4``                 -- asymmetric INT4, group 128, fp16 scale/zero
* ``w4a16_gemm``                -- Y = X deq(Wq)^T, fp32 accumulate, fp16 out
* ``repack_int4``               -- packed weights -> contiguous decode tiles
* ``w4a16_gemm_repacked``       -- the decode matmul (M <= 16) over the tiles
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["AwqError", "lib", "act_stats", "act_mean", "candidate_scales", "search_scale",
           "pack_int4", "pack_int3", "w4a16_gemm", "w3a16_gemm", "w4a16_gemm_scaled",
           "repack_int4", "w4a16_gemm_repacked", "repack_int3", "w3a16_gemm_repacked",
           "gram", "search_scale_gram",
           "set_weight_prefetch",
           "sync_status",
           "ALPHA_GRID",
           "GROUP"]

GROUP = 128
ALPHA_GRID = tuple(i / 20.0 for i in range(20))
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libawq_b300.so")

_STATUS = {0: "AWQ_OK", 1: "AWQ_ERR_INVALID_ARG", 2: "AWQ_ERR_SHAPE", 3: "AWQ_ERR_ALIGN",
           4: "AWQ_ERR_DEVICE", 5: "AWQ_ERR_WORKSPACE", 6: "AWQ_ERR_CUDA", 7: "AWQ_ERR_TIMEOUT",
           8: "AWQ_ERR_NONFINITE", 9: "AWQ_ERR_OVERFLOW"}


class AwqError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where}: {_STATUS.get(code, code)}: {msg}")
        self.code = code


_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_sz = ctypes.c_size_t

# (name, restype, argtypes)
SIGNATURES = (
    ("awq_act_stats", _int, [_p, _i64, _i64, _i64, _int, _p, _p]),
    ("awq_act_mean", _int, [_p, _i64, _i64, _p, _p]),
    ("awq_candidate_scales", _int, [_p, _i64, _p, _int, _p, _p, _sz, _p]),
    ("awq_candidate_scales_workspace_size", _sz, [_i64, _int]),
    ("awq_search_scale", _int, [_p, _i64, _i64, _i64, _p, _i64, _i64, _p, _p, _int, _int, _p, _p,
                                _p, _p, _p, _sz, _p]),
    ("awq_search_workspace_size", _sz, [_i64, _i64, _i64, _int]),
    ("awq_search_scale_noalloc", _int, [_p, _i64, _i64, _i64, _p, _i64, _i64, _p, _p, _int, _int,
                                        _p, _p, _p, _p, _p]),
    ("awq_pack_int4", _int, [_p, _i64, _i64, _i64, _p, _int, _p, _p, _p, _p]),
    ("awq_pack_int3", _int, [_p, _i64, _i64, _i64, _p, _int, _p, _p, _p, _p]),
    ("w3a16_gemm", _int, [_p, _i64, _i64, _i64, _p, _p, _p, _i64, _int, _p, _i64, _p]),
    ("w4a16_gemm", _int, [_p, _i64, _i64, _i64, _p, _p, _p, _i64, _int, _p, _i64, _p, _sz, _p]),
    ("w4a16_gemm_workspace_size", _sz, [_i64, _i64, _i64]),
    ("w4a16_gemm_scaled", _int, [_p, _i64, _i64, _i64, _p, _p, _p, _p, _i64, _int, _p, _i64, _p,
                                 _sz, _p]),
    ("w4a16_gemm_scaled_workspace_size", _sz, [_i64, _i64, _i64]),
    ("awq_repack_int4_bytes", _sz, [_i64, _i64]),
    ("awq_repack_int3_bytes", _sz, [_i64, _i64]),
    ("awq_repack_int3", _int, [_p, _p, _p, _i64, _i64, _int, _p, _sz, _p]),
    ("w3a16_gemm_repacked", _int, [_p, _i64, _i64, _i64, _p, _i64, _int, _p, _i64, _p]),
    ("awq_gram_workspace_size", _sz, [_i64, _i64]),
    ("awq_gram", _int, [_p, _i64, _i64, _i64, _p, _p, _sz, _p]),
    ("awq_search_gram_workspace_size", _sz, [_i64, _i64, _int]),
    ("awq_search_scale_gram", _int, [_p, _i64, _i64, _i64, _p, _p, _p, _int, _int, _p, _p, _p, _p,
                                     _p, _sz, _p]),
    ("awq_search_scale_gram_int3", _int, [_p, _i64, _i64, _i64, _p, _p, _p, _int, _int, _p, _p, _p,
                                          _p, _p, _sz, _p]),
    ("awq_search_mse", _int, [_p, _i64, _i64, _i64, _p, _i64, _i64, _p, _int, _int, _p, _p, _p,
                              _p, _sz, _p]),
    ("awq_search_mse_workspace_size", _sz, [_i64, _i64, _i64, _int]),
    ("awq_search_scale_int3", _int, [_p, _i64, _i64, _i64, _p, _i64, _i64, _p, _p, _int, _int, _p,
                                     _p, _p, _p, _p, _sz, _p]),
    ("awq_repack_int4", _int, [_p, _p, _p, _i64, _i64, _int, _p, _sz, _p]),
    ("w4a16_gemm_repacked", _int, [_p, _i64, _i64, _i64, _p, _p, _i64, _int, _p, _i64, _p]),
    ("awq_set_weight_prefetch", _int, [_int]),
    ("awq_selftest_wait_timeout", _int, [_i64, _p]),
    ("awq_sync_status", _int, [_p]),
    ("awq_last_error_string", ctypes.c_char_p, []),
    ("awq_version", _int, []),
)

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m weight_only_bit_stats_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _check(code: int, where: str) -> None:
    if code != 0:
        raise AwqError(code, where, lib().awq_last_error_string().decode())


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() >= 1 and t.stride(-1) != 1:
        raise ValueError(f"{name} must have a contiguous last dimension")
    return t


def _ld(t: torch.Tensor) -> int:
    return t.stride(0) if t.dim() == 2 else t.shape[-1]


def act_stats(X: torch.Tensor, abs_sum: torch.Tensor | None = None, out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Exact per-channel sum of |x| * 2^24 (int64 [K]).  With ``abs_sum``
    given, this batch is added to it (streamed calibration); otherwise the
    sums are written to ``out`` (or a new tensor)."""
    _dev(X, torch.float16, "X")
    T, K = X.shape
    acc = abs_sum is not None
    if acc:
        out = abs_sum
    elif out is None:
        out = torch.empty(K, dtype=torch.int64, device=X.device)
    _dev(out, torch.int64, "abs_sum")
    _check(lib().awq_act_stats(X.data_ptr(), T, K, _ld(X), int(acc), out.data_ptr(),
                               _stream(stream)), "awq_act_stats")
    return out


def act_mean(abs_sum: torch.Tensor, n_tokens: int, out: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """mean |x| per channel, fp64 [K]."""
    _dev(abs_sum, torch.int64, "abs_sum")
    if out is None:
        out = torch.empty(abs_sum.shape[0], dtype=torch.float64, device=abs_sum.device)
    _check(lib().awq_act_mean(abs_sum.data_ptr(), int(n_tokens), abs_sum.shape[0], out.data_ptr(),
                              _stream(stream)), "awq_act_mean")
    return out


def _alphas(alphas) -> tuple[ctypes.Array, int]:
    a = [float(x) for x in alphas]
    return (ctypes.c_double * len(a))(*a), len(a)


def candidate_scales(mean_abs: torch.Tensor, alphas=ALPHA_GRID, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """All candidate scales, fp32 [n_alpha, K]."""
    _dev(mean_abs, torch.float64, "mean_abs")
    K = mean_abs.shape[0]
    arr, n = _alphas(alphas)
    if out is None:
        out = torch.empty((n, K), dtype=torch.float32, device=mean_abs.device)
    ws_n = lib().awq_candidate_scales_workspace_size(K, n)
    ws = workspace if workspace is not None else \
        torch.empty(max(ws_n, 16), dtype=torch.uint8, device=mean_abs.device)
    _check(lib().awq_candidate_scales(mean_abs.data_ptr(), K, arr, n, out.data_ptr(),
                                      ws.data_ptr(), ws.numel(), _stream(stream)),
           "awq_candidate_scales")
    return out


def search_mse(W: torch.Tensor, Xcal: torch.Tensor, s_alpha: torch.Tensor,
               workspace: torch.Tensor | None = None, out=None, stream=None):
    """The search on given candidate scales s_alpha [n_alpha, K]: returns
    (s, mse, best) like ``search_scale``."""
    _dev(W, torch.float16, "W")
    _dev(Xcal, torch.float16, "Xcal")
    _dev(s_alpha, torch.float32, "s_alpha")
    N, K = W.shape
    T = Xcal.shape[0]
    na = s_alpha.shape[0]
    if out is None:
        s = torch.empty(K, dtype=torch.float32, device=W.device)
        mse = torch.empty(na, dtype=torch.float64, device=W.device)
        best = torch.empty(1, dtype=torch.int32, device=W.device)
    else:
        s, mse, best = out
    n = lib().awq_search_mse_workspace_size(N, K, T, na)
    if workspace is None:
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=W.device)
    _check(lib().awq_search_mse(W.data_ptr(), N, K, _ld(W), Xcal.data_ptr(), T, _ld(Xcal),
                                s_alpha.data_ptr(), na, GROUP, s.data_ptr(), mse.data_ptr(),
                                best.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                _stream(stream)), "awq_search_mse")
    return s, mse, best


def search_workspace(N: int, K: int, T: int, n_alpha: int, device) -> torch.Tensor:
    n = lib().awq_search_workspace_size(N, K, T, n_alpha)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def gram(Xcal: torch.Tensor, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """G/T = Xcal^T Xcal / T as fp16 [K, K]."""
    _dev(Xcal, torch.float16, "Xcal")
    T, K = Xcal.shape
    if out is None:
        out = torch.empty((K, K), dtype=torch.float16, device=Xcal.device)
    _dev(out, torch.float16, "G")
    n = lib().awq_gram_workspace_size(T, K)
    if workspace is None:
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=Xcal.device)
    _check(lib().awq_gram(Xcal.data_ptr(), T, K, _ld(Xcal), out.data_ptr(), workspace.data_ptr(),
                          workspace.numel(), _stream(stream)), "awq_gram")
    return out


def search_scale_gram(W: torch.Tensor, G: torch.Tensor, mean_abs: torch.Tensor,
                      alphas=ALPHA_GRID, workspace: torch.Tensor | None = None,
                      return_candidates: bool = False, out=None, stream=None, bits: int = 4):
    """The alpha search through G/T from ``gram``: returns (s, mse, best)
    like ``search_scale`` (and the candidate scales when asked)."""
    if bits not in (3, 4):
        raise ValueError("bits must be 3 or 4")
    _dev(W, torch.float16, "W")
    _dev(G, torch.float16, "G")
    _dev(mean_abs, torch.float64, "mean_abs")
    N, K = W.shape
    arr, na = _alphas(alphas)
    if out is None:
        s = torch.empty(K, dtype=torch.float32, device=W.device)
        mse = torch.empty(na, dtype=torch.float64, device=W.device)
        best = torch.empty(1, dtype=torch.int32, device=W.device)
    else:
        s, mse, best = out
    cand = torch.empty((na, K), dtype=torch.float32, device=W.device) if return_candidates else None
    n = lib().awq_search_gram_workspace_size(N, K, na)
    if workspace is None:
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=W.device)
    fn = lib().awq_search_scale_gram if bits == 4 else lib().awq_search_scale_gram_int3
    _check(fn(W.data_ptr(), N, K, _ld(W), G.data_ptr(), mean_abs.data_ptr(),
              arr, na, GROUP, s.data_ptr(), mse.data_ptr(), best.data_ptr(),
              cand.data_ptr() if cand is not None else None,
              workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "awq_search_scale_gram" if bits == 4 else "awq_search_scale_gram_int3")
    return (s, mse, best, cand) if return_candidates else (s, mse, best)


def search_scale(W: torch.Tensor, Xcal: torch.Tensor, mean_abs: torch.Tensor, alphas=ALPHA_GRID,
                 workspace: torch.Tensor | None = None, return_candidates: bool = False,
                 out=None, stream=None, bits: int = 4):
    """alpha grid search (``bits`` 4, or 3 for the levels of ``pack_int3``).
    Returns ``(s fp32 [K], mse fp64 [n_alpha], best int32 [1])`` (+ all
    candidate scales [n_alpha, K] when ``return_candidates``), all on the
    device."""
    if bits not in (3, 4):
        raise ValueError("bits must be 3 or 4")
    _dev(W, torch.float16, "W")
    _dev(Xcal, torch.float16, "Xcal")
    _dev(mean_abs, torch.float64, "mean_abs")
    N, K = W.shape
    T = Xcal.shape[0]
    arr, n = _alphas(alphas)
    dev = W.device
    if out is not None:
        s, mse, best = out
    else:
        s = torch.empty(K, dtype=torch.float32, device=dev)
        mse = torch.empty(n, dtype=torch.float64, device=dev)
        best = torch.empty(1, dtype=torch.int32, device=dev)
    cands = torch.empty((n, K), dtype=torch.float32, device=dev) if return_candidates else None
    if workspace is None:
        workspace = search_workspace(N, K, T, n, dev)
    fn = lib().awq_search_scale if bits == 4 else lib().awq_search_scale_int3
    _check(fn(W.data_ptr(), N, K, _ld(W), Xcal.data_ptr(), T, _ld(Xcal),
              mean_abs.data_ptr(), arr, n, GROUP, s.data_ptr(), mse.data_ptr(),
              best.data_ptr(), cands.data_ptr() if cands is not None else None,
              workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "awq_search_scale" if bits == 4 else "awq_search_scale_int3")
    return (s, mse, best, cands) if return_candidates else (s, mse, best)


def pack_int4(W: torch.Tensor, s: torch.Tensor | None = None, out=None, stream=None):
    """INT4 pack of W diag(s): ``(qweight int32 [N, K/8] (uint32 bits),
    scales fp16 [N, K/128], zeros fp16 [N, K/128])``."""
    _dev(W, torch.float16, "W")
    N, K = W.shape
    if s is not None:
        _dev(s, torch.float32, "s")
    if out is None:
        out = (torch.empty((N, K // 8), dtype=torch.int32, device=W.device),
               torch.empty((N, K // GROUP), dtype=torch.float16, device=W.device),
               torch.empty((N, K // GROUP), dtype=torch.float16, device=W.device))
    qw, sc, ze = out
    _check(lib().awq_pack_int4(W.data_ptr(), N, K, _ld(W), s.data_ptr() if s is not None else None,
                               GROUP, qw.data_ptr(), sc.data_ptr(), ze.data_ptr(), _stream(stream)),
           "awq_pack_int4")
    return qw, sc, ze


def pack_int3(W: torch.Tensor, s: torch.Tensor | None = None, out=None, stream=None):
    """3-bit pack of W diag(s): ``(planes int32 [N, 3K/32] (uint32 bits),
    scales fp16 [N, K/128], zeros fp16 [N, K/128])``."""
    _dev(W, torch.float16, "W")
    N, K = W.shape
    if s is not None:
        _dev(s, torch.float32, "s")
    if out is None:
        out = (torch.empty((N, K // 32 * 3), dtype=torch.int32, device=W.device),
               torch.empty((N, K // GROUP), dtype=torch.float16, device=W.device),
               torch.empty((N, K // GROUP), dtype=torch.float16, device=W.device))
    pl, sc, ze = out
    _check(lib().awq_pack_int3(W.data_ptr(), N, K, _ld(W), s.data_ptr() if s is not None else None,
                               GROUP, pl.data_ptr(), sc.data_ptr(), ze.data_ptr(), _stream(stream)),
           "awq_pack_int3")
    return pl, sc, ze


def w3a16_gemm(X: torch.Tensor, planes: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = X deq(Wq)^T over the 3-bit planes of ``pack_int3``, fp16 [M, N]
    (decode kernel for M <= 16, tensor cores above)."""
    _dev(X, torch.float16, "X")
    _dev(planes, torch.int32, "planes")
    _dev(scales, torch.float16, "scales")
    _dev(zeros, torch.float16, "zeros")
    M, K = X.shape
    N = planes.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=X.device)
    _check(lib().w3a16_gemm(X.data_ptr(), M, K, _ld(X), planes.data_ptr(), scales.data_ptr(),
                            zeros.data_ptr(), N, GROUP, Y.data_ptr(), _ld(Y), _stream(stream)),
           "w3a16_gemm")
    return Y


def w4a16_gemm(X: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = X deq(Wq)^T, fp16 [M, N]."""
    _dev(X, torch.float16, "X")
    _dev(qweight, torch.int32, "qweight")
    _dev(scales, torch.float16, "scales")
    _dev(zeros, torch.float16, "zeros")
    M, K = X.shape
    N = qweight.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=X.device)
    ws_n = lib().w4a16_gemm_workspace_size(M, N, K)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=X.device) if ws_n else None
    _check(lib().w4a16_gemm(X.data_ptr(), M, K, _ld(X), qweight.data_ptr(), scales.data_ptr(),
                            zeros.data_ptr(), N, GROUP, Y.data_ptr(), _ld(Y),
                            ws.data_ptr() if ws is not None else None, ws_n, _stream(stream)),
           "w4a16_gemm")
    return Y


def repack_int4(qweight: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The packed weights regrouped into contiguous decode tiles (uint8
    [awq_repack_int4_bytes(N, K)]), one 1088-byte tile per 16 rows x 128
    input channels."""
    _dev(qweight, torch.int32, "qweight")
    _dev(scales, torch.float16, "scales")
    _dev(zeros, torch.float16, "zeros")
    N, K8 = qweight.shape
    K = K8 * 8
    nbytes = lib().awq_repack_int4_bytes(N, K)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=qweight.device)
    _dev(out, torch.uint8, "tiles")
    _check(lib().awq_repack_int4(qweight.data_ptr(), scales.data_ptr(), zeros.data_ptr(), N, K,
                                 GROUP, out.data_ptr(), out.numel(), _stream(stream)),
           "awq_repack_int4")
    return out


def w4a16_gemm_repacked(X: torch.Tensor, tiles: torch.Tensor, N: int,
                        inv_s: torch.Tensor | None = None, out: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Y = X deq(Wq)^T over the decode tiles of an [N, K] weight, M <= 16;
    with ``inv_s`` the input is fp16(X * inv_s)."""
    _dev(X, torch.float16, "X")
    _dev(tiles, torch.uint8, "tiles")
    if inv_s is not None:
        _dev(inv_s, torch.float32, "inv_s")
    M, K = X.shape
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=X.device)
    _check(lib().w4a16_gemm_repacked(X.data_ptr(), M, K, _ld(X),
                                     inv_s.data_ptr() if inv_s is not None else None,
                                     tiles.data_ptr(), N, GROUP, Y.data_ptr(), _ld(Y),
                                     _stream(stream)), "w4a16_gemm_repacked")
    return Y


def repack_int3(planes: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The 3-bit planes regrouped into contiguous decode tiles (uint8
    [awq_repack_int3_bytes(N, K)]), one 832-byte tile per 16 rows x 128
    input channels."""
    _dev(planes, torch.int32, "planes")
    _dev(scales, torch.float16, "scales")
    _dev(zeros, torch.float16, "zeros")
    N, W3 = planes.shape
    K = W3 // 3 * 32
    nbytes = lib().awq_repack_int3_bytes(N, K)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=planes.device)
    _dev(out, torch.uint8, "tiles")
    _check(lib().awq_repack_int3(planes.data_ptr(), scales.data_ptr(), zeros.data_ptr(), N, K,
                                 GROUP, out.data_ptr(), out.numel(), _stream(stream)),
           "awq_repack_int3")
    return out


def w3a16_gemm_repacked(X: torch.Tensor, tiles: torch.Tensor, N: int,
                        out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = X deq(Wq)^T over the 3-bit decode tiles of an [N, K] weight, M <= 16."""
    _dev(X, torch.float16, "X")
    _dev(tiles, torch.uint8, "tiles")
    M, K = X.shape
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=X.device)
    _check(lib().w3a16_gemm_repacked(X.data_ptr(), M, K, _ld(X), tiles.data_ptr(), N, GROUP,
                                     Y.data_ptr(), _ld(Y), _stream(stream)), "w3a16_gemm_repacked")
    return Y


def w4a16_gemm_scaled(X: torch.Tensor, inv_s: torch.Tensor, qweight: torch.Tensor,
                      scales: torch.Tensor, zeros: torch.Tensor,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = fp16(X * inv_s) deq(Wq)^T with the input scaling fused, fp16 [M, N]."""
    _dev(X, torch.float16, "X")
    _dev(inv_s, torch.float32, "inv_s")
    _dev(qweight, torch.int32, "qweight")
    _dev(scales, torch.float16, "scales")
    _dev(zeros, torch.float16, "zeros")
    M, K = X.shape
    N = qweight.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.float16, device=X.device)
    ws_n = lib().w4a16_gemm_scaled_workspace_size(M, N, K)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=X.device) if ws_n else None
    _check(lib().w4a16_gemm_scaled(X.data_ptr(), M, K, _ld(X), inv_s.data_ptr(),
                                   qweight.data_ptr(), scales.data_ptr(), zeros.data_ptr(), N,
                                   GROUP, Y.data_ptr(), _ld(Y),
                                   ws.data_ptr() if ws is not None else None, ws_n,
                                   _stream(stream)), "w4a16_gemm_scaled")
    return Y


def set_weight_prefetch(enable: bool) -> None:
    """Allow decode matmuls to fetch their packed weights before the previous
    kernel in the stream completes (see ``awq_set_weight_prefetch``); only
    valid when no kernel writing a matmul's weights runs immediately before
    it in the same stream."""
    _check(lib().awq_set_weight_prefetch(1 if enable else 0), "awq_set_weight_prefetch")


def sync_status(stream=None) -> None:
    """Synchronise and raise if a kernel flagged a device-side condition."""
    _check(lib().awq_sync_status(_stream(stream)), "awq_sync_status")
