"""Seeded synthetic inputs for the AWQ hot path.

This module only draws random numbers and rounds them to fp16; it holds none
of the method's arithmetic.  Both the CPU oracle and the CUDA library are fed
the exact bytes produced here, so the two sides always see identical inputs.

Generator (counter based, so any slice can be drawn independently):

* ``splitmix64``: the i-th 64-bit word of stream ``seed`` is the SplitMix64
  finaliser applied to ``seed + (i + 1) * 0x9E3779B97F4A7C15`` (mod 2**64),
  the published SplitMix64 step (Steele, Lea, Flood, OOPSLA 2014).
* normals: Box-Muller on consecutive word pairs ``(2j, 2j+1)``:
  ``u1 = ((w0 >> 11) + 1) * 2**-53`` in (0, 1], ``u2 = (w1 >> 11) * 2**-53``,
  ``r = sqrt(-2 ln u1)``, giving ``r cos(2 pi u2)`` and ``r sin(2 pi u2)``.
* fp16: the fp64 value is rounded to the nearest fp16 (ties to even) by
  numpy's float64 -> float16 conversion.

Workload recipe (the synthetic stand-in for the pages' calibration text):

* weights ``W ~ N(0, sigma^2)`` fp16 ``[N, K]``;
* activations ``X ~ N(0, 1)`` fp16 ``[T, K]`` where ``round(0.01 K)`` input
  channels, picked by a seeded Fisher-Yates shuffle, are multiplied by 20
  before rounding (the "1% salient channels" of the pages);
* calibration and matmul activations of one layer share the outlier channels.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_MASK64 = (1 << 64) - 1
_CHUNK = 1 << 24
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

# Seed bases; a layer ``l`` and linear ``j`` (0..6 for q,k,v,o,gate,up,down)
# adds ``16 * l + j``.
SEED_W = 0xA0A00000
SEED_XCAL = 0xB0B00000
SEED_CHANNELS = 0xC0C00000
SEED_XMM = 0xD0D00000


def layer_seed(base: int, layer: int, linear: int) -> int:
    return (base + 16 * layer + linear) & _MASK64


def _lib():
    """Compile (once, in-tree) and load the C draw helper."""
    global _LIB
    if _LIB is not None:
        return _LIB
    src = os.path.join(_HERE, "_synth.c")
    out_dir = os.path.join(_HERE, "_build")
    so = os.path.join(out_dir, "libsynth.so")
    if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
        os.makedirs(out_dir, exist_ok=True)
        tmp = so + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-ffp-contract=off", src, "-o", tmp, "-lm"])
        os.replace(tmp, so)
    lib = ctypes.CDLL(so)
    lib.sg_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                  ctypes.c_void_p]
    lib.sg_normals.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                               ctypes.c_double, ctypes.c_void_p]
    _LIB = lib
    return lib


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Words ``offset .. offset+n-1`` of the SplitMix64 stream ``seed``."""
    out = np.empty(n, dtype=np.uint64)
    if n:
        _lib().sg_splitmix64(seed & _MASK64, offset, n, out.ctypes.data)
    return out


def normals(seed: int, n: int, scale: float = 1.0, offset: int = 0) -> np.ndarray:
    """``scale`` times standard normals ``offset .. offset+n-1`` of stream
    ``seed`` (Box-Muller), fp64."""
    out = np.empty(n, dtype=np.float64)
    if n:
        _lib().sg_normals(seed & _MASK64, offset, n, float(scale), out.ctypes.data)
    return out


def _fp16_normals(seed: int, n: int, scale: float) -> np.ndarray:
    """fp16 rounding of ``scale * normal``, drawn in chunks to bound memory."""
    out = np.empty(n, dtype=np.float16)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        out[lo:hi] = normals(seed, hi - lo, scale, lo).astype(np.float16)
    return out


def outlier_channels(seed: int, K: int, frac: float = 0.01) -> np.ndarray:
    """Sorted indices of ``round(frac*K)`` channels chosen by a seeded
    Fisher-Yates shuffle of ``0..K-1`` (the first ``n`` after shuffling)."""
    n_out = int(round(frac * K))
    perm = np.arange(K, dtype=np.int64)
    if n_out == 0:
        return perm[:0]
    w = splitmix64(seed, K)
    # Durstenfeld's in-place form, front to back, stopping after n_out picks.
    for i in range(min(n_out, K - 1)):
        j = i + int(w[i] % np.uint64(K - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:n_out])


def gen_weights(seed: int, N: int, K: int, sigma: float) -> np.ndarray:
    """fp16 ``[N, K]`` weights drawn from ``N(0, sigma^2)``."""
    return _fp16_normals(seed, N * K, sigma).reshape(N, K)


def gen_acts(seed: int, T: int, K: int, channels: np.ndarray | None = None,
             mult: float = 20.0) -> np.ndarray:
    """fp16 ``[T, K]`` activations ``N(0,1)`` with ``channels`` scaled by
    ``mult`` (in fp64, before the single rounding to fp16)."""
    out = np.empty((T, K), dtype=np.float16)
    rows = max(1, _CHUNK // max(K, 1))
    for r0 in range(0, T, rows):
        r1 = min(T, r0 + rows)
        x = normals(seed, (r1 - r0) * K, 1.0, r0 * K).reshape(r1 - r0, K)
        if channels is not None and len(channels):
            x[:, channels] *= mult
        out[r0:r1] = x.astype(np.float16)
    return out


def fp16_bits(a: np.ndarray) -> np.ndarray:
    """View an fp16 array as its uint16 bit patterns (no copy)."""
    return np.ascontiguousarray(a).view(np.uint16)


# Workloads: named by what they are, with their sizes.
LLAMA7B_DECODE_PROJ = (  # (name, N, K)
    ("qkv", 12288, 4096),
    ("o", 4096, 4096),
    ("gate_up", 22016, 4096),
    ("down", 4096, 11008),
)
LLAMA13B_DECODE_PROJ = (("gate_up", 27648, 5120), ("down", 5120, 13824))
LLAMA70B_PREFILL_PROJ = (("gate_up", 57344, 8192), ("down", 8192, 28672))
LLAMA7B_LAYER_LINEARS = (  # (name, N, K)
    ("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
    ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008),
)


# A LLaMA-7B-shaped decoder layer's linears read four distinct inputs:
# q, k, v the attention input; o the attention output; gate, up the MLP
# input; down the MLP hidden state.  (input name, K) per input, and the
# input index of each linear in LLAMA7B_LAYER_LINEARS.
LLAMA7B_LAYER_INPUTS = (("attn_in", 4096), ("attn_out", 4096), ("mlp_in", 4096),
                        ("mlp_hidden", 11008))
LLAMA7B_LINEAR_INPUT = (0, 0, 0, 1, 2, 2, 3)


def layer_activations(layer: int, index: int, T: int, K: int) -> np.ndarray:
    """Calibration activations of input ``index`` of decoder ``layer``: fp16
    ``[T, K]`` N(0,1) with the input's own 1% outlier channels x20 (seeds
    offset by 8 so they never collide with a linear's own seeds)."""
    ch = outlier_channels(layer_seed(SEED_CHANNELS, layer, 8 + index), K)
    return gen_acts(layer_seed(SEED_XCAL, layer, 8 + index), T, K, ch)


def layer_inputs(layer: int, linear: int, N: int, K: int, T_cal: int,
                 M: int = 0, sigma: float = 0.02):
    """The seeded inputs of one linear layer.

    Returns ``(W, Xcal, Xmm, channels)``: fp16 weights ``[N,K]``, calibration
    activations ``[T_cal, K]``, matmul activations ``[M, K]`` (``None`` when
    ``M == 0``) and the outlier channel indices they share.
    """
    ch = outlier_channels(layer_seed(SEED_CHANNELS, layer, linear), K)
    W = gen_weights(layer_seed(SEED_W, layer, linear), N, K, sigma)
    Xcal = gen_acts(layer_seed(SEED_XCAL, layer, linear), T_cal, K, ch) if T_cal else None
    Xmm = gen_acts(layer_seed(SEED_XMM, layer, linear), M, K, ch) if M else None
    return W, Xcal, Xmm, ch
