"""The C-ABI library without a GPU: it builds, loads, exports every function
declared in include/awq.h, and rejects bad arguments on the host before any
device work (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "awq.h")


@pytest.fixture(scope="module")
def capi():
    from weight_only_bit_stats_b300 import build
    build.build()
    import weight_only_bit_stats_b300 as wb
    return wb.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("awq_act_stats", "awq_search_scale", "awq_pack_int4", "w4a16_gemm"):
        assert n in names


def test_every_declared_symbol_is_exported(capi):
    import weight_only_bit_stats_b300 as wb
    names = declared_functions()
    bound = {n for n, _, _ in wb.SIGNATURES}
    for n in names:
        assert hasattr(capi, n), f"{n} not exported"
        assert n in bound, f"{n} has no binding signature"


def test_version_and_workspace_sizes(capi):
    assert capi.awq_version() >= 100
    assert capi.w4a16_gemm_workspace_size(1, 4096, 4096) == 0
    n = capi.awq_search_workspace_size(12288, 4096, 512, 20)
    # s_alpha + 1/s (fp32) + r (fp64) per alpha and channel, plus partials
    assert n >= 20 * 4096 * (4 + 4 + 8) + 20 * 96 * 4 * 8
    assert capi.awq_search_workspace_size(0, 4096, 512, 20) == 0
    assert capi.awq_candidate_scales_workspace_size(4096, 20) >= 20 * 4096 * 8
    # decode tiles: 1088 bytes per (16-row slab, group of 128), N rounded up to 16
    assert capi.awq_repack_int4_bytes(12288, 4096) == 768 * 32 * 1088
    assert capi.awq_repack_int4_bytes(136, 384) == 9 * 3 * 1088
    assert capi.awq_repack_int4_bytes(16, 100) == 0
    assert capi.awq_repack_int3_bytes(12288, 4096) == 768 * 32 * 832
    # Gram route: the transposed calibration copy (T padded to 64) and the
    # search workspace over K columns in place of T tokens
    assert capi.awq_gram_workspace_size(300, 1024) >= 1024 * 320 * 2
    assert capi.awq_search_gram_workspace_size(4096, 4096, 20) == \
        capi.awq_search_workspace_size(4096, 4096, 4096, 20)
    assert capi.awq_search_mse_workspace_size(12288, 4096, 512, 20) == \
        capi.awq_search_workspace_size(12288, 4096, 512, 20)


def test_host_argument_checks(capi):
    """Bad arguments are refused before any device call."""
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) & ~15
    # null pointers
    assert capi.awq_pack_int4(None, 8, 128, 128, None, 128, None, None, None, None) == 1
    # group must be 128, K a multiple of 128
    assert capi.awq_pack_int4(base, 8, 128, 128, None, 64, base, base, base, None) == 2
    assert capi.awq_pack_int4(base, 8, 100, 100, None, 128, base, base, base, None) == 2
    # misaligned weight pointer
    assert capi.awq_pack_int4(base + 2, 8, 128, 128, None, 128, base, base, base, None) == 3
    # gemm: N % 8, ldx < K
    assert capi.w4a16_gemm(base, 1, 128, 128, base, base, base, 12, 128, base, 12, None, 0,
                           None) == 2
    assert capi.w4a16_gemm(base, 1, 256, 128, base, base, base, 16, 128, base, 16, None, 0,
                           None) == 2
    # search: too many alphas; missing workspace
    alphas = (ctypes.c_double * 65)(*([0.0] * 65))
    assert capi.awq_search_scale(base, 8, 128, 128, base, 4, 128, base, alphas, 65, 128, base,
                                 None, base, None, base, 4096, None) == 1
    assert capi.awq_search_scale(base, 8, 128, 128, base, 4, 128, base, alphas, 2, 128, base,
                                 None, base, None, None, 0, None) == 5
    # stats: bad accumulate flag
    assert capi.awq_act_stats(base, 4, 128, 128, 2, base, None) == 1
    # stats: the exact int64 sums hold for fewer than 2^23 tokens per call
    assert capi.awq_act_stats(base, 1 << 23, 128, 128, 0, base, None) == 2
    assert capi.awq_act_stats(base, 1 << 23, 128, 128, 1, base, None) == 2
    # decode weight prefetch: a flag, 0 or 1 only (host-side setting)
    assert capi.awq_set_weight_prefetch(2) == 1
    assert capi.awq_set_weight_prefetch(1) == 0 and capi.awq_set_weight_prefetch(0) == 0
    # timeout self-test: the limit is checked before any device call
    assert capi.awq_selftest_wait_timeout(0, None) == 1
    # 3-bit pack: null pointer, group, K, misaligned W and planes
    assert capi.awq_pack_int3(None, 8, 128, 128, None, 128, None, None, None, None) == 1
    assert capi.awq_pack_int3(base, 8, 128, 128, None, 64, base, base, base, None) == 2
    assert capi.awq_pack_int3(base, 8, 96, 96, None, 128, base, base, base, None) == 2
    assert capi.awq_pack_int3(base + 2, 8, 128, 128, None, 128, base, base, base, None) == 3
    assert capi.awq_pack_int3(base, 8, 128, 128, None, 128, base + 2, base, base, None) == 3
    # 3-bit matmul: planes 16-byte aligned for M > 16 (tensor-core path), N % 8, misaligned X
    assert capi.w3a16_gemm(base, 17, 128, 128, base + 4, base, base, 8, 128, base, 8, None) == 3
    assert capi.w3a16_gemm(base, 1, 128, 128, base, base, base, 12, 128, base, 12, None) == 2
    assert capi.w3a16_gemm(base + 2, 1, 128, 128, base, base, base, 8, 128, base, 8, None) == 3
    assert capi.w3a16_gemm(None, 1, 128, 128, base, base, base, 8, 128, base, 8, None) == 1
    # repack: K % 128, tiles buffer too small, misaligned tiles
    assert capi.awq_repack_int4(base, base, base, 16, 100, 128, base, 4096, None) == 2
    assert capi.awq_repack_int4(base, base, base, 16, 128, 128, base, 1087, None) == 5
    assert capi.awq_repack_int4(base, base, base, 16, 128, 128, base + 8, 4096, None) == 3
    # repacked matmul: decode sizes only, N % 8, misaligned X or tiles
    assert capi.w4a16_gemm_repacked(base, 17, 128, 128, None, base, 16, 128, base, 16, None) == 2
    assert capi.w4a16_gemm_repacked(base, 1, 128, 128, None, base, 12, 128, base, 12, None) == 2
    assert capi.w4a16_gemm_repacked(base + 2, 1, 128, 128, None, base, 16, 128, base, 16,
                                    None) == 3
    assert capi.w4a16_gemm_repacked(base, 1, 128, 128, None, base + 8, 16, 128, base, 16,
                                    None) == 3
    # 3-bit repack and repacked matmul: planes alignment, decode sizes only
    assert capi.awq_repack_int3(base + 4, base, base, 16, 128, 128, base, 4096, None) == 3
    assert capi.w3a16_gemm_repacked(base, 17, 128, 128, base, 16, 128, base, 16, None) == 2
    # Gram route: K % 128, misaligned G, missing workspace
    assert capi.awq_gram(base, 64, 100, 100, base, base, 1 << 20, None) == 2
    assert capi.awq_gram(base, 64, 128, 128, base + 2, base, 1 << 20, None) == 3
    assert capi.awq_gram(base, 64, 128, 128, base, None, 0, None) == 5
    assert capi.awq_search_scale_gram(base, 8, 128, 128, base, base, alphas, 65, 128, base, None,
                                      base, None, base, 4096, None) == 1
    assert capi.awq_search_scale_gram(base, 12, 128, 128, base, base, alphas, 2, 128, base, None,
                                      base, None, base, 4096, None) == 2
    assert capi.awq_search_scale_gram(base, 8, 128, 128, base, base, alphas, 2, 128, base, None,
                                      base, None, None, 0, None) == 5
    # search on given candidates: n_alpha range, null candidates, K % 128,
    # misaligned candidates, workspace (all before any device call)
    assert capi.awq_search_mse(base, 8, 128, 128, base, 4, 128, base, 65, 128, base, None, base,
                               base, 4096, None) == 1
    assert capi.awq_search_mse(base, 8, 128, 128, base, 4, 128, None, 2, 128, base, None, base,
                               base, 4096, None) == 1
    assert capi.awq_search_mse(base, 8, 100, 100, base, 4, 100, base, 2, 128, base, None, base,
                               base, 4096, None) == 2
    assert capi.awq_search_mse(base, 8, 128, 128, base, 4, 128, base + 4, 2, 128, base, None, base,
                               base, 4096, None) == 3
    assert capi.awq_search_mse(base, 8, 128, 128, base, 4, 128, base, 2, 128, base, None, base,
                               None, 0, None) == 5
    assert capi.awq_last_error_string()


def test_host_argument_checks_remaining_calls(capi):
    """The entry points not exercised above refuse bad arguments on the host
    too, with the documented codes (1 invalid argument, 2 shape, 3 alignment,
    5 workspace), before any device call."""
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) & ~15
    alphas = (ctypes.c_double * 65)(*([0.0] * 65))
    # mean of the statistics: token count, null pointers
    assert capi.awq_act_mean(base, 0, 128, base, None) == 1
    assert capi.awq_act_mean(None, 4, 128, base, None) == 1
    assert capi.awq_act_mean(base, 4, 128, None, None) == 1
    # candidate scales: K, n_alpha range, null pointers, workspace
    ws = capi.awq_candidate_scales_workspace_size(128, 2)
    assert ws > 0 and capi.awq_candidate_scales_workspace_size(0, 2) == 0
    assert capi.awq_candidate_scales(base, 0, alphas, 2, base, base, ws, None) == 1
    assert capi.awq_candidate_scales(base, 128, alphas, 0, base, base, ws, None) == 1
    assert capi.awq_candidate_scales(base, 128, alphas, 65, base, base, ws, None) == 1
    assert capi.awq_candidate_scales(None, 128, alphas, 2, base, base, ws, None) == 1
    assert capi.awq_candidate_scales(base, 128, None, 2, base, base, ws, None) == 1
    assert capi.awq_candidate_scales(base, 128, alphas, 2, None, base, ws, None) == 1
    assert capi.awq_candidate_scales(base, 128, alphas, 2, base, None, ws, None) == 5
    assert capi.awq_candidate_scales(base, 128, alphas, 2, base, base, ws - 1, None) == 5
    assert capi.awq_candidate_scales(base, 128, alphas, 2, base, base + 8, ws, None) == 5
    # 3-bit search: the same checks as the 4-bit search
    args = dict(W=base, N=8, K=128, ldw=128, X=base, T=4, ldx=128, m=base, n_alpha=2,
                group=128, s=base, best=base, ws=base, ws_bytes=4096)

    def s3(**kw):
        a = dict(args, **kw)
        return capi.awq_search_scale_int3(a["W"], a["N"], a["K"], a["ldw"], a["X"], a["T"],
                                          a["ldx"], a["m"], alphas, a["n_alpha"], a["group"],
                                          a["s"], None, a["best"], None, a["ws"], a["ws_bytes"],
                                          None)
    assert s3(n_alpha=65) == 1 and s3(n_alpha=0) == 1 and s3(T=0) == 1
    assert s3(W=None) == 1 and s3(best=None) == 1
    assert s3(K=100, ldw=100, ldx=100) == 2 and s3(N=12) == 2 and s3(group=64) == 2
    assert s3(ldx=132) == 2
    assert s3(W=base + 2) == 3 and s3(s=base + 4) == 3
    assert s3(ws=None, ws_bytes=0) == 5 and s3(ws_bytes=16) == 5
    # 3-bit search through the Gram matrix

    def g3(**kw):
        a = dict(args, **kw)
        return capi.awq_search_scale_gram_int3(a["W"], a["N"], a["K"], a["ldw"], a["X"], a["m"],
                                               alphas, a["n_alpha"], a["group"], a["s"], None,
                                               a["best"], None, a["ws"], a["ws_bytes"], None)
    assert g3(n_alpha=65) == 1 and g3(X=None) == 1
    assert g3(N=12) == 2 and g3(K=100, ldw=100) == 2
    assert g3(X=base + 2) == 3
    assert g3(ws=None, ws_bytes=0) == 5
    # allocation-free search: sizes and n_alpha first, then the scratch size
    # (a problem larger than the library's 16 MiB array)
    assert capi.awq_search_scale_noalloc(base, 8, 128, 128, base, 4, 128, base, alphas, 65, 128,
                                         base, None, base, None, None) == 1
    assert capi.awq_search_scale_noalloc(base, 0, 128, 128, base, 4, 128, base, alphas, 2, 128,
                                         base, None, base, None, None) == 1
    assert capi.awq_search_workspace_size(8, 65536, 4, 64) > 16 << 20
    assert capi.awq_search_scale_noalloc(base, 8, 65536, 65536, base, 4, 65536, base, alphas, 64,
                                         128, base, None, base, None, None) == 5
    # fused input scaling: null inv_s, then the matmul's own checks, and a
    # misaligned inv_s
    assert capi.w4a16_gemm_scaled(base, 1, 128, 128, None, base, base, base, 16, 128, base, 16,
                                  None, 0, None) == 1
    assert capi.w4a16_gemm_scaled(base, 1, 128, 128, base, base, base, base, 12, 128, base, 12,
                                  None, 0, None) == 2
    assert capi.w4a16_gemm_scaled(base, 1, 128, 128, base + 4, base, base, base, 16, 128, base,
                                  16, None, 0, None) == 3
    # its workspace: none at decode sizes; at least fp16(X / s) for M > 16
    assert capi.w4a16_gemm_scaled_workspace_size(16, 4096, 4096) == 0
    assert capi.w4a16_gemm_scaled_workspace_size(300, 4096, 4096) >= 300 * 4096 * 2
    assert capi.w4a16_gemm_scaled_workspace_size(300, 4096, 100) == 0
    assert capi.w4a16_gemm_scaled_workspace_size(300, 0, 4096) == 0
    # the status word needs a device: without one the call reports that
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert capi.awq_sync_status(None) in (4, 6)


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    import weight_only_bit_stats_b300 as wb
    with pytest.raises(ValueError):
        wb.pack_int4(torch.zeros(8, 128, dtype=torch.float16))
