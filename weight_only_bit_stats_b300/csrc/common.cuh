// Device-side building blocks shared by the library's kernels: status bits,
// warp reductions, the INT4 group quantiser, and thin inline-PTX wrappers for
// mbarrier, TMA (cp.async.bulk.tensor) and the 5th-generation tensor core
// (tcgen05 MMA with TMEM accumulators) on sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace awq {

constexpr int kGroup = 128;

// Bits of the device status word (see awq_sync_status).
constexpr unsigned kStatusNonFinite = 1u;
constexpr unsigned kStatusTimeout = 2u;
constexpr unsigned kStatusOverflow = 4u;

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void set_status(unsigned* status, unsigned bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// min / max that return NaN when either input is NaN (fminf / fmaxf ignore
// NaN), so a lane's reduction of its values is non-finite exactly when one
// of them is.
__device__ __forceinline__ float fmin_nan(float a, float b) {
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Three-input forms (one instruction on sm_100 and later).
__device__ __forceinline__ float fmin3_nan(float a, float b, float c) {
    float r;
    asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float fmax3_nan(float a, float b, float c) {
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// INT4 group quantiser (asymmetric, group of 128).
//
// For one row-group with scaled weights w':
//   lo, hi = min, max of w'
//   scale  = fp16_rn(max(fp32(fp32(hi - lo) / 15), 2^-14))
//   z      = clamp(rint(fp32(-lo / scale)), 0, 15)
//   q      = clamp(rint(fp32(w' / scale)) + z, 0, 15)
// Every rounding is a single IEEE fp32 operation written as an _rn
// intrinsic, so no FMA contraction can change a level.
// ---------------------------------------------------------------------------

// rint(x), ties to even, for |x| < 2^22: x + 1.5*2^23 lies in [2^23, 2^24)
// where fp32 values are the integers, so the sum is x rounded to an integer
// (ties to even, as 1.5*2^23 is even), and subtracting the constant is exact.
// For larger |x| the result is off by at most 2 (callers only use it there
// after a check that sends such x to the exact path).
__device__ __forceinline__ float rint_small(float x) {
    const float c = 12582912.0f;   // 1.5 * 2^23
    return __fsub_rn(__fadd_rn(x, c), c);
}

// rint(fp32(a / b)) wherever it can change a level, given rb = fp32(1 / b)
// correctly rounded.  Every caller clamps the result (plus a zero-point in
// 0..15) to 0..15, so only |a / b| < 32 needs the exact integer; beyond that
// any value of the same sign and at least 16 in magnitude clamps alike.
// t0 = fp32(a * rb) carries two roundings of at most 2^-24 relative each,
// so |t0 - fp32(a / b)| <= 3 * 2^-24 |t0| < 2^-16 for |t0| < 32.  Hence
// when t0 is more than 2^-16 away from the nearest half-integer (the test
// below), fp32(a / b) rounds to the same integer as t0.  Near a tie the
// quotient is formed by IEEE division.  For |t0| >= 32 the fast value keeps
// the sign and stays >= 16 in magnitude (rint_small errs by at most 2 past
// 2^22), so the clamped level is the same; Inf and NaN reach the same clamp
// on both paths.  The fast path uses no XU instruction.
constexpr float kTieBand = 0.4999847412109375f;   // 0.5 - 2^-16

__device__ __forceinline__ bool near_tie(float t0, float rt) {
    return fabsf(__fsub_rn(t0, rt)) > kTieBand;
}

__device__ __forceinline__ float rint_quot(float a, float b, float rb) {
    const float t0 = __fmul_rn(a, rb);
    const float rt = rint_small(t0);
    if (near_tie(t0, rt)) return rintf(__fdiv_rn(a, b));
    return rt;
}

// rint_quot for 8 values of one divisor (per lane; lanes may differ),
// without a branch per value: the fast roundings first, then -- only if some
// lane of the warp met a near-tie -- the exact quotient for those values.
// All 32 lanes of the warp must call it together (the vote).
__device__ __forceinline__ void rint_quot8(const float* a, float b, float rb, float* r) {
    bool tie = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float t0 = __fmul_rn(a[j], rb);
        r[j] = rint_small(t0);
        tie |= near_tie(t0, r[j]);
    }
    if (__any_sync(0xffffffffu, tie)) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (near_tie(__fmul_rn(a[j], rb), r[j])) r[j] = rintf(__fdiv_rn(a[j], b));
    }
}

struct GroupQuant {
    float scale;    // exact value of the fp16 scale
    float rcp;      // fp32(1 / scale), correctly rounded
    float zf;       // zero-point, an integer 0..15
    __half scale_h;
    bool finite;    // false when the fp16 scale overflowed
};

// Group parameters from the group's min and max (already reduced), for
// levels 0..qmax (15 at 4 bits, 7 at 3 bits): d = fp32(range / qmax) is one
// IEEE division whatever qmax is.
__device__ __forceinline__ GroupQuant group_quant_from_range(float lo, float hi,
                                                            float qmax = 15.0f) {
    GroupQuant g;
    float range = __fsub_rn(hi, lo);
    float d = __fdiv_rn(range, qmax);
    d = fmaxf(d, 6.103515625e-05f);              // 2^-14, least normal fp16
    g.scale_h = __float2half_rn(d);
    g.scale = __half2float(g.scale_h);
    g.finite = isfinite(g.scale);
    g.rcp = __frcp_rn(g.scale);
    // the zero-point is an integer level: -0 and negatives clamp to +0
    float z = rint_quot(-lo, g.scale, g.rcp);
    g.zf = z > 0.0f ? fminf(z, qmax) : 0.0f;
    return g;
}

// One warp holds a group, 4 scaled weights per lane.
__device__ __forceinline__ GroupQuant group_quant_params(float lo_lane, float hi_lane) {
    return group_quant_from_range(warp_min(lo_lane), warp_max(hi_lane));
}

__device__ __forceinline__ float quant_level(float wp, const GroupQuant& g) {
    const float t = rint_quot(wp, g.scale, g.rcp);
    return fminf(fmaxf(__fadd_rn(t, g.zf), 0.0f), 15.0f);
}

// (q - z) for a scaled weight: clamp(rint(w' / scale), -z, 15 - z), which is
// clamp(rint(w' / scale) + z, 0, 15) - z exactly (small integers).
__device__ __forceinline__ float quant_level_mz(float wp, float scale, float rcp, float neg_z,
                                                float top_z) {
    return fminf(fmaxf(rint_quot(wp, scale, rcp), neg_z), top_z);
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers, TMA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch: let the next kernel in the stream start
// beside this one; wait until the previous kernel has completed and its
// writes are visible (returns at once when not launched as a dependent).
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// after kWaitLimitNs or as soon as *abort is set by another thread; on
// giving up it sets *abort and the timeout status bit and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned* status,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort = 1;
                set_status(status, kStatusTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
// c0 is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// An L2 cache policy that keeps lines in L2 in preference to others.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_2d with an L2 cache policy for the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map,
                                                 uint64_t* bar, int c0, int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// 3-D tiled TMA load of one box (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// L2 policy for data read once: its lines are the first candidates for
// eviction, so a stream of weights does not push reused data out of L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Plain (untiled) bulk copy of `bytes` contiguous bytes from global to shared
// memory, completing on `bar`.  Both addresses 16-byte aligned and bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Ask L2 to fetch `bytes` contiguous bytes (16-byte aligned, a multiple of
// 16).  L2 is coherent with every SM's writes, so this is safe even ahead of
// a dependency on the kernel that writes the data: a line fetched early is
// updated in L2 by a later write, and the data are read only after the wait.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                     reinterpret_cast<uint64_t>(gsrc)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads, fences.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, fp16 inputs, fp32 accumulation.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Instruction descriptor for kind::f16: fp16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int M, int N) {
    return (1u << 4)                          // D format: f32
           | (0u << 7) | (0u << 10)           // A, B format: f16
           | (0u << 15) | (0u << 16)          // A, B K-major
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Shared-memory matrix descriptor of a K-major operand tile stored in the
// 128-byte swizzled layout: rows of 64 fp16 (128 B), 8-row atoms of 1024 B,
// atom base 1024-byte aligned.  `smem_addr` may be advanced by 32 B per
// 16-element K step inside the atom.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                        // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                        // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                        // layout: 128-byte swizzle
    return d;
}

// Byte offset of element (row, k) inside a [rows x 64] fp16 tile stored in
// the 128-byte swizzled layout (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t k) {
    return row * 128u + ((((k >> 3) ^ (row & 7u)) & 7u) << 4) + ((k & 7u) << 1);
}

// 32 lanes x 32 consecutive fp32 columns from TMEM (this warp's lane quarter).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Host: unique id of the calling thread's current CUDA context, 0 when it
// has none yet (defined in capi.cu).  Unlike a device ordinal or a context
// handle, an id is never reused within the process, so state that belongs
// to one context (symbol addresses, function attributes) is keyed on it and
// is looked up again in the new primary context after a cudaDeviceReset.
unsigned long long context_id();

// Host: raise a kernel's dynamic shared-memory limit once per device and
// context.  The attribute call is driver work on the launch path; repeating
// it per launch adds host latency that a short kernel cannot hide.
template <auto Kernel>
inline cudaError_t smem_attr_once(int bytes) {
    static std::atomic<unsigned long long> done_ctx[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long id = context_id();
    if (id != 0 && done_ctx[dev & 63].load(std::memory_order_acquire) == id) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done_ctx[dev & 63].store(context_id(), std::memory_order_release);
    return e;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace awq
