// ds41_common.cuh - shared device helpers and host-side error handling of
// libds41 (the CUDA path).  Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ds41.h"

namespace ds41 {

// ---------------------------------------------------------------------------
// Host-side error handling (ds41_common.cu)
// ---------------------------------------------------------------------------
int fail(int code, const char* fmt, ...);
int cuda_check(cudaError_t e, const char* what);
int launch_check(const char* what);
// Device address of the status word of the current device (set-up per device).
int status_word(unsigned int** out);
bool aligned16(const void* p);

#define DS41_REQUIRE(cond, code, ...)              \
    do {                                           \
        if (!(cond)) return ::ds41::fail((code), __VA_ARGS__); \
    } while (0)

// ---------------------------------------------------------------------------
// bf16 bit helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
__device__ __forceinline__ uint16_t f2bf(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));  // round to nearest even
}

// ---------------------------------------------------------------------------
// fp4 (e2m1) rounding, e8m0 and e4m3 scales
// ---------------------------------------------------------------------------
// Grid index 0..7 of {0,.5,1,1.5,2,3,4,6} nearest |t| (|t| <= 6 after the
// clamp).  A value on a midpoint goes to the neighbour with the even index, so
// each interval is closed on its even-index end.
__device__ __forceinline__ int e2m1_idx(float t) {
    const float a = fabsf(t);
    int i = 7;
    i = (a <= 5.0f) ? 6 : i;
    i = (a < 3.5f) ? 5 : i;
    i = (a <= 2.5f) ? 4 : i;
    i = (a < 1.75f) ? 3 : i;
    i = (a <= 1.25f) ? 2 : i;
    i = (a < 0.75f) ? 1 : i;
    i = (a <= 0.25f) ? 0 : i;
    return i;
}

// Magnitude of grid index i, as a float (exact): 0 and 0.5 below index 2,
// then (1 or 1.5) * 2^(i/2 - 1).
__device__ __forceinline__ float e2m1_mag(int i) {
    if (i < 2) return 0.5f * (float)i;
    const float m = (i & 1) ? 1.5f : 1.0f;
    return m * __uint_as_float((uint32_t)((i >> 1) + 126) << 23);
}

// 4-bit code: sign in bit 3 (taken from t, so a negative value that rounds to
// zero keeps its sign), index in bits 0..2.
__device__ __forceinline__ uint32_t e2m1_code(float t) {
    return ((__float_as_uint(t) >> 28) & 8u) | (uint32_t)e2m1_idx(t);
}

// Value of a code (signed, -0 preserved).
__device__ __forceinline__ float e2m1_val(uint32_t c) {
    const float m = e2m1_mag((int)(c & 7u));
    return (c & 8u) ? -m : m;
}

// Smallest power of two >= x, x a positive normal float.
__device__ __forceinline__ float pow2_ceil_pos(float x) {
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x007fffffu) == 0u) return x;
    return __uint_as_float((u & 0x7f800000u) + 0x00800000u);
}

// Entry j of the window part of query token t's index row, for a call of m
// tokens from start_pos (window win): the row that holds position
// q = start_pos + t - win + 1 + j, or -1 before position 0.  With no earlier
// positions the rows are the call's own kv rows (q); a single token reads the
// ring (slot q mod win); a chunk reads rows_a, the ring's old contents
// (slot q mod win) followed by the chunk's kv rows (win + q - start_pos).
__device__ __forceinline__ int32_t window_index(int64_t start_pos, int64_t m, int64_t win,
                                                int64_t t, int64_t j) {
    const int64_t q = start_pos + t - win + 1 + j;
    if (q < 0) return -1;
    if (start_pos == 0) return (int32_t)q;
    if (m == 1 || q < start_pos) {
        // q mod win, by a 32-bit division when both fit
        if (((q | win) >> 31) == 0) return (int32_t)((uint32_t)q % (uint32_t)win);
        return (int32_t)(q % win);
    }
    return (int32_t)(win + (q - start_pos));
}

// The power-of-two block scale s = pow2_ceil(amax / 6) (the quotient
// correctly rounded) and rs = 1/s, both exact, for an amax that is a bf16
// magnitude or the floor 6 * 2^-126 (at most 8 significant bits, normal).
// Writing amax = M 2^E with 1 <= M < 2: amax / 6 = (M / 1.5) 2^(E-2), so s is
// 2^(E-2) when M <= 1.5 and 2^(E-1) when M > 1.5; the rounded quotient never
// crosses the power of two, since M - 1.5 >= 2^-7 whenever it is positive.
// This holds for every positive finite bf16 magnitude (checked against the
// divide for all of them); an infinite amax takes the divide.
__device__ __forceinline__ float e8m0_scale_bf16(float amax, float* rs) {
    const uint32_t u = __float_as_uint(amax);
    if (u >= 0x7f800000u) {
        const float s = pow2_ceil_pos(__fdiv_rn(amax, 6.0f));
        *rs = __frcp_rn(s);
        return s;
    }
    const uint32_t e = (u >> 23) - 2u + ((u & 0x007fffffu) > 0x00400000u ? 1u : 0u);
    *rs = __uint_as_float((254u - e) << 23);
    return __uint_as_float(e << 23);
}

// f32 -> e4m3 (OCP "fn") with round-to-nearest-even and saturation at the
// largest finite value (448), via the hardware conversion.  Returns the byte.
__device__ __forceinline__ uint32_t f32_to_e4m3_sat(float x) {
    uint16_t r;
    // cvt packs two inputs: the first operand lands in the upper byte.
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
    return (uint32_t)(r & 0xffu);
}

// e4m3 byte -> f32 (exact), via the hardware conversion to f16.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
    uint32_t h2;
    const uint16_t in = (uint16_t)(c & 0xffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((uint16_t)(h2 & 0xffffu)));
}

// One element of the fp4 round trip with scale s: clamp(v/s) -> e2m1 -> * s.
// Division and product are single IEEE operations (never contracted).
__device__ __forceinline__ float fp4_elem(float v, float s, uint32_t* code) {
    float t = __fdiv_rn(v, s);
    t = fminf(fmaxf(t, -6.0f), 6.0f);
    const uint32_t c = e2m1_code(t);
    *code = c;
    return __fmul_rn(e2m1_val(c), s);
}

// The same element path for a power-of-two scale s with rs = 1/s (exact for
// a power of two, subnormal results included): v * rs rounds exactly as v / s.
__device__ __forceinline__ float fp4_elem_pow2(float v, float s, float rs, uint32_t* code) {
    float t = __fmul_rn(v, rs);
    t = fminf(fmaxf(t, -6.0f), 6.0f);
    const uint32_t c = e2m1_code(t);
    *code = c;
    return __fmul_rn(e2m1_val(c), s);
}

// Hardware e2m1 conversion: two f32 values -> two 4-bit codes (round to
// nearest, ties to the even code, saturating at +-6; a negative value that
// rounds to zero keeps its sign).  The first value lands in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint16_t r;
    asm("{\n.reg .b8 b0;\ncvt.rn.satfinite.e2m1x2.f32 b0, %1, %2;\nmov.b16 %0, {b0, b0};\n}"
        : "=h"(r)
        : "f"(hi), "f"(lo));
    return (uint32_t)(r & 0xffu);
}

// Two e2m1 codes (one byte, first element in the low nibble) -> their exact
// values as two floats.
__device__ __forceinline__ float2 e2m1x2_to_float2(uint32_t byte) {
    uint32_t h2;
    const uint16_t in = (uint16_t)(byte & 0xffu);
    asm("{\n.reg .b8 b0, b1;\nmov.b16 {b0, b1}, %1;\ncvt.rn.f16x2.e2m1x2 %0, b0;\n}"
        : "=r"(h2)
        : "h"(in));
    return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// The fp4 round trip of 8 values t[] already divided by their block scale s:
// codes (element k in nibble k) and bf16(e2m1(t) * s) packed in a uint4.
// |t| > 6 saturates to 6, which is what clamping first and rounding gives.
__device__ __forceinline__ uint4 e2m1_round8(const float t[8], float s, uint32_t* codes) {
    uint32_t c = 0;
#pragma unroll
    for (int k = 0; k < 8; k += 2) c |= cvt_e2m1x2(t[k], t[k + 1]) << (4 * k);
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        const float2 g = e2m1x2_to_float2(c >> (4 * k));
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(g.x, s), __fmul_rn(g.y, s));
        o[k / 2] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *codes = c;
    return out;
}

// ---------------------------------------------------------------------------
// Vector loads / stores and async copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ---------------------------------------------------------------------------
// Warp-level bf16 tensor-core helpers (m16n8k16, f32 accumulate)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const uint32_t l = f2bf(lo), h = f2bf(hi);
    return l | (h << 16);
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor on the stream finishes;
// pdl_wait() blocks until the predecessor has completed and its writes are
// visible (a no-op without such a predecessor), pdl_trigger() lets the next
// kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The rule every kernel of the library follows: pdl_wait() comes before the
// first global memory access, and pdl_trigger() after pdl_wait(), so that a
// kernel launches only once everything two places before it in the stream
// has completed.  The one exception that reads before its wait is the
// few-token attention (q, an input of the step); every kernel that precedes it
// waits before triggering.  The few-token attention and the host copy kernel
// trigger first: every kernel that can follow them waits before touching
// memory.  The long persistent tensor-core kernels trigger only when a CTA's
// work is done, not at their start: their dependents' CTAs would otherwise
// sit resident and waiting beside them for their whole run (measured: the
// prefill step 708 -> 724 us with early triggers).

// Launch with programmatic stream serialization (the kernel calls pdl_wait()
// before its first global memory access).
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      const char* what, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int rc = cuda_check(cudaLaunchKernelEx(&cfg, kern, args...), what);
    if (rc) return rc;
    return launch_check(what);
}

// ---------------------------------------------------------------------------
// mbarriers and TMA bulk copies (global -> shared, completion by byte count)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// make barrier initialisation visible to the async proxy and the cluster
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// One contiguous copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global memory into this CTA's shared memory; completes
// `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Wait for phase `parity` of `bar` to complete, giving up after max_iter
// polls (each poll may suspend the thread for a short while).  Returns false
// on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t max_iter) {
    for (uint32_t i = 0; i < max_iter; i++) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}
constexpr uint32_t kWaitPolls = 1u << 22;  // bound of every mbarrier wait (~1 s)

// The shared::cluster address of `p` (this CTA's shared memory) in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// One bulk copy of `bytes` (a multiple of 16, both ends 16-byte aligned) from
// this CTA's shared memory into another CTA's, completing `bytes`
// transactions on the mbarrier at cluster address `bar` (in the receiver).
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];\n" ::"r"(dst),
        "r"(smem_u32(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Raise a DS41_E_* code in the device status word (first error wins).
__device__ __forceinline__ void raise_status(unsigned int* status, unsigned int code) {
    if (status) atomicCAS(status, 0u, code);
}

}  // namespace ds41
