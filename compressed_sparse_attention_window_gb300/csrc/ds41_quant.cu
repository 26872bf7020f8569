// ds41_quant.cu - the two fp4 block quantisers and the YaRN RoPE table.
//
// metrale_model_arch/deepseek_v41_ref/compress.rs: fp4_quant_e8m0_inplace
// (power-of-two scales, block 32), fp4_quant_e4m3_inplace (e4m3 scales, block
// 16), yarn_freqs_cis.
#include <math.h>

#include "ds41_common.cuh"

namespace ds41 {

// Each thread owns 8 consecutive values (one 16-byte load); a block of BLOCK
// values spans BLOCK/8 neighbouring lanes, which reduce amax with shuffles.
template <int BLOCK, bool E4M3>
__global__ void __launch_bounds__(256) fp4_quant_kernel(const uint4* __restrict__ x,
                                                        uint4* __restrict__ y,
                                                        uint32_t* __restrict__ codes,
                                                        uint8_t* __restrict__ scales,
                                                        int64_t n8) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    pdl_trigger();
    constexpr int LANES = BLOCK / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // Threads past the end still take part in the shuffles (n8 is a multiple
    // of LANES, so a whole block is either in or out).
    const bool live = i < n8;
    uint4 raw = live ? x[i] : make_uint4(0, 0, 0, 0);
    const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
    float v[8];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        v[k] = bf2f(h[k]);
        amax = fmaxf(amax, fabsf(v[k]));
    }
#pragma unroll
    for (int off = 1; off < LANES; off <<= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float s;
    uint32_t sbyte;
    float rs = 0.0f;
    if (E4M3) {
        amax = fmaxf(amax, 0.01171875f);  // 6 * 2^-9
        sbyte = f32_to_e4m3_sat(__fdiv_rn(amax, 6.0f));
        s = e4m3_to_f32(sbyte);
    } else {
        amax = fmaxf(amax, __uint_as_float(0x01c00000u));  // 6 * 2^-126
        s = e8m0_scale_bf16(amax, &rs);  // amax: a bf16 magnitude or the floor
        sbyte = (__float_as_uint(s) >> 23) & 0xffu;  // biased exponent = e8m0
    }
    if (!live) return;
    float tq[8];
#pragma unroll
    for (int k = 0; k < 8; k++) tq[k] = E4M3 ? __fdiv_rn(v[k], s) : __fmul_rn(v[k], rs);
    uint32_t packed;
    const uint4 out = e2m1_round8(tq, s, &packed);
    y[i] = out;
    if (codes) codes[i] = packed;
    if (scales && (threadIdx.x % LANES) == 0) scales[i / LANES] = (uint8_t)sbyte;
}

template <int BLOCK, bool E4M3>
static int quant_launch(const ds41_bf16* x, ds41_bf16* y, uint8_t* codes, uint8_t* scales,
                        int64_t rows, int64_t cols, ds41_stream_t stream, const char* name) {
    DS41_REQUIRE(x && y, DS41_E_ARG, "%s: x and y must be non-null", name);
    DS41_REQUIRE(rows >= 0 && cols >= 0, DS41_E_ARG, "%s: negative size", name);
    DS41_REQUIRE(cols % BLOCK == 0, DS41_E_ARG, "%s: cols=%lld is not a multiple of %d", name,
                 (long long)cols, BLOCK);
    DS41_REQUIRE(rows * cols < (int64_t(1) << 31), DS41_E_ARG, "%s: tensor too large", name);
    DS41_REQUIRE(aligned16(x) && aligned16(y), DS41_E_ARG, "%s: x/y not 16-byte aligned", name);
    DS41_REQUIRE(!codes || (reinterpret_cast<uintptr_t>(codes) & 3u) == 0, DS41_E_ARG,
                 "%s: codes not 4-byte aligned", name);
    const int64_t n8 = rows * cols / 8;
    if (n8 == 0) return DS41_OK;
    const int threads = 256;
    const int64_t blocks = (n8 + threads - 1) / threads;
    return launch_pdl(fp4_quant_kernel<BLOCK, E4M3>, dim3((unsigned)blocks), dim3(threads), 0,
                      (cudaStream_t)stream, name, reinterpret_cast<const uint4*>(x),
                      reinterpret_cast<uint4*>(y), reinterpret_cast<uint32_t*>(codes), scales, n8);
}

// ---------------------------------------------------------------------------
// YaRN RoPE table.  One thread per (position, frequency).  The frequency is
// recomputed by every thread (a handful of flops); pow, cos and sin are taken
// in double and rounded once, which gives the correctly rounded f32 value in
// all but vanishingly rare cases.
// ---------------------------------------------------------------------------
__device__ float yarn_freq(int k, int dim, float lo, float span, float base, float factor) {
    const float ex = __fdiv_rn((float)(2 * k), (float)dim);
    const float pw = (float)pow((double)base, (double)ex);
    const float f = __fdiv_rn(1.0f, pw);
    float ramp = __fdiv_rn(__fsub_rn((float)k, lo), span);
    ramp = fminf(fmaxf(ramp, 0.0f), 1.0f);
    const float keep = __fsub_rn(1.0f, ramp);
    const float scaled = __fdiv_rn(f, factor);
    return __fadd_rn(__fmul_rn(scaled, __fsub_rn(1.0f, keep)), __fmul_rn(f, keep));
}

__global__ void yarn_table_kernel(float2* __restrict__ out, int64_t seqlen, int dim, float lo,
                                  float span, float base, float factor) {
    const int half = dim / 2;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= seqlen * half) return;
    const int k = (int)(i % half);
    const int64_t p = i / half;
    const float f = yarn_freq(k, dim, lo, span, base, factor);
    const float ang = __fmul_rn((float)p, f);
    double sd, cd;
    sincos((double)ang, &sd, &cd);
    out[i] = make_float2((float)cd, (float)sd);
}

}  // namespace ds41

using namespace ds41;

extern "C" int ds41_fp4_quant_e8m0(const ds41_bf16* x, ds41_bf16* y, uint8_t* codes,
                                   uint8_t* scales, int64_t rows, int64_t cols,
                                   ds41_stream_t stream) {
    return quant_launch<32, false>(x, y, codes, scales, rows, cols, stream, "ds41_fp4_quant_e8m0");
}

extern "C" int ds41_fp4_quant_e4m3(const ds41_bf16* x, ds41_bf16* y, uint8_t* codes,
                                   uint8_t* scales, int64_t rows, int64_t cols,
                                   ds41_stream_t stream) {
    return quant_launch<16, true>(x, y, codes, scales, rows, cols, stream, "ds41_fp4_quant_e4m3");
}

extern "C" int ds41_yarn_freqs_cis(float* out, int64_t dim, int64_t seqlen,
                                   int64_t original_seq_len, float base, float factor,
                                   float beta_fast, float beta_slow, ds41_stream_t stream) {
    const char* name = "ds41_yarn_freqs_cis";
    DS41_REQUIRE(out, DS41_E_ARG, "%s: out is NULL", name);
    DS41_REQUIRE(dim >= 2 && dim % 2 == 0 && dim <= 4096, DS41_E_ARG, "%s: dim=%lld", name,
                 (long long)dim);
    DS41_REQUIRE(seqlen >= 0 && seqlen <= (int64_t(1) << 24), DS41_E_ARG, "%s: seqlen=%lld",
                 name, (long long)seqlen);
    DS41_REQUIRE(original_seq_len > 0 && base > 1.0f && factor > 0.0f && beta_fast > 0.0f &&
                     beta_slow > 0.0f,
                 DS41_E_ARG, "%s: bad YaRN constants", name);
    // The correction range is taken in double, as the page does, on the host
    // (two scalars per table, not per element).
    const double two_pi = 6.283185307179586476925286766559;
    auto corr = [&](double rot) {
        return (double)dim * log((double)original_seq_len / (rot * two_pi)) /
               (2.0 * log((double)base));
    };
    const float lo = (float)fmax(floor(corr((double)beta_fast)), 0.0);
    const float hi = (float)fmin(ceil(corr((double)beta_slow)), (double)(dim - 1));
    const float span = fmaxf(hi - lo, 1e-3f);
    const int64_t n = seqlen * (dim / 2);
    if (n == 0) return DS41_OK;
    const int threads = 256;
    yarn_table_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0,
                         (cudaStream_t)stream>>>(reinterpret_cast<float2*>(out), seqlen, (int)dim,
                                                 lo, span, base, factor);
    return launch_check(name);
}
