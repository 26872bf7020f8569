// ds41_out_proj.cu - the output side of the layer: o rotated back (inverse
// RoPE at each token's position), the grouped wo_a projection rounded to
// bf16, and the wo_b projection.
//
// metrale_model_arch/deepseek_v41_ref/compress.rs, attention_any after
// sparse_attn: apply_rotary(o, .., inverse = true) with each head at its
// token's position; o split into `groups` groups of nh*hd/groups values, each
// projected by its own o_rank rows of wo_a and rounded to bf16 (to_bf16_rne);
// then linear_bf16 with wo_b [dim, groups*o_rank].
//
// Design.  The rotation touches the last rd dims of every head only, so one
// small kernel rotates those pairs back in place (each product rounded, then
// the sum, as the forward rotation of the latent rows) and rounds them to
// bf16, the operand type of the tensor cores.  The two projections are plain
// GEMMs and go to cuBLAS: a strided batch of `groups` products (bf16 in, f32
// accumulation, bf16 out, which is the rounding the definition asks for) and
// one product with an f32 result.
#include <cublas_v2.h>

#include <mutex>

#include "ds41_common.cuh"

namespace ds41 {

// One thread per rotary pair (token t, head h, pair i): the pair at dims
// hd - rd + 2 i, + 1 of head h rotated by table column i of position
// start_pos + t with the angle negated.
__global__ void inv_rope_kernel(uint16_t* o, const float2* fc, int64_t m, int nh, int hd, int rd,
                                int64_t start_pos) {
    const int half = rd / 2;
    const int64_t total = m * nh * half;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total;
         k += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(k % half);
        const int64_t th = k / half;  // t * nh + h
        const int64_t t = th / nh;
        uint32_t* pr = reinterpret_cast<uint32_t*>(o + th * hd + (hd - rd) + 2 * i);
        const uint32_t v = *pr;
        const float x0 = bf2f((uint16_t)(v & 0xffffu)), x1 = bf2f((uint16_t)(v >> 16));
        const float2 cs = fc[(start_pos + t) * half + i];
        const float c = cs.x, s = -cs.y;
        const float y0 = __fsub_rn(__fmul_rn(x0, c), __fmul_rn(x1, s));
        const float y1 = __fadd_rn(__fmul_rn(x0, s), __fmul_rn(x1, c));
        *pr = (uint32_t)f2bf(y0) | ((uint32_t)f2bf(y1) << 16);
    }
}

// One cuBLAS handle for the library, used under a lock (a handle serves one
// call at a time; the stream is set per call).
static std::mutex g_blas_mu;
static cublasHandle_t g_blas = nullptr;

static int blas_check(cublasStatus_t s, const char* what) {
    if (s == CUBLAS_STATUS_SUCCESS) return DS41_OK;
    return fail(DS41_E_CUDA, "%s: cuBLAS status %d", what, (int)s);
}

}  // namespace ds41

using namespace ds41;

extern "C" int ds41_attn_out_proj(ds41_bf16* o, const float* freqs_cis, int64_t max_pos,
                                  const ds41_bf16* wo_a, const ds41_bf16* wo_b, ds41_bf16* og,
                                  float* out, int64_t m, int64_t start_pos, int64_t nh, int64_t hd,
                                  int64_t rd, int64_t groups, int64_t o_rank, int64_t dim,
                                  ds41_stream_t stream) {
    const char* name = "ds41_attn_out_proj";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 31), DS41_E_RANGE, "%s: m=%lld", name, (long long)m);
    DS41_REQUIRE(start_pos >= 0 && start_pos + m <= max_pos, DS41_E_RANGE,
                 "%s: positions %lld .. %lld are past the %lld rows of freqs_cis", name,
                 (long long)start_pos, (long long)(start_pos + m - 1), (long long)max_pos);
    DS41_REQUIRE(nh >= 1 && hd >= 8 && hd % 8 == 0 && rd >= 0 && rd % 2 == 0 && rd <= hd,
                 DS41_E_ARG, "%s: nh=%lld hd=%lld rd=%lld", name, (long long)nh, (long long)hd,
                 (long long)rd);
    DS41_REQUIRE(groups >= 1 && (nh * hd) % groups == 0 && ((nh * hd) / groups) % 8 == 0,
                 DS41_E_ARG, "%s: groups=%lld must split nh*hd=%lld into multiples of 8", name,
                 (long long)groups, (long long)(nh * hd));
    DS41_REQUIRE(o_rank >= 1 && (groups * o_rank) % 8 == 0 && dim >= 1 && dim % 4 == 0, DS41_E_ARG,
                 "%s: o_rank=%lld dim=%lld (groups*o_rank a multiple of 8, dim of 4)", name,
                 (long long)o_rank, (long long)dim);
    DS41_REQUIRE(nh * hd < (int64_t(1) << 31) && groups * o_rank < (int64_t(1) << 31) &&
                     dim < (int64_t(1) << 31),
                 DS41_E_ARG, "%s: sizes beyond 32-bit GEMM dimensions", name);
    DS41_REQUIRE(o && wo_a && wo_b && og && out && (rd == 0 || freqs_cis), DS41_E_ARG,
                 "%s: o, wo_a, wo_b, og, out (and freqs_cis when rd > 0) must be non-null", name);
    DS41_REQUIRE(aligned16(o) && aligned16(wo_a) && aligned16(wo_b) && aligned16(og) &&
                     aligned16(out) && (rd == 0 || aligned16(freqs_cis)),
                 DS41_E_ARG, "%s: every pointer must be 16-byte aligned", name);
    cudaStream_t st = (cudaStream_t)stream;
    if (rd > 0) {
        const int64_t pairs = m * nh * (rd / 2);
        const int threads = 256;
        const int64_t blocks = (pairs + threads - 1) / threads;
        inv_rope_kernel<<<(unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16), threads, 0, st>>>(
            reinterpret_cast<uint16_t*>(o), reinterpret_cast<const float2*>(freqs_cis), m, (int)nh,
            (int)hd, (int)rd, start_pos);
        if (int rc = launch_check(name)) return rc;
    }
    const int gw = (int)((nh * hd) / groups), gr = (int)(groups * o_rank);
    const float one = 1.0f, zero = 0.0f;
    std::lock_guard<std::mutex> lk(g_blas_mu);
    if (!g_blas) {
        if (int rc = blas_check(cublasCreate(&g_blas), "ds41_attn_out_proj: cublasCreate")) {
            g_blas = nullptr;
            return rc;
        }
    }
    if (int rc = blas_check(cublasSetStream(g_blas, st), name)) return rc;
    // og[t, g*o_rank + r] = bf16(sum_i o[t, g*gw + i] wo_a[g*o_rank + r, i]): column-major,
    // og^T_g [o_rank, m] = wo_a_g [o_rank, gw] . o_g^T [gw, m], one batch entry per group
    if (int rc = blas_check(
            cublasGemmStridedBatchedEx(g_blas, CUBLAS_OP_T, CUBLAS_OP_N, (int)o_rank, (int)m, gw,
                                       &one, wo_a, CUDA_R_16BF, gw, (long long)o_rank * gw, o,
                                       CUDA_R_16BF, (int)(nh * hd), (long long)gw, &zero, og,
                                       CUDA_R_16BF, gr, (long long)o_rank, (int)groups,
                                       CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT),
            "ds41_attn_out_proj: grouped wo_a product"))
        return rc;
    // out [m, dim] = og . wo_b^T: column-major out^T [dim, m] = wo_b [dim, gr] . og^T [gr, m]
    if (int rc = blas_check(cublasGemmEx(g_blas, CUBLAS_OP_T, CUBLAS_OP_N, (int)dim, (int)m, gr,
                                         &one, wo_b, CUDA_R_16BF, gr, og, CUDA_R_16BF, gr, &zero,
                                         out, CUDA_R_32F, (int)dim, CUBLAS_COMPUTE_32F,
                                         CUBLAS_GEMM_DEFAULT),
                            "ds41_attn_out_proj: wo_b product"))
        return rc;
    return DS41_OK;
}
