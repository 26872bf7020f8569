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
// bf16, the operand type of the tensor cores.  Both projections are one
// operation, a grouped linear map
//   Y[t, n] = sum_{k < Kd} X[t, (n / rows_per_group) Kd + k] W[n, k]
// (wo_a: X = o, Kd = gw, rows_per_group = o_rank, Y = og rounded to bf16;
// wo_b: X = og, Kd = groups o_rank, one group, Y = out in f32), in one of two
// kernels:
// * few tokens (the weights streamed once from HBM dominate): a warp per
//   weight row reads it with 16-byte loads, four in flight per lane, and
//   keeps one f32 partial sum per token; a warp reduction finishes the row.
// * many tokens (a dense contraction): tcgen05 tiles of 128 weight rows x
//   BN tokens (D = W X^T, the weight rows on the lanes of D), 64-wide K steps
//   through a 4-stage TMA pipeline, two accumulators in tensor memory so the
//   epilogue of one tile overlaps the MMAs of the next, persistent CTAs
//   walking the weight-row tiles of one token block before the next (the
//   weights stay in L2 across token blocks).
#include "ds41_tc.cuh"

namespace ds41 {

// One thread per rotary pair (token t, head h, pair i): the pair at dims
// hd - rd + 2 i, + 1 of head h rotated by table column i of position
// start_pos + t with the angle negated.
__global__ void inv_rope_kernel(uint16_t* o, const float2* fc, int64_t m, int nh, int hd, int rd,
                                int64_t start_pos) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    pdl_trigger();
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

// The grouped linear map of the few-token kernel and the tensor-core kernel.
struct Lin {
    const uint16_t* X;     // [m][ldx] bf16
    const uint16_t* W;     // [N][Kd] bf16
    void* Y;               // [m][N]: bf16 (RNE) or f32
    int64_t ldx, N;
    int Kd, rows_per_group, m;
    int out_bf16;
};

// ---------------------------------------------------------------------------
// Few tokens: a warp per weight row, MT tokens at a time
// ---------------------------------------------------------------------------
constexpr int GEMV_THREADS = 256;
constexpr int GEMV_UNROLL = 4;  // 16-byte loads of the row in flight per lane

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void dot8(float& acc, uint4 w, uint4 x) {
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w}, xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int e = 0; e < 4; e++) {
        acc = __fmaf_rn(__uint_as_float(wv[e] << 16), __uint_as_float(xv[e] << 16), acc);
        acc = __fmaf_rn(__uint_as_float(wv[e] & 0xffff0000u), __uint_as_float(xv[e] & 0xffff0000u),
                        acc);
    }
}

template <int MT>
__global__ void __launch_bounds__(GEMV_THREADS) proj_gemv_kernel(Lin a, int t0) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * GEMV_THREADS + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * GEMV_THREADS) >> 5;
    const int mt = min(MT, a.m - t0);
    const int k8 = a.Kd / 8;  // 16-byte vectors per row
    for (int64_t n = warp; n < a.N; n += nwarps) {
        const uint4* wr = reinterpret_cast<const uint4*>(a.W + n * a.Kd);
        const int64_t xoff = (n / a.rows_per_group) * a.Kd;
        float acc[MT];
#pragma unroll
        for (int t = 0; t < MT; t++) acc[t] = 0.0f;
        for (int v0 = lane; v0 < k8; v0 += 32 * GEMV_UNROLL) {
            uint4 wv[GEMV_UNROLL];
#pragma unroll
            for (int u = 0; u < GEMV_UNROLL; u++) {
                const int v = v0 + 32 * u;
                wv[u] = v < k8 ? ld_stream(wr + v) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < GEMV_UNROLL; u++) {
                const int v = v0 + 32 * u;
                if (v >= k8) break;
#pragma unroll
                for (int t = 0; t < MT; t++) {
                    if (t < mt) {
                        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(
                                                   a.X + (int64_t)(t0 + t) * a.ldx + xoff) + v);
                        dot8(acc[t], wv[u], xv);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < MT; t++) {
            float s = acc[t];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            acc[t] = s;
        }
        if (lane == 0) {
            for (int t = 0; t < mt; t++) {
                const int64_t at = (int64_t)(t0 + t) * a.N + n;
                if (a.out_bf16) reinterpret_cast<uint16_t*>(a.Y)[at] = f2bf(acc[t]);
                else reinterpret_cast<float*>(a.Y)[at] = acc[t];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Many tokens: tcgen05 tiles D[128 weight rows][BN tokens] = W X^T
// ---------------------------------------------------------------------------
namespace pj {

using namespace tc;

constexpr int BM = 128;            // weight rows per tile (the lanes of D)
constexpr int BK = 64;             // K per stage (one 128-byte swizzled row)
constexpr int STAGES = 4;
constexpr int THREADS = 256;       // warp 0 TMA, warp 1 MMA, warps 4..7 epilogue
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KiB

template <int BN>
struct Cfg {
    static constexpr uint32_t B_BYTES = BN * BK * 2;
    static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
    static constexpr uint32_t BAR_OFF = STAGES * STAGE;
    static constexpr uint32_t SMEM = BAR_OFF + 256 + 1024;
    static constexpr uint32_t IDESC = idesc_bf16(BM, BN, 0, 0);
    static_assert(SMEM <= 232448, "shared memory budget");
};

enum { B_FULL, B_EMPTY = B_FULL + STAGES, B_AFULL = B_EMPTY + STAGES, B_AEMPTY = B_AFULL + 2,
       B_FINAL = B_AEMPTY + 2, NBAR };

struct Params {
    Lin a;
    int n_mt, n_nt;  // weight-row tiles, token tiles
    unsigned int* status;
};

// One CTA per SM walks its tiles: D[128 weight rows][BN tokens] in tensor
// memory (two accumulators), the K steps through STAGES shared-memory stages.
template <int BN>
__global__ void __launch_bounds__(THREADS, 1)
    proj_tc_kernel(const __grid_constant__ CUtensorMap map_w,
                   const __grid_constant__ CUtensorMap map_x, const Params p) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::BAR_OFF + NBAR * 8);
    volatile int* abort_f = reinterpret_cast<volatile int*>(sm + C::BAR_OFF + NBAR * 8 + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = p.n_mt * p.n_nt;
    const int ksteps = p.a.Kd / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&bars[B_FULL + s], 1);
            mbar_init(&bars[B_EMPTY + s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&bars[B_AFULL + b], 1);
            mbar_init(&bars[B_AEMPTY + b], 4);
        }
        mbar_init(&bars[B_FINAL], 1);
        *abort_f = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(
                smem_u32(tmem_slot))
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0, armed[STAGES] = {};
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
                const int mt = tile % p.n_mt, nt = tile / p.n_mt;
                const int g = (mt * BM) / p.a.rows_per_group;
                for (int k = 0; k < ksteps; k++, it++) {
                    const int s = it % STAGES;
                    if (it >= STAGES && !wait_bar(&bars[B_EMPTY + s], ((it / STAGES) - 1) & 1,
                                                  abort_f, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[B_FULL + s], C::STAGE);
                    armed[s]++;
                    const uint32_t st = sbase + s * C::STAGE;
                    tma_load_2d(st, &map_w, k * BK, mt * BM, &bars[B_FULL + s]);
                    tma_load_2d(st + A_BYTES, &map_x, g * p.a.Kd + k * BK, nt * BN,
                                &bars[B_FULL + s]);
                }
            }
            for (int s = 0; s < STAGES; s++)
                if (armed[s]) drain_bar(&bars[B_FULL + s], (armed[s] - 1) & 1, p.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t it = 0, lt = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x, lt++) {
                const int ab = lt & 1;
                if (lt >= 2 &&
                    !wait_bar(&bars[B_AEMPTY + ab], ((lt - 2) >> 1) & 1, abort_f, p.status))
                    break;
                const uint32_t d = tmem + 256 * ab;
                for (int k = 0; k < ksteps; k++, it++) {
                    const int s = it % STAGES;
                    if (!wait_bar(&bars[B_FULL + s], (it / STAGES) & 1, abort_f, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = sbase + s * C::STAGE;
                    const uint64_t ad = sdesc(st, 16, 1024), bd = sdesc(st + A_BYTES, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; kk++)
                        tc_mma(d, ad + ((kk * 32) >> 4), bd + ((kk * 32) >> 4), C::IDESC,
                               (k > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&bars[B_EMPTY + s]);
                }
                if (ok) tc_commit(&bars[B_AFULL + ab]);
            }
            tc_commit(&bars[B_FINAL]);
            drain_bar(&bars[B_FINAL], 0, p.status);
        }
    } else if (warp >= 4) {
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        uint32_t lt = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, lt++) {
            const int ab = lt & 1;
            if (!wait_bar(&bars[B_AFULL + ab], (lt >> 1) & 1, abort_f, p.status)) break;
            tc_fence_after();
            const int mt = tile % p.n_mt, nt = tile / p.n_mt;
            const int64_t n = (int64_t)mt * BM + 32 * q + lane;
            const int tbase = nt * BN;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t r[32];
                tc_ld32(tmem + lane_off + 256 * ab + c0, r);
                tc_wait_ld();
                if (c0 + 32 >= BN) {  // the accumulator is in registers: release it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_AEMPTY + ab]);
                }
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    const int t = tbase + c0 + j;
                    if (t < p.a.m) {
                        const int64_t at = (int64_t)t * p.a.N + n;
                        if (p.a.out_bf16)
                            reinterpret_cast<uint16_t*>(p.a.Y)[at] = f2bf(__uint_as_float(r[j]));
                        else
                            reinterpret_cast<float*>(p.a.Y)[at] = __uint_as_float(r[j]);
                    }
                }
            }
        }
    }

    // a long persistent kernel: its dependents may start launching once this
    // CTA's work is done (an early trigger would keep their CTAs resident and
    // waiting beside this kernel for its whole run)
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem)
                     : "memory");
}

template <int BN>
int launch_tc(const Lin& a, int sms, unsigned int* status, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int rc = get_encode(&enc);
    if (rc) return rc;
    CUtensorMap mw, mx;
    if ((rc = make_map_bf16(enc, &mw, a.W, a.N, a.Kd, BK, BM))) return rc;
    if ((rc = make_map_bf16(enc, &mx, a.X, a.m, a.ldx, BK, BN))) return rc;
    Params p;
    p.a = a;
    p.n_mt = (int)(a.N / BM);
    p.n_nt = (a.m + BN - 1) / BN;
    p.status = status;
    const int ntiles = p.n_mt * p.n_nt;
    const int grid = ntiles < sms ? ntiles : sms;
    rc = cuda_check(cudaFuncSetAttribute(proj_tc_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cfg<BN>::SMEM),
                    "ds41_attn_out_proj: tensor-core kernel attributes");
    if (rc) return rc;
    return launch_pdl(proj_tc_kernel<BN>, dim3((unsigned)grid), dim3(THREADS), Cfg<BN>::SMEM, st,
                      "ds41_attn_out_proj: tensor-core projection", mw, mx, p);
}

}  // namespace pj

static int device_sms() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

constexpr int GEMV_MAX_M = 16;  // up to here the weight stream dominates

// One grouped linear map: few tokens on the CUDA cores, many on tcgen05.
static int run_lin(const Lin& a, cudaStream_t st) {
    const int sms = device_sms();
    const bool tc_shape = a.N % pj::BM == 0 && a.rows_per_group % pj::BM == 0 &&
                          a.Kd % pj::BK == 0 && a.ldx % 8 == 0;
    if (a.m > GEMV_MAX_M && tc_shape) {
        unsigned int* status = nullptr;
        int rc = status_word(&status);
        if (rc) return rc;
        if (a.m <= 64) return pj::launch_tc<64>(a, sms, status, st);
        if (a.m <= 128) return pj::launch_tc<128>(a, sms, status, st);
        return pj::launch_tc<256>(a, sms, status, st);
    }
    const int64_t warps = a.N;
    int64_t blocks = (warps * 32 + GEMV_THREADS - 1) / GEMV_THREADS;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    // tokens in chunks of up to 8: the smallest kernel that covers the chunk
    for (int t0 = 0; t0 < a.m; t0 += 8) {
        const int rem = a.m - t0;
        auto kern = rem > 4 ? proj_gemv_kernel<8>
                    : rem > 2 ? proj_gemv_kernel<4>
                    : rem > 1 ? proj_gemv_kernel<2>
                              : proj_gemv_kernel<1>;
        if (int rc = launch_pdl(kern, dim3((unsigned)blocks), dim3(GEMV_THREADS), 0, st,
                                "ds41_attn_out_proj: projection", a, t0))
            return rc;
    }
    return DS41_OK;
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
        if (int rc = launch_pdl(inv_rope_kernel,
                                dim3((unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16)),
                                dim3(threads), 0, st, name, reinterpret_cast<uint16_t*>(o),
                                reinterpret_cast<const float2*>(freqs_cis), m, (int)nh, (int)hd,
                                (int)rd, start_pos))
            return rc;
    }
    const int gw = (int)((nh * hd) / groups), gr = (int)(groups * o_rank);
    // og[t, g*o_rank + r] = bf16(sum_i o[t, g*gw + i] wo_a[g*o_rank + r, i])
    Lin a1{o, wo_a, og, nh * hd, gr, gw, (int)o_rank, (int)m, 1};
    if (int rc = run_lin(a1, st)) return rc;
    // out[t, j] = sum_k og[t, k] wo_b[j, k]
    Lin a2{og, wo_b, out, gr, dim, gr, (int)dim, (int)m, 0};
    return run_lin(a2, st);
}
