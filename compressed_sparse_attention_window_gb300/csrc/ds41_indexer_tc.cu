// ds41_indexer_tc.cu - the fp4 indexer scores of many query tokens on the
// 5th-generation tensor cores (tcgen05), for 64 indexer heads of dim 128.
//
// metrale_model_arch/attn_v41/forward.rs calls the indexer; the header of
// metrale_model_arch/deepseek_v41_ref/compress.rs fixes its precision (q and
// k take the e2m1 round trip with power-of-two scales per block of 32, the
// scores are bf16).  Score of query t against compressed row s, for
// s < (start_pos + t + 1) / ratio:
//   acc = 0; for h in 0..63: acc = fma(w[t,h], max(<qh[t,h], kh[s]>, 0), acc)
//   score = bf16(acc)          (-0 -> +0; rows not visible yet score -inf)
//
// The quantised k arrives as bf16 values, q as it is: the kernel takes each
// group's q through the same round trip in shared memory (each fp4 value
// times its power-of-two scale is exact in bf16), so one bf16 MMA gives the
// dot products; they are exact in f32, so any summation order gives the same
// bits.  A tile is 128 compressed rows x 4 tokens:
//
//   D = Kh Qh^T    M = 128 rows, N = 256 (4 tokens x 64 heads), K = 128
//
// With rows as the lanes of D, the thread that owns row s holds all 64 head
// dots of a token, so the ordered head chain runs inside one thread.
//
// Persistent CTAs walk groups of 4 tokens (later groups, which see more rows,
// first); per group the row tiles run over the rows its last token can see.
// Warp 0 issues the TMA copies (the group's 256 q rows and 4 x 64 weights,
// then the row tiles through two stages), warp 1 owns tensor memory and (one
// lane) issues the MMAs into two D buffers, warps 4..11 quantise each group's
// q in place and then run its head chains (warp 4 + 4p + q: lane quarter q,
// tokens 2p and 2p + 1).  Every wait is bounded; a timeout raises
// DS41_E_TIMEOUT and the roles exit.
#include "ds41_internal.cuh"
#include "ds41_tc.cuh"

namespace ds41 {
namespace tci {

using namespace tc;

constexpr int HI = 64;            // indexer heads
constexpr int DI = 128;           // indexer dim
constexpr int TT = 4;             // tokens per group
constexpr int ROWS = 128;         // compressed rows per tile
constexpr int THREADS = 384;

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t QBLK = TT * HI * 64 * 2;            // [256 q rows][64 dims]: 32 KiB
constexpr uint32_t Q_BYTES = 2 * QBLK;                 // one group's q (2 blocks of 64 dims)
constexpr uint32_t KBLK = ROWS * 64 * 2;               // [128 rows][64 dims]: 16 KiB
constexpr uint32_t K_BYTES = 2 * KBLK;                 // one row tile
constexpr int KST = 2;                                 // row-tile stages
constexpr uint32_t Q_OFF = 0;                          // 2 q stages
constexpr uint32_t K_OFF = 2 * Q_BYTES;                // KST row-tile stages
constexpr uint32_t W_OFF = K_OFF + KST * K_BYTES;      // 2 x [4][64] f32 weights
constexpr uint32_t W_BYTES = TT * HI * 4;
constexpr uint32_t BAR_OFF = W_OFF + 2 * W_BYTES;
constexpr uint32_t SMEM_BYTES = BAR_OFF + 256 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

enum {
    B_QFULL, B_QEMPTY = B_QFULL + 2, B_WFULL = B_QEMPTY + 2, B_WEMPTY = B_WFULL + 2,
    B_KFULL = B_WEMPTY + 2, B_KEMPTY = B_KFULL + KST, B_DFULL = B_KEMPTY + KST,
    B_DEMPTY = B_DFULL + 2, B_QREADY = B_DEMPTY + 2,  // 2: the group's q quantised in place
    B_EPI = B_QREADY + 2, B_FINAL, NBAR
};
static_assert(NBAR * 8 + 8 <= 256, "barrier area");

constexpr uint32_t TM_COLS = 512;  // two D buffers of 256 columns
constexpr int EPI_THREADS = 256;   // warps 4..11
constexpr uint32_t IDESC = idesc_bf16(128, TT * HI, 0, 0);

struct Params {
    const float* w;
    uint16_t* scores;
    int m;
    int64_t n_c, ratio, start_pos;
    int fill_hidden;
    unsigned int* status;
};

__device__ __forceinline__ int64_t visible(int64_t t, const Params& p) {
    const int64_t v = (p.start_pos + t + 1) / p.ratio;
    return v < p.n_c ? v : p.n_c;
}

// Group k of this CTA -> its first token and the number of row tiles its
// last token can see.
__device__ __forceinline__ void group_of(int j, const Params& p, int& t0, int& tcount, int& ntile) {
    const int G = (p.m + TT - 1) / TT;
    const int gi = G - 1 - (int)(blockIdx.x + (int64_t)j * gridDim.x);
    t0 = gi * TT;
    tcount = min(TT, p.m - t0);
    const int64_t vis = visible(t0 + tcount - 1, p);
    ntile = (int)((vis + ROWS - 1) / ROWS);
}

// A group's q in place: the q stage holds 256 bf16 rows of 128 as two
// 64-column blocks with the 128-byte swizzle (as the tiled copy lands them);
// every block of 32 values becomes bf16(e2m1(v / s) * s) with
// s = 2^ceil(log2(max(amax, 6 * 2^-126) / 6)), exactly as fp4_quant_e8m0.
// Thread `tid` of `nthr` takes blocks tid, tid + nthr, ... of the first `rows`
// rows (rows past the group's tokens are zero-filled and stay zero), two at a
// time so that their dependent steps interleave; the maximum is a tree (the
// maximum of a set does not depend on the order).
__device__ __forceinline__ void quant_q_inplace(uint8_t* qst, int rows, int tid, int nthr) {
    const int nb = rows * 4;
#pragma unroll 1
    for (int id0 = tid; id0 < nb; id0 += 2 * nthr) {
        float v[2][32];
        uint8_t* rowp[2];
        int nn[2], cb[2];
        bool live[2];
#pragma unroll
        for (int b = 0; b < 2; b++) {
            const int id = id0 + b * nthr;
            live[b] = id < nb;
            // a second block past the end reads this thread's first block
            // again (before this thread stores it) and is never stored
            const int idc = live[b] ? id : id0;
            const int n = idc >> 2, j = idc & 3;
            nn[b] = n;
            cb[b] = (j & 1) * 4;
            rowp[b] = qst + (j >> 1) * QBLK + n * 128;
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++) {
                const uint4 u = *reinterpret_cast<const uint4*>(rowp[b] + (((cb[b] + c4) ^ (n & 7)) << 4));
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    v[b][c4 * 8 + 2 * e] = __uint_as_float(w4[e] << 16);
                    v[b][c4 * 8 + 2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < 2; b++) {
            float mx[16];
#pragma unroll
            for (int e = 0; e < 16; e++) mx[e] = fmaxf(fabsf(v[b][2 * e]), fabsf(v[b][2 * e + 1]));
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                for (int e = 0; e < w; e++) mx[e] = fmaxf(mx[e], mx[e + w]);
            const float amax = fmaxf(mx[0], __uint_as_float(0x01c00000u));  // 6 * 2^-126
            float rs;
            const float sc = e8m0_scale_bf16(amax, &rs);
#pragma unroll
            for (int c4 = 0; c4 < 4; c4++) {
                float t[8];
#pragma unroll
                for (int e = 0; e < 8; e++) t[e] = __fmul_rn(v[b][c4 * 8 + e], rs);
                uint32_t codes;
                const uint4 o = e2m1_round8(t, sc, &codes);
                if (live[b])
                    *reinterpret_cast<uint4*>(rowp[b] + (((cb[b] + c4) ^ (nn[b] & 7)) << 4)) = o;
            }
        }
    }
}

__global__ void __launch_bounds__(THREADS, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_k, const Params p) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BAR_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + BAR_OFF + NBAR * 8);
    volatile int* abort_f = reinterpret_cast<volatile int*>(sm + BAR_OFF + NBAR * 8 + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = (p.m + TT - 1) / TT;
    const int ngroups = (int)((G - (int64_t)blockIdx.x + gridDim.x - 1) / gridDim.x);

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; b++) {
            mbar_init(&bars[B_QFULL + b], 1);
            mbar_init(&bars[B_QEMPTY + b], 1);
            mbar_init(&bars[B_WFULL + b], 1);
            mbar_init(&bars[B_WEMPTY + b], EPI_THREADS / 32);
            mbar_init(&bars[B_DFULL + b], 1);
            mbar_init(&bars[B_DEMPTY + b], EPI_THREADS / 32);
            mbar_init(&bars[B_QREADY + b], 1);
        }
        for (int b = 0; b < KST; b++) {
            mbar_init(&bars[B_KFULL + b], 1);
            mbar_init(&bars[B_KEMPTY + b], 1);
        }
        mbar_init(&bars[B_EPI], EPI_THREADS / 32);
        mbar_init(&bars[B_FINAL], 1);
        *abort_f = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                smem_u32(tmem_slot)),
            "r"(TM_COLS)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer (one lane)
        // ------------------------------------------------------------------
        if (lane == 0) {
            uint32_t kt = 0, q_armed[2] = {0, 0}, w_armed[2] = {0, 0}, k_armed[KST] = {};
            bool ok = true;
            int jq = 0;  // groups with tiles so far
            for (int j = 0; j < ngroups && ok; j++) {
                int t0, tcount, ntile;
                group_of(j, p, t0, tcount, ntile);
                if (ntile == 0) continue;
                const int qs = jq & 1;
                if (jq >= 2 &&
                    !(wait_bar(&bars[B_QEMPTY + qs], ((jq - 2) >> 1) & 1, abort_f, p.status) &&
                      wait_bar(&bars[B_WEMPTY + qs], ((jq - 2) >> 1) & 1, abort_f, p.status)))
                    break;
                mbar_arrive_expect_tx(&bars[B_QFULL + qs], Q_BYTES);
                q_armed[qs]++;
                for (int kb = 0; kb < 2; kb++)
                    tma_load_2d(sbase + Q_OFF + qs * Q_BYTES + kb * QBLK, &map_q, kb * 64, t0 * HI,
                                &bars[B_QFULL + qs]);
                const uint32_t wbytes = (uint32_t)tcount * HI * 4;
                mbar_arrive_expect_tx(&bars[B_WFULL + qs], wbytes);
                w_armed[qs]++;
                bulk_g2s(sm + W_OFF + qs * W_BYTES, p.w + (int64_t)t0 * HI, wbytes,
                         &bars[B_WFULL + qs]);
                for (int i = 0; i < ntile; i++, kt++) {
                    const int ks = kt % KST;
                    if (kt >= KST && !wait_bar(&bars[B_KEMPTY + ks], ((kt - KST) / KST) & 1, abort_f,
                                               p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[B_KFULL + ks], K_BYTES);
                    k_armed[ks]++;
                    for (int kb = 0; kb < 2; kb++)
                        tma_load_2d(sbase + K_OFF + ks * K_BYTES + kb * KBLK, &map_k, kb * 64,
                                    i * ROWS, &bars[B_KFULL + ks]);
                }
                jq++;
            }
            // let every copy this CTA started land before the CTA exits
            for (int b = 0; b < 2; b++) {
                if (q_armed[b]) drain_bar(&bars[B_QFULL + b], (q_armed[b] - 1) & 1, p.status);
                if (w_armed[b]) drain_bar(&bars[B_WFULL + b], (w_armed[b] - 1) & 1, p.status);
            }
            for (int b = 0; b < KST; b++)
                if (k_armed[b]) drain_bar(&bars[B_KFULL + b], (k_armed[b] - 1) & 1, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer (one lane): D[kt % 2] = Kh(tile) Qh(group)^T
        // ------------------------------------------------------------------
        if (lane == 0) {
            uint32_t jq = 0, kt = 0;
            bool ok = true;
            for (int j = 0; j < ngroups && ok; j++) {
                int t0, tcount, ntile;
                group_of(j, p, t0, tcount, ntile);
                if (ntile == 0) continue;
                const int qs = jq & 1;
                if (!wait_bar(&bars[B_QREADY + qs], (jq >> 1) & 1, abort_f, p.status)) break;
                const uint64_t qd = sdesc(sbase + Q_OFF + qs * Q_BYTES, 16, 1024);
                for (int i = 0; i < ntile; i++, kt++) {
                    const int ks = kt % KST, db = kt & 1;
                    if (!wait_bar(&bars[B_KFULL + ks], (kt / KST) & 1, abort_f, p.status) ||
                        (kt >= 2 &&
                         !wait_bar(&bars[B_DEMPTY + db], ((kt - 2) >> 1) & 1, abort_f, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t kd = sdesc(sbase + K_OFF + ks * K_BYTES, 16, 1024);
                    const uint32_t d = tmem + 256 * db;
#pragma unroll
                    for (int kk = 0; kk < DI / 16; kk++)
                        tc_mma(d, kd + (((kk >> 2) * KBLK + (kk & 3) * 32) >> 4),
                               qd + (((kk >> 2) * QBLK + (kk & 3) * 32) >> 4), IDESC,
                               kk > 0 ? 1u : 0u);
                    tc_commit(&bars[B_KEMPTY + ks]);
                    tc_commit(&bars[B_DFULL + db]);
                    if (i == ntile - 1) tc_commit(&bars[B_QEMPTY + qs]);
                }
                jq++;
            }
            tc_commit(&bars[B_FINAL]);
            drain_bar(&bars[B_FINAL], 0, p.status);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------------
        // Head chains: thread = compressed row 32 q + lane of the tile,
        // tokens 2 pr and 2 pr + 1 of the group.  The same warps quantise
        // each group's q first.  (Quantising the next group's q while a
        // group's tiles run measured slower: the quantisation then took about
        // twice as long, beside the MMAs reading their operands from shared
        // memory.)
        // ------------------------------------------------------------------
        const int q = warp & 3, pr = (warp - 4) >> 2;
        const int etid = threadIdx.x - 128;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        uint32_t jq = 0, kt = 0, epi_ph = 0;
        for (int j = 0; j < ngroups; j++) {
            int t0, tcount, ntile;
            group_of(j, p, t0, tcount, ntile);
            const int64_t all_tiles = (p.n_c + ROWS - 1) / ROWS;
            if (ntile > 0) {
                const int ws = jq & 1;
                {
                    // the group's q quantised in place, before its head chains
                    if (!wait_bar(&bars[B_QFULL + ws], (jq >> 1) & 1, abort_f, p.status)) break;
                    quant_q_inplace(sm + Q_OFF + ws * Q_BYTES, tcount * HI, etid, EPI_THREADS);
                    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                    if (!warps_sync(&bars[B_EPI], epi_ph, abort_f, p.status)) break;
                    if (etid == 0) mbar_arrive(&bars[B_QREADY + ws]);
                }
                if (!wait_bar(&bars[B_WFULL + ws], (jq >> 1) & 1, abort_f, p.status)) break;
                const float* wsm = reinterpret_cast<const float*>(sm + W_OFF + ws * W_BYTES);
                // rows each of this thread's two tokens can see (one 64-bit
                // division per token and group, not per score)
                int64_t vis_u[2];
#pragma unroll
                for (int u = 0; u < 2; u++)
                    vis_u[u] = 2 * pr + u < tcount ? visible(t0 + 2 * pr + u, p) : 0;
                bool ok = true;
                for (int i = 0; i < ntile; i++, kt++) {
                    const int db = kt & 1;
                    if (!wait_bar(&bars[B_DFULL + db], (kt >> 1) & 1, abort_f, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int64_t s = (int64_t)i * ROWS + 32 * q + lane;
                    // both tokens' 64 head dots, then the buffer goes back to
                    // the MMA issuer before the chains run
                    uint32_t dv[2][64];
#pragma unroll
                    for (int u = 0; u < 2; u++) {
                        const uint32_t col = tmem + lane_off + 256 * db + 64 * (2 * pr + u);
                        tc_ld32(col, *reinterpret_cast<uint32_t(*)[32]>(dv[u]));
                        tc_ld32(col + 32, *reinterpret_cast<uint32_t(*)[32]>(dv[u] + 32));
                    }
                    tc_wait_ld();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_DEMPTY + db]);
                    // the two tokens' chains side by side, each in head order;
                    // the weights come four heads per 16-byte load
                    const float4* w0 = reinterpret_cast<const float4*>(wsm + (2 * pr) * HI);
                    const float4* w1 = w0 + HI / 4;
                    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
                    for (int h4 = 0; h4 < HI / 4; h4++) {
                        const float4 x0 = w0[h4], x1 = w1[h4];
                        const float c0[4] = {x0.x, x0.y, x0.z, x0.w};
                        const float c1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int h = 4 * h4 + e;
                            a0 = __fmaf_rn(c0[e], fmaxf(__uint_as_float(dv[0][h]), 0.0f), a0);
                            a1 = __fmaf_rn(c1[e], fmaxf(__uint_as_float(dv[1][h]), 0.0f), a1);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; u++) {
                        const int tt = 2 * pr + u;
                        if (tt >= tcount || s >= p.n_c) continue;
                        uint16_t out = 0xff80u;  // -inf: not visible yet
                        if (s < vis_u[u]) {
                            out = f2bf(u == 0 ? a0 : a1);
                            if (out == 0x8000u) out = 0u;
                        }
                        p.scores[(int64_t)(t0 + tt) * p.n_c + s] = out;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_WEMPTY + ws]);
                jq++;
                if (!ok) break;
            }
            // rows no token of the group can see yet, when the scores are an output
            if (p.fill_hidden) {
                for (int64_t tile = ntile; tile < all_tiles; tile++) {
                    const int64_t s = tile * ROWS + 32 * q + lane;
                    if (s >= p.n_c) continue;
                    for (int u = 0; u < 2; u++) {
                        const int tt = 2 * pr + u;
                        if (tt < tcount) p.scores[(int64_t)(t0 + tt) * p.n_c + s] = 0xff80u;
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
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(TM_COLS)
                     : "memory");
}

}  // namespace tci

bool indexer_tc_supported(int64_t m, int64_t Hi, int64_t Di, int sms) {
    return Hi == tci::HI && Di == tci::DI && (m + tci::TT - 1) / tci::TT >= sms &&
           m * Hi < (int64_t(1) << 31);
}

int indexer_tc_launch(const uint16_t* q_idx, const uint16_t* kq, const float* w, uint16_t* scores,
                      int64_t m, int64_t n_c, int64_t ratio, int64_t start_pos, bool fill_hidden,
                      unsigned int* status, int sms, cudaStream_t st) {
    using namespace tci;
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int rc = get_encode(&enc);
    if (rc) return rc;
    CUtensorMap mq, mk;
    if ((rc = make_map_bf16(enc, &mq, q_idx, m * HI, DI, 64, TT * HI))) return rc;
    if ((rc = make_map_bf16(enc, &mk, kq, n_c, DI, 64, ROWS))) return rc;
    Params p;
    p.w = w;
    p.scores = scores;
    p.m = (int)m;
    p.n_c = n_c;
    p.ratio = ratio;
    p.start_pos = start_pos;
    p.fill_hidden = fill_hidden ? 1 : 0;
    p.status = status;
    const int64_t G = (m + TT - 1) / TT;
    const int grid = (int)(G < sms ? G : sms);
    rc = cuda_check(cudaFuncSetAttribute(indexer_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES),
                    "ds41_indexer_topk: tensor-core kernel attributes");
    if (rc) return rc;
    return launch_pdl(indexer_tc_kernel, dim3((unsigned)grid), dim3(THREADS), SMEM_BYTES, st,
                      "ds41_indexer_topk: tensor-core scores kernel", mq, mk, p);
}

}  // namespace ds41
