// ds41_indexer_mxf4.cu - the fp4 indexer scores on a packed mxf4 key cache,
// with block-scaled tcgen05 MMAs (kind::mxf4) on the e2m1 codes and their
// e8m0 block-32 scales.
//
// metrale_model_arch/attn_v41/forward.rs calls the indexer; the header of
// metrale_model_arch/deepseek_v41_ref/compress.rs fixes its precision: q and
// k take the e2m1 round trip with power-of-two scales per block of 32
// (fp4_quant_e8m0_inplace), the scores are bf16.  Those operands are exactly
// mxf4: an e2m1 code per element and an e8m0 scale per block of 32, so the
// key cache is kept in that form (64 bytes of codes + 4 scale bytes per row
// of 128, instead of 256 bytes of bf16) and the tensor core multiplies the
// codes with the scales applied in hardware.  Score of query t against
// compressed row s, for s < (start_pos + t + 1) / ratio:
//   acc = 0; for h in 0..63: acc = fma(w[t,h], max(<qh[t,h], kh[s]>, 0), acc)
//   score = bf16(acc)          (-0 -> +0; rows not visible yet score -inf)
// The dot products of these fp4 values are exact in f32, so the MMA's sum
// gives the same bits as the ordered one.
//
// A tile is 128 compressed rows x (up to 2 tokens x 64 heads):
//
//   D = Kh Qh^T    M = 128 rows, N = 64 per token, K = 128 (two MMAs of 64)
//
// with the A operand (key codes) and the B operand (query codes) K-major in
// shared memory with the 64-byte swizzle, and the scale factors in tensor
// memory: per 128 rows, 4 columns, lane r (of every lane quarter) holding in
// column j the 4 scale bytes of row r + 32 j; the MMA over dims 0..63 takes
// bytes 0-1 (scale-factor id 0), the one over 64..127 bytes 2-3 (id 2).
//
// Roles (384 threads): warp 0 issues the TMA copies (the group's q rows in
// bf16, the weights, the key-code tiles through 6 stages); warp 1 owns tensor
// memory and (one lane) issues the MMAs into two D buffers; warps 2..3
// quantise the q of the CTA's next group into codes + scale bytes in shared
// memory while warps 4..11 run the head chains of this one (the CTA's first
// group they quantise themselves); warps 4..7 write the scale factors into
// tensor memory, and warp 4 + 4 p + q holds lane quarter q of D and token p
// of the group for the head chains.
// Groups of 2 tokens go to persistent CTAs (heaviest first) when there are at
// least as many groups as SMs; otherwise the row tiles of each group are
// split over several CTAs.  Every wait is bounded; a timeout raises
// DS41_E_TIMEOUT and the roles exit.
#include "ds41_internal.cuh"
#include "ds41_step1.cuh"
#include "ds41_tc.cuh"

namespace ds41 {
namespace mx {

using namespace tc;

constexpr int HI = 64;             // indexer heads
constexpr int DI = 128;            // indexer dim
constexpr int TT = 2;              // tokens per group
constexpr int NMAX = TT * HI;      // 128 B-operand rows
constexpr int ROWS = 128;          // compressed rows per tile
constexpr int KST = 6;             // key-code tile stages
constexpr int THREADS = 384;
constexpr int EPI_THREADS = 256;   // warps 4..11

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t QBLK = NMAX * 64 * 2;               // [128 q rows][64 dims] bf16: 16 KiB
constexpr uint32_t Q_BYTES = 2 * QBLK;                 // one group's q
constexpr uint32_t QP_BYTES = NMAX * 64;               // packed q codes [128][64 B]: 8 KiB
constexpr uint32_t K_BYTES = ROWS * 64;                // packed key codes [128][64 B]: 8 KiB
constexpr uint32_t Q_OFF = 0;                          // 2 stages (1024-aligned)
constexpr uint32_t QP_OFF = Q_OFF + 2 * Q_BYTES;       // 2 buffers (512-aligned)
constexpr uint32_t K_OFF = QP_OFF + 2 * QP_BYTES;      // KST stages (512-aligned)
constexpr uint32_t W_OFF = K_OFF + KST * K_BYTES;      // 2 x [2][64] f32 weights
constexpr uint32_t W_BYTES = NMAX * 4;
constexpr uint32_t SFQ_OFF = W_OFF + 2 * W_BYTES;      // 2 x [128] scale words of q
constexpr uint32_t SFQ_BYTES = NMAX * 4;
constexpr uint32_t BAR_OFF = SFQ_OFF + 2 * SFQ_BYTES;
constexpr uint32_t SMEM_BYTES = BAR_OFF + 512 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(QP_OFF % 512 == 0 && K_OFF % 512 == 0, "64-byte swizzle atoms");

enum {
    B_QFULL, B_QEMPTY = B_QFULL + 2, B_QREADY = B_QEMPTY + 2, B_QPEMPTY = B_QREADY + 2,
    B_WFULL = B_QPEMPTY + 2, B_WEMPTY = B_WFULL + 2, B_KFULL = B_WEMPTY + 2,
    B_KEMPTY = B_KFULL + KST, B_SFFULL = B_KEMPTY + KST, B_SFEMPTY = B_SFFULL + 2,
    B_DFULL = B_SFEMPTY + 2, B_DEMPTY = B_DFULL + 2, B_QPFULL = B_DEMPTY + 2,
    B_EPI = B_QPFULL + 2, B_QW, B_FINAL, NBAR
};
static_assert(NBAR * 8 + 8 <= 512, "barrier area");

// tensor-memory columns
constexpr uint32_t TM_COLS = 512;
constexpr uint32_t D_COL = 0;      // two D buffers of 128 columns
constexpr uint32_t SFA_COL = 256;  // two key scale-factor buffers of 4 columns
constexpr uint32_t SFB_COL = 264;  // two query scale-factor buffers of 4 columns

// Instruction descriptor of kind::mxf4 with e8m0 scales: e2m1 A and B
// (format 1), K-major, f32 accumulator, M = 128, N, and the scale-factor ids.
__host__ __device__ constexpr uint32_t idesc_mxf4(int N, int sfa_id, int sfb_id) {
    return ((uint32_t)sfb_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           (1u << 23) | ((uint32_t)(ROWS >> 4) << 24) | ((uint32_t)sfa_id << 29);
}

// Shared-memory descriptor of a K-major operand with the 64-byte swizzle
// (rows of 64 bytes, 8-row groups 512 bytes apart).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(512 >> 4) << 32) |
           (1ull << 46) | (4ull << 61);
}

__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], "
        "[%5], p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc));
}

// 4 columns of this warp's 32 lanes (32x32b shape)
__device__ __forceinline__ void tc_st4(uint32_t taddr, const uint32_t (&r)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

constexpr int QW_THREADS = 64;     // warps 2..3: q of the next group


// A group's q, N bf16 rows of 128 (two 64-column blocks with the 128-byte
// swizzle, as the tiled copy lands them) -> e2m1 codes (rows of 64 bytes with
// the 64-byte swizzle) and one e8m0 scale byte per block of 32, exactly as
// fp4_quant_e8m0: s = 2^ceil(log2(max(amax, 6 * 2^-126) / 6)), codes =
// e2m1(x / s).  Thread `tid` of `nthr` takes blocks tid, tid + nthr, ...
__device__ __forceinline__ void quant_group(const uint8_t* qsrc, uint8_t* qdst, uint8_t* sfq, int N,
                                            int tid, int nthr) {
#pragma unroll 1
    for (int id = tid; id < N * 4; id += nthr) {
        const int n = id >> 2, kb = id & 3;
        const uint8_t* row = qsrc + (kb >> 1) * QBLK + n * 128;
        float v[32];
        float amax = 0.0f;
#pragma unroll
        for (int c4 = 0; c4 < 4; c4++) {
            const int c = (kb & 1) * 4 + c4;
            const uint4 u = *reinterpret_cast<const uint4*>(row + ((c ^ (n & 7)) << 4));
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                v[c4 * 8 + 2 * e] = __uint_as_float(w4[e] << 16);
                v[c4 * 8 + 2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
            }
        }
#pragma unroll
        for (int e = 0; e < 32; e++) amax = fmaxf(amax, fabsf(v[e]));
        amax = fmaxf(amax, __uint_as_float(0x01c00000u));  // 6 * 2^-126
        float rs;
        const float sc = e8m0_scale_bf16(amax, &rs);  // amax: a bf16 magnitude or the floor
        uint32_t cw[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            uint32_t c = 0;
#pragma unroll
            for (int k = 0; k < 8; k += 2)
                c |= cvt_e2m1x2(__fmul_rn(v[8 * e + k], rs), __fmul_rn(v[8 * e + k + 1], rs))
                     << (4 * k);
            cw[e] = c;
        }
        *reinterpret_cast<uint4*>(qdst + n * 64 + ((kb ^ ((n >> 1) & 3)) << 4)) =
            make_uint4(cw[0], cw[1], cw[2], cw[3]);
        sfq[n * 4 + kb] = (uint8_t)(__float_as_uint(sc) >> 23);
    }
}

struct Params {
    const float* w;
    const uint32_t* k_scales;  // [n_c] words: the 4 scale bytes of a key row
    uint16_t* scores;
    int m;
    int G;          // token groups
    int ys;         // CTAs per group (1: persistent over groups)
    int main_ctas;  // CTAs of the score grid; the ones past it do step 1
    int64_t n_c, ratio, start_pos;
    int fill_hidden;
    unsigned int* status;
    RingArgs ring;    // fused few-token step: ring write + window indices
    LatentArgs lat;   // ... and the latent groups (lat.G == 0: none)
};

__device__ __forceinline__ int64_t visible(int64_t t, const Params& p) {
    const int64_t v = (p.start_pos + t + 1) / p.ratio;
    return v < p.n_c ? v : p.n_c;
}

// The CTA's j-th work item: a group (first token, token count, row tiles its
// last token can see) and the tiles of it this CTA takes (first, stride).
struct Item {
    int t0, tcount, ntile, tile0, tstride;
};
__device__ __forceinline__ int n_items(const Params& p) {
    if (p.ys > 1) return 1;
    return (int)((p.G - (int64_t)blockIdx.x + p.main_ctas - 1) / p.main_ctas);
}
__device__ __forceinline__ Item item_of(int j, const Params& p) {
    Item it;
    int gi;
    if (p.ys > 1) {
        gi = (int)(blockIdx.x % p.G);
        it.tile0 = (int)(blockIdx.x / p.G);
        it.tstride = p.ys;
    } else {
        gi = p.G - 1 - (int)(blockIdx.x + (int64_t)j * p.main_ctas);  // later groups see more
        it.tile0 = 0;
        it.tstride = 1;
    }
    it.t0 = gi * TT;
    it.tcount = min(TT, p.m - it.t0);
    const int64_t vis = visible(it.t0 + it.tcount - 1, p);
    it.ntile = (int)((vis + ROWS - 1) / ROWS);
    return it;
}
// tiles of the item this CTA computes
__device__ __forceinline__ int item_tiles(const Item& it) {
    return it.tile0 < it.ntile ? (it.ntile - it.tile0 + it.tstride - 1) / it.tstride : 0;
}

// The 4 scale words of key rows r0 + lane + 32 j (rows past n_c: scale 1, their
// codes are zero-filled by the copy).
__device__ __forceinline__ void load_sfa(const Params& p, int64_t r0, int lane, uint32_t (&v)[4]) {
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int64_t r = r0 + lane + 32 * j;
        v[j] = r < p.n_c ? __ldg(p.k_scales + r) : 0x7f7f7f7fu;
    }
}

__global__ void __launch_bounds__(THREADS, 1)
    indexer_mxf4_kernel(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k, const Params p) {
    // launched with programmatic stream serialization: the kernel before (the
    // previous step's attention, which reads the ring this kernel writes) is
    // waited for here, before the first memory access; only then may a
    // dependent kernel start launching (the decode attention reads q before
    // its own wait, so everything before this kernel must be complete)
    pdl_wait();
    const bool front = p.ring.ring != nullptr;  // the fused few-token step: a short kernel
    if (front) pdl_trigger();
    if ((int)blockIdx.x >= p.main_ctas) {
        // Fused front of a few-token step: the CTAs past the score grid do
        // step 1 (ring write + window indices, then the latent groups).
        const int side = (int)blockIdx.x - p.main_ctas, nside = (int)gridDim.x - p.main_ctas;
        if (side == 0) ring_write_cta(p.ring);
        const int hd8 = p.lat.hd / 8;
        for (int g = side; g < p.lat.G; g += nside)
            for (int k0 = 0; k0 < hd8; k0 += THREADS) latent_write_item(p.lat, g, k0 + threadIdx.x);
        return;
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + BAR_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + BAR_OFF + NBAR * 8);
    volatile int* abort_f = reinterpret_cast<volatile int*>(sm + BAR_OFF + NBAR * 8 + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nit = n_items(p);

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; b++) {
            mbar_init(&bars[B_QFULL + b], 1);
            mbar_init(&bars[B_QEMPTY + b], 1);
            mbar_init(&bars[B_QREADY + b], 1);
            mbar_init(&bars[B_QPEMPTY + b], 1);
            mbar_init(&bars[B_WFULL + b], 1);
            mbar_init(&bars[B_WEMPTY + b], 8);
            mbar_init(&bars[B_SFFULL + b], 4);
            mbar_init(&bars[B_SFEMPTY + b], 1);
            mbar_init(&bars[B_DFULL + b], 1);
            mbar_init(&bars[B_DEMPTY + b], 8);
            mbar_init(&bars[B_QPFULL + b], 1);
        }
        for (int s = 0; s < KST; s++) {
            mbar_init(&bars[B_KFULL + s], 1);
            mbar_init(&bars[B_KEMPTY + s], 1);
        }
        mbar_init(&bars[B_EPI], EPI_THREADS / 32);
        mbar_init(&bars[B_QW], QW_THREADS / 32);
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
            uint32_t jq = 0, kt = 0, q_armed[2] = {0, 0}, w_armed[2] = {0, 0}, k_armed[KST] = {};
            bool ok = true;
            for (int j = 0; j < nit && ok; j++) {
                const Item it = item_of(j, p);
                const int nt = item_tiles(it);
                if (nt == 0) continue;
                const int qs = jq & 1;
                if (jq >= 2 && !(wait_bar(&bars[B_QEMPTY + qs], ((jq - 2) >> 1) & 1, abort_f, p.status) &&
                                 wait_bar(&bars[B_WEMPTY + qs], ((jq - 2) >> 1) & 1, abort_f, p.status)))
                    break;
                mbar_arrive_expect_tx(&bars[B_QFULL + qs], Q_BYTES);
                q_armed[qs]++;
                for (int kb = 0; kb < 2; kb++)
                    tma_load_2d(sbase + Q_OFF + qs * Q_BYTES + kb * QBLK, &map_q, kb * 64, it.t0 * HI,
                                &bars[B_QFULL + qs]);
                const uint32_t wbytes = (uint32_t)it.tcount * HI * 4;
                mbar_arrive_expect_tx(&bars[B_WFULL + qs], wbytes);
                w_armed[qs]++;
                bulk_g2s(sm + W_OFF + qs * W_BYTES, p.w + (int64_t)it.t0 * HI, wbytes,
                         &bars[B_WFULL + qs]);
                for (int i = 0; i < nt; i++, kt++) {
                    const int ks = kt % KST;
                    if (kt >= KST && !wait_bar(&bars[B_KEMPTY + ks], ((kt / KST) - 1) & 1, abort_f,
                                               p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[B_KFULL + ks], K_BYTES);
                    k_armed[ks]++;
                    tma_load_2d(sbase + K_OFF + ks * K_BYTES, &map_k, 0,
                                (it.tile0 + i * it.tstride) * ROWS, &bars[B_KFULL + ks]);
                }
                jq++;
            }
            // let every copy this CTA started land before the CTA exits
            for (int b = 0; b < 2; b++) {
                if (q_armed[b]) drain_bar(&bars[B_QFULL + b], (q_armed[b] - 1) & 1, p.status);
                if (w_armed[b]) drain_bar(&bars[B_WFULL + b], (w_armed[b] - 1) & 1, p.status);
            }
            for (int s = 0; s < KST; s++)
                if (k_armed[s]) drain_bar(&bars[B_KFULL + s], (k_armed[s] - 1) & 1, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer (one lane): D[kt % 2] = Kh(tile) Qh(group)^T, block-scaled
        // ------------------------------------------------------------------
        if (lane == 0) {
            uint32_t jq = 0, kt = 0;
            bool ok = true;
            for (int j = 0; j < nit && ok; j++) {
                const Item it = item_of(j, p);
                const int nt = item_tiles(it);
                if (nt == 0) continue;
                const int qs = jq & 1;
                if (!wait_bar(&bars[B_QREADY + qs], (jq >> 1) & 1, abort_f, p.status)) break;
                const uint32_t N = (uint32_t)it.tcount * HI;
                const uint64_t qd = sdesc_sw64(sbase + QP_OFF + qs * QP_BYTES);
                for (int i = 0; i < nt; i++, kt++) {
                    const int ks = kt % KST, db = kt & 1;
                    if (!wait_bar(&bars[B_KFULL + ks], (kt / KST) & 1, abort_f, p.status) ||
                        !wait_bar(&bars[B_SFFULL + db], (kt >> 1) & 1, abort_f, p.status) ||
                        (kt >= 2 &&
                         !wait_bar(&bars[B_DEMPTY + db], ((kt - 2) >> 1) & 1, abort_f, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t kd = sdesc_sw64(sbase + K_OFF + ks * K_BYTES);
#pragma unroll
                    for (int k = 0; k < 2; k++)
                        mma_mxf4(tmem + D_COL + 128 * db, kd + ((32 * k) >> 4), qd + ((32 * k) >> 4),
                                 idesc_mxf4((int)N, 2 * k, 2 * k), tmem + SFA_COL + 4 * db,
                                 tmem + SFB_COL + 4 * qs, k > 0 ? 1u : 0u);
                    tc_commit(&bars[B_KEMPTY + ks]);
                    tc_commit(&bars[B_SFEMPTY + db]);
                    tc_commit(&bars[B_DFULL + db]);
                    if (i == nt - 1) tc_commit(&bars[B_QPEMPTY + qs]);
                }
                jq++;
            }
            tc_commit(&bars[B_FINAL]);
            drain_bar(&bars[B_FINAL], 0, p.status);
        }
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------------------------
        // q of the CTA's second and later groups, one group ahead of the head
        // chains (the first group's q is quantised by the epilogue warps)
        // ------------------------------------------------------------------
        const int qt = threadIdx.x - 64;
        uint32_t jq = 0, qw_ph = 0;
        for (int j = 0; j < nit; j++) {
            const Item it = item_of(j, p);
            if (item_tiles(it) == 0) continue;
            const int qs = jq & 1;
            if (jq >= 1) {
                // the packed buffer is free once the MMAs of group jq - 2 are done
                if ((jq >= 2 && !wait_bar(&bars[B_QPEMPTY + qs], ((jq - 2) >> 1) & 1, abort_f,
                                          p.status)) ||
                    !wait_bar(&bars[B_QFULL + qs], (jq >> 1) & 1, abort_f, p.status))
                    break;
                quant_group(sm + Q_OFF + qs * Q_BYTES, sm + QP_OFF + qs * QP_BYTES,
                            sm + SFQ_OFF + qs * SFQ_BYTES, it.tcount * HI, qt, QW_THREADS);
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                if (!warps_sync(&bars[B_QW], qw_ph, abort_f, p.status)) break;
                if (qt == 0) {
                    mbar_arrive(&bars[B_QPFULL + ((jq - 1) & 1)]);
                    mbar_arrive(&bars[B_QEMPTY + qs]);
                }
            }
            jq++;
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------------
        // q quantisation, scale factors, head chains: thread = compressed
        // row 32 q + lane of the tile, token pr of the group
        // ------------------------------------------------------------------
        const int q = warp & 3, pr = (warp - 4) >> 2, etid = threadIdx.x - 128;
        const bool sfw = pr == 0;  // warps 4..7 write the scale factors
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const int64_t all_tiles = (p.n_c + ROWS - 1) / ROWS;
        uint32_t jq = 0, kt = 0, epi_ph = 0;
        bool ok = true;
        for (int j = 0; j < nit && ok; j++) {
            const Item it = item_of(j, p);
            const int nt = item_tiles(it);
            if (nt > 0) {
                const int qs = jq & 1;
                uint32_t sfa_next[4] = {0, 0, 0, 0}, sfa_after[4] = {0, 0, 0, 0};
                if (sfw) {
                    load_sfa(p, (int64_t)it.tile0 * ROWS, lane, sfa_next);
                    if (nt > 1) load_sfa(p, (int64_t)(it.tile0 + it.tstride) * ROWS, lane, sfa_after);
                }
                // (1) the group's q as e2m1 codes + e8m0 scale bytes: the first
                // group here, every later one by warps 2..3 while this group's
                // predecessor ran its head chains
                const int N = it.tcount * HI;
                uint8_t* sfq = sm + SFQ_OFF + qs * SFQ_BYTES;
                if (jq == 0) {
                    if (!wait_bar(&bars[B_QFULL + qs], 0, abort_f, p.status)) {
                        ok = false;
                        break;
                    }
                    quant_group(sm + Q_OFF + qs * Q_BYTES, sm + QP_OFF + qs * QP_BYTES, sfq, N, etid,
                                EPI_THREADS);
                    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                    if (!warps_sync(&bars[B_EPI], epi_ph, abort_f, p.status)) {
                        ok = false;
                        break;
                    }
                } else if (!wait_bar(&bars[B_QPFULL + ((jq - 1) & 1)], ((jq - 1) >> 1) & 1, abort_f,
                                     p.status)) {
                    ok = false;
                    break;
                }
                if (sfw) {
                    // query scale factors: lane r, column j = row r + 32 j
                    const uint32_t* sw = reinterpret_cast<const uint32_t*>(sfq);
                    uint32_t v4[4];
#pragma unroll
                    for (int jj = 0; jj < 4; jj++) {
                        const int n = lane + 32 * jj;
                        v4[jj] = n < N ? sw[n] : 0x7f7f7f7fu;
                    }
                    tc_st4(tmem + lane_off + SFB_COL + 4 * qs, v4);
                    tc_wait_st();
                }
                tc_fence_before();
                if (!warps_sync(&bars[B_EPI], epi_ph, abort_f, p.status)) {
                    ok = false;
                    break;
                }
                if (etid == 0) {
                    mbar_arrive(&bars[B_QREADY + qs]);
                    if (jq == 0) mbar_arrive(&bars[B_QEMPTY + qs]);
                }
                if (!wait_bar(&bars[B_WFULL + qs], (jq >> 1) & 1, abort_f, p.status)) {
                    ok = false;
                    break;
                }
                const float* wt = reinterpret_cast<const float*>(sm + W_OFF + qs * W_BYTES) + pr * HI;
                const bool live = pr < it.tcount;
                const int64_t t = it.t0 + pr;
                const int64_t vis_t = live ? visible(t, p) : 0;
                for (int i = 0; i < nt; i++, kt++) {
                    const int db = kt & 1;
                    if (sfw) {
                        // key scale factors of this tile, and the next one's ahead
                        const int first = i == 0 ? 0 : 1;
                        for (int a = first; a < 2 && i + a < nt; a++) {
                            const uint32_t kk = kt + a;
                            const int sb = kk & 1;
                            if (kk >= 2 && !wait_bar(&bars[B_SFEMPTY + sb], ((kk - 2) >> 1) & 1,
                                                     abort_f, p.status)) {
                                ok = false;
                                break;
                            }
                            tc_st4(tmem + lane_off + SFA_COL + 4 * sb, sfa_next);
                            tc_wait_st();
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bars[B_SFFULL + sb]);
#pragma unroll
                            for (int e = 0; e < 4; e++) sfa_next[e] = sfa_after[e];
                            if (i + a + 2 < nt)
                                load_sfa(p, (int64_t)(it.tile0 + (i + a + 2) * it.tstride) * ROWS,
                                         lane, sfa_after);
                        }
                        if (!ok) break;
                    }
                    if (!wait_bar(&bars[B_DFULL + db], (kt >> 1) & 1, abort_f, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t dv[64];
                    if (live) {
                        tc_ld32(tmem + lane_off + D_COL + 128 * db + 64 * pr,
                                *reinterpret_cast<uint32_t(*)[32]>(dv));
                        tc_ld32(tmem + lane_off + D_COL + 128 * db + 64 * pr + 32,
                                *reinterpret_cast<uint32_t(*)[32]>(dv + 32));
                        tc_wait_ld();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_DEMPTY + db]);
                    const int64_t s = (int64_t)(it.tile0 + i * it.tstride) * ROWS + 32 * q + lane;
                    if (live && s < p.n_c) {
                        uint16_t out = 0xff80u;  // -inf: not visible yet
                        if (s < vis_t) {
                            float a = 0.0f;
#pragma unroll
                            for (int h = 0; h < HI; h++)
                                a = __fmaf_rn(wt[h], fmaxf(__uint_as_float(dv[h]), 0.0f), a);
                            out = f2bf(a);
                            if (out == 0x8000u) out = 0u;
                        }
                        p.scores[t * p.n_c + s] = out;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_WEMPTY + qs]);
                jq++;
                if (!ok) break;
            }
            // rows no token of the group can see yet, when the scores are an output
            if (p.fill_hidden && pr < it.tcount) {
                const int first = it.ntile > it.tile0
                                      ? it.tile0 + ((it.ntile - it.tile0 + it.tstride - 1) / it.tstride) * it.tstride
                                      : it.tile0;
                for (int64_t tile = first; tile < all_tiles; tile += it.tstride) {
                    const int64_t s = tile * ROWS + 32 * q + lane;
                    if (s < p.n_c) p.scores[(int64_t)(it.t0 + pr) * p.n_c + s] = 0xff80u;
                }
            }
        }
    }

    // many tokens: a long persistent kernel, whose dependents may start
    // launching once this CTA's work is done
    if (!front) pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                     "r"(TM_COLS)
                     : "memory");
}

}  // namespace mx

bool indexer_mxf4_supported(int64_t Hi, int64_t Di) { return Hi == mx::HI && Di == mx::DI; }

int indexer_mxf4_launch(const uint16_t* q_idx, const uint8_t* k_codes, const uint8_t* k_scales,
                        const float* w, uint16_t* scores, int64_t m, int64_t n_c, int64_t ratio,
                        int64_t start_pos, bool fill_hidden, unsigned int* status, int sms,
                        cudaStream_t st, const RingArgs* ring, const LatentArgs* lat) {
    using namespace mx;
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int rc = get_encode(&enc);
    if (rc) return rc;
    CUtensorMap mq, mk;
    if ((rc = make_map_bf16(enc, &mq, q_idx, m * HI, DI, 64, NMAX))) return rc;
    if ((rc = make_map_u8_sw64(enc, &mk, k_codes, n_c, DI / 2, ROWS))) return rc;
    Params p;
    p.w = w;
    p.k_scales = reinterpret_cast<const uint32_t*>(k_scales);
    p.scores = scores;
    p.m = (int)m;
    p.G = (int)((m + TT - 1) / TT);
    p.n_c = n_c;
    p.ratio = ratio;
    p.start_pos = start_pos;
    p.fill_hidden = fill_hidden ? 1 : 0;
    p.status = status;
    int grid;
    if (p.G >= sms) {
        p.ys = 1;
        grid = sms;
    } else {
        // few groups: split each group's row tiles over ys CTAs
        const int64_t tiles = (n_c + ROWS - 1) / ROWS;
        int64_t ys = sms / p.G;
        if (ys > tiles) ys = tiles;
        if (ys < 1) ys = 1;
        p.ys = (int)ys;
        grid = p.G * p.ys;
        if (p.ys == 1) grid = p.G;
    }
    p.main_ctas = grid;
    p.ring = ring ? *ring : RingArgs{};
    p.lat = lat ? *lat : LatentArgs{};
    if (ring) grid += (lat && lat->G > 1) ? 2 : 1;  // step-1 CTAs of the fused step
    rc = cuda_check(cudaFuncSetAttribute(indexer_mxf4_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES),
                    "indexer mxf4 kernel attributes");
    if (rc) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    rc = cuda_check(cudaLaunchKernelEx(&cfg, indexer_mxf4_kernel, mq, mk, p),
                    "ds41_indexer_topk_mxf4: scores kernel");
    if (rc) return rc;
    return launch_check("ds41_indexer_topk_mxf4: scores kernel");
}

}  // namespace ds41
