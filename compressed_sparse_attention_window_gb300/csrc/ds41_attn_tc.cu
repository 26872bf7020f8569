// ds41_attn_tc.cu - sparse attention with a per-head sink on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory), for many query tokens
// with 64-head groups and head_dim 512.
//
// metrale_model_arch/deepseek_v41_ref/compress.rs, attention_any: sparse_attn
// over the merged index row (window rows of rows_a, then the top-k rows of the
// compressed cache), scale = head_dim^-0.5, one row per position serving as key
// and value, the sink an extra logit of the softmax denominator.
//
//   o[t,h] = sum_v e^{s_v} row_v / (e^{sink_h} + sum_v e^{s_v}),
//   s_v = scale * <q[t,h], row_v>
//
// Design.  A persistent CTA per SM walks its work items (token, 64 heads).
// Per item a plan warp turns the index row into chunks of 128 rows: for each
// source (rows_a, rows_b) whose selected rows lie in a compact range the
// chunks are consecutive rows of that range, loaded by tiled TMA copies, with
// a 128-bit mask of the selected rows; otherwise (or when the range would take
// more chunks than the rows themselves) the selected rows are listed and
// gathered by the softmax warps as 16-byte cp.async pieces, which they fetch
// while the tensor core works through PV of the chunk before.  Duplicate
// indices force the list form (each copy then counts once per occurrence, as
// the definition does).
//
//   S  = Q R^T       M = 64 heads, N = 128 rows, K = 512  (S in tensor memory)
//   O^T += R^T P^T   M = 128 of hd (4 tiles), N = 64 heads, K = 128 rows
//
// A tcgen05.mma instruction costs some 50-70 cycles of issue however small,
// so the chunk is as wide as the one row buffer shared memory holds next to Q
// (128 rows, 128 KiB) and the MMA sequences are fully unrolled on
// precomputed descriptors.  The row buffer is managed in four pairs of
// 64-column blocks with a barrier each: PV tile t reads pair t only and
// releases it when done, so the next chunk's loads and the parts of its S
// follow the PV tile by tile instead of waiting for the whole chunk.  With heads as
// the rows of S, the four threads of a quad own one head's scores, so the
// running max and the denominator need two shuffles.  The reference max of a
// head moves only when a chunk exceeds it by 2^4 (and on the first chunk), so
// O is rescaled in tensor memory only on those chunks; the bound trades
// accuracy for rescales (the largest weight of a head is then up to 2^4
// instead of exactly 1 and takes a bf16 rounding too: with 2^8 the worst error
// on peaked softmaxes doubled, with 2^4 it stays within 1.3x of an exact
// running maximum).
//
// Warp roles (384 threads): warp 0 issues the TMA copies (Q, consecutive-row
// chunks), warp 1 owns tensor memory and (one lane) issues the MMAs, warp 2
// builds the per-item plans one item ahead, warps 4..7 compute the
// probabilities and gather the listed chunks' rows (warp 4+q block pair q),
// warps 8..11 rescale the columns of O whose head's reference moved and write
// the normalised output of each item (warp 4+q and 8+q use lane quarter q of
// tensor memory).  The softmax warps never wait for the output stores.  Every hand-off is an mbarrier
// with a bounded wait; a timeout raises DS41_E_TIMEOUT, and each role then
// drains what it started and exits.
#include "ds41_internal.cuh"
#include "ds41_tc.cuh"

namespace ds41 {
namespace tc {

constexpr int HD = 512;
constexpr int NH = 64;            // heads per work item
constexpr int RC = 128;           // rows per chunk
constexpr int NKP = 4;            // pairs of 64-column blocks of the row buffer
constexpr int THREADS = 384;
constexpr int MAXK = 1024;        // longest index row this kernel takes
constexpr int DCAP = 2048;        // longest row range loaded as consecutive rows
constexpr int MAXCH = 2 * DCAP / RC;  // chunks per item: two consecutive-row sources at most
constexpr int OOB_ROW = 1 << 29;  // a row coordinate beyond every tensor (reads as zero)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 4.0f;
constexpr int CORR_FEW = 8;        // moved heads rescaled column by column

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t Q_KB = 64 * 64 * 2;                // Q block [64 heads][64 dims]: 8 KiB
constexpr uint32_t R_KB = RC * 64 * 2;                // row block [128 rows][64 dims]: 16 KiB
constexpr uint32_t Q_OFF = 0;                         // 8 Q blocks
constexpr uint32_t R_OFF = 8 * Q_KB;                  // 8 row blocks (4 pairs)
constexpr uint32_t R_BYTES = 8 * R_KB;
constexpr uint32_t P_OFF = R_OFF + R_BYTES;           // P: 2 blocks of [64 heads][64 rows] bf16
constexpr uint32_t P_BLK = 8192;
constexpr uint32_t PLAN_OFF = P_OFF + 2 * P_BLK;      // 2 plans
constexpr uint32_t PLAN_DESC = 0;                     // MAXCH x 2 uint4
constexpr uint32_t PLAN_LIST = MAXCH * 32;            // int32 row list
constexpr uint32_t PLAN_N = PLAN_LIST + (MAXK + RC + 4) * 4;  // chunk count (the list
                                                      // has room for a 4-aligned start and a
                                                      // full chunk read past its end)
constexpr uint32_t PLAN_BYTES = PLAN_N + 64;
constexpr uint32_t BM_OFF = PLAN_OFF + 2 * PLAN_BYTES;  // 2 sources x DCAP bits
constexpr uint32_t BM_WORDS = DCAP / 32;
constexpr uint32_t MISC_OFF = BM_OFF + 2 * BM_WORDS * 4;
constexpr uint32_t MISC_BYTES = 3072;
constexpr uint32_t SMEM_BYTES = MISC_OFF + MISC_BYTES + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(PLAN_OFF % 16 == 0 && PLAN_BYTES % 16 == 0, "plan alignment");

// barriers
enum {
    B_QFULL, B_QEMPTY,
    B_RFULL,                               // NKP: block pair of the chunk landed
    B_REMPTY = B_RFULL + NKP,              // NKP: PV tile done with the block pair
    B_DONE = B_REMPTY + NKP,               // PV of the chunk complete (P free, O up to date)
    B_SFULL, B_SEMPTY,                     // S of the chunk in tensor memory / read
    B_CORR,                                // rescale factors of the chunk written
    B_PFULL,                               // P written and O rescaled
    B_ODONE, B_OFREE,
    B_INVL, B_INVLFREE = B_INVL + 2,       // 2 each: per-item normalisers
    B_PLANFULL = B_INVLFREE + 2, B_PLANEMPTY = B_PLANFULL + 2,
    B_FINAL = B_PLANEMPTY + 2, NBAR
};
// misc area layout
constexpr uint32_t M_BAR = 0;                   // NBAR x 8
constexpr uint32_t M_TMEM = 512;                // tensor memory base address
constexpr uint32_t M_ABORT = 516;               // set when any wait gave up
constexpr uint32_t M_FLAG = 528;                // 4 ints: a warp's heads moved their reference
constexpr uint32_t M_CORR = 1024;               // 64 floats
constexpr uint32_t M_INVL = 2048;               // 2 x 64 floats
static_assert(NBAR * 8 <= 512 && M_INVL + 512 <= MISC_BYTES, "misc layout");

// tensor memory columns
constexpr uint32_t TM_S = 0;     // S at columns 0 .. 127
constexpr uint32_t TM_O = 128;   // O^T tile mt at column 128 + 64 mt
constexpr uint32_t TM_COLS = 512;

struct Params {
    const uint16_t* rows_a;  // [n_a][HD]
    const uint16_t* rows_b;  // [n_c][HD]
    int64_t n_a, n_c;
    const int32_t* idx;
    int K;
    int nh;
    int m;
    float scale_log2;
    const float* sink;
    uint16_t* o;
    float* lse;
    unsigned int* status;
};

constexpr uint32_t IDESC_S = idesc_bf16(64, RC, 0, 0);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 64, 1, 0);

// Work item k of this CTA -> (token, head group): items are taken from the
// end (longest index rows first when later tokens see more rows).
__device__ __forceinline__ void item_of(int j, int m, int hg, int& t, int& g) {
    const int64_t k = (int64_t)blockIdx.x + (int64_t)j * gridDim.x;
    const int64_t r = (int64_t)m * hg - 1 - k;
    t = (int)(r / hg);
    g = (int)(r % hg);
}

constexpr uint32_t NEG_INF_BITS = 0xff800000u;

// 2^x by the special function unit, denormal results flushed to zero: a
// head's denominator is at least 1 (its reference maximum is the maximum of
// some chunk, whose weight is 1), so a weight below 2^-126 changes nothing.
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// two floats to bf16 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// four 8x8 b16 fragments to shared memory, lane l giving the address of row
// l % 8 of fragment l / 8
__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                            uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};\n" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_max(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// Block pair kp of a listed chunk (descriptor d, d1 of the plan), fetched by
// one warp as 16-byte cp.async pieces into the row blocks' 128-byte swizzled
// layout (the layout the tiled copies produce); rows past the list are zero.
// Lane l copies piece l % 16 of rows 64 (l / 16) .. 64 (l / 16) + 63, so each
// instruction reads two 256-byte row segments.  Returns once the pieces have
// landed and a proxy fence has made them visible to the tensor core.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ void gather_pair(const Params& p, const uint8_t* plan, uint4 d, uint4 d1, int kp,
                            uint32_t sbase, int lane) {
    const int* list = reinterpret_cast<const int*>(plan + PLAN_LIST) + (d.x & 0x3FFFFFFFu);
    const int cnt = __popc(d.y) + __popc(d.z) + __popc(d.w) + __popc(d1.x);
    const uint16_t* src = ((d.x >> 30) & 1u) ? p.rows_b : p.rows_a;
    const int c = lane & 15;                  // 16-byte piece of the pair's 256 bytes
    const int blk = 2 * kp + (c >> 3);        // 64-column block
    const int cc = c & 7;                     // 16-byte column within the block
    const uint16_t* col = src + blk * 64 + cc * 8;
    const uint32_t dst0 = sbase + R_OFF + blk * R_KB;
    const int r0 = 64 * (lane >> 4);
#pragma unroll 4
    for (int m4 = 0; m4 < 64; m4 += 4) {
        const int r = r0 + m4;
        const int4 rows = *reinterpret_cast<const int4*>(list + r);  // list has RC slack entries
        const int rr[4] = {rows.x, rows.y, rows.z, rows.w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int rk = r + k;
            const uint32_t dst = dst0 + rk * 128 + ((cc ^ (rk & 7)) << 4);
            if (rk < cnt)
                cp_async16(dst, col + (int64_t)rr[k] * HD);
            else
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};\n" ::"r"(dst), "r"(0u)
                             : "memory");
        }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncwarp();
}

// ---------------------------------------------------------------------------
// Plan warp: index row of one item -> chunk descriptors
//   desc[2i].x: row (consecutive chunk) or list offset (listed chunk) in bits
//               0..29, source in bit 30 (0 rows_a, 1 rows_b), listed in bit 31
//   desc[2i].y/z/w, desc[2i+1].x: mask of the chunk's rows 0..31, 32..63,
//               64..95, 96..127 (row r selected iff its bit is set)
// ---------------------------------------------------------------------------
__device__ void plan_item(const Params& p, int t, uint8_t* plan, uint32_t* bm, int lane) {
    constexpr int KPL = MAXK / 32;  // index entries per lane
    uint4* desc = reinterpret_cast<uint4*>(plan + PLAN_DESC);
    int* list = reinterpret_cast<int*>(plan + PLAN_LIST);
    const int32_t* irow = p.idx + (int64_t)t * p.K;
    const int64_t n_rows = p.n_a + p.n_c;
    const int na = (int)p.n_a;

    // the whole index row in registers (entry 32 k + lane), all loads in flight
    // at once; invalid entries become -1
    int vals[KPL];
#pragma unroll
    for (int k = 0; k < KPL; k++) {
        const int j = 32 * k + lane;
        vals[k] = j < p.K ? __ldg(irow + j) : -1;
    }
    int cnt[2] = {0, 0}, mn[2] = {INT_MAX, INT_MAX}, mx[2] = {-1, -1};
#pragma unroll
    for (int k = 0; k < KPL; k++) {
        const int v = vals[k];
        if (v < -1 || (int64_t)v >= n_rows) {
            raise_status(p.status, DS41_E_INDEX);
            vals[k] = -1;
        } else if (v >= 0) {
            const int s = v >= na;
            const int y = s ? v - na : v;
            cnt[s]++;
            mn[s] = min(mn[s], y);
            mx[s] = max(mx[s], y);
        }
    }
    bool dense[2];
    int range[2];
#pragma unroll
    for (int s = 0; s < 2; s++) {
        cnt[s] = warp_sum(cnt[s]);
        mn[s] = warp_min(mn[s]);
        mx[s] = warp_max(mx[s]);
        range[s] = cnt[s] ? mx[s] - mn[s] + 1 : 0;
        // consecutive rows where they take no more chunks than the list
        dense[s] = cnt[s] > 0 && range[s] <= DCAP &&
                   (range[s] + RC - 1) / RC <= (cnt[s] + RC - 1) / RC;
        if (dense[s]) {
            const int nw = 4 * ((range[s] + RC - 1) / RC);
            for (int w = lane; w < nw; w += 32) bm[s * BM_WORDS + w] = 0u;
        }
    }
    __syncwarp();
    if (dense[0] || dense[1]) {
        bool dup[2] = {false, false};
#pragma unroll
        for (int k = 0; k < KPL; k++) {
            const int v = vals[k];
            if (v < 0) continue;
            const int s = v >= na;
            if (!dense[s]) continue;
            const int bit = (s ? v - na : v) - mn[s];
            const uint32_t b = 1u << (bit & 31);
            const uint32_t old = atomicOr(&bm[s * BM_WORDS + (bit >> 5)], b);
            if (old & b) dup[s] = true;
        }
        // a repeated row must count once per occurrence: list it instead
        if (__any_sync(0xffffffffu, dup[0])) dense[0] = false;
        if (__any_sync(0xffffffffu, dup[1])) dense[1] = false;
    }
    __syncwarp();
    const uint32_t lt = (1u << lane) - 1u;
    int pos = 0, off[2] = {0, 0};
#pragma unroll
    for (int s = 0; s < 2; s++) {
        if (dense[s] || cnt[s] == 0) continue;
        pos = (pos + 3) & ~3;  // a listed chunk's rows start 16-byte aligned
        off[s] = pos;
#pragma unroll
        for (int k = 0; k < KPL; k++) {
            const int v = vals[k];
            const bool take = v >= 0 && ((v >= na) == (s == 1));
            const uint32_t bal = __ballot_sync(0xffffffffu, take);
            if (take) list[pos + __popc(bal & lt)] = s ? v - na : v;
            pos += __popc(bal);
        }
    }
    // consecutive-row chunks first, then listed ones: the copy engine's loads
    // of an item then all precede its gathers, so the producer's wait for the
    // chunk before each of its loads never runs ahead of the barrier's phase
    int nch = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int s = k & 1;
        if (cnt[s] == 0 || dense[s] != (k < 2)) continue;
        const uint32_t sbit = (uint32_t)s << 30;
        if (dense[s]) {
            const int nck = (range[s] + RC - 1) / RC;
            for (int base = 0; base < nck; base += 32) {
                const int i = base + lane;
                uint4 mk = make_uint4(0u, 0u, 0u, 0u);
                if (i < nck) mk = *reinterpret_cast<const uint4*>(bm + s * BM_WORDS + 4 * i);
                const bool keep = (mk.x | mk.y | mk.z | mk.w) != 0u;
                const uint32_t bal = __ballot_sync(0xffffffffu, keep);
                if (keep) {
                    const int at = nch + __popc(bal & lt);
                    desc[2 * at] = make_uint4((uint32_t)(mn[s] + RC * i) | sbit, mk.x, mk.y, mk.z);
                    desc[2 * at + 1] = make_uint4(mk.w, 0u, 0u, 0u);
                }
                nch += __popc(bal);
            }
        } else {
            const int nck = (cnt[s] + RC - 1) / RC;
            for (int i = lane; i < nck; i += 32) {
                const int n = min(RC, cnt[s] - RC * i);
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int nb = n - 32 * k;
                    w[k] = nb >= 32 ? 0xffffffffu : (nb > 0 ? ((1u << nb) - 1u) : 0u);
                }
                desc[2 * (nch + i)] =
                    make_uint4((uint32_t)(off[s] + RC * i) | sbit | 0x80000000u, w[0], w[1], w[2]);
                desc[2 * (nch + i) + 1] = make_uint4(w[3], 0u, 0u, 0u);
            }
            nch += nck;
        }
    }
    if (nch == 0) {  // nothing valid: one fully masked chunk of out-of-range (zero) rows
        if (lane == 0) {
            desc[0] = make_uint4((uint32_t)OOB_ROW, 0u, 0u, 0u);
            desc[1] = make_uint4(0u, 0u, 0u, 0u);
        }
        nch = 1;
    }
    if (lane == 0) *reinterpret_cast<int*>(plan + PLAN_N) = nch;
    __syncwarp();
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_ad,
                   const __grid_constant__ CUtensorMap map_bd,
                   const Params p) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + MISC_OFF + M_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + MISC_OFF + M_TMEM);
    volatile int* abort_f = reinterpret_cast<volatile int*>(sm + MISC_OFF + M_ABORT);
    int* flags = reinterpret_cast<int*>(sm + MISC_OFF + M_FLAG);
    float* corr_s = reinterpret_cast<float*>(sm + MISC_OFF + M_CORR);
    float* invl_s = reinterpret_cast<float*>(sm + MISC_OFF + M_INVL);
    uint32_t* bm = reinterpret_cast<uint32_t*>(sm + BM_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hg = p.nh / NH;
    const int64_t items = (int64_t)p.m * hg;
    const int ntok =
        (int)((items - (int64_t)blockIdx.x + gridDim.x - 1) / (int64_t)gridDim.x);

    if (threadIdx.x == 0) {
        mbar_init(&bars[B_QFULL], 1);
        mbar_init(&bars[B_QEMPTY], 1);
        for (int k = 0; k < NKP; k++) {
            mbar_init(&bars[B_RFULL + k], 1);
            mbar_init(&bars[B_REMPTY + k], 1);
        }
        mbar_init(&bars[B_DONE], 1);
        mbar_init(&bars[B_SFULL], 1);
        mbar_init(&bars[B_SEMPTY], 4);
        mbar_init(&bars[B_CORR], 4);
        mbar_init(&bars[B_PFULL], 8);
        for (int b = 0; b < 2; b++) {
            mbar_init(&bars[B_INVL + b], 4);
            mbar_init(&bars[B_INVLFREE + b], 4);
            mbar_init(&bars[B_PLANFULL + b], 1);
            mbar_init(&bars[B_PLANEMPTY + b], 10);  // producer, MMA issuer, 4 softmax, 4 correction
        }
        mbar_init(&bars[B_ODONE], 1);
        mbar_init(&bars[B_OFREE], 4);
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
        // TMA producer (one lane): per chunk, block pair k is loaded as soon
        // as the previous chunk's PV tile k has released it
        // ------------------------------------------------------------------
        if (lane == 0) {
            uint32_t g = 0;
            uint32_t q_armed = 0;
            for (int j = 0; j < ntok; j++) {
                int t, hgi;
                item_of(j, p.m, hg, t, hgi);
                const int slot = j & 1;
                if (!wait_bar(&bars[B_PLANFULL + slot], (j >> 1) & 1, abort_f, p.status)) break;
                if (j >= 1 && !wait_bar(&bars[B_QEMPTY], (j - 1) & 1, abort_f, p.status)) break;
                mbar_arrive_expect_tx(&bars[B_QFULL], 8 * Q_KB);
                q_armed++;
                const int qrow = t * p.nh + hgi * NH;
                for (int kb = 0; kb < 8; kb++)
                    tma_load_2d(sbase + Q_OFF + kb * Q_KB, &map_q, kb * 64, qrow, &bars[B_QFULL]);
                const uint8_t* plan = sm + PLAN_OFF + slot * PLAN_BYTES;
                const uint4* desc = reinterpret_cast<const uint4*>(plan + PLAN_DESC);
                const int nch = *reinterpret_cast<const int*>(plan + PLAN_N);
                bool ok = true;
                for (int i = 0; i < nch && ok; i++, g++) {
                    const uint4 d = desc[2 * i];
                    // a listed chunk's rows are gathered by the softmax warps
                    if (d.x & 0x80000000u) continue;
                    const int pos = (int)(d.x & 0x3FFFFFFFu);
                    const bool src_b = (d.x >> 30) & 1u;
                    const CUtensorMap* mp = src_b ? &map_bd : &map_ad;
                    for (int kp = 0; kp < NKP; kp++) {
                        if (g >= 1 && !wait_bar(&bars[B_REMPTY + kp], (g - 1) & 1, abort_f, p.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&bars[B_RFULL + kp], 2 * R_KB);
                        const uint32_t rb = sbase + R_OFF + 2 * kp * R_KB;
                        for (int kb = 0; kb < 2; kb++)
                            tma_load_2d(rb + kb * R_KB, mp, (2 * kp + kb) * 64, pos,
                                        &bars[B_RFULL + kp]);
                    }
                }
                if (!ok) break;
                mbar_arrive(&bars[B_PLANEMPTY + slot]);
            }
            // let every copy this CTA started land before the CTA exits: the
            // last chunk's block pairs land after every earlier chunk's (a pair
            // is loaded only once the PV of the chunk before has read it)
            if (q_armed) drain_bar(&bars[B_QFULL], (q_armed - 1) & 1, p.status);
            if (g >= 1)
                for (int kp = 0; kp < NKP; kp++)
                    drain_bar(&bars[B_RFULL + kp], (g - 1) & 1, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer (one lane).  PV tiles first: tile k of PV(g) releases
        // block pair k, whose load for chunk g + 1 then feeds part k of
        // S(g + 1), so S of the next chunk follows the PV tile by tile.
        // ------------------------------------------------------------------
        if (lane == 0) {
            int s_tok = 0, s_i = 0, s_n = -1, s_kp = 0;
            int p_tok = 0, p_i = 0, p_mt = 0;
            uint32_t sg = 0, pg = 0;
            uint32_t nring = 0;  // chunk counts of the last four items, 8 bits each
            uint32_t idle = 0;
            const uint32_t q_s = sbase + Q_OFF;
            const uint32_t r_s = sbase + R_OFF;
            const uint32_t p_s = sbase + P_OFF;
            while (p_tok < ntok) {
                bool prog = false;
                if (pg < sg) {
                    const bool ok =
                        p_mt > 0 ||
                        (mbar_test(&bars[B_PFULL], pg & 1) &&
                         (p_i > 0 || p_tok == 0 || mbar_test(&bars[B_OFREE], (p_tok - 1) & 1)));
                    if (ok) {
                        if (p_mt == 0) tc_fence_after();
                        // O^T tile p_mt += R^T P^T over the 128 rows of the chunk
                        // (P in two K blocks of 64 rows)
                        const uint64_t vd = sdesc(r_s + 2 * p_mt * R_KB, R_KB, 1024);
                        const uint64_t pd = sdesc(p_s, 16, 1024);
                        const uint32_t acc0 = p_i > 0 ? 1u : 0u;
                        const uint32_t d = tmem + TM_O + 64 * p_mt;
#pragma unroll
                        for (int kk = 0; kk < RC / 16; kk++)
                            tc_mma(d, vd + ((kk * 2048) >> 4),
                                   pd + (((kk >> 2) * P_BLK + (kk & 3) * 32) >> 4), IDESC_PV,
                                   kk > 0 ? 1u : acc0);
                        tc_commit(&bars[B_REMPTY + p_mt]);
                        if (++p_mt == 4) {
                            p_mt = 0;
                            tc_commit(&bars[B_DONE]);
                            const int pn = (int)((nring >> (8 * (p_tok & 3))) & 0xffu);
                            if (p_i == pn - 1) tc_commit(&bars[B_ODONE]);
                            pg++;
                            if (++p_i == pn) {
                                p_tok++;
                                p_i = 0;
                            }
                        }
                        prog = true;
                    }
                }
                if (s_tok < ntok && s_tok < p_tok + 3 && sg <= pg + 1) {
                    if (s_n < 0 && mbar_test(&bars[B_PLANFULL + (s_tok & 1)], (s_tok >> 1) & 1)) {
                        s_n = *reinterpret_cast<const int*>(sm + PLAN_OFF +
                                                            (s_tok & 1) * PLAN_BYTES + PLAN_N);
                        nring = (nring & ~(0xffu << (8 * (s_tok & 3)))) | ((uint32_t)s_n << (8 * (s_tok & 3)));
                        mbar_arrive(&bars[B_PLANEMPTY + (s_tok & 1)]);  // done with the plan
                    }
                    if (s_n > 0) {
                        const bool ok =
                            mbar_test(&bars[B_RFULL + s_kp], sg & 1) &&
                            (s_kp > 0 ||
                             ((sg < 1 || mbar_test(&bars[B_SEMPTY], (sg - 1) & 1)) &&
                              (s_i > 0 || mbar_test(&bars[B_QFULL], s_tok & 1))));
                        if (ok) {
                            tc_fence_after();
                            // part s_kp of S = Q R^T: the 64-column blocks 2 s_kp and
                            // 2 s_kp + 1, 8 MMAs on descriptors stepped by offsets in
                            // 16-byte units
                            const uint32_t kb0 = 2 * s_kp;
                            const uint64_t qd = sdesc(q_s + kb0 * Q_KB, 16, 1024);
                            const uint64_t rd = sdesc(r_s + kb0 * R_KB, 16, 1024);
#pragma unroll
                            for (int kk = 0; kk < 8; kk++)
                                tc_mma(tmem + TM_S, qd + (((kk >> 2) * Q_KB + (kk & 3) * 32) >> 4),
                                       rd + (((kk >> 2) * R_KB + (kk & 3) * 32) >> 4), IDESC_S,
                                       (s_kp > 0 || kk > 0) ? 1u : 0u);
                            if (++s_kp == NKP) {
                                s_kp = 0;
                                tc_commit(&bars[B_SFULL]);
                                if (s_i == s_n - 1) tc_commit(&bars[B_QEMPTY]);
                                sg++;
                                if (++s_i == s_n) {
                                    s_tok++;
                                    s_i = 0;
                                    s_n = -1;
                                }
                            }
                            prog = true;
                        }
                    }
                }
                if (prog) {
                    idle = 0;
                } else {
                    if (*abort_f) break;
                    if (++idle > (1u << 25)) {
                        *abort_f = 1;
                        raise_status(p.status, DS41_E_TIMEOUT);
                        break;
                    }
                    __nanosleep(32);
                }
            }
            // every MMA issued so far completes before tensor memory is freed
            tc_commit(&bars[B_FINAL]);
            drain_bar(&bars[B_FINAL], 0, p.status);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------------
        // Plan warp, one item ahead of the consumers
        // ------------------------------------------------------------------
        for (int j = 0; j < ntok; j++) {
            int t, hgi;
            item_of(j, p.m, hg, t, hgi);
            const int slot = j & 1;
            if (j >= 2 && !wait_bar(&bars[B_PLANEMPTY + slot], ((j - 2) >> 1) & 1, abort_f,
                                    p.status))
                break;
            plan_item(p, t, sm + PLAN_OFF + slot * PLAN_BYTES, bm, lane);
            if (lane == 0) mbar_arrive(&bars[B_PLANFULL + slot]);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------------
        // Softmax: warp 4+q reads lane quarter q.  With M = 64 the scores of
        // head 16q + r sit in lane 32q + r (r < 16), one column per row of
        // the chunk; the 16x256b reads give thread l the heads hA = 16q + l/4
        // and hB = hA + 8, 32 columns each.
        // ------------------------------------------------------------------
        const int q = warp - 4;
        const int qi = lane & 3;
        const int hA = 16 * q + (lane >> 2), hB = hA + 8;
        // |scale| in log2 units, at least 1e-30 so that a zero scale keeps
        // -inf (an unselected row) at -inf: its logits become s * 1e-30,
        // which is 0 in float arithmetic for every finite bf16 score product
        const bool neg = p.scale_log2 < 0.0f;
        const float sc = fmaxf(fabsf(p.scale_log2), 1e-30f);
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        uint32_t g = 0;
        // Softmax warp q also gathers block pair q of every listed chunk (the
        // tensor-memory lane quarter and the pair share the index): the first
        // chunk here, every later one once PV of the chunk before it has
        // released the pair, which is when this warp has nothing else to do.
        bool start_ok = true;
        if (ntok > 0) {
            start_ok = wait_bar(&bars[B_PLANFULL], 0, abort_f, p.status);
            const uint4* d0s = reinterpret_cast<const uint4*>(sm + PLAN_OFF + PLAN_DESC);
            if (start_ok && (d0s[0].x & 0x80000000u)) {
                gather_pair(p, sm + PLAN_OFF, d0s[0], d0s[1], q, sbase, lane);
                if (lane == 0) mbar_arrive(&bars[B_RFULL + q]);
            }
        }
        for (int j = 0; j < ntok && start_ok; j++) {
            int t, hgi;
            item_of(j, p.m, hg, t, hgi);
            const int slot = j & 1;
            if (!wait_bar(&bars[B_PLANFULL + slot], (j >> 1) & 1, abort_f, p.status)) break;
            const uint8_t* plan = sm + PLAN_OFF + slot * PLAN_BYTES;
            const uint4* desc = reinterpret_cast<const uint4*>(plan + PLAN_DESC);
            const int nch = *reinterpret_cast<const int*>(plan + PLAN_N);
            // per head: reference max (log2 units) and this thread's part of the
            // denominator (the quad's four parts add up to it)
            float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;
            bool bad = false;
            for (int i = 0; i < nch; i++, g++) {
                const uint4 d0 = desc[2 * i];
                const uint32_t m3 = desc[2 * i + 1].x;
                __syncwarp();
                if (i == nch - 1 && lane == 0)
                    mbar_arrive(&bars[B_PLANEMPTY + slot]);  // this warp's last read of the plan
                if (!wait_bar(&bars[B_SFULL], g & 1, abort_f, p.status)) {
                    bad = true;
                    break;
                }
                tc_fence_after();
                uint32_t sr[64];
                tc_ld16x256(tmem + lane_off + TM_S, *reinterpret_cast<uint32_t(*)[32]>(sr));
                tc_ld16x256(tmem + lane_off + TM_S + 64, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
                tc_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_SEMPTY]);
                // raw scores, -inf where the row is not selected (a chunk with
                // every row selected skips the masking): register 4 jr + e (+2)
                // holds column 8 jr + 2 qi + e, jr = 0..15.  With a negative
                // scale the scores change sign so that sc = |scale log2 e|.
                if (neg) {
#pragma unroll
                    for (int k = 0; k < 64; k++) sr[k] ^= 0x80000000u;
                }
                if ((d0.y & d0.z & d0.w & m3) != 0xffffffffu) {
                    const uint32_t mw[4] = {d0.y >> (2 * qi), d0.z >> (2 * qi),
                                            d0.w >> (2 * qi), m3 >> (2 * qi)};
#pragma unroll
                    for (int jr = 0; jr < 16; jr++) {
#pragma unroll
                        for (int e = 0; e < 2; e++) {
                            const bool sel = (mw[jr >> 2] >> (8 * (jr & 3) + e)) & 1u;
                            if (!sel) {
                                sr[4 * jr + e] = NEG_INF_BITS;
                                sr[4 * jr + 2 + e] = NEG_INF_BITS;
                            }
                        }
                    }
                }
                float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
                for (int jr = 0; jr < 16; jr++) {
                    mxA = fmaxf(mxA, fmaxf(__uint_as_float(sr[4 * jr]), __uint_as_float(sr[4 * jr + 1])));
                    mxB = fmaxf(mxB, fmaxf(__uint_as_float(sr[4 * jr + 2]), __uint_as_float(sr[4 * jr + 3])));
                }
                mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
                mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
                mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
                mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
                // chunk maxima in log2 units (sc > 0, so -inf stays -inf)
                mxA *= sc;
                mxB *= sc;
                float cA = 1.0f, cB = 1.0f;
                if (i == 0) {
                    mA = mxA;
                    mB = mxB;
                } else {
                    if (mxA > mA + RESCALE_LOG2) {
                        cA = ex2_ftz(mA - mxA);
                        mA = mxA;
                        lA *= cA;
                    }
                    if (mxB > mB + RESCALE_LOG2) {
                        cB = ex2_ftz(mB - mxB);
                        mB = mxB;
                        lB *= cB;
                    }
                }
                // hand the rescale factors of this chunk to the correction warps,
                // with the mask of this warp's heads that moved (bit r: head
                // 16 q + r; the four lanes of a quad agree, so lane 4 r speaks
                // for heads hA and hB of quad r)
                const uint32_t mvA = __ballot_sync(0xffffffffu, cA != 1.0f);
                const uint32_t mvB = __ballot_sync(0xffffffffu, cB != 1.0f);
                if (qi == 0) {
                    corr_s[hA] = cA;
                    corr_s[hB] = cB;
                }
                if (lane == 0) {
                    uint32_t m16 = 0;
#pragma unroll
                    for (int r = 0; r < 8; r++)
                        m16 |= (((mvA >> (4 * r)) & 1u) << r) | (((mvB >> (4 * r)) & 1u) << (8 + r));
                    flags[q] = (int)m16;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_CORR]);
                // probabilities 2^(sc s - m), the denominator, P (bf16) for the
                // PV MMA; an unselected row (-inf) gives 0
                const float nmA = (mA == -INFINITY) ? 0.0f : -mA;
                const float nmB = (mB == -INFINITY) ? 0.0f : -mB;
                uint32_t pkA[16], pkB[16];
#pragma unroll
                for (int jr = 0; jr < 16; jr++) {
                    const float a0 = ex2_ftz(fmaf(__uint_as_float(sr[4 * jr]), sc, nmA));
                    const float a1 = ex2_ftz(fmaf(__uint_as_float(sr[4 * jr + 1]), sc, nmA));
                    const float b0 = ex2_ftz(fmaf(__uint_as_float(sr[4 * jr + 2]), sc, nmB));
                    const float b1 = ex2_ftz(fmaf(__uint_as_float(sr[4 * jr + 3]), sc, nmB));
                    lA += a0 + a1;
                    lB += b0 + b1;
                    pkA[jr] = pack_bf16x2_rn(a0, a1);
                    pkB[jr] = pack_bf16x2_rn(b0, b1);
                }
                // P is free once PV(g - 1) is done
                if (g >= 1 && !wait_bar(&bars[B_DONE], (g - 1) & 1, abort_f, p.status)) {
                    bad = true;
                    break;
                }
                {
                    // row h of P block k: 8 chunks of 16 bytes (8 rows each),
                    // swizzled by h % 8.  The registers of column block jr are
                    // the 8x8 fragments (heads 16 q .. 16 q + 7 | + 8 .. + 15,
                    // columns 8 jr ..): four fragments per stmatrix, lane l
                    // giving the address of row l % 8 of fragment l / 8.
                    const int fr = lane >> 3;                 // fragment of this lane's address
                    const int h = 16 * q + 8 * (fr & 1) + (lane & 7);
                    const uint32_t rowa = sbase + P_OFF + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll
                    for (int jp = 0; jp < 8; jp++) {
                        const int jr = 2 * jp + (fr >> 1);
                        const uint32_t addr = rowa + (jr >> 3) * P_BLK + (((jr & 7) ^ (h & 7)) << 4);
                        stmatrix_x4(addr, pkA[2 * jp], pkB[2 * jp], pkA[2 * jp + 1], pkB[2 * jp + 1]);
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_PFULL]);
                // the next chunk (of this item or the next), if its rows are listed
                const uint8_t* nplan = plan;
                int ni = i + 1;
                if (ni == nch) {
                    ni = -1;
                    if (j + 1 < ntok) {
                        const int ns = (j + 1) & 1;
                        if (!wait_bar(&bars[B_PLANFULL + ns], ((j + 1) >> 1) & 1, abort_f, p.status)) {
                            bad = true;
                            break;
                        }
                        nplan = sm + PLAN_OFF + ns * PLAN_BYTES;
                        ni = 0;
                    }
                }
                if (ni >= 0) {
                    const uint4* nd = reinterpret_cast<const uint4*>(nplan + PLAN_DESC);
                    const uint4 dn = nd[2 * ni];
                    if (dn.x & 0x80000000u) {
                        if (!wait_bar(&bars[B_REMPTY + q], g & 1, abort_f, p.status)) {
                            bad = true;
                            break;
                        }
                        gather_pair(p, nplan, dn, nd[2 * ni + 1], q, sbase, lane);
                        if (lane == 0) mbar_arrive(&bars[B_RFULL + q]);
                    }
                }
            }
            if (bad) break;
            // ---- normalisers of this item for the correction warps ----
            lA += __shfl_xor_sync(0xffffffffu, lA, 1);
            lB += __shfl_xor_sync(0xffffffffu, lB, 1);
            lA += __shfl_xor_sync(0xffffffffu, lA, 2);
            lB += __shfl_xor_sync(0xffffffffu, lB, 2);
            if (j >= 2 && !wait_bar(&bars[B_INVLFREE + slot], ((j - 2) >> 1) & 1, abort_f, p.status))
                break;
            if (qi < 2) {
                const int hl = qi == 0 ? hA : hB;
                const float mr = qi == 0 ? mA : mB;
                const float l = qi == 0 ? lA : lB;
                const int h = hgi * NH + hl;
                const float sk = p.sink[h] * LOG2E;
                const float M = fmaxf(mr, sk);
                const float Mr = (M == -INFINITY) ? 0.0f : M;
                const float a = exp2f(mr - Mr);
                const float L = l * a + exp2f(sk - Mr);
                invl_s[slot * 64 + hl] = (L > 0.0f) ? a / L : 0.0f;
                if (p.lse) p.lse[(int64_t)t * p.nh + h] = (Mr + log2f(L)) / LOG2E;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_INVL + slot]);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------------------------
        // Correction + epilogue: warp 8+q owns lanes 32q.. of O^T (head dims
        // 128 mt + 32 q + lane of tile mt, one column per head).
        // ------------------------------------------------------------------
        const int q = warp - 8;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        uint32_t g = 0;
        for (int j = 0; j < ntok; j++) {
            int t, hgi;
            item_of(j, p.m, hg, t, hgi);
            const int slot = j & 1;
            if (!wait_bar(&bars[B_PLANFULL + slot], (j >> 1) & 1, abort_f, p.status)) break;
            const int nch =
                *reinterpret_cast<const int*>(sm + PLAN_OFF + slot * PLAN_BYTES + PLAN_N);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_PLANEMPTY + slot]);  // each warp read nch
            bool bad = false;
            for (int i = 0; i < nch; i++, g++) {
                if (!wait_bar(&bars[B_CORR], g & 1, abort_f, p.status)) {
                    bad = true;
                    break;
                }
                // heads whose reference moved (head h is column h of every O^T
                // tile): a few are rescaled column by column, more in groups of
                // 16 columns (the heads of one softmax warp)
                const uint32_t f0 = (uint32_t)flags[0], f1 = (uint32_t)flags[1];
                const uint32_t f2 = (uint32_t)flags[2], f3 = (uint32_t)flags[3];
                const uint64_t mv = (uint64_t)(f0 | (f1 << 16)) | ((uint64_t)(f2 | (f3 << 16)) << 32);
                const int nmv = __popcll(mv);
                if (nmv) {
                    // O^T holds the chunks before this one once PV(g-1) is done
                    if (!wait_bar(&bars[B_DONE], (g - 1) & 1, abort_f, p.status)) {
                        bad = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ta = tmem + lane_off + TM_O;
                    if (nmv <= CORR_FEW) {
                        uint32_t hv[CORR_FEW][4];
                        int hs[CORR_FEW];
                        uint64_t rest = mv;
#pragma unroll
                        for (int k = 0; k < CORR_FEW; k++) {
                            hs[k] = __ffsll((long long)rest) - 1;  // -1 once none are left
                            rest &= rest - 1;
                            if (k < nmv) {
#pragma unroll
                                for (int mt = 0; mt < 4; mt++) tc_ld1(ta + 64 * mt + hs[k], hv[k][mt]);
                            }
                        }
                        tc_wait_ld();
#pragma unroll
                        for (int k = 0; k < CORR_FEW; k++) {
                            if (k < nmv) {
                                const float c = corr_s[hs[k]];
#pragma unroll
                                for (int mt = 0; mt < 4; mt++) {
                                    hv[k][mt] = __float_as_uint(__uint_as_float(hv[k][mt]) * c);
                                    tc_st1(ta + 64 * mt + hs[k], hv[k][mt]);
                                }
                            }
                        }
                    } else {
#pragma unroll 1
                        for (int w = 0; w < 4; w++) {
                            if (!((mv >> (16 * w)) & 0xffffu)) continue;
                            float c[16];
#pragma unroll
                            for (int k = 0; k < 16; k += 4) {
                                const float4 v = *reinterpret_cast<const float4*>(corr_s + 16 * w + k);
                                c[k] = v.x;
                                c[k + 1] = v.y;
                                c[k + 2] = v.z;
                                c[k + 3] = v.w;
                            }
                            uint32_t ov[4][16];
#pragma unroll
                            for (int mt = 0; mt < 4; mt++) tc_ld16(ta + 64 * mt + 16 * w, ov[mt]);
                            tc_wait_ld();
#pragma unroll
                            for (int mt = 0; mt < 4; mt++) {
#pragma unroll
                                for (int k = 0; k < 16; k++)
                                    ov[mt][k] = __float_as_uint(__uint_as_float(ov[mt][k]) * c[k]);
                                tc_st16(ta + 64 * mt + 16 * w, ov[mt]);
                            }
                        }
                    }
                    tc_wait_st();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_PFULL]);
            }
            if (bad) break;
            // ---- epilogue of this item ----
            if (!wait_bar(&bars[B_INVL + slot], (j >> 1) & 1, abort_f, p.status)) break;
            if (!wait_bar(&bars[B_ODONE], j & 1, abort_f, p.status)) break;
            tc_fence_after();
            const float* inv = invl_s + slot * 64;
            uint16_t* obase = p.o + ((int64_t)t * p.nh + hgi * NH) * HD;
#pragma unroll 1
            for (int mt = 0; mt < 4; mt++) {
                const int dd = 128 * mt + 32 * q + lane;
#pragma unroll 1
                for (int hh = 0; hh < 2; hh++) {
                    uint32_t ov[32];
                    tc_ld32(tmem + lane_off + TM_O + 64 * mt + 32 * hh, ov);
                    tc_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; k++) {
                        const int c = 32 * hh + k;
                        obase[(int64_t)c * HD + dd] = f2bf(__uint_as_float(ov[k]) * inv[c]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_INVLFREE + slot]);
                mbar_arrive(&bars[B_OFREE]);
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

// ---------------------------------------------------------------------------
// Host side: tensor maps and the launch
// ---------------------------------------------------------------------------
}  // namespace tc

bool attn_tc_supported(int64_t m, int64_t nh, int64_t hd, int64_t K, int sms) {
    return hd == tc::HD && nh % tc::NH == 0 && K >= 1 && K <= tc::MAXK &&
           m * (nh / tc::NH) >= sms && m * nh < (int64_t(1) << 31);
}

int attn_tc_launch(const uint16_t* q, const uint16_t* rows_a, int64_t n_a, const uint16_t* rows_b,
                   int64_t n_c, const int32_t* idx, int64_t K, const float* sink, float scale,
                   uint16_t* o, float* lse, int64_t m, int64_t nh, unsigned int* status,
                   int sms, cudaStream_t st) {
    using namespace tc;
    if (n_a >= OOB_ROW || n_c >= OOB_ROW)
        return fail(DS41_E_RANGE, "ds41_sparse_attn_sink_fwd: %lld + %lld rows exceed the row range",
                    (long long)n_a, (long long)n_c);
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int rc = get_encode(&enc);
    if (rc) return rc;
    CUtensorMap mq, mad, mbd;
    if ((rc = make_map_bf16(enc, &mq, q, m * nh, HD, 64, 64))) return rc;
    if ((rc = make_map_bf16(enc, &mad, rows_a, n_a, HD, 64, RC))) return rc;
    if ((rc = make_map_bf16(enc, &mbd, rows_b, n_c, HD, 64, RC))) return rc;
    Params p;
    p.n_a = n_a;
    p.n_c = n_c;
    p.idx = idx;
    p.K = (int)K;
    p.nh = (int)nh;
    p.m = (int)m;
    p.scale_log2 = scale * LOG2E;
    p.rows_a = rows_a;
    p.rows_b = rows_b;
    p.sink = sink;
    p.o = o;
    p.lse = lse;
    p.status = status;
    const int64_t items = m * (nh / NH);
    const int grid = (int)(items < sms ? items : sms);
    auto kern = attn_tc_kernel;
    rc = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES),
                    "ds41_sparse_attn_sink_fwd: tensor-core kernel attributes");
    if (rc) return rc;
    // A plain launch: launched programmatically behind the top-k kernel, its
    // CTAs (a whole SM's shared memory each) wait resident beside that kernel,
    // and the step measured slower (prefill 704 -> 724 us, chunked prefill
    // 234 -> 255 us).  Its own trigger still lets the next kernel launch early.
    kern<<<grid, THREADS, SMEM_BYTES, st>>>(mq, mad, mbd, p);
    return launch_check("ds41_sparse_attn_sink_fwd: tensor-core kernel");
}

}  // namespace ds41
