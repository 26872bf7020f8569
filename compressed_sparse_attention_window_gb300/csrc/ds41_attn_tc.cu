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
// Per item a plan warp turns the index row into chunks of 64 rows: for each
// source (rows_a, rows_b) whose selected rows lie in a compact range the
// chunks are consecutive rows of that range, loaded by tiled TMA copies, with
// a 64-bit mask of the selected rows; otherwise the selected rows are listed
// and fetched by TMA gather4 copies.  Duplicate indices force the list form
// (each copy then counts once per occurrence, as the definition does).
//
//   S  = Q R^T       M = 64 heads, N = 64 rows, K = 512   (S in tensor memory)
//   O^T += R^T P^T   M = 128 of hd (4 tiles), N = 64 heads, K = 64 rows
//
// With heads as the rows of S, one thread owns one head's scores, so the
// running max and the denominator need no reductions across threads.  The
// reference max of a head moves only when a chunk exceeds it by 2^4 (and on the
// first chunk), so O is rescaled in tensor memory only on those rare chunks.
// The bound trades accuracy for rescales: the largest weight of a head is then
// up to 2^4 instead of exactly 1 and takes a bf16 rounding too; with 2^8 the
// worst error on peaked softmaxes doubled, with 2^4 it stays within 1.3x of an
// exact running maximum while N(0,1) scores almost never move the reference.
//
// Warp roles (256 threads): warp 0 issues TMA copies, warp 1 owns tensor
// memory and (one lane) issues the MMAs, warp 2 builds the per-item plans one
// item ahead, warps 4..7 run the softmax and the epilogue (warp 4+q reads
// lane quarter q of tensor memory).  Shared memory: Q (64 KiB), two row chunks
// (2 x 64 KiB), two P tiles (2 x 8 KiB), two plans.  Tensor memory: two S
// buffers (64 columns each) and O^T (4 x 64 columns).  Every wait is bounded;
// a timeout raises DS41_E_TIMEOUT and the CTA drains its copies and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ds41_internal.cuh"

namespace ds41 {
namespace tc {

constexpr int HD = 512;
constexpr int NH = 64;            // heads per work item
constexpr int RC = 64;            // rows per chunk
constexpr int THREADS = 256;
constexpr int MAXK = 1024;        // longest index row this kernel takes
constexpr int DCAP = 2048;        // longest row range loaded as consecutive rows
constexpr int MAXCH = 64;         // chunks per item (dense <= DCAP/64 per source, lists <= MAXK/64)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_LOG2 = 4.0f;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t KB_BYTES = RC * 64 * 2;            // one 64-column block of 64 rows: 8 KiB
constexpr uint32_t Q_OFF = 0;                         // 8 blocks of [64 heads][64 dims]
constexpr uint32_t R_OFF = 65536;                     // 2 buffers x 8 blocks of [64 rows][64 dims]
constexpr uint32_t R_BYTES = 65536;
constexpr uint32_t P_OFF = R_OFF + 2 * R_BYTES;       // 2 buffers of [64 heads][64 rows] bf16
constexpr uint32_t P_BYTES = 8192;
constexpr uint32_t PLAN_OFF = P_OFF + 2 * P_BYTES;    // 2 plans
constexpr uint32_t PLAN_DESC = 0;                     // MAXCH x uint4
constexpr uint32_t PLAN_LIST = MAXCH * 16;            // MAXK x int32
constexpr uint32_t PLAN_N = PLAN_LIST + MAXK * 4;     // chunk count
constexpr uint32_t PLAN_BYTES = PLAN_N + 64;
constexpr uint32_t BM_OFF = PLAN_OFF + 2 * PLAN_BYTES;  // 2 sources x DCAP bits
constexpr uint32_t BM_WORDS = DCAP / 32;
constexpr uint32_t MISC_OFF = BM_OFF + 2 * BM_WORDS * 4;
constexpr uint32_t MISC_BYTES = 1024;
constexpr uint32_t SMEM_BYTES = MISC_OFF + MISC_BYTES + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(PLAN_OFF % 16 == 0 && PLAN_BYTES % 16 == 0, "plan alignment");

// barriers
enum {
    B_QFULL, B_QEMPTY, B_RFULL, B_RFULL1, B_SFULL, B_SFULL1, B_SEMPTY, B_SEMPTY1, B_PFULL,
    B_PFULL1, B_DONE, B_DONE1, B_ODONE, B_OFREE, B_PLANFULL, B_PLANFULL1, B_PLANEMPTY,
    B_PLANEMPTY1, B_FINAL, NBAR
};
// misc area layout
constexpr uint32_t M_BAR = 0;                   // NBAR x 8
constexpr uint32_t M_TMEM = 256;                // tensor memory base address
constexpr uint32_t M_ABORT = 260;               // set when any wait gave up
constexpr uint32_t M_VOTE = 272;                // 2 x 4 ints
constexpr uint32_t M_CORR = 320;                // 64 floats
constexpr uint32_t M_INVL = 576;                // 64 floats
static_assert(NBAR * 8 <= 256 && M_INVL + 256 <= MISC_BYTES, "misc layout");

// tensor memory columns
constexpr uint32_t TM_S = 0;     // S buffer b at column 64 b
constexpr uint32_t TM_O = 128;   // O^T tile mt at column 128 + 64 mt
constexpr uint32_t TM_COLS = 512;

struct Params {
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

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0,
                                            int y1, int y2, int y3, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
        "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
            smem_u32(bar))
        : "memory");
}
// 32 consecutive columns of this warp's 32 lanes: r[i] = column col + i of
// lane (lane quarter base + lane id).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
        "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
        "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void named_sync_softmax() {
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, start / leading /
// stride byte offsets (each encoded >> 4), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: bf16 A and B, f32 accumulator, the
// majorness of A and B (0 = K-major, 1 = M/N-major), N and M.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t IDESC_S = idesc_bf16(64, 64, 0, 0);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 64, 1, 0);

// A bounded wait that also gives up once another role has given up.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_f,
                                         unsigned int* status) {
    for (uint32_t i = 0; i < kWaitPolls; i++) {
        uint32_t done;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 63u) == 63u && *abort_f) return false;
    }
    *abort_f = 1;
    raise_status(status, DS41_E_TIMEOUT);
    return false;
}

// Work item k of this CTA -> (token, head group): items are taken from the
// end (longest index rows first when later tokens see more rows).
__device__ __forceinline__ void item_of(int j, int m, int hg, int& t, int& g) {
    const int64_t k = (int64_t)blockIdx.x + (int64_t)j * gridDim.x;
    const int64_t r = (int64_t)m * hg - 1 - k;
    t = (int)(r / hg);
    g = (int)(r % hg);
}

// ---------------------------------------------------------------------------
// Plan warp: index row of one item -> chunk descriptors
//   desc.x: bit 0 source (0 rows_a, 1 rows_b), bit 1 listed rows
//   desc.y: first row of a consecutive chunk, or offset into the row list
//   desc.z/w: mask of the chunk's 64 rows (row r selected iff bit r)
// ---------------------------------------------------------------------------
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

__device__ void plan_item(const Params& p, int t, uint8_t* plan, uint32_t* bm, int lane) {
    uint4* desc = reinterpret_cast<uint4*>(plan + PLAN_DESC);
    int* list = reinterpret_cast<int*>(plan + PLAN_LIST);
    const int32_t* irow = p.idx + (int64_t)t * p.K;
    const int64_t n_rows = p.n_a + p.n_c;
    const int na = (int)p.n_a;

    int cnt[2] = {0, 0}, mn[2] = {INT_MAX, INT_MAX}, mx[2] = {-1, -1};
    for (int j = lane; j < p.K; j += 32) {
        const int v = irow[j];
        if (v == -1) continue;
        if (v < -1 || (int64_t)v >= n_rows) {
            raise_status(p.status, DS41_E_INDEX);
            continue;
        }
        const int s = v >= na;
        const int y = s ? v - na : v;
        cnt[s]++;
        mn[s] = min(mn[s], y);
        mx[s] = max(mx[s], y);
    }
    bool dense[2];
    int range[2];
#pragma unroll
    for (int s = 0; s < 2; s++) {
        cnt[s] = warp_sum(cnt[s]);
        mn[s] = warp_min(mn[s]);
        mx[s] = warp_max(mx[s]);
        range[s] = cnt[s] ? mx[s] - mn[s] + 1 : 0;
        dense[s] = cnt[s] > 0 && range[s] <= DCAP && range[s] <= 2 * cnt[s] + RC;
        if (dense[s]) {
            const int nw = ((range[s] + RC - 1) / RC) * 2;
            for (int w = lane; w < nw; w += 32) bm[s * BM_WORDS + w] = 0u;
        }
    }
    __syncwarp();
    if (dense[0] || dense[1]) {
        bool dup[2] = {false, false};
        for (int j = lane; j < p.K; j += 32) {
            const int v = irow[j];
            if (v < 0 || (int64_t)v >= n_rows) continue;
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
        off[s] = pos;
        for (int base = 0; base < p.K; base += 32) {
            const int j = base + lane;
            const int v = j < p.K ? irow[j] : -1;
            const bool take = v >= 0 && (int64_t)v < n_rows && ((v >= na) == (s == 1));
            const uint32_t bal = __ballot_sync(0xffffffffu, take);
            if (take) list[pos + __popc(bal & lt)] = s ? v - na : v;
            pos += __popc(bal);
        }
    }
    int nch = 0;
#pragma unroll
    for (int s = 0; s < 2; s++) {
        if (cnt[s] == 0) continue;
        if (dense[s]) {
            const int nck = (range[s] + RC - 1) / RC;
            for (int base = 0; base < nck; base += 32) {
                const int i = base + lane;
                uint32_t lo = 0, hi = 0;
                if (i < nck) {
                    lo = bm[s * BM_WORDS + 2 * i];
                    hi = bm[s * BM_WORDS + 2 * i + 1];
                }
                const bool keep = (lo | hi) != 0u;
                const uint32_t bal = __ballot_sync(0xffffffffu, keep);
                if (keep)
                    desc[nch + __popc(bal & lt)] =
                        make_uint4((uint32_t)s, (uint32_t)(mn[s] + RC * i), lo, hi);
                nch += __popc(bal);
            }
        } else {
            const int nck = (cnt[s] + RC - 1) / RC;
            for (int i = lane; i < nck; i += 32) {
                const int n = min(RC, cnt[s] - RC * i);
                const uint32_t lo = n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
                const uint32_t hi = n >= 64 ? 0xffffffffu : (n > 32 ? ((1u << (n - 32)) - 1u) : 0u);
                desc[nch + i] = make_uint4((uint32_t)s | 2u, (uint32_t)(off[s] + RC * i), lo, hi);
            }
            nch += nck;
        }
    }
    if (nch == 0) {  // nothing valid: one fully masked chunk of out-of-range (zero) rows
        if (lane == 0) desc[0] = make_uint4(0u, 1u << 30, 0u, 0u);
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
                   const __grid_constant__ CUtensorMap map_ag,
                   const __grid_constant__ CUtensorMap map_bd,
                   const __grid_constant__ CUtensorMap map_bg, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + MISC_OFF + M_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + MISC_OFF + M_TMEM);
    volatile int* abort_f = reinterpret_cast<volatile int*>(sm + MISC_OFF + M_ABORT);
    int* vote = reinterpret_cast<int*>(sm + MISC_OFF + M_VOTE);
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
        for (int b = 0; b < 2; b++) {
            mbar_init(&bars[B_RFULL + b], 1);
            mbar_init(&bars[B_SFULL + b], 1);
            mbar_init(&bars[B_SEMPTY + b], 4);
            mbar_init(&bars[B_PFULL + b], 4);
            mbar_init(&bars[B_DONE + b], 1);
            mbar_init(&bars[B_PLANFULL + b], 1);
            mbar_init(&bars[B_PLANEMPTY + b], 2);
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
        // TMA producer (one lane)
        // ------------------------------------------------------------------
        if (lane == 0) {
            uint32_t g = 0;
            uint32_t q_armed = 0, r_armed[2] = {0, 0};
            for (int j = 0; j < ntok; j++) {
                int t, hgi;
                item_of(j, p.m, hg, t, hgi);
                const int slot = j & 1;
                if (!wait_bar(&bars[B_PLANFULL + slot], (j >> 1) & 1, abort_f, p.status)) break;
                if (j >= 1 && !wait_bar(&bars[B_QEMPTY], (j - 1) & 1, abort_f, p.status)) break;
                mbar_arrive_expect_tx(&bars[B_QFULL], 8 * KB_BYTES);
                q_armed++;
                const int qrow = t * p.nh + hgi * NH;
                for (int kb = 0; kb < 8; kb++)
                    tma_load_2d(sbase + Q_OFF + kb * KB_BYTES, &map_q, kb * 64, qrow,
                                &bars[B_QFULL]);
                const uint8_t* plan = sm + PLAN_OFF + slot * PLAN_BYTES;
                const uint4* desc = reinterpret_cast<const uint4*>(plan + PLAN_DESC);
                const int* list = reinterpret_cast<const int*>(plan + PLAN_LIST);
                const int nch = *reinterpret_cast<const int*>(plan + PLAN_N);
                bool ok = true;
                for (int i = 0; i < nch; i++, g++) {
                    const int b = g & 1;
                    if (g >= 2 && !wait_bar(&bars[B_DONE + b], ((g - 2) >> 1) & 1, abort_f,
                                            p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[B_RFULL + b], 8 * KB_BYTES);
                    r_armed[b]++;
                    const uint4 d = desc[i];
                    const uint32_t rb = sbase + R_OFF + b * R_BYTES;
                    if (!(d.x & 2u)) {
                        const CUtensorMap* mp = (d.x & 1u) ? &map_bd : &map_ad;
                        for (int kb = 0; kb < 8; kb++)
                            tma_load_2d(rb + kb * KB_BYTES, mp, kb * 64, (int)d.y,
                                        &bars[B_RFULL + b]);
                    } else {
                        const CUtensorMap* mp = (d.x & 1u) ? &map_bg : &map_ag;
                        const int cnt = __popc(d.z) + __popc(d.w);
                        const int* lr = list + d.y;
                        for (int gq = 0; gq < RC / 4; gq++) {
                            int y[4];
#pragma unroll
                            for (int k = 0; k < 4; k++) {
                                const int r = 4 * gq + k;
                                y[k] = r < cnt ? lr[r] : (1 << 30);  // beyond the list: zero fill
                            }
                            for (int kb = 0; kb < 8; kb++)
                                tma_gather4(rb + kb * KB_BYTES + gq * 512, mp, kb * 64, y[0], y[1],
                                            y[2], y[3], &bars[B_RFULL + b]);
                        }
                    }
                }
                if (!ok) break;
                mbar_arrive(&bars[B_PLANEMPTY + slot]);
            }
            // let every copy this CTA started land before the CTA exits
            if (q_armed) wait_bar(&bars[B_QFULL], (q_armed - 1) & 1, abort_f, p.status);
            for (int b = 0; b < 2; b++)
                if (r_armed[b]) wait_bar(&bars[B_RFULL + b], (r_armed[b] - 1) & 1, abort_f, p.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer (one lane): S(g) may run one chunk ahead of PV(g-1)
        // ------------------------------------------------------------------
        if (lane == 0) {
            int s_tok = 0, s_i = 0, s_n = -1;
            int p_tok = 0, p_i = 0;
            uint32_t sg = 0, pg = 0;
            int nring[4] = {0, 0, 0, 0};
            uint32_t idle = 0;
            const uint32_t q_s = sbase + Q_OFF;
            while (p_tok < ntok) {
                bool prog = false;
                if (s_tok < ntok) {
                    if (s_n < 0 && mbar_test(&bars[B_PLANFULL + (s_tok & 1)], (s_tok >> 1) & 1)) {
                        s_n = *reinterpret_cast<const int*>(sm + PLAN_OFF +
                                                            (s_tok & 1) * PLAN_BYTES + PLAN_N);
                        nring[s_tok & 3] = s_n;
                    }
                    if (s_n > 0 && sg < pg + 2) {
                        const int b = sg & 1;
                        const bool ok =
                            mbar_test(&bars[B_RFULL + b], (sg >> 1) & 1) &&
                            (sg < 2 || mbar_test(&bars[B_SEMPTY + b], ((sg - 2) >> 1) & 1)) &&
                            (s_i > 0 || mbar_test(&bars[B_QFULL], s_tok & 1));
                        if (ok) {
                            tc_fence_after();
                            const uint32_t r_s = sbase + R_OFF + b * R_BYTES;
                            const uint32_t d = tmem + TM_S + 64 * b;
#pragma unroll 4
                            for (int kk = 0; kk < HD / 16; kk++) {
                                const uint32_t off = (kk >> 2) * KB_BYTES + (kk & 3) * 32;
                                tc_mma(d, sdesc(q_s + off, 16, 1024), sdesc(r_s + off, 16, 1024),
                                       IDESC_S, kk > 0);
                            }
                            tc_commit(&bars[B_SFULL + b]);
                            if (s_i == s_n - 1) tc_commit(&bars[B_QEMPTY]);
                            sg++;
                            if (++s_i == s_n) {
                                s_tok++;
                                s_i = 0;
                                s_n = -1;
                            }
                            prog = true;
                        }
                    }
                }
                if (pg < sg) {
                    const int b = pg & 1;
                    const bool ok =
                        mbar_test(&bars[B_PFULL + b], (pg >> 1) & 1) &&
                        (p_i > 0 || p_tok == 0 || mbar_test(&bars[B_OFREE], (p_tok - 1) & 1));
                    if (ok) {
                        tc_fence_after();
                        const uint32_t r_s = sbase + R_OFF + b * R_BYTES;
                        const uint32_t p_s = sbase + P_OFF + b * P_BYTES;
#pragma unroll
                        for (int mt = 0; mt < 4; mt++) {
                            const uint32_t d = tmem + TM_O + 64 * mt;
#pragma unroll
                            for (int kk = 0; kk < RC / 16; kk++)
                                tc_mma(d, sdesc(r_s + 2 * mt * KB_BYTES + kk * 2048, KB_BYTES, 1024),
                                       sdesc(p_s + kk * 32, 16, 1024), IDESC_PV,
                                       (p_i > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(&bars[B_DONE + b]);
                        const int pn = nring[p_tok & 3];
                        if (p_i == pn - 1) tc_commit(&bars[B_ODONE]);
                        pg++;
                        if (++p_i == pn) {
                            p_tok++;
                            p_i = 0;
                        }
                        prog = true;
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
            wait_bar(&bars[B_FINAL], 0, abort_f, p.status);
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
    } else if (warp >= 4) {
        // ------------------------------------------------------------------
        // Softmax + epilogue: warp 4+q reads lane quarter q; with M = 64 the
        // scores of head 16q + l sit in lane 32q + l (l < 16), one column per
        // row of the chunk.
        // ------------------------------------------------------------------
        const int q = warp - 4;
        const int tid = threadIdx.x - 128;
        const bool own = lane < 16;
        const int hl = 16 * q + lane;  // this thread's head (own lanes)
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        uint32_t g = 0;
        bool bad = false;  // a wait of this thread gave up
        for (int j = 0; j < ntok; j++) {
            int t, hgi;
            item_of(j, p.m, hg, t, hgi);
            const int slot = j & 1;
            if (!wait_bar(&bars[B_PLANFULL + slot], (j >> 1) & 1, abort_f, p.status)) bad = true;
            const uint8_t* plan = sm + PLAN_OFF + slot * PLAN_BYTES;
            const uint4* desc = reinterpret_cast<const uint4*>(plan + PLAN_DESC);
            const int nch = bad ? 1 : *reinterpret_cast<const int*>(plan + PLAN_N);
            float m_ref = -INFINITY, l = 0.0f;
            bool stop = false;
            for (int i = 0; i < nch; i++, g++) {
                const int b = g & 1;
                const uint4 d = bad ? make_uint4(0, 0, 0, 0) : desc[i];
                if (!bad && !wait_bar(&bars[B_SFULL + b], (g >> 1) & 1, abort_f, p.status))
                    bad = true;
                tc_fence_after();
                uint32_t s0[32], s1[32];
                tc_ld32(tmem + lane_off + TM_S + 64 * b, s0);
                tc_ld32(tmem + lane_off + TM_S + 64 * b + 32, s1);
                tc_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_SEMPTY + b]);
                // scaled scores (log2 units) and the chunk max over selected rows
                float mx = -INFINITY;
#pragma unroll
                for (int k = 0; k < 32; k++) {
                    const float x0 = __uint_as_float(s0[k]) * p.scale_log2;
                    const float x1 = __uint_as_float(s1[k]) * p.scale_log2;
                    s0[k] = __float_as_uint(((d.z >> k) & 1u) ? x0 : -INFINITY);
                    s1[k] = __float_as_uint(((d.w >> k) & 1u) ? x1 : -INFINITY);
                    mx = fmaxf(mx, fmaxf(__uint_as_float(s0[k]), __uint_as_float(s1[k])));
                }
                bool need = false;
                if (i == 0) m_ref = mx;
                else need = own && mx > m_ref + RESCALE_LOG2;
                // one vote per chunk: a rescale anywhere, or a wait that gave up
                const uint32_t v = (__any_sync(0xffffffffu, need) ? 1u : 0u) |
                                   (__any_sync(0xffffffffu, bad) ? 2u : 0u);
                if (lane == 0) vote[b * 4 + q] = (int)v;
                named_sync_softmax();
                const int all = vote[b * 4 + 0] | vote[b * 4 + 1] | vote[b * 4 + 2] | vote[b * 4 + 3];
                if (all & 2) {
                    stop = true;
                    break;
                }
                if (i == nch - 1 && tid == 0) mbar_arrive(&bars[B_PLANEMPTY + slot]);
                if (all & 1) {
                    // move the reference of the heads that need it; rescale O^T
                    float corr = 1.0f;
                    if (need) {
                        corr = exp2f(m_ref - mx);
                        m_ref = mx;
                        l *= corr;
                    }
                    if (own) corr_s[hl] = corr;
                    if (!wait_bar(&bars[B_DONE + ((g - 1) & 1)], ((g - 1) >> 1) & 1, abort_f,
                                  p.status))
                        bad = true;
                    tc_fence_after();
                    named_sync_softmax();
                    if (!bad) {
#pragma unroll 1
                        for (int mt = 0; mt < 4; mt++) {
#pragma unroll 1
                            for (int hh = 0; hh < 2; hh++) {
                                uint32_t ov[32];
                                const uint32_t ta = tmem + lane_off + TM_O + 64 * mt + 32 * hh;
                                tc_ld32(ta, ov);
                                tc_wait_ld();
#pragma unroll
                                for (int k = 0; k < 32; k++)
                                    ov[k] = __float_as_uint(__uint_as_float(ov[k]) *
                                                            corr_s[32 * hh + k]);
                                tc_st32(ta, ov);
                            }
                        }
                        tc_wait_st();
                    }
                }
                // probabilities, the denominator, P (bf16) for the PV MMA
                const float mu = (m_ref == -INFINITY) ? 0.0f : m_ref;
                float lsum = 0.0f;
                uint32_t pk[32];
#pragma unroll
                for (int k = 0; k < 16; k++) {
                    const float a0 = exp2f(__uint_as_float(s0[2 * k]) - mu);
                    const float a1 = exp2f(__uint_as_float(s0[2 * k + 1]) - mu);
                    const float c0 = exp2f(__uint_as_float(s1[2 * k]) - mu);
                    const float c1 = exp2f(__uint_as_float(s1[2 * k + 1]) - mu);
                    lsum += (a0 + a1) + (c0 + c1);
                    pk[k] = pack_bf16x2(a0, a1);
                    pk[16 + k] = pack_bf16x2(c0, c1);
                }
                l += lsum;
                if (g >= 2 && !bad &&
                    !wait_bar(&bars[B_DONE + b], ((g - 2) >> 1) & 1, abort_f, p.status))
                    bad = true;
                if (own) {
                    // row hl of P: 128 bytes = 8 chunks of 16, swizzled by hl % 8
                    uint8_t* prow = sm + P_OFF + b * P_BYTES + (hl >> 3) * 1024 + (hl & 7) * 128;
#pragma unroll
                    for (int c = 0; c < 8; c++)
                        *reinterpret_cast<uint4*>(prow + ((c ^ (hl & 7)) << 4)) =
                            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                }
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_PFULL + b]);
            }
            if (stop) break;
            // ---- epilogue of this item ----
            const int h = hgi * NH + hl;
            if (own) {
                const float sk = p.sink[h] * LOG2E;
                const float M = fmaxf(m_ref, sk);
                const float Mr = (M == -INFINITY) ? 0.0f : M;
                const float a = exp2f(m_ref - Mr);
                const float L = l * a + exp2f(sk - Mr);
                invl_s[hl] = (L > 0.0f) ? a / L : 0.0f;
                if (p.lse) p.lse[(int64_t)t * p.nh + h] = (Mr + log2f(L)) / LOG2E;
            }
            if (!bad && !wait_bar(&bars[B_ODONE], j & 1, abort_f, p.status)) bad = true;
            tc_fence_after();
            named_sync_softmax();
            if (!bad) {
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
                            obase[(int64_t)c * HD + dd] = f2bf(__uint_as_float(ov[k]) * invl_s[c]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_OFREE]);
        }
    }

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
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::mutex g_encode_mu;

static int get_encode(PFN_cuTensorMapEncodeTiled_v12000* out) {
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult qr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &qr);
        if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn)
            return fail(DS41_E_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return DS41_OK;
}

// 2-D bf16 map over [rows][512] with a box of 64 columns x box_rows rows and
// the 128-byte swizzle; elements outside the tensor read as zero.
static int make_map(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* m, const void* ptr,
                    int64_t rows, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)HD, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)HD * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DS41_E_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return DS41_OK;
}

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
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    int rc = get_encode(&enc);
    if (rc) return rc;
    CUtensorMap mq, mad, mag, mbd, mbg;
    if ((rc = make_map(enc, &mq, q, m * nh, 64))) return rc;
    if ((rc = make_map(enc, &mad, rows_a, n_a, RC))) return rc;
    if ((rc = make_map(enc, &mag, rows_a, n_a, 1))) return rc;
    if ((rc = make_map(enc, &mbd, rows_b, n_c, RC))) return rc;
    if ((rc = make_map(enc, &mbg, rows_b, n_c, 1))) return rc;
    Params p;
    p.n_a = n_a;
    p.n_c = n_c;
    p.idx = idx;
    p.K = (int)K;
    p.nh = (int)nh;
    p.m = (int)m;
    p.scale_log2 = scale * LOG2E;
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
    kern<<<grid, THREADS, SMEM_BYTES, st>>>(mq, mad, mag, mbd, mbg, p);
    return launch_check("ds41_sparse_attn_sink_fwd: tensor-core kernel");
}

}  // namespace ds41
