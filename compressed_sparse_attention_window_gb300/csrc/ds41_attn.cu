// ds41_attn.cu - step 3 of the forward: sparse attention of every head over
// the gathered window + compressed rows, with a per-head sink logit.
//
// metrale_model_arch/deepseek_v41_ref/compress.rs, attention_any: sparse_attn
// (q, kv_rows, sink, idx, m, nh, hd, topk, scale) with scale = head_dim^-0.5;
// metrale_model_arch/attn_v41/forward.rs passes rows_a, rows_b and the merged
// idx to attend_and_project.  One row per position is both key and value.
//
//   o[t,h] = sum_v e^{s_v} row_v / (e^{sink_h} + sum_v e^{s_v}),
//   s_v = scale * <q[t,h], row_v>
//
// One CTA handles one query token, 64 heads, and a contiguous range of its
// index row (a split).  Eight warps: warp w owns heads 16*(w%4).. and half
// w/4 of the head dim.  Per chunk of 32 gathered rows the two warps of a head
// group each form the partial scores of their half, exchange them through
// shared memory, and both run the same online softmax on the full scores;
// each then accumulates P*V for its half of the output columns.  Rows are
// gathered with cp.async (double-buffered); tensor-core MMAs are bf16 with f32
// accumulation.  With several splits the unnormalised (m, l, O) of each split
// goes to the workspace and a merge kernel adds the sink once.  In the whole
// step, when the CTAs fit one wave with one split each, every CTA builds its
// token's index row itself from the indexer scores (SEL).
#include <cooperative_groups.h>

#include <mutex>

#include "ds41_internal.cuh"
#include "ds41_topk.cuh"

namespace ds41 {

constexpr int ATT_NC = 32;       // gathered rows per chunk
constexpr int ATT_STAGE = 4096;  // indices of a CTA's range staged in shared memory
constexpr int ATT_HEADS = 64;    // heads per CTA
constexpr int ATT_THREADS = 256;
constexpr float LOG2E = 1.4426950408889634f;

template <int HD>
struct AttnSmem {
    static constexpr int CPR = HD / 8;  // 16-byte chunks per row
    static constexpr size_t q_bytes = (size_t)ATT_HEADS * HD * 2;
    static constexpr size_t kv_bytes = (size_t)ATT_NC * HD * 2;
    static constexpr size_t sx_bytes = (size_t)2 * ATT_HEADS * ATT_NC * 4;
    static constexpr size_t total =
        q_bytes + 2 * kv_bytes + sx_bytes + 2 * ATT_NC * 4 + (size_t)ATT_STAGE * 4;
};

__device__ __forceinline__ int aswz(int row, int c) { return c ^ (row & 7); }

// SEL: the CTA builds its token's merged index row itself, from the
// indexer scores of the kernel before (tk; one split, K <= ATT_STAGE, at most
// WTK_MAX visible scores): the window entries, then warp 0 ranks the visible
// scores (warp_topk), and head group 0 writes the row to tk.idx_out.
template <int HD, bool SEL>
__global__ void __launch_bounds__(ATT_THREADS, 1) sparse_attn_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ rows_a, int64_t n_a,
    const uint16_t* __restrict__ rows_b, int64_t n_c, const int32_t* __restrict__ idx, int K,
    const float* __restrict__ sink, float scale_log2, uint16_t* __restrict__ o,
    float* __restrict__ lse, int nh, int chunks_per_split, float* __restrict__ part_o,
    float2* __restrict__ part_ml, unsigned int* status, DecTopk tk) {
    // the rows the query can see (a 64-bit division, from the arguments
    // alone) while the kernel before finishes
    int64_t vis = 0;
    if constexpr (SEL) {
        vis = (tk.start_pos + (int64_t)blockIdx.x + 1) / tk.ratio;
        if (vis > tk.n_c) vis = tk.n_c;
    }
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    pdl_trigger();
    using SM = AttnSmem<HD>;
    constexpr int CPR = SM::CPR;
    constexpr int HALF = HD / 2;
    constexpr int NT = HALF / 8;  // output n-tiles per warp
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t* qs = reinterpret_cast<uint16_t*>(smem);
    uint16_t* kvs = reinterpret_cast<uint16_t*>(smem + SM::q_bytes);
    float* sx = reinterpret_cast<float*>(smem + SM::q_bytes + 2 * SM::kv_bytes);
    int* vflag = reinterpret_cast<int*>(smem + SM::q_bytes + 2 * SM::kv_bytes + SM::sx_bytes);
    int* sidx = vflag + 2 * ATT_NC;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = warp & 3, half = warp >> 2;
    const int64_t t = blockIdx.x;
    const int split = blockIdx.y;
    const int splits = gridDim.y;
    const int h0 = blockIdx.z * ATT_HEADS;
    const int64_t n_rows = n_a + n_c;

    const int nchunks_total = (K + ATT_NC - 1) / ATT_NC;
    const int c_begin = split * chunks_per_split;
    int c_end = c_begin + chunks_per_split;
    if (c_end > nchunks_total) c_end = nchunks_total;
    const int32_t* irow = idx + t * (int64_t)K;

    // Q of 64 heads (rows beyond nh are zero).
    for (int id = tid; id < ATT_HEADS * CPR; id += ATT_THREADS) {
        const int r = id / CPR, c = id % CPR;
        const int h = h0 + r;
        const bool live = h < nh;
        const uint16_t* src = q + ((t * nh + (live ? h : 0)) * (int64_t)HD) + c * 8;
        cp_async16(smem_u32(qs + r * HD + aswz(r, c) * 8), src, live);
    }
    // The indices of this CTA's range go to shared memory in one coalesced
    // pass, so the gathers below do not wait on a global load per row.
    const int jr0 = c_begin * ATT_NC;
    const int nst = max(0, min(min(K, c_end * ATT_NC) - jr0, ATT_STAGE));
    if constexpr (SEL) {
        // [window entries | the kk best visible rows, ascending | -1] (one
        // split: jr0 = 0 and nst = K)
        const int win = tk.win;
        const int kk = (int)(vis < tk.ctopk ? vis : tk.ctopk);
        for (int j = tid; j < K; j += ATT_THREADS) {
            if (j < win) sidx[j] = window_index(tk.start_pos, tk.m, win, t, j);
            else if (j - win >= kk) sidx[j] = -1;
            else if (vis <= tk.ctopk) sidx[j] = (int)(tk.offset + (j - win));
        }
        if (vis > tk.ctopk && warp == 0) {
            int* hist = reinterpret_cast<int*>(sx);  // free until the chunks below
            warp_topk(tk.scores + t * tk.n_c, (int)vis, kk, hist, hist + 256,
                      [&](int pos, int r) { sidx[win + pos] = (int)(tk.offset + r); });
        }
        __syncthreads();
        if (blockIdx.z == 0)
            for (int j = tid; j < K; j += ATT_THREADS) tk.idx_out[t * (int64_t)K + j] = sidx[j];
    } else {
        for (int j = tid; j < nst; j += ATT_THREADS) sidx[j] = irow[jr0 + j];
    }
    __syncthreads();
    auto load_chunk = [&](int chunk, int buf) {
        uint16_t* dst = kvs + buf * (ATT_NC * HD);
        for (int id = tid; id < ATT_NC * CPR; id += ATT_THREADS) {
            const int r = id / CPR, c = id % CPR;
            const int j = chunk * ATT_NC + r;
            int64_t v = -1;
            if (j - jr0 < nst) v = sidx[j - jr0];
            else if (j < K) v = irow[j];
            bool ok = v >= 0 && v < n_rows;
            if (c == 0) {
                if (j < K && (v < -1 || v >= n_rows)) raise_status(status, DS41_E_INDEX);
                vflag[buf * ATT_NC + r] = ok ? 1 : 0;
            }
            const uint16_t* src = rows_a;
            if (ok) src = (v < n_a) ? rows_a + v * HD : rows_b + (v - n_a) * HD;
            cp_async16(smem_u32(dst + r * HD + aswz(r, c) * 8), src + c * 8, ok);
        }
    };

    float oacc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; j++) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.0f;
    float mrow[2] = {-INFINITY, -INFINITY};  // running max (log2 units) of rows lane/4, +8
    float lrow[2] = {0.0f, 0.0f};            // this thread's partial denominators

    if (c_begin < c_end) load_chunk(c_begin, 0);
    cp_async_commit();

    for (int chunk = c_begin; chunk < c_end; chunk++) {
        const int buf = (chunk - c_begin) & 1;
        if (chunk + 1 < c_end) load_chunk(chunk + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const uint16_t* kv = kvs + buf * (ATT_NC * HD);

        // partial scores of this half: [16 heads] x [32 rows]
        float sacc[4][4];
#pragma unroll
        for (int j = 0; j < 4; j++) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.0f;
#pragma unroll 4
        for (int kk = 0; kk < HALF / 16; kk++) {
            uint32_t a0, a1, a2, a3;
            {
                const int r = g * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = half * (HALF / 8) + kk * 2 + (lane >> 4);
                ldsm_x4(smem_u32(qs + r * HD + aswz(r, c) * 8), a0, a1, a2, a3);
            }
#pragma unroll
            for (int jj = 0; jj < 2; jj++) {
                uint32_t b0, b1, b2, b3;
                const int r = jj * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = half * (HALF / 8) + kk * 2 + ((lane >> 3) & 1);
                ldsm_x4(smem_u32(kv + r * HD + aswz(r, c) * 8), b0, b1, b2, b3);
                mma_bf16(sacc[2 * jj], a0, a1, a2, a3, b0, b1);
                mma_bf16(sacc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        // exchange halves
        float* mine = sx + half * (ATT_HEADS * ATT_NC);
        const float* other = sx + (half ^ 1) * (ATT_HEADS * ATT_NC);
        const int ra = g * 16 + (lane >> 2), rb = ra + 8;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int col = j * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2*>(mine + ra * ATT_NC + col) = make_float2(sacc[j][0], sacc[j][1]);
            *reinterpret_cast<float2*>(mine + rb * ATT_NC + col) = make_float2(sacc[j][2], sacc[j][3]);
        }
        asm volatile("bar.sync %0, 64;\n" ::"r"(1 + g));
        float sv[4][4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int col = j * 8 + 2 * (lane & 3);
            const float2 xa = *reinterpret_cast<const float2*>(other + ra * ATT_NC + col);
            const float2 xb = *reinterpret_cast<const float2*>(other + rb * ATT_NC + col);
            // the same sum, in the same order, in both warps of the pair
            const float s0 = half ? xa.x + sacc[j][0] : sacc[j][0] + xa.x;
            const float s1 = half ? xa.y + sacc[j][1] : sacc[j][1] + xa.y;
            const float s2 = half ? xb.x + sacc[j][2] : sacc[j][2] + xb.x;
            const float s3 = half ? xb.y + sacc[j][3] : sacc[j][3] + xb.y;
            const bool v0 = vflag[buf * ATT_NC + col] != 0;
            const bool v1 = vflag[buf * ATT_NC + col + 1] != 0;
            sv[j][0] = v0 ? s0 * scale_log2 : -INFINITY;
            sv[j][1] = v1 ? s1 * scale_log2 : -INFINITY;
            sv[j][2] = v0 ? s2 * scale_log2 : -INFINITY;
            sv[j][3] = v1 ? s3 * scale_log2 : -INFINITY;
        }
        // online softmax on rows ra (sv[.][0..1]) and rb (sv[.][2..3])
        float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            mx[0] = fmaxf(mx[0], fmaxf(sv[j][0], sv[j][1]));
            mx[1] = fmaxf(mx[1], fmaxf(sv[j][2], sv[j][3]));
        }
#pragma unroll
        for (int i = 0; i < 2; i++) {
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
        }
        float corr[2], muse[2];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            muse[i] = (mx[i] == -INFINITY) ? 0.0f : mx[i];
            corr[i] = exp2f(mrow[i] - muse[i]);
            mrow[i] = mx[i];
            lrow[i] *= corr[i];
        }
        uint32_t pa[2][4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float p0 = exp2f(sv[j][0] - muse[0]), p1 = exp2f(sv[j][1] - muse[0]);
            const float p2 = exp2f(sv[j][2] - muse[1]), p3 = exp2f(sv[j][3] - muse[1]);
            lrow[0] += p0 + p1;
            lrow[1] += p2 + p3;
            // C fragment of n-tile j -> A fragment of k-step j/2
            pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
            pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
        }
#pragma unroll
        for (int j = 0; j < NT; j++) {
            oacc[j][0] *= corr[0];
            oacc[j][1] *= corr[0];
            oacc[j][2] *= corr[1];
            oacc[j][3] *= corr[1];
        }
        // O += P * V over this half's columns
#pragma unroll
        for (int ks = 0; ks < 2; ks++) {
            // A fragment order: a0 (row ra, k 0-7), a1 (row rb, k 0-7),
            // a2 (row ra, k 8-15), a3 (row rb, k 8-15)
            const uint32_t a0 = pa[ks][0], a1 = pa[ks][1], a2 = pa[ks][2], a3 = pa[ks][3];
#pragma unroll
            for (int jj = 0; jj < NT / 2; jj++) {
                uint32_t b0, b1, b2, b3;
                const int r = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = half * (HALF / 8) + jj * 2 + (lane >> 4);
                ldsm_x4_t(smem_u32(kv + r * HD + aswz(r, c) * 8), b0, b1, b2, b3);
                mma_bf16(oacc[2 * jj], a0, a1, a2, a3, b0, b1);
                mma_bf16(oacc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();  // buffer and exchange area are reused next chunk
    }
    cp_async_wait<0>();

    // reduce the per-thread denominators over the quad
#pragma unroll
    for (int i = 0; i < 2; i++) {
        lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 1);
        lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 2);
    }
    const int rows[2] = {g * 16 + (lane >> 2), g * 16 + (lane >> 2) + 8};
    if (splits == 1) {
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const int h = h0 + rows[i];
            if (h >= nh) continue;
            const float sk = sink[h] * LOG2E;
            const float mfin = fmaxf(mrow[i], sk);
            const float mref = (mfin == -INFINITY) ? 0.0f : mfin;
            const float a = exp2f(mrow[i] - mref);
            const float L = lrow[i] * a + exp2f(sk - mref);
            const float inv = (L > 0.0f) ? a / L : 0.0f;
            uint16_t* orow = o + (t * nh + h) * (int64_t)HD + half * HALF;
#pragma unroll
            for (int j = 0; j < NT; j++) {
                const int col = j * 8 + 2 * (lane & 3);
                const float x0 = oacc[j][2 * i] * inv, x1 = oacc[j][2 * i + 1] * inv;
                *reinterpret_cast<uint32_t*>(orow + col) = pack_bf16x2(x0, x1);
            }
            if (lse && half == 0 && (lane & 3) == 0) lse[t * nh + h] = (mref + log2f(L)) / LOG2E;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const int h = h0 + rows[i];
            if (h >= nh) continue;
            const int64_t pidx = (t * splits + split) * (int64_t)nh + h;
            float* prow = part_o + pidx * HD + half * HALF;
#pragma unroll
            for (int j = 0; j < NT; j++) {
                const int col = j * 8 + 2 * (lane & 3);
                *reinterpret_cast<float2*>(prow + col) = make_float2(oacc[j][2 * i], oacc[j][2 * i + 1]);
            }
            if (half == 0 && (lane & 3) == 0) part_ml[pidx] = make_float2(mrow[i], lrow[i]);
        }
    }
}

// Merge the splits of one (token, head): M = max(sink, m_s),
// L = e^{sink - M} + sum_s l_s e^{m_s - M}, o = sum_s O_s e^{m_s - M} / L.
template <int HD>
__global__ void __launch_bounds__(128) attn_merge_kernel(const float* __restrict__ part_o,
                                                         const float2* __restrict__ part_ml,
                                                         const float* __restrict__ sink,
                                                         uint16_t* __restrict__ o,
                                                         float* __restrict__ lse, int nh,
                                                         int splits) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    pdl_trigger();
    const int64_t t = blockIdx.x;
    const int h = blockIdx.y;
    const float sk = sink[h] * LOG2E;
    float M = sk;
    for (int s = 0; s < splits; s++) M = fmaxf(M, part_ml[(t * splits + s) * nh + h].x);
    const float Mref = (M == -INFINITY) ? 0.0f : M;
    float L = exp2f(sk - Mref);
    for (int s = 0; s < splits; s++) {
        const float2 ml = part_ml[(t * splits + s) * nh + h];
        L += ml.y * exp2f(ml.x - Mref);
    }
    const float invL = (L > 0.0f) ? 1.0f / L : 0.0f;
    for (int d = threadIdx.x * 2; d < HD; d += blockDim.x * 2) {
        float a0 = 0.0f, a1 = 0.0f;
        for (int s = 0; s < splits; s++) {
            const int64_t pidx = (t * splits + s) * (int64_t)nh + h;
            const float wgt = exp2f(part_ml[pidx].x - Mref);
            const float2 v = *reinterpret_cast<const float2*>(part_o + pidx * HD + d);
            a0 += v.x * wgt;
            a1 += v.y * wgt;
        }
        *reinterpret_cast<uint32_t*>(o + (t * nh + h) * (int64_t)HD + d) =
            pack_bf16x2(a0 * invL, a1 * invL);
    }
    if (lse && threadIdx.x == 0) lse[t * nh + h] = (Mref + log2f(L)) / LOG2E;
}

// ---------------------------------------------------------------------------
constexpr int TKD_CAP = 4096;  // most score keys one CTA ranks in the fused decode step
constexpr int TKD_WHIST = 10752;  // per-warp histograms of the local selection, in its area

// Split halves of a cluster barrier: every CTA arrives once it has started,
// and waits before its first access to another CTA's shared memory.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}

// The selection of dec_topk when every visible score fits in registers
// (vis <= TKD_CAP, at most TKD_CAP / NTH per thread): each CTA ranks all of
// them itself, with the same two 8-bit histogram passes, threshold and tie
// rule (the lowest-numbered ties) as the cluster version, and keeps the picks
// whose positions fall in its own slice [j0, j1).  Thread (w, l) holds the run of
// kpt consecutive scores starting at kpt (32 w + l), so index order is warp,
// lane, register; the histograms are per warp (no same-address atomics across
// warps), and positions come from one warp scan.  No cluster traffic.
template <int NTH>
__device__ void dec_topk_local(const DecTopk& tk, int64_t t, int vis, int kk, int win, int j0, int j1,
                               int* sidx, uint8_t* area, int32_t* orow, bool write_idx) {
    constexpr int NW = NTH / 32;
    constexpr int KMAX = TKD_CAP / NTH;  // 16 with 8 warps
    static_assert(NTH * KMAX == TKD_CAP && KMAX % 8 == 0, "keys per thread");
    int* hist = reinterpret_cast<int*>(area + 8192);
    int* hist2 = hist + 256;
    int* wsum = hist2 + 256;
    int* sel = wsum + 64;
    int* whist = reinterpret_cast<int*>(area + TKD_WHIST);  // [NW][256]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (kk <= 0) return;
    const int kpt = (vis + NTH - 1) / NTH;
    const int i0 = kpt * tid;  // first score of this thread
    const uint16_t* sc = tk.scores + t * tk.n_c;
    uint32_t key[KMAX];
    const bool vec = (kpt & 7) == 0 && ((reinterpret_cast<uintptr_t>(sc) & 15u) == 0);
#pragma unroll
    for (int v = 0; v < KMAX / 8; v++) {
        const int b0 = i0 + 8 * v;
        if (8 * v >= kpt || b0 >= vis) continue;
        if (vec && b0 + 8 <= vis) {  // whole groups of eight only: nothing past vis is read
            uint4 u = __ldg(reinterpret_cast<const uint4*>(sc + b0));
            const uint16_t* h = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
            for (int e = 0; e < 8; e++) key[8 * v + e] = order_key(h[e]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++)
                if (8 * v + e < kpt && b0 + e < vis) key[8 * v + e] = order_key(sc[b0 + e]);
        }
    }
    // keys past vis (or past kpt) take no part: n_mine counts the live ones
    const int n_mine = max(0, min(kpt, vis - i0));
    int* wh = whist + warp * 256;
#pragma unroll
    for (int e = 0; e < 8; e++) wh[lane + 32 * e] = 0;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < KMAX; e++)
        if (e < n_mine) atomicAdd(&wh[key[e] >> 8], 1);
    __syncthreads();
    for (int b = tid; b < 256; b += NTH) {
        int v = 0;
#pragma unroll
        for (int w = 0; w < NW; w++) {
            v += whist[w * 256 + b];
            whist[w * 256 + b] = 0;
        }
        hist[b] = v;
    }
    __syncthreads();
    if (tid < 32) find_bucket(hist, kk, 0, &sel[0], &sel[1]);
    __syncthreads();
    const uint32_t hb = (uint32_t)sel[0];
#pragma unroll
    for (int e = 0; e < KMAX; e++)
        if (e < n_mine && (key[e] >> 8) == hb) atomicAdd(&wh[key[e] & 0xffu], 1);
    __syncthreads();
    for (int b = tid; b < 256; b += NTH) {
        int v = 0;
#pragma unroll
        for (int w = 0; w < NW; w++) v += whist[w * 256 + b];
        hist2[b] = v;
    }
    __syncthreads();
    if (tid < 32) find_bucket(hist2, kk, sel[1], &sel[2], &sel[3]);
    __syncthreads();
    const uint32_t T = (hb << 8) | (uint32_t)sel[2];
    const int need_eq = kk - sel[3];
    // this thread's keys above and at the threshold as bit masks (bit e:
    // key e), so that every key's rank among them is one population count
    uint32_t gm = 0, qm = 0;
#pragma unroll
    for (int e = 0; e < KMAX; e++) {
        gm |= (e < n_mine && key[e] > T) ? (1u << e) : 0u;
        qm |= (e < n_mine && key[e] == T) ? (1u << e) : 0u;
    }
    const int n_gt = __popc(gm), n_eq = __popc(qm);
    // exclusive prefixes over the lanes of the warp, then over the warps
    int x_gt = n_gt, x_eq = n_eq;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, x_gt, off);
        const int b = __shfl_up_sync(0xffffffffu, x_eq, off);
        if (lane >= off) {
            x_gt += a;
            x_eq += b;
        }
    }
    if (lane == 31) {
        wsum[warp] = x_gt;
        wsum[32 + warp] = x_eq;
    }
    __syncthreads();
    int gt = x_gt - n_gt, eq = x_eq - n_eq;
    for (int w = 0; w < warp; w++) {
        gt += wsum[w];
        eq += wsum[32 + w];
    }
    const int v0 = (int)(tk.offset + i0);
#pragma unroll
    for (int e = 0; e < KMAX; e++) {
        const uint32_t below = (1u << e) - 1u;
        const int eqb = eq + __popc(qm & below);  // keys at T before this one
        const bool take = ((gm >> e) & 1u) || (((qm >> e) & 1u) && eqb < need_eq);
        const int j = win + gt + __popc(gm & below) + min(eqb, need_eq);  // merged-row position
        if (take && j >= j0 && j < j1) {
            sidx[j - j0] = v0 + e;
            if (write_idx) orow[j] = v0 + e;
        }
    }
}

// Fill sidx[0 .. j1 - j0) with slice [j0, j1) of the merged index row
// [window indices | the min(ctopk, visible) best compressed rows in ascending
// order | -1].  Every CTA ranks the visible scores itself (dec_topk_local):
// the host fuses the selection into the attention only while they fit one
// CTA's registers (n_c <= TKD_CAP); longer score rows go through the
// separate top-k kernel, which measured faster than any selection split over
// the attention's cluster.
template <int NTH>
__device__ void dec_topk(const DecTopk& tk, int64_t t, int64_t vis, int K, int j0, int j1, int* sidx,
                         uint8_t* area, bool write_idx, unsigned int* status) {
    const int tid = threadIdx.x;
    const int win = tk.win;
    const int kk = (int)(vis < tk.ctopk ? vis : tk.ctopk);
    int32_t* orow = tk.idx_out + t * (int64_t)K;
    // window entries, the picks when every visible row is kept, and padding
    for (int j = j0 + tid; j < j1; j += NTH) {
        int v;
        if (j < win) {
            // the same entry the front writes to win_idx, worked out here
            // rather than read back
            v = window_index(tk.start_pos, tk.m, win, t, j);
        } else if (j - win >= kk) {
            v = -1;
        } else if (vis <= tk.ctopk) {
            v = (int)(tk.offset + (j - win));
        } else {
            continue;  // a pick: stored by the ranking below
        }
        sidx[j - j0] = v;
        if (write_idx) orow[j] = v;
    }
    if (vis <= tk.ctopk) return;  // the same branch in every CTA of the cluster
    if (vis > TKD_CAP) {
        raise_status(status, DS41_E_RANGE);  // excluded by the host plan
        return;
    }
    dec_topk_local<NTH>(tk, t, (int)vis, kk, win, j0, j1, sidx, area, orow, write_idx);
}

// Few-token (decode) path: constants and the shared memory map of
// sparse_attn_decode_kernel below.
// ---------------------------------------------------------------------------
constexpr int DEC_HEADS = 16;
constexpr int DEC_NC = 48;  // gathered rows per chunk: a 16-CTA slice of 640 rows (40) in one chunk
constexpr int DEC_SPS = DEC_NC + 8;  // padded row stride of the partial scores (no bank conflicts)
constexpr int DEC_STAGE = 2048;      // indices of a CTA's slice staged in shared memory
// warps per CTA: 8 when the head dim gives every warp at least two n-tiles
template <int HD>
__host__ __device__ constexpr int dec_warps() { return HD >= 128 ? 8 : 4; }

template <int HD>
struct DecSmem {
    // Rows of q and of the gathered kv are padded to HD + 8 bf16 (a 16-byte
    // multiple): eight consecutive rows then start on eight different 4-bank
    // groups, so ldmatrix reads them without conflicts, and every row can be
    // the destination of one contiguous bulk copy.
    static constexpr int RS = HD + 8;
    static constexpr size_t q_bytes = (size_t)DEC_HEADS * RS * 2;
    static constexpr size_t kv_bytes = (size_t)DEC_NC * RS * 2;  // one buffer
    static constexpr size_t sp_bytes = (size_t)dec_warps<HD>() * DEC_HEADS * DEC_SPS * 4;
    static constexpr size_t bar_off = q_bytes + 2 * kv_bytes + sp_bytes;
    static constexpr size_t base_end = bar_off + 4 * 8 + 2 * DEC_NC * 4 + 2 * DEC_HEADS * 4 +
                                       (size_t)DEC_STAGE * 4;
    // Cluster exchange, written by the other CTAs (push) so that every read
    // after the barrier is local: the unnormalised O slices [16 ranks][16
    // heads][HD / CL] (first, in the fused step, the two histograms of the
    // row selection, [16 ranks][256] each), and (m, l) [16 ranks][2][16].
    static constexpr size_t xch_off = (base_end + 15) & ~size_t(15);
    static constexpr size_t xch_bytes =
        (size_t)DEC_HEADS * HD * 4 > 32768 ? (size_t)DEC_HEADS * HD * 4 : 32768;
    static constexpr size_t spush_off = xch_off + xch_bytes;
    static constexpr size_t total = spush_off + 16 * 2 * DEC_HEADS * 4;
    // the decode step that selects its own rows: score keys of this CTA's
    // slice, its histogram, the cluster sum, warp counts, selection, and the
    // per-slice totals pushed by the other CTAs [16][2]
    static constexpr size_t tk_off = total;
    static constexpr size_t tk_bytes = TKD_WHIST + (size_t)dec_warps<HD>() * 256 * 4;
    static_assert(2 * 4096 + 256 * 4 + 256 * 4 + 64 * 4 + 32 + 16 * 2 * 4 <= TKD_WHIST, "selection area");
    static constexpr size_t fused_total = tk_off + tk_bytes;
    static_assert(q_bytes % 16 == 0 && kv_bytes % 16 == 0 && sp_bytes % 16 == 0, "alignment");
};

// Few-token (decode) path.  A cluster of CL CTAs shares one (token, group of
// 16 heads); CTA r of the cluster takes slice r of the index row.  Rows move
// by TMA bulk copies (one per 1 KiB row) completing on mbarriers: the 16 q
// rows, then chunks of DEC_NC gathered rows, double-buffered, each warp
// copying its own share of a chunk.  The warps split the head dim for S (each
// reduces over its slice of hd); every score is then summed once over the
// partials in a fixed order, so all warps read the same scores and derive the
// same softmax statistics; for P*V each warp owns a slice of the output
// columns.  At the end each CTA pushes its (m, l) and the slices of its
// unnormalised O into the CTAs that reduce them (bulk copies into
// distributed shared memory); CTA r reduces the r-th slice of the columns
// over the cluster, adds the sink and writes o.  No scratch memory and no
// second launch.  In the fused step every CTA first ranks the scores itself (up to
// TKD_CAP of them) and keeps the picks of its own slice.  PACKED: the
// compressed rows may arrive packed (e2m1 codes + e4m3 scales) and are
// expanded in shared memory; a separate instantiation, so that the code runs
// only where packed rows are possible (the kernel's time goes largely to
// fetching its instructions: it runs once per launch on each SM).
template <int HD, bool FUSED, bool PACKED>
__global__ void __launch_bounds__(32 * dec_warps<HD>(), 1) sparse_attn_decode_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ rows_a, int64_t n_a,
    const uint16_t* __restrict__ rows_b, int64_t n_c, const int32_t* __restrict__ idx, int K,
    const float* __restrict__ sink, float scale_log2, uint16_t* __restrict__ o,
    float* __restrict__ lse, int nh, unsigned int* status, DecTopk tk, PackedRows pk) {
    namespace cg = cooperative_groups;
    using SM = DecSmem<HD>;
    constexpr int NW = dec_warps<HD>();
    constexpr int NTH = 32 * NW;
    constexpr int RS = SM::RS;
    constexpr int QW = HD / NW;      // head-dim columns per warp
    constexpr int NT = QW / 8;       // output n-tiles per warp
    constexpr uint32_t ROWB = HD * 2;  // bytes of one row
    // A packed compressed row (e2m1 codes + e4m3 block-16 scale codes) lands
    // at the tail of its padded row buffer and is expanded in place.
    constexpr uint32_t PKB = HD / 2 + HD / 16;
    constexpr uint32_t PKO = ((uint32_t)RS * 2 - PKB) & ~15u;
    static_assert(PKO + PKB <= (uint32_t)RS * 2 && PKO % 16 == 0, "packed row placement");
    const bool packed = PACKED && HD == 512 && pk.codes != nullptr;
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t* qs = reinterpret_cast<uint16_t*>(smem);
    uint16_t* kvs = reinterpret_cast<uint16_t*>(smem + SM::q_bytes);
    float* sp = reinterpret_cast<float*>(smem + SM::q_bytes + 2 * SM::kv_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::bar_off);  // q, kv0, kv1, exchange
    int* vflag = reinterpret_cast<int*>(smem + SM::bar_off + 4 * 8);
    float* stat = reinterpret_cast<float*>(vflag + 2 * DEC_NC);  // [2][16]: m then l
    int* sidx = reinterpret_cast<int*>(stat + 2 * DEC_HEADS);      // [DEC_STAGE]

    cg::cluster_group cluster = cg::this_cluster();
    const int CL = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t t = blockIdx.z;
    const int h0 = blockIdx.y * DEC_HEADS;
    const int64_t n_rows = n_a + n_c;
    const int32_t* irow = idx + t * (int64_t)K;

    // this CTA's slice of the index row
    const int per = (K + CL - 1) / CL;
    const int j0 = rank * per;
    const int j1 = min(K, j0 + per);
    const int nchunks = j1 > j0 ? (j1 - j0 + DEC_NC - 1) / DEC_NC : 0;

    // the next kernel (the following step's front) may start launching; it
    // waits for this one to complete before it touches memory
    pdl_trigger();
    if (tid == 0) {
        mbar_init(&bars[0], 1);   // q
        mbar_init(&bars[1], NW);  // kv buffer 0: one arrival a warp (load_chunk)
        mbar_init(&bars[2], NW);  // kv buffer 1
        mbar_init(&bars[3], 1);   // cluster exchange
        mbar_init_fence();
    }
    __syncthreads();
    cluster_arrive_relaxed();  // this CTA has started (waited on before any remote store)
    // q rows of this head group (rows past nh are zero); q is an input, so it
    // is read before waiting for the previous kernel.
    if (warp == 0) {
        const int hv = max(0, min(DEC_HEADS, nh - h0));
        if (lane == 0) mbar_arrive_expect_tx(&bars[0], (uint32_t)hv * ROWB);
        __syncwarp();
        if (lane < DEC_HEADS) {
            uint16_t* dst = qs + lane * RS;
            if (lane < hv) {
                bulk_g2s(dst, q + (t * nh + h0 + lane) * (int64_t)HD, ROWB, &bars[0]);
            } else {
                for (int c = 0; c < HD / 8; c++) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
            }
        }
    }
    // The rows the query can see (a 64-bit division, from the arguments
    // alone) while the kernel before finishes; the indices, the ring and the
    // cache may come from it.
    int64_t vis = 0;
    if constexpr (FUSED) {
        vis = (tk.start_pos + t + 1) / tk.ratio;
        if (vis > tk.n_c) vis = tk.n_c;
    }
    pdl_wait();
    const int nst = max(0, min(j1 - j0, DEC_STAGE));
    if constexpr (FUSED) {
        // select this query's rows here (the scores come from the kernel before)
        dec_topk<NTH>(tk, t, vis, K, j0, j1, sidx, smem + SM::tk_off, blockIdx.y == 0, status);
    } else {
        for (int j = tid; j < nst; j += NTH) sidx[j] = irow[j0 + j];
    }
    __syncthreads();
    // Every warp copies its own share of the chunk's rows, one bulk copy per
    // valid row (rows w * RPW .. w * RPW + RPW - 1 of the chunk, one a lane):
    // a warp issues its copies one after another (a microbenchmark: about
    // 40 ns apart), so spreading them over the warps lands the chunk sooner.
    // The chunk's barrier takes one arrival a warp, each carrying that warp's
    // byte count, so it cannot complete before every warp has announced its
    // bytes.  Invalid rows are zeroed (their scores are masked, and 0 * row
    // must stay finite in P*V).
    constexpr int RPW = (DEC_NC + NW - 1) / NW;  // rows per warp
    static_assert(RPW <= 32, "one row a lane");
    auto load_chunk = [&](int chunk, int buf) {
        const int r = warp * RPW + lane;
        const bool mine = lane < RPW && r < DEC_NC;
        const int j = j0 + chunk * DEC_NC + r;
        const bool in = mine && j < j1;
        int64_t v = -1;
        if (in) v = (j - j0 < nst) ? sidx[j - j0] : irow[j];
        const bool ok = v >= 0 && v < n_rows;
        if (in && (v < -1 || v >= n_rows)) raise_status(status, DS41_E_INDEX);
        const uint32_t nok = __popc(__ballot_sync(0xffffffffu, ok));
        const uint32_t npk = __popc(__ballot_sync(0xffffffffu, ok && packed && v >= n_a));
        // order this buffer's earlier generic-proxy writes before the copies
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        if (lane == 0) mbar_arrive_expect_tx(&bars[1 + buf], (nok - npk) * ROWB + npk * PKB);
        __syncwarp();
        if (!mine) return;
        uint16_t* dst = kvs + buf * (DEC_NC * RS) + r * RS;
        int flag = 0;
        if (ok) {
            if (packed && v >= n_a) {
                uint8_t* d8 = reinterpret_cast<uint8_t*>(dst) + PKO;
                bulk_g2s(d8, pk.codes + (v - n_a) * (HD / 2), HD / 2, &bars[1 + buf]);
                bulk_g2s(d8 + HD / 2, pk.scales + (v - n_a) * (HD / 16), HD / 16, &bars[1 + buf]);
                flag = 2;
            } else {
                const uint16_t* src = (v < n_a) ? rows_a + v * HD : rows_b + (v - n_a) * HD;
                bulk_g2s(dst, src, ROWB, &bars[1 + buf]);
                flag = 1;
            }
        } else {
            for (int c = 0; c < HD / 8; c++) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
        }
        vflag[buf * DEC_NC + r] = flag;
    };
    // Packed rows of a landed chunk -> bf16 in place, a warp per row: lane b
    // holds block b (16 values: 8 code bytes, one scale byte) in registers
    // before any lane writes, then writes bf16(e2m1 * scale), the exact value
    // the latent write stored in the bf16 cache.
    auto expand_chunk = [&](int buf) {
        uint16_t* kvb = kvs + buf * (DEC_NC * RS);
        for (int r = warp; r < DEC_NC; r += NW) {
            if (vflag[buf * DEC_NC + r] != 2) continue;  // the same for the whole warp
            uint8_t* row = reinterpret_cast<uint8_t*>(kvb + r * RS);
            uint2 cb[(HD / 16 + 31) / 32];
            uint32_t sb[(HD / 16 + 31) / 32];
#pragma unroll
            for (int u = 0; u < (HD / 16 + 31) / 32; u++) {
                const int b = lane + 32 * u;
                if (b < HD / 16) {
                    cb[u] = *reinterpret_cast<const uint2*>(row + PKO + 8 * b);
                    sb[u] = row[PKO + HD / 2 + b];
                }
            }
            __syncwarp();
#pragma unroll
            for (int u = 0; u < (HD / 16 + 31) / 32; u++) {
                const int b = lane + 32 * u;
                if (b >= HD / 16) continue;
                const float s = e4m3_to_f32(sb[u]);
                uint32_t w[8];
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const uint32_t byte = ((k < 4 ? cb[u].x : cb[u].y) >> (8 * (k & 3))) & 0xffu;
                    const float2 g = e2m1x2_to_float2(byte);
                    w[k] = (uint32_t)f2bf(__fmul_rn(g.x, s)) | ((uint32_t)f2bf(__fmul_rn(g.y, s)) << 16);
                }
                uint4* out = reinterpret_cast<uint4*>(row + 32 * b);
                out[0] = make_uint4(w[0], w[1], w[2], w[3]);
                out[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        // these generic writes come before later bulk copies into the buffer
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncthreads();
    };
    constexpr int NCT = DEC_NC / 8;   // n-tiles of 8 rows per chunk
    constexpr int NKS = DEC_NC / 16;  // k-steps of 16 rows per chunk in P*V

    float oacc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; j++) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.0f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.0f, 0.0f};
    const int ra = lane >> 2, rb = ra + 8;
    bool failed = false;

    if (nchunks > 0) load_chunk(0, 0);
    for (int chunk = 0; chunk < nchunks; chunk++) {
        const int buf = chunk & 1;
        if (chunk + 1 < nchunks) load_chunk(chunk + 1, buf ^ 1);
        if (chunk == 0 && !mbar_wait(&bars[0], 0, kWaitPolls)) failed = true;
        if (!mbar_wait(&bars[1 + buf], (chunk >> 1) & 1, kWaitPolls)) failed = true;
        __syncthreads();  // zero-filled rows and flags of warp 0 are visible
        if (packed) expand_chunk(buf);
        const uint16_t* kv = kvs + buf * (DEC_NC * RS);
        float sacc[NCT][4];
#pragma unroll
        for (int j = 0; j < NCT; j++) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.0f;
#pragma unroll 1
        for (int kk = 0; kk < QW / 16; kk++) {
            uint32_t a0, a1, a2, a3;
            {
                const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = warp * (QW / 8) + kk * 2 + (lane >> 4);
                ldsm_x4(smem_u32(qs + r * RS + c * 8), a0, a1, a2, a3);
            }
#pragma unroll
            for (int jj = 0; jj < NKS; jj++) {
                uint32_t b0, b1, b2, b3;
                const int r = jj * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = warp * (QW / 8) + kk * 2 + ((lane >> 3) & 1);
                ldsm_x4(smem_u32(kv + r * RS + c * 8), b0, b1, b2, b3);
                mma_bf16(sacc[2 * jj], a0, a1, a2, a3, b0, b1);
                mma_bf16(sacc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        // partial scores of the NW slices of hd, one block a warp
        float* mine = sp + warp * (DEC_HEADS * DEC_SPS);
#pragma unroll
        for (int j = 0; j < NCT; j++) {
            const int col = j * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2*>(mine + ra * DEC_SPS + col) = make_float2(sacc[j][0], sacc[j][1]);
            *reinterpret_cast<float2*>(mine + rb * DEC_SPS + col) = make_float2(sacc[j][2], sacc[j][3]);
        }
        __syncthreads();
        // every score summed once over the warps' partials, in the warps'
        // order, then scaled (or masked) in place of warp 0's block; every
        // warp then reads the same final scores (each warp summing all the
        // partials itself read eight times the bytes)
        for (int e = tid; e < DEC_HEADS * DEC_NC; e += NTH) {
            const int h = e / DEC_NC, c = e - h * DEC_NC;
            float x = sp[h * DEC_SPS + c];
#pragma unroll
            for (int w = 1; w < NW; w++) x += sp[w * DEC_HEADS * DEC_SPS + h * DEC_SPS + c];
            sp[h * DEC_SPS + c] = vflag[buf * DEC_NC + c] != 0 ? x * scale_log2 : -INFINITY;
        }
        __syncthreads();
        float sv[NCT][4];
#pragma unroll
        for (int j = 0; j < NCT; j++) {
            const int col = j * 8 + 2 * (lane & 3);
            const float2 xa = *reinterpret_cast<const float2*>(sp + ra * DEC_SPS + col);
            const float2 xb = *reinterpret_cast<const float2*>(sp + rb * DEC_SPS + col);
            sv[j][0] = xa.x;
            sv[j][1] = xa.y;
            sv[j][2] = xb.x;
            sv[j][3] = xb.y;
        }
        float mx[2] = {mrow[0], mrow[1]};
#pragma unroll
        for (int j = 0; j < NCT; j++) {
            mx[0] = fmaxf(mx[0], fmaxf(sv[j][0], sv[j][1]));
            mx[1] = fmaxf(mx[1], fmaxf(sv[j][2], sv[j][3]));
        }
#pragma unroll
        for (int i = 0; i < 2; i++) {
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
            mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
        }
        float corr[2], muse[2];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            muse[i] = (mx[i] == -INFINITY) ? 0.0f : mx[i];
            corr[i] = exp2f(mrow[i] - muse[i]);
            mrow[i] = mx[i];
            lrow[i] *= corr[i];
        }
        uint32_t pa[NKS][4];
#pragma unroll
        for (int j = 0; j < NCT; j++) {
            const float p0 = exp2f(sv[j][0] - muse[0]), p1 = exp2f(sv[j][1] - muse[0]);
            const float p2 = exp2f(sv[j][2] - muse[1]), p3 = exp2f(sv[j][3] - muse[1]);
            lrow[0] += p0 + p1;
            lrow[1] += p2 + p3;
            pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
            pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
        }
#pragma unroll
        for (int j = 0; j < NT; j++) {
            oacc[j][0] *= corr[0];
            oacc[j][1] *= corr[0];
            oacc[j][2] *= corr[1];
            oacc[j][3] *= corr[1];
        }
#pragma unroll
        for (int ks = 0; ks < NKS; ks++) {
#pragma unroll
            for (int jj = 0; jj < NT / 2; jj++) {
                uint32_t b0, b1, b2, b3;
                const int r = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = warp * (QW / 8) + jj * 2 + (lane >> 4);
                ldsm_x4_t(smem_u32(kv + r * RS + c * 8), b0, b1, b2, b3);
                mma_bf16(oacc[2 * jj], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
                mma_bf16(oacc[2 * jj + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
            }
        }
        __syncthreads();  // this buffer is refilled two chunks later
    }
    if (failed) {
        // a copy never completed (only a broken index or address could do
        // this): report it and leave this CTA's contribution empty
        raise_status(status, DS41_E_TIMEOUT);
        mrow[0] = mrow[1] = -INFINITY;
        lrow[0] = lrow[1] = 0.0f;
#pragma unroll
        for (int j = 0; j < NT; j++) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.0f;
    }
    if (nchunks == 0 && !mbar_wait(&bars[0], 0, kWaitPolls)) raise_status(status, DS41_E_TIMEOUT);

#pragma unroll
    for (int i = 0; i < 2; i++) {
        lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 1);
        lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 2);
    }
    // Push this CTA's (m, l) into every CTA of the cluster and each slice of
    // its unnormalised O, as bf16 pairs (half the exchanged bytes; the same
    // relative rounding as the bf16 output), into the CTA that reduces those
    // columns; every read afterwards is local.  Both are staged in this CTA's
    // shared memory first ((m, l) in stat, the O slices in sp, laid out as the
    // receivers' blocks) and moved by bulk copies, two per receiver, that
    // complete on the receiver's exchange barrier: each CTA waits only for the
    // bytes it receives.  A sender cannot see when its copies have read the
    // staging, so sp and stat stay untouched until the closing cluster barrier,
    // which every CTA passes only once all copies have landed.
    const int cols = HD / CL;
    float* spush = reinterpret_cast<float*>(smem + SM::spush_off);    // [16 ranks][2][16]
    uint32_t* opush = reinterpret_cast<uint32_t*>(smem + SM::xch_off);  // [CL ranks][16][cols/2]
    uint32_t* ostage = reinterpret_cast<uint32_t*>(sp);                 // [CL][16][cols/2]
    static_assert((size_t)DEC_HEADS * HD * 2 <= SM::sp_bytes && (SM::bar_off + 32 + 2 * DEC_NC * 4) % 16 == 0,
                  "O staging; (m, l) staging moved as 16-byte multiples");
    if (warp == 0 && (lane & 3) == 0) {
        stat[ra] = mrow[0];
        stat[rb] = mrow[1];
        stat[DEC_HEADS + ra] = lrow[0];
        stat[DEC_HEADS + rb] = lrow[1];
    }
#pragma unroll
    for (int j = 0; j < NT; j++) {
        const int col = warp * QW + j * 8 + 2 * (lane & 3);
        const int qo = col / cols, cc = (col - qo * cols) >> 1;
        uint32_t* dst = ostage + qo * DEC_HEADS * (cols / 2);
        dst[ra * (cols / 2) + cc] = pack_bf16x2(oacc[j][0], oacc[j][1]);
        dst[rb * (cols / 2) + cc] = pack_bf16x2(oacc[j][2], oacc[j][3]);
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // staged bytes, for the copies
    __syncthreads();
    cluster_wait();  // every CTA of the cluster has started: its exchange barrier is initialised
    if (tid == 0) {
        const uint32_t oblk = (uint32_t)DEC_HEADS * (cols / 2) * 4;  // one receiver's O block
        const uint32_t mlb = 2 * DEC_HEADS * 4;                      // (m, l) of one sender
        mbar_arrive_expect_tx(&bars[3], (uint32_t)CL * (oblk + mlb));
        for (int qd = 0; qd < CL; qd++) {
            const uint32_t rbar = cluster_addr(&bars[3], qd);
            bulk_s2cluster(cluster_addr(opush, qd) + (uint32_t)rank * oblk, ostage + qd * (oblk / 4),
                           oblk, rbar);
            bulk_s2cluster(cluster_addr(spush, qd) + (uint32_t)rank * mlb, stat, mlb, rbar);
        }
    }
    if (!mbar_wait(&bars[3], 0, kWaitPolls)) raise_status(status, DS41_E_TIMEOUT);
    cluster_arrive_relaxed();  // every block this CTA receives has landed

    // Weights e^{m_r - M} / L for every (head, rank): one thread per pair,
    // the max and the sum over the ranks by shuffles within 16-lane groups.
    float* wts = reinterpret_cast<float*>(kvs);  // [16 ranks][16 heads]; the row buffers are idle now
    for (int pidx = tid; pidx < DEC_HEADS * 16; pidx += NTH) {
        const int hh = pidx >> 4, r = pidx & 15;
        const int h = h0 + hh;
        float mr = -INFINITY, lr = 0.0f;
        if (r < CL) {
            mr = spush[r * 2 * DEC_HEADS + hh];
            lr = spush[r * 2 * DEC_HEADS + DEC_HEADS + hh];
        }
        const float sk = (h < nh) ? sink[h] * LOG2E : -INFINITY;
        float M = fmaxf(mr, sk);
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float Mref = (M == -INFINITY) ? 0.0f : M;
        const float e = exp2f(mr - Mref);
        float L = lr * e;
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        L += exp2f(sk - Mref);
        const float inv = (L > 0.0f) ? 1.0f / L : 0.0f;
        wts[r * DEC_HEADS + hh] = e * inv;
        if (lse && rank == 0 && r == 0 && h < nh) lse[t * nh + h] = (Mref + log2f(L)) / LOG2E;
    }
    __syncthreads();
    // CTA `rank` reduces columns [c0, c0 + cols) of the 16 heads, 4 at a time.
    const int c0 = rank * cols;
    for (int e = tid; e < DEC_HEADS * (cols / 4); e += NTH) {
        const int hh = e / (cols / 4), cl4 = 4 * (e % (cols / 4));
        const int h = h0 + hh;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int r = 0; r < 16; r++) {
            if (r < CL) {
                const uint2 u = *reinterpret_cast<const uint2*>(opush + (r * DEC_HEADS + hh) * (cols / 2) + cl4 / 2);
                const float4 v = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                                             __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
                const float wgt = wts[r * DEC_HEADS + hh];
                acc.x += v.x * wgt;
                acc.y += v.y * wgt;
                acc.z += v.z * wgt;
                acc.w += v.w * wgt;
            }
        }
        if (h < nh) {
            const uint2 packed = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
            *reinterpret_cast<uint2*>(o + (t * nh + h) * (int64_t)HD + c0 + cl4) = packed;
        }
    }
    // no CTA leaves while a copy into or out of its shared memory may be in
    // flight: each has arrived once its own blocks landed
    cluster_wait();
}

struct AttnPlan {
    int splits, chunks_per_split, head_groups;
    int cluster;  // > 0: the few-token path with this many CTAs per cluster
    int tc;       // > 0: the tensor-core path on this many SMs
    size_t part_o_bytes, part_ml_bytes;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static AttnPlan plan_attn(int64_t m, int64_t nh, int64_t hd, int64_t K, int sms) {
    AttnPlan p;
    p.cluster = 0;
    p.tc = 0;
    // Few tokens: one cluster per (token, 16 heads) when that leaves most SMs
    // to the row slices; no scratch, no merge launch.
    const int64_t dec_groups = m * ((nh + DEC_HEADS - 1) / DEC_HEADS);
    if (dec_groups * 4 <= sms) {
        int cl = 16;
        while (cl > 1 && (dec_groups * cl > 2 * sms || (K + cl - 1) / cl < 8)) cl >>= 1;
        p.cluster = cl;
        p.splits = 1;
        p.chunks_per_split = 0;
        p.head_groups = (int)((nh + DEC_HEADS - 1) / DEC_HEADS);
        p.part_o_bytes = p.part_ml_bytes = 0;
        return p;
    }
    p.head_groups = (int)((nh + ATT_HEADS - 1) / ATT_HEADS);
    // Many tokens, hd 512, whole 64-head groups: persistent tcgen05 kernel.
    if (attn_tc_supported(m, nh, hd, K, sms)) {
        p.tc = sms;
        p.splits = 1;
        p.chunks_per_split = 0;
        p.part_o_bytes = p.part_ml_bytes = 0;
        return p;
    }
    const int chunks = (int)((K + ATT_NC - 1) / ATT_NC);
    const int64_t ctas = m * p.head_groups;
    int splits = 1;
    if (ctas < sms) {
        splits = (int)((sms + ctas - 1) / ctas);
        if (splits > chunks) splits = chunks;
    }
    p.chunks_per_split = (chunks + splits - 1) / splits;
    p.splits = (chunks + p.chunks_per_split - 1) / p.chunks_per_split;
    if (p.splits > 1) {
        p.part_o_bytes = align256((size_t)m * p.splits * nh * hd * 4);
        p.part_ml_bytes = align256((size_t)m * p.splits * nh * 8);
    } else {
        p.part_o_bytes = p.part_ml_bytes = 0;
    }
    return p;
}

static int device_sms() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

template <int HD>
static int launch_attn_decode(const AttnPlan& p, const uint16_t* q, const uint16_t* rows_a,
                              int64_t n_a, const uint16_t* rows_b, int64_t n_c,
                              const int32_t* idx, int64_t K, const float* sink, float scale,
                              uint16_t* o, float* lse, int64_t m, int64_t nh,
                              unsigned int* status, cudaStream_t st, bool pdl,
                              const DecTopk* tk = nullptr, const PackedRows* pk = nullptr) {
    const size_t smem = tk ? DecSmem<HD>::fused_total : DecSmem<HD>::total;
    auto kern = tk ? sparse_attn_decode_kernel<HD, true, false>
                   : sparse_attn_decode_kernel<HD, false, false>;
    const bool packed = pk && HD == 512 && pk->codes != nullptr;
    if constexpr (HD == 512) {
        if (packed)
            kern = tk ? sparse_attn_decode_kernel<HD, true, true>
                      : sparse_attn_decode_kernel<HD, false, true>;
    }
    const DecTopk tkv = tk ? *tk : DecTopk{};
    const PackedRows pkv = packed ? *pk : PackedRows{nullptr, nullptr};
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (p.cluster > 8) cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.cluster, (unsigned)p.head_groups, (unsigned)m);
    cfg.blockDim = dim3(32 * dec_warps<HD>());  // NOLINT
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    int rc = cuda_check(cudaLaunchKernelEx(&cfg, kern, q, rows_a, n_a, rows_b, n_c, idx, (int)K,
                                           sink, scale * LOG2E, o, lse, (int)nh, status, tkv,
                                           pkv),
                        "ds41_sparse_attn_sink_fwd: decode kernel");
    if (rc) return rc;
    return launch_check("ds41_sparse_attn_sink_fwd: decode kernel");
}

template <int HD>
static int launch_attn(const AttnPlan& p, const uint16_t* q, const uint16_t* rows_a, int64_t n_a,
                       const uint16_t* rows_b, int64_t n_c, const int32_t* idx, int64_t K,
                       const float* sink, float scale, uint16_t* o, float* lse, int64_t m,
                       int64_t nh, uint8_t* ws, unsigned int* status, cudaStream_t st,
                       bool pdl = false, const DecTopk* tk = nullptr,
                       const PackedRows* pk = nullptr) {
    if (p.cluster > 0)
        return launch_attn_decode<HD>(p, q, rows_a, n_a, rows_b, n_c, idx, K, sink, scale, o, lse,
                                      m, nh, status, st, pdl, tk, pk);
    if constexpr (HD == 512) {
        if (p.tc > 0)
            return attn_tc_launch(q, rows_a, n_a, rows_b, n_c, idx, K, sink, scale, o, lse, m, nh,
                                  status, p.tc, st);
    }
    const size_t smem = AttnSmem<HD>::total;
    // with tk (one split only, see attn_topk_fusable) the kernel selects the
    // rows itself and writes the index rows to tk->idx_out
    auto kern = tk ? sparse_attn_kernel<HD, true> : sparse_attn_kernel<HD, false>;
    const DecTopk tkv = tk ? *tk : DecTopk{};
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    float* part_o = p.splits > 1 ? reinterpret_cast<float*>(ws) : nullptr;
    float2* part_ml = p.splits > 1 ? reinterpret_cast<float2*>(ws + p.part_o_bytes) : nullptr;
    dim3 grid((unsigned)m, (unsigned)p.splits, (unsigned)p.head_groups);
    int rc = launch_pdl(kern, grid, dim3(ATT_THREADS), smem, st,
                        "ds41_sparse_attn_sink_fwd: attention kernel", q, rows_a, n_a, rows_b, n_c,
                        idx, (int)K, sink, scale * LOG2E, o, lse, (int)nh, p.chunks_per_split,
                        part_o, part_ml, status, tkv);
    if (rc || p.splits == 1) return rc;
    return launch_pdl(attn_merge_kernel<HD>, dim3((unsigned)m, (unsigned)nh), dim3(128), 0, st,
                      "ds41_sparse_attn_sink_fwd: merge kernel", (const float*)part_o,
                      (const float2*)part_ml, sink, o, lse, (int)nh, p.splits);
}

}  // namespace ds41

using namespace ds41;

extern "C" size_t ds41_sparse_attn_workspace_bytes(int64_t m, int64_t nh, int64_t hd, int64_t K) {
    if (m < 1 || nh < 1 || hd < 1 || K < 1) return 0;
    AttnPlan p = plan_attn(m, nh, hd, K, device_sms());
    return p.part_o_bytes + p.part_ml_bytes;
}

extern "C" int ds41_sparse_attn_sink_fwd(const ds41_bf16* q, const ds41_bf16* rows_a,
                                         int64_t n_a, const ds41_bf16* rows_b, int64_t n_c,
                                         const int32_t* idx, int64_t K, const float* sink,
                                         float scale, ds41_bf16* o, float* lse, int64_t m,
                                         int64_t nh, int64_t hd, void* ws, size_t ws_bytes,
                                         ds41_stream_t stream) {
    const char* name = "ds41_sparse_attn_sink_fwd";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 31), DS41_E_RANGE, "%s: m=%lld", name,
                 (long long)m);
    DS41_REQUIRE(nh >= 1 && nh <= 65535 * ATT_HEADS, DS41_E_ARG, "%s: nh=%lld", name,
                 (long long)nh);
    DS41_REQUIRE(hd == 64 || hd == 128 || hd == 256 || hd == 512, DS41_E_ARG,
                 "%s: hd=%lld must be 64, 128, 256 or 512", name, (long long)hd);
    DS41_REQUIRE(K >= 1 && K < (int64_t(1) << 30), DS41_E_ARG, "%s: K=%lld", name, (long long)K);
    DS41_REQUIRE(n_a >= 0 && n_c >= 0 && n_a + n_c >= 1, DS41_E_ARG, "%s: n_a=%lld n_c=%lld",
                 name, (long long)n_a, (long long)n_c);
    DS41_REQUIRE(q && idx && sink && o && (n_a == 0 || rows_a) && (n_c == 0 || rows_b),
                 DS41_E_ARG, "%s: null tensor pointer", name);
    DS41_REQUIRE(aligned16(q) && aligned16(o) && (n_a == 0 || aligned16(rows_a)) &&
                     (n_c == 0 || aligned16(rows_b)),
                 DS41_E_ARG, "%s: q/o/rows must be 16-byte aligned", name);
    unsigned int* status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    AttnPlan p = plan_attn(m, nh, hd, K, device_sms());
    const size_t need = p.part_o_bytes + p.part_ml_bytes;
    DS41_REQUIRE(need == 0 || (ws && ws_bytes >= need), DS41_E_WORKSPACE,
                 "%s: workspace of %zu bytes needed, %zu given", name, need, ws ? ws_bytes : 0);
    DS41_REQUIRE(need == 0 || aligned16(ws), DS41_E_ARG, "%s: ws must be 16-byte aligned", name);
    const uint16_t* ra = n_a ? rows_a : rows_b;
    const uint16_t* rb = n_c ? rows_b : rows_a;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    switch (hd) {
        case 64: return launch_attn<64>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, wsb, status, st);
        case 128: return launch_attn<128>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, wsb, status, st);
        case 256: return launch_attn<256>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, wsb, status, st);
        default: return launch_attn<512>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, wsb, status, st);
    }
}

// ---------------------------------------------------------------------------
// Internal entry for the fused step (ds41_forward.cu): arguments already
// checked by the caller.
// ---------------------------------------------------------------------------
namespace ds41 {

size_t attn_ws_bytes(int64_t m, int64_t nh, int64_t hd, int64_t K) {
    if (m < 1 || nh < 1 || hd < 1 || K < 1) return 0;
    AttnPlan p = plan_attn(m, nh, hd, K, device_sms());
    return p.part_o_bytes + p.part_ml_bytes;
}

int attn_run(const uint16_t* q, const uint16_t* rows_a, int64_t n_a, const uint16_t* rows_b,
             int64_t n_c, const int32_t* idx, int64_t K, const float* sink, float scale,
             uint16_t* o, float* lse, int64_t m, int64_t nh, int64_t hd, uint8_t* ws,
             size_t ws_bytes, bool pdl, cudaStream_t st, const char* name, const DecTopk* tk,
             const PackedRows* pk) {
    unsigned int* status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    AttnPlan p = plan_attn(m, nh, hd, K, device_sms());
    const size_t need = p.part_o_bytes + p.part_ml_bytes;
    DS41_REQUIRE(need == 0 || (ws && ws_bytes >= need), DS41_E_WORKSPACE,
                 "%s: workspace of %zu bytes needed, %zu given", name, need, ws ? ws_bytes : 0);
    const uint16_t* ra = n_a ? rows_a : rows_b;
    const uint16_t* rb = n_c ? rows_b : rows_a;
    switch (hd) {
        case 64: return launch_attn<64>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, ws, status, st, pdl, tk);
        case 128: return launch_attn<128>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, ws, status, st, pdl, tk);
        case 256: return launch_attn<256>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, ws, status, st, pdl, tk);
        default: return launch_attn<512>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, ws, status, st, pdl, tk, pk);
    }
}

bool attn_is_cluster_path(int64_t m, int64_t nh, int64_t hd, int64_t K) {
    return plan_attn(m, nh, hd, K, device_sms()).cluster > 0;
}

bool attn_topk_fusable(int64_t m, int64_t nh, int64_t hd, int64_t K, int64_t n_c) {
    const int sms = device_sms();
    const AttnPlan p = plan_attn(m, nh, hd, K, sms);
    if (p.cluster >= 4) {
        const int64_t per = (K + p.cluster - 1) / p.cluster;
        return per <= DEC_STAGE && n_c <= TKD_CAP;
    }
    // the generic kernel in one wave of CTAs, one split each: every CTA ranks
    // its token's scores with one warp (SEL)
    return p.cluster == 0 && p.tc == 0 && p.splits == 1 && m * p.head_groups <= sms &&
           K <= ATT_STAGE && n_c <= WTK_MAX;
}

}  // namespace ds41

// ---------------------------------------------------------------------------
// The same attention for callers that cannot allocate device memory.  The
// split partials live in one file-scope device array instead of a
// caller-provided workspace.
// ---------------------------------------------------------------------------
namespace ds41 {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static constexpr int kNoAllocMaxDevices = 64;
static uint8_t* g_noalloc_ptr[kNoAllocMaxDevices];
static std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device.  The array's
// name is only a host-side stand-in in host code, so its address is looked
// up once per device, with that device current, and cached.
static int noalloc_scratch(uint8_t** out) {
    int dev = 0;
    int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (rc) return rc;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(DS41_E_CUDA, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        rc = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                        "cudaGetSymbolAddress(no-alloc scratch)");
        if (rc) return rc;
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return DS41_OK;
}

}  // namespace ds41

extern "C" size_t ds41_sparse_attn_noalloc_capacity(void) { return ds41::kNoAllocScratchBytes; }

extern "C" int ds41_sparse_attn_sink_fwd_noalloc(const ds41_bf16* q, const ds41_bf16* rows_a,
                                                 int64_t n_a, const ds41_bf16* rows_b,
                                                 int64_t n_c, const int32_t* idx, int64_t K,
                                                 const float* sink, float scale, ds41_bf16* o,
                                                 float* lse, int64_t m, int64_t nh, int64_t hd,
                                                 ds41_stream_t stream) {
    const char* name = "ds41_sparse_attn_sink_fwd_noalloc";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 31), DS41_E_RANGE, "%s: m=%lld", name,
                 (long long)m);
    DS41_REQUIRE(nh >= 1 && nh <= 65535 * ATT_HEADS, DS41_E_ARG, "%s: nh=%lld", name,
                 (long long)nh);
    DS41_REQUIRE(hd == 64 || hd == 128 || hd == 256 || hd == 512, DS41_E_ARG,
                 "%s: hd=%lld must be 64, 128, 256 or 512", name, (long long)hd);
    DS41_REQUIRE(K >= 1 && K < (int64_t(1) << 30), DS41_E_ARG, "%s: K=%lld", name, (long long)K);
    DS41_REQUIRE(n_a >= 0 && n_c >= 0 && n_a + n_c >= 1, DS41_E_ARG, "%s: n_a=%lld n_c=%lld",
                 name, (long long)n_a, (long long)n_c);
    DS41_REQUIRE(q && idx && sink && o && (n_a == 0 || rows_a) && (n_c == 0 || rows_b),
                 DS41_E_ARG, "%s: null tensor pointer", name);
    DS41_REQUIRE(aligned16(q) && aligned16(o) && (n_a == 0 || aligned16(rows_a)) &&
                     (n_c == 0 || aligned16(rows_b)),
                 DS41_E_ARG, "%s: q/o/rows must be 16-byte aligned", name);
    AttnPlan p = plan_attn(m, nh, hd, K, device_sms());
    const size_t need = p.part_o_bytes + p.part_ml_bytes;
    DS41_REQUIRE(need <= kNoAllocScratchBytes, DS41_E_WORKSPACE,
                 "%s: these sizes need %zu bytes of scratch, more than the %zu bytes of the "
                 "static scratch array; use ds41_sparse_attn_sink_fwd with a workspace",
                 name, need, kNoAllocScratchBytes);
    unsigned int* status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    uint8_t* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    const uint16_t* ra = n_a ? rows_a : rows_b;
    const uint16_t* rb = n_c ? rows_b : rows_a;
    cudaStream_t st = (cudaStream_t)stream;
    switch (hd) {
        case 64: return launch_attn<64>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, scratch, status, st);
        case 128: return launch_attn<128>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, scratch, status, st);
        case 256: return launch_attn<256>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, scratch, status, st);
        default: return launch_attn<512>(p, q, ra, n_a, rb, n_c, idx, K, sink, scale, o, lse, m, nh, scratch, status, st);
    }
}
