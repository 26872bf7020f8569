// ds41_indexer.cu - step 2 of the forward: fp4 indexer scores, per-query
// top-k, and the merge of window and compressed indices.
//
// metrale_model_arch/attn_v41/forward.rs calls the indexer (its body is not
// on the pages) and merges [window indices | indexer picks] per token; the
// header of metrale_model_arch/deepseek_v41_ref/compress.rs fixes the indexer
// precision: q and k take the e2m1 round trip with power-of-two scales per
// block of 32 (fp4_quant_e8m0_inplace) and the scores are bf16 values.
//
// Score of query t against compressed row s (s < (start_pos + t + 1)/ratio):
//   acc = 0; for h in 0..Hi-1: acc = fma(w[t,h], max(<qh[t,h], kh[s]>, 0), acc)
//   score = bf16(acc)
// The dot products of fp4 values are exact in f32 for inputs whose block
// scales stay within a moderate range, so the tensor-core sum equals the
// ordered sum bit for bit; the head sum is an explicit fma chain in head
// order, identical on every architecture.
#include <cooperative_groups.h>

#include "ds41_internal.cuh"
#include "ds41_step1.cuh"
#include "ds41_topk.cuh"

namespace ds41 {

constexpr int IDX_ROWS = 64;     // compressed rows per tile (16 per warp)
constexpr int IDX_N = 128;       // (token, head) columns per CTA
constexpr int IDX_THREADS = 256;

template <int CPR>
__device__ __forceinline__ int swz(int n, int c) {
    if (CPR >= 8) return c ^ (n & 7);
    if (CPR == 4) return c ^ ((n >> 1) & 3);
    return c;
}

// Quantise 8 consecutive values held by this lane; BLOCK/8 = 4 neighbouring
// lanes hold one block of 32.  Returns the bf16 round-trip values packed.
__device__ __forceinline__ uint4 q8_chunk(uint4 raw, bool live) {
    const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
    float v[8];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        v[k] = live ? bf2f(h[k]) : 0.0f;
        amax = fmaxf(amax, fabsf(v[k]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __uint_as_float(0x01c00000u));  // 6 * 2^-126
    float rs;
    const float s = e8m0_scale_bf16(amax, &rs);  // amax: a bf16 magnitude or the floor
#pragma unroll
    for (int k = 0; k < 8; k++) v[k] = __fmul_rn(v[k], rs);
    uint32_t codes;
    return e2m1_round8(v, s, &codes);
}

__device__ __forceinline__ int64_t visible_rows(int64_t t, int64_t start_pos, int64_t ratio,
                                                int64_t n_c) {
    const int64_t v = (start_pos + t + 1) / ratio;
    return v < n_c ? v : n_c;
}

// Grid: x = token groups of TT tokens, y = row-tile splits.  Each CTA
// quantises the q of its tokens once into shared memory, then walks its row
// tiles: k tile -> shared (quantised on the fly, or copied when kq holds the
// pre-quantised keys), 4 warps x 16 rows x 128 columns of bf16 MMA, the
// accumulator through shared memory, then one thread per (row, token) runs the
// ordered head chain and writes the bf16 score.  NARROW: at most IDX_N / 2
// live (token, head) columns (one token of 64 heads), so the eight warps split
// those instead of computing on padding.
template <int DI, bool KQ_INLINE, bool NARROW>
__global__ void __launch_bounds__(IDX_THREADS) indexer_scores_kernel(
    const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_src,
    const float* __restrict__ w, uint16_t* __restrict__ scores, int m, int Hi, int hpad, int TT,
    int64_t n_c, int64_t ratio, int64_t start_pos, bool fill_hidden, int ymain, int nkb,
    RingArgs ring, LatentArgs lat) {
    constexpr int CPR = DI / 8;  // 16-byte chunks per row
    // q rows and score columns held: the narrow form holds only the live half
    constexpr int QN = NARROW ? IDX_N / 2 : IDX_N;
    // Every input (and the ring and cache this kernel writes) may belong to the
    // kernel before, e.g. the previous step's attention reading the ring: this
    // kernel is launched with programmatic stream serialization, so it waits
    // for that kernel here, before its first memory access, and only its
    // launch overlaps it.  Only then may the next kernel start launching: the
    // decode attention reads q (an input of the step) before its own wait, so
    // everything before this kernel must be complete when it launches.
    // The rows each token of the group can see (one 64-bit division per
    // token, from the arguments alone) are worked out while it waits.
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * TT;
    const int tcount = min(TT, m - t0);
    __shared__ int64_t vis_s[IDX_N];
    for (int tt = tid; tt < tcount; tt += IDX_THREADS)
        vis_s[tt] = visible_rows(t0 + tt, start_pos, ratio, n_c);
    const int64_t vis_last = visible_rows(t0 + tcount - 1, start_pos, ratio, n_c);
    pdl_wait();
    pdl_trigger();
    if ((int)blockIdx.y >= ymain) {
        // Fused front of a few-token step: the CTAs past the score grid do
        // step 1 (ring write + window indices, then the latent groups).
        const int side = (int)(blockIdx.y - ymain) * gridDim.x + blockIdx.x;
        const int nside = (int)(gridDim.y - ymain) * gridDim.x;
        if (side == 0) ring_write_cta(ring);
        const int hd8 = lat.hd / 8;
        for (int g = side; g < lat.G; g += nside)
            for (int k0 = 0; k0 < hd8; k0 += IDX_THREADS) latent_write_item(lat, g, k0 + threadIdx.x);
        return;
    }
    extern __shared__ __align__(128) uint8_t smem[];
    // nkb key buffers: 2, or 1 when every CTA takes at most one tile (the
    // host launches a CTA per tile then, so more CTAs fit an SM)
    uint16_t* qs = reinterpret_cast<uint16_t*>(smem);                 // [QN][DI]
    uint16_t* ksb = qs + QN * DI;                                      // nkb x [IDX_ROWS][DI]
    float* cs = reinterpret_cast<float*>(ksb + nkb * IDX_ROWS * DI);  // [IDX_ROWS][QN + 1]
    float* wsm = cs + IDX_ROWS * (QN + 1);                             // [QN]


    // q of this CTA's tokens as rows n = tt * hpad + h: staged raw with
    // cp.async (padding rows zero-filled), then quantised in place.  The
    // quantisation loop stays rolled: a decode call runs this code once per
    // SM, so compact code (fewer instruction-cache misses) beats unrolling.
    for (int id = tid; id < QN * CPR; id += IDX_THREADS) {
        const int n = id / CPR, c = id % CPR;
        const int tt = n / hpad, h = n % hpad;
        const bool live = tt < tcount && h < Hi;
        const uint16_t* src = q_idx + ((int64_t)(t0 + (live ? tt : 0)) * Hi + (live ? h : 0)) * DI;
        cp_async16(smem_u32(qs + n * DI + swz<CPR>(n, c) * 8), src + c * 8, live);
    }
    const int64_t tiles_vis = (vis_last + IDX_ROWS - 1) / IDX_ROWS;
    // When the scores are a caller-visible output, rows no query of this
    // group can see yet are written as -inf too.
    const int64_t tiles = fill_hidden ? (n_c + IDX_ROWS - 1) / IDX_ROWS : tiles_vis;
    cp_async_commit();  // group of q
    // Key tiles go through two buffers: the CTA's first two tiles are fetched
    // together with q, so the three loads overlap (a decode CTA takes one or
    // two tiles), and q is quantised while they are in flight; each later
    // tile is fetched as soon as the tile two before it is done.
    auto fetch_k = [&](int64_t tile, uint16_t* ks) {
        const int64_t r0 = tile * IDX_ROWS;
        for (int id = tid; id < IDX_ROWS * CPR; id += IDX_THREADS) {
            const int r = id / CPR, c = id % CPR;
            const int64_t row = r0 + r;
            const bool live = row < n_c;
            cp_async16(smem_u32(ks + r * DI + swz<CPR>(r, c) * 8),
                       k_src + (live ? row : 0) * DI + c * 8, live);
        }
    };
    for (int b = 0; b < 2; b++) {
        const int64_t tile = (int64_t)blockIdx.y + (int64_t)b * ymain;
        if (b < nkb && tile < tiles_vis) fetch_k(tile, ksb + b * IDX_ROWS * DI);
        cp_async_commit();  // one group per buffer (empty when there is no such tile)
    }
    for (int n = tid; n < QN; n += IDX_THREADS) {
        const int tt = n / hpad, h = n % hpad;
        wsm[n] = (tt < tcount && h < Hi) ? w[(int64_t)(t0 + tt) * Hi + h] : 0.0f;
    }
    cp_async_wait<2>();  // this thread's q copies have landed
    __syncthreads();
    // only the live rows (tokens of the group x Hi heads), rounded up to whole
    // passes of the block: q8_chunk shuffles over the full warp, and the
    // padding rows past the live ones are zero (they stay zero)
    const int live_rows = (tcount - 1) * hpad + Hi;
    const int q_iters = min(QN * CPR,
                            (live_rows * CPR + IDX_THREADS - 1) / IDX_THREADS * IDX_THREADS);
#pragma unroll 1
    for (int id = tid; id < q_iters; id += IDX_THREADS) {
        const int n = id / CPR, c = id % CPR;
        uint4* p = reinterpret_cast<uint4*>(qs + n * DI + swz<CPR>(n, c) * 8);
        *p = q8_chunk(*p, true);
    }

    int it = 0;  // this CTA's visible tiles so far: tile it uses buffer it & 1
    for (int64_t tile = blockIdx.y; tile < tiles; tile += ymain) {
        const int64_t r0 = tile * IDX_ROWS;
        if (tile >= tiles_vis) {
            for (int p = tid; p < IDX_ROWS * tcount; p += IDX_THREADS) {
                const int tt = p / IDX_ROWS, r = p % IDX_ROWS;
                if (r0 + r < n_c) scores[(int64_t)(t0 + tt) * n_c + r0 + r] = 0xff80u;
            }
            continue;
        }
        if (it >= nkb && nkb == 1) break;  // one buffer: one tile a CTA (the host plan)
        uint16_t* ks = ksb + (it & 1) * IDX_ROWS * DI;
        cp_async_wait<1>();  // this thread's copies of this tile (the next may be in flight)
        __syncthreads();     // everyone's copies; previous tile's readers are done with cs
        if (KQ_INLINE) {
            // raw keys -> fp4 round trip, in place (rows past n_c are zero)
#pragma unroll 1
            for (int id = tid; id < IDX_ROWS * CPR; id += IDX_THREADS) {
                const int r = id / CPR, c = id % CPR;
                uint4* p = reinterpret_cast<uint4*>(ks + r * DI + swz<CPR>(r, c) * 8);
                *p = q8_chunk(*p, true);
            }
            __syncthreads();
        }

        // 8 warps: warp w owns rows 16*(w%4).. and columns WN*(w/4)..
        constexpr int WN = NARROW ? IDX_N / 4 : IDX_N / 2;  // columns per warp
        const int wr = (warp & 3) * 16, wc = (warp >> 2) * WN;
        float acc[WN / 8][4];
#pragma unroll
        for (int j = 0; j < WN / 8; j++)
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
#pragma unroll 1
        for (int kk = 0; kk < DI / 16; kk++) {
            uint32_t a0, a1, a2, a3;
            {
                const int r = wr + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = kk * 2 + (lane >> 4);
                ldsm_x4(smem_u32(ks + r * DI + swz<CPR>(r, c) * 8), a0, a1, a2, a3);
            }
#pragma unroll
            for (int jj = 0; jj < WN / 16; jj++) {
                uint32_t b0, b1, b2, b3;
                const int n = wc + jj * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = kk * 2 + ((lane >> 3) & 1);
                ldsm_x4(smem_u32(qs + n * DI + swz<CPR>(n, c) * 8), b0, b1, b2, b3);
                mma_bf16(acc[2 * jj], a0, a1, a2, a3, b0, b1);
                mma_bf16(acc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
            }
        }
#pragma unroll
        for (int j = 0; j < WN / 8; j++) {
            const int r = wr + (lane >> 2);
            const int col = wc + j * 8 + 2 * (lane & 3);
            cs[r * (QN + 1) + col] = acc[j][0];
            cs[r * (QN + 1) + col + 1] = acc[j][1];
            cs[(r + 8) * (QN + 1) + col] = acc[j][2];
            cs[(r + 8) * (QN + 1) + col + 1] = acc[j][3];
        }
        __syncthreads();  // cs written; every warp is done reading ks
        {
            // refill this buffer with the tile two after this one
            const int64_t next = tile + 2 * (int64_t)ymain;
            if (nkb == 2 && next < tiles_vis) fetch_k(next, ks);
            cp_async_commit();
        }

        for (int p = tid; p < IDX_ROWS * tcount; p += IDX_THREADS) {
            const int tt = p / IDX_ROWS, r = p % IDX_ROWS;
            const int64_t s = r0 + r;
            if (s >= n_c) continue;
            const int t = t0 + tt;
            const int64_t vis = vis_s[tt];
            uint16_t out = 0xff80u;  // -inf: not visible yet
            if (s < vis) {
                const float* col = cs + r * (QN + 1) + tt * hpad;
                const float* wt = wsm + tt * hpad;
                float a = 0.0f;
                if (Hi == 64) {
                    // the same chain unrolled: its loads no longer wait in turn
#pragma unroll
                    for (int h = 0; h < 64; h++) a = __fmaf_rn(wt[h], fmaxf(col[h], 0.0f), a);
                } else {
                    for (int h = 0; h < Hi; h++) a = __fmaf_rn(wt[h], fmaxf(col[h], 0.0f), a);
                }
                out = f2bf(a);
                if (out == 0x8000u) out = 0u;
            }
            scores[(int64_t)t * n_c + s] = out;
        }
        it++;
    }
    cp_async_wait<0>();  // no copy of this CTA outlives it
}

// ---------------------------------------------------------------------------
// Top-k select + merge.  One CTA per query.  Scores map to 16-bit keys whose
// unsigned order is the float order; two 8-bit histogram passes find the key
// T of the k-th largest score, then one ordered pass keeps every row with a
// larger key and the lowest-numbered rows with key T, writing them in
// ascending row order.
// ---------------------------------------------------------------------------
// Top-k of many short rows (at most TKW_MAX visible scores): one warp per
// query, eight queries a CTA, no block-wide barrier.  Lane l holds the run of
// kpl consecutive order keys from kpl * l in registers (index order lane,
// register); the two 8-bit histogram passes go into the warp's own shared
// histogram, the warp finds the threshold, and one warp scan places the picks
// (the lowest-numbered ties first), merged after the window indices.
// ---------------------------------------------------------------------------
constexpr int TKW_WARPS = 8;
constexpr int TKW_MAX = WTK_MAX;          // 1024 visible scores

__global__ void __launch_bounds__(32 * TKW_WARPS) topk_warp_kernel(
    const uint16_t* __restrict__ scores, const int32_t* __restrict__ win_idx,
    int32_t* __restrict__ idx, int64_t m, int64_t n_c, int win, int ctopk, int64_t ratio,
    int64_t start_pos, int64_t offset) {
    __shared__ __align__(16) int hist_all[TKW_WARPS][256];
    __shared__ int sel_all[TKW_WARPS][4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t = (int64_t)blockIdx.x * TKW_WARPS + warp;
    // the rows this query can see (a 64-bit division, from the arguments
    // alone) while the kernel before finishes
    const int64_t vis64 = t < m ? visible_rows(t, start_pos, ratio, n_c) : 0;
    pdl_wait();     // the scores (and window indices) come from the previous kernel
    pdl_trigger();
    if (t >= m) return;  // whole warps only: the rest of the CTA syncs nothing with it
    const int K = win + ctopk;
    int32_t* out = idx + t * K;
    for (int j = lane; j < win; j += 32) out[j] = win_idx[t * win + j];
    const int vis = (int)vis64;  // <= TKW_MAX (host plan)
    const int kk = vis < ctopk ? vis : ctopk;
    if (vis <= ctopk) {
        for (int j = lane; j < ctopk; j += 32) out[win + j] = (j < vis) ? (int32_t)(offset + j) : -1;
        return;
    }
    warp_topk(scores + t * n_c, vis, kk, hist_all[warp], sel_all[warp],
              [&](int pos, int r) { out[win + pos] = (int32_t)(offset + r); });
    for (int j = kk + lane; j < ctopk; j += 32) out[win + j] = -1;
}

// ---------------------------------------------------------------------------
struct KeySrc {
    const uint16_t* g;
    const uint16_t* s;
    __device__ __forceinline__ uint32_t operator()(int64_t i) const {
        return s ? (uint32_t)s[i] : order_key(g[i]);
    }
};

__global__ void __launch_bounds__(1024) topk_merge_kernel(
    const uint16_t* __restrict__ scores, const int32_t* __restrict__ win_idx,
    int32_t* __restrict__ idx, int64_t n_c, int win, int ctopk, int64_t ratio, int64_t start_pos,
    int64_t offset, int keys_cap) {
    extern __shared__ __align__(16) uint16_t skeys[];
    __shared__ int hist[256];
    __shared__ int wsum[64];
    __shared__ int sel[4];
    const int t = blockIdx.x;
    // the rows this query can see (a 64-bit division, from the arguments
    // alone) while the kernel before finishes
    const int64_t vis = visible_rows(t, start_pos, ratio, n_c);
    pdl_wait();     // the scores (and window indices) come from the previous kernel
    pdl_trigger();
    const int K = win + ctopk;
    int32_t* out = idx + (int64_t)t * K;
    const uint16_t* sc = scores + (int64_t)t * n_c;
    for (int j = threadIdx.x; j < win; j += blockDim.x) out[j] = win_idx[(int64_t)t * win + j];
    const int kk = (int)(vis < ctopk ? vis : ctopk);
    if (vis <= ctopk) {
        for (int j = threadIdx.x; j < ctopk; j += blockDim.x)
            out[win + j] = (j < vis) ? (int32_t)(offset + j) : -1;
        return;
    }
    KeySrc key{sc, nullptr};
    if (vis <= keys_cap) {
        // 8 scores per 16-byte load when the row is aligned, else one by one
        const bool vec = ((reinterpret_cast<uintptr_t>(sc) & 15u) == 0);
        const int64_t n8 = vec ? vis / 8 : 0;
        for (int64_t i = threadIdx.x; i < n8; i += blockDim.x) {
            uint4 v = __ldg(reinterpret_cast<const uint4*>(sc) + i);
            const uint16_t* h = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
            for (int e = 0; e < 8; e++) skeys[i * 8 + e] = (uint16_t)order_key(h[e]);
        }
        for (int64_t i = n8 * 8 + threadIdx.x; i < vis; i += blockDim.x)
            skeys[i] = (uint16_t)order_key(sc[i]);
        __syncthreads();
        key.s = skeys;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    // pass 1: high byte.  Close scores share a bin, so the lanes of a warp
    // that hold the same bin add their count with one atomic.
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t base = threadIdx.x - lane; base < vis; base += blockDim.x) {
        const int64_t s = base + lane;
        const uint32_t bin = s < vis ? key(s) >> 8 : 0x10000u;
        const uint32_t mm = __match_any_sync(0xffffffffu, bin);
        if (bin < 256u && lane == __ffs(mm) - 1) atomicAdd(&hist[bin], __popc(mm));
    }
    __syncthreads();
    if (threadIdx.x < 32) find_bucket(hist, kk, 0, &sel[0], &sel[1]);
    __syncthreads();
    const uint32_t hb = (uint32_t)sel[0];
    const int above1 = sel[1];
    __syncthreads();
    // pass 2: low byte inside bucket hb
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t base = threadIdx.x - lane; base < vis; base += blockDim.x) {
        const int64_t s = base + lane;
        uint32_t bin = 0x10000u;
        if (s < vis) {
            const uint32_t k = key(s);
            if ((k >> 8) == hb) bin = k & 0xffu;
        }
        const uint32_t mm = __match_any_sync(0xffffffffu, bin);
        if (bin < 256u && lane == __ffs(mm) - 1) atomicAdd(&hist[bin], __popc(mm));
    }
    __syncthreads();
    if (threadIdx.x < 32) find_bucket(hist, kk, above1, &sel[2], &sel[3]);
    __syncthreads();
    const uint32_t T = (hb << 8) | (uint32_t)sel[2];
    const int need_eq = kk - sel[3];
    // pass 3: each warp takes a contiguous block of the visible keys, its
    // lanes interleaved (conflict-free shared-memory reads); ballots count the
    // keys above T and equal to T, a scan over the warps turns the counts into
    // output offsets (the equal keys taken are the lowest-numbered need_eq of
    // them), and every block is written in ascending row order.
    const int64_t wseg = ((vis + nwarps - 1) / nwarps + 31) & ~int64_t(31);
    const int64_t w_lo = min(vis, (int64_t)warp * wseg);
    const int64_t w_hi = min(vis, w_lo + wseg);
    const uint32_t lt = (1u << lane) - 1u;
    int n_gt = 0, n_eq = 0;
    for (int64_t b0 = w_lo; b0 < w_hi; b0 += 32) {
        const int64_t s = b0 + lane;
        const uint32_t k = s < w_hi ? key(s) : 0u;
        n_gt += __popc(__ballot_sync(0xffffffffu, s < w_hi && k > T));
        n_eq += __popc(__ballot_sync(0xffffffffu, s < w_hi && k == T));
    }
    if (lane == 0) {
        wsum[warp] = n_gt;
        wsum[32 + warp] = n_eq;
    }
    __syncthreads();
    if (warp == 0) {
        const int a = lane < nwarps ? wsum[lane] : 0;
        const int e = lane < nwarps ? wsum[32 + lane] : 0;
        int xa = a, xe = e;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int oa = __shfl_up_sync(0xffffffffu, xa, off);
            const int oe = __shfl_up_sync(0xffffffffu, xe, off);
            if (lane >= off) {
                xa += oa;
                xe += oe;
            }
        }
        __syncwarp();
        if (lane < nwarps) {
            wsum[lane] = xa - a;
            wsum[32 + lane] = xe - e;
        }
    }
    __syncthreads();
    int eq_rank = wsum[32 + warp];
    int pos = wsum[warp] + min(eq_rank, need_eq);
    for (int64_t b0 = w_lo; b0 < w_hi; b0 += 32) {
        const int64_t s = b0 + lane;
        const uint32_t k = s < w_hi ? key(s) : 0u;
        const bool eq = s < w_hi && k == T;
        const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
        const bool take = (s < w_hi && k > T) || (eq && eq_rank + __popc(eqb & lt) < need_eq);
        const uint32_t tb = __ballot_sync(0xffffffffu, take);
        const int at = pos + __popc(tb & lt);
        if (take && at < kk) out[win + at] = (int32_t)(offset + s);
        pos += __popc(tb);
        eq_rank += __popc(eqb);
    }
    for (int j = kk + threadIdx.x; j < ctopk; j += blockDim.x) out[win + j] = -1;
}

// ---------------------------------------------------------------------------
// Top-k of few long rows: a cluster of TK_CL CTAs per query, CTA r holding
// slice r of the visible scores (up to TK_SMALL keys, staged in shared
// memory; longer slices: topk_cluster_big_kernel).  The same two histogram
// passes and the ordered pass as above, with the histograms summed over the
// cluster through
// distributed shared memory (every CTA derives the same threshold) and a
// cluster-wide prefix of the per-CTA counts, so the picks still come out in
// ascending row order.
// ---------------------------------------------------------------------------
constexpr int TK_CL = 8;
constexpr int TK_THREADS = 512;
constexpr int TK_SLICE_CAP = 8192;  // keys of a slice
constexpr int TK_SMALL = 2048;      // slices up to this size: keys staged in shared memory

__global__ void __launch_bounds__(TK_THREADS) topk_cluster_kernel(
    const uint16_t* __restrict__ scores, const int32_t* __restrict__ win_idx,
    int32_t* __restrict__ idx, int64_t n_c, int win, int ctopk, int64_t ratio, int64_t start_pos,
    int64_t offset) {
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    __shared__ __align__(16) uint16_t skeys[TK_SLICE_CAP];
    __shared__ int hist1[256], hist2[256], ghist[256];
    __shared__ int wsum[64];
    __shared__ int sel[4];
    __shared__ int tot[2];
    const int t = blockIdx.x / TK_CL;
    // the rows this query can see (a 64-bit division, from the arguments
    // alone) while the kernel before finishes
    const int64_t vis = visible_rows(t, start_pos, ratio, n_c);
    pdl_wait();  // the scores (and window indices) come from the previous kernel
    pdl_trigger();
    const int r = (int)cl.block_rank();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int K = win + ctopk;
    int32_t* out = idx + (int64_t)t * K;
    const uint16_t* sc = scores + (int64_t)t * n_c;
    if (r == 0)
        for (int j = threadIdx.x; j < win; j += blockDim.x) out[j] = win_idx[(int64_t)t * win + j];
    const int kk = (int)(vis < ctopk ? vis : ctopk);
    if (vis <= ctopk) {  // the same branch in every CTA of the cluster
        if (r == 0)
            for (int j = threadIdx.x; j < ctopk; j += blockDim.x)
                out[win + j] = (j < vis) ? (int32_t)(offset + j) : -1;
        return;
    }
    const int64_t seg = ((vis + TK_CL - 1) / TK_CL + 7) & ~int64_t(7);
    const int64_t lo = min(vis, (int64_t)r * seg);
    const int n = (int)(min(vis, lo + seg) - lo);
    const bool vec = ((reinterpret_cast<uintptr_t>(sc + lo) & 15u) == 0);
    const int n8 = vec ? n / 8 : 0;
    for (int i = threadIdx.x; i < n8; i += blockDim.x) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(sc + lo) + i);
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
        for (int e = 0; e < 8; e++) skeys[i * 8 + e] = (uint16_t)order_key(h[e]);
    }
    for (int i = n8 * 8 + threadIdx.x; i < n; i += blockDim.x) skeys[i] = (uint16_t)order_key(sc[lo + i]);
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist1[i] = hist2[i] = 0;
    __syncthreads();
    // pass 1: high byte of this slice
    for (int base = threadIdx.x - lane; base < n; base += blockDim.x) {
        const int i = base + lane;
        const uint32_t bin = i < n ? (uint32_t)skeys[i] >> 8 : 0x10000u;
        const uint32_t mm = __match_any_sync(0xffffffffu, bin);
        if (bin < 256u && lane == __ffs(mm) - 1) atomicAdd(&hist1[bin], __popc(mm));
    }
    cl.sync();  // every slice's histogram is complete
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        int v = 0;
        for (int q = 0; q < TK_CL; q++) v += cl.map_shared_rank(hist1, q)[i];
        ghist[i] = v;
    }
    __syncthreads();
    if (threadIdx.x < 32) find_bucket(ghist, kk, 0, &sel[0], &sel[1]);
    __syncthreads();
    const uint32_t hb = (uint32_t)sel[0];
    const int above1 = sel[1];
    // pass 2: low byte inside bucket hb
    for (int base = threadIdx.x - lane; base < n; base += blockDim.x) {
        const int i = base + lane;
        uint32_t bin = 0x10000u;
        if (i < n && ((uint32_t)skeys[i] >> 8) == hb) bin = skeys[i] & 0xffu;
        const uint32_t mm = __match_any_sync(0xffffffffu, bin);
        if (bin < 256u && lane == __ffs(mm) - 1) atomicAdd(&hist2[bin], __popc(mm));
    }
    cl.sync();
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        int v = 0;
        for (int q = 0; q < TK_CL; q++) v += cl.map_shared_rank(hist2, q)[i];
        ghist[i] = v;
    }
    __syncthreads();
    if (threadIdx.x < 32) find_bucket(ghist, kk, above1, &sel[2], &sel[3]);
    __syncthreads();
    const uint32_t T = (hb << 8) | (uint32_t)sel[2];
    const int need_eq = kk - sel[3];
    // pass 3: per-warp blocks of the slice, counted with ballots
    const int wseg = ((n + nwarps - 1) / nwarps + 31) & ~31;
    const int w_lo = min(n, warp * wseg), w_hi = min(n, w_lo + wseg);
    const uint32_t lt = (1u << lane) - 1u;
    int n_gt = 0, n_eq = 0;
    for (int b0 = w_lo; b0 < w_hi; b0 += 32) {
        const int i = b0 + lane;
        const uint32_t k = i < w_hi ? skeys[i] : 0u;
        n_gt += __popc(__ballot_sync(0xffffffffu, i < w_hi && k > T));
        n_eq += __popc(__ballot_sync(0xffffffffu, i < w_hi && k == T));
    }
    if (lane == 0) {
        wsum[warp] = n_gt;
        wsum[32 + warp] = n_eq;
    }
    __syncthreads();
    if (warp == 0) {
        const int a = lane < nwarps ? wsum[lane] : 0;
        const int e = lane < nwarps ? wsum[32 + lane] : 0;
        int xa = a, xe = e;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int oa = __shfl_up_sync(0xffffffffu, xa, off);
            const int oe = __shfl_up_sync(0xffffffffu, xe, off);
            if (lane >= off) {
                xa += oa;
                xe += oe;
            }
        }
        __syncwarp();
        if (lane < nwarps) {
            wsum[lane] = xa - a;
            wsum[32 + lane] = xe - e;
        }
        if (lane == 31) {
            tot[0] = xa;
            tot[1] = xe;
        }
    }
    cl.sync();  // every slice's totals are published
    int gt_before = 0, eq_before = 0;
    for (int q = 0; q < r; q++) {
        const int* rt = cl.map_shared_rank(tot, q);
        gt_before += rt[0];
        eq_before += rt[1];
    }
    int eq_rank = eq_before + wsum[32 + warp];
    int pos = gt_before + wsum[warp] + min(eq_rank, need_eq);
    for (int b0 = w_lo; b0 < w_hi; b0 += 32) {
        const int i = b0 + lane;
        const uint32_t k = i < w_hi ? skeys[i] : 0u;
        const bool eq = i < w_hi && k == T;
        const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
        const bool take = (i < w_hi && k > T) || (eq && eq_rank + __popc(eqb & lt) < need_eq);
        const uint32_t tb = __ballot_sync(0xffffffffu, take);
        const int at = pos + __popc(tb & lt);
        if (take && at < kk) out[win + at] = (int32_t)(offset + lo + i);
        pos += __popc(tb);
        eq_rank += __popc(eqb);
    }
    if (r == 0)
        for (int j = kk + threadIdx.x; j < ctopk; j += blockDim.x) out[win + j] = -1;
    cl.sync();  // the totals stay readable until every CTA has read them
}

// ---------------------------------------------------------------------------
// The same for long slices (more than TK_SMALL keys a CTA): CTA r holds
// slice r of the visible scores as 16-bit order keys in registers (a run of
// consecutive keys per thread, so index order is warp, lane, register).  The
// same two 8-bit histogram passes (per-warp histograms), with every slice's
// histogram pushed into every CTA of the cluster, so each CTA derives the same
// threshold from local sums; with the second pass each slice also pushes its
// count of keys above the threshold's bucket, from which every CTA knows how
// many picks and ties the earlier slices hold.  The picks, in ascending row
// order, go straight to global memory: two cluster barriers, and no CTA reads
// another's shared memory.
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(TK_THREADS) topk_cluster_big_kernel(
    const uint16_t* __restrict__ scores, const int32_t* __restrict__ win_idx,
    int32_t* __restrict__ idx, int64_t n_c, int win, int ctopk, int64_t ratio, int64_t start_pos,
    int64_t offset, unsigned int* status) {
    namespace cg = cooperative_groups;
    constexpr int NW = TK_THREADS / 32;
    constexpr uint32_t HB1 = 256 * 4;  // bytes a slice pushes in round 1 (its histogram)
    constexpr uint32_t HB2 = 260 * 4;  // round 2: its histogram, then its count above bucket hb
    constexpr int KMAX = TK_SLICE_CAP / TK_THREADS;
    cg::cluster_group cl = cg::this_cluster();
    __shared__ __align__(16) int whist[NW][256];      // per-warp histograms
    __shared__ __align__(16) int hist[256];           // this slice's pass-1 histogram (round 1's bytes)
    __shared__ __align__(16) int hpush1[TK_CL][256];  // every slice's pass-1 histogram (pushed)
    __shared__ __align__(16) int stage2[260];         // round 2's bytes: histogram, count above hb
    __shared__ __align__(16) int hpush2[TK_CL][260];  // every slice's round-2 bytes (pushed)
    __shared__ __align__(8) uint64_t xbar[2];         // the two exchange rounds
    __shared__ int ghist[256];
    __shared__ int wsum[64];
    __shared__ int sel[8];
    if (threadIdx.x == 0) {
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        mbar_init_fence();
    }
    __syncthreads();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");  // this CTA has started
    const int t = blockIdx.x / TK_CL;
    // the rows this query can see (a 64-bit division, from the arguments
    // alone) while the kernel before finishes
    const int64_t vis = visible_rows(t, start_pos, ratio, n_c);
    pdl_wait();  // the scores (and window indices) come from the previous kernel
    pdl_trigger();
    const int r = (int)cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = win + ctopk;
    int32_t* out = idx + (int64_t)t * K;
    const uint16_t* sc = scores + (int64_t)t * n_c;
    if (r == 0)
        for (int j = tid; j < win; j += TK_THREADS) out[j] = win_idx[(int64_t)t * win + j];
    const int kk = (int)(vis < ctopk ? vis : ctopk);
    if (vis <= ctopk) {  // the same branch in every CTA of the cluster
        if (r == 0)
            for (int j = tid; j < ctopk; j += TK_THREADS)
                out[win + j] = (j < vis) ? (int32_t)(offset + j) : -1;
        asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
        return;
    }
    const int64_t seg = ((vis + TK_CL - 1) / TK_CL + 7) & ~int64_t(7);
    const int64_t lo = min(vis, (int64_t)r * seg);
    const int n = (int)(min(vis, lo + seg) - lo);  // <= TK_SLICE_CAP (host plan)
    const int kpt = (n + TK_THREADS - 1) / TK_THREADS;
    const int i0 = kpt * tid;
    const uint16_t* ss = sc + lo;
    uint32_t key[KMAX];
    const bool vec = (kpt & 7) == 0 && ((reinterpret_cast<uintptr_t>(ss) & 15u) == 0);
#pragma unroll
    for (int v = 0; v < KMAX / 8; v++) {
        const int b0 = i0 + 8 * v;
        if (8 * v >= kpt || b0 >= n) continue;
        if (vec && b0 + 8 <= n) {  // whole groups of eight only: nothing past the slice is read
            uint4 u = __ldg(reinterpret_cast<const uint4*>(ss + b0));
            const uint16_t* h = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
            for (int e = 0; e < 8; e++) key[8 * v + e] = order_key(h[e]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++)
                if (8 * v + e < kpt && b0 + e < n) key[8 * v + e] = order_key(ss[b0 + e]);
        }
    }
    const int n_mine = max(0, min(kpt, n - i0));
    int* wh = whist[warp];
#pragma unroll
    for (int e = 0; e < 8; e++) wh[lane + 32 * e] = 0;
    __syncwarp();
    // pass 1: high byte of this slice
#pragma unroll
    for (int e = 0; e < KMAX; e++)
        if (e < n_mine) atomicAdd(&wh[key[e] >> 8], 1);
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");  // every CTA has started
    // Sums of four bins a thread; the slice's histogram then goes to every
    // CTA of the cluster by bulk copies that complete on the receiver's own
    // round barrier, so each CTA waits only for the bytes it receives.  The
    // staged bytes (hist, stage2) stay untouched until the closing barrier.
    if (tid < 64) {
        int4 v = make_int4(0, 0, 0, 0);
#pragma unroll
        for (int w = 0; w < NW; w++) {
            int4* h = reinterpret_cast<int4*>(&whist[w][4 * tid]);
            const int4 x = *h;
            v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
            *h = make_int4(0, 0, 0, 0);
        }
        *reinterpret_cast<int4*>(&hist[4 * tid]) = v;
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&xbar[0], TK_CL * HB1);
        for (int q = 0; q < TK_CL; q++)
            bulk_s2cluster(cluster_addr(&hpush1[r][0], q), hist, HB1, cluster_addr(&xbar[0], q));
    }
    if (!mbar_wait(&xbar[0], 0, kWaitPolls)) raise_status(status, DS41_E_TIMEOUT);
    for (int b = tid; b < 256; b += TK_THREADS) {
        int v = 0;
#pragma unroll
        for (int q = 0; q < TK_CL; q++) v += hpush1[q][b];
        ghist[b] = v;
    }
    __syncthreads();
    if (tid < 32) find_bucket(ghist, kk, 0, &sel[0], &sel[1]);
    __syncthreads();
    const uint32_t hb = (uint32_t)sel[0];
    const int above1 = sel[1];
    // pass 2: low byte inside bucket hb
#pragma unroll
    for (int e = 0; e < KMAX; e++)
        if (e < n_mine && (key[e] >> 8) == hb) atomicAdd(&wh[key[e] & 0xffu], 1);
    if (warp == 0) {
        int a = 0;
        for (int b = (int)hb + 1 + lane; b < 256; b += 32) a += hist[b];
        a = __reduce_add_sync(0xffffffffu, a);
        if (lane == 0) *reinterpret_cast<int4*>(&stage2[256]) = make_int4(a, 0, 0, 0);
    }
    __syncthreads();
    if (tid < 64) {
        int4 v = make_int4(0, 0, 0, 0);
#pragma unroll
        for (int w = 0; w < NW; w++) {
            const int4 x = *reinterpret_cast<const int4*>(&whist[w][4 * tid]);
            v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
        }
        *reinterpret_cast<int4*>(&stage2[4 * tid]) = v;
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(&xbar[1], TK_CL * HB2);
        for (int q = 0; q < TK_CL; q++)
            bulk_s2cluster(cluster_addr(&hpush2[r][0], q), stage2, HB2, cluster_addr(&xbar[1], q));
    }
    if (!mbar_wait(&xbar[1], 0, kWaitPolls)) raise_status(status, DS41_E_TIMEOUT);
    // every block this CTA receives has landed; no CTA leaves before all have
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
    for (int b = tid; b < 256; b += TK_THREADS) {
        int v = 0;
#pragma unroll
        for (int q = 0; q < TK_CL; q++) v += hpush2[q][b];
        ghist[b] = v;
    }
    __syncthreads();
    if (tid < 32) find_bucket(ghist, kk, above1, &sel[2], &sel[3]);
    __syncthreads();
    const uint32_t T = (hb << 8) | (uint32_t)sel[2];
    const int need_eq = kk - sel[3];
    if (warp == 0) {
        // keys above and at the threshold in the slices before this one
        const int tl = sel[2];
        int g = 0, e = 0;
        for (int q = 0; q < r; q++) {
            int a = 0;
            for (int b = tl + 1 + lane; b < 256; b += 32) a += hpush2[q][b];
            g += __reduce_add_sync(0xffffffffu, a) + hpush2[q][256];
            e += hpush2[q][tl];
        }
        if (lane == 0) {
            sel[4] = g;
            sel[5] = e;
        }
    }
    // this thread's keys above and at the threshold as bit masks (bit e:
    // key e), so that every key's rank among them is one population count
    static_assert(KMAX <= 32, "one mask word");
    uint32_t gm = 0, qm = 0;
#pragma unroll
    for (int e = 0; e < KMAX; e++) {
        gm |= (e < n_mine && key[e] > T) ? (1u << e) : 0u;
        qm |= (e < n_mine && key[e] == T) ? (1u << e) : 0u;
    }
    const int n_gt = __popc(gm), n_eq = __popc(qm);
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
    int gt = sel[4] + x_gt - n_gt, eq = sel[5] + x_eq - n_eq;
    for (int w = 0; w < warp; w++) {
        gt += wsum[w];
        eq += wsum[32 + w];
    }
    const int32_t v0 = (int32_t)(offset + lo + i0);
#pragma unroll
    for (int e = 0; e < KMAX; e++) {
        const uint32_t below = (1u << e) - 1u;  // bits 0 .. e-1
        const int eqb = eq + __popc(qm & below);
        if (((gm >> e) & 1u) || (((qm >> e) & 1u) && eqb < need_eq))
            out[win + gt + __popc(gm & below) + min(eqb, need_eq)] = v0 + e;
    }
    if (r == 0)
        for (int j = kk + tid; j < ctopk; j += TK_THREADS) out[win + j] = -1;
    // no CTA leaves while a copy into or out of its shared memory may be in flight
    asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct IndexerPlan {
    int hpad, TT, groups;
    bool prequant;  // keys quantised once into the workspace
    bool tc;        // many tokens: scores on the tcgen05 tensor cores (q quantised in the kernel)
    size_t kq_bytes, sc_bytes;
};

int device_sm_count() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

// Workspace: [quantised keys | scores], each 256-byte aligned.
static IndexerPlan plan_indexer(int64_t m, int64_t Hi, int64_t Di, int64_t n_c, bool scores_given) {
    IndexerPlan p;
    p.hpad = (int)((Hi + 7) / 8 * 8);
    p.TT = IDX_N / p.hpad;
    if (p.TT < 1) p.TT = 1;
    p.groups = (int)((m + p.TT - 1) / p.TT);
    p.prequant = p.groups > 4;
    p.tc = p.prequant && indexer_tc_supported(m, Hi, Di, device_sm_count());
    p.kq_bytes = p.prequant ? align256((size_t)n_c * Di * 2) : 0;
    p.sc_bytes = scores_given ? 0 : align256((size_t)m * n_c * 2);
    return p;
}

template <int DI>
static int launch_scores(const IndexerPlan& p, const uint16_t* q, const uint16_t* k, const float* w,
                         uint16_t* scores, int64_t m, int64_t Hi, int64_t n_c, int64_t ratio,
                         int64_t start_pos, bool fill_hidden, cudaStream_t st,
                         const RingArgs* ring = nullptr, const LatentArgs* lat = nullptr) {
    // Row-tile splits: enough CTAs to cover the GPU when there are few tokens.
    const int64_t tiles = (n_c + IDX_ROWS - 1) / IDX_ROWS;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // every group's live columns fit in half the tile: one token of <= 64 heads
    const bool narrow = (int64_t)p.hpad * (m < p.TT ? m : p.TT) <= IDX_N / 2;
    const int qn = narrow ? IDX_N / 2 : IDX_N;
    int64_t ysplit = (2 * (int64_t)sms + p.groups - 1) / p.groups;
    int nkb = 2;
    if (narrow && p.groups * tiles <= 4 * (int64_t)sms) {
        // a CTA per tile and one key buffer: four CTAs fit an SM, and no CTA
        // runs two tiles in turn (long decode: 512 tiles)
        ysplit = tiles;
        nkb = 1;
    }
    if (ysplit > tiles) ysplit = tiles;
    if (ysplit < 1) ysplit = 1;
    const size_t smem = (size_t)qn * DI * 2 + (size_t)nkb * IDX_ROWS * DI * 2 +
                        (size_t)IDX_ROWS * (qn + 1) * 4 + qn * 4;
    const bool side = ring != nullptr;
    const RingArgs ra = side ? *ring : RingArgs{};
    const LatentArgs la = side ? *lat : LatentArgs{};
    dim3 grid((unsigned)p.groups, (unsigned)(ysplit + (side ? 1 : 0)));
    auto kern = p.prequant ? (narrow ? indexer_scores_kernel<DI, false, true>
                                     : indexer_scores_kernel<DI, false, false>)
                           : (narrow ? indexer_scores_kernel<DI, true, true>
                                     : indexer_scores_kernel<DI, true, false>);
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    // programmatic stream serialization: the kernel may launch while the one
    // before it runs (it waits for it before touching memory)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(IDX_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int rc = cuda_check(cudaLaunchKernelEx(&cfg, kern, q, k, w, scores, (int)m, (int)Hi, p.hpad,
                                           p.TT, n_c, ratio, start_pos, fill_hidden, (int)ysplit,
                                           nkb, ra, la),
                        "ds41_indexer_topk: scores kernel");
    if (rc) return rc;
    return launch_check("ds41_indexer_topk: scores kernel");
}

}  // namespace ds41

using namespace ds41;

extern "C" size_t ds41_indexer_workspace_bytes(int64_t m, int64_t Hi, int64_t Di, int64_t n_c,
                                               int scores_out_given) {
    if (m < 1 || Hi < 1 || Di < 1 || n_c < 1) return 0;
    IndexerPlan p = plan_indexer(m, Hi, Di, n_c, scores_out_given != 0);
    return p.kq_bytes + p.sc_bytes;
}

extern "C" int ds41_indexer_topk(const ds41_bf16* q_idx, const ds41_bf16* k_idx, const float* w,
                                 const int32_t* win_idx, int32_t* idx, ds41_bf16* scores,
                                 int64_t m, int64_t Hi, int64_t Di, int64_t n_c, int64_t win,
                                 int64_t ratio, int64_t start_pos, int64_t topk, int64_t offset,
                                 void* ws, size_t ws_bytes, ds41_stream_t stream) {
    const char* name = "ds41_indexer_topk";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 31), DS41_E_RANGE, "%s: m=%lld", name,
                 (long long)m);
    DS41_REQUIRE(Hi >= 1 && Hi <= 128, DS41_E_ARG, "%s: Hi=%lld must be in 1..128", name,
                 (long long)Hi);
    DS41_REQUIRE(Di == 32 || Di == 64 || Di == 128 || Di == 256, DS41_E_ARG,
                 "%s: Di=%lld must be 32, 64, 128 or 256", name, (long long)Di);
    DS41_REQUIRE(n_c >= 1 && n_c < (int64_t(1) << 31), DS41_E_ARG, "%s: n_c=%lld", name,
                 (long long)n_c);
    DS41_REQUIRE(win >= 0 && win <= (int64_t(1) << 20), DS41_E_ARG, "%s: win=%lld", name,
                 (long long)win);
    DS41_REQUIRE(ratio >= 1 && start_pos >= 0, DS41_E_ARG, "%s: ratio=%lld start_pos=%lld", name,
                 (long long)ratio, (long long)start_pos);
    DS41_REQUIRE(topk >= 1, DS41_E_RANGE, "%s: topk=%lld", name, (long long)topk);
    DS41_REQUIRE(q_idx && k_idx && w && idx && (win == 0 || win_idx), DS41_E_ARG,
                 "%s: null tensor pointer", name);
    DS41_REQUIRE(aligned16(q_idx) && aligned16(k_idx), DS41_E_ARG,
                 "%s: q_idx/k_idx must be 16-byte aligned", name);
    const int64_t ctopk = topk < n_c ? topk : n_c;
    DS41_REQUIRE(win + ctopk < (int64_t(1) << 30), DS41_E_RANGE, "%s: merged row too long", name);
    IndexerPlan p = plan_indexer(m, Hi, Di, n_c, scores != nullptr);
    const size_t need = p.kq_bytes + p.sc_bytes;
    DS41_REQUIRE(need == 0 || (ws && ws_bytes >= need), DS41_E_WORKSPACE,
                 "%s: workspace of %zu bytes needed, %zu given", name, need, ws ? ws_bytes : 0);
    DS41_REQUIRE(need == 0 || aligned16(ws), DS41_E_ARG, "%s: ws must be 16-byte aligned", name);
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    uint16_t* kq = p.prequant ? reinterpret_cast<uint16_t*>(wsb) : nullptr;
    uint16_t* sc = scores ? scores : reinterpret_cast<uint16_t*>(wsb + p.kq_bytes);
    int rc;
    if (p.prequant) {
        rc = ds41_fp4_quant_e8m0(k_idx, kq, nullptr, nullptr, n_c, Di, stream);
        if (rc) return rc;
    }
    const uint16_t* ksrc = p.prequant ? kq : k_idx;
    const bool fill = scores != nullptr;
    if (p.tc && aligned16(w)) {
        // the scores on the tensor cores, q quantised in the kernel
        unsigned int* status = nullptr;
        rc = status_word(&status);
        if (rc) return rc;
        rc = indexer_tc_launch(q_idx, kq, w, sc, m, n_c, ratio, start_pos, fill, status,
                               device_sm_count(), st);
    } else switch (Di) {
        case 32: rc = launch_scores<32>(p, q_idx, ksrc, w, sc, m, Hi, n_c, ratio, start_pos, fill, st); break;
        case 64: rc = launch_scores<64>(p, q_idx, ksrc, w, sc, m, Hi, n_c, ratio, start_pos, fill, st); break;
        case 128: rc = launch_scores<128>(p, q_idx, ksrc, w, sc, m, Hi, n_c, ratio, start_pos, fill, st); break;
        default: rc = launch_scores<256>(p, q_idx, ksrc, w, sc, m, Hi, n_c, ratio, start_pos, fill, st); break;
    }
    if (rc) return rc;
    return launch_topk(sc, win_idx, idx, m, n_c, win, ctopk, ratio, start_pos, offset, false, st);
}

extern "C" size_t ds41_indexer_mxf4_workspace_bytes(int64_t m, int64_t n_c,
                                                    int scores_out_given) {
    if (m < 1 || n_c < 1 || scores_out_given) return 0;
    return align256((size_t)m * n_c * 2);
}

extern "C" int ds41_indexer_topk_mxf4(const ds41_bf16* q_idx, const uint8_t* k_codes,
                                      const uint8_t* k_scales, const float* w,
                                      const int32_t* win_idx, int32_t* idx, ds41_bf16* scores,
                                      int64_t m, int64_t Hi, int64_t Di, int64_t n_c, int64_t win,
                                      int64_t ratio, int64_t start_pos, int64_t topk,
                                      int64_t offset, void* ws, size_t ws_bytes,
                                      ds41_stream_t stream) {
    const char* name = "ds41_indexer_topk_mxf4";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 25), DS41_E_RANGE, "%s: m=%lld", name,
                 (long long)m);
    DS41_REQUIRE(indexer_mxf4_supported(Hi, Di), DS41_E_ARG,
                 "%s: Hi=%lld Di=%lld; the packed-key path takes 64 heads of dim 128", name,
                 (long long)Hi, (long long)Di);
    DS41_REQUIRE(n_c >= 1 && n_c < (int64_t(1) << 31), DS41_E_ARG, "%s: n_c=%lld", name,
                 (long long)n_c);
    DS41_REQUIRE(win >= 0 && win <= (int64_t(1) << 20), DS41_E_ARG, "%s: win=%lld", name,
                 (long long)win);
    DS41_REQUIRE(ratio >= 1 && start_pos >= 0, DS41_E_ARG, "%s: ratio=%lld start_pos=%lld", name,
                 (long long)ratio, (long long)start_pos);
    DS41_REQUIRE(topk >= 1, DS41_E_RANGE, "%s: topk=%lld", name, (long long)topk);
    DS41_REQUIRE(q_idx && k_codes && k_scales && w && idx && (win == 0 || win_idx), DS41_E_ARG,
                 "%s: null tensor pointer", name);
    DS41_REQUIRE(aligned16(q_idx) && aligned16(k_codes) && aligned16(k_scales) && aligned16(w),
                 DS41_E_ARG, "%s: q_idx/k_codes/k_scales/w must be 16-byte aligned", name);
    const int64_t ctopk = topk < n_c ? topk : n_c;
    DS41_REQUIRE(win + ctopk < (int64_t(1) << 30), DS41_E_RANGE, "%s: merged row too long", name);
    const size_t need = ds41_indexer_mxf4_workspace_bytes(m, n_c, scores != nullptr);
    DS41_REQUIRE(need == 0 || (ws && ws_bytes >= need), DS41_E_WORKSPACE,
                 "%s: workspace of %zu bytes needed, %zu given", name, need, ws ? ws_bytes : 0);
    DS41_REQUIRE(need == 0 || aligned16(ws), DS41_E_ARG, "%s: ws must be 16-byte aligned", name);
    cudaStream_t st = (cudaStream_t)stream;
    uint16_t* sc = scores ? scores : static_cast<uint16_t*>(ws);
    unsigned int* status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    rc = indexer_mxf4_launch(q_idx, k_codes, k_scales, w, sc, m, n_c, ratio, start_pos,
                             scores != nullptr, status, device_sm_count(), st);
    if (rc) return rc;
    return launch_topk(sc, win_idx, idx, m, n_c, win, ctopk, ratio, start_pos, offset, false, st);
}

// ---------------------------------------------------------------------------
// Pieces of the fused step (ds41_forward.cu).
// ---------------------------------------------------------------------------
namespace ds41 {

size_t front_scores_bytes(int64_t m, int64_t n_c) { return align256((size_t)m * n_c * 2); }

bool front_fusable(int64_t m, int64_t Hi, int64_t Di, int64_t n_c) {
    if (n_c < 1 || Hi < 1 || Hi > 128) return false;
    if (!(Di == 32 || Di == 64 || Di == 128 || Di == 256)) return false;
    IndexerPlan p = plan_indexer(m, Hi, Di, n_c, false);
    return !p.prequant;
}

int launch_front(const uint16_t* q_idx, const uint16_t* k_idx, const float* w, uint16_t* scores,
                 int64_t m, int64_t Hi, int64_t Di, int64_t n_c, int64_t ratio,
                 int64_t start_pos, const RingArgs& ring, const LatentArgs& lat,
                 cudaStream_t st) {
    IndexerPlan p = plan_indexer(m, Hi, Di, n_c, true);
    switch (Di) {
        case 32: return launch_scores<32>(p, q_idx, k_idx, w, scores, m, Hi, n_c, ratio, start_pos, false, st, &ring, &lat);
        case 64: return launch_scores<64>(p, q_idx, k_idx, w, scores, m, Hi, n_c, ratio, start_pos, false, st, &ring, &lat);
        case 128: return launch_scores<128>(p, q_idx, k_idx, w, scores, m, Hi, n_c, ratio, start_pos, false, st, &ring, &lat);
        default: return launch_scores<256>(p, q_idx, k_idx, w, scores, m, Hi, n_c, ratio, start_pos, false, st, &ring, &lat);
    }
}

int launch_topk(const uint16_t* scores, const int32_t* win_idx, int32_t* idx, int64_t m,
                int64_t n_c, int64_t win, int64_t ctopk, int64_t ratio, int64_t start_pos,
                int64_t offset, bool pdl, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        na++;
    }
    int rc;
    // Many queries with rows of 513..1024 scores: a warp per query (shorter
    // rows gain nothing over one CTA per query).
    if (n_c > TKW_MAX / 2 && n_c <= TKW_MAX && m * 32 > (int64_t)device_sm_count()) {
        cfg.gridDim = dim3((unsigned)((m + TKW_WARPS - 1) / TKW_WARPS));
        cfg.blockDim = dim3(32 * TKW_WARPS);
        cfg.dynamicSmemBytes = 0;
        cfg.attrs = attr;
        cfg.numAttrs = na;
        rc = cuda_check(cudaLaunchKernelEx(&cfg, topk_warp_kernel, scores, win_idx, idx, m, n_c,
                                           (int)win, (int)ctopk, ratio, start_pos, offset),
                        "top-k warp kernel");
        if (rc) return rc;
        return launch_check("top-k warp kernel");
    }
    // Few queries with long rows: a cluster per query splits each row over
    // TK_CL SMs.  Otherwise one CTA per query.
    if (m * TK_CL <= 2 * (int64_t)device_sm_count() && n_c >= 1024 &&
        n_c <= (int64_t)TK_CL * TK_SLICE_CAP) {
        cfg.gridDim = dim3((unsigned)(m * TK_CL));
        cfg.blockDim = dim3(TK_THREADS);
        cfg.dynamicSmemBytes = 0;
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = TK_CL;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        na++;
        cfg.attrs = attr;
        cfg.numAttrs = na;
        const bool big = n_c > (int64_t)TK_CL * TK_SMALL;
        if (big) {
            unsigned int* status = nullptr;
            if ((rc = status_word(&status))) return rc;
            rc = cuda_check(cudaLaunchKernelEx(&cfg, topk_cluster_big_kernel, scores, win_idx, idx,
                                               n_c, (int)win, (int)ctopk, ratio, start_pos, offset,
                                               status),
                            "top-k cluster kernel");
        } else {
            rc = cuda_check(cudaLaunchKernelEx(&cfg, topk_cluster_kernel, scores, win_idx, idx, n_c,
                                               (int)win, (int)ctopk, ratio, start_pos, offset),
                            "top-k cluster kernel");
        }
        if (rc) return rc;
        return launch_check("top-k cluster kernel");
    }
    const int threads = n_c >= 8192 ? 1024 : (n_c >= 1024 ? 512 : 256);
    const int keys_cap = (int)(n_c < 49152 ? n_c : 49152);  // up to 96 KiB of staged keys
    const size_t ksm = ((size_t)keys_cap * 2 + 15) & ~size_t(15);
    if (ksm > 48 * 1024)
        cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ksm);
    cfg.gridDim = dim3((unsigned)m);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = ksm;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    rc = cuda_check(cudaLaunchKernelEx(&cfg, topk_merge_kernel, scores, win_idx, idx, n_c,
                                       (int)win, (int)ctopk, ratio, start_pos, offset, keys_cap),
                    "top-k kernel");
    if (rc) return rc;
    return launch_check("top-k kernel");
}

}  // namespace ds41
