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
#include "ds41_common.cuh"

namespace ds41 {

constexpr int IDX_ROWS = 64;     // compressed rows per tile (16 per warp)
constexpr int IDX_N = 128;       // (token, head) columns per CTA
constexpr int IDX_THREADS = 128;

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
    const float s = pow2_ceil_pos(__fdiv_rn(amax, 6.0f));
    uint4 out;
    uint16_t* o = reinterpret_cast<uint16_t*>(&out);
#pragma unroll
    for (int k = 0; k < 8; k++) {
        uint32_t c;
        o[k] = f2bf(fp4_elem(v[k], s, &c));
    }
    return out;
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
// ordered head chain and writes the bf16 score.
template <int DI, bool KQ_INLINE>
__global__ void __launch_bounds__(IDX_THREADS) indexer_scores_kernel(
    const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_src,
    const float* __restrict__ w, uint16_t* __restrict__ scores, int m, int Hi, int hpad, int TT,
    int64_t n_c, int64_t ratio, int64_t start_pos, bool fill_hidden) {
    constexpr int CPR = DI / 8;  // 16-byte chunks per row
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t* qs = reinterpret_cast<uint16_t*>(smem);                 // [IDX_N][DI]
    uint16_t* ks = qs + IDX_N * DI;                                    // [IDX_ROWS][DI]
    float* cs = reinterpret_cast<float*>(ks + IDX_ROWS * DI);         // [IDX_ROWS][IDX_N + 1]
    float* wsm = cs + IDX_ROWS * (IDX_N + 1);                          // [IDX_N]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * TT;
    const int tcount = min(TT, m - t0);

    // q of this CTA's tokens, quantised, as rows n = tt * hpad + h.
    for (int id = tid; id < IDX_N * CPR; id += IDX_THREADS) {
        const int n = id / CPR, c = id % CPR;
        const int tt = n / hpad, h = n % hpad;
        const bool live = tt < tcount && h < Hi;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (live)
            raw = reinterpret_cast<const uint4*>(q_idx + ((int64_t)(t0 + tt) * Hi + h) * DI)[c];
        uint4 qv = q8_chunk(raw, live);
        if (!live) qv = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(qs + n * DI + swz<CPR>(n, c) * 8) = qv;
    }
    for (int n = tid; n < IDX_N; n += IDX_THREADS) {
        const int tt = n / hpad, h = n % hpad;
        wsm[n] = (tt < tcount && h < Hi) ? w[(int64_t)(t0 + tt) * Hi + h] : 0.0f;
    }

    const int64_t vis_last = visible_rows(t0 + tcount - 1, start_pos, ratio, n_c);
    const int64_t tiles_vis = (vis_last + IDX_ROWS - 1) / IDX_ROWS;
    // When the scores are a caller-visible output, rows no query of this
    // group can see yet are written as -inf too.
    const int64_t tiles = fill_hidden ? (n_c + IDX_ROWS - 1) / IDX_ROWS : tiles_vis;

    for (int64_t tile = blockIdx.y; tile < tiles; tile += gridDim.y) {
        const int64_t r0 = tile * IDX_ROWS;
        if (tile >= tiles_vis) {
            for (int p = tid; p < IDX_ROWS * tcount; p += IDX_THREADS) {
                const int tt = p / IDX_ROWS, r = p % IDX_ROWS;
                if (r0 + r < n_c) scores[(int64_t)(t0 + tt) * n_c + r0 + r] = 0xff80u;
            }
            continue;
        }
        __syncthreads();  // previous tile's readers are done with ks / cs
        for (int id = tid; id < IDX_ROWS * CPR; id += IDX_THREADS) {
            const int r = id / CPR, c = id % CPR;
            const int64_t row = r0 + r;
            const bool live = row < n_c;
            uint16_t* dst = ks + r * DI + swz<CPR>(r, c) * 8;
            if (KQ_INLINE) {
                uint4 raw = make_uint4(0, 0, 0, 0);
                if (live) raw = reinterpret_cast<const uint4*>(k_src + row * DI)[c];
                uint4 kv = q8_chunk(raw, live);
                if (!live) kv = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(dst) = kv;
            } else {
                cp_async16(smem_u32(dst), k_src + (live ? row : 0) * DI + c * 8, live);
            }
        }
        if (!KQ_INLINE) {
            cp_async_commit();
            cp_async_wait<0>();
        }
        __syncthreads();

        float acc[IDX_N / 8][4];
#pragma unroll
        for (int j = 0; j < IDX_N / 8; j++)
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < DI / 16; kk++) {
            uint32_t a0, a1, a2, a3;
            {
                const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = kk * 2 + (lane >> 4);
                ldsm_x4(smem_u32(ks + r * DI + swz<CPR>(r, c) * 8), a0, a1, a2, a3);
            }
#pragma unroll
            for (int jj = 0; jj < IDX_N / 16; jj++) {
                uint32_t b0, b1, b2, b3;
                const int n = jj * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = kk * 2 + ((lane >> 3) & 1);
                ldsm_x4(smem_u32(qs + n * DI + swz<CPR>(n, c) * 8), b0, b1, b2, b3);
                mma_bf16(acc[2 * jj], a0, a1, a2, a3, b0, b1);
                mma_bf16(acc[2 * jj + 1], a0, a1, a2, a3, b2, b3);
            }
        }
#pragma unroll
        for (int j = 0; j < IDX_N / 8; j++) {
            const int r = warp * 16 + (lane >> 2);
            const int col = j * 8 + 2 * (lane & 3);
            cs[r * (IDX_N + 1) + col] = acc[j][0];
            cs[r * (IDX_N + 1) + col + 1] = acc[j][1];
            cs[(r + 8) * (IDX_N + 1) + col] = acc[j][2];
            cs[(r + 8) * (IDX_N + 1) + col + 1] = acc[j][3];
        }
        __syncthreads();

        for (int p = tid; p < IDX_ROWS * tcount; p += IDX_THREADS) {
            const int tt = p / IDX_ROWS, r = p % IDX_ROWS;
            const int64_t s = r0 + r;
            if (s >= n_c) continue;
            const int t = t0 + tt;
            const int64_t vis = visible_rows(t, start_pos, ratio, n_c);
            uint16_t out = 0xff80u;  // -inf: not visible yet
            if (s < vis) {
                const float* col = cs + r * (IDX_N + 1) + tt * hpad;
                const float* wt = wsm + tt * hpad;
                float a = 0.0f;
                for (int h = 0; h < Hi; h++) a = __fmaf_rn(wt[h], fmaxf(col[h], 0.0f), a);
                out = f2bf(a);
                if (out == 0x8000u) out = 0u;
            }
            scores[(int64_t)t * n_c + s] = out;
        }
    }
}

// ---------------------------------------------------------------------------
// Top-k select + merge.  One CTA per query.  Scores map to 16-bit keys whose
// unsigned order is the float order; two 8-bit histogram passes find the key
// T of the k-th largest score, then one ordered pass keeps every row with a
// larger key and the lowest-numbered rows with key T, writing them in
// ascending row order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t order_key(uint16_t b) {
    return (b & 0x8000u) ? (uint32_t)(~b & 0xffffu) : (uint32_t)(b | 0x8000u);
}

// Block-wide exclusive prefix count of a per-thread flag (blockDim multiple of
// 32, <= 1024).  Returns this thread's rank; *total gets the block total.
__device__ __forceinline__ int block_rank(bool flag, int* wsum, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    __syncthreads();
    if (lane == 0) wsum[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
        int v = lane < nw ? wsum[lane] : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane < nw) wsum[lane] = incl - v;
        if (lane == 31) wsum[32] = incl;
    }
    __syncthreads();
    *total = wsum[32];
    return wsum[warp] + in_warp;
}

__global__ void __launch_bounds__(1024) topk_merge_kernel(
    const uint16_t* __restrict__ scores, const int32_t* __restrict__ win_idx,
    int32_t* __restrict__ idx, int64_t n_c, int win, int ctopk, int64_t ratio, int64_t start_pos,
    int64_t offset) {
    __shared__ int hist[256];
    __shared__ int wsum[33];
    __shared__ int sel[4];
    const int t = blockIdx.x;
    const int K = win + ctopk;
    int32_t* out = idx + (int64_t)t * K;
    const uint16_t* sc = scores + (int64_t)t * n_c;
    for (int j = threadIdx.x; j < win; j += blockDim.x) out[j] = win_idx[(int64_t)t * win + j];
    const int64_t vis = visible_rows(t, start_pos, ratio, n_c);
    const int kk = (int)(vis < ctopk ? vis : ctopk);
    if (vis <= ctopk) {
        for (int j = threadIdx.x; j < ctopk; j += blockDim.x)
            out[win + j] = (j < vis) ? (int32_t)(offset + j) : -1;
        return;
    }
    // pass 1: high byte
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t s = threadIdx.x; s < vis; s += blockDim.x)
        atomicAdd(&hist[order_key(sc[s]) >> 8], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        int cum = 0, b = 255;
        for (; b > 0; b--) {
            if (cum + hist[b] >= kk) break;
            cum += hist[b];
        }
        sel[0] = b;
        sel[1] = cum;  // keys in higher buckets
    }
    __syncthreads();
    const uint32_t hb = (uint32_t)sel[0];
    const int above1 = sel[1];
    __syncthreads();
    // pass 2: low byte inside bucket hb
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t s = threadIdx.x; s < vis; s += blockDim.x) {
        const uint32_t k = order_key(sc[s]);
        if ((k >> 8) == hb) atomicAdd(&hist[k & 0xffu], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int cum = above1, b = 255;
        for (; b > 0; b--) {
            if (cum + hist[b] >= kk) break;
            cum += hist[b];
        }
        sel[2] = b;
        sel[3] = cum;  // keys strictly above T
    }
    __syncthreads();
    const uint32_t T = (hb << 8) | (uint32_t)sel[2];
    const int need_eq = kk - sel[3];
    // pass 3: ordered selection
    int base_out = 0, base_eq = 0;
    for (int64_t s0 = 0; s0 < vis; s0 += blockDim.x) {
        const int64_t s = s0 + threadIdx.x;
        const uint32_t k = (s < vis) ? order_key(sc[s]) : 0u;
        const bool gt = (s < vis) && k > T;
        const bool eq = (s < vis) && k == T;
        int n_eq;
        const int r_eq = block_rank(eq, wsum, &n_eq);
        const bool take = gt || (eq && base_eq + r_eq < need_eq);
        int n_take;
        const int r_take = block_rank(take, wsum, &n_take);
        if (take && base_out + r_take < kk) out[win + base_out + r_take] = (int32_t)(offset + s);
        base_out += n_take;
        base_eq += n_eq;
    }
    for (int j = kk + threadIdx.x; j < ctopk; j += blockDim.x) out[win + j] = -1;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct IndexerPlan {
    int hpad, TT, groups;
    bool prequant;
    size_t kq_bytes, sc_bytes;
};

static IndexerPlan plan_indexer(int64_t m, int64_t Hi, int64_t Di, int64_t n_c, bool scores_given) {
    IndexerPlan p;
    p.hpad = (int)((Hi + 7) / 8 * 8);
    p.TT = IDX_N / p.hpad;
    if (p.TT < 1) p.TT = 1;
    p.groups = (int)((m + p.TT - 1) / p.TT);
    p.prequant = p.groups > 4;
    p.kq_bytes = p.prequant ? align256((size_t)n_c * Di * 2) : 0;
    p.sc_bytes = scores_given ? 0 : align256((size_t)m * n_c * 2);
    return p;
}

template <int DI>
static int launch_scores(const IndexerPlan& p, const uint16_t* q, const uint16_t* k, const float* w,
                         uint16_t* scores, int64_t m, int64_t Hi, int64_t n_c, int64_t ratio,
                         int64_t start_pos, bool fill_hidden, cudaStream_t st) {
    const size_t smem = (size_t)IDX_N * DI * 2 + (size_t)IDX_ROWS * DI * 2 +
                        (size_t)IDX_ROWS * (IDX_N + 1) * 4 + IDX_N * 4;
    // Row-tile splits: enough CTAs to cover the GPU when there are few tokens.
    const int64_t tiles = (n_c + IDX_ROWS - 1) / IDX_ROWS;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t ysplit = (2 * (int64_t)sms + p.groups - 1) / p.groups;
    if (ysplit > tiles) ysplit = tiles;
    if (ysplit < 1) ysplit = 1;
    dim3 grid((unsigned)p.groups, (unsigned)ysplit);
    if (p.prequant) {
        auto kern = indexer_scores_kernel<DI, false>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, IDX_THREADS, smem, st>>>(q, k, w, scores, (int)m, (int)Hi, p.hpad, p.TT, n_c,
                                              ratio, start_pos, fill_hidden);
    } else {
        auto kern = indexer_scores_kernel<DI, true>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, IDX_THREADS, smem, st>>>(q, k, w, scores, (int)m, (int)Hi, p.hpad, p.TT, n_c,
                                              ratio, start_pos, fill_hidden);
    }
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
    switch (Di) {
        case 32: rc = launch_scores<32>(p, q_idx, ksrc, w, sc, m, Hi, n_c, ratio, start_pos, fill, st); break;
        case 64: rc = launch_scores<64>(p, q_idx, ksrc, w, sc, m, Hi, n_c, ratio, start_pos, fill, st); break;
        case 128: rc = launch_scores<128>(p, q_idx, ksrc, w, sc, m, Hi, n_c, ratio, start_pos, fill, st); break;
        default: rc = launch_scores<256>(p, q_idx, ksrc, w, sc, m, Hi, n_c, ratio, start_pos, fill, st); break;
    }
    if (rc) return rc;
    int threads = n_c >= 8192 ? 1024 : (n_c >= 1024 ? 512 : 256);
    topk_merge_kernel<<<(unsigned)m, threads, 0, st>>>(sc, win_idx, idx, n_c, (int)win, (int)ctopk,
                                                        ratio, start_pos, offset);
    return launch_check("ds41_indexer_topk: top-k kernel");
}
