// ds41_step1.cuh - step 1 of the forward as device functions: the window
// ring write with the window indices, and the compressed latent write.  Used
// by their own kernels (ds41_window.cu) and by the fused few-token front
// kernel (ds41_indexer.cu).
//
// metrale_model_arch/attn_v41/forward.rs, AttnV41::forward: "the window ring"
// copies, window_topk_idxs, and the latent branch (rope, fp4_quant with
// LATENT_BLOCK, copy to cache row start_pos / ratio).  The same steps appear
// in attention_any of metrale_model_arch/deepseek_v41_ref/compress.rs.
#pragma once

#include "ds41_common.cuh"

namespace ds41 {

// Non-negative remainder.
__device__ __forceinline__ int64_t pmod(int64_t a, int64_t b) {
    const int64_t r = a % b;
    return r < 0 ? r + b : r;
}

struct RingArgs {
    const uint4* kv;
    uint4* ring;
    uint4* rows_a;
    int32_t* win_idx;
    int64_t m, hd8, win, start_pos;
    bool chunk;
    __host__ __device__ int64_t total() const {
        return win * hd8 + (chunk ? m * hd8 : 0) + m * win;
    }
};

// Work item i of the ring write, over three independent parts:
//   A  win * hd/8 vectors: ring slot j takes the newest of this call's
//      positions q with q mod win == j (if any).  In chunk mode the slot's
//      old contents are first copied to rows_a[j] by the same thread, so the
//      read happens before the overwrite.
//   B  (chunk mode) m * hd/8 vectors: rows_a[win + t] = kv[t].
//   C  m * win window indices.
__device__ __forceinline__ void ring_write_item(const RingArgs& a, int64_t i) {
    const int64_t nA = a.win * a.hd8;
    const int64_t nB = a.chunk ? a.m * a.hd8 : 0;
    const int64_t nC = a.m * a.win;
    if (i < nA) {
        const int64_t j = i / a.hd8, v = i % a.hd8;
        if (a.chunk) a.rows_a[j * a.hd8 + v] = a.ring[j * a.hd8 + v];
        const int64_t last = a.start_pos + a.m - 1;
        const int64_t q = last - pmod(last - j, a.win);
        if (q >= a.start_pos) a.ring[j * a.hd8 + v] = a.kv[(q - a.start_pos) * a.hd8 + v];
        return;
    }
    i -= nA;
    if (i < nB) {
        a.rows_a[a.win * a.hd8 + i] = a.kv[i];
        return;
    }
    i -= nB;
    if (i < nC) {
        const int64_t t = i / a.win, j = i % a.win;
        a.win_idx[i] = window_index(a.start_pos, a.m, a.win, t, j);
    }
}

// The whole ring write done by one CTA (the fused few-token front kernel):
// the chunk copy of the old ring first, a barrier, then only the slots that
// receive a row, then the window indices.  32-bit index math (the few-token
// path has m * win and win * hd/8 far below 2^31).
__device__ __forceinline__ void ring_write_cta(const RingArgs& a) {
    const int hd8 = (int)a.hd8, win = (int)a.win, m = (int)a.m;
    const int tid = threadIdx.x, nt = blockDim.x;
    if (a.chunk) {
        for (int i = tid; i < win * hd8; i += nt) a.rows_a[i] = a.ring[i];
        for (int i = tid; i < m * hd8; i += nt) a.rows_a[win * hd8 + i] = a.kv[i];
        __syncthreads();
    }
    const int64_t last = a.start_pos + a.m - 1;
    const int64_t first = (a.start_pos > last - a.win + 1) ? a.start_pos : last - a.win + 1;
    const int nnew = (int)(last - first + 1);  // <= win positions, distinct slots
    for (int i = tid; i < nnew * hd8; i += nt) {
        const int pi = i / hd8, v = i - pi * hd8;
        const int64_t p = first + pi;
        const int slot = (int)(p % a.win);
        a.ring[(int64_t)slot * hd8 + v] = a.kv[(p - a.start_pos) * hd8 + v];
    }
    for (int i = tid; i < m * win; i += nt) {
        const int t = i / win, j = i - t * win;
        a.win_idx[i] = window_index(a.start_pos, a.m, a.win, t, j);
    }
}

struct LatentArgs {
    const uint4* latent;
    const float2* freqs;
    uint4* cache;
    uint32_t* codes;
    uint8_t* scales;
    int hd, rd, G;
    int64_t first_row, ratio;
};

// Group g, dims 8k..8k+7 of the row (k may run past hd/8: such lanes only
// take part in the shuffle).  A rotary pair (2i, 2i+1) never straddles two
// lanes because the rotary part starts at an even dim; a block of 16 dims
// spans lanes k and k^1, so the caller runs whole warps with k0 even.
__device__ __forceinline__ void latent_write_item(const LatentArgs& a, int g, int k) {
    const int hd8 = a.hd / 8;
    const bool live = k < hd8;
    const int64_t row = a.first_row + g;
    const int64_t lpos = row * a.ratio;  // first position of the group
    float x[8];
    if (live) {
        uint4 raw = a.latent[(int64_t)g * hd8 + k];
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
        for (int e = 0; e < 8; e++) x[e] = bf2f(h[e]);
        const int rope0 = a.hd - a.rd;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const int d = 8 * k + e;
            if (d >= rope0) {
                const float2 cs = a.freqs[lpos * (a.rd / 2) + (d - rope0) / 2];
                const float x0 = x[e], x1 = x[e + 1];
                const float y0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
                const float y1 = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
                x[e] = bf2f(f2bf(y0));  // the rotated row is a bf16 buffer
                x[e + 1] = bf2f(f2bf(y1));
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; e++) x[e] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; e++) amax = fmaxf(amax, fabsf(x[e]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, 0.01171875f);  // 6 * 2^-9
    const uint32_t sbyte = f32_to_e4m3_sat(__fdiv_rn(amax, 6.0f));
    const float s = e4m3_to_f32(sbyte);
    if (!live) return;
    float tq[8];
#pragma unroll
    for (int e = 0; e < 8; e++) tq[e] = __fdiv_rn(x[e], s);
    uint32_t packed;
    const uint4 out = e2m1_round8(tq, s, &packed);
    a.cache[row * hd8 + k] = out;
    if (a.codes) a.codes[row * hd8 + k] = packed;
    if (a.scales && (k & 1) == 0) a.scales[row * (a.hd / 16) + k / 2] = (uint8_t)sbyte;
}

}  // namespace ds41
