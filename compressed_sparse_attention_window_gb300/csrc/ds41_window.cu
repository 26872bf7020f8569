// ds41_window.cu - step 1 of the forward: the sliding-window ring (with the
// window indices of every query) and the compressed latent rows.
//
// metrale_model_arch/attn_v41/forward.rs, AttnV41::forward: "the window ring"
// copies, window_topk_idxs, and the latent branch (rope, fp4_quant with
// LATENT_BLOCK, copy to cache row start_pos / ratio).  The same steps appear
// in attention_any of metrale_model_arch/deepseek_v41_ref/compress.rs.
#include "ds41_common.cuh"

namespace ds41 {

// Non-negative remainder.
__device__ __forceinline__ int64_t pmod(int64_t a, int64_t b) {
    const int64_t r = a % b;
    return r < 0 ? r + b : r;
}

// One flat launch over three independent parts:
//   A  win * hd/8 vectors: ring slot j takes the newest of this call's
//      positions q with q mod win == j (if any).  In chunk mode the slot's
//      old contents are first copied to rows_a[j] by the same thread, so the
//      read happens before the overwrite.
//   B  (chunk mode) m * hd/8 vectors: rows_a[win + t] = kv[t].
//   C  m * win window indices.
__global__ void __launch_bounds__(256) ring_write_kernel(const uint4* __restrict__ kv,
                                                         uint4* __restrict__ ring,
                                                         uint4* __restrict__ rows_a,
                                                         int32_t* __restrict__ win_idx, int64_t m,
                                                         int64_t hd8, int64_t win,
                                                         int64_t start_pos, bool chunk) {
    const int64_t nA = win * hd8;
    const int64_t nB = chunk ? m * hd8 : 0;
    const int64_t nC = m * win;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < nA) {
        const int64_t j = i / hd8, v = i % hd8;
        if (chunk) rows_a[j * hd8 + v] = ring[j * hd8 + v];
        const int64_t last = start_pos + m - 1;
        const int64_t q = last - pmod(last - j, win);
        if (q >= start_pos) ring[j * hd8 + v] = kv[(q - start_pos) * hd8 + v];
        return;
    }
    i -= nA;
    if (i < nB) {
        rows_a[win * hd8 + i] = kv[i];
        return;
    }
    i -= nB;
    if (i < nC) {
        const int64_t t = i / win, j = i % win;
        const int64_t p = start_pos + t;
        const int64_t q = p - win + 1 + j;
        int64_t v;
        if (q < 0) v = -1;
        else if (start_pos == 0) v = q;
        else if (m == 1) v = q % win;
        else if (q < start_pos) v = q % win;
        else v = win + (q - start_pos);
        win_idx[i] = (int32_t)v;
    }
}

// One CTA per completed group.  Thread k owns dims 8k..8k+7 of the row; a
// rotary pair (2i, 2i+1) never straddles two threads because the rotary part
// starts at an even dim.  Blocks of 16 dims span two neighbouring lanes.
__global__ void latent_write_kernel(const uint4* __restrict__ latent,
                                    const float2* __restrict__ freqs, uint4* __restrict__ cache,
                                    uint32_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                    int hd, int rd, int64_t first_row, int64_t ratio) {
    const int g = blockIdx.x;
    const int k = threadIdx.x;
    const int hd8 = hd / 8;
    const bool live = k < hd8;
    const int64_t row = first_row + g;
    const int64_t lpos = row * ratio;  // first position of the group
    float x[8];
    if (live) {
        uint4 raw = latent[(int64_t)g * hd8 + k];
        const uint16_t* h = reinterpret_cast<const uint16_t*>(&raw);
#pragma unroll
        for (int e = 0; e < 8; e++) x[e] = bf2f(h[e]);
        const int rope0 = hd - rd;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const int d = 8 * k + e;
            if (d >= rope0) {
                const float2 cs = freqs[lpos * (rd / 2) + (d - rope0) / 2];
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
    uint4 out;
    uint16_t* o = reinterpret_cast<uint16_t*>(&out);
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 8; e++) {
        uint32_t c;
        o[e] = f2bf(fp4_elem(x[e], s, &c));
        packed |= c << (4 * e);
    }
    cache[row * hd8 + k] = out;
    if (codes) codes[row * hd8 + k] = packed;
    if (scales && (k & 1) == 0) scales[row * (hd / 16) + k / 2] = (uint8_t)sbyte;
}

}  // namespace ds41

using namespace ds41;

extern "C" int64_t ds41_rows_a_len(int64_t m, int64_t win, int64_t start_pos) {
    if (start_pos == 0) return m;
    if (m == 1) return win;
    return win + m;
}

extern "C" int ds41_window_ring_write(const ds41_bf16* kv, ds41_bf16* ring, ds41_bf16* rows_a,
                                      int32_t* win_idx, int64_t* n_a, int64_t m, int64_t hd,
                                      int64_t win, int64_t start_pos, ds41_stream_t stream) {
    const char* name = "ds41_window_ring_write";
    DS41_REQUIRE(m >= 1, DS41_E_RANGE, "%s: m=%lld tokens, need at least 1", name, (long long)m);
    DS41_REQUIRE(start_pos >= 0 && start_pos + m < (int64_t(1) << 31), DS41_E_RANGE,
                 "%s: start_pos=%lld out of range", name, (long long)start_pos);
    DS41_REQUIRE(win >= 1 && win <= (int64_t(1) << 20), DS41_E_ARG, "%s: win=%lld", name,
                 (long long)win);
    DS41_REQUIRE(hd >= 8 && hd % 8 == 0, DS41_E_ARG, "%s: hd=%lld must be a multiple of 8", name,
                 (long long)hd);
    const bool chunk = start_pos > 0 && m > 1;
    DS41_REQUIRE(kv && ring && win_idx, DS41_E_ARG, "%s: kv, ring and win_idx must be non-null",
                 name);
    DS41_REQUIRE(!chunk || rows_a, DS41_E_ARG,
                 "%s: rows_a is required for a chunk of m > 1 tokens past position 0", name);
    DS41_REQUIRE(aligned16(kv) && aligned16(ring) && (!chunk || aligned16(rows_a)), DS41_E_ARG,
                 "%s: kv/ring/rows_a must be 16-byte aligned", name);
    if (n_a) *n_a = ds41_rows_a_len(m, win, start_pos);
    const int64_t hd8 = hd / 8;
    const int64_t total = win * hd8 + (chunk ? m * hd8 : 0) + m * win;
    const int threads = 256;
    ring_write_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0,
                        (cudaStream_t)stream>>>(
        reinterpret_cast<const uint4*>(kv), reinterpret_cast<uint4*>(ring),
        reinterpret_cast<uint4*>(rows_a), win_idx, m, hd8, win, start_pos, chunk);
    return launch_check(name);
}

extern "C" int ds41_compress_latent_write(const ds41_bf16* latent, const float* freqs_cis,
                                          int64_t max_pos, ds41_bf16* cache, int64_t cache_rows,
                                          uint8_t* cache_codes, uint8_t* cache_scales, int64_t G,
                                          int64_t hd, int64_t rd, int64_t ratio,
                                          int64_t start_pos, int64_t m, ds41_stream_t stream) {
    const char* name = "ds41_compress_latent_write";
    DS41_REQUIRE(ratio >= 1, DS41_E_ARG, "%s: ratio=%lld", name, (long long)ratio);
    DS41_REQUIRE(m >= 1 && start_pos >= 0, DS41_E_RANGE, "%s: m=%lld start_pos=%lld", name,
                 (long long)m, (long long)start_pos);
    const int64_t want = (start_pos + m) / ratio - start_pos / ratio;
    DS41_REQUIRE(G == want, DS41_E_ARG,
                 "%s: G=%lld but %lld tokens at %lld complete %lld groups of %lld", name,
                 (long long)G, (long long)m, (long long)start_pos, (long long)want,
                 (long long)ratio);
    if (G == 0) return DS41_OK;
    DS41_REQUIRE(hd >= 16 && hd % 16 == 0 && hd <= 8192, DS41_E_ARG,
                 "%s: hd=%lld must be a multiple of 16 (<= 8192)", name, (long long)hd);
    DS41_REQUIRE(rd > 0 && rd % 2 == 0 && rd <= hd, DS41_E_ARG, "%s: rd=%lld", name,
                 (long long)rd);
    DS41_REQUIRE((start_pos + m) / ratio <= cache_rows, DS41_E_RANGE,
                 "%s: cache holds %lld rows, need %lld", name, (long long)cache_rows,
                 (long long)((start_pos + m) / ratio));
    DS41_REQUIRE(start_pos + m <= max_pos, DS41_E_RANGE, "%s: RoPE table has %lld rows, need %lld",
                 name, (long long)max_pos, (long long)(start_pos + m));
    DS41_REQUIRE(latent && freqs_cis && cache, DS41_E_ARG,
                 "%s: latent, freqs_cis and cache must be non-null", name);
    DS41_REQUIRE(aligned16(latent) && aligned16(cache) && aligned16(freqs_cis), DS41_E_ARG,
                 "%s: pointers must be 16-byte aligned", name);
    DS41_REQUIRE(!cache_codes || (reinterpret_cast<uintptr_t>(cache_codes) & 3u) == 0, DS41_E_ARG,
                 "%s: cache_codes must be 4-byte aligned", name);
    const int threads = (int)(((hd / 8) + 31) / 32 * 32);
    latent_write_kernel<<<(unsigned)G, threads, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const uint4*>(latent), reinterpret_cast<const float2*>(freqs_cis),
        reinterpret_cast<uint4*>(cache), reinterpret_cast<uint32_t*>(cache_codes), cache_scales,
        (int)hd, (int)rd, start_pos / ratio, ratio);
    return launch_check(name);
}
