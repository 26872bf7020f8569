// ds41_window.cu - step 1 of the forward: the sliding-window ring (with the
// window indices of every query) and the compressed latent rows.
//
// metrale_model_arch/attn_v41/forward.rs, AttnV41::forward: "the window ring"
// copies, window_topk_idxs, and the latent branch (rope, fp4_quant with
// LATENT_BLOCK, copy to cache row start_pos / ratio).  The same steps appear
// in attention_any of metrale_model_arch/deepseek_v41_ref/compress.rs.
#include "ds41_step1.cuh"

namespace ds41 {

// One thread per work item (see ring_write_item).
__global__ void __launch_bounds__(256) ring_write_kernel(RingArgs a) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    pdl_trigger();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < a.total()) ring_write_item(a, i);
}

// One CTA per completed group, one lane per 8 dims (whole warps).
__global__ void latent_write_kernel(LatentArgs a) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    pdl_trigger();
    latent_write_item(a, blockIdx.x, threadIdx.x);
}

}  // namespace ds41

using namespace ds41;

extern "C" int64_t ds41_rows_a_len(int64_t m, int64_t win, int64_t start_pos) {
    if (start_pos == 0) return m;
    if (m == 1) return win;
    return win + m;
}

extern "C" int ds41_step_sizes(int64_t m, int64_t start_pos, int64_t win, int64_t ratio,
                               int64_t topk, int64_t* out) {
    const char* name = "ds41_step_sizes";
    DS41_REQUIRE(out, DS41_E_ARG, "%s: out is NULL", name);
    DS41_REQUIRE(m >= 1 && start_pos >= 0 && start_pos + m < (int64_t(1) << 31), DS41_E_RANGE,
                 "%s: m=%lld start_pos=%lld", name, (long long)m, (long long)start_pos);
    DS41_REQUIRE(win >= 1 && ratio >= 1 && topk >= 1, DS41_E_ARG,
                 "%s: win=%lld ratio=%lld topk=%lld", name, (long long)win, (long long)ratio,
                 (long long)topk);
    const int64_t n_c = (start_pos + m) / ratio;  // compress_len
    const int64_t ctopk = n_c == 0 ? 0 : (topk < n_c ? topk : n_c);
    out[0] = ds41_rows_a_len(m, win, start_pos);
    out[1] = n_c;
    out[2] = n_c - start_pos / ratio;  // groups this call completes
    out[3] = ctopk;
    out[4] = win + ctopk;
    return DS41_OK;
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
    RingArgs ra{reinterpret_cast<const uint4*>(kv), reinterpret_cast<uint4*>(ring),
                reinterpret_cast<uint4*>(rows_a), win_idx, m, hd / 8, win, start_pos, chunk};
    const int64_t total = ra.total();
    const int threads = 256;
    return launch_pdl(ring_write_kernel, dim3((unsigned)((total + threads - 1) / threads)),
                      dim3(threads), 0, (cudaStream_t)stream, name, ra);
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
    LatentArgs la{reinterpret_cast<const uint4*>(latent), reinterpret_cast<const float2*>(freqs_cis),
                  reinterpret_cast<uint4*>(cache), reinterpret_cast<uint32_t*>(cache_codes),
                  cache_scales, (int)hd, (int)rd, (int)G, start_pos / ratio, ratio};
    return launch_pdl(latent_write_kernel, dim3((unsigned)G), dim3(threads), 0,
                      (cudaStream_t)stream, name, la);
}
