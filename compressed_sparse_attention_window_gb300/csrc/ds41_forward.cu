// ds41_forward.cu - the whole step of one layer's compressed sparse attention
// forward in one call: window ring + window indices, latent write, indexer
// scores + top-k + merge, sparse attention with the sink.
//
// metrale_model_arch/attn_v41/forward.rs, AttnV41::forward runs these steps
// in this order for m tokens at start_pos; metrale_model_arch/
// deepseek_v41_ref/compress.rs, attention_any does the same on the CPU.
//
// Few-token calls (decode) take three launches: (1) one grid whose CTAs
// compute the indexer scores while its last CTA writes the ring, the window
// indices and the latent rows (these are independent of each other); (2)
// the top-k + merge; (3) the cluster attention.  (2) and (3) are launched
// with programmatic stream serialization, so each starts while its
// predecessor finishes and waits on the device (griddepcontrol) only where it
// reads the predecessor's output.  Larger calls run the four entry points in
// sequence.
#include "ds41_internal.cuh"
#include "ds41_step1.cuh"
#include "ds41_tc.cuh"

using namespace ds41;

static int64_t ctopk_of(int64_t topk, int64_t n_c) { return n_c == 0 ? 0 : (topk < n_c ? topk : n_c); }

static bool use_fused(int64_t m, int64_t start_pos, int64_t nh, int64_t hd, int64_t win,
                      int64_t ratio, int64_t topk, int64_t Hi, int64_t Di) {
    const int64_t n_c = (start_pos + m) / ratio;
    if (n_c < 1) return false;
    const int64_t K = win + ctopk_of(topk, n_c);
    // the fused front feeds the few-token cluster attention, or the generic
    // attention when its CTAs select their rows themselves
    return front_fusable(m, Hi, Di, n_c) &&
           (attn_is_cluster_path(m, nh, hd, K) || attn_topk_fusable(m, nh, hd, K, n_c));
}

extern "C" size_t ds41_csa_workspace_bytes(int64_t m, int64_t start_pos, int64_t nh, int64_t hd,
                                           int64_t win, int64_t ratio, int64_t topk, int64_t Hi,
                                           int64_t Di) {
    if (m < 1 || ratio < 1 || win < 1) return 0;
    const int64_t n_c = (start_pos + m) / ratio;
    const int64_t K = win + ctopk_of(topk, n_c);
    size_t a = 0;
    if (n_c > 0) {
        a = use_fused(m, start_pos, nh, hd, win, ratio, topk, Hi, Di)
                ? front_scores_bytes(m, n_c)
                : ds41_indexer_workspace_bytes(m, Hi, Di, n_c, 0);
    }
    const size_t b = attn_ws_bytes(m, nh, hd, K);
    return a > b ? a : b;
}

extern "C" int ds41_csa_forward(const ds41_bf16* q, const ds41_bf16* kv, ds41_bf16* ring,
                                ds41_bf16* rows_a, const ds41_bf16* latent,
                                const float* freqs_cis, int64_t max_pos, ds41_bf16* cache,
                                int64_t cache_rows, const ds41_bf16* q_idx,
                                const ds41_bf16* k_idx, const float* w, const float* sink,
                                float scale, int32_t* win_idx, int32_t* idx, ds41_bf16* o,
                                float* lse, int64_t m, int64_t start_pos, int64_t nh, int64_t hd,
                                int64_t rd, int64_t win, int64_t ratio, int64_t topk, int64_t Hi,
                                int64_t Di, void* ws, size_t ws_bytes, ds41_stream_t stream) {
    const char* name = "ds41_csa_forward";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 31), DS41_E_RANGE, "%s: m=%lld", name,
                 (long long)m);
    DS41_REQUIRE(start_pos >= 0 && start_pos + m < (int64_t(1) << 31), DS41_E_RANGE,
                 "%s: start_pos=%lld", name, (long long)start_pos);
    DS41_REQUIRE(ratio >= 1 && win >= 1 && topk >= 1, DS41_E_ARG,
                 "%s: ratio=%lld win=%lld topk=%lld", name, (long long)ratio, (long long)win,
                 (long long)topk);
    const int64_t n_c = (start_pos + m) / ratio;
    const int64_t G = n_c - start_pos / ratio;
    const int64_t ctopk = ctopk_of(topk, n_c);
    const int64_t K = win + ctopk;
    const int64_t n_a = ds41_rows_a_len(m, win, start_pos);
    const size_t need = ds41_csa_workspace_bytes(m, start_pos, nh, hd, win, ratio, topk, Hi, Di);
    DS41_REQUIRE(need == 0 || (ws && ws_bytes >= need), DS41_E_WORKSPACE,
                 "%s: workspace of %zu bytes needed, %zu given", name, need, ws ? ws_bytes : 0);
    cudaStream_t st = (cudaStream_t)stream;
    const bool chunk = start_pos > 0 && m > 1;
    const ds41_bf16* rows_a_used = start_pos == 0 ? kv : (m == 1 ? ring : rows_a);

    if (!use_fused(m, start_pos, nh, hd, win, ratio, topk, Hi, Di)) {
        int rc = ds41_window_ring_write(kv, ring, rows_a, win_idx, nullptr, m, hd, win, start_pos,
                                        stream);
        if (rc) return rc;
        if (G > 0) {
            rc = ds41_compress_latent_write(latent, freqs_cis, max_pos, cache, cache_rows, nullptr,
                                            nullptr, G, hd, rd, ratio, start_pos, m, stream);
            if (rc) return rc;
        }
        const int32_t* att_idx = win_idx;
        if (n_c > 0) {
            rc = ds41_indexer_topk(q_idx, k_idx, w, win_idx, idx, nullptr, m, Hi, Di, n_c, win,
                                   ratio, start_pos, topk, n_a, ws, ws_bytes, stream);
            if (rc) return rc;
            att_idx = idx;
        }
        return ds41_sparse_attn_sink_fwd(q, rows_a_used, n_a, n_c ? cache : nullptr, n_c, att_idx,
                                         K, sink, scale, o, lse, m, nh, hd, ws, ws_bytes, stream);
    }

    // ---- few-token fused path: the same checks the separate entry points make
    DS41_REQUIRE(hd >= 64 && hd <= 512 && (hd & (hd - 1)) == 0, DS41_E_ARG,
                 "%s: hd=%lld must be 64, 128, 256 or 512", name, (long long)hd);
    DS41_REQUIRE(nh >= 1 && rd > 0 && rd % 2 == 0 && rd <= hd, DS41_E_ARG, "%s: nh=%lld rd=%lld",
                 name, (long long)nh, (long long)rd);
    DS41_REQUIRE(n_c <= cache_rows, DS41_E_RANGE, "%s: cache holds %lld rows, need %lld", name,
                 (long long)cache_rows, (long long)n_c);
    DS41_REQUIRE(G == 0 || start_pos + m <= max_pos, DS41_E_RANGE,
                 "%s: RoPE table has %lld rows, need %lld", name, (long long)max_pos,
                 (long long)(start_pos + m));
    DS41_REQUIRE(q && kv && ring && cache && q_idx && k_idx && w && sink && win_idx && idx && o &&
                     (G == 0 || (latent && freqs_cis)) && (!chunk || rows_a),
                 DS41_E_ARG, "%s: null tensor pointer", name);
    DS41_REQUIRE(aligned16(q) && aligned16(kv) && aligned16(ring) && aligned16(cache) &&
                     aligned16(q_idx) && aligned16(k_idx) && aligned16(o) &&
                     (G == 0 || (aligned16(latent) && aligned16(freqs_cis))) &&
                     (!chunk || aligned16(rows_a)) && aligned16(ws),
                 DS41_E_ARG, "%s: pointers must be 16-byte aligned", name);
    RingArgs ra{reinterpret_cast<const uint4*>(kv), reinterpret_cast<uint4*>(ring),
                reinterpret_cast<uint4*>(rows_a), win_idx, m, hd / 8, win, start_pos, chunk};
    LatentArgs la{reinterpret_cast<const uint4*>(latent),
                  reinterpret_cast<const float2*>(freqs_cis), reinterpret_cast<uint4*>(cache),
                  nullptr, nullptr, (int)hd, (int)rd, (int)G, start_pos / ratio, ratio};
    uint16_t* scores = static_cast<uint16_t*>(ws);
    int rc = launch_front(q_idx, k_idx, w, scores, m, Hi, Di, n_c, ratio, start_pos, ra, la, st);
    if (rc) return rc;
    if (attn_topk_fusable(m, nh, hd, K, n_c)) {
        // the attention clusters select their rows from the scores themselves
        const DecTopk tk{scores, win_idx, idx, n_c, ratio, start_pos, n_a, (int)win, (int)ctopk, m};
        return attn_run(q, rows_a_used, n_a, cache, n_c, idx, K, sink, scale, o, lse, m, nh, hd,
                        nullptr, 0, true, st, name, &tk);
    }
    rc = launch_topk(scores, win_idx, idx, m, n_c, win, ctopk, ratio, start_pos, n_a, true, st);
    if (rc) return rc;
    return attn_run(q, rows_a_used, n_a, cache, n_c, idx, K, sink, scale, o, lse, m, nh, hd,
                    nullptr, 0, true, st, name);
}

// ---------------------------------------------------------------------------
// The step on packed fp4 caches: the indexer keys as mxf4 (e2m1 codes + e8m0
// block-32 scales) read by the block-scaled tensor-core scores, and the latent
// rows also written as e2m1 codes + e4m3 block-16 scales.
// ---------------------------------------------------------------------------
static bool fp4_fused(int64_t m, int64_t nh, int64_t hd, int64_t K, int64_t n_c) {
    return n_c >= 1 && m <= 8 && attn_is_cluster_path(m, nh, hd, K);
}

extern "C" size_t ds41_csa_fp4_workspace_bytes(int64_t m, int64_t start_pos, int64_t nh,
                                               int64_t hd, int64_t win, int64_t ratio,
                                               int64_t topk) {
    if (m < 1 || ratio < 1 || win < 1 || start_pos < 0) return 0;
    const int64_t n_c = (start_pos + m) / ratio;
    const int64_t K = win + ctopk_of(topk, n_c);
    const size_t a = n_c > 0 ? ds41_indexer_mxf4_workspace_bytes(m, n_c, 0) : 0;
    const size_t b = fp4_fused(m, nh, hd, K, n_c) ? 0 : attn_ws_bytes(m, nh, hd, K);
    return a > b ? a : b;
}

extern "C" int ds41_csa_forward_fp4(const ds41_bf16* q, const ds41_bf16* kv, ds41_bf16* ring,
                                    ds41_bf16* rows_a, const ds41_bf16* latent,
                                    const float* freqs_cis, int64_t max_pos, ds41_bf16* cache,
                                    uint8_t* cache_codes, uint8_t* cache_scales,
                                    int64_t cache_rows, const ds41_bf16* q_idx,
                                    const uint8_t* k_codes, const uint8_t* k_scales,
                                    const float* w, const float* sink, float scale,
                                    int32_t* win_idx, int32_t* idx, ds41_bf16* o, float* lse,
                                    int64_t m, int64_t start_pos, int64_t nh, int64_t hd,
                                    int64_t rd, int64_t win, int64_t ratio, int64_t topk,
                                    int64_t Hi, int64_t Di, void* ws, size_t ws_bytes,
                                    ds41_stream_t stream) {
    const char* name = "ds41_csa_forward_fp4";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 25), DS41_E_RANGE, "%s: m=%lld", name,
                 (long long)m);
    DS41_REQUIRE(start_pos >= 0 && start_pos + m < (int64_t(1) << 31), DS41_E_RANGE,
                 "%s: start_pos=%lld", name, (long long)start_pos);
    DS41_REQUIRE(ratio >= 1 && win >= 1 && topk >= 1, DS41_E_ARG,
                 "%s: ratio=%lld win=%lld topk=%lld", name, (long long)ratio, (long long)win,
                 (long long)topk);
    DS41_REQUIRE(indexer_mxf4_supported(Hi, Di), DS41_E_ARG,
                 "%s: Hi=%lld Di=%lld; the packed-key path takes 64 heads of dim 128", name,
                 (long long)Hi, (long long)Di);
    const int64_t n_c = (start_pos + m) / ratio;
    const int64_t G = n_c - start_pos / ratio;
    const int64_t ctopk = ctopk_of(topk, n_c);
    const int64_t K = win + ctopk;
    const int64_t n_a = ds41_rows_a_len(m, win, start_pos);
    const size_t need = ds41_csa_fp4_workspace_bytes(m, start_pos, nh, hd, win, ratio, topk);
    DS41_REQUIRE(need == 0 || (ws && ws_bytes >= need), DS41_E_WORKSPACE,
                 "%s: workspace of %zu bytes needed, %zu given", name, need, ws ? ws_bytes : 0);
    DS41_REQUIRE((cache_codes == nullptr) == (cache_scales == nullptr), DS41_E_ARG,
                 "%s: cache_codes and cache_scales go together", name);
    cudaStream_t st = (cudaStream_t)stream;
    const bool chunk = start_pos > 0 && m > 1;
    const ds41_bf16* rows_a_used = start_pos == 0 ? kv : (m == 1 ? ring : rows_a);
    uint8_t* wsb = static_cast<uint8_t*>(ws);

    if (!fp4_fused(m, nh, hd, K, n_c)) {
        int rc = ds41_window_ring_write(kv, ring, rows_a, win_idx, nullptr, m, hd, win, start_pos,
                                        stream);
        if (rc) return rc;
        if (G > 0) {
            rc = ds41_compress_latent_write(latent, freqs_cis, max_pos, cache, cache_rows,
                                            cache_codes, cache_scales, G, hd, rd, ratio,
                                            start_pos, m, stream);
            if (rc) return rc;
        }
        const int32_t* att_idx = win_idx;
        if (n_c > 0) {
            rc = ds41_indexer_topk_mxf4(q_idx, k_codes, k_scales, w, win_idx, idx, nullptr, m, Hi,
                                        Di, n_c, win, ratio, start_pos, topk, n_a, ws, ws_bytes,
                                        stream);
            if (rc) return rc;
            att_idx = idx;
        }
        return ds41_sparse_attn_sink_fwd(q, rows_a_used, n_a, n_c ? cache : nullptr, n_c, att_idx,
                                         K, sink, scale, o, lse, m, nh, hd, ws, ws_bytes, stream);
    }

    // ---- few-token fused path: the same checks the separate entry points make
    DS41_REQUIRE(hd >= 64 && hd <= 512 && (hd & (hd - 1)) == 0 && hd % 16 == 0, DS41_E_ARG,
                 "%s: hd=%lld must be 64, 128, 256 or 512", name, (long long)hd);
    DS41_REQUIRE(nh >= 1 && rd > 0 && rd % 2 == 0 && rd <= hd, DS41_E_ARG, "%s: nh=%lld rd=%lld",
                 name, (long long)nh, (long long)rd);
    DS41_REQUIRE(n_c <= cache_rows, DS41_E_RANGE, "%s: cache holds %lld rows, need %lld", name,
                 (long long)cache_rows, (long long)n_c);
    DS41_REQUIRE(G == 0 || start_pos + m <= max_pos, DS41_E_RANGE,
                 "%s: RoPE table has %lld rows, need %lld", name, (long long)max_pos,
                 (long long)(start_pos + m));
    DS41_REQUIRE(q && kv && ring && cache && q_idx && k_codes && k_scales && w && sink &&
                     win_idx && idx && o && (G == 0 || (latent && freqs_cis)) && (!chunk || rows_a),
                 DS41_E_ARG, "%s: null tensor pointer", name);
    DS41_REQUIRE(aligned16(q) && aligned16(kv) && aligned16(ring) && aligned16(cache) &&
                     aligned16(q_idx) && aligned16(k_codes) && aligned16(k_scales) &&
                     aligned16(w) && aligned16(o) &&
                     (!cache_codes || (aligned16(cache_codes) && aligned16(cache_scales))) &&
                     (G == 0 || (aligned16(latent) && aligned16(freqs_cis))) &&
                     (!chunk || aligned16(rows_a)) && aligned16(ws),
                 DS41_E_ARG, "%s: pointers must be 16-byte aligned", name);
    RingArgs ra{reinterpret_cast<const uint4*>(kv), reinterpret_cast<uint4*>(ring),
                reinterpret_cast<uint4*>(rows_a), win_idx, m, hd / 8, win, start_pos, chunk};
    LatentArgs la{reinterpret_cast<const uint4*>(latent),
                  reinterpret_cast<const float2*>(freqs_cis), reinterpret_cast<uint4*>(cache),
                  reinterpret_cast<uint32_t*>(cache_codes), cache_scales, (int)hd, (int)rd, (int)G,
                  start_pos / ratio, ratio};
    uint16_t* scores = reinterpret_cast<uint16_t*>(wsb);
    unsigned int* status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    rc = indexer_mxf4_launch(q_idx, k_codes, k_scales, w, scores, m, n_c, ratio, start_pos, false,
                             status, device_sm_count(), st, &ra, &la);
    if (rc) return rc;
    // with the packed latent rows given, the attention gathers them packed
    const PackedRows pk{cache_codes, cache_scales};
    const PackedRows* pkp = (cache_codes && hd == 512) ? &pk : nullptr;
    if (attn_topk_fusable(m, nh, hd, K, n_c)) {
        const DecTopk tk{scores, win_idx, idx, n_c, ratio, start_pos, n_a, (int)win, (int)ctopk, m};
        return attn_run(q, rows_a_used, n_a, cache, n_c, idx, K, sink, scale, o, lse, m, nh, hd,
                        nullptr, 0, true, st, name, &tk, pkp);
    }
    rc = launch_topk(scores, win_idx, idx, m, n_c, win, ctopk, ratio, start_pos, n_a, true, st);
    if (rc) return rc;
    return attn_run(q, rows_a_used, n_a, cache, n_c, idx, K, sink, scale, o, lse, m, nh, hd,
                    nullptr, 0, true, st, name, nullptr, pkp);
}

// The step with its per-step inputs and its output in host memory: one copy
// per input into the caller's device buffers, the step, and one copy of o
// back, all on the caller's stream.
// ---------------------------------------------------------------------------
// Copies between host buffers and device buffers for the host entry points.
// When the host side is device-mapped page-locked memory (cudaHostAlloc,
// cudaHostRegister) and the copy is small, a kernel moves the bytes with
// 16-byte loads and stores through the mapping: for the tens of KB of a
// decode step this finishes sooner than a copy-engine transfer, whose
// start-up dominates at that size.  Everything else goes through
// cudaMemcpyAsync.
// ---------------------------------------------------------------------------
__global__ void copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16) {
    // launched with programmatic stream serialization: the kernel after this
    // one may start launching now, and this one waits for the kernel before
    // it (whose output it may read, or whose inputs it may overwrite) before
    // its first memory access
    pdl_trigger();
    pdl_wait();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

constexpr size_t kKernelCopyMax = size_t(4) << 20;  // larger copies use the copy engines

// The device address of `bytes` bytes of host memory when it is page-locked
// memory of the current device's context, mapped into its address space, and
// the span is at most kKernelCopyMax bytes, a multiple of 16; else NULL.
static void* mapped_small(const void* host, size_t bytes) {
    cudaPointerAttributes a;
    int dev = -1;
    if (bytes == 0 || bytes > kKernelCopyMax || bytes % 16 != 0 || cudaGetDevice(&dev) != cudaSuccess)
        return nullptr;
    if (cudaPointerGetAttributes(&a, host) == cudaSuccess && a.type == cudaMemoryTypeHost &&
        a.device == dev)
        return a.devicePointer;
    cudaGetLastError();  // not registered with CUDA: clear the query's error
    return nullptr;
}

static int host_copy(void* dst, const void* src, size_t bytes, bool h2d, cudaStream_t st,
                     const char* what) {
    if (bytes == 0) return DS41_OK;
    void* mapped = mapped_small(h2d ? src : dst, bytes);
    const void* s = h2d ? mapped : src;
    void* d = h2d ? dst : mapped;
    if (mapped && ((reinterpret_cast<uintptr_t>(s) | reinterpret_cast<uintptr_t>(d)) & 15u) == 0) {
        const int64_t n16 = (int64_t)(bytes / 16);
        const int64_t cap = 4 * (int64_t)device_sm_count();
        const int64_t blocks = (n16 + 255) / 256;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(blocks < cap ? blocks : cap));
        cfg.blockDim = dim3(256);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const int rc = cuda_check(cudaLaunchKernelEx(&cfg, copy16_kernel,
                                                     static_cast<const uint4*>(s),
                                                     static_cast<uint4*>(d), n16),
                                  what);
        if (rc) return rc;
        return launch_check(what);
    }
    return cuda_check(cudaMemcpyAsync(dst, src, bytes,
                                      h2d ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost, st),
                      what);
}

// Where the step writes o for a host entry point: the device address of h_o
// when it is mapped page-locked memory (mapped_small) and the step has few
// tokens, so that the attention's stores go straight over the host link
// (measured on the decode step: 20.6 -> 18.6 us a step against a copy kernel
// after it); NULL otherwise (the step writes the device buffer o, which is
// then copied into h_o).
constexpr int64_t kDirectOutTokens = 16;
static ds41_bf16* direct_out(ds41_bf16* h_o, int64_t m, int64_t nh, int64_t hd) {
    if (m > kDirectOutTokens) return nullptr;
    void* d = mapped_small(h_o, (size_t)(m * nh * hd) * 2);
    return (reinterpret_cast<uintptr_t>(d) & 15u) == 0 ? static_cast<ds41_bf16*>(d) : nullptr;
}

extern "C" int ds41_csa_forward_host(
    const ds41_bf16* h_q, const ds41_bf16* h_kv, const ds41_bf16* h_latent, const ds41_bf16* h_q_idx,
    const float* h_w, ds41_bf16* h_o, ds41_bf16* q, ds41_bf16* kv, ds41_bf16* ring, ds41_bf16* rows_a,
    ds41_bf16* latent, const float* freqs_cis, int64_t max_pos, ds41_bf16* cache, int64_t cache_rows,
    ds41_bf16* q_idx, const ds41_bf16* k_idx, float* w, const float* sink, float scale,
    int32_t* win_idx, int32_t* idx, ds41_bf16* o, float* lse, int64_t m, int64_t start_pos,
    int64_t nh, int64_t hd, int64_t rd, int64_t win, int64_t ratio, int64_t topk, int64_t Hi,
    int64_t Di, void* ws, size_t ws_bytes, ds41_stream_t stream) {
    const char* name = "ds41_csa_forward_host";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 31) && start_pos >= 0 && ratio >= 1 && nh >= 1 &&
                     hd >= 1 && Hi >= 1 && Di >= 1,
                 DS41_E_ARG, "%s: m=%lld start_pos=%lld ratio=%lld", name, (long long)m,
                 (long long)start_pos, (long long)ratio);
    const int64_t G = (start_pos + m) / ratio - start_pos / ratio;
    DS41_REQUIRE(h_q && h_kv && h_q_idx && h_w && h_o && q && kv && q_idx && w && o &&
                     (G == 0 || (h_latent && latent)),
                 DS41_E_ARG, "%s: null pointer", name);
    cudaStream_t st = (cudaStream_t)stream;
    struct Copy {
        void* dst;
        const void* src;
        size_t bytes;
    };
    const Copy in[5] = {{q, h_q, (size_t)(m * nh * hd) * 2},
                        {kv, h_kv, (size_t)(m * hd) * 2},
                        {latent, h_latent, (size_t)(G * hd) * 2},
                        {q_idx, h_q_idx, (size_t)(m * Hi * Di) * 2},
                        {w, h_w, (size_t)(m * Hi) * 4}};
    for (const Copy& c : in) {
        if (c.bytes == 0) continue;
        const int rc = host_copy(c.dst, c.src, c.bytes, true, st, "ds41_csa_forward_host: input copy");
        if (rc) return rc;
    }
    // o straight into h_o when the mapping allows it (see direct_out)
    ds41_bf16* d_o = direct_out(h_o, m, nh, hd);
    const int rc = ds41_csa_forward(q, kv, ring, rows_a, latent, freqs_cis, max_pos, cache, cache_rows,
                                    q_idx, k_idx, w, sink, scale, win_idx, idx, d_o ? d_o : o, lse,
                                    m, start_pos, nh, hd, rd, win, ratio, topk, Hi, Di, ws, ws_bytes,
                                    stream);
    if (rc || d_o) return rc;
    return host_copy(h_o, o, (size_t)(m * nh * hd) * 2, false, st, "ds41_csa_forward_host: output copy");
}

extern "C" size_t ds41_step_inputs_bytes(int64_t m, int64_t start_pos, int64_t nh, int64_t hd,
                                         int64_t ratio, int64_t Hi, int64_t Di) {
    if (m < 1 || start_pos < 0 || ratio < 1) return 0;
    const int64_t G = (start_pos + m) / ratio - start_pos / ratio;
    return (size_t)(m * nh * hd + m * hd + G * hd + m * Hi * Di) * 2 + (size_t)(m * Hi) * 4;
}

// The same with the step's inputs in one block on each side: one copy in.
extern "C" int ds41_csa_forward_host_packed(
    const void* h_in, void* d_in, ds41_bf16* h_o, ds41_bf16* ring, ds41_bf16* rows_a,
    const float* freqs_cis, int64_t max_pos, ds41_bf16* cache, int64_t cache_rows,
    const ds41_bf16* k_idx, const float* sink, float scale, int32_t* win_idx, int32_t* idx,
    ds41_bf16* o, float* lse, int64_t m, int64_t start_pos, int64_t nh, int64_t hd, int64_t rd,
    int64_t win, int64_t ratio, int64_t topk, int64_t Hi, int64_t Di, void* ws, size_t ws_bytes,
    ds41_stream_t stream) {
    const char* name = "ds41_csa_forward_host_packed";
    const size_t bytes = ds41_step_inputs_bytes(m, start_pos, nh, hd, ratio, Hi, Di);
    DS41_REQUIRE(bytes > 0 && h_in && d_in && h_o && o, DS41_E_ARG, "%s: m=%lld, null pointer",
                 name, (long long)m);
    const int64_t G = (start_pos + m) / ratio - start_pos / ratio;
    char* d = static_cast<char*>(d_in);
    ds41_bf16* q = reinterpret_cast<ds41_bf16*>(d);
    ds41_bf16* kv = q + m * nh * hd;
    ds41_bf16* latent = kv + m * hd;
    ds41_bf16* q_idx = latent + G * hd;
    float* w = reinterpret_cast<float*>(q_idx + m * Hi * Di);
    cudaStream_t st = (cudaStream_t)stream;
    int rc = host_copy(d_in, h_in, bytes, true, st, "ds41_csa_forward_host_packed: input copy");
    if (rc) return rc;
    ds41_bf16* d_o = direct_out(h_o, m, nh, hd);  // o straight into h_o (see direct_out)
    rc = ds41_csa_forward(q, kv, ring, rows_a, G > 0 ? latent : nullptr, freqs_cis, max_pos, cache,
                          cache_rows, q_idx, k_idx, w, sink, scale, win_idx, idx, d_o ? d_o : o, lse,
                          m, start_pos, nh, hd, rd, win, ratio, topk, Hi, Di, ws, ws_bytes, stream);
    if (rc || d_o) return rc;
    return host_copy(h_o, o, (size_t)(m * nh * hd) * 2, false, st,
                     "ds41_csa_forward_host_packed: output copy");
}

// ---------------------------------------------------------------------------
// A prepared host step: the packed host step recorded once into a CUDA graph
// ---------------------------------------------------------------------------
struct ds41_host_step {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" int ds41_host_step_create(
    ds41_host_step** out, const void* h_in, void* d_in, ds41_bf16* h_o, ds41_bf16* ring,
    ds41_bf16* rows_a, const float* freqs_cis, int64_t max_pos, ds41_bf16* cache,
    int64_t cache_rows, const ds41_bf16* k_idx, const float* sink, float scale, int32_t* win_idx,
    int32_t* idx, ds41_bf16* o, float* lse, int64_t m, int64_t start_pos, int64_t nh, int64_t hd,
    int64_t rd, int64_t win, int64_t ratio, int64_t topk, int64_t Hi, int64_t Di, void* ws,
    size_t ws_bytes) {
    const char* name = "ds41_host_step_create";
    DS41_REQUIRE(out, DS41_E_ARG, "%s: out is NULL", name);
    *out = nullptr;
    DS41_REQUIRE(ds41_step_inputs_bytes(m, start_pos, nh, hd, ratio, Hi, Di) > 0 && h_in && d_in &&
                     h_o && o,
                 DS41_E_ARG, "%s: m=%lld, null pointer", name, (long long)m);
    // resources the step looks up on first use, outside the recording
    unsigned int* status = nullptr;
    int rc = status_word(&status);
    if (rc) return rc;
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    if ((rc = tc::get_encode(&enc))) return rc;
    cudaStream_t cs;
    if ((rc = cuda_check(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking),
                         "ds41_host_step_create: stream")))
        return rc;
    rc = cuda_check(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal),
                    "ds41_host_step_create: begin capture");
    if (rc) {
        cudaStreamDestroy(cs);
        return rc;
    }
    const int step_rc = ds41_csa_forward_host_packed(
        h_in, d_in, h_o, ring, rows_a, freqs_cis, max_pos, cache, cache_rows, k_idx, sink, scale,
        win_idx, idx, o, lse, m, start_pos, nh, hd, rd, win, ratio, topk, Hi, Di, ws, ws_bytes,
        (ds41_stream_t)cs);
    cudaGraph_t g = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (step_rc || ce != cudaSuccess || !g) {
        if (g) cudaGraphDestroy(g);
        if (step_rc) return step_rc;  // its message stands
        cudaGetLastError();
        return fail(DS41_E_CUDA, "%s: capture failed: %s", name, cudaGetErrorString(ce));
    }
    cudaGraphExec_t ex = nullptr;
    rc = cuda_check(cudaGraphInstantiate(&ex, g, 0), "ds41_host_step_create: instantiate");
    if (rc) {
        cudaGraphDestroy(g);
        return rc;
    }
    *out = new ds41_host_step{g, ex};
    return DS41_OK;
}

extern "C" int ds41_host_step_launch(ds41_host_step* h, ds41_stream_t stream) {
    DS41_REQUIRE(h, DS41_E_ARG, "ds41_host_step_launch: handle is NULL");
    return cuda_check(cudaGraphLaunch(h->exec, (cudaStream_t)stream), "ds41_host_step_launch");
}

extern "C" int ds41_host_step_destroy(ds41_host_step* h) {
    if (!h) return DS41_OK;
    cudaGraphExecDestroy(h->exec);
    cudaGraphDestroy(h->graph);
    delete h;
    return DS41_OK;
}

// ---------------------------------------------------------------------------
// A layer that reuses the last source layer's compressed rows and picks
// ---------------------------------------------------------------------------
// idx row t = the window indices of t, then the shared picks of t.
__global__ void merge_shared_kernel(const int32_t* win_idx, const int32_t* cidx, int32_t* idx,
                                    int64_t m, int win, int ctopk) {
    pdl_wait();     // the kernel before may still be running (programmatic launch)
    pdl_trigger();
    const int K = win + ctopk;
    const int64_t total = m * K;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total;
         k += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = k / K;
        const int j = (int)(k % K);
        idx[k] = j < win ? win_idx[t * win + j] : cidx[t * ctopk + (j - win)];
    }
}

extern "C" int ds41_csa_forward_reuse(const ds41_bf16* q, const ds41_bf16* kv, ds41_bf16* ring,
                                      ds41_bf16* rows_a, const ds41_bf16* cache,
                                      const int32_t* cidx, int64_t ctopk, const float* sink,
                                      float scale, int32_t* win_idx, int32_t* idx, ds41_bf16* o,
                                      float* lse, int64_t m, int64_t start_pos, int64_t nh,
                                      int64_t hd, int64_t win, int64_t ratio, void* ws,
                                      size_t ws_bytes, ds41_stream_t stream) {
    const char* name = "ds41_csa_forward_reuse";
    DS41_REQUIRE(m >= 1 && m < (int64_t(1) << 31), DS41_E_RANGE, "%s: m=%lld", name,
                 (long long)m);
    DS41_REQUIRE(start_pos >= 0 && start_pos + m < (int64_t(1) << 31), DS41_E_RANGE,
                 "%s: start_pos=%lld", name, (long long)start_pos);
    DS41_REQUIRE(ratio >= 1 && win >= 1 && win <= (int64_t(1) << 20), DS41_E_ARG,
                 "%s: ratio=%lld win=%lld", name, (long long)ratio, (long long)win);
    const int64_t n_c = (start_pos + m) / ratio;
    DS41_REQUIRE(ctopk >= 0 && ctopk <= n_c && ctopk <= (int64_t(1) << 20), DS41_E_ARG,
                 "%s: ctopk=%lld with %lld compressed rows", name, (long long)ctopk,
                 (long long)n_c);
    DS41_REQUIRE(ctopk == 0 || (cidx && idx && cache), DS41_E_ARG,
                 "%s: cidx, idx and cache are required when ctopk > 0", name);
    // the attention's own checks, made before the ring write is enqueued
    DS41_REQUIRE(nh >= 1 && nh <= 65535 && (hd == 64 || hd == 128 || hd == 256 || hd == 512),
                 DS41_E_ARG, "%s: nh=%lld hd=%lld (hd must be 64, 128, 256 or 512)", name,
                 (long long)nh, (long long)hd);
    DS41_REQUIRE(q && sink && o && aligned16(q) && aligned16(o) && (ctopk == 0 || aligned16(cache)),
                 DS41_E_ARG, "%s: q, sink and o must be non-null; q, o, cache 16-byte aligned",
                 name);
    const size_t need = ds41_sparse_attn_workspace_bytes(m, nh, hd, win + ctopk);
    DS41_REQUIRE(need == 0 || (ws && ws_bytes >= need), DS41_E_WORKSPACE,
                 "%s: workspace of %zu bytes needed, %zu given", name, need, ws ? ws_bytes : 0);
    DS41_REQUIRE(need == 0 || aligned16(ws), DS41_E_ARG, "%s: ws must be 16-byte aligned", name);
    const int64_t n_a = ds41_rows_a_len(m, win, start_pos);
    int rc = ds41_window_ring_write(kv, ring, rows_a, win_idx, nullptr, m, hd, win, start_pos,
                                    stream);
    if (rc) return rc;
    const int32_t* att_idx = win_idx;
    if (ctopk > 0) {
        const int64_t total = m * (win + ctopk);
        const int threads = 256;
        const int64_t blocks = (total + threads - 1) / threads;
        if ((rc = launch_pdl(merge_shared_kernel,
                             dim3((unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16)),
                             dim3(threads), 0, (cudaStream_t)stream, name,
                             (const int32_t*)win_idx, cidx, idx, m, (int)win, (int)ctopk)))
            return rc;
        att_idx = idx;
    }
    const ds41_bf16* rows_a_used = start_pos == 0 ? kv : (m == 1 ? ring : rows_a);
    return ds41_sparse_attn_sink_fwd(q, rows_a_used, n_a, ctopk ? cache : nullptr,
                                     ctopk ? n_c : 0, att_idx, win + ctopk, sink, scale, o, lse,
                                     m, nh, hd, ws, ws_bytes, stream);
}
