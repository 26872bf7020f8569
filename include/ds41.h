/*
 * ds41.h - C ABI of libds41: one layer's compressed sparse attention forward
 * (DeepSeek-V4.1 style) for m tokens at start_pos, as hand-written CUDA for
 * GB300 (sm_103a).
 *
 * The operations follow three pages of the metrale_model_arch crate:
 *   forward.rs  = metrale_model_arch/attn_v41/forward.rs, AttnV41::forward
 *   compress.rs = metrale_model_arch/deepseek_v41_ref/compress.rs, the CPU
 *                 reference (attention_any and its helpers)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensor pointers are DEVICE pointers owned by the caller (for example
 *   torch allocations).  The entry points allocate no device memory.  Entry
 *   points that need scratch memory take (ws, ws_bytes); the matching
 *   *_workspace_bytes function says how much.  Host pointers are marked
 *   "host".
 * - bf16 tensors are passed as uint16_t bit patterns (ds41_bf16).
 * - Layouts are row-major and contiguous; every device pointer must be 16-byte
 *   aligned.
 * - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *   stream) and runs asynchronously; no entry point synchronises the host.
 * - Every entry point returns DS41_OK (0) or an error code.  On DS41_E_ARG and
 *   DS41_E_RANGE nothing was enqueued.  ds41_last_error() gives the message of
 *   the calling thread's last failure.
 * - Kernels that read indices check them; an out-of-range index is skipped
 *   (never dereferenced) and raises DS41_E_INDEX in the device status word,
 *   read with ds41_device_status().
 */
#ifndef DS41_H_
#define DS41_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t ds41_bf16;               /* bfloat16 bit pattern */
typedef struct CUstream_st* ds41_stream_t; /* same type as cudaStream_t */

enum {
    DS41_OK = 0,
    DS41_E_ARG = 1,       /* null / misaligned pointer, unsupported size */
    DS41_E_RANGE = 2,     /* a limit of the forward: token count, position, top-k */
    DS41_E_CUDA = 3,      /* a CUDA call or launch failed */
    DS41_E_INDEX = 4,     /* a device-side index check tripped (device status) */
    DS41_E_WORKSPACE = 5, /* ws is NULL or smaller than *_workspace_bytes */
    DS41_E_TIMEOUT = 6    /* a bounded device-side wait gave up (device status) */
};

/* Message of the calling thread's last error ("" if none).  The pointer stays
 * valid until the thread's next failing call. */
const char* ds41_last_error(void);

/* Reads (and with reset != 0 clears) the device status word of the current
 * device: 0, or the DS41_E_* code a kernel raised.  Synchronises the device. */
int ds41_device_status(int32_t* status /* host */, int reset);

/* ------------------------------------------------------------------------ */
/* fp4 block quantisers                                                      */
/* ------------------------------------------------------------------------ */
/* compress.rs, fp4_quant_e8m0_inplace (the indexer's q and k): per block of
 * 32 values along a row, amax (floored at 6*2^-126), scale s = the power of
 * two at or above amax/6, each value v -> bf16(e2m1(clamp(v/s, -6, 6)) * s),
 * where e2m1 rounds to the grid {0,.5,1,1.5,2,3,4,6} with ties to the even
 * code.
 *   x      [rows, cols] bf16 input;  y [rows, cols] bf16 output (may equal x)
 *   codes  nullable [rows, cols/2] uint8: e2m1 codes, element 2j in the low
 *          nibble of byte j; bit 3 of a code is the sign
 *   scales nullable [rows, cols/32] uint8: the biased exponent of s (e8m0)
 *   cols % 32 == 0.  rows * cols < 2^31. */
int ds41_fp4_quant_e8m0(const ds41_bf16* x, ds41_bf16* y, uint8_t* codes, uint8_t* scales,
                        int64_t rows, int64_t cols, ds41_stream_t stream);

/* compress.rs, fp4_quant_e4m3_inplace (the compressed KV latent): per block
 * of 16, amax floored at 6*2^-9, s = e4m3(amax/6) (round to nearest even,
 * saturating at 448), then the same element path as above.
 *   scales nullable [rows, cols/16] uint8: the e4m3 code of s.  cols % 16 == 0. */
int ds41_fp4_quant_e4m3(const ds41_bf16* x, ds41_bf16* y, uint8_t* codes, uint8_t* scales,
                        int64_t rows, int64_t cols, ds41_stream_t stream);

/* ------------------------------------------------------------------------ */
/* RoPE table                                                                 */
/* ------------------------------------------------------------------------ */
/* compress.rs, yarn_freqs_cis: out [seqlen, dim/2, 2] f32 of (cos, sin) of
 * p * f_i, where f_i = base^(-2i/dim) blended towards f_i / factor by the YaRN
 * ramp between floor(corr(beta_fast)) and ceil(corr(beta_slow)),
 * corr(r) = dim * ln(original_seq_len / (2 pi r)) / (2 ln base).  Built once
 * per model; the latent write reads it.  dim even, >= 2. */
int ds41_yarn_freqs_cis(float* out, int64_t dim, int64_t seqlen, int64_t original_seq_len,
                        float base, float factor, float beta_fast, float beta_slow,
                        ds41_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Step 1a: window ring and window indices                                    */
/* ------------------------------------------------------------------------ */
/* Rows the window indices point into (rows_a): m at start_pos 0, win for a
 * single-token step past position 0, win + m for a chunk of m > 1 tokens past
 * position 0.  Host function, no device work. */
int64_t ds41_rows_a_len(int64_t m, int64_t win, int64_t start_pos);

/* The row counts of a call of m tokens at start_pos (host function, no device
 * work), written to the host array out[5]:
 *   out[0] n_a   = ds41_rows_a_len(m, win, start_pos), the offset of the picks
 *   out[1] n_c   = (start_pos + m)/ratio, compress_len of forward.rs and
 *                  compress.rs (compressed rows that exist after the call)
 *   out[2] G     = n_c - start_pos/ratio, the groups the call completes (the
 *                  latent rows it writes, from cache row start_pos/ratio on)
 *   out[3] ctopk = min(topk, n_c) (0 when n_c == 0: no indexer runs)
 *   out[4] K     = win + ctopk, the length of a merged index row
 * DS41_E_ARG for a NULL out or win, ratio or topk below 1; DS41_E_RANGE for
 * m < 1, start_pos < 0 or start_pos + m >= 2^31. */
int ds41_step_sizes(int64_t m, int64_t start_pos, int64_t win, int64_t ratio, int64_t topk,
                    int64_t* out /* host [5] */);

/* forward.rs, "the window ring" block, and compress.rs attention_any's ring
 * update: the row of position q goes to ring slot q mod win; when m > win
 * only the newest row of each slot is kept.  Also writes the window indices
 * (forward.rs calls window_topk_idxs): win_idx[t][j] is the rows_a index of
 * position p - win + 1 + j (p = start_pos + t), or -1 when that position is
 * negative.  rows_a is
 *   start_pos == 0        : kv itself (index = position);
 *   start_pos > 0, m == 1 : the ring after this write (index = q mod win);
 *   start_pos > 0, m > 1  : the ring as it was before this call, then kv
 *                           (q < start_pos -> q mod win, else
 *                           win + q - start_pos); this function writes it.
 *   kv      [m, hd] bf16 new rows;     ring [win, hd] bf16, updated in place
 *   rows_a  [win + m, hd] bf16 output, required only when start_pos > 0 and
 *           m > 1 (ignored otherwise, may be NULL)
 *   win_idx [m, win] int32 output
 *   n_a     nullable host int64 output: ds41_rows_a_len(m, win, start_pos)
 *   m >= 1, hd % 8 == 0, win >= 1. */
int ds41_window_ring_write(const ds41_bf16* kv, ds41_bf16* ring, ds41_bf16* rows_a,
                           int32_t* win_idx, int64_t* n_a, int64_t m, int64_t hd, int64_t win,
                           int64_t start_pos, ds41_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Step 1b: compressed latent rows                                            */
/* ------------------------------------------------------------------------ */
/* forward.rs, "if let Some(groups) = latent_groups" (rope, fp4_quant with
 * LATENT_BLOCK, copy into the cache at row start_pos/ratio) and the same
 * branch of compress.rs attention_any.  The call completes
 * G = (start_pos + m)/ratio - start_pos/ratio groups; group g becomes cache
 * row c = start_pos/ratio + g.  Its RoPE position is c * ratio (g*ratio at
 * start_pos 0, start_pos + 1 - ratio for the single decode group).  The row
 * is rotated (last rd dims, adjacent pairs, table row c * ratio), rounded to
 * bf16, then sent through the e4m3 fp4 round trip (block 16).
 *   latent     [G, hd] bf16, before RoPE
 *   freqs_cis  [max_pos, rd/2, 2] f32 (cos, sin), from ds41_yarn_freqs_cis
 *   cache      [cache_rows, hd] bf16, rows c written
 *   cache_codes  nullable [cache_rows, hd/2] uint8 e2m1 codes of row c
 *   cache_scales nullable [cache_rows, hd/16] uint8 e4m3 scale codes of row c
 *   G must equal (start_pos + m)/ratio - start_pos/ratio (G == 0 is a no-op);
 *   hd % 16 == 0, rd even, 0 < rd <= hd, (start_pos + m)/ratio <= cache_rows,
 *   start_pos + m <= max_pos. */
int ds41_compress_latent_write(const ds41_bf16* latent, const float* freqs_cis, int64_t max_pos,
                               ds41_bf16* cache, int64_t cache_rows, uint8_t* cache_codes,
                               uint8_t* cache_scales, int64_t G, int64_t hd, int64_t rd,
                               int64_t ratio, int64_t start_pos, int64_t m, ds41_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Steps 2a + 2b: fp4 indexer scores, per-query top-k, index merge            */
/* ------------------------------------------------------------------------ */
/* Scratch bytes ds41_indexer_topk needs (scores_out given or not). */
size_t ds41_indexer_workspace_bytes(int64_t m, int64_t Hi, int64_t Di, int64_t n_c,
                                    int scores_out_given);

/* forward.rs / compress.rs call the indexer (its body is not on the pages)
 * and then merge: idx row t = the window indices of t, then the indexer's
 * ctopk = min(topk, n_c) picks, already offset by n_a (= offset).  The
 * compress.rs header fixes the precision: q and k take the e2m1 round trip
 * with power-of-two scales per block of 32 and the scores are bf16 values.
 * This library computes, for query t at p = start_pos + t and every
 * compressed row s < (p + 1)/ratio (rows that are complete at p):
 *   qh = Q8(q_idx[t, h, :]), kh = Q8(k_idx[s, :])       (as ds41_fp4_quant_e8m0)
 *   dot = sum_d qh[d] * kh[d]                             (exact for fp4 values
 *                                                          of moderate range)
 *   acc = 0; for h = 0 .. Hi-1: acc = fma(w[t, h], max(dot, 0), acc)   (f32)
 *   score[t, s] = bf16(acc)  (-0 stored as +0; rows not yet visible: -inf)
 * then keeps the min(topk, visible) highest scores, ties to the lower row, as
 * offset + s, and pads with -1.  The picks of a row are in ascending s.
 *   q_idx  [m, Hi, Di] bf16;  k_idx [n_c, Di] bf16;  w [m, Hi] f32
 *   win_idx [m, win] int32 (from ds41_window_ring_write)
 *   idx    [m, win + ctopk] int32 output
 *   scores nullable [m, n_c] bf16 output
 *   Di % 32 == 0, Di <= 256, 1 <= Hi <= 128, n_c >= 1 (with n_c == 0 call
 *   nothing: the merged row is the window row alone), 1 <= topk. */
int ds41_indexer_topk(const ds41_bf16* q_idx, const ds41_bf16* k_idx, const float* w,
                      const int32_t* win_idx, int32_t* idx, ds41_bf16* scores, int64_t m,
                      int64_t Hi, int64_t Di, int64_t n_c, int64_t win, int64_t ratio,
                      int64_t start_pos, int64_t topk, int64_t offset, void* ws, size_t ws_bytes,
                      ds41_stream_t stream);

/* Scratch bytes ds41_indexer_topk_mxf4 needs: the scores of the top-k when
 * they are not an output (scores_out_given == 0), else 0. */
size_t ds41_indexer_mxf4_workspace_bytes(int64_t m, int64_t n_c, int scores_out_given);

/* ds41_indexer_topk on a packed mxf4 key cache.  The compress.rs header puts
 * the indexer's k through the e2m1 round trip with power-of-two scales per
 * block of 32 (fp4_quant_e8m0_inplace); those values are exactly an e2m1 code
 * per element and an e8m0 scale per block, which is how this call takes the
 * keys: 68 bytes per row of 128 instead of 256.  ds41_fp4_quant_e8m0 writes
 * them (its codes and scales outputs) from bf16 keys.  The scores, picks,
 * merge and errors are those of ds41_indexer_topk on the bf16 keys the codes
 * and scales encode (Q8 of those keys gives back the same values), bit for
 * bit.  The dot products run as block-scaled tensor-core MMAs on the codes;
 * q is quantised inside the kernel.
 *   q_idx    [m, Hi, Di] bf16
 *   k_codes  [n_c, Di/2] uint8: e2m1 codes, element 2j in the low nibble of
 *            byte j, bit 3 of a code the sign
 *   k_scales [n_c, Di/32] uint8: biased exponents (e8m0) of the block scales
 *   w [m, Hi] f32, win_idx [m, win], idx [m, win + ctopk], scores nullable
 *            [m, n_c] bf16: as ds41_indexer_topk
 *   Hi == 64 and Di == 128 (DS41_E_ARG otherwise); q_idx, k_codes, k_scales
 *   and w 16-byte aligned. */
int ds41_indexer_topk_mxf4(const ds41_bf16* q_idx, const uint8_t* k_codes, const uint8_t* k_scales,
                           const float* w, const int32_t* win_idx, int32_t* idx, ds41_bf16* scores,
                           int64_t m, int64_t Hi, int64_t Di, int64_t n_c, int64_t win,
                           int64_t ratio, int64_t start_pos, int64_t topk, int64_t offset,
                           void* ws, size_t ws_bytes, ds41_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Step 3: sparse attention with a per-head sink                              */
/* ------------------------------------------------------------------------ */
/* Scratch bytes ds41_sparse_attn_sink_fwd needs. */
size_t ds41_sparse_attn_workspace_bytes(int64_t m, int64_t nh, int64_t hd, int64_t K);

/* compress.rs attention_any: sparse_attn(q, kv_rows, sink, idx, ...) with
 * scale = head_dim^-0.5 (the body of sparse_attn is not on the pages), and
 * forward.rs attend_and_project's rows_a / rows_b / idx / topk arguments.
 * For every query t and head h, over the valid entries v of idx row t
 * (v < n_a -> rows_a[v], n_a <= v < n_a + n_c -> rows_b[v - n_a], -1 skipped):
 *   s_v = scale * <q[t, h], row_v>
 *   o[t, h] = sum_v e^{s_v} row_v / (e^{sink[h]} + sum_v e^{s_v})
 * One row serves as key and value.  The sink is a logit in the denominator
 * only (-inf gives a plain softmax).  f32 accumulation, bf16 output.
 *   q [m, nh, hd] bf16;  rows_a [n_a, hd];  rows_b [n_c, hd] (NULL if n_c == 0)
 *   idx [m, K] int32;  sink [nh] f32
 *   o [m, nh, hd] bf16 output;  lse nullable [m, nh] f32 output: the natural
 *   log of the denominator above, e^{lse} = e^{sink} + sum_v e^{s_v}
 *   hd % 64 == 0, hd <= 512, nh >= 1, K >= 1. */
int ds41_sparse_attn_sink_fwd(const ds41_bf16* q, const ds41_bf16* rows_a, int64_t n_a,
                              const ds41_bf16* rows_b, int64_t n_c, const int32_t* idx, int64_t K,
                              const float* sink, float scale, ds41_bf16* o, float* lse, int64_t m,
                              int64_t nh, int64_t hd, void* ws, size_t ws_bytes,
                              ds41_stream_t stream);

/* ------------------------------------------------------------------------ */
/* The whole step                                                             */
/* ------------------------------------------------------------------------ */
/* Scratch bytes ds41_csa_forward needs for these sizes. */
size_t ds41_csa_workspace_bytes(int64_t m, int64_t start_pos, int64_t nh, int64_t hd, int64_t win,
                                int64_t ratio, int64_t topk, int64_t Hi, int64_t Di);

/* forward.rs, AttnV41::forward (and compress.rs attention_any): the whole
 * compressed sparse attention step of one layer for m tokens at start_pos, in
 * the pages' order: the window ring write and window indices
 * (ds41_window_ring_write), the latent write of the groups this call
 * completes (ds41_compress_latent_write), the indexer top-k and merge
 * (ds41_indexer_topk, offset = ds41_rows_a_len), and sparse attention with
 * the sink (ds41_sparse_attn_sink_fwd).  Arguments and layouts are those of
 * the four calls; the results are the same.  rows_a ([win + m, hd]) is
 * needed only for a chunk of m > 1 tokens past position 0; latent /
 * freqs_cis only when the call completes a group; lse is nullable.  idx is
 * [m, win + min(topk, n_c)] with n_c = (start_pos + m)/ratio (unused when
 * n_c == 0).  Few-token calls, and calls whose attention runs in one wave of
 * CTAs with one split (each CTA then selects its token's rows from the scores
 * itself), run in two or three launches chained on the device (programmatic
 * dependent launch), larger ones as the four calls. */
int ds41_csa_forward(const ds41_bf16* q, const ds41_bf16* kv, ds41_bf16* ring, ds41_bf16* rows_a,
                     const ds41_bf16* latent, const float* freqs_cis, int64_t max_pos,
                     ds41_bf16* cache, int64_t cache_rows, const ds41_bf16* q_idx,
                     const ds41_bf16* k_idx, const float* w, const float* sink, float scale,
                     int32_t* win_idx, int32_t* idx, ds41_bf16* o, float* lse, int64_t m,
                     int64_t start_pos, int64_t nh, int64_t hd, int64_t rd, int64_t win,
                     int64_t ratio, int64_t topk, int64_t Hi, int64_t Di, void* ws,
                     size_t ws_bytes, ds41_stream_t stream);

/* Scratch bytes ds41_csa_forward_fp4 needs for these sizes. */
size_t ds41_csa_fp4_workspace_bytes(int64_t m, int64_t start_pos, int64_t nh, int64_t hd,
                                    int64_t win, int64_t ratio, int64_t topk);

/* ds41_csa_forward on packed fp4 caches (the pages' precision, kept in its
 * packed form).  The indexer keys are an mxf4 cache, as
 * ds41_indexer_topk_mxf4 takes them: k_codes [n_c, Di/2] e2m1 codes and
 * k_scales [n_c, Di/32] e8m0 bytes (68 bytes per row of 128 instead of 256).
 * The latent write (forward.rs latent branch: fp4_quant with LATENT_BLOCK)
 * writes the new compressed rows to `cache` (bf16) and, when cache_codes /
 * cache_scales are given, also as e2m1 codes [cache_rows, hd/2] and e4m3
 * block-16 scale codes [cache_rows, hd/16] (288 bytes per row of 512
 * instead of 1024).  With them given, few-token calls at hd 512 gather the
 * compressed rows in that packed form and expand them in shared memory to
 * exactly the bf16 values (so cache_codes / cache_scales must hold the packed
 * form of every row below n_c that the call does not write itself);
 * many-token calls read the bf16 cache.  Every other argument, the results
 * and the errors are those of ds41_csa_forward, bit for bit (the codes and
 * scales encode the same values).  Hi == 64 and Di == 128 (DS41_E_ARG
 * otherwise); k_codes, k_scales, w, cache_codes and cache_scales 16-byte
 * aligned; cache_codes and cache_scales both given or both NULL.  Few-token
 * calls run in two or three launches chained on the device (the scores
 * kernel's extra CTAs do the ring and latent writes), larger ones as the
 * separate calls. */
int ds41_csa_forward_fp4(const ds41_bf16* q, const ds41_bf16* kv, ds41_bf16* ring,
                         ds41_bf16* rows_a, const ds41_bf16* latent, const float* freqs_cis,
                         int64_t max_pos, ds41_bf16* cache, uint8_t* cache_codes,
                         uint8_t* cache_scales, int64_t cache_rows, const ds41_bf16* q_idx,
                         const uint8_t* k_codes, const uint8_t* k_scales, const float* w,
                         const float* sink, float scale, int32_t* win_idx, int32_t* idx,
                         ds41_bf16* o, float* lse, int64_t m, int64_t start_pos, int64_t nh,
                         int64_t hd, int64_t rd, int64_t win, int64_t ratio, int64_t topk,
                         int64_t Hi, int64_t Di, void* ws, size_t ws_bytes, ds41_stream_t stream);

/* forward.rs, AttnV41::forward, for a layer that is neither a kv source
 * nor an index source: it writes its own window ring and window indices,
 * takes the compressed rows (rows_b) and the compressed picks of the last
 * source layer (the shared slots compress_kv and topk_idxs), merges its
 * window indices with those picks, and attends.  No latent write, no indexer.
 *   q [m, nh, hd], kv [m, hd], ring [win, hd], rows_a as ds41_csa_forward
 *   cache [>= n_c, hd] bf16: the source layer's compressed rows, n_c =
 *       (start_pos + m)/ratio of them visible
 *   cidx [m, ctopk] int32: the source layer's picks, already offset by
 *       ds41_rows_a_len (as ds41_indexer_topk writes them after the window
 *       part of its idx rows); ctopk = min(topk, n_c), NULL when 0
 *   win_idx [m, win] and idx [m, win + ctopk] int32 outputs (idx row t = the
 *       window indices of t, then cidx row t; idx is unused when ctopk == 0)
 *   o, lse, sink, scale as ds41_sparse_attn_sink_fwd.
 * Scratch: ds41_sparse_attn_workspace_bytes(m, nh, hd, win + ctopk).  Errors:
 * those of ds41_window_ring_write and ds41_sparse_attn_sink_fwd, all checked
 * before anything is enqueued; an index in cidx past n_a + n_c raises
 * DS41_E_INDEX on the device and is skipped. */
int ds41_csa_forward_reuse(const ds41_bf16* q, const ds41_bf16* kv, ds41_bf16* ring,
                           ds41_bf16* rows_a, const ds41_bf16* cache, const int32_t* cidx,
                           int64_t ctopk, const float* sink, float scale, int32_t* win_idx,
                           int32_t* idx, ds41_bf16* o, float* lse, int64_t m, int64_t start_pos,
                           int64_t nh, int64_t hd, int64_t win, int64_t ratio, void* ws,
                           size_t ws_bytes, ds41_stream_t stream);

/* ds41_csa_forward for a caller whose per-step inputs and output live in
 * host memory (no counterpart on the pages, whose reference computes on the host): the
 * inputs h_q [m, nh, hd], h_kv [m, hd], h_latent [G, hd] (read only when the
 * call completes G > 0 groups, G = (start_pos + m)/ratio - start_pos/ratio;
 * may be NULL otherwise), h_q_idx [m, Hi, Di] and h_w [m, Hi] are copied into
 * the device buffers q, kv, latent, q_idx and w (caller-owned, same shapes),
 * ds41_csa_forward runs on them, and o is copied into h_o [m, nh, hd]; the
 * other arguments are ds41_csa_forward's.  When h_o is page-locked memory
 * mapped for the current device, m <= 16 and o takes at most 4 MiB (a
 * multiple of 16 bytes), the step writes o straight into h_o through the
 * mapping instead and the device buffer o is left unwritten.  Everything is enqueued on `stream`
 * in that order; the call returns without waiting, and h_o holds the result
 * once the stream has reached that point (cudaStreamSynchronize).  The copies
 * are asynchronous only for page-locked host memory (cudaHostAlloc /
 * cudaHostRegister); pageable buffers work but the copies then block the
 * calling thread.  A copy of at most 4 MiB, a multiple of 16 bytes, between
 * 16-byte aligned device memory and page-locked memory mapped for the current
 * device runs as a small kernel on the stream that moves the bytes through
 * the mapping (for a decode step's tens of KB this ends sooner than a
 * copy-engine transfer); other copies use cudaMemcpyAsync.  The host buffers must stay valid and unmodified until the
 * stream has passed the copies.  Errors: ds41_csa_forward's, DS41_E_ARG for a
 * NULL pointer, DS41_E_CUDA when a copy cannot be enqueued (the copies
 * enqueued before stay enqueued). */
int ds41_csa_forward_host(const ds41_bf16* h_q, const ds41_bf16* h_kv, const ds41_bf16* h_latent,
                          const ds41_bf16* h_q_idx, const float* h_w, ds41_bf16* h_o,
                          ds41_bf16* q, ds41_bf16* kv, ds41_bf16* ring, ds41_bf16* rows_a,
                          ds41_bf16* latent, const float* freqs_cis, int64_t max_pos,
                          ds41_bf16* cache, int64_t cache_rows, ds41_bf16* q_idx,
                          const ds41_bf16* k_idx, float* w, const float* sink, float scale,
                          int32_t* win_idx, int32_t* idx, ds41_bf16* o, float* lse, int64_t m,
                          int64_t start_pos, int64_t nh, int64_t hd, int64_t rd, int64_t win,
                          int64_t ratio, int64_t topk, int64_t Hi, int64_t Di, void* ws,
                          size_t ws_bytes, ds41_stream_t stream);

/* Bytes of one step's inputs packed back to back as [q | kv | latent | q_idx |
 * w] (the layout ds41_csa_forward_host_packed takes): 2 (m nh hd + m hd +
 * G hd + m Hi Di) + 4 m Hi, G as above; 0 for m < 1, start_pos < 0 or
 * ratio < 1. */
size_t ds41_step_inputs_bytes(int64_t m, int64_t start_pos, int64_t nh, int64_t hd,
                              int64_t ratio, int64_t Hi, int64_t Di);

/* ds41_csa_forward_host with the step's inputs in one block on each side:
 * h_in (host) and d_in (device, 16-byte aligned) each hold q, kv, latent,
 * q_idx and w back to back in that order, ds41_step_inputs_bytes bytes, so
 * they go over in one copy; the kernels read the inputs from d_in.  Same
 * results, stream behaviour and errors as ds41_csa_forward_host. */
int ds41_csa_forward_host_packed(const void* h_in, void* d_in, ds41_bf16* h_o, ds41_bf16* ring,
                                 ds41_bf16* rows_a, const float* freqs_cis, int64_t max_pos,
                                 ds41_bf16* cache, int64_t cache_rows, const ds41_bf16* k_idx,
                                 const float* sink, float scale, int32_t* win_idx, int32_t* idx,
                                 ds41_bf16* o, float* lse, int64_t m, int64_t start_pos,
                                 int64_t nh, int64_t hd, int64_t rd, int64_t win, int64_t ratio,
                                 int64_t topk, int64_t Hi, int64_t Di, void* ws, size_t ws_bytes,
                                 ds41_stream_t stream);

/* A prepared host step: what one ds41_csa_forward_host_packed call enqueues
 * (the input copy, the step's kernels, the output copy), recorded once into a
 * CUDA graph for fixed buffers, as a serving loop runs a layer's step again
 * and again.  Each ds41_host_step_launch then enqueues the whole step with one
 * graph launch instead of a copy, two kernel launches and a copy, which takes
 * less host time per step and leaves fewer gaps between the operations on the
 * GPU.  No counterpart on the pages (their runtime launches the kernels
 * directly).  The handle is opaque and owned by the caller. */
typedef struct ds41_host_step ds41_host_step;

/* Records the step into *out.  Arguments as ds41_csa_forward_host_packed,
 * minus the stream; every pointer and size is fixed in the recording, so the
 * buffers must outlive the handle and each launch reads whatever h_in holds
 * when the copy runs.  Nothing runs at creation (the recording is made on a
 * private stream in capture mode).  Errors: those of
 * ds41_csa_forward_host_packed's argument checks (nothing is recorded then),
 * DS41_E_ARG for a NULL out, DS41_E_CUDA when the capture or the graph's
 * instantiation fails; *out is NULL on any error. */
int ds41_host_step_create(ds41_host_step** out, const void* h_in, void* d_in, ds41_bf16* h_o,
                          ds41_bf16* ring, ds41_bf16* rows_a, const float* freqs_cis,
                          int64_t max_pos, ds41_bf16* cache, int64_t cache_rows,
                          const ds41_bf16* k_idx, const float* sink, float scale,
                          int32_t* win_idx, int32_t* idx, ds41_bf16* o, float* lse, int64_t m,
                          int64_t start_pos, int64_t nh, int64_t hd, int64_t rd, int64_t win,
                          int64_t ratio, int64_t topk, int64_t Hi, int64_t Di, void* ws,
                          size_t ws_bytes);

/* Enqueues the recorded step on `stream` (one graph launch); returns without
 * waiting, and h_o holds the result once the stream has passed the step.
 * Launches of one handle run one after another.  Results are the same bits
 * as ds41_csa_forward_host_packed with the same arguments.  Errors: DS41_E_ARG
 * for a NULL handle, DS41_E_CUDA when the launch fails. */
int ds41_host_step_launch(ds41_host_step* h, ds41_stream_t stream);

/* Frees the recording (NULL is a no-op).  Launches still pending complete
 * first: the driver frees an executable graph that is in flight once it has
 * finished.  Returns DS41_OK. */
int ds41_host_step_destroy(ds41_host_step* h);

/* ------------------------------------------------------------------------ */
/* Step 3 without caller-provided scratch                                     */
/* ------------------------------------------------------------------------ */
/* No counterpart on the pages: this entry point exists for callers that
 * cannot allocate device memory.  Examples are serving runtimes that reserve
 * all device memory when they start and forbid any allocation afterwards
 * (cudaMalloc can synchronise the device and fragment a carefully packed
 * pool), and plugin hosts that hand a kernel its input and output buffers and
 * no allocator.  Such callers can still run the split (flash-decoding) path
 * of ds41_sparse_attn_sink_fwd, whose partial results need scratch memory.
 *
 * Same arguments, same computation and same results as
 * ds41_sparse_attn_sink_fwd, minus ws / ws_bytes.  The split partials go to
 * one static device array of ds41_sparse_attn_noalloc_capacity() bytes
 * (16 MiB) that every GPU loading this library holds until the process
 * exits.  Sizes whose partials need more (ds41_sparse_attn_workspace_bytes
 * larger than the capacity) are rejected with DS41_E_WORKSPACE and nothing is
 * enqueued.  The call allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  Every call shares the one array and it keeps the last call's
 * contents; nothing in it has to start at zero, because each split writes its
 * partial before the merge reads it.  Calls whose work overlaps on the GPU
 * (on different streams, or on different host threads) race on the array:
 * order them on one stream.  All tensors must be on the current device, whose
 * array the call uses. */
size_t ds41_sparse_attn_noalloc_capacity(void);

int ds41_sparse_attn_sink_fwd_noalloc(const ds41_bf16* q, const ds41_bf16* rows_a, int64_t n_a,
                                      const ds41_bf16* rows_b, int64_t n_c, const int32_t* idx,
                                      int64_t K, const float* sink, float scale, ds41_bf16* o,
                                      float* lse, int64_t m, int64_t nh, int64_t hd,
                                      ds41_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Self-test of the bounded device waits                                      */
/* ------------------------------------------------------------------------ */
/* No counterpart on the pages.  Every mbarrier wait in the tensor-core and
 * decode kernels gives up after a bound (about a second): it sets the
 * kernel's abort flag, raises DS41_E_TIMEOUT in the device status word, and
 * the kernel drains its copies, frees its tensor memory and returns, so the
 * context stays usable.  This call runs that path on purpose: one CTA that
 * holds 32 columns of tensor memory waits `polls` polls (1 .. 2^22) on an
 * mbarrier of count 1.  With arrive == 0 nobody arrives, the wait runs out
 * and DS41_E_TIMEOUT is raised; with arrive != 0 the thread arrives first and
 * the wait completes.
 *   result [2] int32 device output (16-byte aligned): result[0] = 1 if the
 *          wait completed, 0 if it gave up; result[1] = the abort flag as
 *          another warp reads it afterwards.
 * Errors: DS41_E_ARG (bad pointer or polls), DS41_E_CUDA (launch). */
int ds41_selftest_wait_timeout(uint32_t polls, int arrive, int32_t* result, ds41_stream_t stream);

/* ------------------------------------------------------------------------ */
/* The output side of the layer                                               */
/* ------------------------------------------------------------------------ */
/* compress.rs, attention_any after sparse_attn: o is rotated back
 * (apply_rotary with inverse = true, each head at its token's position),
 * split into `groups` groups of gw = nh*hd/groups values, and each group is
 * projected by its own o_rank rows of wo_a, every result rounded to bf16
 * (to_bf16_rne); then linear_bf16 with wo_b (body not on the pages: read as
 * og . wo_b^T with an unrounded f32 result).  This library computes
 *   o[t, h, hd-rd+2i .. +1] <- the pair rotated by -angle of table column i
 *       at position start_pos + t, each product rounded, then the sum, and
 *       the result rounded to bf16 (IN PLACE: o is overwritten)
 *   og[t, g*o_rank + r] = bf16(sum_i o[t, g*gw + i] * wo_a[g*o_rank + r, i])
 *   out[t, j] = sum_k og[t, k] * wo_b[j, k]                           (f32)
 * with f32 accumulation, so og can differ from a differently ordered sum by
 * one bf16 step.  Few tokens (m <= 16) run on the CUDA cores, a warp per
 * weight row (the weight stream from HBM bounds them); more tokens run as
 * tcgen05 tensor-core tiles of 128 weight rows when o_rank, dim and
 * groups*o_rank are multiples of 128 and gw of 64 (else the CUDA-core
 * kernel in chunks of 8 tokens).
 *   o        [m, nh, hd] bf16, in/out (the attention output; rotated back)
 *   freqs_cis [max_pos, rd/2, 2] f32 (cos, sin), as ds41_yarn_freqs_cis
 *   wo_a     [groups*o_rank, gw] bf16;  wo_b [dim, groups*o_rank] bf16
 *   og       [m, groups*o_rank] bf16 output;  out [m, dim] f32 output
 *   All caller-owned device memory, 16-byte aligned.  hd % 8 == 0, rd even
 *   and <= hd (rd = 0: no rotation, freqs_cis may be NULL), gw % 8 == 0,
 *   groups*o_rank % 8 == 0, dim % 4 == 0, start_pos + m <= max_pos.
 * Errors: DS41_E_ARG / DS41_E_RANGE before anything is enqueued; DS41_E_CUDA
 * when a launch fails (the launches before it stay enqueued).  Thread-safe;
 * the work runs on the current device. */
int ds41_attn_out_proj(ds41_bf16* o, const float* freqs_cis, int64_t max_pos,
                       const ds41_bf16* wo_a, const ds41_bf16* wo_b, ds41_bf16* og, float* out,
                       int64_t m, int64_t start_pos, int64_t nh, int64_t hd, int64_t rd,
                       int64_t groups, int64_t o_rank, int64_t dim, ds41_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DS41_H_ */
