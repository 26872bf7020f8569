// ds41_internal.cuh - host-side pieces shared between translation units of
// libds41 (not part of the C ABI).
#pragma once

#include "ds41_common.cuh"

namespace ds41 {

struct RingArgs;
struct LatentArgs;

int device_sm_count();

// few-token fused front: step 1 + indexer scores in one launch
bool front_fusable(int64_t m, int64_t Hi, int64_t Di, int64_t n_c);
size_t front_scores_bytes(int64_t m, int64_t n_c);
int launch_front(const uint16_t* q_idx, const uint16_t* k_idx, const float* w, uint16_t* scores,
                 int64_t m, int64_t Hi, int64_t Di, int64_t n_c, int64_t ratio,
                 int64_t start_pos, const RingArgs& ring, const LatentArgs& lat,
                 cudaStream_t st);
int launch_topk(const uint16_t* scores, const int32_t* win_idx, int32_t* idx, int64_t m,
                int64_t n_c, int64_t win, int64_t ctopk, int64_t ratio, int64_t start_pos,
                int64_t offset, bool pdl, cudaStream_t st);

// The per-query top-k of the few-token step done by the decode attention
// clusters themselves (no separate launch, no reload of the index row): the
// arguments of the merge, as in the top-k kernels of the indexer.
struct DecTopk {
    const uint16_t* scores;   // [m][n_c] bf16 indexer scores
    const int32_t* win_idx;   // [m][win] window indices
    int32_t* idx_out;         // [m][K] merged index rows (written by head group 0)
    int64_t n_c, ratio, start_pos, offset;
    int win, ctopk;
    int64_t m;                // tokens of the call (the window entries follow from it)
};

// The compressed rows (rows_b) in their packed form: e2m1 codes [n_c][hd/2]
// and e4m3 block-16 scale codes [n_c][hd/16], as the latent write stores them.
struct PackedRows {
    const uint8_t* codes;
    const uint8_t* scales;
};

// sparse attention with an explicit plan choice; pdl launches the few-token
// kernel with programmatic stream serialization; tk (few-token cluster path
// only) makes the attention select its rows from the scores first; pk
// (few-token cluster path, hd 512 only) makes it gather the compressed rows
// packed and expand them in shared memory
int attn_run(const uint16_t* q, const uint16_t* rows_a, int64_t n_a, const uint16_t* rows_b,
             int64_t n_c, const int32_t* idx, int64_t K, const float* sink, float scale,
             uint16_t* o, float* lse, int64_t m, int64_t nh, int64_t hd, uint8_t* ws,
             size_t ws_bytes, bool pdl, cudaStream_t st, const char* name,
             const DecTopk* tk = nullptr, const PackedRows* pk = nullptr);
// whether the few-token attention can select its own rows for these sizes
bool attn_topk_fusable(int64_t m, int64_t nh, int64_t hd, int64_t K, int64_t n_c);
size_t attn_ws_bytes(int64_t m, int64_t nh, int64_t hd, int64_t K);
bool attn_is_cluster_path(int64_t m, int64_t nh, int64_t hd, int64_t K);

// many-token indexer scores on the tcgen05 tensor cores (ds41_indexer_tc.cu):
// q_idx [m*64][128] as given (the kernel takes it through the fp4 round trip),
// kq [n_c][128] the keys' fp4 round-trip values in bf16
bool indexer_tc_supported(int64_t m, int64_t Hi, int64_t Di, int sms);
int indexer_tc_launch(const uint16_t* q_idx, const uint16_t* kq, const float* w, uint16_t* scores,
                      int64_t m, int64_t n_c, int64_t ratio, int64_t start_pos, bool fill_hidden,
                      unsigned int* status, int sms, cudaStream_t st);

// indexer scores on a packed mxf4 key cache (ds41_indexer_mxf4.cu): q_idx
// bf16 [m][64][128], k_codes [n_c][64] e2m1 codes, k_scales [n_c][4] e8m0
bool indexer_mxf4_supported(int64_t Hi, int64_t Di);
// With ring (and lat), extra CTAs past the score grid do step 1 of the
// fused few-token step.
int indexer_mxf4_launch(const uint16_t* q_idx, const uint8_t* k_codes, const uint8_t* k_scales,
                        const float* w, uint16_t* scores, int64_t m, int64_t n_c, int64_t ratio,
                        int64_t start_pos, bool fill_hidden, unsigned int* status, int sms,
                        cudaStream_t st, const RingArgs* ring = nullptr,
                        const LatentArgs* lat = nullptr);

// many-token attention on the tcgen05 tensor cores (ds41_attn_tc.cu)
bool attn_tc_supported(int64_t m, int64_t nh, int64_t hd, int64_t K, int sms);
int attn_tc_launch(const uint16_t* q, const uint16_t* rows_a, int64_t n_a, const uint16_t* rows_b,
                   int64_t n_c, const int32_t* idx, int64_t K, const float* sink, float scale,
                   uint16_t* o, float* lse, int64_t m, int64_t nh, unsigned int* status,
                   int sms, cudaStream_t st);

}  // namespace ds41
