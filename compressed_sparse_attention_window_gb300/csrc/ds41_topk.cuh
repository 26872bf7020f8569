// ds41_topk.cuh - pieces of the per-query top-k shared by the top-k kernels
// and the decode attention that selects its own rows: 16-bit order keys of
// bf16 scores and the bucket search over a 256-bin histogram.
#pragma once

#include "ds41_common.cuh"

namespace ds41 {

// bf16 score -> 16-bit key whose unsigned order is the float order
__device__ __forceinline__ uint32_t order_key(uint16_t b) {
    return (b & 0x8000u) ? (uint32_t)(~b & 0xffffu) : (uint32_t)(b | 0x8000u);
}

// Warp 0: the bucket b (of 256) holding the kk-th largest key, counting
// `above` keys already known to be larger; *bucket = b, *cum = above + keys
// in buckets above b.  Lane l owns buckets 8l .. 8l+7.
__device__ __forceinline__ void find_bucket(const int* hist, int kk, int above, int* bucket,
                                            int* cum) {
    const int lane = threadIdx.x & 31;
    int v[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        v[i] = hist[8 * lane + i];
        sum += v[i];
    }
    // keys in the buckets of lanes l .. 31
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_down_sync(0xffffffffu, incl, off);
        if (lane + off < 32) incl += o;
    }
    int c = above + incl - sum;  // keys in buckets of higher lanes
    const bool mine = (c < kk && c + sum >= kk) || (lane == 0 && c + sum < kk);
    if (mine) {
        int b = 8 * lane + 7;
#pragma unroll
        for (int i = 7; i > 0; i--, b--) {
            if (c + v[i] >= kk) break;
            c += v[i];
        }
        *bucket = b;
        *cum = c;
    }
}

// Keys of the visible scores, staged in shared memory when they fit
// (keys_cap entries), read from global memory otherwise.
}  // namespace ds41
