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

// One warp ranks the vis (1 <= kk < vis <= WTK_MAX) scores sc[0 .. vis) of a
// query and hands each of the kk best to put(position, row): positions
// 0 .. kk-1 in ascending row order, ties at the threshold key going to the
// lowest-numbered rows.  Lane l holds the run of ceil(vis / 32) consecutive
// keys from that many times l (index order lane, register); the two 8-bit
// histogram passes use the warp's own 256-entry hist (and sel[4]), and one
// warp scan of the per-lane counts places the picks (each lane's keys above
// and at the threshold as bit masks, so that a pick's rank among them is one
// population count).
constexpr int WTK_KPL = 32;            // keys per lane at most
constexpr int WTK_MAX = 32 * WTK_KPL;  // 1024 visible scores
template <class Put>
__device__ __forceinline__ void warp_topk(const uint16_t* sc, int vis, int kk, int* hist, int* sel,
                                          Put put) {
    const int lane = threadIdx.x & 31;
    const int kpl = (vis + 31) / 32;
    const int i0 = kpl * lane;
    const int n_mine = max(0, min(kpl, vis - i0));
    uint32_t key[WTK_KPL];
    const bool vec = (kpl & 7) == 0 && ((reinterpret_cast<uintptr_t>(sc) & 15u) == 0);
#pragma unroll
    for (int v = 0; v < WTK_KPL / 8; v++) {
        const int b0 = i0 + 8 * v;
        if (8 * v >= n_mine) continue;
        if (vec && 8 * v + 8 <= n_mine) {  // whole groups of eight only
            uint4 u = __ldg(reinterpret_cast<const uint4*>(sc + b0));
            const uint16_t* h = reinterpret_cast<const uint16_t*>(&u);
#pragma unroll
            for (int e = 0; e < 8; e++) key[8 * v + e] = order_key(h[e]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++)
                if (8 * v + e < n_mine) key[8 * v + e] = order_key(__ldg(sc + b0 + e));
        }
    }
#pragma unroll
    for (int e = 0; e < 8; e++) hist[lane + 32 * e] = 0;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < WTK_KPL; e++)
        if (e < n_mine) atomicAdd(&hist[key[e] >> 8], 1);
    __syncwarp();
    find_bucket(hist, kk, 0, &sel[0], &sel[1]);
    __syncwarp();
    const uint32_t hb = (uint32_t)sel[0];
    const int above1 = sel[1];
#pragma unroll
    for (int e = 0; e < 8; e++) hist[lane + 32 * e] = 0;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < WTK_KPL; e++)
        if (e < n_mine && (key[e] >> 8) == hb) atomicAdd(&hist[key[e] & 0xffu], 1);
    __syncwarp();
    find_bucket(hist, kk, above1, &sel[2], &sel[3]);
    __syncwarp();
    const uint32_t T = (hb << 8) | (uint32_t)sel[2];
    const int need_eq = kk - sel[3];
    uint32_t gm = 0, qm = 0;
#pragma unroll
    for (int e = 0; e < WTK_KPL; e++) {
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
    const int gt = x_gt - n_gt, eq = x_eq - n_eq;
#pragma unroll
    for (int e = 0; e < WTK_KPL; e++) {
        const uint32_t below = (1u << e) - 1u;  // bits 0 .. e-1
        const int eqb = eq + __popc(qm & below);
        if (((gm >> e) & 1u) || (((qm >> e) & 1u) && eqb < need_eq))
            put(gt + __popc(gm & below) + min(eqb, need_eq), i0 + e);
    }
}

}  // namespace ds41
