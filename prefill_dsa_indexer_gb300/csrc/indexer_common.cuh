// indexer_common.cuh -- work planning shared by the indexer kernels.
//
// A launch covers groups [group0, group0 + num_groups) of G consecutive rows
// (one request each).  Every CTA computes, in shared memory, each group's
// request, its longest visible context and the prefix sums of its key-tile
// counts (128 or 256 keys per tile); the tiles of all groups then form one list that the
// persistent grid splits into equal contiguous shares (key-balanced).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace dsa {

constexpr int kIdxTileKeys = 128;

// Sequential walk over a CTA's contiguous range of the global tile list.
struct TileWalker {
    const int32_t *prefix;  // [num_groups + 1] tile prefix sums (shared memory)
    int g;
    __device__ void seek(int32_t w, int num_groups) {
        int lo = 0, hi = num_groups;  // largest g < num_groups with prefix[g] <= w
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (prefix[mid] <= w) lo = mid;
            else hi = mid;
        }
        g = lo;
    }
    __device__ void advance(int32_t w) {
        while (prefix[g + 1] <= w) ++g;
    }
};

// Fill greq/gmax/prefix for the launch's groups.  Must be followed by
// __syncthreads() and then plan_scan() by warp 0.
template <int G, int TK = kIdxTileKeys>
__device__ __forceinline__ void plan_groups(const IndexerArgs &a, int32_t *prefix, int32_t *greq, int32_t *gmax) {
    for (int g = threadIdx.x; g < a.num_groups; g += blockDim.x) {
        const int row0 = (a.group0 + g) * G;
        const int req = a.row_req[row0];
        int mx = 0;
        bool bad = req < 0 || req >= a.num_requests;
        for (int j = 0; j < G; ++j) {
            const int c = a.row_ctx[row0 + j];
            if (a.row_req[row0 + j] != req || c < 0 || c > a.max_ctx) bad = true;
            mx = max(mx, min(max(c, 0), a.max_ctx));
        }
        if (bad) {
            report(a.status, DSA_ERR_BOUNDS);
            mx = 0;
        }
        greq[g] = req;
        gmax[g] = mx;
        prefix[g + 1] = (mx + TK - 1) / TK;
    }
    if (threadIdx.x == 0) prefix[0] = 0;
}

// Inclusive scan of prefix[1..ng] in place, by one warp.
__device__ __forceinline__ void plan_scan(int32_t *prefix, int ng, int lane) {
    const int per = (ng + 31) / 32;
    const int b = 1 + lane * per, e = min(ng + 1, b + per);
    int sum = 0;
    for (int i = b; i < e; ++i) sum += prefix[i];
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int run = incl - sum;
    for (int i = b; i < e; ++i) {
        run += prefix[i];
        prefix[i] = run;
    }
}

// This CTA's contiguous share [begin, end) of `total` tiles.
__device__ __forceinline__ void plan_share(int32_t total, int32_t &begin, int32_t &end) {
    const int32_t P = static_cast<int32_t>(gridDim.x), b = static_cast<int32_t>(blockIdx.x);
    const int32_t per = total / P, rem = total % P;
    begin = b * per + (b < rem ? b : rem);
    end = begin + per + (b < rem ? 1 : 0);
}

}  // namespace dsa
