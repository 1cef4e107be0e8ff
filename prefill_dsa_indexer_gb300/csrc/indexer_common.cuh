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

// sum_h w[h] * max(0, acc[h]) over the 32 indexer heads of one (row, key), with packed
// two-wide fp32 FMAs (the weights are a shared-memory broadcast, 16-byte aligned).  Half of the
// ReLUs are a max (integer/ALU pipe) and half are x + |x| = 2 max(0, x), exact, on the FMA
// pipe; those terms are halved at the end (exact), which balances the two pipes.
__device__ __forceinline__ float head_relu_sum(const uint32_t (&acc)[32], const float *w) {
    float2 a0 = make_float2(0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
    auto rl = [&](int h) { return fmaxf(__uint_as_float(acc[h]), 0.f); };
    auto r2 = [&](int h) {
        const float x = __uint_as_float(acc[h]);
        return x + fabsf(x);
    };
#pragma unroll
    for (int h = 0; h < 32; h += 8) {
        const float4 wa = *reinterpret_cast<const float4 *>(w + h);
        const float4 wb = *reinterpret_cast<const float4 *>(w + h + 4);
        a0 = __ffma2_rn(make_float2(wa.x, wa.y), make_float2(rl(h), rl(h + 1)), a0);
        b0 = __ffma2_rn(make_float2(wa.z, wa.w), make_float2(r2(h + 2), r2(h + 3)), b0);
        a1 = __ffma2_rn(make_float2(wb.x, wb.y), make_float2(rl(h + 4), rl(h + 5)), a1);
        b1 = __ffma2_rn(make_float2(wb.z, wb.w), make_float2(r2(h + 6), r2(h + 7)), b1);
    }
    return fmaf(0.5f, (b0.x + b0.y) + (b1.x + b1.y), (a0.x + a0.y) + (a1.x + a1.y));
}

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
