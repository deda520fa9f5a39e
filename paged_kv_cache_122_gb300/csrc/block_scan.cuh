// Block-wide exclusive prefix sum of one int64 per thread (warp shuffles,
// then one pass over the warp totals).
#pragma once

#include <cstdint>

namespace pk {

// `warp_sums` is shared memory with room for blockDim.x / 32 + 1 values.
// Returns this thread's exclusive prefix; *total receives the block sum.
// Contains two __syncthreads(): every thread of the block must call it.
template <int kThreads>
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t *warp_sums, int64_t *total) {
    static_assert(kThreads % 32 == 0 && kThreads <= 1024, "block size");
    constexpr int kWarps = kThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t s = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kWarps) warp_sums[lane] = s;          // inclusive over warps
        if (lane == kWarps - 1) warp_sums[kWarps] = s;   // block total
    }
    __syncthreads();
    *total = warp_sums[kWarps];
    return (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
}

}  // namespace pk
