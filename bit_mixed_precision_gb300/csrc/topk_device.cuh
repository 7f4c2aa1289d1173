// Block-wide top-k by radix select on float32 keys, with ties resolved to
// the lower index, and block-wide prefix scans.  One CTA of kBlock threads
// owns one unit; n may exceed kBlock (threads stride over the elements).
#pragma once

#include "kvq_common.cuh"

namespace kvq {

constexpr int kTopkBlock = 1024;

// Monotone map float32 -> uint32: a > b as floats  <=>  key(a) > key(b).
__device__ __forceinline__ uint32_t orderable(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkShared {
    uint32_t hist[256];
    uint32_t warp_tot[kTopkBlock / 32];
    uint32_t bcast[4];
};

// Exclusive scan of one uint32 per thread across the block; returns the
// thread's exclusive prefix, writes the block total to *total.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, TopkShared& sh, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        uint32_t w = lane < nw ? sh.warp_tot[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) sh.warp_tot[lane] = w;          // inclusive warp prefix
    }
    __syncthreads();
    const uint32_t before = warp ? sh.warp_tot[warp - 1] : 0u;
    const uint32_t tot = sh.warp_tot[(blockDim.x >> 5) - 1];
    __syncthreads();
    *total = tot;
    return before + x - v;
}

// Finds the k-th largest key among n elements (k >= 1, k <= n):
// *kstar = its value, *take_eq = how many elements equal to it belong to
// the top k (the rest of the top k is strictly greater).
// The digit holding the k-th largest among the 256 counts of sh.hist (bins
// taken from the top), by warp 0: each lane sums eight bins, one warp scan.
// Writes the bin to sh.bcast[0] and the rank left inside it to sh.bcast[1].
__device__ __forceinline__ void radix_pick_bin(TopkShared& sh, uint32_t remaining) {
    const int lane = threadIdx.x & 31;
    uint32_t c[8], sum = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        c[q] = sh.hist[255 - 8 * lane - q];
        sum += c[q];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const uint32_t excl = incl - sum;                   // elements in the bins above this lane's eight
    if (excl < remaining && remaining <= incl) {        // exactly one lane: remaining <= the total
        uint32_t cum = excl;
        int bin = 255 - 8 * lane - 7;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (cum + c[q] >= remaining) {
                bin = 255 - 8 * lane - q;
                break;
            }
            cum += c[q];
        }
        sh.bcast[0] = (uint32_t)bin;
        sh.bcast[1] = remaining - cum;
    }
}

// start_shift < 24: every key shares the bits above start_shift + 8 with
// `prefix` (the caller knows them, e.g. from the keys' minimum and maximum),
// and the passes start at that digit.
template <typename KeyFn>
__device__ void block_radix_select(KeyFn key, int n, int k, TopkShared& sh, uint32_t* kstar,
                                   uint32_t* take_eq, int start_shift = 24, uint32_t prefix = 0) {
    uint32_t mask = start_shift >= 24 ? 0u : ~0u << (start_shift + 8);
    prefix &= mask;
    uint32_t remaining = (uint32_t)k;
    for (int shift = start_shift; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) sh.hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint32_t kv = key(i);
            if ((kv & mask) == prefix) atomicAdd(&sh.hist[(kv >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) radix_pick_bin(sh, remaining);
        __syncthreads();
        prefix |= sh.bcast[0] << shift;
        mask |= 255u << shift;
        remaining = sh.bcast[1];
        __syncthreads();
    }
    *kstar = prefix;
    *take_eq = remaining;
}

}  // namespace kvq
