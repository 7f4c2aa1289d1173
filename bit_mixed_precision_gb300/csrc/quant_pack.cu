// kv_quant_pack: asymmetric b-bit quantisation with fp16 scale/zero and
// packing into 32-bit words (MiniKV verdict JSON, key_machinery: 16 INT2
// codes per INT32 word; review page "Core claim": per-channel keys and
// per-token values).  Memory-bound; one thread per (group, channel) for
// the channel grouping (coalesced across channels) and one thread per
// (token, group) for the token grouping (contiguous G-element runs).
#include "kvq_internal.h"
#include "pack_device.cuh"

namespace kvq {

KVQ_DEFINE_STATUS(quant)

template <typename T>
__global__ void quant_channel_kernel(const T* __restrict__ x, int T_len, int D,
                                     const int32_t* __restrict__ gather, int gstride, int n,
                                     int bits, int G, int cap, uint32_t* __restrict__ codes,
                                     uint16_t* __restrict__ scale, uint16_t* __restrict__ zero) {
    const int grp = blockIdx.x;
    const int unit = blockIdx.y;
    const int words_per_group = G * bits / 32;
    const T* xu = x + (size_t)unit * T_len * D;
    const int32_t* gu = gather ? gather + (size_t)unit * gstride : nullptr;
    // positions of the group, checked once
    bool ok = true;
    if (gu) {
        for (int i = threadIdx.x; i < G; i += blockDim.x) {
            int t = gu[grp * G + i];
            if (t < 0 || t >= T_len) ok = false;
        }
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(&g_status_quant, kDevCheck);
        return;
    }
    uint32_t* cu = codes + ((size_t)unit * (cap * bits / 32) + (size_t)grp * words_per_group) * D;
    uint16_t* su = scale + ((size_t)unit * (cap / G) + grp) * D;
    uint16_t* zu = zero + ((size_t)unit * (cap / G) + grp) * D;
    auto row = [&](int i) -> const T* {
        int t = gu ? gu[grp * G + i] : grp * G + i;
        return xu + (size_t)t * D;
    };
    for (int c = threadIdx.x; c < D; c += blockDim.x)
        quant_channel_group<T>(row, G, c, bits, cu, D, su + c, zu + c);
}

template <typename T>
__global__ void quant_token_kernel(const T* __restrict__ x, int T_len, int D,
                                   const int32_t* __restrict__ gather, int gstride, int n, int bits,
                                   int G, int cap, int units, uint32_t* __restrict__ codes,
                                   uint16_t* __restrict__ scale, uint16_t* __restrict__ zero) {
    const int groups = D / G;
    const size_t total = (size_t)units * n * groups;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int g = (int)(idx % groups);
        const size_t rowi = idx / groups;            // unit * n + i
        const int i = (int)(rowi % n);
        const int unit = (int)(rowi / n);
        const size_t orow = (size_t)unit * cap + i;  // output row
        int t = gather ? gather[(size_t)unit * gstride + i] : i;
        if (t < 0 || t >= T_len) {
            atomicOr(&g_status_quant, kDevCheck);
            continue;
        }
        const T* src = x + ((size_t)unit * T_len + t) * D + (size_t)g * G;
        auto load = [&](int k) -> float { return Elem<T>::to_f(src[k]); };
        uint32_t* cw = codes + orow * (D * bits / 32) + (size_t)g * (G * bits / 32);
        quant_token_group(load, G, bits, cw, scale + orow * groups + g, zero + orow * groups + g);
    }
}

cudaError_t launch_quant_pack_strided(const void* x, int dt, int units, int T, int D,
                                      const int32_t* gather, int gstride, int n, int bits, int G,
                                      int axis, int cap, uint32_t* codes, uint16_t* scale,
                                      uint16_t* zero, cudaStream_t s) {
    if (n == 0 || units == 0) return cudaSuccess;
    if (axis == KVQ_AXIS_CHANNEL) {
        dim3 grid(n / G, units);
        int threads = D < 256 ? ((D + 31) / 32) * 32 : 256;
        if (dt == KVQ_F16)
            quant_channel_kernel<__half><<<grid, threads, 0, s>>>(
                (const __half*)x, T, D, gather, gstride, n, bits, G, cap, codes, scale, zero);
        else
            quant_channel_kernel<__nv_bfloat16><<<grid, threads, 0, s>>>(
                (const __nv_bfloat16*)x, T, D, gather, gstride, n, bits, G, cap, codes, scale, zero);
    } else {
        size_t total = (size_t)units * n * (D / G);
        int threads = 128;
        size_t blocks = (total + threads - 1) / threads;
        if (blocks > 152 * 64) blocks = 152 * 64;
        if (dt == KVQ_F16)
            quant_token_kernel<__half><<<(unsigned)blocks, threads, 0, s>>>(
                (const __half*)x, T, D, gather, gstride, n, bits, G, cap, units, codes, scale, zero);
        else
            quant_token_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, s>>>(
                (const __nv_bfloat16*)x, T, D, gather, gstride, n, bits, G, cap, units, codes, scale,
                zero);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_pack(const void* x, int dt, int units, int T, int D,
                              const int32_t* gather, int n, int bits, int G, int axis,
                              uint32_t* codes, uint16_t* scale, uint16_t* zero, cudaStream_t s) {
    return launch_quant_pack_strided(x, dt, units, T, D, gather, n, n, bits, G, axis, n, codes,
                                     scale, zero, s);
}

}  // namespace kvq
