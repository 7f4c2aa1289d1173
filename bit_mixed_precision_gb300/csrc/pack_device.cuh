// Device routines that quantise and pack one group, used by kv_quant_pack
// and by the policy kernels (prefill-end build, residual flush, tier moves).
#pragma once

#include "kvq_common.cuh"

namespace kvq {

// Channel grouping: a group is G consecutive rows (tokens) of one channel c.
// row(i) returns a pointer to the D elements of token i of the group.
// Words are written at codes[w * D + c] for w < G*bits/32 (packed along
// tokens, LSB first); scale/zero at *s_out / *z_out.
template <typename T, typename RowFn>
__device__ __forceinline__ void quant_channel_group(RowFn row, int G, int c, int bits,
                                                    uint32_t* codes, int D, uint16_t* s_out,
                                                    uint16_t* z_out) {
    float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
    for (int i = 0; i < G; ++i) {
        float x = Elem<T>::to_f(row(i)[c]);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
    }
    QParams p = quant_params(__fadd_rn(mn, 0.0f), __fadd_rn(mx, 0.0f), bits);
    const int per = 32 / bits;
    for (int w = 0; w < G / per; ++w) {
        uint32_t word = 0;
        for (int k = 0; k < per; ++k) {
            float x = Elem<T>::to_f(row(w * per + k)[c]);
            word |= quant_code(x, p, bits) << (bits * k);
        }
        codes[(size_t)w * D + c] = word;
    }
    *s_out = p.s_bits;
    *z_out = p.z_bits;
}

// Token grouping: G consecutive channels of one token.  src points at the
// first of the G elements (any float-convertible source via Load), codes at
// the first of its G*bits/32 words.
template <typename Load>
__device__ __forceinline__ void quant_token_group(Load load, int G, int bits, uint32_t* codes,
                                                  uint16_t* s_out, uint16_t* z_out) {
    float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
    for (int i = 0; i < G; ++i) {
        float x = load(i);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
    }
    QParams p = quant_params(__fadd_rn(mn, 0.0f), __fadd_rn(mx, 0.0f), bits);
    const int per = 32 / bits;
    for (int w = 0; w < G / per; ++w) {
        uint32_t word = 0;
        for (int k = 0; k < per; ++k) word |= quant_code(load(w * per + k), p, bits) << (bits * k);
        codes[w] = word;
    }
    *s_out = p.s_bits;
    *z_out = p.z_bits;
}

// Groups of 32 held in registers (every value loaded once): the quantiser
// parameters of the group, and its BITS words written at out[w * stride].
template <int BITS>
__device__ __forceinline__ void pack32(const float (&v)[32], const QParams& p, uint32_t* out, size_t stride) {
    constexpr int per = 32 / BITS;
#pragma unroll
    for (int w = 0; w < BITS; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < per; ++k) word |= quant_code(v[w * per + k], p, BITS) << (BITS * k);
        out[(size_t)w * stride] = word;
    }
}

__device__ __forceinline__ QParams params32(const float (&v)[32], int bits) {
    float mn = __int_as_float(0x7f800000), mx = -__int_as_float(0x7f800000);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        mn = fminf(mn, v[i]);
        mx = fmaxf(mx, v[i]);
    }
    return quant_params(__fadd_rn(mn, 0.0f), __fadd_rn(mx, 0.0f), bits);
}

// Code k of a token-grouped packed row.
__device__ __forceinline__ uint32_t code_at(const uint32_t* words, int k, int bits) {
    const int per = 32 / bits;
    return (words[k / per] >> (bits * (k % per))) & ((1u << bits) - 1u);
}

}  // namespace kvq
