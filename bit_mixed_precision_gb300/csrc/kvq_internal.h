// Host-side declarations shared by the translation units of libkvq.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

// Records the thread-local message returned by kvq_last_error().
void set_error(const char* fmt, ...);

cudaError_t launch_quant_pack(const void* x, int dt, int units, int T, int D,
                              const int32_t* gather, int n, int bits, int G, int axis,
                              uint32_t* codes, uint16_t* scale, uint16_t* zero, cudaStream_t s);

// Same with a gather row stride and an output capacity (tokens per unit of
// the destination buffers); the first n gathered rows are packed.
cudaError_t launch_quant_pack_strided(const void* x, int dt, int units, int T, int D,
                                      const int32_t* gather, int gstride, int n, int bits, int G,
                                      int axis, int cap, uint32_t* codes, uint16_t* scale,
                                      uint16_t* zero, cudaStream_t s);

// o == NULL: pass 2 only (lse given).  q_first: the first query counted in colscore.
kvq_status run_prefill(const void* q, const void* k, const void* v, int dt, int B, int Hq,
                       int Hkv, int T, int D, float sm_scale, void* o, float* lse,
                       float* colscore, int q_first, cudaStream_t s);

cudaError_t launch_select(const float* score, int units, int T, const int32_t* k_hh, int kmax,
                          int w, int32_t* idx_out, int32_t* n_out, cudaStream_t s);

cudaError_t launch_score_reduce(const float* cs, int B, int Hq, int Hkv, int T, int mode,
                                float* out, cudaStream_t s);

size_t decode_workspace_bytes(const kvq_cache& c);
int decode_launches(const kvq_cache& c);
void set_withhold_copy(int on);
cudaError_t launch_decode(const void* q, const void* k_new, const void* v_new, const kvq_cache& c,
                          float sm_scale, void* o, float* lse_out, void* ws, cudaStream_t s);

// Device address of the library's static decode scratch on the current device.
cudaError_t static_decode_scratch(void** out);

kvq_status run_policy(const kvq_cache& c, int mode, const kvq_policy_params* p, int step,
                      cudaStream_t s);

// DiffKV page pools: reset, and release of finished units.
kvq_status run_pages_init(const kvq_cache& c, cudaStream_t s);
kvq_status run_pages_release(const kvq_cache& c, const int32_t* mask, cudaStream_t s);

// MiniKV prefill-end build from column scores in one launch (selection + packing + residual).
kvq_status run_minikv_fused_build(const kvq_cache& c, const void* k, const void* v, int T, const float* score,
                                  const int32_t* k_hh, int kmax, int w, int32_t* idx_out, cudaStream_t s);

}  // namespace kvq
