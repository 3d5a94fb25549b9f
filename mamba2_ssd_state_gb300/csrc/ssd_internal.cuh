// ssd_internal.cuh -- declarations shared by the translation units of libssd.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdint>

#include "../../include/ssd.h"

namespace ssd {

// Activation load/store in fp32 registers.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// dt preprocessing: softplus(raw + bias) (log1p(e^v), identity above 20) or the plain sum.
__device__ __forceinline__ float dt_prep(float raw, float bias, int softplus) {
  float v = raw + bias;
  if (!softplus) return v;
  return v > 20.f ? v : log1pf(expf(v));
}

__device__ __forceinline__ void set_status(uint32_t* st, uint32_t bit) {
  if (st) atomicOr(st, bit);
}

// Launchers (each returns cudaSuccess or the launch error).
cudaError_t launch_state_update(const ssd_update_args& a, cudaStream_t s);
// pdl: launch as a programmatic dependent of the previous kernel on the stream (which
// must not write z or w; the kernel waits for it before reading x).
cudaError_t launch_gated_rmsnorm(const void* x, const void* z, const void* w, void* out,
                                 int64_t rows, int d, int gs, float eps, ssd_dtype act,
                                 ssd_dtype wt, cudaStream_t s, bool pdl = false);
cudaError_t launch_scan_simt(const ssd_scan_args& a, cudaStream_t s);

// Tensor-core scan: supported shapes, the workspace its plan wants (0 = no split) and the
// launch (SSD_ERR_UNSUPPORTED for shapes it cannot take, SSD_ERR_INVALID_ARG for a forced
// split without a large enough workspace).
// ws_limit caps the workspace of the splits the planner may choose (SIZE_MAX: no cap).
bool scan_tc_supported(const ssd_scan_args& a);
size_t scan_tc_workspace_size(const ssd_scan_args& a, size_t ws_limit = SIZE_MAX);
ssd_status launch_scan_tc(const ssd_scan_args& a, cudaStream_t s, size_t ws_limit = SIZE_MAX);

// Decode-side ops (decode.cu).
bool decode_n_supported(int N);
cudaError_t launch_state_copy(const float* src, int64_t src_stride, int src_slots,
                              const int32_t* src_idx, float* dst, int64_t dst_stride,
                              int dst_slots, const int32_t* dst_idx, int n, int64_t slot_elems,
                              uint32_t* status, cudaStream_t st);
cudaError_t launch_state_update_multi(const ssd_update_args& a, int ntok, float* inter,
                                      cudaStream_t st);
cudaError_t launch_decode_layer(const ssd_update_args& a, const void* z, const void* w,
                                ssd_dtype wt, int group_size, float eps, void* out,
                                cudaStream_t st);

// Library-owned scan scratch (scan_noalloc.cu): its size, and its address on the current
// device (NULL if the lookup failed).
size_t scan_static_scratch_bytes();
void* scan_static_scratch();

}  // namespace ssd
