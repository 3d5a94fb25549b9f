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

#ifndef SSD_WAIT_LIMIT_CYCLES
#define SSD_WAIT_LIMIT_CYCLES 4000000000LL  // about 2 s
#endif

// Hand-off of finished rows of y from the scan to the gated norm of the scan + norm call,
// so that the norm runs while the scan still works on later chunks.  For every 128-token
// chunk of every sequence and every norm group there is a counter: each output warp of
// the scan, once its 32 rows of one 64-channel head block of a chunk are written and
// ordered by a warp barrier, adds one to it (a release reduction nobody waits for), so a
// chunk-group is complete when its counter reaches 4 per 64-channel block of the group.
// The norm kernel takes
// chunk-groups in chunk-major order (chunk 0 of every sequence, then chunk 1, ...), as
// kReadyParts tasks of 32 rows, and polls each one's counter before it reads the rows.
// A split scan runs the segments of a sequence side by side, so there the order is chunk
// c of every segment of every sequence before chunk c + 1.
// Chunk ids: chunk c of sequence s (tokens from t0 = cu_seqlens[s]) is floor(t0 / 128) +
// s + c, distinct for nondecreasing cu_seqlens and below ceil(T / 128) + nseq.
constexpr int kReadyParts = 4;
struct ReadyQueue {
  int* cnt;       // [nid * ngroups] contributions so far (zeroed before the call)
  int* head;      // next task a norm block takes
  int* abort;     // set when a wait gave up: every later wait gives up at once
  long long nid;  // chunk ids: ceil(T / 128) + nseq
  int ngroups;    // norm groups per row
  int gs;         // channels per norm group
  int target;     // contributions that complete a chunk-group: 4 per 64 channels
  int segc;       // chunks per segment of a split scan (0: unsplit)
};
static_assert(128 % kReadyParts == 0, "tasks of whole rows");
// Count inc contributions to (chunk id, group): a reduction with release semantics at GPU
// scope (nobody waits for it).  Call after a warp or block barrier with every thread whose
// stores the contributions stand for: the barrier orders their stores before the caller's
// release, and a release carries what was ordered before it, so a reader that sees the
// count (and then fences) sees the stores.
__device__ __forceinline__ void ready_count(const ReadyQueue& rq, long long id, int grp,
                                            int inc) {
  if (id < 0 || id >= rq.nid) return;  // only for cu_seqlens that are not nondecreasing
  int* p = rq.cnt + id * rq.ngroups + grp;
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(inc) : "memory");
}
// Workspace of the counters for T tokens in nseq sequences (256-byte multiple; zero it
// before each call), and the counters laid out at ws.
size_t ready_queue_bytes(int64_t T, int nseq, int ngroups);
ReadyQueue ready_queue_at(void* ws, int64_t T, int nseq, int ngroups, int gs, int segc);

// Launchers (each returns cudaSuccess or the launch error).
cudaError_t launch_state_update(const ssd_update_args& a, cudaStream_t s);
// pdl: launch as a programmatic dependent of the previous kernel on the stream (which
// must not write z or w; the kernel waits for it before reading x).
cudaError_t launch_gated_rmsnorm(const void* x, const void* z, const void* w, void* out,
                                 int64_t rows, int d, int gs, float eps, ssd_dtype act,
                                 ssd_dtype wt, cudaStream_t s, bool pdl = false);
cudaError_t launch_scan_simt(const ssd_scan_args& a, cudaStream_t s);
// The gated norm that follows a ReadyQueue's counters (launched as a programmatic
// dependent of the scan that fills them; it does not wait for the scan's completion).  False when this
// activation / weight type, group size or alignment has no such kernel.
bool norm_ready_supported(const void* x, const void* z, const void* w, const void* out, int d,
                          int gs, ssd_dtype act);
cudaError_t launch_norm_ready(const void* x, const void* z, const void* w, void* out,
                              const int32_t* cu, int nseq, int T, int d, int gs, float eps,
                              ssd_dtype act, ssd_dtype wt, const ReadyQueue& rq,
                              uint32_t* status, cudaStream_t st);

// Tensor-core scan: supported shapes, the workspace its plan wants (0 = no split) and the
// launch (SSD_ERR_UNSUPPORTED for shapes it cannot take, SSD_ERR_INVALID_ARG for a forced
// split without a large enough workspace).
// ws_limit caps the workspace of the splits the planner may choose (SIZE_MAX: no cap).
bool scan_tc_supported(const ssd_scan_args& a);
size_t scan_tc_workspace_size(const ssd_scan_args& a, size_t ws_limit = SIZE_MAX);
ssd_status launch_scan_tc(const ssd_scan_args& a, cudaStream_t s, size_t ws_limit = SIZE_MAX);
// True when the call's plan (given the workspace it wants) runs a scan that can fill a
// ReadyQueue: 64-channel blocks, unsplit or split with two heads per CTA, in at most two
// waves of CTAs.  *split_bytes is then that split's workspace (0: unsplit) and *segc its
// segment length.  launch_scan_tc_ready launches it so (rq from ready_queue_at; the
// split's workspace in a.workspace).
bool scan_tc_ready_plan(const ssd_scan_args& a, size_t* split_bytes, int* segc);
ssd_status launch_scan_tc_ready(const ssd_scan_args& a, const ReadyQueue& rq, cudaStream_t s);

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
