// ssd_api.cu -- the C ABI of libssd.so (declared in include/ssd.h): host-side argument
// validation and kernel dispatch.  Nothing here computes any part of the ops; every
// step runs in the kernels of the other translation units.
#include <cstring>

#include "ssd_internal.cuh"

using namespace ssd;

namespace {

inline bool bad_dtype(ssd_dtype d) { return d != SSD_F32 && d != SSD_BF16; }

ssd_status validate_scan(const ssd_scan_args* a) {
  if (!a || a->struct_size < sizeof(ssd_scan_args)) return SSD_ERR_INVALID_ARG;
  if (!a->A || !a->cu_seqlens) return SSD_ERR_INVALID_ARG;
  if (a->T > 0 && (!a->x || !a->dt || !a->B || !a->C || !a->y)) return SSD_ERR_INVALID_ARG;
  if (a->nseq < 1 || a->T < 0 || a->H < 1 || a->P < 1 || a->G < 1 || a->N < 1)
    return SSD_ERR_INVALID_ARG;
  if (a->H % a->G != 0) return SSD_ERR_INVALID_ARG;
  if (a->chunk_size < 1 || a->chunk_size > 256) return SSD_ERR_INVALID_ARG;
  if (bad_dtype(a->act_dtype)) return SSD_ERR_INVALID_ARG;
  if (a->x_stride_t != 0 && a->x_stride_t < (int64_t)a->H * a->P) return SSD_ERR_INVALID_ARG;
  if (a->B_stride_t != 0 && a->B_stride_t < (int64_t)a->G * a->N) return SSD_ERR_INVALID_ARG;
  if (a->C_stride_t != 0 && a->C_stride_t < (int64_t)a->G * a->N) return SSD_ERR_INVALID_ARG;
  if (a->impl < SSD_IMPL_AUTO || a->impl > SSD_IMPL_TC) return SSD_ERR_INVALID_ARG;
  if (a->p_block != 0 && a->p_block != 16 && a->p_block != 32 && a->p_block != 64)
    return SSD_ERR_INVALID_ARG;
  if (a->seg_chunks < -1) return SSD_ERR_INVALID_ARG;
  if (a->head_block < 0 || a->head_block > 2) return SSD_ERR_INVALID_ARG;
  if (a->workspace_bytes > 0 && !a->workspace) return SSD_ERR_INVALID_ARG;
  if (a->nseq > 65535 || a->H > 65535) return SSD_ERR_UNSUPPORTED;  // grid limits
  return SSD_OK;
}

ssd_status validate_update(const ssd_update_args* a) {
  if (!a || a->struct_size < sizeof(ssd_update_args)) return SSD_ERR_INVALID_ARG;
  if (!a->state_pool || !a->A) return SSD_ERR_INVALID_ARG;
  if (a->batch > 0 &&
      (!a->state_indices || !a->x || !a->dt || !a->B || !a->C || !a->y))
    return SSD_ERR_INVALID_ARG;
  if (a->num_slots < 1 || a->batch < 0 || a->H < 1 || a->P < 1 || a->G < 1 || a->N < 1)
    return SSD_ERR_INVALID_ARG;
  if (a->H % a->G != 0) return SSD_ERR_INVALID_ARG;
  if (bad_dtype(a->act_dtype)) return SSD_ERR_INVALID_ARG;
  if (a->slot_stride != 0 && a->slot_stride < (int64_t)a->H * a->P * a->N)
    return SSD_ERR_INVALID_ARG;
  if (a->batch > 65535) return SSD_ERR_UNSUPPORTED;  // grid limit
  return SSD_OK;
}

// Workspace of the overlapped scan + norm (0 = the call runs the norm after the scan):
// the tensor-core scan unsplit in 64-channel blocks, bf16, a norm group of whole blocks,
// a norm kernel for this group size and alignment, and enough tokens: on short inputs
// the norm is short and the fixed costs (the counters' memset, the norm grid's tail)
// outweigh the overlap (one Nemotron-H sequence: 50 against 42 us at 1024 tokens, 73
// against 71 at 2048, 93 against 102 at 3072).
constexpr int32_t kReadyMinTokens = 3072;

// The workspace is the split's (if the plan splits), then the counters.
size_t gated_norm_ready_bytes(const ssd_scan_args& a, const void* z, const void* w,
                              int32_t group_size, const void* out, size_t* split_bytes,
                              int* segc) {
  const int64_t d = (int64_t)a.H * a.P;
  if (a.impl == SSD_IMPL_SIMT || a.act_dtype != SSD_BF16 || group_size % 64 != 0) return 0;
  if (a.T < kReadyMinTokens) return 0;
  // the norm's task counter (an int) runs over chunk positions x sequences x groups x
  // parts; chunk positions are at most ceil(T / 128), or twice that when split (whole
  // segments of positions)
  const int64_t positions = ((int64_t)a.T + 127) / 128 * a.nseq * 2;
  if (positions * (d / group_size) * kReadyParts >= 0x7f000000LL) return 0;  // + the grid
  if (!norm_ready_supported(a.y, z, w, out, (int)d, group_size, a.act_dtype)) return 0;
  if (!scan_tc_ready_plan(a, split_bytes, segc)) return 0;
  return *split_bytes + ready_queue_bytes(a.T, a.nseq, (int)(d / group_size));
}

}  // namespace

extern "C" {

ssd_status ssd_chunk_scan(const ssd_scan_args* args, ssd_stream_t stream) {
  ssd_status v = validate_scan(args);
  if (v != SSD_OK) return v;
  const ssd_scan_args& a = *args;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool tc_ok = scan_tc_supported(a);
  if (a.impl == SSD_IMPL_TC || (a.impl == SSD_IMPL_AUTO && tc_ok)) {
    if (!tc_ok) return SSD_ERR_UNSUPPORTED;
    return launch_scan_tc(a, st);
  }
  if (a.N > 256) return SSD_ERR_UNSUPPORTED;
  return launch_scan_simt(a, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_chunk_scan_static_ws(const ssd_scan_args* args, ssd_stream_t stream) {
  ssd_status v = validate_scan(args);
  if (v != SSD_OK) return v;
  const ssd_scan_args& a = *args;
  if (a.workspace || a.workspace_bytes) return SSD_ERR_INVALID_ARG;  // the library's own
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool tc_ok = scan_tc_supported(a);
  if (a.impl == SSD_IMPL_TC || (a.impl == SSD_IMPL_AUTO && tc_ok)) {
    if (!tc_ok) return SSD_ERR_UNSUPPORTED;
    const size_t cap = scan_static_scratch_bytes();
    // an explicit split must fit the array; the automatic plan keeps to it
    if (a.seg_chunks >= 1 && scan_tc_workspace_size(a) > cap) return SSD_ERR_UNSUPPORTED;
    const size_t need = scan_tc_workspace_size(a, cap);
    ssd_scan_args b = a;
    if (need > 0) {
      b.workspace = scan_static_scratch();
      if (!b.workspace) return SSD_ERR_CUDA;
      b.workspace_bytes = cap;
    }
    return launch_scan_tc(b, st, cap);
  }
  if (a.N > 256) return SSD_ERR_UNSUPPORTED;
  return launch_scan_simt(a, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_chunk_scan_gated_norm(const ssd_scan_args* args, const void* z,
                                     const void* norm_weight, ssd_dtype weight_dtype,
                                     int32_t group_size, float eps, void* out,
                                     ssd_stream_t stream) {
  if (!args || args->struct_size < sizeof(ssd_scan_args)) return SSD_ERR_INVALID_ARG;
  ssd_scan_args a = *args;  // y is optional here: the scan then writes into out
  if (!a.y) a.y = out;
  ssd_status v = validate_scan(&a);
  if (v != SSD_OK) return v;
  const int64_t d = (int64_t)a.H * a.P;
  if (!norm_weight || bad_dtype(weight_dtype) || !(eps >= 0.f)) return SSD_ERR_INVALID_ARG;
  if (group_size < 1 || d % group_size != 0) return SSD_ERR_INVALID_ARG;
  if (d > 0x7fffffffLL || ((int64_t)a.T * (d / group_size) + 7) / 8 > 0x7fffffffLL)
    return SSD_ERR_UNSUPPORTED;  // grid limits of the norm
  if (a.T == 0) return ssd_chunk_scan(&a, stream);  // final states only
  // the norm may read z while the scan still runs: z must not share bytes with y or out
  const size_t bytes = (size_t)a.T * (size_t)d * (a.act_dtype == SSD_BF16 ? 2 : 4);
  auto overlap = [bytes](const void* p, const void* q) {
    const uintptr_t u = (uintptr_t)p, w = (uintptr_t)q;
    return u < w + bytes && w < u + bytes;
  };
  if (z && (overlap(z, a.y) || overlap(z, out))) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the overlapped form: the norm consumes the scan's finished chunks while it runs
  size_t split_bytes = 0;
  int segc = 0;
  const size_t need =
      gated_norm_ready_bytes(a, z, norm_weight, group_size, out, &split_bytes, &segc);
  if (need > 0 && a.workspace && ((uintptr_t)a.workspace & 255u) == 0 &&
      a.workspace_bytes >= need) {
    const int ngroups = (int)(d / group_size);
    void* counters = static_cast<char*>(a.workspace) + split_bytes;
    if (cudaMemsetAsync(counters, 0, need - split_bytes, st) != cudaSuccess) return SSD_ERR_CUDA;
    const ReadyQueue rq = ready_queue_at(counters, a.T, a.nseq, ngroups, group_size, segc);
    ssd_scan_args b = a;  // the scan sees the split's part of the workspace only
    b.workspace = split_bytes ? a.workspace : nullptr;
    b.workspace_bytes = split_bytes;
    v = launch_scan_tc_ready(b, rq, st);
    if (v != SSD_OK) return v;
    return launch_norm_ready(a.y, z, norm_weight, out, a.cu_seqlens, a.nseq, a.T, (int)d,
                             group_size, eps, a.act_dtype, weight_dtype, rq, a.d_status,
                             st) == cudaSuccess
               ? SSD_OK
               : SSD_ERR_CUDA;
  }
  v = ssd_chunk_scan(&a, stream);
  if (v != SSD_OK) return v;
  return launch_gated_rmsnorm(a.y, z, norm_weight, out, a.T, (int)d, group_size, eps,
                              a.act_dtype, weight_dtype, st, /*pdl=*/true) == cudaSuccess
             ? SSD_OK
             : SSD_ERR_CUDA;
}

size_t ssd_chunk_scan_gated_norm_workspace_size(const ssd_scan_args* args, const void* z,
                                                const void* norm_weight, int32_t group_size,
                                                const void* out) {
  if (!args || args->struct_size < sizeof(ssd_scan_args)) return 0;
  ssd_scan_args a = *args;
  if (!a.y) a.y = const_cast<void*>(out);  // only its address is looked at
  if (validate_scan(&a) != SSD_OK || a.T == 0 || !norm_weight || !out) return 0;
  const int64_t d = (int64_t)a.H * a.P;
  if (group_size < 1 || d % group_size != 0) return 0;
  // the overlapped form's (its split's and the counters), else a split the scan would
  // choose (the norm then follows the scan)
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  size_t split_bytes = 0;
  int segc = 0;
  const size_t ready =
      gated_norm_ready_bytes(a, z, norm_weight, group_size, out, &split_bytes, &segc);
  if (ready > 0) return ready;
  return a.impl == SSD_IMPL_SIMT ? 0 : scan_tc_workspace_size(a);
}

size_t ssd_chunk_scan_workspace_size(const ssd_scan_args* args) {
  if (validate_scan(args) != SSD_OK) return 0;
  const ssd_scan_args& a = *args;
  if (a.impl == SSD_IMPL_SIMT) return 0;
  return scan_tc_workspace_size(a);
}

ssd_status ssd_state_update(const ssd_update_args* args, ssd_stream_t stream) {
  ssd_status v = validate_update(args);
  if (v != SSD_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_state_update(*args, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_state_copy(const float* src_pool, int64_t src_slot_stride, int32_t src_slots,
                          const int32_t* src_idx, float* dst_pool, int64_t dst_slot_stride,
                          int32_t dst_slots, const int32_t* dst_idx, int32_t n,
                          int64_t slot_elems, uint32_t* d_status, ssd_stream_t stream) {
  if (n < 0 || slot_elems < 1 || src_slots < 1 || dst_slots < 1) return SSD_ERR_INVALID_ARG;
  if (n == 0) return SSD_OK;
  if (!src_pool || !dst_pool || !src_idx || !dst_idx) return SSD_ERR_INVALID_ARG;
  const int64_t ss = src_slot_stride ? src_slot_stride : slot_elems;
  const int64_t ds = dst_slot_stride ? dst_slot_stride : slot_elems;
  if (ss < slot_elems || ds < slot_elems) return SSD_ERR_INVALID_ARG;
  // float4 copies: 16-byte aligned slots
  if (slot_elems % 4 || ss % 4 || ds % 4 || ((uintptr_t)src_pool & 15u) ||
      ((uintptr_t)dst_pool & 15u))
    return SSD_ERR_UNSUPPORTED;
  if (n > 65535) return SSD_ERR_UNSUPPORTED;  // grid limit
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_state_copy(src_pool, ss, src_slots, src_idx, dst_pool, ds, dst_slots, dst_idx, n,
                           slot_elems, d_status, st) == cudaSuccess
             ? SSD_OK
             : SSD_ERR_CUDA;
}

ssd_status ssd_state_update_multi(const ssd_update_args* args, int32_t ntok,
                                  float* inter_states, ssd_stream_t stream) {
  ssd_status v = validate_update(args);
  if (v != SSD_OK) return v;
  if (ntok < 1) return SSD_ERR_INVALID_ARG;
  const ssd_update_args& a = *args;
  if (a.batch == 0) return SSD_OK;
  if (!decode_n_supported(a.N)) return SSD_ERR_UNSUPPORTED;
  if (a.slot_stride % 4 || ((uintptr_t)a.state_pool & 15u) || ((uintptr_t)inter_states & 15u))
    return SSD_ERR_UNSUPPORTED;
  // B and C are read four values at a time: rows must start on that boundary
  const uintptr_t vec = 4u * (a.act_dtype == SSD_BF16 ? 2u : 4u);
  if (((uintptr_t)a.B % vec) || ((uintptr_t)a.C % vec)) return SSD_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_state_update_multi(a, ntok, inter_states, st) == cudaSuccess ? SSD_OK
                                                                             : SSD_ERR_CUDA;
}

ssd_status ssd_decode_layer_step(const ssd_update_args* args, const void* z,
                                 const void* norm_weight, ssd_dtype weight_dtype,
                                 int32_t group_size, float eps, void* out,
                                 ssd_stream_t stream) {
  if (!args || args->struct_size < sizeof(ssd_update_args)) return SSD_ERR_INVALID_ARG;
  ssd_update_args chk = *args;  // y is optional here
  if (!chk.y) chk.y = out;
  ssd_status v = validate_update(&chk);
  if (v != SSD_OK) return v;
  const ssd_update_args& a = *args;
  if (!norm_weight || bad_dtype(weight_dtype) || !(eps >= 0.f)) return SSD_ERR_INVALID_ARG;
  if (group_size < a.P || group_size % a.P || (a.H * a.P) % group_size)
    return SSD_ERR_INVALID_ARG;
  if (a.batch > 0 && (!z || !out)) return SSD_ERR_INVALID_ARG;
  if (a.batch == 0) return SSD_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_decode_layer(a, z, norm_weight, weight_dtype, group_size, eps, out, st) ==
                 cudaSuccess
             ? SSD_OK
             : SSD_ERR_CUDA;
}

ssd_status gated_rmsnorm(const void* x, const void* z, const void* weight, void* out,
                         int64_t rows, int32_t d, int32_t group_size, float eps, ssd_dtype act,
                         ssd_dtype wt, ssd_stream_t stream) {
  if (!weight || rows < 0 || d < 1 || group_size < 1 || d % group_size != 0)
    return SSD_ERR_INVALID_ARG;
  if (rows > 0 && (!x || !out)) return SSD_ERR_INVALID_ARG;
  if (bad_dtype(act) || bad_dtype(wt) || !(eps >= 0.f)) return SSD_ERR_INVALID_ARG;
  if ((rows * (int64_t)(d / group_size) + 7) / 8 > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return launch_gated_rmsnorm(x, z, weight, out, rows, d, group_size, eps, act, wt, st) ==
                 cudaSuccess
             ? SSD_OK
             : SSD_ERR_CUDA;
}

ssd_status ssd_read_status(uint32_t* d_status, int32_t clear, uint32_t* bits_out,
                           ssd_stream_t stream) {
  if (!d_status) return SSD_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  if (cudaMemcpyAsync(&bits, d_status, sizeof(bits), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return SSD_ERR_CUDA;
  if (clear && cudaMemsetAsync(d_status, 0, sizeof(uint32_t), st) != cudaSuccess)
    return SSD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
  if (bits_out) *bits_out = bits;
  if (bits & SSD_DEV_A_NOT_NEG) return SSD_ERR_A_NOT_NEGATIVE;
  if (bits & SSD_DEV_INDEX_OOR) return SSD_ERR_INDEX;
  if (bits & SSD_DEV_SEQ_META) return SSD_ERR_SEQ_META;
  if (bits & SSD_DEV_TIMEOUT) return SSD_ERR_TIMEOUT;
  return SSD_OK;
}

const char* ssd_status_string(ssd_status s) {
  switch (s) {
    case SSD_OK: return "SSD_OK";
    case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG";
    case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED";
    case SSD_ERR_A_NOT_NEGATIVE: return "SSD_ERR_A_NOT_NEGATIVE";
    case SSD_ERR_INDEX: return "SSD_ERR_INDEX";
    case SSD_ERR_SEQ_META: return "SSD_ERR_SEQ_META";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA";
    case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT";
  }
  return "SSD_ERR_UNKNOWN";
}

int32_t ssd_version(void) { return 100; }

}  // extern "C"
