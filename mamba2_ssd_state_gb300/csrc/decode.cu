// decode.cu -- decode-side ops around the pooled state cache:
//
//   * state slot copy: snapshot / restore of whole slots between two pools (the prefix-cache
//     state copies of the atlas page "serving-engine #69", SsmStatePool, and the rollback
//     of a speculative step);
//   * multi-token state update: k tokens per request in one pass over the state (the
//     decode-rollback ring of the same page: the state after every token can be kept,
//     so a caller that accepts only m of k draft tokens restores the m-th);
//   * decode layer step: state update, D skip and the silu-gated RMSNorm of
//     vt::Mamba2StateUpdate + vt::RmsNormGatedGroup (vllm.cpp page "W2 finish
//     (KERNEL-SSM-MAMBA)") behind one call.
//
// The copy and the multi-token update are HBM streams of fp32 state rows.  The update uses
// the layout of state_update.cu: a CTA of 256 threads per (request, head), each lane
// owning 4 consecutive n of a state row, N/4 lanes per row, shuffles for the y reduction
// over n.
#include <algorithm>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

// ------------------------------------------------------------------------- slot copy

constexpr int kCopyThreads = 256, kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) state_copy_kernel(
    const float* __restrict__ src, int64_t src_stride, int src_slots,
    const int32_t* __restrict__ src_idx, float* __restrict__ dst, int64_t dst_stride,
    int dst_slots, const int32_t* __restrict__ dst_idx, int64_t nvec, uint32_t* status) {
  const int i = blockIdx.y;
  const int s = src_idx[i], d = dst_idx[i];
  const bool oor = s < -1 || s >= src_slots || d < -1 || d >= dst_slots;
  if (oor) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, SSD_DEV_INDEX_OOR);
    return;
  }
  if (s < 0 || d < 0) return;  // a -1 on either side: nothing to copy
  const float4* sp = reinterpret_cast<const float4*>(src + (size_t)s * src_stride);
  float4* dp = reinterpret_cast<float4*>(dst + (size_t)d * dst_stride);
  const int64_t step = (int64_t)gridDim.x * kCopyThreads * kCopyUnroll;
  for (int64_t v0 = (int64_t)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x; v0 < nvec;
       v0 += step) {
    float4 t[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {  // every load before any store
      const int64_t v = v0 + (int64_t)u * kCopyThreads;
      if (v < nvec) t[u] = __ldcs(sp + v);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t v = v0 + (int64_t)u * kCopyThreads;
      if (v < nvec) dp[v] = t[u];
    }
  }
}

// ------------------------------------------------------------ shared update helpers

template <typename TA>
__device__ __forceinline__ void load4(const TA* p, float v[4]) {
  if constexpr (sizeof(TA) == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
    const uint2 t = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  }
}

// The slot a request updates, or -1 (a -1 row, an out-of-range slot, or a head whose A is
// not < 0: those never touch the pool); thread 0 raises the status bits.
__device__ __forceinline__ int slot_of(const ssd_update_args& a, int b, int h) {
  const int s = a.state_indices[b];
  const bool oor = s < -1 || s >= a.num_slots;
  const bool a_ok = a.A[h] < 0.f;  // sign test: NaN, +0 and -0 fail
  if (threadIdx.x == 0) {
    if (oor) set_status(a.d_status, SSD_DEV_INDEX_OOR);
    if (!a_ok) set_status(a.d_status, SSD_DEV_A_NOT_NEG);
  }
  return (s >= 0 && !oor && a_ok) ? s : -1;
}

// ---------------------------------------------------------------- multi-token update

// Token t of request b sits at row b * ntok + t of x, dt, B, C and y.
template <typename TA, int N>
__global__ void __launch_bounds__(256) state_update_multi_kernel(const ssd_update_args a,
                                                                 int ntok, float* inter) {
  constexpr int LPR = N / 4;     // lanes per state row
  constexpr int RPW = 32 / LPR;  // rows per warp
  constexpr int RPI = 8 * RPW;   // rows per CTA pass
  constexpr int KMAX = 8;        // state rows (float4 each) a thread keeps in registers
  const int h = blockIdx.x, b = blockIdx.y;
  const int H = a.H, P = a.P, G = a.G;
  const int s = slot_of(a, b, h);
  if (s < 0) {  // y of every token is 0
    for (int e = threadIdx.x; e < ntok * P; e += blockDim.x)
      reinterpret_cast<TA*>(a.y)[(((size_t)b * ntok + e / P) * H + h) * P + e % P] =
          from_f32<TA>(0.f);
    return;
  }
  const int g = h / (H / G);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q = lane % LPR, rw = lane / LPR;
  const float Ah = a.A[h], Dh = a.D ? a.D[h] : 0.f, bias = a.dt_bias ? a.dt_bias[h] : 0.f;
  const size_t PN = (size_t)P * N;
  const size_t slot_stride = a.slot_stride ? (size_t)a.slot_stride : (size_t)H * PN;
  float* S = a.state_pool + (size_t)s * slot_stride + (size_t)h * PN;

  for (int base = warp * RPW; base < P; base += RPI * KMAX) {  // warp-uniform
    const int p0 = base + rw;
    float4 st[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int p = p0 + k * RPI;
      st[k] = p < P ? __ldcs(reinterpret_cast<const float4*>(S + (size_t)p * N + 4 * q))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // a token's small inputs (B, C, x, dt) are loaded one token ahead
    float bn[4], cn[4], xn[KMAX], dtn;
    auto load_tok = [&](int t) {
      const size_t row = (size_t)b * ntok + t;
      load4<TA>(reinterpret_cast<const TA*>(a.B) + (row * G + g) * N + 4 * q, bn);
      load4<TA>(reinterpret_cast<const TA*>(a.C) + (row * G + g) * N + 4 * q, cn);
      const TA* xr = reinterpret_cast<const TA*>(a.x) + (row * H + h) * P;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int p = p0 + k * RPI;
        xn[k] = p < P ? to_f32(xr[p]) : 0.f;
      }
      dtn = a.dt[row * H + h];
    };
    load_tok(0);
    for (int t = 0; t < ntok; ++t) {
      const size_t row = (size_t)b * ntok + t;
      float bv[4], cv[4], xv[KMAX];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bv[k] = bn[k];
        cv[k] = cn[k];
      }
#pragma unroll
      for (int k = 0; k < KMAX; ++k) xv[k] = xn[k];
      const float dt = dt_prep(dtn, bias, a.dt_softplus);
      if (t + 1 < ntok) load_tok(t + 1);
      const float dA = expf(dt * Ah);
      TA* yr = reinterpret_cast<TA*>(a.y) + (row * H + h) * P;
      float* ir = inter ? inter + (row * H + h) * PN : nullptr;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int p = p0 + k * RPI;
        const float dx = dt * xv[k];
        float4& v = st[k];
        v.x = fmaf(dA, v.x, dx * bv[0]);
        v.y = fmaf(dA, v.y, dx * bv[1]);
        v.z = fmaf(dA, v.z, dx * bv[2]);
        v.w = fmaf(dA, v.w, dx * bv[3]);
        float acc = cv[0] * v.x;
        acc = fmaf(cv[1], v.y, acc);
        acc = fmaf(cv[2], v.z, acc);
        acc = fmaf(cv[3], v.w, acc);
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (p < P) {
          if (q == 0) yr[p] = from_f32<TA>(fmaf(Dh, xv[k], acc));
          if (ir) __stcs(reinterpret_cast<float4*>(ir + (size_t)p * N + 4 * q), v);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int p = p0 + k * RPI;
      if (p < P) __stcs(reinterpret_cast<float4*>(S + (size_t)p * N + 4 * q), st[k]);
    }
  }
}

template <typename TA, int N>
cudaError_t launch_multi_n(const ssd_update_args& a, int ntok, float* inter, cudaStream_t st) {
  state_update_multi_kernel<TA, N><<<dim3(a.H, a.batch), 256, 0, st>>>(a, ntok, inter);
  return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_multi_t(const ssd_update_args& a, int ntok, float* inter, cudaStream_t st) {
  switch (a.N) {
    case 128: return launch_multi_n<TA, 128>(a, ntok, inter, st);
    case 64: return launch_multi_n<TA, 64>(a, ntok, inter, st);
    case 32: return launch_multi_n<TA, 32>(a, ntok, inter, st);
    case 16: return launch_multi_n<TA, 16>(a, ntok, inter, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool decode_n_supported(int N) { return N == 16 || N == 32 || N == 64 || N == 128; }

cudaError_t launch_state_copy(const float* src, int64_t src_stride, int src_slots,
                              const int32_t* src_idx, float* dst, int64_t dst_stride,
                              int dst_slots, const int32_t* dst_idx, int n, int64_t slot_elems,
                              uint32_t* status, cudaStream_t st) {
  const int64_t nvec = slot_elems / 4;
  const int64_t per_block = (int64_t)kCopyThreads * kCopyUnroll;
  const unsigned gx = (unsigned)std::min<int64_t>(256, (nvec + per_block - 1) / per_block);
  state_copy_kernel<<<dim3(gx, (unsigned)n), kCopyThreads, 0, st>>>(
      src, src_stride, src_slots, src_idx, dst, dst_stride, dst_slots, dst_idx, nvec, status);
  return cudaGetLastError();
}

cudaError_t launch_state_update_multi(const ssd_update_args& a, int ntok, float* inter,
                                      cudaStream_t st) {
  return a.act_dtype == SSD_BF16 ? launch_multi_t<__nv_bfloat16>(a, ntok, inter, st)
                                 : launch_multi_t<float>(a, ntok, inter, st);
}

// One decode token of a mixer layer after its projections: the state update writes y
// (into `out` when the caller does not want y: the norm then runs in place, each element
// read before it is written by the same thread), then the gated norm.  A kernel that
// fused the two through a thread-block cluster per norm group measured slower at every
// batch size on GB300 (batch 256 of 128 heads: 472 us vs 295 us; batch 1: 6.1 vs 5.6 us,
// CUDA-graph timed): y's round trip is under 2% of the state traffic, and the cluster
// serialised each CTA's heads.
cudaError_t launch_decode_layer(const ssd_update_args& a, const void* z, const void* w,
                                ssd_dtype wt, int group_size, float eps, void* out,
                                cudaStream_t st) {
  ssd_update_args u = a;
  if (!u.y) u.y = out;
  cudaError_t e = launch_state_update(u, st);
  if (e != cudaSuccess) return e;
  return launch_gated_rmsnorm(u.y, z, w, out, (int64_t)a.batch, a.H * a.P, group_size, eps,
                              a.act_dtype, wt, st);
}

}  // namespace ssd
