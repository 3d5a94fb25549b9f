// decode.cu -- decode-side ops around the pooled state cache:
//
//   * state slot copy: snapshot / restore of whole slots between two pools (the prefix-cache
//     state copies of the atlas page "serving-engine #69", SsmStatePool, and the rollback
//     of a speculative step);
//   * multi-token state update: k tokens per request in one pass over the state (the
//     decode-rollback ring of the same page: the state after every token can be kept,
//     so a caller that accepts only m of k draft tokens restores the m-th);
//   * fused decode layer step: state update, D skip and the silu-gated RMSNorm of
//     vt::Mamba2StateUpdate + vt::RmsNormGatedGroup (vllm.cpp page "W2 finish
//     (KERNEL-SSM-MAMBA)") in one kernel, so y never goes back to HBM.
//
// All three are HBM read-modify-write streams of fp32 state rows.  The update kernels use
// the layout of state_update.cu: a CTA of 256 threads per (request, head), each lane
// owning 4 consecutive n of a state row, N/4 lanes per row, shuffles for the y reduction
// over n.  The fused step gathers the heads of one norm group in a thread-block cluster:
// each CTA updates its heads, the CTAs exchange their partial sums of g^2 through
// distributed shared memory, and each CTA normalises its own channels.
#include <cooperative_groups.h>

#include <algorithm>

#include "ssd_internal.cuh"

namespace cg = cooperative_groups;

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
    for (int t = 0; t < ntok; ++t) {
      const size_t row = (size_t)b * ntok + t;
      float bv[4], cv[4], xv[KMAX];
      load4<TA>(reinterpret_cast<const TA*>(a.B) + (row * G + g) * N + 4 * q, bv);
      load4<TA>(reinterpret_cast<const TA*>(a.C) + (row * G + g) * N + 4 * q, cv);
      const TA* xr = reinterpret_cast<const TA*>(a.x) + (row * H + h) * P;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int p = p0 + k * RPI;
        xv[k] = p < P ? to_f32(xr[p]) : 0.f;
      }
      const float dt = dt_prep(a.dt[row * H + h], bias, a.dt_softplus);
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

// ------------------------------------------------------------- fused decode layer step

// silu(z) = z / (1 + e^-z).  bf16 activations take the fast exponential and division
// (relative error near 2^-21 over the range that matters); a tanh-based sigmoid is
// cheaper but loses relative accuracy where sigmoid(z) is small, which a large y then
// carries into the normalised output.  fp32 takes the full-precision form.
__device__ __forceinline__ float silu_of(float z, bool fast) {
  if (!fast) return z / (1.f + expf(-z));
  return __fdividef(z, 1.f + __expf(-z));
}

struct LayerParams {
  const void* z;
  const void* w;
  void* out;
  int group_size;  // channels per norm group (a whole number of heads)
  int hpc;         // heads per CTA
  float eps;
};

// Grid (ngroups * CS, batch), cluster (CS, 1, 1): the CS CTAs of a cluster share one
// norm group of one request; CTA `rank` owns heads [rank * hpc, (rank + 1) * hpc) of it.
template <typename TA, typename TW, int N>
__global__ void __launch_bounds__(256) decode_layer_kernel(const ssd_update_args a,
                                                           const LayerParams lp) {
  constexpr int LPR = N / 4, RPW = 32 / LPR, RPI = 8 * RPW, KMAX = 8;
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int grp = blockIdx.x / cs, b = blockIdx.y;
  const int H = a.H, P = a.P, G = a.G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q = lane % LPR, rw = lane / LPR;
  extern __shared__ float ys[];  // [hpc * P]: y of this CTA's channels, then g
  __shared__ float red[8];
  __shared__ float part;         // this CTA's sum of g^2, read by the whole cluster
  const int h0 = (grp * lp.group_size) / P + rank * lp.hpc;
  const size_t PN = (size_t)P * N;
  const size_t slot_stride = a.slot_stride ? (size_t)a.slot_stride : (size_t)H * PN;

  for (int hh = 0; hh < lp.hpc; ++hh) {
    const int h = h0 + hh;
    float* yh = ys + hh * P;
    const int s = slot_of(a, b, h);
    if (s < 0) {
      for (int p = threadIdx.x; p < P; p += blockDim.x) yh[p] = 0.f;
      continue;
    }
    const int g = h / (H / G);
    float bv[4], cv[4];
    load4<TA>(reinterpret_cast<const TA*>(a.B) + ((size_t)b * G + g) * N + 4 * q, bv);
    load4<TA>(reinterpret_cast<const TA*>(a.C) + ((size_t)b * G + g) * N + 4 * q, cv);
    const float dt = dt_prep(a.dt[(size_t)b * H + h], a.dt_bias ? a.dt_bias[h] : 0.f,
                             a.dt_softplus);
    const float dA = expf(dt * a.A[h]);
    const float Dh = a.D ? a.D[h] : 0.f;
    float* S = a.state_pool + (size_t)s * slot_stride + (size_t)h * PN;
    const TA* xb = reinterpret_cast<const TA*>(a.x) + ((size_t)b * H + h) * P;
    for (int base = warp * RPW; base < P; base += RPI * KMAX) {
      const int p0 = base + rw;
      float4 st[KMAX];
      float xv[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int p = p0 + k * RPI;
        if (p < P) {
          st[k] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)p * N + 4 * q));
          xv[k] = to_f32(xb[p]);
        } else {
          st[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          xv[k] = 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const int p = p0 + k * RPI;
        const float dx = dt * xv[k];
        float4 v = st[k];
        v.x = fmaf(dA, v.x, dx * bv[0]);
        v.y = fmaf(dA, v.y, dx * bv[1]);
        v.z = fmaf(dA, v.z, dx * bv[2]);
        v.w = fmaf(dA, v.w, dx * bv[3]);
        float acc = cv[0] * v.x;
        acc = fmaf(cv[1], v.y, acc);
        acc = fmaf(cv[2], v.z, acc);
        acc = fmaf(cv[3], v.w, acc);
        if (p < P) __stcs(reinterpret_cast<float4*>(S + (size_t)p * N + 4 * q), v);
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (p < P && q == 0) yh[p] = fmaf(Dh, xv[k], acc);
      }
    }
  }
  __syncthreads();
  // gate (y is optional output) and the partial sum of g^2
  const int nc = lp.hpc * P;
  const size_t c0 = (size_t)h0 * P;  // first channel of this CTA within the row
  const TA* zr = reinterpret_cast<const TA*>(lp.z) + (size_t)b * H * P + c0;
  TA* yout = a.y ? reinterpret_cast<TA*>(a.y) + (size_t)b * H * P + c0 : nullptr;
  constexpr bool kFast = sizeof(TA) == 2;
  float ss = 0.f;
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    if (yout) yout[c] = from_f32<TA>(ys[c]);
    const float gv = ys[c] * silu_of(to_f32(zr[c]), kFast);  // y stays fp32 here
    ys[c] = gv;
    ss = fmaf(gv, gv, ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    part = t;
  }
  cluster.sync();  // every CTA's partial sum is in place
  float total = 0.f;
  for (int r = 0; r < cs; ++r) total += *cluster.map_shared_rank(&part, r);
  const float inv = rsqrtf(total / (float)lp.group_size + lp.eps);
  const TW* wr = reinterpret_cast<const TW*>(lp.w) + (size_t)(grp * lp.group_size) +
                 (size_t)rank * nc;
  TA* orow = reinterpret_cast<TA*>(lp.out) + (size_t)b * H * P + c0;
  for (int c = threadIdx.x; c < nc; c += blockDim.x)
    orow[c] = from_f32<TA>(ys[c] * inv * to_f32(wr[c]));
  cluster.sync();  // no CTA leaves while another may still read its partial sum
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

template <typename TA, typename TW, int N>
cudaError_t launch_layer_n(const ssd_update_args& a, const LayerParams& lp, int cs,
                           cudaStream_t st) {
  const int ngroups = a.H * a.P / lp.group_size;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(ngroups * cs), (unsigned)a.batch);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = (size_t)lp.hpc * a.P * sizeof(float);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<TA, TW, N>, a, lp);
}

template <typename TA, typename TW>
cudaError_t launch_layer_t(const ssd_update_args& a, const LayerParams& lp, int cs,
                           cudaStream_t st) {
  switch (a.N) {
    case 128: return launch_layer_n<TA, TW, 128>(a, lp, cs, st);
    case 64: return launch_layer_n<TA, TW, 64>(a, lp, cs, st);
    case 32: return launch_layer_n<TA, TW, 32>(a, lp, cs, st);
    case 16: return launch_layer_n<TA, TW, 16>(a, lp, cs, st);
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

// Cluster size: the largest of 8, 4, 2, 1 that divides the heads of a norm group.
int decode_layer_cluster(int heads_per_group) {
  for (int cs : {8, 4, 2}) if (heads_per_group % cs == 0) return cs;
  return 1;
}

cudaError_t launch_decode_layer(const ssd_update_args& a, const void* z, const void* w,
                                ssd_dtype wt, int group_size, float eps, void* out,
                                cudaStream_t st) {
  const int hpg = group_size / a.P;
  const int cs = decode_layer_cluster(hpg);
  LayerParams lp{z, w, out, group_size, hpg / cs, eps};
  if (a.act_dtype == SSD_BF16)
    return wt == SSD_BF16 ? launch_layer_t<__nv_bfloat16, __nv_bfloat16>(a, lp, cs, st)
                          : launch_layer_t<__nv_bfloat16, float>(a, lp, cs, st);
  return wt == SSD_BF16 ? launch_layer_t<float, __nv_bfloat16>(a, lp, cs, st)
                        : launch_layer_t<float, float>(a, lp, cs, st);
}

}  // namespace ssd
