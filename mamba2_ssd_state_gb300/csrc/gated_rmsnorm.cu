// gated_rmsnorm.cu -- silu-gated RMSNorm with per-group variance (vt::RmsNormGatedGroup of
// the vllm.cpp page "W2 finish (KERNEL-SSM-MAMBA)"; its mutation rows M7 "whole-row
// variance, not per-group" and M8 "sigmoid instead of silu" fix the two parts).
//
//   g = x * silu(z);  out = g * rsqrt(mean_group(g^2) + eps) * w
//
// HBM-bound: x and z are read once and out written once (6 bytes per element in bf16).
// One warp owns one (row, group); in the vector path every lane keeps its
// VPT * 8 gated values in registers between the reduction and the write, so the op is a
// single pass over memory with 16-byte loads and stores and a warp-shuffle reduction.
//
// Launched as a programmatic dependent of the scan (the scan + norm call), a block may
// start while the scan is still running: it loads z, an input of the whole call, then
// waits (griddepcontrol.wait) for the scan to complete before it reads x, the scan's y.
// Launched plainly, the wait returns at once.
#include "ssd_internal.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }
// bf16 outputs carry 2^-9 relative rounding, so the bf16 path evaluates the sigmoid as
// 0.5 + 0.5 tanh(z/2) with the hardware tanh approximation (relative error about 2^-11,
// one special-function op instead of an exponential and a reciprocal); fp32 keeps expf
// and an IEEE division.
__device__ __forceinline__ float tanh_approx(float v) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float silu_fast(float z) {
  return z * fmaf(0.5f, tanh_approx(0.5f * z), 0.5f);
}
template <typename TA> __device__ __forceinline__ float gate(float z) {
  if constexpr (sizeof(TA) == 2) return silu_fast(z);
  else return silu(z);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// 8 activations per 16-byte vector (bf16) or two float4 (fp32).
template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float v[8]) {
    uint4 t = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&t);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float v[8]) {
    uint4 t;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&t);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = t;
  }
};
template <> struct Vec8<float> {
  static __device__ __forceinline__ void load(const float* p, float v[8]) {
    float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ void store(float* p, const float v[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

// group_size == TPG * 8 * VPT: the TPG threads of a group (one to eight warps) each hold
// VPT 8-element vectors, thread t vectors t + TPG i, so every load instruction of a warp
// covers 32 consecutive vectors (coalesced), and at most 4 vectors per thread keep the
// register count low enough for several blocks per SM.  Warp partial sums meet in
// shared memory when a group spans several warps.
template <typename TA, typename TW, int VPT, int TPG>
__global__ void __launch_bounds__(256) norm_vec_kernel(const TA* x,
                                                       const TA* __restrict__ z,
                                                       const TW* __restrict__ w, TA* out,
                                                       int64_t units, int d, int gs, float eps) {
  constexpr int GPB = 256 / TPG;  // groups per block
  __shared__ float part[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tig = threadIdx.x % TPG;
  const int64_t unit = (int64_t)blockIdx.x * GPB + threadIdx.x / TPG;
  const bool valid = unit < units;
  const int ngroups = d / gs;
  const int64_t row = valid ? unit / ngroups : 0;
  const int col0 = valid ? (int)(unit % ngroups) * gs : 0;
  const size_t base = (size_t)row * d + col0;
  float g[VPT][8];
  float ss = 0.f;
  if (valid && z) {  // z first: it may be read before the producer of x has finished
#pragma unroll
    for (int i = 0; i < VPT; ++i) Vec8<TA>::load(z + base + 8 * (tig + TPG * i), g[i]);
  }
  tc::griddep_wait();
  if (valid) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int off = 8 * (tig + TPG * i);
      float xv[8];
      Vec8<TA>::load(x + base + off, xv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        g[i][e] = z ? xv[e] * gate<TA>(g[i][e]) : xv[e];
        ss = fmaf(g[i][e], g[i][e], ss);
      }
    }
  }
  ss = warp_sum(ss);
  if constexpr (TPG > 32) {
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    constexpr int WPG = TPG / 32;  // warps per group
    const int w0 = (warp / WPG) * WPG;
    ss = 0.f;
#pragma unroll
    for (int k = 0; k < WPG; ++k) ss += part[w0 + k];
  }
  if (!valid) return;
  const float r = rsqrtf(ss / (float)gs + eps);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int off = 8 * (tig + TPG * i);
    float wv[8], o[8];
    Vec8<TW>::load(w + col0 + off, wv);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = g[i][e] * r * wv[e];
    Vec8<TA>::store(out + base + off, o);
  }
}

// Any group size: one warp per (row, group), two passes (the second re-reads x and z,
// which are still in L1/L2 for the group just reduced).
template <typename TA, typename TW>
__global__ void __launch_bounds__(256) norm_generic_kernel(const TA* x,
                                                           const TA* __restrict__ z,
                                                           const TW* __restrict__ w, TA* out,
                                                           int64_t units, int d, int gs,
                                                           float eps) {
  tc::griddep_wait();  // x may be the output of the kernel before (see norm_vec_kernel)
  const int64_t unit = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (unit >= units) return;
  const int lane = threadIdx.x & 31;
  const int ngroups = d / gs;
  const int64_t row = unit / ngroups;
  const int col0 = (int)(unit % ngroups) * gs;
  const size_t base = (size_t)row * d + col0;
  float ss = 0.f;
  for (int k = lane; k < gs; k += 32) {
    float gv = to_f32(x[base + k]);
    if (z) gv *= gate<TA>(to_f32(z[base + k]));
    ss = fmaf(gv, gv, ss);
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / (float)gs + eps);
  for (int k = lane; k < gs; k += 32) {
    float gv = to_f32(x[base + k]);
    if (z) gv *= gate<TA>(to_f32(z[base + k]));
    out[base + k] = from_f32<TA>(gv * r * to_f32(w[col0 + k]));
  }
}

// 256-thread blocks on `st`; with pdl the launch may begin before the previous kernel on
// the stream has completed (programmatic stream serialisation).
template <typename... P, typename... A>
cudaError_t launch256(void (*kernel)(P...), int64_t blocks, bool pdl, cudaStream_t st,
                      A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename TA, typename TW>
cudaError_t launch_typed(const void* x, const void* z, const void* w, void* out, int64_t rows,
                         int d, int gs, float eps, bool pdl, cudaStream_t st) {
  const int64_t units = rows * (int64_t)(d / gs);
  const int64_t blocks = (units + 7) / 8;
  const TA* xp = static_cast<const TA*>(x);
  const TA* zp = static_cast<const TA*>(z);
  const TW* wp = static_cast<const TW*>(w);
  TA* op = static_cast<TA*>(out);
  const bool aligned = ((uintptr_t)x % 16 == 0) && ((uintptr_t)out % 16 == 0) &&
                       (z == nullptr || (uintptr_t)z % 16 == 0) && ((uintptr_t)w % 16 == 0) &&
                       ((size_t)d * sizeof(TA)) % 16 == 0;
  // vector path: the smallest group of threads (32..256) with at most 4 vectors each
  int tpg = 0, vpt = 0;
  if (aligned && gs % 8 == 0) {
    for (int t = 32; t <= 256; t *= 2) {
      const int nvec = gs / 8;
      if (nvec % t == 0 && nvec / t <= 4) {
        tpg = t;
        vpt = nvec / t;
        break;
      }
    }
  }
  const int gpb = tpg ? 256 / tpg : 8;
  const int64_t vblocks = (units + gpb - 1) / gpb;
#define SSD_NORM_CASE(V, T)                                                                 \
  if (vpt == V && tpg == T)                                                                  \
    return launch256(norm_vec_kernel<TA, TW, V, T>, vblocks, pdl, st, xp, zp, wp, op, units, d, \
                     gs, eps);
  SSD_NORM_CASE(1, 32) SSD_NORM_CASE(2, 32) SSD_NORM_CASE(3, 32) SSD_NORM_CASE(4, 32)
  SSD_NORM_CASE(3, 64) SSD_NORM_CASE(4, 64) SSD_NORM_CASE(3, 128) SSD_NORM_CASE(4, 128)
  SSD_NORM_CASE(3, 256) SSD_NORM_CASE(4, 256)
#undef SSD_NORM_CASE
  return launch256(norm_generic_kernel<TA, TW>, blocks, pdl, st, xp, zp, wp, op, units, d, gs,
                   eps);
}

}  // namespace

cudaError_t launch_gated_rmsnorm(const void* x, const void* z, const void* w, void* out,
                                 int64_t rows, int d, int gs, float eps, ssd_dtype act,
                                 ssd_dtype wt, cudaStream_t st, bool pdl) {
  if (rows == 0) return cudaSuccess;
  using bf = __nv_bfloat16;
  if (act == SSD_BF16)
    return wt == SSD_BF16 ? launch_typed<bf, bf>(x, z, w, out, rows, d, gs, eps, pdl, st)
                          : launch_typed<bf, float>(x, z, w, out, rows, d, gs, eps, pdl, st);
  return wt == SSD_BF16 ? launch_typed<float, bf>(x, z, w, out, rows, d, gs, eps, pdl, st)
                        : launch_typed<float, float>(x, z, w, out, rows, d, gs, eps, pdl, st);
}

}  // namespace ssd
