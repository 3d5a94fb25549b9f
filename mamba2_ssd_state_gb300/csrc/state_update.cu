// state_update.cu -- decode-time selective state update over a pooled fp32 state cache
// (vt::Mamba2StateUpdate of the vllm.cpp page "W2 finish (KERNEL-SSM-MAMBA)"; mutation
// table rows M5 "ignore state_indices", M6 "NULL row as slot 0", M9 "drop the A < 0
// check" fix its index and sign handling).
//
// The op is a pure HBM read-modify-write: each active (row, head) streams its
// [P, N] fp32 slot state once in and once out (2 * 4 * P * N bytes), everything else
// is small.  Design for GB300:
//   * one CTA of 256 threads per (row b, head h); grid (H, batch);
//   * each lane owns 4 consecutive n of a state row (one 16-byte float4); N/4 lanes
//     share a row, so the y reduction over n is a shuffle within those lanes;
//   * all KMAX float4 loads of a thread are issued before any arithmetic (up to 32 KB
//     per CTA in flight), with streaming cache hints since every byte is touched once;
//   * -1 rows, out-of-range slots and heads with A not < 0 never touch the pool.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

template <typename TA>
__device__ __forceinline__ void load4(const TA* p, float v[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float v[4]) {
  float4 t = *reinterpret_cast<const float4*>(p);
  v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float v[4]) {
  uint2 t = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&t.x);
  __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162*>(&t.y);
  float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}

// Returns the slot to update, or -1 when this (b, h) must not touch the pool (in which
// case y[b, h, :] is zeroed and the status bits are set by thread 0).
template <typename TA>
__device__ __forceinline__ int guard_row(const ssd_update_args& a, int b, int h) {
  const int s = a.state_indices[b];
  const bool oor = (s < -1 || s >= a.num_slots);
  const bool a_ok = a.A[h] < 0.f;  // sign test: NaN, +0 and -0 fail
  if (s >= 0 && !oor && a_ok) return s;
  if (threadIdx.x == 0) {
    if (oor) set_status(a.d_status, SSD_DEV_INDEX_OOR);
    if (!a_ok) set_status(a.d_status, SSD_DEV_A_NOT_NEG);
  }
  TA* yrow = reinterpret_cast<TA*>(a.y) + ((size_t)b * a.H + h) * a.P;
  for (int p = threadIdx.x; p < a.P; p += blockDim.x) yrow[p] = from_f32<TA>(0.f);
  return -1;
}

template <typename TA, int N>
__global__ void __launch_bounds__(256) state_update_vec_kernel(const ssd_update_args a) {
  constexpr int LPR = N / 4;       // lanes per state row
  constexpr int RPW = 32 / LPR;    // rows per warp
  constexpr int RPI = 8 * RPW;     // rows per CTA pass (8 warps)
  constexpr int KMAX = 8;          // float4 loads in flight per thread
  const int h = blockIdx.x, b = blockIdx.y;
  const int s = guard_row<TA>(a, b, h);
  if (s < 0) return;
  const int H = a.H, P = a.P;
  const int g = h / (H / a.G);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q = lane % LPR, rw = lane / LPR;

  float bv[4], cv[4];
  load4<TA>(reinterpret_cast<const TA*>(a.B) + ((size_t)b * a.G + g) * N + 4 * q, bv);
  load4<TA>(reinterpret_cast<const TA*>(a.C) + ((size_t)b * a.G + g) * N + 4 * q, cv);
  const float dt = dt_prep(a.dt[(size_t)b * H + h], a.dt_bias ? a.dt_bias[h] : 0.f,
                           a.dt_softplus);
  const float dA = expf(dt * a.A[h]);
  const float Dh = a.D ? a.D[h] : 0.f;
  const size_t slot_stride = a.slot_stride ? (size_t)a.slot_stride : (size_t)H * P * N;
  float* S = a.state_pool + (size_t)s * slot_stride + (size_t)h * P * N;
  const TA* xb = reinterpret_cast<const TA*>(a.x) + ((size_t)b * H + h) * P;
  TA* yb = reinterpret_cast<TA*>(a.y) + ((size_t)b * H + h) * P;

  // `base` is warp-uniform so every lane runs the same iterations (the shuffles need all 32)
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
      if (p < P && q == 0) yb[p] = from_f32<TA>(fmaf(Dh, xv[k], acc));
    }
  }
}

// Any N: one warp per state row, lanes strided over n.
template <typename TA>
__global__ void __launch_bounds__(256) state_update_generic_kernel(const ssd_update_args a) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int s = guard_row<TA>(a, b, h);
  if (s < 0) return;
  const int H = a.H, P = a.P, N = a.N;
  const int g = h / (H / a.G);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const TA* Bb = reinterpret_cast<const TA*>(a.B) + ((size_t)b * a.G + g) * N;
  const TA* Cb = reinterpret_cast<const TA*>(a.C) + ((size_t)b * a.G + g) * N;
  const float dt = dt_prep(a.dt[(size_t)b * H + h], a.dt_bias ? a.dt_bias[h] : 0.f,
                           a.dt_softplus);
  const float dA = expf(dt * a.A[h]);
  const float Dh = a.D ? a.D[h] : 0.f;
  const size_t slot_stride = a.slot_stride ? (size_t)a.slot_stride : (size_t)H * P * N;
  float* S = a.state_pool + (size_t)s * slot_stride + (size_t)h * P * N;
  const TA* xb = reinterpret_cast<const TA*>(a.x) + ((size_t)b * H + h) * P;
  TA* yb = reinterpret_cast<TA*>(a.y) + ((size_t)b * H + h) * P;
  for (int p = warp; p < P; p += blockDim.x / 32) {
    const float xv = to_f32(xb[p]);
    const float dx = dt * xv;
    float acc = 0.f;
    for (int n = lane; n < N; n += 32) {
      float v = fmaf(dA, S[(size_t)p * N + n], dx * to_f32(Bb[n]));
      S[(size_t)p * N + n] = v;
      acc = fmaf(to_f32(Cb[n]), v, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) yb[p] = from_f32<TA>(fmaf(Dh, xv, acc));
  }
}

template <typename TA>
cudaError_t launch_typed(const ssd_update_args& a, cudaStream_t st) {
  dim3 grid(a.H, a.batch);
  const size_t slot_stride = a.slot_stride ? (size_t)a.slot_stride : (size_t)a.H * a.P * a.N;
  const bool aligned = ((uintptr_t)a.state_pool % 16 == 0) && (slot_stride % 4 == 0) &&
                       ((uintptr_t)a.B % (4 * sizeof(TA)) == 0) &&
                       ((uintptr_t)a.C % (4 * sizeof(TA)) == 0);
  if (aligned && a.N == 128)
    state_update_vec_kernel<TA, 128><<<grid, 256, 0, st>>>(a);
  else if (aligned && a.N == 64)
    state_update_vec_kernel<TA, 64><<<grid, 256, 0, st>>>(a);
  else if (aligned && a.N == 32)
    state_update_vec_kernel<TA, 32><<<grid, 256, 0, st>>>(a);
  else if (aligned && a.N == 16)
    state_update_vec_kernel<TA, 16><<<grid, 256, 0, st>>>(a);
  else
    state_update_generic_kernel<TA><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_state_update(const ssd_update_args& a, cudaStream_t st) {
  if (a.batch == 0) return cudaSuccess;
  return a.act_dtype == SSD_BF16 ? launch_typed<__nv_bfloat16>(a, st) : launch_typed<float>(a, st);
}

}  // namespace ssd
