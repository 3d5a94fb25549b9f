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
// One (row, group) unit: the threads of a 256-thread block with the same threadIdx / TPG
// work on it; every thread of the block calls this (valid or not), since groups of more
// than a warp meet at block barriers.  pdl: wait for the kernel before (the producer of
// x) after loading z.
template <typename TA, typename TW, int VPT, int TPG, bool kPdl>
__device__ __forceinline__ void norm_unit(const TA* x, const TA* __restrict__ z,
                                          const TW* __restrict__ w, TA* out, bool valid,
                                          size_t base, int col0, int gs, float eps,
                                          float* part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tig = threadIdx.x % TPG;
  float g[VPT][8];
  float ss = 0.f;
  if (valid && z) {  // z first: it may be read before the producer of x has finished
#pragma unroll
    for (int i = 0; i < VPT; ++i) Vec8<TA>::load(z + base + 8 * (tig + TPG * i), g[i]);
  }
  if constexpr (kPdl) tc::griddep_wait();
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
    __syncthreads();  // part is rewritten by the next unit
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

template <typename TA, typename TW, int VPT, int TPG>
__global__ void __launch_bounds__(256) norm_vec_kernel(const TA* x,
                                                       const TA* __restrict__ z,
                                                       const TW* __restrict__ w, TA* out,
                                                       int64_t units, int d, int gs, float eps) {
  constexpr int GPB = 256 / TPG;  // groups per block
  __shared__ float part[8];
  const int64_t unit = (int64_t)blockIdx.x * GPB + threadIdx.x / TPG;
  const bool valid = unit < units;
  const int ngroups = d / gs;
  const int64_t row = valid ? unit / ngroups : 0;
  const int col0 = valid ? (int)(unit % ngroups) * gs : 0;
  norm_unit<TA, TW, VPT, TPG, true>(x, z, w, out, valid, (size_t)row * d + col0, col0, gs, eps,
                                    part);
}

// The norm of the scan + norm call, fed by the scan's ready counters.  Tasks go in
// chunk-major order — chunk 0 of every sequence, then chunk 1, ... — which follows the
// order in which a scan grid finishes chunks; each is kReadyParts tasks of 32 rows per
// norm group.  Each block takes the next task with an atomic, waits (bounded) until the
// task's chunk-group counter is complete, and normalises the rows with the per-unit
// arithmetic of norm_vec_kernel, so its outputs are bit for bit those of the standalone
// norm.  The blocks start once every scan CTA has started (programmatic dependent
// launch), on SMs the scan leaves free, and never wait for the scan grid itself until
// their last task is done.
template <typename TA, typename TW, int VPT, int TPG>
__global__ void __launch_bounds__(256) norm_ready_kernel(const TA* x,
                                                         const TA* __restrict__ z,
                                                         const TW* __restrict__ w, TA* out,
                                                         const int32_t* __restrict__ cu,
                                                         int nseq, int T, int d, int gs,
                                                         float eps, ReadyQueue rq,
                                                         uint32_t* status) {
  constexpr int GPB = 256 / TPG;  // rows per block step
  constexpr int kRows = 128 / kReadyParts;
  __shared__ float part[8];
  __shared__ int red[8];
  __shared__ int task[3];  // sequence (-1: none left), chunk, part * ngroups + group
  // the chunk-major task list spans max_s(chunks of s) chunk positions of nseq sequences,
  // taken as nsegm segments of segc positions, position c of every segment before c + 1
  int mine = 0;
  for (int s = threadIdx.x; s < nseq; s += blockDim.x) {
    const int t0 = cu[s], t1 = cu[s + 1];
    if (0 <= t0 && t0 <= t1 && t1 <= T) mine = max(mine, (t1 - t0 + 127) / 128);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mine = max(mine, __shfl_xor_sync(0xffffffffu, mine, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mine;
  __syncthreads();
  int maxc = 0;
  for (int k = 0; k < 8; ++k) maxc = max(maxc, red[k]);
  const int per_pos = rq.ngroups * kReadyParts;  // tasks per (chunk, sequence)
  const int segc = rq.segc > 0 ? min(rq.segc, max(maxc, 1)) : max(maxc, 1);
  const int nsegm = (maxc + segc - 1) / segc;
  const long long total = (long long)segc * nsegm * nseq * per_pos;
  for (;;) {
    if (threadIdx.x == 0) {
      int ts = -1, tc = 0, tk = 0;
      for (;;) {  // the next task of a chunk that exists
        const long long idx = atomicAdd(rq.head, 1);
        if (idx >= total) break;
        const long long pos = idx / per_pos;
        const long long q = pos / nseq;
        const int s = (int)(pos % nseq);
        const int c = (int)(q % nsegm) * segc + (int)(q / nsegm);
        const int t0 = cu[s], t1 = cu[s + 1];
        if (!(0 <= t0 && t0 <= t1 && t1 <= T) || c >= (t1 - t0 + 127) / 128) continue;
        ts = s;
        tc = c;
        tk = (int)(idx % per_pos);
        // wait until every output warp of the scan has counted this chunk-group
        const int grp = tk % rq.ngroups;
        const long long id = (long long)(t0 / 128) + s + c;
        const volatile int* cnt = rq.cnt + id * rq.ngroups + grp;
        const long long t_start = clock64();
        while (*cnt < rq.target) {
          if (*(volatile int*)rq.abort) {
            ts = -1;
            break;
          }
          if (clock64() - t_start > SSD_WAIT_LIMIT_CYCLES) {
            atomicExch(rq.abort, 1);
            set_status(status, SSD_DEV_TIMEOUT);
            ts = -1;
            break;
          }
          __nanosleep(128);
        }
        __threadfence();  // the rows the counter stands for are visible from here on
        break;
      }
      task[0] = ts;
      task[1] = tc;
      task[2] = tk;
    }
    __syncthreads();
    const int s = task[0], c = task[1], tk = task[2];
    __syncthreads();
    if (s < 0) break;
    const int grp = tk % rq.ngroups, k = tk / rq.ngroups;
    const int t1 = cu[s + 1];
    const int r0 = cu[s] + 128 * c + kRows * k;
    const int r1 = min(t1, r0 + kRows);
    const int col0 = grp * gs;
    for (int rb = r0; rb < r1; rb += GPB) {  // the same trip count in every thread
      const int row = rb + threadIdx.x / TPG;
      norm_unit<TA, TW, VPT, TPG, false>(x, z, w, out, row < r1, (size_t)row * d + col0, col0,
                                         gs, eps, part);
    }
  }
  // end no earlier than the scan grid, so that work after this call on the stream finds
  // the scan's final states written too
  tc::griddep_wait();
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
constexpr int kReadyBlocksPerSm = 4;  // resident ready-queue norm blocks per free SM

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

// Vector path: the smallest group of threads (32..256) with at most 4 vectors each, for
// 16-byte aligned rows; false (generic path) otherwise.
bool vec_shape(const void* x, const void* z, const void* w, const void* out, int d, int gs,
               size_t act_bytes, int* tpg, int* vpt) {
  *tpg = *vpt = 0;
  const bool aligned = ((uintptr_t)x % 16 == 0) && ((uintptr_t)out % 16 == 0) &&
                       (z == nullptr || (uintptr_t)z % 16 == 0) && ((uintptr_t)w % 16 == 0) &&
                       ((size_t)d * act_bytes) % 16 == 0;
  if (!aligned || gs % 8 != 0) return false;
  for (int t = 32; t <= 256; t *= 2) {
    const int nvec = gs / 8;
    if (nvec % t == 0 && nvec / t <= 4) {
      *tpg = t;
      *vpt = nvec / t;
      return true;
    }
  }
  return false;
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
  int tpg, vpt;
  vec_shape(x, z, w, out, d, gs, sizeof(TA), &tpg, &vpt);
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

// The ready-queue norm: a persistent grid of a few blocks per SM.
template <typename TA, typename TW>
cudaError_t launch_ready_typed(const void* x, const void* z, const void* w, void* out,
                               const int32_t* cu, int nseq, int T, int d, int gs, float eps,
                               const ReadyQueue& rq, uint32_t* status, cudaStream_t st) {
  int tpg, vpt;
  if (!vec_shape(x, z, w, out, d, gs, sizeof(TA), &tpg, &vpt)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  const int64_t blocks = (int64_t)kReadyBlocksPerSm * sms;
  const TA* xp = static_cast<const TA*>(x);
  const TA* zp = static_cast<const TA*>(z);
  const TW* wp = static_cast<const TW*>(w);
  TA* op = static_cast<TA*>(out);
#define SSD_READY_CASE(V, TP)                                                                \
  if (vpt == V && tpg == TP)                                                                  \
    return launch256(norm_ready_kernel<TA, TW, V, TP>, blocks, true, st, xp, zp, wp, op, cu,   \
                     nseq, T, d, gs, eps, rq, status);
  SSD_READY_CASE(1, 32) SSD_READY_CASE(2, 32) SSD_READY_CASE(3, 32) SSD_READY_CASE(4, 32)
  SSD_READY_CASE(3, 64) SSD_READY_CASE(4, 64) SSD_READY_CASE(3, 128) SSD_READY_CASE(4, 128)
  SSD_READY_CASE(3, 256) SSD_READY_CASE(4, 256)
#undef SSD_READY_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

bool norm_ready_supported(const void* x, const void* z, const void* w, const void* out, int d,
                          int gs, ssd_dtype act) {
  int tpg, vpt;
  return vec_shape(x, z, w, out, d, gs, act == SSD_BF16 ? 2 : 4, &tpg, &vpt);
}

cudaError_t launch_norm_ready(const void* x, const void* z, const void* w, void* out,
                              const int32_t* cu, int nseq, int T, int d, int gs, float eps,
                              ssd_dtype act, ssd_dtype wt, const ReadyQueue& rq,
                              uint32_t* status, cudaStream_t st) {
  using bf = __nv_bfloat16;
  if (act == SSD_BF16)
    return wt == SSD_BF16
               ? launch_ready_typed<bf, bf>(x, z, w, out, cu, nseq, T, d, gs, eps, rq, status, st)
               : launch_ready_typed<bf, float>(x, z, w, out, cu, nseq, T, d, gs, eps, rq, status,
                                               st);
  return wt == SSD_BF16
             ? launch_ready_typed<float, bf>(x, z, w, out, cu, nseq, T, d, gs, eps, rq, status, st)
             : launch_ready_typed<float, float>(x, z, w, out, cu, nseq, T, d, gs, eps, rq, status,
                                                st);
}

size_t ready_queue_bytes(int64_t T, int nseq, int ngroups) {
  const int64_t nid = (T + 127) / 128 + nseq;
  const size_t bytes = (size_t)nid * ngroups * sizeof(int) + 4 * sizeof(int);
  return (bytes + 255) / 256 * 256;
}

ReadyQueue ready_queue_at(void* ws, int64_t T, int nseq, int ngroups, int gs, int segc) {
  const int64_t nid = (T + 127) / 128 + nseq;
  int* p = static_cast<int*>(ws);
  ReadyQueue rq;
  rq.cnt = p;
  rq.head = p + (size_t)nid * ngroups;
  rq.abort = rq.head + 1;
  rq.nid = nid;
  rq.ngroups = ngroups;
  rq.gs = gs;
  rq.target = 4 * (gs / 64);
  rq.segc = segc;
  return rq;
}

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
