// scan_simt.cu -- token-sequential fp32 SIMT evaluation of the Mamba2 SSD scan
// (vt::Mamba2ChunkScan of the vllm.cpp page "W2 finish (KERNEL-SSM-MAMBA)").
//
// This is the precision path: it walks the recurrence
//     h_t = exp(dt_t A) h_{t-1} + dt_t B_t x_t^T,   y_t = C_t . h_t + D x_t
// one token at a time in fp32, so each output carries only the error of a length-K
// recurrence and a length-N dot product -- the error model behind the pages' fp32 bar
// rtol(K) = 4 (K + 2) 2^-24 (same page, section "Evidence" and the #675 message).  The
// chunked decomposition is exact, so walking the tokens gives the chunked result for
// any chunk_size; the tensor-core path is the one that tiles by chunk.
//
// Layout of the work: one warp per (sequence, head, channel p); a lane owns the state
// entries n = lane + 32 k (k < NPL) in registers.  No shared memory, no block barrier:
// every warp marches over its sequence independently, prefetching token t + 1's inputs
// while it computes token t.
#include "ssd_internal.cuh"

namespace ssd {
namespace {

template <typename TA, int NPL>
__global__ void __launch_bounds__(256) scan_simt_kernel(const ssd_scan_args a) {
  const int s = blockIdx.z, h = blockIdx.y;
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int H = a.H, P = a.P, G = a.G, N = a.N;
  const int g = h / (H / G);

  if (blockIdx.x == 0 && blockIdx.y == 0 && s == 0 && threadIdx.x == 0) {
    if (a.cu_seqlens[0] != 0 || a.cu_seqlens[a.nseq] != a.T) set_status(a.d_status, SSD_DEV_SEQ_META);
  }
  const int t0 = a.cu_seqlens[s], t1 = a.cu_seqlens[s + 1];
  if (!(0 <= t0 && t0 <= t1 && t1 <= a.T)) {
    if (threadIdx.x == 0) set_status(a.d_status, SSD_DEV_SEQ_META);
    return;
  }
  if (p >= P) return;  // warp-uniform

  const int64_t xs = a.x_stride_t ? a.x_stride_t : (int64_t)H * P;
  const int64_t bs = a.B_stride_t ? a.B_stride_t : (int64_t)G * N;
  const int64_t cs = a.C_stride_t ? a.C_stride_t : (int64_t)G * N;
  const TA* X = reinterpret_cast<const TA*>(a.x) + (size_t)h * P + p;
  const TA* Bg = reinterpret_cast<const TA*>(a.B) + (size_t)g * N;
  const TA* Cg = reinterpret_cast<const TA*>(a.C) + (size_t)g * N;
  TA* Y = reinterpret_cast<TA*>(a.y) + (size_t)h * P + p;
  const float Ah = a.A[h];
  const size_t PN = (size_t)P * N;
  float* fin = a.final_states ? a.final_states + ((size_t)s * H + h) * PN + (size_t)p * N : nullptr;

  if (!(Ah < 0.f)) {  // sign test; the head produces zeros
    if (lane == 0) {
      if (p == 0) set_status(a.d_status, SSD_DEV_A_NOT_NEG);
      for (int t = t0; t < t1; ++t) Y[(size_t)t * H * P] = from_f32<TA>(0.f);
    }
    if (fin)
      for (int n = lane; n < N; n += 32) fin[n] = 0.f;
    return;
  }

  float st[NPL];
  const bool has_init =
      a.initial_states && (a.has_initial_state == nullptr || a.has_initial_state[s] != 0);
#pragma unroll
  for (int k = 0; k < NPL; ++k) {
    const int n = lane + 32 * k;
    st[k] = (has_init && n < N) ? a.initial_states[((size_t)s * H + h) * PN + (size_t)p * N + n]
                                : 0.f;
  }
  const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
  const float Dh = a.D ? a.D[h] : 0.f;

  // prefetched inputs of the next token
  float nxt_dt = 0.f, nxt_x = 0.f, nxt_b[NPL], nxt_c[NPL];
  auto fetch = [&](int t) {
    nxt_dt = a.dt[(size_t)t * H + h];
    nxt_x = to_f32(X[(size_t)t * xs]);
#pragma unroll
    for (int k = 0; k < NPL; ++k) {
      const int n = lane + 32 * k;
      nxt_b[k] = n < N ? to_f32(Bg[(size_t)t * bs + n]) : 0.f;
      nxt_c[k] = n < N ? to_f32(Cg[(size_t)t * cs + n]) : 0.f;
    }
  };
  if (t0 < t1) fetch(t0);
  for (int t = t0; t < t1; ++t) {
    const float dt = dt_prep(nxt_dt, bias, a.dt_softplus);
    const float xv = nxt_x;
    float bv[NPL], cv[NPL];
#pragma unroll
    for (int k = 0; k < NPL; ++k) {
      bv[k] = nxt_b[k];
      cv[k] = nxt_c[k];
    }
    if (t + 1 < t1) fetch(t + 1);
    const float dA = expf(dt * Ah);
    const float dx = dt * xv;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < NPL; ++k) {
      st[k] = fmaf(dA, st[k], dx * bv[k]);
      acc = fmaf(cv[k], st[k], acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) Y[(size_t)t * H * P] = from_f32<TA>(fmaf(Dh, xv, acc));
  }
  if (fin) {
#pragma unroll
    for (int k = 0; k < NPL; ++k) {
      const int n = lane + 32 * k;
      if (n < N) fin[n] = st[k];
    }
  }
}

template <typename TA>
cudaError_t launch_typed(const ssd_scan_args& a, cudaStream_t st) {
  dim3 grid((a.P + 7) / 8, a.H, a.nseq);
  const int npl = (a.N + 31) / 32;
  switch (npl) {
    case 1: scan_simt_kernel<TA, 1><<<grid, 256, 0, st>>>(a); break;
    case 2: scan_simt_kernel<TA, 2><<<grid, 256, 0, st>>>(a); break;
    case 3: scan_simt_kernel<TA, 3><<<grid, 256, 0, st>>>(a); break;
    case 4: scan_simt_kernel<TA, 4><<<grid, 256, 0, st>>>(a); break;
    case 5: case 6: scan_simt_kernel<TA, 6><<<grid, 256, 0, st>>>(a); break;
    default: scan_simt_kernel<TA, 8><<<grid, 256, 0, st>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_simt(const ssd_scan_args& a, cudaStream_t st) {
  return a.act_dtype == SSD_BF16 ? launch_typed<__nv_bfloat16>(a, st) : launch_typed<float>(a, st);
}

}  // namespace ssd
