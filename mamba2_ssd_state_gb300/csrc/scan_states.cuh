// scan_states.cuh -- the state pass and the state fold of the two-head scan's split form
// (included by scan_tc.cu after scan_pair.cuh).
//
// A sequence cut into segments of segc chunks runs each segment as its own two-head chain
// (scan_pair_kernel<true>), entered with the state the sequence has at the segment's first
// token, so that every output is written once.  Those entering states come from two small
// passes that run before it:
//
// 1. scan_state_kernel, one CTA per (segment that is not its sequence's last, head pair,
//    64 channels): the state the segment leaves when it is entered with zero,
//        L = sum_t 2^(cs_end - cs_t) dt_t B_t^T x_t     (base-2 decay, over the segment),
//    and its total decay d = cs_end = sum_t dt_t A log2(e).  The decay from each token to
//    the segment's end folds into the weight of its x row, so L is one product
//    B_seg^T (w o x_seg) accumulated in one TMEM tile over the segment's chunks, with no
//    state step between chunks: nothing chains them, and the pass streams x and B at the
//    memory's pace.  The chunks are taken last to first, so each token's decay to the end
//    is its chunk's suffix sum plus a carry from the chunks already done.
// 2. scan_fold_kernel: per sequence and state element, the entering state of segment k,
//        E_0 = initial state,   E_{k+1} = 2^(d_k) E_k + L_k,
//    written over L_k (the slot of segment k then holds the state segment k + 1 enters with).
//
// The three grids run back to back with programmatic stream serialisation: each sets up
// while the one before drains and waits for it before reading what it wrote.

namespace ssd {
namespace {

namespace statepass {

constexpr int kStages = 3;               // TMA ring: B and x of both heads per stage
constexpr int kStage = 65536;            // B (2 x 16 KB boxes) | x head 0 | x head 1
constexpr int kWRing = 8;                // weights ring: the decay warps run this far ahead
constexpr int kWBuf = kStages * kStage;  // float [kWRing][2][QT] weights w
constexpr int kDtBuf = kWBuf + kWRing * 2 * QT * 4;  // float [kDtRing][2][QT] dt
constexpr int kBar = kDtBuf + kDtRing * 2 * QT * 4;
constexpr int kNumBar = 3 * kStages + 2 * kWRing + 1;
constexpr int kFlags = kBar + kNumBar * 8;
constexpr int kSmemBytes = kFlags + 16 + 1024;
constexpr int kScaleWarps = 8;
constexpr int kThreads = 32 * (4 + kScaleWarps);  // producer, MMA, 2 decay, 8 scale
static_assert(kSmemBytes <= 232448, "dynamic shared memory per CTA");
static_assert(kBar % 8 == 0, "mbarriers need 8-byte alignment");

}  // namespace statepass

// Warp roles (384 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA issuer, warps
// 2-3 decay warps (one per head: dt, the suffix sums, the weights w), warps 4-11 scale
// warps (w o x in place in the stage, then the accumulator out to the workspace).
__global__ void __launch_bounds__(statepass::kThreads, 1)
    scan_state_kernel(const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmB, const TcParams prm) {
  using namespace statepass;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int npair = prm.H / 2;
  const int pbk = unit % prm.npb;
  const int hp = (unit / prm.npb) % npair;
  const int j = unit / (prm.npb * npair);  // the segment
  const int h0 = 2 * hp, p0 = pbk * 64;
  const int H = prm.H, P = prm.P;
  const int g = h0 / (H / prm.G);

  __shared__ int seg_info[5];
  if (warp == 0) {
    int ss = -1, kk = 0, nn = 0, a = 0, b = 0;
    find_segment_warp(prm.cu, prm.nseq, prm.segc, j, ss, kk, nn, a, b);
    if (lane == 0) {
      seg_info[0] = ss;
      seg_info[1] = kk;
      seg_info[2] = nn;
      seg_info[3] = a;
      seg_info[4] = b;
    }
  }
  __syncthreads();
  const int s = seg_info[0], kseg = seg_info[1], nseg_s = seg_info[2];
  const int t0 = seg_info[3], t1 = seg_info[4];
  // a sequence's last segment needs no pass (its chain writes the final state); malformed
  // lengths are reported by the scan kernel
  if (s < 0 || kseg + 1 >= nseg_s || !(0 <= t0 && t0 <= t1 && t1 <= prm.T)) return;
  const int nch = prm.segc;  // a segment before the last is whole: segc full chunks
  const int tb = t0 + kseg * prm.segc * QT;
  const float A0 = prm.A[h0], A1 = prm.A[h0 + 1];
  const size_t PN = (size_t)P * NSTATE;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);
  uint64_t* full = bars;                 // [kStages] B and x landed
  uint64_t* xs_ready = bars + kStages;   // [kStages] w o x in place (8 scale warps)
  uint64_t* empty = bars + 2 * kStages;  // [kStages] read by the tensor core
  uint64_t* w_full = bars + 3 * kStages;  // [kWRing] weights of both heads (2 decay warps)
  uint64_t* w_empty = w_full + kWRing;    // [kWRing] weights read (8 scale warps)
  uint64_t* acc_full = w_empty + kWRing;  //  every product accumulated
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kFlags + 4);
  float* wbuf = reinterpret_cast<float*>(sm + kWBuf);
  float* dtbuf = reinterpret_cast<float*>(sm + kDtBuf);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&xs_ready[i], kScaleWarps);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kWRing; ++i) {
      mbar_init(&w_full[i], 2);
      mbar_init(&w_empty[i], kScaleWarps);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) griddep_launch_dependents();
  auto wwait = [&](uint64_t* bar, uint32_t par) -> bool {
    return warp_wait(bar, par, abort_flag, kWaitLimit);
  };
  // chunk i of the walk is chunk nch - 1 - i of the segment
  auto chunk_tok = [&](int i) { return tb + (nch - 1 - i) * QT; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (lane 0)
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int sg = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[sg], ((i / kStages) - 1) & 1, abort_flag, kWaitLimit))
          break;
        uint8_t* stg = sm + sg * kStage;
        const int tok = chunk_tok(i);
        mbar_arrive_expect_tx(&full[sg], kStage);
        tma_load_3d(stg, &tmB, &full[sg], 0, g, tok);
        tma_load_3d(stg + 16384, &tmB, &full[sg], 64, g, tok);
        tma_load_3d(stg + 32768, &tmX, &full[sg], p0, h0, tok);
        tma_load_3d(stg + 49152, &tmX, &full[sg], p0, h0 + 1, tok);
        issued = i + 1;
        if (i + kStages < nch) {  // the stage after next, into L2
          const int tp = chunk_tok(i + kStages);
          tma_prefetch_3d(&tmB, 0, g, tp);
          tma_prefetch_3d(&tmB, 64, g, tp);
          tma_prefetch_3d(&tmX, p0, h0, tp);
          tma_prefetch_3d(&tmX, p0, h0 + 1, tp);
        }
      }
      // every copy issued must have landed before the CTA's shared memory is released
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        mbar_wait_drain(&full[i % kStages], (i / kStages) & 1, kWaitLimit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lane 0)
    if (lane == 0) {
      // L^T[n][e p] += B^T (w o x): A = B read MN-major (two 64-row atoms 16 KB apart), B
      // operand = w o x of both heads MN-major (the two heads' tiles are the two 64-column
      // atoms of N = 128, 16 KB apart); K = 16 tokens per MMA
      constexpr uint32_t idS = make_idesc_bf16(128, 128, true, true);
      for (int i = 0; i < nch; ++i) {
        const int sg = i % kStages;
        if (!mbar_wait(&xs_ready[sg], (i / kStages) & 1, abort_flag, kWaitLimit)) break;
        tc_fence_after();
        const uint32_t base = smem_u32(sm + sg * kStage);
        const uint64_t dB = make_sdesc(base, 16384, 1024, kSw128);
        const uint64_t dX = make_sdesc(base + 32768, 16384, 1024, kSw128);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem, dB + kk * 128, dX + kk * 128, idS, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&empty[sg]);
      }
      mma_commit(acc_full);  // also the teardown's drain: every MMA issued has retired
      mbar_wait_drain(acc_full, 0, kWaitLimit);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ decay warps (one per head)
    const int e = warp - 2;
    const int hh = h0 + e;
    const float Ae = e ? A1 : A0;
    const bool bad = !(Ae < 0.f);  // such a head's outputs are zero: its state is unused
    const float a2 = bad ? 0.f : Ae * kLog2e;
    const float bias = prm.dt_bias ? prm.dt_bias[hh] : 0.f;
    // dt of the next kDtRing chunks in flight (a strided gather into the shared ring);
    // lane l copies and reads tokens 4 l .. 4 l + 3
    float* dring = dtbuf + e * QT + 4 * lane;
    auto fetch_dt = [&](int i) {
      float* dst = dring + (i % kDtRing) * 2 * QT;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int tok = chunk_tok(i) + 4 * lane + u;
        const bool v = i < nch && tok < t1;
        cp_async4(dst + u, v ? prm.dt + (size_t)tok * H + hh : prm.dt, v);
      }
      cp_async_commit();
    };
    for (int r = 0; r < kDtRing; ++r) fetch_dt(r);
    float carry = 0.f;  // log2 decay over the chunks already walked (the later ones)
    for (int i = 0; i < nch; ++i) {
      const int sw = i % kWRing;
      // weights slot sw was last read by the scale warps for chunk i - kWRing
      if (i >= kWRing && !wwait(&w_empty[sw], ((i / kWRing) - 1) & 1)) break;
      cp_async_wait<kDtRing - 1>();  // chunk i's copies have landed
      const float4 r4 = *reinterpret_cast<const float4*>(dring + (i % kDtRing) * 2 * QT);
      float raw[4] = {r4.x, r4.y, r4.z, r4.w}, d[4], cs[4];
      const float run =
          chunk_decay(raw, bias, a2, chunk_tok(i) + 4 * lane, t1, bad, prm.dt_softplus, d, cs);
      fetch_dt(i + kDtRing);  // into the slot just read (its values are in registers)
      // w_t = 2^(decay from t to the segment's end) dt_t: the rest of this chunk, then
      // every later chunk
      float w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) w[u] = ex2(run - cs[u] + carry) * d[u];
      *reinterpret_cast<float4*>(wbuf + (sw * 2 + e) * QT + 4 * lane) =
          make_float4(w[0], w[1], w[2], w[3]);
      carry += run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&w_full[sw]);
    }
    cp_async_wait<0>();  // no copy may land after the CTA's shared memory is released
    if (lane == 0 && pbk == 0 && !*abort_flag) prm.ws_d[(size_t)j * H + hh] = carry;
  } else {
    // ------------------------------------------------------------ scale warps
    const int ts = threadIdx.x - 128;  // 0..255
    for (int i = 0; i < nch; ++i) {
      const int sg = i % kStages;
      const int sw = i % kWRing;
      if (!wwait(&full[sg], (i / kStages) & 1)) break;
      if (!wwait(&w_full[sw], (i / kWRing) & 1)) break;
      uint8_t* xt = sm + sg * kStage + 32768;
      const float* wb = wbuf + sw * 2 * QT;
      // 2048 16-byte pieces (two heads x 128 rows x 8): the swizzle moves pieces only
      // within their 128-byte row, so piece q of head q / 1024 belongs to row (q / 8) % 128
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int q = ts + 256 * m;
        const float w = wb[(q >> 10) * QT + ((q >> 3) & 127)];
        uint4 xv = *reinterpret_cast<const uint4*>(xt + 16 * q);
        __nv_bfloat162* e2 = reinterpret_cast<__nv_bfloat162*>(&xv);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 f = __bfloat1622float2(e2[t]);
          float a, bb;
          mul_f32x2(a, bb, f.x, f.y, w, w);
          e2[t] = __floats2bfloat162_rn(a, bb);
        }
        *reinterpret_cast<uint4*>(xt + 16 * q) = xv;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&xs_ready[sg]);
        mbar_arrive(&w_empty[sw]);
      }
    }
    // the accumulator: TMEM lane n = state row, column 64 e + p; warp w reads the lanes of
    // its quadrant w % 4, head (w - 4) / 4
    if (wwait(acc_full, 0) && !*abort_flag) {
      tc_fence_after();
      const int q = warp & 3, e = (warp - 4) >> 2;
      const int n = 32 * q + lane;
      const uint32_t lrow = (uint32_t)(32 * q) << 16;
      float* out = prm.ws_h + ((size_t)j * H + h0 + e) * PN + (size_t)p0 * NSTATE + n;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[32];
        tmem_ld32(tmem + lrow + 64 * e + 32 * half, v);
#pragma unroll
        for (int t = 0; t < 32; ++t) out[(size_t)(32 * half + t) * NSTATE] = v[t];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(prm.status, SSD_DEV_TIMEOUT);
}

// Index of the first segment of sequence s among the batch's segments (one warp; every
// lane gets the result).
__device__ inline int first_segment_warp(const int32_t* cu, int s, int segc) {
  const int lane = threadIdx.x & 31;
  int n = 0;
  for (int i = lane; i < s; i += 32) n += seg_count(cu[i + 1] - cu[i], segc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
  return n;
}

// One thread per four consecutive state elements (h, p, n..n+3) of one sequence
// (blockIdx.y); it walks the sequence's segments in order.
constexpr int kFoldThreads = 256;

__global__ void __launch_bounds__(kFoldThreads)
    scan_fold_kernel(const TcParams prm) {
  __shared__ int info[2];
  const int s = blockIdx.y;
  if (threadIdx.x < 32) {
    const int t0 = prm.cu[s], t1 = prm.cu[s + 1];
    const bool okl = 0 <= t0 && t0 <= t1 && t1 <= prm.T;
    const int j0 = first_segment_warp(prm.cu, s, prm.segc);
    if (threadIdx.x == 0) {
      info[0] = j0;
      info[1] = okl ? seg_count(t1 - t0, prm.segc) : 1;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int j0 = info[0], nseg_s = info[1];
  if (nseg_s < 2) return;
  const size_t PN = (size_t)prm.P * NSTATE;
  const size_t HPN = (size_t)prm.H * PN;
  const size_t e4 = ((size_t)blockIdx.x * kFoldThreads + threadIdx.x) * 4;
  if (e4 >= HPN) return;
  const int h = (int)(e4 / PN);
  const bool has_init = prm.init && (prm.has_init == nullptr || prm.has_init[s] != 0);
  float4 acc = has_init ? *reinterpret_cast<const float4*>(prm.init + (size_t)s * HPN + e4)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
  griddep_wait();  // the local states and decays are the state pass's
  // the walk is a chain of multiply-adds, but its loads are not: kFoldAhead of them in
  // flight (the chain's pace would otherwise be one memory round trip per segment)
  constexpr int kFoldAhead = 4;
  float* slot = prm.ws_h + (size_t)j0 * HPN + e4;
  const float* dseg = prm.ws_d + (size_t)j0 * prm.H + h;
  const int nfold = nseg_s - 1;  // local states to fold: segments 0 .. nseg_s - 2
  float4 ring[kFoldAhead];
  float dring[kFoldAhead];
#pragma unroll
  for (int k = 0; k < kFoldAhead; ++k) {
    if (k < nfold) {
      ring[k] = *reinterpret_cast<const float4*>(slot + (size_t)k * HPN);
      dring[k] = dseg[(size_t)k * prm.H];
    }
  }
  for (int k0 = 0; k0 < nfold; k0 += kFoldAhead) {
#pragma unroll
    for (int u = 0; u < kFoldAhead; ++u) {
      const int k = k0 + u;
      if (k < nfold) {
        const float4 l = ring[u];
        const float dec = ex2(dring[u]);
        if (k + kFoldAhead < nfold) {  // the load kFoldAhead segments on
          ring[u] = *reinterpret_cast<const float4*>(slot + (size_t)(k + kFoldAhead) * HPN);
          dring[u] = dseg[(size_t)(k + kFoldAhead) * prm.H];
        }
        acc.x = fmaf(dec, acc.x, l.x);
        acc.y = fmaf(dec, acc.y, l.y);
        acc.z = fmaf(dec, acc.z, l.z);
        acc.w = fmaf(dec, acc.w, l.w);
        // the state segment k + 1 enters with, over segment k's local one (already read)
        *reinterpret_cast<float4*>(slot + (size_t)k * HPN) = acc;
      }
    }
  }
}

}  // namespace
}  // namespace ssd
