// scan_tc.cu -- the chunked Mamba2 SSD scan on GB300 tensor cores (tcgen05 + TMEM + TMA).
//
// The op is vt::Mamba2ChunkScan of the vllm.cpp page "W2 finish (KERNEL-SSM-MAMBA)"; its
// mutation table (section "Evidence": M1 inter-chunk state term, M2 initial_states, M3
// states[c-1] feeding chunk c, M4 the D skip) names the parts computed here.  With
// a_t = dt_t A and, inside a chunk, cs_i = sum_{r<=i} a_r:
//     CB[i,j]  = C_i . B_j                                   (tensor core, fp32 in TMEM)
//     M[i,j]   = CB[i,j] exp(cs_i - cs_j) dt_j,  j <= i       (segsum decay, epilogue)
//     Y        = M x                                          (tensor core, A from TMEM)
//     S^T      = B^T (w o x),  w_j = exp(cs_last - cs_j) dt_j (chunk state, tensor core)
//     Yoff     = C h_{c-1}^T                                  (tensor core)
//     y_i      = Y_i + exp(cs_i) Yoff_i + D x_i               (epilogue, bf16 out)
//     h_c      = exp(cs_last) h_{c-1} + S                      (state pass, fp32 registers)
//
// One CTA owns one (sequence, head, block of PB channels) chain and walks its chunks in
// order, so the state never leaves the SM: states[c-1] feeds chunk c in place, and HBM
// sees only x, B, C, dt in and y (plus the per-sequence initial / final states).  The
// channel split PB (64, 32 or 16) trades redundant C.B^T work for more chains when a
// workload has few (sequence, head) pairs.
//
// Warp roles (320 threads):
//   warp 0    TMA producer: C, B (two 64-wide 128B-swizzled boxes each) and x per chunk
//             into a 2-stage ring guarded by full/empty mbarriers.
//   warp 1    TMEM owner (512 columns) and the single MMA-issuing thread.
//   warps 2-9 epilogue: two warps per TMEM lane quadrant, each taking half of the
//             columns.  dt/softplus/cumsum, the decay mask (CB -> M written back to
//             TMEM as bf16), w o x into shared memory, y, and the fp32 state h.
// Every wait is bounded; a wait that runs out raises a CTA-wide abort flag, every role
// then drains what it has in flight and the kernel returns with SSD_DEV_TIMEOUT set.
//
// The chunk is the 128-row tcgen05 tile: sequences are split into 128-token chunks
// starting at their first token.  Chunked evaluation is exact for any chunk length, so
// the result equals the requested chunk_size's up to rounding.
#include <cudaTypedefs.h>

#include <mutex>

#include "ssd_internal.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int QT = 128;          // chunk length = tcgen05 M
constexpr int NSTATE = 128;      // state size N of this kernel
constexpr int NST = 2;           // TMA ring depth
constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitLimit = 4000000000LL;  // SM cycles (about 2 s)

// TMEM columns
constexpr uint32_t kColCB = 0;    // two fp32 128x128 C.B^T buffers: [0,128) and [128,256)
constexpr uint32_t kColM = 256;   // bf16 decay-masked M, 64 columns (two values per column)
constexpr uint32_t kColY = 320;   // Y, then Yoff, then S, PB columns each

struct TcParams {
  const float* dt;
  const float* dt_bias;
  const float* A;
  const float* D;
  const float* init;
  const uint8_t* has_init;
  const int32_t* cu;
  __nv_bfloat16* y;
  float* fin;
  uint32_t* status;
  int nseq, T, H, P, G, npb, dt_softplus;
};

template <int PB>
struct Layout {
  static constexpr int kXRow = PB * 2;                 // bytes per token row of x / x' / h^T
  static constexpr int kXBytes = QT * kXRow;
  static constexpr int kXPad = (kXBytes + 1023) / 1024 * 1024;
  static constexpr int kStageC = 0;                    // C: two [128 x 64] bf16 boxes
  static constexpr int kStageB = 32768;                // B: two boxes
  static constexpr int kStageX = 65536;                // x: one [128 x PB] box
  static constexpr int kStage = 65536 + kXPad;
  static constexpr int kXs = NST * kStage;             // w o x
  static constexpr int kHT = kXs + kXPad;              // h^T, [N rows][PB] bf16
  static constexpr int kHTPad = (NSTATE * kXRow + 1023) / 1024 * 1024;
  static constexpr int kDt = kHT + kHTPad;             // float [2][QT]
  static constexpr int kCs = kDt + 2 * QT * 4;         // float [2][QT] (base-2 cumsum)
  static constexpr int kBar = kCs + 2 * QT * 4;        // mbarriers
  static constexpr int kNumBar = 2 * NST + 4 + 4 + 6;
  static constexpr int kFlags = kBar + kNumBar * 8;    // abort flag, TMEM base
  static constexpr int kEnd = kFlags + 16;
  static constexpr int kSmemBytes = kEnd + 1024;       // + alignment slack
  static constexpr int kSwB = PB == 64 ? 3 : PB == 32 ? 2 : 1;  // Swizzle<B,4,3>
  static constexpr uint32_t kSwCode = PB == 64 ? kSw128 : PB == 32 ? kSw64 : kSw32;
  static constexpr uint32_t kTxBytes = 65536 + kXBytes;
};

template <int PB>
__global__ void __launch_bounds__(kThreads, 1)
    scan_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams prm) {
  using L = Layout<PB>;
  constexpr int PH = PB / 2;  // columns per epilogue half
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int pbk = unit % prm.npb;
  const int h = (unit / prm.npb) % prm.H;
  const int s = unit / (prm.npb * prm.H);
  const int p0 = pbk * PB;
  const int H = prm.H, P = prm.P;
  const int g = h / (H / prm.G);

  if (unit == 0 && threadIdx.x == 0 && (prm.cu[0] != 0 || prm.cu[prm.nseq] != prm.T))
    set_status(prm.status, SSD_DEV_SEQ_META);
  const int t0 = prm.cu[s], t1 = prm.cu[s + 1];
  if (!(0 <= t0 && t0 <= t1 && t1 <= prm.T)) {
    if (threadIdx.x == 0) set_status(prm.status, SSD_DEV_SEQ_META);
    return;
  }
  const float Ah = prm.A[h];
  const size_t PN = (size_t)P * NSTATE;
  float* fin = prm.fin ? prm.fin + ((size_t)s * H + h) * PN + (size_t)p0 * NSTATE : nullptr;
  if (!(Ah < 0.f)) {  // sign test (NaN, +0, -0 fail): the chain produces zeros
    if (threadIdx.x == 0 && pbk == 0) set_status(prm.status, SSD_DEV_A_NOT_NEG);
    for (int e = threadIdx.x; e < (t1 - t0) * PB; e += kThreads)
      prm.y[((size_t)(t0 + e / PB) * H + h) * P + p0 + e % PB] = __float2bfloat16_rn(0.f);
    if (fin)
      for (int e = threadIdx.x; e < PB * NSTATE; e += kThreads) fin[e] = 0.f;
    return;
  }
  const int nch = (t1 - t0 + QT - 1) / QT;

  float* dt_s = reinterpret_cast<float*>(sm + L::kDt);
  float* cs_s = reinterpret_cast<float*>(sm + L::kCs);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* full = bars;                 // [NST]  TMA landed
  uint64_t* empty = bars + NST;          // [NST]  stage free (MMA commit + 8 epilogue warps)
  uint64_t* cb_full = bars + 2 * NST;    // [2]    C.B^T ready in TMEM
  uint64_t* cb_empty = cb_full + 2;      // [2]    C.B^T consumed (8 warps)
  uint64_t* pro_full = cb_empty + 2;     // [2]    dt / cumsum of a chunk in smem (4 warps)
  uint64_t* pro_empty = pro_full + 2;    // [2]    dt / cumsum buffer consumed (8 warps)
  uint64_t* m_ready = pro_empty + 2;     //        M in TMEM and w o x in smem (8 warps)
  uint64_t* acc_full = m_ready + 1;      //        Y and S done
  uint64_t* yoff_full = m_ready + 2;     //        Yoff done
  uint64_t* acc_empty = m_ready + 3;     //        Y, Yoff, S read (8 warps)
  uint64_t* h_ready = m_ready + 4;       //        h^T in smem (8 warps)
  uint64_t* drain = m_ready + 5;         //        teardown: all MMAs retired
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kFlags + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&cb_full[i], 1);
      mbar_init(&cb_empty[i], 8);
      mbar_init(&pro_full[i], 4);
      mbar_init(&pro_empty[i], 8);
    }
    mbar_init(m_ready, 8);
    mbar_init(acc_full, 1);
    mbar_init(yoff_full, 1);
    mbar_init(acc_empty, 8);
    mbar_init(h_ready, 8);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        const int st = c % NST;
        if (c >= NST && !mbar_wait(&empty[st], ((c / NST) - 1) & 1, abort_flag, kWaitLimit))
          break;
        uint8_t* stg = sm + st * L::kStage;
        const int tok = t0 + c * QT;
        mbar_arrive_expect_tx(&full[st], L::kTxBytes);
        tma_load_3d(stg + L::kStageC, &tmC, &full[st], 0, g, tok);
        tma_load_3d(stg + L::kStageC + 16384, &tmC, &full[st], 64, g, tok);
        tma_load_3d(stg + L::kStageB, &tmB, &full[st], 0, g, tok);
        tma_load_3d(stg + L::kStageB + 16384, &tmB, &full[st], 64, g, tok);
        tma_load_3d(stg + L::kStageX, &tmX, &full[st], p0, h, tok);
        issued = c + 1;
      }
      // every copy issued must have landed before the CTA's shared memory is released
      for (int c = issued > NST ? issued - NST : 0; c < issued; ++c)
        mbar_wait_drain(&full[c % NST], (c / NST) & 1, kWaitLimit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idCB = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idY = make_idesc_bf16(128, PB, false, true);
      constexpr uint32_t idS = make_idesc_bf16(128, PB, true, true);
      constexpr uint32_t idO = make_idesc_bf16(128, PB, false, true);
      const uint32_t colY = tmem + kColY, colO = tmem + kColY + PB, colS = tmem + kColY + 2 * PB;
      const uint32_t sXs = smem_u32(sm + L::kXs), sHT = smem_u32(sm + L::kHT);
      bool ok = true;
      auto issue_cb = [&](int c) -> bool {
        const int st = c % NST, cb = c & 1;
        if (!mbar_wait(&full[st], (c / NST) & 1, abort_flag, kWaitLimit)) return false;
        if (c >= 2 && !mbar_wait(&cb_empty[cb], ((c >> 1) - 1) & 1, abort_flag, kWaitLimit))
          return false;
        tc_fence_after();
        const uint32_t sC = smem_u32(sm + st * L::kStage + L::kStageC);
        const uint32_t sB = smem_u32(sm + st * L::kStage + L::kStageB);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // K = N = 128 in steps of 16 (32 bytes)
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tmem + kColCB + cb * 128, make_sdesc(sC + ko, 16, 1024, kSw128),
                 make_sdesc(sB + ko, 16, 1024, kSw128), idCB, kk > 0);
        }
        mma_commit(&cb_full[cb]);
        return true;
      };
      if (nch > 0) ok = issue_cb(0);
      for (int c = 0; ok && c < nch; ++c) {
        const int st = c % NST;
        if (c + 1 < nch && !(ok = issue_cb(c + 1))) break;
        if (!(ok = mbar_wait(m_ready, c & 1, abort_flag, kWaitLimit))) break;
        if (c >= 1 && !(ok = mbar_wait(acc_empty, (c - 1) & 1, abort_flag, kWaitLimit))) break;
        tc_fence_after();
        const uint32_t sX = smem_u32(sm + st * L::kStage + L::kStageX);
        const uint32_t sB = smem_u32(sm + st * L::kStage + L::kStageB);
        const uint32_t sC = smem_u32(sm + st * L::kStage + L::kStageC);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // Y = M x : K = 128 tokens, M from TMEM (8 cols/step)
          mma_ts(colY, tmem + kColM + kk * 8,
                 make_sdesc(sX + kk * 16 * L::kXRow, L::kXBytes, 8 * L::kXRow, L::kSwCode), idY,
                 kk > 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // S^T = B^T (w o x): A = B read MN-major
          mma_ss(colS, make_sdesc(sB + kk * 2048, 16384, 1024, kSw128),
                 make_sdesc(sXs + kk * 16 * L::kXRow, L::kXBytes, 8 * L::kXRow, L::kSwCode), idS,
                 kk > 0);
        mma_commit(acc_full);
        if (!(ok = mbar_wait(h_ready, c & 1, abort_flag, kWaitLimit))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // Yoff = C h^T : K = N = 128
          const uint32_t ko = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(colO, make_sdesc(sC + ko, 16, 1024, kSw128),
                 make_sdesc(sHT + kk * 16 * L::kXRow, L::kHTPad, 8 * L::kXRow, L::kSwCode), idO,
                 kk > 0);
        }
        mma_commit(yoff_full);
        mma_commit(&empty[st]);
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0, kWaitLimit);
    }
  } else {
    // ------------------------------------------------------------ epilogue (8 warps)
    const int hf = (warp - 2) >> 2;        // column half
    const int q = warp & 3;                // TMEM lane quadrant of this warp
    const int r = 32 * q + lane;           // token row i (or state row n)
    const uint32_t lrow = (uint32_t)(32 * q) << 16;
    const float bias = prm.dt_bias ? prm.dt_bias[h] : 0.f;
    const float Dh = prm.D ? prm.D[h] : 0.f;
    const float a2 = Ah * kLog2e;
    auto ewait = [&](uint64_t* bar, uint32_t par) -> bool {
      const bool ok = mbar_wait(bar, par, abort_flag, kWaitLimit);
      return __all_sync(0xffffffffu, ok);
    };
    // dt and the base-2 cumulative decay of chunk c, computed by the four hf == 0 warps
    // (each warp forms the sums of the lower quadrants itself, so no cross-warp step).
    auto prologue = [&](int c) -> bool {
      if (hf != 0) return true;
      const int b = c & 1;
      if (c >= 2 && !ewait(&pro_empty[b], ((c >> 1) - 1) & 1)) return false;
      float own_dt = 0.f, own_a = 0.f, pre = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int tok = t0 + c * QT + 32 * k + lane;
        const float d = tok < t1 ? dt_prep(prm.dt[(size_t)tok * H + h], bias, prm.dt_softplus)
                                 : 0.f;
        const float av = d * a2;
        if (k < q) {
          float sum = av;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
          pre += sum;
        }
        if (k == q) {
          own_dt = d;
          own_a = av;
        }
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float nb = __shfl_up_sync(0xffffffffu, own_a, off);
        if (lane >= off) own_a += nb;
      }
      dt_s[b * QT + r] = own_dt;
      cs_s[b * QT + r] = pre + own_a;
      __syncwarp();
      if (lane == 0) mbar_arrive(&pro_full[b]);
      return true;
    };

    // state rows n = r, channels p0 + hf*PH + k
    float hreg[PH];
    const bool has_init =
        prm.init && (prm.has_init == nullptr || prm.has_init[s] != 0);
#pragma unroll
    for (int k = 0; k < PH; ++k)
      hreg[k] = has_init ? prm.init[((size_t)s * H + h) * PN + (size_t)(p0 + hf * PH + k) * NSTATE + r]
                         : 0.f;
    auto write_hT = [&]() {
#pragma unroll
      for (int k8 = 0; k8 < PH / 8; ++k8) {
        uint4 v;
        v.x = pack_bf16(hreg[8 * k8 + 0], hreg[8 * k8 + 1]);
        v.y = pack_bf16(hreg[8 * k8 + 2], hreg[8 * k8 + 3]);
        v.z = pack_bf16(hreg[8 * k8 + 4], hreg[8 * k8 + 5]);
        v.w = pack_bf16(hreg[8 * k8 + 6], hreg[8 * k8 + 7]);
        const uint32_t off = swz((uint32_t)(r * L::kXRow + 16 * (hf * PH / 8 + k8)), L::kSwB);
        *reinterpret_cast<uint4*>(sm + L::kHT + off) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(h_ready);
    };
    write_hT();

    bool ok = (nch == 0) || prologue(0);
    for (int c = 0; ok && c < nch; ++c) {
      const int st = c % NST, b = c & 1;
      const uint8_t* xt = sm + st * L::kStage + L::kStageX;
      if (!(ok = ewait(&full[st], (c / NST) & 1))) break;
      if (!(ok = ewait(&pro_full[b], (c >> 1) & 1))) break;
      if (!(ok = ewait(&cb_full[b], (c >> 1) & 1))) break;
      tc_fence_after();
      const float* dtb = dt_s + b * QT;
      const float* csb = cs_s + b * QT;
      const float cs_i = csb[r];
      const float cs_last = csb[QT - 1];
      const float dt_r = dtb[r];

      // (b) decay mask: M[i, j] = CB[i, j] 2^(cs_i - cs_j) dt_j for j <= i, bf16 into TMEM
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int jb = hf + 2 * jj;  // 32-column block
        uint32_t pk[16];
        if (jb > q) {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = 0u;
        } else {
          float v[32];
          tmem_ld32(tmem + lrow + kColCB + b * 128 + jb * 32, v);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int j = jb * 32 + e;
            float m0 = v[e] * ex2(cs_i - csb[j]) * dtb[j];
            float m1 = v[e + 1] * ex2(cs_i - csb[j + 1]) * dtb[j + 1];
            if (jb == q && e > lane) m0 = 0.f;
            if (jb == q && e + 1 > lane) m1 = 0.f;
            pk[e / 2] = pack_bf16(m0, m1);
          }
        }
        tmem_st16(tmem + lrow + kColM + jb * 16, pk);
      }
      tmem_st_wait();

      // (c) w o x for token row j = r: 16-byte chunks, the swizzle only permutes chunks
      //     within a row, so the row is scaled in place of its physical chunks
      {
        const float w = ex2(cs_last - cs_i) * dt_r;
        const uint4* src = reinterpret_cast<const uint4*>(xt + r * L::kXRow);
        uint4* dst = reinterpret_cast<uint4*>(sm + L::kXs + r * L::kXRow);
        constexpr int CPH = PB / 16;  // chunks per half row
#pragma unroll
        for (int k = 0; k < CPH; ++k) {
          uint4 v = src[hf * CPH + k];
          __nv_bfloat162* e2 = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 f = __bfloat1622float2(e2[e]);
            e2[e] = __floats2bfloat162_rn(f.x * w, f.y * w);
          }
          dst[hf * CPH + k] = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&cb_empty[b]);
        mbar_arrive(m_ready);
      }

      // next chunk's dt / cumsum while the tensor core runs
      if (c + 1 < nch && !(ok = prologue(c + 1))) break;

      // (d) y = Y + 2^cs_i Yoff + D x, rows i = r, channels of this half
      if (!(ok = ewait(acc_full, c & 1))) break;
      if (!(ok = ewait(yoff_full, c & 1))) break;
      tc_fence_after();
      {
        float yv[PH], yo[PH];
        tmem_ld<PH>(tmem + lrow + kColY + hf * PH, yv);
        tmem_ld<PH>(tmem + lrow + kColY + PB + hf * PH, yo);
        const float e_i = ex2(cs_i);
        const int tok = t0 + c * QT + r;
#pragma unroll
        for (int k8 = 0; k8 < PH / 8; ++k8) {
          const uint32_t off = swz((uint32_t)(r * L::kXRow + 16 * (hf * PH / 8 + k8)), L::kSwB);
          uint4 xv = *reinterpret_cast<const uint4*>(xt + off);
          const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xv);
          uint4 o;
          uint32_t* o32 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 xf = __bfloat1622float2(x2[e]);
            const int k = 8 * k8 + 2 * e;
            const float y0 = fmaf(e_i, yo[k], yv[k]) + Dh * xf.x;
            const float y1 = fmaf(e_i, yo[k + 1], yv[k + 1]) + Dh * xf.y;
            o32[e] = pack_bf16(y0, y1);
          }
          if (tok < t1)
            *reinterpret_cast<uint4*>(prm.y + ((size_t)tok * H + h) * P + p0 + hf * PH + 8 * k8) = o;
        }
      }
      // (e) state pass: h = 2^cs_last h + S, rows n = r
      {
        float sv[PH];
        tmem_ld<PH>(tmem + lrow + kColY + 2 * PB + hf * PH, sv);
        const float e_l = ex2(cs_last);
#pragma unroll
        for (int k = 0; k < PH; ++k) hreg[k] = fmaf(e_l, hreg[k], sv[k]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(acc_empty);
        mbar_arrive(&pro_empty[b]);
        mbar_arrive(&empty[st]);
      }
      if (c + 1 < nch) write_hT();
    }
    if (ok && fin) {
#pragma unroll
      for (int k = 0; k < PH; ++k) fin[(size_t)(hf * PH + k) * NSTATE + r] = hreg[k];
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) set_status(prm.status, SSD_DEV_TIMEOUT);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 tensor map: dims (d0 innermost, d1, d2) with byte strides s1, s2.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b2, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, 1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int PB>
ssd_status launch_pb(const ssd_scan_args& a, cudaStream_t st) {
  using L = Layout<PB>;
  const int64_t xs = a.x_stride_t ? a.x_stride_t : (int64_t)a.H * a.P;
  const int64_t bs = a.B_stride_t ? a.B_stride_t : (int64_t)a.G * a.N;
  const int64_t cs = a.C_stride_t ? a.C_stride_t : (int64_t)a.G * a.N;
  const uint64_t T = a.T > 0 ? (uint64_t)a.T : 1;
  CUtensorMap mX, mB, mC;
  const CUtensorMapSwizzle xsw = PB == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : PB == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
  if (!make_map(&mX, a.x, a.P, a.H, T, (uint64_t)a.P * 2, (uint64_t)xs * 2, PB, QT, xsw) ||
      !make_map(&mB, a.B, NSTATE, a.G, T, NSTATE * 2, (uint64_t)bs * 2, 64, QT,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mC, a.C, NSTATE, a.G, T, NSTATE * 2, (uint64_t)cs * 2, 64, QT,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return SSD_ERR_CUDA;
  static bool attr_set = false;  // per template instance
  if (!attr_set) {
    if (cudaFuncSetAttribute(scan_tc_kernel<PB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kSmemBytes) != cudaSuccess)
      return SSD_ERR_CUDA;
    attr_set = true;
  }
  TcParams prm;
  prm.dt = a.dt;
  prm.dt_bias = a.dt_bias;
  prm.A = a.A;
  prm.D = a.D;
  prm.init = a.initial_states;
  prm.has_init = a.has_initial_state;
  prm.cu = a.cu_seqlens;
  prm.y = static_cast<__nv_bfloat16*>(a.y);
  prm.fin = a.final_states;
  prm.status = a.d_status;
  prm.nseq = a.nseq;
  prm.T = a.T;
  prm.H = a.H;
  prm.P = a.P;
  prm.G = a.G;
  prm.npb = a.P / PB;
  prm.dt_softplus = a.dt_softplus;
  const long long grid = (long long)a.nseq * a.H * prm.npb;
  scan_tc_kernel<PB><<<(unsigned)grid, kThreads, L::kSmemBytes, st>>>(mX, mB, mC, prm);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool scan_tc_supported(const ssd_scan_args& a, int* pb_out) {
  if (a.act_dtype != SSD_BF16 || a.N != NSTATE || a.P % 16 != 0 || a.T < 1) return false;
  if (a.chunk_size != 64 && a.chunk_size != 128 && a.chunk_size != 256) return false;
  const int64_t xs = a.x_stride_t ? a.x_stride_t : (int64_t)a.H * a.P;
  const int64_t bs = a.B_stride_t ? a.B_stride_t : (int64_t)a.G * a.N;
  const int64_t cs = a.C_stride_t ? a.C_stride_t : (int64_t)a.G * a.N;
  auto al16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  if (!al16(a.x) || !al16(a.B) || !al16(a.C) || !al16(a.y)) return false;
  if ((xs * 2) % 16 || (bs * 2) % 16 || (cs * 2) % 16) return false;
  if ((long long)a.nseq * a.H * (a.P / 16) > 0x7fffffffLL) return false;
  int pb = a.p_block;
  if (pb) {
    if (a.P % pb) return false;
  } else {
    // Fewest waves of CTAs over 148+ SMs, with a per-chunk cost model in which a CTA's
    // time grows slowly with its channel block (the C.B^T product and the decay mask do
    // not depend on it): cost(PB) ~ 1 + PB/64.
    double best = 1e30;
    for (int cand : {64, 32, 16}) {
      if (a.P % cand) continue;
      const long long ctas = (long long)a.nseq * a.H * (a.P / cand);
      const long long waves = (ctas + 147) / 148;
      const double cost = (double)waves * (1.0 + cand / 64.0);
      if (cost < best - 1e-9) {
        best = cost;
        pb = cand;
      }
    }
  }
  if (pb != 16 && pb != 32 && pb != 64) return false;
  *pb_out = pb;
  return true;
}

ssd_status launch_scan_tc(const ssd_scan_args& a, int pb, cudaStream_t st) {
  switch (pb) {
    case 64: return launch_pb<64>(a, st);
    case 32: return launch_pb<32>(a, st);
    case 16: return launch_pb<16>(a, st);
  }
  return SSD_ERR_UNSUPPORTED;
}

}  // namespace ssd
