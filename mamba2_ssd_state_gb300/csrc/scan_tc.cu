// scan_tc.cu -- the chunked Mamba2 SSD scan on GB300 tensor cores (tcgen05 + TMEM + TMA).
//
// The op is vt::Mamba2ChunkScan of the vllm.cpp page "W2 finish (KERNEL-SSM-MAMBA)"; its
// mutation table (section "Evidence": M1 inter-chunk state term, M2 initial_states, M3
// states[c-1] feeding chunk c, M4 the D skip) names the parts computed here.  With
// a_t = dt_t A and, inside a chunk, cs_i = sum_{r<=i} a_r:
//     CB[i,j]  = C_i . B_j                                   (tensor core, fp32 in TMEM)
//     M[i,j]   = CB[i,j] exp(cs_i - cs_j) dt_j,  j <= i       (segsum decay, mask warps)
//     Y        = M x                                          (tensor core, A from TMEM)
//     S^T      = B^T (w o x),  w_j = exp(cs_last - cs_j) dt_j (chunk state, tensor core)
//     Yoff     = C h_{c-1}^T                                  (tensor core)
//     y_i      = Y_i + exp(cs_i) Yoff_i + D x_i               (fp32, bf16 out)
//     h_c      = exp(cs_last) h_{c-1} + S                      (state pass, fp32 registers)
//
// One CTA owns one (sequence, head, block of PB channels) chain and walks its chunks in
// order, so the state never leaves the SM: states[c-1] feeds chunk c in place, and HBM
// sees only x, B, C, dt in and y out (plus the per-sequence initial / final states).
// The channel split PB (64, 32 or 16) trades redundant C.B^T work for more chains when a
// workload has few (sequence, head) pairs.
//
// Warp roles (480 threads), pipelined across chunks:
//   warp 0      TMA producer (one lane): B and C of a chunk (two 64-wide 128B-swizzled
//               boxes each) into their own rings, freed by the tensor core as soon as
//               their last product is done, x into a ring freed by the mask and output
//               warps, plus L2 prefetches further ahead.
//   warp 1      TMEM owner (512 columns); one lane issues every MMA, in whatever order
//               their inputs become ready.
//   warps 2-9   mask warps (two per TMEM lane quadrant): first w o x into shared memory
//               (so the chunk state S, which needs no mask, starts early and frees B),
//               then C.B^T -> M (bf16, written back to TMEM as the A operand of Y = M x).
//   warps 10-13 output warps (one per quadrant): first the state, h = 2^cs_last h + S
//               in fp32 registers and h^T (bf16) for the next chunk's Yoff, then
//               y = Y + 2^cs_i Yoff + D x, then the final state.
//   warp 14     decay warp: dt (softplus), the base-2 cumulative decay, the column
//               factors of the mask and the chunk-state weights w, chunks ahead.
// TMEM: C.B^T (128 columns), M (64), Y x2, S (x2 for PB <= 32), Yoff x2 (PB each).  Y, Yoff and h^T are
// double-buffered, so chunk c+1's products run while chunk c's outputs are read; the
// state chain per chunk is S -> h -> h^T -> Yoff of the next chunk.  Every wait is
// bounded; a wait that runs out raises a CTA-wide abort flag, every role then drains
// what it has in flight and the kernel returns with SSD_DEV_TIMEOUT set.
//
// Decay mask arithmetic: exp(cs_i - cs_j) = 2^(cs2_i - cs2_a) * 2^(cs2_a - cs2_j) with the
// anchor a the first token of j's 8-token group, so the mask costs two multiplies per
// element (and four exponentials per row and 32-column block) instead of an exponential.
// The decay warp checks, per 32-column block, that the factors stay in range (column factors
// within 2^100, row factors within 2^20); a block that fails takes the exact per-element
// exponential.  With dt >= 0 only eight tokens decaying by more than
// 2^100 fail, so strong decays stay on the two-multiply path.
//
// The decay warp's lane l owns tokens 4 l .. 4 l + 3 of a chunk: one sequential prefix and
// one warp scan for the cumulative decay, a few shuffles for the block bounds.  (Its chain
// of dependent shuffles paces the pipeline when it is long: one scan per 32-token block and
// full-warp reductions took four times as many.)
//
// Few long sequences leave most SMs idle (a chain is one CTA).  The planner may then cut
// each sequence into segments of segc chunks, every segment its own chain started from a
// zero state that leaves its local end state in a caller-provided workspace.  A small
// tensor-core fix-up kernel, launched to overlap this kernel's tail, then chains those
// end states into the state each later segment entered with, adds that state's
// contribution to the segment's outputs and writes the final states.
//
// The chunk is the 128-row tcgen05 tile: sequences are split into 128-token chunks
// starting at their first token.  Chunked evaluation is exact for any chunk length, so
// the result equals the requested chunk_size's up to rounding.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "scan_segments.cuh"
#include "ssd_internal.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int QT = 128;          // chunk length = tcgen05 M
constexpr int NSTATE = 128;      // state size N of this kernel
constexpr int NBB = 2;           // TMA ring depth of B
constexpr int NB = 3;            // depth of the decay buffer ring
constexpr int kMaskWarps = 8, kOutWarps = 4;
constexpr int kDecayWarp = 2 + kMaskWarps + kOutWarps;
constexpr int kThreads = 32 * (kDecayWarp + 1);
template <bool kReady> constexpr int tc_threads() { return kThreads; }
constexpr float kLog2e = 1.4426950408889634f;
// Log2 bounds of the factorised decay mask: a column factor stays within 2^kColFactorLimit
// (so a row factor that underflows to zero drops only terms below 2^-26 of the row's own
// diagonal), a row factor within 2^kRowFactorLimit (its exponent is clamped there, so the
// rows above a group, whose entries the causal mask zeroes, keep finite products too).
constexpr float kColFactorLimit = 100.f;
constexpr float kRowFactorLimit = 20.f;
constexpr long long kWaitLimit = SSD_WAIT_LIMIT_CYCLES;  // SM cycles a wait may take

#ifdef SSD_FAULT_INJECT
// Test builds only: the decay warp of every CTA withholds the "decay ready" arrival of
// this chunk (-1 = none), so every role's bounded wait runs out and the kernel must
// abort cleanly with SSD_DEV_TIMEOUT.
__device__ int g_inject_withhold_chunk = -1;
#endif

// TMEM columns (fp32 unless noted)
constexpr uint32_t kColCB = 0;    // C.B^T, 128 columns
constexpr uint32_t kColM = 128;   // bf16 decay-masked M, 64 columns (two values per column)
constexpr uint32_t kColAcc = 192; // Y[2], S, Yoff[2]: PB columns each (5 PB <= 320)

// decay buffer: per chunk, float arrays of QT
constexpr int kProCs = 0, kProDt = QT, kProColf = 2 * QT, kProW = 3 * QT, kProSafe = 4 * QT;
constexpr int kProStride = 4 * QT + 8;  // floats
// Chunks of dt in flight per decay warp: copied asynchronously into a shared ring, since
// a plain load still in flight would hold up the warp's next mbarrier arrive (a release)
// until it landed.
constexpr int kDtRing = 4;

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
  float* ws_h;    // split sequences: a state per segment [nseg, H, P, N] (one head: the
                  // segment's local end state; two heads: the state the next one enters with)
  float* ws_cs;   // split one-head scan: log2 decay from the segment start to each token [T, H]
  float* ws_d;    // split two-head scan: total log2 decay of each segment [nseg, H]
  int nseq, T, H, P, G, npb, dt_softplus, segc;
  ReadyQueue rq;  // unsplit two-head scan of the scan + norm call: finished rows; cnt NULL = off
};

template <int PB>
struct Layout {
  static constexpr int NX = PB == 64 ? 2 : 3;          // TMA ring depth of x
  static constexpr int NBC = PB == 64 ? 2 : 3;         // TMA ring depth of C
  static constexpr int kXRow = PB * 2;                 // bytes per token row of x / x' / h^T
  static constexpr int kXBytes = QT * kXRow;
  static constexpr int kXPad = (kXBytes + 1023) / 1024 * 1024;
  static constexpr int kB = 0;                         // NBB x B tile (two [128 x 64] boxes)
  static constexpr int kC = NBB * 32768;               // NBC x C tile
  static constexpr int kX = kC + NBC * 32768;          // NX x x tile
  // w o x tiles and S accumulators: two of each where shared and tensor memory allow,
  // so the mask warps prepare chunk c+1 while S of chunk c still reads its tile
  static constexpr int NXS = PB <= 32 ? 2 : 1;
  static constexpr int kXs = kX + NX * kXPad;          // NXS x w o x
  static constexpr int kHT = kXs + NXS * kXPad;        // h^T x 2, [N rows][PB] bf16 each
  static constexpr int kHTPad = (NSTATE * kXRow + 1023) / 1024 * 1024;
  static constexpr int kPro = kHT + 2 * kHTPad;        // float [NB][kProStride]
  static constexpr int kDtR = kPro + NB * kProStride * 4;  // float [kDtRing][QT] dt
  static constexpr int kBar = kDtR + kDtRing * QT * 4;
  static constexpr int kNumBar = 2 * NBB + 2 * NBC + 2 * NX + 2 * NB + 12 + 3 * NXS;
  static constexpr int kFlags = kBar + kNumBar * 8;    // abort flag, TMEM base
  static constexpr int kEnd = kFlags + 16;
  static constexpr int kSmemBytes = kEnd + 1024;       // + alignment slack
  static constexpr int kSwB = PB == 64 ? 3 : PB == 32 ? 2 : 1;  // Swizzle<B,4,3>
  static constexpr uint32_t kSwCode = PB == 64 ? kSw128 : PB == 32 ? kSw64 : kSw32;
  // accumulator columns
  static constexpr uint32_t kY0 = kColAcc, kS = kColAcc + 2 * PB, kO0 = kColAcc + (2 + NXS) * PB;
  static_assert(kO0 + 2 * PB <= 512, "TMEM columns");
  static_assert(kSmemBytes <= 232448, "dynamic shared memory per CTA");
};

// softplus for the bf16 path: exp(v) alone below -8 (log1p(e) = e (1 - e/2 ...), relative
// error < 2e-4 there), else log(1 + e^v) with the fast exponential and logarithm; the
// error stays far below bf16's 2^-9.
__device__ __forceinline__ float softplus_fast(float v) {
  if (v > 20.f) return v;
  const float e = __expf(v);
  return v < -8.f ? e : __logf(1.f + e);
}

// The decay of one head over one 128-token chunk, by one warp whose lane l owns tokens
// 4 l .. 4 l + 3: a sequential prefix over its four tokens, then one warp scan of the lane
// sums (a scan per 32-token column block would put four times the shuffle latency on the
// warp's chain).  raw = dt of the lane's tokens before the bias; tok0 = the lane's first
// token.  d = dt after the optional softplus (zero past the sequence end and for a
// failing head), cs = the inclusive base-2 cumulative decay from the chunk's first token.
// Returns the chunk's total (the same in every lane).
__device__ __forceinline__ float chunk_decay(const float (&raw)[4], float bias, float a2,
                                             int tok0, int t1, bool bad, bool softplus,
                                             float (&d)[4], float (&cs)[4]) {
  const int lane = threadIdx.x & 31;
  float run = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float v0 = raw[u] + bias;
    d[u] = (tok0 + u < t1 && !bad) ? (softplus ? softplus_fast(v0) : v0) : 0.f;
    run += d[u] * a2;
    cs[u] = run;
  }
  float incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float nb = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += nb;
  }
  float base = __shfl_up_sync(0xffffffffu, incl, 1);  // the sum over the lanes before
  if (lane == 0) base = 0.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) cs[u] += base;
  return __shfl_sync(0xffffffffu, incl, 31);
}

// What the mask, state and output roles read of a chunk's decay, from chunk_decay's output
// (lane l's tokens 4 l .. 4 l + 3) into pb: cs, dt, the mask's column factors
// 2^(anchor - cs_j) dt_j with the anchor the first token of j's 8-token group, the chunk
// state's weights 2^(cs_last - cs_j) dt_j, and per 32-column block whether its factorised
// mask is safe: in each of its 8-token groups the column factors' exponent anchor - cs_j
// stays within kColFactorLimit and the row factors' largest exponent (the largest cs from
// the group's first token on, less the anchor) within kRowFactorLimit.  (With dt >= 0 the
// cumulative decay never increases, so the row factors stay at most 1 and a block fails
// only where 8 tokens decay by more than 2^kColFactorLimit.)
__device__ __forceinline__ void put_decay(float* pb, const float (&d)[4], const float (&cs)[4],
                                          float cs_last) {
  const int lane = threadIdx.x & 31;
  const float anchor = __shfl_sync(0xffffffffu, cs[0], lane & ~1);  // lanes 2g, 2g + 1: group g
  float span = fmaxf(fmaxf(anchor - cs[0], anchor - cs[1]), fmaxf(anchor - cs[2], anchor - cs[3]));
  float gmax = fmaxf(fmaxf(cs[0], cs[1]), fmaxf(cs[2], cs[3]));
  span = fmaxf(span, __shfl_xor_sync(0xffffffffu, span, 1));
  gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, 1));
#pragma unroll
  for (int off = 2; off < 32; off <<= 1) {  // the largest cs from the group's first token on
    const float n = __shfl_down_sync(0xffffffffu, gmax, off);
    if (lane + off < 32) gmax = fmaxf(gmax, n);
  }
  const unsigned safe =
      __ballot_sync(0xffffffffu, span <= kColFactorLimit && gmax - anchor <= kRowFactorLimit);
  float cf[4], w[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    cf[u] = ex2(anchor - cs[u]) * d[u];
    w[u] = ex2(cs_last - cs[u]) * d[u];
  }
  *reinterpret_cast<float4*>(pb + kProCs + 4 * lane) = make_float4(cs[0], cs[1], cs[2], cs[3]);
  *reinterpret_cast<float4*>(pb + kProDt + 4 * lane) = make_float4(d[0], d[1], d[2], d[3]);
  *reinterpret_cast<float4*>(pb + kProColf + 4 * lane) = make_float4(cf[0], cf[1], cf[2], cf[3]);
  *reinterpret_cast<float4*>(pb + kProW + 4 * lane) = make_float4(w[0], w[1], w[2], w[3]);
  if ((lane & 7) == 0)  // block lane / 8: its four groups, lanes lane .. lane + 7
    pb[kProSafe + (lane >> 3)] = ((safe >> lane) & 0xffu) == 0xffu ? 1.f : 0.f;
}

// The row factors of the factorised mask of the 32-column block at pbc = pb + kProCs + 32 jb
// for token row cs_i: 2^(cs_i - anchor) of its four 8-token groups, the exponent clamped to
// kRowFactorLimit (which only the rows above a group, masked, reach).
__device__ __forceinline__ void mask_row_factors(float cs_i, const float* pbc, float (&rowf)[4]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) rowf[g] = ex2(fminf(cs_i - pbc[8 * g], kRowFactorLimit));
}

// kReady: the unsplit scan of the scan + norm call, which fills the norm's ready queue
// (64-channel blocks only; its own instantiation).
template <int PB, bool kSplit, bool kReady = false>
__global__ void __launch_bounds__(tc_threads<kReady>(), 1)
    scan_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams prm) {
  using L = Layout<PB>;
  constexpr int NX = L::NX, NBC = L::NBC, NXS = L::NXS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int pbk = unit % prm.npb;
  const int h = (unit / prm.npb) % prm.H;
  const int j = unit / (prm.npb * prm.H);  // the sequence, or the segment when split
  const int p0 = pbk * PB;
  const int H = prm.H, P = prm.P;
  const int g = h / (H / prm.G);
  const float Ah = prm.A[h];  // issued first: nothing below depends on it until the test

  int s = j, kseg = 0, nseg_s = 1, t0, t1;
  if constexpr (kSplit) {  // a separate instance: the plain chain carries none of this
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
    s = seg_info[0];
    kseg = seg_info[1];
    nseg_s = seg_info[2];
    t0 = seg_info[3];
    t1 = seg_info[4];
    if (s < 0) return;  // past the batch's last segment
  } else if constexpr (kReady) {
    // the scan + norm call keeps batch order: remapping the slots measured slower there,
    // by 2-7% even where the order stays the same (a single sequence)
    t0 = prm.cu[s];
    t1 = prm.cu[s + 1];
  } else {  // the sequences longest first (scan_segments.cuh)
    lpt_sequence_warp(prm.cu, prm.nseq, prm.T, j, s, t0, t1);
  }
  if (unit == 0 && threadIdx.x == 0 && (prm.cu[0] != 0 || prm.cu[prm.nseq] != prm.T))
    set_status(prm.status, SSD_DEV_SEQ_META);
  if (!(0 <= t0 && t0 <= t1 && t1 <= prm.T)) {
    if (threadIdx.x == 0) set_status(prm.status, SSD_DEV_SEQ_META);
    return;
  }
  const size_t PN = (size_t)P * NSTATE;
  // this CTA's chunks: [c0, c0 + nch) of the sequence, first token tb
  const int nch_s = (t1 - t0 + QT - 1) / QT;
  const int c0 = kSplit ? kseg * prm.segc : 0;
  const int nch = kSplit ? max(0, min(prm.segc, nch_s - c0)) : nch_s;
  const int tb = t0 + c0 * QT;
  const int te = min(t1, tb + nch * QT);
  const bool split = nseg_s > 1;
  // where this CTA's end state goes: the final state, or (split) the segment's local one
  auto end_state = [&]() -> float* {
    if (split) return prm.ws_h + ((size_t)j * H + h) * PN + (size_t)p0 * NSTATE;
    return prm.fin ? prm.fin + ((size_t)s * H + h) * PN + (size_t)p0 * NSTATE : nullptr;
  };
  // the scan + norm call: this CTA's norm group, the id of the sequence's first chunk
  // (unsplit: tb is the sequence start), and the count of chunk cc's rows of y
  const bool ready = kReady && !kSplit && PB == 64 && prm.rq.cnt != nullptr;
  const int grp = ready ? (h * P + p0) / prm.rq.gs : 0;
  const long long id0 = (long long)(tb / QT) + s;
  if (!(Ah < 0.f)) {  // sign test (NaN, +0, -0 fail): the chain produces zeros
    if (threadIdx.x == 0 && pbk == 0 && kseg == 0) set_status(prm.status, SSD_DEV_A_NOT_NEG);
    for (int e = threadIdx.x; e < (te - tb) * PB; e += tc_threads<kReady>())
      prm.y[((size_t)(tb + e / PB) * H + h) * P + p0 + e % PB] = __float2bfloat16_rn(0.f);
    // the first segment zeroes the final state (the fix-up kernel skips such heads)
    float* fin = (prm.fin && kseg == 0)
                     ? prm.fin + ((size_t)s * H + h) * PN + (size_t)p0 * NSTATE
                     : nullptr;
    if (fin)
      for (int e = threadIdx.x; e < PB * NSTATE; e += tc_threads<kReady>()) fin[e] = 0.f;
    if (ready) {  // the zero rows count for every chunk at once
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0)
        for (int cc = 0; cc < nch; ++cc) ready_count(prm.rq, id0 + cc, grp, kOutWarps);
    }
    return;
  }

  float* pro = reinterpret_cast<float*>(sm + L::kPro);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* b_full = bars;                  // [NBB] B landed
  uint64_t* b_empty = b_full + NBB;         // [NBB] B free (MMA commit after S)
  uint64_t* c_full = b_empty + NBB;         // [NBC] C landed
  uint64_t* c_empty = c_full + NBC;         // [NBC] C free (MMA commit after Yoff)
  uint64_t* x_full = c_empty + NBC;         // [NX]  x landed
  uint64_t* x_empty = x_full + NX;          // [NX]  x free (8 mask + 4 output warps)
  uint64_t* pro_full = x_empty + NX;        // [NB]  decay of a chunk ready (decay warp)
  uint64_t* pro_empty = pro_full + NB;      // [NB]  consumed (8 mask + 4 output warps)
  // Single barriers track one phase per chunk; a resource with two buffers gets one
  // barrier per buffer, so no waiter can fall two phases behind its barrier.
  uint64_t* cb_full = pro_empty + NB;       //       C.B^T in TMEM
  uint64_t* cb_empty = cb_full + 1;         //       C.B^T read (8 mask warps)
  uint64_t* xs_ready = cb_full + 2;         // [NXS] w o x in smem (8 mask warps)
  uint64_t* s_full = xs_ready + NXS;        // [NXS] S done (also frees its w o x tile)
  uint64_t* s_empty = s_full + NXS;         // [NXS] S read (4 output warps)
  uint64_t* m_ready = s_empty + NXS;        //       M in TMEM (8 mask warps)
  uint64_t* y_full = m_ready + 1;           // [2]   Y buffer done (also frees M)
  uint64_t* h_ready = y_full + 2;           // [2]   h^T buffer written (4 output warps)
  uint64_t* yoff_full = h_ready + 2;        // [2]   Yoff buffer done
  uint64_t* y_empty = yoff_full + 2;        // [2]   Y and Yoff buffers read (4 output warps)
  uint64_t* drain = y_empty + 2;            //       teardown: all MMAs retired
  static_assert(L::kNumBar == 2 * NBB + 2 * NBC + 2 * NX + 2 * NB + 12 + 3 * NXS,
                "barrier block size must match the barriers laid out here");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kFlags + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < NBC; ++i) {
      mbar_init(&c_full[i], 1);
      mbar_init(&c_empty[i], 1);
    }
    for (int i = 0; i < NX; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], kMaskWarps + kOutWarps);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&pro_full[i], 1);
      mbar_init(&pro_empty[i], kMaskWarps + kOutWarps);
    }
    mbar_init(cb_full, 1);
    mbar_init(cb_empty, kMaskWarps);
    for (int i = 0; i < NXS; ++i) {
      mbar_init(&xs_ready[i], kMaskWarps);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kOutWarps);
    }
    mbar_init(m_ready, kMaskWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&y_full[i], 1);
      mbar_init(&h_ready[i], kOutWarps);
      mbar_init(&yoff_full[i], 1);
      mbar_init(&y_empty[i], kOutWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // thread 0 is the TMA producer: chunk 0's tiles are on their way while the rest of
    // the CTA sets up (the barriers they complete are the ones just initialised here)
    for (int c = 1; c < 4 && c < nch; ++c) {  // L2 prefetch of the next chunks
      tma_prefetch_3d(&tmB, 0, g, tb + c * QT);
      tma_prefetch_3d(&tmB, 64, g, tb + c * QT);
      tma_prefetch_3d(&tmC, 0, g, tb + c * QT);
      tma_prefetch_3d(&tmC, 64, g, tb + c * QT);
      tma_prefetch_3d(&tmX, p0, h, tb + c * QT);
    }
    if (nch > 0) {
      mbar_arrive_expect_tx(&b_full[0], 32768);
      tma_load_3d(sm + L::kB, &tmB, &b_full[0], 0, g, tb);
      tma_load_3d(sm + L::kB + 16384, &tmB, &b_full[0], 64, g, tb);
      mbar_arrive_expect_tx(&c_full[0], 32768);
      tma_load_3d(sm + L::kC, &tmC, &c_full[0], 0, g, tb);
      tma_load_3d(sm + L::kC + 16384, &tmC, &c_full[0], 64, g, tb);
      mbar_arrive_expect_tx(&x_full[0], L::kXBytes);
      tma_load_3d(sm + L::kX, &tmX, &x_full[0], p0, h, tb);
    }
  }
  // the decay warp's dt ring (kDtRing chunks in flight, the first ones during the set-up);
  // lane l copies and reads tokens 4 l .. 4 l + 3 of a chunk
  float* dt_ring = reinterpret_cast<float*>(sm + L::kDtR) + 4 * lane;
  auto fetch_dt = [&](int c) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tok = tb + c * QT + 4 * lane + u;
      const bool v = c < nch && tok < t1;
      cp_async4(dt_ring + (c % kDtRing) * QT + u, v ? prm.dt + (size_t)tok * H + h : prm.dt, v);
    }
    cp_async_commit();
  };
  if (warp == kDecayWarp)
    for (int c = 0; c < kDtRing; ++c) fetch_dt(c);
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // a programmatic dependent (the fix-up kernel of split sequences, the norm of the
  // scan + norm call) may be scheduled once every CTA holds its tensor memory; it waits
  // for this grid to complete before it reads anything this grid writes
  if (threadIdx.x == 0) griddep_launch_dependents();
  auto wwait = [&](uint64_t* bar, uint32_t par) -> bool {
    return warp_wait(bar, par, abort_flag, kWaitLimit);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (lane 0)
    if (lane == 0) {
      constexpr int kAhead = 4;  // L2 prefetch distance, in chunks
      auto prefetch = [&](int c) {
        const int tok = tb + c * QT;
        tma_prefetch_3d(&tmB, 0, g, tok);
        tma_prefetch_3d(&tmB, 64, g, tok);
        tma_prefetch_3d(&tmC, 0, g, tok);
        tma_prefetch_3d(&tmC, 64, g, tok);
        tma_prefetch_3d(&tmX, p0, h, tok);
      };
      // chunk 0's tiles and the prefetch of chunks 1..3 were issued during the set-up
      int nb_iss = nch > 0, nc_iss = nch > 0, nx_iss = nch > 0;
      for (int c = 0; c < nch; ++c) {
        const int tok = tb + c * QT;
        if (c + kAhead < nch) prefetch(c + kAhead);
        if (c == 0) continue;
        const int sb = c % NBB, sc = c % NBC, sx = c % NX;
        if (c >= NBB && !mbar_wait(&b_empty[sb], ((c / NBB) - 1) & 1, abort_flag, kWaitLimit))
          break;
        uint8_t* bt = sm + L::kB + sb * 32768;
        mbar_arrive_expect_tx(&b_full[sb], 32768);
        tma_load_3d(bt, &tmB, &b_full[sb], 0, g, tok);
        tma_load_3d(bt + 16384, &tmB, &b_full[sb], 64, g, tok);
        nb_iss = c + 1;
        if (c >= NBC && !mbar_wait(&c_empty[sc], ((c / NBC) - 1) & 1, abort_flag, kWaitLimit))
          break;
        uint8_t* ct = sm + L::kC + sc * 32768;
        mbar_arrive_expect_tx(&c_full[sc], 32768);
        tma_load_3d(ct, &tmC, &c_full[sc], 0, g, tok);
        tma_load_3d(ct + 16384, &tmC, &c_full[sc], 64, g, tok);
        nc_iss = c + 1;
        if (c >= NX && !mbar_wait(&x_empty[sx], ((c / NX) - 1) & 1, abort_flag, kWaitLimit))
          break;
        mbar_arrive_expect_tx(&x_full[sx], L::kXBytes);
        tma_load_3d(sm + L::kX + sx * L::kXPad, &tmX, &x_full[sx], p0, h, tok);
        nx_iss = c + 1;
      }
      // every copy issued must have landed before the CTA's shared memory is released
      for (int c = nb_iss > NBB ? nb_iss - NBB : 0; c < nb_iss; ++c)
        mbar_wait_drain(&b_full[c % NBB], (c / NBB) & 1, kWaitLimit);
      for (int c = nc_iss > NBC ? nc_iss - NBC : 0; c < nc_iss; ++c)
        mbar_wait_drain(&c_full[c % NBC], (c / NBC) & 1, kWaitLimit);
      for (int c = nx_iss > NX ? nx_iss - NX : 0; c < nx_iss; ++c)
        mbar_wait_drain(&x_full[c % NX], (c / NX) & 1, kWaitLimit);
    }
  } else if (warp == kDecayWarp) {
    // ------------------------------------------------------------ decay warp
    const float bias = prm.dt_bias ? prm.dt_bias[h] : 0.f;
    const float a2 = Ah * kLog2e;
    // split sequences: each token's log2 decay from its segment start, for the fix-up
    float* cs_out = (kSplit && split && pbk == 0) ? prm.ws_cs + h : nullptr;
    float seg_off = 0.f;
    for (int c = 0; c < nch; ++c) {
      const int b = c % NB;
      if (c >= NB && !wwait(&pro_empty[b], ((c / NB) - 1) & 1)) break;
      cp_async_wait<kDtRing - 1>();  // chunk c's copies have landed
      // dt, base-2 decay a = dt A log2(e), inclusive cumulative sum over the 128 tokens
      const float4 r4 = *reinterpret_cast<const float4*>(dt_ring + (c % kDtRing) * QT);
      float raw[4] = {r4.x, r4.y, r4.z, r4.w}, d[4], cs[4];
      const float cs_last =
          chunk_decay(raw, bias, a2, tb + c * QT + 4 * lane, t1, false, prm.dt_softplus, d, cs);
      fetch_dt(c + kDtRing);  // into the slot just read (its values are in registers)
      if (kSplit && cs_out) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int tok = tb + c * QT + 4 * lane + u;
          if (tok < t1) cs_out[(size_t)tok * H] = seg_off + cs[u];
        }
        seg_off += cs_last;
      }
      put_decay(pro + b * kProStride, d, cs, cs_last);
      __syncwarp();
#ifdef SSD_FAULT_INJECT
      if (lane == 0 && c != g_inject_withhold_chunk) mbar_arrive(&pro_full[b]);
#else
      if (lane == 0) mbar_arrive(&pro_full[b]);
#endif
    }
    cp_async_wait<0>();  // no copy may land after the CTA's shared memory is released
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lane 0)
    if (lane == 0) {
      constexpr uint32_t idCB = make_idesc_bf16(128, 128, false, false);
      constexpr uint32_t idY = make_idesc_bf16(128, PB, false, true);
      constexpr uint32_t idS = make_idesc_bf16(128, PB, true, true);
      constexpr uint32_t idO = make_idesc_bf16(128, PB, false, true);
      // Descriptors are built once; a K step only advances the start-address field
      // (bits 0-13, in 16-byte units), which stays inside the field for every tile here.
      auto kstep_k = [](int kk) -> uint64_t {  // K-major, 128B swizzle: 64-wide K blocks
        return (uint64_t)((kk >> 2) * (16384 >> 4) + (kk & 3) * (32 >> 4));
      };
      // per-buffer descriptors: the buffers of a ring are evenly spaced, so buffer i's
      // descriptor is buffer 0's plus i times the spacing (in 16-byte units)
      const uint64_t dB_k0 = make_sdesc(smem_u32(sm + L::kB), 16, 1024, kSw128);
      const uint64_t dB_mn0 = make_sdesc(smem_u32(sm + L::kB), 16384, 1024, kSw128);
      const uint64_t dC_k0 = make_sdesc(smem_u32(sm + L::kC), 16, 1024, kSw128);
      const uint64_t dX0 = make_sdesc(smem_u32(sm + L::kX), L::kXBytes, 8 * L::kXRow, L::kSwCode);
      const uint64_t dHT0 = make_sdesc(smem_u32(sm + L::kHT), L::kHTPad, 8 * L::kXRow, L::kSwCode);
      const uint64_t dXs = make_sdesc(smem_u32(sm + L::kXs), L::kXBytes, 8 * L::kXRow, L::kSwCode);
      // Issue whichever product is ready, each kind in chunk order:
      //   CB(k)    B, C of k landed; C.B^T of k-1 read by the mask warps
      //   S(k)     CB(k) issued; w o x of k; S of k-1 read          -> frees B of k
      //   Yoff(k)  CB(k) issued; h^T = h_{k-1}; Yoff buffer of k-2 read -> frees C of k
      //   Y(k)     M of k; Y buffer of k-2 read
      int ncb = 0, ns = 0, nyo = 0, ny = 0;
      long long t_idle = 0;
      while (ns < nch || ny < nch || nyo < nch) {
        bool progress = false;
        // S(k) uses w o x tile and accumulator k % NXS, the ((k / NXS) & 1) phase of their
        // barriers; the accumulator is free once S(k - NXS) has been read
        if (ns < ncb && mbar_test_wait(&xs_ready[ns % NXS], (ns / NXS) & 1) &&
            (ns < NXS || mbar_test_wait(&s_empty[ns % NXS], ((ns / NXS) - 1) & 1))) {
          tc_fence_after();
          // S^T = B^T (w o x): A = B read MN-major, 16 token rows (2 KB) per K step
          const uint64_t da = dB_mn0 + (uint64_t)((ns % NBB) * (32768 >> 4));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + L::kS + (ns % NXS) * PB, da + kk * 128,
                   dXs + (uint64_t)((ns % NXS) * (L::kXPad >> 4)) + kk * L::kXRow, idS, kk > 0);
          mma_commit(&s_full[ns % NXS]);
          mma_commit(&b_empty[ns % NBB]);
          ++ns;
          progress = true;
        }
        // h_j sits in h^T buffer j & 1 as that buffer's ((j + 1) >> 1)-th value
        if (nyo < ncb && mbar_test_wait(&h_ready[(nyo + 1) & 1], (nyo >> 1) & 1) &&
            (nyo < 2 || mbar_test_wait(&y_empty[nyo & 1], ((nyo >> 1) - 1) & 1))) {
          tc_fence_after();
          const uint64_t da = dC_k0 + (uint64_t)((nyo % NBC) * (32768 >> 4));
          const uint64_t db = dHT0 + (uint64_t)(((nyo + 1) & 1) * (L::kHTPad >> 4));  // h_{k-1}
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // Yoff = C h^T : K = N = 128
            mma_ss(tmem + L::kO0 + (nyo & 1) * PB, da + kstep_k(kk), db + kk * L::kXRow, idO,
                   kk > 0);
          mma_commit(&yoff_full[nyo & 1]);
          mma_commit(&c_empty[nyo % NBC]);
          ++nyo;
          progress = true;
        }
        if (ncb < nch && mbar_test_wait(&b_full[ncb % NBB], (ncb / NBB) & 1) &&
            mbar_test_wait(&c_full[ncb % NBC], (ncb / NBC) & 1) &&
            (ncb == 0 || mbar_test_wait(cb_empty, (ncb - 1) & 1))) {
          tc_fence_after();
          const uint64_t da = dC_k0 + (uint64_t)((ncb % NBC) * (32768 >> 4));
          const uint64_t db = dB_k0 + (uint64_t)((ncb % NBB) * (32768 >> 4));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // K = N = 128 in steps of 16 (32 bytes)
            mma_ss(tmem + kColCB, da + kstep_k(kk), db + kstep_k(kk), idCB, kk > 0);
          mma_commit(cb_full);
          ++ncb;
          progress = true;
        }
        if (ny < ncb && mbar_test_wait(m_ready, ny & 1) &&
            (ny < 2 || mbar_test_wait(&y_empty[ny & 1], ((ny >> 1) - 1) & 1))) {
          tc_fence_after();
          const uint64_t db = dX0 + (uint64_t)((ny % NX) * (L::kXPad >> 4));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // Y = M x : K = 128 tokens, M from TMEM (8 cols/step)
            mma_ts(tmem + L::kY0 + (ny & 1) * PB, tmem + kColM + kk * 8, db + kk * L::kXRow, idY,
                   kk > 0);
          mma_commit(&y_full[ny & 1]);
          ++ny;
          progress = true;
        }
        if (progress) {
          t_idle = 0;
        } else {
          if (*abort_flag) break;
          const long long now = clock64();
          if (t_idle == 0) t_idle = now;
          else if (now - t_idle > kWaitLimit) {
            *abort_flag = 1;
            break;
          }
          __nanosleep(32);
        }
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0, kWaitLimit);
    }
  } else if (warp < 2 + kMaskWarps) {
    // ------------------------------------------------------------ mask warps
    const int hf = (warp - 2) >> 2;        // which two of the four 32-column blocks
    const int q = warp & 3;                // TMEM lane quadrant of this warp
    const int r = 32 * q + lane;           // token row i (and token row j for w o x)
    const uint32_t lrow = (uint32_t)(32 * q) << 16;
    constexpr int CPH = PB / 16;           // 16-byte chunks of a row per warp half
    for (int c = 0; c < nch; ++c) {
      const int sx = c % NX, b = c % NB;
      if (!wwait(&pro_full[b], (c / NB) & 1)) break;
      if (!wwait(&x_full[sx], (c / NX) & 1)) break;
      const float* pb = pro + b * kProStride;
      // (1) w o x for token row j = r: logical 16-byte chunks of this half at their
      //     swizzled positions (the same in x and in w o x); the buffer is free once the
      //     previous chunk's S product is done
      // this chunk's w o x tile was last read by S(c - NXS)
      if (c >= NXS && !wwait(&s_full[c % NXS], ((c / NXS) - 1) & 1)) break;
      {
        const float w = pb[kProW + r];
        const uint8_t* xt = sm + L::kX + sx * L::kXPad;
#pragma unroll
        for (int k = 0; k < CPH; ++k) {
          const uint32_t off = swz((uint32_t)(r * L::kXRow + 16 * (hf * CPH + k)), L::kSwB);
          uint4 xv = *reinterpret_cast<const uint4*>(xt + off);
          __nv_bfloat162* e2 = reinterpret_cast<__nv_bfloat162*>(&xv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(e2[e]);
            float a, b;
            mul_f32x2(a, b, f.x, f.y, w, w);
            e2[e] = __floats2bfloat162_rn(a, b);
          }
          *reinterpret_cast<uint4*>(sm + L::kXs + (c % NXS) * L::kXPad + off) = xv;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&xs_ready[c % NXS]);
      // (2) the decay mask from C.B^T
      if (!wwait(cb_full, c & 1)) break;
      tc_fence_after();
      const float cs_i = pb[kProCs + r];
      const int nblk = (hf <= q) + (hf + 2 <= q);  // column blocks at or below the diagonal
      float v[2][32];
      if (nblk == 2)
        tmem_ld32x2(tmem + lrow + kColCB + hf * 32, tmem + lrow + kColCB + (hf + 2) * 32, v[0],
                    v[1]);
      else if (nblk == 1)
        tmem_ld32(tmem + lrow + kColCB + hf * 32, v[0]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cb_empty);
      uint32_t pk[2][16];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int jb = hf + 2 * jj;  // 32-column block
        if (jb > q) {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[jj][e] = 0u;
          continue;
        }
        float* m = v[jj];  // the mask is formed in place of C.B^T
        if (pb[kProSafe + jb] != 0.f) {
          float rowf[4];
          mask_row_factors(cs_i, pb + kProCs + 32 * jb, rowf);
          const float4* cf = reinterpret_cast<const float4*>(pb + kProColf + 32 * jb);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 f = cf[e4];
            const float rf = rowf[e4 >> 1];
            float t0, t1, t2, t3;  // rowf * colf, then times C.B^T, two lanes at a time
            mul_f32x2(t0, t1, rf, rf, f.x, f.y);
            mul_f32x2(t2, t3, rf, rf, f.z, f.w);
            mul_f32x2(m[4 * e4 + 0], m[4 * e4 + 1], m[4 * e4 + 0], m[4 * e4 + 1], t0, t1);
            mul_f32x2(m[4 * e4 + 2], m[4 * e4 + 3], m[4 * e4 + 2], m[4 * e4 + 3], t2, t3);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = 32 * jb + e;
            m[e] *= ex2(cs_i - pb[kProCs + j]) * pb[kProDt + j];
          }
        }
        if (jb == q) {  // causal mask on the diagonal block
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e > lane) m[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[jj][e] = pack_bf16(m[2 * e], m[2 * e + 1]);
      }
      // M of the previous chunk is free once its Y product is done
      if (c >= 1 && !wwait(&y_full[(c - 1) & 1], ((c - 1) >> 1) & 1)) break;
      tc_fence_after();
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
        tmem_st16(tmem + lrow + kColM + (hf + 2 * jj) * 16, pk[jj]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(m_ready);
        mbar_arrive(&x_empty[sx]);
        mbar_arrive(&pro_empty[b]);
      }
    }
  } else {
    // ------------------------------------------------------------ output warps
    const int q = warp & 3;
    const int r = 32 * q + lane;           // token row i of y, state row n of h
    const uint32_t lrow = (uint32_t)(32 * q) << 16;
    float hreg[PB];                        // h[n = r][p0 + k]
    const bool has_init =
        kseg == 0 && prm.init && (prm.has_init == nullptr || prm.has_init[s] != 0);
#pragma unroll
    for (int k = 0; k < PB; ++k)
      hreg[k] = has_init ? prm.init[((size_t)s * H + h) * PN + (size_t)(p0 + k) * NSTATE + r] : 0.f;
    // h_j goes to h^T buffer j & 1 (h_{-1}, the initial state, to buffer 1)
    auto write_hT = [&](int buf) {
      uint8_t* ht = sm + L::kHT + buf * L::kHTPad;
#pragma unroll
      for (int k8 = 0; k8 < PB / 8; ++k8) {
        uint4 v;
        v.x = pack_bf16(hreg[8 * k8 + 0], hreg[8 * k8 + 1]);
        v.y = pack_bf16(hreg[8 * k8 + 2], hreg[8 * k8 + 3]);
        v.z = pack_bf16(hreg[8 * k8 + 4], hreg[8 * k8 + 5]);
        v.w = pack_bf16(hreg[8 * k8 + 6], hreg[8 * k8 + 7]);
        *reinterpret_cast<uint4*>(ht + swz((uint32_t)(r * L::kXRow + 16 * k8), L::kSwB)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&h_ready[buf]);
    };
    write_hT(1);
    const float Dh = prm.D ? prm.D[h] : 0.f;
    // the scan + norm call: this warp's rows of chunk cc are written; count them, lane 0's
    // release covering the warp's stores.  Done one chunk late, when the stores have long
    // landed.
    auto release_rows = [&](int cc) {
      __syncwarp();
      if (lane == 0) ready_count(prm.rq, id0 + cc, grp, 1);
    };
    bool ok = true;
    int c = 0;
    for (; c < nch; ++c) {
      const int b = c % NB, sx = c % NX;
      if (!(ok = wwait(&pro_full[b], (c / NB) & 1))) break;
      if (!(ok = wwait(&s_full[c % NXS], (c / NXS) & 1))) break;
      tc_fence_after();
      const float* pb = pro + b * kProStride;
      // state first: h = 2^cs_last h + S, then h^T for the next chunk's Yoff
      const float e_l = ex2(pb[kProCs + QT - 1]);
#pragma unroll
      for (int sl = 0; sl < PB / 16; ++sl) {
        float sv[16];
        tmem_ld16(tmem + lrow + L::kS + (c % NXS) * PB + 16 * sl, sv);
#pragma unroll
        for (int e = 0; e < 16; e += 2)
          fma_f32x2(hreg[16 * sl + e], hreg[16 * sl + e + 1], e_l, e_l, hreg[16 * sl + e],
                    hreg[16 * sl + e + 1], sv[e], sv[e + 1]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[c % NXS]);
      if (c + 1 < nch) write_hT(c & 1);
      // then y = Y + 2^cs_i Yoff + D x
      if (!(ok = wwait(&y_full[c & 1], (c >> 1) & 1))) break;
      if (!(ok = wwait(&yoff_full[c & 1], (c >> 1) & 1))) break;
      if (!(ok = wwait(&x_full[sx], (c / NX) & 1))) break;
      if (ready && c > 0) release_rows(c - 1);
      tc_fence_after();
      const float e_i = ex2(pb[kProCs + r]);
      const int tok = tb + c * QT + r;
      __nv_bfloat16* yrow = prm.y + ((size_t)tok * H + h) * P + p0;
      const uint8_t* xt = sm + L::kX + sx * L::kXPad;
      const uint32_t colY = tmem + lrow + L::kY0 + (c & 1) * PB;
      const uint32_t colO = tmem + lrow + L::kO0 + (c & 1) * PB;
#pragma unroll
      for (int sl = 0; sl < PB / 16; ++sl) {
        float yv[16], yo[16];
        tmem_ld16x2(colY + 16 * sl, colO + 16 * sl, yv, yo);
        uint4 xr[2];
        xr[0] = *reinterpret_cast<const uint4*>(xt + swz((uint32_t)(r * L::kXRow + 32 * sl), L::kSwB));
        xr[1] = *reinterpret_cast<const uint4*>(xt + swz((uint32_t)(r * L::kXRow + 32 * sl + 16), L::kSwB));
        const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(xr);
        uint4 o[2];
        uint32_t* o32 = reinterpret_cast<uint32_t*>(o);
#pragma unroll
        for (int e = 0; e < 8; ++e) {  // y = D x + (2^cs_i Yoff + Y), two channels at a time
          const float2 xf = __bfloat1622float2(x2[e]);
          float a, b;
          fma_f32x2(a, b, e_i, e_i, yo[2 * e], yo[2 * e + 1], yv[2 * e], yv[2 * e + 1]);
          fma_f32x2(a, b, Dh, Dh, xf.x, xf.y, a, b);
          o32[e] = pack_bf16(a, b);
        }
        if (tok < t1) {
          reinterpret_cast<uint4*>(yrow + 16 * sl)[0] = o[0];
          reinterpret_cast<uint4*>(yrow + 16 * sl)[1] = o[1];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&y_empty[c & 1]);
        mbar_arrive(&x_empty[sx]);
        mbar_arrive(&pro_empty[b]);
      }
    }
    if (ready && c == nch && nch > 0) release_rows(nch - 1);
    // the final state, or a segment's local end state (the fix-up kernel chains those)
    float* hout = ok ? end_state() : nullptr;
    if (hout) {
#pragma unroll
      for (int k = 0; k < PB; ++k) hout[(size_t)k * NSTATE + r] = hreg[k];
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag) {
    set_status(prm.status, SSD_DEV_TIMEOUT);
    if (ready) atomicExch(prm.rq.abort, 1);  // the norm stops waiting for these rows
  }
}

#ifdef SSD_FAULT_INJECT
}  // namespace
extern "C" SSD_API int ssd_test_withhold_chunk(int chunk) {
  return (int)cudaMemcpyToSymbol(g_inject_withhold_chunk, &chunk, sizeof(int));
}
namespace {
#endif
}  // namespace
}  // namespace ssd

#include "scan_pair.cuh"
#include "scan_states.cuh"

namespace ssd {
namespace {

// ------------------------------------------------------------------ split sequences
//
// When a sequence is split into segments, segment k > 0 was scanned from a zero state and
// left its local end state L_k.  With d_k the segment's total log2 decay, the state that
// entered segment k is
//     H_1 = L_0,   H_{i+1} = 2^{d_i} H_i + L_i,
// the final state is 2^{d_last} H_last + L_last, and the outputs of segment k miss
//     y_t += 2^{cs'_t} C_t H_k^T,   cs'_t = sum of dt A log2(e) from the segment start to t.
// The scan kernel leaves L_k and every token's cs'_t (d_k is cs' at the segment's last
// token) in the workspace.  One fix-up CTA per (later segment, head, channel block) forms
// H_k from the L_i, adds that term chunk by chunk (tensor core: C H_k^T; y tiles in and
// out by TMA through a three-deep shared ring) and, for the last segment, writes the
// final state.  It is launched with programmatic stream
// serialisation: its set-up and its C loads overlap the scan kernel's tail, and it waits
// for the scan to complete before it reads what the scan wrote.

constexpr int kMaxSegs = 64;      // segments per sequence (the planner keeps to it)
constexpr int kFixThreads = 192;  // warp 0 TMA, warp 1 TMEM + MMA, warps 2-5 epilogue

struct FixParams {
  const float* A;
  const int32_t* cu;
  __nv_bfloat16* y;
  const float* ws_h;   // local end states of the segments [nseg, H, P, N]
  const float* ws_cs;  // log2 decay from the segment start to each token [T, H]
  float* fin;
  uint32_t* status;
  int nseq, T, H, P, G, npb, segc;
};

template <int PB>
struct FixLayout {
  static constexpr int kXRow = PB * 2;
  static constexpr int kC = 0;                          // 2 x C tile (32 KB each)
  static constexpr int kHT = 65536;                     // H_k^T, [N rows][PB] bf16
  static constexpr int kHTPad = (NSTATE * kXRow + 1023) / 1024 * 1024;
  static constexpr int kYPad = (QT * kXRow + 1023) / 1024 * 1024;  // a [128 tokens][PB] y tile
  static constexpr int NY = 3;                                     // y tile ring depth
  static constexpr int kY = kHT + kHTPad;                          // NY x y tile
  static constexpr int kBar = kY + NY * kYPad;
  static constexpr int kNumBar = 10 + 2 * NY;
  static constexpr int kFlags = kBar + kNumBar * 8;
  static constexpr int kSmemBytes = kFlags + 16 + 1024;
  static constexpr int kSwB = PB == 64 ? 3 : PB == 32 ? 2 : 1;
  static constexpr uint32_t kSwCode = PB == 64 ? kSw128 : PB == 32 ? kSw64 : kSw32;
  static_assert(kBar % 8 == 0, "mbarriers need 8-byte alignment");
};

template <int PB>
__global__ void __launch_bounds__(kFixThreads, 1)
    scan_fixup_kernel(const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmY, const FixParams prm) {
  using L = FixLayout<PB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int pbk = unit % prm.npb;
  const int h = (unit / prm.npb) % prm.H;
  const int j = unit / (prm.npb * prm.H);
  const int p0 = pbk * PB;
  const int H = prm.H, P = prm.P;
  __shared__ int seg_info[5];
  if (threadIdx.x < 32) {
    int ss = -1, kk = 0, nn = 0, a = 0, b = 0;
    find_segment_warp(prm.cu, prm.nseq, prm.segc, j, ss, kk, nn, a, b);
    if (threadIdx.x == 0) {
      seg_info[0] = ss;
      seg_info[1] = kk;
      seg_info[2] = nn;
      seg_info[3] = a;
      seg_info[4] = b;
    }
  }
  __syncthreads();
  // A CTA with nothing to do still waits for the scan grid before it leaves, so that this
  // grid never completes before the scan does: a programmatic dependent of this kernel
  // (the norm of the scan + norm call) relies on that to read the scan's outputs.
  const int s = seg_info[0], kseg = seg_info[1], nseg_s = seg_info[2];
  if (s < 0 || kseg == 0) {  // a first segment has nothing to add
    griddep_wait();
    return;
  }
  const int t0 = seg_info[3], t1 = seg_info[4];
  const float Ah = prm.A[h];
  // malformed lengths are reported by the scan kernel; it zeroed heads with A not < 0
  if (!(0 <= t0 && t0 <= t1 && t1 <= prm.T) || !(Ah < 0.f)) {
    griddep_wait();
    return;
  }
  if (nseg_s > kMaxSegs) {  // the planner never gets here; a malformed batch might
    if (threadIdx.x == 0) set_status(prm.status, SSD_DEV_SEQ_META);
    griddep_wait();
    return;
  }
  const int seg_tokens = prm.segc * QT;
  const int nch_s = (t1 - t0 + QT - 1) / QT;
  const int c0 = kseg * prm.segc;
  const int nch = max(0, min(prm.segc, nch_s - c0));
  const int tb = t0 + c0 * QT;
  const bool last = kseg == nseg_s - 1;
  const int gidx = h / (H / prm.G);
  const size_t PN = (size_t)P * NSTATE;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
  uint64_t* c_full = bars;         // [2] C landed
  uint64_t* c_empty = bars + 2;    // [2] C read by the tensor core
  uint64_t* acc_full = bars + 4;   // [2] C H_k^T of a chunk in TMEM
  uint64_t* acc_empty = bars + 6;  // [2] read by the 4 epilogue warps
  uint64_t* h_ready = bars + 8;    //     H_k^T in shared memory
  uint64_t* drain = bars + 9;      //     teardown: all MMAs retired
  constexpr int NY = L::NY;
  uint64_t* y_full = bars + 10;    // [NY] y tile landed
  uint64_t* y_free = y_full + NY;  // [NY] y tile written back (its store read the tile)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::kFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kFlags + 4);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c_full[i], 1);
      mbar_init(&c_empty[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(h_ready, 4);
    mbar_init(drain, 1);
    for (int i = 0; i < NY; ++i) {
      mbar_init(&y_full[i], 1);
      mbar_init(&y_free[i], 1);
    }
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
  // a programmatic dependent (the norm of the scan + norm call) may be scheduled now; it
  // waits for this grid, and so for the scan kernel before it, to complete
  if (threadIdx.x == 0) griddep_launch_dependents();
  auto wwait = [&](uint64_t* bar, uint32_t par) -> bool {
    return warp_wait(bar, par, abort_flag, kWaitLimit);
  };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer: C and y of every chunk
    if (lane == 0) {
      constexpr int kYBytes = QT * L::kXRow;
      auto load_c = [&](int c) {
        uint8_t* ct = sm + L::kC + (c & 1) * 32768;
        mbar_arrive_expect_tx(&c_full[c & 1], 32768);
        tma_load_3d(ct, &tmC, &c_full[c & 1], 0, gidx, tb + c * QT);
        tma_load_3d(ct + 16384, &tmC, &c_full[c & 1], 64, gidx, tb + c * QT);
      };
      int c_issued = 0, y_issued = 0;
      for (; c_issued < nch && c_issued < 2; ++c_issued) load_c(c_issued);  // inputs only
      griddep_wait();  // y below is the scan kernel's output
      for (int c = 0; c < nch; ++c) {
        if (c >= 2) {
          if (!mbar_wait(&c_empty[c & 1], ((c >> 1) - 1) & 1, abort_flag, kWaitLimit)) break;
          load_c(c);
          c_issued = c + 1;
        }
        if (c >= NY &&
            !mbar_wait(&y_free[c % NY], ((c / NY) - 1) & 1, abort_flag, kWaitLimit))
          break;
        mbar_arrive_expect_tx(&y_full[c % NY], kYBytes);
        tma_load_3d(sm + L::kY + (c % NY) * L::kYPad, &tmY, &y_full[c % NY], p0, h, tb + c * QT);
        y_issued = c + 1;
      }
      for (int c = c_issued > 2 ? c_issued - 2 : 0; c < c_issued; ++c)
        mbar_wait_drain(&c_full[c & 1], (c >> 1) & 1, kWaitLimit);
      for (int c = y_issued > NY ? y_issued - NY : 0; c < y_issued; ++c)
        mbar_wait_drain(&y_full[c % NY], (c / NY) & 1, kWaitLimit);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer: Yfix = C H_k^T
    if (lane == 0) {
      constexpr uint32_t idO = make_idesc_bf16(128, PB, false, true);
      const uint64_t dC0 = make_sdesc(smem_u32(sm + L::kC), 16, 1024, kSw128);
      const uint64_t dH = make_sdesc(smem_u32(sm + L::kHT), L::kHTPad, 8 * L::kXRow, L::kSwCode);
      bool ok = mbar_wait(h_ready, 0, abort_flag, kWaitLimit);
      for (int c = 0; ok && c < nch; ++c) {
        const int st = c & 1;
        if (!(ok = mbar_wait(&c_full[st], (c >> 1) & 1, abort_flag, kWaitLimit))) break;
        if (c >= 2 && !(ok = mbar_wait(&acc_empty[st], ((c >> 1) - 1) & 1, abort_flag, kWaitLimit)))
          break;
        tc_fence_after();
        const uint64_t da = dC0 + (uint64_t)(st * (32768 >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // K = N = 128 in steps of 16
          const uint64_t ko = (uint64_t)((kk >> 2) * (16384 >> 4) + (kk & 3) * (32 >> 4));
          mma_ss(tmem + st * PB, da + ko, dH + kk * L::kXRow, idO, kk > 0);
        }
        mma_commit(&acc_full[st]);
        mma_commit(&c_empty[st]);
      }
      mma_commit(drain);
      mbar_wait_drain(drain, 0, kWaitLimit);
    }
  } else {
    // ------------------------------------------------ epilogue warps (one per TMEM quadrant)
    const int q = warp & 3;
    const int r = 32 * q + lane;  // state row n of H_k^T, token row of a chunk
    const uint32_t lrow = (uint32_t)(32 * q) << 16;
    // everything below reads what the scan kernel wrote
    griddep_wait();
    // d_i: the decay from segment i's start to its last token, as the scan kernel left it
    auto seg_decay = [&](int i) -> float {
      const int te = min(t1, t0 + (i + 1) * seg_tokens);
      return prm.ws_cs[(size_t)(te - 1) * H + h];
    };
    // 1. H_k from the local end states: H_1 = L_0, H_{i+1} = 2^{d_i} H_i + L_i
    const float* loc0 = prm.ws_h + ((size_t)(j - kseg) * H + h) * PN + (size_t)p0 * NSTATE + r;
    float hin[PB];
#pragma unroll
    for (int k = 0; k < PB; ++k) hin[k] = loc0[(size_t)k * NSTATE];
    for (int i = 1; i < kseg; ++i) {
      const float d = ex2(seg_decay(i));
      const float* li = loc0 + (size_t)i * H * PN;
#pragma unroll
      for (int k = 0; k < PB; ++k) hin[k] = fmaf(d, hin[k], li[(size_t)k * NSTATE]);
    }
    {
      uint8_t* ht = sm + L::kHT;
#pragma unroll
      for (int k8 = 0; k8 < PB / 8; ++k8) {
        uint4 w;
        w.x = pack_bf16(hin[8 * k8 + 0], hin[8 * k8 + 1]);
        w.y = pack_bf16(hin[8 * k8 + 2], hin[8 * k8 + 3]);
        w.z = pack_bf16(hin[8 * k8 + 4], hin[8 * k8 + 5]);
        w.w = pack_bf16(hin[8 * k8 + 6], hin[8 * k8 + 7]);
        *reinterpret_cast<uint4*>(ht + swz((uint32_t)(r * L::kXRow + 16 * k8), L::kSwB)) = w;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(h_ready);
    }
    if (last && prm.fin) {  // final state = 2^{d_last} H_last + L_last
      const float d = ex2(seg_decay(kseg));
      const float* ll = loc0 + (size_t)kseg * H * PN;
      // every load first: a store between them could alias the next load and would
      // serialise the whole row on memory latency
#pragma unroll
      for (int k = 0; k < PB; ++k) hin[k] = fmaf(d, hin[k], ll[(size_t)k * NSTATE]);
      float* f = prm.fin + ((size_t)s * H + h) * PN + (size_t)p0 * NSTATE + r;
#pragma unroll
      for (int k = 0; k < PB; ++k) f[(size_t)k * NSTATE] = hin[k];
    }
    // 2. per chunk: y += 2^{cs'} Yfix, cs' the decay from the segment start to the row's
    // token.  The y tile comes in by TMA; each thread updates its row in shared memory;
    // a full tile goes back by one TMA store, the rows of a sequence's last, partial
    // tile by plain stores (a tile store would overwrite the next sequence's rows).
    float csn = 0.f;  // this row's decay for the next chunk, loaded a chunk ahead
    auto load_cs = [&](int c) {
      const int tok = tb + c * QT + r;
      csn = tok < t1 ? prm.ws_cs[(size_t)tok * H + h] : 0.f;
    };
    if (nch > 0) load_cs(0);
    int done_c = 0;
    for (int c = 0; c < nch; ++c) {
      const int st = c & 1;
      const int tok = tb + c * QT + r;
      const bool full_tile = tb + (c + 1) * QT <= t1;
      const float scale = ex2(csn);
      if (c + 1 < nch) load_cs(c + 1);
      const int sy = c % NY;
      // A wait that fails (an abort) skips this chunk's work, but every epilogue warp still
      // reaches the named barrier below, which ORs the failures, so they all leave the
      // loop there together: a warp leaving early would strand the others in the barrier.
      const bool ok = wwait(&acc_full[st], (c >> 1) & 1) && wwait(&y_full[sy], (c / NY) & 1);
      tc_fence_after();
      uint8_t* yt = sm + L::kY + sy * L::kYPad;
#pragma unroll
      for (int sl = 0; sl < PB / 16; ++sl) {
        if (!ok) break;
        float fv[16];
        tmem_ld16(tmem + lrow + st * PB + 16 * sl, fv);
        uint4* q0 = reinterpret_cast<uint4*>(yt + swz((uint32_t)(r * L::kXRow + 32 * sl), L::kSwB));
        uint4* q1 =
            reinterpret_cast<uint4*>(yt + swz((uint32_t)(r * L::kXRow + 32 * sl + 16), L::kSwB));
        uint4 yv[2] = {*q0, *q1};
        __nv_bfloat162* y2 = reinterpret_cast<__nv_bfloat162*>(yv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 yf = __bfloat1622float2(y2[e]);
          y2[e] = __floats2bfloat162_rn(fmaf(scale, fv[2 * e], yf.x),
                                        fmaf(scale, fv[2 * e + 1], yf.y));
        }
        if (full_tile) {
          *q0 = yv[0];
          *q1 = yv[1];
        } else if (tok < t1) {
          uint4* dst = reinterpret_cast<uint4*>(prm.y + ((size_t)tok * H + h) * P + p0 + 16 * sl);
          dst[0] = yv[0];
          dst[1] = yv[1];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&acc_empty[st]);
      if (full_tile) fence_proxy_async_smem();  // the tile store reads what the threads wrote
      if (named_bar_sync_or(1, 128, !ok)) break;  // the same decision in every epilogue warp
      if (r == 0) {
        // a tile may be refilled once its store has read it; that wait is deferred by one
        // chunk (one store group left in flight), so the store overlaps the next chunk
        if (full_tile) {
          tma_store_3d(&tmY, yt, p0, h, tb + c * QT);
          bulk_commit_group();
        }
        if (c > 0) {
          bulk_wait_read_one();
          mbar_arrive(&y_free[(c - 1) % NY]);
        }
      }
      done_c = c + 1;
    }
    if (r == 0) {
      bulk_wait_all();  // every tile store complete before the kernel ends
      if (done_c > 0) mbar_arrive(&y_free[(done_c - 1) % NY]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
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

constexpr int kMaxDevices = 64;

int current_device() {
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices ? dev : 0;
}

// SM count of the current device, looked up once per device (148 if it cannot be read).
int sm_count() {
  static std::atomic<int> sms[kMaxDevices];
  const int dev = current_device();
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// How one call runs: heads per CTA hb (1, or 2 for the pair kernel), channel block PB,
// segment length segc (0 = sequences are not split), the segment count the grid covers
// and the workspace that needs.
struct ScanPlan {
  int hb = 1;
  int pb = 0;
  int segc = 0;
  long long nseg = 0;
  size_t ws_bytes = 0;
};

// Upper bound of the segment count of a batch of nseq sequences and T tokens:
// max(1, ceil(nch_s / segc)) <= 1 + nch_s / segc and sum nch_s <= (T + 127 nseq) / 128.
long long seg_capacity(const ssd_scan_args& a, int segc) {
  return (long long)a.nseq + ((long long)a.T + (long long)(kScanChunk - 1) * a.nseq) /
                                 ((long long)kScanChunk * segc);
}

// Workspace of a split: the segments' local end states [nseg, H, P, N] fp32 (a multiple
// of 512 bytes), then each token's decay from its segment start [T, H] fp32.
size_t ws_states_bytes(const ssd_scan_args& a, long long nseg) {
  return (size_t)nseg * a.H * a.P * NSTATE * sizeof(float);
}
// The states, then one float per (token, head) (one head per CTA: each token's decay from
// its segment's start) or per (segment, head) (two heads: each segment's total decay).
size_t ws_bytes_for(const ssd_scan_args& a, long long nseg) {
  const size_t cs = (size_t)std::max<long long>(a.T, nseg) * a.H * sizeof(float);
  return (ws_states_bytes(a, nseg) + cs + 255) / 256 * 256;
}

// Smallest segment length that keeps every sequence within kMaxSegs segments: no
// sequence has more than ceil(T / 128) chunks.
int min_segc(const ssd_scan_args& a) {
  const long long nch_max = ((long long)a.T + kScanChunk - 1) / kScanChunk;
  return (int)std::max<long long>(1, (nch_max + kMaxSegs - 1) / kMaxSegs);
}

// The pair kernel takes two heads of one group per CTA, 64 channels each.
bool pair_ok(const ssd_scan_args& a) {
  return a.H % 2 == 0 && (a.H / a.G) % 2 == 0 && a.P % 64 == 0 &&
         (a.p_block == 0 || a.p_block == 64);
}

// Cost model in units of one 128-token chunk of a one-head 64-channel CTA in its steady
// state (about 2 us).  The host sees only T and nseq (the lengths live on the device),
// so sequences are taken as equally long.  One CTA per SM, grids run in waves of one CTA
// per SM.  A one-head CTA of channel block PB that runs n chunks costs about
// kRamp + n (1 + PB/256) (the mask and C.B^T work does not shrink with PB; kRamp is the
// pipeline fill of its first chunk); a pair CTA kPairRamp + n (kPairChunk0 + kPairChunk1 w)
// for two heads, w the fraction of the SMs its wave occupies (the chunks slow down as more
// chains share the memory system).  A one-head split adds the fix-up grid over the later
// segments, one CTA per (segment, head, channel block): a fixed cost per wave (its launch,
// set-up and first tile), one chained step per segment before it (the entering state) and
// per chunk 0.4 of a scan chunk when up to 96 fix-up CTAs run at once, rising to 1.1 for a
// wave of 128 or more (each chunk reads and writes a y tile; measured at 24 and at 128
// heads).  (kFixBase also carries what a split costs the scan grid itself beyond its
// chunks.)  A two-head split runs instead, before the scan, the state pass over every
// segment but a sequence's last (one CTA per segment and head pair, kStateChunk per chunk)
// and the fold (a fixed cost plus its state traffic, kFoldUnitBytes per unit).  Fitted to
// one Nemotron-H-shaped sequence of 4K, 16K and 64K tokens, the Nemotron-H varlen batch and
// Mamba2-130M-shaped batches of 2 x 2K and 1 x 16K tokens, at several segment lengths.
constexpr double kRamp = 3.0, kFixBase = 5.0, kFixPerSeg = 0.4;
constexpr double kFixChunkLo = 0.4, kFixChunkHi = 1.1;
constexpr double kPairRamp = 3.0, kPairChunk0 = 1.5, kPairChunk1 = 0.4;
constexpr double kStateRamp = 1.0, kStateChunk = 0.7, kFoldBase = 3.0;
constexpr double kFoldUnitBytes = 12e6;

double plan_cost(const ssd_scan_args& a, int hb, int pb, int segc) {
  const int sms = sm_count();
  const long long per = ((long long)a.T + a.nseq - 1) / a.nseq;
  const long long nch = std::max<long long>(1, (per + kScanChunk - 1) / kScanChunk);
  const long long nseg = segc > 0 ? (nch + segc - 1) / segc : 1;
  const long long chain = segc > 0 ? std::min<long long>(segc, nch) : nch;
  const long long per_seg = (long long)(a.H / hb) * (a.P / pb);
  const long long ctas = (long long)a.nseq * nseg * per_seg;
  const long long waves = (ctas + sms - 1) / sms;
  double cost = 0.0;
  if (hb == 2) {
    for (long long w = 0; w < waves; ++w) {
      const double busy = (double)std::min<long long>(sms, ctas - w * sms) / sms;
      cost += kPairRamp + chain * (kPairChunk0 + kPairChunk1 * busy);
    }
  } else {
    cost = (double)waves * (kRamp + chain * (1.0 + pb / 256.0));
  }
  if (nseg > 1 && hb == 2) {
    const long long st_ctas = (long long)a.nseq * (nseg - 1) * per_seg;
    const long long st_waves = (st_ctas + sms - 1) / sms;
    const double fold_bytes =
        (double)a.nseq * (nseg - 1) * a.H * a.P * NSTATE * 2.0 * sizeof(float);
    cost += st_waves * (kStateRamp + chain * kStateChunk) + kFoldBase + fold_bytes / kFoldUnitBytes;
  } else if (nseg > 1) {
    const long long fix_ctas = (long long)a.nseq * (nseg - 1) * a.H * (a.P / pb);
    const long long fix_waves = (fix_ctas + sms - 1) / sms;
    const double busy =
        std::min(1.0, std::max(0.0, (double)(std::min<long long>(fix_ctas, sms) - 96) / 32.0));
    const double per_chunk = kFixChunkLo + (kFixChunkHi - kFixChunkLo) * busy;
    cost += fix_waves * (kFixBase + kFixPerSeg * nseg + per_chunk * chain);
  }
  return cost;
}

constexpr int kMaxSplitSeqs = 1024;  // each CTA walks the sequence table to find its segment

// The norm kernel of the overlapped scan + norm starts only once every scan CTA has
// started, so that form pays only when the scan grid takes at most two waves (one CTA per
// SM): then the norm runs beside the scan's last wave.  Deeper grids leave it no time.
constexpr int kReadyMaxWaves = 2;

// A plan the overlapped scan + norm can run: 64-channel blocks, unsplit or split with two
// heads per CTA (the one-head split's fix-up rewrites y), at most kReadyMaxWaves waves.
bool ready_eligible(const ssd_scan_args& a, int hb, int pb, int segc) {
  if (pb != 64 || (segc > 0 && hb != 2)) return false;
  const long long nseg = segc > 0 ? seg_capacity(a, segc) : a.nseq;
  return nseg * (a.H / hb) * (a.P / 64) <= (long long)kReadyMaxWaves * sm_count();
}

// The cheapest plan under the cost model (ready_only: among those the overlapped scan +
// norm can run).  Splits are considered only when allowed, and only those whose workspace
// fits in ws_limit bytes.  *cost_out (if given) is the plan's modelled cost.
bool plan_scan(const ssd_scan_args& a, bool allow_split, ScanPlan* out,
               size_t ws_limit = SIZE_MAX, bool ready_only = false,
               double* cost_out = nullptr) {
  ScanPlan best;
  double best_cost = 1e300;
  const long long per = ((long long)a.T + a.nseq - 1) / a.nseq;
  const int nch = (int)std::max<long long>(1, (per + kScanChunk - 1) / kScanChunk);
  const int lo = min_segc(a);
  const int hb_lo = a.head_block == 2 ? 2 : 1, hb_hi = a.head_block == 1 ? 1 : 2;
  for (int hb = hb_lo; hb <= hb_hi; ++hb) {
    if (hb == 2 && !pair_ok(a)) continue;
    for (int pb : {64, 32, 16}) {
      if (a.P % pb || (a.p_block && a.p_block != pb) || (hb == 2 && pb != 64)) continue;
      auto consider = [&](int segc) {
        if (segc > 0 && ws_bytes_for(a, seg_capacity(a, segc)) > ws_limit) return;
        if (ready_only && !ready_eligible(a, hb, pb, segc)) return;
        const double c = plan_cost(a, hb, pb, segc);
        if (c < best_cost - 1e-9) {
          best_cost = c;
          best.hb = hb;
          best.pb = pb;
          best.segc = segc;
        }
      };
      if (a.seg_chunks >= 1) {
        consider(std::max(a.seg_chunks, lo));
      } else {
        consider(0);
        if (allow_split && a.seg_chunks == 0 && a.nseq <= kMaxSplitSeqs)
          for (int segc = lo; segc < nch; ++segc) consider(segc);
      }
    }
  }
  if (best.pb == 0) return false;
  if (best.segc > 0) {
    best.nseg = seg_capacity(a, best.segc);
    best.ws_bytes = ws_bytes_for(a, best.nseg);
  } else {
    best.nseg = a.nseq;
  }
  if (best.nseg * (a.H / best.hb) * (a.P / best.pb) > 0x7fffffffLL) return false;
  *out = best;
  if (cost_out) *cost_out = best_cost;
  return true;
}

// Opt in to the kernel's dynamic shared memory once per device.
template <typename K>
bool opt_in(K kernel, int bytes, std::atomic<bool>* done) {
  const int dev = current_device();
  if (done[dev].load(std::memory_order_acquire)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  done[dev].store(true, std::memory_order_release);
  return true;
}

template <int PB>
ssd_status launch_pb(const ssd_scan_args& a, const ScanPlan& plan, cudaStream_t st,
                     const ReadyQueue* rq = nullptr) {
  using L = Layout<PB>;
  const bool pair = plan.hb == 2;
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
  // dynamic shared memory above 48 KB is opted into once per kernel and device
  static std::atomic<bool> set_one[kMaxDevices], set_one_split[kMaxDevices],
      set_pair[kMaxDevices], set_pair_split[kMaxDevices], set_pair_ready[kMaxDevices],
      set_pair_split_ready[kMaxDevices], set_one_ready[kMaxDevices], set_fix[kMaxDevices],
      set_state[kMaxDevices];
  const bool split = plan.segc > 0;
  bool ok;
  if (pair && rq)
    ok = split ? opt_in(scan_pair_kernel<true, true>, pair::kSmemBytes, set_pair_split_ready)
               : opt_in(scan_pair_kernel<false, true>, pair::kSmemBytes, set_pair_ready);
  else if (pair)
    ok = split ? opt_in(scan_pair_kernel<true>, pair::kSmemBytes, set_pair_split)
               : opt_in(scan_pair_kernel<false>, pair::kSmemBytes, set_pair);
  else if (rq) {
    if constexpr (PB == 64) ok = opt_in(scan_tc_kernel<PB, false, true>, L::kSmemBytes, set_one_ready);
    else return SSD_ERR_UNSUPPORTED;
  } else
    ok = split ? opt_in(scan_tc_kernel<PB, true>, L::kSmemBytes, set_one_split)
               : opt_in(scan_tc_kernel<PB, false>, L::kSmemBytes, set_one);
  if (ok && split && pair) ok = opt_in(scan_state_kernel, statepass::kSmemBytes, set_state);
  if (ok && split && !pair) ok = opt_in(scan_fixup_kernel<PB>, FixLayout<PB>::kSmemBytes, set_fix);
  if (!ok) return SSD_ERR_CUDA;
  // split workspace: a state per segment, then (one head) every token's log2 decay from
  // its segment's start or (two heads) every segment's total log2 decay
  float* ws_h = split ? static_cast<float*>(a.workspace) : nullptr;
  float* ws_tail = split ? ws_h + ws_states_bytes(a, plan.nseg) / sizeof(float) : nullptr;
  float* ws_cs = pair ? nullptr : ws_tail;
  float* ws_d = pair ? ws_tail : nullptr;
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
  prm.ws_h = ws_h;
  prm.ws_cs = ws_cs;
  prm.ws_d = ws_d;
  prm.nseq = a.nseq;
  prm.T = a.T;
  prm.H = a.H;
  prm.P = a.P;
  prm.G = a.G;
  prm.npb = a.P / PB;
  prm.dt_softplus = a.dt_softplus;
  prm.segc = plan.segc;
  prm.rq = ReadyQueue{};
  if (rq) {
    if ((split && !pair) || PB != 64) return SSD_ERR_UNSUPPORTED;
    prm.rq = *rq;
  }
  const long long grid = plan.nseg * (a.H / plan.hb) * prm.npb;
  // programmatic stream serialisation: the grid may start while the one before it drains;
  // it waits for that grid's completion before it reads what that grid wrote
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  auto pdl_cfg = [&](dim3 g, int threads, int smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = g;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cfg;
  };
  if (pair && split) {
    // the state pass and the fold, then every segment from the state it enters with
    scan_state_kernel<<<(unsigned)grid, statepass::kThreads, statepass::kSmemBytes, st>>>(mX, mB, prm);
    if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
    const long long fold_x = ((long long)a.H * a.P * NSTATE / 4 + kFoldThreads - 1) / kFoldThreads;
    cudaLaunchConfig_t cf = pdl_cfg(dim3((unsigned)fold_x, (unsigned)a.nseq), kFoldThreads, 0);
    if (cudaLaunchKernelEx(&cf, scan_fold_kernel, prm) != cudaSuccess) return SSD_ERR_CUDA;
    cudaLaunchConfig_t cs3 = pdl_cfg(dim3((unsigned)grid), pair::kPairThreads, pair::kSmemBytes);
    const cudaError_t e = rq ? cudaLaunchKernelEx(&cs3, scan_pair_kernel<true, true>, mX, mB, mC, prm)
                             : cudaLaunchKernelEx(&cs3, scan_pair_kernel<true>, mX, mB, mC, prm);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  }
  if (pair && rq) {
    scan_pair_kernel<false, true><<<(unsigned)grid, pair::pair_threads<true>(), pair::kSmemBytes, st>>>(mX, mB, mC, prm);
  } else if (pair) {
    scan_pair_kernel<false><<<(unsigned)grid, pair::kPairThreads, pair::kSmemBytes, st>>>(mX, mB, mC, prm);
  } else if (rq) {
    if constexpr (PB == 64)
      scan_tc_kernel<PB, false, true><<<(unsigned)grid, tc_threads<true>(), L::kSmemBytes, st>>>(mX, mB, mC, prm);
  } else {
    if (split)
      scan_tc_kernel<PB, true><<<(unsigned)grid, kThreads, L::kSmemBytes, st>>>(mX, mB, mC, prm);
    else
      scan_tc_kernel<PB, false><<<(unsigned)grid, kThreads, L::kSmemBytes, st>>>(mX, mB, mC, prm);
  }
  if (cudaGetLastError() != cudaSuccess) return SSD_ERR_CUDA;
  if (!split) return SSD_OK;
  FixParams fp;
  fp.A = a.A;
  fp.cu = a.cu_seqlens;
  fp.y = prm.y;
  fp.ws_h = ws_h;
  fp.ws_cs = ws_cs;
  fp.fin = a.final_states;
  fp.status = a.d_status;
  fp.nseq = a.nseq;
  fp.T = a.T;
  fp.H = a.H;
  fp.P = a.P;
  fp.G = a.G;
  fp.npb = prm.npb;
  fp.segc = plan.segc;
  // the fix-up grid may start while the scan grid drains; it waits for the scan's
  // completion before it reads the scan's outputs
  cudaLaunchConfig_t cfg =
      pdl_cfg(dim3((unsigned)(plan.nseg * a.H * prm.npb)), kFixThreads, FixLayout<PB>::kSmemBytes);
  CUtensorMap mY;  // y as the fix-up reads and writes it: tiles of [128 tokens][PB channels]
  if (!make_map(&mY, a.y, a.P, a.H, T, (uint64_t)a.P * 2, (uint64_t)a.H * a.P * 2, PB, QT, xsw))
    return SSD_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, scan_fixup_kernel<PB>, mC, mY, fp) != cudaSuccess)
    return SSD_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

bool scan_tc_supported(const ssd_scan_args& a) {
  if (a.act_dtype != SSD_BF16 || a.N != NSTATE || a.P % 16 != 0 || a.T < 1) return false;
  if (a.chunk_size != 64 && a.chunk_size != 128 && a.chunk_size != 256) return false;
  const int64_t xs = a.x_stride_t ? a.x_stride_t : (int64_t)a.H * a.P;
  const int64_t bs = a.B_stride_t ? a.B_stride_t : (int64_t)a.G * a.N;
  const int64_t cs = a.C_stride_t ? a.C_stride_t : (int64_t)a.G * a.N;
  auto al16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
  if (!al16(a.x) || !al16(a.B) || !al16(a.C) || !al16(a.y)) return false;
  if ((xs * 2) % 16 || (bs * 2) % 16 || (cs * 2) % 16) return false;
  if (a.p_block && a.P % a.p_block) return false;
  ScanPlan plan;
  return plan_scan(a, false, &plan);
}

size_t scan_tc_workspace_size(const ssd_scan_args& a, size_t ws_limit) {
  if (!scan_tc_supported(a) || a.seg_chunks < 0) return 0;
  ScanPlan plan;
  if (!plan_scan(a, true, &plan, ws_limit)) return 0;
  return plan.ws_bytes;
}

namespace {
// The plan a call runs: the cheapest (splits within ws_limit when allowed), run unsplit
// when the caller's workspace is too small for the split it chose.
ssd_status final_plan(const ssd_scan_args& a, size_t ws_limit, ScanPlan* plan) {
  if (!plan_scan(a, a.seg_chunks >= 0, plan, ws_limit)) {
    if (a.seg_chunks >= 1) return SSD_ERR_UNSUPPORTED;
    if (!plan_scan(a, false, plan)) return SSD_ERR_UNSUPPORTED;
  }
  if (plan->segc > 0) {
    const bool ws_ok = a.workspace && ((uintptr_t)a.workspace & 255u) == 0 &&
                       a.workspace_bytes >= plan->ws_bytes;
    if (!ws_ok) {
      if (a.seg_chunks >= 1) return SSD_ERR_INVALID_ARG;
      if (!plan_scan(a, false, plan)) return SSD_ERR_UNSUPPORTED;  // run unsplit
    }
  }
  return SSD_OK;
}
}  // namespace

ssd_status launch_scan_tc(const ssd_scan_args& a, cudaStream_t st, size_t ws_limit) {
  ScanPlan plan;
  const ssd_status v = final_plan(a, ws_limit, &plan);
  if (v != SSD_OK) return v;
  switch (plan.pb) {
    case 64: return launch_pb<64>(a, plan, st);
    case 32: return launch_pb<32>(a, plan, st);
    case 16: return launch_pb<16>(a, plan, st);
  }
  return SSD_ERR_UNSUPPORTED;
}

// The overlapped scan + norm takes the cheapest plan it can run when the cost model puts
// that plan within kReadySlack of the cheapest plan overall: the norm it hides behind the
// scan is worth more than the difference.
constexpr double kReadySlack = 1.15;

bool ready_plan(const ssd_scan_args& a, ScanPlan* plan) {
  ScanPlan all;
  double c_all = 0.0, c_ready = 0.0;
  const bool allow = a.seg_chunks >= 0;
  if (!plan_scan(a, allow, &all, SIZE_MAX, false, &c_all)) return false;
  if (!plan_scan(a, allow, plan, SIZE_MAX, true, &c_ready)) return false;
  return c_ready <= kReadySlack * c_all;
}

bool scan_tc_ready_plan(const ssd_scan_args& a, size_t* split_bytes, int* segc) {
  if (!scan_tc_supported(a)) return false;
  ScanPlan plan;
  if (!ready_plan(a, &plan)) return false;
  *split_bytes = plan.segc > 0 ? plan.ws_bytes : 0;
  *segc = plan.segc;
  return true;
}

ssd_status launch_scan_tc_ready(const ssd_scan_args& a, const ReadyQueue& rq, cudaStream_t st) {
  ScanPlan plan;
  if (!ready_plan(a, &plan) || plan.segc != rq.segc) return SSD_ERR_UNSUPPORTED;
  if (plan.segc > 0 && !(a.workspace && ((uintptr_t)a.workspace & 255u) == 0 &&
                         a.workspace_bytes >= plan.ws_bytes))
    return SSD_ERR_INVALID_ARG;
  return launch_pb<64>(a, plan, st, &rq);
}

}  // namespace ssd
