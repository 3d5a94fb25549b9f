// scan_pair.cuh -- the tensor-core chunked scan over pairs of heads (included by
// scan_tc.cu, which defines TcParams, the constants and the helpers used here).
//
// The products of a chunk are those of the single-head kernel (C.B^T, the decay mask,
// Y = M x, the chunk state, Yoff = C h^T, y = Y + 2^cs_i Yoff + D x), but one CTA owns two
// heads h0, h0 + 1 of the same group, all 64 channels of a channel block each.  The two
// heads read the same B and C tiles, so per chunk:
//   - C.B^T is computed once (8 MMAs at N = 128) and masked twice, once per head;
//   - the chunk state of both heads is one product, S^T = B^T [w0 o x0 | w1 o x1] (N = 128);
//   - Yoff of both heads is one product, C [h0^T | h1^T] (N = 128);
//   - only Y = M x stays per head (two chains of N = 64).
// That halves the tensor-core instructions, the TMA traffic of B and C and the pipeline
// handoffs per head and chunk compared with one head per CTA.
//
// Tensor memory (512 columns, single-buffered):
//   [0, 128)    C.B^T (fp32), then the two bf16 masks in place: the mask of head e for
//               32-column block jb goes to columns [32 jb + 16 e, 32 jb + 16 e + 16), which
//               lie inside the columns of C.B^T block jb that the same warp has just read
//   [128, 256)  Y of head 0 | head 1
//   [256, 384)  the state h^T (row n, columns p of head 0 | head 1), fp32: the output
//               warps store 2^cs_last h_{c-1} there and the chunk-state product
//               accumulates onto it, so h_c never leaves tensor memory
//   [384, 512)  Yoff of head 0 | head 1
// Shared memory: one B tile and one C tile (32 KB each), two x buffers (two heads each),
// the w o x tile and the bf16 h^T tile of both heads (32 KB each), the decay ring.
//
// Warp roles (640 threads): warp 0 TMA producer, warp 1 TMEM owner and MMA issuer,
// warps 2-3 decay warps (one per head), warps 4-11 mask warps (w o x, then the two
// masks), warps 12-15 state warps (the state step: h_c -> h^T and 2^cs_last h_c, on the
// chain that feeds the next chunk's products), warps 16-19 epilogue warps (y of both
// heads).  Y and Yoff are single-buffered, so the epilogue is on the loop that frees them
// for the next chunk; the state step runs in warps of its own beside it.  The epilogue
// writes each row of y with full 32-byte sector stores straight from registers: no
// shared-memory staging, which would add to the traffic of the shared-memory data path
// the tensor core reads its operands from.  The x buffer of a chunk is released as soon
// as the epilogue has read x for D x.
//
// Split sequences: a CTA may run one segment of segc chunks of a sequence (kSplit).  It
// enters the segment with the sequence's true state at that point, computed beforehand
// by the state pass and fold of scan_states.cuh, so its outputs are final and only the
// sequence's last segment writes the final state.

namespace ssd {
namespace {

namespace pair {

constexpr int PBP = 64;                 // channels per head in a CTA
constexpr int kPairMaskWarps = 8, kPairStateWarps = 4, kPairEpiWarps = 4;
constexpr int kDecay0 = 2, kMask0 = 4, kState0 = kMask0 + kPairMaskWarps;
constexpr int kEpi0 = kState0 + kPairStateWarps;
constexpr int kPairThreads = 32 * (kEpi0 + kPairEpiWarps);
template <bool kReady> constexpr int pair_threads() { return kPairThreads; }
constexpr int kTile = 16384;            // one head's [128 rows][64] bf16 tile
constexpr int kB = 0;                   // B tile, two 64-wide 128B-swizzled boxes
constexpr int kC = 32768;               // C tile
constexpr int kX = 65536;               // 2 buffers x 2 heads x kTile
constexpr int kXs = kX + 4 * kTile;     // w o x, 2 heads
constexpr int kHT = kXs + 2 * kTile;    // h^T bf16, 2 heads: [n rows][64 p]
constexpr int kPro = kHT + 2 * kTile;   // float [NB][2][kProStride]
constexpr int kDtR = kPro + NB * 2 * kProStride * 4;  // float [kDtRing][2][QT] dt
constexpr int kBar = kDtR + kDtRing * 2 * QT * 4;
constexpr int kNumBar = 2 * 2 + 2 + 2 + 2 * NB + 10;
constexpr int kFlags = kBar + kNumBar * 8;
constexpr int kSmemBytes = kFlags + 16 + 1024;
static_assert(kSmemBytes <= 232448, "dynamic shared memory per CTA");
static_assert(kBar % 8 == 0, "mbarriers need 8-byte alignment");
constexpr uint32_t kColPCB = 0, kColY = 128, kColH = 256, kColO = 384;

}  // namespace pair

// kSplit: each CTA runs one segment of a split sequence from the state it enters with
// (left by scan_state_kernel and scan_fold_kernel, scan_states.cuh).  kReady: the scan of
// the scan + norm call, which counts finished rows for the norm (a separate instantiation:
// the counting code costs the plain scan time even unexecuted).
template <bool kSplit, bool kReady = false>
__global__ void __launch_bounds__(pair::pair_threads<kReady>(), 1)
    scan_pair_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const TcParams prm) {
  using namespace pair;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int npair = prm.H / 2;
  const int pbk = unit % prm.npb;
  const int hp = (unit / prm.npb) % npair;
  const int j = unit / (prm.npb * npair);  // the sequence, or the segment when split
  const int h0 = 2 * hp;
  const int p0 = pbk * PBP;
  const int H = prm.H, P = prm.P;
  const int g = h0 / (H / prm.G);  // both heads: H / G is even
  const float A0 = prm.A[h0], A1 = prm.A[h0 + 1];

  int s = j, kseg = 0, nseg_s = 1, t0, t1;
  if constexpr (kSplit) {
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
    if (s < 0) {  // past the batch's last segment
      griddep_wait();
      return;
    }
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
    if (kSplit) griddep_wait();
    return;
  }
  const size_t PN = (size_t)P * NSTATE;
  const int nch_s = (t1 - t0 + QT - 1) / QT;
  const int c0 = kSplit ? kseg * prm.segc : 0;
  const int nch = kSplit ? max(0, min(prm.segc, nch_s - c0)) : nch_s;
  const int tb = t0 + c0 * QT;
  const int te = min(t1, tb + nch * QT);
  // per head: the sign test of A (NaN, +0, -0 fail); a failing head's outputs are zero
  const bool bad0 = !(A0 < 0.f), bad1 = !(A1 < 0.f);
  if ((bad0 || bad1) && threadIdx.x == 0 && pbk == 0 && kseg == 0)
    set_status(prm.status, SSD_DEV_A_NOT_NEG);
  // the first segment zeroes a failing head's final state
  for (int e = 0; e < 2; ++e) {
    if (!(e ? bad1 : bad0) || !prm.fin || kseg != 0) continue;
    float* fin = prm.fin + ((size_t)s * H + h0 + e) * PN + (size_t)p0 * NSTATE;
    for (int i = threadIdx.x; i < PBP * NSTATE; i += pair_threads<kReady>()) fin[i] = 0.f;
  }
  // the scan + norm call: where this CTA's two 64-channel head blocks lie among the norm
  // groups, and the id of the segment's first chunk (the sequence's chunk ids run from
  // t0 / 128 + s, and the segment starts c0 chunks in)
  const bool ready = kReady && prm.rq.cnt != nullptr;
  const int grp0 = ready ? (h0 * P + p0) / prm.rq.gs : 0;
  const int grp1 = ready ? ((h0 + 1) * P + p0) / prm.rq.gs : 0;
  const long long id0 = (long long)(tb / QT) + s;
  // count `per` contributions of each head block to chunk cc (after a barrier with every
  // thread whose y stores they stand for)
  auto publish = [&](int cc, int per) {
    if (grp0 == grp1) {
      ready_count(prm.rq, id0 + cc, grp0, 2 * per);
    } else {
      ready_count(prm.rq, id0 + cc, grp0, per);
      ready_count(prm.rq, id0 + cc, grp1, per);
    }
  };
  if (bad0 && bad1) {
    for (int e = threadIdx.x; e < (te - tb) * 2 * PBP; e += pair_threads<kReady>()) {
      const int tok = tb + e / (2 * PBP), hh = h0 + (e / PBP) % 2;
      prm.y[((size_t)tok * H + hh) * P + p0 + e % PBP] = __float2bfloat16_rn(0.f);
    }
    if (ready) {
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0)
        for (int cc = 0; cc < nch; ++cc) publish(cc, kPairEpiWarps);
    }
    if (kSplit) griddep_wait();
    return;
  }

  float* pro = reinterpret_cast<float*>(sm + kPro);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kBar);
  uint64_t* x_full = bars;               // [2]  x of both heads landed
  uint64_t* x_empty = bars + 2;          // [2]  x read (8 mask + 4 epilogue warps)
  uint64_t* b_full = bars + 4;           //      B landed
  uint64_t* b_empty = bars + 5;          //      B read by C.B^T and S (tensor core)
  uint64_t* c_full = bars + 6;           //      C landed
  uint64_t* c_empty = bars + 7;          //      C read by C.B^T and Yoff (tensor core)
  uint64_t* pro_full = bars + 8;         // [NB] decay of both heads ready (2 decay warps)
  uint64_t* pro_empty = pro_full + NB;   // [NB] consumed (8 mask + 4 epilogue warps)
  uint64_t* cb_full = pro_empty + NB;    //      C.B^T in TMEM
  uint64_t* xs_ready = cb_full + 1;      //      w o x in smem (8 mask warps)
  uint64_t* m_ready = cb_full + 2;       //      both masks in TMEM (8 mask warps)
  uint64_t* y_full = cb_full + 3;        //      Y of both heads done (frees the masks)
  uint64_t* s_full = cb_full + 4;        //      S accumulated onto the state (frees w o x)
  uint64_t* o_full = cb_full + 5;        //      Yoff done (frees h^T)
  uint64_t* h_ready = cb_full + 6;       //      scaled state in TMEM, h^T in smem (4 state)
  uint64_t* y_empty = cb_full + 7;       //      Y and Yoff read (4 epilogue warps)
  uint64_t* drain = cb_full + 8;         //      teardown: all MMAs retired
  static_assert(kNumBar == 8 + 2 * NB + 10, "barrier block size");
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kFlags + 4);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], kPairMaskWarps + kPairEpiWarps);
    }
    mbar_init(b_full, 1);
    mbar_init(b_empty, 1);
    mbar_init(c_full, 1);
    mbar_init(c_empty, 1);
    for (int i = 0; i < NB; ++i) {
      mbar_init(&pro_full[i], 2);
      mbar_init(&pro_empty[i], kPairMaskWarps + kPairEpiWarps);
    }
    mbar_init(cb_full, 1);
    mbar_init(xs_ready, kPairMaskWarps);
    mbar_init(m_ready, kPairMaskWarps);
    mbar_init(y_full, 1);
    mbar_init(s_full, 1);
    mbar_init(o_full, 1);
    mbar_init(h_ready, kPairStateWarps);
    mbar_init(y_empty, kPairEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // thread 0 is the TMA producer: chunk 0's tiles (and chunk 1's x) are on their way
    // while the rest of the CTA sets up
    for (int c = 1; c < 4 && c < nch; ++c) {
      tma_prefetch_3d(&tmB, 0, g, tb + c * QT);
      tma_prefetch_3d(&tmB, 64, g, tb + c * QT);
      tma_prefetch_3d(&tmC, 0, g, tb + c * QT);
      tma_prefetch_3d(&tmC, 64, g, tb + c * QT);
      if (c >= 2) {
        tma_prefetch_3d(&tmX, p0, h0, tb + c * QT);
        tma_prefetch_3d(&tmX, p0, h0 + 1, tb + c * QT);
      }
    }
    for (int c = 0; c < 2 && c < nch; ++c) {
      mbar_arrive_expect_tx(&x_full[c], 2 * kTile);
      tma_load_3d(sm + kX + c * 2 * kTile, &tmX, &x_full[c], p0, h0, tb + c * QT);
      tma_load_3d(sm + kX + c * 2 * kTile + kTile, &tmX, &x_full[c], p0, h0 + 1, tb + c * QT);
    }
    if (nch > 0) {
      mbar_arrive_expect_tx(b_full, 32768);
      tma_load_3d(sm + kB, &tmB, b_full, 0, g, tb);
      tma_load_3d(sm + kB + 16384, &tmB, b_full, 64, g, tb);
      mbar_arrive_expect_tx(c_full, 32768);
      tma_load_3d(sm + kC, &tmC, c_full, 0, g, tb);
      tma_load_3d(sm + kC + 16384, &tmC, c_full, 64, g, tb);
    }
  }
  // the decay warps' dt ring (kDtRing chunks in flight); lane l copies and reads tokens
  // 4 l .. 4 l + 3 of a chunk
  float* dt_ring = reinterpret_cast<float*>(sm + kDtR);
  auto fetch_dt = [&](int e, int c) {
    float* dst = dt_ring + ((c % kDtRing) * 2 + e) * QT + 4 * lane;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int tok = tb + c * QT + 4 * lane + u;
      const bool v = c < nch && tok < t1;
      cp_async4(dst + u, v ? prm.dt + (size_t)tok * H + h0 + e : prm.dt, v);
    }
    cp_async_commit();
  };
  if (warp >= kDecay0 && warp < kMask0)  // the first chunks, during the set-up
    for (int c = 0; c < kDtRing; ++c) fetch_dt(warp - kDecay0, c);
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (lane 0)
    if (lane == 0) {
      constexpr int kAhead = 4;  // L2 prefetch distance, in chunks
      int nb = nch > 0, nc = nch > 0, nx = min(nch, 2), npf = min(nch, 4);
      long long t_idle = 0;
      while (nb < nch || nc < nch || nx < nch) {
        bool progress = false;
        // the next chunk's B and C as soon as the tensor core is done with the current
        // ones (one buffer each), x two chunks ahead
        if (nb < nch && mbar_test_wait(b_empty, (nb - 1) & 1)) {
          mbar_arrive_expect_tx(b_full, 32768);
          tma_load_3d(sm + kB, &tmB, b_full, 0, g, tb + nb * QT);
          tma_load_3d(sm + kB + 16384, &tmB, b_full, 64, g, tb + nb * QT);
          ++nb;
          progress = true;
        }
        if (nc < nch && mbar_test_wait(c_empty, (nc - 1) & 1)) {
          mbar_arrive_expect_tx(c_full, 32768);
          tma_load_3d(sm + kC, &tmC, c_full, 0, g, tb + nc * QT);
          tma_load_3d(sm + kC + 16384, &tmC, c_full, 64, g, tb + nc * QT);
          ++nc;
          progress = true;
        }
        if (nx < nch && mbar_test_wait(&x_empty[nx & 1], ((nx >> 1) - 1) & 1)) {
          uint8_t* xt = sm + kX + (nx & 1) * 2 * kTile;
          mbar_arrive_expect_tx(&x_full[nx & 1], 2 * kTile);
          tma_load_3d(xt, &tmX, &x_full[nx & 1], p0, h0, tb + nx * QT);
          tma_load_3d(xt + kTile, &tmX, &x_full[nx & 1], p0, h0 + 1, tb + nx * QT);
          ++nx;
          progress = true;
        }
        while (npf < nch && npf < min(nb, nc) + kAhead) {
          const int tok = tb + npf * QT;
          tma_prefetch_3d(&tmB, 0, g, tok);
          tma_prefetch_3d(&tmB, 64, g, tok);
          tma_prefetch_3d(&tmC, 0, g, tok);
          tma_prefetch_3d(&tmC, 64, g, tok);
          tma_prefetch_3d(&tmX, p0, h0, tok);
          tma_prefetch_3d(&tmX, p0, h0 + 1, tok);
          ++npf;
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
          __nanosleep(64);
        }
      }
      // every copy issued must have landed before the CTA's shared memory is released
      if (nb > 0) mbar_wait_drain(b_full, (nb - 1) & 1, kWaitLimit);
      if (nc > 0) mbar_wait_drain(c_full, (nc - 1) & 1, kWaitLimit);
      for (int c = nx > 2 ? nx - 2 : 0; c < nx; ++c)
        mbar_wait_drain(&x_full[c & 1], (c >> 1) & 1, kWaitLimit);
    }
  } else if (warp >= kDecay0 && warp < kMask0) {
    // ------------------------------------------------------------ decay warps (one per head)
    const int e = warp - kDecay0;
    const bool bad = e ? bad1 : bad0;
    const float bias = prm.dt_bias ? prm.dt_bias[h0 + e] : 0.f;
    const float a2 = bad ? 0.f : (e ? A1 : A0) * kLog2e;
    for (int c = 0; c < nch; ++c) {
      const int b = c % NB;
      if (c >= NB && !wwait(&pro_empty[b], ((c / NB) - 1) & 1)) break;
      cp_async_wait<kDtRing - 1>();  // chunk c's copies have landed
      float raw[4], d[4], cs[4];
      const float4 r4 =
          *reinterpret_cast<const float4*>(dt_ring + ((c % kDtRing) * 2 + e) * QT + 4 * lane);
      raw[0] = r4.x;
      raw[1] = r4.y;
      raw[2] = r4.z;
      raw[3] = r4.w;
      const float cs_last =
          chunk_decay(raw, bias, a2, tb + c * QT + 4 * lane, t1, bad, prm.dt_softplus, d, cs);
      fetch_dt(e, c + kDtRing);  // into the slot just read (its values are in registers)
      put_decay(pro + (b * 2 + e) * kProStride, d, cs, cs_last);
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
      constexpr uint32_t idY = make_idesc_bf16(128, PBP, false, true);
      constexpr uint32_t idS = make_idesc_bf16(128, 2 * PBP, true, true);
      constexpr uint32_t idO = make_idesc_bf16(128, 2 * PBP, false, true);
      auto kstep_k = [](int kk) -> uint64_t {  // K-major, 128B swizzle: 64-wide K blocks
        return (uint64_t)((kk >> 2) * (16384 >> 4) + (kk & 3) * (32 >> 4));
      };
      // B read K-major (C.B^T) and MN-major (the chunk state's A = B^T, two 64-row atoms
      // 16 KB apart); C K-major; x, w o x and h^T MN-major with the two heads' tiles as
      // the two 64-column atoms of N = 128, 16 KB apart
      const uint64_t dB_k = make_sdesc(smem_u32(sm + kB), 16, 1024, kSw128);
      const uint64_t dB_mn = make_sdesc(smem_u32(sm + kB), 16384, 1024, kSw128);
      const uint64_t dC_k = make_sdesc(smem_u32(sm + kC), 16, 1024, kSw128);
      const uint64_t dX0 = make_sdesc(smem_u32(sm + kX), kTile, 1024, kSw128);
      const uint64_t dXs = make_sdesc(smem_u32(sm + kXs), kTile, 1024, kSw128);
      const uint64_t dHT = make_sdesc(smem_u32(sm + kHT), kTile, 1024, kSw128);
      int ncb = 0, ny = 0, ns = 0, no = 0;
      long long t_idle = 0;
      while (ny < nch || ns < nch || no < nch) {
        bool progress = false;
        // S(k): w o x of k; the scaled state of k-1 in TMEM; B of k.  The state region
        // always holds a valid state (zeros without an initial state), so S accumulates.
        if (ns < nch && mbar_test_wait(xs_ready, ns & 1) && mbar_test_wait(h_ready, ns & 1) &&
            mbar_test_wait(b_full, ns & 1)) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + kColH, dB_mn + kk * 128, dXs + kk * 128, idS, 1u);
          mma_commit(s_full);
          if (ncb > ns) mma_commit(b_empty);
          ++ns;
          progress = true;
        }
        // Yoff(k): C of k; h^T of k-1; Yoff of k-1 read
        if (no < nch && mbar_test_wait(c_full, no & 1) && mbar_test_wait(h_ready, no & 1) &&
            (no == 0 || mbar_test_wait(y_empty, (no - 1) & 1))) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + kColO, dC_k + kstep_k(kk), dHT + kk * 128, idO, kk > 0);
          mma_commit(o_full);
          if (ncb > no) mma_commit(c_empty);
          ++no;
          progress = true;
        }
        // C.B^T(k): B, C of k; Y of k-1 done (its masks live in these columns)
        if (ncb < nch && ncb == ny && mbar_test_wait(b_full, ncb & 1) &&
            mbar_test_wait(c_full, ncb & 1) && (ncb == 0 || mbar_test_wait(y_full, (ncb - 1) & 1))) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + kColPCB, dC_k + kstep_k(kk), dB_k + kstep_k(kk), idCB, kk > 0);
          mma_commit(cb_full);
          if (ns > ncb) mma_commit(b_empty);
          if (no > ncb) mma_commit(c_empty);
          ++ncb;
          progress = true;
        }
        // Y(k) = M x for both heads: the masks of k; Y of k-1 read
        if (ny < ncb && mbar_test_wait(m_ready, ny & 1) &&
            (ny == 0 || mbar_test_wait(y_empty, (ny - 1) & 1))) {
          tc_fence_after();
          const uint64_t db = dX0 + (uint64_t)((ny & 1) * (2 * kTile >> 4));
#pragma unroll
          for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + kColY + e * PBP, tmem + kColPCB + 32 * (kk >> 1) + 16 * e + 8 * (kk & 1),
                     db + (uint64_t)(e * (kTile >> 4)) + kk * 128, idY, kk > 0);
          mma_commit(y_full);
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
  } else if (warp < kState0) {
    // ------------------------------------------------------------ mask warps
    const int hf = (warp - kMask0) >> 2;   // which two of the four 32-column blocks
    const int q = warp & 3;                // TMEM lane quadrant of this warp
    const int r = 32 * q + lane;           // token row i (and token row j for w o x)
    const uint32_t lrow = (uint32_t)(32 * q) << 16;
    for (int c = 0; c < nch; ++c) {
      const int sx = c & 1, b = c % NB;
      if (!wwait(&pro_full[b], (c / NB) & 1)) break;
      if (!wwait(&x_full[sx], (c >> 1) & 1)) break;
      // the w o x tile was last read by S(c - 1)
      if (c >= 1 && !wwait(s_full, (c - 1) & 1)) break;
      // (1) w o x of both heads for token row j = r, this warp's half of the row's 16-byte
      //     chunks, at their swizzled positions (the same in x and in w o x)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float w = pro[(b * 2 + e) * kProStride + kProW + r];
        const uint8_t* xt = sm + kX + sx * 2 * kTile + e * kTile;
        uint8_t* xs = sm + kXs + e * kTile;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t off = swz((uint32_t)(r * 128 + 16 * (hf * 4 + k)), 3);
          uint4 xv = *reinterpret_cast<const uint4*>(xt + off);
          __nv_bfloat162* e2 = reinterpret_cast<__nv_bfloat162*>(&xv);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(e2[t]);
            float a, bb;
            mul_f32x2(a, bb, f.x, f.y, w, w);
            e2[t] = __floats2bfloat162_rn(a, bb);
          }
          *reinterpret_cast<uint4*>(xs + off) = xv;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(xs_ready);
      // (2) the two decay masks from C.B^T, each block written back into the columns of
      //     C.B^T it came from
      if (!wwait(cb_full, c & 1)) break;
      tc_fence_after();
#pragma unroll 1
      for (int jj = 0; jj < 2; ++jj) {
        const int jb = hf + 2 * jj;  // 32-column block
        uint32_t pk[16];
        if (jb > q) {  // above the diagonal: zero for both heads
#pragma unroll
          for (int t = 0; t < 16; ++t) pk[t] = 0u;
          tmem_st16(tmem + lrow + kColPCB + 32 * jb, pk);
          tmem_st16(tmem + lrow + kColPCB + 32 * jb + 16, pk);
          continue;
        }
        float v[32];
        tmem_ld32(tmem + lrow + kColPCB + 32 * jb, v);
        // column 32 jb + t of row r is kept when t <= tmax (causal)
        const int tmax = jb < q ? 31 : lane;
        if (jb == q) {  // C.B^T zeroed above the diagonal (the factorised products stay finite)
#pragma unroll
          for (int t = 0; t < 32; ++t)
            if (t > lane) v[t] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float* pb = pro + (b * 2 + e) * kProStride;
          if (pb[kProSafe + jb] != 0.f) {
            float rowf[4];
            mask_row_factors(pb[kProCs + r], pb + kProCs + 32 * jb, rowf);
            const float4* cf = reinterpret_cast<const float4*>(pb + kProColf + 32 * jb);
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const float4 f = cf[e4];
              const float rf = rowf[e4 >> 1];
              float u0, u1, u2, u3, m0, m1, m2, m3;
              mul_f32x2(u0, u1, rf, rf, f.x, f.y);
              mul_f32x2(u2, u3, rf, rf, f.z, f.w);
              mul_f32x2(m0, m1, v[4 * e4 + 0], v[4 * e4 + 1], u0, u1);
              mul_f32x2(m2, m3, v[4 * e4 + 2], v[4 * e4 + 3], u2, u3);
              pk[2 * e4] = pack_bf16(m0, m1);
              pk[2 * e4 + 1] = pack_bf16(m2, m3);
            }
          } else {
            // the exact decay, one exponential per element (its masked entries may
            // overflow where cs falls steeply, so they are selected away: 0 * inf is NaN)
            const float cs_i = pb[kProCs + r];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const int jt = 32 * jb + 2 * t;
              const float f0 = ex2(cs_i - pb[kProCs + jt]) * pb[kProDt + jt];
              const float f1 = ex2(cs_i - pb[kProCs + jt + 1]) * pb[kProDt + jt + 1];
              pk[t] = pack_bf16(2 * t <= tmax ? v[2 * t] * f0 : 0.f, 2 * t + 1 <= tmax ? v[2 * t + 1] * f1 : 0.f);
            }
          }
          tmem_st16(tmem + lrow + kColPCB + 32 * jb + 16 * e, pk);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(m_ready);
        mbar_arrive(&x_empty[sx]);
        mbar_arrive(&pro_empty[b]);
      }
    }
  } else if (warp < kEpi0) {
    // ------------------------------------------------------------ state warps
    const int q = warp & 3;
    const int r = 32 * q + lane;           // state row n of h
    const uint32_t lrow = (uint32_t)(32 * q) << 16;
    // the state the chain enters with: the initial state (or zero), or for a later
    // segment of a split sequence the one the state fold left in the segment before's slot
    const bool has_init = prm.init && (prm.has_init == nullptr || prm.has_init[s] != 0);
    const float* entry = kSplit && kseg > 0 ? prm.ws_h + (size_t)(j - 1) * H * PN
                         : has_init        ? prm.init + (size_t)s * H * PN
                                           : nullptr;
    // where the end state of head e goes: the final state, written by a sequence's last
    // segment (the state pass has the others')
    auto end_state = [&](int e) -> float* {
      if (kSplit && kseg + 1 < nseg_s) return nullptr;
      const size_t hoff = (size_t)(h0 + e) * PN + (size_t)p0 * NSTATE + r;
      return prm.fin ? prm.fin + (size_t)s * H * PN + hoff : nullptr;
    };
    // h^T (bf16, row n = r, 16 channels of head e from `col`) into the shared tile
    auto put_hT = [&](int e, int col, const float (&v)[16]) {
      uint8_t* ht = sm + kHT + e * kTile;
#pragma unroll
      for (int k8 = 0; k8 < 2; ++k8) {
        uint4 w;
        w.x = pack_bf16(v[8 * k8 + 0], v[8 * k8 + 1]);
        w.y = pack_bf16(v[8 * k8 + 2], v[8 * k8 + 3]);
        w.z = pack_bf16(v[8 * k8 + 4], v[8 * k8 + 5]);
        w.w = pack_bf16(v[8 * k8 + 6], v[8 * k8 + 7]);
        *reinterpret_cast<uint4*>(ht + swz((uint32_t)(r * 128 + 2 * col + 16 * k8), 3)) = w;
      }
    };
    auto st_scaled = [&](uint32_t taddr, float a, const float (&v)[16]) {
      uint32_t o[16];
#pragma unroll
      for (int t = 0; t < 16; t += 2) {
        float u0, u1;
        mul_f32x2(u0, u1, a, a, v[t], v[t + 1]);
        o[t] = __float_as_uint(u0);
        o[t + 1] = __float_as_uint(u1);
      }
      tmem_st16(taddr, o);
    };
    bool ok = true;
    if (nch == 0) {
      // an empty sequence: the end state is the initial state
#pragma unroll 1
      for (int e = 0; e < 2; ++e) {
        float* hout = end_state(e);
        if (!hout || (e ? bad1 : bad0)) continue;
        const float* src = entry ? entry + (size_t)(h0 + e) * PN + (size_t)p0 * NSTATE + r : nullptr;
        for (int p = 0; p < PBP; ++p)
          hout[(size_t)p * NSTATE] = entry ? src[(size_t)p * NSTATE] : 0.f;
      }
    } else if ((ok = wwait(&pro_full[0], 0))) {
      // the entering state: 2^cs_last(0) h_{-1} into TMEM (the chunk state accumulates onto
      // it), h_{-1}^T in bf16 for Yoff of chunk 0
      if (kSplit && kseg > 0) griddep_wait();  // the state fold's output
#pragma unroll 1
      for (int e = 0; e < 2; ++e) {
        const float a0 = ex2(pro[e * kProStride + kProCs + QT - 1]);
        const float* src = entry ? entry + (size_t)(h0 + e) * PN + (size_t)p0 * NSTATE + r : nullptr;
#pragma unroll 1
        for (int sl = 0; sl < PBP / 16; ++sl) {
          float v[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) v[t] = entry ? src[(size_t)(16 * sl + t) * NSTATE] : 0.f;
          put_hT(e, 16 * sl, v);
          st_scaled(tmem + lrow + kColH + e * PBP + 16 * sl, a0, v);
        }
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(h_ready);
    }
    for (int c = 0; ok && c < nch; ++c) {
      const bool last = c + 1 == nch;
      // h_c is in TMEM once S(c) is done; the h^T tile is free once Yoff(c) is
      if (!(ok = wwait(s_full, c & 1))) break;
      if (!(ok = wwait(o_full, c & 1))) break;
      if (!last && !(ok = wwait(&pro_full[(c + 1) % NB], ((c + 1) / NB) & 1))) break;
      tc_fence_after();
#pragma unroll 1
      for (int e = 0; e < 2; ++e) {
        const float an =
            last ? 1.f : ex2(pro[(((c + 1) % NB) * 2 + e) * kProStride + kProCs + QT - 1]);
        float* hout = last ? end_state(e) : nullptr;
        const bool zero = e ? bad1 : bad0;
#pragma unroll
        for (int sl = 0; sl < PBP / 16; sl += 2) {
          float v[16], w[16];
          tmem_ld16x2(tmem + lrow + kColH + e * PBP + 16 * sl,
                      tmem + lrow + kColH + e * PBP + 16 * sl + 16, v, w);
          if (last) {
            if (hout) {
#pragma unroll
              for (int t = 0; t < 16; ++t) {
                hout[(size_t)(16 * sl + t) * NSTATE] = zero ? 0.f : v[t];
                hout[(size_t)(16 * sl + 16 + t) * NSTATE] = zero ? 0.f : w[t];
              }
            }
          } else {
            put_hT(e, 16 * sl, v);
            put_hT(e, 16 * sl + 16, w);
            st_scaled(tmem + lrow + kColH + e * PBP + 16 * sl, an, v);
            st_scaled(tmem + lrow + kColH + e * PBP + 16 * sl + 16, an, w);
          }
        }
      }
      if (!last) {
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(h_ready);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;
    const int r = 32 * q + lane;           // token row i of y
    const uint32_t lrow = (uint32_t)(32 * q) << 16;
    const float D0 = prm.D ? prm.D[h0] : 0.f, D1 = prm.D ? prm.D[h0 + 1] : 0.f;
    const bool wide = ((uintptr_t)prm.y & 31u) == 0;  // 32-byte stores need 32-byte rows
    // the scan + norm call: this warp's rows of chunk cc are written; count them (one
    // contribution per head block), lane 0's release covering the warp's stores.  Done one
    // chunk late, when the stores have long landed, so the release waits for little.
    auto release_rows = [&](int cc) {
      __syncwarp();
      if (lane == 0) publish(cc, 1);
    };
    int c = 0;
    for (; c < nch; ++c) {
      const int b = c % NB, sx = c & 1;
      if (!wwait(y_full, c & 1)) break;
      if (!wwait(o_full, c & 1)) break;
      if (!wwait(&x_full[sx], (c >> 1) & 1)) break;
      if (!wwait(&pro_full[b], (c / NB) & 1)) break;
      if (ready && c > 0) release_rows(c - 1);
      tc_fence_after();
      const int tok = tb + c * QT + r;
#pragma unroll 1
      for (int e = 0; e < 2; ++e) {
        // y = Y + 2^cs_i Yoff + D x
        const float e_i = ex2(pro[(b * 2 + e) * kProStride + kProCs + r]);
        const bool zero = e ? bad1 : bad0;
        const float De = e ? D1 : D0;
        __nv_bfloat16* yrow = prm.y + ((size_t)tok * H + h0 + e) * P + p0;
        const uint8_t* xt = sm + kX + sx * 2 * kTile + e * kTile;
#pragma unroll
        for (int sl = 0; sl < PBP / 16; ++sl) {
          float yv[16], yo[16];
          tmem_ld16x2(tmem + lrow + kColY + e * PBP + 16 * sl,
                      tmem + lrow + kColO + e * PBP + 16 * sl, yv, yo);
          uint4 xr[2];
          xr[0] = *reinterpret_cast<const uint4*>(xt + swz((uint32_t)(r * 128 + 32 * sl), 3));
          xr[1] = *reinterpret_cast<const uint4*>(xt + swz((uint32_t)(r * 128 + 32 * sl + 16), 3));
          const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(xr);
          uint32_t o32[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const float2 xf = __bfloat1622float2(x2[t]);
            float a, bb;
            fma_f32x2(a, bb, e_i, e_i, yo[2 * t], yo[2 * t + 1], yv[2 * t], yv[2 * t + 1]);
            fma_f32x2(a, bb, De, De, xf.x, xf.y, a, bb);
            o32[t] = zero ? 0u : pack_bf16(a, bb);
          }
          if (tok < t1) {  // 16 channels = one full 32-byte sector of the row
            if (wide) {
              st_global_v8(yrow + 16 * sl, o32);
            } else {
              reinterpret_cast<uint4*>(yrow + 16 * sl)[0] = make_uint4(o32[0], o32[1], o32[2], o32[3]);
              reinterpret_cast<uint4*>(yrow + 16 * sl)[1] = make_uint4(o32[4], o32[5], o32[6], o32[7]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(y_empty);
        mbar_arrive(&x_empty[sx]);
        mbar_arrive(&pro_empty[b]);
      }
    }
    if (ready && c == nch && nch > 0) release_rows(nch - 1);
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
  // a split scan's grid ends no earlier than the state passes before it, so that whatever
  // waits for this grid finds their writes done as well
  if (kSplit) griddep_wait();
}

}  // namespace
}  // namespace ssd
