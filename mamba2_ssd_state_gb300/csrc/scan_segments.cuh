// scan_segments.cuh -- how the tensor-core scan splits a packed batch into segments.
//
// Sequence s has nch_s = ceil(len_s / 128) chunks and nseg_s = max(1, ceil(nch_s / segc))
// segments of at most segc chunks; segments are numbered over the batch in sequence
// order.  An empty sequence keeps one segment (with no chunk) so its final state is
// still written.
#pragma once

#include <stdint.h>

namespace ssd {

constexpr int kScanChunk = 128;  // tokens per chunk of the tensor-core scan

__host__ __device__ inline int seg_count(int len, int segc) {
  const int nch = len > 0 ? (len + kScanChunk - 1) / kScanChunk : 0;
  return nch == 0 ? 1 : (nch + segc - 1) / segc;
}

// Segment j of the batch, found by all 32 lanes of one warp: its sequence s, its index k
// within s, the segment count of s and the sequence's token range [t0, t1); false when j
// lies past the last segment.  Lane l reads the lengths of sequences base + l, so a batch
// of up to 32 sequences costs one round trip to memory.  Malformed lengths count as
// empty (the kernels report them separately).  The results are the same in every lane.
__device__ inline bool find_segment_warp(const int32_t* cu, int nseq, int segc, int j, int& s,
                                         int& k, int& nseg_s, int& t0, int& t1) {
  const int lane = threadIdx.x & 31;
  int off = 0;  // segments of the sequences before base
  for (int base = 0; base < nseq; base += 32) {
    const int i = base + lane;
    int a = 0, b = 0, n = 0;
    if (i < nseq) {
      a = cu[i];
      b = cu[i + 1];
      n = seg_count(b - a, segc);
    }
    int incl = n;  // inclusive prefix sum of the segment counts over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, i < nseq && off + incl > j);
    if (hit) {
      const int src = __ffs(hit) - 1;
      s = base + src;
      k = j - off - __shfl_sync(0xffffffffu, incl - n, src);
      nseg_s = __shfl_sync(0xffffffffu, n, src);
      t0 = __shfl_sync(0xffffffffu, a, src);
      t1 = __shfl_sync(0xffffffffu, b, src);
      return true;
    }
    off += __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;
}

// The scheduling order of an unsplit scan grid: slot j (the j-th group of a sequence's
// CTAs in the grid) runs the j-th longest sequence by chunk count, ties in index order (the
// longest-processing-time-first rule).  The longest chain of chunks sets the scan's time
// when it starts late: in batch order, a long sequence packed after short ones starts only
// as they finish.  Batches of more than kLptMaxSeqs sequences fill many waves, where the
// order hardly moves the tail: they run in batch order.  Every warp of the CTA calls it and
// gets the sequence and its token range [t0, t1) in all lanes, from one load per lane and 32
// shuffles (no shared memory, no block barrier).  Malformed lengths rank as empty; the
// caller checks the range it gets.
constexpr int kLptMaxSeqs = 32;
__device__ inline void lpt_sequence_warp(const int32_t* cu, int nseq, int T, int j, int& s,
                                         int& t0, int& t1) {
  if (nseq <= 1 || nseq > kLptMaxSeqs) {
    s = j;
    t0 = cu[j];
    t1 = cu[j + 1];
    return;
  }
  const int lane = threadIdx.x & 31;
  int a = 0, b = 0, n = -1;  // past the batch: below every sequence
  if (lane < nseq) {
    a = cu[lane];
    b = cu[lane + 1];
    n = (0 <= a && a <= b && b <= T) ? (b - a + kScanChunk - 1) / kScanChunk : 0;
  }
  int rank = 0;  // sequences ahead of this lane's in the order
#pragma unroll
  for (int src = 0; src < 32; ++src) {
    const int o = __shfl_sync(0xffffffffu, n, src);
    rank += (o > n || (o == n && src < lane)) ? 1 : 0;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < nseq && rank == j);
  s = hit ? __ffs(hit) - 1 : j;  // ranks are a permutation of 0..nseq-1: always a hit
  t0 = __shfl_sync(0xffffffffu, a, s & 31);
  t1 = __shfl_sync(0xffffffffu, b, s & 31);
}

}  // namespace ssd
