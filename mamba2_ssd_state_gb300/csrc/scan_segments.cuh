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

}  // namespace ssd
