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

// Segment j of the batch: its sequence s, its index k within s and the segment count of
// s; false when j lies past the last segment.  Malformed lengths count as empty (the
// kernels report them separately).
__device__ inline bool find_segment(const int32_t* cu, int nseq, int segc, int j, int& s,
                                    int& k, int& nseg_s) {
  int off = 0;
  for (int i = 0; i < nseq; ++i) {
    const int n = seg_count(cu[i + 1] - cu[i], segc);
    if (j < off + n) {
      s = i;
      k = j - off;
      nseg_s = n;
      return true;
    }
    off += n;
  }
  return false;
}

}  // namespace ssd
