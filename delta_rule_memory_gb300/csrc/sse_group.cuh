// sse_group.cuh - the per-(batch, head) table that groups the SSE visits by
// partition (SSE deck, "Varlen groups tokens while preserving causal order"):
// written by the group kernel (sse_chunk.cu), read by the chunked prefills of
// the additive write (sse_chunk.cu) and of the delta write (gdn_chunk.cu).
//
// Every partition's visits form one time-ordered subsequence; a unit is one
// chunk of 64 visits of one partition.  The shared partition visits every
// token, so it owns units [0, ceil(T/64)); routed partition p owns units
// [first[p], first[p+1]).
#pragma once

#include <stdint.h>

namespace sdm {
namespace ssegrp {

constexpr int kVisits = 64;  // visits per unit
constexpr int kMaxTopk = 8;
constexpr int kMaxN = 64;

// ---- group table of one (batch, head), in 32-bit words
constexpr int kGFirst = 0;   // first unit of routed partition p (p = 0..N-1); [N] = units in total
constexpr int kGCnt = 72;    // visits of routed partition p
constexpr int kGOff = 136;   // offset of p's visit list among the entries
constexpr int kGHdr = 200;   // then the entries: (token << 4) | rank, partition by partition, time order

__host__ __device__ inline int units_max(int T, int N, int topk) {
  // shared: ceil(T/C); routed: sum_p ceil(n_p/C) <= floor((topk*T + (C-1)*N)/C)
  return (T + kVisits - 1) / kVisits +
         static_cast<int>((static_cast<long>(topk) * T + static_cast<long>(kVisits - 1) * N) / kVisits);
}
__host__ __device__ inline long group_words(int T, int topk) {
  return kGHdr + ((static_cast<long>(topk) * T + 3) & ~3L);
}

// words of one routing record: topk partitions, topk gates (fp32 bits), the
// key-softmax max and inverse normaliser, padded to a multiple of 4
__host__ __device__ inline int rec_words(int topk) { return (2 * topk + 2 + 3) & ~3; }

}  // namespace ssegrp
}  // namespace sdm
