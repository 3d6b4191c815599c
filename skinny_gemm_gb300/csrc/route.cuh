// route.cuh -- token gathering for the routed-expert (mm_id) kernels.
#pragma once

#include <cstdint>

#include "launch.h"

namespace w4a16 {

// Collect, in token order, up to `cap` (<= kMaxChunk) tokens t >= s_state[0]
// with ids[t] == e (or, when e < 0, with ids[t] outside 0..E-1) into s_tok.
// All threads of the CTA call it; warp 0 scans 32 ids per step with a
// ballot.  On return s_state[0] is the scan position for the next call and
// the return value is the number of tokens collected (0 = none left).
__device__ __forceinline__ int gather_tokens(const int32_t* __restrict__ ids, int T, int E, int e, int* s_tok,
                                             int* s_state, int cap = kMaxChunk) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    int pos = s_state[0];
    int cnt = 0;
    while (pos < T && cnt < cap) {
      const int t = pos + lane;
      bool match = false;
      if (t < T) {
        const int v = ids[t];
        match = (e >= 0) ? (v == e) : (v < 0 || v >= E);
      }
      const unsigned mask = __ballot_sync(0xffffffffu, match);
      const int rank = __popc(mask & ((1u << lane) - 1u));
      const int n = __popc(mask);
      const int need = cap - cnt;
      if (n <= need) {
        if (match) s_tok[cnt + rank] = t;
        cnt += n;
        pos += 32;
      } else {
        if (match && rank < need) s_tok[cnt + rank] = t;
        const unsigned last = __ballot_sync(0xffffffffu, match && rank == need - 1);
        pos += (__ffs(last) - 1) + 1;
        cnt = cap;
      }
    }
    if (lane == 0) {
      s_state[0] = pos < T ? pos : T;
      s_state[1] = cnt;
    }
  }
  __syncthreads();
  const int cnt = s_state[1];
  __syncthreads();  // everyone has read the count before it can change
  return cnt;
}

}  // namespace w4a16
