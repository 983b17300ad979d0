// Ordered compaction of a per-token selection bitmap into a query head's list:
// S = set bits of `sel` inside the LSH region [lo, hi), ascending, followed by the
// exact tokens [0, lo) and [hi, n) with bit 31 set (sinks and window, u = 1;
// MagicPIG arXiv 2410.16179v2 Algorithm 1 and §4.4 "On-device cache").
#pragma once

#include "mp_internal.h"

namespace mp {

// Called by all 256 threads of a block. `sel` may live in shared or global memory;
// word i covers tokens 32i .. 32i+31. If !valid, S is empty.
__device__ __forceinline__ void write_list(const uint32_t* sel, bool valid, int lo, int hi, int n,
                                           uint32_t* lst, int32_t* sample_count, int32_t* list_len) {
  __shared__ int wsum[8];
  __shared__ int s_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwords = (hi + 31) >> 5;
  const int w0 = lo >> 5;
  const int nw = nwords - w0;
  const int per = (nw + blockDim.x - 1) / blockDim.x;
  const int my0 = w0 + threadIdx.x * per, my1 = min(nwords, my0 + per);
  auto word_at = [&](int wi) -> uint32_t {
    uint32_t v = sel[wi];
    const int base = wi << 5;
    if (base < lo) v &= ~((1u << (lo - base)) - 1u);  // lo - base in 1..31
    if (base + 32 > hi) v &= (1u << (hi - base)) - 1u; // hi - base in 1..31
    return v;
  };
  int local = 0;
  if (valid)
    for (int wi = my0; wi < my1; ++wi) local += __popc(word_at(wi));
  int x = local;
#pragma unroll
  for (int k = 1; k < 32; k <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, k);
    if (lane >= k) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int i = 0; i < 8; ++i) {
      const int v = wsum[i];
      wsum[i] = run;
      run += v;
    }
    s_total = run;
  }
  __syncthreads();
  int pos = wsum[warp] + x - local;
  if (valid) {
    for (int wi = my0; wi < my1; ++wi) {
      uint32_t v = word_at(wi);
      while (v) {
        const int b = __ffs(v) - 1;
        v &= v - 1;
        lst[pos++] = uint32_t((wi << 5) + b);
      }
    }
  }
  const int ns = s_total;
  const int nexact = lo + (n - hi);
  for (int i = threadIdx.x; i < nexact; i += blockDim.x) {
    const int tok = i < lo ? i : hi + (i - lo);
    lst[ns + i] = uint32_t(tok) | kExactFlag;
  }
  if (threadIdx.x == 0) {
    *sample_count = ns;
    *list_len = ns + nexact;
  }
}

}  // namespace mp
