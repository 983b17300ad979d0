// Ordered compaction of a per-token selection bitmap into a query head's list:
// S = set bits of `sel` inside the LSH region [lo, hi), ascending, followed by the
// exact tokens [0, lo) and [hi, n) with bit 31 set (sinks and window, u = 1;
// MagicPIG arXiv 2410.16179v2 Algorithm 1 and §4.4 "On-device cache").
#pragma once

#include "mp_internal.h"

namespace mp {

// Called by all threads of a block (a multiple of 32, at most 256). `sel` may live in
// shared or global memory; word i covers tokens origin + 32i .. origin + 32i + 31
// (origin <= lo). If !valid, S is empty.
__device__ __forceinline__ void write_list(const uint32_t* sel, bool valid, int lo, int hi, int n,
                                           uint32_t* lst, int32_t* sample_count, int32_t* list_len,
                                           int origin = 0) {
  __shared__ int wsum[8];
  __shared__ int s_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rl = lo - origin, rh = hi - origin;  // the region in bit positions of sel
  const int nwords = (rh + 31) >> 5;
  const int w0 = rl >> 5;
  const int nw = nwords - w0;
  const int per = (nw + blockDim.x - 1) / blockDim.x;
  const int my0 = w0 + threadIdx.x * per, my1 = min(nwords, my0 + per);
  auto word_at = [&](int wi) -> uint32_t {
    uint32_t v = sel[wi];
    const int base = wi << 5;
    if (base < rl) v &= ~((1u << (rl - base)) - 1u);  // rl - base in 1..31
    if (base + 32 > rh) v &= (1u << (rh - base)) - 1u; // rh - base in 1..31
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
    for (int i = 0; i < int(blockDim.x >> 5); ++i) {
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
        lst[pos++] = uint32_t(origin + (wi << 5) + b);
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
