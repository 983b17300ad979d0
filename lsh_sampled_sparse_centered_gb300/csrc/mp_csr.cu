// Hash-table construction: for every (KV head, table) a bucketed id list (CSR)
// of the prefill tokens [n_sink, n_prefill), keyed by their K-bit code. Within a
// bucket ids are ascending (stable counting sort).
// The hash tables HT of MagicPIG (arXiv 2410.16179v2) Algorithm 1 and §4.4(4);
// the pages build them on the CPU per KV head, here one CTA builds one table.
#include "mp_internal.h"

namespace mp {

// One CTA per (unit, table). The token range is cut into `nseg` contiguous segments,
// one per warp. Pass 1: per-warp bucket histograms in shared memory. Then per bucket
// the segment prefix and the bucket starts (exclusive scan). Pass 2: each warp walks
// its segment in order and scatters ids; __match_any_sync ranks equal codes inside a
// 32-token step, so the order of ids within a bucket is the token order.
__global__ void __launch_bounds__(512) k_csr_build(const uint16_t* __restrict__ codes,
                                                   uint32_t* __restrict__ off, uint32_t* __restrict__ ids,
                                                   int L, int cap, int nb, int lo, int hi) {
  extern __shared__ uint32_t sm[];
  const int nseg = blockDim.x >> 5;
  uint32_t* hist = sm;                 // [nseg][nb]
  uint32_t* scan = sm + nseg * nb;     // [blockDim.x] per-thread partial sums
  const int64_t table = blockIdx.x;    // unit * L + t
  const uint16_t* c = codes + table * cap;
  uint32_t* o = off + table * (nb + 1);
  uint32_t* id = ids + table * cap;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = hi - lo;
  const int span = (n + nseg - 1) / nseg;
  const int s0 = lo + warp * span, s1 = min(hi, s0 + span);

  for (int i = threadIdx.x; i < nseg * nb; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  uint32_t* h = hist + warp * nb;
  for (int tok = s0 + lane; tok < s1; tok += 32) atomicAdd(&h[c[tok]], 1u);
  __syncthreads();

  // per bucket: exclusive prefix over the segments; each thread owns `per`
  // consecutive buckets and keeps their totals in `scan` for the block scan below
  const int per = (nb + blockDim.x - 1) / blockDim.x;
  const int b0 = threadIdx.x * per, b1 = min(nb, b0 + per);
  uint32_t local = 0;
  for (int b = b0; b < b1; ++b) {
    uint32_t run = 0;
    for (int s = 0; s < nseg; ++s) {
      const uint32_t v = hist[s * nb + b];
      hist[s * nb + b] = run;
      run += v;
    }
    local += run;
    scan[b] = run;  // bucket total
  }
  __syncthreads();
  // block exclusive scan of `local` (per-thread totals)
  __shared__ uint32_t wsum[32];
  uint32_t x = local;
#pragma unroll
  for (int k = 1; k < 32; k <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, k);
    if (lane >= k) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t v = lane < nseg ? wsum[lane] : 0;
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, v, k);
      if (lane >= k) v += y;
    }
    if (lane < nseg) wsum[lane] = v;
  }
  __syncthreads();
  uint32_t base = x - local + (warp > 0 ? wsum[warp - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    const uint32_t total = scan[b];
    o[b] = base;
    for (int s = 0; s < nseg; ++s) hist[s * nb + b] += base;
    base += total;
  }
  if (threadIdx.x == 0) o[nb] = uint32_t(n);
  __syncthreads();

  // pass 2: stable scatter
  for (int t0 = s0; t0 < s1; t0 += 32) {
    const int tok = t0 + lane;
    const bool act = tok < s1;
    const unsigned mask = __ballot_sync(0xffffffffu, act);
    if (act) {
      const uint32_t code = c[tok];
      const unsigned peers = __match_any_sync(mask, code);
      const int leader = __ffs(peers) - 1;
      const int rank = __popc(peers & ((1u << lane) - 1u));
      uint32_t pos = 0;
      if (lane == leader) {
        pos = h[code];
        h[code] = pos + __popc(peers);
      }
      pos = __shfl_sync(peers, pos, leader);
      id[pos + rank] = uint32_t(tok);
    }
    __syncwarp();
  }
}

cudaError_t launch_csr_build(const Geometry& g, int n_prefill, const TablesPtrs& t, cudaStream_t st) {
  const int lo = min(g.s, n_prefill), hi = n_prefill;
  // segments (warps): as many as fit 200 KB of histograms, at most 16
  // `scan` holds one slot per bucket, rounded up to whole per-thread chunks
  auto smem_for = [&](int ns) {
    const int th = 32 * ns;
    const int per = (g.nb + th - 1) / th;
    return (size_t(ns) * g.nb + size_t(per) * th) * sizeof(uint32_t);
  };
  int nseg = 16;
  while (nseg > 1 && smem_for(nseg) > 200 * 1024) --nseg;
  const int threads = 32 * nseg;
  const size_t smem = smem_for(nseg);
  cudaFuncSetAttribute(k_csr_build, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  k_csr_build<<<int64_t(g.units) * g.L, threads, smem, st>>>(t.codes, t.off, t.ids, g.L, g.cap, g.nb, lo, hi);
  return cudaGetLastError();
}

}  // namespace mp
