// Hash-table construction: for every (KV head, table) the prefill tokens
// [n_sink, n_prefill) bucketed by their K-bit code, one bucketed segment of up to
// 32768 tokens at a time (16-bit ids relative to the segment's first token, 16-bit
// bucket starts). These are the hash tables HT of MagicPIG (arXiv 2410.16179v2)
// Algorithm 1 and §4.4(4); the pages build them on the CPU per KV head, here one CTA
// sorts one segment of one table in shared memory and writes it out coalesced. The
// order of the ids inside a bucket is whatever the shared-memory atomics give: the
// tables are only ever read as sets.
#include "mp_internal.h"

namespace mp {

// 16 warps, three CTAs per SM (68 KB of shared memory each): while one CTA scans its
// counts or writes its ids out, the others keep the shared-memory atomics busy (32 warps,
// two per SM, measured 5.93 against 5.47 ms on the 32-layer build)
constexpr int kCsrThreads = 512;
static_assert(kCsrThreads % 32 == 0 && kCsrThreads <= 1024, "the per-warp sums fit one warp's scan");

// One CTA per (unit x table, segment). Pass 1: bucket counts with shared-memory atomics.
// Block scan of the counts gives the bucket starts (written out as the offsets). Pass 2:
// every token takes a slot of its bucket with a shared-memory atomic on the bucket's
// cursor. The codes are read as 16-byte chunks of 8 (from the 16-byte boundary at or
// below the segment's first code: the codes region is padded to 256 bytes, so the
// chunks never leave it), and the ids leave shared memory as 16-byte chunks too, so
// that the memory instruction queue carries the atomics and few loads and stores.
__device__ __forceinline__ uint32_t code_of(const uint4& v, int e) {
  const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
  return (w >> (16 * (e & 1))) & 0xffffu;
}

__global__ void __launch_bounds__(kCsrThreads, 3) k_csr_build(const uint16_t* __restrict__ codes,
                                                           uint16_t* __restrict__ off, uint16_t* __restrict__ ids,
                                                           int cap, int nb, int nseg, int lo, int hi,
                                                           uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smraw[];
  const int64_t table = blockIdx.x;  // unit * L + t
  const int s = blockIdx.y;
  const int a = lo + s * kCsrSeg;
  const int m = min(hi, a + kCsrSeg) - a;  // tokens of this segment (>= 1)
  uint32_t* cursor = reinterpret_cast<uint32_t*>(smraw);  // [nb]
  // segment ids in bucket order; id j sits at element j + r, r = the misalignment of the
  // destination, so that 16-byte chunks of this buffer are 16-byte chunks of the output
  uint16_t* sorted = reinterpret_cast<uint16_t*>(smraw + ((size_t(nb) * 4 + 15) & ~size_t(15)));
  __shared__ uint32_t wsum[kCsrThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uintptr_t ca = reinterpret_cast<uintptr_t>(codes + table * cap + a);
  const int skip = int(ca & 15u) >> 1;  // codes of the first chunk before the segment
  const uint4* cv = reinterpret_cast<const uint4*>(ca & ~uintptr_t(15));
  const int nch = (skip + m + 7) >> 3;
  uint16_t* dst = ids + table * cap + int64_t(s) * kCsrSeg;
  const int r = int(reinterpret_cast<uintptr_t>(dst) & 15u) >> 1;

  for (int i = tid; i < nb; i += kCsrThreads) cursor[i] = 0u;
  __syncthreads();
  // pass 1 reads the codes from HBM; pass 2 reads them again, from L2
#pragma unroll 2
  for (int ch = tid; ch < nch; ch += kCsrThreads) {
    const uint4 v = __ldg(cv + ch);
    const int i0 = ch * 8 - skip;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (unsigned(i0 + e) < unsigned(m) && in_range(code_of(v, e) < uint32_t(nb), status))
        atomicAdd(&cursor[code_of(v, e)], 1u);
  }
  __syncthreads();

  // exclusive scan of the counts: thread i owns buckets [i*per, (i+1)*per)
  const int per = (nb + kCsrThreads - 1) / kCsrThreads;
  const int b0 = min(nb, tid * per), b1 = min(nb, b0 + per);
  uint32_t local = 0;
  for (int b = b0; b < b1; ++b) local += cursor[b];
  uint32_t x = local;
#pragma unroll
  for (int k = 1; k < 32; k <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, k);
    if (lane >= k) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    // one lane per warp of the block (lanes past the last warp carry zeros)
    uint32_t v = lane < kCsrThreads / 32 ? wsum[lane] : 0u;
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, v, k);
      if (lane >= k) v += y;
    }
    if (lane < kCsrThreads / 32) wsum[lane] = v;
  }
  __syncthreads();
  // offsets of the table, bucket-major with the segments innermost: the starts of one
  // bucket in all segments (and those of the next bucket) share a cache line
  uint16_t* o = off + table * int64_t(nb + 1) * nseg + s;
  uint32_t base = x - local + (warp > 0 ? wsum[warp - 1] : 0u);
  for (int b = b0; b < b1; ++b) {
    const uint32_t cnt = cursor[b];
    cursor[b] = base + uint32_t(r);
    o[int64_t(b) * nseg] = uint16_t(base);
    base += cnt;
  }
  if (tid == 0) o[int64_t(nb) * nseg] = uint16_t(m);
  __syncthreads();

  // pass 2: placement (the cursors start at bucket start + r)
#pragma unroll 2
  for (int ch = tid; ch < nch; ch += kCsrThreads) {
    const uint4 v = __ldcs(cv + ch);
    const int i0 = ch * 8 - skip;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (unsigned(i0 + e) < unsigned(m) && in_range(code_of(v, e) < uint32_t(nb), status))
        sorted[atomicAdd(&cursor[code_of(v, e)], 1u)] = uint16_t(i0 + e);
  }
  __syncthreads();
  // out: whole 16-byte chunks inside the segment as one store, the ragged ends by element
  const int nout = (r + m + 7) >> 3;
  uint4* dv = reinterpret_cast<uint4*>(dst - r);
  const uint4* sv = reinterpret_cast<const uint4*>(sorted);
  for (int k = tid; k < nout; k += kCsrThreads) {
    const int j0 = 8 * k - r;
    if (j0 >= 0 && j0 + 8 <= m) {
      dv[k] = sv[k];
    } else {
      for (int e = 0; e < 8; ++e)
        if (unsigned(j0 + e) < unsigned(m)) dst[j0 + e] = sorted[8 * k + e];
    }
  }
}

cudaError_t launch_csr_build(const Geometry& g, int n_prefill, const TablesPtrs& t, cudaStream_t st) {
  const int lo = min(g.s, n_prefill), hi = n_prefill;
  if (hi <= lo) return cudaSuccess;
  const int segs = (hi - lo + kCsrSeg - 1) / kCsrSeg;
  const size_t smem = ((size_t(g.nb) * 4 + 15) & ~size_t(15)) + size_t(kCsrSeg + 16) * 2;
  cudaFuncSetAttribute(k_csr_build, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  dim3 grid(g.units * g.L, segs);
  k_csr_build<<<grid, kCsrThreads, smem, st>>>(t.codes, t.off, t.ids, g.cap, g.nb, g.nseg, lo, hi, &t.hdr->status);
  return cudaGetLastError();
}

}  // namespace mp
