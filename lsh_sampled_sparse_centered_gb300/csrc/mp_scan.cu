// Scan match mode: the codes of every token kept as bit-planes (for each KV head,
// table t and bit b, one bit per token), streamed once per decode step for all the
// query heads of a KV head. A token is sampled when its code equals the query's in
// at least `threshold` tables (MagicPIG arXiv 2410.16179v2 §4.3 "Hash function
// selection"); the per-table equality of a 32-token word is the AND over the K planes
// of (plane XNOR query bit), and the count ">= 1" / ">= 2" is kept with two
// bit-sliced words (ones, twos).
#include "mp_compact.cuh"
#include "mp_internal.h"

namespace mp {

// planes[(ut*K + b)*cw + w] for tokens [0, n_prefill) from the code store; one warp per
// 32-token word: __ballot_sync of bit b over the 32 codes is plane word b.
__global__ void __launch_bounds__(256) k_planes_build(const uint16_t* __restrict__ codes, uint32_t* __restrict__ planes,
                                                      int K, int cap, int cw, int n0) {
  const int64_t ut = blockIdx.y;
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= cw) return;
  const int tok = w * 32 + lane;
  const uint32_t code = tok < n0 ? codes[ut * cap + tok] : 0u;
  for (int b = 0; b < K; ++b) {
    const uint32_t word = __ballot_sync(0xffffffffu, (code >> b) & 1u);
    if (lane == b) planes[(ut * K + b) * cw + w] = word;
  }
}

cudaError_t launch_planes_build(const Geometry& g, int n_prefill, const TablesPtrs& t, cudaStream_t st) {
  if (g.K == 0) return cudaSuccess;
  dim3 grid((g.cw + 7) / 8, g.units * g.L);
  k_planes_build<<<grid, 256, 0, st>>>(t.codes, t.planes, g.K, g.cap, g.cw, n_prefill);
  return cudaGetLastError();
}

// After an append: copy the new token's code bits into the planes (one thread per
// (unit, table); each plane word touched by exactly one thread).
__global__ void k_planes_append(const uint16_t* __restrict__ codes, uint32_t* __restrict__ planes, int units_L,
                                int K, int cap, int cw, int pos) {
  const int64_t ut = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (ut >= units_L) return;
  const uint32_t code = codes[ut * cap + pos];
  const uint32_t bit = 1u << (pos & 31);
  for (int b = 0; b < K; ++b) {
    uint32_t* p = planes + (ut * K + b) * cw + (pos >> 5);
    *p = ((code >> b) & 1u) ? (*p | bit) : (*p & ~bit);
  }
}

cudaError_t launch_planes_append(const Geometry& g, int pos, const TablesPtrs& t, cudaStream_t st) {
  if (g.K == 0) return cudaSuccess;
  const int n = g.units * g.L;
  k_planes_append<<<(n + 255) / 256, 256, 0, st>>>(t.codes, t.planes, n, g.K, g.cap, g.cw, pos);
  return cudaGetLastError();
}

// Stream the planes of one KV head over 4 words (128 tokens) per thread for up to 8
// query heads at a time; write each head's selection bitmap. Threshold <= 2 keeps
// the bit-sliced (ones, twos) pair; larger thresholds keep a 3-bit bit-sliced counter
// per token and a sticky "reached" word (the count rises by at most 1 per table, so it
// passes through the threshold exactly once).
constexpr int kScanThreads = 128;

template <bool kGeneral>
__global__ void __launch_bounds__(kScanThreads) k_scan(const uint32_t* __restrict__ planes,
                                                       const uint16_t* __restrict__ qcodes,
                                                       uint32_t* __restrict__ sbits, int L, int K, int cw,
                                                       int nwords, int group, int threshold) {
  constexpr int H = kGeneral ? 4 : 8;  // query heads per pass
  extern __shared__ uint16_t qc[];     // [group][L]
  const int unit = blockIdx.y;
  for (int i = threadIdx.x; i < group * L; i += blockDim.x) qc[i] = qcodes[int64_t(unit) * group * L + i];
  __syncthreads();
  const int w4 = (blockIdx.x * kScanThreads + threadIdx.x) * 4;
  if (w4 >= nwords) return;
  const uint32_t* pu = planes + int64_t(unit) * L * K * cw + w4;
  const uint32_t t0m = (threshold & 1) ? 0xffffffffu : 0u;
  const uint32_t t1m = (threshold & 2) ? 0xffffffffu : 0u;
  const uint32_t t2m = (threshold & 4) ? 0xffffffffu : 0u;
  for (int g0 = 0; g0 < group; g0 += H) {
    const int ng = min(H, group - g0);
    // kGeneral: a = bit 0, b = bit 1, c = bit 2 of the count, r = reached; else a = ones, b = twos
    uint32_t a[H][4], b[H][4], c[H][4], r[H][4];
#pragma unroll
    for (int g = 0; g < H; ++g)
#pragma unroll
      for (int i = 0; i < 4; ++i) a[g][i] = b[g][i] = c[g][i] = r[g][i] = 0u;
    for (int t = 0; t < L; ++t) {
      uint32_t eq[H][4];
      uint32_t code[H];
#pragma unroll
      for (int g = 0; g < H; ++g) {
        code[g] = g < ng ? qc[(g0 + g) * L + t] : 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) eq[g][i] = 0xffffffffu;
      }
      const uint32_t* pt = pu + int64_t(t) * K * cw;
      for (int bb = 0; bb < K; ++bb) {
        const uint4 p = *reinterpret_cast<const uint4*>(pt + int64_t(bb) * cw);
#pragma unroll
        for (int g = 0; g < H; ++g) {
          // (qbit ? plane : ~plane) = plane ^ (qbit - 1)
          const uint32_t m = ((code[g] >> bb) & 1u) - 1u;
          eq[g][0] &= p.x ^ m;
          eq[g][1] &= p.y ^ m;
          eq[g][2] &= p.z ^ m;
          eq[g][3] &= p.w ^ m;
        }
      }
#pragma unroll
      for (int g = 0; g < H; ++g)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t e = eq[g][i];
          if (kGeneral) {
            const uint32_t c0 = a[g][i] & e;  // carry into bit 1
            a[g][i] ^= e;
            const uint32_t c1 = b[g][i] & c0;  // carry into bit 2
            b[g][i] ^= c0;
            c[g][i] ^= c1;
            r[g][i] |= ~(a[g][i] ^ t0m) & ~(b[g][i] ^ t1m) & ~(c[g][i] ^ t2m);
          } else {
            b[g][i] |= a[g][i] & e;
            a[g][i] |= e;
          }
        }
    }
    for (int g = 0; g < ng; ++g) {
      const int qh = unit * group + g0 + g;
      const uint32_t* sel = kGeneral ? r[g] : (threshold >= 2 ? b[g] : a[g]);
      uint4 v;
      v.x = sel[0];
      v.y = sel[1];
      v.z = sel[2];
      v.w = sel[3];
      *reinterpret_cast<uint4*>(sbits + int64_t(qh) * cw + w4) = v;
    }
  }
}

cudaError_t launch_scan(const Geometry& g, int n, const TablesPtrs& t, const DecodePtrs& dp, cudaStream_t st) {
  const int lo = min(g.s, n);
  const int hi = max(lo, n - g.w);
  const int nwords = (hi + 31) >> 5;
  if (nwords == 0) return cudaSuccess;
  dim3 grid((nwords + 4 * kScanThreads - 1) / (4 * kScanThreads), g.units);
  const size_t smem = size_t(g.group) * g.L * sizeof(uint16_t);
  if (g.threshold >= 3) {
    cudaFuncSetAttribute(k_scan<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    k_scan<true><<<grid, kScanThreads, smem, st>>>(t.planes, dp.qcodes, dp.sbits, g.L, g.K, g.cw, nwords,
                                                   g.group, g.threshold);
  } else {
    cudaFuncSetAttribute(k_scan<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    k_scan<false><<<grid, kScanThreads, smem, st>>>(t.planes, dp.qcodes, dp.sbits, g.L, g.K, g.cw, nwords,
                                                    g.group, g.threshold);
  }
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) k_compact(DevHeader* hdr, const uint32_t* __restrict__ sbits,
                                                 uint32_t* __restrict__ lists, int32_t* __restrict__ list_len,
                                                 int32_t* __restrict__ sample_count, uint32_t* __restrict__ counters,
                                                 int n, int s, int w, int cap, int cw) {
  const int qh = blockIdx.x;
  const int lo = min(s, n);
  const int hi = max(lo, n - w);
  const bool built = hdr->magic == kMagic;
  if (threadIdx.x == 0) {
    counters[qh] = 0u;
    if (qh == 0) counters[gridDim.x] = 0u;  // the attention's work queue
    if (!built) atomicOr(&hdr->status, MP_STATUS_NOT_BUILT);
    else if (hi > hdr->appended_end) atomicOr(&hdr->status, MP_STATUS_APPEND_GAP);
  }
  write_list(sbits + int64_t(qh) * cw, built && hi > lo, lo, hi, n, lists + int64_t(qh) * cap, &sample_count[qh],
             &list_len[qh]);
}

cudaError_t launch_compact(const Geometry& g, int n, const TablesPtrs& t, const DecodePtrs& dp, cudaStream_t st) {
  k_compact<<<g.queries, 256, 0, st>>>(t.hdr, dp.sbits, dp.lists, dp.list_len, dp.sample_count, dp.counters, n,
                                       g.s, g.w, g.cap, g.cw);
  return cudaGetLastError();
}

}  // namespace mp
