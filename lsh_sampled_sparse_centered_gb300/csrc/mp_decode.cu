// Decode step: sampled-set construction from the bucketed tables, then the
// importance-weighted attention over the sampled keys plus the exact sink/window
// tokens, split across CTAs with a fused log-sum-exp combine.
// (A shared-memory-staged variant with one bulk asynchronous copy per K/V row was
// measured 1.4x slower than the register gathers below on the 96K workload and removed.)
// MagicPIG (arXiv 2410.16179v2): Algorithm 1, Eq. 9-11, §4.4 "On-device cache".
#include <math_constants.h>

#include <algorithm>
#include <atomic>

#include "mp_compact.cuh"
#include "mp_internal.h"

namespace mp {

// ---------------------------------------------------------------------------------
// sampled set: one CTA per query head
// ---------------------------------------------------------------------------------
// Bitmaps over the tokens [lo, n), bit j <-> token lo + j (lo = n_sink when the region is
// not empty): `seen1` marks tokens met in >= 1 table's bucket, `seen2` in >= 2. With
// threshold 2 the sampled set is seen2 restricted to [lo, n - window); with threshold 1
// it is seen1. Compaction writes S in ascending token order, then the exact tokens (bit
// 31 set). The bitmaps reach n rather than n - window so that a bucketed token (always
// < n_prefill <= n in a decode that covers the prefill) needs no range test; the window
// bits are masked off by the compaction.
constexpr int kMatchWarps = 8;
constexpr int kChunkUnroll = 2;  // 16-byte chunks of ids in flight per thread

// Exclusive scan of v[0..n) in place by the whole block; v[n] receives the total.
__device__ __forceinline__ void block_exclusive_scan(uint32_t* v, int n) {
  __shared__ uint32_t wsum[kMatchWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int i0 = min(n, int(threadIdx.x) * per), i1 = min(n, i0 + per);
  uint32_t local = 0;
  for (int i = i0; i < i1; ++i) local += v[i];
  uint32_t x = local;
#pragma unroll
  for (int k = 1; k < 32; k <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, k);
    if (lane >= k) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  uint32_t before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kMatchWarps; ++w) {
    before += (w < warp) ? wsum[w] : 0u;
    total += wsum[w];
  }
  uint32_t run = before + x - local;
  for (int i = i0; i < i1; ++i) {
    const uint32_t c = v[i];
    v[i] = run;
    run += c;
  }
  if (threadIdx.x == 0) v[n] = total;
  __syncthreads();
}

// One thread's share [cb, ce) of a head's id chunks, kChunkUnroll chunks at a time (all
// loads issued before the first mark). Run r = (table, segment) holds the ids of the
// query's bucket in that segment; id i of segment sg is token lo + 32768 sg + i, i.e. bit
// 32768 sg + i of the bitmaps. BYTES: one byte counter per token instead of the two
// bitmaps (thresholds >= 3). CLIP: drop tokens at or beyond rh (a decode over fewer
// tokens than the prefill). The bounds-checking build also tests every bit position
// against the nbits bits of the bitmaps.
template <bool BYTES, bool CLIP>
__device__ __forceinline__ void walk_chunks(const uint4* __restrict__ cbase, const uint2* bkt, const uint32_t* pre,
                                            int r, uint32_t cb, uint32_t ce, uint32_t rh, uint32_t nbits,
                                            uint32_t* seen1, uint32_t* seen2, uint32_t* cnt, uint32_t* status) {
  const uint32_t s1 = uint32_t(__cvta_generic_to_shared(seen1));
  const uint32_t s2off = uint32_t(__cvta_generic_to_shared(seen2)) - s1;
  for (uint32_t c = cb; c < ce; c += kChunkUnroll) {
    uint4 v[kChunkUnroll];
    uint32_t vm[kChunkUnroll], sgb[kChunkUnroll];  // vm: bit q <-> slot q is an id of the run
#pragma unroll
    for (int u = 0; u < kChunkUnroll; ++u) {
      const uint32_t cc = c + u;
      vm[u] = 0u;
      sgb[u] = 0u;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (cc < ce) {
        while (cc >= pre[r + 1]) ++r;
        const uint2 e = bkt[r];
        const uint32_t k = cc - pre[r];  // chunk index within the run
        const int32_t first = int32_t((e.y >> 16) & 7u) - int32_t(8u * k);  // ids before the run
        const int32_t end = first + int32_t(e.y & 0xffffu);
        const uint32_t f = uint32_t(max(first, 0)), l = uint32_t(min(end, 8));
        vm[u] = (0xffu >> (8u - l)) & (0xffu << f);
        sgb[u] = ((e.y >> 19) & 15u) * uint32_t(kCsrSeg);
        v[u] = __ldg(cbase + e.x + k);
      }
    }
#pragma unroll
    for (int u = 0; u < kChunkUnroll; ++u)
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint32_t word = (q < 2) ? v[u].x : (q < 4) ? v[u].y : (q < 6) ? v[u].z : v[u].w;
        const uint32_t id = (q & 1) ? (word >> 16) : (word & 0xffffu);
        const uint32_t j = sgb[u] + id;  // bit position
        uint32_t okm = vm[u] & (1u << q);
        if (CLIP) okm = (j < rh) ? okm : 0u;
#if MP_CHECK
        if (okm && !in_range(j < nbits, status)) okm = 0u;
#else
        (void)nbits;
        (void)status;
#endif
        if (BYTES) {
          if (okm) atomicAdd(&cnt[j >> 2], 1u << (8 * (id & 3u)));
        } else {
          // seen1 |= bit; when it was set already, seen2 |= bit (both predicated, no branch)
          const uint32_t bit = __funnelshift_l(0u, 1u, id);
          const uint32_t a = s1 + ((j >> 5) << 2);
          asm volatile(
              "{\n\t.reg .pred p, q;\n\t.reg .b32 o;\n\t"
              "setp.ne.b32 p, %2, 0;\n\t"
              "mov.b32 o, 0;\n\t"
              "@p atom.shared.or.b32 o, [%0], %1;\n\t"
              "and.b32 o, o, %1;\n\t"
              "setp.ne.b32 q, o, 0;\n\t"
              "@q red.shared.or.b32 [%3], %1;\n\t}" ::"r"(a),
              "r"(bit), "r"(okm), "r"(a + s2off)
              : "memory");
        }
      }
  }
}

__global__ void __launch_bounds__(kMatchWarps * 32, 5) k_match_csr(DevHeader* hdr,
                                                   const uint16_t* __restrict__ qcodes,
                                                   const uint16_t* __restrict__ codes,
                                                   const uint16_t* __restrict__ off,
                                                   const uint16_t* __restrict__ ids, uint32_t* __restrict__ lists,
                                                   int32_t* __restrict__ list_len, int32_t* __restrict__ sample_count,
                                                   uint32_t* __restrict__ counters, int n, int s, int w, int L,
                                                   int nb, int cap, int nseg, int group, int threshold) {
  extern __shared__ __align__(16) uint32_t sm[];
  const int qh = blockIdx.x;
  const int unit = qh / group;  // [layer][batch][q_head] -> [layer][batch][kv_head]
  const int lo = min(s, n);
  const int hi = max(lo, n - w);
  const int nwords = (n - lo + 31) >> 5;  // bitmap words over [lo, n)
  // threshold <= 2: two bitmaps (met in >= 1 table, in >= 2 tables);
  // threshold >= 3: one byte counter per token (L <= 255), then a selection bitmap
  const bool bytes = threshold >= 3;
  uint32_t* seen1 = sm;
  uint32_t* seen2 = sm + nwords;
  uint32_t* cnt = sm + nwords;  // [nwords * 8] byte counters (threshold >= 3)
  const int body = bytes ? nwords * 9 : nwords * 2;
  uint2* bkt = reinterpret_cast<uint2*>(sm + ((body + 1) & ~1));  // [L * nseg] runs of ids
  uint32_t* pre = reinterpret_cast<uint32_t*>(bkt + L * nseg);     // [L * nseg + 1] chunk prefix
  uint16_t* qc = reinterpret_cast<uint16_t*>(pre + L * nseg + 1);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const bool built = hdr->magic == kMagic;
  const int n0 = hdr->n_prefill;
  const int app_end = hdr->appended_end;
  if (threadIdx.x == 0) {
    counters[qh] = 0u;
    if (qh == 0) counters[gridDim.x] = 0u;  // the attention's work queue
    if (!built) atomicOr(&hdr->status, MP_STATUS_NOT_BUILT);
    else if (hi > app_end) atomicOr(&hdr->status, MP_STATUS_APPEND_GAP);
  }
  for (int i = threadIdx.x; i < (body >> 2); i += blockDim.x) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = (body & ~3) + threadIdx.x; i < body; i += blockDim.x) sm[i] = 0u;
  for (int t = threadIdx.x; t < L; t += blockDim.x) qc[t] = qcodes[int64_t(qh) * L + t];
  __syncthreads();

  if (built && hi > lo) {
    // Tokens hashed at build time: the query's bucket in every (table, segment), one run
    // of ids each. Every run is covered by the 16-byte chunks that hold it; the chunks of
    // all runs of the head are numbered consecutively (a block scan of the per-run chunk
    // counts) and split evenly over the threads, so each thread has about the same number
    // of chunks and marks every id of its chunks itself.
    const int64_t tbase = int64_t(unit) * L;
    const int lo_b = min(s, n0);  // first token bucketed at build time (= lo here)
    const int nsu = n0 > lo_b ? (n0 - lo_b + kCsrSeg - 1) / kCsrSeg : 0;
    const int runs = L * nsu;
    const uintptr_t idb = reinterpret_cast<uintptr_t>(ids + tbase * cap);  // the unit's id arrays
    const uintptr_t idb16 = idb & ~uintptr_t(15);
    // run r = t * nsu + sg: {first chunk (16-byte units from idb16), size | skip << 16 | sg << 19},
    // skip = ids of the first chunk before the run; pre[r] = chunks of runs before r
    for (int t = threadIdx.x; t < L; t += blockDim.x) {
      const bool code_ok = in_range(qc[t] < uint32_t(nb), &hdr->status);
      const uint16_t* o = off + (tbase + t) * int64_t(nb + 1) * nseg + int64_t(code_ok ? qc[t] : 0) * nseg;
      for (int sg = 0; sg < nsu; ++sg) {
        const uint32_t b0 = __ldg(o + sg), b1 = __ldg(o + nseg + sg);
        // a run lies inside its segment (whose tokens number min(32768, n0 - lo_b - 32768 sg))
        const bool run_ok = code_ok && in_range(b0 <= b1 && int(b1) <= min(kCsrSeg, n0 - lo_b - sg * kCsrSeg),
                                                &hdr->status);
        const uint32_t sz = run_ok ? b1 - b0 : 0u;
        const uintptr_t a = idb + 2u * (uint64_t(t) * uint64_t(cap) + uint64_t(sg) * kCsrSeg + b0);
        const uint32_t c0 = uint32_t((a - idb16) >> 4);
        bkt[t * nsu + sg] = make_uint2(c0, sz | (uint32_t((a & 15u) >> 1) << 16) | (uint32_t(sg) << 19));
        pre[t * nsu + sg] = sz ? uint32_t(((a + 2u * sz - 1u) >> 4) - (a >> 4) + 1u) : 0u;
      }
    }
    __syncthreads();
    block_exclusive_scan(pre, runs);  // pre[runs] = total chunks
    const uint32_t total = pre[runs];
    const uint32_t cb = uint32_t((uint64_t(total) * threadIdx.x) / blockDim.x);
    const uint32_t ce = uint32_t((uint64_t(total) * (threadIdx.x + 1)) / blockDim.x);
    if (cb < ce) {
      // the last run r with pre[r] <= cb (then pre[r + 1] > cb)
      int r = 0, rh = runs;
      while (rh - r > 1) {
        const int mid = (r + rh) >> 1;
        if (pre[mid] <= cb) r = mid;
        else rh = mid;
      }
      const uint4* cbase = reinterpret_cast<const uint4*>(idb16);
      // bucketed tokens lie below n0; with n0 <= n they all have a bit (lo_b = lo)
      const uint32_t rel_hi = uint32_t(hi - lo), nbits = uint32_t(nwords) * 32u;
      uint32_t* st = &hdr->status;
      if (n0 <= n) {
        if (bytes) walk_chunks<true, false>(cbase, bkt, pre, r, cb, ce, rel_hi, nbits, seen1, seen2, cnt, st);
        else walk_chunks<false, false>(cbase, bkt, pre, r, cb, ce, rel_hi, nbits, seen1, seen2, cnt, st);
      } else {
        if (bytes) walk_chunks<true, true>(cbase, bkt, pre, r, cb, ce, rel_hi, nbits, seen1, seen2, cnt, st);
        else walk_chunks<false, true>(cbase, bkt, pre, r, cb, ce, rel_hi, nbits, seen1, seen2, cnt, st);
      }
    }
    // tokens appended after the build that have left the window: compare codes
    const int a0 = max(lo, n0), a1 = min(hi, app_end);
    for (int tok = a0 + warp; tok < a1; tok += kMatchWarps) {
      int c = 0;
      for (int t = lane; t < L; t += 32) c += (codes[(tbase + t) * cap + tok] == qc[t]) ? 1 : 0;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) c += __shfl_xor_sync(0xffffffffu, c, k);
      if (lane == 0) {
        const int j = tok - lo;
        if (bytes) {
          atomicAdd(&cnt[j >> 2], uint32_t(min(c, 255)) << (8 * (j & 3)));
        } else {
          const uint32_t bit = 1u << (j & 31);
          if (c >= 1) atomicOr(&seen1[j >> 5], bit);
          if (c >= 2) atomicOr(&seen2[j >> 5], bit);
        }
      }
    }
  }
  __syncthreads();
  if (bytes) {
    // selection bitmap: counter >= threshold (reuses the first words)
    const int sw = (hi - lo + 31) >> 5;
    for (int wi = threadIdx.x; wi < sw; wi += blockDim.x) {
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t c4 = cnt[wi * 8 + j];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (((c4 >> (8 * k)) & 0xFFu) >= uint32_t(threshold)) m |= 1u << (4 * j + k);
      }
      seen1[wi] = m;
    }
    __syncthreads();
  }
  // compaction of [lo, hi)
  write_list(threshold == 2 ? seen2 : seen1, built, lo, hi, n, lists + int64_t(qh) * cap, &sample_count[qh],
             &list_len[qh], lo);
}

cudaError_t launch_match_csr(const Geometry& g, int n, const TablesPtrs& t, const DecodePtrs& dp,
                             cudaStream_t st) {
  const int lo = std::min(g.s, n);
  const int nwords = (n - lo + 31) >> 5;
  const int body = g.threshold >= 3 ? nwords * 9 : nwords * 2;
  const size_t smem = size_t(body + 1) * 4 + size_t(g.L) * g.nseg * 12 + 4 + size_t(g.L) * 2 + 16;
  cudaFuncSetAttribute(k_match_csr, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  k_match_csr<<<g.queries, kMatchWarps * 32, smem, st>>>(t.hdr, dp.qcodes, t.codes, t.off, t.ids, dp.lists,
                                                         dp.list_len, dp.sample_count, dp.counters, n, g.s, g.w, g.L,
                                                         g.nb, g.cap, g.nseg, g.group, g.threshold);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// inclusion probability u = P[Binomial(L, x) >= T], x = p^K  (Eq. 10 / Eq. 11; T = 2
// on the pages). The printed closed form 1 - sum_{j<T} C(L,j) x^j (1-x)^(L-j)
// cancels when L*x is small; there the tail sum_{j>=T} is added term by term instead
// (ratio of consecutive terms (L-j)/(j+1) * x/(1-x)).
// ---------------------------------------------------------------------------------
__device__ __forceinline__ float inclusion_prob(float x, int L, int threshold) {
  if (x >= 1.f) return 1.f;
  if (x <= 0.f) return 0.f;
  const float Lf = float(L);
  if (threshold <= 1) return -expm1f(Lf * log1pf(-x));
  if (L < threshold) return 0.f;
  const float l1x = log1pf(-x);
  const float r = __fdividef(x, 1.f - x);
  if (threshold == 2) {
    if (Lf * x < 0.1f) {
      // consecutive terms shrink by (L-j)/(j+1) * x/(1-x) < 0.04, so six terms reach
      // fp32 precision; the unrolled loop has constant reciprocals
      float term = 0.5f * Lf * (Lf - 1.f) * x * x * expf((Lf - 2.f) * l1x);
      float sum = term;
#pragma unroll
      for (int j = 2; j < 8; ++j) {
        term *= fmaxf(Lf - float(j), 0.f) * (1.f / float(j + 1)) * r;
        sum += term;
      }
      return sum;
    }
    // 1 - (1-x)^(L-1) (1 + (L-1) x)
    return -expm1f((Lf - 1.f) * l1x + log1pf((Lf - 1.f) * x));
  }
  const float T = float(threshold);
  if (Lf * x < 0.5f * T) {
    float lc = 0.f;  // log C(L, T) as a sum of T logs (T <= 7)
    for (int i = 1; i <= threshold; ++i) lc += logf((Lf - T + float(i)) / float(i));
    float term = expf(lc + T * logf(x) + (Lf - T) * l1x);
    float sum = term;
    for (int j = threshold; j < L && j < threshold + 24; ++j) {
      term *= (Lf - float(j)) / float(j + 1) * r;
      sum += term;
      if (term < 1e-9f * sum) break;
    }
    return sum;
  }
  float term = expf(Lf * l1x);
  float head = term;
  for (int j = 0; j < threshold - 1; ++j) {
    term *= (Lf - float(j)) / float(j + 1) * r;
    head += term;
  }
  return 1.f - head;
}

// -log u evaluated directly (cosines outside the table, or no table for this config)
__device__ __noinline__ float neg_log_u(float cs, int K, int L, int threshold) {
  const float p = 1.f - acosf(cs) * (1.f / CUDART_PI_F);
  // x = p^K by squaring (K <= 12)
  float x = 1.f, pb = p;
#pragma unroll
  for (int bit = 0; bit < 4; ++bit) {
    if ((K >> bit) & 1) x *= pb;
    pb *= pb;
  }
  return -logf(fmaxf(inclusion_prob(x, L, threshold), 1e-30f));
}

// lut[i] = -log u at the cosine kLutLo + i (kLutHi - kLutLo) / kLutN, evaluated exactly as
// the attention evaluates it outside the table; the header records which (K, L,
// threshold) it holds.
__global__ void k_logu_lut(float* __restrict__ lut, DevHeader* hdr, int K, int L, int threshold) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i <= kLutN) lut[i] = neg_log_u(kLutLo + float(i) * ((kLutHi - kLutLo) / float(kLutN)), K, L, threshold);
  if (i == 0) hdr->lut_key = lut_key_of(K, L, threshold);
}

cudaError_t launch_logu_lut(const Geometry& g, const TablesPtrs& t, cudaStream_t st) {
  k_logu_lut<<<(kLutN + 1 + 127) / 128, 128, 0, st>>>(t.lut, t.hdr, g.K, g.L, g.threshold);
  return cudaGetLastError();
}

constexpr int kAttThreads = 128;
constexpr float kLazyMargin = 8.f;  // weights below e^8 between raises of the reference

// ---------------------------------------------------------------------------------
// attention with register gathers: each warp walks groups of list entries, every
// lane loading one 16-byte slice of a K row and of a V row (a warp covers 32/LPR rows
// per load, LPR = lanes per row), so a group of U x RPI rows (U = 8) is in flight per warp
// without shared-memory staging; the online softmax state (m, l, acc) lives in
// registers and the warps of a CTA merge through shared memory at the end.
// ---------------------------------------------------------------------------------
constexpr int kGatherUnroll = 8;

// 16 bytes of a K or V row: read-only, and not kept in L1 (the rows are streamed; the
// query heads that share a row meet it in L2)
__device__ __forceinline__ uint4 ld_na(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
constexpr int kListChunk = 2048;

// a 16-byte slice of a row as packed fp32 pairs: 4 pairs of bf16, or 2 pairs of fp32
__device__ __forceinline__ void pairs_of(const uint4& v, const __nv_bfloat16*, uint64_t (&f)[4]) {
  f[0] = bf2_to_f2(v.x);
  f[1] = bf2_to_f2(v.y);
  f[2] = bf2_to_f2(v.z);
  f[3] = bf2_to_f2(v.w);
}
__device__ __forceinline__ void pairs_of(const uint4& v, const float*, uint64_t (&f)[2]) {
  f[0] = (uint64_t(v.y) << 32) | v.x;
  f[1] = (uint64_t(v.w) << 32) | v.z;
}

// Transposed butterfly over the LPR lanes of a row set: on entry s[u] is this lane's
// partial sum for row u (u < 8) of its sub-group. Three halving steps (lane offsets
// LPR/2, LPR/4, LPR/8) each exchange half of the remaining rows, leaving every lane one
// row, ju = 4*[lane & LPR/2] + 2*[lane & LPR/4] + [lane & LPR/8], summed over 8 lanes;
// the offsets below LPR/8 finish the sum. 7 shuffles for 8 rows instead of 8*log2(LPR).
template <int LPR>
__device__ __forceinline__ float reduce_rows8(float (&s)[8], int lane) {
  static_assert(LPR >= 8 && LPR <= 32, "row sets of 8..32 lanes");
#pragma unroll
  for (int lvl = 0; lvl < 3; ++lvl) {
    const int o = (LPR / 2) >> lvl, half = 4 >> lvl;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = up ? s[j] : s[j + half];
      const float keep = up ? s[j + half] : s[j];
      s[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float r = s[0];
#pragma unroll
  for (int o = LPR / 16; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}
// the lane of sub-group `sub` that holds row u after reduce_rows8
template <int LPR>
__device__ __forceinline__ int row_lane(int sub, int u) {
  return sub * LPR + (u >> 2) * (LPR / 2) + ((u >> 1) & 1) * (LPR / 4) + (u & 1) * (LPR / 8);
}

// CQ (center_query): p = 1 - theta(q - c, k - c)/pi instead of 1 - theta(q, k - c)/pi.
// bf16 rows run four CTAs per SM in both readings (the centered one then spills 24 bytes
// and still measured 181 us against 189 us at three per SM on the 32-layer step).
// Per row the kernel accumulates q.(k - c) and |k - c|^2 (and, for CQ, c.(k - c)); the
// logit's q.k is q.(k - c) + q.c with q.c constant per head, and the cosine's numerator
// q.(k - c) (or (q - c).(k - c) = q.(k - c) - c.(k - c)) is formed without subtracting two
// large dot products, which keeps it accurate when the keys sit far from the origin
// (narrow key cones).
template <typename T, int D, bool CQ>
__global__ void __launch_bounds__(kAttThreads, sizeof(T) == 2 ? 4 : 3) k_attend_gather(
    const uint32_t* __restrict__ lists, const int32_t* __restrict__ list_len, const float* __restrict__ center,
    const T* __restrict__ keys, const T* __restrict__ values, const T* __restrict__ q, float* __restrict__ out,
    float* __restrict__ partials, uint32_t* __restrict__ counters, const float* __restrict__ lut,
    const DevHeader* hdr, int cap, int group, int K, int L, int threshold, int P, int queries, uint32_t* status) {
  constexpr int VE = 16 / int(sizeof(T));  // elements per 16-byte slice
  constexpr int LPR = D / VE;              // lanes per row
  constexpr int RPI = 32 / LPR;            // rows per warp-wide load
  constexpr int U = kGatherUnroll;
  static_assert(U == 8, "reduce_rows8 takes 8 rows per lane");
  constexpr int GR = RPI * U;              // rows per group
  constexpr int NW = kAttThreads / 32;
  __shared__ float sm_m[NW], sm_l[NW];
  __shared__ float sm_acc[NW][D];
  __shared__ int sm_last;
  __shared__ uint32_t sl[kListChunk];
  // persistent: the CTAs take items (query head, slice) = (item / P, item % P) from a
  // work queue (counters[queries], zeroed by the match kernel), so that a CTA that
  // drew short slices takes more of them
  __shared__ int s_item;
  // the -log u table holds this config's (K, L, threshold) once the tables are built
  __shared__ float s_lut[kLutN + 1];
  const bool use_lut = hdr->lut_key == lut_key_of(K, L, threshold);
  if (use_lut)
    for (int i = threadIdx.x; i <= kLutN; i += kAttThreads) s_lut[i] = __ldg(lut + i);
  for (;;) {
  if (threadIdx.x == 0) s_item = int(atomicAdd(&counters[queries], 1u));
  __syncthreads();
  const int item = s_item;
  if (item >= queries * P) break;
  const int qh = item / P, split = item - (item / P) * P;
  const int unit = qh / group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane / LPR, part = lane % LPR;
  const int len = list_len[qh];
  const int per = (len + P - 1) / P;
  const int beg = min(len, split * per), end = min(len, beg + per);
  const uint32_t* lst = lists + int64_t(qh) * cap;
  const T* kbase = keys + int64_t(unit) * cap * D + part * VE;
  const T* vbase = values + int64_t(unit) * cap * D + part * VE;

  constexpr int NP = VE / 2;  // packed pairs per slice
  uint64_t q2[NP], c2[NP];
  float qq = 0.f, qc = 0.f;  // |q|^2 (CQ: |q - c|^2) and q.c
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    const float q0 = to_f(q[int64_t(qh) * D + part * VE + 2 * i]);
    const float q1 = to_f(q[int64_t(qh) * D + part * VE + 2 * i + 1]);
    const float c0 = center[int64_t(unit) * D + part * VE + 2 * i];
    const float c1 = center[int64_t(unit) * D + part * VE + 2 * i + 1];
    q2[i] = pk2(q0, q1);
    c2[i] = pk2(c0, c1);
    if (CQ) {
      const float m0 = q0 - c0, m1 = q1 - c1;
      qq = fmaf(m0, m0, fmaf(m1, m1, qq));
    } else {
      qq = fmaf(q0, q0, fmaf(q1, q1, qq));
    }
    qc = fmaf(q0, c0, fmaf(q1, c1, qc));
  }
#pragma unroll
  for (int o = LPR / 2; o >= 1; o >>= 1) {
    qq += __shfl_xor_sync(0xffffffffu, qq, o);
    qc += __shfl_xor_sync(0xffffffffu, qc, o);
  }
  const float qnorm = sqrtf(qq);  // norm of the hashed query
  const float inv_qnorm = qnorm > 0.f ? 1.f / qnorm : 0.f;
  // this lane's row of the group after reduce_rows8
  const int ju = 4 * ((lane & (LPR / 2)) != 0) + 2 * ((lane & (LPR / 4)) != 0) + ((lane & (LPR / 8)) != 0);
  const float scale = rsqrtf(float(D));

  float m_run = -CUDART_INF_F, l_run = 0.f;
  uint64_t acc2[NP];
#pragma unroll
  for (int i = 0; i < NP; ++i) acc2[i] = 0ull;

  // the slice's list entries go through shared memory (one round trip per chunk), so
  // that each group only waits for its K and V rows
  for (int c0 = beg; c0 < end; c0 += kListChunk) {
  const int cn = min(kListChunk, end - c0);
  for (int i = tid; i < cn; i += kAttThreads) sl[i] = __ldg(&lst[c0 + i]);
  __syncthreads();
  const int ngroups = (cn + GR - 1) / GR;
  for (int gi = warp; gi < ngroups; gi += NW) {
    const int e0 = gi * GR + sub;
    uint32_t ent[U];
    uint4 kv[U], vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * RPI;
      ent[u] = e < cn ? sl[e] : 0xffffffffu;
      // a list entry names a token of the unit's rows [0, capacity)
      if (ent[u] != 0xffffffffu && !in_range((ent[u] & ~kExactFlag) < uint32_t(cap), status)) ent[u] = 0xffffffffu;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (ent[u] != 0xffffffffu) {
        const int64_t tok = int64_t(ent[u] & ~kExactFlag);
        kv[u] = ld_na(reinterpret_cast<const uint4*>(kbase + tok * D));
        vv[u] = ld_na(reinterpret_cast<const uint4*>(vbase + tok * D));
      } else {
        kv[u] = make_uint4(0u, 0u, 0u, 0u);
        vv[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // per row: q.(k - c), |k - c|^2 (and c.(k - c) for CQ), reduced so that every lane
    // ends with one row of the group and evaluates the scalar part of its logit
    float sa[U], sn[U], sc[CQ ? U : 1];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint64_t k2[NP];
      pairs_of(kv[u], static_cast<const T*>(nullptr), k2);
      uint64_t a2 = 0ull, n2 = 0ull, m2 = 0ull;
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        const uint64_t d2 = sub2(k2[i], c2[i]);
        a2 = fma2(q2[i], d2, a2);
        n2 = fma2(d2, d2, n2);
        if (CQ) m2 = fma2(c2[i], d2, m2);
      }
      sa[u] = lo2(a2) + hi2(a2);
      sn[u] = lo2(n2) + hi2(n2);
      if (CQ) sc[CQ ? u : 0] = lo2(m2) + hi2(m2);
    }
    const float rqd = reduce_rows8<LPR>(sa, lane);  // q.(k - c)
    const float rkk = reduce_rows8<LPR>(sn, lane);
    float rnum = rqd;  // the cosine's numerator: q.(k - c), or (q - c).(k - c)
    if constexpr (CQ) rnum -= reduce_rows8<LPR>(sc, lane);
    const int je = gi * GR + ju * RPI + sub;
    uint32_t rent = je < cn ? sl[je] : 0xffffffffu;
#if MP_CHECK
    if ((rent & ~kExactFlag) >= uint32_t(cap)) rent = 0xffffffffu;  // skipped above, recorded there
#endif
    float lg = -CUDART_INF_F;
    if (rent != 0xffffffffu) {
      lg = (rqd + qc) * scale;  // q.k / sqrt(d)
      if (!(rent & kExactFlag)) {
        // p = 1 - theta(q, k - c)/pi (CQ: theta(q - c, k - c)), u = P[Bin(L, p^K) >= threshold]
        // (Eq. 10/11)
        float cs;
        if constexpr (CQ) {
          const float kn = sqrtf(rkk);
          cs = (qnorm > 0.f && kn > 0.f) ? rnum / (qnorm * kn) : 0.f;
        } else {
          cs = rkk > 0.f ? rnum * rsqrtf(rkk) * inv_qnorm : 0.f;
        }
        cs = fminf(1.f, fmaxf(-1.f, cs));
        if (use_lut && cs >= kLutLo && cs <= kLutHi) {
          // -log u interpolated on the build-time table (staged in shared memory)
          const float tt = (cs - kLutLo) * (float(kLutN) / (kLutHi - kLutLo));
          const int i = min(int(tt), kLutN - 1);
          const float a = s_lut[i], b = s_lut[i + 1];
          lg += fmaf(tt - float(i), b - a, a);
        } else {
          lg += neg_log_u(cs, K, L, threshold);
        }
      }
    }
    // The weights are exp(logit - m_run) for a reference m_run. With the query as it is,
    // the reference is raised (to the running maximum, rescaling l and acc) only when a
    // logit exceeds it by more than kLazyMargin: one vote per group instead of a maximum
    // reduction, weights below e^kLazyMargin; the final normalisation and the merges
    // (which carry each partial's reference) make the result independent of it. The
    // centered-query instance keeps the exact running maximum (at its register limit the
    // vote measured slower).
    const bool raise = CQ ? true : __any_sync(0xffffffffu, lg > m_run + kLazyMargin);
    float m_new = m_run;
    if (raise) {
      float mg = lg;  // group maximum (every row sits in LPR/8 lanes)
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
      m_new = fmaxf(m_run, mg);
    }
    if (m_new == -CUDART_INF_F) continue;  // warp-uniform: nothing valid yet
    const float alpha = raise ? ((m_run == -CUDART_INF_F) ? 0.f : __expf(m_run - m_new)) : 1.f;
    // each lane's weights for its rows: the row lane's logit, shifted by the reference
    const float pw = (lg == -CUDART_INF_F) ? 0.f : __expf(lg - m_new);
    float ps = 0.f;
    if (raise) {
      const uint64_t al2 = pk2(alpha, alpha);
#pragma unroll
      for (int i = 0; i < NP; ++i) acc2[i] = mul2(acc2[i], al2);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float p = __shfl_sync(0xffffffffu, pw, row_lane<LPR>(sub, u));
      ps += p;
      const uint64_t p2 = pk2(p, p);
      uint64_t v2[NP];
      pairs_of(vv[u], static_cast<const T*>(nullptr), v2);
#pragma unroll
      for (int i = 0; i < NP; ++i) acc2[i] = fma2(p2, v2[i], acc2[i]);
    }
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    l_run = l_run * alpha + ps;
    m_run = m_new;
  }
  __syncthreads();  // before the next chunk overwrites the staged entries
  }
  float acc[VE];
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    acc[2 * i] = lo2(acc2[i]);
    acc[2 * i + 1] = hi2(acc2[i]);
  }
  // rows of the other sub-groups of lanes hold the same dims: fold them
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int i = 0; i < VE; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], o);
  if (lane < LPR)
#pragma unroll
    for (int i = 0; i < VE; ++i) sm_acc[warp][part * VE + i] = acc[i];
  if (lane == 0) {
    sm_m[warp] = m_run;
    sm_l[warp] = l_run;
  }
  __syncthreads();
  // merge the warps of this CTA
  float M = -CUDART_INF_F;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w]);
  float f[NW];
  float lt = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    f[w] = (sm_m[w] == -CUDART_INF_F) ? 0.f : __expf(sm_m[w] - M);
    lt = fmaf(sm_l[w], f[w], lt);
  }
  if (P == 1) {
    for (int dd = tid; dd < D; dd += kAttThreads) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) a = fmaf(sm_acc[w][dd], f[w], a);
      out[int64_t(qh) * D + dd] = lt > 0.f ? a / lt : 0.f;
    }
    __syncthreads();  // shared state is reused by the next item
    continue;
  }
  float* part_out = partials + (int64_t(qh) * kSplitsMax + split) * (D + 2);
  for (int dd = tid; dd < D; dd += kAttThreads) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) a = fmaf(sm_acc[w][dd], f[w], a);
    part_out[2 + dd] = a;
  }
  if (tid == 0) {
    part_out[0] = M;
    part_out[1] = lt;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t done = atomicAdd(&counters[qh], 1u);
    sm_last = (done == uint32_t(P - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (sm_last) {
    __threadfence();
    const float* base = partials + int64_t(qh) * kSplitsMax * (D + 2);
    float MM = -CUDART_INF_F;
    for (int p = 0; p < P; ++p) MM = fmaxf(MM, __ldcg(&base[p * (D + 2)]));
    for (int dd = tid; dd < D; dd += kAttThreads) {
      float l2 = 0.f, a2 = 0.f;
      if (MM != -CUDART_INF_F) {
        for (int p = 0; p < P; ++p) {
          const float mp = __ldcg(&base[p * (D + 2)]);
          if (mp == -CUDART_INF_F) continue;
          const float fp = __expf(mp - MM);
          l2 = fmaf(__ldcg(&base[p * (D + 2) + 1]), fp, l2);
          a2 = fmaf(__ldcg(&base[p * (D + 2) + 2 + dd]), fp, a2);
        }
      }
      out[int64_t(qh) * D + dd] = l2 > 0.f ? a2 / l2 : 0.f;
    }
    if (tid == 0) counters[qh] = 0u;
  }
  __syncthreads();  // shared state is reused by the next item
  }
}

template <typename T, int D, bool CQ>
static cudaError_t launch_attend_t(const Geometry& g, int splits, const TablesPtrs& t, const void* keys,
                                   const void* values, const void* q, float* out, const DecodePtrs& dp,
                                   cudaStream_t st) {
  // persistent grid: as many CTAs as can be resident at once, each walking items. The
  // resident count per SM is cached per device; callers on several host threads may fill
  // the cache at once, each writing the same value.
  static std::atomic<int> per_sm[64];
  int dev = 0;
  cudaGetDevice(&dev);
  int occ = per_sm[dev & 63].load(std::memory_order_relaxed);
  if (occ == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_attend_gather<T, D, CQ>, kAttThreads, 0) !=
            cudaSuccess ||
        occ < 1)
      occ = 1;
    per_sm[dev & 63].store(occ, std::memory_order_relaxed);
  }
  const int64_t items = int64_t(splits) * g.queries;
  const int grid = int(std::min<int64_t>(items, int64_t(occ) * device_sm_count()));
  k_attend_gather<T, D, CQ><<<grid, kAttThreads, 0, st>>>(
      dp.lists, dp.list_len, t.center, static_cast<const T*>(keys), static_cast<const T*>(values),
      static_cast<const T*>(q), out, dp.partials, dp.counters, t.lut, t.hdr, g.cap, g.group, g.K, g.L, g.threshold, splits,
      g.queries, &t.hdr->status);
  return cudaGetLastError();
}

cudaError_t launch_attend(const Geometry& g, int n, int splits, const TablesPtrs& t, const void* keys,
                          const void* values, const void* q, float* out, const DecodePtrs& dp,
                          cudaStream_t st) {
  (void)n;
  if (g.center_query) {
    if (g.dtype == MP_DTYPE_BF16) {
      if (g.d == 128) return launch_attend_t<__nv_bfloat16, 128, true>(g, splits, t, keys, values, q, out, dp, st);
      return launch_attend_t<__nv_bfloat16, 64, true>(g, splits, t, keys, values, q, out, dp, st);
    }
    if (g.d == 128) return launch_attend_t<float, 128, true>(g, splits, t, keys, values, q, out, dp, st);
    return launch_attend_t<float, 64, true>(g, splits, t, keys, values, q, out, dp, st);
  }
  if (g.dtype == MP_DTYPE_BF16) {
    if (g.d == 128) return launch_attend_t<__nv_bfloat16, 128, false>(g, splits, t, keys, values, q, out, dp, st);
    return launch_attend_t<__nv_bfloat16, 64, false>(g, splits, t, keys, values, q, out, dp, st);
  }
  if (g.d == 128) return launch_attend_t<float, 128, false>(g, splits, t, keys, values, q, out, dp, st);
  return launch_attend_t<float, 64, false>(g, splits, t, keys, values, q, out, dp, st);
}

}  // namespace mp
