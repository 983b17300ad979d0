// Decode step: sampled-set construction from the bucketed tables, then the
// importance-weighted attention over the sampled keys plus the exact sink/window
// tokens, split across CTAs with a fused log-sum-exp combine.
// MagicPIG (arXiv 2410.16179v2): Algorithm 1, Eq. 9-11, §4.4 "On-device cache".
#include <math_constants.h>

#include "mp_compact.cuh"
#include "mp_internal.h"

namespace mp {

// ---------------------------------------------------------------------------------
// sampled set: one CTA per query head
// ---------------------------------------------------------------------------------
// Bitmaps over token ids [0, n - window): `seen1` marks tokens met in >= 1 table's
// bucket, `seen2` in >= 2. With threshold 2 the sampled set is seen2 restricted to
// [n_sink, n - window); with threshold 1 it is seen1. Compaction writes S in
// ascending token order, then the exact tokens (bit 31 set).
__global__ void __launch_bounds__(256) k_match_csr(DevHeader* hdr,
                                                   const uint16_t* __restrict__ qcodes,
                                                   const uint16_t* __restrict__ codes,
                                                   const uint32_t* __restrict__ off,
                                                   const uint32_t* __restrict__ ids, uint32_t* __restrict__ lists,
                                                   int32_t* __restrict__ list_len, int32_t* __restrict__ sample_count,
                                                   uint32_t* __restrict__ counters, int n, int s, int w, int L,
                                                   int nb, int cap, int group, int threshold) {
  extern __shared__ uint32_t sm[];
  const int qh = blockIdx.x;
  const int unit = qh / group;  // [layer][batch][q_head] -> [layer][batch][kv_head]
  const int lo = min(s, n);
  const int hi = max(lo, n - w);
  const int nwords = (hi + 31) >> 5;
  uint32_t* seen1 = sm;
  uint32_t* seen2 = sm + nwords;
  uint16_t* qc = reinterpret_cast<uint16_t*>(sm + 2 * nwords);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  const bool built = hdr->magic == kMagic;
  const int n0 = hdr->n_prefill;
  const int app_end = hdr->appended_end;
  if (threadIdx.x == 0) {
    counters[qh] = 0u;
    if (!built) atomicOr(&hdr->status, MP_STATUS_NOT_BUILT);
    else if (hi > app_end) atomicOr(&hdr->status, MP_STATUS_APPEND_GAP);
  }
  for (int i = threadIdx.x; i < 2 * nwords; i += blockDim.x) sm[i] = 0u;
  for (int t = threadIdx.x; t < L; t += blockDim.x) qc[t] = qcodes[int64_t(qh) * L + t];
  __syncthreads();

  if (built && hi > lo) {
    // tokens hashed at build time: walk the query's bucket in every table
    const int64_t tbase = int64_t(unit) * L;
    for (int t = warp; t < L; t += 8) {
      const uint32_t* o = off + (tbase + t) * (nb + 1);
      const int code = qc[t];
      const uint32_t b0 = o[code], b1 = o[code + 1];
      const uint32_t* id = ids + (tbase + t) * cap;
      for (uint32_t i = b0 + lane; i < b1; i += 32) {
        const uint32_t tok = id[i];
        if (tok < uint32_t(hi)) {
          const uint32_t bit = 1u << (tok & 31);
          const uint32_t old = atomicOr(&seen1[tok >> 5], bit);
          if (old & bit) atomicOr(&seen2[tok >> 5], bit);
        }
      }
    }
    // tokens appended after the build that have left the window: compare codes
    const int a0 = max(lo, n0), a1 = min(hi, app_end);
    for (int tok = a0 + warp; tok < a1; tok += 8) {
      int cnt = 0;
      for (int t = lane; t < L; t += 32)
        cnt += (codes[(tbase + t) * cap + tok] == qc[t]) ? 1 : 0;
#pragma unroll
      for (int k = 16; k > 0; k >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, k);
      if (lane == 0) {
        const uint32_t bit = 1u << (tok & 31);
        if (cnt >= 1) atomicOr(&seen1[tok >> 5], bit);
        if (cnt >= 2) atomicOr(&seen2[tok >> 5], bit);
      }
    }
  }
  __syncthreads();

  // compaction of [lo, hi)
  write_list(threshold >= 2 ? seen2 : seen1, built, lo, hi, n, lists + int64_t(qh) * cap, &sample_count[qh],
             &list_len[qh]);
}

cudaError_t launch_match_csr(const Geometry& g, int n, const TablesPtrs& t, const DecodePtrs& dp,
                             cudaStream_t st) {
  const int lo = min(g.s, n);
  const int hi = max(lo, n - g.w);
  const int nwords = (hi + 31) >> 5;
  const size_t smem = size_t(2 * nwords) * 4 + size_t(g.L) * 2 + 16;
  cudaFuncSetAttribute(k_match_csr, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  k_match_csr<<<g.queries, 256, smem, st>>>(t.hdr, dp.qcodes, t.codes, t.off, t.ids, dp.lists,
                                            dp.list_len, dp.sample_count, dp.counters, n, g.s, g.w, g.L,
                                            g.nb, g.cap, g.group, g.threshold);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// inclusion probability u = P[Binomial(L, x) >= T], x = p^K  (Eq. 10 / Eq. 11)
// ---------------------------------------------------------------------------------
// The printed closed form cancels when L*x is small; there the tail is summed
// term by term: C(L,2) x^2 (1-x)^(L-2) * (1 + ratio + ...). Elsewhere
// 1 - (1-x)^(L-1) (1 + (L-1) x) is evaluated as -expm1(log1p(-x)(L-1) + log1p((L-1)x)).
__device__ __forceinline__ float inclusion_prob(float x, int L, int threshold) {
  if (x >= 1.f) return 1.f;
  if (x <= 0.f) return 0.f;
  const float Lf = float(L);
  if (threshold <= 1) return -expm1f(Lf * log1pf(-x));
  if (L < 2) return 0.f;
  if (Lf * x < 0.1f) {
    const float r = x / (1.f - x);
    float term = 0.5f * Lf * (Lf - 1.f) * x * x * expf((Lf - 2.f) * log1pf(-x));
    float sum = term;
    for (int j = 2; j < L && j < 14; ++j) {
      term *= (Lf - float(j)) / float(j + 1) * r;
      sum += term;
      if (term < 1e-9f * sum) break;
    }
    return sum;
  }
  return -expm1f((Lf - 1.f) * log1pf(-x) + log1pf((Lf - 1.f) * x));
}

// ---------------------------------------------------------------------------------
// bounded mbarrier / bulk-copy helpers (inline PTX)
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Returns false if the phase did not complete within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------------
// attention over list entries, split-K across CTAs, fused combine
// ---------------------------------------------------------------------------------
constexpr int kRows = 32;     // list entries per tile
constexpr int kStages = 2;
constexpr int kAttThreads = 128;

template <typename T, int D>
struct AttSmem {
  T k[kStages][kRows][D];
  T v[kStages][kRows][D];
  float logit[kRows];
  float e[kRows];
  float red[kAttThreads];
  uint64_t bar[kStages];
  int last;
};

template <typename T>
__device__ __forceinline__ void load_pair(const T* p, float& a, float& b);
template <>
__device__ __forceinline__ void load_pair<__nv_bfloat16>(const __nv_bfloat16* p, float& a, float& b) {
  const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(p);
  a = __bfloat162float(v.x);
  b = __bfloat162float(v.y);
}
template <>
__device__ __forceinline__ void load_pair<float>(const float* p, float& a, float& b) {
  const float2 v = *reinterpret_cast<const float2*>(p);
  a = v.x;
  b = v.y;
}

// One CTA = one slice of one query head's list. Per tile of 32 entries: the K and V
// rows are gathered into shared memory by bulk asynchronous copies (one 128/256/512-B
// copy per row, completion counted on an mbarrier), a warp per row forms the logit
// q.k/sqrt(d) - log u (u = 1 for exact tokens) and an online softmax keeps
// (m, l, acc[d]). Slices of a head are merged by the CTA that finishes last.
template <typename T, int D>
__global__ void __launch_bounds__(kAttThreads) k_attend(
    DevHeader* hdr, const uint32_t* __restrict__ lists, const int32_t* __restrict__ list_len,
    const float* __restrict__ center, const T* __restrict__ keys, const T* __restrict__ values,
    const T* __restrict__ q, float* __restrict__ out, float* __restrict__ partials, uint32_t* __restrict__ counters,
    int cap, int group, int K, int L, int threshold) {
  extern __shared__ __align__(128) unsigned char smraw[];
  AttSmem<T, D>& S = *reinterpret_cast<AttSmem<T, D>*>(smraw);
  const int qh = blockIdx.y, split = blockIdx.x, P = gridDim.x;
  const int unit = qh / group;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int len = list_len[qh];
  const int per = (len + P - 1) / P;
  const int beg = min(len, split * per), end = min(len, beg + per);
  const uint32_t* lst = lists + int64_t(qh) * cap;
  const T* kbase = keys + int64_t(unit) * cap * D;
  const T* vbase = values + int64_t(unit) * cap * D;
  constexpr uint32_t kRowBytes = D * sizeof(T);
  constexpr int kPer = D / 64;  // element pairs per lane

  // the lane's share of q and c: elements 2*lane + 64*i, +1
  float qr[2 * kPer], cr[2 * kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = 2 * lane + 64 * i;
    qr[2 * i] = to_f(q[int64_t(qh) * D + j]);
    qr[2 * i + 1] = to_f(q[int64_t(qh) * D + j + 1]);
    cr[2 * i] = center[int64_t(unit) * D + j];
    cr[2 * i + 1] = center[int64_t(unit) * D + j + 1];
  }
  float qq = 0.f;
#pragma unroll
  for (int i = 0; i < 2 * kPer; ++i) qq = fmaf(qr[i], qr[i], qq);
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) qq += __shfl_xor_sync(0xffffffffu, qq, k);
  const float qnorm = sqrtf(qq);
  const float scale = rsqrtf(float(D));

  if (tid == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(&S.bar[s], kRows);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();

  const int ntiles = (end - beg + kRows - 1) / kRows;
  auto issue = [&](int tile) {
    const int st = tile % kStages;
    if (tid < kRows) {
      const int e = beg + tile * kRows + tid;
      if (e < end) {
        const uint32_t tok = lst[e] & ~kExactFlag;
        mbar_arrive_expect_tx(&S.bar[st], 2 * kRowBytes);
        bulk_g2s(&S.k[st][tid][0], kbase + int64_t(tok) * D, kRowBytes, &S.bar[st]);
        bulk_g2s(&S.v[st][tid][0], vbase + int64_t(tok) * D, kRowBytes, &S.bar[st]);
      } else {
        mbar_arrive(&S.bar[st]);
      }
    }
  };

  constexpr int RS = kAttThreads / D;  // threads per output dim (1 for d=128, 2 for d=64)
  const int dim = tid % D, rphase = tid / D;
  float m_run = -CUDART_INF_F, l_run = 0.f, acc = 0.f;

  if (ntiles > 0) issue(0);
  for (int tile = 0; tile < ntiles; ++tile) {
    const int st = tile % kStages;
    if (tile + 1 < ntiles) issue(tile + 1);
    const bool got = mbar_wait_bounded(&S.bar[st], uint32_t((tile / kStages) & 1));
    if (__syncthreads_or(!got)) {
      // give up on this head; wait (bounded) for the copies still in flight so that
      // none lands after the CTA has released its shared memory
      if (tid == 0) atomicOr(&hdr->status, MP_STATUS_WAIT_TIMEOUT);
      (void)mbar_wait_bounded(&S.bar[st], uint32_t((tile / kStages) & 1));
      if (tile + 1 < ntiles)
        (void)mbar_wait_bounded(&S.bar[(tile + 1) % kStages], uint32_t(((tile + 1) / kStages) & 1));
      m_run = -CUDART_INF_F;
      l_run = 0.f;
      acc = 0.f;
      break;
    }
    const int nvalid = min(kRows, end - (beg + tile * kRows));
    // logits: one warp per row
    for (int r = warp; r < kRows; r += kAttThreads / 32) {
      float lg = -CUDART_INF_F;
      if (r < nvalid) {
        const uint32_t ent = lst[beg + tile * kRows + r];
        float dot = 0.f, dotc = 0.f, kk = 0.f;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          float k0, k1;
          load_pair<T>(&S.k[st][r][2 * lane + 64 * i], k0, k1);
          const float c0 = k0 - cr[2 * i], c1 = k1 - cr[2 * i + 1];
          dot = fmaf(qr[2 * i], k0, fmaf(qr[2 * i + 1], k1, dot));
          dotc = fmaf(qr[2 * i], c0, fmaf(qr[2 * i + 1], c1, dotc));
          kk = fmaf(c0, c0, fmaf(c1, c1, kk));
        }
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) {
          dot += __shfl_xor_sync(0xffffffffu, dot, k);
          dotc += __shfl_xor_sync(0xffffffffu, dotc, k);
          kk += __shfl_xor_sync(0xffffffffu, kk, k);
        }
        lg = dot * scale;
        if (!(ent & kExactFlag)) {
          // p = 1 - theta(q, k - c)/pi, u = P[Bin(L, p^K) >= threshold]  (Eq. 10/11)
          const float kn = sqrtf(kk);
          float cs = (qnorm > 0.f && kn > 0.f) ? dotc / (qnorm * kn) : 0.f;
          cs = fminf(1.f, fmaxf(-1.f, cs));
          const float p = 1.f - acosf(cs) * (1.f / CUDART_PI_F);
          float x = 1.f;
          for (int b = 0; b < K; ++b) x *= p;
          const float u = fmaxf(inclusion_prob(x, L, threshold), 1e-30f);
          lg -= logf(u);
        }
      }
      if (lane == 0) S.logit[r] = lg;
    }
    __syncthreads();
    // online softmax: every thread derives the same max and rescale factor
    float mt = -CUDART_INF_F;
    for (int r = 0; r < nvalid; ++r) mt = fmaxf(mt, S.logit[r]);
    const float m_new = fmaxf(m_run, mt);
    const float alpha = (m_run == -CUDART_INF_F) ? 0.f : __expf(m_run - m_new);
    if (tid < kRows) S.e[tid] = (tid < nvalid && S.logit[tid] != -CUDART_INF_F) ? __expf(S.logit[tid] - m_new) : 0.f;
    __syncthreads();
    float esum = 0.f;
    for (int r = 0; r < nvalid; ++r) esum += S.e[r];
    l_run = l_run * alpha + esum;
    m_run = m_new;
    float a = 0.f;
    for (int r = rphase; r < nvalid; r += RS) a = fmaf(S.e[r], to_f(S.v[st][r][dim]), a);
    acc = acc * alpha + a;
    __syncthreads();
  }
  // fold the RS row phases of each dim
  if (RS > 1) {
    S.red[tid] = acc;
    __syncthreads();
    if (tid < D) {
      float v = 0.f;
      for (int r = 0; r < RS; ++r) v += S.red[r * D + tid];
      acc = v;
    }
  }
  if (P == 1) {
    if (tid < D) out[int64_t(qh) * D + tid] = (l_run > 0.f) ? acc / l_run : 0.f;
    return;
  }
  float* part = partials + (int64_t(qh) * kSplitsMax + split) * (D + 2);
  if (tid < D) part[2 + tid] = acc;
  if (tid == 0) {
    part[0] = m_run;
    part[1] = l_run;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t done = atomicAdd(&counters[qh], 1u);
    S.last = (done == uint32_t(P - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!S.last) return;
  __threadfence();
  if (tid < D) {
    const float* base = partials + int64_t(qh) * kSplitsMax * (D + 2);
    float M = -CUDART_INF_F;
    for (int p = 0; p < P; ++p) M = fmaxf(M, __ldcg(&base[p * (D + 2)]));
    float lt = 0.f, at = 0.f;
    if (M != -CUDART_INF_F) {
      for (int p = 0; p < P; ++p) {
        const float mp = __ldcg(&base[p * (D + 2)]);
        if (mp == -CUDART_INF_F) continue;
        const float f = __expf(mp - M);
        lt = fmaf(__ldcg(&base[p * (D + 2) + 1]), f, lt);
        at = fmaf(__ldcg(&base[p * (D + 2) + 2 + tid]), f, at);
      }
    }
    out[int64_t(qh) * D + tid] = lt > 0.f ? at / lt : 0.f;
  }
  if (tid == 0) counters[qh] = 0u;
}

template <typename T, int D>
static cudaError_t launch_attend_t(const Geometry& g, int splits, const TablesPtrs& t, const void* keys,
                                   const void* values, const void* q, float* out, const DecodePtrs& dp,
                                   cudaStream_t st) {
  const size_t smem = sizeof(AttSmem<T, D>);
  cudaFuncSetAttribute(k_attend<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  dim3 grid(splits, g.queries);
  k_attend<T, D><<<grid, kAttThreads, smem, st>>>(
      t.hdr, dp.lists, dp.list_len, t.center, static_cast<const T*>(keys), static_cast<const T*>(values),
      static_cast<const T*>(q), out, dp.partials, dp.counters, g.cap, g.group, g.K, g.L, g.threshold);
  return cudaGetLastError();
}

cudaError_t launch_attend(const Geometry& g, int n, int splits, const TablesPtrs& t, const void* keys,
                          const void* values, const void* q, float* out, const DecodePtrs& dp,
                          cudaStream_t st) {
  (void)n;
  if (g.dtype == MP_DTYPE_BF16) {
    if (g.d == 128) return launch_attend_t<__nv_bfloat16, 128>(g, splits, t, keys, values, q, out, dp, st);
    return launch_attend_t<__nv_bfloat16, 64>(g, splits, t, keys, values, q, out, dp, st);
  }
  if (g.d == 128) return launch_attend_t<float, 128>(g, splits, t, keys, values, q, out, dp, st);
  return launch_attend_t<float, 64>(g, splits, t, keys, values, q, out, dp, st);
}

}  // namespace mp
