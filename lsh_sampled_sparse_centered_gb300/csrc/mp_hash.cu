// Build-time and decode-time SimHash on CUDA cores:
//  - W preparation (transpose to [KLp][d], zero padding, bf16 copy),
//  - key centering (mean of keys [n_sink, n_prefill) per KV head, and beta = W^T c),
//  - hashing of arbitrary rows (queries, appended keys, fp32 prefill keys) into
//    L packed K-bit codes.
// MagicPIG (arXiv 2410.16179v2) §2.2 SimHash, §4.3 "Hash function selection" and
// "Data pre-processing", Algorithm 1 'Encode'.
#include "mp_internal.h"

namespace mp {

// ---------------------------------------------------------------------------------
// W [n_w][d][K*L] fp32 -> wt32 [n_w][TC][d] fp32 and (bf16 configs) wt16 [n_w][3][TC][d]
// in tile-aligned column order: 256-column tile n holds tables n*tpt .. n*tpt+tpt-1,
// column n*256 + i*K + b is bit b of the tile's i-th table; the other columns are zero.
// wt16 holds W as three bf16 terms: hi = bf16(W), mid = bf16(W - hi), lo = bf16(W - hi -
// mid); each step removes at least 8 mantissa bits, so hi + mid + lo = W exactly. If any
// mid or lo term is nonzero the header's w_terms3 flag (and the informational status
// bit) tells the tensor-core kernels to add the two extra terms.
// ---------------------------------------------------------------------------------
__global__ void k_prepare_w(const float* __restrict__ W, float* __restrict__ wt32,
                            __nv_bfloat16* __restrict__ wt16, int d, int K, int L, int tpt, int kltc,
                            DevHeader* hdr) {
  const int m = blockIdx.y;
  const int jc = blockIdx.x;  // one tensor-core column per block, d threads
  const int kl = K * L;
  const int n = jc >> 8, within = jc & 255;
  const int i = within / K, b = within - i * K;
  const int t = n * tpt + i;
  const bool live = i < tpt && t < L;
  bool inexact = false;
  for (int dd = threadIdx.x; dd < d; dd += blockDim.x) {
    const float v = live ? W[(int64_t(m) * d + dd) * kl + t * K + b] : 0.f;
    wt32[(int64_t(m) * kltc + jc) * d + dd] = v;
    if (wt16) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const float r1 = v - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
      const int64_t o = ((int64_t(m) * 3) * kltc + jc) * d + dd;
      wt16[o] = hi;
      wt16[o + int64_t(kltc) * d] = mid;
      wt16[o + 2 * int64_t(kltc) * d] = lo;
      inexact |= (r1 != 0.f);
    }
  }
  if (inexact) {
    atomicOr(&hdr->status, MP_STATUS_W_NOT_BF16);
    atomicOr(&hdr->w_terms3, 1u);
  }
}

cudaError_t launch_prepare_w(const Geometry& g, const float* W, const TablesPtrs& t, cudaStream_t st) {
  if (g.kltc == 0) return cudaSuccess;
  dim3 grid(g.kltc, g.n_w);
  k_prepare_w<<<grid, 128, 0, st>>>(W, t.wt32, t.wt16, g.d, g.K, g.L, g.tpt, g.kltc, t.hdr);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// centering: per unit, partial sums over `parts` token ranges, then the mean and
// beta = W^T c. Deterministic (fixed summation order).
// ---------------------------------------------------------------------------------
// 16-byte loads: a row of d elements is read by d/VE lanes (VE = 8 bf16 or 4 fp32),
// 256/(d/VE) rows per step; the partial sums of the row phases meet in shared memory.
template <typename T>
__global__ void __launch_bounds__(256) k_center_parts(const T* __restrict__ keys, float* __restrict__ cparts,
                                                      int d, int cap, int lo, int hi, int parts) {
  constexpr int VE = 16 / int(sizeof(T));
  extern __shared__ float red[];  // [256 / (d / VE)][d]
  const int u = blockIdx.y, part = blockIdx.x;
  const int lpr = d / VE, rpi = 256 / lpr;
  const int span = (hi - lo + parts - 1) / parts;
  const int t0 = lo + part * span;
  const int t1 = min(hi, t0 + span);
  const int pl = threadIdx.x % lpr, ph = threadIdx.x / lpr;
  const T* base = keys + int64_t(u) * cap * d + pl * VE;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int t = t0 + ph;
  for (; t + 3 * rpi < t1; t += 4 * rpi) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldg(reinterpret_cast<const uint4*>(base + int64_t(t + k * rpi) * d));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (sizeof(T) == 2) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[k]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(h[i]);
          acc[2 * i] += f.x;
          acc[2 * i + 1] += f.y;
        }
      } else {
        acc[0] += __uint_as_float(v[k].x);
        acc[1] += __uint_as_float(v[k].y);
        acc[2] += __uint_as_float(v[k].z);
        acc[3] += __uint_as_float(v[k].w);
      }
    }
  }
  for (; t < t1; t += rpi) {
    const T* row = base + int64_t(t) * d;
#pragma unroll
    for (int i = 0; i < VE; ++i) acc[i] += to_f(row[i]);
  }
#pragma unroll
  for (int i = 0; i < VE; ++i) red[ph * d + pl * VE + i] = acc[i];
  __syncthreads();
  for (int dim = threadIdx.x; dim < d; dim += blockDim.x) {
    float sum = 0.f;
    for (int p = 0; p < rpi; ++p) sum += red[p * d + dim];
    cparts[(int64_t(u) * parts + part) * d + dim] = sum;
  }
}

// The mean key of each unit from its partial sums (fixed summation order), and the
// header fields of a built table set.
__global__ void k_center_mean(const float* __restrict__ cparts, float* __restrict__ center, int d, int parts,
                              int count, DevHeader* hdr, int n_prefill, int no_center) {
  const int u = blockIdx.x;
  for (int dim = threadIdx.x; dim < d; dim += blockDim.x) {
    float s = 0.f;
    for (int p = 0; p < parts; ++p) s += cparts[(int64_t(u) * parts + p) * d + dim];
    center[int64_t(u) * d + dim] = (count > 0 && !no_center) ? s / float(count) : 0.f;
  }
  if (u == 0 && threadIdx.x == 0) {
    hdr->n_prefill = n_prefill;
    hdr->appended_end = n_prefill;
    __threadfence();
    hdr->magic = kMagic;
  }
}

// -beta = -W^T c (fp32 W) for kBetaUnits units x 128 tensor-core columns per CTA, in
// tile-aligned column order, stored as fp32 and as three bf16 terms hi + mid + lo (each
// the bf16 rounding of what is left, an exact split of the fp32 value): the tensor-core
// hash adds them through one extra K step against rows of ones. Thread j owns column
// j of the block and reads its W row once per W matrix met in the unit tile.
constexpr int kBetaUnits = 16;
constexpr int kBetaCols = 128;

__global__ void __launch_bounds__(kBetaCols, 4) k_center_beta(const float* __restrict__ center,
                                                          __nv_bfloat16* __restrict__ beta,
                                                          __nv_bfloat16* __restrict__ ones,
                                                          float* __restrict__ negbeta, const float* __restrict__ wt32,
                                                          int units, int d, int kltc, int units_per_w,
                                                          int64_t w_stride) {
  extern __shared__ float cs[];  // [kBetaUnits][d]
  const int u0 = blockIdx.x * kBetaUnits;
  const int nu = min(kBetaUnits, units - u0);
  for (int i = threadIdx.x; i < nu * d; i += blockDim.x) cs[i] = center[int64_t(u0) * d + i];
  if (blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) ones[i] = __float2bfloat16_rn((i & 15) < 3 ? 1.f : 0.f);
  __syncthreads();
  const int j = blockIdx.y * kBetaCols + threadIdx.x;
  if (j >= kltc) return;
  float acc[kBetaUnits];
#pragma unroll
  for (int i = 0; i < kBetaUnits; ++i) acc[i] = 0.f;
  // units of the tile that share a W matrix are done together, one pass over the W row
  for (int ua = 0; ua < nu;) {
    const int wi = (u0 + ua) / units_per_w;
    const int ub = min(nu, (wi + 1) * units_per_w - u0);  // first unit of the next W matrix
    const float4* row = reinterpret_cast<const float4*>(wt32 + int64_t(wi) * w_stride + int64_t(j) * d);
    for (int q = 0; q < d / 4; ++q) {
      const float4 w = __ldg(row + q);
#pragma unroll
      for (int i = 0; i < kBetaUnits; ++i)
        if (i >= ua && i < ub) {
          const float4 c = reinterpret_cast<const float4*>(cs + i * d)[q];
          acc[i] = fmaf(w.x, c.x, fmaf(w.y, c.y, fmaf(w.z, c.z, fmaf(w.w, c.w, acc[i]))));
        }
    }
    ua = ub;
  }
#pragma unroll
  for (int i = 0; i < kBetaUnits; ++i) {
    if (i >= nu) continue;
    const int64_t u = u0 + i;
    const float nb = -acc[i];
    negbeta[u * kltc + j] = nb;
    const __nv_bfloat16 hi = __float2bfloat16_rn(nb);
    const float r1 = nb - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    __nv_bfloat16* o = beta + (u * kltc + j) * 16;
    o[0] = hi;
    o[1] = mid;
    o[2] = lo;
#pragma unroll
    for (int k = 3; k < 16; ++k) o[k] = __float2bfloat16_rn(0.f);
  }
}

cudaError_t launch_center(const Geometry& g, const void* keys, int n_prefill, const TablesPtrs& t,
                          cudaStream_t st) {
  const int lo = min(g.s, n_prefill), hi = n_prefill;
  const int threads = 256;
  dim3 grid(g.parts, g.units);
  // row phases per block x d floats of partial sums
  if (g.dtype == MP_DTYPE_BF16)
    k_center_parts<__nv_bfloat16><<<grid, threads, size_t(threads / (g.d / 8)) * g.d * sizeof(float), st>>>(
        static_cast<const __nv_bfloat16*>(keys), t.cparts, g.d, g.cap, lo, hi, g.parts);
  else
    k_center_parts<float><<<grid, threads, size_t(threads / (g.d / 4)) * g.d * sizeof(float), st>>>(
        static_cast<const float*>(keys), t.cparts, g.d, g.cap, lo, hi, g.parts);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_center_mean<<<g.units, 128, 0, st>>>(t.cparts, t.center, g.d, g.parts, hi - lo, t.hdr, n_prefill, g.no_center);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // -beta only for the tensor-core paths (bf16 configurations)
  if (t.wt16 && g.kltc > 0) {
    const int64_t w_stride = g.w_per_layer ? int64_t(g.kltc) * g.d : 0;
    dim3 gb((g.units + kBetaUnits - 1) / kBetaUnits, (g.kltc + kBetaCols - 1) / kBetaCols);
    k_center_beta<<<gb, kBetaCols, size_t(kBetaUnits) * g.d * sizeof(float), st>>>(
        t.center, t.beta, t.ones, t.negbeta, t.wt32, g.units, g.d, g.kltc, g.batch * g.kvh, w_stride);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// SimHash of rows on CUDA cores: a CTA hashes R rows against one 256-column tile of
// W (whole tables, tile-aligned order). The fp32 W tile
// is copied into shared memory with 16-byte loads, rows padded to an odd
// number of words so that thread j reading column j hits distinct banks. Thread j
// keeps the R projections of column j in registers; a warp ballot per row turns the
// signs into bits and the bits are cut into K-bit codes.
// ---------------------------------------------------------------------------------
constexpr int kHashCols = 256;

// four consecutive fp32 W elements of a shared-memory row as two packed pairs
__device__ __forceinline__ void w4(const float* p, uint64_t& a, uint64_t& b) {
  a = pk2(p[0], p[1]);
  b = pk2(p[2], p[3]);
}

template <typename T, typename WT, int R>
__global__ void __launch_bounds__(kHashCols) k_hash_rows(HashRowsArgs a, int d, int K, int L, int tpt, int kltc) {
  extern __shared__ float xs[];  // [R][d] centered rows, then the W tile [256][wstride words]
  __shared__ uint32_t bits[R][kHashCols / 32 + 1];
  const int wstride = d * int(sizeof(WT)) / 4 + 1;  // words per W row (odd)
  uint32_t* wsm = reinterpret_cast<uint32_t*>(xs + R * d);
  const int g = blockIdx.z, n = blockIdx.y;
  const int r0 = blockIdx.x * R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (a.mark_hdr && tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
    if (a.mark_hdr->magic != kMagic) atomicOr(&a.mark_hdr->status, MP_STATUS_NOT_BUILT);
    else atomicMax(&a.mark_hdr->appended_end, a.mark_pos + 1);
  }
  // W tile: 256 consecutive rows of d elements, one contiguous block in global memory
  const WT* wsrc = static_cast<const WT*>(a.wt) + int64_t(g / a.groups_per_w) * a.w_stride +
                   int64_t(n) * kHashCols * d;
  {
    // 8 loads in flight per thread before their shared-memory stores
    constexpr int EPV = 16 / int(sizeof(WT));  // elements per 16-byte vector
    constexpr int B = 8;
    const int nvec = kHashCols * d / EPV;
    for (int c0 = 0; c0 < nvec; c0 += B * kHashCols) {
      uint4 v[B];
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int c = c0 + k * kHashCols + tid;
        if (c < nvec) v[k] = __ldg(reinterpret_cast<const uint4*>(wsrc) + c);
      }
#pragma unroll
      for (int k = 0; k < B; ++k) {
        const int c = c0 + k * kHashCols + tid;
        if (c < nvec) {
          const int e = c * EPV, row = e / d, wcol = (e - row * d) * int(sizeof(WT)) / 4;
          uint32_t* dst = wsm + row * wstride + wcol;
          dst[0] = v[k].x;
          dst[1] = v[k].y;
          dst[2] = v[k].z;
          dst[3] = v[k].w;
        }
      }
    }
  }
  const T* src = static_cast<const T*>(a.src) + int64_t(g) * a.src_gs;
  for (int i = tid; i < R * d; i += blockDim.x) {
    const int r = i / d, dim = i - r * d;
    float v = 0.f;
    if (r0 + r < a.rows) {
      v = to_f(src[int64_t(a.row0 + r0 + r) * a.src_rs + dim]);
      if (a.center) v -= a.center[(int64_t(g) * a.c_gs + int64_t((r0 + r) / a.c_div) * a.c_rs) * d + dim];
    }
    xs[i] = v;
  }
  __syncthreads();
  const WT* wrow = reinterpret_cast<const WT*>(wsm + tid * wstride);
  // even and odd dimensions accumulate in the two halves of a packed pair
  uint64_t acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0ull;
  for (int d0 = 0; d0 < d; d0 += 4) {
    uint64_t wa, wb;
    w4(wrow + d0, wa, wb);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(xs + r * d + d0);
      acc[r] = fma2(wa, pk2(x.x, x.y), acc[r]);
      acc[r] = fma2(wb, pk2(x.z, x.w), acc[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t m = __ballot_sync(0xffffffffu, lo2(acc[r]) + hi2(acc[r]) > 0.f);
    if (lane == 0) bits[r][warp] = m;
  }
  if (tid < R) bits[tid][kHashCols / 32] = 0u;
  __syncthreads();
  const uint32_t mask = (1u << K) - 1u;
  for (int i = tid; i < R * tpt; i += blockDim.x) {
    const int r = i / tpt, tl = i - r * tpt;
    const int t = n * tpt + tl;
    if (r0 + r >= a.rows || t >= L) continue;
    const int c0 = tl * K;
    const uint64_t v = uint64_t(bits[r][c0 >> 5]) | (uint64_t(bits[r][(c0 >> 5) + 1]) << 32);
    const uint32_t code = uint32_t(v >> (c0 & 31)) & mask;
    a.out[int64_t(g) * a.out_gs + int64_t(a.row0 + r0 + r) * a.out_rs + int64_t(t) * a.out_ts] = uint16_t(code);
  }
}

template <typename T, typename WT, int R>
static void launch_rows_tw(const Geometry& g, const HashRowsArgs& a, cudaStream_t st) {
  dim3 grid((a.rows + R - 1) / R, g.nt, a.groups);
  const int wstride = g.d * int(sizeof(WT)) / 4 + 1;
  const size_t smem = size_t(R) * g.d * sizeof(float) + size_t(kHashCols) * wstride * 4;
  cudaFuncSetAttribute(k_hash_rows<T, WT, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  k_hash_rows<T, WT, R><<<grid, kHashCols, smem, st>>>(a, g.d, g.K, g.L, g.tpt, g.kltc);
}

template <int R>
static void launch_rows_t(const Geometry& g, const HashRowsArgs& a, cudaStream_t st) {
  // the fp32 W, exact for any W (the tensor-core paths reach the same values through
  // W's three-term bf16 split)
  if (g.dtype == MP_DTYPE_BF16) launch_rows_tw<__nv_bfloat16, float, R>(g, a, st);
  else launch_rows_tw<float, float, R>(g, a, st);
}

// Row tile of 32, 16 or 8 rows: the largest that still gives two CTAs per SM.
cudaError_t launch_hash_rows(const Geometry& g, const HashRowsArgs& a, cudaStream_t st) {
  if (a.rows <= 0 || a.groups <= 0 || g.nt == 0) return cudaSuccess;
  const int64_t want = 2 * int64_t(device_sm_count());
  auto ctas = [&](int r) { return int64_t((a.rows + r - 1) / r) * g.nt * a.groups; };
  if (a.rows > 16 && ctas(32) >= want) launch_rows_t<32>(g, a, st);
  else if (a.rows > 8 && ctas(16) >= want) launch_rows_t<16>(g, a, st);
  else launch_rows_t<8>(g, a, st);
  return cudaGetLastError();
}

__global__ void k_mark_appended(DevHeader* hdr, int pos) {
  if (hdr->magic != kMagic) {
    atomicOr(&hdr->status, MP_STATUS_NOT_BUILT);
    return;
  }
  atomicMax(&hdr->appended_end, pos + 1);
}

cudaError_t launch_mark_appended(const Geometry&, int pos, const TablesPtrs& t, cudaStream_t st) {
  k_mark_appended<<<1, 1, 0, st>>>(t.hdr, pos);
  return cudaGetLastError();
}

}  // namespace mp
