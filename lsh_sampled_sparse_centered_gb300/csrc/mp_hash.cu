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
// W [n_w][d][K*L] fp32  ->  wt32 [n_w][KLp][d] fp32 (column j = t*K + b, zero padded)
//                       ->  wt16 [n_w][TC][d] bf16 in tensor-core column order: tile
//                           n holds tables n*tpt .. n*tpt+tpt-1, column n*256 + i*K + b
//                           is bit b of the tile's i-th table; the rest is zero.
// ---------------------------------------------------------------------------------
__global__ void k_prepare_w(const float* __restrict__ W, float* __restrict__ wt32,
                            __nv_bfloat16* __restrict__ wt16, int d, int K, int L, int kl, int klp, int tpt,
                            int kltc, uint32_t* status) {
  // tile transpose: 32 columns x 32 d-rows per block
  __shared__ float tile[32][33];
  const int m = blockIdx.z;
  const int j0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int dd = d0 + r, j = j0 + tx;
    tile[r][tx] = (dd < d && j < kl) ? W[(int64_t(m) * d + dd) * kl + j] : 0.f;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int j = j0 + r, dd = d0 + tx;
    if (j < klp && dd < d) wt32[(int64_t(m) * klp + j) * d + dd] = tile[tx][r];
  }
  if (!wt16) return;
  // tensor-core order: this block also writes TC columns jc in [j0, j0 + 32)
  bool inexact = false;
  for (int r = ty; r < 32; r += 8) {
    const int jc = j0 + r, dd = d0 + tx;
    if (jc >= kltc || dd >= d) continue;
    const int n = jc >> 8, within = jc & 255;
    const int i = within / K, b = within - i * K;
    const int t = n * tpt + i;
    float v = 0.f;
    if (i < tpt && t < L) v = W[(int64_t(m) * d + dd) * kl + t * K + b];
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    wt16[(int64_t(m) * kltc + jc) * d + dd] = h;
    inexact |= (__bfloat162float(h) != v);
  }
  if (inexact) atomicOr(status, MP_STATUS_W_NOT_BF16);
}

cudaError_t launch_prepare_w(const Geometry& g, const float* W, const TablesPtrs& t, cudaStream_t st) {
  const int cols = max(g.klp, g.kltc);
  dim3 grid((cols + 31) / 32, (g.d + 31) / 32, g.n_w), block(32, 8);
  k_prepare_w<<<grid, block, 0, st>>>(W, t.wt32, t.wt16, g.d, g.K, g.L, g.kl, g.klp, g.tpt, g.kltc,
                                      &t.hdr->status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// centering: per unit, partial sums over `parts` token ranges, then the mean and
// beta = W^T c. Deterministic (fixed summation order).
// ---------------------------------------------------------------------------------
template <typename T>
__global__ void k_center_parts(const T* __restrict__ keys, float* __restrict__ cparts, int d, int cap,
                               int lo, int hi, int parts) {
  extern __shared__ float red[];  // [blockDim.x]
  const int u = blockIdx.y, part = blockIdx.x;
  const int span = (hi - lo + parts - 1) / parts;
  const int t0 = lo + part * span;
  const int t1 = min(hi, t0 + span);
  const int dim = threadIdx.x % d, phase = threadIdx.x / d, nph = blockDim.x / d;
  const T* base = keys + int64_t(u) * cap * d;
  float acc = 0.f;
  for (int t = t0 + phase; t < t1; t += nph) acc += to_f(base[int64_t(t) * d + dim]);
  red[threadIdx.x] = acc;
  __syncthreads();
  if (phase == 0) {
    float s = 0.f;
    for (int p = 0; p < nph; ++p) s += red[p * d + dim];
    cparts[(int64_t(u) * parts + part) * d + dim] = s;
  }
}

__global__ void k_center_final(const float* __restrict__ cparts, float* __restrict__ center,
                               float* __restrict__ beta, const __nv_bfloat16* __restrict__ wt16, int d,
                               int kltc, int parts, int count, int units_per_w, int64_t w_stride,
                               DevHeader* hdr, int n_prefill) {
  extern __shared__ float c[];  // [d]
  const int u = blockIdx.x;
  for (int dim = threadIdx.x; dim < d; dim += blockDim.x) {
    float s = 0.f;
    for (int p = 0; p < parts; ++p) s += cparts[(int64_t(u) * parts + p) * d + dim];
    const float v = count > 0 ? s / float(count) : 0.f;
    c[dim] = v;
    center[int64_t(u) * d + dim] = v;
  }
  __syncthreads();
  // beta = W^T c in tensor-core column order (used by the tensor-core hash)
  if (wt16) {
    const __nv_bfloat16* w = wt16 + int64_t(u / units_per_w) * w_stride;
    for (int j = threadIdx.x; j < kltc; j += blockDim.x) {
      const __nv_bfloat16* row = w + int64_t(j) * d;
      float s = 0.f;
      for (int dim = 0; dim < d; ++dim) s = fmaf(__bfloat162float(row[dim]), c[dim], s);
      beta[int64_t(u) * kltc + j] = s;
    }
  }
  if (u == 0 && threadIdx.x == 0) {
    hdr->n_prefill = n_prefill;
    hdr->appended_end = n_prefill;
    __threadfence();
    hdr->magic = kMagic;
  }
}

cudaError_t launch_center(const Geometry& g, const void* keys, int n_prefill, const TablesPtrs& t,
                          cudaStream_t st) {
  const int lo = min(g.s, n_prefill), hi = n_prefill;
  const int threads = 256;
  dim3 grid(g.parts, g.units);
  if (g.dtype == MP_DTYPE_BF16)
    k_center_parts<__nv_bfloat16><<<grid, threads, threads * sizeof(float), st>>>(
        static_cast<const __nv_bfloat16*>(keys), t.cparts, g.d, g.cap, lo, hi, g.parts);
  else
    k_center_parts<float><<<grid, threads, threads * sizeof(float), st>>>(
        static_cast<const float*>(keys), t.cparts, g.d, g.cap, lo, hi, g.parts);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t w_stride = g.w_per_layer ? int64_t(g.kltc) * g.d : 0;
  k_center_final<<<g.units, 256, g.d * sizeof(float), st>>>(t.cparts, t.center, t.beta, t.wt16, g.d,
                                                          g.kltc, g.parts, hi - lo, g.batch * g.kvh,
                                                          w_stride, t.hdr, n_prefill);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// SimHash of rows on CUDA cores. One warp = 32 rows x one table; one thread holds
// the K projections of its (row, table) and packs them into the code directly.
// Rows are staged (centered, fp32) in shared memory, the block's W columns too.
// ---------------------------------------------------------------------------------
constexpr int kHashRows = 32;
constexpr int kHashTables = 8;  // tables (warps) per block

template <typename T>
__global__ void __launch_bounds__(256) k_hash_rows(HashRowsArgs a, int d, int K, int L, int klp) {
  extern __shared__ float sm[];
  float* xs = sm;                              // [32][d+1]
  float* ws = sm + kHashRows * (d + 1);        // [kHashTables*K][d]
  const int g = blockIdx.z;
  const int r0 = blockIdx.x * kHashRows;
  const int t0 = blockIdx.y * kHashTables;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* src = static_cast<const T*>(a.src) + int64_t(g) * a.src_gs;
  // stage rows
  for (int i = threadIdx.x; i < kHashRows * d; i += blockDim.x) {
    const int r = i / d, dim = i % d;
    float v = 0.f;
    if (r0 + r < a.rows) {
      v = to_f(src[int64_t(a.row0 + r0 + r) * a.src_rs + dim]);
      if (a.center) v -= a.center[(int64_t(g) * a.c_gs + int64_t(r0 + r) * a.c_rs) * d + dim];
    }
    xs[r * (d + 1) + dim] = v;
  }
  // stage W columns of this block's tables
  const float* w = a.wt32 + int64_t(g / a.groups_per_w) * a.w_stride;
  const int ncol = kHashTables * K;
  for (int i = threadIdx.x; i < ncol * d; i += blockDim.x) {
    const int c = i / d, dim = i % d;
    const int j = t0 * K + c;
    ws[i] = (j < klp) ? w[int64_t(j) * d + dim] : 0.f;
  }
  __syncthreads();
  const int t = t0 + warp;
  const int r = r0 + lane;
  if (t >= L || r >= a.rows) return;
  float acc[kMaxK];
#pragma unroll
  for (int b = 0; b < kMaxK; ++b) acc[b] = 0.f;
  const float* x = xs + lane * (d + 1);
  const float* wc = ws + warp * K * d;
  for (int dim = 0; dim < d; ++dim) {
    const float xv = x[dim];
#pragma unroll
    for (int b = 0; b < kMaxK; ++b)
      if (b < K) acc[b] = fmaf(xv, wc[b * d + dim], acc[b]);
  }
  uint32_t code = 0;
#pragma unroll
  for (int b = 0; b < kMaxK; ++b)
    if (b < K && acc[b] > 0.f) code |= 1u << b;
  a.out[int64_t(g) * a.out_gs + int64_t(a.row0 + r) * a.out_rs + int64_t(t) * a.out_ts] = uint16_t(code);
}

cudaError_t launch_hash_rows(const Geometry& g, const HashRowsArgs& a, cudaStream_t st) {
  if (a.rows <= 0 || a.groups <= 0) return cudaSuccess;
  dim3 grid((a.rows + kHashRows - 1) / kHashRows, (g.L + kHashTables - 1) / kHashTables, a.groups);
  const size_t smem = (size_t(kHashRows) * (g.d + 1) + size_t(kHashTables) * g.K * g.d) * sizeof(float);
  if (g.dtype == MP_DTYPE_BF16) {
    cudaFuncSetAttribute(k_hash_rows<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    k_hash_rows<__nv_bfloat16><<<grid, 256, smem, st>>>(a, g.d, g.K, g.L, g.klp);
  } else {
    cudaFuncSetAttribute(k_hash_rows<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    k_hash_rows<float><<<grid, 256, smem, st>>>(a, g.d, g.K, g.L, g.klp);
  }
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
