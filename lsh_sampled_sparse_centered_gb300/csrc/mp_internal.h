// Internal declarations shared by the translation units of libmagicpig.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "magicpig.h"

namespace mp {

constexpr uint32_t kMagic = 0x4D504947u;  // "MPIG"
constexpr int kMaxK = 12;
constexpr int kMaxL = 1024;
constexpr int kMaxCapacity = 1 << 19;
constexpr int kMaxCapacityCounters = 196608;  // bucket walk with threshold > 2: one byte per token
constexpr int kCsrSeg = 32768;                // tokens per bucketed segment (16-bit local ids)
constexpr int kSplitsMax = 64;
constexpr uint32_t kExactFlag = 0x80000000u;

// First 256 bytes of the tables buffer.
struct DevHeader {
  uint32_t magic;
  int32_t n_prefill;     // tokens hashed at build time
  int32_t appended_end;  // one past the last token whose code is stored
  uint32_t status;       // MP_STATUS_* bits
  uint32_t w_terms3;     // nonzero: W is not bf16-representable, the tensor-core paths add
                         // the mid and lo bf16 terms of the split W = hi + mid + lo
  uint32_t lut_key;      // (K, L, threshold) the -log u table was written for (lut_key_of)
  int32_t pad[58];
};
static_assert(sizeof(DevHeader) == 256, "header size");

// Sizes derived from an mp_config.
struct Geometry {
  int layers, batch, kvh, qh, d, K, L, s, w, cap, dtype, w_per_layer, threshold;
  int no_center;  // 1: keys hashed uncentered (c = 0)
  int center_query;  // 1: queries hashed as q - c and p taken from cos(q - c, k - c)
  int group;    // q_heads / kv_heads
  int units;    // layers * batch * kv_heads
  int queries;  // layers * batch * q_heads
  int kl;       // K*L
  int nb;       // 2^K
  int tpt;      // tables per 256-column tensor-core tile: floor(256 / K)
  int nt;       // tensor-core column tiles: ceil(L / tpt)
  int kltc;     // nt * 256
  int match;    // MP_MATCH_CSR or MP_MATCH_SCAN (AUTO resolved)
  int cw;       // bit-plane words per table row: ceil(cap/32) rounded up to a multiple of 4
  int nseg;     // bucketed segments per table: ceil(cap / kCsrSeg)
  int parts;    // partial sums per unit for the center
  int n_w;      // number of W matrices
};

struct TablesPtrs {
  DevHeader* hdr;
  float* center;
  __nv_bfloat16* beta;   // [U][kltc][16]: -W^T c as three bf16 terms per column
  __nv_bfloat16* ones;   // [128][16]: (1, 1, 1, 0, ...) per row
  float* negbeta;        // [U][kltc]: -W^T c
  float* wt32;
  __nv_bfloat16* wt16;   // [n_w][3][kltc][d]: hi, mid, lo bf16 terms of W (W = hi + mid + lo)
  float* cparts;
  uint16_t* codes;
  uint16_t* off;   // [U][L][nseg][nb+1]
  uint16_t* ids;   // [U][L][cap]
  uint32_t* planes;
  float* lut;  // [kLutN + 1]: -log u on the cosine grid kLutLo + i (kLutHi - kLutLo) / kLutN
};

// -log u as a table over the cosine of the hashed query with k - c (written at build
// time, interpolated by the attention): kLutN intervals on [kLutLo, kLutHi]. Outside
// that range (u near 0 below it; the square-root edge of 1 - acos(c)/pi at c = 1 above
// it) the attention evaluates u directly.
constexpr int kLutN = 4096;
constexpr float kLutLo = -0.5f, kLutHi = 0.99f;
__host__ __device__ constexpr uint32_t lut_key_of(int K, int L, int threshold) {
  return 0x80000000u | uint32_t(K) | (uint32_t(L) << 8) | (uint32_t(threshold) << 20);
}

struct DecodePtrs {
  uint16_t* qcodes;
  int32_t* list_len;
  int32_t* sample_count;
  uint32_t* lists;
  float* partials;
  uint32_t* counters;
  uint32_t* sbits;
};

// Rows to hash: row r (0-based) of group g lives at
//   src + g*src_gs + (row0 + r)*src_rs          (elements)
// and is centered with  center + (g*c_gs + (r / c_div)*c_rs)*d  (if center != nullptr;
// c_div > 1 when several rows share a center, e.g. the query heads of a KV head).
// Codes go to out + g*out_gs + (row0 + r)*out_rs + t*out_ts.
struct HashRowsArgs {
  const void* src;
  int64_t src_gs, src_rs;
  int rows, groups, row0;
  const float* center;
  int64_t c_gs, c_rs;
  int c_div;
  const void* wt;         // [n_w][kltc][d], tile-aligned column order: bf16 (bf16 configs) or fp32
  int64_t w_stride;       // elements between consecutive W matrices (0: shared)
  int groups_per_w;       // group g uses W matrix g / groups_per_w
  uint16_t* out;
  int64_t out_gs, out_rs, out_ts;
  DevHeader* mark_hdr;    // appends: raise the appended end to mark_pos + 1 (nullptr: no-op)
  int mark_pos;
};

// Rows hashed on the tensor cores (bf16 rows and W, d = 64 or 128): `groups` groups of
// `rows` rows, row r of group g at x + (g * rows + r) * x_rs elements; group g uses W
// matrix g / groups_per_w (when W is per layer). negbeta != nullptr: row r of group g is
// centered by adding the -beta of unit (g * rows + r) / nb_div in the epilogue (appended
// keys: nb_div = 1; queries: nb_div = the query heads per KV head). mark != 0: the launch
// also raises the appended end to mark_pos + 1 (appends).
struct RowsHashTc {
  const __nv_bfloat16* x;
  int64_t x_rs;
  int rows, groups, groups_per_w;
  const __nv_bfloat16* wt16;
  const float* negbeta;  // [U][kltc]
  int nb_div;
  uint16_t* out;
  int64_t out_gs, out_rs, out_ts;
  DevHeader* hdr;
  int mark;
  int mark_pos;
};

// ---- launchers (each returns cudaError_t of the launch) ----
cudaError_t launch_hash_rows_tc(const Geometry& g, const RowsHashTc& h0, const RowsHashTc* h1, cudaStream_t st);
cudaError_t launch_prepare_w(const Geometry& g, const float* W, const TablesPtrs& t, cudaStream_t st);
cudaError_t launch_center(const Geometry& g, const void* keys, int n_prefill, const TablesPtrs& t,
                          cudaStream_t st);
cudaError_t launch_hash_rows(const Geometry& g, const HashRowsArgs& a, cudaStream_t st);
cudaError_t launch_hash_keys_tc(const Geometry& g, const void* keys, int n_prefill, const TablesPtrs& t,
                                cudaStream_t st, bool* used);
cudaError_t launch_csr_build(const Geometry& g, int n_prefill, const TablesPtrs& t, cudaStream_t st);
cudaError_t launch_mark_appended(const Geometry& g, int pos, const TablesPtrs& t, cudaStream_t st);
cudaError_t launch_logu_lut(const Geometry& g, const TablesPtrs& t, cudaStream_t st);
cudaError_t launch_match_csr(const Geometry& g, int n, const TablesPtrs& t, const DecodePtrs& dp,
                             cudaStream_t st);
cudaError_t launch_planes_build(const Geometry& g, int n_prefill, const TablesPtrs& t, cudaStream_t st);
cudaError_t launch_planes_append(const Geometry& g, int pos, const TablesPtrs& t, cudaStream_t st);
cudaError_t launch_scan(const Geometry& g, int n, const TablesPtrs& t, const DecodePtrs& dp, cudaStream_t st);
cudaError_t launch_compact(const Geometry& g, int n, const TablesPtrs& t, const DecodePtrs& dp, cudaStream_t st);
cudaError_t launch_attend(const Geometry& g, int n, int splits, const TablesPtrs& t, const void* keys,
                          const void* values, const void* q, float* out, const DecodePtrs& dp,
                          cudaStream_t st);

int device_sm_count();

// MP_CHECK=1 builds the bounds-checking library: kernels test every index that comes
// from data (codes, bucket offsets, list entries) against its buffer before using it,
// record a failure in the status word (MP_STATUS_BAD_INDEX) and skip that access. In
// the ordinary build the tests compile away.
#ifndef MP_CHECK
#define MP_CHECK 0
#endif

#ifdef __CUDACC__
// true when `ok`; in the bounds-checking build a false `ok` also sets MP_STATUS_BAD_INDEX
__device__ __forceinline__ bool in_range(bool ok, uint32_t* status) {
#if MP_CHECK
  if (!ok) atomicOr(status, MP_STATUS_BAD_INDEX);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Limit of every spin-wait on an mbarrier: the wait gives up after this long.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// Packed fp32 pairs (PTX .f32x2 arithmetic, sm_100 and later): one instruction works on
// two lanes of a 64-bit register, each half rounded exactly like the scalar
// instruction, so a pair op equals two scalar fmaf / __fadd_rn / __fmul_rn calls.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// two bf16 (low element first) as a packed fp32 pair: widening is exact
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
#endif

}  // namespace mp
