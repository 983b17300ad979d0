// SimHash of bf16 prefill keys on the 5th-generation tensor cores (tcgen05).
//
// For every unit (layer, sequence, KV head) the projections Y = K_u W (keys
// [n_prefill, d] times W [d, K*L]) run as a bf16 GEMM with fp32 accumulation in
// tensor memory; the epilogue subtracts beta = W^T c (centering, MagicPIG arXiv
// 2410.16179v2 §4.3 "Data pre-processing"), keeps the sign of each projection and
// packs K signs into each table's code (§2.2 SimHash, §4.3 "Hash function selection").
// bf16 x bf16 products are exact in fp32, so with bf16-representable W the only
// rounding is the fp32 accumulation.
//
// Structure: persistent CTAs, one per SM, each walking 128-key tiles. Warp 0 streams
// key tiles (A, 128 x d) and W column tiles (B, 256 x d) with TMA into 128B-swizzled
// shared memory; warp 1 issues tcgen05.mma (M=128, N=256, K=16 steps) into one of two
// 256-column fp32 accumulators in tensor memory; warps 2..9 read the accumulator with
// tcgen05.ld, form the codes and store them. W columns are laid out so that every
// 256-column tile holds floor(256/K) whole tables: no code straddles two tiles.
// All waits are bounded: on expiry the kernel records MP_STATUS_WAIT_TIMEOUT and stops.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mp_internal.h"

namespace mp {

namespace {

constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kThreads = 320;  // 10 warps
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(saddr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after kWaitLimitNs (setting *abort) or as soon as another
// role has given up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort = 1u;
        return false;
      }
    }
  }
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(saddr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(saddr(bar))
      : "memory");
}
// K-major operand in 128B-swizzled rows of 64 bf16 (the TMA SWIZZLE_128B layout):
// 8-row atoms 1024 B apart (SBO), leading offset unused, descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= uint64_t((addr & 0x3FFFFu) >> 4);
  d |= uint64_t(1) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
               : "memory");
}
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int D>
struct GemmSmem {
  static constexpr int kSub = D / 64;  // 64-element (128 B) swizzle columns per row
  // A: [2 slots][kSub][128 rows][64], B: [2 slots][kSub][256 rows][64]; every sub-tile 1024-aligned
  __nv_bfloat16 a[2][kSub][kTileM * 64];
  __nv_bfloat16 b[2][kSub][kTileN * 64];
  uint64_t a_full[2], a_empty[2], b_full[2], b_empty[2], acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  uint32_t abort;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    k_hash_keys_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmW,
                   const float* __restrict__ beta, uint16_t* __restrict__ codes, DevHeader* hdr, int units,
                   int units_per_w, int w_per_layer, int cap, int n0, int L, int K, int tpt, int nt) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  // align the dynamic shared memory to 1024 B for the swizzle atoms
  const uint32_t base = saddr(smraw);
  GemmSmem<D>& S = *reinterpret_cast<GemmSmem<D>*>(smraw + ((1024 - (base & 1023)) & 1023));
  constexpr int kSub = GemmSmem<D>::kSub;
  constexpr uint32_t kABytes = kTileM * D * 2;
  constexpr uint32_t kBBytes = kTileN * D * 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (n0 + kTileM - 1) / kTileM;
  const int items = units * mt;
  volatile uint32_t* abort = &S.abort;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.a_full[i], 1);
      mbar_init(&S.a_empty[i], 1);
      mbar_init(&S.b_full[i], 1);
      mbar_init(&S.b_empty[i], 1);
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_empty[i], kEpiWarps);
    }
    S.abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&S.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t bc = 0;
      int li = 0;
      for (int item = blockIdx.x; item < items && !*abort; item += gridDim.x, ++li) {
        const int u = item / mt, m0 = (item - u * mt) * kTileM;
        const int as = li & 1;
        if (!mbar_wait(&S.a_empty[as], ((li >> 1) & 1) ^ 1, abort)) break;
        mbar_expect_tx(&S.a_full[as], kABytes);
        for (int s = 0; s < kSub; ++s) tma_load_2d(&S.a[as][s][0], &tmK, s * 64, u * cap + m0, &S.a_full[as]);
        const int wrow = (w_per_layer ? (u / units_per_w) : 0) * nt * kTileN;
        bool ok = true;
        for (int n = 0; n < nt; ++n, ++bc) {
          const int bs = bc & 1;
          if (!mbar_wait(&S.b_empty[bs], ((bc >> 1) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&S.b_full[bs], kBBytes);
          for (int s = 0; s < kSub; ++s)
            tma_load_2d(&S.b[bs][s][0], &tmW, s * 64, wrow + n * kTileN, &S.b_full[bs]);
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kTileN >> 3) << 17) |
                             (uint32_t(kTileM >> 4) << 24);
      uint32_t bc = 0, ac = 0;
      int li = 0;
      for (int item = blockIdx.x; item < items && !*abort; item += gridDim.x, ++li) {
        const int as = li & 1;
        if (!mbar_wait(&S.a_full[as], (li >> 1) & 1, abort)) break;
        fence_after();
        bool ok = true;
        for (int n = 0; n < nt; ++n, ++bc, ++ac) {
          const int bs = bc & 1, cs = ac & 1;
          if (!mbar_wait(&S.b_full[bs], (bc >> 1) & 1, abort) ||
              !mbar_wait(&S.acc_empty[cs], ((ac >> 1) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t d_tmem = tmem + uint32_t(cs * kTileN);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int s = kk >> 2, off = (kk & 3) * 32;
            const uint64_t da = sw128_desc(saddr(&S.a[as][s][0]) + off);
            const uint64_t db = sw128_desc(saddr(&S.b[bs][s][0]) + off);
            mma_bf16(d_tmem, da, db, idesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&S.b_empty[bs]);
          mma_commit(&S.acc_full[cs]);
        }
        if (!ok) break;
        mma_commit(&S.a_empty[as]);
      }
    }
  } else {
    // ---------------- epilogue: 8 warps, 2 per TMEM lane quarter ----------------
    const int e = warp - 2;
    const int quarter = warp & 3;      // TMEM lanes 32*quarter .. +31 are reachable by this warp
    const int half = e >> 2;           // which half of the tile's tables
    const int t_split = (tpt + 1) >> 1;
    const int tl0 = half ? t_split : 0, tl1 = half ? tpt : t_split;
    const uint32_t mask = (K >= 32) ? 0xffffffffu : ((1u << K) - 1u);
    uint32_t ac = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
      const int u = item / mt, m0 = (item - u * mt) * kTileM;
      const int row = m0 + quarter * 32 + lane;
      const bool store = row < n0;
      const float* bu = beta + int64_t(u) * nt * kTileN;
      bool ok = true;
      for (int n = 0; n < nt; ++n, ++ac) {
        const int cs = ac & 1;
        // warp-uniform outcome: the tcgen05.ld below must be executed by all 32 lanes
        if (!__all_sync(0xffffffffu, mbar_wait(&S.acc_full[cs], (ac >> 1) & 1, abort))) {
          *abort = 1u;
          ok = false;
          break;
        }
        fence_after();
        const int tfirst = n * tpt + tl0;
        const int tlast = min(n * tpt + tl1, L);  // exclusive
        if (tfirst < tlast) {
          const int c0 = tl0 * K, c1 = (tlast - n * tpt) * K;  // column range within the tile
          const uint32_t tbase = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(cs * kTileN);
          uint64_t buf = 0;
          int have = 0, t = tfirst;
          for (int ch = c0 >> 5; ch * 32 < c1; ++ch) {
            uint32_t r[32];
            tmem_ld32(tbase + uint32_t(ch * 32), r);
            const float* bb = bu + n * kTileN + ch * 32;
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 b4 = __ldg(reinterpret_cast<const float4*>(bb + j));
              // sign bit of (beta - y) is set iff y - beta > 0
              word = __funnelshift_l(__float_as_uint(b4.x - __uint_as_float(r[j + 0])), word, 1);
              word = __funnelshift_l(__float_as_uint(b4.y - __uint_as_float(r[j + 1])), word, 1);
              word = __funnelshift_l(__float_as_uint(b4.z - __uint_as_float(r[j + 2])), word, 1);
              word = __funnelshift_l(__float_as_uint(b4.w - __uint_as_float(r[j + 3])), word, 1);
            }
            word = __brev(word);  // bit j <-> column ch*32 + j
            const int lo = max(c0, ch * 32);
            const int sh = lo - ch * 32;
            buf |= uint64_t(word >> sh) << have;
            have += 32 - sh;
            while (have >= K && t < tlast) {
              if (store) codes[(int64_t(u) * L + t) * cap + row] = uint16_t(uint32_t(buf) & mask);
              buf >>= K;
              have -= K;
              ++t;
            }
          }
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.acc_empty[cs]);
      }
      if (!ok) break;
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (threadIdx.x == 0 && S.abort) atomicOr(&hdr->status, MP_STATUS_WAIT_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc(const Geometry& g, const void* keys, int n_prefill, const TablesPtrs& t, cudaStream_t st) {
  CUtensorMap mk, mw;
  if (!make_map(&mk, keys, uint64_t(g.d), uint64_t(g.units) * g.cap, kTileM)) return cudaErrorInvalidValue;
  if (!make_map(&mw, t.wt16, uint64_t(g.d), uint64_t(g.n_w) * g.kltc, kTileN)) return cudaErrorInvalidValue;
  const size_t smem = sizeof(GemmSmem<D>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_hash_keys_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const int mt = (n_prefill + kTileM - 1) / kTileM;
  const int items = g.units * mt;
  const int grid = std::min(items, device_sm_count());
  k_hash_keys_tc<D><<<grid, kThreads, smem, st>>>(mk, mw, t.beta, t.codes, t.hdr, g.units, g.batch * g.kvh,
                                                  g.w_per_layer, g.cap, n_prefill, g.L, g.K, g.tpt, g.nt);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hash_keys_tc(const Geometry& g, const void* keys, int n_prefill, const TablesPtrs& t,
                                cudaStream_t st, bool* used) {
  *used = false;
  if (g.dtype != MP_DTYPE_BF16 || g.K == 0 || n_prefill < 1 || !t.wt16) return cudaSuccess;
  cudaError_t e = (g.d == 128) ? launch_tc<128>(g, keys, n_prefill, t, st) : launch_tc<64>(g, keys, n_prefill, t, st);
  if (e == cudaSuccess) *used = true;
  return e;
}

}  // namespace mp
