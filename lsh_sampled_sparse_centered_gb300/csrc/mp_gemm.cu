// SimHash of bf16 prefill keys on the 5th-generation tensor cores (tcgen05).
//
// For every unit (layer, sequence, KV head) the centered projections
// Y = (K_u - c) W = K_u W - beta (keys [n_prefill, d], W [d, K*L], beta = W^T c;
// centering: MagicPIG arXiv 2410.16179v2 §4.3 "Data pre-processing") run as a bf16
// GEMM with fp32 accumulation in tensor memory. -beta enters the accumulator through
// one extra K step: a tile of rows (1, 1, 1, 0, ...) times the per-unit split of -beta
// into three bf16 terms (exact). The epilogue keeps the sign of each projection and
// packs K signs into each table's code (§2.2 SimHash, §4.3 "Hash function selection").
// bf16 x bf16 products are exact in fp32, so with bf16-representable W the only
// rounding is the fp32 accumulation; a W that bf16 cannot hold enters as its exact
// split hi + mid + lo, one pass of K steps per term into the same accumulator.
//
// The same file holds the swap-AB kernel that hashes the few rows of a decode step
// (queries, appended keys): there the W columns are the M dimension, so a warp ballot
// over tensor-memory lanes gives a row's sign bits directly.
//
// Structure: persistent CTAs, one per SM, each walking 128-key tiles. Warp 0 streams
// key tiles (A, 128 x d) and W column tiles (B, 256 x d) with TMA into 128B-swizzled
// shared memory; warp 1 issues tcgen05.mma (M=128, N=256, K=16 steps) into one of two
// 256-column fp32 accumulators in tensor memory; warps 2..13 (three per tensor-memory
// lane quarter, each owning a part of the tile's tables) read the accumulator with
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
constexpr int kEpiWarps = 12;  // kParts per TMEM lane quarter
constexpr int kParts = kEpiWarps / 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
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
// try_wait with a suspend-time hint (ns): a waiting thread sleeps until the phase
// completes or the hint expires instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(saddr(bar)), "r"(parity), "r"(1000000u)
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
// K-major operand of one K step (16 bf16 = 32 B per row) in the TMA SWIZZLE_32B layout:
// 8-row atoms 256 B apart.
__device__ __forceinline__ uint64_t sw32_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= uint64_t((addr & 0x3FFFFu) >> 4);
  d |= uint64_t(1) << 16;
  d |= uint64_t(256 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(6) << 61;
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
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Sign bits of 32 accumulator columns: bit j <-> column j is 1 iff y_j >= +0, i.e.
// y - beta > 0 up to an exact zero, which lies in the near-tie band. Four independent
// shift chains (columns j, j+8, j+16, j+24) keep the dependency chains short.
__device__ __forceinline__ uint32_t sign_word(const uint32_t (&r)[32]) {
  uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w0 = __funnelshift_l(r[i], w0, 1);
    w1 = __funnelshift_l(r[8 + i], w1, 1);
    w2 = __funnelshift_l(r[16 + i], w2, 1);
    w3 = __funnelshift_l(r[24 + i], w3, 1);
  }
  // w_k holds the sign bits of columns 8k..8k+7, column 8k at bit 7
  return ~__brev((w0 << 24) | (w1 << 16) | (w2 << 8) | w3);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// sign bits of 16 accumulator columns in bits 0..15 (as sign_word)
__device__ __forceinline__ uint32_t sign_word16(const uint32_t (&r)[16]) {
  uint32_t w0 = 0, w1 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w0 = __funnelshift_l(r[i], w0, 1);
    w1 = __funnelshift_l(r[8 + i], w1, 1);
  }
  return ~__brev((w0 << 24) | (w1 << 16)) & 0xffffu;
}

// Codes of one part of a 256-column tile with K known at compile time. The tile's used
// 32-column chunks are split evenly over the kParts warps of a lane quarter; a part
// cuts the codes of the tables that start in its chunks, and when its last table runs
// into the next part's first chunk it also reads that chunk's first 16 columns. The
// column, word and shift of every code are constants, so cutting a code is one or two
// shifts.
template <int KC, int PART>
__device__ __forceinline__ void epi_tile_k(uint32_t tbase, uint16_t* codes, int64_t u, int L, int cap, int row,
                                           bool store, int n) {
  constexpr int TPT = 256 / KC;
  constexpr int NCT = (TPT * KC + 31) / 32;  // chunks holding whole tables
  constexpr int CH0 = PART * NCT / kParts, CH1 = (PART + 1) * NCT / kParts;  // this part's chunks
  constexpr int TL0 = (CH0 * 32 + KC - 1) / KC;
  constexpr int TL1c = (CH1 * 32 + KC - 1) / KC;
  constexpr int TL1 = TL1c < TPT ? TL1c : TPT;  // tables starting in [CH0, CH1)
  if constexpr (TL0 < TL1) {
    constexpr int NCH = CH1 - CH0;
    constexpr bool NEXT = (TL1 - 1) * KC + KC > CH1 * 32;  // the last table reaches chunk CH1
    static_assert(!NEXT || (TL1 - 1) * KC + KC <= CH1 * 32 + 16, "a code reaches at most 16 columns on");
    uint32_t words[NCH + 1];
    // every load of the part in flight before one wait (at most three chunks and a half)
    static_assert(NCH <= 3, "at most three chunks per part");
    uint32_t r0[32], r1[32], r2[32], rx[16];
    tmem_ld32(tbase + uint32_t(CH0 * 32), r0);
    if constexpr (NCH > 1) tmem_ld32(tbase + uint32_t((CH0 + 1) * 32), r1);
    if constexpr (NCH > 2) tmem_ld32(tbase + uint32_t((CH0 + 2) * 32), r2);
    if constexpr (NEXT) tmem_ld16(tbase + uint32_t(CH1 * 32), rx);
    tmem_wait_ld();
    words[0] = sign_word(r0);
    if constexpr (NCH > 1) words[1] = sign_word(r1);
    if constexpr (NCH > 2) words[2] = sign_word(r2);
    words[NCH] = NEXT ? sign_word16(rx) : 0u;
    constexpr uint32_t MASK = (1u << KC) - 1u;
#pragma unroll
    for (int tl = TL0; tl < TL1; ++tl) {
      const int c = tl * KC, wi = c / 32 - CH0, sh = c % 32;
      uint32_t code = words[wi] >> sh;
      if (sh + KC > 32) code |= words[wi + 1] << (32 - sh);
      const int t = n * TPT + tl;
      if (store && t < L) codes[(u * L + t) * cap + row] = uint16_t(code & MASK);
    }
  }
}

template <int D>
struct GemmSmem {
  static constexpr int kSub = D / 64;  // 64-element (128 B) swizzle columns per row
  // A: [2 slots][kSub][128 rows][64], B: [2 slots][kSub][256 rows][64]; every sub-tile 1024-aligned
  __nv_bfloat16 a[2][kSub][kTileM * 64];
  __nv_bfloat16 b[2][kSub][kTileN * 64];
  __nv_bfloat16 b1[2][kTileN * 16];  // -beta split of the stage's columns (32-byte swizzle)
  __nv_bfloat16 a1[kTileM * 16];     // rows (1, 1, 1, 0, ...) (32-byte swizzle)
  uint64_t a_full[2], a_empty[2], b_full[2], b_empty[2], acc_full[2], acc_empty[2], ones_full;
  uint32_t tmem_base;
  uint32_t abort;
};

template <int D, int KT>
__global__ void __launch_bounds__(kThreads, 1)
    k_hash_keys_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmBias, const __grid_constant__ CUtensorMap tmOnes,
                   uint16_t* __restrict__ codes, DevHeader* hdr, int units,
                   int units_per_w, int w_per_layer, int cap, int n0, int L, int K, int tpt, int nt, int kltc) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  // align the dynamic shared memory to 1024 B for the swizzle atoms
  const uint32_t base = saddr(smraw);
  GemmSmem<D>& S = *reinterpret_cast<GemmSmem<D>*>(smraw + ((1024 - (base & 1023)) & 1023));
  constexpr int kSub = GemmSmem<D>::kSub;
  constexpr uint32_t kABytes = kTileM * D * 2;
  constexpr uint32_t kWBytes = kTileN * D * 2;                    // one bf16 term of the W columns
  constexpr uint32_t kBBytes = kWBytes + kTileN * 16 * 2;         // + their -beta split (first term)
  constexpr uint32_t kOnesBytes = kTileM * 16 * 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (n0 + kTileM - 1) / kTileM;
  // bf16 terms of W to accumulate: 1, or 3 (hi, mid, lo) when W is not bf16-representable
  const int terms = hdr->w_terms3 ? 3 : 1;
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
    mbar_init(&S.ones_full, 1);
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
      mbar_expect_tx(&S.ones_full, kOnesBytes);
      tma_load_2d(&S.a1[0], &tmOnes, 0, 0, &S.ones_full);
      uint32_t bc = 0;
      int li = 0;
      for (int item = blockIdx.x; item < items && !*abort; item += gridDim.x, ++li) {
        const int u = item / mt, m0 = (item - u * mt) * kTileM;
        const int as = li & 1;
        if (!mbar_wait(&S.a_empty[as], ((li >> 1) & 1) ^ 1, abort)) break;
        mbar_expect_tx(&S.a_full[as], kABytes);
        for (int s = 0; s < kSub; ++s) tma_load_2d(&S.a[as][s][0], &tmK, s * 64, u * cap + m0, &S.a_full[as]);
        const int wrow = (w_per_layer ? (u / units_per_w) : 0) * 3 * kltc;  // [n_w][3][kltc] rows
        bool ok = true;
        for (int n = 0; n < nt && ok; ++n) {
          for (int j = 0; j < terms; ++j, ++bc) {
            const int bs = bc & 1;
            if (!mbar_wait(&S.b_empty[bs], ((bc >> 1) & 1) ^ 1, abort)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&S.b_full[bs], j == 0 ? kBBytes : kWBytes);
            for (int s = 0; s < kSub; ++s)
              tma_load_2d(&S.b[bs][s][0], &tmW, s * 64, wrow + j * kltc + n * kTileN, &S.b_full[bs]);
            if (j == 0) tma_load_2d(&S.b1[bs][0], &tmBias, 0, u * kltc + n * kTileN, &S.b_full[bs]);
          }
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
      const bool have_ones = mbar_wait(&S.ones_full, 0, abort);
      for (int item = blockIdx.x; have_ones && item < items && !*abort; item += gridDim.x, ++li) {
        const int as = li & 1;
        if (!mbar_wait(&S.a_full[as], (li >> 1) & 1, abort)) break;
        fence_after();
        bool ok = true;
        for (int n = 0; n < nt && ok; ++n, ++ac) {
          const int cs = ac & 1;
          if (!mbar_wait(&S.acc_empty[cs], ((ac >> 1) & 1) ^ 1, abort)) {
            ok = false;
            break;
          }
          const uint32_t d_tmem = tmem + uint32_t(cs * kTileN);
          for (int j = 0; j < terms; ++j, ++bc) {
            const int bs = bc & 1;
            if (!mbar_wait(&S.b_full[bs], (bc >> 1) & 1, abort)) {
              ok = false;
              break;
            }
            fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int s = kk >> 2, off = (kk & 3) * 32;
              const uint64_t da = sw128_desc(saddr(&S.a[as][s][0]) + off);
              const uint64_t db = sw128_desc(saddr(&S.b[bs][s][0]) + off);
              mma_bf16(d_tmem, da, db, idesc, (j > 0 || kk > 0) ? 1u : 0u);
            }
            // extra K step (with the first term): ones x (-beta split) adds -W^T c to every row
            if (j == 0) mma_bf16(d_tmem, sw32_desc(saddr(&S.a1[0])), sw32_desc(saddr(&S.b1[bs][0])), idesc, 1u);
            mma_commit(&S.b_empty[bs]);
          }
          if (!ok) break;
          mma_commit(&S.acc_full[cs]);
        }
        if (!ok) break;
        mma_commit(&S.a_empty[as]);
      }
    }
  } else {
    // ---------------- epilogue: 12 warps, 3 per TMEM lane quarter ----------------
    const int e = warp - 2;
    const int quarter = warp & 3;      // TMEM lanes 32*quarter .. +31 are reachable by this warp
    const int part = e >> 2;           // which part of the tile's tables
    const int t_per = (tpt + kParts - 1) / kParts;
    const int tl0 = min(tpt, part * t_per), tl1 = min(tpt, tl0 + t_per);
    const uint32_t mask = (1u << K) - 1u;
    uint32_t ac = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
      const int u = item / mt, m0 = (item - u * mt) * kTileM;
      const int row = m0 + quarter * 32 + lane;
      const bool store = row < n0;
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
        if constexpr (KT > 0) {
          const uint32_t tbase = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(cs * kTileN);
          if (part == 0) epi_tile_k<KT, 0>(tbase, codes, u, L, cap, row, store, n);
          else if (kParts > 1 && part == 1) epi_tile_k<KT, (kParts > 1 ? 1 : 0)>(tbase, codes, u, L, cap, row, store, n);
          else if (kParts > 2 && part == 2) epi_tile_k<KT, (kParts > 2 ? 2 : 0)>(tbase, codes, u, L, cap, row, store, n);
          else if (kParts > 3) epi_tile_k<KT, (kParts > 3 ? 3 : 0)>(tbase, codes, u, L, cap, row, store, n);
        } else if (tfirst < tlast) {
          const int c0 = tl0 * K, c1 = (tlast - n * tpt) * K;  // column range within the tile
          const uint32_t tbase = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(cs * kTileN);
          const int ch_last = (c1 - 1) >> 5;
          uint64_t buf = 0;
          int have = 0, t = tfirst;
          auto consume = [&](const uint32_t (&r)[32], int ch) {
            const uint32_t word = sign_word(r);  // bit j <-> column ch*32 + j
            const int sh = max(c0, ch * 32) - ch * 32;
            buf |= uint64_t(word >> sh) << have;
            have += 32 - sh;
            while (have >= K && t < tlast) {
              if (store) codes[(int64_t(u) * L + t) * cap + row] = uint16_t(uint32_t(buf) & mask);
              buf >>= K;
              have -= K;
              ++t;
            }
          };
          for (int ch = c0 >> 5; ch <= ch_last; ch += 2) {
            uint32_t r0[32], r1[32];
            tmem_ld32(tbase + uint32_t(ch * 32), r0);
            if (ch + 1 <= ch_last) tmem_ld32(tbase + uint32_t((ch + 1) * 32), r1);
            tmem_wait_ld();
            consume(r0, ch);
            if (ch + 1 <= ch_last) consume(r1, ch + 1);
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

// ---------------------------------------------------------------------------------
// SimHash of a few rows per W matrix (decode queries, appended keys) on the tensor
// cores, with the roles of the operands swapped: A = 256 W columns (two M = 128
// halves), B = up to 256 rows (N), so that a tensor-memory lane is a W column and a
// ballot across a warp's lanes gives one row's sign bits of 32 columns at once.
// One launch hashes one or two row sets (a decode step's appended keys and its
// queries): per W group the sets are laid end to end, each rounded up to 32 rows, and
// row blocks of up to 256 of these rows share one load of a W tile. One CTA per (W
// group, 256-column tile, row block): thread 0 issues the TMA loads (the rows in boxes
// of 32, each from its set's tensor map) and the MMAs, then all 8 warps read the
// accumulator (warp w: half w / 4, lanes of quarter w % 4), add -beta where the set is
// centered, ballot the signs into a shared [row][32-column block] bitmap, and cut the
// codes.
// ---------------------------------------------------------------------------------
constexpr int kRowsWarps = 8;

template <int D>
struct RowsLayout {
  static constexpr int kSub = D / 64;
  static constexpr uint32_t kABytes = 256u * 64u * 2u;  // one 64-element slab of 256 W columns
  __host__ __device__ static constexpr uint32_t a_off(int s) { return uint32_t(s) * kABytes; }
  __host__ __device__ static constexpr uint32_t b_off(int s, int nr) {
    return uint32_t(kSub) * kABytes + uint32_t(s) * uint32_t(nr) * 128u;
  }
  __host__ __device__ static constexpr uint32_t bits_off(int nr) { return b_off(kSub, nr); }
  __host__ __device__ static constexpr uint32_t ctl_off(int nr) { return bits_off(nr) + uint32_t(nr) * 9u * 4u; }
  __host__ __device__ static constexpr uint32_t bytes(int nr) { return ctl_off(nr) + 64u; }  // 3 barriers + slots
};

// One set of rows hashed by k_hash_rows_tc.
struct RowSetTc {
  int rows;              // rows per group
  int nr32;              // rows rounded up to a multiple of 32
  const float* negbeta;  // -beta [U][kltc] added to row r of group g: unit (g * rows + r) / nb_div
                         // (nullptr: rows hashed as they are)
  int nb_div;
  uint16_t* out;
  int64_t out_gs, out_rs, out_ts;
};

struct RowsTcArgs {
  RowSetTc set[2];   // set[1].rows = 0 when one set is hashed
  int vrows;         // set[0].nr32 + set[1].nr32
  int nr;            // rows per CTA (multiple of 32, <= 256)
  int groups_per_w;  // group g uses W matrix g / groups_per_w
  int w_rows;        // W rows between consecutive W matrices (0: shared)
  int kltc;
  DevHeader* hdr;    // status word
  int mark;          // appends: raise the appended end to mark_pos + 1
  int mark_pos;
};

template <int D>
__global__ void __launch_bounds__(kRowsWarps * 32)
    k_hash_rows_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX0,
                   const __grid_constant__ CUtensorMap tmX1, const RowsTcArgs a, int L, int K, int tpt) {
  using Lay = RowsLayout<D>;
  constexpr int kSub = Lay::kSub;
  extern __shared__ __align__(1024) unsigned char smraw[];
  const uint32_t sbase = saddr(smraw);
  unsigned char* sm = smraw + ((1024 - (sbase & 1023)) & 1023);
  const int nr = a.nr;
  uint32_t* bits = reinterpret_cast<uint32_t*>(sm + Lay::bits_off(nr));  // [nr][9]
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + Lay::ctl_off(nr));
  uint64_t* accb = full + 1;
  uint64_t* mdone = full + 2;  // the MMAs of one W term have read the A tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 3);
  volatile uint32_t* abort = tmem_slot + 1;
  const int g = blockIdx.z, n = blockIdx.y, rb = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = rb * nr;                  // first row of this CTA in the group's row list
  const int nrow = min(nr, a.vrows - v0);  // rows of this CTA (multiple of 32)
  uint32_t ncols = 32;
  while (ncols < uint32_t(2 * nrow)) ncols <<= 1;
  // row v of the group's list belongs to set 1 from set[0].nr32 on
  const int split = a.set[0].nr32;

  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    mbar_init(accb, 1);
    mbar_init(mdone, 1);
    *abort = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (a.mark && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
      if (a.hdr->magic != kMagic) atomicOr(&a.hdr->status, MP_STATUS_NOT_BUILT);
      else atomicMax(&a.hdr->appended_end, a.mark_pos + 1);
    }
  }
  for (int i = threadIdx.x; i < nrow; i += blockDim.x) bits[i * 9 + 8] = 0u;
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    // W terms (1, or hi, mid, lo when W is not bf16-representable) go through the one A
    // buffer in turn; the rows are loaded with the first term
    const int terms = a.hdr->w_terms3 ? 3 : 1;
    const int wrow = (g / a.groups_per_w) * a.w_rows + n * 256;
    // D[col][row]: M = 128 W columns per half, N = nrow rows
    const uint32_t idesc =
        (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(nrow >> 3) << 17) | (uint32_t(128 >> 4) << 24);
    for (int j = 0; j < terms; ++j) {
      if (j > 0 && !mbar_wait(mdone, (j - 1) & 1, abort)) break;
      mbar_expect_tx(full, uint32_t(kSub) * (Lay::kABytes + (j == 0 ? uint32_t(nrow) * 128u : 0u)));
      for (int s = 0; s < kSub; ++s) {
        tma_load_2d(sm + Lay::a_off(s), &tmW, s * 64, wrow + j * a.kltc, full);
        if (j == 0)
          for (int b = 0; b < nrow / 32; ++b) {
            const int v = v0 + 32 * b, st = v >= split ? 1 : 0;
            const int xrow = g * a.set[st].rows + v - (st ? split : 0);
            tma_load_2d(sm + Lay::b_off(s, nr) + uint32_t(b) * 4096u, st ? &tmX1 : &tmX0, s * 64, xrow, full);
          }
      }
      if (!mbar_wait(full, j & 1, abort)) break;
      fence_after();
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int s = kk >> 2, off = (kk & 3) * 32;
          const uint64_t da = sw128_desc(saddr(sm + Lay::a_off(s)) + uint32_t(h) * 16384u + off);
          const uint64_t db = sw128_desc(saddr(sm + Lay::b_off(s, nr)) + off);
          mma_bf16(tmem + uint32_t(h * nrow), da, db, idesc, (j > 0 || kk > 0) ? 1u : 0u);
        }
      mma_commit(j + 1 < terms ? mdone : accb);
    }
  }
  __syncwarp();
  // epilogue: all warps. Each 32-row chunk lies in one set. Row j of chunk ch is row
  // local + j of its set, centered (if the set is) with unit (g * rows + local + j) /
  // nb_div, walked as a quotient and remainder so that no division runs per row; the
  // -beta of the first chunk is fetched before the wait for the accumulator.
  const int h = warp >> 2, quarter = warp & 3;
  const int col = h * 128 + quarter * 32 + lane;  // column within the 256-column tile
  float nb[32];
  auto fetch_nb = [&](int ch) {
    const int v = v0 + 32 * ch, st = v >= split ? 1 : 0;
    const RowSetTc& S = a.set[st];
    const int local = v - (st ? split : 0);
    const float* nbc = S.negbeta ? S.negbeta + int64_t(n) * 256 + col : nullptr;
    const int row_base = g * S.rows + local;
    int unit = row_base / S.nb_div, rem = row_base - unit * S.nb_div;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      nb[j] = (nbc && local + j < S.rows) ? __ldg(nbc + int64_t(unit) * a.kltc) : 0.f;
      if (++rem == S.nb_div) {
        rem = 0;
        ++unit;
      }
    }
  };
  fetch_nb(0);
  const bool ok = __all_sync(0xffffffffu, mbar_wait(accb, 0, abort));
  if (ok) {
    fence_after();
    for (int ch = 0; ch < nrow / 32; ++ch) {
      if (ch > 0) fetch_nb(ch);
      uint32_t r[32];
      tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + uint32_t(h * nrow + ch * 32), r);
      tmem_wait_ld();
      uint32_t mine = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t w = __ballot_sync(0xffffffffu, __uint_as_float(r[j]) + nb[j] > 0.f);
        if (lane == j) mine = w;
      }
      bits[(ch * 32 + lane) * 9 + h * 4 + quarter] = mine;
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
  }
  if (*abort) {
    if (threadIdx.x == 0) atomicOr(&a.hdr->status, MP_STATUS_WAIT_TIMEOUT);
    return;
  }
  const uint32_t mask = (1u << K) - 1u;
  for (int i = threadIdx.x; i < nrow * tpt; i += blockDim.x) {
    const int row = i / tpt, tl = i - row * tpt;
    const int t = n * tpt + tl;
    const int v = v0 + row, st = v >= split ? 1 : 0;
    const RowSetTc& S = a.set[st];
    const int local = v - (st ? split : 0);
    if (t >= L || local >= S.rows) continue;
    const int c0 = tl * K;
    const uint64_t w = uint64_t(bits[row * 9 + (c0 >> 5)]) | (uint64_t(bits[row * 9 + (c0 >> 5) + 1]) << 32);
    S.out[int64_t(g) * S.out_gs + int64_t(local) * S.out_rs + int64_t(t) * S.out_ts] =
        uint16_t(uint32_t(w >> (c0 & 31)) & mask);
  }
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

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
              CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// rows `row_bytes` apart (a multiple of 16)
bool make_map_strided(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                      uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int KT>
cudaError_t launch_tc(const Geometry& g, const void* keys, int n_prefill, const TablesPtrs& t, cudaStream_t st) {
  CUtensorMap mk, mw, mb, mo;
  if (!make_map(&mk, keys, uint64_t(g.d), uint64_t(g.units) * g.cap, 64, kTileM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mw, t.wt16, uint64_t(g.d), uint64_t(g.n_w) * 3 * g.kltc, 64, kTileN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mb, t.beta, 16, uint64_t(g.units) * g.kltc, 16, kTileN, CU_TENSOR_MAP_SWIZZLE_32B) ||
      !make_map(&mo, t.ones, 16, kTileM, 16, kTileM, CU_TENSOR_MAP_SWIZZLE_32B))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(GemmSmem<D>) + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(k_hash_keys_tc<D, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  const int mt = (n_prefill + kTileM - 1) / kTileM;
  const int items = g.units * mt;
  const int grid = std::min(items, device_sm_count());
  k_hash_keys_tc<D, KT><<<grid, kThreads, smem, st>>>(mk, mw, mb, mo, t.codes, t.hdr, g.units, g.batch * g.kvh,
                                                  g.w_per_layer, g.cap, n_prefill, g.L, g.K, g.tpt, g.nt, g.kltc);
  return cudaGetLastError();
}

static RowSetTc row_set(const RowsHashTc& h) {
  RowSetTc r;
  r.rows = h.rows;
  r.nr32 = (h.rows + 31) / 32 * 32;
  r.negbeta = h.negbeta;
  r.nb_div = h.nb_div > 0 ? h.nb_div : 1;
  r.out = h.out;
  r.out_gs = h.out_gs;
  r.out_rs = h.out_rs;
  r.out_ts = h.out_ts;
  return r;
}

template <int D>
cudaError_t launch_rows_tc(const Geometry& g, const RowsHashTc& h0, const RowsHashTc* h1, cudaStream_t st) {
  RowsTcArgs a;
  a.set[0] = row_set(h0);
  if (h1) {
    a.set[1] = row_set(*h1);
  } else {
    a.set[1] = a.set[0];
    a.set[1].rows = 0;
    a.set[1].nr32 = 0;
  }
  a.vrows = a.set[0].nr32 + a.set[1].nr32;
  // rows per CTA: the largest of 256, 128, 64, 32 whose grid still gives every SM two
  // CTAs (every CTA loads a whole W tile, so fewer, fuller CTAs move fewer bytes when the
  // grid is large enough; otherwise smaller row blocks spread the work and shorten each
  // CTA's epilogue: on the 32-layer decode step 32-row blocks, 384 CTAs, measured 12.3 µs
  // against 13.5 µs for 64-row blocks, 192 CTAs)
  a.nr = 32;
  for (int cand = 256; cand >= 32; cand >>= 1)
    if (int64_t((a.vrows + cand - 1) / cand) * g.nt * h0.groups >= 2 * int64_t(device_sm_count())) {
      a.nr = std::min(cand, a.vrows);
      break;
    }
  a.groups_per_w = h0.groups_per_w;
  a.w_rows = g.w_per_layer ? 3 * g.kltc : 0;
  a.kltc = g.kltc;
  a.hdr = h0.hdr;
  a.mark = h0.mark || (h1 && h1->mark);
  a.mark_pos = h0.mark ? h0.mark_pos : (h1 ? h1->mark_pos : 0);
  CUtensorMap mw, mx0, mx1;
  if (!make_map(&mw, h0.wt16, uint64_t(g.d), uint64_t(g.n_w) * 3 * g.kltc, 64, 256, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_strided(&mx0, h0.x, uint64_t(g.d), uint64_t(h0.rows) * h0.groups, uint64_t(h0.x_rs) * 2, 64, 32,
                        CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (h1) {
    if (!make_map_strided(&mx1, h1->x, uint64_t(g.d), uint64_t(h1->rows) * h1->groups, uint64_t(h1->x_rs) * 2, 64,
                          32, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    mx1 = mx0;
  }
  const size_t smem = RowsLayout<D>::bytes(a.nr) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_hash_rows_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.vrows + a.nr - 1) / a.nr, g.nt, h0.groups);
  k_hash_rows_tc<D><<<grid, kRowsWarps * 32, smem, st>>>(mw, mx0, mx1, a, g.L, g.K, g.tpt);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_hash_rows_tc(const Geometry& g, const RowsHashTc& h0, const RowsHashTc* h1, cudaStream_t st) {
  if (h1 && h1->rows <= 0) h1 = nullptr;
  if (h0.rows <= 0 || h0.groups <= 0 || g.nt == 0) return cudaSuccess;
  if (h1 && (h1->groups != h0.groups || h1->groups_per_w != h0.groups_per_w)) return cudaErrorInvalidValue;
  return g.d == 128 ? launch_rows_tc<128>(g, h0, h1, st) : launch_rows_tc<64>(g, h0, h1, st);
}

cudaError_t launch_hash_keys_tc(const Geometry& g, const void* keys, int n_prefill, const TablesPtrs& t,
                                cudaStream_t st, bool* used) {
  *used = false;
  if (g.dtype != MP_DTYPE_BF16 || g.K == 0 || n_prefill < 1 || !t.wt16) return cudaSuccess;
  // K = 7..12 with d = 128 get an epilogue specialised for K; other shapes the generic one
  cudaError_t e;
  if (g.d == 128) {
    switch (g.K) {
      case 7: e = launch_tc<128, 7>(g, keys, n_prefill, t, st); break;
      case 8: e = launch_tc<128, 8>(g, keys, n_prefill, t, st); break;
      case 9: e = launch_tc<128, 9>(g, keys, n_prefill, t, st); break;
      case 10: e = launch_tc<128, 10>(g, keys, n_prefill, t, st); break;
      case 11: e = launch_tc<128, 11>(g, keys, n_prefill, t, st); break;
      case 12: e = launch_tc<128, 12>(g, keys, n_prefill, t, st); break;
      default: e = launch_tc<128, 0>(g, keys, n_prefill, t, st); break;
    }
  } else {
    e = launch_tc<64, 0>(g, keys, n_prefill, t, st);
  }
  if (e == cudaSuccess) *used = true;
  return e;
}

}  // namespace mp
