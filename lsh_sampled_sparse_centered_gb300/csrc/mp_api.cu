// Host side of the C ABI: validation, buffer layouts and the launch sequence of
// each call. No device memory is allocated here; every buffer is the caller's.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "mp_internal.h"

namespace mp {

static uint64_t align256(uint64_t x) { return (x + 255u) & ~uint64_t(255u); }

// AUTO: the mode that moves fewer bytes per query head and decode step.
//   CSR : L buckets of ~m/2^K ids (2 B) + per 32K-token segment 4 B of offsets, per table
//   SCAN: m tokens x L tables x K bits, read once for the G query heads of a KV head
static int resolve_match(const mp_config* c) {
  if (c->match_mode != MP_MATCH_AUTO) return c->match_mode;
  const double m = std::max(1, c->capacity - c->n_sink - c->window);
  const double G = double(c->q_heads / c->kv_heads);
  const double csr = c->L * (m / std::ldexp(1.0, c->K)) * 2.0 + c->L * (4.0 * std::ceil(m / 32768.0) + 2.0);
  const double scan = m * c->L * c->K / 8.0 / G;
  return scan < csr ? MP_MATCH_SCAN : MP_MATCH_CSR;
}

static int check_config(const mp_config* c) {
  if (!c) return MP_ERR_INVALID_ARG;
  if (c->layers < 1 || c->batch < 1 || c->kv_heads < 1 || c->q_heads < 1) return MP_ERR_INVALID_ARG;
  if (c->q_heads % c->kv_heads != 0) return MP_ERR_INVALID_ARG;
  if (c->K < 0 || c->L < 1 || c->n_sink < 0 || c->window < 0 || c->capacity < 1) return MP_ERR_INVALID_ARG;
  if (c->dtype != MP_DTYPE_F32 && c->dtype != MP_DTYPE_BF16) return MP_ERR_INVALID_ARG;
  if (c->w_per_layer != 0 && c->w_per_layer != 1) return MP_ERR_INVALID_ARG;
  if (c->match_mode != MP_MATCH_AUTO && c->match_mode != MP_MATCH_CSR && c->match_mode != MP_MATCH_SCAN)
    return MP_ERR_INVALID_ARG;
  if (c->threshold < 1 || c->threshold > c->L) return MP_ERR_INVALID_ARG;
  for (int i = 0; i < 2; ++i)
    if (c->reserved[i] != 0) return MP_ERR_INVALID_ARG;
  if (c->no_centering != 0 && c->no_centering != 1) return MP_ERR_INVALID_ARG;
  if (c->center_query != 0 && c->center_query != 1) return MP_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return MP_ERR_UNSUPPORTED;
  if (c->K > kMaxK || c->L > kMaxL || c->capacity > kMaxCapacity) return MP_ERR_UNSUPPORTED;
  // thresholds above 2: at most 7 (3-bit counters in the scan), L <= 255 (byte counters
  // in the bucket walk) and, for the bucket walk, one counter byte per token in shared memory
  if (c->threshold > 7) return MP_ERR_UNSUPPORTED;
  if (c->threshold > 2 && c->L > 255) return MP_ERR_UNSUPPORTED;
  if (c->threshold > 2 && resolve_match(c) == MP_MATCH_CSR && c->capacity > kMaxCapacityCounters)
    return MP_ERR_UNSUPPORTED;
  if (resolve_match(c) == MP_MATCH_CSR) {
    // the match kernel keeps per-token bitmaps (or byte counters), one bucket run and
    // its chunk prefix per (table, 32768-token segment) and the query codes in shared memory
    const int64_t words = (int64_t(c->capacity) + 31) / 32;
    const int64_t nseg = (int64_t(c->capacity) + kCsrSeg - 1) / kCsrSeg;
    const int64_t smem = words * 4 * (c->threshold > 2 ? 9 : 2) + int64_t(c->L) * (nseg * 12 + 2) + 24;
    if (smem > 227 * 1024) return MP_ERR_UNSUPPORTED;
  }
  // grid limits: units and queries index blockIdx.x / y
  const int64_t q = int64_t(c->layers) * c->batch * c->q_heads;
  if (q > (1 << 30)) return MP_ERR_UNSUPPORTED;
  return MP_OK;
}

static Geometry geometry(const mp_config* c) {
  Geometry g;
  g.layers = c->layers;
  g.batch = c->batch;
  g.kvh = c->kv_heads;
  g.qh = c->q_heads;
  g.d = c->head_dim;
  g.K = c->K;
  g.L = c->L;
  g.s = c->n_sink;
  g.w = c->window;
  g.cap = c->capacity;
  g.dtype = c->dtype;
  g.w_per_layer = c->w_per_layer;
  g.threshold = c->threshold;
  g.no_center = c->no_centering;
  g.center_query = c->center_query;
  g.group = c->q_heads / c->kv_heads;
  g.units = c->layers * c->batch * c->kv_heads;
  g.queries = c->layers * c->batch * c->q_heads;
  g.kl = c->K * c->L;
  g.nb = 1 << c->K;
  g.tpt = c->K > 0 ? 256 / c->K : 0;
  g.nt = c->K > 0 ? (c->L + g.tpt - 1) / g.tpt : 0;
  g.kltc = g.nt * 256;
  g.match = resolve_match(c);
  g.cw = (((c->capacity + 31) / 32) + 3) & ~3;
  g.nseg = (c->capacity + kCsrSeg - 1) / kCsrSeg;
  g.parts = 32;
  g.n_w = c->w_per_layer ? c->layers : 1;
  return g;
}

static void tables_layout(const Geometry& g, mp_tables_layout* o) {
  std::memset(o, 0, sizeof(*o));
  const uint64_t U = uint64_t(g.units), d = uint64_t(g.d), L = uint64_t(g.L), cap = uint64_t(g.cap);
  uint64_t off = 0;
  o->header = off;
  off += 256;
  o->center = off;
  off = align256(off + U * d * 4);
  o->beta = off;
  off = align256(off + U * uint64_t(g.kltc) * 16 * 2);
  o->ones = off;
  off = align256(off + 128 * 16 * 2);
  o->negbeta_f32 = off;
  off = align256(off + U * uint64_t(g.kltc) * 4);
  o->wt_f32 = off;
  off = align256(off + uint64_t(g.n_w) * g.kltc * d * 4);
  if (g.dtype == MP_DTYPE_BF16) {
    o->wt_bf16 = off;
    off = align256(off + uint64_t(g.n_w) * 3 * g.kltc * d * 2);
  }
  o->center_parts = off;
  off = align256(off + U * uint64_t(g.parts) * d * 4);
  o->codes = off;
  off = align256(off + U * L * cap * 2);
  if (g.match == MP_MATCH_CSR) {
    o->csr_offsets = off;
    off = align256(off + U * L * uint64_t(g.nseg) * (uint64_t(g.nb) + 1) * 2);
    o->csr_ids = off;
    off = align256(off + U * L * cap * 2 + 16);  // +16: aligned 16-byte chunk reads past the last id
  } else {
    o->planes = off;
    off = align256(off + U * L * uint64_t(g.K) * g.cw * 4);
  }
  o->logu_lut = off;
  off = align256(off + uint64_t(kLutN + 1) * 4);
  o->total_bytes = off;
  o->n_buckets = g.nb;
  o->parts = g.parts;
  o->tc_cols = g.kltc;
  o->match_mode = g.match;
  o->cap_words = g.cw;
}

static void decode_layout(const Geometry& g, mp_decode_layout* o) {
  std::memset(o, 0, sizeof(*o));
  const uint64_t Q = uint64_t(g.queries);
  uint64_t off = 0;
  o->q_codes = off;
  off = align256(off + Q * g.L * 2);
  o->list_len = off;
  off = align256(off + Q * 4);
  o->sample_count = off;
  off = align256(off + Q * 4);
  o->lists = off;
  off = align256(off + Q * uint64_t(g.cap) * 4);
  o->partials = off;
  off = align256(off + Q * kSplitsMax * uint64_t(g.d + 2) * 4);
  o->counters = off;
  off = align256(off + (Q + 1) * 4);
  if (g.match == MP_MATCH_SCAN) {
    o->sample_bits = off;
    off = align256(off + Q * uint64_t(g.cw) * 4);
  }
  o->total_bytes = off;
  o->splits_max = kSplitsMax;
}

static TablesPtrs tables_ptrs(const Geometry& g, void* base) {
  mp_tables_layout l;
  tables_layout(g, &l);
  char* b = static_cast<char*>(base);
  TablesPtrs t;
  t.hdr = reinterpret_cast<DevHeader*>(b + l.header);
  t.center = reinterpret_cast<float*>(b + l.center);
  t.beta = reinterpret_cast<__nv_bfloat16*>(b + l.beta);
  t.ones = reinterpret_cast<__nv_bfloat16*>(b + l.ones);
  t.negbeta = reinterpret_cast<float*>(b + l.negbeta_f32);
  t.wt32 = reinterpret_cast<float*>(b + l.wt_f32);
  t.wt16 = l.wt_bf16 ? reinterpret_cast<__nv_bfloat16*>(b + l.wt_bf16) : nullptr;
  t.cparts = reinterpret_cast<float*>(b + l.center_parts);
  t.codes = reinterpret_cast<uint16_t*>(b + l.codes);
  t.off = l.csr_offsets ? reinterpret_cast<uint16_t*>(b + l.csr_offsets) : nullptr;
  t.ids = l.csr_ids ? reinterpret_cast<uint16_t*>(b + l.csr_ids) : nullptr;
  t.planes = l.planes ? reinterpret_cast<uint32_t*>(b + l.planes) : nullptr;
  t.lut = reinterpret_cast<float*>(b + l.logu_lut);
  return t;
}

static DecodePtrs decode_ptrs(const Geometry& g, void* base) {
  mp_decode_layout l;
  decode_layout(g, &l);
  char* b = static_cast<char*>(base);
  DecodePtrs p;
  p.qcodes = reinterpret_cast<uint16_t*>(b + l.q_codes);
  p.list_len = reinterpret_cast<int32_t*>(b + l.list_len);
  p.sample_count = reinterpret_cast<int32_t*>(b + l.sample_count);
  p.lists = reinterpret_cast<uint32_t*>(b + l.lists);
  p.partials = reinterpret_cast<float*>(b + l.partials);
  p.counters = reinterpret_cast<uint32_t*>(b + l.counters);
  p.sbits = l.sample_bits ? reinterpret_cast<uint32_t*>(b + l.sample_bits) : nullptr;
  return p;
}

// MP_FAULT_INJECT=build|append|decode|all makes the named calls fail before any
// launch (host-side fault injection for error-path tests).
static bool injected(const char* what) {
  const char* e = std::getenv("MP_FAULT_INJECT");
  if (!e || !*e) return false;
  return std::strcmp(e, "all") == 0 || std::strcmp(e, what) == 0;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count() {
  // per-device cache; callers on several host threads may fill it concurrently
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;  // GB300
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// Hash path for bf16 keys, queries and appends: tensor cores unless MP_HASH_PATH=simt.
static bool use_simt_hash() {
  const char* e = std::getenv("MP_HASH_PATH");
  return e && std::strcmp(e, "simt") == 0;
}

// Decode-time rows (queries, appended keys) go through the swap-AB tensor-core kernel
// for bf16 with d = 64 or 128.
static bool rows_on_tensor_cores(const Geometry& g, const TablesPtrs& t) {
  return g.dtype == MP_DTYPE_BF16 && (g.d == 64 || g.d == 128) && g.K > 0 && g.nt > 0 && t.wt16 &&
         !use_simt_hash();
}

// Number of slices per query head for the attention: about 1024 list entries per
// slice (estimated from the closed-form budget at p = 1/2); when that leaves fewer work
// items than resident CTAs of the persistent grid (four per SM), the largest number of
// slices that still fits in one wave of the grid, as long as a slice keeps ~128 entries;
// at most kSplitsMax. The time of the launch is about the number of waves times a
// slice's length, so a slice count that spills into a second wave is slower than the
// one below it (measured on 256 query heads of 128K tokens: 2 slices 69 us, 3 slices
// 83 us, 5 slices 76 us).
static int choose_splits(const Geometry& g, int n) {
  const double x = std::ldexp(1.0, -g.K);
  double frac;
  if (g.threshold == 1) frac = 1.0 - std::pow(1.0 - x, g.L);
  else frac = 1.0 - std::pow(1.0 - x, g.L) - g.L * x * std::pow(1.0 - x, g.L - 1);
  const int lo = std::min(g.s, n);
  const int hi = std::max(lo, n - g.w);
  const double est = double(n - (hi - lo)) + frac * double(hi - lo);
  int s = int(std::ceil(est / 1024.0));
  const int64_t resident = 4 * int64_t(device_sm_count());
  if (int64_t(s) * g.queries < resident) {
    const int fill = int(resident / g.queries);  // slices per head of one full wave
    s = std::max(s, std::min(fill, int(est / 128.0)));
  }
  if (s < 1) s = 1;
  if (s > kSplitsMax) s = kSplitsMax;
  return s;
}

// ---- optional per-launch event timing ----
enum KernelId {
  K_PREPARE_W, K_CENTER, K_HASH_KEYS_SIMT, K_HASH_KEYS_TC, K_CSR_BUILD, K_HASH_APPEND, K_MARK_APPENDED,
  K_HASH_QUERY, K_MATCH_CSR, K_ATTEND, K_PLANES_BUILD, K_PLANES_APPEND, K_SCAN, K_COMPACT, K_HASH_STEP, K_LOGU_LUT,
  K_COUNT
};
static const char* kKernelNames[K_COUNT] = {"prepare_w", "center", "hash_keys_simt", "hash_keys_tc",
                                            "csr_build", "hash_append", "mark_appended", "hash_query",
                                            "match_csr", "attend", "planes_build", "planes_append",
                                            "scan", "compact", "hash_step", "logu_lut"};
struct ProfRec {
  int id;
  cudaEvent_t a, b;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<ProfRec> g_prof;
static std::vector<cudaEvent_t> g_pool;

static cudaEvent_t pool_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Brackets one launcher call with events when profiling is on.
class ProfScope {
 public:
  ProfScope(cudaStream_t st, int id) : st_(st), id_(id) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (!g_prof_on) return;
    a_ = pool_event();
    b_ = pool_event();
    if (a_ && b_) cudaEventRecord(a_, st_);
  }
  ~ProfScope() {
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (!a_ || !b_) return;
    cudaEventRecord(b_, st_);
    g_prof.push_back({id_, a_, b_});
  }

 private:
  cudaStream_t st_;
  int id_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

}  // namespace mp

using namespace mp;

extern "C" {

int mp_abi_version(void) { return MP_ABI_VERSION; }

const char* mp_status_string(int code) {
  switch (code) {
    case MP_OK: return "ok";
    case MP_ERR_INVALID_ARG: return "invalid argument";
    case MP_ERR_UNSUPPORTED: return "unsupported configuration";
    case MP_ERR_CAPACITY: return "token index or length beyond capacity";
    case MP_ERR_CUDA: return "CUDA error";
    case MP_ERR_INJECTED: return "injected failure";
    case MP_ERR_SCRATCH: return "scratch buffer too small";
    default: return "unknown error";
  }
}

int mp_config_check(const mp_config* cfg) { return check_config(cfg); }

int mp_tables_layout_get(const mp_config* cfg, mp_tables_layout* out) {
  const int rc = check_config(cfg);
  if (rc != MP_OK) return rc;
  if (!out) return MP_ERR_INVALID_ARG;
  tables_layout(geometry(cfg), out);
  return MP_OK;
}

int mp_decode_layout_get(const mp_config* cfg, mp_decode_layout* out) {
  const int rc = check_config(cfg);
  if (rc != MP_OK) return rc;
  if (!out) return MP_ERR_INVALID_ARG;
  decode_layout(geometry(cfg), out);
  return MP_OK;
}

int mp_build_tables(const mp_config* cfg, const void* keys, int32_t n_prefill, const float* W,
                    void* tables, void* stream) {
  int rc = check_config(cfg);
  if (rc != MP_OK) return rc;
  // W may be null only when it has no columns (K = 0)
  if (!keys || !tables || (!W && cfg->K > 0)) return MP_ERR_INVALID_ARG;
  if (!aligned16(keys) || !aligned16(W) || (reinterpret_cast<uintptr_t>(tables) & 255u))
    return MP_ERR_INVALID_ARG;
  if (n_prefill < 1 || n_prefill > cfg->capacity) return MP_ERR_CAPACITY;
  if (injected("build")) return MP_ERR_INJECTED;
  const Geometry g = geometry(cfg);
  const TablesPtrs t = tables_ptrs(g, tables);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();  // clear a stale error so that it is not blamed on this call
  if (cudaMemsetAsync(t.hdr, 0, sizeof(DevHeader), st) != cudaSuccess) return MP_ERR_CUDA;
  {
    ProfScope ps(st, K_PREPARE_W);
    if (launch_prepare_w(g, W, t, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  {
    ProfScope ps(st, K_LOGU_LUT);
    if (launch_logu_lut(g, t, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  {
    ProfScope ps(st, K_CENTER);
    if (launch_center(g, keys, n_prefill, t, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  bool done = false;
  if (g.K == 0) {
    // no projections: every code of every table is the empty code 0
    if (cudaMemsetAsync(t.codes, 0, size_t(g.units) * g.L * g.cap * sizeof(uint16_t), st) != cudaSuccess)
      return MP_ERR_CUDA;
    done = true;
  }
  if (!done && g.dtype == MP_DTYPE_BF16 && !use_simt_hash()) {
    ProfScope ps(st, K_HASH_KEYS_TC);
    if (launch_hash_keys_tc(g, keys, n_prefill, t, st, &done) != cudaSuccess) return MP_ERR_CUDA;
  }
  if (!done) {
    HashRowsArgs a;
    std::memset(&a, 0, sizeof(a));
    a.src = keys;
    a.src_gs = int64_t(g.cap) * g.d;
    a.src_rs = g.d;
    a.rows = n_prefill;
    a.groups = g.units;
    a.row0 = 0;
    a.center = t.center;
    a.c_gs = 1;
    a.c_rs = 0;
    a.c_div = 1;
    a.wt = t.wt32;
    a.w_stride = g.w_per_layer ? int64_t(g.kltc) * g.d : 0;
    a.groups_per_w = g.batch * g.kvh;
    a.out = t.codes;
    a.out_gs = int64_t(g.L) * g.cap;
    a.out_rs = 1;
    a.out_ts = g.cap;
    ProfScope ps(st, K_HASH_KEYS_SIMT);
    if (launch_hash_rows(g, a, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  if (g.match == MP_MATCH_CSR) {
    ProfScope ps(st, K_CSR_BUILD);
    if (launch_csr_build(g, n_prefill, t, st) != cudaSuccess) return MP_ERR_CUDA;
  } else {
    ProfScope ps(st, K_PLANES_BUILD);
    if (launch_planes_build(g, n_prefill, t, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}

}  // extern "C"

namespace mp {

// Rows of a decode step's append: the key at token `pos` of every (layer, sequence,
// KV head), one group per layer, centered with its unit's build-time center.
static HashRowsArgs append_rows_simt(const Geometry& g, const TablesPtrs& t, const void* keys, int pos) {
  HashRowsArgs a;
  std::memset(&a, 0, sizeof(a));
  a.src = static_cast<const char*>(keys) + int64_t(pos) * g.d * (g.dtype == MP_DTYPE_BF16 ? 2 : 4);
  a.src_gs = int64_t(g.batch) * g.kvh * g.cap * g.d;  // one group per layer
  a.src_rs = int64_t(g.cap) * g.d;                     // one row per (sequence, KV head)
  a.rows = g.batch * g.kvh;
  a.groups = g.layers;
  a.row0 = 0;
  a.center = t.center;
  a.c_gs = g.batch * g.kvh;
  a.c_rs = 1;
  a.c_div = 1;
  a.wt = t.wt32;
  a.w_stride = g.w_per_layer ? int64_t(g.kltc) * g.d : 0;
  a.groups_per_w = 1;
  a.out = t.codes + pos;
  a.out_gs = int64_t(g.batch) * g.kvh * g.L * g.cap;
  a.out_rs = int64_t(g.L) * g.cap;
  a.out_ts = g.cap;
  // the hash kernel also records the new appended end (no projections when K = 0:
  // then a one-thread kernel does it)
  a.mark_hdr = g.nt > 0 ? t.hdr : nullptr;
  a.mark_pos = pos;
  return a;
}

static RowsHashTc append_rows_tc(const Geometry& g, const TablesPtrs& t, const void* keys, int pos) {
  RowsHashTc h;
  std::memset(&h, 0, sizeof(h));
  h.x = static_cast<const __nv_bfloat16*>(keys) + int64_t(pos) * g.d;
  h.x_rs = int64_t(g.cap) * g.d;
  h.rows = g.batch * g.kvh;
  h.groups = g.layers;
  h.groups_per_w = 1;
  h.wt16 = t.wt16;
  h.negbeta = t.negbeta;
  h.nb_div = 1;
  h.out = t.codes + pos;
  h.out_gs = int64_t(g.batch) * g.kvh * g.L * g.cap;
  h.out_rs = int64_t(g.L) * g.cap;
  h.out_ts = g.cap;
  h.hdr = t.hdr;
  h.mark = 1;
  h.mark_pos = pos;
  return h;
}

// Rows of a decode step's query hash (Algorithm 1 'Encode'): the query as it is, or
// (center_query) the query minus the center of its KV head, query head j of a
// sequence using KV head j / group.
static HashRowsArgs query_rows_simt(const Geometry& g, const TablesPtrs& t, const void* q, const DecodePtrs& dp) {
  HashRowsArgs a;
  std::memset(&a, 0, sizeof(a));
  a.src = q;
  a.src_gs = int64_t(g.batch) * g.qh * g.d;
  a.src_rs = g.d;
  a.rows = g.batch * g.qh;
  a.groups = g.layers;
  a.row0 = 0;
  a.center = g.center_query ? t.center : nullptr;
  a.c_gs = int64_t(g.batch) * g.kvh;
  a.c_rs = 1;
  a.c_div = g.group;
  a.wt = t.wt32;
  a.w_stride = g.w_per_layer ? int64_t(g.kltc) * g.d : 0;
  a.groups_per_w = 1;
  a.out = dp.qcodes;
  a.out_gs = int64_t(g.batch) * g.qh * g.L;
  a.out_rs = g.L;
  a.out_ts = 1;
  return a;
}

static RowsHashTc query_rows_tc(const Geometry& g, const TablesPtrs& t, const void* q, const DecodePtrs& dp) {
  RowsHashTc h;
  std::memset(&h, 0, sizeof(h));
  h.x = static_cast<const __nv_bfloat16*>(q);
  h.x_rs = g.d;
  h.rows = g.batch * g.qh;
  h.groups = g.layers;
  h.groups_per_w = 1;
  h.wt16 = t.wt16;
  h.negbeta = g.center_query ? t.negbeta : nullptr;
  h.nb_div = g.group;
  h.out = dp.qcodes;
  h.out_gs = int64_t(g.batch) * g.qh * g.L;
  h.out_rs = g.L;
  h.out_ts = 1;
  h.hdr = t.hdr;
  return h;
}

// After the appended key's codes are stored: its bit-planes (scan mode) and, with no
// projections (K = 0), the appended end.
static int finish_append(const Geometry& g, const TablesPtrs& t, int pos, cudaStream_t st) {
  if (g.match == MP_MATCH_SCAN) {
    ProfScope ps(st, K_PLANES_APPEND);
    if (launch_planes_append(g, pos, t, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  if (g.nt == 0) {
    ProfScope ps(st, K_MARK_APPENDED);
    if (launch_mark_appended(g, pos, t, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  return MP_OK;
}

// The query codes of K = 0 (every code is the empty code 0).
static int zero_query_codes(const Geometry& g, const DecodePtrs& dp, cudaStream_t st) {
  return cudaMemsetAsync(dp.qcodes, 0, size_t(g.queries) * g.L * sizeof(uint16_t), st) == cudaSuccess ? MP_OK
                                                                                                     : MP_ERR_CUDA;
}

// Sampled sets (Algorithm 1 'Query') plus exact tokens, then the split-K
// importance-weighted attention with its fused combine.
static int match_and_attend(const Geometry& g, const TablesPtrs& t, const DecodePtrs& dp, int n, const void* keys,
                            const void* values, const void* q, float* out, cudaStream_t st) {
  if (g.match == MP_MATCH_CSR) {
    ProfScope ps(st, K_MATCH_CSR);
    if (launch_match_csr(g, n, t, dp, st) != cudaSuccess) return MP_ERR_CUDA;
  } else {
    {
      ProfScope ps(st, K_SCAN);
      if (launch_scan(g, n, t, dp, st) != cudaSuccess) return MP_ERR_CUDA;
    }
    ProfScope ps(st, K_COMPACT);
    if (launch_compact(g, n, t, dp, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  const int splits = choose_splits(g, n);
  ProfScope ps(st, K_ATTEND);
  if (launch_attend(g, n, splits, t, keys, values, q, out, dp, st) != cudaSuccess) return MP_ERR_CUDA;
  return MP_OK;
}

static int check_decode_args(const mp_config* cfg, void* tables, const void* keys, const void* values, int32_t n,
                             const void* q, float* out, void* scratch, size_t scratch_bytes) {
  if (!tables || !keys || !values || !q || !out || !scratch) return MP_ERR_INVALID_ARG;
  if (!aligned16(keys) || !aligned16(values) || !aligned16(q) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(tables) & 255u) || (reinterpret_cast<uintptr_t>(scratch) & 255u))
    return MP_ERR_INVALID_ARG;
  if (n < 1 || n > cfg->capacity) return MP_ERR_CAPACITY;
  mp_decode_layout dl;
  decode_layout(geometry(cfg), &dl);
  if (scratch_bytes < dl.total_bytes) return MP_ERR_SCRATCH;
  return MP_OK;
}

}  // namespace mp

extern "C" {

int mp_append(const mp_config* cfg, void* tables, const void* keys, int32_t pos, void* stream) {
  int rc = check_config(cfg);
  if (rc != MP_OK) return rc;
  if (!keys || !tables) return MP_ERR_INVALID_ARG;
  if (!aligned16(keys) || (reinterpret_cast<uintptr_t>(tables) & 255u)) return MP_ERR_INVALID_ARG;
  if (pos < 0 || pos >= cfg->capacity) return MP_ERR_CAPACITY;
  if (injected("append")) return MP_ERR_INJECTED;
  const Geometry g = geometry(cfg);
  const TablesPtrs t = tables_ptrs(g, tables);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  if (rows_on_tensor_cores(g, t)) {
    const RowsHashTc h = append_rows_tc(g, t, keys, pos);
    ProfScope ps(st, K_HASH_APPEND);
    if (launch_hash_rows_tc(g, h, nullptr, st) != cudaSuccess) return MP_ERR_CUDA;
  } else {
    const HashRowsArgs a = append_rows_simt(g, t, keys, pos);
    ProfScope ps(st, K_HASH_APPEND);
    if (launch_hash_rows(g, a, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  if ((rc = finish_append(g, t, pos, st)) != MP_OK) return rc;
  return cudaGetLastError() == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}

int mp_decode_attention(const mp_config* cfg, void* tables, const void* keys, const void* values,
                        int32_t n, const void* q, float* out, void* scratch, size_t scratch_bytes,
                        void* stream) {
  int rc = check_config(cfg);
  if (rc != MP_OK) return rc;
  if ((rc = check_decode_args(cfg, tables, keys, values, n, q, out, scratch, scratch_bytes)) != MP_OK) return rc;
  if (injected("decode")) return MP_ERR_INJECTED;
  const Geometry g = geometry(cfg);
  const TablesPtrs t = tables_ptrs(g, tables);
  const DecodePtrs dp = decode_ptrs(g, scratch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  if (g.K == 0) {
    if ((rc = zero_query_codes(g, dp, st)) != MP_OK) return rc;
  } else if (rows_on_tensor_cores(g, t)) {
    const RowsHashTc h = query_rows_tc(g, t, q, dp);
    ProfScope ps(st, K_HASH_QUERY);
    if (launch_hash_rows_tc(g, h, nullptr, st) != cudaSuccess) return MP_ERR_CUDA;
  } else {
    const HashRowsArgs a = query_rows_simt(g, t, q, dp);
    ProfScope ps(st, K_HASH_QUERY);
    if (launch_hash_rows(g, a, st) != cudaSuccess) return MP_ERR_CUDA;
  }
  if ((rc = match_and_attend(g, t, dp, n, keys, values, q, out, st)) != MP_OK) return rc;
  return cudaGetLastError() == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}

int mp_decode_step(const mp_config* cfg, void* tables, const void* keys, const void* values, int32_t pos,
                   const void* q, float* out, void* scratch, size_t scratch_bytes, void* stream) {
  int rc = check_config(cfg);
  if (rc != MP_OK) return rc;
  if (pos < 0 || pos >= cfg->capacity) return MP_ERR_CAPACITY;
  if ((rc = check_decode_args(cfg, tables, keys, values, pos + 1, q, out, scratch, scratch_bytes)) != MP_OK)
    return rc;
  if (injected("append") || injected("decode")) return MP_ERR_INJECTED;
  const Geometry g = geometry(cfg);
  const TablesPtrs t = tables_ptrs(g, tables);
  const DecodePtrs dp = decode_ptrs(g, scratch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  // the appended keys and the queries of the step, hashed by one launch (the appended
  // codes are stored before the match kernel reads them: stream order)
  if (g.K == 0) {
    if ((rc = zero_query_codes(g, dp, st)) != MP_OK) return rc;
  } else if (rows_on_tensor_cores(g, t)) {
    const RowsHashTc ha = append_rows_tc(g, t, keys, pos);
    const RowsHashTc hq = query_rows_tc(g, t, q, dp);
    ProfScope ps(st, K_HASH_STEP);
    if (launch_hash_rows_tc(g, ha, &hq, st) != cudaSuccess) return MP_ERR_CUDA;
  } else {
    const HashRowsArgs aa = append_rows_simt(g, t, keys, pos);
    const HashRowsArgs aq = query_rows_simt(g, t, q, dp);
    ProfScope ps(st, K_HASH_STEP);
    if (launch_hash_rows(g, aa, st) != cudaSuccess || launch_hash_rows(g, aq, st) != cudaSuccess)
      return MP_ERR_CUDA;
  }
  if ((rc = finish_append(g, t, pos, st)) != MP_OK) return rc;
  if ((rc = match_and_attend(g, t, dp, pos + 1, keys, values, q, out, st)) != MP_OK) return rc;
  return cudaGetLastError() == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}

int mp_profile_enable(int on) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (auto& r : g_prof) {
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_prof.clear();
  g_prof_on = on != 0;
  return MP_OK;
}

int mp_profile_read(mp_kernel_time* out, int32_t capacity, int32_t* count) {
  if (!count || (capacity > 0 && !out)) return MP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(g_prof_mu);
  double ms[K_COUNT] = {0};
  int n[K_COUNT] = {0};
  int rc = MP_OK;
  for (auto& r : g_prof) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      rc = MP_ERR_CUDA;
    ms[r.id] += t;
    n[r.id] += 1;
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_prof.clear();
  int k = 0;
  for (int i = 0; i < K_COUNT; ++i) {
    if (n[i] == 0) continue;
    if (k < capacity) {
      std::memset(&out[k], 0, sizeof(out[k]));
      std::strncpy(out[k].name, kKernelNames[i], sizeof(out[k].name) - 1);
      out[k].launches = n[i];
      out[k].total_ms = ms[i];
    }
    ++k;
  }
  *count = k;
  return rc;
}

int mp_get_status(const void* tables, uint32_t* status, void* stream) {
  if (!tables || !status) return MP_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const DevHeader* h = static_cast<const DevHeader*>(tables);
  if (cudaMemcpyAsync(status, &h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MP_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MP_ERR_CUDA;
  return MP_OK;
}

}  // extern "C"
