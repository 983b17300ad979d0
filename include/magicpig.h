/*
 * magicpig.h — C ABI of an LSH-sampled sparse decode-attention library for one
 * GB300 GPU (sm_103a).
 *
 * The method is the one of "MagicPIG: LSH Sampling for Efficient LLM Generation"
 * (arXiv 2410.16179v2):
 *   - keys are centered by their mean before hashing (§4.3 "Data pre-processing";
 *     config.no_centering = 1 gives the pages' ablation without it);
 *   - each key and each query gets L SimHash codes of K bits from K·L random
 *     projections W ∈ R^{d×(K·L)} (§2.2 SimHash; §4.3 "Hash function selection";
 *     Algorithm 1 'Encode');
 *   - a key is sampled when its code equals the query's in at least T tables
 *     (T = config.threshold; the pages take T = 2: §4.3; Algorithm 1 'Query');
 *   - the output is the self-normalised importance-sampling estimate
 *     softmax(q·k/√d − log u) V over the sampled keys, with u = P[Bin(L, p^K) >= T]
 *     (for T = 2: 1 − (1 − p^K)^L − L p^K (1 − p^K)^(L−1)) and p = 1 − θ(q, k − c)/π
 *     (Eq. 9–11);
 *   - sink tokens and a local window are attended exactly with u = 1 (§4.4
 *     "On-device cache"; §5.1 Baselines: 4 sinks and a 64-token window).
 *
 * Tensor layouts (all row-major, C order, dense):
 *   keys, values : [layers][batch][kv_heads][capacity][head_dim]   (the pages' K, V ∈ R^{n×d} per head)
 *   q            : [layers][batch][q_heads][head_dim]              (the pages' q ∈ R^{1×d} per head)
 *   W            : [layers or 1][head_dim][K·L] float32            (the pages' W ∈ R^{d×(K·L)})
 *   out          : [layers][batch][q_heads][head_dim] float32
 * Query head j of a sequence reads KV head j / (q_heads / kv_heads) (grouped-query attention).
 * Element type of keys, values and q: MP_DTYPE_BF16 or MP_DTYPE_F32 (config.dtype).
 *
 * Ownership: every pointer passed in is owned by the caller. Device pointers must
 * be device memory of the current device; the library allocates and frees nothing,
 * never synchronises (except mp_get_status) and enqueues all work on the caller's
 * stream (`stream` is a cudaStream_t; NULL is the legacy default stream).
 *
 * Errors: every call returns MP_OK (0) or a negative MP_ERR_* code and enqueues
 * nothing when it fails validation. Faults detected by kernels while they run are
 * ORed into a device status word kept in the tables (MP_STATUS_* bits), read with
 * mp_get_status.
 */
#ifndef MAGICPIG_H_
#define MAGICPIG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MP_API __attribute__((visibility("default")))
#else
#define MP_API
#endif

#define MP_ABI_VERSION 4 /* 2: mp_config.no_centering, mp_tables_layout.negbeta_f32, three-term W;
                            3: mp_config.center_query; 4: mp_tables_layout.logu_lut */

/* return codes */
#define MP_OK 0
#define MP_ERR_INVALID_ARG (-1) /* null pointer, bad shape, inconsistent config */
#define MP_ERR_UNSUPPORTED (-2) /* valid but not implemented (e.g. head_dim not 64/128) */
#define MP_ERR_CAPACITY (-3)    /* a token index or length beyond config.capacity */
#define MP_ERR_CUDA (-4)        /* a CUDA runtime call or kernel launch failed */
#define MP_ERR_INJECTED (-5)    /* failure injected on the host by MP_FAULT_INJECT */
#define MP_ERR_SCRATCH (-6)     /* scratch buffer smaller than required */

/* device status bits (mp_get_status) */
#define MP_STATUS_W_NOT_BF16 0x1u   /* informational, bf16 configs: W is not bf16-representable, so the
                                       tensor-core hashing runs on its three-term bf16 split (three
                                       times the MMA work; results as exact as with fp32 W) */
#define MP_STATUS_WAIT_TIMEOUT 0x2u /* a bounded wait on an mbarrier gave up */
#define MP_STATUS_APPEND_GAP 0x4u   /* decode needed codes of a token never appended */
#define MP_STATUS_NOT_BUILT 0x8u    /* decode or append on tables that were never built */
#define MP_STATUS_BAD_INDEX 0x10u   /* bounds-checking build only (compiled with MP_CHECK=1): a
                                       kernel met an index outside its buffer (a code of 2^K or
                                       more, a bucket run past its segment, a list entry past the
                                       capacity) and skipped that access */

/* element types */
#define MP_DTYPE_F32 0
#define MP_DTYPE_BF16 1

/* how the sampled set is found */
#define MP_MATCH_AUTO 0 /* choose by bytes moved per query head (fewer wins) */
#define MP_MATCH_CSR 1  /* bucketed tables: one id list per (KV head, table, code) */
#define MP_MATCH_SCAN 2 /* stream bit-planes of every code, shared by the query heads of a KV head */

typedef struct mp_config {
  int32_t layers;      /* independent attention layers handled by one call */
  int32_t batch;       /* independent sequences */
  int32_t kv_heads;    /* KV heads per sequence */
  int32_t q_heads;     /* query heads per sequence, a multiple of kv_heads */
  int32_t head_dim;    /* d: 64 or 128 */
  int32_t K;           /* bits per table, 0..12 (0: every key collides in every table) */
  int32_t L;           /* tables, 1..1024 */
  int32_t n_sink;      /* initial tokens always attended exactly (pages: 4) */
  int32_t window;      /* most recent tokens always attended exactly (pages: 64) */
  int32_t capacity;    /* maximum tokens per sequence (prefill + appended), <= 2^19 */
  int32_t dtype;       /* MP_DTYPE_BF16 or MP_DTYPE_F32 (keys, values, q) */
  int32_t w_per_layer; /* 1: W holds one matrix per layer; 0: one matrix shared by all layers */
  int32_t match_mode;  /* MP_MATCH_AUTO, MP_MATCH_CSR or MP_MATCH_SCAN */
  int32_t threshold;   /* minimum colliding tables for a key to be sampled, 1..7 (pages: 2);
                          above 2 it needs L <= 255 and, in CSR mode, capacity <= 196608 */
  int32_t no_centering; /* 0 (default): keys are centered by their prefill mean before hashing
                           (pages §4.3 "Data pre-processing"); 1: hashed uncentered, c = 0 (the
                           pages' centering ablation) */
  int32_t center_query; /* 0 (default): the query is hashed as it is, p = 1 - theta(q, k - c)/pi
                           (the pages center the keys only, §4.3); 1: the query is hashed after
                           subtracting its KV head's center and p = 1 - theta(q - c, k - c)/pi,
                           the probability that the two vectors whose signs are compared share a
                           table's code (§2.2 SimHash). The logits use the raw q and k either way */
  int32_t reserved[2]; /* must be zero */
} mp_config;

/* Byte offsets (from the start of the tables buffer) of the arrays the library keeps
 * between calls. U = layers·batch·kv_heads units, NB = 2^K buckets, TC = columns of
 * the tile-aligned projection layout: 256-column tiles, each holding floor(256/K)
 * whole tables (column 256·n + i·K + b is bit b of table n·floor(256/K) + i), the
 * rest zero. Exposed for tests and tools; the contents are library-private. */
typedef struct mp_tables_layout {
  uint64_t total_bytes;
  uint64_t header;       /* 256 B: magic, prefill length, appended length, status word */
  uint64_t center;       /* float [U][d]: mean key of tokens [n_sink, n_prefill) */
  uint64_t beta;         /* bf16 [U][TC][16]: -W^T·center split into three bf16 terms (elements 0..2,
                            the rest zero), tile-aligned column order; with `ones` it is the
                            extra K step of the tensor-core projection that subtracts W^T·center */
  uint64_t ones;         /* bf16 [128][16]: rows of (1, 1, 1, 0, ..., 0) */
  uint64_t negbeta_f32;  /* float [U][TC]: -W^T·center in tile-aligned column order (centering of
                            appended keys hashed on the tensor cores) */
  uint64_t wt_f32;       /* float [layers or 1][TC][d]: W transposed, tile-aligned column order */
  uint64_t wt_bf16;      /* bf16  [layers or 1][3][TC][d] (bf16 configs only, else 0): W split into
                            three bf16 terms hi, mid, lo with hi + mid + lo = W exactly (mid and lo
                            are zero when W is bf16-representable) */
  uint64_t center_parts; /* float [U][parts][d]: partial sums while building */
  uint64_t codes;        /* uint16 [U][L][capacity]: code of every hashed token, table-major */
  uint64_t csr_offsets;  /* uint16 [U][L][NB+1][NS]: per table, bucket b and 32768-token segment s of
                            [n_sink, n_prefill), the start of bucket b within segment s (element
                            [NB][s]: the segment's length) (CSR mode, else 0); NS = ceil(capacity / 32768) */
  uint64_t csr_ids;      /* uint16 [U][L][capacity]: element 32768*s + i is the i-th id of segment s in
                            bucket order, as an offset from the segment's first token; the order inside
                            a bucket is unspecified (CSR mode, else 0) */
  uint64_t planes;       /* uint32 [U][L][K][CW]: bit-planes, word w bit i = bit b of the code of token
                            32w+i (scan mode, else 0); CW = capacity/32 rounded up to a multiple of 4 */
  uint64_t logu_lut;     /* float [4097]: -log u of the config's (K, L, threshold) at the cosines
                            -0.5 + 1.49·i/4096 (Eq. 10/11), written by mp_build_tables; the attention
                            interpolates it and evaluates u directly outside [-0.5, 0.99] */
  int32_t n_buckets;     /* NB */
  int32_t parts;
  int32_t tc_cols;       /* TC */
  int32_t match_mode;    /* the mode in use: MP_MATCH_CSR or MP_MATCH_SCAN (AUTO resolved) */
  int32_t cap_words;     /* CW */
} mp_tables_layout;

/* Byte offsets in the decode scratch buffer. Q = layers·batch·q_heads. */
typedef struct mp_decode_layout {
  uint64_t total_bytes;
  uint64_t q_codes;      /* uint16 [Q][L]: query codes */
  uint64_t list_len;     /* int32 [Q]: entries in the list (sampled + exact) */
  uint64_t sample_count; /* int32 [Q]: sampled entries |S| (they come first) */
  uint64_t lists;        /* uint32 [Q][capacity]: token ids, S ascending then exact tokens
                            (bit 31 set on exact tokens) */
  uint64_t partials;     /* float [Q][splits_max][d+2]: split-K partial (m, l, acc[d]) */
  uint64_t counters;     /* uint32 [Q + 1]: split-K completion counters, then the attention's
                            work-queue head */
  uint64_t sample_bits;  /* uint32 [Q][CW]: sampled-token bitmaps (scan mode, else 0) */
  int32_t splits_max;
  int32_t reserved;
} mp_decode_layout;

/* Validate a configuration. MP_OK or MP_ERR_INVALID_ARG / MP_ERR_UNSUPPORTED. */
MP_API int mp_config_check(const mp_config* cfg);

/* Layout and size of the tables buffer (device memory the caller allocates, at least
 * 256-byte aligned; contents need no initialisation). */
MP_API int mp_tables_layout_get(const mp_config* cfg, mp_tables_layout* out);

/* Layout and size of the decode scratch buffer (device memory, 256-byte aligned,
 * no initialisation needed; reusable across calls on the same stream). */
MP_API int mp_decode_layout_get(const mp_config* cfg, mp_decode_layout* out);

/* Build the hash tables from the prefill keys [0, n_prefill) of every
 * (layer, sequence, KV head): center with the mean of keys [n_sink, n_prefill)
 * (§4.3 "Data pre-processing"), SimHash every prefill key into L K-bit codes with
 * the projections W (§2.2, §4.3, Algorithm 1 'Encode'; on bf16 keys the projection
 * runs on tensor cores, through W's exact three-term bf16 split when W is not
 * bf16-representable, which the informational MP_STATUS_W_NOT_BF16 bit reports),
 * and bucket the ids of tokens [n_sink, n_prefill) per (head, table, code) —
 * the hash tables HT of Algorithm 1.
 *   keys    : device, layout above; rows [0, n_prefill) are read.
 *   W       : device float32, [layers or 1][d][K·L] per config.w_per_layer (may be NULL when K = 0).
 *   tables  : device, mp_tables_layout_get(cfg).total_bytes.
 * 1 <= n_prefill <= capacity, else MP_ERR_CAPACITY. Resets the status word. */
MP_API int mp_build_tables(const mp_config* cfg, const void* keys, int32_t n_prefill,
                    const float* W, void* tables, void* stream);

/* Hash the key at token index `pos` of every (layer, sequence, KV head) into all
 * L tables (one decode-step append). The caller has already written
 * keys[..][pos][:]. Uses the center fixed at build time. Tokens appended this way
 * are matched by comparing stored codes once they leave the window.
 * 0 <= pos < capacity, else MP_ERR_CAPACITY. pos is meant to be the next token,
 * pos >= n_prefill; the host cannot check that bound (n_prefill lives in the device
 * header). An append at pos < n_prefill rewrites that token's stored code (and its
 * bit-planes in scan mode) but not its place in the CSR buckets built at build time. */
MP_API int mp_append(const mp_config* cfg, void* tables, const void* keys, int32_t pos, void* stream);

/* One decode step for every query head (Algorithm 1 with the exact sink/window
 * cache of §4.4): hash q (or q - c with config.center_query), collect S = {i in [n_sink, n - window) :
 * code equal in >= threshold tables}, and write
 *   out = softmax([q·k_S/√d − log u_S, q·k_T/√d]) [V_S; V_T]
 * with T the sinks [0, n_sink) and the window [n - window, n), u = 1 on T.
 *   keys, values : device, layout above; rows [0, n) are read.
 *   n            : tokens visible to the query, 1 <= n <= capacity.
 *   q            : device [layers][batch][q_heads][d] in config.dtype.
 *   out          : device float32 [layers][batch][q_heads][d].
 *   scratch      : device, at least mp_decode_layout_get(cfg).total_bytes (scratch_bytes).
 * Writes only out, scratch and the status word of tables. */
MP_API int mp_decode_attention(const mp_config* cfg, void* tables, const void* keys,
                        const void* values, int32_t n, const void* q, float* out,
                        void* scratch, size_t scratch_bytes, void* stream);

/* One decode step of a growing sequence: mp_append(cfg, tables, keys, pos) followed by
 * mp_decode_attention(..., n = pos + 1, ...), with the same results, in fewer launches:
 * the appended key of every (layer, sequence, KV head) and every query are hashed
 * together (on the tensor cores, one launch that loads each W tile once for both).
 * This is the step of the pages' decoding loop (Algorithm 1 per generated token, the
 * new key entering the tables; §4.4): the caller has already written keys[..][pos][:]
 * and values[..][pos][:].
 *   pos : the new token, 0 <= pos < capacity (else MP_ERR_CAPACITY); meant to be the
 *         next token after the prefill and earlier appends (see mp_append).
 * Other arguments, errors and writes as mp_append and mp_decode_attention. */
MP_API int mp_decode_step(const mp_config* cfg, void* tables, const void* keys, const void* values,
                          int32_t pos, const void* q, float* out, void* scratch, size_t scratch_bytes,
                          void* stream);

/* Size of the scratch array built into the library for mp_decode_attention_static. */
#define MP_STATIC_SCRATCH_BYTES (32u << 20)

/* The decode step of mp_decode_attention for callers that cannot allocate device
 * memory for its scratch buffer: for example a plugin whose host application owns
 * all device memory, a server that reserved its whole memory budget up front, or a
 * latency-critical loop that must not call cudaMalloc because it can block on the
 * device. No counterpart on the pages: it is a deployment variant of the same call.
 * Same arguments and results as mp_decode_attention, minus scratch and scratch_bytes.
 * The scratch lives in a fixed device array of MP_STATIC_SCRATCH_BYTES (32 MiB)
 * compiled into the library and held by every GPU that loads it until the process
 * exits. Calls whose mp_decode_layout_get(cfg).total_bytes exceeds that size are
 * rejected with MP_ERR_SCRATCH before anything is enqueued. The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress, with that device
 * current) and keeps it for the life of the process; make that first call before any
 * stream capture. The kept address assumes the device's primary context lives as long
 * as the process: after cudaDeviceReset the module is loaded again and the array may
 * move, so a process that resets a device must not call this entry point afterwards. Allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine). All calls share the array
 * and it keeps the last call's contents; the counters that must start at zero are
 * reset on the device by every call. Calls whose kernels overlap on the GPU race on
 * the shared array: order them on one stream (or by events). */
MP_API int mp_decode_attention_static(const mp_config* cfg, void* tables, const void* keys,
                                      const void* values, int32_t n, const void* q, float* out,
                                      void* stream);

/* Copy the device status word to *status (synchronises `stream`). */
MP_API int mp_get_status(const void* tables, uint32_t* status, void* stream);

/* Human-readable name of a return code. */
MP_API const char* mp_status_string(int code);

/* MP_ABI_VERSION of the loaded library. */
MP_API int mp_abi_version(void);

/* ---- measurement instrumentation (no counterpart on the pages) ----
 * When enabled, every kernel launch of the calls above is bracketed by a pair of
 * CUDA events recorded on the caller's stream. mp_profile_read synchronises those
 * events, returns per-kernel launch counts and summed device time, and clears the
 * record. Disabled by default; enabling it adds two event records per launch. */
typedef struct mp_kernel_time {
  char name[32];
  int32_t launches;
  int32_t reserved;
  double total_ms;
} mp_kernel_time;

/* on = 1 starts recording (clearing earlier records), on = 0 stops. */
MP_API int mp_profile_enable(int on);

/* Writes up to `capacity` entries (one per kernel name seen) and their number to *count. */
MP_API int mp_profile_read(mp_kernel_time* out, int32_t capacity, int32_t* count);

#ifdef __cplusplus
}
#endif

#endif /* MAGICPIG_H_ */
