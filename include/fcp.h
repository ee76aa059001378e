/*
 * fcp.h -- C ABI of libfcp: document-masked context-parallel attention on one
 * GB300 (sm_103a).
 *
 * Sources of the operations (web pages this library restates):
 *   [FlashCP]  "FlashCP: Load-Balanced Communication-Efficient Context
 *              Parallelism for LLM Training" (arXiv 2606.08476).
 *   [CPGuide]  "LLM Context Parallel in Production: Breaking Long-Context
 *              Bottlenecks with Sequence Sharding, Ring/Ulysses Communication,
 *              and Causal Load Balancing".
 *
 * Conventions
 *   - Every call returns an int status (FCP_OK = 0). Argument checks are done
 *     on the host, synchronously, before anything is launched; a call that
 *     returns an error has launched nothing.
 *   - Device calls are asynchronous on the given stream (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).
 *   - The library never allocates device memory. Every device buffer is owned
 *     by the caller. Host memory is allocated only for a plan object, freed by
 *     fcp_plan_free.
 *   - Token-major varlen layout: Q and O are [T][Hq][d], K and V [T][Hkv][d],
 *     all contiguous, row-major; LSE is [Hq][T] fp32, natural log.
 *   - Query head h reads KV head h / (Hq/Hkv) (contiguous GQA groups).
 *   - Supported: d in {64, 128}, Hq % Hkv == 0 (any group size, MHA included), T < 2^31.
 *   - All device pointers must be 16-byte aligned.
 */
#ifndef FCP_H
#define FCP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------ */
/* Status codes and enums                                                    */
/* ------------------------------------------------------------------------ */
enum {
  FCP_OK = 0,
  FCP_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent tables   */
  FCP_ERR_UNSUPPORTED = 2,   /* e.g. d not in {64,128}, Hq % Hkv != 0          */
  FCP_ERR_CUDA = 3,          /* a CUDA runtime call failed                     */
  FCP_ERR_TIMEOUT = 4,       /* a bounded device wait expired (see status)     */
  FCP_ERR_INFEASIBLE = 5,    /* the policy cannot shard this input (e.g. T%2N) */
  FCP_ERR_CAPACITY = 6,      /* a caller buffer is too small                   */
  FCP_ERR_MISSING_PART = 7   /* a partial result is missing or duplicated      */
};

enum {
  FCP_POLICY_LLAMA3 = 0,     /* [FlashCP] §2.2/§2.3: sequence in 2N chunks, i & 2N-1-i */
  FCP_POLICY_PER_DOC = 1,    /* [FlashCP] §2.3: every doc in 2N chunks, i & 2N-1-i    */
  FCP_POLICY_WHOLE_DOC = 2,  /* [FlashCP] Algorithm 1 with R = infinity               */
  FCP_POLICY_HYBRID = 3,     /* [FlashCP] Algorithm 1 with target imbalance R         */
  FCP_POLICY_HYBRID_TILES = 4 /* Algorithm 1 with R, a piece's workload in kernel tiles:
                                 sum over its query tiles of the key tiles of the causal
                                 prefix, plus one per query tile (instead of W)        */
};

enum {
  FCP_OUT_BF16 = 0,          /* final output: O bf16 [T][Hq][d]                   */
  FCP_OUT_F32 = 1            /* partial output for a merge: O fp32 [T][Hq][d]     */
};

/* The human-readable name of a status code (static string). */
const char* fcp_strerror(int status);

/* ------------------------------------------------------------------------ */
/* Plans (host)                                                              */
/* ------------------------------------------------------------------------ */

/* A half-open global token range [start, end) inside document `doc`. */
typedef struct {
  int32_t doc;
  int32_t start;
  int32_t end;
} fcp_range;

typedef struct fcp_plan fcp_plan_t;   /* opaque, host-owned */

/* Per-shard view. Pointers are owned by the plan and valid until fcp_plan_free. */
typedef struct {
  int32_t n_pieces;            /* query pieces, ascending, each inside one doc */
  const fcp_range* pieces;
  int32_t n_need;              /* per document touched: [doc start, last piece end) */
  const fcp_range* kv_need;
  int32_t n_remote;            /* needed keys held by other shards, ascending     */
  const fcp_range* kv_remote;
  int64_t tokens;              /* sum of piece lengths                            */
  int64_t useful_pairs;        /* sum of W_i = (2 p_i + s_i + 1) s_i / 2           */
  int64_t remote_rows;         /* rows in kv_remote                                */
  int64_t kbuf_base;           /* first row of this shard in an all-shards kbuf    */
  /* Tiles of 128 x 128 the kernels visit for this shard, per query head
   * (useful pairs only enter tiles that hold at least one):              */
  int64_t fwd_tiles;           /* forward query-tile x key-tile pairs              */
  int64_t fwd_qtiles;          /* forward query tiles                              */
  int64_t fwd_masked;          /* forward tiles needing a per-element mask         */
  int64_t bwd_tiles;           /* backward key-tile x query-tile pairs             */
  int64_t bwd_ktiles;          /* backward work units (per KV head): the shard's   */
                               /* distinct key tiles (a key tile shared by two     */
                               /* pieces of one document is one unit)              */
} fcp_shard_view;

typedef struct {
  int32_t cp;                  /* N */
  int32_t n_docs;
  int64_t T;
  double imbalance;            /* max_j W_j / mean_j W_j ([FlashCP] §4.3)         */
  int64_t max_pairs;
  int64_t total_pairs;         /* = sum over docs of L(L+1)/2                      */
  int64_t eq4_tokens;          /* Eq. 4 volume / (H * D): 4 (C/N) (N-1)            */
  int64_t eq5_tokens;          /* Eq. 5 volume / (H * D): 4 max_j sum_{S^} s (N-1) */
  int64_t remote_rows_total;   /* receiver-side exact need, all shards             */
  int64_t remote_rows_max;
  int64_t eq2_max_dev;         /* max_j |tokens_j - C/N| (0 unless Per-Doc rounding) */
  int32_t iterations;          /* Algorithm 1 outer passes (1 for other policies)  */
  int32_t n_per_doc;           /* documents sharded Per-Doc                        */
} fcp_plan_stats_t;

/*
 * fcp_plan -- build a CP sharding plan from document lengths.
 * Source: [FlashCP] §3.1 (problem: D = [d_1..d_n], CP size N, shards s_i with
 * prefix p_i, W_i = (2p_i+s_i+1)s_i/2, Eq. 1 and Eq. 2), §2.2-§2.3 (Llama3 CP,
 * Per-Doc chunk pairing), §3.2 (a shard needs its documents' prefix keys,
 * S^ excludes last shards), §3.3-§3.4 and Algorithm 1 (Whole-Doc, hybrid).
 *   doclens  host int32[n_docs], each >= 1, sum = T (the packed sequence).
 *   cp       N >= 1 shards.
 *   policy   FCP_POLICY_*.
 *   target_imbalance  R for FCP_POLICY_HYBRID / _HYBRID_TILES (ignored
 *            otherwise; > 0). The plan's reported imbalance is always by W.
 *   out      receives a new plan, to be freed with fcp_plan_free.
 * Errors: FCP_ERR_INVALID_ARG (null, n_docs < 1, a length < 1, T >= 2^31),
 *         FCP_ERR_INFEASIBLE (Llama3 needs T % 2N == 0; Whole-Doc and hybrid
 *         need T % N == 0).
 */
int fcp_plan(const int32_t* doclens, int32_t n_docs, int32_t cp, int32_t policy,
             double target_imbalance, fcp_plan_t** out);

void fcp_plan_free(fcp_plan_t* plan);

/* Shard j's pieces, needed and remote KV ranges ([FlashCP] §3.2). */
int fcp_plan_shard(const fcp_plan_t* plan, int32_t shard, fcp_shard_view* out);

/* Shard j's query token ids, ascending, into host idx[cap]; *n = count.
 * FCP_ERR_CAPACITY if cap is too small (then *n holds the needed count). */
int fcp_plan_query_indices(const fcp_plan_t* plan, int32_t shard, int32_t* idx,
                           int64_t cap, int64_t* n);

/* Whole-plan statistics (workload imbalance, Eq. 4 / Eq. 5 volumes). */
int fcp_plan_stats(const fcp_plan_t* plan, fcp_plan_stats_t* out);

/* Per-document policy flags: out[i] = 1 if doc i is sharded Per-Doc. */
int fcp_plan_per_doc_flags(const fcp_plan_t* plan, int32_t* out, int32_t n_docs);

/* ------------------------------------------------------------------------ */
/* Device plan                                                               */
/* ------------------------------------------------------------------------ */

/* Handle to a plan's work tables in caller-owned device memory. Filled by
 * fcp_plan_upload; treat the fields as read-only. */
typedef struct {
  const fcp_plan_t* host;      /* the plan uploaded; must outlive this handle      */
  const int32_t* base;         /* device buffer given to fcp_plan_upload          */
  int64_t bytes;
  int32_t n_shards;
  int32_t T;
  int64_t total_remote_rows;   /* rows of an all-shards kbuf/vbuf                  */
  int32_t tables[16];          /* int32 offsets of the tables inside base          */
  int32_t counts[16];          /* table lengths                                    */
} fcp_dev_plan;

/* Bytes needed to upload `plan` (a multiple of 256). */
int64_t fcp_plan_device_bytes(const fcp_plan_t* plan);

/*
 * fcp_plan_upload -- copy the plan's work tables (query tiles, key segments,
 * backward key tiles, gather runs) into dev_buf[bytes] on `stream`.
 * The copy reads host memory owned by `plan`: keep the plan alive until the
 * stream has passed the copy. Errors: FCP_ERR_CAPACITY if bytes is too small,
 * FCP_ERR_CUDA if the copy cannot be queued.
 */
int fcp_plan_upload(const fcp_plan_t* plan, void* dev_buf, int64_t bytes, void* stream,
                    fcp_dev_plan* out);

/*
 * fcp_plan_device_image -- copy the plan's work tables, exactly the bytes
 * fcp_plan_upload would send (fcp_plan_device_bytes of them), into host
 * memory dst[bytes]. The image holds offsets only, so it may be copied to any
 * 16-byte-aligned device buffer by the caller, e.g. from pinned memory with an
 * asynchronous copy that does not wait for the stream (a copy from pageable
 * memory, as fcp_plan_upload makes, can block the host until the stream has
 * drained). No CUDA call. Errors: FCP_ERR_INVALID_ARG for a null argument,
 * FCP_ERR_CAPACITY if bytes is too small.
 */
int fcp_plan_device_image(const fcp_plan_t* plan, void* dst, int64_t bytes);

/*
 * fcp_plan_bind -- fill `out` for a device buffer dev_buf[bytes] that holds
 * (or will hold, before any device call reads it) the plan's image, copied by
 * the caller. No CUDA call. Errors: FCP_ERR_INVALID_ARG for a null argument or
 * a dev_buf that is not 16-byte aligned, FCP_ERR_CAPACITY if bytes is too
 * small.
 */
int fcp_plan_bind(const fcp_plan_t* plan, const void* dev_buf, int64_t bytes, fcp_dev_plan* out);

/* ------------------------------------------------------------------------ */
/* Device operations                                                         */
/* ------------------------------------------------------------------------ */

typedef struct {
  int32_t T;      /* tokens of the packed sequence                     */
  int32_t hq;     /* query heads                                       */
  int32_t hkv;    /* KV heads                                          */
  int32_t d;      /* head dim, 64 or 128                               */
  float scale;    /* softmax scale; 0 selects 1/sqrt(d)                */
} fcp_dims;

/* Workspace the device calls on `plan` need, in bytes: an error word and the
 * attention kernels' work counter (set by each call before use), e4m3 copies
 * of Q, K and the received K rows with their scales (fcp_attn_fwd_qk8), the
 * backward's row statistics D_i = <dO_i, O_i> ([Hq][T] fp32), fp16 copies of
 * Q and dO ([T][Hq][d] each, the backward's tensor-core operands) and of V and
 * the plan's received V rows (the forward's P*V operands). The caller
 * zero-fills a new workspace once before its first call: the error word must
 * start at zero (fcp_get_device_status clears it after reporting an error),
 * and a one-shard backward reads the fp16 Q and dO rows of whole 128-row
 * tiles, rows of other shards included, which must hold finite values (their
 * probabilities are zero, but 0 * NaN is not); each call writes the rows of
 * its own shard before reading them. Calls that share a workspace must be
 * ordered on the GPU (one stream, or synchronised): two at once would race on
 * these contents. */
int64_t fcp_workspace_bytes(fcp_dims dims, const fcp_plan_t* plan);

/*
 * fcp_gather_kv -- sharding-aware KV exchange on one GPU ([FlashCP] §3.2: a
 * shard receives only the prefix keys of its documents that other shards
 * hold, compacted into one contiguous buffer without per-document padding).
 * Copies, for shard `shard` (or every shard if shard == -1), the rows of its
 * kv_remote ranges from K and V [T][Hkv][d] bf16 into kbuf, vbuf
 * [rows][Hkv][d] bf16, in ascending kv_remote order. For shard == -1 the
 * shards' buffers are concatenated (shard j starts at its kbuf_base); for one
 * shard, kbuf row 0 is its first remote row. row_bytes = Hkv*d*2.
 * Sizes (caller-owned, not checked here: the call takes no buffer sizes):
 * kbuf and vbuf hold at least plan->total_remote_rows rows for shard == -1,
 * or that shard's remote_rows (fcp_plan_shard) for one shard; the attention
 * calls read them with the same layout.
 */
int fcp_gather_kv(const void* k, const void* v, const fcp_dev_plan* plan, int32_t shard,
                  int32_t hkv, int32_t d, void* kbuf, void* vbuf, void* stream);

/*
 * fcp_attn_fwd -- document-masked attention forward for one shard (or all).
 * Source: [FlashCP] §2.1 and Fig. 1(a) (intra-document causal mask), §3.2
 * (a shard computes with its own keys plus the received prefix keys).
 * For every query i of the shard and head h (g = h / (Hq/Hkv)):
 *   s_ij = scale <q_ih, k_jg>, j in doc(i), j <= i, j in [kv_lo, kv_hi)
 *   LSE_ih = ln sum_j exp(s_ij), O_ih = sum_j exp(s_ij - LSE_ih) v_jg.
 * Keys owned by the shard are read from k/v at their global rows; remote keys
 * from kbuf/vbuf as laid out by fcp_gather_kv for the same `shard` value.
 *   kv_lo, kv_hi  restrict keys to a global block [kv_lo, kv_hi) (a ring
 *                 step); pass 0, T for the full key set.
 *   out_dtype     FCP_OUT_BF16: out is bf16; FCP_OUT_F32: fp32 partial.
 *   out, lse      written only at the shard's query rows. A row without any
 *                 key in the block gets O = 0 and LSE = -inf.
 *   ws            workspace of fcp_workspace_bytes(dims, plan) bytes.
 */
int fcp_attn_fwd(const void* q, const void* k, const void* v, const void* kbuf,
                 const void* vbuf, const fcp_dev_plan* plan, int32_t shard,
                 int32_t kv_lo, int32_t kv_hi, fcp_dims dims, int32_t out_dtype,
                 void* out, float* lse, void* ws, int64_t ws_bytes, void* stream);

/*
 * fcp_quant_e4m3 -- FP8 (OCP E4M3) copy of a bf16 array with one
 * power-of-two scale ("LLM Context Parallel in Production" lists FP8 among
 * the precisions of CP attention): out[i] = e4m3(x[i] * 2^k), k the largest
 * integer with max|x| * 2^k <= 448, rounded to nearest (ties to even) and
 * saturated to +-448; *scale_out = 2^k (device float). Scaling by a power of
 * two is exact, so out[i] / 2^k is the dequantised value.
 *   n        elements, a multiple of 8; x 16-byte aligned, out 8-byte aligned.
 *   scratch  4 bytes of device memory (4-byte aligned) for max|x|.
 */
int fcp_quant_e4m3(const void* x, int64_t n, void* out, float* scale_out, void* scratch, void* stream);

/*
 * fcp_attn_fwd_qk8 -- fcp_attn_fwd with the scores Q K^T computed on e4m3
 * copies of Q, K and the received K rows (fcp_quant_e4m3: Q with its own
 * scale, K and its received rows with K's), the product unscaled exactly
 * in the softmax; P V runs on fp16 operands as in fcp_attn_fwd. d = 128 only
 * (FCP_ERR_UNSUPPORTED otherwise). Arguments and results as fcp_attn_fwd;
 * the workspace (same size) holds the e4m3 copies. The result is the
 * attention of the dequantised Q and K with V.
 */
int fcp_attn_fwd_qk8(const void* q, const void* k, const void* v, const void* kbuf,
                     const void* vbuf, const fcp_dev_plan* plan, int32_t shard,
                     int32_t kv_lo, int32_t kv_hi, fcp_dims dims, int32_t out_dtype,
                     void* out, float* lse, void* ws, int64_t ws_bytes, void* stream);

/*
 * fcp_round_bf16 -- bf16 copy of an fp32 array, each element rounded to the
 * nearest bf16 value (ties to even). The final output of the forward is bf16
 * ([FlashCP] trains in bf16); a caller that keeps the fp32 output of
 * fcp_attn_fwd for the backward's D_i = <dO_i, O_i> rounds it once with this
 * call for its own use. Equals fcp_attn_fwd's FCP_OUT_BF16 output bit for bit.
 *   x    fp32 [n], out bf16 [n]; n a multiple of 8; both 16-byte aligned.
 * Errors: FCP_ERR_INVALID_ARG (n not a multiple of 8, null or misaligned
 * pointers when n > 0).
 */
int fcp_round_bf16(const float* x, int64_t n, void* out, void* stream);

/*
 * fcp_attn_fwd_ring -- the same forward in ring order, without a gathered
 * key buffer ([CPGuide] "Ring Attention": at step s of the ring, shard j
 * holds the KV block of shard (j - s) mod N and merges its partial result by
 * the online softmax; [FlashCP] §2.2 ("Reduced Kernel Efficiency") and §4
 * attribute a cost to this blockwise execution and its partial-result
 * processing, against the gather-then-compute design of fcp_gather_kv +
 * fcp_attn_fwd).
 * Every key a query needs is read from its owner's rows of k/v (owner = the
 * shard that holds that token in the plan), owners visited in ring order
 * (own rows first).
 *   ring_step -1: all owners in one pass, the softmax state carried across
 *             them (the fused ring: no partial results are stored). Output
 *             equals fcp_attn_fwd's up to the summation order.
 *             s in [0, N): only the keys of owner (j - s) mod N for each
 *             query of shard j -- the partial (O, LSE) of ring step s, to be
 *             combined with fcp_merge; a row with no such key gets O = 0,
 *             LSE = -inf.
 *   Other arguments as fcp_attn_fwd (no kbuf/vbuf, no key block). The
 *   workspace is the same (its received-row part is unused).
 */
int fcp_attn_fwd_ring(const void* q, const void* k, const void* v, const fcp_dev_plan* plan,
                      int32_t shard, int32_t ring_step, fcp_dims dims, int32_t out_dtype, void* out,
                      float* lse, void* ws, int64_t ws_bytes, void* stream);

/*
 * fcp_merge -- combine B partial results over disjoint key blocks
 * ([CPGuide] "Core Principle: Split Q, Circulate KV" and "Ring Attention":
 * online softmax keeps each block's row maximum and exponential sum).
 *   LSE = ln sum_b exp(LSE_b), O = sum_b exp(LSE_b - LSE) O_b.
 *   o_parts   fp32 [B][rows][hq][d]; lse_parts fp32 [B][hq][rows].
 *   out       bf16 [rows][hq][d]; lse_out fp32 [hq][rows].
 * A row empty in every block (all LSE_b = -inf) gets O = 0, LSE = -inf.
 * Limits: 1 <= B <= d/4 (32 for d = 128, 16 for d = 64), rows * hq < 2^30
 * (FCP_ERR_UNSUPPORTED otherwise).
 */
int fcp_merge(const float* o_parts, const float* lse_parts, int32_t B, int64_t rows,
              int32_t hq, int32_t d, void* out, float* lse_out, void* stream);

/*
 * fcp_merge_ring -- fcp_merge of the N ring-step partials of a plan, with the
 * check a distributed merge needs before it combines anything ([CPGuide]
 * "Ring Attention": shard j folds in the partial of every ring step; the
 * guide's go-live checklist asks that a lost or faulty rank be reported, not
 * silently absorbed). The partials are those of fcp_attn_fwd_ring(ring_step =
 * s) for every shard at once, fp32, one per step; part_step[b] (host) names
 * the ring step that produced partial b -- in a distributed run, the tag each
 * received partial carries.
 *   o_parts   fp32 [B][T][hq][d]; lse_parts fp32 [B][hq][T] (T = the plan's).
 *   out       bf16 [T][hq][d]; lse_out fp32 [hq][T].
 * Errors, all before any launch: FCP_ERR_MISSING_PART unless B equals the
 * plan's shard count N and part_step holds every step 0..N-1 exactly once (a
 * lost partial, a duplicated one, or a tag outside the ring); the errors of
 * fcp_merge otherwise.
 */
int fcp_merge_ring(const fcp_dev_plan* plan, const float* o_parts, const float* lse_parts,
                   const int32_t* part_step, int32_t B, int32_t hq, int32_t d, void* out,
                   float* lse_out, void* stream);

/*
 * fcp_attn_bwd -- exact gradient of fcp_attn_fwd (full key set) for one shard
 * or all. P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D_i = <dO_i, O_i>,
 * dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q. [FlashCP] Fig. 6 /
 * Eq. 4 name the backward pass and the ReduceScatter of KV gradients; here
 * that reduction is a scatter-add at the keys' global rows.
 *   out, lse  the forward's output and LSE at the shard's rows; out_dtype
 *             (FCP_OUT_BF16 or FCP_OUT_F32) says how `out` is stored. D_i is
 *             formed from it, so an fp32 `out` gives the more exact gradient.
 *   dout      bf16 [T][Hq][d].
 *   dq        fp32 [T][Hq][d]: written (=) at the shard's query rows.
 *   dk, dv    fp32 [T][Hkv][d]: ACCUMULATED (+=) at global key rows, remote
 *             keys included; zero them before the first shard.
 */
int fcp_attn_bwd(const void* q, const void* k, const void* v, const void* kbuf,
                 const void* vbuf, const void* out, int32_t out_dtype, const float* lse,
                 const void* dout, const fcp_dev_plan* plan, int32_t shard, fcp_dims dims,
                 float* dq, float* dk, float* dv, void* ws, int64_t ws_bytes, void* stream);

/* Size of the device array that fcp_attn_fwd_noalloc uses as its scratch. */
#define FCP_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * fcp_attn_fwd_noalloc -- fcp_attn_fwd without a caller workspace and without
 * any device allocation. The paper has no counterpart: this entry point exists
 * for callers that cannot allocate device memory at call time -- for example a
 * serving or training process that reserved all device memory up front (or
 * handed it to another allocator) and forbids allocation on its request path,
 * where a cudaMalloc would synchronise the device and can fail once memory is
 * fragmented.
 *   Arguments, layouts and results are those of fcp_attn_fwd, minus ws and
 *   ws_bytes. The scratch (an error word, the kernel's work counter and fp16
 *   copies of V and of the received V rows) is one file-scope device array of
 *   FCP_NOALLOC_SCRATCH_BYTES bytes, held by every GPU that loads the library
 *   until the process exits.
 *   Limit: 256 + align256(T*Hkv*d*2) + align256(R*Hkv*d*2) bytes must fit in
 *   that array, R = the received rows of this call (all shards' for shard ==
 *   -1); larger inputs return FCP_ERR_CAPACITY before anything is launched.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture. Nothing is allocated, by this library or through any allocating
 *   library routine.
 *   Every call shares the array and overwrites what the previous call left in
 *   it (the error word is cleared at the start of each call): calls whose work
 *   can overlap on the GPU -- on different streams without ordering -- race and
 *   must not be issued. Device-side timeouts of this variant are recorded in
 *   the shared array only, and so is an input of V (or of the received V rows)
 *   beyond the fp16 range |x| > 65504, which fcp_attn_fwd reports as
 *   FCP_ERR_UNSUPPORTED: this variant gives inf/NaN in O and LSE for such
 *   input without an error. Use fcp_attn_fwd with a workspace to detect both.
 */
int fcp_attn_fwd_noalloc(const void* q, const void* k, const void* v, const void* kbuf,
                         const void* vbuf, const fcp_dev_plan* plan, int32_t shard,
                         int32_t kv_lo, int32_t kv_hi, fcp_dims dims, int32_t out_dtype,
                         void* out, float* lse, void* stream);

/*
 * fcp_get_device_status -- read the workspace error word (synchronizes the
 * stream). FCP_ERR_TIMEOUT if a bounded pipeline wait expired in a previous
 * call on this workspace; FCP_ERR_UNSUPPORTED if an input exceeded the fp16
 * range of its tensor-core operands (|x| > 65504: V in the forward, Q, dO, K
 * or V in the backward); FCP_ERR_INVALID_ARG if, in the checked build of the
 * library (compiled with FCP_DEVICE_CHECKS=1), a kernel found a plan-table
 * index out of range and skipped that work unit; FCP_OK otherwise. Clears
 * the word.
 */
int fcp_get_device_status(void* ws, void* stream);

/* Limit of every bounded device wait, in nanoseconds (default 2 s; 0 restores
 * the default). A negative value makes a wait give up at its first
 * unsatisfied try: a test hook that exercises the timeout path (the kernel
 * sets the error word, drains its copies and MMAs, frees TMEM and returns)
 * without a hang. */
void fcp_debug_set_wait_limit(int64_t ns);

/*
 * fcp_debug_rescale_events -- diagnostic read of the forward kernels' rescale
 * counter in the workspace header (synchronizes the stream, then clears it).
 * The online softmax ([CPGuide] "Core Principle: Split Q, Circulate KV")
 * keeps a running row maximum m; the kernels rescale the accumulated O only
 * when a later key tile raises m by more than 2^8 (log2 units), so that the
 * unnormalised probabilities stay <= 2^8. *count receives the number of such
 * rescales (one count per 32-row warp and event) made by fcp_attn_fwd,
 * fcp_attn_fwd_qk8 and fcp_attn_fwd_ring on this workspace since the last
 * read; a new, zero-filled workspace starts at 0. Errors: FCP_ERR_INVALID_ARG
 * for a null argument, FCP_ERR_CUDA if the read fails.
 */
int fcp_debug_rescale_events(void* ws, void* stream, int64_t* count);

#ifdef __cplusplus
}
#endif
#endif /* FCP_H */
