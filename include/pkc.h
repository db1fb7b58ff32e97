/*
 * pkc.h -- C ABI of libpkc, shared-prefix ("cascade") batch-decode attention
 * over a paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * Every attention call returns attention STATES: for a query q and a set I
 * of cached keys/values,
 *     s_i  = sm_scale * (q . k_i)
 *     LSE  = s(I) = log sum_{i in I} exp(s_i)          (natural log)
 *     O    = v(I) = sum_{i in I} exp(s_i - s(I)) v_i
 * and states of disjoint sets combine with the merge operator (+)
 * (FlashInfer tutorial "Attention States and Recursive Attention", the
 * definitions of s(I), v(I) and the binary / n-ary merge equations; blog
 * "Cascade Inference: Memory Bandwidth Efficient Shared Prefix Batch
 * Decoding", section "Recursive Attention").  An empty set has the identity
 * state O = 0, LSE = -inf.
 *
 * Conventions shared by all calls
 *  - Pointers named *_host are host memory; every other tensor pointer is
 *    device memory.  The caller owns every buffer; the library allocates no
 *    device memory.
 *  - Tensors are dense and row-major (C order) in the layouts stated below.
 *    Device pointers to 16-bit tensors must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *    device work is enqueued on it asynchronously; no call synchronises the
 *    host except pkc_device_status.
 *  - Return value: PKC_OK or a pkc_status code; on error nothing has been
 *    enqueued and pkc_last_error() describes the problem.  No call aborts
 *    the process or traps on the device.  Faults found by kernels (a bad
 *    page id, a plan that does not match cache_seqlens, a wait that timed
 *    out) are recorded in the workspace status word, read with
 *    pkc_device_status.
 *  - head_dim must be 128 for the attention calls (PKC_ERR_UNSUPPORTED
 *    otherwise).  num_qo_heads must be a multiple of num_kv_heads; query
 *    head h reads KV head h / (num_qo_heads / num_kv_heads) (GQA head
 *    groups, FlashInfer MLSys'25 notes, appendix A "head-group fusion").
 */
#ifndef PKC_H_
#define PKC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKC_OK = 0,
  PKC_ERR_INVALID_ARG = 1, /* bad pointer, size, stride or dtype */
  PKC_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head_dim) */
  PKC_ERR_WORKSPACE = 3,   /* workspace too small or misaligned */
  PKC_ERR_BLOCK_TABLE = 4, /* device: page id < 0 or >= num_pages in use */
  PKC_ERR_CUDA = 5,        /* a CUDA runtime call failed */
  PKC_ERR_TIMEOUT = 6,     /* device: a bounded wait ran out */
  PKC_ERR_PLAN = 7         /* plan buffer invalid or inconsistent */
} pkc_status;

/* Element types.  PKC_E4M3 (8-bit float: 1 sign, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinities, S.1111.111 is NaN; largest
 * finite 448) is accepted only for a KV cache (pkc_paged_decode_state_fp8). */
typedef enum { PKC_F32 = 0, PKC_F16 = 1, PKC_BF16 = 2, PKC_E4M3 = 3 } pkc_dtype;

/* Library version, major * 10000 + minor * 100 + patch. */
int pkc_version(void);

/* Message for the last error returned on the calling thread ("" if none). */
const char* pkc_last_error(void);

/* ------------------------------------------------------------------------
 * Merge operator
 * ---------------------------------------------------------------------- */

/*
 * Binary merge of two attention states per (token, head):
 *   v_out = (v_a e^{s_a} + v_b e^{s_b}) / (e^{s_a} + e^{s_b})
 *   s_out = log(e^{s_a} + e^{s_b})
 * ("Attention States and Recursive Attention", binary merge equation),
 * evaluated with the larger s subtracted first; a side with s = -inf is
 * empty and two empty sides give (0, -inf).
 *
 * v_a, v_b, v_out: [n_tokens, n_heads, head_dim] of v_dtype (F32, F16 or
 * BF16); s_a, s_b, s_out: [n_tokens, n_heads] float32 natural-log LSE.
 * v_out may be v_a (in place); s_out may be s_a.  head_dim * element size
 * must be a multiple of 16 bytes and all pointers 16-byte aligned.
 */
int pkc_merge_state(const void* v_a, const float* s_a, const void* v_b,
                    const float* s_b, void* v_out, float* s_out,
                    int64_t n_tokens, int n_heads, int head_dim, int v_dtype,
                    void* stream);

/*
 * n-ary merge over axis 1 ("Attention States and Recursive Attention",
 * n-ary merge equation): v_out = sum_i softmax_i(s_i) v_i,
 * s_out = log sum_i exp(s_i).  v: [n_tokens, n_states, n_heads, head_dim]
 * of v_dtype; s: [n_tokens, n_states, n_heads] float32; v_out
 * [n_tokens, n_heads, head_dim]; s_out [n_tokens, n_heads].  n_states >= 1.
 */
int pkc_merge_states(const void* v, const float* s, void* v_out, float* s_out,
                     int64_t n_tokens, int n_states, int n_heads, int head_dim,
                     int v_dtype, void* stream);

/*
 * The n-ary merge above with a result of another element type: float32
 * states (v_dtype PKC_F32) merged into an fp16 or bf16 v_out (out_dtype),
 * the weighted sum formed in float32 and rounded once (nearest even).
 * Equal types are pkc_merge_states.  This is the last step of a KV-sharded
 * decode ("Attention States and Recursive Attention", Applications: the
 * states of KV subsets computed on different devices are merged in any
 * order): the gathered float32 states [n_states, B*Hq, 128] of the shards
 * are a [1, n_states, B*Hq, 128] input.  head_dim / 4 must divide 32 or be
 * a multiple of 32; PKC_ERR_INVALID_ARG for other type pairs.
 */
int pkc_merge_states_to(const void* v, const float* s, void* v_out,
                        float* s_out, int64_t n_tokens, int n_states,
                        int n_heads, int head_dim, int v_dtype, int out_dtype,
                        void* stream);

/* ------------------------------------------------------------------------
 * Load-balanced plan (host only)
 * ---------------------------------------------------------------------- */

/*
 * The plan is the CPU-side schedule of KV chunks onto CTAs (FlashInfer
 * MLSys'25 notes, A3 "load-balanced scheduling", steps 1-7, and appendix D
 * "split-K direct write"):
 *   1. a work unit is a (request, query tile of tile_q rows), request-major;
 *   2. L_kv = ceil(sum_i ceil(qo_len_i / tile_q) * kv_len_i / num_ctas), >= 1;
 *   3. each unit's KV is cut into consecutive chunks of at most L_kv tokens,
 *      numbered w unit by unit (a unit with kv_len 0 has no chunk);
 *   4. chunks are sorted longest first (equal lengths keep ascending w);
 *   5. a min-priority queue of (cost, CTA index) starts at (0, c) for every
 *      CTA; each chunk goes to the popped CTA, whose cost grows by
 *      alpha * l_q + beta * l_kv (l_q = the tile's query rows);
 *   6. a unit with one chunk writes its output directly; chunks of units
 *      with >= 2 chunks get partial slots numbered in w order, and a
 *      contraction merges them in ascending KV order.
 *
 * The plan is an int32 buffer of pkc_plan_words(...) words; its layout is
 * given by the PKC_PLAN_* header indices below (all offsets in words from
 * the start of the buffer):
 *   cta_indptr[num_ctas + 1]    CSR: CTA c runs work cta_work[...] in pop order
 *   cta_work[n_work]            work index w
 *   work_unit, work_kv_begin, work_kv_end, work_partial [n_work] each
 *                               (work_partial = -1: direct write)
 *   unit_req, unit_qtile, unit_kv_len, unit_n_chunks, unit_partial_begin
 *                               [n_units] each (partial_begin -1 if unsplit)
 *   unit_list[n_split + n_empty] split units then empty units, unit order
 *   cta_cost[num_ctas]          final cost per CTA, as float64 (2 words each)
 *   work_order[n_work]          the chunks w in the order of step 4
 *   order_rec[n_work][4]        for work_order[i]: (unit, kv_begin, kv_end,
 *                               partial), 16-byte aligned; the queue a
 *                               dynamically scheduled decode takes chunks
 *                               from (pkc_set_decode_schedule)
 * The plan depends on lengths only: it is the same for every head.
 */
enum {
  PKC_PLAN_MAGIC = 0, /* == PKC_PLAN_MAGIC_VALUE */
  PKC_PLAN_TOTAL_WORDS,
  PKC_PLAN_NUM_CTAS,
  PKC_PLAN_TILE_Q,
  PKC_PLAN_N_REQ,
  PKC_PLAN_KV_CHUNK, /* L_kv */
  PKC_PLAN_N_UNITS,
  PKC_PLAN_N_WORK,
  PKC_PLAN_N_PARTIALS,
  PKC_PLAN_N_SPLIT,
  PKC_PLAN_N_EMPTY,
  PKC_PLAN_OFF_CTA_INDPTR,
  PKC_PLAN_OFF_CTA_WORK,
  PKC_PLAN_OFF_WORK_UNIT,
  PKC_PLAN_OFF_WORK_KV_BEGIN,
  PKC_PLAN_OFF_WORK_KV_END,
  PKC_PLAN_OFF_WORK_PARTIAL,
  PKC_PLAN_OFF_UNIT_REQ,
  PKC_PLAN_OFF_UNIT_QTILE,
  PKC_PLAN_OFF_UNIT_KV_LEN,
  PKC_PLAN_OFF_UNIT_N_CHUNKS,
  PKC_PLAN_OFF_UNIT_PARTIAL_BEGIN,
  PKC_PLAN_OFF_UNIT_LIST,
  PKC_PLAN_OFF_CTA_COST,
  PKC_PLAN_OFF_WORK_ORDER,
  PKC_PLAN_OFF_ORDER_REC,
  PKC_PLAN_HEADER_WORDS = 32
};
#define PKC_PLAN_MAGIC_VALUE 0x504b4331 /* "PKC1" */

/*
 * Words needed for a plan of n requests.  qo_len_host [n] may be NULL for
 * decode (every request has one query row).  The bound uses
 * n_work <= num_ctas + n_units.
 */
int pkc_plan_words(const int32_t* qo_len_host, int n, int tile_q,
                   int num_ctas, size_t* words);

/*
 * Compute the plan on the host into plan_host [plan_words].  qo_len_host
 * may be NULL (all 1); kv_len_host [n] >= 0.  Deterministic: equal inputs
 * give bit-identical buffers.  Pinned host memory for plan_host makes the
 * later upload truly asynchronous.
 */
int pkc_plan(const int32_t* qo_len_host, const int32_t* kv_len_host, int n,
             int tile_q, int num_ctas, double alpha, double beta,
             int32_t* plan_host, size_t plan_words);

/*
 * Copy a plan into the plan region of a workspace (cudaMemcpyAsync on
 * `stream`).  plan_host must stay valid until the copy has run.  Every
 * planned call reads the plan from the workspace: it must have been
 * uploaded there (pkc_workspace_init clears only the status block).
 */
int pkc_plan_upload(const int32_t* plan_host, void* workspace,
                    size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Workspace
 * ---------------------------------------------------------------------- */

/*
 * Bytes of device workspace for a problem.  The workspace holds, in order
 * and each 256-byte aligned: a status block (256 B); the plan region
 * (pkc_plan_words for `batch` decode requests and num_ctas CTAs, 0 when
 * num_ctas is 0); the suffix states [batch, Hq, D+1] float32; the suffix
 * partials [2 * num_ctas, Hq, D+1] float32 (appendix D bound
 * 2 * #CTA * T_q * H * (D+1) with T_q = 1); the fused contraction's
 * arrival counters [batch, Hq] int32 (zeroed by every call that uses them);
 * and prefix_splits copies of [batch, Hq, D+1] float32 for prefix partial
 * states.
 *   num_ctas: CTAs of the plan the calls will use (0 if none).
 *   prefix_splits: partial-state slots for the shared prefix (0 if no
 *                  prefix).  The prefix stage spreads the KV tiles of all
 *                  (128-row query tile, KV head) pairs evenly over one
 *                  thread block per SM; a pair cut between blocks needs one
 *                  slot per piece (at most 1 + ceil(pair tiles / tiles per
 *                  block)).  With fewer slots the calls use fewer blocks;
 *                  4 covers the workloads of the pages, 64 any problem.
 */
int pkc_workspace_size(int batch, int num_qo_heads, int head_dim,
                       int num_ctas, int prefix_splits, size_t* bytes);

/* Zero the status block.  Call once after allocating a workspace. */
int pkc_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Read (and clear) the device status word: *status = PKC_OK or the first
 * PKC_ERR_BLOCK_TABLE / PKC_ERR_PLAN / PKC_ERR_TIMEOUT a kernel recorded
 * since the last read.  Synchronises `stream`.
 */
int pkc_device_status(void* workspace, void* stream, int32_t* status);

/* ------------------------------------------------------------------------
 * Attention states
 * ---------------------------------------------------------------------- */

/*
 * Single-query paged decode state (blog "Cascade Inference", step 2 of the
 * algorithm; Hugging Face "Paged attention", decoding path).  For every
 * request b and query head h, the state of q[b, h] over the
 * cache_seqlens[b] cached tokens of b:
 *   q        [batch, num_qo_heads, 128] of dtype (F16 or BF16)
 *   k_cache, v_cache [num_pages, page_size, num_kv_heads, 128] of dtype
 *   block_table [batch, block_table_stride] int32: token t of request b is
 *            in page block_table[b, t / page_size], slot t % page_size;
 *            entries past the last used page are never read (-1 allowed)
 *   cache_seqlens [batch] int32 >= 0
 *   plan_host: NULL, or a plan of these lengths (tile_q 1) that was
 *            uploaded into this workspace with pkc_plan_upload.  NULL runs
 *            one chunk per request.  The kernels compare the workspace's
 *            copy (magic word, total words, request count) with plan_host
 *            before reading it: a plan never uploaded is reported as
 *            PKC_ERR_PLAN on the device, and nothing is computed.
 *   o        [batch, num_qo_heads, 128] of dtype; lse [batch, num_qo_heads]
 *            float32 natural log.  A request with 0 tokens gets (0, -inf).
 */
int pkc_paged_decode_state(const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* block_table,
                           int block_table_stride,
                           const int32_t* cache_seqlens, int batch,
                           int num_qo_heads, int num_kv_heads, int head_dim,
                           int page_size, int64_t num_pages, float sm_scale,
                           const int32_t* plan_host, void* workspace,
                           size_t workspace_bytes, void* o, float* lse,
                           int dtype, void* stream);

/*
 * Paged decode that allocates nothing (the pages have no counterpart; this
 * is a deployment convenience).  Same computation, arguments and outputs as
 * pkc_paged_decode_state, for callers that cannot call cudaMalloc or own no
 * spare device memory for a workspace -- e.g. code running inside another
 * framework's pre-reserved memory pool, or under a fixed memory budget.
 * The split-KV scratch (status word, uploaded plan, partial states) lives in
 * an 8 MiB array declared in device memory by the library itself.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  Under CUDA's lazy
 *     module loading (the default) that lookup is also when the driver
 *     places the 8 MiB array in that device's memory, where it stays until
 *     the process exits.  So make that first call before any stream
 *     capture and before the caller's memory pool reserves the rest of the
 *     device; a call with batch 0 (no other pointer is read) does only the
 *     set-up.
 *   - The plan (plan_host, as in pkc_paged_decode_state, or NULL) is copied
 *     into the array by this call (cudaMemcpyAsync from the host buffer,
 *     in stream order); no pkc_plan_upload is needed.  If the call is made
 *     inside a stream capture, that copy becomes a graph node that reads
 *     plan_host at every replay: the buffer must then stay alive, and its
 *     contents at replay time are the plan used.  It needs
 *     256 + plan + 2 * num_ctas * num_qo_heads * 129 * 4 bytes (rounded to
 *     256-byte blocks) <= 8 MiB, else PKC_ERR_WORKSPACE with the numbers.
 *   - Every call shares the one array and leaves its contents behind; the
 *     call clears the status word itself.  Calls whose kernels overlap on
 *     the GPU (different streams, or different host threads) race on the
 *     array: serialise them.
 *   - device_status: NULL, or a device int32 that receives the call's status
 *     word (PKC_OK or the PKC_ERR_* a kernel recorded) in stream order.
 * Calls no cudaMalloc / cudaFree and no allocating library routine.
 */
int pkc_paged_decode_state_noalloc(
    const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_table, int block_table_stride,
    const int32_t* cache_seqlens, int batch, int num_qo_heads,
    int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
    float sm_scale, const int32_t* plan_host, void* o, float* lse,
    int32_t* device_status, int dtype, void* stream);

/*
 * Paged decode state over an FP8 KV cache (MLSys'25 notes, appendix F,
 * "FP8-FP16 mixed-precision attention": queries and outputs stay fp16, the
 * KV cache is stored in fp8).  Same computation, plan and workspace as
 * pkc_paged_decode_state, with:
 *   q [batch, num_qo_heads, 128] fp16;  o [batch, num_qo_heads, 128] fp16
 *   k_cache, v_cache [num_pages, page_size, num_kv_heads, 128] of one-byte
 *            e4m3 codes (PKC_E4M3)
 *   k_scale, v_scale > 0, finite: the cached values are k_scale * e4m3(code)
 *            and v_scale * e4m3(code) (one scale per tensor; 1 for codes
 *            stored unscaled)
 * so the scores are sm_scale * k_scale * (q . e4m3(k)) and O is v_scale
 * times the softmax-weighted sum of e4m3(v).  The codes are widened to
 * fp16 exactly; products accumulate in fp32.  page_size must be a power of
 * two with min(page_size, 16) * H >= 8, H = the largest of 8, 4, 2, 1 that
 * divides num_kv_heads (else PKC_ERR_UNSUPPORTED).  Slots outside a
 * request's sequence are never used, whatever bytes they hold.
 */
int pkc_paged_decode_state_fp8(const void* q, const void* k_cache,
                               const void* v_cache,
                               const int32_t* block_table,
                               int block_table_stride,
                               const int32_t* cache_seqlens, int batch,
                               int num_qo_heads, int num_kv_heads,
                               int head_dim, int page_size, int64_t num_pages,
                               float sm_scale, float k_scale, float v_scale,
                               const int32_t* plan_host, void* workspace,
                               size_t workspace_bytes, void* o, float* lse,
                               void* stream);

/*
 * In-place append of one new token per request to the paged cache
 * (Hugging Face "Paged attention", decoding path: the next token of request
 * b is written to page block_table[b][len / page_size], slot
 * len % page_size, len = cache_seqlens[b]; then the length grows by one).
 *   k_new, v_new [batch, num_kv_heads, 128] of dtype: the new token's K, V
 *   k_cache, v_cache [num_pages, page_size, num_kv_heads, 128] of dtype,
 *            written in place
 *   block_table [batch, block_table_stride] int32: the caller allocates
 *            the next page before the token that starts it
 *   cache_seqlens [batch] int32, incremented in place (device memory)
 *   append_mask: NULL (every request appends) or [batch] uint8 in device
 *            memory: only requests with a nonzero entry append
 *   dtype: PKC_F16, PKC_BF16 or PKC_E4M3 (an fp8 cache: k_new / v_new are
 *            e4m3 codes too)
 * A request whose next page id is negative or >= num_pages is skipped (its
 * cache and length untouched) and PKC_ERR_BLOCK_TABLE is recorded in the
 * workspace status word.  Every pointer except the mask must be 16-byte
 * aligned.
 */
int pkc_append_kv(const void* k_new, const void* v_new, void* k_cache,
                  void* v_cache, const int32_t* block_table,
                  int block_table_stride, int32_t* cache_seqlens,
                  const uint8_t* append_mask, int batch, int num_kv_heads,
                  int head_dim, int page_size, int64_t num_pages, int dtype,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Multi-query prefix state (blog "Cascade Inference", step 1 of the
 * algorithm): every request's queries against the KV of the shared prefix
 * of its group, on the tensor cores (tcgen05, TMEM accumulators).
 *   q [batch, num_qo_heads, 128] of dtype
 *   k_prefix, v_prefix [L, num_kv_heads, 128] of dtype, L = last indptr
 *   prefix_kv_indptr_host [n_prefix + 1]: prefix j is tokens
 *            indptr[j] .. indptr[j+1]-1
 *   prefix_req_indptr_host [n_prefix + 1]: requests indptr[j] ..
 *            indptr[j+1]-1 share prefix j (cumulative-length convention of
 *            Hugging Face "Paged attention", varlen path); requests outside
 *            every group get the empty state
 *   o [batch, num_qo_heads, 128] float32; lse [batch, num_qo_heads] float32
 * 1 <= n_prefix <= 256.  Uses the prefix-partials region of the workspace.
 */
int pkc_prefix_attention_state(
    const void* q, const void* k_prefix, const void* v_prefix,
    const int32_t* prefix_kv_indptr_host,
    const int32_t* prefix_req_indptr_host, int n_prefix, int batch,
    int num_qo_heads, int num_kv_heads, int head_dim, float sm_scale,
    void* workspace, size_t workspace_bytes, float* o, float* lse, int dtype,
    void* stream);

/*
 * Cascade decode (blog "Cascade Inference", the three-step algorithm):
 * prefix state (tensor cores) (+) paged suffix state (load-balanced split
 * KV) -> final O [batch, num_qo_heads, 128] of dtype and LSE [batch,
 * num_qo_heads] float32, equal to attention over prefix u suffix.
 * Arguments as in the two calls above; cache_seqlens counts suffix tokens
 * only; plan_host as in pkc_paged_decode_state.
 * The prefix and suffix stages do not depend on each other: the three
 * kernels go on `stream` as a chain of programmatic dependents, so that the
 * suffix decode runs next to the prefix kernel and each waits in hardware
 * for the grid before it (the decode only before its blocks exit).  The call
 * stays ordered on `stream` after the work already queued there, under
 * CUDA-graph capture too; the library creates no stream.
 */
int pkc_cascade_decode(
    const void* q, const void* k_prefix, const void* v_prefix,
    const int32_t* prefix_kv_indptr_host,
    const int32_t* prefix_req_indptr_host, int n_prefix, const void* k_cache,
    const void* v_cache, const int32_t* block_table, int block_table_stride,
    const int32_t* cache_seqlens, int batch, int num_qo_heads,
    int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
    float sm_scale, const int32_t* plan_host, void* workspace,
    size_t workspace_bytes, void* o, float* lse, int dtype, void* stream);

/*
 * The cascade decode above returning the attention state unrounded: o is
 * float32 [batch, num_qo_heads, 128] (every other argument as in
 * pkc_cascade_decode, q and the caches of dtype).  For states that are
 * merged further with (+) -- a KV-sharded decode, where each device computes
 * the state of its part of every request's keys ("Attention States and
 * Recursive Attention", Applications) -- so the result is rounded only once,
 * after the last merge.
 */
int pkc_cascade_decode_state(
    const void* q, const void* k_prefix, const void* v_prefix,
    const int32_t* prefix_kv_indptr_host,
    const int32_t* prefix_req_indptr_host, int n_prefix, const void* k_cache,
    const void* v_cache, const int32_t* block_table, int block_table_stride,
    const int32_t* cache_seqlens, int batch, int num_qo_heads,
    int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
    float sm_scale, const int32_t* plan_host, void* workspace,
    size_t workspace_bytes, float* o, float* lse, int dtype, void* stream);

/*
 * Multi-level cascade decode: the cascade above with prefix groups given as
 * request ranges that may overlap.  Group j holds requests
 * prefix_req_begin[j] <= b < prefix_req_end[j] and prefix tokens
 * prefix_kv_indptr[j] .. prefix_kv_indptr[j+1]-1 of k/v_prefix; a request
 * attends to the prefixes of every group holding it (e.g. level 0: one
 * system prompt for all requests; level 1: a prompt per request group),
 * then to its own cached tokens.  The state of the union is the (+) of the
 * parts' states (tutorial "Attention States and Recursive Attention"), so
 * each group is computed once for all its requests, as in the two-level
 * cascade (blog "Cascade Inference").  Other arguments as in
 * pkc_cascade_decode.  Groups that share a request use disjoint partial
 * slots: the workspace's prefix_splits must cover, for every request, the
 * slots of all its groups (else fewer prefix blocks are used, and
 * PKC_ERR_WORKSPACE when even one block per group does not fit).
 * 1 <= n_prefix <= 256; 0 <= begin <= end <= batch.
 */
int pkc_cascade_decode_multilevel(
    const void* q, const void* k_prefix, const void* v_prefix,
    const int32_t* prefix_kv_indptr_host, const int32_t* prefix_req_begin_host,
    const int32_t* prefix_req_end_host, int n_prefix, const void* k_cache,
    const void* v_cache, const int32_t* block_table, int block_table_stride,
    const int32_t* cache_seqlens, int batch, int num_qo_heads,
    int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
    float sm_scale, const int32_t* plan_host, void* workspace,
    size_t workspace_bytes, void* o, float* lse, int dtype, void* stream);

/*
 * Cascade decode with the shared prefixes kept in the page pool (MLSys'25
 * notes, A3 "composable formats": the prefix is a block of the same paged
 * KV, read in place, not copied out).  As pkc_cascade_decode_multilevel,
 * except:
 *   prefix_pages: device int32 page ids into k_cache / v_cache; group j's
 *            prefix tokens are, in order, the slots of pages
 *            prefix_pages[prefix_page_indptr[j] .. prefix_page_indptr[j+1]-1]
 *            (the last page filled only up to the group's length)
 *   prefix_page_indptr_host [n_prefix + 1]: cumulative page counts; group j
 *            needs at least ceil(len_j / page_size) pages, len_j =
 *            prefix_kv_indptr[j+1] - prefix_kv_indptr[j]
 * page_size must divide 128 and be >= 8 (PKC_ERR_UNSUPPORTED otherwise).
 * A page id < 0 or >= num_pages in a list is read as zeros and recorded as
 * PKC_ERR_BLOCK_TABLE.  Slots past a group's length may hold anything.
 */
int pkc_cascade_decode_paged_prefix(
    const void* q, const int32_t* prefix_pages,
    const int32_t* prefix_page_indptr_host, const int32_t* prefix_kv_indptr_host,
    const int32_t* prefix_req_begin_host, const int32_t* prefix_req_end_host,
    int n_prefix, const void* k_cache, const void* v_cache,
    const int32_t* block_table, int block_table_stride,
    const int32_t* cache_seqlens, int batch, int num_qo_heads,
    int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
    float sm_scale, const int32_t* plan_host, void* workspace,
    size_t workspace_bytes, void* o, float* lse, int dtype, void* stream);

/* ------------------------------------------------------------------------
 * Stage timing
 * ---------------------------------------------------------------------- */

/*
 * Optional timing hook for the calling thread.  When events is non-NULL,
 * the NEXT pkc_cascade_decode call on this thread records events[0] on its
 * stream right before its first kernel (after the host builds that kernel's
 * TMA descriptors), then events[1], events[2], events[3]
 * after the prefix, suffix-decode and contraction kernels; the hook is then
 * cleared.  A timed call runs its stages one after the other on `stream`
 * (the decode does not overlap the prefix), so that each pair of events
 * brackets one kernel.
 * events: n_events >= 4 cudaEvent_t handles created by the caller; NULL
 * clears the hook.
 */
int pkc_set_stage_events(void* const* events, int n_events);

/*
 * Diagnostics: the failure path of the kernels' bounded waits, without a
 * fault.  Launches one block on `stream` whose thread waits on an mbarrier
 * that nothing arrives at, through the bounded wait all kernels use.  After
 * the limit (2 s of %globaltimer) the wait records PKC_ERR_TIMEOUT in the
 * workspace status word and returns; the kernel then ends normally and the
 * context stays usable.  *gave_up_host receives 1 if the wait gave up as
 * designed (0 otherwise); the call synchronises `stream`.  The workspace
 * needs PKC status bytes only (pkc_workspace_size(0, 1, ...)).
 */
int pkc_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int32_t* gave_up_host,
                              void* stream);

/*
 * Kernel used by the paged decode over a 16-bit cache (process-wide):
 *   0 = automatic (default): tensor-core kernel for grouped heads
 *       (num_qo_heads / num_kv_heads >= 2), CUDA-core kernel otherwise
 *   1 = always the CUDA-core kernel
 *   2 = the tensor-core kernel wherever it applies (page size a power of
 *       two, min(page_size, 16) * heads per block >= 8), else CUDA cores
 * Both compute the same states; the switch exists for measurement and
 * tests.  An FP8 cache always uses the tensor-core kernel.  Returns
 * PKC_ERR_INVALID_ARG for any other value.
 */
int pkc_set_decode_kernel(int which);

/*
 * Schedule of a planned paged decode (process-wide):
 *   1 = dynamic (default): one block per planned CTA; the blocks take the
 *       plan's chunks (x the KV-head groups) from a queue in the plan's
 *       longest-first order (order_rec), so blocks that run ahead take the
 *       short chunks at the end and all finish together.  The queue's
 *       counters live in the workspace's status block; the last block resets
 *       them, so a workspace must not be shared by two decodes in flight.
 *   0 = static: block c runs CTA c's list of the plan (the pages' greedy
 *       assignment), one block per (CTA, KV-head group).
 * The states are the same either way; chunks and partial slots come from the
 * plan.  Returns PKC_ERR_INVALID_ARG for any other value.
 */
int pkc_set_decode_schedule(int dynamic);

/*
 * Where split states are contracted into the output (process-wide):
 *   0 = (default) a standalone contraction kernel after the attention
 *       kernels, launched as a programmatic dependent of the suffix decode:
 *       its blocks start while the decode's last blocks run, load the prefix
 *       pieces and plan words, and wait in hardware (griddepcontrol.wait)
 *       for the decode grid before reading the suffix states.
 *   2 = the same kernel launched plainly after the decode (for measurement).
 *   1 = fused: the attention kernels do it themselves (MLSys'25
 *       notes, A3: attention and contraction in one persistent kernel).
 *       Every kernel that writes a state that is not yet a final output --
 *       a chunk's partial state, a cascade's suffix state, a prefix piece --
 *       adds one to the arrival counter of its (request, KV head) pair;
 *       the warp whose count is the pair's last merges the pair's sources
 *       with (+) and writes the final O and LSE.  No kernel waits for
 *       another.  A planned pkc_paged_decode_state is then one kernel
 *       launch, a cascade the prefix and decode kernels.  Each such call
 *       first zeroes its counters (cudaMemsetAsync of batch * num_kv_heads
 *       int32 in the workspace).  Cascades with more than 16 prefix groups
 *       use the standalone kernel.
       The standalone kernel was faster on every workload measured: the
 *       fused merges stall decode warps that keep HBM busy.
 * All modes give the same bits: one routine merges a row's sources in the
 * same order.  pkc_prefix_attention_state and
 * pkc_paged_decode_state_noalloc always use the standalone kernel.
 * Returns PKC_ERR_INVALID_ARG for any other value.
 */
int pkc_set_contraction(int mode);

/*
 * Thread blocks of the prefix stage in the cascade calls and
 * pkc_prefix_attention_state, process-wide.
 *   - n > 0: at most n blocks (one per SM).
 *   - n = 0 (the default): automatic.
 *
 * Automatic mode.  The prefix takes every SM, except in a cascade call with
 * a plan.  There the prefix runs next to the suffix decode,
 * which is bound by HBM and saturates it on about 100 SMs.  When every
 * prefix group's K/V tiles are read by two or more 128-row query tiles, the
 * prefix is bound by the tensor pipe rather than HBM.  It then gets SMs of
 * its own, so that the two stages overlap.  Let p_min be the SM count on
 * which the prefix is expected to take at most 0.8 of the decode's time,
 * and at least 16; the estimate uses 4.5 TFLOP/s per SM (a conservative
 * rate) against 6.5 TB/s for the decode.
 *   - Dynamic decode schedule (pkc_set_decode_schedule): the prefix gets a
 *     quarter of the SMs, or p_min if that is more, as long as 96 SMs remain
 *     for the decode.
 *   - Static schedule: the prefix gets the SMs the plan's CTAs leave free,
 *     if at least p_min.
 *
 * Decode blocks.  Under the dynamic schedule, with the prefix on fewer than
 * all SMs (also for n > 0), the decode runs one persistent block on each
 * remaining SM, at most one per plan CTA.  The two grids together never
 * exceed the SMs.  Those blocks take the plan's chunks from the shared
 * queue, so the chunks stay those of the plan.
 *
 * Alignment.  Any prefix block count is then lowered, to no less than 3/4
 * of it, to the largest value at which the query row tiles sharing a K/V
 * tile are computed by different blocks at the same moment.  The second
 * read of each such tile then hits L2.  Only groups whose K/V exceeds 16 MB
 * count; smaller ones stay in L2.
 *
 * A timed call (pkc_set_stage_events) keeps the same split.  The states are
 * the same for any block count up to rounding: the prefix's pieces, and so
 * its partial states, depend on it.
 * Returns PKC_ERR_INVALID_ARG for n < 0.
 * Reference: blog "Cascade Inference" (the prefix and suffix stages are
 * independent until the final merge).
 */
int pkc_set_prefix_ctas(int n);

/*
 * Small-batch cascade (process-wide; default 16).  A cascade call without a
 * plan (pkc_cascade_decode, pkc_cascade_decode_state) whose every prefix
 * group has at most max_rows query rows per KV head (requests x query heads
 * per KV head), whose groups are contiguous and do not overlap, and whose
 * prefixes (and the first prefix offset) are whole pages, runs as one
 * CUDA-core decode launch: each request attends to its group's prefix, read
 * as the first pages of its keys from the contiguous prefix tensors (viewed
 * as [tokens / page_size, page_size, Hkv, 128]), then to its cached suffix,
 * and the final state is written directly.  With so few rows per prefix the
 * multi-query kernel has no reuse to exploit (blog "Cascade Inference",
 * "Multi-query vs single-query kernels": the cascade pays off when many
 * queries share the prefix), while its fixed latency and the contraction
 * launch make up the step.  The state is the same attention state either way
 * (up to rounding).  0 disables the path.  PKC_ERR_INVALID_ARG for n < 0.
 */
int pkc_set_cascade_small(int max_rows);

/*
 * Diagnostics: the thread-block counts of the prefix kernel and of the
 * suffix decode in the calling thread's last cascade call
 * (pkc_cascade_decode, _multilevel, _paged_prefix) that got as far as the
 * decode launch; 0 and 0 before any.  Host only, no device work.  Returns
 * PKC_ERR_INVALID_ARG for NULL pointers.
 */
int pkc_last_launch_blocks(int* prefix_blocks, int* decode_blocks);

#ifdef __cplusplus
}
#endif

#endif /* PKC_H_ */
