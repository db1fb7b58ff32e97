/*
 * Oracle for the paged-KV cascade decode library -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load or call this file.  It shares no code, header, table or helper with
 * the CUDA library and never calls it.
 *
 * What it computes is the plain definition of an attention state, in
 * float64, with no blocking, fusion or reordering beyond the definition:
 *
 *   s_i  = sm_scale * (q . k_i)                 pre-softmax score
 *   s(I) = log sum_{i in I} exp(s_i)            generalised score (LSE)
 *   v(I) = sum_{i in I} exp(s_i) v_i / exp(s(I))
 *
 * (FlashInfer tutorial "Attention States and Recursive Attention", the
 * definitions of s(I) and v(I); blog "Cascade Inference: Memory Bandwidth
 * Efficient Shared Prefix Batch Decoding", section "Recursive Attention";
 * the FlashInfer MLSys'25 notes, A2 "Attention Composition", LSE(T) and
 * O(T)).  The pages write s_i = q k_i^T without a scale; the scale
 * 1/sqrt(d) of the workloads is applied to the score and the LSE is taken
 * over scaled scores.  The maximum is subtracted before exp, as both pages
 * say is done "in practice" for stability; it cancels exactly.
 *
 * The key set I of a (request b, query head h) row is the shared prefix of
 * every group b belongs to (one group in the two-level cascade, several in
 * a multi-level one) followed by b's own cached tokens, found through the
 * block table (Hugging Face "Paged attention", decoding path, indexing
 * mechanism): token t of request b lives in physical page
 * block_table[b][t / page_size], slot t % page_size, for
 * 0 <= t < cache_seqlens[b].  Cache layout is [num_pages, page_size,
 * H_kv, D], head dim contiguous; query head h reads KV head h / (H_qo/H_kv)
 * (GQA head groups, MLSys'25 notes appendix A).  An empty key set gives the
 * identity state v = 0, s = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_E4M3 = 3 };
enum { ORC_OK = 0, ORC_BAD_PAGE = 1, ORC_BAD_ARG = 2, ORC_NOMEM = 3 };
enum { ORC_MAX_GROUPS = 256 };

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double pkc_oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  else if (e == 31)
    mag = f ? NAN : INFINITY;
  else
    mag = ldexp((double)(f + 1024), e - 25); /* (1 + f/1024) * 2^(e-15) */
  return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 (1 sign, 8 exponent
 * with bias 127, 7 fraction bits). */
double pkc_oracle_bf16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int f = h & 0x7f;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -133); /* f * 2^-126 * 2^-7 */
  else if (e == 255)
    mag = f ? NAN : INFINITY;
  else
    mag = ldexp((double)(f + 128), e - 134); /* (1 + f/128) * 2^(e-127) */
  return sign ? -mag : mag;
}

/* 8-bit float E4M3 in the OCP "FP8 Formats for Deep Learning" form (the
 * "e4m3fn" of the libraries): 1 sign, 4 exponent bits with bias 7, 3
 * fraction bits.  Exponent field 0 is subnormal, f * 2^-9; there are no
 * infinities: S.1111.111 is NaN and S.1111.ffff (f < 7) is an ordinary
 * number, the largest 1.75 * 2^8 = 448.  The pages name "fp8" KV with fp16
 * queries and outputs (MLSys'25 notes, appendix F) without fixing the
 * variant; E4M3 is the one used for KV caches. */
double pkc_oracle_e4m3_to_f64(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int f = c & 7;
  double mag;
  if (e == 15 && f == 7)
    mag = NAN;
  else if (e == 0)
    mag = ldexp((double)f, -9); /* f/8 * 2^(1-7) */
  else
    mag = ldexp((double)(f + 8), e - 10); /* (1 + f/8) * 2^(e-7) */
  return sign ? -mag : mag;
}

static double elem(const void* x, int64_t i, int dtype) {
  if (dtype == ORC_F32) return (double)((const float*)x)[i];
  if (dtype == ORC_F16) return pkc_oracle_f16_to_f64(((const uint16_t*)x)[i]);
  if (dtype == ORC_E4M3) return pkc_oracle_e4m3_to_f64(((const uint8_t*)x)[i]);
  return pkc_oracle_bf16_to_f64(((const uint16_t*)x)[i]);
}

/*
 * Resolve every cached token of every request to its (page, slot).
 * out_page / out_slot are laid out request after request, sum(seqlens)
 * entries.  Entries of the block table at or past ceil(len / page_size) are
 * never read.  Returns ORC_BAD_PAGE if a page id that must be read is
 * negative or >= num_pages.
 */
int pkc_oracle_resolve(const int32_t* block_table, int64_t stride,
                       const int32_t* seqlens, int batch, int page_size,
                       int64_t num_pages, int32_t* out_page,
                       int32_t* out_slot) {
  int64_t k = 0;
  for (int b = 0; b < batch; ++b) {
    if (seqlens[b] < 0) return ORC_BAD_ARG;
    for (int32_t t = 0; t < seqlens[b]; ++t) {
      int32_t page = block_table[(int64_t)b * stride + t / page_size];
      if (page < 0 || page >= num_pages) return ORC_BAD_PAGE;
      out_page[k] = page;
      out_slot[k] = t % page_size;
      ++k;
    }
  }
  return ORC_OK;
}

typedef struct {
  /* queries [batch, hq, d] */
  const void* q;
  int batch, hq, hkv, d, dtype;
  double sm_scale;
  /* shared prefixes: k/v_prefix [sum Lp, hkv, d]; requests
   * req_begin[j] <= b < req_end[j] share prefix j, whose tokens are
   * kv_indptr[j] .. kv_indptr[j+1]-1.  Ranges may overlap: a request in
   * several groups (a multi-level cascade) attends to all their prefixes,
   * in group order.  n_prefix == 0 means no prefix. */
  const void* k_prefix;
  const void* v_prefix;
  const int32_t* prefix_kv_indptr;
  const int32_t* prefix_req_begin;
  const int32_t* prefix_req_end;
  int n_prefix;
  /* paged suffix: k/v_cache [num_pages, page_size, hkv, d]; NULL cache
   * means no suffix. */
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* cache_seqlens;
  int page_size;
  int64_t num_pages;
  /* element type of the paged cache, and its per-tensor scales: a cached
   * key is k_scale * k_cache[...], a cached value v_scale * v_cache[...]
   * (1 and 1 for 16-bit caches) */
  int kv_dtype;
  double k_scale, v_scale;
} orc_problem;

/* The prefix segments of row b's key list: (first prefix token, length)
 * of each group containing b, in group order. */
typedef struct {
  int n;
  int64_t total;
  int64_t lo[ORC_MAX_GROUPS], len[ORC_MAX_GROUPS];
} orc_segments;

/* Address (in elements) of the key/value vector of token t of row b. */
static int resolve_token(const orc_problem* p, int b, int kvh, int64_t t,
                         const orc_segments* sg, const void** kbase,
                         const void** vbase, int64_t* off) {
  if (t < sg->total) {
    int i = 0;
    while (t >= sg->len[i]) t -= sg->len[i++];
    *kbase = p->k_prefix;
    *vbase = p->v_prefix;
    *off = ((sg->lo[i] + t) * p->hkv + kvh) * (int64_t)p->d;
    return ORC_OK;
  }
  const int64_t n_pref = sg->total;
  int64_t ts = t - n_pref;
  int32_t page = p->block_table[(int64_t)b * p->bt_stride + ts / p->page_size];
  if (page < 0 || page >= p->num_pages) return ORC_BAD_PAGE;
  int64_t slot = ts % p->page_size;
  *kbase = p->k_cache;
  *vbase = p->v_cache;
  *off = (((int64_t)page * p->page_size + slot) * p->hkv + kvh) * (int64_t)p->d;
  return ORC_OK;
}

/* The attention state of one (request b, query head h) row. */
static int one_row(const orc_problem* p, int b, int h, double* o, double* lse,
                   double* s /* scratch, >= row length */) {
  int g = p->hq / p->hkv;
  int kvh = h / g;
  int64_t n_suf = 0;
  orc_segments sg;
  sg.n = 0;
  sg.total = 0;
  for (int j = 0; j < p->n_prefix; ++j) {
    if (p->prefix_req_begin[j] <= b && b < p->prefix_req_end[j]) {
      sg.lo[sg.n] = p->prefix_kv_indptr[j];
      sg.len[sg.n] = p->prefix_kv_indptr[j + 1] - p->prefix_kv_indptr[j];
      sg.total += sg.len[sg.n];
      ++sg.n;
    }
  }
  if (p->k_cache) n_suf = p->cache_seqlens[b];
  int64_t n = sg.total + n_suf;
  for (int x = 0; x < p->d; ++x) o[x] = 0.0;
  if (n == 0) {
    *lse = -INFINITY; /* empty key set: identity state */
    return ORC_OK;
  }
  const int64_t qoff = ((int64_t)b * p->hq + h) * p->d;
  /* s_i = sm_scale * q . k_i */
  for (int64_t t = 0; t < n; ++t) {
    const void *kb, *vb;
    int64_t off;
    int rc = resolve_token(p, b, kvh, t, &sg, &kb, &vb, &off);
    if (rc) return rc;
    const int cached = t >= sg.total;
    const int kd = cached ? p->kv_dtype : p->dtype;
    const double ks = cached ? p->k_scale : 1.0;
    double dot = 0.0;
    for (int x = 0; x < p->d; ++x)
      dot += elem(p->q, qoff + x, p->dtype) * (ks * elem(kb, off + x, kd));
    s[t] = p->sm_scale * dot;
  }
  /* s(I) = m + log sum exp(s_i - m) */
  double m = -INFINITY;
  for (int64_t t = 0; t < n; ++t) m = s[t] > m ? s[t] : m;
  double sum = 0.0;
  for (int64_t t = 0; t < n; ++t) sum += exp(s[t] - m);
  *lse = m + log(sum);
  /* v(I) = sum exp(s_i - m) v_i / sum exp(s_i - m) */
  for (int64_t t = 0; t < n; ++t) {
    const void *kb, *vb;
    int64_t off;
    resolve_token(p, b, kvh, t, &sg, &kb, &vb, &off);
    const int cached = t >= sg.total;
    const int vd = cached ? p->kv_dtype : p->dtype;
    const double vs = cached ? p->v_scale : 1.0;
    double w = exp(s[t] - m) / sum;
    for (int x = 0; x < p->d; ++x) o[x] += w * (vs * elem(vb, off + x, vd));
  }
  return ORC_OK;
}

/*
 * Attention states for a list of rows.  rows[2*r] = request, rows[2*r+1] =
 * query head.  q and the prefixes are of dtype; the paged cache of kv_dtype
 * with scales k_scale, v_scale (see orc_problem).  o_out [n_rows, d], lse_out [n_rows], float64.  Rows run in
 * parallel over n_threads OpenMP threads (0 = the runtime's default); each
 * row is computed by one thread in the order above.
 */
int pkc_oracle_attention_rows(
    const void* q, int batch, int hq, int hkv, int d, int dtype,
    double sm_scale, const void* k_prefix, const void* v_prefix,
    const int32_t* prefix_kv_indptr, const int32_t* prefix_req_begin,
    const int32_t* prefix_req_end, int n_prefix, const void* k_cache,
    const void* v_cache,
    const int32_t* block_table, int64_t bt_stride,
    const int32_t* cache_seqlens, int page_size, int64_t num_pages,
    int kv_dtype, double k_scale, double v_scale,
    const int32_t* rows, int64_t n_rows, int n_threads, double* o_out,
    double* lse_out) {
  if (hkv <= 0 || hq % hkv != 0 || d <= 0 || n_prefix < 0 || n_prefix > ORC_MAX_GROUPS) return ORC_BAD_ARG;
  orc_problem p = {q, batch, hq, hkv, d, dtype, sm_scale, k_prefix, v_prefix,
                   prefix_kv_indptr, prefix_req_begin, prefix_req_end, n_prefix, k_cache,
                   v_cache, block_table, bt_stride, cache_seqlens, page_size,
                   num_pages, kv_dtype, k_scale, v_scale};
  int64_t max_n = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t n = 0;
    for (int j = 0; j < n_prefix; ++j)
      if (prefix_req_begin[j] <= b && b < prefix_req_end[j])
        n += prefix_kv_indptr[j + 1] - prefix_kv_indptr[j];
    if (k_cache) n += cache_seqlens[b];
    if (n > max_n) max_n = n;
  }
  int err = ORC_OK;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_n > 0 ? max_n : 1));
    if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      err = ORC_NOMEM;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t r = 0; r < n_rows; ++r) {
        int rc = one_row(&p, rows[2 * r], rows[2 * r + 1], o_out + r * d,
                         lse_out + r, s);
        if (rc) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
          err = rc;
        }
      }
      free(s);
    }
  }
  return err;
}

/* Number of OpenMP threads a parallel region would use by default. */
int pkc_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
