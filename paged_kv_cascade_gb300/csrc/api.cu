// C ABI entry points: argument checks, workspace layout, and the launch
// sequences that compose the kernels into the public calls.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "pkc.h"
#include "pkc_internal.h"

namespace pkc {

static thread_local char g_err[1024] = "";
static thread_local cudaEvent_t g_stage_events[4] = {nullptr, nullptr, nullptr, nullptr};
// Block counts of the calling thread's last cascade call (pkc_last_launch_blocks).
static thread_local int g_last_prefix_blocks = 0, g_last_decode_blocks = 0;

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_error(int e, const char* what) {
  if (e == -1) return set_error(PKC_ERR_CUDA, "%s: TMA tensor map encoding failed", what);
  return set_error(PKC_ERR_CUDA, "%s: %s", what, cudaGetErrorString((cudaError_t)e));
}

int num_sms() {
  static int cache[128] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

static size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int batch, int hq, int d, int num_ctas) {
  WsLayout L;
  size_t off = PKC_STATUS_BYTES;
  L.plan = off;
  off += al256(num_ctas > 0 ? 4 * (size_t)plan_layout(batch, num_ctas).total : 0);
  const size_t rows = (size_t)batch * hq;
  L.suffix_o = off;   off += al256(4 * rows * d);
  L.suffix_lse = off; off += al256(4 * rows);
  const size_t prow = (size_t)2 * num_ctas * hq;
  L.part_o = off;     off += al256(4 * prow * d);
  L.part_lse = off;   off += al256(4 * prow);
  L.arrive = off;     off += al256(4 * rows);  // per (request, KV head) <= per (request, query head)
  L.fixed_end = off;
  L.prefix = off;
  L.prefix_split = al256(4 * rows * d) + al256(4 * rows);
  return L;
}

}  // namespace pkc

using namespace pkc;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_attn_dims(int batch, int hq, int hkv, int head_dim, int dtype) {
  if (batch < 0) return set_error(PKC_ERR_INVALID_ARG, "batch must be >= 0 (got %d)", batch);
  if (head_dim != PKC_HEAD_DIM)
    return set_error(PKC_ERR_UNSUPPORTED, "head_dim %d is not supported (only 128)", head_dim);
  if (hkv <= 0 || hq <= 0 || hq % hkv != 0)
    return set_error(PKC_ERR_INVALID_ARG, "num_qo_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                     hq, hkv);
  const int g = hq / hkv;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return set_error(PKC_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", g);
  if (dtype != PKC_F16 && dtype != PKC_BF16)
    return set_error(PKC_ERR_INVALID_ARG, "dtype must be PKC_F16 or PKC_BF16 (got %d)", dtype);
  return PKC_OK;
}

int check_plan(const int32_t* plan, int batch) {
  if (!plan) return PKC_OK;
  if (plan[PKC_PLAN_MAGIC] != PKC_PLAN_MAGIC_VALUE) return set_error(PKC_ERR_PLAN, "plan: bad magic word");
  if (plan[PKC_PLAN_N_REQ] != batch)
    return set_error(PKC_ERR_PLAN, "plan was made for %d requests, call has batch %d", plan[PKC_PLAN_N_REQ], batch);
  if (plan[PKC_PLAN_TILE_Q] != 1 || plan[PKC_PLAN_N_UNITS] != batch)
    return set_error(PKC_ERR_PLAN, "decode needs a plan with tile_q 1 and one query row per request");
  if (plan[PKC_PLAN_NUM_CTAS] < 1) return set_error(PKC_ERR_PLAN, "plan: num_ctas < 1");
  return PKC_OK;
}

int check_ws(const void* ws, size_t bytes, size_t need) {
  if (!ws) return set_error(PKC_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return set_error(PKC_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (bytes < need) return set_error(PKC_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", bytes, need);
  return PKC_OK;
}

struct PrefixSetup {
  PrefixParams pp;
  int n_tiles = 0;
  int64_t tokens = 0;
};

// Validate the prefix description and lay out its work: the flat KV tiles
// of all (row tile, KV head) pairs split evenly over one block per SM, as
// long as the pieces of any pair fit the workspace's partial slots.
int setup_prefix(PrefixSetup& S, const int32_t* kv_indptr, const int32_t* req_begin, const int32_t* req_end,
                 int n_prefix, int batch, int hq, int hkv, float sm_scale, uint8_t* ws, size_t ws_bytes,
                 const WsLayout& L, int32_t* status, int max_blocks) {
  if (n_prefix < 1 || n_prefix > PKC_MAX_PREFIX)
    return set_error(PKC_ERR_INVALID_ARG, "n_prefix must be in [1, %d] (got %d)", PKC_MAX_PREFIX, n_prefix);
  if (!kv_indptr || !req_begin || !req_end) return set_error(PKC_ERR_INVALID_ARG, "prefix arrays are NULL");
  if (kv_indptr[0] < 0) return set_error(PKC_ERR_INVALID_ARG, "prefix_kv_indptr must start >= 0");
  for (int j = 0; j < n_prefix; ++j) {
    if (kv_indptr[j + 1] < kv_indptr[j])
      return set_error(PKC_ERR_INVALID_ARG, "prefix_kv_indptr must be non-decreasing (at %d)", j);
    if (req_begin[j] < 0 || req_end[j] < req_begin[j] || req_end[j] > batch)
      return set_error(PKC_ERR_INVALID_ARG, "prefix group %d: requests [%d, %d) outside [0, batch %d]", j,
                       req_begin[j], req_end[j], batch);
  }
  PrefixParams& p = S.pp;
  std::memset(&p, 0, sizeof(p));
  p.batch = batch;
  p.hq = hq;
  p.hkv = hkv;
  p.g = hq / hkv;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.n_prefix = n_prefix;
  // Flat KV tiles over the (row tile, KV head) pairs of every group.
  int tiles = 0;
  int64_t T = 0;
  for (int j = 0; j <= n_prefix; ++j) {
    p.kv_indptr[j] = kv_indptr[j];
    p.tile_indptr[j] = tiles;
    if (T > INT32_MAX) return set_error(PKC_ERR_UNSUPPORTED, "prefix: too many KV tiles (%lld)", (long long)T);
    p.kvt_indptr[j] = (int32_t)T;
    if (j < n_prefix) {
      p.req_begin[j] = req_begin[j];
      p.req_end[j] = req_end[j];
      const int rows = (req_end[j] - req_begin[j]) * p.g;
      const int rt = (rows + 127) / 128;
      const int kvt = (kv_indptr[j + 1] - kv_indptr[j] + 127) / 128;
      tiles += rt;
      T += (int64_t)rt * hkv * kvt;
    }
  }
  S.n_tiles = tiles;
  S.tokens = kv_indptr[n_prefix];
  const size_t avail = ws_bytes > L.fixed_end ? (ws_bytes - L.fixed_end) / L.prefix_split : 0;
  if (avail < 1) return set_error(PKC_ERR_WORKSPACE, "workspace has no room for prefix partial states");
  const int max_slots = (int)std::min<size_t>(avail, PKC_MAX_PREFIX_SPLITS);
  // One block per SM, or max_blocks (fewer if there are fewer tiles).
  // Group j needs as many partial slots as the most pieces any of its pairs
  // is cut into; groups sharing a request get disjoint slot ranges (first
  // fit in group order), and every request's slots must fit the workspace.
  int C = (int)std::min<int64_t>(std::max(1, std::min(max_blocks, num_sms())), T);
  // The 128-row query tiles of one (group, KV head) read the same K/V
  // tiles, Hkv * kvt flat tiles apart.  When that distance is a whole number
  // of blocks' shares (D C divisible by T), block i and block i + D C / T
  // reach the two copies of every K/V tile at the same moment and the
  // second read hits L2; otherwise they drift apart by a fraction of a
  // share and the second read goes to HBM (GQA prefix next to the decode:
  // 40 or 48 blocks 296 us per step, 44 or 52 blocks 313 us).  So C is the
  // largest count, down to 3/4 of the candidate, that aligns every group
  // with two or more row tiles whose K/V (all heads) is larger than 16 MB;
  // a smaller group's K/V, read by several row tiles, stays in the 126 MB L2.
  {
    std::vector<int64_t> dist;
    for (int j = 0; j < n_prefix; ++j) {
      const int kvt = (kv_indptr[j + 1] - kv_indptr[j] + 127) / 128;
      const int64_t kv_bytes = (int64_t)(kv_indptr[j + 1] - kv_indptr[j]) * hkv * PKC_HEAD_DIM * 4;
      if (kvt > 0 && p.tile_indptr[j + 1] - p.tile_indptr[j] >= 2 && kv_bytes > (16ll << 20))
        dist.push_back((int64_t)hkv * kvt);
    }
    if (!dist.empty()) {
      for (int c = C; c >= 1 && 4 * c >= 3 * C; --c) {
        bool aligned = true;
        for (const int64_t d : dist) aligned = aligned && (d * c) % T == 0;
        if (aligned) {
          C = c;
          break;
        }
      }
    }
  }
  if (T * C >= INT32_MAX) return set_error(PKC_ERR_UNSUPPORTED, "prefix: too many KV tiles (%lld)", (long long)T);
  int slots = 0;
  std::vector<int> need(n_prefix), base(n_prefix);
  while (C > 0) {
    for (int j = 0; j < n_prefix; ++j) {
      need[j] = 0;
      const int kvt = (kv_indptr[j + 1] - kv_indptr[j] + 127) / 128;
      if (kvt == 0) continue;
      const int n_pairs = (p.tile_indptr[j + 1] - p.tile_indptr[j]) * hkv;
      for (int q = 0; q < n_pairs; ++q) {
        const int64_t a = p.kvt_indptr[j] + (int64_t)q * kvt;
        need[j] = std::max(need[j], prefix_block_of(a + kvt - 1, T, C) - prefix_block_of(a, T, C) + 1);
      }
    }
    slots = 1;
    for (int j = 0; j < n_prefix; ++j) {
      base[j] = 0;
      for (int i = 0; i < j; ++i)  // after every earlier group that shares a request
        if (need[i] > 0 && req_begin[i] < req_end[j] && req_begin[j] < req_end[i])
          base[j] = std::max(base[j], base[i] + need[i]);
      slots = std::max(slots, base[j] + need[j]);
    }
    if (slots <= max_slots) break;
    --C;
  }
  if (T > 0 && C == 0)
    return set_error(PKC_ERR_WORKSPACE, "workspace has too few prefix partial slots for %d overlapping groups",
                     n_prefix);
  for (int j = 0; j < n_prefix; ++j) p.slot_base[j] = base[j];
  p.n_blocks = C;
  p.total_tiles = T;
  p.splits = std::max(1, slots);
  p.out_o = reinterpret_cast<float*>(ws + L.prefix);
  p.out_lse = reinterpret_cast<float*>(ws + L.prefix + al256(4 * (size_t)batch * hq * PKC_HEAD_DIM));
  p.split_stride_o = (int64_t)(L.prefix_split / 4);
  p.split_stride_lse = (int64_t)(L.prefix_split / 4);
  p.status = status;
  return PKC_OK;
}

// Request ranges [indptr[j], indptr[j+1]) of the contiguous groups of the
// two-level calls (validated; setup_prefix checks the bounds).
int indptr_ranges(const int32_t* req_indptr, int n_prefix, int32_t* begin, int32_t* end) {
  if (!req_indptr) return set_error(PKC_ERR_INVALID_ARG, "prefix_req_indptr is NULL");
  if (n_prefix < 1 || n_prefix > PKC_MAX_PREFIX)
    return set_error(PKC_ERR_INVALID_ARG, "n_prefix must be in [1, %d] (got %d)", PKC_MAX_PREFIX, n_prefix);
  if (req_indptr[0] < 0) return set_error(PKC_ERR_INVALID_ARG, "prefix_req_indptr must start >= 0");
  for (int j = 0; j < n_prefix; ++j) {
    if (req_indptr[j + 1] < req_indptr[j])
      return set_error(PKC_ERR_INVALID_ARG, "prefix_req_indptr must be non-decreasing (at %d)", j);
    begin[j] = req_indptr[j];
    end[j] = req_indptr[j + 1];
  }
  return PKC_OK;
}

// Blocks of the prefix kernel in a cascade call (pkc_set_prefix_ctas).
std::atomic<int> g_prefix_ctas{0};

// How a planned cascade shares the SMs between its two independent stages.
// The suffix decode is bound by HBM and, with its producer's integer row
// masks, saturates it on about 100 SMs (GQA suffix of 1.8 GB: 148 / 112 /
// 100 CTAs take 267 / 270 / 272 us).  A prefix whose K/V tiles are each
// read by two or more 128-row query tiles is bound by the tensor pipe
// instead (about 6 TFLOP/s per SM on SMs of its own: 34.4 GFLOP in 175 us
// on 32 SMs, 145 us on 40; the estimate below uses 4.5, since a prefix that
// outlasts the decode lengthens the step: the three-level GQA cascade, whose
// prefix needs about 90 % of its decode's time on a quarter of the SMs,
// took 317 us split against 283 us unsplit), so the two stages can overlap
// instead of queueing for SMs.  The two grids together never exceed the SMs: which of
// the two streams' kernels starts first is not fixed, and a prefix over
// every SM that started first would hold the decode back.
// The prefix needs p_min SMs to be expected to finish in 0.8 of the
// decode's time.
//  - Dynamic schedule: the decode's persistent blocks take the plan's
//    chunks from a queue, so their number is free.  The prefix gets a
//    quarter of the SMs or p_min if that is more, as long as the decode
//    keeps kMinDecodeSms, and the decode the rest (GQA cascade step 319 ->
//    294 us on 32 + 120 SMs; three-level GQA cascade 277 -> 254 us on
//    40 + 112, where 30 prefix SMs outlasted the decode: 317 us).
//  - Static schedule: each decode block runs one plan CTA's list; the
//    prefix gets the SMs the plan leaves free if they are at least p_min.
// Otherwise (a prefix that is itself HBM-bound, a short suffix) the prefix
// takes every SM and the decode one block per plan CTA.
constexpr int kMinPrefixSms = 16;
constexpr int kMinDecodeSms = 96;  // 148 / 100 / 88 decode blocks: 267 / 272 / 284 us
constexpr double kPrefixFlopsPerSm = 4.5e12;  // tensor-pipe bound prefix, per SM (conservative)
constexpr double kDecodeBytesPerS = 6.5e12;   // HBM-bound suffix decode
struct StageSplit {
  int prefix_blocks;  // at most this many prefix blocks (setup_prefix may use fewer)
  int decode_blocks;  // 0: one per plan CTA; -1: the SMs the prefix leaves; else this many
};
StageSplit stage_split(const int32_t* kv_indptr, const int32_t* req_begin, const int32_t* req_end, int n_prefix,
                       int g, int hkv, int elem_bytes, const int32_t* plan_host, bool next_to_decode) {
  const int sms = num_sms();
  const bool dynamic = plan_host && decode_schedule_dynamic();
  const int forced = g_prefix_ctas.load();
  if (forced > 0) return {std::min(forced, sms), next_to_decode && dynamic && forced < sms ? -1 : 0};
  const StageSplit all{sms, 0};
  if (!next_to_decode || !plan_host) return all;
  double flops = 0.0;
  for (int j = 0; j < n_prefix; ++j) {
    const int64_t tokens = kv_indptr[j + 1] - kv_indptr[j];
    const int64_t row_tiles = ((int64_t)(req_end[j] - req_begin[j]) * g + 127) / 128;
    if (tokens == 0 || row_tiles == 0) continue;
    if (row_tiles < 2) return all;  // each K/V tile read once: HBM-bound
    flops += 4.0 * PKC_HEAD_DIM * 128.0 * (double)row_tiles * (double)tokens * hkv;
  }
  if (flops <= 0.0) return all;
  int64_t suffix_tokens = 0;
  const int32_t* kv_len = plan_host + plan_host[PKC_PLAN_OFF_UNIT_KV_LEN];
  for (int u = 0; u < plan_host[PKC_PLAN_N_UNITS]; ++u) suffix_tokens += kv_len[u];
  const double t_decode = (double)suffix_tokens * 2.0 * hkv * PKC_HEAD_DIM * elem_bytes / kDecodeBytesPerS;
  if (t_decode <= 0.0) return all;
  const double need = flops / (0.8 * t_decode * kPrefixFlopsPerSm);
  if (need > sms) return all;
  const int p_min = std::max(kMinPrefixSms, (int)std::ceil(need));
  if (dynamic) {
    const int blocks = std::max(sms - (3 * sms) / 4, p_min);
    if (blocks > sms - kMinDecodeSms) return all;
    return {blocks, -1};
  }
  const int free_sms = sms - plan_host[PKC_PLAN_NUM_CTAS];
  return free_sms >= p_min ? StageSplit{free_sms, 0} : all;
}

void fill_contract_prefix(ContractParams& c, const PrefixSetup& S) {
  c.prefix_o = S.pp.out_o;
  c.prefix_lse = S.pp.out_lse;
  c.prefix_stride_o = S.pp.split_stride_o;
  c.prefix_stride_lse = S.pp.split_stride_lse;
  c.prefix_splits = S.pp.splits;
  c.n_prefix = S.pp.n_prefix;
  c.hkv = S.pp.hkv;
  c.g = S.pp.g;
  c.prefix_blocks = S.pp.n_blocks;
  c.prefix_tiles = S.pp.total_tiles;
  std::memcpy(c.prefix_req_begin, S.pp.req_begin, sizeof(c.prefix_req_begin));
  std::memcpy(c.prefix_req_end, S.pp.req_end, sizeof(c.prefix_req_end));
  std::memcpy(c.prefix_slot_base, S.pp.slot_base, sizeof(c.prefix_slot_base));
  std::memcpy(c.prefix_kv_indptr, S.pp.kv_indptr, sizeof(c.prefix_kv_indptr));
  std::memcpy(c.prefix_kvt_indptr, S.pp.kvt_indptr, sizeof(c.prefix_kvt_indptr));
}

// Copy the plan-array offsets the contraction kernel needs.
void contract_plan_offsets(ContractParams& c, const int32_t* plan_host) {
  if (!plan_host) return;
  c.plan_words = plan_host[PKC_PLAN_TOTAL_WORDS];
  c.off_unit_list = plan_host[PKC_PLAN_OFF_UNIT_LIST];
  c.off_unit_req = plan_host[PKC_PLAN_OFF_UNIT_REQ];
  c.off_unit_n_chunks = plan_host[PKC_PLAN_OFF_UNIT_N_CHUNKS];
  c.off_unit_partial_begin = plan_host[PKC_PLAN_OFF_UNIT_PARTIAL_BEGIN];
}

// Small-batch cascade (pkc_set_cascade_small): a cascade call without a plan
// whose every prefix group has at most this many query rows per KV head
// (requests x G) reads its prefixes through the decode kernel, as pages of
// the prefix tensors.  0: never.
std::atomic<int> g_cascade_small_rows{16};

// Contraction fused into the attention kernels (1) or the standalone
// contraction kernel after them (0, default): pkc_set_contraction.  Fused,
// the merges at the ends of work items stall decode warps that keep HBM
// busy, and a prefix stage that finishes last merges whole row tiles on a
// few blocks: measured slower on every benchmark workload (headline 296 vs
// 293 us, long prompt 266 vs 181 us, tiny 24 vs 15 us).
std::atomic<int> g_fused_contraction{0};

// The fused contraction's view of a call: the same sources, offsets and
// output as the standalone kernel's ContractParams (c), plus the counters.
void fill_fuse(FuseParams& f, const ContractParams& c, int hkv, int32_t* arrive) {
  std::memset(&f, 0, sizeof(f));
  f.enabled = 1;
  f.arrive = arrive;
  f.batch = c.batch;
  f.hq = c.hq;
  f.hkv = hkv;
  f.g = c.hq / hkv;
  f.plan = c.plan;
  f.plan_words = c.plan_words;
  f.off_unit_list = c.off_unit_list;
  f.off_unit_req = c.off_unit_req;
  f.off_unit_n_chunks = c.off_unit_n_chunks;
  f.off_unit_partial_begin = c.off_unit_partial_begin;
  f.suffix_o = c.suffix_o;
  f.suffix_lse = c.suffix_lse;
  f.part_o = c.part_o;
  f.part_lse = c.part_lse;
  if (c.prefix_o && c.n_prefix <= PKC_FUSE_MAX_PREFIX) {
    f.prefix_o = c.prefix_o;
    f.prefix_lse = c.prefix_lse;
    f.prefix_stride_o = c.prefix_stride_o;
    f.prefix_stride_lse = c.prefix_stride_lse;
    f.n_prefix = c.n_prefix;
    f.prefix_blocks = c.prefix_blocks;
    f.prefix_tiles = c.prefix_tiles;
    for (int j = 0; j < c.n_prefix; ++j) {
      f.prefix_req_begin[j] = c.prefix_req_begin[j];
      f.prefix_req_end[j] = c.prefix_req_end[j];
      f.prefix_slot_base[j] = c.prefix_slot_base[j];
    }
    for (int j = 0; j <= c.n_prefix; ++j) {
      f.prefix_kv_indptr[j] = c.prefix_kv_indptr[j];
      f.prefix_kvt_indptr[j] = c.prefix_kvt_indptr[j];
    }
  }
  f.o = c.o;
  f.lse = c.lse;
  f.out_dtype = c.out_dtype;
}

}  // namespace

extern "C" {

int pkc_version(void) { return PKC_VERSION; }

int pkc_set_stage_events(void* const* events, int n_events) {
  if (events && n_events < 4) return set_error(PKC_ERR_INVALID_ARG, "set_stage_events: need 4 events");
  for (int i = 0; i < 4; ++i) g_stage_events[i] = events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  return PKC_OK;
}

const char* pkc_last_error(void) { return g_err; }

int pkc_merge_state(const void* v_a, const float* s_a, const void* v_b, const float* s_b, void* v_out,
                    float* s_out, int64_t n_tokens, int n_heads, int head_dim, int v_dtype, void* stream) {
  if (n_tokens < 0 || n_heads < 0 || head_dim <= 0)
    return set_error(PKC_ERR_INVALID_ARG, "merge_state: negative size");
  if (v_dtype != PKC_F32 && v_dtype != PKC_F16 && v_dtype != PKC_BF16)
    return set_error(PKC_ERR_INVALID_ARG, "merge_state: bad dtype %d", v_dtype);
  const int esz = v_dtype == PKC_F32 ? 4 : 2;
  if ((head_dim * esz) % 16 != 0)
    return set_error(PKC_ERR_UNSUPPORTED, "merge_state: head_dim * element size must be a multiple of 16 bytes");
  const int cpr = head_dim * esz / 16;
  if (cpr > 32 ? cpr % 32 != 0 : 32 % cpr != 0)
    return set_error(PKC_ERR_UNSUPPORTED, "merge_state: head_dim*esize/16 must divide 32 or be a multiple of 32");
  if (n_tokens * n_heads == 0) return PKC_OK;
  if (!v_a || !s_a || !v_b || !s_b || !v_out || !s_out)
    return set_error(PKC_ERR_INVALID_ARG, "merge_state: NULL pointer");
  if (!aligned16(v_a) || !aligned16(v_b) || !aligned16(v_out))
    return set_error(PKC_ERR_INVALID_ARG, "merge_state: v pointers must be 16-byte aligned");
  const int e = launch_merge_state(v_a, s_a, v_b, s_b, v_out, s_out, n_tokens * n_heads, head_dim, v_dtype, stream);
  return e ? cuda_error(e, "merge_state launch") : PKC_OK;
}

int pkc_merge_states(const void* v, const float* s, void* v_out, float* s_out, int64_t n_tokens, int n_states,
                     int n_heads, int head_dim, int v_dtype, void* stream) {
  if (n_tokens < 0 || n_heads < 0 || head_dim <= 0 || n_states < 1)
    return set_error(PKC_ERR_INVALID_ARG, "merge_states: bad size (n_states >= 1 required)");
  if (v_dtype != PKC_F32 && v_dtype != PKC_F16 && v_dtype != PKC_BF16)
    return set_error(PKC_ERR_INVALID_ARG, "merge_states: bad dtype %d", v_dtype);
  const int esz = v_dtype == PKC_F32 ? 4 : 2;
  if ((head_dim * esz) % 16 != 0)
    return set_error(PKC_ERR_UNSUPPORTED, "merge_states: head_dim * element size must be a multiple of 16 bytes");
  const int cpr = head_dim * esz / 16;
  if (cpr > 32 ? cpr % 32 != 0 : 32 % cpr != 0)
    return set_error(PKC_ERR_UNSUPPORTED, "merge_states: head_dim*esize/16 must divide 32 or be a multiple of 32");
  if (n_tokens * n_heads == 0) return PKC_OK;
  if (!v || !s || !v_out || !s_out) return set_error(PKC_ERR_INVALID_ARG, "merge_states: NULL pointer");
  if (!aligned16(v) || !aligned16(v_out))
    return set_error(PKC_ERR_INVALID_ARG, "merge_states: v pointers must be 16-byte aligned");
  const int e = launch_merge_states(v, s, v_out, s_out, n_tokens, n_states, n_heads, head_dim, v_dtype, stream);
  return e ? cuda_error(e, "merge_states launch") : PKC_OK;
}

int pkc_merge_states_to(const void* v, const float* s, void* v_out, float* s_out, int64_t n_tokens, int n_states,
                        int n_heads, int head_dim, int v_dtype, int out_dtype, void* stream) {
  if (out_dtype == v_dtype)
    return pkc_merge_states(v, s, v_out, s_out, n_tokens, n_states, n_heads, head_dim, v_dtype, stream);
  if (v_dtype != PKC_F32 || (out_dtype != PKC_F16 && out_dtype != PKC_BF16))
    return set_error(PKC_ERR_INVALID_ARG,
                     "merge_states_to: fp32 states into an fp16 / bf16 result, or equal types (got %d -> %d)",
                     v_dtype, out_dtype);
  if (n_tokens < 0 || n_heads < 0 || n_states < 1)
    return set_error(PKC_ERR_INVALID_ARG, "merge_states_to: bad size (n_states >= 1 required)");
  const int cpr = head_dim / 4;  // 16-byte chunks of an fp32 row
  if (head_dim <= 0 || head_dim % 4 != 0 || (cpr > 32 ? cpr % 32 != 0 : 32 % cpr != 0))
    return set_error(PKC_ERR_UNSUPPORTED, "merge_states_to: head_dim/4 must divide 32 or be a multiple of 32");
  if (n_tokens * n_heads == 0) return PKC_OK;
  if (!v || !s || !v_out || !s_out) return set_error(PKC_ERR_INVALID_ARG, "merge_states_to: NULL pointer");
  if (!aligned16(v) || !aligned16(v_out))
    return set_error(PKC_ERR_INVALID_ARG, "merge_states_to: v pointers must be 16-byte aligned");
  const int e = launch_merge_states_to(v, s, v_out, s_out, n_tokens, n_states, n_heads, head_dim, v_dtype, out_dtype,
                                       stream);
  return e ? cuda_error(e, "merge_states_to launch") : PKC_OK;
}

int pkc_workspace_size(int batch, int num_qo_heads, int head_dim, int num_ctas, int prefix_splits, size_t* bytes) {
  if (!bytes || batch < 0 || num_qo_heads <= 0 || head_dim <= 0 || num_ctas < 0 || prefix_splits < 0)
    return set_error(PKC_ERR_INVALID_ARG, "workspace_size: bad argument");
  const WsLayout L = ws_layout(batch, num_qo_heads, head_dim, num_ctas);
  *bytes = L.fixed_end + (size_t)prefix_splits * L.prefix_split;
  return PKC_OK;
}

int pkc_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (int rc = check_ws(workspace, workspace_bytes, PKC_STATUS_BYTES)) return rc;
  const cudaError_t e = cudaMemsetAsync(workspace, 0, PKC_STATUS_BYTES, (cudaStream_t)stream);
  return e ? cuda_error(e, "workspace_init") : PKC_OK;
}

int pkc_device_status(void* workspace, void* stream, int32_t* status) {
  if (!workspace || !status) return set_error(PKC_ERR_INVALID_ARG, "device_status: NULL pointer");
  cudaStream_t st = (cudaStream_t)stream;
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (!e) e = cudaStreamSynchronize(st);
  if (!e) e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), st);
  if (e) return cuda_error(e, "device_status");
  *status = v;
  return PKC_OK;
}

int pkc_plan_upload(const int32_t* plan_host, void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan_host) return set_error(PKC_ERR_INVALID_ARG, "plan_upload: plan is NULL");
  if (plan_host[PKC_PLAN_MAGIC] != PKC_PLAN_MAGIC_VALUE) return set_error(PKC_ERR_PLAN, "plan_upload: bad magic");
  const size_t words = (size_t)plan_host[PKC_PLAN_TOTAL_WORDS];
  if (int rc = check_ws(workspace, workspace_bytes, PKC_STATUS_BYTES + 4 * words)) return rc;
  const cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(workspace) + PKC_STATUS_BYTES, plan_host, 4 * words,
                                        cudaMemcpyHostToDevice, (cudaStream_t)stream);
  return e ? cuda_error(e, "plan_upload") : PKC_OK;
}

}  // extern "C"

namespace {
// Paged decode (+ contraction of split chunks) for both cache kinds.
int paged_decode_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                      int block_table_stride, const int32_t* cache_seqlens, int batch, int num_qo_heads,
                      int num_kv_heads, int head_dim, int page_size, int64_t num_pages, float sm_scale,
                      float k_scale, float v_scale, const int32_t* plan_host, void* workspace,
                      size_t workspace_bytes, void* o, float* lse, int dtype, int kv_dtype, void* stream) {
  if (int rc = check_attn_dims(batch, num_qo_heads, num_kv_heads, head_dim, dtype)) return rc;
  if (int rc = check_plan(plan_host, batch)) return rc;
  if (page_size < 1 || block_table_stride < 1 || num_pages < 0)
    return set_error(PKC_ERR_INVALID_ARG, "page_size and block_table_stride must be >= 1, num_pages >= 0");
  if (kv_dtype == PKC_E4M3) {
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
      return set_error(PKC_ERR_INVALID_ARG, "paged_decode_state_fp8: k_scale and v_scale must be finite and > 0");
    if (mma_decode_heads_per_block(num_kv_heads, page_size) == 0)
      return set_error(PKC_ERR_UNSUPPORTED,
                       "paged_decode_state_fp8: page_size %d with %d KV heads is not supported (page_size must "
                       "be a power of two and min(page_size, 16) x heads per block >= 8)",
                       page_size, num_kv_heads);
  }
  const int num_ctas = plan_host ? plan_host[PKC_PLAN_NUM_CTAS] : 0;
  const WsLayout L = ws_layout(batch, num_qo_heads, head_dim, num_ctas);
  if (int rc = check_ws(workspace, workspace_bytes, L.fixed_end)) return rc;
  if (batch == 0) return PKC_OK;
  if (!q || !k_cache || !v_cache || !block_table || !cache_seqlens || !o || !lse)
    return set_error(PKC_ERR_INVALID_ARG, "paged_decode_state: NULL pointer");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return set_error(PKC_ERR_INVALID_ARG, "paged_decode_state: q, caches and o must be 16-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  DecodeParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.q = q; dp.k_cache = k_cache; dp.v_cache = v_cache;
  dp.block_table = block_table; dp.cache_seqlens = cache_seqlens;
  dp.bt_stride = block_table_stride; dp.num_pages = num_pages;
  dp.batch = batch; dp.hq = num_qo_heads; dp.hkv = num_kv_heads; dp.page_size = page_size;
  dp.scale_log2 = sm_scale * k_scale * 1.4426950408889634f;
  dp.v_scale = v_scale;
  dp.plan = plan_host ? reinterpret_cast<const int32_t*>(ws + L.plan) : nullptr;
  dp.plan_words = plan_host ? plan_host[PKC_PLAN_TOTAL_WORDS] : 0;
  dp.o_direct = o; dp.lse_direct = lse; dp.direct_f32 = 0;
  dp.part_o = reinterpret_cast<float*>(ws + L.part_o);
  dp.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  dp.status = status;
  // Split requests' chunk partials are contracted into the output: by the
  // decode kernel itself (fused; counters zeroed first), or by the
  // contraction kernel after it.
  ContractParams cp;
  std::memset(&cp, 0, sizeof(cp));
  cp.batch = batch; cp.hq = num_qo_heads; cp.mode = kContractPlanUnits; cp.plan = dp.plan;
  cp.hkv = num_kv_heads; cp.g = num_qo_heads / num_kv_heads;
  contract_plan_offsets(cp, plan_host);
  cp.part_o = dp.part_o; cp.part_lse = dp.part_lse;
  cp.o = o; cp.lse = lse; cp.out_dtype = dtype; cp.status = status;
  const bool fused = plan_host && g_fused_contraction.load() != 0;
  if (fused) {
    int32_t* arrive = reinterpret_cast<int32_t*>(ws + L.arrive);
    const cudaError_t me = cudaMemsetAsync(arrive, 0, 4 * (size_t)batch * num_kv_heads, (cudaStream_t)stream);
    if (me) return cuda_error(me, "paged decode: counter reset");
    fill_fuse(dp.fuse, cp, num_kv_heads, arrive);
  }
  int e = launch_paged_decode(dp, plan_host ? num_ctas : batch, dtype, kv_dtype, stream);
  if (e == -1) return set_error(PKC_ERR_CUDA, "paged decode: could not build TMA tensor maps");
  if (e) return cuda_error(e, "paged decode launch");
  if (plan_host && !fused) {
    e = launch_contract(cp, batch, stream, true);
    if (e) return cuda_error(e, "contraction launch");
  }
  return PKC_OK;
}
}  // namespace

extern "C" {

int pkc_paged_decode_state(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                           int block_table_stride, const int32_t* cache_seqlens, int batch, int num_qo_heads,
                           int num_kv_heads, int head_dim, int page_size, int64_t num_pages, float sm_scale,
                           const int32_t* plan_host, void* workspace, size_t workspace_bytes, void* o, float* lse,
                           int dtype, void* stream) {
  return paged_decode_impl(q, k_cache, v_cache, block_table, block_table_stride, cache_seqlens, batch,
                           num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale, 1.f, 1.f,
                           plan_host, workspace, workspace_bytes, o, lse, dtype, dtype, stream);
}

int pkc_paged_decode_state_fp8(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int block_table_stride, const int32_t* cache_seqlens,
                               int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                               int64_t num_pages, float sm_scale, float k_scale, float v_scale,
                               const int32_t* plan_host, void* workspace, size_t workspace_bytes, void* o,
                               float* lse, void* stream) {
  return paged_decode_impl(q, k_cache, v_cache, block_table, block_table_stride, cache_seqlens, batch,
                           num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale, k_scale, v_scale,
                           plan_host, workspace, workspace_bytes, o, lse, PKC_F16, PKC_E4M3, stream);
}

int pkc_append_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache, const int32_t* block_table,
                  int block_table_stride, int32_t* cache_seqlens, const uint8_t* append_mask, int batch,
                  int num_kv_heads, int head_dim, int page_size, int64_t num_pages, int dtype, void* workspace,
                  size_t workspace_bytes, void* stream) {
  if (batch < 0 || num_kv_heads <= 0 || page_size < 1 || block_table_stride < 1 || num_pages < 0)
    return set_error(PKC_ERR_INVALID_ARG, "append_kv: bad size");
  if (head_dim != PKC_HEAD_DIM)
    return set_error(PKC_ERR_UNSUPPORTED, "append_kv: head_dim must be %d (got %d)", PKC_HEAD_DIM, head_dim);
  if (dtype != PKC_F16 && dtype != PKC_BF16 && dtype != PKC_E4M3)
    return set_error(PKC_ERR_INVALID_ARG, "append_kv: dtype must be PKC_F16, PKC_BF16 or PKC_E4M3 (got %d)", dtype);
  if (int rc = check_ws(workspace, workspace_bytes, PKC_STATUS_BYTES)) return rc;
  if (batch == 0) return PKC_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !cache_seqlens)
    return set_error(PKC_ERR_INVALID_ARG, "append_kv: NULL pointer");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return set_error(PKC_ERR_INVALID_ARG, "append_kv: K/V pointers must be 16-byte aligned");
  AppendParams ap;
  std::memset(&ap, 0, sizeof(ap));
  ap.k_new = k_new; ap.v_new = v_new; ap.k_cache = k_cache; ap.v_cache = v_cache;
  ap.block_table = block_table; ap.cache_seqlens = cache_seqlens; ap.mask = append_mask;
  ap.bt_stride = block_table_stride; ap.num_pages = num_pages;
  ap.hkv = num_kv_heads; ap.page_size = page_size;
  ap.row_bytes = PKC_HEAD_DIM * (dtype == PKC_E4M3 ? 1 : 2);
  ap.status = static_cast<int32_t*>(workspace);
  const int e = launch_append_kv(ap, batch, stream);
  return e ? cuda_error(e, "append_kv launch") : PKC_OK;
}

int pkc_set_decode_kernel(int which) {
  if (set_decode_kernel(which) != 0)
    return set_error(PKC_ERR_INVALID_ARG, "set_decode_kernel: which must be 0, 1 or 2 (got %d)", which);
  return PKC_OK;
}

int pkc_set_decode_schedule(int dynamic) {
  if (set_decode_schedule(dynamic) != 0)
    return set_error(PKC_ERR_INVALID_ARG, "set_decode_schedule: dynamic must be 0 or 1 (got %d)", dynamic);
  return PKC_OK;
}

int pkc_last_launch_blocks(int* prefix_blocks, int* decode_blocks) {
  if (!prefix_blocks || !decode_blocks) return set_error(PKC_ERR_INVALID_ARG, "last_launch_blocks: NULL pointer");
  *prefix_blocks = g_last_prefix_blocks;
  *decode_blocks = g_last_decode_blocks;
  return PKC_OK;
}

int pkc_set_contraction(int mode) {
  if (mode < 0 || mode > 2)
    return set_error(PKC_ERR_INVALID_ARG, "set_contraction: mode must be 0, 1 or 2 (got %d)", mode);
  g_fused_contraction.store(mode == 1 ? 1 : 0);
  set_contract_pdl(mode == 0 ? 1 : 0);
  return PKC_OK;
}

int pkc_set_cascade_small(int max_rows) {
  if (max_rows < 0) return set_error(PKC_ERR_INVALID_ARG, "set_cascade_small: max_rows must be >= 0 (got %d)", max_rows);
  g_cascade_small_rows.store(max_rows);
  return PKC_OK;
}

int pkc_set_prefix_ctas(int n) {
  if (n < 0) return set_error(PKC_ERR_INVALID_ARG, "set_prefix_ctas: n must be >= 0 (got %d)", n);
  g_prefix_ctas.store(n);
  return PKC_OK;
}

int pkc_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int32_t* gave_up_host, void* stream) {
  if (!gave_up_host) return set_error(PKC_ERR_INVALID_ARG, "selftest_wait_timeout: NULL result pointer");
  if (int rc = check_ws(workspace, workspace_bytes, PKC_STATUS_BYTES)) return rc;
  int32_t* status = static_cast<int32_t*>(workspace);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemsetAsync(status + 32, 0, sizeof(int32_t), st);
  if (!e) e = (cudaError_t)launch_wait_timeout(status, stream);
  int32_t v = 0;
  if (!e) e = cudaMemcpyAsync(&v, status + 32, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (!e) e = cudaStreamSynchronize(st);
  if (e) return cuda_error(e, "selftest_wait_timeout");
  *gave_up_host = v;
  return PKC_OK;
}

int pkc_prefix_attention_state(const void* q, const void* k_prefix, const void* v_prefix,
                               const int32_t* prefix_kv_indptr_host, const int32_t* prefix_req_indptr_host,
                               int n_prefix, int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                               float sm_scale, void* workspace, size_t workspace_bytes, float* o, float* lse,
                               int dtype, void* stream) {
  if (int rc = check_attn_dims(batch, num_qo_heads, num_kv_heads, head_dim, dtype)) return rc;
  const WsLayout L = ws_layout(batch, num_qo_heads, head_dim, 0);
  if (int rc = check_ws(workspace, workspace_bytes, L.fixed_end)) return rc;
  if (batch == 0) return PKC_OK;
  if (!q || !k_prefix || !v_prefix || !o || !lse) return set_error(PKC_ERR_INVALID_ARG, "prefix_attention_state: NULL pointer");
  if (!aligned16(q) || !aligned16(k_prefix) || !aligned16(v_prefix) || !aligned16(o))
    return set_error(PKC_ERR_INVALID_ARG, "prefix_attention_state: tensors must be 16-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  int32_t rb[PKC_MAX_PREFIX], re[PKC_MAX_PREFIX];
  if (int rc = indptr_ranges(prefix_req_indptr_host, n_prefix, rb, re)) return rc;
  PrefixSetup S;
  const StageSplit split = stage_split(prefix_kv_indptr_host, rb, re, n_prefix, num_qo_heads / num_kv_heads,
                                       num_kv_heads, 2, nullptr, false);
  if (int rc = setup_prefix(S, prefix_kv_indptr_host, rb, re, n_prefix, batch, num_qo_heads, num_kv_heads, sm_scale,
                            ws, workspace_bytes, L, status, split.prefix_blocks))
    return rc;
  int e = launch_prefix(S.pp, q, k_prefix, v_prefix, S.tokens, dtype, stream);
  if (e == -1) return set_error(PKC_ERR_CUDA, "prefix: could not build TMA tensor maps");
  if (e) return cuda_error(e, "prefix launch");
  ContractParams cp;
  std::memset(&cp, 0, sizeof(cp));
  cp.batch = batch; cp.hq = num_qo_heads; cp.mode = kContractAllRequests;
  fill_contract_prefix(cp, S);
  cp.o = o; cp.lse = lse; cp.out_dtype = PKC_F32; cp.status = status;
  e = launch_contract(cp, batch, stream);
  return e ? cuda_error(e, "contraction launch") : PKC_OK;
}

}  // extern "C"

namespace {
// The cascade for prefix groups given as request ranges (overlapping ranges:
// a multi-level cascade).
// prefix_pages (device) / page_indptr (host): a paged prefix read from the
// cache's page pool (k_prefix, v_prefix unused); nullptr: contiguous prefixes.
int cascade_impl(const void* q, const void* k_prefix, const void* v_prefix, const int32_t* prefix_kv_indptr_host,
                 const int32_t* req_begin, const int32_t* req_end, int n_prefix, const void* k_cache,
                 const void* v_cache, const int32_t* block_table, int block_table_stride, const int32_t* cache_seqlens,
                 int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
                 float sm_scale, const int32_t* plan_host, void* workspace, size_t workspace_bytes, void* o,
                 float* lse, int dtype, void* stream, const int32_t* prefix_pages = nullptr,
                 const int32_t* page_indptr = nullptr, int o_dtype = -1) {
  if (o_dtype < 0) o_dtype = dtype;
  if (prefix_pages) {
    k_prefix = k_cache;
    v_prefix = v_cache;
  }
  if (int rc = check_attn_dims(batch, num_qo_heads, num_kv_heads, head_dim, dtype)) return rc;
  if (int rc = check_plan(plan_host, batch)) return rc;
  if (page_size < 1 || block_table_stride < 1 || num_pages < 0)
    return set_error(PKC_ERR_INVALID_ARG, "page_size and block_table_stride must be >= 1, num_pages >= 0");
  const int num_ctas = plan_host ? plan_host[PKC_PLAN_NUM_CTAS] : 0;
  const WsLayout L = ws_layout(batch, num_qo_heads, head_dim, num_ctas);
  if (int rc = check_ws(workspace, workspace_bytes, L.fixed_end)) return rc;
  if (batch == 0) return PKC_OK;
  // The prefix tensors may be NULL when no group has a prefix token (a
  // shard of the keys that holds none of the prefixes).
  const bool no_prefix_tokens =
      prefix_kv_indptr_host && n_prefix >= 1 && prefix_kv_indptr_host[n_prefix] == prefix_kv_indptr_host[0];
  if (!q || ((!k_prefix || !v_prefix) && !no_prefix_tokens) || !k_cache || !v_cache || !block_table ||
      !cache_seqlens || !o || !lse)
    return set_error(PKC_ERR_INVALID_ARG, "cascade_decode: NULL pointer");
  if (!aligned16(q) || !aligned16(k_prefix) || !aligned16(v_prefix) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(o))
    return set_error(PKC_ERR_INVALID_ARG, "cascade_decode: tensors must be 16-byte aligned");
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  cudaEvent_t ev[4];
  for (int i = 0; i < 4; ++i) ev[i] = g_stage_events[i];
  g_stage_events[0] = g_stage_events[1] = g_stage_events[2] = g_stage_events[3] = nullptr;
  const bool timed = ev[0] || ev[1] || ev[2] || ev[3];
  PrefixSetup S;
  // The same split whether or not the call is timed, so that stage events
  // never change the result's rounding.
  const StageSplit split = stage_split(prefix_kv_indptr_host, req_begin, req_end, n_prefix,
                                       num_qo_heads / num_kv_heads, num_kv_heads, 2, plan_host, true);
  if (int rc = setup_prefix(S, prefix_kv_indptr_host, req_begin, req_end, n_prefix, batch, num_qo_heads,
                            num_kv_heads, sm_scale, ws, workspace_bytes, L, status, split.prefix_blocks))
    return rc;
  // Small batches: a shared prefix read by one 128-row query tile that holds
  // a handful of rows gives the tensor cores nothing to share, and the
  // prefix kernel's fixed latency and the contraction launch dominate such
  // a step.  Then the decode kernel reads each request's prefix itself, as
  // the first pages of its keys (the prefix tensors viewed as pages), and
  // writes the final state: one launch, no partial states.  Needs no plan,
  // contiguous non-overlapping groups of whole pages, and a contiguous
  // prefix.
  {
    const int small_rows = g_cascade_small_rows.load();
    bool small = small_rows > 0 && !plan_host && !prefix_pages && n_prefix <= PKC_FUSE_MAX_PREFIX &&
                 prefix_kv_indptr_host[0] % page_size == 0;
    for (int j = 0; small && j < n_prefix; ++j) {
      small = (prefix_kv_indptr_host[j + 1] - prefix_kv_indptr_host[j]) % page_size == 0 &&
              (req_end[j] - req_begin[j]) * (num_qo_heads / num_kv_heads) <= small_rows &&
              (j == 0 || req_begin[j] == req_end[j - 1]);
    }
    if (small) {
      DecodeParams dp;
      std::memset(&dp, 0, sizeof(dp));
      dp.q = q; dp.k_cache = k_cache; dp.v_cache = v_cache;
      dp.block_table = block_table; dp.cache_seqlens = cache_seqlens;
      dp.bt_stride = block_table_stride; dp.num_pages = num_pages;
      dp.batch = batch; dp.hq = num_qo_heads; dp.hkv = num_kv_heads; dp.page_size = page_size;
      dp.scale_log2 = sm_scale * 1.4426950408889634f;
      dp.v_scale = 1.f;
      dp.o_direct = o; dp.lse_direct = lse; dp.direct_f32 = o_dtype == PKC_F32 ? 1 : 0;
      dp.status = status;
      dp.prefix_as_pages = 1;
      dp.prefix_k = k_prefix; dp.prefix_v = v_prefix;
      dp.prefix_pages = prefix_kv_indptr_host[n_prefix] / page_size;
      dp.pre_n = n_prefix;
      for (int j = 0; j < n_prefix; ++j) dp.pre_req_indptr[j] = req_begin[j];
      dp.pre_req_indptr[n_prefix] = req_end[n_prefix - 1];
      for (int j = 0; j <= n_prefix; ++j) dp.pre_kv_indptr[j] = prefix_kv_indptr_host[j];
      // KV heads per block: the largest of 8, 4, 2, 1 dividing Hkv that still
      // gives every SM a block, else 1 (more blocks for a latency-bound step).
      dp.hg = 1;
      for (int hg = 8; hg >= 2; hg /= 2)
        if (num_kv_heads % hg == 0 && (int64_t)batch * (num_kv_heads / hg) >= num_sms()) {
          dp.hg = hg;
          break;
        }
      for (int i = 0; i < 2; ++i)
        if (ev[i]) cudaEventRecord(ev[i], (cudaStream_t)stream);
      g_last_prefix_blocks = 0;
      g_last_decode_blocks = batch * (num_kv_heads / dp.hg);
      const int e = launch_paged_decode(dp, batch, dtype, dtype, stream);
      if (e == -1) return set_error(PKC_ERR_CUDA, "cascade: could not build TMA tensor maps");
      if (e) return cuda_error(e, "cascade (small batch) decode launch");
      for (int i = 2; i < 4; ++i)
        if (ev[i]) cudaEventRecord(ev[i], (cudaStream_t)stream);
      return PKC_OK;
    }
  }
  // Decode blocks: one per plan CTA, or (dynamic schedule) fewer persistent
  // blocks taking the plan's chunks from the queue; the chunks are the
  // plan's either way.
  int decode_blocks = plan_host ? num_ctas : batch;
  if (plan_host && S.pp.n_blocks > 0) {
    if (split.decode_blocks == -1) decode_blocks = std::max(1, std::min(num_ctas, num_sms() - S.pp.n_blocks));
    else if (split.decode_blocks > 0) decode_blocks = std::min(num_ctas, split.decode_blocks);
  }
  if (prefix_pages) {
    if (!page_indptr) return set_error(PKC_ERR_INVALID_ARG, "paged prefix: prefix_page_indptr is NULL");
    if (page_size < 8 || 128 % page_size != 0)
      return set_error(PKC_ERR_UNSUPPORTED, "paged prefix: page_size must divide 128 and be >= 8 (got %d)",
                       page_size);
    if (page_indptr[0] < 0) return set_error(PKC_ERR_INVALID_ARG, "prefix_page_indptr must start >= 0");
    for (int j = 0; j < n_prefix; ++j) {
      const int len = prefix_kv_indptr_host[j + 1] - prefix_kv_indptr_host[j];
      if (page_indptr[j + 1] - page_indptr[j] < (len + page_size - 1) / page_size)
        return set_error(PKC_ERR_INVALID_ARG, "paged prefix: group %d has %d tokens but %d pages", j, len,
                         page_indptr[j + 1] - page_indptr[j]);
    }
    S.pp.prefix_pages = prefix_pages;
    for (int j = 0; j <= n_prefix; ++j) S.pp.page_indptr[j] = page_indptr[j];
    S.pp.page_size = page_size;
    S.pp.num_pages = num_pages;
  }
  auto mark = [&](int i) {
    if (ev[i]) cudaEventRecord(ev[i], (cudaStream_t)stream);
  };
  // The prefix and suffix stages are independent.  Unless per-stage timing
  // is asked for, all three launches go on the caller's stream as a chain of
  // programmatic dependents: the decode starts as soon as every prefix block
  // has started (on the SMs the prefix leaves, or those it releases) and
  // waits for the prefix grid only before its blocks exit; the contraction
  // starts once every decode block has, and waits for the decode grid (and
  // so the prefix's) before it reads either stage's states.  (With the
  // prefix on a side stream joined before the contraction, the join
  // serialised the contraction behind the decode: it started 2.5-3 us after
  // the decode's last block.)  Timed, the stages run one after the other.
  auto run_prefix = [&](void* st, cudaEvent_t start) -> int {
    const int r = launch_prefix(S.pp, q, k_prefix, v_prefix, S.tokens, dtype, st, start);
    if (r == -1) return set_error(PKC_ERR_CUDA, "prefix: could not build TMA tensor maps");
    if (r) return cuda_error(r, "prefix launch");
    return PKC_OK;
  };
  // 3. (planned now, launched last or fused) contraction + merge: prefix
  // pieces (+) suffix states -> final O, LSE
  ContractParams cp;
  std::memset(&cp, 0, sizeof(cp));
  cp.batch = batch; cp.hq = num_qo_heads; cp.mode = kContractAllRequests;
  cp.plan = plan_host ? reinterpret_cast<const int32_t*>(ws + L.plan) : nullptr;
  contract_plan_offsets(cp, plan_host);
  cp.suffix_o = reinterpret_cast<const float*>(ws + L.suffix_o);
  cp.suffix_lse = reinterpret_cast<const float*>(ws + L.suffix_lse);
  cp.part_o = reinterpret_cast<const float*>(ws + L.part_o);
  cp.part_lse = reinterpret_cast<const float*>(ws + L.part_lse);
  fill_contract_prefix(cp, S);
  cp.o = o; cp.lse = lse; cp.out_dtype = o_dtype; cp.status = status;
  // Fused: both stages' kernels count the sources they write, and the
  // writer of a (request, KV head) pair's last source merges the pair; the
  // counters are zeroed first, on the caller's stream before the prefix.
  const bool fused = g_fused_contraction.load() != 0 && n_prefix <= PKC_FUSE_MAX_PREFIX;
  FuseParams fuse;
  std::memset(&fuse, 0, sizeof(fuse));
  if (fused) {
    int32_t* arrive = reinterpret_cast<int32_t*>(ws + L.arrive);
    const cudaError_t me = cudaMemsetAsync(arrive, 0, 4 * (size_t)batch * num_kv_heads, (cudaStream_t)stream);
    if (me) return cuda_error(me, "cascade: counter reset");
    fill_fuse(fuse, cp, num_kv_heads, arrive);
    S.pp.fuse = fuse;
  }
  int e = 0;
  // 1. shared prefix: multi-query states on the tensor cores (stage event 0
  // is recorded right before the kernel, after its tensor maps are built)
  if (int rc = run_prefix(stream, ev[0])) return rc;
  mark(1);
  // 2. unique suffixes: paged decode states (unsplit -> suffix states)
  DecodeParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.q = q; dp.k_cache = k_cache; dp.v_cache = v_cache;
  dp.block_table = block_table; dp.cache_seqlens = cache_seqlens;
  dp.bt_stride = block_table_stride; dp.num_pages = num_pages;
  dp.batch = batch; dp.hq = num_qo_heads; dp.hkv = num_kv_heads; dp.page_size = page_size;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  dp.v_scale = 1.f;
  dp.plan = plan_host ? reinterpret_cast<const int32_t*>(ws + L.plan) : nullptr;
  dp.plan_words = plan_host ? plan_host[PKC_PLAN_TOTAL_WORDS] : 0;
  dp.o_direct = ws + L.suffix_o; dp.lse_direct = reinterpret_cast<float*>(ws + L.suffix_lse); dp.direct_f32 = 1;
  dp.part_o = reinterpret_cast<float*>(ws + L.part_o);
  dp.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  dp.status = status;
  dp.fuse = fuse;
  // the prefix's programmatic dependent, when this call launched a prefix grid
  dp.after_prefix = !timed && S.pp.n_blocks > 0 && S.pp.total_tiles > 0 ? 1 : 0;
  g_last_prefix_blocks = S.pp.n_blocks;
  g_last_decode_blocks = decode_blocks;
  e = launch_paged_decode(dp, decode_blocks, dtype, dtype, stream);
  if (e) return cuda_error(e, "paged decode launch");
  mark(2);
  if (!fused) {
    cp.prefix_after_wait = dp.after_prefix;  // prefix pieces only after the contraction's wait
    e = launch_contract(cp, batch, stream, !timed);
    if (e) return cuda_error(e, "contraction launch");
  }
  mark(3);
  return PKC_OK;
}
}  // namespace

extern "C" {

int pkc_cascade_decode(const void* q, const void* k_prefix, const void* v_prefix,
                       const int32_t* prefix_kv_indptr_host, const int32_t* prefix_req_indptr_host, int n_prefix,
                       const void* k_cache, const void* v_cache, const int32_t* block_table, int block_table_stride,
                       const int32_t* cache_seqlens, int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                       int page_size, int64_t num_pages, float sm_scale, const int32_t* plan_host, void* workspace,
                       size_t workspace_bytes, void* o, float* lse, int dtype, void* stream) {
  int32_t rb[PKC_MAX_PREFIX], re[PKC_MAX_PREFIX];
  if (int rc = check_attn_dims(batch, num_qo_heads, num_kv_heads, head_dim, dtype)) return rc;
  if (int rc = indptr_ranges(prefix_req_indptr_host, n_prefix, rb, re)) return rc;
  return cascade_impl(q, k_prefix, v_prefix, prefix_kv_indptr_host, rb, re, n_prefix, k_cache, v_cache, block_table,
                      block_table_stride, cache_seqlens, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                      num_pages, sm_scale, plan_host, workspace, workspace_bytes, o, lse, dtype, stream);
}

int pkc_cascade_decode_state(const void* q, const void* k_prefix, const void* v_prefix,
                             const int32_t* prefix_kv_indptr_host, const int32_t* prefix_req_indptr_host,
                             int n_prefix, const void* k_cache, const void* v_cache, const int32_t* block_table,
                             int block_table_stride, const int32_t* cache_seqlens, int batch, int num_qo_heads,
                             int num_kv_heads, int head_dim, int page_size, int64_t num_pages, float sm_scale,
                             const int32_t* plan_host, void* workspace, size_t workspace_bytes, float* o, float* lse,
                             int dtype, void* stream) {
  int32_t rb[PKC_MAX_PREFIX], re[PKC_MAX_PREFIX];
  if (int rc = check_attn_dims(batch, num_qo_heads, num_kv_heads, head_dim, dtype)) return rc;
  if (int rc = indptr_ranges(prefix_req_indptr_host, n_prefix, rb, re)) return rc;
  return cascade_impl(q, k_prefix, v_prefix, prefix_kv_indptr_host, rb, re, n_prefix, k_cache, v_cache, block_table,
                      block_table_stride, cache_seqlens, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                      num_pages, sm_scale, plan_host, workspace, workspace_bytes, o, lse, dtype, stream, nullptr,
                      nullptr, PKC_F32);
}

int pkc_cascade_decode_paged_prefix(
    const void* q, const int32_t* prefix_pages, const int32_t* prefix_page_indptr_host,
    const int32_t* prefix_kv_indptr_host, const int32_t* prefix_req_begin_host, const int32_t* prefix_req_end_host,
    int n_prefix, const void* k_cache, const void* v_cache, const int32_t* block_table, int block_table_stride,
    const int32_t* cache_seqlens, int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
    int64_t num_pages, float sm_scale, const int32_t* plan_host, void* workspace, size_t workspace_bytes, void* o,
    float* lse, int dtype, void* stream) {
  if (!prefix_pages) return set_error(PKC_ERR_INVALID_ARG, "paged prefix: prefix_pages is NULL");
  return cascade_impl(q, k_cache, v_cache, prefix_kv_indptr_host, prefix_req_begin_host, prefix_req_end_host,
                      n_prefix, k_cache, v_cache, block_table, block_table_stride, cache_seqlens, batch, num_qo_heads,
                      num_kv_heads, head_dim, page_size, num_pages, sm_scale, plan_host, workspace, workspace_bytes, o,
                      lse, dtype, stream, prefix_pages, prefix_page_indptr_host);
}

int pkc_cascade_decode_multilevel(
    const void* q, const void* k_prefix, const void* v_prefix, const int32_t* prefix_kv_indptr_host,
    const int32_t* prefix_req_begin_host, const int32_t* prefix_req_end_host, int n_prefix, const void* k_cache,
    const void* v_cache, const int32_t* block_table, int block_table_stride, const int32_t* cache_seqlens, int batch,
    int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int64_t num_pages, float sm_scale,
    const int32_t* plan_host, void* workspace, size_t workspace_bytes, void* o, float* lse, int dtype,
    void* stream) {
  return cascade_impl(q, k_prefix, v_prefix, prefix_kv_indptr_host, prefix_req_begin_host, prefix_req_end_host,
                      n_prefix, k_cache, v_cache, block_table, block_table_stride, cache_seqlens, batch, num_qo_heads,
                      num_kv_heads, head_dim, page_size, num_pages, sm_scale, plan_host, workspace, workspace_bytes, o,
                      lse, dtype, stream);
}

}  // extern "C"
