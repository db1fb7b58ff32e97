// Host-side load-balanced plan (FlashInfer MLSys'25 notes, A3 "Dynamic-aware
// runtime", load-balanced scheduling steps 1-7; appendix D "split-K direct
// write" and the partial-output bound).  Runs on the CPU once per
// generation step; the result is a flat int32 buffer that pkc_plan_upload
// copies into the device workspace.
#include <algorithm>
#include <cstring>
#include <functional>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "pkc.h"
#include "pkc_internal.h"

namespace pkc {

PlanLayout plan_layout(int64_t n_units, int num_ctas) {
  PlanLayout L;
  const int64_t cap_work = (int64_t)num_ctas + n_units;
  int64_t o = PKC_PLAN_HEADER_WORDS;
  L.cta_indptr = o;         o += num_ctas + 1;
  L.cta_work = o;           o += cap_work;
  L.work_unit = o;          o += cap_work;
  L.work_kv_begin = o;      o += cap_work;
  L.work_kv_end = o;        o += cap_work;
  L.work_partial = o;       o += cap_work;
  L.unit_req = o;           o += n_units;
  L.unit_qtile = o;         o += n_units;
  L.unit_kv_len = o;        o += n_units;
  L.unit_n_chunks = o;      o += n_units;
  L.unit_partial_begin = o; o += n_units;
  L.unit_list = o;          o += n_units;
  o += (o & 1);  // float64 costs start on an 8-byte boundary
  L.cta_cost = o;           o += 2 * (int64_t)num_ctas;
  L.work_order = o;         o += cap_work;
  o = (o + 3) & ~int64_t(3);  // 16-byte records
  L.order_rec = o;          o += 4 * cap_work;
  L.total = o;
  return L;
}

}  // namespace pkc

using pkc::set_error;

extern "C" int pkc_plan_words(const int32_t* qo_len_host, int n, int tile_q,
                              int num_ctas, size_t* words) {
  if (n < 0 || tile_q < 1 || num_ctas < 1 || !words)
    return set_error(PKC_ERR_INVALID_ARG, "pkc_plan_words: n >= 0, tile_q >= 1, num_ctas >= 1 required");
  int64_t n_units = 0;
  for (int i = 0; i < n; ++i) {
    int64_t q = qo_len_host ? qo_len_host[i] : 1;
    if (q < 0) return set_error(PKC_ERR_INVALID_ARG, "pkc_plan_words: negative qo_len");
    n_units += (q + tile_q - 1) / tile_q;
  }
  if (n_units > INT32_MAX / 8)
    return set_error(PKC_ERR_INVALID_ARG, "pkc_plan_words: too many work units");
  *words = (size_t)pkc::plan_layout(n_units, num_ctas).total;
  return PKC_OK;
}

extern "C" int pkc_plan(const int32_t* qo_len_host, const int32_t* kv_len_host,
                        int n, int tile_q, int num_ctas, double alpha,
                        double beta, int32_t* plan, size_t plan_words) {
  if (!kv_len_host && n > 0) return set_error(PKC_ERR_INVALID_ARG, "pkc_plan: kv_len is NULL");
  if (!plan) return set_error(PKC_ERR_INVALID_ARG, "pkc_plan: plan buffer is NULL");
  size_t need = 0;
  int rc = pkc_plan_words(qo_len_host, n, tile_q, num_ctas, &need);
  if (rc) return rc;
  if (plan_words < need)
    return set_error(PKC_ERR_INVALID_ARG, "pkc_plan: plan buffer has %zu words, needs %zu", plan_words, need);

  // Step 1: work units (request, query tile), request-major.
  struct Unit { int32_t req, qtile, lq, kv; };
  std::vector<Unit> units;
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    int32_t q = qo_len_host ? qo_len_host[i] : 1;
    int32_t kv = kv_len_host[i];
    if (kv < 0) return set_error(PKC_ERR_INVALID_ARG, "pkc_plan: negative kv_len at %d", i);
    int32_t tiles = (q + tile_q - 1) / tile_q;
    for (int32_t j = 0; j < tiles; ++j)
      units.push_back({i, j, std::min(tile_q, q - j * tile_q), kv});
    total += (int64_t)tiles * kv;
  }
  const int64_t n_units = (int64_t)units.size();
  // Step 3: largest chunk L_kv = ceil(total / #CTA), at least one token.
  const int64_t L = std::max<int64_t>(1, (total + num_ctas - 1) / num_ctas);
  if (L > INT32_MAX) return set_error(PKC_ERR_INVALID_ARG, "pkc_plan: KV too long");

  // Step 4: cut each unit into consecutive chunks of <= L_kv tokens.
  struct Chunk { int32_t unit, b, e; };
  std::vector<Chunk> work;
  std::vector<int32_t> n_chunks(n_units, 0), first_chunk(n_units, 0);
  for (int64_t u = 0; u < n_units; ++u) {
    first_chunk[u] = (int32_t)work.size();
    for (int64_t b = 0; b < units[u].kv; b += L)
      work.push_back({(int32_t)u, (int32_t)b, (int32_t)std::min<int64_t>(b + L, units[u].kv)});
    n_chunks[u] = (int32_t)work.size() - first_chunk[u];
  }
  const int64_t n_work = (int64_t)work.size();

  // Step 5: longest first, equal lengths in ascending w.
  std::vector<int32_t> order(n_work);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
    return (work[x].e - work[x].b) > (work[y].e - work[y].b);
  });

  // Steps 6-7: min-priority queue of (cost, CTA index).
  using Entry = std::pair<double, int32_t>;
  std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> pq;
  for (int32_t c = 0; c < num_ctas; ++c) pq.push({0.0, c});
  std::vector<std::vector<int32_t>> lists(num_ctas);
  for (int32_t w : order) {
    Entry top = pq.top();
    pq.pop();
    lists[top.second].push_back(w);
    const Unit& un = units[work[w].unit];
    top.first = top.first + (alpha * un.lq + beta * (double)(work[w].e - work[w].b));
    pq.push(top);
  }
  std::vector<double> cost(num_ctas, 0.0);
  while (!pq.empty()) {
    cost[pq.top().second] = pq.top().first;
    pq.pop();
  }

  // Partial slots: chunks of split units, numbered in w order.
  std::vector<int32_t> partial(n_work, -1), partial_begin(n_units, -1);
  int32_t slot = 0;
  for (int64_t u = 0; u < n_units; ++u) {
    if (n_chunks[u] >= 2) {
      partial_begin[u] = slot;
      for (int32_t k = 0; k < n_chunks[u]; ++k) partial[first_chunk[u] + k] = slot++;
    }
  }

  // Serialise.
  const pkc::PlanLayout Lay = pkc::plan_layout(n_units, num_ctas);
  std::memset(plan, 0, sizeof(int32_t) * (size_t)Lay.total);
  int32_t* h = plan;
  h[PKC_PLAN_MAGIC] = PKC_PLAN_MAGIC_VALUE;
  h[PKC_PLAN_TOTAL_WORDS] = (int32_t)Lay.total;
  h[PKC_PLAN_NUM_CTAS] = num_ctas;
  h[PKC_PLAN_TILE_Q] = tile_q;
  h[PKC_PLAN_N_REQ] = n;
  h[PKC_PLAN_KV_CHUNK] = (int32_t)L;
  h[PKC_PLAN_N_UNITS] = (int32_t)n_units;
  h[PKC_PLAN_N_WORK] = (int32_t)n_work;
  h[PKC_PLAN_N_PARTIALS] = slot;
  h[PKC_PLAN_OFF_CTA_INDPTR] = (int32_t)Lay.cta_indptr;
  h[PKC_PLAN_OFF_CTA_WORK] = (int32_t)Lay.cta_work;
  h[PKC_PLAN_OFF_WORK_UNIT] = (int32_t)Lay.work_unit;
  h[PKC_PLAN_OFF_WORK_KV_BEGIN] = (int32_t)Lay.work_kv_begin;
  h[PKC_PLAN_OFF_WORK_KV_END] = (int32_t)Lay.work_kv_end;
  h[PKC_PLAN_OFF_WORK_PARTIAL] = (int32_t)Lay.work_partial;
  h[PKC_PLAN_OFF_UNIT_REQ] = (int32_t)Lay.unit_req;
  h[PKC_PLAN_OFF_UNIT_QTILE] = (int32_t)Lay.unit_qtile;
  h[PKC_PLAN_OFF_UNIT_KV_LEN] = (int32_t)Lay.unit_kv_len;
  h[PKC_PLAN_OFF_UNIT_N_CHUNKS] = (int32_t)Lay.unit_n_chunks;
  h[PKC_PLAN_OFF_UNIT_PARTIAL_BEGIN] = (int32_t)Lay.unit_partial_begin;
  h[PKC_PLAN_OFF_UNIT_LIST] = (int32_t)Lay.unit_list;
  h[PKC_PLAN_OFF_CTA_COST] = (int32_t)Lay.cta_cost;
  h[PKC_PLAN_OFF_WORK_ORDER] = (int32_t)Lay.work_order;
  h[PKC_PLAN_OFF_ORDER_REC] = (int32_t)Lay.order_rec;

  int32_t k = 0;
  for (int32_t c = 0; c < num_ctas; ++c) {
    h[Lay.cta_indptr + c] = k;
    for (int32_t w : lists[c]) h[Lay.cta_work + k++] = w;
  }
  h[Lay.cta_indptr + num_ctas] = k;
  for (int64_t w = 0; w < n_work; ++w) {
    h[Lay.work_unit + w] = work[w].unit;
    h[Lay.work_kv_begin + w] = work[w].b;
    h[Lay.work_kv_end + w] = work[w].e;
    h[Lay.work_partial + w] = partial[w];
  }
  int32_t n_split = 0, n_empty = 0;
  for (int64_t u = 0; u < n_units; ++u) {
    h[Lay.unit_req + u] = units[u].req;
    h[Lay.unit_qtile + u] = units[u].qtile;
    h[Lay.unit_kv_len + u] = units[u].kv;
    h[Lay.unit_n_chunks + u] = n_chunks[u];
    h[Lay.unit_partial_begin + u] = partial_begin[u];
    if (n_chunks[u] >= 2) h[Lay.unit_list + n_split++] = (int32_t)u;
  }
  for (int64_t u = 0; u < n_units; ++u)
    if (n_chunks[u] == 0) h[Lay.unit_list + n_split + n_empty++] = (int32_t)u;
  h[PKC_PLAN_N_SPLIT] = n_split;
  h[PKC_PLAN_N_EMPTY] = n_empty;
  std::memcpy(h + Lay.cta_cost, cost.data(), sizeof(double) * (size_t)num_ctas);
  // The chunks in the order of step 4, and one 16-byte record per chunk in
  // that order, for a kernel that takes them from a shared queue.
  for (int64_t i = 0; i < n_work; ++i) {
    const int32_t w = order[i];
    h[Lay.work_order + i] = w;
    int32_t* r = h + Lay.order_rec + 4 * i;
    r[0] = work[w].unit;
    r[1] = work[w].b;
    r[2] = work[w].e;
    r[3] = partial[w];
  }
  return PKC_OK;
}
