// Internal declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>

#include "pkc.h"

#define PKC_VERSION 100  // 0.1.0
#define PKC_HEAD_DIM 128
#define PKC_MAX_PREFIX 256
#define PKC_MAX_PREFIX_SPLITS 64
// The status block at the start of every workspace: word 0 is the status
// word (pkc_device_status), words 16-17 the dynamic decode queue's counters,
// word 32 the result of pkc_selftest_wait_timeout.
#define PKC_STATUS_BYTES 256

namespace pkc {

// Record an error message for pkc_last_error(); returns `code`.
int set_error(int code, const char* fmt, ...);
int cuda_error(int cuda_code, const char* what);

// Word offsets of the plan arrays (see pkc.h, "Load-balanced plan").
struct PlanLayout {
  int64_t cta_indptr, cta_work, work_unit, work_kv_begin, work_kv_end,
      work_partial, unit_req, unit_qtile, unit_kv_len, unit_n_chunks,
      unit_partial_begin, unit_list, cta_cost, work_order, order_rec, total;
};
PlanLayout plan_layout(int64_t n_units, int num_ctas);

// Byte offsets of the workspace regions (see pkc.h, pkc_workspace_size).
struct WsLayout {
  size_t arrive;           // fused contraction's arrival counters [batch * hq] int32
  size_t plan;             // plan region
  size_t suffix_o, suffix_lse;
  size_t part_o, part_lse;
  size_t prefix;           // first prefix split
  size_t prefix_split;     // bytes per prefix split ([B, Hq, D] + [B, Hq])
  size_t fixed_end;        // bytes before the prefix splits
};
WsLayout ws_layout(int batch, int hq, int d, int num_ctas);

// ---------------------------------------------------------------------------
// Kernel parameter blocks (plain data, passed by value to the kernels)
// ---------------------------------------------------------------------------

// Prefix groups a fused contraction can follow; calls with more groups use
// the standalone contraction kernel.
#define PKC_FUSE_MAX_PREFIX 16

// The contraction fused into the attention kernels (contract_common.cuh):
// the sources of every (request, KV head) pair, the pair's arrival counter
// and the final output.  Field names follow ContractParams, so one merge
// routine serves both.
struct FuseParams {
  int enabled;              // 1: the kernel that writes a pair's last source merges the pair
  int32_t* arrive;          // [batch * hkv] arrival counters, zeroed before each call
  int batch, hq, hkv, g;
  const int32_t* plan;      // device plan (decode plans: unit = request) or nullptr
  int32_t plan_words;       // the host plan's total words (the device copy must match)
  int32_t off_unit_list, off_unit_req, off_unit_n_chunks, off_unit_partial_begin;
  const float* suffix_o;    // direct suffix states (a cascade) or nullptr
  const float* suffix_lse;
  const float* part_o;      // partial states of split requests' chunks
  const float* part_lse;
  const float* prefix_o;    // prefix pieces [split, B, Hq, D] or nullptr
  const float* prefix_lse;
  int64_t prefix_stride_o, prefix_stride_lse;
  int n_prefix;
  int prefix_blocks;
  int64_t prefix_tiles;
  int32_t prefix_req_begin[PKC_FUSE_MAX_PREFIX];
  int32_t prefix_req_end[PKC_FUSE_MAX_PREFIX];
  int32_t prefix_slot_base[PKC_FUSE_MAX_PREFIX];
  int32_t prefix_kv_indptr[PKC_FUSE_MAX_PREFIX + 1];
  int32_t prefix_kvt_indptr[PKC_FUSE_MAX_PREFIX + 1];
  void* o;                  // final O [B, Hq, D] of out_dtype, LSE [B, Hq]
  float* lse;
  int out_dtype;
};

struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* cache_seqlens;
  int64_t bt_stride;
  int64_t num_pages;
  int batch, hq, hkv, page_size;
  float scale_log2;       // sm_scale * log2(e)
  const int32_t* plan;    // device copy of the plan, or nullptr
  int32_t plan_words;     // the host plan's total words (the device copy must match)
  int after_prefix;       // launched as the prefix kernel's programmatic dependent (cascade)
  void* o_direct;         // unsplit outputs: [B, Hq, D] (dtype or f32)
  float* lse_direct;      // [B, Hq]
  int direct_f32;         // 1: o_direct is float32 (suffix states)
  float* part_o;          // partial slots [slot, Hq, D]
  float* part_lse;        // [slot, Hq]
  int32_t* status;
  float v_scale;          // V = v_scale * stored V (1 for 16-bit caches)
  int dynamic;            // 1: blocks take the plan's chunks from a shared queue
  int32_t* sched;         // the queue's two counters (in the status block)
  FuseParams fuse;        // fused contraction (fuse.enabled) or none
  // Small-batch cascade (prefix_as_pages = 1; CUDA-core kernel, no plan):
  // each request's keys are its group's shared prefix, read as pages of the
  // contiguous prefix tensors (prefix_k / prefix_v viewed as
  // [prefix_pages, page_size, Hkv, 128]), then its cached suffix.  Group j
  // holds requests pre_req_indptr[j] .. pre_req_indptr[j+1]-1 and prefix
  // tokens pre_kv_indptr[j] .. pre_kv_indptr[j+1]-1, whole pages.
  int prefix_as_pages;
  const void* prefix_k;
  const void* prefix_v;
  int64_t prefix_pages;
  int pre_n;
  int32_t pre_req_indptr[PKC_FUSE_MAX_PREFIX + 1];
  int32_t pre_kv_indptr[PKC_FUSE_MAX_PREFIX + 1];
  int hg;                 // CUDA-core kernel: KV heads per block (0: the largest of 8, 4, 2, 1 dividing Hkv)
};

// Element kinds of a paged KV cache.
enum KvKind { kKvF16 = 0, kKvBF16 = 1, kKvE4M3 = 2 };

enum ContractMode {
  kContractPlanUnits = 0,  // rows = the plan's split + empty units
  kContractAllRequests = 1 // rows = every request
};

// Prefix groups hold contiguous request ranges that may overlap (a
// multi-level cascade: a request shares several prefixes).  Groups that
// share a request write their pieces to disjoint partial-slot ranges.
//
// Prefix work split: the prefix stage's KV tiles are laid out flat, pair
// after pair, where a pair is (128-row query tile, KV head) of one prefix
// group (group j's pairs are q = row_tile * Hkv + kv_head, each covering
// ceil(L_j / 128) KV tiles).  With T tiles over C thread blocks, block i
// takes tiles [floor(i T / C), floor((i+1) T / C)); a pair that spans
// several blocks is computed in pieces whose partial states are merged by
// the contraction.  The piece of block i in a pair starting at tile A is
// partial slot slot_base[group] + i - block_of(A).
#if defined(__CUDACC__)
#define PKC_HD __host__ __device__
#else
#define PKC_HD
#endif
PKC_HD inline int64_t prefix_block_begin(int i, int64_t T, int C) { return (int64_t)i * T / C; }
PKC_HD inline int prefix_block_of(int64_t x, int64_t T, int C) { return (int)(((x + 1) * C - 1) / T); }

struct ContractParams {
  int batch, hq;
  int mode;
  const int32_t* plan;      // device plan or nullptr
  int32_t plan_words;       // the host plan's total words (the device copy must match)
  int prefix_after_wait;    // the prefix stage may still run until griddepcontrol.wait returns
  // Word offsets of the plan arrays, copied from the host plan (they depend
  // only on batch and CTA count) so the kernel's first loads are the arrays.
  int32_t off_unit_list, off_unit_req, off_unit_n_chunks, off_unit_partial_begin;
  const float* suffix_o;    // direct suffix states or nullptr (no suffix)
  const float* suffix_lse;
  const float* part_o;
  const float* part_lse;
  const float* prefix_o;    // [split, B, Hq, D] or nullptr (no prefix)
  const float* prefix_lse;  // [split, B, Hq]
  int64_t prefix_stride_o, prefix_stride_lse;
  int prefix_splits;
  int n_prefix;
  int hkv, g;                                      // KV heads, query heads per KV head
  int prefix_blocks;                               // C of the prefix work split
  int64_t prefix_tiles;                            // T of the prefix work split
  int32_t prefix_req_begin[PKC_MAX_PREFIX];       // group j holds requests [begin, end)
  int32_t prefix_req_end[PKC_MAX_PREFIX];          //   (ranges may overlap: levels)
  int32_t prefix_slot_base[PKC_MAX_PREFIX];        // first partial slot of group j
  int32_t prefix_kv_indptr[PKC_MAX_PREFIX + 1];    // prefix tokens per group
  int32_t prefix_kvt_indptr[PKC_MAX_PREFIX + 1];   // first flat KV tile of each group
  void* o;
  float* lse;
  int out_dtype;
  int32_t* status;
};

struct PrefixParams {
  int batch, hq, hkv, g;
  float scale_log2;
  int n_prefix;
  int splits;                               // partial slots per row (most pieces of one pair)
  int n_blocks;                             // C: thread blocks of the work split
  int64_t total_tiles;                      // T: flat KV tiles over all pairs
  int32_t kv_indptr[PKC_MAX_PREFIX + 1];
  int32_t req_begin[PKC_MAX_PREFIX];        // group j holds requests [begin, end)
  int32_t req_end[PKC_MAX_PREFIX];
  int32_t slot_base[PKC_MAX_PREFIX];        // first partial slot of group j's pieces
  int32_t tile_indptr[PKC_MAX_PREFIX + 1];  // cumulative 128-row tiles
  int32_t kvt_indptr[PKC_MAX_PREFIX + 1];   // first flat KV tile of each group
  float* out_o;                             // [split, B, Hq, D]
  float* out_lse;                           // [split, B, Hq]
  int64_t split_stride_o, split_stride_lse;
  int32_t* status;
  // Paged prefix (the prefix KV stays in the page pool [num_pages,
  // page_size, Hkv, 128]): group j's tokens are pages
  // prefix_pages[page_indptr[j] ..] in order, the last one partly filled.
  // page_size divides 128.  nullptr prefix_pages: contiguous prefixes.
  const int32_t* prefix_pages;              // device
  int32_t page_indptr[PKC_MAX_PREFIX + 1];
  int page_size;
  int64_t num_pages;
  FuseParams fuse;                          // fused contraction (fuse.enabled) or none
};

struct AppendParams {
  const void* k_new;       // [batch, Hkv, 128] of the cache's element type
  const void* v_new;
  void* k_cache;           // [num_pages, page_size, Hkv, 128]
  void* v_cache;
  const int32_t* block_table;
  int32_t* cache_seqlens;  // incremented in place
  const uint8_t* mask;     // [batch] or nullptr (all append)
  int64_t bt_stride, num_pages;
  int hkv, page_size, row_bytes;  // row_bytes: one head's 128 elements
  int32_t* status;
};

// Launchers (defined in the .cu files); return a cudaError_t value.
int launch_merge_state(const void* va, const float* sa, const void* vb,
                       const float* sb, void* vo, float* so, int64_t rows,
                       int head_dim, int dtype, void* stream);
int launch_merge_states(const void* v, const float* s, void* vo, float* so,
                        int64_t n_tokens, int n_states, int n_heads,
                        int head_dim, int dtype, void* stream);
// The same with an output of out_dtype (fp32 states into a 16-bit result).
int launch_merge_states_to(const void* v, const float* s, void* vo, float* so,
                           int64_t n_tokens, int n_states, int n_heads,
                           int head_dim, int dtype, int out_dtype, void* stream);
// Paged decode: q of dtype (PKC_F16 / PKC_BF16) against a cache of
// kv_dtype (the same, or PKC_E4M3 with an fp16 q); picks the tensor-core
// kernel or the CUDA-core kernel.
int launch_paged_decode(const DecodeParams& p, int grid_x, int dtype, int kv_dtype,
                        void* stream);
int set_decode_kernel(int which);  // 0 auto, 1 CUDA cores, 2 tensor cores
int set_decode_schedule(int dynamic);  // 1 shared queue (default), 0 the plan's CTA lists
int decode_schedule_dynamic();         // the current choice of set_decode_schedule
int launch_wait_timeout(int32_t* status, void* stream);  // diagnostics (diag.cu)
int launch_paged_decode_simt(const DecodeParams& p, int grid_x, int dtype,
                             void* stream);
int launch_paged_decode_mma(const DecodeParams& p, int grid_x, int kv_kind,
                            void* stream);
// The instantiations with the fused contraction (p.fuse.enabled); mk, mv
// are the CUtensorMaps of the K and V pools.
int launch_paged_decode_mma_fused(const DecodeParams& p, int grid_x, int kv_kind, int hg,
                                  const void* mk, const void* mv, void* stream);
int launch_paged_decode_simt_fused(const DecodeParams& p, int grid_x, int dtype, int hg,
                                   const void* mk, const void* mv, const void* prefix_maps,
                                   void* stream);
// KV heads per block of the tensor-core kernel, or 0 if it cannot take
// this head count and page size.
int mma_decode_heads_per_block(int hkv, int page_size);
// after_decode: the kernel right before it on the stream is the suffix
// decode (it may then be launched as that grid's programmatic dependent).
int launch_contract(const ContractParams& p, int n_rows, void* stream, bool after_decode = false);
int set_contract_pdl(int on);  // 1: contraction as a programmatic dependent (default)
int launch_append_kv(const AppendParams& p, int batch, void* stream);
// q/k/v tensor maps are built inside; returns cudaError_t or -1 when the
// driver entry point for tensor maps is unavailable.
// Contiguous prefixes: k/v_prefix [prefix_tokens, Hkv, 128].  Paged
// prefixes (p.prefix_pages set): k/v_prefix are the page pools.
// start_event (a cudaEvent_t, or nullptr) is recorded on the stream right
// before the kernel launch, after the host work of building the maps.
int launch_prefix(const PrefixParams& p, const void* q, const void* k_prefix,
                  const void* v_prefix, int64_t prefix_tokens, int dtype,
                  void* stream, void* start_event = nullptr);

int num_sms();

// Encode a TMA tiled tensor map (a 128-byte CUtensorMap at `map`) over a
// 16-bit (PKC_F16, PKC_BF16) or byte (PKC_E4M3) tensor; dims[0] is the
// contiguous dimension.  Returns false if the
// driver entry point is unavailable or the encoding is rejected.
bool encode_tiled_map(void* map, const void* base, int dtype, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);

}  // namespace pkc
