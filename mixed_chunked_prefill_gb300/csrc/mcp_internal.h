// Internal definitions shared by the host planner (host.cpp) and the CUDA
// kernels (*.cu).  Plain C++ data; no CUDA types.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "mcp.h"

namespace mcp {

enum ItemKind : int32_t { kDecodeItem = 0, kPrefillItem = 1 };

constexpr int kDecodeMaxRows = 16;   // query rows of one kv head on the decode path (m16 tile)
constexpr int kDecodeMaxHeads = 8;   // kv heads one decode item covers (one consumer warp each)
constexpr int kTileRows = 128;       // query rows of a tensor-core tile (TMEM lanes)
constexpr int kKvTile = 128;         // keys per tensor-core KV tile
constexpr int kPageSize = 16;        // tokens per KV block the kernels step over (a cache
                                     // page holds 1, 2 or 4 such blocks at page size 16,
                                     // 32, 64; at page size 8 a block spans two pages)
constexpr int kFwdThreads = 320;     // 10 warps: TMA producer, MMA issuer, 8 compute / producer

// kv heads covered by one decode item: the largest power of two <= 8 dividing H_kv
inline int decode_head_group(int num_kv_heads) {
  int g = 1;
  while (g * 2 <= kDecodeMaxHeads && num_kv_heads % (g * 2) == 0) g *= 2;
  return g;
}

// One unit of work of the fused kernel (one CTA).  32 bytes.
struct WorkItem {
  int32_t seg;         // segment index in the stream
  int16_t kv_head;     // first kv head covered
  int8_t kind;         // ItemKind
  int8_t num_heads;    // kv heads covered (decode: the head group; tensor-core tile: 1)
  int32_t q_begin;     // first query token of the item, counted inside the segment
  int32_t q_count;     // query tokens covered
  int32_t kv_begin;    // first key position (multiple of 16, or of 128 for tiles)
  int32_t kv_end;      // one past the last key position the item reads
  int32_t part_row;    // -1: write out/lse directly; else first partial row of the first head
  int32_t part_head_stride;  // partial rows between consecutive kv heads of the item
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

// A row group whose KV range was split: its num_splits partial results sit at
// rows part_row + k * rows (k < num_splits) of the partial buffers.  32 bytes.
struct CombineEntry {
  int32_t seg;
  int32_t kv_head;
  int32_t q_begin;
  int32_t q_count;
  int32_t num_splits;
  int32_t part_row;
  int32_t rows;      // q_count * G
  int32_t row_base;  // rows of all entries are numbered consecutively: this entry's first
};
static_assert(sizeof(CombineEntry) == 32, "CombineEntry layout");
// merged rows per combine block (one warp each); the plan stores, after the
// combine entries, the entry of the first row of every such block
constexpr int kCombineRowsPerBlock = 8;

struct FwdArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* cu_seqlens_q;
  const int32_t* seqlens_k;
  void* out;
  float* lse;
  const WorkItem* items;
  const CombineEntry* combine;
  float* part_o;
  float* part_lse;
  int32_t* error_word;
  int32_t num_items;
  int32_t num_combine;
  int32_t combine_rows;
  int32_t total_q;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t max_pages_per_seq;
  int32_t num_pages;
  float sm_scale;
  // non-paged K/V [total_k, H_kv, D] (cu_seqlens_k != nullptr): segment s's
  // keys are rows cu_seqlens_k[s] .. cu_seqlens_k[s+1]-1; block tables unused
  const int32_t* cu_seqlens_k = nullptr;
  int64_t total_k = 0;
  int32_t test_stall = 0;  // mcp_plan_options.test_stall of the plan
};

// Launchers (return a cudaError_t value; 0 = success).  Defined in *.cu.
int launch_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                  int32_t num_tokens, int32_t row_bytes, int64_t num_slots, void* k_cache,
                  void* v_cache, int32_t* error_word, void* stream);
int launch_mixed_attn(const FwdArgs& a, void* stream);
int launch_copy_pages(const void* k_src, const void* v_src, int32_t src_num_pages, void* k_dst,
                      void* v_dst, int32_t dst_num_pages, int32_t page_bytes,
                      const int32_t* src_pages, const int32_t* dst_pages, int32_t num,
                      int32_t* error_word, void* stream);
int launch_gather_rows(const void* src, int32_t num_src_rows, int32_t row_bytes,
                       const int32_t* rows, int32_t num_rows, void* dst, int32_t* error_word,
                       void* stream);
int launch_combine(const FwdArgs& a, void* stream);
int launch_merge_states(const float* o_parts, const float* lse_parts, int32_t n, int32_t rows,
                        int32_t heads, int32_t head_dim, void* out, float* lse_out, void* stream);
// Record `msg` as this thread's mcp_last_error() and return `status`.
// Defined in host.cpp.
int32_t set_error_code(int32_t status, const char* msg);
// Message of the last launcher failure that was not a CUDA error (e.g. a tensor
// map the driver rejected), "" otherwise.
const char* launch_detail();

// Host-side checks of mcp_mixed_attn_fwd's arguments other than the
// workspace: the plan, non-NULL tensors and their alignment.  MCP_OK when the
// plan has no work item.  Defined in host.cpp.
mcp_status check_fwd_args(const mcp_plan* plan, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* block_tables,
                          const int32_t* cu_seqlens_q, const int32_t* seqlens_k, const void* out,
                          const float* lse);

// mcp_mixed_attn_plan_host in one pass: fills *plan and resizes `lists` to the
// first plan->off_part_o bytes of the workspace layout (at least one byte),
// holding the work items and combine entries.  Defined in host.cpp.
mcp_status plan_to_host(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                        const int32_t* h_seqlens_k, const mcp_plan_options* opts, mcp_plan* plan,
                        std::vector<unsigned char>& lists);

}  // namespace mcp
