/*
 * mcp.h -- C ABI of the mixed chunked-prefill + decode paged-attention library
 * (GB300, sm_103a).
 *
 * One step of a chunked-prefill serving engine packs decode segments (one
 * query token each) and prefill chunks (many query tokens) into one token
 * stream.  For every layer the step (1) writes each new token's K/V into its
 * physical page through a slot mapping, then (2) runs one fused attention
 * forward over the whole stream, each segment against its own paged KV with the
 * query segment right-aligned to the end of its KV segment.
 *
 * Pages this follows (title, section):
 *   [W] wangyu.me, "大语言模型推理优化（二）：Chunked Prefill" -- sections
 *       "组装长序列", "记录 KV Cache 的长度", "Flash Attention 的 varlen 接口",
 *       "输入组装".
 *   [L] lpnh.cn, "技术融合剖析：Chunked Prefill如何借助FlashAttention/FlashInfer
 *       实现混合批次推理" -- sections 3.1 (packed Q/K/V and cu_seqlens),
 *       4.1 (block tables), 4.2 (append_paged_kv_cache).
 *   [K] kwkr.cn, hybrid-batch Chunked Prefill page -- sections
 *       "混合批次计算图与内存访问不对称性" (paged KV scattered in HBM),
 *       "平铺策略 / 掩码特化" (one fused kernel, mask only on the chunk's
 *       diagonal), "Triton 混合算子内核设计与实现" (online softmax).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every tensor is caller-owned.  Device tensors are dense, row-major,
 *    16-byte aligned; bf16 is IEEE bfloat16 stored as 2 bytes.
 *  - The library allocates no device memory at run time.  Calls that need
 *    scratch take a caller-provided device workspace sized by
 *    mcp_mixed_attn_plan().  The one exception is mcp_mixed_attn_fwd_noalloc,
 *    whose scratch is a fixed 16 MiB device array that the library holds on
 *    every GPU it is loaded on, for as long as the process runs.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Device work is enqueued asynchronously on it; host-only calls ignore it.
 *  - Return value: MCP_OK, or an mcp_status error.  Argument errors are found on
 *    the host before anything is launched; nothing is written in that case.
 *    mcp_last_error() gives a one-line description of the last failure on the
 *    calling thread.  No C++ exception crosses this boundary.
 *  - Layouts (shapes are [outer, ..., inner]):
 *      q, out        [T, H_q, D]        bf16   T = cu_seqlens_q[S]
 *      k_new, v_new  [T, H_kv, D]       bf16
 *      k/v cache     [num_pages, P, H_kv, D] bf16 ("NHD" pages, K and V apart)
 *      block_tables  [S, max_pages_per_seq] int32, logical -> physical page
 *      cu_seqlens_q  [S + 1] int32, exclusive prefix sum of query lengths
 *      seqlens_k     [S] int32, KV length of each segment INCLUDING this
 *                    step's tokens ([W] "记录 KV Cache 的长度")
 *      slot_mapping  [T] int64, physical_page * P + offset; < 0 = skip
 *      lse           [T, H_q] float32, natural-log sum of exp of the scores
 *    Query head h uses kv head h / (H_q / H_kv) (grouped-query attention;
 *    with H_q == H_kv this is [K]'s multi-head indexing).
 */
#ifndef MCP_H_
#define MCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MCP_ABI_VERSION 1

typedef enum mcp_status {
  MCP_OK = 0,
  MCP_ERR_INVALID_ARG = 1,         /* bad pointer, size, layout or metadata        */
  MCP_ERR_UNSUPPORTED = 2,         /* valid but not built (e.g. head_dim 80)       */
  MCP_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace smaller than the plan needs        */
  MCP_ERR_CUDA = 4,                /* a CUDA runtime/driver call failed            */
  MCP_ERR_TIMEOUT = 5,             /* a device-side bounded wait gave up           */
  MCP_ERR_DEVICE_CHECK = 6         /* a device-side range check failed             */
} mcp_status;

/* Static string for a status code (never NULL). */
const char* mcp_status_string(int32_t status);

/* One-line description of the last non-OK return on this thread ("" if none). */
const char* mcp_last_error(void);

/* MCP_ABI_VERSION of the loaded library. */
int32_t mcp_abi_version(void);

/* How the loaded library was built: MCP_BUILD_CHECKED when it was compiled
 * with MCP_CHECKED defined (a debugging build whose mcp_paged_kv_append also
 * checks on the device that its slots are distinct), else 0. */
#define MCP_BUILD_CHECKED 0x1
int32_t mcp_build_flags(void);

/* ------------------------------------------------------------------------- */
/* a1: paged KV append                                                       */
/* ------------------------------------------------------------------------- */
/*
 * Copy each new token's K and V rows into its physical slot of the paged
 * caches: for t in [0, num_tokens) with s = slot_mapping[t] >= 0,
 *   k_cache[s / P][s % P][:][:] = k_new[t][:][:]   (and the same for v).
 * Tokens with s < 0 are padding and are skipped.  This is the "write new K/V
 * through slot_mapping, then run attention" step of [W] "输入组装" and [L] 4.2
 * (physical address translation, scattered writes).  Slots must be distinct
 * within one call (the result is then independent of thread order; [L] 4.2's
 * atomics are not needed); a slot mapping with a repeated slot gives an
 * undefined cache row, except in MCP_CHECKED builds (mcp_build_flags()), where
 * a second kernel compares every pair of slots and sets MCP_DEVERR_SLOT_DUP
 * (O(num_tokens^2) work: a debugging aid).  mcp_build_slot_mapping never
 * produces one.  Slots >= num_pages * P are not written and are
 * reported by mcp_check_device_errors() as MCP_ERR_DEVICE_CHECK.
 *
 * k_new, v_new  device, bf16 [num_tokens, num_kv_heads, head_dim]
 * slot_mapping  device, int64 [num_tokens]
 * k_cache, v_cache device, bf16 [num_pages, page_size, num_kv_heads, head_dim]
 * error_word    device int32, or NULL; receives device-check bits (see below)
 * Requirements: num_tokens >= 0; (num_kv_heads * head_dim) % 8 == 0.
 * Bit-exact: the bytes of the new rows are copied unchanged.
 */
mcp_status mcp_paged_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                               int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                               int32_t page_size, int32_t num_pages, void* k_cache, void* v_cache,
                               int32_t* error_word, void* stream);

/*
 * Host helper for step assembly: the slot of every new token of the step
 * ([W] "输入组装").  Segment s's tokens are its last Lq_s KV positions,
 * Lq_s = cu_seqlens_q[s+1] - cu_seqlens_q[s], so token t of segment s sits at
 * position pos = seqlens_k[s] - Lq_s + (t - cu_seqlens_q[s]) and gets
 *   slot = block_tables[s][pos / P] * P + pos % P.
 * All pointers are HOST memory.  slot_mapping receives cu_seqlens_q[S] values.
 * Returns MCP_ERR_INVALID_ARG on malformed metadata, a page id outside
 * [0, num_pages), or two new tokens that land in the same slot (a physical page
 * listed twice in the block tables); slot_mapping is then partly written.
 */
mcp_status mcp_build_slot_mapping(const int32_t* block_tables, int32_t num_seqs,
                                  int32_t max_pages_per_seq, int32_t page_size, int32_t num_pages,
                                  const int32_t* cu_seqlens_q, const int32_t* seqlens_k,
                                  int64_t* slot_mapping);

/* ------------------------------------------------------------------------- */
/* a2..a9: mixed attention forward                                           */
/* ------------------------------------------------------------------------- */

typedef struct mcp_attn_desc {
  int32_t num_seqs;          /* S, segments in the stream                        */
  int32_t total_q;           /* T = cu_seqlens_q[S]                              */
  int32_t num_q_heads;       /* H_q                                              */
  int32_t num_kv_heads;      /* H_kv; must divide H_q                            */
  int32_t head_dim;          /* D: 64, 96, 128 or 256 (96 zero-padded to 128)   */
  int32_t page_size;         /* P: 1, 8, 16, 32 or 64                           */
  int32_t max_pages_per_seq; /* row length of block_tables                       */
  int32_t num_pages;         /* pages in each cache tensor                       */
  float sm_scale;            /* score scale > 0, e.g. 1/sqrt(D) ([K] kernel launch) */
} mcp_attn_desc;

typedef struct mcp_plan_options {
  int32_t num_sms;              /* 0 = query the current device                  */
  int32_t decode_split_tokens;  /* KV tokens per decode work item; 0 = auto      */
  int32_t prefill_split_tokens; /* KV tokens per prefill work item; 0 = auto     */
  int32_t test_stall;           /* 0 in production.  1 (for failure-detection    */
                                /* tests): every tensor-core item leaves its Q   */
                                /* tile unloaded and every device wait gives up  */
                                /* after ~1 ms, so those items end through the   */
                                /* bounded-wait abort path: no output rows, the  */
                                /* error word reports MCP_ERR_TIMEOUT            */
  int32_t reserved[4];          /* must be 0                                     */
} mcp_plan_options;

/* Filled by mcp_mixed_attn_plan(); read by mcp_mixed_attn_fwd().  Plain data:
 * it may be copied; its fields describe the workspace layout. */
typedef struct mcp_plan {
  int32_t magic;
  int32_t num_items;          /* work items (CTAs of the fused kernel)           */
  int32_t num_decode_items;   /* items on the decode (split-KV) path             */
  int32_t num_prefill_items;  /* items on the tensor-core chunk path             */
  int32_t num_combine;        /* row groups merged by the combine kernel         */
  int32_t decode_split_tokens;
  int32_t prefill_split_tokens;
  int32_t num_sms;
  int64_t partial_rows;       /* rows of split partial results                   */
  int64_t off_items, off_combine, off_part_o, off_part_lse, off_error;
  int64_t workspace_bytes;    /* bytes the workspace must have                   */
  mcp_attn_desc desc;         /* the description the plan was built for          */
  int32_t combine_rows;       /* query rows (token, head) merged by the combine  */
  int32_t test_stall;         /* mcp_plan_options.test_stall                     */
  int32_t reserved[6];
} mcp_plan;

/*
 * Plan one step.  Validates the step's metadata on the host and splits it
 * into work items for the fused kernel:
 *  - a segment with Lq * G <= 16 (G = H_q / H_kv) goes to the decode path:
 *    one item per (kv head, KV range); its G*Lq query rows share each K/V page;
 *  - any other segment goes to the tensor-core path: one item per (kv head,
 *    tile of 128/G query tokens, KV range), the G query heads of a kv head
 *    packed into 128 rows.
 * Long KV ranges are split; the combine kernel merges the splits.  Items are
 * ordered so the longest go first and tiles reading the same K/V run side by
 * side.
 *
 * h_cu_seqlens_q [S+1], h_seqlens_k [S]: HOST copies of the step metadata.
 * opts: may be NULL (all defaults).
 * Requirements ([W] "Flash Attention 的 varlen 接口"): cu_seqlens_q[0] == 0,
 * non-decreasing, cu_seqlens_q[S] == total_q; 0 <= Lq_s <= seqlens_k[s],
 * seqlens_k[s] >= 1 when Lq_s > 0; ceil(seqlens_k[s] / P) <= max_pages_per_seq.
 *
 * workspace == NULL: sizing only; *plan receives the work counts and
 *   plan->workspace_bytes; nothing is copied and `stream` is unused.
 * workspace != NULL: device memory of workspace_bytes >= plan->workspace_bytes,
 *   256-byte aligned.  The work lists are copied into it on `stream` (from a
 *   host buffer that is staged before this call returns) and its device error
 *   word is cleared.  A workspace must not be re-planned while a previous
 *   mcp_mixed_attn_fwd that uses it is still running on another stream.
 */
mcp_status mcp_mixed_attn_plan(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                               const int32_t* h_seqlens_k, const mcp_plan_options* opts,
                               mcp_plan* plan, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Same plan as mcp_mixed_attn_plan, written to HOST memory instead of a
 * device workspace: host_buffer receives the first plan->off_part_o bytes of
 * the workspace layout (the work items at plan->off_items, the combine
 * entries at plan->off_combine and, right after them, the combine's index of
 * the entry holding the first row of each block of 8 merged rows, int32).
 * A caller that copies those bytes to the
 * start of its device workspace and zeroes the 4-byte error word at
 * plan->off_error gets the same state mcp_mixed_attn_plan uploads.
 * host_buffer == NULL: sizing only.  Host only; needs no GPU when
 * opts->num_sms > 0.  Item layout (32 bytes, little-endian): int32 segment,
 * int16 first kv head, int8 kind (0 decode, 1 tensor-core tile), int8 number of
 * kv heads covered, int32 first query token inside the segment, int32 query
 * token count, int32 first key, int32 one past the last key, int32 partial row
 * of the first head (-1 = written directly), int32 partial rows between heads.
 * Combine entry (32 bytes, int32): segment, kv head, first query token, query
 * token count, number of splits, first partial row, rows per split, 0.
 */
mcp_status mcp_mixed_attn_plan_host(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                                    const int32_t* h_seqlens_k, const mcp_plan_options* opts,
                                    mcp_plan* plan, void* host_buffer, size_t host_bytes);

/*
 * The fused mixed attention forward ([W] "Flash Attention 的 varlen 接口":
 * the i-th query segment attends only to the i-th KV segment, right-aligned
 * causal; [K] "平铺策略 / 掩码特化": one kernel for prefill chunks and
 * decodes).  For every segment s, query head h and query i in [0, Lq_s):
 *   s_j  = sm_scale * <q[i,h], k_j>  for KV positions j <= i + (Lk_s - Lq_s)
 *   out[i,h] = sum_j softmax(s)_j v_j,   lse[i,h] = ln sum_j exp(s_j)
 * with k_j, v_j the kv head h / G of position j, read through block_tables.
 * Runs the fused kernel and, when the plan split a KV range, the combine
 * kernel, both on `stream`.  The caches must already hold this step's K/V
 * (mcp_paged_kv_append earlier on the same stream).
 *
 * q        device bf16 [T, H_q, D]
 * k_cache, v_cache device bf16 [num_pages, P, H_kv, D]
 * block_tables, cu_seqlens_q, seqlens_k: DEVICE copies of the metadata the
 *          plan was built from (same values).
 * out      device bf16 [T, H_q, D]  (rounded to nearest even from fp32)
 * lse      device float32 [T, H_q], or NULL
 * workspace: the one the plan was uploaded into.
 * Rows of segments with Lq = 0 do not exist; no other output row is skipped.
 */
mcp_status mcp_mixed_attn_fwd(const mcp_plan* plan, const void* q, const void* k_cache,
                              const void* v_cache, const int32_t* block_tables,
                              const int32_t* cu_seqlens_q, const int32_t* seqlens_k, void* out,
                              float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronise `stream`, read the device error word of `workspace` (the one
 * mcp_mixed_attn_fwd and the plan's kernels write; or any int32 error word
 * given to mcp_paged_kv_append) and clear it.  Returns MCP_OK,
 * MCP_ERR_TIMEOUT (a bounded device wait gave up) or MCP_ERR_DEVICE_CHECK
 * (an out-of-range page or slot was skipped).
 */
mcp_status mcp_check_device_errors(int32_t* error_word, void* stream);

/* Device address of the error word inside a workspace laid out by `plan`. */
int32_t* mcp_workspace_error_word(const mcp_plan* plan, void* workspace);

/* ------------------------------------------------------------------------- */
/* a8 standalone: merge split attention states                               */
/* ------------------------------------------------------------------------- */
/*
 * Merge n attention results over disjoint key sets (split-KV): for each row r
 * and head h, with M = max_k lse[k,r,h] and w_k = exp(lse[k,r,h] - M),
 *   out[r,h,:] = sum_k w_k o[k,r,h,:] / sum_k w_k,  lse_out = M + ln sum_k w_k.
 * A part with lse = -inf carries weight 0.  Not on the pages: it is the plain
 * identity that makes split-KV equal to unsplit attention.
 *
 * o_parts   device float32 [n, rows, heads, head_dim], each part normalised
 * lse_parts device float32 [n, rows, heads]
 * out       device bf16 [rows, heads, head_dim];  lse_out float32 or NULL
 */
mcp_status mcp_merge_states(const float* o_parts, const float* lse_parts, int32_t n, int32_t rows,
                            int32_t heads, int32_t head_dim, void* out, float* lse_out,
                            void* stream);

/* ------------------------------------------------------------------------- */
/* mixed attention forward without a workspace                              */
/* ------------------------------------------------------------------------- */
/*
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory when they run a step (e.g. inside a framework
 * whose memory pool owns every device allocation, or a server that must not
 * grow its device footprint after start-up).  It plans the step on the host
 * exactly like mcp_mixed_attn_plan and runs mcp_mixed_attn_fwd, but keeps the
 * work lists, split partials and error word in a fixed 16 MiB device array
 * owned by the library instead of a caller workspace.  It allocates no device
 * memory (the planner's host-side working lists use ordinary host memory).
 *
 * Inputs and outputs are those of mcp_mixed_attn_plan (host metadata, opts may
 * be NULL) and mcp_mixed_attn_fwd (device tensors, stream).
 * error_word: NULL, or receives the device address of the error word of this
 *   call (valid until the next call; pass it to mcp_check_device_errors).
 * Limits:
 *  - a step whose plan needs more than 16 MiB of scratch returns
 *    MCP_ERR_WORKSPACE_TOO_SMALL before anything is launched;
 *  - every GPU that loads the library holds the 16 MiB array until exit;
 *  - argument errors (bad metadata, NULL or misaligned tensors) are returned
 *    before the array is touched or anything is enqueued;
 *  - all calls share that array (it keeps the last call's contents; this call
 *    clears what must start at zero), so calls whose GPU work overlaps -- on
 *    different streams or from different threads -- race; order them;
 *  - the first call on each device looks up the array's device address; make
 *    that first call before any CUDA stream capture.
 */
mcp_status mcp_mixed_attn_fwd_noalloc(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                                      const int32_t* h_seqlens_k, const mcp_plan_options* opts,
                                      const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, const int32_t* cu_seqlens_q,
                                      const int32_t* seqlens_k, void* out, float* lse,
                                      int32_t** error_word, void* stream);

/* ------------------------------------------------------------------------- */
/* Sampled rows: logits_indices, attention for listed rows, row gather       */
/* ------------------------------------------------------------------------- */
/*
 * [W] "采样：只有该出字的请求才出字": the output layer computes logits only at
 * the last position of every segment, logits_indices = query_start_loc[1:] - 1,
 * and the sampler keeps them only for decode segments and for chunks that
 * finish their prompt.  Host-only: h_out receives the index of the last token
 * of every segment with at least one token this step, in segment order, and
 * *count their number (at most num_seqs).  h_sample_mask [S] (or NULL = all):
 * segments with mask 0 are left out.  A segment without tokens contributes no
 * index (the printed formula would name the previous segment's last token).
 */
mcp_status mcp_build_logits_indices(int32_t num_seqs, const int32_t* h_cu_seqlens_q,
                                    const uint8_t* h_sample_mask, int32_t* h_out,
                                    int32_t* count);

/*
 * Plan attention for the listed query rows only (e.g. logits_indices in the
 * last layer, where only the sampled positions feed the output head).
 * h_rows [num_rows]: HOST token indices into the packed stream, strictly
 * increasing, each in [0, total_q).  Each listed token attends exactly as in
 * the full step (its segment's paged KV, right-aligned causal); rows of out /
 * lse not listed are not written by mcp_mixed_attn_fwd with this plan.
 * Consecutive listed tokens of one segment share a work item.  Everything
 * else as mcp_mixed_attn_plan (workspace NULL = sizing only).
 */
mcp_status mcp_mixed_attn_plan_rows(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                                    const int32_t* h_seqlens_k, const int32_t* h_rows,
                                    int32_t num_rows, const mcp_plan_options* opts,
                                    mcp_plan* plan, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* mcp_mixed_attn_plan_rows that writes the work lists into a HOST buffer (as
 * mcp_mixed_attn_plan_host; host_buffer NULL = sizing only). */
mcp_status mcp_mixed_attn_plan_rows_host(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                                         const int32_t* h_seqlens_k, const int32_t* h_rows,
                                         int32_t num_rows, const mcp_plan_options* opts,
                                         mcp_plan* plan, void* host_buffer, size_t host_bytes);

/*
 * dst[i][:] = src[rows[i]][:] for i < num_rows (device; rows of row_bytes
 * bytes, bit-exact) -- e.g. the attention output [T, H_q, D] at
 * logits_indices, packed for the output head.  row_bytes % 16 == 0; src, dst
 * 16-byte aligned; rows: device int32.  An index outside [0, num_src_rows)
 * writes a zero row and sets MCP_DEVERR_ROW_RANGE in error_word (if not NULL).
 */
mcp_status mcp_gather_rows(const void* src, int32_t num_src_rows, int32_t row_bytes,
                           const int32_t* rows, int32_t num_rows, void* dst, int32_t* error_word,
                           void* stream);

/* ------------------------------------------------------------------------- */
/* KV page copies between pools: swap-out / swap-in                          */
/* ------------------------------------------------------------------------- */
/*
 * [X] m.xxqk.cn "动态批处理中的抢占与优先级调度", section "Prefill 算力霸占与抢占
 * 策略演进": when the KV pool runs out, a preempted sequence's KV pages are
 * copied out to host memory (swap-out) and copied back into free pages once
 * memory is available again (swap-in).  For i < num:
 *   k_dst[dst_pages[i]] = k_src[src_pages[i]]   (whole pages of page_bytes
 *   v_dst[dst_pages[i]] = v_src[src_pages[i]]    bytes, bit-exact)
 * Pools: k_src / v_src with src_num_pages pages, k_dst / v_dst with
 * dst_num_pages pages; each pool is device memory or page-locked host memory
 * (a swap pool), read and written by the kernel directly.  page_bytes =
 * page_size * num_kv_heads * head_dim * 2 for the caches of this library; a
 * multiple of 16.  src_pages, dst_pages: int32 [num], device (or page-locked
 * host) memory.  Destination pages must be distinct; when src and dst are
 * the same pool, no destination page may also be a source page.  A page id
 * outside its pool skips that page and sets MCP_DEVERR_PAGE_RANGE in
 * error_word (if not NULL).  Asynchronous on `stream`.
 */
mcp_status mcp_kv_copy_pages(const void* k_src, const void* v_src, int32_t src_num_pages,
                             void* k_dst, void* v_dst, int32_t dst_num_pages, int32_t page_bytes,
                             const int32_t* src_pages, const int32_t* dst_pages, int32_t num,
                             int32_t* error_word, void* stream);

/* ------------------------------------------------------------------------- */
/* Step builder: the chunked-prefill scheduler (host-only)                   */
/* ------------------------------------------------------------------------- */
/*
 * Decides, step by step, which requests run and with how many tokens, and
 * builds the step's metadata.  [W] wangyu.me sections "Token 预算：
 * max_num_batched_tokens" and "调度器：running 优先，waiting 填充": each request
 * tracks num_computed_tokens; a step has a token budget; running requests go
 * first (decodes and unfinished prompts, in arrival order), then waiting
 * requests fill what is left, a prompt taking as many tokens as the budget
 * allows; long_prefill_token_threshold (0 = none) caps one chunk, for running
 * and newly admitted prompts alike.
 * [W] "采样": the step's logits_indices are the last token of every segment;
 * only decodes and chunks that finish their prompt sample.  [X] m.xxqk.cn
 * "动态批处理中的抢占与优先级调度": waiting requests are admitted by priority
 * (higher first, then arrival); when the KV page pool cannot hold a running
 * request's next tokens, the lowest-priority, latest-arrived running request
 * is preempted -- recomputed (its pages are freed and it re-enters the
 * waiting queue with all its tokens as prompt) or swapped (its pages are
 * listed for swap-out to host pool pages and swapped back in, into free
 * device pages, when it resumes).  Page 16-token granularity, one page table
 * row per request.  The object and its arrays live in host memory.
 */
typedef struct mcp_sched_config {
  int32_t max_num_batched_tokens;       /* token budget of one step (>= 1)           */
  int32_t long_prefill_token_threshold; /* 0 = none, else max tokens of one chunk    */
  int32_t max_num_seqs;                 /* segments in one step (>= 1)               */
  int32_t num_pages;                    /* device KV pool pages                      */
  int32_t page_size;                    /* tokens per page (1, 8, 16, 32 or 64)      */
  int32_t max_pages_per_seq;            /* block-table row length                    */
  int32_t preempt_swap;                 /* 0 = recompute, 1 = swap to the host pool  */
  int32_t num_host_pages;               /* host swap pool pages (swap mode)          */
  int32_t reserved[4];                  /* must be 0                                 */
} mcp_sched_config;

typedef struct mcp_sched mcp_sched; /* opaque */

/* One step's plan.  Arrays are owned by the scheduler and stay valid until
 * the next mcp_sched_schedule() / mcp_sched_destroy().  Execute the step as:
 * swap-out copies, swap-in copies, then append + attention with the arrays. */
typedef struct mcp_sched_output {
  int32_t num_seqs;            /* segments of the step (0 = nothing runnable)      */
  int32_t total_q;             /* tokens of the step                               */
  const int64_t* request_ids;  /* [num_seqs]                                       */
  const int32_t* cu_seqlens_q; /* [num_seqs + 1]                                   */
  const int32_t* seqlens_k;    /* [num_seqs]: tokens in the cache after the step   */
  const int32_t* block_tables; /* [num_seqs, max_pages_per_seq], -1 padded         */
  const uint8_t* sample_mask;  /* [num_seqs]: 1 = the segment samples a token      */
  const int32_t* logits_indices; /* [num_logits]: last token of sampling segments  */
  int32_t num_logits;
  int32_t num_swap_out;        /* device page -> host page copies, before the step */
  const int32_t* swap_out_device_pages;
  const int32_t* swap_out_host_pages;
  int32_t num_swap_in;         /* host page -> device page copies, before the step */
  const int32_t* swap_in_host_pages;
  const int32_t* swap_in_device_pages;
  int32_t num_preempted;       /* requests preempted while building this step      */
  const int64_t* preempted_ids;
  int32_t reserved[4];
} mcp_sched_output;

mcp_status mcp_sched_create(const mcp_sched_config* config, mcp_sched** sched);
/* Queue a request: a prompt of prompt_len tokens, then up to max_new_tokens
 * sampled tokens; ids must be unique among live requests. */
mcp_status mcp_sched_add_request(mcp_sched* sched, int64_t request_id, int32_t prompt_len,
                                 int32_t max_new_tokens, int32_t priority);
/* Build the next step (out receives views of the scheduler's arrays). */
mcp_status mcp_sched_schedule(mcp_sched* sched, mcp_sched_output* out);
/* The last scheduled step ran: advance num_computed_tokens, add one sampled
 * token to every sampling segment, retire requests that reached
 * max_new_tokens (their pages return to the pool).  *num_finished (if not
 * NULL) receives how many finished; their ids go to finished_ids (if not
 * NULL, room for num_seqs ids). */
mcp_status mcp_sched_finish_step(mcp_sched* sched, int32_t* num_finished, int64_t* finished_ids);
/* Counts: waiting, running, swapped, finished requests; free device pages. */
mcp_status mcp_sched_stats(const mcp_sched* sched, int32_t* waiting, int32_t* running,
                           int32_t* swapped, int64_t* finished, int32_t* free_pages);
mcp_status mcp_sched_destroy(mcp_sched* sched);

/* ------------------------------------------------------------------------- */
/* One step from host memory, two steps in flight                            */
/* ------------------------------------------------------------------------- */
/*
 * The whole step of [W] "输入组装" from host arrays: the step's metadata and
 * new tokens are copied to the device, the new K/V are appended to the paged
 * caches (a1), the fused forward runs (a2..a9), and out (and lse) are copied
 * back to host memory.  Up to two steps are in flight: while step n's kernels
 * run on the caller's stream, step n+1 is planned on the host and its inputs
 * are copied in on a second stream, and step n's outputs are copied out on a
 * third.  Each in-flight step has its own staging slot (device inputs,
 * outputs, metadata and workspace; page-locked metadata, slot mapping and
 * work lists), so no step overwrites buffers another still reads.  The
 * append of step n+1 runs after the forward of step n on the caller's stream.
 *
 * Memory is caller-owned: mcp_host_step_arena_bytes() sizes a device arena and
 * a page-locked host arena for two slots.  The library keeps only a small host
 * object (two streams, six events) between mcp_host_step_create() and
 * mcp_host_step_destroy().  One object is used by one host thread at a time.
 */
typedef struct mcp_host_step_limits {
  int32_t max_tokens;        /* T of any step                                    */
  int32_t max_seqs;          /* S of any step                                    */
  int32_t max_pages_per_seq; /* row length of every step's block_tables          */
  int32_t reserved0;         /* must be 0                                        */
  int64_t workspace_bytes;   /* device workspace per slot (work lists + split
                                partials, see mcp_plan); 0 = 64 MiB              */
  int64_t list_bytes;        /* page-locked work-list bytes per slot; 0 = 4 MiB  */
  int32_t reserved[4];       /* must be 0                                        */
} mcp_host_step_limits;

typedef struct mcp_host_step mcp_host_step; /* opaque */

/*
 * Bytes of the device arena and of the page-locked host arena for `limits`.
 * shape supplies num_q_heads, num_kv_heads, head_dim, page_size, num_pages and
 * sm_scale (validated as in mcp_mixed_attn_plan; its num_seqs, total_q and
 * max_pages_per_seq are ignored).  Host-only.
 */
mcp_status mcp_host_step_arena_bytes(const mcp_attn_desc* shape, const mcp_host_step_limits* limits,
                                     size_t* device_bytes, size_t* host_bytes);

/*
 * device_arena: device memory of the current device, 256-byte aligned.
 * host_arena: page-locked host memory (cudaHostAlloc or cudaHostRegister),
 * 256-byte aligned; rejected with MCP_ERR_INVALID_ARG if it is not page-locked.
 * stream: the stream the kernels run on.  *step receives the object.
 */
mcp_status mcp_host_step_create(const mcp_attn_desc* shape, const mcp_host_step_limits* limits,
                                void* device_arena, size_t device_bytes, void* host_arena,
                                size_t host_bytes, void* stream, mcp_host_step** step);

/*
 * Enqueue one step.  HOST pointers: cu_seqlens_q [S+1], seqlens_k [S] and
 * block_tables [S, max_pages_per_seq] int32 are read before the call returns;
 * q [T, H_q, D], k_new / v_new [T, H_kv, D] bf16 are read by the asynchronous
 * copy-in (keep them unchanged until mcp_host_step_wait(ticket) returns;
 * page-locked memory lets the copies overlap the kernels); out [T, H_q, D]
 * bf16 and lse [T, H_q] float32 (or NULL) are written by the copy-out (valid
 * after mcp_host_step_wait(ticket)).  k_cache, v_cache: device caches as in
 * mcp_paged_kv_append.  *ticket receives the step's number (0, 1, ...).
 * Metadata errors (including a block-table page outside the pool) are
 * returned before anything is enqueued.  Blocks only while the step two
 * before this one is still running (its slot is reused); if that step failed
 * on the device and was not waited for, its error is returned here and
 * nothing is enqueued.
 */
mcp_status mcp_host_step_run(mcp_host_step* step, int32_t num_seqs, const int32_t* cu_seqlens_q,
                             const int32_t* seqlens_k, const int32_t* block_tables,
                             const void* q, const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, void* out, float* lse, int64_t* ticket);

/*
 * Block until step `ticket` has finished (its outputs are in host memory) and
 * return its device-side check: MCP_ERR_TIMEOUT or MCP_ERR_DEVICE_CHECK as in
 * mcp_check_device_errors().  A step whose slot was already reused has been
 * checked by then: MCP_OK.
 */
mcp_status mcp_host_step_wait(mcp_host_step* step, int64_t ticket);

/* Wait for every step in flight, then free the object (NULL is ignored). */
mcp_status mcp_host_step_destroy(mcp_host_step* step);

/* ------------------------------------------------------------------------- */
/* Non-paged varlen forward                                                   */
/* ------------------------------------------------------------------------- */
/*
 * [W] "Flash Attention 的 varlen 接口": the same right-aligned causal attention
 * over packed, non-paged K and V -- k, v [total_k, H_kv, D] bf16 (device), the
 * keys of segment s being rows cu_seqlens_k[s] .. cu_seqlens_k[s+1]-1
 * (cu_seqlens_k [S+1] int32, device, non-decreasing, cu_seqlens_k[0] = 0,
 * cu_seqlens_k[S] = total_k <= 2^30).  Plan with mcp_mixed_attn_plan (or
 * _plan_rows) from HOST cu_seqlens_q and seqlens_k = diff(cu_seqlens_k), with
 * page_size 16, max_pages_per_seq >= ceil(max seqlens_k / 16) and any
 * num_pages >= 1 (no page pool is read).  q, out, lse, workspace as in
 * mcp_mixed_attn_fwd; there is no append (the keys are given).
 */
mcp_status mcp_mixed_attn_fwd_varlen(const mcp_plan* plan, const void* q, const void* k,
                                     const void* v, const int32_t* cu_seqlens_q,
                                     const int32_t* cu_seqlens_k, int64_t total_k, void* out,
                                     float* lse, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* Device-check bits written to an error word. */
#define MCP_DEVERR_TIMEOUT 0x1      /* a bounded mbarrier wait gave up           */
#define MCP_DEVERR_PAGE_RANGE 0x2   /* a block-table page id outside the pool    */
#define MCP_DEVERR_SLOT_RANGE 0x4   /* an append slot outside the pool           */
#define MCP_DEVERR_ROW_RANGE 0x8    /* a gathered row index outside the source   */
#define MCP_DEVERR_ITEM_KIND 0x10   /* a work item this head_dim has no path for */
#define MCP_DEVERR_SLOT_DUP 0x20    /* two append tokens share a slot (MCP_CHECKED) */

#ifdef __cplusplus
}
#endif

#endif /* MCP_H_ */
