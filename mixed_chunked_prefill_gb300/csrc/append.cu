// Row and page copies around the step: the paged KV append (scatter each new
// token's K/V row into its physical slot), the row gather of the sampled
// positions, and whole-page copies between page pools (swap-out / swap-in).
//
// [W] "输入组装": the new tokens' K/V are written into the paged cache through
// slot_mapping before attention runs; [L] 4.2 (append_paged_kv_cache):
// physical-address translation and scattered (non-contiguous) writes.
// Slots are distinct within one call, so plain stores suffice.
//
// HBM-bound copy: each token row is H_kv * D * 2 bytes, moved as 16-byte
// vectors; consecutive threads take consecutive vectors of a row, so both the
// read of k_new / v_new and the write into the page are coalesced.
#include <cuda_runtime.h>
#include <stdint.h>

#include "mcp.h"
#include "mcp_internal.h"

namespace mcp {
namespace {

__global__ void __launch_bounds__(256) paged_kv_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slots, int64_t total_vec, int32_t vec_per_tok, int64_t num_slots,
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int32_t* err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_vec;
       i += stride) {
    const int64_t t = i / vec_per_tok;
    const int64_t c = i - t * vec_per_tok;
    const int64_t slot = slots[t];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (err && c == 0) atomicOr(err, MCP_DEVERR_SLOT_RANGE);
      continue;
    }
    const int64_t dst = slot * vec_per_tok + c;
    k_cache[dst] = k_new[i];
    v_cache[dst] = v_new[i];
  }
}

// dst[i] = src[rows[i]] ([W] "采样：只有该出字的请求才出字": the output rows at
// logits_indices), 16-byte vectors, consecutive threads on consecutive vectors
// of a row.  An index outside the source is reported and its row zeroed.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src,
                                                          int32_t num_src_rows,
                                                          const int32_t* __restrict__ rows,
                                                          int64_t total_vec, int32_t vec_per_row,
                                                          uint4* __restrict__ dst, int32_t* err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_vec;
       i += stride) {
    const int64_t r = i / vec_per_row;
    const int64_t c = i - r * vec_per_row;
    const int32_t from = rows[r];
    if (from < 0 || from >= num_src_rows) {
      if (err && c == 0) atomicOr(err, MCP_DEVERR_ROW_RANGE);
      dst[i] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    dst[i] = src[static_cast<int64_t>(from) * vec_per_row + c];
  }
}

// Whole-page copies between two page pools: dst[dst_pages[i]] = src[src_pages[i]]
// for K and V.  Either pool may be page-locked host memory (swap-out / swap-in
// of a preempted sequence's pages) or device memory (copy-on-write).  A page
// id outside its pool is reported and that page skipped.
__global__ void __launch_bounds__(256) copy_pages_kernel(
    const uint4* __restrict__ k_src, const uint4* __restrict__ v_src, int32_t src_pages_total,
    uint4* __restrict__ k_dst, uint4* __restrict__ v_dst, int32_t dst_pages_total,
    const int32_t* __restrict__ src_pages, const int32_t* __restrict__ dst_pages,
    int64_t total_vec, int32_t vec_per_page, int32_t* err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_vec;
       i += stride) {
    const int64_t p = i / vec_per_page;
    const int64_t c = i - p * vec_per_page;
    const int32_t sp = src_pages[p], dp = dst_pages[p];
    if (sp < 0 || sp >= src_pages_total || dp < 0 || dp >= dst_pages_total) {
      if (err && c == 0) atomicOr(err, MCP_DEVERR_PAGE_RANGE);
      continue;
    }
    const int64_t from = static_cast<int64_t>(sp) * vec_per_page + c;
    const int64_t to = static_cast<int64_t>(dp) * vec_per_page + c;
    k_dst[to] = k_src[from];
    v_dst[to] = v_src[from];
  }
}

#ifdef MCP_CHECKED
// Checked builds only: flag two tokens of one append that share a slot.  Each
// block stages a 1024-slot window of the mapping in shared memory and every
// token of the grid-stride loop compares its slot with the window's later
// tokens; the blocks cover all windows.  O(T^2) compares: a debugging aid.
__global__ void __launch_bounds__(256) slot_dup_check_kernel(const int64_t* __restrict__ slots,
                                                             int32_t num_tokens, int32_t* err) {
  constexpr int kWin = 1024;
  __shared__ int64_t win[kWin];
  const int32_t nwin = (num_tokens + kWin - 1) / kWin;
  for (int32_t wi = blockIdx.x; wi < nwin; wi += gridDim.x) {
    const int32_t w0 = wi * kWin;
    const int32_t wn = num_tokens - w0 < kWin ? num_tokens - w0 : kWin;
    __syncthreads();
    for (int32_t i = threadIdx.x; i < wn; i += blockDim.x) win[i] = slots[w0 + i];
    __syncthreads();
    // tokens t < w0 + wn against window tokens u > t
    const int32_t tend = w0 + wn;
    for (int32_t t = threadIdx.x; t < tend; t += blockDim.x) {
      const int64_t s = slots[t];
      if (s < 0) continue;
      const int32_t u0 = t + 1 > w0 ? t + 1 - w0 : 0;
      for (int32_t u = u0; u < wn; ++u)
        if (win[u] == s) {
          if (err) atomicOr(err, MCP_DEVERR_SLOT_DUP);
          break;
        }
    }
  }
}
#endif

int grid_for(int64_t total) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(blocks > cap ? cap : blocks);
}

}  // namespace

int launch_gather_rows(const void* src, int32_t num_src_rows, int32_t row_bytes,
                       const int32_t* rows, int32_t num_rows, void* dst, int32_t* error_word,
                       void* stream) {
  if (num_rows <= 0) return 0;
  const int32_t vec = row_bytes / 16;
  const int64_t total = static_cast<int64_t>(num_rows) * vec;
  gather_rows_kernel<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), num_src_rows, rows, total, vec, static_cast<uint4*>(dst),
      error_word);
  return static_cast<int>(cudaGetLastError());
}

int launch_copy_pages(const void* k_src, const void* v_src, int32_t src_num_pages, void* k_dst,
                      void* v_dst, int32_t dst_num_pages, int32_t page_bytes,
                      const int32_t* src_pages, const int32_t* dst_pages, int32_t num,
                      int32_t* error_word, void* stream) {
  if (num <= 0) return 0;
  const int32_t vec = page_bytes / 16;
  const int64_t total = static_cast<int64_t>(num) * vec;
  copy_pages_kernel<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_src), static_cast<const uint4*>(v_src), src_num_pages,
      static_cast<uint4*>(k_dst), static_cast<uint4*>(v_dst), dst_num_pages, src_pages, dst_pages,
      total, vec, error_word);
  return static_cast<int>(cudaGetLastError());
}

int launch_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                  int32_t num_tokens, int32_t row_bytes, int64_t num_slots, void* k_cache,
                  void* v_cache, int32_t* error_word, void* stream) {
  if (num_tokens <= 0) return 0;
  const int32_t vec_per_tok = row_bytes / 16;
  const int64_t total = static_cast<int64_t>(num_tokens) * vec_per_tok;
  paged_kv_append_kernel<<<grid_for(total), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, total,
      vec_per_tok, num_slots, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      error_word);
#ifdef MCP_CHECKED
  if (num_tokens > 1) {
    const int32_t nwin = (num_tokens + 1023) / 1024;
    slot_dup_check_kernel<<<nwin, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        slot_mapping, num_tokens, error_word);
  }
#endif
  return static_cast<int>(cudaGetLastError());
}

}  // namespace mcp
