// mcp_mixed_attn_fwd_noalloc: the mixed attention forward with its scratch in
// a fixed, library-owned device array instead of a caller-provided workspace.
//
// Who needs this: callers that cannot allocate device memory at the point where
// they run a step -- for example code running under a framework whose memory
// pool owns all device allocations and forbids stray cudaMalloc calls, or a
// runtime that must not grow its device footprint after start-up.  They can
// hand over inputs and outputs, but not scratch.  This entry point needs no
// workspace: the work lists, split partials and the error word live in
// `g_scratch` below.
//
// Costs and limits of that choice:
//  * every GPU that loads the library holds kScratchBytes (16 MiB) of device
//    memory for g_scratch until the process exits;
//  * a step whose plan needs more scratch than that is rejected with
//    MCP_ERR_WORKSPACE_TOO_SMALL (use mcp_mixed_attn_fwd with a workspace);
//  * all calls share the one array, so two calls whose GPU work overlaps (on
//    different streams, or from different threads) race; calls must be
//    ordered, e.g. on one stream;
//  * the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress); make that first call before any stream capture.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "mcp.h"
#include "mcp_internal.h"

namespace {

constexpr size_t kScratchBytes = 16u << 20;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code `g_scratch` names a host-side stand-in, not
// the device memory: only the address from cudaGetSymbolAddress may be given
// to kernels.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

thread_local std::vector<unsigned char> g_lists;

mcp_status fail_with(mcp_status status, const char* msg) {
  return static_cast<mcp_status>(mcp::set_error_code(status, msg));
}

}  // namespace

extern "C" mcp_status mcp_mixed_attn_fwd_noalloc(
    const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q, const int32_t* h_seqlens_k,
    const mcp_plan_options* opts, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* cu_seqlens_q, const int32_t* seqlens_k,
    void* out, float* lse, int32_t** error_word, void* stream) {
  try {
    // Plan once, into host memory (the plan and its work lists together).
    mcp_plan plan;
    mcp_status st = mcp::plan_to_host(desc, h_cu_seqlens_q, h_seqlens_k, opts, &plan, g_lists);
    if (st != MCP_OK) return st;
    if (plan.workspace_bytes > static_cast<int64_t>(kScratchBytes)) {
      char msg[200];
      snprintf(msg, sizeof(msg),
               "step needs %lld bytes of scratch; the fixed scratch holds %zu "
               "(use mcp_mixed_attn_fwd with a workspace)",
               static_cast<long long>(plan.workspace_bytes), kScratchBytes);
      return fail_with(MCP_ERR_WORKSPACE_TOO_SMALL, msg);
    }
    // Every argument error is found here, before the shared scratch is touched
    // or anything is enqueued.
    st = mcp::check_fwd_args(&plan, q, k_cache, v_cache, block_tables, cu_seqlens_q, seqlens_k,
                             out, lse);
    if (st != MCP_OK) return st;
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
      char msg[200];
      snprintf(msg, sizeof(msg), "scratch address lookup: %s", cudaGetErrorString(e));
      return fail_with(MCP_ERR_CUDA, msg);
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (plan.off_part_o > 0)
      e = cudaMemcpyAsync(scratch, g_lists.data(), static_cast<size_t>(plan.off_part_o),
                          cudaMemcpyHostToDevice, cs);
    // the error word must start at zero; nothing else in the scratch is read
    // before this call's kernels write it
    if (e == cudaSuccess)
      e = cudaMemsetAsync(static_cast<char*>(scratch) + plan.off_error, 0, 256, cs);
    if (e != cudaSuccess) {
      char msg[200];
      snprintf(msg, sizeof(msg), "scratch upload: %s", cudaGetErrorString(e));
      return fail_with(MCP_ERR_CUDA, msg);
    }
    if (error_word)
      *error_word = reinterpret_cast<int32_t*>(static_cast<char*>(scratch) + plan.off_error);
    return mcp_mixed_attn_fwd(&plan, q, k_cache, v_cache, block_tables, cu_seqlens_q, seqlens_k,
                              out, lse, scratch, kScratchBytes, stream);
  } catch (const std::bad_alloc&) {
    return fail_with(MCP_ERR_INVALID_ARG, "host allocation failed while planning");
  } catch (...) {
    return fail_with(MCP_ERR_INVALID_ARG, "unexpected host error");
  }
}
