// Split-KV combine and the standalone state merge.
//
// When the planner splits a row group's KV range into n parts, each part k
// leaves (O_k normalised by its own sum, LSE_k natural log).  The exact
// unsplit result is, with M = max_k LSE_k and w_k = exp(LSE_k - M),
//   O = sum_k w_k O_k / sum_k w_k,   LSE = M + ln sum_k w_k.
// Parts with LSE = -inf (no visible key) carry weight 0.  Not on the pages:
// this is the identity that makes split-KV equal to unsplit attention.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mcp_internal.h"
#include "ptx.cuh"

namespace mcp {
namespace {

constexpr float kLog2e = 1.44269504088896341f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per merged row.  The rows of all entries are numbered
// consecutively (entry e owns rows [row_base, row_base + rows)), so the grid
// covers exactly the rows that have parts, whatever the mix of short decode
// entries and 128-row chunk tiles.  The plan stores, right after the
// entries, the entry of each block's first row; a warp steps forward from it
// to its own row's entry (a block's 8 rows span at most 8 entries).  Lane k
// holds the LSE of part k (32 parts per pass); lane l accumulates columns
// [l * D/32, (l + 1) * D/32) of O.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineEntry* __restrict__ ents,
                                                      int num_ents, int total_rows,
                                                      const int32_t* __restrict__ cu_q,
                                                      const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse, int hq, int G) {
  constexpr int V = D / 32;
  const int r = blockIdx.x * kCombineRowsPerBlock + (threadIdx.x >> 5);
  if (r >= total_rows) return;
  const int lane = threadIdx.x & 31;
  // the entry holding flat row r: the last one with row_base <= r
  const int32_t* block_ent = reinterpret_cast<const int32_t*>(ents + num_ents);
  int lo = __ldg(&block_ent[blockIdx.x]);
  while (lo + 1 < num_ents && __ldg(&ents[lo + 1].row_base) <= r) ++lo;
  const CombineEntry e = ents[lo];
  const int row = r - e.row_base;
  const int n = e.num_splits;
  const int64_t pr0 = static_cast<int64_t>(e.part_row) + row;  // part k: row pr0 + k * e.rows

  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  float L = 0.f, M = neg_inf();
  if (V == 4 && n <= 8) {
    // few parts (every split chunk tile, most decodes): the LSEs and every
    // part's slice of O are loaded at once, one memory latency for the row
    float4 ov[8];
    const float lk = lane < n ? part_lse[pr0 + static_cast<int64_t>(lane) * e.rows] : neg_inf();
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < n)
        ov[j] = __ldg(reinterpret_cast<const float4*>(
            part_o + (pr0 + static_cast<int64_t>(j) * e.rows) * D + lane * V));
    M = warp_max(lk);
    const float w = (lk == neg_inf()) ? 0.f : ptx::ex2((lk - M) * kLog2e);
    L = w;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < n) {
        const float wj = __shfl_sync(0xffffffffu, w, j);
        acc[0] += wj * ov[j].x;
        acc[1] += wj * ov[j].y;
        acc[2] += wj * ov[j].z;
        acc[3] += wj * ov[j].w;
      }
    }
  } else {
  for (int k = lane; k < n; k += 32) M = fmaxf(M, part_lse[pr0 + static_cast<int64_t>(k) * e.rows]);
  M = warp_max(M);
  for (int k0 = 0; k0 < n; k0 += 32) {
    const int k = k0 + lane;
    const float lk = k < n ? part_lse[pr0 + static_cast<int64_t>(k) * e.rows] : neg_inf();
    const float w = (lk == neg_inf()) ? 0.f : ptx::ex2((lk - M) * kLog2e);
    L += w;
    const int cnt = n - k0 < 32 ? n - k0 : 32;
#pragma unroll 4
    for (int j = 0; j < cnt; ++j) {
      const float wj = __shfl_sync(0xffffffffu, w, j);
      const float* src = part_o + (pr0 + static_cast<int64_t>(k0 + j) * e.rows) * D + lane * V;
      if constexpr (V == 4) {
        const float4 o = __ldg(reinterpret_cast<const float4*>(src));
        acc[0] += wj * o.x;
        acc[1] += wj * o.y;
        acc[2] += wj * o.z;
        acc[3] += wj * o.w;
      } else if constexpr (V == 2) {
        const float2 o = __ldg(reinterpret_cast<const float2*>(src));
        acc[0] += wj * o.x;
        acc[1] += wj * o.y;
      } else {
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] += wj * __ldg(src + v);
      }
    }
  }
  }
  L = warp_sum(L);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int tok = e.q_begin + row / G;
  const int g = row - (row / G) * G;
  const int64_t orow = static_cast<int64_t>(cu_q[e.seg] + tok) * hq + e.kv_head * G + g;
  if constexpr (V == 4) {
    uint2* dst = reinterpret_cast<uint2*>(out + orow * D + lane * V);
    *dst = make_uint2(ptx::pack_bf16x2(acc[0] * inv, acc[1] * inv),
                      ptx::pack_bf16x2(acc[2] * inv, acc[3] * inv));
  } else if constexpr (V == 2) {
    *reinterpret_cast<uint32_t*>(out + orow * D + lane * V) = ptx::pack_bf16x2(acc[0] * inv, acc[1] * inv);
  } else {
#pragma unroll
    for (int v = 0; v < V; ++v) out[orow * D + lane * V + v] = __float2bfloat16_rn(acc[v] * inv);
  }
  if (lse && lane == 0) lse[orow] = L > 0.f ? M + logf(L) : neg_inf();
}

// Standalone merge: one warp per (row, head); o_parts [n, rows, heads, D].
__global__ void __launch_bounds__(128) merge_states_kernel(const float* __restrict__ o_parts,
                                                           const float* __restrict__ lse_parts,
                                                           int n, int rows, int heads, int D,
                                                           __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse_out) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t rh = static_cast<int64_t>(rows) * heads;
  if (idx >= rh) return;
  float M = neg_inf();
  for (int k = 0; k < n; ++k) M = fmaxf(M, lse_parts[k * rh + idx]);
  float L = 0.f;
  for (int k = 0; k < n; ++k) {
    const float lk = lse_parts[k * rh + idx];
    L += (lk == neg_inf()) ? 0.f : ptx::ex2((lk - M) * kLog2e);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  for (int d = lane; d < D; d += 32) {
    float a = 0.f;
    for (int k = 0; k < n; ++k) {
      const float lk = lse_parts[k * rh + idx];
      if (lk == neg_inf()) continue;
      a += ptx::ex2((lk - M) * kLog2e) * o_parts[(k * rh + idx) * D + d];
    }
    out[idx * D + d] = __float2bfloat16_rn(a * inv);
  }
  if (lse_out && lane == 0) lse_out[idx] = L > 0.f ? M + logf(L) : neg_inf();
}

}  // namespace

int launch_combine(const FwdArgs& a, void* stream) {
  if (a.num_combine <= 0 || a.combine_rows <= 0) return 0;
  const int G = a.num_q_heads / a.num_kv_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int blocks = (a.combine_rows + kCombineRowsPerBlock - 1) / kCombineRowsPerBlock;
  if (a.head_dim == 128) {
    combine_kernel<128><<<blocks, 256, 0, st>>>(
        a.combine, a.num_combine, a.combine_rows, a.cu_seqlens_q, a.part_o, a.part_lse,
        static_cast<__nv_bfloat16*>(a.out), a.lse, a.num_q_heads, G);
  } else if (a.head_dim == 256) {
    combine_kernel<256><<<blocks, 256, 0, st>>>(
        a.combine, a.num_combine, a.combine_rows, a.cu_seqlens_q, a.part_o, a.part_lse,
        static_cast<__nv_bfloat16*>(a.out), a.lse, a.num_q_heads, G);
  } else if (a.head_dim == 96) {
    combine_kernel<96><<<blocks, 256, 0, st>>>(
        a.combine, a.num_combine, a.combine_rows, a.cu_seqlens_q, a.part_o, a.part_lse,
        static_cast<__nv_bfloat16*>(a.out), a.lse, a.num_q_heads, G);
  } else {
    combine_kernel<64><<<blocks, 256, 0, st>>>(
        a.combine, a.num_combine, a.combine_rows, a.cu_seqlens_q, a.part_o, a.part_lse,
        static_cast<__nv_bfloat16*>(a.out), a.lse, a.num_q_heads, G);
  }
  return static_cast<int>(cudaGetLastError());
}

int launch_merge_states(const float* o_parts, const float* lse_parts, int32_t n, int32_t rows,
                        int32_t heads, int32_t head_dim, void* out, float* lse_out, void* stream) {
  const int64_t rh = static_cast<int64_t>(rows) * heads;
  if (rh == 0) return 0;
  const int64_t blocks = (rh + 3) / 4;
  merge_states_kernel<<<static_cast<int>(blocks), 128, 0, static_cast<cudaStream_t>(stream)>>>(
      o_parts, lse_parts, n, rows, heads, head_dim, static_cast<__nv_bfloat16*>(out), lse_out);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace mcp
