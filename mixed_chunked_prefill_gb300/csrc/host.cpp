// Host side of the C ABI: argument validation, the slot-mapping builder, the
// per-step work planner, workspace layout and kernel launches.
//
// The planner turns one step's metadata into the fused kernel's work list.
// [W] "Flash Attention 的 varlen 接口": segments are independent (the i-th
// query segment sees only the i-th KV segment), and "prefill and decode are
// just segments of different lengths" -- so the planner only decides how to
// cut each segment into units that keep all SMs busy: decode segments by KV
// range (split-KV), chunks by 128-row query tile and KV range.  Items are
// ordered longest-first (list scheduling over the SMs by the hardware block
// dispatcher approximates LPT) with decode and tensor-core work interleaved in
// proportion to their estimated cost, so HBM streaming and tensor-core tiles
// run side by side.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "mcp.h"
#include "mcp_internal.h"

namespace {

thread_local char g_err[512] = "";

mcp_status fail(mcp_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

mcp_status okay() {
  g_err[0] = 0;
  return MCP_OK;
}

mcp_status cuda_fail(int e, const char* what) {
  const char* detail = mcp::launch_detail();
  if (e == -1 && detail && detail[0]) return fail(MCP_ERR_CUDA, "%s: %s", what, detail);
  return fail(MCP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(static_cast<cudaError_t>(e)));
}

constexpr int32_t kPlanMagic = 0x4D435031;  // "MCP1"

int64_t align256(int64_t x) { return (x + 255) & ~static_cast<int64_t>(255); }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

mcp_status validate_desc(const mcp_attn_desc* d) {
  if (!d) return fail(MCP_ERR_INVALID_ARG, "desc is NULL");
  if (d->num_seqs < 0) return fail(MCP_ERR_INVALID_ARG, "num_seqs %d < 0", d->num_seqs);
  if (d->total_q < 0) return fail(MCP_ERR_INVALID_ARG, "total_q %d < 0", d->total_q);
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0)
    return fail(MCP_ERR_INVALID_ARG, "head counts must be positive (%d, %d)", d->num_q_heads,
                d->num_kv_heads);
  if (d->num_q_heads % d->num_kv_heads != 0)
    return fail(MCP_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                d->num_q_heads, d->num_kv_heads);
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(MCP_ERR_UNSUPPORTED, "head_dim %d (built: 64, 128)", d->head_dim);
  if (d->page_size != mcp::kPageSize)
    return fail(MCP_ERR_UNSUPPORTED, "page_size %d (built: 16)", d->page_size);
  if (d->num_q_heads / d->num_kv_heads > mcp::kTileRows)
    return fail(MCP_ERR_UNSUPPORTED, "group size %d > 128", d->num_q_heads / d->num_kv_heads);
  if (d->num_kv_heads > 32767)
    return fail(MCP_ERR_UNSUPPORTED, "num_kv_heads %d > 32767", d->num_kv_heads);
  if (d->num_pages <= 0) return fail(MCP_ERR_INVALID_ARG, "num_pages %d <= 0", d->num_pages);
  if (d->num_seqs > 0 && d->max_pages_per_seq <= 0)
    return fail(MCP_ERR_INVALID_ARG, "max_pages_per_seq %d <= 0", d->max_pages_per_seq);
  if (!std::isfinite(d->sm_scale) || d->sm_scale <= 0.f)
    return fail(MCP_ERR_INVALID_ARG, "sm_scale must be finite and > 0");
  return MCP_OK;
}

// Shared metadata checks ([W] "记录 KV Cache 的长度": Lk counts this step's
// tokens, so Lq <= Lk; cu_seqlens_q is an exclusive prefix sum).
mcp_status validate_meta(int32_t S, int32_t total_q, int32_t page_size, int32_t max_pages,
                         const int32_t* cu, const int32_t* sk) {
  if (!cu) return fail(MCP_ERR_INVALID_ARG, "cu_seqlens_q is NULL");
  if (S > 0 && !sk) return fail(MCP_ERR_INVALID_ARG, "seqlens_k is NULL");
  if (cu[0] != 0) return fail(MCP_ERR_INVALID_ARG, "cu_seqlens_q[0] = %d, expected 0", cu[0]);
  for (int32_t s = 0; s < S; ++s) {
    const int64_t lq = static_cast<int64_t>(cu[s + 1]) - cu[s];
    if (lq < 0) return fail(MCP_ERR_INVALID_ARG, "cu_seqlens_q decreases at segment %d", s);
    if (sk[s] < 0) return fail(MCP_ERR_INVALID_ARG, "seqlens_k[%d] = %d < 0", s, sk[s]);
    if (lq > sk[s])
      return fail(MCP_ERR_INVALID_ARG,
                  "segment %d has %lld query tokens but KV length %d (KV length must include "
                  "this step's tokens)",
                  s, static_cast<long long>(lq), sk[s]);
    if (cdiv(sk[s], page_size) > max_pages)
      return fail(MCP_ERR_INVALID_ARG, "segment %d needs %lld pages > max_pages_per_seq %d", s,
                  static_cast<long long>(cdiv(sk[s], page_size)), max_pages);
  }
  if (total_q >= 0 && cu[S] != total_q)
    return fail(MCP_ERR_INVALID_ARG, "cu_seqlens_q[S] = %d but total_q = %d", cu[S], total_q);
  return MCP_OK;
}

struct Built {
  std::vector<mcp::WorkItem> items;
  std::vector<mcp::CombineEntry> comb;
  int64_t part_rows = 0;
  int n_dec = 0, n_pre = 0;
  int dsplit = 0, psplit = 0;
};

// Even split of [0, len) into pieces of at most `cap`, each a multiple of `gran`.
void even_split(int64_t len, int64_t cap, int64_t gran, int64_t* n, int64_t* size) {
  int64_t k = std::max<int64_t>(1, cdiv(len, cap));
  int64_t sz = round_up(cdiv(len, k), gran);
  *size = sz;
  *n = cdiv(len, sz);
}

void build(const mcp_attn_desc& d, const int32_t* cu, const int32_t* sk, int num_sms,
           const mcp_plan_options* o, Built& b) {
  const int G = d.num_q_heads / d.num_kv_heads;
  const int TQ = mcp::kTileRows / G;
  const int H = d.num_kv_heads;
  const int HG = mcp::decode_head_group(H);
  const int dopt = o ? o->decode_split_tokens : 0;
  const int popt = o ? o->prefill_split_tokens : 0;

  auto count = [&](int64_t ds, int64_t ps) {
    int64_t n = 0;
    for (int s = 0; s < d.num_seqs; ++s) {
      const int64_t lq = cu[s + 1] - cu[s], lk = sk[s];
      if (lq == 0) continue;
      if (lq * G <= mcp::kDecodeMaxRows) {
        int64_t k, z;
        even_split(lk, ds, mcp::kPageSize, &k, &z);
        n += k * (H / HG);
      } else {
        for (int64_t qb = 0; qb < lq; qb += TQ) {
          const int64_t vis = lk - lq + std::min<int64_t>(lq, qb + TQ);
          int64_t k, z;
          even_split(vis, ps, mcp::kKvTile, &k, &z);
          n += k * H;
        }
      }
    }
    return n;
  };

  // Decode splits: about eight decode items per SM (each item streams its KV
  // range for a whole kv-head group), never below 1024 tokens.
  int64_t ds;
  if (dopt > 0) {
    ds = round_up(dopt, mcp::kPageSize);
  } else {
    int64_t dec_tokens = 0;
    for (int s = 0; s < d.num_seqs; ++s) {
      const int64_t lq = cu[s + 1] - cu[s];
      if (lq > 0 && lq * G <= mcp::kDecodeMaxRows) dec_tokens += sk[s] * (H / HG);
    }
    ds = std::max<int64_t>(1024, round_up(cdiv(dec_tokens, 8LL * num_sms), mcp::kPageSize));
  }
  int64_t ps = popt > 0 ? round_up(popt, mcp::kKvTile) : 32768;
  while (count(ds, ps) < 2LL * num_sms) {
    bool changed = false;
    if (dopt <= 0 && ds > 1024) { ds = std::max<int64_t>(1024, ds / 2); changed = true; }
    if (popt <= 0 && ps > 2048) { ps /= 2; changed = true; }
    if (!changed) break;
  }
  b.dsplit = static_cast<int>(ds);
  b.psplit = static_cast<int>(ps);

  // Rough per-SM cost model (ns) used only for ordering: a decode key streams
  // 4*D bytes of K/V per kv head at ~45 GB/s per SM; a tensor-core key-tile
  // does 4*128*D flops at ~6 TFLOP/s per SM.
  struct Entry {
    mcp::WorkItem it;
    double cost;
    int64_t group;
  };
  std::vector<Entry> dec, pre;
  for (int s = 0; s < d.num_seqs; ++s) {
    const int64_t lq = cu[s + 1] - cu[s], lk = sk[s], hist = lk - lq;
    if (lq == 0) continue;
    if (lq * G <= mcp::kDecodeMaxRows) {
      int64_t n, sz;
      even_split(lk, ds, mcp::kPageSize, &n, &sz);
      const int rows = static_cast<int>(lq * G);
      for (int h0 = 0; h0 < H; h0 += HG) {
        int64_t base = -1;
        if (n > 1) {
          // head j of the group, split k: partial rows base + j*n*rows + k*rows
          base = b.part_rows;
          b.part_rows += n * rows * HG;
          for (int j = 0; j < HG; ++j)
            b.comb.push_back({s, h0 + j, 0, static_cast<int32_t>(lq), static_cast<int32_t>(n),
                              static_cast<int32_t>(base + j * n * rows), rows, 0});
        }
        for (int64_t k = 0; k < n; ++k) {
          mcp::WorkItem it;
          it.seg = s;
          it.kv_head = static_cast<int16_t>(h0);
          it.kind = mcp::kDecodeItem;
          it.num_heads = static_cast<int8_t>(HG);
          it.q_begin = 0;
          it.q_count = static_cast<int32_t>(lq);
          it.kv_begin = static_cast<int32_t>(k * sz);
          it.kv_end = static_cast<int32_t>(std::min(lk, (k + 1) * sz));
          it.part_row = static_cast<int32_t>(n > 1 ? base + k * rows : -1);
          it.part_head_stride = static_cast<int32_t>(n * rows);
          dec.push_back({it, (it.kv_end - it.kv_begin) * 4.0 * d.head_dim * HG / 45.0, 0});
        }
      }
    } else {
      for (int64_t qb = 0; qb < lq; qb += TQ) {
        const int64_t qc = std::min<int64_t>(TQ, lq - qb);
        const int64_t vis = hist + qb + qc;
        int64_t n, sz;
        even_split(vis, ps, mcp::kKvTile, &n, &sz);
        const int rows = static_cast<int>(qc * G);
        for (int h = 0; h < H; ++h) {
          int64_t base = -1;
          if (n > 1) {
            base = b.part_rows;
            b.part_rows += n * rows;
            b.comb.push_back({s, h, static_cast<int32_t>(qb), static_cast<int32_t>(qc),
                              static_cast<int32_t>(n), static_cast<int32_t>(base), rows, 0});
          }
          for (int64_t k = 0; k < n; ++k) {
            mcp::WorkItem it;
            it.seg = s;
            it.kv_head = static_cast<int16_t>(h);
            it.kind = mcp::kPrefillItem;
            it.num_heads = 1;
            it.q_begin = static_cast<int32_t>(qb);
            it.q_count = static_cast<int32_t>(qc);
            it.kv_begin = static_cast<int32_t>(k * sz);
            it.kv_end = static_cast<int32_t>(std::min(vis, (k + 1) * sz));
            it.part_row = static_cast<int32_t>(n > 1 ? base + k * rows : -1);
            it.part_head_stride = 0;
            const double tiles = static_cast<double>(cdiv(it.kv_end - it.kv_begin, mcp::kKvTile));
            // tiles reading the same K/V (same segment, kv head, split) share a group
            const int64_t gid = (static_cast<int64_t>(s) * H + h) * 4096 + k;
            pre.push_back({it, 300.0 + tiles * 4.0 * 128 * 128 * d.head_dim / 6000.0, gid});
          }
        }
      }
    }
  }
  b.n_dec = static_cast<int>(dec.size());
  b.n_pre = static_cast<int>(pre.size());

  std::stable_sort(dec.begin(), dec.end(),
                   [](const Entry& a, const Entry& c) { return a.cost > c.cost; });
  // prefill: groups by descending total cost, tiles of a group kept together
  {
    std::vector<std::pair<int64_t, double>> gc;
    std::stable_sort(pre.begin(), pre.end(),
                     [](const Entry& a, const Entry& c) { return a.group < c.group; });
    for (size_t i = 0; i < pre.size(); ++i) {
      if (gc.empty() || gc.back().first != pre[i].group) gc.push_back({pre[i].group, 0.0});
      gc.back().second += pre[i].cost;
    }
    std::vector<int64_t> rank_of;
    std::vector<size_t> order(gc.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](size_t a, size_t c) { return gc[a].second > gc[c].second; });
    std::vector<Entry> sorted;
    sorted.reserve(pre.size());
    std::vector<size_t> start(gc.size() + 1, 0);
    {
      size_t gi = 0;
      for (size_t i = 0; i < pre.size(); ++i) {
        if (i > 0 && pre[i].group != pre[i - 1].group) ++gi;
        start[gi + 1] = i + 1;
      }
    }
    for (size_t oi : order) {
      const size_t a = start[oi], e = start[oi + 1];
      std::vector<Entry> grp(pre.begin() + a, pre.begin() + e);
      std::stable_sort(grp.begin(), grp.end(),
                       [](const Entry& x, const Entry& y) { return x.cost > y.cost; });
      sorted.insert(sorted.end(), grp.begin(), grp.end());
    }
    pre.swap(sorted);
  }
  // interleave the two lists in proportion to their total cost
  double td = 0, tp = 0;
  for (auto& e : dec) td += e.cost;
  for (auto& e : pre) tp += e.cost;
  b.items.reserve(dec.size() + pre.size());
  size_t i = 0, j = 0;
  double ad = 0, ap = 0;
  while (i < dec.size() || j < pre.size()) {
    const bool take_dec =
        j >= pre.size() || (i < dec.size() && (ad / std::max(td, 1e-9)) <= (ap / std::max(tp, 1e-9)));
    if (take_dec) {
      ad += dec[i].cost;
      b.items.push_back(dec[i++].it);
    } else {
      ap += pre[j].cost;
      b.items.push_back(pre[j++].it);
    }
  }
}

thread_local std::vector<unsigned char> g_staging;

}  // namespace

namespace mcp {
int32_t set_error_code(int32_t status, const char* msg) {
  snprintf(g_err, sizeof(g_err), "%s", msg ? msg : "");
  return status;
}
}  // namespace mcp

extern "C" {

const char* mcp_status_string(int32_t s) {
  switch (s) {
    case MCP_OK: return "MCP_OK";
    case MCP_ERR_INVALID_ARG: return "MCP_ERR_INVALID_ARG";
    case MCP_ERR_UNSUPPORTED: return "MCP_ERR_UNSUPPORTED";
    case MCP_ERR_WORKSPACE_TOO_SMALL: return "MCP_ERR_WORKSPACE_TOO_SMALL";
    case MCP_ERR_CUDA: return "MCP_ERR_CUDA";
    case MCP_ERR_TIMEOUT: return "MCP_ERR_TIMEOUT";
    case MCP_ERR_DEVICE_CHECK: return "MCP_ERR_DEVICE_CHECK";
    default: return "MCP_ERR_UNKNOWN";
  }
}

const char* mcp_last_error(void) { return g_err; }

int32_t mcp_abi_version(void) { return MCP_ABI_VERSION; }

mcp_status mcp_paged_kv_append(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                               int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                               int32_t page_size, int32_t num_pages, void* k_cache, void* v_cache,
                               int32_t* error_word, void* stream) {
  if (num_tokens < 0) return fail(MCP_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_pages <= 0)
    return fail(MCP_ERR_INVALID_ARG, "sizes must be positive (heads %d, dim %d, page %d, pages %d)",
                num_kv_heads, head_dim, page_size, num_pages);
  if ((static_cast<int64_t>(num_kv_heads) * head_dim) % 8 != 0)
    return fail(MCP_ERR_INVALID_ARG, "num_kv_heads * head_dim = %lld is not a multiple of 8",
                static_cast<long long>(num_kv_heads) * head_dim);
  if (num_tokens == 0) return okay();
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache)
    return fail(MCP_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(MCP_ERR_INVALID_ARG, "tensor not 16-byte aligned");
  const int32_t row_bytes = num_kv_heads * head_dim * 2;
  const int e = mcp::launch_append(k_new, v_new, slot_mapping, num_tokens, row_bytes,
                                   static_cast<int64_t>(num_pages) * page_size, k_cache, v_cache,
                                   error_word, stream);
  if (e != 0) return cuda_fail(e, "paged_kv_append launch");
  return okay();
}

mcp_status mcp_build_slot_mapping(const int32_t* block_tables, int32_t num_seqs,
                                  int32_t max_pages_per_seq, int32_t page_size, int32_t num_pages,
                                  const int32_t* cu_seqlens_q, const int32_t* seqlens_k,
                                  int64_t* slot_mapping) {
  if (num_seqs < 0) return fail(MCP_ERR_INVALID_ARG, "num_seqs %d < 0", num_seqs);
  if (page_size <= 0 || num_pages <= 0)
    return fail(MCP_ERR_INVALID_ARG, "page_size %d / num_pages %d must be positive", page_size,
                num_pages);
  if (num_seqs > 0 && (max_pages_per_seq <= 0 || !block_tables))
    return fail(MCP_ERR_INVALID_ARG, "block_tables missing or max_pages_per_seq <= 0");
  mcp_status st = validate_meta(num_seqs, -1, page_size, max_pages_per_seq, cu_seqlens_q, seqlens_k);
  if (st != MCP_OK) return st;
  if (cu_seqlens_q[num_seqs] > 0 && !slot_mapping)
    return fail(MCP_ERR_INVALID_ARG, "slot_mapping is NULL");
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
    const int32_t hist = seqlens_k[s] - lq;
    for (int32_t t = cu_seqlens_q[s]; t < cu_seqlens_q[s + 1]; ++t) {
      const int64_t pos = hist + (t - cu_seqlens_q[s]);
      const int32_t page = block_tables[static_cast<int64_t>(s) * max_pages_per_seq + pos / page_size];
      if (page < 0 || page >= num_pages)
        return fail(MCP_ERR_INVALID_ARG, "block_tables[%d][%lld] = %d outside [0, %d)", s,
                    static_cast<long long>(pos / page_size), page, num_pages);
      slot_mapping[t] = static_cast<int64_t>(page) * page_size + pos % page_size;
    }
  }
  return okay();
}

}  // extern "C"

namespace {

// Validate, build the work lists and fill *plan (no device access unless the
// SM count has to be queried).
mcp_status plan_common(const mcp_attn_desc* desc, const int32_t* cu, const int32_t* sk,
                       const mcp_plan_options* opts, mcp_plan* plan, Built& b) {
  mcp_status st = validate_desc(desc);
  if (st != MCP_OK) return st;
  if (!plan) return fail(MCP_ERR_INVALID_ARG, "plan is NULL");
  if (opts) {
    for (int i = 0; i < 5; ++i)
      if (opts->reserved[i] != 0) return fail(MCP_ERR_INVALID_ARG, "opts->reserved must be 0");
    if (opts->num_sms < 0 || opts->decode_split_tokens < 0 || opts->prefill_split_tokens < 0)
      return fail(MCP_ERR_INVALID_ARG, "negative plan option");
  }
  st = validate_meta(desc->num_seqs, desc->total_q, desc->page_size, desc->max_pages_per_seq, cu, sk);
  if (st != MCP_OK) return st;
  int num_sms = opts ? opts->num_sms : 0;
  if (num_sms <= 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "SM count query: %s", cudaGetErrorString(e));
  }
  build(*desc, cu, sk, num_sms, opts, b);
  if (b.part_rows > INT32_MAX || static_cast<int64_t>(b.items.size()) > INT32_MAX)
    return fail(MCP_ERR_UNSUPPORTED, "step too large for one plan");
  mcp_plan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.magic = kPlanMagic;
  pl.num_items = static_cast<int32_t>(b.items.size());
  pl.num_decode_items = b.n_dec;
  pl.num_prefill_items = b.n_pre;
  pl.num_combine = static_cast<int32_t>(b.comb.size());
  int64_t crow = 0;
  for (mcp::CombineEntry& e : b.comb) {
    e.row_base = static_cast<int32_t>(crow);
    crow += e.rows;
  }
  pl.combine_rows = static_cast<int32_t>(crow);
  pl.decode_split_tokens = b.dsplit;
  pl.prefill_split_tokens = b.psplit;
  pl.num_sms = num_sms;
  pl.partial_rows = b.part_rows;
  pl.off_items = 0;
  pl.off_combine = align256(static_cast<int64_t>(b.items.size()) * sizeof(mcp::WorkItem));
  pl.off_part_o =
      align256(pl.off_combine + static_cast<int64_t>(b.comb.size()) * sizeof(mcp::CombineEntry));
  pl.off_part_lse = align256(pl.off_part_o + b.part_rows * desc->head_dim * 4);
  pl.off_error = align256(pl.off_part_lse + b.part_rows * 4);
  pl.workspace_bytes = pl.off_error + 256;
  pl.desc = *desc;
  *plan = pl;
  return MCP_OK;
}

void write_lists(const mcp_plan& pl, const Built& b, unsigned char* dst) {
  std::memset(dst, 0, static_cast<size_t>(pl.off_part_o));
  if (!b.items.empty()) std::memcpy(dst, b.items.data(), b.items.size() * sizeof(mcp::WorkItem));
  if (!b.comb.empty())
    std::memcpy(dst + pl.off_combine, b.comb.data(), b.comb.size() * sizeof(mcp::CombineEntry));
}

}  // namespace

extern "C" {

mcp_status mcp_mixed_attn_plan(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                               const int32_t* h_seqlens_k, const mcp_plan_options* opts,
                               mcp_plan* plan, void* workspace, size_t workspace_bytes,
                               void* stream) {
  try {
    Built b;
    mcp_status st = plan_common(desc, h_cu_seqlens_q, h_seqlens_k, opts, plan, b);
    if (st != MCP_OK) return st;
    const mcp_plan& pl = *plan;
    if (!workspace) return okay();
    if (!aligned(workspace, 256)) return fail(MCP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    if (static_cast<int64_t>(workspace_bytes) < pl.workspace_bytes)
      return fail(MCP_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %lld needed", workspace_bytes,
                  static_cast<long long>(pl.workspace_bytes));
    const size_t nbytes = static_cast<size_t>(pl.off_part_o);
    g_staging.resize(nbytes);
    write_lists(pl, b, g_staging.data());
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (nbytes > 0)
      e = cudaMemcpyAsync(workspace, g_staging.data(), nbytes, cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(static_cast<char*>(workspace) + pl.off_error, 0, 256, cs);
    if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "plan upload: %s", cudaGetErrorString(e));
    return okay();
  } catch (const std::bad_alloc&) {
    return fail(MCP_ERR_INVALID_ARG, "host allocation failed while planning");
  } catch (...) {
    return fail(MCP_ERR_INVALID_ARG, "unexpected host error while planning");
  }
}

mcp_status mcp_mixed_attn_plan_host(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                                    const int32_t* h_seqlens_k, const mcp_plan_options* opts,
                                    mcp_plan* plan, void* host_buffer, size_t host_bytes) {
  try {
    Built b;
    mcp_status st = plan_common(desc, h_cu_seqlens_q, h_seqlens_k, opts, plan, b);
    if (st != MCP_OK) return st;
    if (!host_buffer) return okay();
    if (static_cast<int64_t>(host_bytes) < plan->off_part_o)
      return fail(MCP_ERR_WORKSPACE_TOO_SMALL, "host buffer %zu bytes < %lld needed", host_bytes,
                  static_cast<long long>(plan->off_part_o));
    write_lists(*plan, b, static_cast<unsigned char*>(host_buffer));
    return okay();
  } catch (const std::bad_alloc&) {
    return fail(MCP_ERR_INVALID_ARG, "host allocation failed while planning");
  } catch (...) {
    return fail(MCP_ERR_INVALID_ARG, "unexpected host error while planning");
  }
}

mcp_status mcp_mixed_attn_fwd(const mcp_plan* plan, const void* q, const void* k_cache,
                              const void* v_cache, const int32_t* block_tables,
                              const int32_t* cu_seqlens_q, const int32_t* seqlens_k, void* out,
                              float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan || plan->magic != kPlanMagic) return fail(MCP_ERR_INVALID_ARG, "plan not initialised");
  const mcp_attn_desc& d = plan->desc;
  if (plan->num_items == 0) return okay();
  if (!q || !k_cache || !v_cache || !block_tables || !cu_seqlens_q || !seqlens_k || !out || !workspace)
    return fail(MCP_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return fail(MCP_ERR_INVALID_ARG, "q / caches / out must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(MCP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(MCP_ERR_INVALID_ARG, "lse not 4-byte aligned");
  if (static_cast<int64_t>(workspace_bytes) < plan->workspace_bytes)
    return fail(MCP_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %lld needed", workspace_bytes,
                static_cast<long long>(plan->workspace_bytes));
  char* ws = static_cast<char*>(workspace);
  mcp::FwdArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.cu_seqlens_q = cu_seqlens_q;
  a.seqlens_k = seqlens_k;
  a.out = out;
  a.lse = lse;
  a.items = reinterpret_cast<const mcp::WorkItem*>(ws + plan->off_items);
  a.combine = reinterpret_cast<const mcp::CombineEntry*>(ws + plan->off_combine);
  a.part_o = reinterpret_cast<float*>(ws + plan->off_part_o);
  a.part_lse = reinterpret_cast<float*>(ws + plan->off_part_lse);
  a.error_word = reinterpret_cast<int32_t*>(ws + plan->off_error);
  a.num_items = plan->num_items;
  a.num_combine = plan->num_combine;
  a.combine_rows = plan->combine_rows;
  a.total_q = d.total_q;
  a.num_q_heads = d.num_q_heads;
  a.num_kv_heads = d.num_kv_heads;
  a.head_dim = d.head_dim;
  a.page_size = d.page_size;
  a.max_pages_per_seq = d.max_pages_per_seq;
  a.num_pages = d.num_pages;
  a.sm_scale = d.sm_scale;
  int e = mcp::launch_mixed_attn(a, stream);
  if (e != 0) return cuda_fail(e, "mixed_attn_fwd launch");
  e = mcp::launch_combine(a, stream);
  if (e != 0) return cuda_fail(e, "combine launch");
  return okay();
}

mcp_status mcp_check_device_errors(int32_t* error_word, void* stream) {
  if (!error_word) return fail(MCP_ERR_INVALID_ARG, "error_word is NULL");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(cs);
  int32_t v = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&v, error_word, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && v != 0) e = cudaMemset(error_word, 0, sizeof(v));
  if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "device error check: %s", cudaGetErrorString(e));
  if (v & MCP_DEVERR_TIMEOUT)
    return fail(MCP_ERR_TIMEOUT, "a device-side wait gave up (error bits 0x%x)", v);
  if (v != 0) return fail(MCP_ERR_DEVICE_CHECK, "device range check failed (error bits 0x%x)", v);
  return okay();
}

int32_t* mcp_workspace_error_word(const mcp_plan* plan, void* workspace) {
  if (!plan || !workspace || plan->magic != kPlanMagic) return nullptr;
  return reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + plan->off_error);
}

mcp_status mcp_merge_states(const float* o_parts, const float* lse_parts, int32_t n, int32_t rows,
                            int32_t heads, int32_t head_dim, void* out, float* lse_out,
                            void* stream) {
  if (n < 1 || rows < 0 || heads < 1 || head_dim < 1)
    return fail(MCP_ERR_INVALID_ARG, "bad sizes (n %d, rows %d, heads %d, dim %d)", n, rows, heads,
                head_dim);
  if (rows == 0) return okay();
  if (!o_parts || !lse_parts || !out) return fail(MCP_ERR_INVALID_ARG, "NULL pointer argument");
  const int e = mcp::launch_merge_states(o_parts, lse_parts, n, rows, heads, head_dim, out, lse_out,
                                         stream);
  if (e != 0) return cuda_fail(e, "merge_states launch");
  return okay();
}

}  // extern "C"
