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
#include <functional>
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
  if (d->head_dim != 64 && d->head_dim != 96 && d->head_dim != 128 && d->head_dim != 256)
    return fail(MCP_ERR_UNSUPPORTED, "head_dim %d (built: 64, 96, 128, 256)", d->head_dim);
  if (d->page_size != 1 && d->page_size != 8 && d->page_size != 16 && d->page_size != 32 &&
      d->page_size != 64)
    return fail(MCP_ERR_UNSUPPORTED, "page_size %d (built: 1, 8, 16, 32, 64)", d->page_size);
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

// A unit of query rows the planner cuts into work items: tokens [qb, qb + qc)
// of segment s, on the decode path (qc * G <= 16 rows) or the tensor-core path.
struct Unit {
  int s;
  int64_t qb, qc;
  bool decode;
};

// Units of a whole step: each decode segment whole, each chunk by 128-row
// tiles.  With `rows` (strictly increasing token indices): only those tokens,
// consecutive tokens of one segment grouped (at most 16 query rows on the
// decode path; a lone token of G > 16 heads takes a tensor-core tile).
std::vector<Unit> plan_units(const mcp_attn_desc& d, const int32_t* cu, const int32_t* rows,
                             int32_t num_rows) {
  const int G = d.num_q_heads / d.num_kv_heads;
  const int TQ = mcp::kTileRows / G;
  // the decode path is built up to head_dim 128 and for pages of 8 or more
  // tokens; at head_dim 256 or 1-token pages every segment takes tensor-core
  // tiles (a decode token fills G of a tile's 128 rows)
  const bool dec_ok = d.head_dim <= 128 && d.page_size >= 8;
  std::vector<Unit> u;
  if (!rows) {
    for (int s = 0; s < d.num_seqs; ++s) {
      const int64_t lq = cu[s + 1] - cu[s];
      if (lq == 0) continue;
      if (dec_ok && lq * G <= mcp::kDecodeMaxRows) {
        u.push_back({s, 0, lq, true});
      } else {
        for (int64_t qb = 0; qb < lq; qb += TQ) u.push_back({s, qb, std::min<int64_t>(TQ, lq - qb), false});
      }
    }
    return u;
  }
  const int64_t dec_max = std::max(1, mcp::kDecodeMaxRows / G);  // tokens per decode unit
  int s = 0;
  for (int32_t i = 0; i < num_rows;) {
    const int32_t t = rows[i];
    while (cu[s + 1] <= t) ++s;
    const bool dec = dec_ok && G <= mcp::kDecodeMaxRows;
    const int64_t cap = dec ? dec_max : TQ;
    int32_t j = i + 1;
    while (j < num_rows && rows[j] == rows[j - 1] + 1 && rows[j] < cu[s + 1] && j - i < cap) ++j;
    u.push_back({s, t - cu[s], j - i, dec});
    i = j;
  }
  return u;
}

void build(const mcp_attn_desc& d, const int32_t* cu, const int32_t* sk, int num_sms,
           const mcp_plan_options* o, Built& b, const int32_t* rows = nullptr,
           int32_t num_rows = 0) {
  const int G = d.num_q_heads / d.num_kv_heads;
  const int H = d.num_kv_heads;
  // head_dim of the kernel that runs the step (96 runs the 128 one): the cost model's D
  const int DK = d.head_dim == 96 ? 128 : d.head_dim;
  const int HG = mcp::decode_head_group(H);
  const int dopt = o ? o->decode_split_tokens : 0;
  const int popt = o ? o->prefill_split_tokens : 0;
  const std::vector<Unit> units = plan_units(d, cu, rows, num_rows);
  // keys visible to the unit's last token (right-aligned causal)
  auto vis_of = [&](const Unit& x) {
    return static_cast<int64_t>(sk[x.s]) - (cu[x.s + 1] - cu[x.s]) + x.qb + x.qc;
  };

  auto count = [&](int64_t ds, int64_t ps) {
    int64_t n = 0;
    for (const Unit& x : units) {
      int64_t k, z;
      if (x.decode) {
        even_split(vis_of(x), ds, mcp::kPageSize, &k, &z);
        n += k * (H / HG);
      } else {
        even_split(vis_of(x), ps, mcp::kKvTile, &k, &z);
        n += k * H;
      }
    }
    return n;
  };

  // Decode splits: about eight decode items per SM (each item streams its KV
  // range for a whole kv-head group), not below 1024 tokens -- or 256 when the
  // step has no tensor-core tiles, so that a few long rows alone (e.g. the
  // sampled rows of a step) still spread over many SMs.
  bool any_tc = false;
  for (const Unit& x : units) any_tc = any_tc || !x.decode;
  const int64_t ds_floor = any_tc ? 1024 : 256;
  int64_t ds;
  if (dopt > 0) {
    ds = round_up(dopt, mcp::kPageSize);
  } else {
    int64_t dec_tokens = 0;
    for (const Unit& x : units)
      if (x.decode) dec_tokens += vis_of(x) * (H / HG);
    ds = std::max<int64_t>(1024, round_up(cdiv(dec_tokens, 8LL * num_sms), mcp::kPageSize));
  }
  int64_t ps = popt > 0 ? round_up(popt, mcp::kKvTile) : 32768;
  while (count(ds, ps) < 2LL * num_sms) {
    bool changed = false;
    if (dopt <= 0 && ds > ds_floor) { ds = std::max<int64_t>(ds_floor, ds / 2); changed = true; }
    if (popt <= 0 && ps > 2048) { ps /= 2; changed = true; }
    if (!changed) break;
  }
  // Chunk split size for steps made (almost) only of tensor-core tiles: the
  // candidate whose list-scheduled makespan over the SMs is shortest (ties
  // within 2% go to the larger split: fewer items and less combine work).
  // Per-item estimates (ns, GB300): ~5 us of set-up and drain plus ~0.75 us
  // per 128-key tile at D = 128.  Splitting too fine pays the set-up per item;
  // too coarse leaves SMs idle in the last wave.  Steps with real decode work
  // keep the rule above: there HBM-bound decode items and tensor-bound tiles
  // overlap on different SMs, which this model does not capture (measured:
  // it chose a split 2.5% slower on the long-context step).
  if (popt <= 0) {
    const double tile_ns = 750.0 * DK / 128.0, item_ns = 5000.0;
    double pre_ns = 0.0, dec_ns = 0.0;
    for (const Unit& x : units) {
      if (x.decode) dec_ns += vis_of(x) * 4.0 * DK * H / 45.0;
      else pre_ns += H * (item_ns + cdiv(vis_of(x), mcp::kKvTile) * tile_ns);
    }
    if (pre_ns > 0.0 && dec_ns < 0.1 * (pre_ns + dec_ns)) {
      // items of a candidate split (same for every candidate that splits no
      // unit differently); evaluating only distinct candidates and none past
      // sixteen items per SM keeps the search to a few list schedules (finer
      // splits than that only add per-item cost in this model)
      auto signature = [&](int64_t cand_ps) {
        uint64_t sig = 1469598103934665603ull;  // FNV-1a over the units' split counts
        for (const Unit& x : units) {
          if (x.decode) continue;
          int64_t n, sz;
          even_split(vis_of(x), cand_ps, mcp::kKvTile, &n, &sz);
          sig = (sig ^ static_cast<uint64_t>(n)) * 1099511628211ull;
        }
        return static_cast<int64_t>(sig & 0x7fffffffffffffffull);
      };
      std::vector<double> cost, load;
      auto makespan = [&](int64_t cand_ps) {
        cost.clear();
        for (const Unit& x : units) {
          int64_t n, sz;
          if (x.decode) {
            even_split(vis_of(x), ds, mcp::kPageSize, &n, &sz);
            for (int64_t k = 0; k < n; ++k)
              for (int h0 = 0; h0 < H; h0 += HG)
                cost.push_back(3000.0 + std::min<int64_t>(sz, vis_of(x) - k * sz) * 4.0 *
                                            DK * HG / 45.0);
          } else {
            even_split(vis_of(x), cand_ps, mcp::kKvTile, &n, &sz);
            for (int64_t k = 0; k < n; ++k) {
              const double tiles = static_cast<double>(
                  cdiv(std::min<int64_t>(sz, vis_of(x) - k * sz), mcp::kKvTile));
              for (int h = 0; h < H; ++h) cost.push_back(item_ns + tiles * tile_ns);
            }
          }
        }
        std::sort(cost.begin(), cost.end(), std::greater<double>());
        load.assign(static_cast<size_t>(std::max(1, num_sms)), 0.0);
        for (double c : cost) {  // longest first onto the least-loaded SM (a min-heap)
          std::pop_heap(load.begin(), load.end(), std::greater<double>());
          load.back() += c;
          std::push_heap(load.begin(), load.end(), std::greater<double>());
        }
        return *std::max_element(load.begin(), load.end());
      };
      const double t0 = makespan(ps);
      const int64_t ps_sig = signature(ps);
      int64_t best = ps, last_sig = -1;
      double best_t = t0;
      for (int64_t cand = 65536; cand >= 2048; cand /= 2) {
        // candidates finer than the rule's split stop past sixteen items per SM
        // (counts grow as cand shrinks); coarser ones are always evaluated
        if (cand < ps && count(ds, cand) > 16LL * std::max(1, num_sms)) break;
        const int64_t sig = signature(cand);
        if (sig == last_sig) continue;  // the previous, larger candidate had the same items
        last_sig = sig;
        const double t = sig == ps_sig ? t0 : makespan(cand);
        if (t < best_t * 0.98 || (t <= best_t * 1.02 && cand > best)) {
          if (t < best_t) best_t = t;
          best = cand;
        }
      }
      ps = best;
    }
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
  for (const Unit& x : units) {
    const int s = x.s;
    const int64_t vis = vis_of(x);
    const int rows_n = static_cast<int>(x.qc * G);
    if (x.decode) {
      int64_t n, sz;
      even_split(vis, ds, mcp::kPageSize, &n, &sz);
      for (int h0 = 0; h0 < H; h0 += HG) {
        int64_t base = -1;
        if (n > 1) {
          // head j of the group, split k: partial rows base + j*n*rows + k*rows
          base = b.part_rows;
          b.part_rows += n * rows_n * HG;
          for (int j = 0; j < HG; ++j)
            b.comb.push_back({s, h0 + j, static_cast<int32_t>(x.qb), static_cast<int32_t>(x.qc),
                              static_cast<int32_t>(n), static_cast<int32_t>(base + j * n * rows_n),
                              rows_n, 0});
        }
        for (int64_t k = 0; k < n; ++k) {
          mcp::WorkItem it;
          it.seg = s;
          it.kv_head = static_cast<int16_t>(h0);
          it.kind = mcp::kDecodeItem;
          it.num_heads = static_cast<int8_t>(HG);
          it.q_begin = static_cast<int32_t>(x.qb);
          it.q_count = static_cast<int32_t>(x.qc);
          it.kv_begin = static_cast<int32_t>(k * sz);
          it.kv_end = static_cast<int32_t>(std::min(vis, (k + 1) * sz));
          it.part_row = static_cast<int32_t>(n > 1 ? base + k * rows_n : -1);
          it.part_head_stride = static_cast<int32_t>(n * rows_n);
          dec.push_back({it, (it.kv_end - it.kv_begin) * 4.0 * DK * HG / 45.0, 0});
        }
      }
    } else {
      int64_t n, sz;
      even_split(vis, ps, mcp::kKvTile, &n, &sz);
      for (int h = 0; h < H; ++h) {
        int64_t base = -1;
        if (n > 1) {
          base = b.part_rows;
          b.part_rows += n * rows_n;
          b.comb.push_back({s, h, static_cast<int32_t>(x.qb), static_cast<int32_t>(x.qc),
                            static_cast<int32_t>(n), static_cast<int32_t>(base), rows_n, 0});
        }
        for (int64_t k = 0; k < n; ++k) {
          mcp::WorkItem it;
          it.seg = s;
          it.kv_head = static_cast<int16_t>(h);
          it.kind = mcp::kPrefillItem;
          it.num_heads = 1;
          it.q_begin = static_cast<int32_t>(x.qb);
          it.q_count = static_cast<int32_t>(x.qc);
          it.kv_begin = static_cast<int32_t>(k * sz);
          it.kv_end = static_cast<int32_t>(std::min(vis, (k + 1) * sz));
          it.part_row = static_cast<int32_t>(n > 1 ? base + k * rows_n : -1);
          it.part_head_stride = 0;
          const double tiles = static_cast<double>(cdiv(it.kv_end - it.kv_begin, mcp::kKvTile));
          // tiles reading the same K/V (same segment, kv head, split) share a group
          const int64_t gid = (static_cast<int64_t>(s) * H + h) * 4096 + k;
          pre.push_back({it, 300.0 + tiles * 4.0 * 128 * 128 * DK / 6000.0, gid});
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

int32_t mcp_build_flags(void) {
#ifdef MCP_CHECKED
  return MCP_BUILD_CHECKED;
#else
  return 0;
#endif
}

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
  // [L] 4.2 writes through atomics; here slots are unique within a call (the
  // append uses plain stores), so two tokens mapped to one slot -- a physical
  // page shared by two block-table rows, or repeated in one -- are rejected.
  const int32_t T = cu_seqlens_q[num_seqs];
  if (T > 1) {
    std::vector<int64_t> sorted(slot_mapping, slot_mapping + T);
    std::sort(sorted.begin(), sorted.end());
    const auto dup = std::adjacent_find(sorted.begin(), sorted.end());
    if (dup != sorted.end())
      return fail(MCP_ERR_INVALID_ARG,
                  "slot %lld is the slot of two new tokens (a physical page appears twice in "
                  "the block tables)", static_cast<long long>(*dup));
  }
  return okay();
}

}  // extern "C"

namespace {

// Validate, build the work lists and fill *plan (no device access unless the
// SM count has to be queried).
mcp_status plan_common(const mcp_attn_desc* desc, const int32_t* cu, const int32_t* sk,
                       const mcp_plan_options* opts, mcp_plan* plan, Built& b,
                       const int32_t* rows = nullptr, int32_t num_rows = 0) {
  mcp_status st = validate_desc(desc);
  if (st != MCP_OK) return st;
  if (!plan) return fail(MCP_ERR_INVALID_ARG, "plan is NULL");
  if (opts) {
    for (int i = 0; i < 4; ++i)
      if (opts->reserved[i] != 0) return fail(MCP_ERR_INVALID_ARG, "opts->reserved must be 0");
    if (opts->num_sms < 0 || opts->decode_split_tokens < 0 || opts->prefill_split_tokens < 0)
      return fail(MCP_ERR_INVALID_ARG, "negative plan option");
    if (opts->test_stall != 0 && opts->test_stall != 1)
      return fail(MCP_ERR_INVALID_ARG, "opts->test_stall must be 0 or 1");
  }
  st = validate_meta(desc->num_seqs, desc->total_q, desc->page_size, desc->max_pages_per_seq, cu, sk);
  if (st != MCP_OK) return st;
  if (rows) {
    if (num_rows < 0) return fail(MCP_ERR_INVALID_ARG, "num_rows %d < 0", num_rows);
    for (int32_t i = 0; i < num_rows; ++i) {
      if (rows[i] < 0 || rows[i] >= desc->total_q)
        return fail(MCP_ERR_INVALID_ARG, "rows[%d] = %d outside [0, %d)", i, rows[i], desc->total_q);
      if (i > 0 && rows[i] <= rows[i - 1])
        return fail(MCP_ERR_INVALID_ARG, "rows must be strictly increasing (rows[%d] = %d)", i,
                    rows[i]);
    }
  }
  int num_sms = opts ? opts->num_sms : 0;
  if (num_sms <= 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "SM count query: %s", cudaGetErrorString(e));
  }
  build(*desc, cu, sk, num_sms, opts, b, rows, num_rows);
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
  // after the entries: for every block of kCombineRowsPerBlock merged rows,
  // the entry that holds its first row (the combine starts its search there)
  const int64_t cidx = (crow + mcp::kCombineRowsPerBlock - 1) / mcp::kCombineRowsPerBlock;
  pl.off_part_o = align256(pl.off_combine +
                           static_cast<int64_t>(b.comb.size()) * sizeof(mcp::CombineEntry) +
                           cidx * static_cast<int64_t>(sizeof(int32_t)));
  pl.off_part_lse = align256(pl.off_part_o + b.part_rows * desc->head_dim * 4);
  pl.off_error = align256(pl.off_part_lse + b.part_rows * 4);
  pl.workspace_bytes = pl.off_error + 256;
  pl.desc = *desc;
  pl.test_stall = opts ? opts->test_stall : 0;
  *plan = pl;
  return MCP_OK;
}

void write_lists(const mcp_plan& pl, const Built& b, unsigned char* dst) {
  std::memset(dst, 0, static_cast<size_t>(pl.off_part_o));
  if (!b.items.empty()) std::memcpy(dst, b.items.data(), b.items.size() * sizeof(mcp::WorkItem));
  if (!b.comb.empty()) {
    std::memcpy(dst + pl.off_combine, b.comb.data(), b.comb.size() * sizeof(mcp::CombineEntry));
    // block index: entry of the first row of each block of merged rows
    int32_t* idx = reinterpret_cast<int32_t*>(dst + pl.off_combine +
                                              b.comb.size() * sizeof(mcp::CombineEntry));
    size_t e = 0;
    for (int64_t r = 0; r < pl.combine_rows; r += mcp::kCombineRowsPerBlock) {
      while (e + 1 < b.comb.size() && b.comb[e + 1].row_base <= r) ++e;
      *idx++ = static_cast<int32_t>(e);
    }
  }
}

}  // namespace

namespace mcp {

mcp_status check_fwd_args(const mcp_plan* plan, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* block_tables,
                          const int32_t* cu_seqlens_q, const int32_t* seqlens_k, const void* out,
                          const float* lse) {
  if (!plan || plan->magic != kPlanMagic) return fail(MCP_ERR_INVALID_ARG, "plan not initialised");
  if (plan->num_items == 0) return MCP_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !cu_seqlens_q || !seqlens_k || !out)
    return fail(MCP_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return fail(MCP_ERR_INVALID_ARG, "q / caches / out must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(MCP_ERR_INVALID_ARG, "lse not 4-byte aligned");
  return MCP_OK;
}

mcp_status plan_to_host(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                        const int32_t* h_seqlens_k, const mcp_plan_options* opts, mcp_plan* plan,
                        std::vector<unsigned char>& lists) {
  try {
    Built b;
    mcp_status st = plan_common(desc, h_cu_seqlens_q, h_seqlens_k, opts, plan, b);
    if (st != MCP_OK) return st;
    lists.resize(static_cast<size_t>(std::max<int64_t>(1, plan->off_part_o)));
    write_lists(*plan, b, lists.data());
    return MCP_OK;
  } catch (const std::bad_alloc&) {
    return fail(MCP_ERR_INVALID_ARG, "host allocation failed while planning");
  } catch (...) {
    return fail(MCP_ERR_INVALID_ARG, "unexpected host error while planning");
  }
}

}  // namespace mcp

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

mcp_status mcp_mixed_attn_plan_rows(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                                    const int32_t* h_seqlens_k, const int32_t* h_rows,
                                    int32_t num_rows, const mcp_plan_options* opts,
                                    mcp_plan* plan, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (!h_rows && num_rows > 0) return fail(MCP_ERR_INVALID_ARG, "rows is NULL");
  static const int32_t kNone = 0;
  try {
    Built b;
    mcp_status st = plan_common(desc, h_cu_seqlens_q, h_seqlens_k, opts, plan, b,
                                h_rows ? h_rows : &kNone, num_rows);
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

mcp_status mcp_mixed_attn_plan_rows_host(const mcp_attn_desc* desc, const int32_t* h_cu_seqlens_q,
                                         const int32_t* h_seqlens_k, const int32_t* h_rows,
                                         int32_t num_rows, const mcp_plan_options* opts,
                                         mcp_plan* plan, void* host_buffer, size_t host_bytes) {
  if (!h_rows && num_rows > 0) return fail(MCP_ERR_INVALID_ARG, "rows is NULL");
  static const int32_t kNone = 0;
  try {
    Built b;
    mcp_status st = plan_common(desc, h_cu_seqlens_q, h_seqlens_k, opts, plan, b,
                                h_rows ? h_rows : &kNone, num_rows);
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

mcp_status mcp_build_logits_indices(int32_t num_seqs, const int32_t* h_cu_seqlens_q,
                                    const uint8_t* h_sample_mask, int32_t* h_out, int32_t* count) {
  if (num_seqs < 0) return fail(MCP_ERR_INVALID_ARG, "num_seqs %d < 0", num_seqs);
  if (!h_cu_seqlens_q || !count || (num_seqs > 0 && !h_out))
    return fail(MCP_ERR_INVALID_ARG, "NULL pointer argument");
  if (h_cu_seqlens_q[0] != 0)
    return fail(MCP_ERR_INVALID_ARG, "cu_seqlens_q[0] = %d, expected 0", h_cu_seqlens_q[0]);
  int32_t n = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t lo = h_cu_seqlens_q[s], hi = h_cu_seqlens_q[s + 1];
    if (hi < lo) return fail(MCP_ERR_INVALID_ARG, "cu_seqlens_q decreases at segment %d", s);
    if (hi == lo) continue;  // no token this step: nothing to sample
    if (h_sample_mask && !h_sample_mask[s]) continue;
    h_out[n++] = hi - 1;
  }
  *count = n;
  return okay();
}

mcp_status mcp_kv_copy_pages(const void* k_src, const void* v_src, int32_t src_num_pages,
                             void* k_dst, void* v_dst, int32_t dst_num_pages, int32_t page_bytes,
                             const int32_t* src_pages, const int32_t* dst_pages, int32_t num,
                             int32_t* error_word, void* stream) {
  if (num < 0 || src_num_pages < 0 || dst_num_pages < 0 || page_bytes <= 0)
    return fail(MCP_ERR_INVALID_ARG, "bad sizes (num %d, pools %d / %d, page bytes %d)", num,
                src_num_pages, dst_num_pages, page_bytes);
  if (page_bytes % 16 != 0)
    return fail(MCP_ERR_INVALID_ARG, "page_bytes %d not a multiple of 16", page_bytes);
  if (num == 0) return okay();
  if (!k_src || !v_src || !k_dst || !v_dst || !src_pages || !dst_pages)
    return fail(MCP_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(k_src, 16) || !aligned(v_src, 16) || !aligned(k_dst, 16) || !aligned(v_dst, 16))
    return fail(MCP_ERR_INVALID_ARG, "pools must be 16-byte aligned");
  const int e = mcp::launch_copy_pages(k_src, v_src, src_num_pages, k_dst, v_dst, dst_num_pages,
                                       page_bytes, src_pages, dst_pages, num, error_word, stream);
  if (e != 0) return cuda_fail(e, "kv_copy_pages launch");
  return okay();
}

mcp_status mcp_gather_rows(const void* src, int32_t num_src_rows, int32_t row_bytes,
                           const int32_t* rows, int32_t num_rows, void* dst, int32_t* error_word,
                           void* stream) {
  if (num_src_rows < 0 || num_rows < 0 || row_bytes <= 0)
    return fail(MCP_ERR_INVALID_ARG, "bad sizes (src rows %d, rows %d, row bytes %d)",
                num_src_rows, num_rows, row_bytes);
  if (row_bytes % 16 != 0) return fail(MCP_ERR_INVALID_ARG, "row_bytes %d not a multiple of 16", row_bytes);
  if (num_rows == 0) return okay();
  if (!src || !rows || !dst) return fail(MCP_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(src, 16) || !aligned(dst, 16) || !aligned(rows, 4))
    return fail(MCP_ERR_INVALID_ARG, "src / dst must be 16-byte aligned");
  const int e = mcp::launch_gather_rows(src, num_src_rows, row_bytes, rows, num_rows, dst,
                                        error_word, stream);
  if (e != 0) return cuda_fail(e, "gather_rows launch");
  return okay();
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
  mcp_status st = mcp::check_fwd_args(plan, q, k_cache, v_cache, block_tables, cu_seqlens_q,
                                      seqlens_k, out, lse);
  if (st != MCP_OK) return st;
  const mcp_attn_desc& d = plan->desc;
  if (plan->num_items == 0) return okay();
  if (!workspace) return fail(MCP_ERR_INVALID_ARG, "NULL pointer argument (workspace)");
  if (!aligned(workspace, 256)) return fail(MCP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
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
  a.test_stall = plan->test_stall;
  int e = mcp::launch_mixed_attn(a, stream);
  if (e != 0) return cuda_fail(e, "mixed_attn_fwd launch");
  e = mcp::launch_combine(a, stream);
  if (e != 0) return cuda_fail(e, "combine launch");
  return okay();
}

mcp_status mcp_mixed_attn_fwd_varlen(const mcp_plan* plan, const void* q, const void* k,
                                     const void* v, const int32_t* cu_seqlens_q,
                                     const int32_t* cu_seqlens_k, int64_t total_k, void* out,
                                     float* lse, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  if (!plan || plan->magic != kPlanMagic) return fail(MCP_ERR_INVALID_ARG, "plan not initialised");
  const mcp_attn_desc& d = plan->desc;
  if (d.page_size != mcp::kPageSize)
    return fail(MCP_ERR_INVALID_ARG, "plan a non-paged step with page_size 16");
  if (total_k < 0 || total_k > (int64_t(1) << 30))
    return fail(MCP_ERR_INVALID_ARG, "total_k %lld outside [0, 2^30]", static_cast<long long>(total_k));
  if (plan->num_items == 0) return okay();
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out || !workspace)
    return fail(MCP_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return fail(MCP_ERR_INVALID_ARG, "q / k / v / out must be 16-byte aligned");
  if (!aligned(workspace, 256)) return fail(MCP_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(MCP_ERR_INVALID_ARG, "lse not 4-byte aligned");
  if (static_cast<int64_t>(workspace_bytes) < plan->workspace_bytes)
    return fail(MCP_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %lld needed", workspace_bytes,
                static_cast<long long>(plan->workspace_bytes));
  char* ws = static_cast<char*>(workspace);
  mcp::FwdArgs a;
  a.q = q;
  a.k_cache = k;
  a.v_cache = v;
  a.block_tables = nullptr;
  a.cu_seqlens_q = cu_seqlens_q;
  a.seqlens_k = nullptr;
  a.cu_seqlens_k = cu_seqlens_k;
  a.total_k = total_k;
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
  a.test_stall = plan->test_stall;
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

// ---------------------------------------------------------------------------
// One step from host memory, two steps in flight ([W] "输入组装": write the new
// K/V through the slot mapping, then attend).  Slot n % 2 stages step n.
// Streams: copy-in (h2d), the caller's stream (kernels), copy-out (d2h);
// events: staged (copy-in done), computed (kernels done), done (copy-out
// done).  A slot is reused only after the host has seen its `done` event, so
// none of its device or page-locked buffers is overwritten while in use.
// ---------------------------------------------------------------------------

namespace {

struct StepLayout {
  // per-slot byte offsets; device slot
  int64_t d_q, d_k, d_v, d_out, d_lse, d_meta, d_slots, d_ws, d_slot_bytes;
  // page-locked host slot
  int64_t h_meta, h_slots, h_lists, h_err, h_slot_bytes;
  int64_t n_meta;  // int32 metadata words: cu (S+1) | seqlens_k (S) | block tables (S * mp)
  int64_t ws_bytes, list_bytes;
};

mcp_status step_limits(const mcp_attn_desc* shape, const mcp_host_step_limits* lim,
                       mcp_host_step_limits& out) {
  if (!lim) return fail(MCP_ERR_INVALID_ARG, "limits is NULL");
  if (!shape) return fail(MCP_ERR_INVALID_ARG, "shape is NULL");
  mcp_attn_desc d = *shape;
  d.num_seqs = 0;
  d.total_q = 0;
  d.max_pages_per_seq = 1;
  mcp_status st = validate_desc(&d);
  if (st != MCP_OK) return st;
  if (lim->reserved0 != 0) return fail(MCP_ERR_INVALID_ARG, "limits->reserved0 must be 0");
  for (int i = 0; i < 4; ++i)
    if (lim->reserved[i] != 0) return fail(MCP_ERR_INVALID_ARG, "limits->reserved must be 0");
  if (lim->max_tokens <= 0 || lim->max_seqs <= 0 || lim->max_pages_per_seq <= 0)
    return fail(MCP_ERR_INVALID_ARG, "limits must be positive (tokens %d, seqs %d, pages %d)",
                lim->max_tokens, lim->max_seqs, lim->max_pages_per_seq);
  if (lim->workspace_bytes < 0 || lim->list_bytes < 0)
    return fail(MCP_ERR_INVALID_ARG, "negative workspace or list bytes");
  out = *lim;
  if (out.workspace_bytes == 0) out.workspace_bytes = int64_t(64) << 20;
  if (out.list_bytes == 0) out.list_bytes = int64_t(4) << 20;
  return MCP_OK;
}

StepLayout step_layout(const mcp_attn_desc& s, const mcp_host_step_limits& lim) {
  StepLayout L;
  const int64_t T = lim.max_tokens, S = lim.max_seqs, mp = lim.max_pages_per_seq;
  const int64_t qrow = static_cast<int64_t>(s.num_q_heads) * s.head_dim * 2;
  const int64_t kvrow = static_cast<int64_t>(s.num_kv_heads) * s.head_dim * 2;
  L.n_meta = (S + 1) + S + S * mp;
  int64_t o = 0;
  L.d_q = o;     o = align256(o + T * qrow);
  L.d_k = o;     o = align256(o + T * kvrow);
  L.d_v = o;     o = align256(o + T * kvrow);
  L.d_out = o;   o = align256(o + T * qrow);
  L.d_lse = o;   o = align256(o + T * s.num_q_heads * 4);
  L.d_meta = o;  o = align256(o + L.n_meta * 4);
  L.d_slots = o; o = align256(o + T * 8);
  L.d_ws = o;    o = align256(o + lim.workspace_bytes);
  L.d_slot_bytes = o;
  o = 0;
  L.h_meta = o;  o = align256(o + L.n_meta * 4);
  L.h_slots = o; o = align256(o + T * 8);
  L.h_lists = o; o = align256(o + lim.list_bytes);
  L.h_err = o;   o = align256(o + 4);
  L.h_slot_bytes = o;
  L.ws_bytes = lim.workspace_bytes;
  L.list_bytes = lim.list_bytes;
  return L;
}

mcp_status error_bits_status(int32_t v) {
  if (v & MCP_DEVERR_TIMEOUT)
    return fail(MCP_ERR_TIMEOUT, "a device-side wait gave up (error bits 0x%x)", v);
  if (v != 0) return fail(MCP_ERR_DEVICE_CHECK, "device range check failed (error bits 0x%x)", v);
  return okay();
}

}  // namespace

struct mcp_host_step {
  struct Slot {
    char* dev;
    unsigned char* host;
    cudaEvent_t staged = nullptr, computed = nullptr, done = nullptr;
    int64_t ticket = -1;  // step staged in this slot and not yet checked, else -1
  };
  mcp_attn_desc shape;
  mcp_host_step_limits lim;
  StepLayout L;
  cudaStream_t compute = nullptr, h2d = nullptr, d2h = nullptr;
  Slot slot[2];
  int64_t next = 0;
  std::vector<int64_t> slots_tmp;  // the next step's slot mapping, built before its slot is free

  // Wait for the slot's step and turn its device error word into a status.
  mcp_status settle(Slot& sl) {
    if (sl.ticket < 0) return okay();
    const cudaError_t e = cudaEventSynchronize(sl.done);
    if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "step %lld: %s", static_cast<long long>(sl.ticket),
                                      cudaGetErrorString(e));
    int32_t* err = reinterpret_cast<int32_t*>(sl.host + L.h_err);
    const int32_t v = *err;
    *err = 0;
    sl.ticket = -1;
    return error_bits_status(v);
  }
};

extern "C" {

mcp_status mcp_host_step_arena_bytes(const mcp_attn_desc* shape, const mcp_host_step_limits* limits,
                                     size_t* device_bytes, size_t* host_bytes) {
  mcp_host_step_limits lim;
  mcp_status st = step_limits(shape, limits, lim);
  if (st != MCP_OK) return st;
  if (!device_bytes || !host_bytes) return fail(MCP_ERR_INVALID_ARG, "NULL size pointer");
  const StepLayout L = step_layout(*shape, lim);
  *device_bytes = static_cast<size_t>(2 * L.d_slot_bytes);
  *host_bytes = static_cast<size_t>(2 * L.h_slot_bytes);
  return okay();
}

mcp_status mcp_host_step_create(const mcp_attn_desc* shape, const mcp_host_step_limits* limits,
                                void* device_arena, size_t device_bytes, void* host_arena,
                                size_t host_bytes, void* stream, mcp_host_step** step) {
  mcp_host_step_limits lim;
  mcp_status st = step_limits(shape, limits, lim);
  if (st != MCP_OK) return st;
  if (!step) return fail(MCP_ERR_INVALID_ARG, "step is NULL");
  *step = nullptr;
  const StepLayout L = step_layout(*shape, lim);
  if (!device_arena || !host_arena) return fail(MCP_ERR_INVALID_ARG, "NULL arena");
  if (!aligned(device_arena, 256) || !aligned(host_arena, 256))
    return fail(MCP_ERR_INVALID_ARG, "arenas must be 256-byte aligned");
  if (static_cast<int64_t>(device_bytes) < 2 * L.d_slot_bytes ||
      static_cast<int64_t>(host_bytes) < 2 * L.h_slot_bytes)
    return fail(MCP_ERR_WORKSPACE_TOO_SMALL, "arenas %zu / %zu bytes < %lld / %lld needed",
                device_bytes, host_bytes, static_cast<long long>(2 * L.d_slot_bytes),
                static_cast<long long>(2 * L.h_slot_bytes));
  cudaPointerAttributes pa;
  cudaError_t e = cudaPointerGetAttributes(&pa, host_arena);
  if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "host arena query: %s", cudaGetErrorString(e));
  if (pa.type != cudaMemoryTypeHost)
    return fail(MCP_ERR_INVALID_ARG, "host arena is not page-locked host memory");
  e = cudaPointerGetAttributes(&pa, device_arena);
  if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "device arena query: %s", cudaGetErrorString(e));
  if (pa.type != cudaMemoryTypeDevice)
    return fail(MCP_ERR_INVALID_ARG, "device arena is not device memory");
  mcp_host_step* h = new (std::nothrow) mcp_host_step();
  if (!h) return fail(MCP_ERR_INVALID_ARG, "host allocation failed");
  h->shape = *shape;
  h->lim = lim;
  h->L = L;
  h->compute = static_cast<cudaStream_t>(stream);
  e = cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
    mcp_host_step::Slot& sl = h->slot[i];
    sl.dev = static_cast<char*>(device_arena) + i * L.d_slot_bytes;
    sl.host = static_cast<unsigned char*>(host_arena) + i * L.h_slot_bytes;
    *reinterpret_cast<int32_t*>(sl.host + L.h_err) = 0;
    e = cudaEventCreateWithFlags(&sl.staged, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sl.computed, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    mcp_host_step_destroy(h);
    return fail(MCP_ERR_CUDA, "host step streams/events: %s", cudaGetErrorString(e));
  }
  *step = h;
  return okay();
}

mcp_status mcp_host_step_run(mcp_host_step* step, int32_t num_seqs, const int32_t* cu_seqlens_q,
                             const int32_t* seqlens_k, const int32_t* block_tables,
                             const void* q, const void* k_new, const void* v_new, void* k_cache,
                             void* v_cache, void* out, float* lse, int64_t* ticket) {
  try {
    if (!step) return fail(MCP_ERR_INVALID_ARG, "step is NULL");
    if (!ticket) return fail(MCP_ERR_INVALID_ARG, "ticket is NULL");
    const mcp_host_step_limits& lim = step->lim;
    const StepLayout& L = step->L;
    if (num_seqs < 0 || num_seqs > lim.max_seqs)
      return fail(MCP_ERR_INVALID_ARG, "num_seqs %d outside [0, %d]", num_seqs, lim.max_seqs);
    if (!cu_seqlens_q) return fail(MCP_ERR_INVALID_ARG, "cu_seqlens_q is NULL");
    if (num_seqs > 0 && (!seqlens_k || !block_tables))
      return fail(MCP_ERR_INVALID_ARG, "seqlens_k / block_tables is NULL");
    const int32_t T = cu_seqlens_q[num_seqs];
    if (T < 0 || T > lim.max_tokens)
      return fail(MCP_ERR_INVALID_ARG, "step has %d tokens, limit %d", T, lim.max_tokens);
    if (T > 0 && (!q || !k_new || !v_new || !out))
      return fail(MCP_ERR_INVALID_ARG, "NULL token buffer");
    if (!k_cache || !v_cache) return fail(MCP_ERR_INVALID_ARG, "NULL cache");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16))
      return fail(MCP_ERR_INVALID_ARG, "caches must be 16-byte aligned");

    // Plan and build the slot mapping (which validates every page id) before
    // waiting for this step's slot: the slot frees when the step two before
    // has copied its output out, and the host work then overlaps it.
    mcp_attn_desc desc = step->shape;
    desc.num_seqs = num_seqs;
    desc.total_q = T;
    desc.max_pages_per_seq = lim.max_pages_per_seq;
    mcp_plan plan;
    Built b;
    mcp_status st = plan_common(&desc, cu_seqlens_q, seqlens_k, nullptr, &plan, b);
    if (st != MCP_OK) return st;
    if (plan.workspace_bytes > L.ws_bytes)
      return fail(MCP_ERR_WORKSPACE_TOO_SMALL, "step needs %lld workspace bytes > limit %lld",
                  static_cast<long long>(plan.workspace_bytes), static_cast<long long>(L.ws_bytes));
    if (plan.off_part_o > L.list_bytes)
      return fail(MCP_ERR_WORKSPACE_TOO_SMALL, "work lists need %lld bytes > limit %lld",
                  static_cast<long long>(plan.off_part_o), static_cast<long long>(L.list_bytes));
    const int64_t S = num_seqs, mp = lim.max_pages_per_seq;
    step->slots_tmp.resize(static_cast<size_t>(std::max(1, T)));
    st = mcp_build_slot_mapping(block_tables, num_seqs, lim.max_pages_per_seq, desc.page_size,
                                desc.num_pages, cu_seqlens_q, seqlens_k, step->slots_tmp.data());
    if (st != MCP_OK) return st;

    mcp_host_step::Slot& sl = step->slot[step->next & 1];
    // the slot's previous step must be finished before its buffers are reused
    st = step->settle(sl);
    if (st != MCP_OK) return st;
    // host staging: metadata, slot mapping, work lists
    int32_t* hm = reinterpret_cast<int32_t*>(sl.host + L.h_meta);
    int64_t* hs = reinterpret_cast<int64_t*>(sl.host + L.h_slots);
    if (T > 0) std::memcpy(hs, step->slots_tmp.data(), static_cast<size_t>(T) * sizeof(int64_t));
    std::memcpy(hm, cu_seqlens_q, (S + 1) * sizeof(int32_t));
    if (S > 0) {
      std::memcpy(hm + S + 1, seqlens_k, S * sizeof(int32_t));
      std::memcpy(hm + 2 * S + 1, block_tables, S * mp * sizeof(int32_t));
    }
    write_lists(plan, b, sl.host + L.h_lists);

    char* dev = sl.dev;
    int32_t* d_meta = reinterpret_cast<int32_t*>(dev + L.d_meta);
    char* ws = dev + L.d_ws;
    const int64_t n_meta = (S + 1) + S + S * mp;
    const int64_t qbytes = static_cast<int64_t>(T) * desc.num_q_heads * desc.head_dim * 2;
    const int64_t kvbytes = static_cast<int64_t>(T) * desc.num_kv_heads * desc.head_dim * 2;
    const size_t lse_bytes = static_cast<size_t>(T) * desc.num_q_heads * 4;
    cudaError_t e = cudaMemcpyAsync(d_meta, hm, n_meta * 4, cudaMemcpyHostToDevice, step->h2d);
    if (e == cudaSuccess && T > 0)
      e = cudaMemcpyAsync(dev + L.d_slots, hs, static_cast<size_t>(T) * 8, cudaMemcpyHostToDevice,
                          step->h2d);
    if (e == cudaSuccess && plan.off_part_o > 0)
      e = cudaMemcpyAsync(ws, sl.host + L.h_lists, plan.off_part_o, cudaMemcpyHostToDevice, step->h2d);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws + plan.off_error, 0, 256, step->h2d);
    if (e == cudaSuccess && T > 0) e = cudaMemcpyAsync(dev + L.d_q, q, qbytes, cudaMemcpyHostToDevice, step->h2d);
    if (e == cudaSuccess && T > 0) e = cudaMemcpyAsync(dev + L.d_k, k_new, kvbytes, cudaMemcpyHostToDevice, step->h2d);
    if (e == cudaSuccess && T > 0) e = cudaMemcpyAsync(dev + L.d_v, v_new, kvbytes, cudaMemcpyHostToDevice, step->h2d);
    if (e == cudaSuccess) e = cudaEventRecord(sl.staged, step->h2d);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(step->compute, sl.staged, 0);
    if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "step copy-in: %s", cudaGetErrorString(e));

    int32_t* err_word = reinterpret_cast<int32_t*>(ws + plan.off_error);
    if (T > 0) {
      const int rc = mcp::launch_append(dev + L.d_k, dev + L.d_v,
                                        reinterpret_cast<const int64_t*>(dev + L.d_slots), T,
                                        desc.num_kv_heads * desc.head_dim * 2,
                                        static_cast<int64_t>(desc.num_pages) * desc.page_size,
                                        k_cache, v_cache, err_word, step->compute);
      if (rc != 0) return cuda_fail(rc, "step append launch");
    }
    st = mcp_mixed_attn_fwd(&plan, dev + L.d_q, k_cache, v_cache, d_meta + 2 * S + 1, d_meta,
                            d_meta + S + 1, dev + L.d_out,
                            lse ? reinterpret_cast<float*>(dev + L.d_lse) : nullptr, ws,
                            static_cast<size_t>(L.ws_bytes), step->compute);
    if (st != MCP_OK) return st;
    e = cudaEventRecord(sl.computed, step->compute);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(step->d2h, sl.computed, 0);
    if (e == cudaSuccess && T > 0)
      e = cudaMemcpyAsync(out, dev + L.d_out, qbytes, cudaMemcpyDeviceToHost, step->d2h);
    if (e == cudaSuccess && T > 0 && lse)
      e = cudaMemcpyAsync(lse, dev + L.d_lse, lse_bytes, cudaMemcpyDeviceToHost, step->d2h);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(sl.host + L.h_err, err_word, 4, cudaMemcpyDeviceToHost, step->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(sl.done, step->d2h);
    if (e != cudaSuccess) return fail(MCP_ERR_CUDA, "step copy-out: %s", cudaGetErrorString(e));
    sl.ticket = step->next;
    *ticket = step->next++;
    return okay();
  } catch (const std::bad_alloc&) {
    return fail(MCP_ERR_INVALID_ARG, "host allocation failed while planning");
  } catch (...) {
    return fail(MCP_ERR_INVALID_ARG, "unexpected host error in a step");
  }
}

mcp_status mcp_host_step_wait(mcp_host_step* step, int64_t ticket) {
  if (!step) return fail(MCP_ERR_INVALID_ARG, "step is NULL");
  if (ticket < 0 || ticket >= step->next)
    return fail(MCP_ERR_INVALID_ARG, "ticket %lld was never issued", static_cast<long long>(ticket));
  for (mcp_host_step::Slot& sl : step->slot)
    if (sl.ticket == ticket) return step->settle(sl);
  return okay();  // its slot was reused, which checked it
}

mcp_status mcp_host_step_destroy(mcp_host_step* step) {
  if (!step) return okay();
  mcp_status st = MCP_OK;
  for (mcp_host_step::Slot& sl : step->slot) {
    const mcp_status s2 = step->settle(sl);
    if (st == MCP_OK) st = s2;
  }
  for (mcp_host_step::Slot& sl : step->slot) {
    if (sl.staged) cudaEventDestroy(sl.staged);
    if (sl.computed) cudaEventDestroy(sl.computed);
    if (sl.done) cudaEventDestroy(sl.done);
  }
  if (step->h2d) cudaStreamDestroy(step->h2d);
  if (step->d2h) cudaStreamDestroy(step->d2h);
  delete step;
  return st == MCP_OK ? okay() : st;
}

}  // extern "C"
