// Fused mixed (chunked-prefill + decode) paged-attention forward for sm_103a.
//
// One launch serves the whole packed token stream ([K] "平铺策略 / 掩码特化":
// one kernel for prefill chunks and decodes; [W] "Flash Attention 的 varlen
// 接口": the i-th query segment attends only to the i-th KV segment,
// right-aligned causal).  Each CTA (10 warps) runs one work item of the host
// plan:
//
//  * tensor-core item -- 128 query rows (the G query heads of one kv head
//    packed with 128/G tokens) against a KV range in 128-key tiles (64 at
//    head_dim 256).  Warp 0
//    loads the Q tile with TMA and then issues O += P V; warp 1 issues
//    S = Q K^T (A = Q, copied once into TMEM by the softmax warps; B = the K
//    tile in shared memory); warps 6-9 load each K/V tile box by box through
//    the block table (8 boxes x D/64 panels of K plus 8 boxes of V for 16-token
//    boxes, twice as many 8-token boxes for 8-token pages), split over four
//    warps because one warp issues its boxes serially; warps 2-5 run the
//    online softmax on S rows read from TMEM, write bf16 P over the scores
//    they read (S buffer t & 1) and rescale O lazily.  Only tiles that cross
//    the diagonal are masked ([K] "掩码特化").
//  * decode item -- the G*Lq (<= 16) query rows of each kv head of a head group
//    (up to 8 heads) against a KV range.  Warps 0 and 1 stream 16 tokens of
//    the group per ring stage -- warp 0 the TMA box of K, warp 1 the box of
//    V, laid out in shared memory as [head][panel][token][64] (two boxes each
//    for 8-token pages) -- through a multi-stage ring; warps 2-9 each own one
//    kv head (ldmatrix + mma.sync m16n8k16, shuffle max/sum, online softmax;
//    with at most 8 rows the products are taken transposed, the keys in M and
//    the rows in N, see decode_n8); several warps share a head when the group
//    is smaller than 8 and merge their states at the end.
//
// head_dim 96 runs the D = 128 instantiation on 96-wide tensors: the tensor
// maps span 96 columns, TMA fills columns 96-127 of every box with zeros, V
// and decode stages take one box per 64-column panel, and only 96 columns of
// O are stored.  head_dim 256 uses 64-key tiles (TMEM: S twice in columns
// 0-127, O in 128-383, Q in 384-511) with two K and V stages, and has no
// decode path: the planner gives its decode tokens tensor-core tiles.  With
// 1-token pages the producers gather K/V rows with cp.async into the same
// layouts (and decode tokens take tensor-core tiles too).
//
// A split KV range writes (O, LSE) partials that combine.cu merges.
//
// Every mbarrier wait is bounded in time.  On time-out the CTA records
// MCP_DEVERR_TIMEOUT in the error word, every role leaves its loop, in-flight
// TMA copies and MMAs are drained (again with a bound), TMEM is freed and the
// CTA exits without writing outputs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <type_traits>

#include "mcp.h"
#include "mcp_internal.h"
#include "ptx.cuh"

namespace mcp {
namespace {

constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;  // 0.5 s per wait
constexpr uint64_t kTestWaitLimitNs = 1000ull * 1000ull;       // 1 ms (test_stall plans)
constexpr float kRescaleThreshold = 8.0f;  // rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kLog2e = 1.44269504088896341f;
constexpr int kDecRingBytes = 192 * 1024;  // decode page ring
constexpr int kMaxDecStages = 48;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;        // 64-column (128-byte) swizzle panels
  // tensor-core item: 128-key tiles up to D = 128; at D = 256 64-key tiles,
  // so that S (twice), O and Q fit the 512 TMEM columns and two K and V
  // stages fit shared memory
  static constexpr int kKvTile = D > 128 ? 64 : 128;
  static constexpr int kQPanel = kTileRows * 128;  // a 64-column panel of Q: 128 rows x 128 B
  static constexpr int kKPanel = kKvTile * 128;    // a 64-column panel of a K tile
  static constexpr int kQBytes = kHalves * kQPanel;
  static constexpr int kKvBytes = kHalves * kKPanel;  // one K (or V) tile
  static constexpr int kKStages = D > 128 ? 2 : 3;  // K of tile t in stage t % kKStages
  static constexpr int kVStages = kKStages;         // V of tile t in stage t % kVStages
  // TMEM columns: S buffers [0, 2 kKvTile), O [kColO, kColO + D), Q [kColQ, kColQ + D/2)
  static constexpr int kColO = 2 * kKvTile;
  static constexpr int kColQ = 384;
  static_assert(kColO + D <= kColQ && kColQ + D / 2 <= 512, "TMEM columns");
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBytes;                          // K stage s at kOffK + s*kKvBytes
  static constexpr int kOffV = kOffK + kKStages * kKvBytes;      // V stage s at kOffV + s*kKvBytes
  static constexpr int kPrefillBytes = kOffV + kVStages * kKvBytes;  // P lives in TMEM
  // decode item: ring of [K block | V block], block = [head][panel][16 tokens][128 B]
  static constexpr int kHeadBlock = kHalves * kPageSize * 128;
  static constexpr int kMergeBytes = 8 * 16 * D * 4 + 2 * 8 * 16 * 4;  // reuses the ring
  static_assert(kMergeBytes <= kDecRingBytes, "merge area");
  // common
  static constexpr int kDataBytes = kPrefillBytes > kDecRingBytes ? kPrefillBytes : kDecRingBytes;
  static constexpr int kOffBar = (kDataBytes + 1023) & ~1023;
  static constexpr int kSmemBytes = kOffBar + 1024 + 1024;  // barriers/flags + alignment slack
  static_assert(kSmemBytes <= 232448, "227 KB dynamic shared memory limit");
};

// barrier slots
enum : int {
  BQ = 0,        // Q tile landed
  BK0 = 1,       // K of stage s landed (BK0 + s, s < 3); two producer warps arrive
  BV0 = 4,       // V of stage s landed; two producer warps arrive
  BE0 = 7,       // P V of the tile in stage s done: V stage free, O updated
  BS0 = 10,      // S buffer s holds Q K^T of tile t (s = t & 1)
  BP0 = 12,      // P of tile t written (BP0 + (t & 1); 128 softmax threads)
  BDRAIN = 14,   // all MMAs of the CTA finished (both issuing warps commit)
  BQT = 15,      // Q copied into TMEM (128 softmax threads)
  BKE0 = 16,     // Q K^T of the tile in stage s done: K stage free
  BFULL0 = 19,   // decode ring stage landed (BFULL0 .. BFULL0+kMaxDecStages-1)
  BEMPTY0 = BFULL0 + kMaxDecStages,  // decode ring stage free
  kNumBars = BEMPTY0 + kMaxDecStages
};
static_assert(kNumBars * 8 + 32 <= 1024, "barrier block");

struct Ctx {
  uint32_t bar;
  volatile int* abort;
  int32_t* err;
  uint64_t limit_ns;  // bound of every wait: kWaitLimitNs, or kTestWaitLimitNs
  __device__ __forceinline__ uint32_t b(int i) const { return bar + 8u * static_cast<uint32_t>(i); }
};

__device__ __noinline__ bool wait_slow(volatile int* abort, int32_t* err, uint32_t bar,
                                       uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
#pragma unroll 1
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      if (err) atomicOr(err, MCP_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Wait for the phase with `parity` of barrier `bar` to complete; false if the
// CTA aborted or the wait ran past c.limit_ns (then the CTA aborts).
__device__ __forceinline__ bool wait_on(const Ctx& c, uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_slow(c.abort, c.err, bar, parity, c.limit_ns);
}

// wait_on for a warp that goes on to .sync.aligned tcgen05 instructions: every
// lane gets the same answer, so a failed wait never leaves part of the warp
// behind (each lane's own wait is bounded, so all of them reach the vote).
__device__ __forceinline__ bool wait_on_warp(const Ctx& c, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_on(c, bar, parity));
}

// Bounded wait that ignores the abort flag: used to let this CTA's own async
// copies / MMAs finish before it exits.
__device__ __noinline__ void drain_wait_slow(volatile int* abort, int32_t* err, uint32_t bar,
                                             uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
#pragma unroll 1
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      if (err) atomicOr(err, MCP_DEVERR_TIMEOUT);
      return;
    }
  }
}
__device__ __forceinline__ void drain_wait(const Ctx& c, uint32_t bar, uint32_t parity) {
  drain_wait_slow(c.abort, c.err, bar, parity, c.limit_ns);
}

struct KParams {
  const WorkItem* items;
  const int32_t* cu_q;
  const int32_t* seqlens_k;
  const int32_t* bt;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int32_t* err;
  int32_t max_pages;
  int32_t num_pages;
  int32_t hq;
  int32_t G;
  int32_t dec_stages;  // decode ring stages (a multiple of the warps sharing one head)
  int32_t spp_log2;    // log2 of TMA boxes per cache page (0 for page size 8 and 16, 1: 32, 2: 64)
  int32_t box_log2;    // log2 of tokens per TMA box: 3 for page size 8, else 4
  int32_t dr;          // head_dim of the tensors (row width of q, out, K/V, partials): the
                       // kernel's D, or 96 run as D = 128 (TMA fills columns 96-127 with 0)
  int32_t panel_boxes; // 1: V and decode boxes cover one 64-column panel each (dr < D)
  int32_t gather;      // 1: 1-token pages; the producers gather K/V rows with cp.async
  int32_t hkv;         // kv heads (row stride of the caches, in head_dim rows)
  const __nv_bfloat16* kc;  // caches [num_pages, 1, H_kv, dr] (gather only)
  const __nv_bfloat16* vc;
  const int32_t* cu_k; // non-paged K/V: first row of each segment's keys (else nullptr)
  float scale_log2;    // sm_scale * log2(e): scores live in log2 units
  int32_t k_box5;      // 1: 8-token boxes of K carry every 64-column panel (one box per 8
                       // keys, landing [panel][8 keys][128 B]); 0: one box per panel
  int32_t test_stall;  // testing only: 1 = tensor-core items never issue their Q-tile load,
                       // so their softmax waits run out (1 ms bound) and the CTA aborts
};

struct Seg {
  int q_start, lq, lk, hist;
};

// The kernels move KV in boxes of B = 16 tokens (page size 16, 32, 64) or
// B = 8 tokens (page size 8).  Box `u` of segment `seg` lives in cache page
// bt[seg][u / (P/B)] at token (u % (P/B)) * B.  box_of packs both as
// (page << spp_log2) | (u % (P/B)); a block-table entry outside the pool gives
// page num_pages (an out-of-range TMA coordinate: the copy fills zeros) and an
// error bit.
__device__ __forceinline__ int box_of(const KParams& p, int seg, int u) {
  // non-paged K/V: the box is rows cu_k[seg] + B u ... of one tensor (the
  // tensor maps then have a single "page" spanning every row)
  if (p.cu_k) return p.cu_k[seg] + (u << p.box_log2);
  const int v = p.bt[static_cast<size_t>(seg) * p.max_pages + (u >> p.spp_log2)];
  const int sub = u & ((1 << p.spp_log2) - 1);
  if (v >= 0 && v < p.num_pages) return (v << p.spp_log2) | sub;
  atomicOr(p.err, MCP_DEVERR_PAGE_RANGE);
  return p.num_pages << p.spp_log2;
}
// cache page and first token of a packed box
__device__ __forceinline__ int blk_page(const KParams& p, int b) {
  return p.cu_k ? 0 : b >> p.spp_log2;
}
__device__ __forceinline__ int blk_tok(const KParams& p, int b) {
  return p.cu_k ? b : (b & ((1 << p.spp_log2) - 1)) << p.box_log2;
}
// a box outside every tensor (TMA fills zeros)
__device__ __forceinline__ int oob_block(const KParams& p) {
  return p.cu_k ? (1 << 30) : p.num_pages << p.spp_log2;
}

// ------------------------------------------------------------------------
// tensor-core item
// ------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void prefill_item(const Ctx& c, const WorkItem& it, const Seg& sg,
                                             const KParams& p, uint32_t base, uint8_t* gb,
                                             uint32_t tmem, const CUtensorMap* tm_q,
                                             const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                             int warp, int lane) {
  using C = Cfg<D>;
  constexpr int kKvTile = C::kKvTile;  // keys per tile (shadows the 128 of the planner)
  const int G = p.G;
  const int TQ = kTileRows / G;
  const int kv0 = it.kv_begin, kv1 = it.kv_end;
  const int ntiles = (kv1 - kv0 + kKvTile - 1) / kKvTile;
  const uint32_t sQ = base + C::kOffQ;
  auto sK = [&](int s) { return base + C::kOffK + static_cast<uint32_t>(s * C::kKvBytes); };
  auto sV = [&](int s) { return base + C::kOffV + static_cast<uint32_t>(s * C::kKvBytes); };

  // Two warps issue the MMAs: warp 1 Q K^T, warp 0 P V.  Each waits only for
  // its own operands, so one warp's barrier waits overlap the other's MMAs
  // (with a single issuer the waits sat between every pair of MMA groups and
  // the tensor pipe idled for them).  Both feed the same in-order tensor pipe;
  // Q K^T(t) waits for P V(t - 2), the last reader of S buffer t & 1.
  constexpr uint32_t kIdQK = ptx::idesc_bf16(128, kKvTile, false);
  constexpr uint32_t kIdPV = ptx::idesc_bf16(128, D, true);
  if (warp == 0) {
    // ---------------------------------------- Q tile (TMA), then P V issuer
    if (lane == 0 && !p.test_stall) {
      ptx::mbar_arrive_expect_tx(c.b(BQ), C::kHalves * G * TQ * 128);
      for (int h = 0; h < C::kHalves; ++h)
        ptx::tma_load_3d(sQ + h * C::kQPanel, tm_q, c.b(BQ), 64 * h, it.kv_head * G,
                         sg.q_start + it.q_begin, ptx::policy_evict_first());
    }
    __syncwarp();
    const uint32_t tS = tmem;              // S buffers: columns [0, kKvTile), [kKvTile, 2 kKvTile)
    const uint32_t tO = tmem + C::kColO;   // O
    // descriptor of stage 0 built once; an MMA adds a byte offset >> 4 to the
    // start-address field (shared addresses stay below 256 KB: no carry out)
    // V stage: boxes of B tokens, each [panel][B tokens][128 B]: 64-column
    // panels B * 128 bytes apart, 8-key groups 1024 bytes apart inside a
    // 16-token box and one box (D/64 KB) apart with 8-token boxes
    const int B = 1 << p.box_log2;
    const uint64_t dV0 = ptx::sdesc_sw128(sV(0), B * 128, B == 16 ? 1024 : C::kHalves * 1024);
    bool ok = true;
    for (int t = 0; ok && t < ntiles; ++t) {
      // P(t) barriers alternate with the tile parity, like the S buffers: the
      // barrier is reused by tile t + 2 only after Q K^T(t + 2), which waits
      // for this P V(t), so no waiter falls two phases behind
      if (!(ok = wait_on(c, c.b(BP0 + (t & 1)), (t >> 1) & 1))) break;
      const int s = t % C::kVStages;
      if (!(ok = wait_on(c, c.b(BV0 + s), (t / C::kVStages) & 1))) break;
      const int nval = kv1 - (kv0 + t * kKvTile);
      if (nval < kKvTile && (nval & (B - 1))) {
        // Rows past the item's last key inside its last box may be unused
        // cache slots holding anything (NaN included); P is 0 there but
        // 0 * NaN would reach O, so those V rows are zeroed.
        const int r0 = nval, nr = ((nval + B - 1) & ~(B - 1)) - nval;
        const int per_half = nr * 8;
        uint8_t* gV = gb + (sV(s) - base);
        for (int i = lane; i < per_half * C::kHalves; i += 32) {
          const int h = i / per_half, rem = i - h * per_half;
          const int r = r0 + rem / 8, ch = rem & 7;
          *reinterpret_cast<uint4*>(gV + (r >> p.box_log2) * (C::kHalves * B * 128) + h * B * 128 +
                                    (r & (B - 1)) * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
      }
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint64_t dv = dV0 + static_cast<uint64_t>((s * C::kKvBytes) >> 4);
        const uint32_t tp = tS + (t & 1) * kKvTile;
        // P (bf16, two keys per 32-bit column) sits in the first 64 columns of S
        // buffer t & 1; MMA kk takes the 16 keys of page kk of the V tile
        ptx::mma_ts(tO, tp, dv, kIdPV, t > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < kKvTile / 16; ++kk)
          ptx::mma_ts(tO, tp + kk * 8, dv + ((kk * C::kHeadBlock) >> 4), kIdPV, 1u);
        ptx::mma_commit(c.b(BE0 + s));
      }
      __syncwarp();
    }
    if (lane == 0) ptx::mma_commit(c.b(BDRAIN));  // arrives once this warp's MMAs are done
    __syncwarp();
    drain_wait(c, c.b(BDRAIN), 0);
    if (!p.test_stall) drain_wait(c, c.b(BQ), 0);  // the Q tile's copy (none was issued)
  } else if (warp >= 6 && p.gather) {
    // ------------------- K/V producers for 1-token pages: cp.async gathers
    // Every key is its own page, so a TMA box would carry one 128-byte row;
    // instead 64 threads per operand (warps 6-7: K, 8-9: V) copy whole key
    // rows in 16-byte pieces into the same swizzled layouts the TMA path
    // fills: K [panel][key][128 B], V [16-key block][panel][16 keys][128 B],
    // 16-byte chunk ch of row r at (ch ^ (r % 8)) * 16.  A thread commits one
    // copy group per tile and, once the group of the tile before has landed,
    // makes it visible to the tensor core (proxy fence) and arrives on that
    // tile's barrier (64 arrivals), keeping two tiles in flight.
    const int pr = warp - 6;
    const bool isK = pr < 2;
    const int tid = (pr & 1) * 32 + lane;
    const __nv_bfloat16* cache = isK ? p.kc : p.vc;
    const int NS = C::kKStages;
    const int full0 = isK ? BK0 : BV0, empty0 = isK ? BKE0 : BE0;
    constexpr int kKeysPer = kKvTile / 64;  // keys of a tile per thread
    constexpr int kChunks = D / 8;          // 16-byte pieces of a key row
    const size_t head_off = static_cast<size_t>(it.kv_head) * p.dr;
    const size_t page_elems = static_cast<size_t>(p.hkv) * p.dr;  // one token per page
    const int32_t* bt_row = p.bt + static_cast<size_t>(it.seg) * p.max_pages;
    // the block-table entries (one page per key) of tile t + 1 are read while
    // tile t's copies are issued, so the dependent load is off the copy path
    int raw_next[kKeysPer];
#pragma unroll
    for (int j = 0; j < kKeysPer; ++j) {
      const int pos = kv0 + tid + 64 * j;
      raw_next[j] = ntiles > 0 && pos < kv1 ? bt_row[pos] : -1;
    }
    int t = 0;
    for (; t < ntiles; ++t) {
      const int s = t % NS;
      int raw[kKeysPer];
#pragma unroll
      for (int j = 0; j < kKeysPer; ++j) {
        raw[j] = raw_next[j];
        const int pos = kv0 + (t + 1) * kKvTile + tid + 64 * j;
        raw_next[j] = t + 1 < ntiles && pos < kv1 ? bt_row[pos] : -1;
      }
      if (t >= NS && !wait_on(c, c.b(empty0 + s), ((t / NS) + 1) & 1)) break;
      const uint32_t stage = isK ? sK(s) : sV(s);
#pragma unroll
      for (int j = 0; j < kKeysPer; ++j) {
        const int key = tid + 64 * j;
        const int pos = kv0 + t * kKvTile + key;
        int page = -1;
        if (pos < kv1) {
          const int v = raw[j];
          if (v >= 0 && v < p.num_pages) page = v;
          else atomicOr(p.err, MCP_DEVERR_PAGE_RANGE);
        }
        const __nv_bfloat16* row =
            page >= 0 ? cache + static_cast<size_t>(page) * page_elems + head_off : cache;
        const uint32_t swz = static_cast<uint32_t>(key & 7);
        const uint32_t kbase = stage + key * 128;
        const uint32_t vbase = stage + (key >> 4) * C::kHeadBlock + (key & 15) * 128;
#pragma unroll
        for (int cc = 0; cc < kChunks; ++cc) {
          const int panel = cc >> 3;
          const uint32_t ch = static_cast<uint32_t>(cc & 7);
          const uint32_t dst = (isK ? kbase + panel * C::kKPanel : vbase + panel * kPageSize * 128) +
                               ((ch ^ swz) << 4);
          // keys past the item and columns past head_dim are written as zeros
          const bool in = page >= 0 && cc * 8 < p.dr;
          ptx::cp_async16(dst, in ? row + cc * 8 : cache, in ? 16u : 0u);
        }
      }
      ptx::cp_async_commit();
      if (t > 0) {
        ptx::cp_async_wait_group<1>();  // the copies of tile t - 1 have landed
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(c.b(full0 + (t - 1) % NS));
      }
    }
    ptx::cp_async_wait_group<0>();
    if (t > 0) {
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(c.b(full0 + (t - 1) % NS));
    }
  } else if (warp >= 6) {
    // -------------------------------------- K/V producers: four warps
    // warp 6: K boxes of keys 0-63, warp 7: K keys 64-127, warp 8: V keys 0-63,
    // warp 9: V keys 64-127.  A box holds B = 16 (or 8) tokens of one page.
    // A K tile arrives as one box per (box, 64-column panel) so that each
    // panel holds 128 consecutive keys (the K-major operand of Q K^T); a V tile
    // arrives as one box per box of tokens, [panel][B tokens][128 B], which
    // P V reads 16 keys per MMA.
    const int pr = warp - 6;
    const bool isK = pr < 2;
    const CUtensorMap* tm = isK ? tm_k : tm_v;
    const uint64_t pol = ptx::policy_evict_last();  // other q tiles re-read these K/V
    const int NS = C::kKStages;
    const int full0 = isK ? BK0 : BV0, empty0 = isK ? BKE0 : BE0;
    // the tile loop for boxes of B tokens; returns the tiles issued
    auto produce = [&](auto box_tok) -> int {
      constexpr int B = decltype(box_tok)::value;
      constexpr int kLog = B == 16 ? 4 : 3;
      constexpr int nu = (kKvTile / 2) / B;  // boxes of a tile this warp loads: 4 or 8
      const int u0 = (pr & 1) * nu;
      // the block-table entries of tile t + 1 are read while tile t is issued,
      // so that the dependent global load is off the stage-refill path
      auto fetch = [&](int tt) -> int {
        const int key0 = kv0 + tt * kKvTile;
        const int nbox = (kv1 - key0 + B - 1) >> kLog;  // boxes of the tile inside the item
        const bool mine = lane < nu && u0 + lane < nbox;
        return mine ? box_of(p, it.seg, (key0 >> kLog) + u0 + lane) : oob_block(p);
      };
      int pg_next = ntiles > 0 ? fetch(0) : oob_block(p);
      int t = 0;
      for (; t < ntiles; ++t) {
        const int s = t % NS;
        const int pg = pg_next;
        if (t + 1 < ntiles) pg_next = fetch(t + 1);
        if (t >= NS && !wait_on(c, c.b(empty0 + s), ((t / NS) + 1) & 1)) break;
        int pgs[nu];
#pragma unroll
        for (int i = 0; i < nu; ++i) pgs[i] = __shfl_sync(0xffffffffu, pg, i);
        if (lane == 0) {
          const uint32_t bar = c.b(full0 + s);
          ptx::mbar_arrive_expect_tx(bar, C::kKvBytes / 2);
          if (isK && B == 8 && p.k_box5) {
            // one box per 8 keys with every panel: [box][panel][8 keys][128 B]
            const uint32_t dst = sK(s);
#pragma unroll
            for (int i = 0; i < nu; ++i)
              ptx::tma_load_5d(dst + (u0 + i) * (C::kHalves * 1024), tm, bar, 0,
                               blk_tok(p, pgs[i]), 0, it.kv_head, blk_page(p, pgs[i]), pol);
          } else if (isK) {
            const uint32_t dst = sK(s);
#pragma unroll
            for (int i = 0; i < nu; ++i)
#pragma unroll
              for (int h = 0; h < C::kHalves; ++h)
                ptx::tma_load_4d(dst + h * C::kKPanel + (u0 + i) * B * 128, tm, bar, 64 * h,
                                 it.kv_head, blk_tok(p, pgs[i]), blk_page(p, pgs[i]), pol);
          } else {
            const uint32_t dst = sV(s);
#pragma unroll
            for (int i = 0; i < nu; ++i) {
              if (!p.panel_boxes) {
                ptx::tma_load_5d(dst + (u0 + i) * (C::kHalves * B * 128), tm, bar, 0,
                                 blk_tok(p, pgs[i]), 0, it.kv_head, blk_page(p, pgs[i]), pol);
              } else {  // one box per 64-column panel, same [panel][B tokens][128 B] layout
#pragma unroll
                for (int h = 0; h < C::kHalves; ++h)
                  ptx::tma_load_4d(dst + (u0 + i) * (C::kHalves * B * 128) + h * B * 128, tm, bar,
                                   64 * h, blk_tok(p, pgs[i]), it.kv_head, blk_page(p, pgs[i]),
                                   pol);
              }
            }
          }
        }
        __syncwarp();
      }
      return t;
    };
    const int t = p.box_log2 == 4 ? produce(std::integral_constant<int, 16>{})
                                  : produce(std::integral_constant<int, 8>{});
    // drain: the last tile this warp issued into each stage
    for (int s = 0; s < NS && s < t; ++s) {
      const int last = s + ((t - 1 - s) / NS) * NS;
      drain_wait(c, c.b(full0 + s), (last / NS) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ Q K^T issuer
    const uint32_t tS = tmem;              // S buffers
    const uint32_t tQ = tmem + C::kColQ;   // Q: D/2 columns, two bf16 per column
    // K tile layouts: one box per panel, [panel][128 keys][128 B] (8-key
    // groups 1024 B apart, panels kKPanel apart); or, with 8-token boxes of
    // every panel (p.k_box5), [box][panel][8 keys][128 B] (8-key groups one
    // box, kHalves KB, apart; panels 1 KB apart)
    const uint32_t k_group = p.k_box5 ? C::kHalves * 1024 : 1024;
    const uint32_t k_panel = p.k_box5 ? 1024 : C::kKPanel;
    const uint64_t dK0 = ptx::sdesc_sw128(sK(0), 16, k_group);
    bool ok = wait_on(c, c.b(BQT), 0);
    for (int t = 0; ok && t < ntiles; ++t) {
      const int s = t % C::kKStages;
      if (!(ok = wait_on(c, c.b(BK0 + s), (t / C::kKStages) & 1))) break;
      if (t >= 2) {
        // S buffer t & 1 still holds P(t - 2) until P V(t - 2) has read it
        const int ps = (t - 2) % C::kVStages;
        if (!(ok = wait_on(c, c.b(BE0 + ps), ((t - 2) / C::kVStages) & 1))) break;
      }
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint64_t dk = dK0 + static_cast<uint64_t>((s * C::kKvBytes) >> 4);
        const uint32_t ts = tS + (t & 1) * kKvTile;
        // A = Q from TMEM (loaded once per item), B = the K tile from shared memory
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_ts(ts, tQ + kk * 8, dk + (((kk >> 2) * k_panel + (kk & 3) * 32) >> 4), kIdQK,
                      kk > 0 ? 1u : 0u);
        ptx::mma_commit(c.b(BS0 + (t & 1)));
        ptx::mma_commit(c.b(BKE0 + s));
      }
      __syncwarp();
    }
    if (lane == 0) ptx::mma_commit(c.b(BDRAIN));
    __syncwarp();
    drain_wait(c, c.b(BDRAIN), 0);
  } else {
    // ------------------------------------------- softmax + epilogue (2-5)
    const int qw = warp & 3;
    const int row = qw * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    const uint32_t tS = tmem + lane_base;
    const uint32_t tO = tmem + C::kColO + lane_base;
    const int tok = it.q_begin + row / G;  // token index inside the segment
    const int g = row - (row / G) * G;
    const bool valid = row < G * TQ && tok < it.q_begin + it.q_count;
    const int tok_c = tok < it.q_begin + it.q_count ? tok : it.q_begin + it.q_count - 1;
    // right-aligned causal: token i sees keys 0 .. hist + i; the item covers keys < kv1
    int jmax = sg.hist + tok_c;
    jmax = jmax < kv1 - 1 ? jmax : kv1 - 1;
    const float sl2 = p.scale_log2;
    float m_ref = neg_inf(), l = 0.f;
    bool ok = wait_on_warp(c, c.b(BQ), 0);
    {
      // Q is read for every KV tile: move this thread's row from the swizzled
      // shared-memory tile into TMEM (K-major, two bf16 per column) once, so
      // Q K^T runs with A in TMEM and only K read from shared memory.
      uint32_t qv[D / 2];
      const uint8_t* qrow = gb + C::kOffQ + row * 128;
#pragma unroll
      for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 v = *reinterpret_cast<const uint4*>(qrow + h * C::kQPanel + ((ch ^ (row & 7)) << 4));
          qv[h * 32 + ch * 4 + 0] = v.x;
          qv[h * 32 + ch * 4 + 1] = v.y;
          qv[h * 32 + ch * 4 + 2] = v.z;
          qv[h * 32 + ch * 4 + 3] = v.w;
        }
#pragma unroll
      for (int j = 0; j < D / 64; ++j) ptx::tmem_st32(tmem + C::kColQ + lane_base + j * 32, qv + j * 32);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.b(BQT));
    }
    for (int t = 0; ok && t < ntiles; ++t) {
      const int s = t & 1;
      if (!(ok = wait_on_warp(c, c.b(BS0 + s), (t >> 1) & 1))) break;
      ptx::tc_fence_after();
      // the scores, and the max of each 32 of them from the load itself
      uint32_t r[kKvTile];
      float mj[kKvTile / 32];
#pragma unroll
      for (int j = 0; j < kKvTile / 32; ++j) ptx::tmem_ld32_max(tS + s * kKvTile + j * 32, r + j * 32, mj[j]);
#pragma unroll
      for (int j = 0; j < kKvTile / 32; ++j) ptx::tmem_wait_ld_dep_max(r + j * 32, mj[j]);
      const int key0 = kv0 + t * kKvTile;
      // max of the raw scores (sm_scale > 0 keeps the order)
      float mx;
      if (key0 + kKvTile - 1 <= jmax) {  // every key of the tile is visible to this row
        mx = kKvTile == 128 ? fmaxf(fmaxf(mj[0], mj[1]), fmaxf(mj[kKvTile / 32 - 2], mj[kKvTile / 32 - 1]))
                            : fmaxf(mj[0], mj[kKvTile / 32 - 1]);
      } else {  // diagonal / last tile: mask keys past this row's last visible key
        float mxp[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) mxp[j] = neg_inf();
#pragma unroll
        for (int i = 0; i < kKvTile; ++i) {
          const float x = (key0 + i <= jmax) ? __uint_as_float(r[i]) : neg_inf();
          r[i] = __float_as_uint(x);
          mxp[i & 7] = fmaxf(mxp[i & 7], x);
        }
        mx = ptx::max3(ptx::max3(mxp[0], mxp[1], mxp[2]), ptx::max3(mxp[3], mxp[4], mxp[5]),
                       fmaxf(mxp[6], mxp[7]));
      }
      const float m_new = fmaxf(m_ref, mx * sl2);
      const bool rescale = m_new > m_ref + kRescaleThreshold;
      float alpha = 1.f;
      if (rescale) {
        alpha = ptx::ex2(m_ref - m_new);
        m_ref = m_new;
      }
      const float neg_m = m_ref == neg_inf() ? 0.f : -m_ref;
      // P = 2^(s * scale_log2 - m).  bf16 pairs of P overwrite the consumed
      // scores in place: r[i/2] after r[i], r[i+1]; the row sum runs in eight
      // independent chains, two per packed add.
      float sp[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) sp[j] = 0.f;
#pragma unroll
      for (int i = 0; i < kKvTile; i += 2) {
        float x0, x1;
        ptx::fma_f32x2(x0, x1, __uint_as_float(r[i]), __uint_as_float(r[i + 1]), sl2, neg_m);
        const float p0 = ptx::ex2(x0);
        const float p1 = ptx::ex2(x1);
        const int j = (i >> 1) & 3;
        ptx::add_f32x2(sp[2 * j], sp[2 * j + 1], p0, p1);
        r[i / 2] = ptx::pack_bf16x2(p0, p1);
      }
      const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      l = l * alpha + sum;
      // P(t) goes to the first 64 columns of S buffer t & 1 (this thread's lane,
      // already read); P V(t-1) reads the other buffer, so no wait is needed here
#pragma unroll
      for (int j = 0; j < kKvTile / 64; ++j) ptx::tmem_st32(tS + s * kKvTile + j * 32, r + j * 32);
      if (t > 0 && __any_sync(0xffffffffu, rescale)) {
        // P V of the previous tile (issued by the other MMA warp) must be done
        // before O is rescaled; its barrier (V stage (t-1) % kVStages) completes
        // next only with P V(t-1+kVStages), which needs P of that tile, so it
        // is at most one phase off.
        const int ps = (t - 1) % C::kVStages;
        if (!(ok = wait_on_warp(c, c.b(BE0 + ps), ((t - 1) / C::kVStages) & 1))) break;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < D / 32; ++j) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + j * 32, o);
          ptx::tmem_wait_ld();
          if (rescale) {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          }
          ptx::tmem_st32(tO + j * 32, o);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.b(BP0 + (t & 1)));
    }
    // every MMA of the item (each issuing warp commits once after its last MMA)
    if (ok && ntiles > 0) ok = wait_on_warp(c, c.b(BDRAIN), 0);
    ptx::tc_fence_after();
    const bool store = ok && valid && !*c.abort;
    const bool direct = it.part_row < 0;
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    const size_t orow = static_cast<size_t>(sg.q_start + tok) * p.hq + it.kv_head * G + g;
#pragma unroll 1
    for (int j = 0; j < D / 32; ++j) {
      uint32_t o[32];
      ptx::tmem_ld32(tO + j * 32, o);
      ptx::tmem_wait_ld();
      if (store && j * 32 < p.dr) {  // columns past the tensors' head_dim are not stored
        if (direct) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow * p.dr + j * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            dst[v] = make_uint4(
                ptx::pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l),
                ptx::pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l),
                ptx::pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l),
                ptx::pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l));
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.part_o + static_cast<size_t>(it.part_row + row) * p.dr + j * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                 __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
        }
      }
    }
    if (store) {
      const float lse = l > 0.f ? (m_ref + log2f(l)) * kLn2 : neg_inf();
      if (direct) {
        if (p.lse) p.lse[orow] = lse;
      } else {
        p.part_lse[it.part_row + row] = lse;
      }
    }
  }
}

// ------------------------------------------------------------------------
// decode item: whole-page TMA ring + mma.sync, one warp per kv head
// ------------------------------------------------------------------------
__device__ __forceinline__ uint32_t keep_pair(uint32_t v, int k, int nvalid) {
  const uint32_t lo = k < nvalid ? 0x0000FFFFu : 0u;
  const uint32_t hi = k + 1 < nvalid ? 0xFFFF0000u : 0u;
  return v & (lo | hi);
}

// The last step of a decode item whose head is shared by several warps: warp
// (hw, po = 0) merges the warps' (m, l, O) states of head hw, left in shared
// memory as mo [8 warps][16 rows][D], mm and ml [8 warps][16 rows], and writes
// the rows (lane -> row lane % 16, columns half lane / 16).
template <int D>
__device__ __forceinline__ void merge_rows(const KParams& p, const WorkItem& it, const Seg& sg,
                                           const float* mo, const float* mm, const float* ml,
                                           int hw, int HG, int ps, int head, int R, int lane) {
  const int G = p.G;
  const bool direct = it.part_row < 0;
  const int r = lane & 15;
  if (r >= R) return;
  const int d0 = (lane >> 4) * (D / 2);
  float M = neg_inf();
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < ps) M = fmaxf(M, mm[(hw + k * HG) * 16 + r]);
  float wt[8], L = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    wt[k] = 0.f;
    if (k < ps) {
      const float mk = mm[(hw + k * HG) * 16 + r];
      wt[k] = mk == neg_inf() ? 0.f : ptx::ex2(mk - M);
      L += wt[k] * ml[(hw + k * HG) * 16 + r];
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int tok = it.q_begin + r / G;
  const int g = r - (r / G) * G;
  const size_t orow = static_cast<size_t>(sg.q_start + tok) * p.hq + head * G + g;
  for (int d = 0; d < D / 2 && d0 + d < p.dr; d += 4) {
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k >= ps) break;
      const float4 v = *reinterpret_cast<const float4*>(mo + ((hw + k * HG) * 16 + r) * D + d0 + d);
      a[0] += wt[k] * v.x;
      a[1] += wt[k] * v.y;
      a[2] += wt[k] * v.z;
      a[3] += wt[k] * v.w;
    }
    if (direct) {
      uint2 pk2 = make_uint2(ptx::pack_bf16x2(a[0] * inv, a[1] * inv), ptx::pack_bf16x2(a[2] * inv, a[3] * inv));
      *reinterpret_cast<uint2*>(p.out + orow * p.dr + d0 + d) = pk2;
    } else {
      *reinterpret_cast<float4*>(p.part_o + static_cast<size_t>(it.part_row + hw * it.part_head_stride + r) * p.dr + d0 + d) =
          make_float4(a[0] * inv, a[1] * inv, a[2] * inv, a[3] * inv);
    }
  }
  if (lane < 16) {
    const float lse = L > 0.f ? (M + log2f(L)) * kLn2 : neg_inf();
    if (direct) {
      if (p.lse) p.lse[orow] = lse;
    } else {
      p.part_lse[it.part_row + hw * it.part_head_stride + r] = lse;
    }
  }
}


// Decode consumer for at most 8 query rows of a kv head (G * Lq <= 8: every
// plain decode with G <= 8).  The scores are taken transposed, S^T = K Q^T,
// with m16n8k16: 16 keys fill M and the query rows N = 8, so one MMA covers
// 16 keys per 16 dims (rows in M would leave 8 of 16 rows empty at G = 8 and
// 12 at G = 4).  Likewise O^T = V^T P^T: 16 dims in M, the rows in N.  The
// MMA count per page is half the row-major form's, and so are the
// accumulator and Q registers.  P^T, the B operand of the second product, is
// moved from the score layout (lane holds keys gid, gid + 8 of rows 2 tig,
// 2 tig + 1) to the B layout (lane holds row gid, keys 2 tig, +1, +8, +9)
// with four shuffles.
template <int D>
__device__ __forceinline__ void decode_n8(const Ctx& c, const WorkItem& it, const Seg& sg,
                                          const KParams& p, uint8_t* gb, uint32_t ring, int NS,
                                          int stage_bytes, int block, int box_bytes, int npg,
                                          int HG, int hw, int ps, int po, int cw, int lane) {
  const int G = p.G;
  const int B = 1 << p.box_log2;
  const int kv0 = it.kv_begin, kv1 = it.kv_end;
  const int head = it.kv_head + hw;
  const int gid = lane >> 2, tig = lane & 3;
  const int R = it.q_count * G;
  const int last_tok = it.q_count - 1;
  const float sl2 = p.scale_log2;
  // rows of the C fragments: 2 tig and 2 tig + 1; their last visible key
  int jm[2];
  bool rv[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int r = 2 * tig + e;
    rv[e] = r < R;
    const int tk = r / G < last_tok ? r / G : last_tok;
    jm[e] = min(sg.hist + it.q_begin + tk, kv1 - 1);
  }
  // Q^T as B fragments: lane holds row gid, dims 16 kk + 2 tig (+1) and + 8 (+9)
  uint32_t qb[D / 16][2];
  {
    const bool vr = gid < R;
    const uint32_t* qr = reinterpret_cast<const uint32_t*>(
        p.q + (static_cast<size_t>(sg.q_start + it.q_begin + (vr ? gid / G : 0)) * p.hq + head * G +
               (vr ? gid % G : 0)) * p.dr);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const bool in = vr && kk * 16 < p.dr;  // columns past the tensors' head_dim are 0
      qb[kk][0] = in ? qr[kk * 8 + tig] : 0u;
      qb[kk][1] = in ? qr[kk * 8 + 4 + tig] : 0u;
    }
  }
  float o[D / 16][4];  // O^T: dims 16 mt + gid (+8) x rows 2 tig (+1)
#pragma unroll
  for (int i = 0; i < D / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m[2] = {neg_inf(), neg_inf()}, l[2] = {0.f, 0.f};
  bool ok = true;
  const int mi = lane >> 3, rr = lane & 7;
  const int hstr = p.panel_boxes ? B * 128 : Cfg<D>::kHalves * B * 128;  // between heads
  const uint32_t pstr = static_cast<uint32_t>(p.panel_boxes ? HG * B * 128 : B * 128);  // panels
  auto row_off = [&](int tk) -> uint32_t {
    return static_cast<uint32_t>((tk >> p.box_log2) * box_bytes + hw * hstr + (tk & (B - 1)) * 128);
  };
  // ldmatrix rows: K as A (keys x dims): matrices (keys 0-7, c) (8-15, c) (0-7, c+1) (8-15, c+1);
  // V^T as A via .trans of V (keys x dims): (keys 0-7, c) (0-7, c+1) (8-15, c) (8-15, c+1)
  const uint32_t offK = row_off((mi & 1) * 8 + rr);
  const int chK = mi >> 1;
  const uint32_t offV = row_off((mi >> 1) * 8 + rr);
  const int chV = mi & 1;
  // P^T gather sources: keys 2 tig and 2 tig + 1 of row gid
  const int srcA = 4 * (2 * tig) + (gid >> 1), srcB = 4 * (2 * tig + 1) + (gid >> 1);
  const bool odd_row = gid & 1;
  for (int pi = po; pi < npg; pi += ps) {
    const int s = pi % NS;
    if (!(ok = wait_on(c, c.b(BFULL0 + s), (pi / NS) & 1))) break;
    const uint32_t kb = ring + s * stage_bytes;
    const uint32_t vb = kb + block;
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int h = kk >> 2, c0 = (kk & 3) * 2;
      uint32_t a[4];
      ptx::ldsm_x4(kb + offK + h * pstr + (((c0 + chK) ^ rr) << 4), a[0], a[1], a[2], a[3]);
      ptx::mma16816((kk & 1) ? sb : sa, a, qb[kk][0], qb[kk][1]);
    }
    const int key0 = kv0 + pi * kPageSize;
    // x[e]: keys gid (e = 0, 1) and gid + 8 (e = 2, 3), rows 2 tig + (e & 1)
    float x[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = key0 + gid + (e >> 1) * 8;
      x[e] = rv[e & 1] && key <= jm[e & 1] ? (sa[e] + sb[e]) * sl2 : neg_inf();
    }
    float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
      mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
    }
    float u[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float nm = fmaxf(m[e], mx[e]);
      if (nm > m[e] + kRescaleThreshold) {
        const float a = ptx::ex2(m[e] - nm);
        m[e] = nm;
        l[e] *= a;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) { o[i][e] *= a; o[i][2 + e] *= a; }
      }
      u[e] = m[e] == neg_inf() ? 0.f : m[e];
    }
    float pv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pv[e] = ptx::ex2(x[e] - u[e & 1]);
    l[0] += pv[0] + pv[2];
    l[1] += pv[1] + pv[3];
    // P^T to the B layout: row gid, keys 2 tig (+1) in b0 and 2 tig + 8 (+9) in b1
    const uint32_t pe = ptx::pack_bf16x2(pv[0], pv[2]);  // row 2 tig:     keys gid, gid + 8
    const uint32_t po_ = ptx::pack_bf16x2(pv[1], pv[3]); // row 2 tig + 1: keys gid, gid + 8
    const uint32_t ae = __shfl_sync(0xffffffffu, pe, srcA), ao = __shfl_sync(0xffffffffu, po_, srcA);
    const uint32_t be = __shfl_sync(0xffffffffu, pe, srcB), bo = __shfl_sync(0xffffffffu, po_, srcB);
    const uint32_t va = odd_row ? ao : ae;  // keys 2 tig, 2 tig + 8 of row gid
    const uint32_t vb2 = odd_row ? bo : be; // keys 2 tig + 1, 2 tig + 9
    const uint32_t b0 = (va & 0xFFFFu) | (vb2 << 16);
    const uint32_t b1 = (va >> 16) | (vb2 & 0xFFFF0000u);
    const int nvalid = kv1 - key0;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      const int h = mt >> 2, c0 = (mt & 3) * 2;
      uint32_t a[4];
      ptx::ldsm_x4_t(vb + offV + h * pstr + (((c0 + chV) ^ rr) << 4), a[0], a[1], a[2], a[3]);
      if (nvalid < kPageSize) {
        // keys past the item's end: unused slots may hold NaN; P is 0 there
        a[0] = keep_pair(a[0], tig * 2, nvalid);
        a[1] = keep_pair(a[1], tig * 2, nvalid);
        a[2] = keep_pair(a[2], 8 + tig * 2, nvalid);
        a[3] = keep_pair(a[3], 8 + tig * 2, nvalid);
      }
      ptx::mma16816(o[mt], a, b0, b1);
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(c.b(BEMPTY0 + s));
  }
  // full row sums over the eight lanes of each row (gid)
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    l[e] += __shfl_xor_sync(0xffffffffu, l[e], 4);
    l[e] += __shfl_xor_sync(0xffffffffu, l[e], 8);
    l[e] += __shfl_xor_sync(0xffffffffu, l[e], 16);
  }
  const bool direct = it.part_row < 0;
  if (ps == 1) {
    // this warp alone saw its head's whole KV range: write from the fragments
    if (!ok || *c.abort) return;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 2 * tig + e;
      if (r >= R) continue;
      const int tok = it.q_begin + r / G;
      const int g = r - (r / G) * G;
      const float inv = l[e] > 0.f ? 1.f / l[e] : 0.f;
      const size_t orow = static_cast<size_t>(sg.q_start + tok) * p.hq + head * G + g;
      if (direct) {
        __nv_bfloat16* dst = p.out + orow * p.dr;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d0 = mt * 16 + gid;
          if (d0 < p.dr) dst[d0] = __float2bfloat16_rn(o[mt][e] * inv);
          if (d0 + 8 < p.dr) dst[d0 + 8] = __float2bfloat16_rn(o[mt][2 + e] * inv);
        }
      } else {
        float* dst = p.part_o + static_cast<size_t>(it.part_row + hw * it.part_head_stride + r) * p.dr;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int d0 = mt * 16 + gid;
          if (d0 < p.dr) dst[d0] = o[mt][e] * inv;
          if (d0 + 8 < p.dr) dst[d0 + 8] = o[mt][2 + e] * inv;
        }
      }
      if (gid == 0) {
        const float lse = l[e] > 0.f ? (m[e] + log2f(l[e])) * kLn2 : neg_inf();
        if (direct) {
          if (p.lse) p.lse[orow] = lse;
        } else {
          p.part_lse[it.part_row + hw * it.part_head_stride + r] = lse;
        }
      }
    }
    return;
  }
  // several warps per head: merge their (m, l, O) through shared memory, in the
  // layout of the 16-row consumer ([warp][16 rows][D]; rows 8-15 unused)
  asm volatile("bar.sync 1, 256;" ::: "memory");
  float* mo = reinterpret_cast<float*>(gb);
  float* mm = mo + 8 * 16 * D;
  float* ml = mm + 8 * 16;
  float* mine = mo + cw * 16 * D;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int r = 2 * tig + e;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      mine[r * D + mt * 16 + gid] = o[mt][e];
      mine[r * D + mt * 16 + gid + 8] = o[mt][2 + e];
    }
    if (gid == 0) {
      mm[cw * 16 + r] = m[e];
      ml[cw * 16 + r] = l[e];
    }
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (po != 0 || !ok || *c.abort) return;
  merge_rows<D>(p, it, sg, mo, mm, ml, hw, HG, ps, head, R, lane);
}

template <int D>
__device__ __forceinline__ void decode_item(const Ctx& c, const WorkItem& it, const Seg& sg,
                                            const KParams& p, uint32_t base, uint8_t* gb,
                                            const CUtensorMap* tm_kd, const CUtensorMap* tm_vd,
                                            int warp, int lane) {
  using C = Cfg<D>;
  const int G = p.G;
  const int HG = it.num_heads;                 // kv heads of the group (1, 2, 4 or 8)
  const int kv0 = it.kv_begin, kv1 = it.kv_end;
  const int npg = (kv1 - kv0 + kPageSize - 1) / kPageSize;
  const int NS = p.dec_stages;
  const int block = HG * C::kHeadBlock;        // K (or V) bytes of 16 tokens for the group
  const int stage_bytes = 2 * block;
  const uint32_t ring = base;
  // a stage holds 16 tokens: one box of 16 or two boxes of 8, each box laid
  // out [head][panel][B tokens][128 B]
  const int B = 1 << p.box_log2;
  const int ups = kPageSize >> p.box_log2;    // boxes per stage: 1 or 2
  const int box_bytes = block / ups;

  // Two producer warps: warp 0 loads the K half of every stage, warp 1 the V
  // half (each arrives on the stage's barrier with its bytes).  One warp
  // issues its TMA boxes one after another, and a single producer capped one
  // CTA's stream near 100 GB/s.
  if (warp < 2) {
    const bool isV = warp == 1;
    const CUtensorMap* tm = isV ? tm_vd : tm_kd;
    const uint32_t half_off = isV ? static_cast<uint32_t>(block) : 0u;
    const uint64_t pol = ptx::policy_evict_first();  // each page is read once
    int issued = 0;
    bool ok = true;
    const int nbox = (kv1 - kv0 + B - 1) >> p.box_log2;  // boxes inside the item
    const int per_batch = 32 / ups;                      // stages whose box ids one fetch covers
    for (int b0 = 0; ok && b0 < npg; b0 += per_batch) {
      const int n = npg - b0 < per_batch ? npg - b0 : per_batch;
      const int ub = b0 * ups + lane;                    // box (inside the item) of this lane
      const int pg = lane < n * ups && ub < nbox ? box_of(p, it.seg, (kv0 >> p.box_log2) + ub)
                                                  : oob_block(p);
      for (int i = 0; i < n; ++i) {
        const int pi = b0 + i;
        const int s = pi % NS;
        if (pi >= NS && !(ok = wait_on(c, c.b(BEMPTY0 + s), ((pi / NS) + 1) & 1))) break;
        const int pga = __shfl_sync(0xffffffffu, pg, i * ups);
        const int pgb = __shfl_sync(0xffffffffu, pg, i * ups + ups - 1);
        if (lane == 0) {
          const uint32_t dst = ring + s * stage_bytes + half_off;
          ptx::mbar_arrive_expect_tx(c.b(BFULL0 + s), block);
          for (int j = 0; j < ups; ++j) {
            const int pgi = j ? pgb : pga;
            const int tok = blk_tok(p, pgi), pgp = blk_page(p, pgi);
            if (!p.panel_boxes) {  // [head][panel][B tokens][128 B]
              ptx::tma_load_5d(dst + j * box_bytes, tm, c.b(BFULL0 + s), 0, tok, 0, it.kv_head, pgp,
                               pol);
            } else {  // one box per panel: [panel][head][B tokens][128 B]
              for (int h = 0; h < C::kHalves; ++h)
                ptx::tma_load_4d(dst + j * box_bytes + h * HG * B * 128, tm, c.b(BFULL0 + s),
                                 64 * h, tok, it.kv_head, pgp, pol);
            }
          }
        }
        __syncwarp();
        issued = pi + 1;
      }
    }
    for (int s = 0; s < NS && s < issued; ++s) {
      const int last = s + ((issued - 1 - s) / NS) * NS;
      drain_wait(c, c.b(BFULL0 + s), (last / NS) & 1);
    }
    return;
  }

  // ---------------------------------------------------- consumers (2-9)
  const int cw = warp - 2;
  const int hw = cw % HG;        // kv head (within the group) of this warp
  const int ps = 8 / HG;         // warps sharing that head
  const int po = cw / HG;        // this warp takes pages po, po + ps, ...
  if (it.q_count * G <= 8) {
    decode_n8<D>(c, it, sg, p, gb, ring, NS, stage_bytes, block, box_bytes, npg, HG, hw, ps, po, cw,
                 lane);
    return;
  }
  const int head = it.kv_head + hw;
  const int gid = lane >> 2, tig = lane & 3;
  const int R = it.q_count * G;
  const int last_tok = it.q_count - 1;
  const int tl = gid / G < last_tok ? gid / G : last_tok;
  const int th = (gid + 8) / G < last_tok ? (gid + 8) / G : last_tok;
  const int jlo = min(sg.hist + it.q_begin + tl, kv1 - 1);
  const int jhi = min(sg.hist + it.q_begin + th, kv1 - 1);
  const bool vlo = gid < R, vhi = gid + 8 < R;
  const float sl2 = p.scale_log2;

  // Q rows (row r = token r / G, head r % G of this kv head) as m16n8k16 A fragments
  uint32_t qa[D / 16][4];
  {
    const uint32_t* qlo = reinterpret_cast<const uint32_t*>(
        p.q + (static_cast<size_t>(sg.q_start + it.q_begin + gid / G) * p.hq + head * G + gid % G) * p.dr);
    const uint32_t* qhi = reinterpret_cast<const uint32_t*>(
        p.q + (static_cast<size_t>(sg.q_start + it.q_begin + (gid + 8) / G) * p.hq + head * G +
               (gid + 8) % G) * p.dr);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const bool in = kk * 16 < p.dr;  // columns past the tensors' head_dim are 0
      qa[kk][0] = vlo && in ? qlo[kk * 8 + tig] : 0u;
      qa[kk][1] = vhi && in ? qhi[kk * 8 + tig] : 0u;
      qa[kk][2] = vlo && in ? qlo[kk * 8 + 4 + tig] : 0u;
      qa[kk][3] = vhi && in ? qhi[kk * 8 + 4 + tig] : 0u;
    }
  }
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mlo = neg_inf(), mhi = neg_inf(), llo = 0.f, lhi = 0.f;
  bool ok = true;
  const int mi = lane >> 3, rr = lane & 7;
  // byte offset of stage row tk (0-15) of this warp's head inside a K or V
  // half-stage, and the stride between 64-column panels
  const int hstr = p.panel_boxes ? B * 128 : C::kHalves * B * 128;  // between heads
  const uint32_t pstr = static_cast<uint32_t>(p.panel_boxes ? HG * B * 128 : B * 128);  // panels
  auto row_off = [&](int tk) -> uint32_t {
    return static_cast<uint32_t>((tk >> p.box_log2) * box_bytes + hw * hstr + (tk & (B - 1)) * 128);
  };
  const uint32_t offK = row_off((mi >> 1) * 8 + rr);  // ldmatrix rows of the K fragments
  const uint32_t offV = row_off((mi & 1) * 8 + rr);   // and of the transposed V fragments
  for (int pi = po; pi < npg; pi += ps) {
    const int s = pi % NS;
    if (!(ok = wait_on(c, c.b(BFULL0 + s), (pi / NS) & 1))) break;
    const uint32_t kb = ring + s * stage_bytes;
    const uint32_t vb = kb + block;
    // two independent accumulator chains (even / odd k-steps) halve the MMA latency chain
    float sa[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float sb[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int h = kk >> 2, c0 = (kk & 3) * 2;
      // matrices: (tok 0-7, c0) (0-7, c0+1) (8-15, c0) (8-15, c0+1)
      const int ch = c0 + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ptx::ldsm_x4(kb + offK + h * pstr + ((ch ^ rr) << 4), b0, b1, b2, b3);
      float(*acc)[4] = (kk & 1) ? sb : sa;
      ptx::mma16816(acc[0], qa[kk], b0, b1);
      ptx::mma16816(acc[1], qa[kk], b2, b3);
    }
    const int key0 = kv0 + pi * kPageSize;
    float x[2][4];
    float xlo = neg_inf(), xhi = neg_inf();
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = key0 + nt * 8 + tig * 2 + e;
        x[nt][e] = key <= jlo ? (sa[nt][e] + sb[nt][e]) * sl2 : neg_inf();
        x[nt][2 + e] = key <= jhi ? (sa[nt][2 + e] + sb[nt][2 + e]) * sl2 : neg_inf();
        xlo = fmaxf(xlo, x[nt][e]);
        xhi = fmaxf(xhi, x[nt][2 + e]);
      }
    xlo = fmaxf(xlo, __shfl_xor_sync(0xffffffffu, xlo, 1));
    xlo = fmaxf(xlo, __shfl_xor_sync(0xffffffffu, xlo, 2));
    xhi = fmaxf(xhi, __shfl_xor_sync(0xffffffffu, xhi, 1));
    xhi = fmaxf(xhi, __shfl_xor_sync(0xffffffffu, xhi, 2));
    const float nlo = fmaxf(mlo, xlo), nhi = fmaxf(mhi, xhi);
    if (nlo > mlo + kRescaleThreshold) {
      const float a = ptx::ex2(mlo - nlo);
      mlo = nlo;
      llo *= a;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) { o[i][0] *= a; o[i][1] *= a; }
    }
    if (nhi > mhi + kRescaleThreshold) {
      const float a = ptx::ex2(mhi - nhi);
      mhi = nhi;
      lhi *= a;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) { o[i][2] *= a; o[i][3] *= a; }
    }
    const float ulo = mlo == neg_inf() ? 0.f : mlo;
    const float uhi = mhi == neg_inf() ? 0.f : mhi;
    float pv[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      pv[nt][0] = ptx::ex2(x[nt][0] - ulo);
      pv[nt][1] = ptx::ex2(x[nt][1] - ulo);
      pv[nt][2] = ptx::ex2(x[nt][2] - uhi);
      pv[nt][3] = ptx::ex2(x[nt][3] - uhi);
      llo += pv[nt][0] + pv[nt][1];
      lhi += pv[nt][2] + pv[nt][3];
    }
    uint32_t pa[4] = {ptx::pack_bf16x2(pv[0][0], pv[0][1]), ptx::pack_bf16x2(pv[0][2], pv[0][3]),
                      ptx::pack_bf16x2(pv[1][0], pv[1][1]), ptx::pack_bf16x2(pv[1][2], pv[1][3])};
    const int nvalid = kv1 - key0;
#pragma unroll
    for (int dd = 0; dd < D / 16; ++dd) {
      const int h = dd >> 2, c0 = (dd & 3) * 2;
      // matrices: (tok 0-7, c0) (8-15, c0) (0-7, c0+1) (8-15, c0+1)
      const int ch = c0 + (mi >> 1);
      uint32_t v0, v1, v2, v3;
      ptx::ldsm_x4_t(vb + offV + h * pstr + ((ch ^ rr) << 4), v0, v1, v2, v3);
      if (nvalid < kPageSize) {
        // keys past the item's end: unused slots may hold NaN; P is 0 there
        v0 = keep_pair(v0, tig * 2, nvalid);
        v1 = keep_pair(v1, 8 + tig * 2, nvalid);
        v2 = keep_pair(v2, tig * 2, nvalid);
        v3 = keep_pair(v3, 8 + tig * 2, nvalid);
      }
      ptx::mma16816(o[2 * dd], pa, v0, v1);
      ptx::mma16816(o[2 * dd + 1], pa, v2, v3);
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(c.b(BEMPTY0 + s));
  }
  // full row sums inside each quad
  llo += __shfl_xor_sync(0xffffffffu, llo, 1);
  llo += __shfl_xor_sync(0xffffffffu, llo, 2);
  lhi += __shfl_xor_sync(0xffffffffu, lhi, 1);
  lhi += __shfl_xor_sync(0xffffffffu, lhi, 2);

  const bool direct = it.part_row < 0;
  if (ps == 1) {
    // this warp alone saw its head's whole KV range: write from the fragments
    if (!ok || *c.abort) return;
    const float ilo = llo > 0.f ? 1.f / llo : 0.f;
    const float ihi = lhi > 0.f ? 1.f / lhi : 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = gid + 8 * half;
      if (r >= R) continue;
      const int tok = it.q_begin + r / G;
      const int g = r - (r / G) * G;
      const float inv = half ? ihi : ilo;
      const size_t orow = static_cast<size_t>(sg.q_start + tok) * p.hq + head * G + g;
      if (direct) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + orow * p.dr);
#pragma unroll
        for (int nb = 0; nb < D / 8; ++nb)
          if (nb * 8 < p.dr)
            dst[(nb * 8 + tig * 2) / 2] = ptx::pack_bf16x2(o[nb][2 * half] * inv, o[nb][2 * half + 1] * inv);
      } else {
        float* dst = p.part_o + static_cast<size_t>(it.part_row + hw * it.part_head_stride + r) * p.dr;
#pragma unroll
        for (int nb = 0; nb < D / 8; ++nb)
          if (nb * 8 < p.dr)
            *reinterpret_cast<float2*>(dst + nb * 8 + tig * 2) =
                make_float2(o[nb][2 * half] * inv, o[nb][2 * half + 1] * inv);
      }
      if (tig == 0) {
        const float m = half ? mhi : mlo;
        const float L = half ? lhi : llo;
        const float lse = L > 0.f ? (m + log2f(L)) * kLn2 : neg_inf();
        if (direct) {
          if (p.lse) p.lse[orow] = lse;
        } else {
          p.part_lse[it.part_row + hw * it.part_head_stride + r] = lse;
        }
      }
    }
    return;
  }
  // several warps per head: merge their (m, l, O) through shared memory.  The
  // ring is idle once every consumer warp has passed the first barrier.
  asm volatile("bar.sync 1, 256;" ::: "memory");
  float* mo = reinterpret_cast<float*>(gb);           // [8 warps][16 rows][D]
  float* mm = mo + 8 * 16 * D;                         // [8 warps][16 rows]
  float* ml = mm + 8 * 16;
  float* mine = mo + cw * 16 * D;
#pragma unroll
  for (int nb = 0; nb < D / 8; ++nb) {
    *reinterpret_cast<float2*>(mine + gid * D + nb * 8 + tig * 2) = make_float2(o[nb][0], o[nb][1]);
    *reinterpret_cast<float2*>(mine + (gid + 8) * D + nb * 8 + tig * 2) = make_float2(o[nb][2], o[nb][3]);
  }
  if (tig == 0) {
    mm[cw * 16 + gid] = mlo;
    mm[cw * 16 + gid + 8] = mhi;
    ml[cw * 16 + gid] = llo;
    ml[cw * 16 + gid + 8] = lhi;
  }
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (po != 0 || !ok || *c.abort) return;
  merge_rows<D>(p, it, sg, mo, mm, ml, hw, HG, ps, head, R, lane);
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    mixed_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_kd,
                          const __grid_constant__ CUtensorMap tm_vd, const KParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem it = p.items[blockIdx.x];
  Ctx c;
  c.bar = base + C::kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + C::kOffBar + kNumBars * 8);
  c.abort = reinterpret_cast<volatile int*>(gb + C::kOffBar + kNumBars * 8 + 16);
  c.err = p.err;
  c.limit_ns = p.test_stall ? kTestWaitLimitNs : kWaitLimitNs;
  const bool prefill = it.kind == kPrefillItem;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;
      if (i >= BK0 && i < BV0 + 3) count = p.gather ? 64 : 2;  // producer warps (threads) per tile
      if (i == BP0 || i == BP0 + 1 || i == BQT) count = 128;  // every softmax thread
      if (i == BDRAIN) count = 2;                       // the Q K^T and the P V issuer
      if (i >= BEMPTY0) count = prefill ? 1 : it.num_heads;  // one warp per head reads a stage
      // a decode stage: the K-half and the V-half producer warps arrive
      if (!prefill && i >= BFULL0 && i < BFULL0 + kMaxDecStages) count = 2;
      ptx::mbar_init(c.b(i), count);
    }
    *c.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (prefill) {
      ptx::prefetch_tmap(&tm_q);
    } else {
      ptx::prefetch_tmap(&tm_kd);
      ptx::prefetch_tmap(&tm_vd);
    }
  }
  if (prefill && warp >= 6 && lane == 0) ptx::prefetch_tmap(warp < 8 ? &tm_k : &tm_v);
  if (prefill && warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  Seg sg;
  sg.q_start = p.cu_q[it.seg];
  sg.lq = p.cu_q[it.seg + 1] - sg.q_start;
  sg.lk = p.cu_k ? p.cu_k[it.seg + 1] - p.cu_k[it.seg] : p.seqlens_k[it.seg];
  sg.hist = sg.lk - sg.lq;

  if (prefill) {
    prefill_item<D>(c, it, sg, p, base, gb, *tmem_slot, &tm_q, &tm_k, &tm_v, warp, lane);
  } else if constexpr (D <= 128) {
    decode_item<D>(c, it, sg, p, base, gb, &tm_kd, &tm_vd, warp, lane);
  } else {
    // the planner sends every segment of a D = 256 step through tensor-core tiles
    if (threadIdx.x == 0) atomicOr(p.err, MCP_DEVERR_ITEM_KIND);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (prefill && warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(*tmem_slot, 512);
  }
}

// ------------------------------------------------------------------------
// host side: tensor maps and launch
// ------------------------------------------------------------------------
thread_local char g_detail[256] = "";

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool encode(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, const char* what) {
  auto fn = encode_fn();
  if (!fn) {
    snprintf(g_detail, sizeof(g_detail), "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_detail, sizeof(g_detail), "tensor map for %s rejected (CUresult %d)", what, (int)r);
    return false;
  }
  return true;
}

// Decode ring stages for head group HG: as many as fit, a multiple of the
// warps that share one head (8 / HG) so each stage is always read by the same
// warps (mbarrier parity waits must never run a phase ahead).
template <int D>
int decode_stages(int HG) {
  const int stage = 2 * HG * Cfg<D>::kHeadBlock;
  const int per_head = kDecodeMaxHeads / HG;
  int ns = kDecRingBytes / stage;
  if (ns > kMaxDecStages) ns = kMaxDecStages;
  ns -= ns % per_head;
  return ns;
}

template <int D>
int launch_fwd_d(const FwdArgs& a, cudaStream_t st) {
  using C = Cfg<D>;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int TQ = kTileRows / G;
  const int HG = decode_head_group(a.num_kv_heads);
  alignas(64) CUtensorMap tq, tk, tv, tkd, tvd;
  // dr: head_dim of the tensors.  dr = 96 runs this D = 128 kernel: every map
  // below spans dr columns and a 64-column box at column 64 gets zeros past
  // column 96 (out-of-range elements), so Q, K and V are zero-padded to 128.
  const int dr = a.head_dim;
  const cuuint64_t dr2 = static_cast<cuuint64_t>(dr) * 2;
  {
    // Q [T, H_q, dr]: dims {d, head, token}; a box is one 64-column panel of
    // the G heads of one kv head for TQ tokens (column 64 h for panel h)
    cuuint64_t dims[3] = {(cuuint64_t)dr, (cuuint64_t)a.num_q_heads,
                          (cuuint64_t)(a.total_q > 0 ? a.total_q : 1)};
    cuuint64_t strides[2] = {dr2, (cuuint64_t)a.num_q_heads * dr2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TQ};
    if (!encode(&tq, a.q, 3, dims, strides, box, "q")) return -1;
  }
  // Paged caches: [num_pages, P, H_kv, dr].  Non-paged K/V: [total_k, H_kv, dr],
  // described as one page of total_k tokens (a block is then addressed by its
  // first row as the token coordinate).
  const bool contig = a.cu_seqlens_k != nullptr;
  const cuuint64_t ntok = contig ? static_cast<cuuint64_t>(a.total_k > 0 ? a.total_k : 1)
                                 : static_cast<cuuint64_t>(a.page_size);
  const cuuint64_t npages = contig ? 1 : static_cast<cuuint64_t>(a.num_pages);
  const cuuint64_t page_stride = ntok * a.num_kv_heads * dr2;
  // tokens per TMA box: 8 for page size 8, else 16 (a larger page is several boxes)
  // (1-token pages: the maps are encoded with 1-token boxes but the producers
  // gather with cp.async and the shared-memory layout is the 16-token one)
  const bool gather = !contig && a.page_size == 1;
  const int box_tok = gather ? 1 : (!contig && a.page_size == 8) ? 8 : kPageSize;
  const bool panel_boxes = dr != D;
  // 8-token boxes of K carry every panel when the rows are full width: half
  // the K boxes of a tile (an 8-key group per panel fills one box exactly)
  const bool k_box5 = box_tok == 8 && !panel_boxes && !gather && D > 64;
  if (k_box5) {
    cuuint64_t dims[5] = {64, ntok, (cuuint64_t)(D / 64), (cuuint64_t)a.num_kv_heads, npages};
    cuuint64_t strides[4] = {(cuuint64_t)a.num_kv_heads * dr2, 128, dr2, page_stride};
    cuuint32_t box[5] = {64, 8, (cuuint32_t)(D / 64), 1, 1};
    if (!encode(&tk, a.k_cache, 5, dims, strides, box, "k_cache")) return -1;
  } else {
    // one 64-column panel of one kv head of box_tok tokens: dims {d, head, token, page}
    cuuint64_t dims[4] = {(cuuint64_t)dr, (cuuint64_t)a.num_kv_heads, ntok, npages};
    cuuint64_t strides[3] = {dr2, (cuuint64_t)a.num_kv_heads * dr2, page_stride};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)box_tok, 1};
    if (!encode(&tk, a.k_cache, 4, dims, strides, box, "k_cache")) return -1;
  }
  if (!panel_boxes) {
    // box_tok tokens of one kv head: dims {d, token, panel, head, page}, so
    // that shared memory receives [panel][token][64] from one box
    cuuint64_t dims[5] = {64, ntok, (cuuint64_t)(D / 64), (cuuint64_t)a.num_kv_heads, npages};
    cuuint64_t strides[4] = {(cuuint64_t)a.num_kv_heads * dr2, 128, dr2, page_stride};
    cuuint32_t box[5] = {64, (cuuint32_t)box_tok, (cuuint32_t)(D / 64), 1, 1};
    if (!encode(&tv, a.v_cache, 5, dims, strides, box, "v_cache")) return -1;
    // box_tok tokens of HG kv heads, dims ordered {d, token, panel, head, page}
    // so that shared memory receives [head][panel][token][64]
    cuuint32_t boxd[5] = {64, (cuuint32_t)box_tok, (cuuint32_t)(D / 64), (cuuint32_t)HG, 1};
    if (!encode(&tkd, a.k_cache, 5, dims, strides, boxd, "k_cache pages")) return -1;
    if (!encode(&tvd, a.v_cache, 5, dims, strides, boxd, "v_cache pages")) return -1;
  } else {
    // a panel boundary inside the row: one box per 64-column panel, dims
    // {d, token, head, page}; a box lands as [token][64] (V) or
    // [head][token][64] (decode, HG heads)
    cuuint64_t dims[4] = {(cuuint64_t)dr, ntok, (cuuint64_t)a.num_kv_heads, npages};
    cuuint64_t strides[3] = {(cuuint64_t)a.num_kv_heads * dr2, dr2, page_stride};
    cuuint32_t box[4] = {64, (cuuint32_t)box_tok, 1, 1};
    if (!encode(&tv, a.v_cache, 4, dims, strides, box, "v_cache")) return -1;
    cuuint32_t boxd[4] = {64, (cuuint32_t)box_tok, (cuuint32_t)HG, 1};
    if (!encode(&tkd, a.k_cache, 4, dims, strides, boxd, "k_cache pages")) return -1;
    if (!encode(&tvd, a.v_cache, 4, dims, strides, boxd, "v_cache pages")) return -1;
  }
  KParams kp;
  kp.items = a.items;
  kp.cu_q = a.cu_seqlens_q;
  kp.seqlens_k = a.seqlens_k;
  kp.bt = a.block_tables;
  kp.q = static_cast<const __nv_bfloat16*>(a.q);
  kp.out = static_cast<__nv_bfloat16*>(a.out);
  kp.lse = a.lse;
  kp.part_o = a.part_o;
  kp.part_lse = a.part_lse;
  kp.err = a.error_word;
  kp.max_pages = a.max_pages_per_seq;
  kp.spp_log2 = contig ? 0 : (a.page_size == 64 ? 2 : (a.page_size == 32 ? 1 : 0));
  kp.box_log2 = box_tok == 8 ? 3 : 4;
  kp.gather = gather ? 1 : 0;
  kp.hkv = a.num_kv_heads;
  kp.kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  kp.vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  kp.dr = dr;
  kp.panel_boxes = panel_boxes ? 1 : 0;
  kp.cu_k = a.cu_seqlens_k;
  kp.num_pages = a.num_pages;
  kp.hq = a.num_q_heads;
  kp.G = G;
  kp.dec_stages = decode_stages<D>(HG);
  kp.scale_log2 = a.sm_scale * kLog2e;
  kp.test_stall = a.test_stall;
  kp.k_box5 = k_box5 ? 1 : 0;
  cudaError_t e = cudaFuncSetAttribute(mixed_attn_fwd_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return static_cast<int>(e);
  mixed_attn_fwd_kernel<D><<<a.num_items, kFwdThreads, C::kSmemBytes, st>>>(tq, tk, tv, tkd, tvd, kp);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace

const char* launch_detail() { return g_detail; }

int launch_mixed_attn(const FwdArgs& a, void* stream) {
  g_detail[0] = 0;
  if (a.num_items <= 0) return 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (a.head_dim == 128 || a.head_dim == 96) return launch_fwd_d<128>(a, st);
  if (a.head_dim == 64) return launch_fwd_d<64>(a, st);
  if (a.head_dim == 256) return launch_fwd_d<256>(a, st);
  snprintf(g_detail, sizeof(g_detail), "head_dim %d not built", a.head_dim);
  return -1;
}

}  // namespace mcp
