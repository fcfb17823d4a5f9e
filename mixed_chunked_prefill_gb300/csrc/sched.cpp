// Step builder: the chunked-prefill scheduler (host-only C++).
//
// [W] wangyu.me "大语言模型推理优化（二）：Chunked Prefill", sections "Token 预算：
// max_num_batched_tokens" and "调度器：running 优先，waiting 填充": every request
// tracks num_computed_tokens (tokens whose K/V are in the cache) and
// num_tokens (prompt + sampled tokens, whose K/V must eventually be there);
// a step spends a token budget on running requests first, then admits
// waiting ones; long_prefill_token_threshold caps one chunk.  Section "采样":
// only decodes and chunks that finish their prompt sample.  [X] m.xxqk.cn
// "动态批处理中的抢占与优先级调度": waiting requests are admitted by priority;
// when pages run out, a running request is preempted by recompute or swap.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "mcp.h"
#include "mcp_internal.h"

namespace {

// Format the message into this thread's mcp_last_error() and return `s`.
mcp_status sfail(mcp_status s, const char* fmt, ...) {
  char msg[256];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof(msg), fmt, ap);
  va_end(ap);
  return static_cast<mcp_status>(mcp::set_error_code(s, msg));
}

enum class St { kWaiting, kRunning, kSwapped, kFinished };

struct Req {
  int64_t id = 0;
  int32_t prompt = 0;     // tokens to compute before the first sample (after a
                          // recompute: every token the request had)
  int32_t max_new = 0;
  int32_t priority = 0;
  int64_t arrival = 0;
  int32_t num_tokens = 0;    // prompt + sampled tokens
  int32_t num_computed = 0;  // tokens whose K/V are in the device cache
  int32_t generated = 0;
  St st = St::kWaiting;
  std::vector<int32_t> pages;       // device pages, logical order
  std::vector<int32_t> host_pages;  // host pool pages while swapped out
};

struct Seg {
  Req* r;
  int32_t n;
  bool sample;
};

}  // namespace

struct mcp_sched {
  mcp_sched_config cfg;
  std::unordered_map<int64_t, Req*> live;
  std::vector<Req*> reqs;  // every live request (owned)
  std::vector<int32_t> free_pages, free_host;
  int64_t arrivals = 0, finished = 0;
  // last step
  std::vector<Seg> segs;
  std::vector<int64_t> ids, preempted;
  std::vector<int32_t> cu, sk, bt, logits, so_dev, so_host, si_host, si_dev;
  std::vector<uint8_t> sample;

  int32_t pages_for(int64_t tokens) const {
    return static_cast<int32_t>((tokens + cfg.page_size - 1) / cfg.page_size);
  }
  static bool before(const Req* a, const Req* b) {  // admission order: priority, then arrival
    if (a->priority != b->priority) return a->priority > b->priority;
    return a->arrival < b->arrival;
  }
  void release(Req* r) {
    for (int32_t p : r->pages) free_pages.push_back(p);
    r->pages.clear();
  }
  // Preempt r: swap its pages to the host pool if configured and there is
  // room, else drop them for recompute.
  void preempt(Req* r) {
    preempted.push_back(r->id);
    if (cfg.preempt_swap && !r->pages.empty() &&
        free_host.size() >= r->pages.size()) {
      for (int32_t p : r->pages) {
        const int32_t h = free_host.back();
        free_host.pop_back();
        so_dev.push_back(p);
        so_host.push_back(h);
        r->host_pages.push_back(h);
      }
      release(r);
      r->st = St::kSwapped;
      return;
    }
    release(r);
    r->prompt = r->num_tokens;  // every token so far becomes prompt again
    r->num_computed = 0;
    r->st = St::kWaiting;
  }
  bool take_pages(Req* r, int32_t n) {
    if (static_cast<int32_t>(free_pages.size()) < n) return false;
    for (int32_t i = 0; i < n; ++i) {
      r->pages.push_back(free_pages.back());
      free_pages.pop_back();
    }
    return true;
  }
  int32_t chunk(const Req* r, int32_t budget) const {
    int32_t n = r->num_tokens - r->num_computed;
    if (cfg.long_prefill_token_threshold > 0 && n > cfg.long_prefill_token_threshold)
      n = cfg.long_prefill_token_threshold;
    return std::min(n, budget);
  }
};

extern "C" {

mcp_status mcp_sched_create(const mcp_sched_config* c, mcp_sched** out) {
  if (!c || !out) return sfail(MCP_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  for (int i = 0; i < 4; ++i)
    if (c->reserved[i] != 0) return sfail(MCP_ERR_INVALID_ARG, "config reserved must be 0");
  if (c->max_num_batched_tokens < 1 || c->max_num_seqs < 1 || c->num_pages < 1 ||
      c->page_size < 1 || c->max_pages_per_seq < 1 || c->long_prefill_token_threshold < 0 ||
      c->num_host_pages < 0 || (c->preempt_swap != 0 && c->preempt_swap != 1))
    return sfail(MCP_ERR_INVALID_ARG, "invalid scheduler config");
  mcp_sched* s = new (std::nothrow) mcp_sched();
  if (!s) return sfail(MCP_ERR_INVALID_ARG, "host allocation failed");
  s->cfg = *c;
  // pages handed out lowest id first
  for (int32_t p = c->num_pages - 1; p >= 0; --p) s->free_pages.push_back(p);
  for (int32_t p = c->num_host_pages - 1; p >= 0; --p) s->free_host.push_back(p);
  *out = s;
  return MCP_OK;
}

mcp_status mcp_sched_add_request(mcp_sched* s, int64_t id, int32_t prompt_len,
                                 int32_t max_new_tokens, int32_t priority) {
  if (!s) return sfail(MCP_ERR_INVALID_ARG, "sched is NULL");
  if (prompt_len < 1 || max_new_tokens < 1)
    return sfail(MCP_ERR_INVALID_ARG, "prompt_len and max_new_tokens must be >= 1");
  if (static_cast<int64_t>(prompt_len) + max_new_tokens >
      static_cast<int64_t>(s->cfg.max_pages_per_seq) * s->cfg.page_size)
    return sfail(MCP_ERR_INVALID_ARG, "request %lld needs more than max_pages_per_seq pages",
                 static_cast<long long>(id));
  if (s->live.count(id)) return sfail(MCP_ERR_INVALID_ARG, "request id %lld already live",
                                      static_cast<long long>(id));
  try {
    Req* r = new Req();
    r->id = id;
    r->prompt = prompt_len;
    r->num_tokens = prompt_len;
    r->max_new = max_new_tokens;
    r->priority = priority;
    r->arrival = s->arrivals++;
    s->live[id] = r;
    s->reqs.push_back(r);
  } catch (...) {
    return sfail(MCP_ERR_INVALID_ARG, "host allocation failed");
  }
  return MCP_OK;
}

mcp_status mcp_sched_schedule(mcp_sched* s, mcp_sched_output* out) {
  if (!s || !out) return sfail(MCP_ERR_INVALID_ARG, "NULL argument");
  try {
    const mcp_sched_config& c = s->cfg;
    s->segs.clear();
    s->preempted.clear();
    s->so_dev.clear(); s->so_host.clear(); s->si_host.clear(); s->si_dev.clear();
    int32_t budget = c.max_num_batched_tokens;
    std::vector<Req*> running, swapped, waiting;
    for (Req* r : s->reqs) {
      if (r->st == St::kRunning) running.push_back(r);
      else if (r->st == St::kSwapped) swapped.push_back(r);
      else if (r->st == St::kWaiting) waiting.push_back(r);
    }
    std::sort(running.begin(), running.end(),
              [](const Req* a, const Req* b) { return a->arrival < b->arrival; });
    std::sort(swapped.begin(), swapped.end(), mcp_sched::before);
    std::sort(waiting.begin(), waiting.end(), mcp_sched::before);
    auto seats = [&]() { return static_cast<int32_t>(s->segs.size()) < c.max_num_seqs; };
    auto schedule = [&](Req* r, int32_t n) {
      const bool sample = r->num_computed + n >= r->prompt && r->num_computed + n == r->num_tokens;
      s->segs.push_back({r, n, sample});
      budget -= n;
    };
    // 1. running first, in arrival order; preempt from the back when pages run out
    for (size_t i = 0; i < running.size() && budget > 0 && seats(); ++i) {
      Req* r = running[i];
      if (r->st != St::kRunning) continue;  // preempted earlier in this step
      const int32_t n = s->chunk(r, budget);
      if (n <= 0) continue;
      const int32_t need = s->pages_for(static_cast<int64_t>(r->num_computed) + n) -
                           static_cast<int32_t>(r->pages.size());
      bool ok = true;
      while (static_cast<int32_t>(s->free_pages.size()) < need) {
        // victim: lowest priority, latest arrival, among running requests not yet scheduled
        Req* victim = nullptr;
        for (size_t j = running.size(); j-- > i + 1;) {
          Req* v = running[j];
          if (v->st != St::kRunning) continue;
          if (!victim || v->priority < victim->priority ||
              (v->priority == victim->priority && v->arrival > victim->arrival))
            victim = v;
        }
        if (!victim) {
          s->preempt(r);
          ok = false;
          break;
        }
        s->preempt(victim);
      }
      if (!ok) continue;
      s->take_pages(r, need);
      schedule(r, n);
    }
    // 2. swapped requests come back when their pages fit
    for (Req* r : swapped) {
      if (budget <= 0 || !seats() || !s->preempted.empty()) break;
      const int32_t n = s->chunk(r, budget);
      const int32_t have = static_cast<int32_t>(r->host_pages.size());
      const int32_t need = std::max(have, s->pages_for(static_cast<int64_t>(r->num_computed) + n));
      if (static_cast<int32_t>(s->free_pages.size()) < need) break;
      s->take_pages(r, need);
      for (int32_t k = 0; k < have; ++k) {
        s->si_host.push_back(r->host_pages[k]);
        s->si_dev.push_back(r->pages[k]);
        s->free_host.push_back(r->host_pages[k]);
      }
      r->host_pages.clear();
      r->st = St::kRunning;
      if (n > 0) schedule(r, n);
    }
    // 3. waiting requests fill the rest, by priority; no preemption to admit
    for (Req* r : waiting) {
      if (budget <= 0 || !seats() || !s->preempted.empty()) break;
      if (r->st != St::kWaiting) continue;
      const int32_t n = s->chunk(r, budget);
      if (n <= 0) break;
      const int32_t need = s->pages_for(n);
      if (!s->take_pages(r, need)) break;
      r->st = St::kRunning;
      schedule(r, n);
    }
    // the step's arrays
    const int32_t S = static_cast<int32_t>(s->segs.size());
    const int32_t mp = c.max_pages_per_seq;
    s->ids.assign(S, 0);
    s->cu.assign(S + 1, 0);
    s->sk.assign(S, 0);
    s->bt.assign(static_cast<size_t>(S) * mp, -1);
    s->sample.assign(S, 0);
    s->logits.clear();
    for (int32_t i = 0; i < S; ++i) {
      const Seg& g = s->segs[i];
      s->ids[i] = g.r->id;
      s->cu[i + 1] = s->cu[i] + g.n;
      s->sk[i] = g.r->num_computed + g.n;
      for (size_t k = 0; k < g.r->pages.size(); ++k) s->bt[static_cast<size_t>(i) * mp + k] = g.r->pages[k];
      s->sample[i] = g.sample ? 1 : 0;
      if (g.sample) s->logits.push_back(s->cu[i + 1] - 1);
    }
    std::memset(out, 0, sizeof(*out));
    out->num_seqs = S;
    out->total_q = s->cu[S];
    out->request_ids = s->ids.data();
    out->cu_seqlens_q = s->cu.data();
    out->seqlens_k = s->sk.data();
    out->block_tables = s->bt.data();
    out->sample_mask = s->sample.data();
    out->logits_indices = s->logits.data();
    out->num_logits = static_cast<int32_t>(s->logits.size());
    out->num_swap_out = static_cast<int32_t>(s->so_dev.size());
    out->swap_out_device_pages = s->so_dev.data();
    out->swap_out_host_pages = s->so_host.data();
    out->num_swap_in = static_cast<int32_t>(s->si_dev.size());
    out->swap_in_host_pages = s->si_host.data();
    out->swap_in_device_pages = s->si_dev.data();
    out->num_preempted = static_cast<int32_t>(s->preempted.size());
    out->preempted_ids = s->preempted.data();
    return MCP_OK;
  } catch (...) {
    return sfail(MCP_ERR_INVALID_ARG, "host allocation failed while scheduling");
  }
}

mcp_status mcp_sched_finish_step(mcp_sched* s, int32_t* num_finished, int64_t* finished_ids) {
  if (!s) return sfail(MCP_ERR_INVALID_ARG, "sched is NULL");
  int32_t nf = 0;
  for (const Seg& g : s->segs) {
    Req* r = g.r;
    r->num_computed += g.n;
    if (!g.sample) continue;
    ++r->generated;
    if (r->generated >= r->max_new) {
      s->release(r);
      r->st = St::kFinished;
      if (finished_ids) finished_ids[nf] = r->id;
      ++nf;
    } else {
      ++r->num_tokens;  // the sampled token is computed by a later step
    }
  }
  s->segs.clear();
  // drop finished requests
  std::vector<Req*> keep;
  for (Req* r : s->reqs) {
    if (r->st == St::kFinished) {
      s->live.erase(r->id);
      delete r;
      ++s->finished;
    } else {
      keep.push_back(r);
    }
  }
  s->reqs.swap(keep);
  if (num_finished) *num_finished = nf;
  return MCP_OK;
}

mcp_status mcp_sched_stats(const mcp_sched* s, int32_t* waiting, int32_t* running,
                           int32_t* swapped, int64_t* finished, int32_t* free_pages) {
  if (!s) return sfail(MCP_ERR_INVALID_ARG, "sched is NULL");
  int32_t w = 0, r = 0, sw = 0;
  for (const Req* q : s->reqs) {
    if (q->st == St::kWaiting) ++w;
    else if (q->st == St::kRunning) ++r;
    else if (q->st == St::kSwapped) ++sw;
  }
  if (waiting) *waiting = w;
  if (running) *running = r;
  if (swapped) *swapped = sw;
  if (finished) *finished = s->finished;
  if (free_pages) *free_pages = static_cast<int32_t>(s->free_pages.size());
  return MCP_OK;
}

mcp_status mcp_sched_destroy(mcp_sched* s) {
  if (!s) return MCP_OK;
  for (Req* r : s->reqs) delete r;
  delete s;
  return MCP_OK;
}

}  // extern "C"
