// Branch scheduler of hierarchical parallel decoding (HPD-Parsing, inference
// workflow and Algorithm 1): FCFS keys with child branches first, gated
// admission of layout requests (KV occupancy threshold tau, concurrency cap
// N_max) that child branches bypass, KV reserved ahead of every verify step
// for the draft window, preemption of the youngest request when the pool
// runs short, zero-copy forks on <FORK>, release by reference count, and the
// layout request's output interleaved with its children's once all of them
// have ended.  Host code over the refcounted KV pool.
#include <algorithm>
#include <cstdint>
#include <memory>
#include <new>
#include <tuple>
#include <vector>

#include "../../include/padoc.h"
#include "padoc_internal.h"

namespace {

enum State { WAITING = 0, RUNNING = 1, ENDED = 2, DONE = 3 };

struct Req {
  int32_t id;
  int64_t arrival;
  int32_t parent;  // -1: a main (layout) request
  int32_t m = 0;   // children the parent had spawned before this one
  int32_t prompt_len = 0, fork_len = 0;
  std::vector<int32_t> out;
  std::vector<int32_t> children;
  int32_t state = WAITING;
  int32_t seq = -1;
};

}  // namespace

struct padoc_sched {
  padoc_kv_pool* pool = nullptr;
  padoc_sched_config cfg{};
  std::vector<Req> reqs;
  std::vector<int32_t> queue;   // waiting request ids
  std::vector<int32_t> active;  // running request ids

  // (0, arrival(parent), -m, arrival(child), id) for a child, (1, arrival, 0, 0, id) for a main request
  std::tuple<int, int64_t, int64_t, int64_t, int32_t> key(int32_t id) const {
    const Req& r = reqs[id];
    if (r.parent < 0) return {1, r.arrival, 0, 0, id};
    return {0, reqs[r.parent].arrival, -static_cast<int64_t>(r.m), r.arrival, id};
  }
  void sort_by_key(std::vector<int32_t>* v) const {
    std::sort(v->begin(), v->end(), [&](int32_t a, int32_t b) { return key(a) < key(b); });
  }
  int64_t stream_len(const Req& r) const {
    return (r.parent < 0 ? r.prompt_len : r.fork_len) + static_cast<int64_t>(r.out.size());
  }
};

namespace {

int pool_len(padoc_kv_pool* pool, int32_t seq, int32_t* len) { return padoc_kv_seq_info(pool, seq, len, nullptr, nullptr); }

// Admission: reserve the cached tokens + K + 1 and rebuild the cached tokens
// (bookkeeping only: the caller prefills them).  Returns 1 admitted, 0 no room.
int admit_kv(padoc_sched* s, Req& r) {
  const int32_t K1 = s->cfg.window + 1;
  const int64_t cached = s->stream_len(r) - 1;
  int32_t seq = -1;
  if (r.parent < 0) {
    int rc = padoc_kv_alloc(s->pool, static_cast<int32_t>(cached + K1), &seq);
    if (rc == PADOC_ERR_OOM) return 0;
    if (rc) return rc;
    rc = padoc_kv_advance(s->pool, seq, static_cast<int32_t>(cached));
    if (rc) return rc;
  } else {
    const Req& p = s->reqs[r.parent];
    int rc = padoc_kv_fork(s->pool, p.seq, r.fork_len, &seq);
    if (rc) return rc;
    const int32_t own = static_cast<int32_t>(cached - r.fork_len);
    rc = padoc_kv_reserve(s->pool, seq, own + K1);
    if (rc == PADOC_ERR_OOM) {
      padoc_kv_release(s->pool, seq);
      return 0;
    }
    if (rc) return rc;
    rc = padoc_kv_advance(s->pool, seq, own);
    if (rc) return rc;
  }
  r.seq = seq;
  return 1;
}

int preempt(padoc_sched* s, int32_t id) {
  Req& r = s->reqs[id];
  const int rc = padoc_kv_release(s->pool, r.seq);
  if (rc) return rc;
  r.seq = -1;
  r.state = WAITING;
  s->active.erase(std::find(s->active.begin(), s->active.end(), id));
  s->queue.push_back(id);
  return PADOC_OK;
}

// Releases an ended request whose children have all ended, then its parent
// if that completes it.
int maybe_release(padoc_sched* s, int32_t id) {
  while (id >= 0) {
    Req& r = s->reqs[id];
    if (r.state != ENDED) return PADOC_OK;
    for (int32_t c : r.children)
      if (s->reqs[c].state != DONE) return PADOC_OK;
    const int rc = padoc_kv_release(s->pool, r.seq);
    if (rc) return rc;
    r.seq = -1;
    r.state = DONE;
    id = r.parent;
  }
  return PADOC_OK;
}

void interleave(const padoc_sched* s, int32_t id, std::vector<int32_t>* out) {
  const Req& r = s->reqs[id];
  size_t k = 0;
  for (int32_t t : r.out) {
    out->push_back(t);
    if (t == s->cfg.fork_token && r.parent < 0 && k < r.children.size()) interleave(s, r.children[k++], out);
  }
}

}  // namespace

extern "C" int padoc_sched_create(padoc_kv_pool* pool, const padoc_sched_config* cfg, padoc_sched** out) {
  if (!pool || !cfg || !out) return padoc::set_error(PADOC_ERR_INVALID, "sched_create: null argument");
  *out = nullptr;
  if (!(cfg->tau >= 0.f && cfg->tau <= 1.f)) return padoc::set_error(PADOC_ERR_INVALID, "sched_create: tau outside [0, 1]");
  if (cfg->n_max < 1 || cfg->window < 0 || cfg->window > 15 || cfg->max_len < 1)
    return padoc::set_error(PADOC_ERR_INVALID, "sched_create: n_max >= 1, window in [0, 15], max_len >= 1");
  try {
    std::unique_ptr<padoc_sched> s(new padoc_sched());
    s->pool = pool;
    s->cfg = *cfg;
    *out = s.release();
  } catch (const std::bad_alloc&) {
    return padoc::set_error(PADOC_ERR_OOM, "sched_create: out of host memory");
  }
  return PADOC_OK;
}

extern "C" int padoc_sched_destroy(padoc_sched* s) {
  if (!s) return PADOC_OK;
  for (Req& r : s->reqs)
    if (r.seq >= 0) padoc_kv_release(s->pool, r.seq);
  delete s;
  return PADOC_OK;
}

extern "C" int padoc_sched_submit(padoc_sched* s, int32_t prompt_len, int64_t arrival, int32_t* request) {
  if (!s || !request) return padoc::set_error(PADOC_ERR_INVALID, "sched_submit: null argument");
  if (prompt_len < 1) return padoc::set_error(PADOC_ERR_INVALID, "sched_submit: prompt_len must be >= 1");
  try {
    Req r;
    r.id = static_cast<int32_t>(s->reqs.size());
    r.arrival = arrival;
    r.parent = -1;
    r.prompt_len = prompt_len;
    s->reqs.push_back(r);
    s->queue.push_back(r.id);
    *request = r.id;
  } catch (const std::bad_alloc&) {
    return padoc::set_error(PADOC_ERR_OOM, "sched_submit: out of host memory");
  }
  return PADOC_OK;
}

extern "C" int padoc_sched_schedule(padoc_sched* s, padoc_sched_step* st) {
  if (!s || !st) return padoc::set_error(PADOC_ERR_INVALID, "sched_schedule: null argument");
  if (st->cap < 0 || (st->cap > 0 && (!st->admitted || !st->preempted || !st->active || !st->active_seq ||
                                       !st->page_seq || !st->branch_offsets)))
    return padoc::set_error(PADOC_ERR_INVALID, "sched_schedule: output arrays missing");
  const int32_t K1 = s->cfg.window + 1;
  std::vector<int32_t> admitted, preempted;
  try {
    // 1. reserve the step's window for every active branch, preempting the
    //    youngest active request while the pool is short
    std::vector<int32_t> order = s->active;
    s->sort_by_key(&order);
    for (int32_t id : order) {
      while (std::find(s->active.begin(), s->active.end(), id) != s->active.end()) {
        const int rc = padoc_kv_reserve(s->pool, s->reqs[id].seq, K1);
        if (rc == PADOC_OK) break;
        if (rc != PADOC_ERR_OOM) return rc;
        int32_t victim = s->active[0];
        for (int32_t a : s->active)
          if (std::make_pair(s->reqs[a].arrival, a) > std::make_pair(s->reqs[victim].arrival, victim)) victim = a;
        const int rc2 = preempt(s, victim);
        if (rc2) return rc2;
        preempted.push_back(victim);
      }
    }
    // 2. admission in key order: main requests through the gate, children
    //    once their parent is resident with the tokens before the <FORK>
    //    cached; a request
    //    the pool cannot hold now keeps its place and the scan goes on
    std::vector<int32_t> q = s->queue;
    s->sort_by_key(&q);
    for (int32_t id : q) {
      if (std::find(preempted.begin(), preempted.end(), id) != preempted.end()) continue;
      Req& r = s->reqs[id];
      if (r.parent < 0) {
        int32_t free_blocks = 0, live = 0;
        padoc_kv_pool_stats(s->pool, &free_blocks, &live);
        const int32_t total = padoc::pool_num_blocks(s->pool);
        const double occ = static_cast<double>(total - free_blocks) / total;
        if (occ > static_cast<double>(s->cfg.tau) || static_cast<int32_t>(s->active.size()) >= s->cfg.n_max) continue;
      } else {
        const Req& p = s->reqs[r.parent];
        if (p.seq < 0) continue;
        int32_t plen = 0;
        const int rc = pool_len(s->pool, p.seq, &plen);
        if (rc) return rc;
        if (plen < r.fork_len) continue;  // its prefix is not cached yet
      }
      const int rc = admit_kv(s, r);
      if (rc < 0) return rc;
      if (rc == 0) continue;  // no room this step: it keeps its place
      r.state = RUNNING;
      s->queue.erase(std::find(s->queue.begin(), s->queue.end(), id));
      s->active.push_back(id);
      admitted.push_back(id);
    }
  } catch (const std::bad_alloc&) {
    return padoc::set_error(PADOC_ERR_OOM, "sched_schedule: out of host memory");
  }
  // 3. the batch: active branches grouped by page (a child's parent, a main
  //    request itself), pages in order of their first branch in key order
  std::vector<int32_t> order = s->active;
  s->sort_by_key(&order);
  std::vector<int32_t> pages;
  std::vector<std::vector<int32_t>> members;
  for (int32_t id : order) {
    const int32_t pg = s->reqs[id].parent < 0 ? id : s->reqs[id].parent;
    auto it = std::find(pages.begin(), pages.end(), pg);
    if (it == pages.end()) {
      pages.push_back(pg);
      members.push_back({id});
    } else {
      members[it - pages.begin()].push_back(id);
    }
  }
  const int32_t n_act = static_cast<int32_t>(order.size());
  if (static_cast<int32_t>(admitted.size()) > st->cap || static_cast<int32_t>(preempted.size()) > st->cap ||
      n_act > st->cap)
    return padoc::set_error(PADOC_ERR_INVALID, "sched_schedule: capacity %d too small (%d active)", st->cap, n_act);
  std::copy(admitted.begin(), admitted.end(), st->admitted);
  std::copy(preempted.begin(), preempted.end(), st->preempted);
  st->n_admitted = static_cast<int32_t>(admitted.size());
  st->n_preempted = static_cast<int32_t>(preempted.size());
  st->n_active = n_act;
  st->n_pages = static_cast<int32_t>(pages.size());
  int32_t k = 0;
  st->branch_offsets[0] = 0;
  for (size_t p = 0; p < pages.size(); ++p) {
    st->page_seq[p] = s->reqs[pages[p]].seq;
    for (int32_t id : members[p]) {
      st->active[k] = id;
      st->active_seq[k] = s->reqs[id].seq;
      ++k;
    }
    st->branch_offsets[p + 1] = k;
  }
  return PADOC_OK;
}

extern "C" int padoc_sched_update(padoc_sched* s, int64_t now, int32_t n, const int32_t* request,
                                  const int32_t* token_offsets, const int32_t* tokens) {
  if (!s || (n > 0 && (!request || !token_offsets || !tokens)))
    return padoc::set_error(PADOC_ERR_INVALID, "sched_update: null argument");
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = request[i];
    if (id < 0 || id >= static_cast<int32_t>(s->reqs.size()) || s->reqs[id].state != RUNNING)
      return padoc::set_error(PADOC_ERR_INVALID, "sched_update: request %d is not running", id);
    if (token_offsets[i + 1] - token_offsets[i] < 1)
      return padoc::set_error(PADOC_ERR_INVALID, "sched_update: request %d has no token", id);
  }
  try {
    for (int32_t i = 0; i < n; ++i) {
      const int32_t id = request[i];
      bool ended = false;
      int32_t taken = 0;
      for (int32_t j = token_offsets[i]; j < token_offsets[i + 1]; ++j) {
        const int32_t t = tokens[j];
        s->reqs[id].out.push_back(t);
        ++taken;
        if (t == s->cfg.fork_token && s->reqs[id].parent < 0) {
          Req c;
          c.id = static_cast<int32_t>(s->reqs.size());
          c.arrival = now;
          c.parent = id;
          c.m = static_cast<int32_t>(s->reqs[id].children.size());
          c.fork_len = static_cast<int32_t>(s->stream_len(s->reqs[id]) - 1);  // the tokens before the <FORK>
          c.out.push_back(s->cfg.child_token);
          s->reqs[id].children.push_back(c.id);
          s->reqs.push_back(c);  // may move reqs: index by id from here on
          s->queue.push_back(c.id);
        }
        if (t == s->cfg.eos_token || static_cast<int32_t>(s->reqs[id].out.size()) >= s->cfg.max_len) {
          ended = true;
          break;
        }
      }
      // the old anchor and the new tokens but the newest are now cached
      const int rc = padoc_kv_advance(s->pool, s->reqs[id].seq, taken);
      if (rc) return rc;
      if (ended) {
        s->reqs[id].state = ENDED;
        s->active.erase(std::find(s->active.begin(), s->active.end(), id));
        int rc2 = padoc_kv_trim(s->pool, s->reqs[id].seq);  // the unused part of its reservation
        if (!rc2) rc2 = maybe_release(s, id);
        if (rc2) return rc2;
      }
    }
  } catch (const std::bad_alloc&) {
    return padoc::set_error(PADOC_ERR_OOM, "sched_update: out of host memory");
  }
  return PADOC_OK;
}

extern "C" int padoc_sched_request(const padoc_sched* s, int32_t request, int32_t* state, int32_t* seq,
                                   int32_t* parent, int64_t* n_out) {
  if (!s || request < 0 || request >= static_cast<int32_t>(s->reqs.size()))
    return padoc::set_error(PADOC_ERR_INVALID, "sched_request: unknown request");
  const Req& r = s->reqs[request];
  if (state) *state = r.state;
  if (seq) *seq = r.seq;
  if (parent) *parent = r.parent;
  if (n_out) *n_out = static_cast<int64_t>(r.out.size());
  return PADOC_OK;
}

extern "C" int padoc_sched_output(const padoc_sched* s, int32_t request, int32_t* tokens, int64_t cap, int64_t* n) {
  if (!s || !n || request < 0 || request >= static_cast<int32_t>(s->reqs.size()))
    return padoc::set_error(PADOC_ERR_INVALID, "sched_output: bad argument");
  const Req& r = s->reqs[request];
  if (r.parent >= 0 || r.state != DONE)
    return padoc::set_error(PADOC_ERR_INVALID, "sched_output: request %d is not a finished main request", request);
  std::vector<int32_t> out;
  try {
    interleave(s, request, &out);
  } catch (const std::bad_alloc&) {
    return padoc::set_error(PADOC_ERR_OOM, "sched_output: out of host memory");
  }
  *n = static_cast<int64_t>(out.size());
  if (tokens) {
    if (cap < *n) return padoc::set_error(PADOC_ERR_INVALID, "sched_output: capacity %lld < %lld", (long long)cap, (long long)*n);
    std::copy(out.begin(), out.end(), tokens);
  }
  return PADOC_OK;
}
