// Host-side continuous-batching scheduler with the budget rule for draft
// lengths (declared in sdv_sched.h).
//
// Draft length: one verify pass hides a fixed number of token rows under the
// weight stream; the live batch takes one row per sequence and the rest is
// shared as drafts, gamma = (budget - B) / B ("Speculative Decoding and
// Batching Compete for the Same Compute Slack on RDNA4", sections "The budget
// is fixed, and the batch is inside it" and "What the budget says to build").
//
// Membership: decided every step.  Under the continuous policy a finished
// sequence's slot is refilled from the arrival-order queue on the next step;
// the two static policies admit only into an empty batch ("Why Static
// Batching Wastes an RX 9070 XT Agent Swarm and Continuous Batching Wins It
// Back", table in "Continuous batching refills the slot instead of freezing
// it").
//
// The slot mirror follows the device's realignment exactly: a sequence that
// accepted a drafts grows by a + 1 positions and holds
// ceil((L + gamma_max + 1) / page) pages afterwards; it finishes once its
// emitted count reaches its output length and then releases every page; the
// survivors are compacted in order.
#include <cstdint>
#include <deque>
#include <new>
#include <vector>

#include "sdv_sched.h"

namespace {

struct Seq {
  long long id;
  int len;    // positions in its KV cache
  int gen;    // tokens emitted so far
  int limit;  // output length at which it finishes
  int pages;  // pages held
};

struct Pending {
  long long id;
  int ctx, out;
};

int ceil_div(long long a, int b) { return static_cast<int>((a + b - 1) / b); }

}  // namespace

struct sdv_sched {
  sdv_sched_config cfg;
  std::vector<Seq> slots;      // live sequences in slot order
  std::deque<Pending> queue;   // arrival order
  int free_pages = 0;
  int group_width = 0;         // frozen width of the current static group
  bool planned = false;
  sdv_sched_step step{};
  sdv_sched_stats stats{};

  int pages_for(long long len) const { return ceil_div(len + cfg.gamma_max + 1, cfg.page_size); }
  // one step of growth: at most gamma_max + 1 new positions per live sequence
  int growth_pages() const { return ceil_div(cfg.gamma_max + 1, cfg.page_size); }
};

extern "C" {

int sdv_sched_gamma(int budget_rows, int live, int gamma_max) {
  if (live <= 0 || gamma_max <= 0) return 0;
  const int g = (budget_rows - live) / live;  // C division truncates toward zero; negatives clamp below
  if (g < 0) return 0;
  return g > gamma_max ? gamma_max : g;
}

sdv_status sdv_sched_create(const sdv_sched_config* cfg, sdv_sched** out) {
  if (!cfg || !out) return SDV_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->max_slots < 1 || cfg->gamma_max < 0 || cfg->budget_rows < 1 || cfg->page_size < 1 ||
      cfg->pool_pages < 0 || cfg->max_pages_per_seq < 1)
    return SDV_ERR_INVALID_ARG;
  if (cfg->policy < SDV_SCHED_CONTINUOUS || cfg->policy > SDV_SCHED_STATIC_SHRINK) return SDV_ERR_INVALID_ARG;
  sdv_sched* s = new (std::nothrow) sdv_sched;
  if (!s) return SDV_ERR_INTERNAL;
  s->cfg = *cfg;
  s->free_pages = cfg->pool_pages;
  s->slots.reserve(static_cast<size_t>(cfg->max_slots));
  s->stats.free_pages = s->free_pages;
  *out = s;
  return SDV_OK;
}

void sdv_sched_destroy(sdv_sched* s) { delete s; }

sdv_status sdv_sched_submit(sdv_sched* s, long long id, int ctx_len, int out_len) {
  if (!s || ctx_len < 0 || out_len < 1) return SDV_ERR_INVALID_ARG;
  // the longest it can get: out_len - 1 tokens before its last step, which adds up to gamma_max + 1
  const long long longest = static_cast<long long>(ctx_len) + out_len + s->cfg.gamma_max;
  const int most = s->pages_for(longest);
  if (most > s->cfg.max_pages_per_seq || most > s->cfg.pool_pages) return SDV_ERR_CAPACITY;
  s->queue.push_back(Pending{id, ctx_len, out_len});
  s->stats.queued = static_cast<int>(s->queue.size());
  return SDV_OK;
}

sdv_status sdv_sched_plan(sdv_sched* s, sdv_sched_step* step, int* admit_ctx, int* admit_out, long long* slot_ids) {
  if (!s || !step || s->planned) return SDV_ERR_INVALID_ARG;
  const sdv_sched_config& c = s->cfg;
  const bool may_admit = c.policy == SDV_SCHED_CONTINUOUS || s->slots.empty();
  if (may_admit && !s->queue.empty() && (!admit_ctx || !admit_out)) return SDV_ERR_INVALID_ARG;
  int admitted = 0;
  if (may_admit) {
    while (!s->queue.empty() && static_cast<int>(s->slots.size()) < c.max_slots) {
      const Pending& q = s->queue.front();
      const int need = s->pages_for(q.ctx);
      // keep one step of growth for every sequence live after this admission
      const long long reserve = static_cast<long long>(s->slots.size() + 1) * s->growth_pages();
      if (need + reserve > s->free_pages) break;
      s->free_pages -= need;
      s->slots.push_back(Seq{q.id, q.ctx, 0, q.out, need});
      admit_ctx[admitted] = q.ctx;
      admit_out[admitted] = q.out;
      ++admitted;
      s->queue.pop_front();
    }
    if (c.policy != SDV_SCHED_CONTINUOUS && admitted > 0) s->group_width = admitted;
  }
  const int live = static_cast<int>(s->slots.size());
  const int gamma = sdv_sched_gamma(c.budget_rows, live, c.gamma_max);
  step->live = live;
  step->width = c.policy == SDV_SCHED_STATIC ? (live > 0 ? s->group_width : 0) : live;
  step->gamma = gamma;
  step->rows = live * (gamma + 1);
  step->drafts = live * gamma;
  step->admitted = admitted;
  if (slot_ids)
    for (int b = 0; b < live; ++b) slot_ids[b] = s->slots[static_cast<size_t>(b)].id;
  s->step = *step;
  s->planned = true;
  s->stats.queued = static_cast<int>(s->queue.size());
  s->stats.admitted += admitted;
  return SDV_OK;
}

sdv_status sdv_sched_complete(sdv_sched* s, const int* accepted, long long* finished_ids, int* n_finished) {
  if (!s || !s->planned) return SDV_ERR_INVALID_ARG;
  const int live = s->step.live;
  if (live > 0 && !accepted) return SDV_ERR_INVALID_ARG;
  for (int b = 0; b < live; ++b)
    if (accepted[b] < 0 || accepted[b] > s->step.gamma) return SDV_ERR_INVALID_ARG;
  int done = 0;
  long long emitted = 0;
  size_t keep = 0;
  for (int b = 0; b < live; ++b) {
    Seq q = s->slots[static_cast<size_t>(b)];
    const int adv = accepted[b] + 1;
    emitted += adv;
    q.len += adv;
    q.gen += adv;
    if (q.gen >= q.limit) {
      s->free_pages += q.pages;
      if (finished_ids) finished_ids[done] = q.id;
      ++done;
      continue;
    }
    const int now = s->pages_for(q.len);
    s->free_pages += q.pages - now;
    q.pages = now;
    s->slots[keep++] = q;  // stable: survivors keep their order
  }
  s->slots.resize(keep);
  if (n_finished) *n_finished = done;
  s->stats.steps += 1;
  s->stats.emitted += emitted;
  s->stats.slot_steps_paid += s->step.width;
  s->stats.slot_steps_live += live;
  s->stats.finished += done;
  s->stats.free_pages = s->free_pages;
  if (s->slots.empty()) s->group_width = 0;
  s->planned = false;
  return SDV_OK;
}

sdv_status sdv_sched_get_stats(const sdv_sched* s, sdv_sched_stats* st) {
  if (!s || !st) return SDV_ERR_INVALID_ARG;
  *st = s->stats;
  st->queued = static_cast<int>(s->queue.size());
  st->free_pages = s->free_pages;
  st->live = static_cast<int>(s->slots.size());
  return SDV_OK;
}

sdv_status sdv_sched_slots(const sdv_sched* s, int* seq_lens, int* gen_counts, int* out_lens, int* num_pages) {
  if (!s) return SDV_ERR_INVALID_ARG;
  for (size_t b = 0; b < s->slots.size(); ++b) {
    const Seq& q = s->slots[b];
    if (seq_lens) seq_lens[b] = q.len;
    if (gen_counts) gen_counts[b] = q.gen;
    if (out_lens) out_lens[b] = q.limit;
    if (num_pages) num_pages[b] = q.pages;
  }
  return SDV_OK;
}

}  // extern "C"
