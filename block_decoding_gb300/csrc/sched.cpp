// Step-level scheduler of cached block decoding: deficit token budget,
// admission and eviction between denoising steps (Sangam abstract; serving
// study, design principles). Host code only; the rules are stated in
// include/dllm_sched.h.

#include "dllm_sched.h"

#include <algorithm>
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

namespace {

enum class St { kQueued, kReady, kDecoding, kDone };

struct Req {
  int id, P, T, nblocks;
  int block = 0;
  int slot = -1;
  St st = St::kQueued;
};

}  // namespace

struct dllm_sched {
  dllm_sched_config c;
  long long D = 0;
  std::vector<int> slot_req;  // request id per slot, -1 = free
  std::vector<int> queue;     // prefill FIFO of request ids
  std::unordered_map<int, Req> reqs;
  std::vector<int> last;      // request ids of the last plan
  bool planned = false;
  std::deque<int> finished;
};

namespace {

bool config_ok(const dllm_sched_config &c) {
  if (c.slots < 1 || c.slots > 4096 || c.blk < 1 || c.blk > 64 || c.vic < 0 || c.quantum < 0 ||
      c.budget_cap < c.quantum || c.max_seq < c.blk || c.policy < 0 || c.policy > 2)
    return false;
  const long long decode_rows = static_cast<long long>(c.slots) * (c.blk + 2LL * c.vic);
  return c.max_step_rows >= decode_rows && c.max_step_rows >= c.max_seq;
}

int free_slot(const dllm_sched &s) {
  for (int i = 0; i < s.c.slots; ++i)
    if (s.slot_req[i] < 0) return i;
  return -1;
}

dllm_sched_entry make_entry(const dllm_sched &s, const Req &r, int kind) {
  const int b0 = r.P + r.block * s.c.blk;
  dllm_sched_entry e{};
  e.slot = r.slot;
  e.req = r.id;
  e.block = r.block;
  e.kind = kind;
  e.b0 = b0;
  if (kind == 1) {
    e.q_pos0 = 0;
    e.q_rows = r.T;
    e.kv_rows = r.T;
  } else {
    const int ws = std::max(0, b0 - s.c.vic);
    const int we = std::min(r.T, b0 + s.c.blk + s.c.vic);
    e.q_pos0 = ws;
    e.q_rows = we - ws;
    e.kv_rows = s.c.dual_cache ? r.T : we;
  }
  return e;
}

void admit(dllm_sched &s, Req &r) {
  if (r.slot < 0) {
    r.slot = free_slot(s);
    s.slot_req[r.slot] = r.id;
  }
  r.st = St::kDecoding;
}

}  // namespace

extern "C" dllm_status dllm_sched_create(const dllm_sched_config *cfg, dllm_sched **out) {
  if (!cfg || !out || !config_ok(*cfg)) return DLLM_ERR_INVALID_ARG;
  dllm_sched *s = new (std::nothrow) dllm_sched;
  if (!s) return DLLM_ERR_INVALID_ARG;
  s->c = *cfg;
  s->slot_req.assign(cfg->slots, -1);
  *out = s;
  return DLLM_OK;
}

extern "C" void dllm_sched_destroy(dllm_sched *s) { delete s; }

extern "C" dllm_status dllm_sched_submit(dllm_sched *s, int req, int prompt_len, int resp_len) {
  if (!s || req < 0 || s->reqs.count(req) || prompt_len < 0 || resp_len < s->c.blk || resp_len % s->c.blk ||
      static_cast<long long>(prompt_len) + resp_len > s->c.max_seq)
    return DLLM_ERR_INVALID_ARG;
  Req r{req, prompt_len, prompt_len + resp_len, resp_len / s->c.blk};
  s->reqs.emplace(req, r);
  s->queue.push_back(req);
  return DLLM_OK;
}

extern "C" int dllm_sched_plan(dllm_sched *s, dllm_sched_entry *out, int cap) {
  if (!s || !out || cap < s->c.slots || s->planned) return -static_cast<int>(DLLM_ERR_INVALID_ARG);
  const bool budgeted = s->c.policy != DLLM_SCHED_PREFILL_FIRST;
  if (s->c.policy == DLLM_SCHED_DEFICIT)
    s->D = std::min<long long>(s->c.budget_cap, s->D + s->c.quantum);
  else if (s->c.policy == DLLM_SCHED_NO_CARRY)
    s->D = s->c.quantum;
  int n = 0;
  long long used = 0;
  s->last.clear();
  // in-flight decodes first, every one of them
  for (int i = 0; i < s->c.slots; ++i) {
    const int id = s->slot_req[i];
    if (id < 0) continue;
    const Req &r = s->reqs.at(id);
    if (r.st != St::kDecoding) continue;
    out[n] = make_entry(*s, r, 0);
    used += out[n].q_rows;
    if (budgeted) s->D -= out[n].q_rows;
    s->last.push_back(id);
    ++n;
  }
  // whole prefills in FIFO order while the budget and the row cap allow
  std::vector<int> admitted;
  int free_slots = 0;
  for (int i = 0; i < s->c.slots; ++i) free_slots += s->slot_req[i] < 0;
  for (const int id : s->queue) {
    const Req &r = s->reqs.at(id);
    if (r.slot < 0 && free_slots == 0) continue;
    const bool fits_rows = used + r.T <= s->c.max_step_rows;
    const bool fits_budget = !budgeted || r.T <= s->D;
    if (!fits_rows || !fits_budget) break;
    admitted.push_back(id);
    if (r.slot < 0) --free_slots;
    used += r.T;
    if (budgeted) s->D -= r.T;
  }
  // work conservation: never plan an empty step while a prefill could run
  if (n == 0 && admitted.empty()) {
    for (const int id : s->queue) {
      const Req &r = s->reqs.at(id);
      if (r.slot < 0 && free_slots == 0) continue;
      admitted.push_back(id);
      if (budgeted) s->D -= r.T;
      break;
    }
  }
  for (const int id : admitted) {
    Req &r = s->reqs.at(id);
    admit(*s, r);
    s->queue.erase(std::find(s->queue.begin(), s->queue.end(), id));
    out[n++] = make_entry(*s, r, 1);
    s->last.push_back(id);
  }
  s->planned = true;
  return n;
}

extern "C" dllm_status dllm_sched_complete(dllm_sched *s, const int32_t *remaining, const uint8_t *eos) {
  if (!s || !remaining || !s->planned) return DLLM_ERR_INVALID_ARG;
  for (const int id : s->last) {
    Req &r = s->reqs.at(id);
    if (remaining[r.slot] > 0) continue;
    const bool ended = eos && eos[r.slot];
    if (r.block + 1 < r.nblocks && !ended) {
      ++r.block;
      r.st = St::kReady;
      s->queue.push_back(id);
    } else {
      r.st = St::kDone;
      s->slot_req[r.slot] = -1;
      r.slot = -1;
      s->finished.push_back(id);
    }
  }
  s->last.clear();
  s->planned = false;
  return DLLM_OK;
}

extern "C" long long dllm_sched_budget(const dllm_sched *s) { return s ? s->D : 0; }

extern "C" int dllm_sched_queued(const dllm_sched *s) { return s ? static_cast<int>(s->queue.size()) : 0; }

extern "C" int dllm_sched_finished(dllm_sched *s, int32_t *req_out, int cap) {
  if (!s || (!req_out && cap > 0)) return 0;
  int n = 0;
  while (n < cap && !s->finished.empty()) {
    req_out[n++] = s->finished.front();
    s->finished.pop_front();
  }
  return n;
}

extern "C" int dllm_sched_pack(const dllm_sched_entry *entries, int n, int slots, int blk, int32_t *q_off,
                               int32_t *kv_off, int32_t *row_req, int32_t *row_pos) {
  if (n < 0 || slots < 1 || blk < 1 || n > slots || (n > 0 && !entries) || !q_off || !kv_off ||
      (n > 0 && (!row_req || !row_pos)))
    return -static_cast<int>(DLLM_ERR_INVALID_ARG);
  std::vector<const dllm_sched_entry *> by_slot(slots, nullptr);
  for (int i = 0; i < n; ++i) {
    const int sl = entries[i].slot;
    if (sl < 0 || sl >= slots || by_slot[sl] || entries[i].q_rows < 0 || entries[i].kv_rows < 0)
      return -static_cast<int>(DLLM_ERR_INVALID_ARG);
    by_slot[sl] = &entries[i];
  }
  long long q = 0, kv = 0;
  int r = 0;
  q_off[0] = kv_off[0] = 0;
  for (int sl = 0; sl < slots; ++sl) {
    const dllm_sched_entry *e = by_slot[sl];
    if (e) {
      q += e->q_rows;
      kv += e->kv_rows;
      if (q > INT32_MAX || kv > INT32_MAX) return -static_cast<int>(DLLM_ERR_INVALID_ARG);
      for (int j = 0; j < blk; ++j, ++r) {
        row_req[r] = sl;
        row_pos[r] = j;
      }
    }
    q_off[sl + 1] = static_cast<int32_t>(q);
    kv_off[sl + 1] = static_cast<int32_t>(kv);
  }
  return r;
}
