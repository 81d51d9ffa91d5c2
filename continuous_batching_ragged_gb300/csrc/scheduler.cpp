// Host scheduler: one iteration-level continuous-batching step per call.
//
// hassanahmed.net, "How Continuous Batching Speeds Up LLM Serving": each pass
// drops finished requests and releases their KV blocks, admits the head of the
// waiting queue while it fits, then runs one forward pass; the KV memory is
// handed out and reclaimed in fixed-size blocks (PagedAttention paragraph).
// Hugging Face blog "Continuous batching from first principles", section
// "Continuous batching": a budget of m tokens per batch, every decoding request
// first at one token each, the remaining room filled with prefill, chunked as
// needed; section "Attention": the pass over the whole prompt yields the first
// new token, each decode pass one more.
//
// The rules the pages leave open are fixed in cb.h (scheduler block).
#include <algorithm>
#include <cstdint>
#include <functional>
#include <queue>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "host_common.h"

namespace {

struct Request {
  int64_t id;
  int64_t arrival;
  int32_t prompt_len;
  int32_t output_len;
  int32_t prefill_len = 0; // tokens of the next prefill: the prompt, or after a preemption every known token
  int32_t computed = 0;    // tokens whose K/V is in the cache
  int32_t generated = 0;   // output tokens produced so far
  int32_t reserved = 0;    // blocks reserved at admission
  std::vector<int32_t> blocks;
};

struct Chosen {
  Request* req;
  int32_t n;
  bool decode;
};

int64_t blocks_needed(const Request& r, int32_t block_size) {
  int64_t tokens = int64_t(r.prompt_len) + int64_t(r.output_len);
  return (tokens + block_size - 1) / block_size;
}

}  // namespace

struct cb_scheduler {
  cb_sched_config cfg;
  int64_t step = 0;
  int64_t finished = 0;
  int64_t reserved_total = 0;
  std::unordered_map<int64_t, Request> all;                 // by id
  std::set<std::pair<int64_t, int64_t>> waiting;            // (arrival, id)
  std::vector<Request*> running;                            // admission order
  std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_blocks;
  std::vector<Chosen> pending;
  bool has_pending = false;
  int64_t num_preempted = 0;
  int64_t recomputed_tokens = 0;
  // output arrays of the last cb_build_batch
  std::vector<int32_t> cu, ctx, bt;
  std::vector<int64_t> slots, ids, evicted, preempted;

  // CB_ADMIT_PROMPT_PREEMPT: give `r`'s blocks back and return it to the
  // waiting queue; its next prefill recomputes every token it knows.
  void preempt(Request* r) {
    for (int32_t b : r->blocks) free_blocks.push(b);
    r->blocks.clear();
    recomputed_tokens += r->computed;
    r->computed = 0;
    r->prefill_len = r->prompt_len + r->generated;
    waiting.emplace(r->arrival, r->id);
    preempted.push_back(r->id);
    ++num_preempted;
  }
  // take `n` blocks, lowest ids first
  void take_blocks(Request* r, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
      r->blocks.push_back(free_blocks.top());
      free_blocks.pop();
    }
  }
};

extern "C" cb_status cb_scheduler_create(const cb_sched_config* config, cb_scheduler** out) {
  if (!config || !out) return cb::fail(CB_ERR_INVALID, "cb_scheduler_create: null argument");
  if (config->token_budget < 1 || config->block_size < 1 || config->num_blocks < 1 ||
      config->max_num_seqs < 0)
    return cb::fail(CB_ERR_INVALID, "cb_scheduler_create: token_budget, block_size and num_blocks "
                                    "must be >= 1 and max_num_seqs >= 0");
  if (config->admission != CB_ADMIT_RESERVE_LIFETIME && config->admission != CB_ADMIT_PROMPT_PREEMPT)
    return cb::fail(CB_ERR_INVALID, "cb_scheduler_create: unknown admission policy %d", config->admission);
  cb_scheduler* s = new (std::nothrow) cb_scheduler();
  if (!s) return cb::fail(CB_ERR_INVALID, "cb_scheduler_create: out of host memory");
  s->cfg = *config;
  for (int32_t b = 0; b < config->num_blocks; ++b) s->free_blocks.push(b);
  *out = s;
  return CB_OK;
}

extern "C" void cb_scheduler_destroy(cb_scheduler* sched) { delete sched; }

extern "C" cb_status cb_add_request(cb_scheduler* s, int64_t id, int64_t arrival_step,
                                    int32_t prompt_len, int32_t output_len) {
  if (!s) return cb::fail(CB_ERR_INVALID, "cb_add_request: null scheduler");
  if (prompt_len < 1 || output_len < 1 || arrival_step < 0)
    return cb::fail(CB_ERR_INVALID, "cb_add_request: prompt_len and output_len must be >= 1, "
                                    "arrival_step >= 0");
  if (s->all.count(id)) return cb::fail(CB_ERR_INVALID, "cb_add_request: duplicate id %lld", (long long)id);
  Request r;
  r.id = id;
  r.arrival = arrival_step;
  r.prompt_len = prompt_len;
  r.output_len = output_len;
  r.prefill_len = prompt_len;
  if (blocks_needed(r, s->cfg.block_size) > s->cfg.num_blocks)
    return cb::fail(CB_ERR_NO_BLOCKS, "cb_add_request: request %lld needs more blocks than the pool",
                    (long long)id);
  s->all.emplace(id, std::move(r));
  s->waiting.emplace(arrival_step, id);
  return CB_OK;
}

extern "C" cb_status cb_build_batch(cb_scheduler* s, cb_batch* out) {
  if (!s || !out) return cb::fail(CB_ERR_INVALID, "cb_build_batch: null argument");
  if (s->has_pending) return cb::fail(CB_ERR_INVALID, "cb_build_batch: previous batch not completed");
  const int32_t B = s->cfg.block_size;

  // 1. evict finished requests and free their blocks
  s->evicted.clear();
  std::vector<Request*> still;
  still.reserve(s->running.size());
  for (Request* r : s->running) {
    if (r->generated == r->output_len) {
      s->evicted.push_back(r->id);
      for (int32_t b : r->blocks) s->free_blocks.push(b);
      s->reserved_total -= r->reserved;
      ++s->finished;
      s->all.erase(r->id);
    } else {
      still.push_back(r);
    }
  }
  s->running.swap(still);

  const bool preempting = s->cfg.admission == CB_ADMIT_PROMPT_PREEMPT;
  s->preempted.clear();
  s->pending.clear();
  int32_t room = s->cfg.token_budget;
  // 2. admit the FIFO head while it has arrived and fits
  auto admit = [&]() {
    while (!s->waiting.empty()) {
      auto head = *s->waiting.begin();
      Request& r = s->all.at(head.second);
      if (r.arrival > s->step) break;
      if (s->cfg.max_num_seqs > 0 && int32_t(s->running.size()) >= s->cfg.max_num_seqs) break;
      if (preempting) {
        // the prefill's blocks, taken now
        const int64_t need = (int64_t(r.prefill_len) + B - 1) / B;
        if (int64_t(s->free_blocks.size()) < need) break;
        s->waiting.erase(s->waiting.begin());
        s->take_blocks(&r, need);
      } else {
        const int64_t need = blocks_needed(r, B);
        if (int64_t(s->cfg.num_blocks) - s->reserved_total < need) break;
        s->waiting.erase(s->waiting.begin());
        r.reserved = int32_t(need);
        s->reserved_total += need;
      }
      s->running.push_back(&r);
    }
  };
  // 3. decode requests first, one token each
  auto choose_decodes = [&]() {
    for (size_t i = 0; i < s->running.size() && room > 0; ++i) {
      Request* r = s->running[i];
      if (r->computed < r->prefill_len) continue;
      if (preempting && r->computed / B >= int32_t(r->blocks.size())) {
        // this token enters a new block: free one by preempting the latest admitted
        while (s->free_blocks.empty() && s->running.back() != r) {
          s->preempt(s->running.back());
          s->running.pop_back();
        }
        if (s->free_blocks.empty()) {           // r is the latest admitted: it goes itself
          s->preempt(r);
          s->running.pop_back();
          break;
        }
        s->take_blocks(r, 1);
      }
      s->pending.push_back({r, 1, true});
      --room;
    }
  };
  if (preempting) {
    // running requests take their blocks before anyone is admitted, and a step
    // that had to preempt admits no one
    choose_decodes();
    if (s->preempted.empty()) admit();
  } else {
    admit();
    choose_decodes();
  }
  const int32_t num_decode = int32_t(s->pending.size());
  // 4. then prefill chunks, greedily in admission order
  for (Request* r : s->running) {
    if (room == 0) break;
    if (r->computed < r->prefill_len) {
      int32_t n = std::min(r->prefill_len - r->computed, room);
      s->pending.push_back({r, n, false});
      room -= n;
    }
  }

  // 5. blocks for the new positions (lowest free id first), 6. metadata
  const int32_t S = int32_t(s->pending.size());
  s->cu.assign(size_t(S) + 1, 0);
  s->ctx.assign(size_t(S), 0);
  s->ids.assign(size_t(S), 0);
  s->slots.clear();
  int32_t width = 0, max_q = 0, max_ctx = 0;
  for (int32_t i = 0; i < S; ++i) {
    Chosen& c = s->pending[i];
    Request* r = c.req;
    for (int32_t k = 0; k < c.n; ++k) {
      int32_t pos = r->computed + k;
      if (pos / B >= int32_t(r->blocks.size())) {
        // reserve-lifetime admission guarantees a free block exists (with
        // preemption every block is already taken)
        s->take_blocks(r, 1);
      }
      s->slots.push_back(int64_t(r->blocks[pos / B]) * B + pos % B);
    }
    s->cu[i + 1] = s->cu[i] + c.n;
    s->ctx[i] = r->computed + c.n;
    s->ids[i] = r->id;
    width = std::max(width, int32_t(r->blocks.size()));
    max_q = std::max(max_q, c.n);
    max_ctx = std::max(max_ctx, s->ctx[i]);
  }
  s->bt.assign(size_t(S) * size_t(width), -1);
  for (int32_t i = 0; i < S; ++i) {
    const std::vector<int32_t>& blk = s->pending[i].req->blocks;
    std::copy(blk.begin(), blk.end(), s->bt.begin() + size_t(i) * width);
  }
  s->has_pending = true;

  out->num_seqs = S;
  out->num_tokens = s->cu[S];
  out->num_decode = num_decode;
  out->max_blocks_per_seq = width;
  out->max_q_len = max_q;
  out->max_context_len = max_ctx;
  out->cu_seqlens_q = s->cu.data();
  out->context_lens = s->ctx.data();
  out->block_tables = s->bt.data();
  out->slot_mapping = s->slots.data();
  out->request_ids = s->ids.data();
  out->num_evicted = int32_t(s->evicted.size());
  out->evicted_ids = s->evicted.data();
  out->num_preempted = int32_t(s->preempted.size());
  out->preempted_ids = s->preempted.data();
  return CB_OK;
}

extern "C" cb_status cb_complete_step(cb_scheduler* s) {
  if (!s) return cb::fail(CB_ERR_INVALID, "cb_complete_step: null scheduler");
  if (!s->has_pending) return cb::fail(CB_ERR_INVALID, "cb_complete_step: no batch was built");
  for (Chosen& c : s->pending) {
    c.req->computed += c.n;
    if (c.decode || c.req->computed == c.req->prefill_len) c.req->generated += 1;
  }
  s->pending.clear();
  s->has_pending = false;
  ++s->step;
  return CB_OK;
}

extern "C" cb_status cb_scheduler_stats(const cb_scheduler* s, cb_sched_stats* out) {
  if (!s || !out) return cb::fail(CB_ERR_INVALID, "cb_scheduler_stats: null argument");
  out->step = s->step;
  out->num_waiting = int32_t(s->waiting.size());
  out->num_running = int32_t(s->running.size());
  out->free_blocks = int32_t(s->free_blocks.size());
  out->reserved_blocks = int32_t(s->reserved_total);
  out->num_finished = s->finished;
  out->num_preempted = s->num_preempted;
  out->recomputed_tokens = s->recomputed_tokens;
  return CB_OK;
}
