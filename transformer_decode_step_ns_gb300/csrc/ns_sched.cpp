// Constant-dense-batch former: host-side formation of each step's rows.
//
// "NanoFlow: ..." page, "Runtime details that keep the pipeline fed": an overlap schedule tuned
// for one dense batch size only holds if every iteration has that size, so the scheduler takes
// the unfinished decode requests first and tops the batch up to exactly the target token count
// with prefill chunks cut at token granularity; requests that outgrow their predicted peak
// memory are moved to the host and reloaded later instead of being recomputed.  Each step's rows
// are written straight into the metadata arrays ns_decode_step takes; KV blocks come from an
// ns_pool (a handle's own pool via ns_kv_get_pool, or a standalone one).
//
// Policy details where the page gives none (stated in full in ns.h):
//   * decode rows first, one per running request, in running order (prompt completion, resumed
//     requests last); at most dense_tokens of them;
//   * then prompts in arrival order, each contributing its next min(room, remaining) tokens as
//     consecutive positions over its own block table, cut to what the free blocks hold; a
//     prompt starts only when the free blocks cover its predicted peak plus what the admitted
//     requests still need to reach theirs and what the preempted ones need to resume;
//   * when the decode rows lack blocks, the last running request is preempted (its cached K/V
//     saved by the caller, its blocks freed); in a step without preemption the preempted
//     requests resume first in, first out, while they fit (new blocks, K/V reloaded);
//   * blocks are reserved as positions cross block boundaries, in row order;
//   * a row samples when it is a decode row or a prompt's last token; a request finishes on
//     eos_token or at max_new_tokens, and its blocks return to the pool in table order.
#include <algorithm>
#include <deque>
#include <map>
#include <string>
#include <vector>

#include "ns.h"
#include "ns_host.h"

namespace {

struct Request {
  int id = 0;
  std::vector<int32_t> prompt;
  int max_new = 0;
  int peak = 0;  // predicted peak, in blocks
  int done = 0;  // prompt tokens already placed in a step
  std::vector<int32_t> gen;
  std::vector<int32_t> table;
  bool finished = false;
  std::deque<std::pair<long long, int>> inflight;  // (step, row) of formed sampling rows
};

struct Row {
  int id, token, pos, samples;
};

struct Move {
  int kind, id, n_tokens;  // kind 0: save from `table`, 1: reload into `table`
  std::vector<int32_t> table;
};

ns_status err(ns_status s, const char* m) {
  ns::set_last_error(m);
  return s;
}

}  // namespace

struct ns_sched_st {
  ns_pool pool = nullptr;
  int D = 0, mb = 0, bs = 0, nb = 0, eos = 0, pred = 0;
  std::map<int, Request> req;
  std::deque<int> prefill;  // ids with prompt left, arrival order
  std::vector<int> running;  // ids decoding, prompt-completion order (resumed ones appended)
  std::deque<int> swapped;  // preempted ids, preemption order
  bool async_mode = false;
  long long seq = 0;                                        // next step number
  std::deque<std::pair<long long, std::vector<Row>>> pending;  // formed, not committed
  std::vector<Row> rows;    // the step being formed
  std::vector<Move> moves;  // saves and reloads the formed step needs first

  int blocks(long long n_pos) const { return static_cast<int>((n_pos + bs - 1) / bs); }
  // running requests that get a decode row: the first D whose formed rows are below max_new
  std::vector<int> decoding() {
    std::vector<int> out;
    for (int id : running) {
      if (static_cast<int>(out.size()) >= D) break;
      const Request& r = req[id];
      if (static_cast<int>(r.gen.size() + r.inflight.size()) < r.max_new) out.push_back(id);
    }
    return out;
  }
  int decode_need() {
    int need = 0;
    for (int id : decoding())
      if (pos_next(req[id]) % bs == 0) ++need;
    return need;
  }

  int free_blocks() const {
    int n = 0;
    ns_pool_free_count(pool, &n);
    return n;
  }
  int pos_next(const Request& r) const {
    return static_cast<int>(r.prompt.size() + r.gen.size() + r.inflight.size()) - 1;
  }
};

extern "C" {

ns_status ns_sched_create(ns_pool pool, int dense_tokens, int max_blocks_per_seq, int eos_token,
                          int predicted_new_tokens, ns_sched* out) {
  if (pool == nullptr || out == nullptr) return err(NS_ERR_INVALID_ARG, "null argument");
  if (dense_tokens < 1 || max_blocks_per_seq < 1 || predicted_new_tokens < 0)
    return err(NS_ERR_INVALID_ARG, "dense_tokens, max_blocks_per_seq positive; predicted_new_tokens >= 0");
  int bs = 0, nb = 0;
  if (ns_pool_geometry(pool, &nb, &bs) != NS_OK) return NS_ERR_INVALID_ARG;
  ns_sched_st* s = new ns_sched_st();
  s->pool = pool;
  s->D = dense_tokens;
  s->mb = max_blocks_per_seq;
  s->bs = bs;
  s->nb = nb;
  s->eos = eos_token;
  s->pred = predicted_new_tokens;
  *out = s;
  return NS_OK;
}

void ns_sched_destroy(ns_sched s) { delete s; }

ns_status ns_sched_add(ns_sched s, int request_id, const int32_t* prompt, int prompt_len,
                       int max_new_tokens) {
  if (s == nullptr || (prompt_len > 0 && prompt == nullptr)) return err(NS_ERR_INVALID_ARG, "null argument");
  if (request_id < 0 || s->req.count(request_id)) return err(NS_ERR_INVALID_ARG, "request id in use or negative");
  if (prompt_len < 1 || max_new_tokens < 1) return err(NS_ERR_INVALID_ARG, "empty prompt or max_new_tokens < 1");
  // negative ids are how a formed row names a device-sampled token: never a prompt's
  for (int i = 0; i < prompt_len; ++i)
    if (prompt[i] < 0) return err(NS_ERR_INVALID_ARG, "negative prompt token id");
  if (static_cast<long long>(prompt_len) + max_new_tokens > static_cast<long long>(s->mb) * s->bs)
    return err(NS_ERR_INVALID_ARG, "prompt + max_new_tokens beyond the block table");
  if (s->blocks(static_cast<long long>(prompt_len) + max_new_tokens - 1) > s->nb)
    return err(NS_ERR_INVALID_ARG, "prompt + max_new_tokens beyond the pool");
  Request r;
  r.id = request_id;
  r.prompt.assign(prompt, prompt + prompt_len);
  r.max_new = max_new_tokens;
  const int predicted = s->pred == 0 ? max_new_tokens : std::min(max_new_tokens, s->pred);
  r.peak = s->blocks(static_cast<long long>(prompt_len) + predicted - 1);
  s->req.emplace(request_id, std::move(r));
  s->prefill.push_back(request_id);
  return NS_OK;
}

ns_status ns_sched_next(ns_sched s, int32_t* token_ids, int32_t* positions, int32_t* block_tables,
                        int32_t* seq_lens, int64_t* slot_mapping, int32_t* row_request,
                        int32_t* row_samples, int* batch) {
  if (s == nullptr || !token_ids || !positions || !block_tables || !seq_lens || !slot_mapping ||
      !row_request || !row_samples || !batch)
    return err(NS_ERR_INVALID_ARG, "null argument");
  if (s->pending.size() >= (s->async_mode ? 2u : 1u)) return err(NS_ERR_INVALID_ARG, "commit the previous step first");
  const int bs = s->bs;
  s->moves.clear();
  // preempt the last running request while the decode rows lack blocks
  bool preempted = false;
  while (s->decode_need() > s->free_blocks()) {
    Request& r = s->req[s->running.back()];
    s->running.pop_back();
    s->moves.push_back({0, r.id, s->pos_next(r), r.table});
    if (!r.table.empty()) ns_pool_release(s->pool, r.table.data(), static_cast<int>(r.table.size()));
    r.table.clear();
    s->swapped.push_back(r.id);
    preempted = true;
  }
  // resume preempted requests, first in first out, while they fit
  while (!preempted && !s->swapped.empty()) {
    Request& r = s->req[s->swapped.front()];
    const int n = s->pos_next(r);
    const int extra = (s->running.size() < static_cast<size_t>(s->D) && n % bs == 0) ? 1 : 0;
    if (s->free_blocks() - s->decode_need() < s->blocks(n) + extra) break;
    s->swapped.pop_front();
    r.table.assign(s->blocks(n), 0);
    if (!r.table.empty()) ns_pool_reserve(s->pool, static_cast<int>(r.table.size()), r.table.data());
    s->moves.push_back({1, r.id, n, r.table});
    s->running.push_back(r.id);
  }
  s->rows.clear();
  for (int id : s->decoding()) {
    Request& r = s->req[id];
    const int p = s->pos_next(r);
    if (p % bs == 0) {
      int32_t b = 0;
      ns_pool_reserve(s->pool, 1, &b);
      r.table.push_back(b);
    }
    // a token not committed yet is the one sampled at the request's row of the previous step
    const int tok = r.inflight.empty() ? r.gen.back() : -(r.inflight.back().second + 1);
    s->rows.push_back({r.id, tok, p, 1});
  }
  int room = s->D - static_cast<int>(s->rows.size());
  for (int id : s->prefill) {
    if (room <= 0) break;
    Request& r = s->req[id];
    if (r.done == 0) {
      // admission against the predicted peaks
      long long owed = 0;
      for (const auto& kv : s->req) {
        const Request& q = kv.second;
        if (!q.table.empty() && !q.finished) owed += std::max(0, q.peak - static_cast<int>(q.table.size()));
      }
      for (int i : s->swapped) owed += s->blocks(static_cast<long long>(s->pos_next(s->req[i])) + 1);
      if (s->free_blocks() < r.peak + owed) break;
    }
    const int left = static_cast<int>(r.prompt.size()) - r.done;
    int c = std::min(room, left);
    const long long fit = (static_cast<long long>(r.table.size()) + s->free_blocks()) * bs - r.done;
    if (fit < c) c = static_cast<int>(std::max(0LL, fit));
    if (c <= 0) break;
    const int want = (r.done + c + bs - 1) / bs - static_cast<int>(r.table.size());
    if (want > 0) {
      std::vector<int32_t> ids(want);
      ns_pool_reserve(s->pool, want, ids.data());
      r.table.insert(r.table.end(), ids.begin(), ids.end());
    }
    for (int k = 0; k < c; ++k) {
      const int p = r.done + k;
      s->rows.push_back({id, r.prompt[p], p, p == static_cast<int>(r.prompt.size()) - 1 ? 1 : 0});
    }
    r.done += c;
    room -= c;
  }
  const int B = static_cast<int>(s->rows.size());
  const long long step = s->seq++;
  for (int b = 0; b < B; ++b) {
    const Row& w = s->rows[b];
    if (!w.samples) continue;
    Request& r = s->req[w.id];
    if (w.pos == static_cast<int>(r.prompt.size()) - 1) {  // the prompt completes: it runs from now
      s->prefill.erase(std::find(s->prefill.begin(), s->prefill.end(), r.id));
      s->running.push_back(r.id);
    }
    r.inflight.push_back({step, b});
  }
  for (int b = 0; b < B; ++b) {
    const Row& w = s->rows[b];
    const std::vector<int32_t>& t = s->req[w.id].table;
    token_ids[b] = w.token;
    positions[b] = w.pos;
    seq_lens[b] = w.pos + 1;
    int32_t* row = block_tables + static_cast<size_t>(b) * s->mb;
    std::fill(row, row + s->mb, 0);
    std::copy(t.begin(), t.end(), row);
    slot_mapping[b] = static_cast<int64_t>(t[w.pos / bs]) * bs + w.pos % bs;
    row_request[b] = w.id;
    row_samples[b] = w.samples;
  }
  *batch = B;
  s->pending.push_back({step, s->rows});
  return NS_OK;
}

ns_status ns_sched_commit(ns_sched s, const int32_t* sampled, int batch, int32_t* finished_ids,
                          int* n_finished) {
  if (s == nullptr || (batch > 0 && sampled == nullptr) || n_finished == nullptr)
    return err(NS_ERR_INVALID_ARG, "null argument");
  if (s->pending.empty()) return err(NS_ERR_INVALID_ARG, "no step to commit");
  if (batch != static_cast<int>(s->pending.front().second.size()))
    return err(NS_ERR_INVALID_ARG, "batch differs from the formed step");
  const long long step = s->pending.front().first;
  const std::vector<Row> rows = std::move(s->pending.front().second);
  s->pending.pop_front();
  int nf = 0;
  for (int b = 0; b < batch; ++b) {
    const Row& w = rows[b];
    if (!w.samples) continue;
    Request& r = s->req[w.id];
    r.inflight.erase(std::find(r.inflight.begin(), r.inflight.end(), std::make_pair(step, b)));
    if (!r.finished) {  // a row formed after the request's eos: its token is dropped
      const int32_t tok = sampled[b];
      r.gen.push_back(tok);
      if (tok == s->eos || static_cast<int>(r.gen.size()) == r.max_new) {
        r.finished = true;
        s->running.erase(std::find(s->running.begin(), s->running.end(), r.id));
        if (finished_ids != nullptr) finished_ids[nf] = r.id;
        ++nf;
      }
    }
    if (r.finished && r.inflight.empty() && !r.table.empty()) {
      ns_pool_release(s->pool, r.table.data(), static_cast<int>(r.table.size()));
      r.table.clear();
    }
  }
  *n_finished = nf;
  return NS_OK;
}

ns_status ns_sched_set_async(ns_sched s, int on) {
  if (s == nullptr) return err(NS_ERR_INVALID_ARG, "null argument");
  if (on && s->pred != 0) return err(NS_ERR_INVALID_ARG, "asynchronous formation needs every peak reserved");
  if (!s->pending.empty()) return err(NS_ERR_INVALID_ARG, "commit the formed steps first");
  s->async_mode = on != 0;
  return NS_OK;
}

ns_status ns_sched_tokens(ns_sched s, int request_id, int32_t* out, int capacity, int* n) {
  if (s == nullptr || n == nullptr || (capacity > 0 && out == nullptr)) return err(NS_ERR_INVALID_ARG, "null argument");
  auto it = s->req.find(request_id);
  if (it == s->req.end()) return err(NS_ERR_INVALID_ARG, "unknown request id");
  const std::vector<int32_t>& g = it->second.gen;
  *n = static_cast<int>(g.size());
  std::copy(g.begin(), g.begin() + std::min(static_cast<int>(g.size()), std::max(capacity, 0)), out);
  return NS_OK;
}

ns_status ns_sched_remove(ns_sched s, int request_id) {
  if (s == nullptr) return err(NS_ERR_INVALID_ARG, "null argument");
  auto it = s->req.find(request_id);
  if (it == s->req.end()) return err(NS_ERR_INVALID_ARG, "unknown request id");
  if (!it->second.finished || !it->second.inflight.empty())
    return err(NS_ERR_INVALID_ARG, "request not finished (or a formed row of it not committed)");
  s->req.erase(it);
  return NS_OK;
}

ns_status ns_sched_counts(ns_sched s, int* waiting, int* running, int* preempted, int* finished) {
  if (s == nullptr || !waiting || !running || !preempted || !finished)
    return err(NS_ERR_INVALID_ARG, "null argument");
  int fin = 0;
  for (const auto& kv : s->req) fin += kv.second.finished ? 1 : 0;
  *waiting = static_cast<int>(s->prefill.size());
  *running = static_cast<int>(s->running.size());
  *preempted = static_cast<int>(s->swapped.size());
  *finished = fin;
  return NS_OK;
}

ns_status ns_sched_moves(ns_sched s, int32_t* kinds, int32_t* request_ids, int32_t* n_tokens,
                         int32_t* tables, int capacity, int* n) {
  if (s == nullptr || n == nullptr) return err(NS_ERR_INVALID_ARG, "null argument");
  if (capacity > 0 && (!kinds || !request_ids || !n_tokens || !tables))
    return err(NS_ERR_INVALID_ARG, "null argument");
  const int m = static_cast<int>(s->moves.size());
  for (int i = 0; i < std::min(m, std::max(capacity, 0)); ++i) {
    const Move& v = s->moves[i];
    kinds[i] = v.kind;
    request_ids[i] = v.id;
    n_tokens[i] = v.n_tokens;
    int32_t* row = tables + static_cast<size_t>(i) * s->mb;
    std::fill(row, row + s->mb, 0);
    std::copy(v.table.begin(), v.table.end(), row);
  }
  *n = m;
  return NS_OK;
}

}  // extern "C"
