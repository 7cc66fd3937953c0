// Continuous batching around the decode plan: a request scheduler with a KV
// page allocator (host only), and the serving-loop step that drives a plan
// with it.
//
// "Cohere Publishes One-Kernel Server for North Mini Code" ("A hand-built
// approach to a specialized server") and "Inside the Megakernel Serving
// Engine for North Mini Code" (architecture paragraph) present the
// megakernel as the engine of a server that admits requests continuously
// into a paged KV cache with ragged lengths.  They leave the host policy
// open; this one reserves each request's pages at admission, admits first
// come first served, feeds the prompt through the decode tasks (one token per
// step, or prefill chunks of several rows) and retires on a token budget or an
// end token (see include/mk.h).
#include <algorithm>
#include <deque>
#include <unordered_map>
#include <vector>

#include "mk.h"

namespace mk {
void set_last_error(const char* msg);
// plan.cu: a step enqueued from host tokens without waiting, its wait, and a
// task list built ahead for a batch's lengths
int plan_step_host_begin(mk_plan* p, const int* h_tokens, mk_stream stream);
int plan_step_host_end(mk_plan* p, int* h_next, mk_stream stream);
void plan_prebuild(mk_plan* p, int batch, const int* seq_lens);
}

struct mk_sched {
  struct Req {
    std::vector<int> prompt;
    int max_new = 0, eos = -1;
    std::vector<int> out;
    std::vector<int> pages;
    int len = 0;      // tokens in the cache
    bool done = false;
  };
  int num_pages = 0, ps = 0, max_batch = 0, max_pages = 0;
  int max_chunk = 1;                    // prompt tokens a request may feed in one step (rows)
  bool had_chunks = false;              // the last batch handed out held a multi-row chunk
  std::vector<int> rows_of;             // rows each active request took in the pending batch
  std::vector<int> free_pages;          // a stack of free page ids
  std::deque<long long> queue;          // submitted, not admitted (arrival order)
  std::vector<long long> active;        // admitted, in batch order
  std::unordered_map<long long, Req> reqs;
  bool pending = false;                 // a batch was handed out and awaits commit or abandon
  bool changed = true;                  // the admitted set differs from the last batch handed out
  int retired = 0;
  long long steps = 0;

  // cached positions a request uses: its prompt, then every output but the last
  static long long positions(const Req& r) { return (long long)r.prompt.size() + r.max_new - 1; }
  long long pages_for(const Req& r) const { return (positions(r) + ps - 1) / ps; }
};

namespace {

int fail(int code, const char* msg) {
  mk::set_last_error(msg);
  return code;
}

}  // namespace

extern "C" {

int mk_sched_create(int num_pages, int page_size, int max_batch, int max_pages_per_seq, mk_sched** out) {
  if (!out || num_pages < 1 || page_size < 1 || max_batch < 1 || max_pages_per_seq < 1)
    return fail(MK_ERR_INVALID, "mk_sched_create: every size must be positive");
  mk_sched* s = new mk_sched;
  s->num_pages = num_pages;
  s->ps = page_size;
  s->max_batch = max_batch;
  s->max_pages = max_pages_per_seq;
  s->free_pages.resize(num_pages);
  for (int i = 0; i < num_pages; ++i) s->free_pages[i] = num_pages - 1 - i;   // page 0 is handed out first
  *out = s;
  return MK_OK;
}

int mk_sched_submit(mk_sched* s, long long rid, const int* prompt, int n_prompt, int max_new_tokens,
                    int eos_token) {
  if (!s || !prompt || n_prompt < 1 || max_new_tokens < 1)
    return fail(MK_ERR_INVALID, "mk_sched_submit: needs a prompt of at least one token and max_new_tokens >= 1");
  if (s->reqs.count(rid)) return fail(MK_ERR_INVALID, "mk_sched_submit: request id already held");
  for (int i = 0; i < n_prompt; ++i)
    if (prompt[i] < 0) return fail(MK_ERR_INVALID, "mk_sched_submit: negative prompt token");
  mk_sched::Req r;
  r.prompt.assign(prompt, prompt + n_prompt);
  r.max_new = max_new_tokens;
  r.eos = eos_token;
  const long long need = s->pages_for(r);
  if (need > s->max_pages || need > s->num_pages)
    return fail(MK_ERR_CAPACITY, "mk_sched_submit: the request's sequence needs more pages than a row or the pool");
  s->reqs.emplace(rid, std::move(r));
  s->queue.push_back(rid);
  return MK_OK;
}

int mk_sched_set_prefill(mk_sched* s, int max_chunk) {
  if (!s || max_chunk < 1 || max_chunk > 8) return fail(MK_ERR_INVALID, "mk_sched_set_prefill: max_chunk in 1 .. 8");
  if (s->pending) return fail(MK_ERR_INVALID, "mk_sched_set_prefill: a batch is pending");
  s->max_chunk = max_chunk;
  return MK_OK;
}

int mk_sched_next_rows(mk_sched* s, int* rows, int* seq_lens, int* page_table, int* tokens, long long* rids,
                       int* chunk_first, int* changed) {
  if (!s || !rows || !seq_lens || !page_table || !tokens || !rids || !chunk_first || !changed)
    return fail(MK_ERR_INVALID, "mk_sched_next_rows: null argument");
  if (s->pending) return fail(MK_ERR_INVALID, "mk_sched_next: the previous batch was neither committed nor abandoned");
  // admission: first come, first served, while a slot and the head's pages are free
  while (!s->queue.empty() && (int)s->active.size() < s->max_batch) {
    mk_sched::Req& r = s->reqs.at(s->queue.front());
    const long long need = s->pages_for(r);
    if (need > (long long)s->free_pages.size()) break;
    r.pages.assign(s->free_pages.end() - need, s->free_pages.end());
    std::reverse(r.pages.begin(), r.pages.end());
    s->free_pages.resize(s->free_pages.size() - need);
    s->active.push_back(s->queue.front());
    s->queue.pop_front();
    s->changed = true;
  }
  // rows: one per request, then the spare rows to requests still in their
  // prompt, in batch order, up to max_chunk each and the prompt's remaining
  // tokens; above 8 rows a chunk ends at the next multiple of 8 (one launch)
  const int A = (int)s->active.size();
  s->rows_of.assign(A, 1);
  int spare = s->max_batch - A;
  for (int a = 0; a < A && spare > 0; ++a) {
    const mk_sched::Req& r = s->reqs.at(s->active[a]);
    const int left = (int)r.prompt.size() - r.len;
    const int extra = std::min(spare, std::min(s->max_chunk, left) - 1);
    if (extra > 0) {
      s->rows_of[a] += extra;
      spare -= extra;
    }
  }
  int row = 0;
  bool chunks = false;
  for (int a = 0; a < A; ++a) {
    if (s->max_batch > 8) s->rows_of[a] = std::min(s->rows_of[a], 8 - row % 8);
    const mk_sched::Req& r = s->reqs.at(s->active[a]);
    const int np = (int)r.prompt.size();
    for (int j = 0; j < s->rows_of[a]; ++j, ++row) {
      seq_lens[row] = r.len + j;
      tokens[row] = r.len + j < np ? r.prompt[r.len + j] : r.out.back();
      rids[row] = s->active[a];
      chunk_first[row] = row - j;
      int* pr = page_table + (size_t)row * s->max_pages;
      for (int i = 0; i < s->max_pages; ++i) pr[i] = i < (int)r.pages.size() ? r.pages[i] : -1;
    }
    chunks |= s->rows_of[a] > 1;
  }
  *rows = row;
  *changed = row > 0 && (s->changed || chunks || s->had_chunks) ? 1 : 0;
  if (row > 0) {
    s->pending = true;
    s->changed = false;
    s->had_chunks = chunks;
  }
  return MK_OK;
}

int mk_sched_next(mk_sched* s, int* batch, int* seq_lens, int* page_table, int* tokens, long long* rids,
                  int* changed) {
  if (!s || !batch || !seq_lens || !page_table || !tokens || !rids || !changed)
    return fail(MK_ERR_INVALID, "mk_sched_next: null argument");
  if (s->max_chunk != 1) return fail(MK_ERR_INVALID, "mk_sched_next: prefill chunks need mk_sched_next_rows");
  std::vector<int> cf(s->max_batch);
  return mk_sched_next_rows(s, batch, seq_lens, page_table, tokens, rids, cf.data(), changed);
}

int mk_sched_peek_rows(const mk_sched* s, int* rows, int* seq_lens, int* page_table, int* tokens, long long* rids,
                       int* chunk_first) {
  if (!s || !rows || !seq_lens || !page_table || !tokens || !rids || !chunk_first)
    return fail(MK_ERR_INVALID, "mk_sched_peek_rows: null argument");
  mk_sched c = *s;   // the prediction runs on a copy; the scheduler itself does not change
  if (c.pending) {
    // commit the pending batch with outputs that are no request's end token
    std::vector<int> fake(c.rows_of.empty() ? 1 : (size_t)c.max_batch, -2);
    const int rc = mk_sched_commit(&c, fake.data());
    if (rc != MK_OK) return rc;
  }
  int changed = 0;
  return mk_sched_next_rows(&c, rows, seq_lens, page_table, tokens, rids, chunk_first, &changed);
}

int mk_sched_commit(mk_sched* s, const int* next_tokens) {
  if (!s || !next_tokens) return fail(MK_ERR_INVALID, "mk_sched_commit: null argument");
  if (!s->pending) return fail(MK_ERR_INVALID, "mk_sched_commit: no batch is pending");
  std::vector<long long> keep;
  keep.reserve(s->active.size());
  int row = 0;
  for (size_t b = 0; b < s->active.size(); ++b) {
    mk_sched::Req& r = s->reqs.at(s->active[b]);
    const int n = s->rows_of[b];
    r.len += n;
    row += n;
    if (r.len >= (int)r.prompt.size()) {   // the last row's input was the last prompt token or an output
      const int tok = next_tokens[row - 1];
      r.out.push_back(tok);
      if ((int)r.out.size() >= r.max_new || (r.eos >= 0 && tok == r.eos)) r.done = true;
    }
    if (r.done) {
      s->free_pages.insert(s->free_pages.end(), r.pages.rbegin(), r.pages.rend());
      r.pages.clear();
      s->retired += 1;
      s->changed = true;
    } else {
      keep.push_back(s->active[b]);
    }
  }
  s->active.swap(keep);
  s->pending = false;
  s->steps += 1;
  return MK_OK;
}

int mk_sched_abandon(mk_sched* s) {
  if (!s) return fail(MK_ERR_INVALID, "mk_sched_abandon: null scheduler");
  if (!s->pending) return fail(MK_ERR_INVALID, "mk_sched_abandon: no batch is pending");
  s->pending = false;
  s->changed = true;
  return MK_OK;
}

int mk_sched_result(const mk_sched* s, long long rid, int* tokens, int cap, int* n_tokens, int* done) {
  if (!s || !n_tokens || !done || cap < 0 || (cap > 0 && !tokens))
    return fail(MK_ERR_INVALID, "mk_sched_result: bad argument");
  auto it = s->reqs.find(rid);
  if (it == s->reqs.end()) return fail(MK_ERR_INVALID, "mk_sched_result: unknown request id");
  const std::vector<int>& o = it->second.out;
  const int n = (int)o.size();
  for (int i = 0; i < std::min(cap, n); ++i) tokens[i] = o[i];
  *n_tokens = n;
  *done = it->second.done ? 1 : 0;
  return MK_OK;
}

int mk_sched_forget(mk_sched* s, long long rid) {
  if (!s) return fail(MK_ERR_INVALID, "mk_sched_forget: null scheduler");
  auto it = s->reqs.find(rid);
  if (it == s->reqs.end() || !it->second.done)
    return fail(MK_ERR_INVALID, "mk_sched_forget: unknown or unfinished request");
  s->reqs.erase(it);
  s->retired -= 1;
  return MK_OK;
}

int mk_sched_stats(const mk_sched* s, int* out, int n) {
  if (!s || !out || n < 0) return fail(MK_ERR_INVALID, "mk_sched_stats: bad argument");
  const int v[5] = {(int)s->queue.size(), (int)s->active.size(), s->retired, (int)s->free_pages.size(),
                    (int)std::min<long long>(s->steps, 0x7fffffff)};
  for (int i = 0; i < std::min(n, 5); ++i) out[i] = v[i];
  return MK_OK;
}

void mk_sched_destroy(mk_sched* s) { delete s; }

int mk_serve_step(mk_sched* s, mk_plan** plan, const mk_model_dims* dims, const mk_weights* w, const mk_kv* kv,
                  const mk_plan_opts* opts, mk_stream stream) {
  if (!s || !plan) return fail(MK_ERR_INVALID, "mk_serve_step: null argument");
  if (!*plan && (!dims || !w || !kv)) return fail(MK_ERR_INVALID, "mk_serve_step: a new plan needs dims, w and kv");
  const int cap = s->max_batch;
  std::vector<int> seq(cap), pt((size_t)cap * s->max_pages), tok(cap), nxt(cap), cf(cap);
  std::vector<long long> rid(cap);
  int B = 0, changed = 0;
  int rc = mk_sched_next_rows(s, &B, seq.data(), pt.data(), tok.data(), rid.data(), cf.data(), &changed);
  if (rc != MK_OK || B == 0) return rc;
  if (!*plan) {
    mk_plan_opts o{};
    if (opts) o = *opts;
    if (o.max_batch == 0) o.max_batch = cap;
    if (o.max_batch < cap || kv->num_pages < s->num_pages) {
      mk_sched_abandon(s);
      return fail(MK_ERR_INVALID, "mk_serve_step: plan capacity below max_batch, or KV pool smaller than the scheduler's");
    }
    o.chunk_first = cf.data();
    rc = mk_plan_create(dims, w, kv, B, seq.data(), pt.data(), s->max_pages, &o, plan);
  } else if (changed) {
    rc = mk_plan_update_rows(*plan, B, seq.data(), pt.data(), s->max_pages, cf.data(), stream);
  }
  if (rc == MK_OK) rc = mk::plan_step_host_begin(*plan, tok.data(), stream);
  if (rc == MK_OK) {
    // while the GPU runs this step, build the task list of the batch the
    // next call will most likely run (no request ending on its end token)
    std::vector<int> pseq(cap), ppt((size_t)cap * s->max_pages), ptok(cap), pcf(cap);
    std::vector<long long> prid(cap);
    int PB = 0;
    if (mk_sched_peek_rows(s, &PB, pseq.data(), ppt.data(), ptok.data(), prid.data(), pcf.data()) == MK_OK && PB > 0)
      mk::plan_prebuild(*plan, PB, pseq.data());
    rc = mk::plan_step_host_end(*plan, nxt.data(), stream);
  }
  if (rc != MK_OK) {
    mk_sched_abandon(s);
    return rc;
  }
  rc = mk_sched_commit(s, nxt.data());
  return rc == MK_OK ? B : rc;
}

}  // extern "C"
