// Host side of libmk: the task-list and dependency-counter builder ("Each SM
// gets a task list, and dependencies are tracked with counters in global
// memory" — "Inside the Megakernel Serving Engine for North Mini Code",
// architecture paragraph) and the C ABI of include/mk.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <new>
#include <thread>
#include <vector>

#include "mk.h"
#include "mk_internal.h"

namespace mk {
cudaError_t launch_megakernel(const Params& p, int nb, int grid, int smem, cudaStream_t st);
cudaError_t launch_rope_table(float2* tab, int npos, int d, double theta, cudaStream_t st);
int max_active_ctas(int nb, int smem);
size_t misc_bytes();
}  // namespace mk

using mk::Task;

namespace {

// Text of the most recent failure inside the library (per thread).
thread_local char g_last_error[256] = "";

int note_cuda(cudaError_t e, const char* what) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
  return MK_ERR_CUDA;
}

struct Shape {
  int L, H, nq, nkv, d, E, k, F, V, ps, G, qkv_rows;
  float eps, theta;
};

int check_dims(const mk_model_dims* m, Shape& s) {
  if (!m) return MK_ERR_INVALID;
  s.L = m->n_layers; s.H = m->hidden; s.nq = m->n_q_heads; s.nkv = m->n_kv_heads; s.d = m->head_dim;
  s.E = m->n_experts; s.k = m->top_k; s.F = m->expert_ffn; s.V = m->vocab; s.ps = m->page_size;
  s.eps = m->rms_eps; s.theta = m->rope_theta;
  if (s.L < 1 || s.H < 8 || s.nq < 1 || s.nkv < 1 || s.E < 1 || s.k < 1 || s.F < 8 || s.V < 1)
    return MK_ERR_INVALID;
  if (s.nq % s.nkv) return MK_ERR_INVALID;
  s.G = s.nq / s.nkv;
  if (s.k > s.E || !(s.eps >= 0.f) || !(s.theta > 0.f)) return MK_ERR_INVALID;
  if (s.H % 8 || s.F % 8 || (s.nq * s.d) % 8) return MK_ERR_INVALID;
  if (s.ps != 16) return MK_ERR_UNSUPPORTED;
  if (s.d != 64 && s.d != 128) return MK_ERR_UNSUPPORTED;
  if (s.G > mk::MAX_G || s.k > mk::MAX_TOPK || s.E > mk::MAX_EXPERTS) return MK_ERR_UNSUPPORTED;
  s.qkv_rows = s.nkv * (s.G + 2) * s.d;
  return MK_OK;
}

struct Counts {
  int qkv_per_g = 0, attn = 0, o = 0, gu = 0, down = 0, lm = 0, comb = 0, heads_per_comb = 1;
  int part_slots = 0, pages_per_chunk = 1, down_rows_max = 1;
};

// Phase-balanced assignment: tasks of one phase go, largest first, to the CTA
// with the least work in this phase (ties: least work so far, then lowest id).
// The CTAs sit in a binary min-heap ordered by exactly that key; a task only
// raises the root's key, so one sift-down per task: O(n log C) per phase.
struct Assigner {
  struct Key {
    double ph, tot;
    int c;
  };
  static bool before(const Key& a, const Key& b) {   // a is the better choice than b
    if (a.ph != b.ph) return a.ph < b.ph;
    if (a.tot != b.tot) return a.tot < b.tot;
    return a.c < b.c;
  }
  int C;
  std::vector<std::vector<Task>> per_cta;
  std::vector<double> total;
  std::vector<Key> heap;
  explicit Assigner(int c) : C(c), per_cta(c), total(c, 0.0) {}
  void sift_down(size_t i) {
    const size_t n = heap.size();
    const Key k = heap[i];
    for (;;) {
      size_t ch = 2 * i + 1;
      if (ch >= n) break;
      if (ch + 1 < n && before(heap[ch + 1], heap[ch])) ++ch;
      if (!before(heap[ch], k)) break;
      heap[i] = heap[ch];
      i = ch;
    }
    heap[i] = k;
  }
  void phase(std::vector<std::pair<double, Task>>& ts) {
    std::stable_sort(ts.begin(), ts.end(),
                     [](const std::pair<double, Task>& a, const std::pair<double, Task>& b) {
                       return a.first > b.first;
                     });
    heap.resize(C);
    for (int c = 0; c < C; ++c) heap[c] = {0.0, total[c], c};
    for (size_t i = heap.size() / 2; i-- > 0;) sift_down(i);
    for (auto& t : ts) {
      Key& k = heap[0];
      k.ph += t.first;
      total[k.c] += t.first;
      k.tot = total[k.c];
      per_cta[k.c].push_back(t.second);
      sift_down(0);
    }
  }
};

Task mk_task(int type, int layer, int wait_ctr, uint32_t wait_cnt) {
  Task t;
  memset(&t, 0, sizeof(t));
  t.type = type;
  t.layer = layer;
  t.wait_ctr = wait_ctr;
  t.wait_cnt = wait_cnt;
  return t;
}

// Pages covering positions [0, len] (the cached tokens plus the new one).
inline int pages_for(int len, int ps) { return len / ps + 1; }


// Query heads per split-KV combine task: the smallest divisor of G that keeps
// the tasks (pairs x G / heads) within one per CTA, else all G heads.
inline int comb_heads(int G, int pairs, int C) {
  for (int h = 1; h <= G; ++h)
    if (G % h == 0 && (long long)pairs * (G / h) <= C) return h;
  return G;
}

// First partial slot of (request b, KV group g): slots run request by request,
// group by group, chunk by chunk.
inline int first_slot(const std::vector<int>& nch, int B, int nkv, int b, int g) {
  int s = 0;
  for (int i = 0; i < b; ++i) s += nch[i] * nkv;
  return s + g * nch[b];
}

// Split n items into `parts` nearly equal contiguous ranges.
inline void split_range(int n, int parts, int i, int& a, int& b) {
  a = (int)((long long)n * i / parts);
  b = (int)((long long)n * (i + 1) / parts);
}

// Builds the task list in global topological order, phase by phase, then
// hands each phase's tasks to CTAs; every CTA's list is a subsequence of one
// topological order, so with all CTAs resident the step cannot deadlock.
int build_tasks(const Shape& s, int B, int bcap, const int* seq_lens, int C, int split_pages,
                std::vector<Task>& out, std::vector<int>& cta_start, Counts& cnt,
                std::vector<int>& open_start, bool nucleus = false, bool tcp = false) {
  if (B < 1 || B > bcap || C < 1) return MK_ERR_INVALID;
  mk::CtrMap cm;
  cm.init(s.L, s.nkv, bcap, s.H / 128);
  Assigner asg(C);
  const int Rg = (s.G + 2) * s.d;
  const int nqd = s.nq * s.d;
  // tile counts
  cnt.qkv_per_g = std::max(1, std::min(Rg, (C + s.nkv - 1) / s.nkv));
  cnt.o = std::max(1, std::min(s.H, C));
  // tensor-core projections: each 128-row tile split into kq (QKV) or ko (O)
  // runs of its 128-column K stages, as many as the CTAs allow, each run at
  // most TC_PROJ_UNITS stages
  const int kst_q = s.H / 128, kst_o = nqd / 128, mt_q = s.qkv_rows / 128, mt_o = s.H / 128;
  int kq = 1, ko = 1;
  if (tcp) {
    kq = std::min(kst_q, std::max(std::max(1, C / mt_q), (kst_q + mk::TC_PROJ_UNITS - 1) / mk::TC_PROJ_UNITS));
    ko = std::min(kst_o, std::max(std::max(1, C / mt_o), (kst_o + mk::TC_PROJ_UNITS - 1) / mk::TC_PROJ_UNITS));
    cnt.qkv_per_g = Rg / 128 * kq;
    cnt.o = mt_o * ko;
  }
  const int umax = std::min(s.E, B * s.k);
  cnt.gu = mk::moe_tiles(umax, s.F, C, bcap, mk::cf_floats(s.E, s.k, s.F, C, bcap));
  cnt.down = std::max(1, std::min(s.H, C));
  cnt.lm = std::max(1, std::min(s.V, 4 * C));
  cnt.down_rows_max = (s.H + cnt.down - 1) / cnt.down;
  // attention chunking
  long long total_pages = 0;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0) return MK_ERR_INVALID;
    total_pages += pages_for(seq_lens[b], s.ps);
  }
  int P = split_pages;
  if (P <= 0) P = (int)std::max<long long>(1, (total_pages * s.nkv + C - 1) / C);
  for (int b = 0; b < B; ++b)   // the split-KV combine takes at most 128 chunks per (request, group)
    P = std::max(P, (pages_for(seq_lens[b], s.ps) + 127) / 128);
  cnt.pages_per_chunk = P;
  std::vector<int> nch(B);
  open_start.assign(B, 0);
  int slots = 0;
  for (int b = 0; b < B; ++b) {
    nch[b] = (pages_for(seq_lens[b], s.ps) + P - 1) / P;
    open_start[b] = (nch[b] - 1) * P;
    slots += nch[b] * s.nkv;
  }
  cnt.part_slots = slots;
  cnt.attn = slots;
  cnt.heads_per_comb = comb_heads(s.G, B * s.nkv, C);
  cnt.comb = B * s.nkv * (s.G / cnt.heads_per_comb);
  const double PB = 2.0 * s.ps * s.d * 2;
  {   // room for every CTA's share up front (the lists grow by one task at a time)
    const long long per_layer = (long long)cnt.qkv_per_g * s.nkv + cnt.attn + cnt.comb + cnt.o + cnt.gu + cnt.down;
    const long long est = (per_layer * s.L + cnt.lm) / C + 2 * s.L + 8;
    for (auto& v : asg.per_cta) v.reserve((size_t)est);
  }

  for (int l = 0; l < s.L; ++l) {
    std::vector<std::pair<double, Task>> ph;
    // QKV projection tiles, per KV group
    for (int mt = 0; tcp && mt < mt_q; ++mt) {
      for (int i = 0; i < kq; ++i) {   // tensor cores: (128-row tile, run of K stages)
        int a, b;
        split_range(kst_q, kq, i, a, b);
        Task t = mk_task(mk::T_QKV, l, l == 0 ? -1 : cm.down + l - 1, (uint32_t)cnt.down);
        t.a[0] = mt * 128;
        t.a[1] = mt * 128 + 128;
        t.a[2] = mt * 128 / Rg;
        t.a[3] = a;
        t.a[4] = b;
        ph.push_back({(double)(b - a) * 128 * 128 * 2, t});
      }
    }
    for (int g = 0; !tcp && g < s.nkv; ++g) {
      for (int i = 0; i < cnt.qkv_per_g; ++i) {
        int a, b;
        split_range(Rg, cnt.qkv_per_g, i, a, b);
        Task t = mk_task(mk::T_QKV, l, l == 0 ? -1 : cm.down + l - 1, (uint32_t)cnt.down);
        t.a[0] = g * Rg + a;
        t.a[1] = g * Rg + b;
        t.a[2] = g;
        ph.push_back({(double)(b - a) * s.H * 2, t});
      }
    }
    asg.phase(ph);
    ph.clear();
    // split-KV attention chunks
    int slot = 0;
    for (int b = 0; b < B; ++b) {
      const int np = pages_for(seq_lens[b], s.ps);
      for (int g = 0; g < s.nkv; ++g) {
        const int first = slot;
        for (int c = 0; c < nch[b]; ++c) {
          Task t = mk_task(mk::T_ATTN, l, cm.qkv + l * s.nkv + g, (uint32_t)cnt.qkv_per_g);
          t.a[0] = b;
          t.a[1] = g;
          t.a[2] = c * P;
          t.a[3] = (c == nch[b] - 1) ? -1 : (c + 1) * P;
          t.a[4] = slot++;
          t.a[5] = first;
          t.a[6] = nch[b];
          const int pages = (c == nch[b] - 1) ? np - c * P : P;
          ph.push_back({pages * PB, t});
        }
      }
    }
    asg.phase(ph);
    ph.clear();
    // split-KV combine, a few query heads per task, once all chunks of (b, g) are in
    for (int b = 0; b < B; ++b) {
      for (int g = 0; g < s.nkv; ++g) {
        for (int h = 0; h < s.G; h += cnt.heads_per_comb) {
          Task t = mk_task(mk::T_COMB, l, cm.attn_idx(l, b, g), (uint32_t)nch[b]);
          t.a[0] = b;
          t.a[1] = g;
          t.a[2] = h;
          t.a[3] = cnt.heads_per_comb;
          t.a[5] = first_slot(nch, B, s.nkv, b, g);
          t.a[6] = nch[b];
          ph.push_back({(double)nch[b] * cnt.heads_per_comb * (s.d + 2) * 4, t});
        }
      }
    }
    asg.phase(ph);
    ph.clear();
    // O projection + residual, each tile with its hidden rows' share of the router logits
    for (int i = 0; tcp && i < cnt.o; ++i) {   // tensor cores: (128-row tile, run of K stages)
      int a, b;
      split_range(kst_o, ko, i % ko, a, b);
      Task t = mk_task(mk::T_OPROJ, l, cm.combine + l, (uint32_t)cnt.comb);
      t.a[0] = i / ko * 128;
      t.a[1] = i / ko * 128 + 128;
      t.a[2] = i;
      t.a[3] = a;
      t.a[4] = b;
      t.a[5] = cnt.o;
      t.a[6] = ko;   // tasks of this 128-row tile (its ticket's count)
      ph.push_back({(double)(b - a + 1) * 128 * 128 * 2, t});
    }
    for (int i = 0; !tcp && i < cnt.o; ++i) {
      int a, b;
      split_range(s.H, cnt.o, i, a, b);
      Task t = mk_task(mk::T_OPROJ, l, cm.combine + l, (uint32_t)cnt.comb);
      t.a[0] = a;
      t.a[1] = b;
      t.a[2] = i;
      ph.push_back({(double)(b - a) * (nqd + s.E) * 2, t});
    }
    asg.phase(ph);
    ph.clear();
    // expert tiles over the distinct selected experts (every tile routes from the
    // O tiles' logit partials): gate/up + down slices
    for (int i = 0; i < cnt.gu; ++i) {
      Task t = mk_task(mk::T_MOE, l, cm.o + l, (uint32_t)cnt.o);
      t.a[0] = i;
      t.a[1] = cnt.gu;
      ph.push_back({(double)umax * s.F * 6.0 * s.H / cnt.gu, t});
    }
    asg.phase(ph);
    ph.clear();
    // reduce: residual + the expert tiles' partials, row tiles of the hidden dim
    for (int i = 0; i < cnt.down; ++i) {
      int a, b;
      split_range(s.H, cnt.down, i, a, b);
      Task t = mk_task(mk::T_RED, l, cm.gu + l, (uint32_t)cnt.gu);
      t.a[0] = a;
      t.a[1] = b;
      t.a[2] = cnt.gu;
      ph.push_back({(double)(b - a) * cnt.gu * B * 4, t});
    }
    asg.phase(ph);
  }
  std::vector<std::pair<double, Task>> ph;
  for (int i = 0; i < cnt.lm; ++i) {
    int a, b;
    split_range(s.V, cnt.lm, i, a, b);
    Task t = mk_task(mk::T_LM, s.L - 1, cm.down + s.L - 1, (uint32_t)cnt.down);
    t.a[0] = a;
    t.a[1] = b;
    t.a[2] = i;
    t.a[3] = cnt.lm;
    ph.push_back({(double)(b - a) * s.H * 2, t});
  }
  asg.phase(ph);
  if (nucleus) {   // one nucleus draw per request, once every LM tile is done
    ph.clear();
    for (int b = 0; b < B; ++b) {
      Task t = mk_task(mk::T_SAMPLE, s.L - 1, cm.lm, (uint32_t)cnt.lm);
      t.a[0] = b;
      ph.push_back({(double)s.V * 4 * 6, t});
    }
    asg.phase(ph);
  }

  out.clear();
  size_t ntot = 0;
  for (int c = 0; c < C; ++c) ntot += asg.per_cta[c].size();
  out.reserve(ntot);
  cta_start.assign(C + 1, 0);
  for (int c = 0; c < C; ++c) {
    cta_start[c] = (int)out.size();
    out.insert(out.end(), asg.per_cta[c].begin(), asg.per_cta[c].end());
  }
  cta_start[C] = (int)out.size();
  return MK_OK;
}

}  // namespace

namespace mk {
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }
}  // namespace mk

// ------------------------------------------------------------------ the plan

namespace {
struct Built;
}

struct mk_plan {
  // A batch capacity above mk::MAX_BATCH makes a group: sub-plan i holds
  // requests [8i, 8i + 8) and the group's calls run the sub-plans one after
  // another on the caller's stream.  A sub-plan with no requests is idle.
  std::vector<mk_plan*> subs;
  std::vector<int> sub_B;
  int group_B = 0;
  Shape s;
  int B = 0, bcap = 0, C = 0, nb = 1, split_opt = 0, drop_task = 0, trace = 0;
  int ucap = 0;                    // the caller's capacity (bcap: the kernel's, 8 on the batch-8 instance)
  int max_pages = 0, num_pages = 0, rope_npos = 0;
  int smem = 0, nstages = 0, stage_bytes = 0, act_floats = 0;
  int replans = 0;
  uint32_t epoch = 0;
  float inv_temp = 0.f;            // temperature sampling: 1 / T, 0 = greedy
  float top_p = 1.f;               // nucleus sampling below 1 (with inv_temp > 0)
  bool nucleus_built = false;      // the task list holds the nucleus draw tasks
  float* d_lg_keep = nullptr;      // [bcap][V] logits kept for the draw
  unsigned long long seed = 0;
  int slot0 = 0;                   // batch slot of the first request (sub-plan i of a group: 8 i)
  unsigned long long timeout_ns = 0;
  std::vector<int> seq, pt, open_start;
  std::vector<int> chunk0;         // rows' prefill chunk starts (empty: no chunks)
  int* d_chunk0 = nullptr;
  bool chunk_stepped = false;      // a step ran on a batch with prefill chunks (an update must come next)
  std::vector<Task> tasks;
  std::vector<int> cta_start;
  Counts cnt;
  mk::CtrMap cm;
  mk::RouteMap rm;
  mk::Params P;
  // device buffers owned by the plan
  std::vector<void*> allocs;
  Task* d_tasks = nullptr;
  size_t tasks_cap = 0;
  int* d_cta = nullptr;
  uint32_t* d_ctr = nullptr;
  int* d_status = nullptr;
  int* d_seq = nullptr;
  int* d_pt = nullptr;
  size_t pt_cap = 0;
  float2* d_rope = nullptr;
  float* d_part = nullptr;
  size_t part_cap_slots = 0;
  unsigned long long* d_trace = nullptr;
  size_t trace_cap = 0;
  unsigned long long* d_strace = nullptr;
  int* d_io_tok = nullptr;
  int* d_io_next = nullptr;
  float* d_io_logits = nullptr;
  // pinned staging for uploads, protected by an event
  // two pinned staging buffers used in turn: an upload waits only for the one
  // two updates back, never for the step in flight
  void* h_stage[2] = {nullptr, nullptr};
  size_t h_stage_cap[2] = {0, 0};
  cudaEvent_t ev_stage[2] = {nullptr, nullptr};
  int stage_i = 0;
  int* h_status = nullptr;
  int* h_next = nullptr;           // pinned [bcap]: next tokens of a step enqueued without waiting
  int* h_tok = nullptr;            // pinned [bcap]: that step's input tokens
  // a task list built ahead for the lengths `pre_seq` (the serving loop builds
  // the next batch's list while the GPU runs the current step)
  bool pre_valid = false;
  std::vector<int> pre_seq;
  Built* pre = nullptr;
};

namespace {

template <class T>
cudaError_t dalloc(mk_plan* p, T** ptr, size_t bytes) {
  void* v = nullptr;
  cudaError_t e = cudaMalloc(&v, bytes ? bytes : 16);
  if (e != cudaSuccess) return e;
  p->allocs.push_back(v);
  *ptr = (T*)v;
  return cudaSuccess;
}

void dfree(mk_plan* p, void* ptr) {
  if (!ptr) return;
  auto it = std::find(p->allocs.begin(), p->allocs.end(), ptr);
  if (it != p->allocs.end()) p->allocs.erase(it);
  cudaFree(ptr);
}

bool aligned16(const void* q) { return q && ((uintptr_t)q % 16) == 0; }

// chunk_first (nullable): row b is part of the prefill chunk that starts at
// row chunk_first[b] <= b.  A chunk's rows are consecutive, hold consecutive
// positions of one request and the same page row; rows of different chunks
// may not share a page.  group: rows per sub-plan (a chunk stays inside one).
int validate_batch(const Shape& s, int B, const int* seq_lens, const int* page_table, int max_pages,
                   int num_pages, const int* chunk_first = nullptr, int group = 0) {
  if (!seq_lens || !page_table || max_pages < 1) return MK_ERR_INVALID;
  std::vector<char> used((size_t)num_pages, 0);
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0) return MK_ERR_INVALID;
    const int np = pages_for(seq_lens[b], s.ps);
    if (np > max_pages) return MK_ERR_CAPACITY;
    const int c = chunk_first ? chunk_first[b] : b;
    if (c != b) {   // a later row of a chunk: the previous row's request, one position on
      if (c < 0 || c > b || chunk_first[b - 1] != c || seq_lens[b] != seq_lens[b - 1] + 1) return MK_ERR_INVALID;
      if (group > 0 && c / group != b / group) return MK_ERR_INVALID;
      for (int i = 0; i < np; ++i) {
        const int pg = page_table[(size_t)b * max_pages + i];
        if (pg < 0 || pg >= num_pages) return MK_ERR_INVALID;
        const int pc = i < pages_for(seq_lens[b - 1], s.ps) ? page_table[(size_t)(b - 1) * max_pages + i] : -1;
        if (pc >= 0 ? pg != pc : used[pg] != 0) return MK_ERR_INVALID;   // same pages as the chunk, new ones unused
        used[pg] = 1;
      }
      continue;
    }
    for (int i = 0; i < np; ++i) {
      const int pg = page_table[(size_t)b * max_pages + i];
      if (pg < 0 || pg >= num_pages) return MK_ERR_INVALID;
      if (used[pg]) return MK_ERR_INVALID;  // two requests may not share a page
      used[pg] = 1;
    }
  }
  return MK_OK;
}

// Stage the bytes in pinned memory and enqueue the copy to `dst` on `st`.
// Host -> device copies of one update, through the next pinned staging buffer
// (each piece at a 16-byte aligned offset).
struct Up {
  void* dst;
  const void* src;
  size_t bytes;
};
cudaError_t upload_many(mk_plan* p, cudaStream_t st, const Up* u, int n) {
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += (u[i].bytes + 15) / 16 * 16;
  if (total == 0) return cudaSuccess;
  const int k = p->stage_i ^ 1;
  cudaError_t e;
  if (p->ev_stage[k]) {
    e = cudaEventSynchronize(p->ev_stage[k]);   // the update two back no longer reads this buffer
    if (e != cudaSuccess) return e;
  }
  if (total > p->h_stage_cap[k]) {
    if (p->h_stage[k]) cudaFreeHost(p->h_stage[k]);
    p->h_stage[k] = nullptr;
    p->h_stage_cap[k] = 0;
    e = cudaMallocHost(&p->h_stage[k], total + total / 2);
    if (e != cudaSuccess) return e;
    p->h_stage_cap[k] = total + total / 2;
  }
  uint8_t* h = (uint8_t*)p->h_stage[k];
  size_t off = 0;
  for (int i = 0; i < n; ++i) {
    if (u[i].bytes == 0) continue;
    memcpy(h + off, u[i].src, u[i].bytes);
    e = cudaMemcpyAsync(u[i].dst, h + off, u[i].bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return e;
    off += (u[i].bytes + 15) / 16 * 16;
  }
  p->stage_i = k;
  return cudaEventRecord(p->ev_stage[k], st);
}

cudaError_t upload(mk_plan* p, void* dst, const void* src, size_t bytes, cudaStream_t st) {
  const Up u = {dst, src, bytes};
  return upload_many(p, st, &u, 1);
}

// A replan in two halves.  build_for is host work only (the task list for the
// plan's current lengths), so a group builds its sub-plans' lists on parallel
// threads.  commit_built grows device buffers if needed, uploads the list (with
// the lengths and page table when with_batch), and resets the counters.
struct Built {
  std::vector<Task> tasks;
  std::vector<int> cs, open;
  Counts cnt;
  int rc = MK_OK;
  bool nucleus = false;
};

bool nucleus_on(const mk_plan* p) { return p->inv_temp > 0.f && p->top_p < 1.f; }

void build_for(const mk_plan* p, Built& b, int B = -1, const int* seq = nullptr) {
  if (B < 0) {
    B = p->B;
    seq = p->seq.data();
  }
  b.rc = build_tasks(p->s, B, p->bcap, seq, p->C, p->split_opt, b.tasks, b.cs, b.cnt, b.open, nucleus_on(p),
                     p->P.tm_qkv != nullptr);
  b.nucleus = nucleus_on(p);
  if (b.rc != MK_OK) return;
  if (p->drop_task > 0 && p->drop_task - 1 < (int)b.tasks.size()) {
    const int victim = p->drop_task - 1;
    b.tasks.erase(b.tasks.begin() + victim);
    for (int c = 0; c <= p->C; ++c)
      if (b.cs[c] > victim) b.cs[c]--;
  }
}

int commit_built(mk_plan* p, Built& b, cudaStream_t st, bool with_batch) {
  if (b.rc != MK_OK) return b.rc;
  std::vector<Task>& tasks = b.tasks;
  std::vector<int>& cs = b.cs;
  cudaError_t e;
  // one device blob: tasks, then the C + 1 CTA offsets (48-byte tasks keep it 16-byte aligned)
  const size_t tbytes = tasks.size() * sizeof(Task), blob_bytes = tbytes + cs.size() * sizeof(int);
  if (blob_bytes > p->tasks_cap) {
    if (p->d_tasks) {
      if (cudaStreamSynchronize(st) != cudaSuccess) return MK_ERR_CUDA;
      dfree(p, p->d_tasks);
      p->d_tasks = nullptr;
    }
    const size_t cap = blob_bytes + blob_bytes / 2 + 4096;
    if ((e = dalloc(p, (uint8_t**)&p->d_tasks, cap)) != cudaSuccess) return MK_ERR_CUDA;
    p->tasks_cap = cap;
  }
  if (p->trace && tasks.size() > p->trace_cap) {
    if (p->d_trace) {
      if (cudaStreamSynchronize(st) != cudaSuccess) return MK_ERR_CUDA;
      dfree(p, p->d_trace);
      p->d_trace = nullptr;
    }
    const size_t cap = tasks.size() + tasks.size() / 2 + 64;
    if (dalloc(p, &p->d_trace, cap * mk::TRACE_SLOTS * sizeof(unsigned long long)) != cudaSuccess)
      return MK_ERR_CUDA;
    p->trace_cap = cap;
  }
  if ((size_t)b.cnt.part_slots > p->part_cap_slots) {
    // grow the attention partial buffer (rare: only when a replan adds chunks)
    if (p->d_part) {
      if (cudaStreamSynchronize(st) != cudaSuccess) return MK_ERR_CUDA;
      dfree(p, p->d_part);
      p->d_part = nullptr;
    }
    size_t cap = (size_t)b.cnt.part_slots * 2 + 16;
    if (dalloc(p, &p->d_part, (size_t)p->s.L * cap * p->s.G * (p->s.d + 4) * sizeof(float)) != cudaSuccess)
      return MK_ERR_CUDA;
    p->part_cap_slots = cap;
  }
  Up ups[5];
  int nu = 0;
  ups[nu++] = {p->d_tasks, tasks.data(), tbytes};
  ups[nu++] = {(uint8_t*)p->d_tasks + tbytes, cs.data(), cs.size() * sizeof(int)};
  if (with_batch) {
    ups[nu++] = {p->d_seq, p->seq.data(), (size_t)p->B * sizeof(int)};
    if (!p->chunk0.empty()) ups[nu++] = {p->d_chunk0, p->chunk0.data(), (size_t)p->B * sizeof(int)};
    ups[nu++] = {p->d_pt, p->pt.data(), p->pt.size() * sizeof(int)};
  }
  if (upload_many(p, st, ups, nu) != cudaSuccess) return MK_ERR_CUDA;
  p->d_cta = (int*)((uint8_t*)p->d_tasks + tbytes);
  if (cudaMemsetAsync(p->d_ctr, 0, (size_t)p->cm.total * mk::CTR_STRIDE * sizeof(uint32_t), st) != cudaSuccess)
    return MK_ERR_CUDA;
  if (cudaMemsetAsync(p->P.rlsum, 0, (size_t)p->s.L * mk::RL_COPIES * p->bcap * p->s.E * sizeof(unsigned long long), st) !=
      cudaSuccess)
    return MK_ERR_CUDA;
  if (p->P.tm_qkv &&
      (cudaMemsetAsync(p->P.qkv_fx, 0, (size_t)p->s.L * p->bcap * p->s.qkv_rows * sizeof(unsigned long long), st) !=
           cudaSuccess ||
       cudaMemsetAsync(p->P.xmid_fx, 0, (size_t)p->s.L * p->bcap * p->s.H * sizeof(unsigned long long), st) !=
           cudaSuccess))
    return MK_ERR_CUDA;
  p->epoch = 0;
  p->tasks.swap(tasks);
  p->cta_start.swap(cs);
  p->cnt = b.cnt;
  p->open_start.swap(b.open);
  p->nucleus_built = b.nucleus;
  p->replans++;
  return MK_OK;
}

// Rebuild tasks for the plan's current lengths, upload them, reset counters.
int replan(mk_plan* p, cudaStream_t st) {
  Built b;
  build_for(p, b);
  return commit_built(p, b, st, false);
}

bool needs_replan(const mk_plan* p) {
  const int P = p->cnt.pages_per_chunk;
  const int slack = std::max(2, P / 2);
  for (int b = 0; b < p->B; ++b) {
    const int open_pages = pages_for(p->seq[b], p->s.ps) - p->open_start[b];
    if (open_pages > P + slack) return true;
  }
  return false;
}

void fill_params(mk_plan* p) {
  mk::Params& P = p->P;
  const Shape& s = p->s;
  P.L = s.L; P.H = s.H; P.nq = s.nq; P.nkv = s.nkv; P.d = s.d; P.E = s.E; P.k = s.k; P.F = s.F;
  P.V = s.V; P.ps = s.ps; P.G = s.G; P.qkv_rows = s.qkv_rows; P.eps = s.eps;
  P.B = p->B; P.bcap = p->bcap; P.max_pages = p->max_pages;
  P.tasks = p->d_tasks; P.cta_start = p->d_cta; P.ctr = p->d_ctr; P.status = p->d_status;
  P.timeout_ns = p->timeout_ns; P.cm = p->cm; P.rm = p->rm;
  P.nstages = p->nstages; P.stage_bytes = p->stage_bytes;
  P.seq_len = p->d_seq; P.page_table = p->d_pt; P.rope = p->d_rope; P.rope_npos = p->rope_npos;
  P.chunk0 = p->chunk0.empty() ? nullptr : p->d_chunk0;
  P.part = p->d_part; P.part_slots = (int)p->part_cap_slots;
  P.lm_tiles = p->cnt.lm; P.down_rows_max = p->cnt.down_rows_max;
  P.cf_pairs = std::max(1, mk::cf_floats(s.E, s.k, s.F, p->C, p->bcap) / p->bcap);
  P.trace = p->trace ? p->d_trace : nullptr;
  P.strace = p->trace >= 2 ? p->d_strace : nullptr;
}

}  // namespace

extern "C" {

const char* mk_last_error(void) { return g_last_error; }

const char* mk_status_string(int st) {
  switch (st) {
    case MK_OK: return "ok";
    case MK_ERR_INVALID: return "invalid argument";
    case MK_ERR_CUDA: return "CUDA runtime error";
    case MK_ERR_DEP_TIMEOUT: return "device dependency wait timed out";
    case MK_ERR_CAPACITY: return "capacity exceeded (batch, pages or positions)";
    case MK_ERR_UNSUPPORTED: return "unsupported shape";
    default: return "unknown status";
  }
}

int mk_plan_inspect(const mk_model_dims* dims, int batch, const int* seq_lens, int num_ctas,
                    int split_pages, int* tasks_out, int max_tasks, int* cta_start_out) {
  Shape s;
  int rc = check_dims(dims, s);
  if (rc != MK_OK) return rc;
  if (!seq_lens || batch < 1 || batch > mk::MAX_BATCH || num_ctas < 1) return MK_ERR_INVALID;
  std::vector<Task> tasks;
  std::vector<int> cs, open;
  Counts cnt;
  rc = build_tasks(s, batch, batch, seq_lens, num_ctas, split_pages, tasks, cs, cnt, open);
  if (rc != MK_OK) return rc;
  if (tasks_out) {
    const int n = std::min<int>(max_tasks, (int)tasks.size());
    for (int i = 0; i < n; ++i) {
      const Task& t = tasks[i];
      int* o = tasks_out + 12 * i;
      o[0] = t.type; o[1] = t.layer;
      for (int j = 0; j < 8; ++j) o[2 + j] = t.a[j];
      o[10] = t.wait_ctr; o[11] = (int)t.wait_cnt;
    }
  }
  if (cta_start_out) memcpy(cta_start_out, cs.data(), cs.size() * sizeof(int));
  return (int)tasks.size();
}

// A usable sampling temperature: 0 (greedy), or finite and positive with a
// finite inverse (the LM tiles scale logits by 1 / T; below about 2.9e-39 the
// inverse overflows to infinity and every key would be NaN or infinite).
static bool temperature_ok(float t) {
  if (t == 0.f) return true;
  return t > 0.f && std::isfinite(t) && std::isfinite(1.0f / t);
}


// The rows' prefill chunk starts, kept only when some row continues a chunk.
static void set_chunks(mk_plan* p, int batch, const int* chunk_first) {
  p->chunk0.clear();
  p->chunk_stepped = false;
  if (!chunk_first) return;
  bool any = false;
  for (int b = 0; b < batch; ++b) any |= chunk_first[b] != b;
  if (any) p->chunk0.assign(chunk_first, chunk_first + batch);
}

// TMA tensor maps of one weight matrix per layer for the tensor-core paths
// (batch instance 8): bf16 [rows, cols] row-major, 64 x 128 boxes, 128-byte
// swizzle.  Uploaded to `dst` (device, L x 128 bytes).  False when the
// driver's encoder is unavailable or refuses a map: the CUDA cores then take
// the work.
// One 2-D tensor map per layer over a [rows][cols] bf16 matrix: boxes of 64
// columns (128 bytes, swizzled) by box_rows rows.
static bool encode_maps(const Shape& s, const void* const* mats, long long rows, long long cols, int box_rows,
                        void* dst) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      !fn || q != cudaDriverEntryPointSuccess)
    return false;
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  std::vector<CUtensorMap> maps((size_t)s.L);
  const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t gstr[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  for (int l = 0; l < s.L; ++l) {
    if (enc(&maps[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(mats[l]), gdim, gstr, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return cudaMemcpy(dst, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice) == cudaSuccess;
}

static void destroy_one(mk_plan* p);

static int create_one(const mk_model_dims* dims, const mk_weights* w, const mk_kv* kv, int batch,
                      const int* seq_lens, const int* page_table, int max_pages_per_seq,
                      const mk_plan_opts* opts, mk_plan** out) {
  if (!out) return MK_ERR_INVALID;
  *out = nullptr;
  Shape s;
  int rc = check_dims(dims, s);
  if (rc != MK_OK) return rc;
  if (!w || !kv || batch < 1) return MK_ERR_INVALID;
  mk_plan_opts o = {};
  if (opts) o = *opts;
  const int ucap = o.max_batch > 0 ? o.max_batch : batch;   // the caller's batch capacity
  if (batch > ucap) return MK_ERR_INVALID;
  if (ucap > mk::MAX_BATCH) return MK_ERR_UNSUPPORTED;
  // The kernel instance: batch 1, 2, else the batch-8 instance, which runs
  // its projections and expert gate/up on the tensor cores when the shape
  // allows (mid shape, 10 steps: batch 3 0.99 -> 0.85 ms, batch 4 1.19 ->
  // 1.04 ms against the batch-4 instance's CUDA cores; batch 2 stays, 0.63
  // against 0.81 ms).  The batch-8 instance always runs at capacity 8 (its
  // buffers, shared memory, expert tiles and coefficient scratch as for 8
  // requests); the caller's capacity still bounds the updates.
  int nb = ucap <= 1 ? 1 : ucap <= 2 ? 2 : ucap <= 4 ? 4 : 8;
  if (nb == 4 && !o.tc_off && mk::tc_moe_shape(s.H, s.F) && mk::tc_proj_shape(s.H, s.nq, s.d, s.G, s.E, 2 * mk::TC_BOX))
    nb = 8;
  const int bcap = nb == 8 ? mk::MAX_BATCH : ucap;
  if (!aligned16(w->embed) || !aligned16(w->final_norm) || !aligned16(w->lm_head)) return MK_ERR_INVALID;
  if (!w->attn_norm || !w->wqkv || !w->wo || !w->ffn_norm || !w->router || !w->w_gate_up || !w->w_down)
    return MK_ERR_INVALID;
  if (!kv->kv_pool || kv->num_pages < 1) return MK_ERR_INVALID;
  for (int l = 0; l < s.L; ++l) {
    if (!aligned16(w->attn_norm[l]) || !aligned16(w->wqkv[l]) || !aligned16(w->wo[l]) ||
        !aligned16(w->ffn_norm[l]) || !aligned16(w->router[l]) || !aligned16(w->w_gate_up[l]) ||
        !aligned16(w->w_down[l]) || !aligned16(kv->kv_pool[l]))
      return MK_ERR_INVALID;
  }
  rc = validate_batch(s, batch, seq_lens, page_table, max_pages_per_seq, kv->num_pages, o.chunk_first);
  if (rc != MK_OK) return rc;
  if (!temperature_ok(o.temperature)) {
    mk::set_last_error("mk_plan_create: temperature must be 0 (greedy) or a finite value whose inverse is finite");
    return MK_ERR_INVALID;
  }
  if (!(o.top_p == 0.f || (o.top_p > 0.f && o.top_p <= 1.f))) {
    mk::set_last_error("mk_plan_create: top_p must be in (0, 1] (0: off)");
    return MK_ERR_INVALID;
  }

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MK_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MK_ERR_CUDA;

  mk_plan* p = new (std::nothrow) mk_plan();
  if (!p) return MK_ERR_CUDA;
  p->s = s;
  p->B = batch;
  p->bcap = bcap;
  p->ucap = ucap;
  p->nb = nb;
  p->C = o.num_ctas > 0 ? std::min(o.num_ctas, sms) : sms;
  p->split_opt = o.split_pages;
  p->drop_task = o.debug_drop_task;
  p->inv_temp = o.temperature > 0.f ? 1.0f / o.temperature : 0.f;
  p->top_p = o.top_p == 0.f ? 1.f : o.top_p;
  p->seed = o.seed;
  p->trace = o.trace >= 2 ? 2 : o.trace ? 1 : 0;
  p->timeout_ns = (unsigned long long)(o.timeout_us > 0 ? o.timeout_us : 2000000) * 1000ull;
  p->max_pages = max_pages_per_seq;
  p->num_pages = kv->num_pages;
  p->seq.assign(seq_lens, seq_lens + batch);
  p->pt.assign(page_table, page_table + (size_t)batch * max_pages_per_seq);
  set_chunks(p, batch, o.chunk_first);
  p->cm.init(s.L, s.nkv, bcap, s.H / 128);
  p->rm.init(std::min(s.E, bcap * s.k), bcap);

  auto fail = [&](int code) {
    if (code == MK_ERR_CUDA && !g_last_error[0]) note_cuda(cudaGetLastError(), "mk_plan_create");
    destroy_one(p);
    return code;
  };
  g_last_error[0] = 0;

  // shared-memory budget: activations + misc + partial sums, the rest is the weight ring
  const int C = p->C;
  const int down_rows_max = (s.H + std::min(s.H, C) - 1) / std::min(s.H, C);
  mk::SmemPlan sp;
  if (!mk::plan_smem(s.H, s.nq, s.d, s.G, s.E, s.F, s.ps, bcap, p->nb, down_rows_max,
                     mk::cf_floats(s.E, s.k, s.F, C, bcap), mk::misc_bytes(), sp))
    return fail(MK_ERR_UNSUPPORTED);
  p->act_floats = sp.act_floats;
  p->stage_bytes = sp.stage_bytes;
  p->nstages = sp.nstages;
  p->smem = sp.smem;
  p->P.act_off = sp.act_off;
  p->P.act_floats = sp.act_floats;
  p->P.misc_off = sp.misc_off;
  p->P.psum_off = sp.psum_off;
  p->P.attn_mrg_floats = sp.attn_mrg_floats;
  p->P.o_halves = sp.o_halves;
  if (mk::max_active_ctas(p->nb, p->smem) < 1) {
    snprintf(g_last_error, sizeof(g_last_error), "megakernel does not fit on an SM with %d bytes of shared memory",
             p->smem);
    return fail(MK_ERR_CUDA);
  }

  cudaStream_t st = 0;
  mk::Params& P = p->P;
  const size_t L = s.L;
  // weight pointer tables
  {
    std::vector<const void*> tab(8 * L);
    for (size_t l = 0; l < L; ++l) {
      tab[0 * L + l] = w->attn_norm[l];
      tab[1 * L + l] = w->wqkv[l];
      tab[2 * L + l] = w->wo[l];
      tab[3 * L + l] = w->ffn_norm[l];
      tab[4 * L + l] = w->router[l];
      tab[5 * L + l] = w->w_gate_up[l];
      tab[6 * L + l] = w->w_down[l];
      tab[7 * L + l] = kv->kv_pool[l];
    }
    const void** d_tab = nullptr;
    if (dalloc(p, &d_tab, tab.size() * sizeof(void*)) != cudaSuccess) return fail(MK_ERR_CUDA);
    if (cudaMemcpy(d_tab, tab.data(), tab.size() * sizeof(void*), cudaMemcpyHostToDevice) != cudaSuccess)
      return fail(MK_ERR_CUDA);
    P.attn_norm = (const uint16_t* const*)(d_tab + 0 * L);
    P.wqkv = (const uint16_t* const*)(d_tab + 1 * L);
    P.wo = (const uint16_t* const*)(d_tab + 2 * L);
    P.ffn_norm = (const uint16_t* const*)(d_tab + 3 * L);
    P.router = (const uint16_t* const*)(d_tab + 4 * L);
    P.w_gate_up = (const uint16_t* const*)(d_tab + 5 * L);
    P.w_down = (const uint16_t* const*)(d_tab + 6 * L);
    P.kv_pool = (uint16_t* const*)(d_tab + 7 * L);
    P.embed = (const uint16_t*)w->embed;
    P.final_norm = (const uint16_t*)w->final_norm;
    P.lm_head = (const uint16_t*)w->lm_head;
  }
  // the batch-8 instance's expert gate/up on the tensor cores
  P.tm_gu = P.tm_qkv = P.tm_o = nullptr;
  P.qkv_fx = P.xmid_fx = nullptr;
  if (p->nb == 8 && mk::tc_moe_shape(s.H, s.F) && !o.tc_off && p->stage_bytes % mk::TC_BOX == 0 &&
      s.H % (128 * (p->stage_bytes / mk::TC_BOX)) == 0 && (long long)p->act_floats * 4 >= 32LL * s.H) {
    void* maps = nullptr;
    if (dalloc(p, (uint8_t**)&maps, L * sizeof(CUtensorMap)) != cudaSuccess) return fail(MK_ERR_CUDA);
    if (encode_maps(s, (const void* const*)w->w_gate_up, (long long)s.E * 2 * s.F, s.H, 64, maps)) P.tm_gu = maps;
  }
  // and the QKV and O projections: B operand slots of a task's K stages (4 KB
  // each) in the activation region
  const int kst_max = std::max(s.H, s.nq * s.d) / 128;
  if (P.tm_gu && mk::tc_proj_shape(s.H, s.nq, s.d, s.G, s.E, p->stage_bytes) &&
      (long long)p->act_floats * 4 >= 4096LL * std::min(mk::TC_PROJ_UNITS, kst_max)) {
    void* mq = nullptr;
    void* mo = nullptr;
    if (dalloc(p, (uint8_t**)&mq, L * sizeof(CUtensorMap)) != cudaSuccess ||
        dalloc(p, (uint8_t**)&mo, L * sizeof(CUtensorMap)) != cudaSuccess ||
        dalloc(p, &P.qkv_fx, L * bcap * s.qkv_rows * sizeof(unsigned long long)) != cudaSuccess ||
        dalloc(p, &P.xmid_fx, L * bcap * s.H * sizeof(unsigned long long)) != cudaSuccess)
      return fail(MK_ERR_CUDA);
    if (encode_maps(s, (const void* const*)w->wqkv, s.qkv_rows, s.H, 128, mq) &&
        encode_maps(s, (const void* const*)w->wo, s.H, (long long)s.nq * s.d, 128, mo)) {
      P.tm_qkv = mq;
      P.tm_o = mo;
    }
  }
  bool ok = true;
  ok &= dalloc(p, &p->d_ctr, (size_t)p->cm.total * mk::CTR_STRIDE * sizeof(uint32_t)) == cudaSuccess;
  ok &= dalloc(p, &p->d_status, 4 * sizeof(int)) == cudaSuccess;
  ok &= dalloc(p, &p->d_seq, (size_t)bcap * sizeof(int)) == cudaSuccess;
  ok &= dalloc(p, &p->d_chunk0, (size_t)bcap * sizeof(int)) == cudaSuccess;
  p->pt_cap = (size_t)bcap * max_pages_per_seq;
  ok &= dalloc(p, &p->d_pt, p->pt_cap * sizeof(int)) == cudaSuccess;
  ok &= dalloc(p, &P.qkv, L * bcap * s.qkv_rows * sizeof(float)) == cudaSuccess;
  ok &= dalloc(p, &P.o, L * bcap * s.nq * s.d * sizeof(float)) == cudaSuccess;
  ok &= dalloc(p, &P.x_mid, L * bcap * s.H * sizeof(float)) == cudaSuccess;
  ok &= dalloc(p, &P.x_out, L * bcap * s.H * sizeof(float)) == cudaSuccess;
  ok &= dalloc(p, &P.rlog, L * bcap * s.E * sizeof(float)) == cudaSuccess;
  ok &= dalloc(p, &P.ids, L * bcap * s.k * sizeof(int)) == cudaSuccess;
  ok &= dalloc(p, &P.gates, L * bcap * s.k * sizeof(float)) == cudaSuccess;
  ok &= dalloc(p, &P.route, L * p->rm.ints * sizeof(int)) == cudaSuccess;
  // expert-tile partials, sized for the most tiles any batch up to the capacity needs
  const int moe_max = mk::moe_tiles(std::min(s.E, bcap * s.k), s.F, C, bcap, mk::cf_floats(s.E, s.k, s.F, C, bcap));
  ok &= dalloc(p, &P.moe_part, (size_t)moe_max * bcap * s.H * sizeof(float)) == cudaSuccess;
  ok &= dalloc(p, &P.moe_mask, (size_t)L * moe_max * sizeof(uint32_t)) == cudaSuccess;
  ok &= dalloc(p, &P.rlsum, L * mk::RL_COPIES * bcap * s.E * sizeof(unsigned long long)) == cudaSuccess;
  const int lm_tiles = std::max(1, std::min(s.V, 4 * C));
  ok &= dalloc(p, &P.lm_val, (size_t)bcap * lm_tiles * sizeof(float)) == cudaSuccess;
  ok &= dalloc(p, &P.lm_idx, (size_t)bcap * lm_tiles * sizeof(int)) == cudaSuccess;
  if (p->trace >= 2)
    ok &= dalloc(p, &p->d_strace, (size_t)C * mk::STRACE_CAP * mk::STRACE_SLOTS * sizeof(unsigned long long)) ==
          cudaSuccess;
  ok &= dalloc(p, &p->d_io_tok, (size_t)bcap * sizeof(int)) == cudaSuccess;
  ok &= dalloc(p, &p->d_io_next, (size_t)bcap * sizeof(int)) == cudaSuccess;
  p->rope_npos = max_pages_per_seq * s.ps;
  ok &= dalloc(p, &p->d_rope, (size_t)p->rope_npos * (s.d / 2) * sizeof(float2)) == cudaSuccess;
  if (!ok) return fail(MK_ERR_CUDA);
  for (int k = 0; k < 2; ++k)
    if (cudaEventCreateWithFlags(&p->ev_stage[k], cudaEventDisableTiming) != cudaSuccess) return fail(MK_ERR_CUDA);
  if (cudaMallocHost(&p->h_status, 4 * sizeof(int)) != cudaSuccess) return fail(MK_ERR_CUDA);
  if (cudaMallocHost(&p->h_next, (size_t)bcap * sizeof(int)) != cudaSuccess) return fail(MK_ERR_CUDA);
  if (cudaMallocHost(&p->h_tok, (size_t)bcap * sizeof(int)) != cudaSuccess) return fail(MK_ERR_CUDA);
  if (cudaMemsetAsync(p->d_status, 0, 4 * sizeof(int), st) != cudaSuccess) return fail(MK_ERR_CUDA);
  if (cudaMemsetAsync(P.route, 0, L * p->rm.ints * sizeof(int), st) != cudaSuccess) return fail(MK_ERR_CUDA);
  if (mk::launch_rope_table(p->d_rope, p->rope_npos, s.d, (double)s.theta, st) != cudaSuccess)
    return fail(MK_ERR_CUDA);
  {
    Built b;
    build_for(p, b);
    rc = commit_built(p, b, st, true);
    if (rc != MK_OK) return fail(rc);
  }
  p->replans = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return fail(MK_ERR_CUDA);
  fill_params(p);
  *out = p;
  return MK_OK;
}

// n_steps decode steps in one launch; step s's next tokens go to row s of
// d_next_token (rows io_stride apart) and feed step s + 1 on the device.
// The checks of a launch of n_steps, with no side effect: a group checks
// every sub-plan before it launches any.
static int steps_check(const mk_plan* p, int n_steps) {
  if (!p->chunk0.empty() && (n_steps > 1 || p->chunk_stepped)) {
    mk::set_last_error("a batch with prefill chunks runs one step, then needs mk_plan_update_rows");
    return MK_ERR_INVALID;
  }
  const Shape& s = p->s;
  for (int b = 0; b < p->B; ++b) {   // every position this launch writes needs its page
    for (int k = 0; k < n_steps; ++k) {
      const int pos = p->seq[b] + k;
      if (pos / s.ps >= p->max_pages || pos >= p->rope_npos) return MK_ERR_CAPACITY;
      const int pg = p->pt[(size_t)b * p->max_pages + pos / s.ps];
      if (pg < 0 || pg >= p->num_pages) return MK_ERR_CAPACITY;
    }
  }
  return MK_OK;
}

static int steps_one(mk_plan* p, const int* d_tokens, int n_steps, float* d_logits, int* d_next_token,
                     int io_stride, mk_stream stream) {
  if (!p || !d_tokens || !d_next_token || n_steps < 1 || io_stride < p->B) return MK_ERR_INVALID;
  int rc0 = steps_check(p, n_steps);
  if (rc0 != MK_OK) return rc0;
  cudaStream_t st = (cudaStream_t)stream;
  const Shape& s = p->s;
  if (needs_replan(p) || p->nucleus_built != nucleus_on(p)) {
    int rc = replan(p, st);
    if (rc != MK_OK) return rc;
  }
  if (p->nucleus_built && !p->d_lg_keep &&
      dalloc(p, &p->d_lg_keep, (size_t)p->bcap * s.V * sizeof(float)) != cudaSuccess)
    return note_cuda(cudaGetLastError(), "nucleus logits buffer");
  // keep epoch * count far from 32-bit wrap-around
  if ((unsigned long long)(p->epoch + n_steps) * 1024ull * 1024ull > 0x7fffffffull) {
    if (cudaMemsetAsync(p->d_ctr, 0, (size_t)p->cm.total * mk::CTR_STRIDE * sizeof(uint32_t), st) !=
        cudaSuccess)
      return MK_ERR_CUDA;
    p->epoch = 0;
  }
  fill_params(p);
  mk::Params P = p->P;
  P.epoch = p->epoch + 1;
  P.nsteps = n_steps;
  P.io_stride = io_stride;
  P.inv_temp = p->inv_temp;
  P.seed_lo = (uint32_t)(p->seed & 0xffffffffull);
  P.seed_hi = (uint32_t)(p->seed >> 32);
  P.slot0 = p->slot0;
  P.top_p = p->top_p;
  P.lg_keep = p->nucleus_built ? p->d_lg_keep : nullptr;
  P.sdone_cnt = p->nucleus_built ? p->B : 1;
  P.tokens = d_tokens;
  P.logits = d_logits;
  P.next_token = d_next_token;
  if (p->d_strace &&
      cudaMemsetAsync(p->d_strace, 0, (size_t)p->C * mk::STRACE_CAP * mk::STRACE_SLOTS * 8, st) != cudaSuccess)
    return note_cuda(cudaGetLastError(), "stage trace reset");
  cudaError_t e = mk::launch_megakernel(P, p->nb, p->C, p->smem, st);
  if (e != cudaSuccess) return note_cuda(e, "megakernel launch");
  p->epoch += (uint32_t)n_steps;
  for (int b = 0; b < p->B; ++b) p->seq[b] += n_steps;
  if (!p->chunk0.empty()) p->chunk_stepped = true;
  return MK_OK;
}

static int step_one(mk_plan* p, const int* d_tokens, float* d_logits, int* d_next_token, mk_stream stream) {
  if (!p) return MK_ERR_INVALID;
  return steps_one(p, d_tokens, 1, d_logits, d_next_token, p->B, stream);
}

static int step_host_one(mk_plan* p, const int* h_tokens, float* h_logits, int* h_next_token, mk_stream stream) {
  if (!p || !h_tokens || !h_next_token) return MK_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t tb = (size_t)p->B * sizeof(int);
  if (h_logits && !p->d_io_logits) {
    if (dalloc(p, &p->d_io_logits, (size_t)p->bcap * p->s.V * sizeof(float)) != cudaSuccess) return MK_ERR_CUDA;
  }
  if (cudaMemcpyAsync(p->d_io_tok, h_tokens, tb, cudaMemcpyHostToDevice, st) != cudaSuccess) return MK_ERR_CUDA;
  int rc = step_one(p, p->d_io_tok, h_logits ? p->d_io_logits : nullptr, p->d_io_next, stream);
  if (rc != MK_OK) return rc;
  if (cudaMemcpyAsync(h_next_token, p->d_io_next, tb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MK_ERR_CUDA;
  if (h_logits &&
      cudaMemcpyAsync(h_logits, p->d_io_logits, (size_t)p->B * p->s.V * sizeof(float), cudaMemcpyDeviceToHost,
                      st) != cudaSuccess)
    return MK_ERR_CUDA;
  if (cudaMemcpyAsync(p->h_status, p->d_status, 4 * sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MK_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MK_ERR_CUDA;
  return p->h_status[0];
}

// A task list built ahead (mk::plan_prebuild) for exactly the plan's new
// lengths; it is used once.
static bool take_prebuilt(mk_plan* p, Built& b) {
  const bool hit = p->pre_valid && p->pre && p->pre->nucleus == nucleus_on(p) && p->pre_seq == p->seq;
  p->pre_valid = false;
  if (hit) b = std::move(*p->pre);
  return hit;
}

// The first half of an update: checks, device capacity, and the new batch on
// the host side of the plan.
static int update_prepare(mk_plan* p, int batch, const int* seq_lens, const int* page_table, int max_pages_per_seq,
                          cudaStream_t st, const int* chunk_first = nullptr) {
  if (!p || batch < 1) return MK_ERR_INVALID;
  if (batch > p->ucap) return MK_ERR_CAPACITY;
  int rc = validate_batch(p->s, batch, seq_lens, page_table, max_pages_per_seq, p->num_pages, chunk_first);
  if (rc != MK_OK) return rc;
  if ((size_t)p->bcap * max_pages_per_seq > p->pt_cap || max_pages_per_seq * p->s.ps > p->rope_npos) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return MK_ERR_CUDA;
    dfree(p, p->d_pt);
    p->d_pt = nullptr;
    p->pt_cap = (size_t)p->bcap * max_pages_per_seq;
    if (dalloc(p, &p->d_pt, p->pt_cap * sizeof(int)) != cudaSuccess) return MK_ERR_CUDA;
    if (max_pages_per_seq * p->s.ps > p->rope_npos) {
      dfree(p, p->d_rope);
      p->d_rope = nullptr;
      p->rope_npos = max_pages_per_seq * p->s.ps;
      if (dalloc(p, &p->d_rope, (size_t)p->rope_npos * (p->s.d / 2) * sizeof(float2)) != cudaSuccess)
        return MK_ERR_CUDA;
      if (mk::launch_rope_table(p->d_rope, p->rope_npos, p->s.d, (double)p->s.theta, st) != cudaSuccess)
        return MK_ERR_CUDA;
    }
  }
  p->B = batch;
  p->max_pages = max_pages_per_seq;
  p->seq.assign(seq_lens, seq_lens + batch);
  p->pt.assign(page_table, page_table + (size_t)batch * max_pages_per_seq);
  set_chunks(p, batch, chunk_first);
  return MK_OK;
}

// The last half: upload the built list with the batch, clear the status word.
static int update_commit(mk_plan* p, Built& b, cudaStream_t st) {
  int rc = commit_built(p, b, st, true);
  if (rc != MK_OK) return rc;
  if (cudaMemsetAsync(p->d_status, 0, 4 * sizeof(int), st) != cudaSuccess) return MK_ERR_CUDA;
  fill_params(p);
  return MK_OK;
}

static int update_one(mk_plan* p, int batch, const int* seq_lens, const int* page_table, int max_pages_per_seq,
                      mk_stream stream, const int* chunk_first = nullptr) {
  cudaStream_t st = (cudaStream_t)stream;
  int rc = update_prepare(p, batch, seq_lens, page_table, max_pages_per_seq, st, chunk_first);
  if (rc != MK_OK) return rc;
  Built b;
  if (!take_prebuilt(p, b)) build_for(p, b);
  return update_commit(p, b, st);
}

static int sync_one(mk_plan* p, mk_stream stream) {
  if (!p) return MK_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(p->h_status, p->d_status, 4 * sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return note_cuda(e, "mk_plan_sync status copy");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return note_cuda(e, "mk_plan_sync");
  return p->h_status[0];
}

static int read_debug_one(mk_plan* p, int what, void* dst, size_t bytes, mk_stream stream) {
  if (!p || !dst) return MK_ERR_INVALID;
  cudaStream_t st = (cudaStream_t)stream;
  const Shape& s = p->s;
  const size_t B = p->B, bc = p->bcap, L = s.L;
  size_t row = 0;
  const uint8_t* src = nullptr;
  switch (what) {
    case MK_DBG_HIDDEN: row = s.H * 4; src = (const uint8_t*)p->P.x_out; break;
    case MK_DBG_EXPERT_IDS: row = s.k * 4; src = (const uint8_t*)p->P.ids; break;
    case MK_DBG_GATES: row = s.k * 4; src = (const uint8_t*)p->P.gates; break;
    case MK_DBG_ROUTER_LOGITS: row = s.E * 4; src = (const uint8_t*)p->P.rlog; break;
    case MK_DBG_SEQ_LENS:
      if (bytes < B * 4) return MK_ERR_INVALID;
      return cudaMemcpyAsync(dst, p->d_seq, B * 4, cudaMemcpyDefault, st) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
    case MK_DBG_TASKS: {
      const size_t n = p->tasks.size();
      if (bytes < n * 12 * 4) return MK_ERR_INVALID;
      if (cudaStreamSynchronize(st) != cudaSuccess) return MK_ERR_CUDA;
      std::vector<int> v(n * 12);
      for (size_t i = 0; i < n; ++i) {
        const Task& t = p->tasks[i];
        v[i * 12 + 0] = t.type;
        v[i * 12 + 1] = t.layer;
        for (int j = 0; j < 8; ++j) v[i * 12 + 2 + j] = t.a[j];
        v[i * 12 + 10] = t.wait_ctr;
        v[i * 12 + 11] = (int)t.wait_cnt;
      }
      return cudaMemcpy(dst, v.data(), n * 12 * 4, cudaMemcpyDefault) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
    }
    case MK_DBG_TRACE: {
      const size_t n = p->tasks.size() * mk::TRACE_SLOTS * sizeof(unsigned long long);
      if (!p->trace || !p->d_trace || bytes < n) return MK_ERR_INVALID;
      return cudaMemcpyAsync(dst, p->d_trace, n, cudaMemcpyDefault, st) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
    }
    case MK_DBG_STAGE_TRACE: {
      const size_t n = (size_t)p->C * mk::STRACE_CAP * mk::STRACE_SLOTS * sizeof(unsigned long long);
      if (p->trace < 2 || !p->d_strace || bytes < n) return MK_ERR_INVALID;
      return cudaMemcpyAsync(dst, p->d_strace, n, cudaMemcpyDefault, st) == cudaSuccess ? MK_OK : MK_ERR_CUDA;
    }
    case MK_DBG_UNION:
      if (bytes < L * 4) return MK_ERR_INVALID;
      return cudaMemcpy2DAsync(dst, 4, p->P.route, (size_t)p->rm.ints * 4, 4, L, cudaMemcpyDefault, st) ==
                     cudaSuccess
                 ? MK_OK
                 : MK_ERR_CUDA;
    default: return MK_ERR_INVALID;
  }
  if (bytes < B * L * row) return MK_ERR_INVALID;
  // device layout [L][bcap][row] -> caller layout [B][L][row]
  for (size_t b = 0; b < B; ++b) {
    if (cudaMemcpy2DAsync((uint8_t*)dst + b * L * row, row, src + b * row, bc * row, row, L, cudaMemcpyDefault,
                          st) != cudaSuccess)
      return MK_ERR_CUDA;
  }
  return MK_OK;
}

static int info_one(const mk_plan* p, int* out, int n) {
  if (!p || !out) return MK_ERR_INVALID;
  const int v[12] = {p->C, (int)p->tasks.size(), p->nstages, p->stage_bytes, p->smem, p->B,
                     p->cnt.attn, p->cnt.gu, p->cnt.lm, p->replans, p->P.tm_gu ? 1 : 0, p->P.tm_qkv ? 1 : 0};
  for (int i = 0; i < n && i < 12; ++i) out[i] = v[i];
  return MK_OK;
}

static void destroy_one(mk_plan* p) {
  if (!p) return;
  for (void* v : p->allocs) cudaFree(v);
  p->allocs.clear();
  for (int k = 0; k < 2; ++k) {
    if (p->h_stage[k]) cudaFreeHost(p->h_stage[k]);
    if (p->ev_stage[k]) cudaEventDestroy(p->ev_stage[k]);
  }
  if (p->h_status) cudaFreeHost(p->h_status);
  if (p->h_next) cudaFreeHost(p->h_next);
  if (p->h_tok) cudaFreeHost(p->h_tok);
  delete p->pre;
  delete p;
}

// ---- the public entry points: one plan, or a group of sub-plans

static void destroy_group(mk_plan* g) {
  for (mk_plan* sp : g->subs) destroy_one(sp);
  delete g;
}

int mk_plan_create(const mk_model_dims* dims, const mk_weights* w, const mk_kv* kv, int batch,
                   const int* seq_lens, const int* page_table, int max_pages_per_seq,
                   const mk_plan_opts* opts, mk_plan** out) {
  if (!out) return MK_ERR_INVALID;
  *out = nullptr;
  mk_plan_opts o = {};
  if (opts) o = *opts;
  const int bcap = o.max_batch > 0 ? o.max_batch : batch;
  if (bcap <= mk::MAX_BATCH) return create_one(dims, w, kv, batch, seq_lens, page_table, max_pages_per_seq, opts, out);
  if (batch < 1 || batch > bcap || !seq_lens || !page_table || max_pages_per_seq < 1) return MK_ERR_INVALID;
  const int M = mk::MAX_BATCH;
  if (o.chunk_first) {   // prefill chunks: each stays inside one sub-plan
    Shape s;
    int rc = check_dims(dims, s);
    if (rc != MK_OK) return rc;
    if (!kv) return MK_ERR_INVALID;
    rc = validate_batch(s, batch, seq_lens, page_table, max_pages_per_seq, kv->num_pages, o.chunk_first, M);
    if (rc != MK_OK) return rc;
  }
  mk_plan* g = new (std::nothrow) mk_plan();
  if (!g) return MK_ERR_CUDA;
  for (int i = 0; i * M < bcap; ++i) {
    const int n = std::max(0, std::min(M, batch - i * M));
    mk_plan_opts so = o;
    so.max_batch = std::min(M, bcap - i * M);
    std::vector<int> cf;
    so.chunk_first = nullptr;
    if (o.chunk_first && n > 0) {
      cf.resize(n);
      for (int b = 0; b < n; ++b) cf[b] = o.chunk_first[i * M + b] - i * M;
      so.chunk_first = cf.data();
    }
    // an idle sub-plan is built over the group's first request and stepped
    // only once an update gives it requests of its own
    const int* sl = n > 0 ? seq_lens + (size_t)i * M : seq_lens;
    const int* pt = n > 0 ? page_table + (size_t)i * M * max_pages_per_seq : page_table;
    mk_plan* sp = nullptr;
    const int rc = create_one(dims, w, kv, n > 0 ? n : 1, sl, pt, max_pages_per_seq, &so, &sp);
    if (rc != MK_OK) {
      destroy_group(g);
      return rc;
    }
    sp->slot0 = i * M;
    g->subs.push_back(sp);
    g->sub_B.push_back(n);
  }
  g->s = g->subs[0]->s;
  g->B = g->group_B = batch;
  g->bcap = bcap;
  *out = g;
  return MK_OK;
}

// A group's sub-plans that hold requests all pass their checks, or none runs.
static int group_check(const mk_plan* p, int n_steps) {
  for (size_t i = 0; i < p->subs.size(); ++i) {
    if (p->sub_B[i] == 0) continue;
    const int rc = steps_check(p->subs[i], n_steps);
    if (rc != MK_OK) return rc;
  }
  return MK_OK;
}

int mk_decode_step(mk_plan* p, const int* d_tokens, float* d_logits, int* d_next_token, mk_stream stream) {
  if (!p || p->subs.empty()) return step_one(p, d_tokens, d_logits, d_next_token, stream);
  if (!d_tokens || !d_next_token) return MK_ERR_INVALID;
  const int rc0 = group_check(p, 1);
  if (rc0 != MK_OK) return rc0;
  const size_t M = mk::MAX_BATCH, V = p->s.V;
  for (size_t i = 0; i < p->subs.size(); ++i) {
    if (p->sub_B[i] == 0) continue;
    const int rc = step_one(p->subs[i], d_tokens + i * M, d_logits ? d_logits + i * M * V : nullptr,
                            d_next_token + i * M, stream);
    if (rc != MK_OK) return rc;
  }
  return MK_OK;
}

int mk_decode_steps(mk_plan* p, const int* d_tokens, int n_steps, float* d_logits, int* d_next_tokens,
                    mk_stream stream) {
  if (!p || p->subs.empty()) return steps_one(p, d_tokens, n_steps, d_logits, d_next_tokens, p ? p->B : 0, stream);
  if (!d_tokens || !d_next_tokens || n_steps < 1) return MK_ERR_INVALID;
  const int rc0 = group_check(p, n_steps);
  if (rc0 != MK_OK) return rc0;
  // requests of different sub-plans are independent: each sub-plan runs its
  // n_steps in one launch of its own, writing its columns of the rows
  const size_t M = mk::MAX_BATCH, V = p->s.V;
  const int stride = p->group_B;
  for (size_t i = 0; i < p->subs.size(); ++i) {
    if (p->sub_B[i] == 0) continue;
    const int rc = steps_one(p->subs[i], d_tokens + i * M, n_steps, d_logits ? d_logits + i * M * V : nullptr,
                             d_next_tokens + i * M, stride, stream);
    if (rc != MK_OK) return rc;
  }
  return MK_OK;
}

int mk_decode_step_host(mk_plan* p, const int* h_tokens, float* h_logits, int* h_next_token, mk_stream stream) {
  if (!p || p->subs.empty()) return step_host_one(p, h_tokens, h_logits, h_next_token, stream);
  if (!h_tokens || !h_next_token) return MK_ERR_INVALID;
  const int rc0 = group_check(p, 1);
  if (rc0 != MK_OK) return rc0;
  const size_t M = mk::MAX_BATCH, V = p->s.V;
  for (size_t i = 0; i < p->subs.size(); ++i) {
    if (p->sub_B[i] == 0) continue;
    const int rc = step_host_one(p->subs[i], h_tokens + i * M, h_logits ? h_logits + i * M * V : nullptr,
                                 h_next_token + i * M, stream);
    if (rc != MK_OK) return rc;
  }
  return MK_OK;
}

int mk_plan_update_rows(mk_plan* p, int batch, const int* seq_lens, const int* page_table, int max_pages_per_seq,
                        const int* chunk_first, mk_stream stream) {
  if (!p || p->subs.empty())
    return update_one(p, batch, seq_lens, page_table, max_pages_per_seq, stream, chunk_first);
  if (batch < 1 || !seq_lens || !page_table || max_pages_per_seq < 1) return MK_ERR_INVALID;
  if (batch > p->bcap) return MK_ERR_CAPACITY;
  const int M = mk::MAX_BATCH;
  // whole-batch check first: pages are shared only within a chunk, and a
  // chunk stays inside one sub-plan
  int rc = validate_batch(p->s, batch, seq_lens, page_table, max_pages_per_seq, p->subs[0]->num_pages, chunk_first, M);
  if (rc != MK_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t n = p->subs.size();
  std::vector<int> nb(n);
  std::vector<std::vector<int>> cf(n);
  for (size_t i = 0; i < n; ++i) {
    nb[i] = std::max(0, std::min(M, batch - (int)i * M));
    if (nb[i] == 0) continue;
    if (chunk_first) {
      cf[i].resize(nb[i]);
      for (int b = 0; b < nb[i]; ++b) cf[i][b] = chunk_first[i * M + b] - (int)i * M;
    }
    rc = update_prepare(p->subs[i], nb[i], seq_lens + i * M, page_table + i * M * max_pages_per_seq,
                        max_pages_per_seq, st, chunk_first ? cf[i].data() : nullptr);
    if (rc != MK_OK) return rc;
  }
  // the task lists are host work: one thread per sub-plan that holds requests
  std::vector<Built> built(n);
  std::vector<std::thread> th;
  for (size_t i = 0; i < n; ++i)
    if (nb[i] > 0 && !take_prebuilt(p->subs[i], built[i])) th.emplace_back([&, i] { build_for(p->subs[i], built[i]); });
  for (auto& t : th) t.join();
  for (size_t i = 0; i < n; ++i) {
    if (nb[i] > 0) {
      rc = update_commit(p->subs[i], built[i], st);
      if (rc != MK_OK) return rc;
    }
    p->sub_B[i] = nb[i];
  }
  p->B = p->group_B = batch;
  return MK_OK;
}

int mk_plan_update(mk_plan* p, int batch, const int* seq_lens, const int* page_table, int max_pages_per_seq,
                   mk_stream stream) {
  return mk_plan_update_rows(p, batch, seq_lens, page_table, max_pages_per_seq, nullptr, stream);
}

int mk_plan_set_sampling(mk_plan* p, float temperature, unsigned long long seed) {
  if (!p || !temperature_ok(temperature)) {
    mk::set_last_error("mk_plan_set_sampling: temperature must be 0 (greedy) or a finite value whose inverse is finite");
    return MK_ERR_INVALID;
  }
  const float it = temperature > 0.f ? 1.0f / temperature : 0.f;
  p->inv_temp = it;
  p->seed = seed;
  for (mk_plan* s : p->subs) {
    s->inv_temp = it;
    s->seed = seed;
  }
  return MK_OK;
}

int mk_plan_set_top_p(mk_plan* p, float top_p) {
  if (!p || !(top_p > 0.f && top_p <= 1.f)) {
    mk::set_last_error("mk_plan_set_top_p: top_p must be in (0, 1]");
    return MK_ERR_INVALID;
  }
  p->top_p = top_p;
  for (mk_plan* s : p->subs) s->top_p = top_p;
  return MK_OK;
}

int mk_plan_sync(mk_plan* p, mk_stream stream) {
  if (!p || p->subs.empty()) return sync_one(p, stream);
  for (size_t i = 0; i < p->subs.size(); ++i) {
    if (p->sub_B[i] == 0) continue;
    const int rc = sync_one(p->subs[i], stream);
    if (rc != MK_OK) return rc;
  }
  return MK_OK;
}

int mk_plan_read_debug(mk_plan* p, int what, void* dst, size_t bytes, mk_stream stream) {
  if (!p || p->subs.empty()) return read_debug_one(p, what, dst, bytes, stream);
  if (!dst) return MK_ERR_INVALID;
  const size_t L = p->s.L;
  size_t per = 0;   // bytes per request
  switch (what) {
    case MK_DBG_HIDDEN: per = L * p->s.H * 4; break;
    case MK_DBG_EXPERT_IDS: case MK_DBG_GATES: per = L * p->s.k * 4; break;
    case MK_DBG_ROUTER_LOGITS: per = L * p->s.E * 4; break;
    case MK_DBG_SEQ_LENS: per = 4; break;
    default: return MK_ERR_UNSUPPORTED;   // per-plan records: read them from a plan of at most 8 requests
  }
  if (bytes < (size_t)p->group_B * per) return MK_ERR_INVALID;
  const size_t M = mk::MAX_BATCH;
  for (size_t i = 0; i < p->subs.size(); ++i) {
    if (p->sub_B[i] == 0) continue;
    const int rc = read_debug_one(p->subs[i], what, (uint8_t*)dst + i * M * per, (size_t)p->sub_B[i] * per, stream);
    if (rc != MK_OK) return rc;
  }
  return MK_OK;
}

int mk_plan_info(const mk_plan* p, int* out, int n) {
  if (!p || p->subs.empty()) return info_one(p, out, n);
  if (!out) return MK_ERR_INVALID;
  int v[12] = {0};
  for (size_t i = 0; i < p->subs.size(); ++i) {
    int w[12];
    info_one(p->subs[i], w, 12);
    if (i == 0)
      for (int j = 0; j < 12; ++j) v[j] = w[j];
    else
      for (int j : {1, 6, 7, 8, 9}) v[j] += w[j];   // tasks, attention / expert / LM tiles, replans
  }
  v[5] = p->group_B;
  for (int i = 0; i < n && i < 12; ++i) out[i] = v[i];
  return MK_OK;
}

void mk_plan_destroy(mk_plan* p) {
  if (!p) return;
  if (p->subs.empty()) destroy_one(p);
  else destroy_group(p);
}

}  // extern "C"

// ------------------------------------------------------------------ serving-loop helpers
// Used by mk_serve_step: a step enqueued from host tokens without waiting
// for it, the wait, and a task list built ahead for the next batch's lengths
// while the GPU runs the current step.
namespace mk {

static int step_host_begin_one(mk_plan* q, const int* h_tokens, mk_stream stream) {
  cudaStream_t st = (cudaStream_t)stream;
  const size_t tb = (size_t)q->B * sizeof(int);
  memcpy(q->h_tok, h_tokens, tb);
  if (cudaMemcpyAsync(q->d_io_tok, q->h_tok, tb, cudaMemcpyHostToDevice, st) != cudaSuccess) return MK_ERR_CUDA;
  const int rc = step_one(q, q->d_io_tok, nullptr, q->d_io_next, stream);
  if (rc != MK_OK) return rc;
  if (cudaMemcpyAsync(q->h_next, q->d_io_next, tb, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MK_ERR_CUDA;
  if (cudaMemcpyAsync(q->h_status, q->d_status, 4 * sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MK_ERR_CUDA;
  return MK_OK;
}

int plan_step_host_begin(mk_plan* p, const int* h_tokens, mk_stream stream) {
  if (!p || !h_tokens) return MK_ERR_INVALID;
  if (p->subs.empty()) return step_host_begin_one(p, h_tokens, stream);
  const int rc0 = group_check(p, 1);
  if (rc0 != MK_OK) return rc0;
  for (size_t i = 0; i < p->subs.size(); ++i) {
    if (p->sub_B[i] == 0) continue;
    const int rc = step_host_begin_one(p->subs[i], h_tokens + i * MAX_BATCH, stream);
    if (rc != MK_OK) return rc;
  }
  return MK_OK;
}

int plan_step_host_end(mk_plan* p, int* h_next, mk_stream stream) {
  if (!p || !h_next) return MK_ERR_INVALID;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return note_cuda(cudaGetLastError(), "serve step");
  if (p->subs.empty()) {
    memcpy(h_next, p->h_next, (size_t)p->B * sizeof(int));
    return p->h_status[0];
  }
  int st = MK_OK;
  for (size_t i = 0; i < p->subs.size(); ++i) {
    if (p->sub_B[i] == 0) continue;
    memcpy(h_next + i * MAX_BATCH, p->subs[i]->h_next, (size_t)p->sub_B[i] * sizeof(int));
    if (st == MK_OK) st = p->subs[i]->h_status[0];
  }
  return st;
}

static void prebuild_one(mk_plan* q, int batch, const int* seq_lens) {
  q->pre_valid = false;
  if (batch < 1 || batch > q->bcap) return;
  if (!q->pre) q->pre = new (std::nothrow) Built();
  if (!q->pre) return;
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] < 0) return;
  build_for(q, *q->pre, batch, seq_lens);
  q->pre_seq.assign(seq_lens, seq_lens + batch);
  q->pre_valid = q->pre->rc == MK_OK;
}

void plan_prebuild(mk_plan* p, int batch, const int* seq_lens) {
  if (!p || !seq_lens) return;
  if (p->subs.empty()) {
    prebuild_one(p, batch, seq_lens);
    return;
  }
  std::vector<std::thread> th;
  for (size_t i = 0; i < p->subs.size(); ++i) {
    const int nb = std::max(0, std::min(MAX_BATCH, batch - (int)i * MAX_BATCH));
    if (nb == 0) {
      p->subs[i]->pre_valid = false;
      continue;
    }
    th.emplace_back([p, i, nb, seq_lens] { prebuild_one(p->subs[i], nb, seq_lens + i * MAX_BATCH); });
  }
  for (auto& t : th) t.join();
}

}  // namespace mk
