// mk_decode_step_noalloc: one decode step that performs no memory allocation.
//
// Some callers cannot call cudaMalloc at the point where they decode: hosts
// that reserve all device memory up front in their own pool and forbid raw
// allocations inside their enqueue callbacks (plugin interfaces of inference
// runtimes, custom-allocator hooks that would recurse), and latency-critical
// loops that cannot afford the device-wide synchronisation cudaMalloc and
// cudaFree may imply.  This entry point serves them: the megakernel's scratch
// (task list, dependency counters, per-layer activations, attention partials,
// RoPE table, pointer tables) lives in one file-scope __device__ array of
// fixed size, and the host-side task list is built in a file-scope host
// array, so neither side allocates.
//
// Costs of that choice, stated for users:
//   * every GPU that loads libmk.so holds MK_NOALLOC_SCRATCH_BYTES (64 MiB) of
//     device memory for this array until the process exits;
//   * all calls share the array (and the host staging array), so calls whose
//     work overlaps on the GPU, or that run concurrently from several host
//     threads, race and produce garbage; serialise them (one stream, one
//     thread at a time);
//   * the first call on a device looks up the array's device address with
//     cudaGetSymbolAddress (with that device current); make that first call
//     before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "mk.h"
#include "mk_internal.h"

namespace mk {
cudaError_t launch_megakernel(const Params& p, int nb, int grid, int smem, cudaStream_t st);
cudaError_t launch_rope_table(float2* tab, int npos, int d, double theta, cudaStream_t st);
int max_active_ctas(int nb, int smem);
size_t misc_bytes();
void set_last_error(const char* msg);
}  // namespace mk

namespace {

constexpr size_t kScratchBytes = 64ull << 20;   // device scratch limit (MK_NOALLOC_SCRATCH_BYTES)
constexpr size_t kHostBytes = 4ull << 20;       // host staging limit (task list, tables)
constexpr int kMaxCtas = 1024;
constexpr int kMaxDevices = 64;

// The device scratch.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

alignas(256) static unsigned char g_host_stage[kHostBytes];
static void* g_dev_base[kMaxDevices];           // device address of the scratch, per device
static int g_cta_count[kMaxCtas + 1];
static int g_cta_cursor[kMaxCtas];

int fail(int code, const char* msg) {
  mk::set_last_error(msg);
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof(buf), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
  mk::set_last_error(buf);
  return MK_ERR_CUDA;
}

struct Shape {
  int L, H, nq, nkv, d, E, k, F, V, ps, G, qkv_rows;
};

int shape_of(const mk_model_dims* m, Shape& s) {
  if (!m) return MK_ERR_INVALID;
  s = Shape{m->n_layers, m->hidden, m->n_q_heads, m->n_kv_heads, m->head_dim, m->n_experts, m->top_k,
            m->expert_ffn, m->vocab, m->page_size, 0, 0};
  if (s.L < 1 || s.H < 8 || s.nq < 1 || s.nkv < 1 || s.E < 1 || s.k < 1 || s.F < 8 || s.V < 1) return MK_ERR_INVALID;
  if (s.nq % s.nkv || s.k > s.E || !(m->rms_eps >= 0.f) || !(m->rope_theta > 0.f)) return MK_ERR_INVALID;
  if (s.H % 8 || s.F % 8 || (s.nq * s.d) % 8) return MK_ERR_INVALID;
  s.G = s.nq / s.nkv;
  if (s.ps != 16 || (s.d != 64 && s.d != 128) || s.G > mk::MAX_G || s.k > mk::MAX_TOPK || s.E > mk::MAX_EXPERTS)
    return MK_ERR_UNSUPPORTED;
  s.qkv_rows = s.nkv * (s.G + 2) * s.d;
  return MK_OK;
}

inline int pages_for(int len, int ps) { return len / ps + 1; }

inline void split_range(int n, int parts, int i, int& a, int& b) {
  a = (int)((long long)n * i / parts);
  b = (int)((long long)n * (i + 1) / parts);
}

struct Counts {
  int qkv_per_g, o, gu, down, lm, P, slots, down_rows_max, ntasks, hpc, comb;
};

// Emits the step's tasks phase by phase in topological order; a phase with n
// tasks goes to n consecutive CTAs starting where the previous phase stopped.
// Called twice: first to count tasks per CTA, then to place them.
template <class Put>
void emit(const Shape& s, int B, const int* seq_lens, int C, Counts& c, Put put) {
  mk::CtrMap cm;
  cm.init(s.L, s.nkv, B);
  const int Rg = (s.G + 2) * s.d;
  const int umax = s.E < B * s.k ? s.E : B * s.k;
  c.qkv_per_g = (C + s.nkv - 1) / s.nkv;
  if (c.qkv_per_g > Rg) c.qkv_per_g = Rg;
  c.o = C < s.H ? C : s.H;
  c.gu = mk::moe_tiles(umax, s.F, C, B, mk::cf_floats(s.E, s.k, s.F, C, B));
  c.down = C < s.H ? C : s.H;
  c.lm = 4 * C < s.V ? 4 * C : s.V;
  c.down_rows_max = (s.H + c.down - 1) / c.down;
  long long total_pages = 0;
  for (int b = 0; b < B; ++b) total_pages += pages_for(seq_lens[b], s.ps);
  long long P = (total_pages * s.nkv + C - 1) / C;
  c.P = P < 1 ? 1 : (int)P;
  for (int b = 0; b < B; ++b) {   // the split-KV combine takes at most 128 chunks per (request, group)
    const int need = (pages_for(seq_lens[b], s.ps) + 127) / 128;
    if (c.P < need) c.P = need;
  }
  c.slots = 0;
  for (int b = 0; b < B; ++b) c.slots += (pages_for(seq_lens[b], s.ps) + c.P - 1) / c.P * s.nkv;
  // query heads per combine task: the smallest divisor of G within one task per CTA, else G
  c.hpc = s.G;
  for (int h = 1; h <= s.G; ++h)
    if (s.G % h == 0 && (long long)B * s.nkv * (s.G / h) <= C) {
      c.hpc = h;
      break;
    }
  c.comb = B * s.nkv * (s.G / c.hpc);
  int rot = 0;
  auto task = [](int type, int layer, int wc, uint32_t wn) {
    mk::Task t;
    memset(&t, 0, sizeof(t));
    t.type = type;
    t.layer = layer;
    t.wait_ctr = wc;
    t.wait_cnt = wn;
    return t;
  };
  auto next = [&]() {
    const int r = rot;
    rot = (rot + 1) % C;
    return r;
  };
  for (int l = 0; l < s.L; ++l) {
    for (int g = 0; g < s.nkv; ++g)
      for (int i = 0; i < c.qkv_per_g; ++i) {
        int a, b;
        split_range(Rg, c.qkv_per_g, i, a, b);
        mk::Task t = task(mk::T_QKV, l, l == 0 ? -1 : cm.down + l - 1, (uint32_t)c.down);
        t.a[0] = g * Rg + a;
        t.a[1] = g * Rg + b;
        t.a[2] = g;
        put(next(), t);
      }
    int slot = 0;
    for (int b = 0; b < B; ++b) {
      const int nch = (pages_for(seq_lens[b], s.ps) + c.P - 1) / c.P;
      for (int g = 0; g < s.nkv; ++g) {
        const int first = slot;
        for (int ch = 0; ch < nch; ++ch) {
          mk::Task t = task(mk::T_ATTN, l, cm.qkv + l * s.nkv + g, (uint32_t)c.qkv_per_g);
          t.a[0] = b;
          t.a[1] = g;
          t.a[2] = ch * c.P;
          t.a[3] = ch == nch - 1 ? -1 : (ch + 1) * c.P;
          t.a[4] = slot++;
          t.a[5] = first;
          t.a[6] = nch;
          put(next(), t);
        }
      }
    }
    slot = 0;
    for (int b = 0; b < B; ++b) {
      const int nch = (pages_for(seq_lens[b], s.ps) + c.P - 1) / c.P;
      for (int g = 0; g < s.nkv; ++g) {
        for (int h = 0; h < s.G; h += c.hpc) {
          mk::Task t = task(mk::T_COMB, l, cm.attn_idx(l, b, g), (uint32_t)nch);
          t.a[0] = b;
          t.a[1] = g;
          t.a[2] = h;
          t.a[3] = c.hpc;
          t.a[5] = slot;
          t.a[6] = nch;
          put(next(), t);
        }
        slot += nch;
      }
    }
    for (int i = 0; i < c.o; ++i) {
      int a, b;
      split_range(s.H, c.o, i, a, b);
      mk::Task t = task(mk::T_OPROJ, l, cm.combine + l, (uint32_t)c.comb);
      t.a[0] = a;
      t.a[1] = b;
      t.a[2] = i;
      put(next(), t);
    }
    for (int i = 0; i < c.gu; ++i) {
      mk::Task t = task(mk::T_MOE, l, cm.o + l, (uint32_t)c.o);
      t.a[0] = i;
      t.a[1] = c.gu;
      put(next(), t);
    }
    for (int i = 0; i < c.down; ++i) {
      int a, b;
      split_range(s.H, c.down, i, a, b);
      mk::Task t = task(mk::T_RED, l, cm.gu + l, (uint32_t)c.gu);
      t.a[0] = a;
      t.a[1] = b;
      t.a[2] = c.gu;
      put(next(), t);
    }
  }
  for (int i = 0; i < c.lm; ++i) {
    int a, b;
    split_range(s.V, c.lm, i, a, b);
    mk::Task t = task(mk::T_LM, s.L - 1, cm.down + s.L - 1, (uint32_t)c.down);
    t.a[0] = a;
    t.a[1] = b;
    t.a[2] = i;
    t.a[3] = c.lm;
    put(next(), t);
  }
}

// Bump allocator over a fixed region (no memory is allocated: it only hands out offsets).
struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = (off + 255) & ~(size_t)255;
    off = o + bytes;
    return o;
  }
};

}  // namespace

extern "C" int mk_decode_step_noalloc(const mk_model_dims* dims, const mk_weights* w, const mk_kv* kv, int batch,
                                      const int* seq_lens, const int* page_table, int max_pages_per_seq,
                                      const int* d_tokens, float* d_logits, int* d_next_token, int* d_status,
                                      mk_stream stream) {
  mk::set_last_error("");
  Shape s;
  int rc = shape_of(dims, s);
  if (rc != MK_OK) return fail(rc, "unsupported or invalid model shape");
  if (!w || !kv || !seq_lens || !page_table || !d_tokens || !d_next_token || batch < 1 || max_pages_per_seq < 1)
    return fail(MK_ERR_INVALID, "null argument or empty batch");
  if (batch > mk::MAX_BATCH) return fail(MK_ERR_UNSUPPORTED, "batch above 8");
  if (!w->attn_norm || !w->wqkv || !w->wo || !w->ffn_norm || !w->router || !w->w_gate_up || !w->w_down ||
      !kv->kv_pool || !w->embed || !w->final_norm || !w->lm_head)
    return fail(MK_ERR_INVALID, "null weight or KV pointer");
  int max_len = 0;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens[b] < 0) return fail(MK_ERR_INVALID, "negative sequence length");
    const int np = pages_for(seq_lens[b], s.ps);
    if (np > max_pages_per_seq) return fail(MK_ERR_CAPACITY, "no page for the next position");
    for (int i = 0; i < np; ++i) {
      const int pg = page_table[(size_t)b * max_pages_per_seq + i];
      if (pg < 0 || pg >= kv->num_pages) return fail(MK_ERR_INVALID, "page table entry out of range");
    }
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  }
  cudaStream_t st = (cudaStream_t)stream;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MK_ERR_UNSUPPORTED, "device ordinal above 63");
  if (!g_dev_base[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
    g_dev_base[dev] = ptr;
  }
  unsigned char* base = (unsigned char*)g_dev_base[dev];
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  const int C = sms < kMaxCtas ? sms : kMaxCtas;
  const int B = batch;
  const int nb = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;

  // count tasks per CTA, then place them CTA-major
  Counts cnt;
  for (int i = 0; i <= C; ++i) g_cta_count[i] = 0;
  emit(s, B, seq_lens, C, cnt, [&](int cta, const mk::Task&) { g_cta_count[cta]++; });
  long long ntasks = 0;
  for (int i = 0; i < C; ++i) ntasks += g_cta_count[i];
  cnt.ntasks = (int)ntasks;

  // host staging layout: weight tables | seq lens | page table | tasks | cta offsets
  const size_t L = s.L;
  Carve hc;
  const size_t h_tab = hc.take(8 * L * sizeof(void*));
  const size_t h_seq = hc.take((size_t)B * sizeof(int));
  const size_t h_pt = hc.take((size_t)B * max_pages_per_seq * sizeof(int));
  const size_t h_tasks = hc.take((size_t)ntasks * sizeof(mk::Task));
  const size_t h_cta = hc.take((size_t)(C + 1) * sizeof(int));
  const size_t h_bytes = hc.off;
  if (h_bytes > kHostBytes) return fail(MK_ERR_CAPACITY, "task list larger than the 4 MiB host staging limit");

  // device scratch layout: the staged blob, then the kernel's working buffers
  const int umax = s.E < B * s.k ? s.E : B * s.k;
  mk::CtrMap cm;
  cm.init(s.L, s.nkv, B);
  mk::RouteMap rm;
  rm.init(umax, B);
  const int npos = max_len + 1;
  Carve dc;
  const size_t d_blob = dc.take(h_bytes);
  const size_t d_ctr = dc.take((size_t)cm.total * mk::CTR_STRIDE * sizeof(uint32_t));
  const size_t d_stat = dc.take(4 * sizeof(int));
  const size_t d_rope = dc.take((size_t)npos * (s.d / 2) * sizeof(float2));
  const size_t d_qkv = dc.take(L * B * s.qkv_rows * sizeof(float));
  const size_t d_part = dc.take(L * (size_t)cnt.slots * s.G * (s.d + 4) * sizeof(float));
  const size_t d_o = dc.take(L * B * s.nq * s.d * sizeof(float));
  const size_t d_xm = dc.take(L * B * s.H * sizeof(float));
  const size_t d_xo = dc.take(L * B * s.H * sizeof(float));
  const size_t d_rl = dc.take(L * B * s.E * sizeof(float));
  const size_t d_ids = dc.take(L * B * s.k * sizeof(int));
  const size_t d_gt = dc.take(L * B * s.k * sizeof(float));
  const size_t d_route = dc.take(L * rm.ints * sizeof(int));
  const size_t d_mp = dc.take((size_t)cnt.gu * B * s.H * sizeof(float));
  const size_t d_rp = dc.take(L * mk::RL_COPIES * B * s.E * sizeof(unsigned long long));
  const size_t d_lmv = dc.take((size_t)B * cnt.lm * sizeof(float));
  const size_t d_lmi = dc.take((size_t)B * cnt.lm * sizeof(int));
  const size_t d_mm = dc.take(L * (size_t)cnt.gu * sizeof(uint32_t));
  if (dc.off > kScratchBytes) {
    char buf[160];
    snprintf(buf, sizeof(buf), "step needs %zu bytes of scratch, above the %zu-byte static limit", dc.off,
             kScratchBytes);
    return fail(MK_ERR_CAPACITY, buf);
  }

  // shared-memory plan (same layout rule as mk_plan_create)
  mk::SmemPlan sp;
  if (!mk::plan_smem(s.H, s.nq, s.d, s.G, s.E, s.F, s.ps, B, nb, cnt.down_rows_max,
                     mk::cf_floats(s.E, s.k, s.F, C, B), mk::misc_bytes(), sp))
    return fail(MK_ERR_UNSUPPORTED, "shape leaves no room for the shared-memory ring");
  const int smem = sp.smem;
  if (mk::max_active_ctas(nb, smem) < 1) return fail(MK_ERR_CUDA, "megakernel does not fit on an SM");

  // fill the host staging array
  unsigned char* hb = g_host_stage;
  const void** tab = (const void**)(hb + h_tab);
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
  memcpy(hb + h_seq, seq_lens, (size_t)B * sizeof(int));
  memcpy(hb + h_pt, page_table, (size_t)B * max_pages_per_seq * sizeof(int));
  int* cta_start = (int*)(hb + h_cta);
  int acc = 0;
  for (int i = 0; i < C; ++i) {
    cta_start[i] = acc;
    g_cta_cursor[i] = acc;
    acc += g_cta_count[i];
  }
  cta_start[C] = acc;
  mk::Task* tasks = (mk::Task*)(hb + h_tasks);
  Counts cnt2;
  emit(s, B, seq_lens, C, cnt2, [&](int cta, const mk::Task& t) { tasks[g_cta_cursor[cta]++] = t; });

  // one upload (the source may be reused as soon as the call returns), zeroed counters and status
  e = cudaMemcpyAsync(base + d_blob, hb, h_bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyAsync(task list)");
  e = cudaMemsetAsync(base + d_ctr, 0, (d_rope - d_ctr), st);
  if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(counters)");
  e = cudaMemsetAsync(base + d_route, 0, L * rm.ints * sizeof(int), st);
  if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(routing)");
  e = cudaMemsetAsync(base + d_rp, 0, L * mk::RL_COPIES * B * s.E * sizeof(unsigned long long), st);
  if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(router sums)");
  e = mk::launch_rope_table((float2*)(base + d_rope), npos, s.d, (double)dims->rope_theta, st);
  if (e != cudaSuccess) return fail_cuda(e, "RoPE table launch");

  mk::Params P;
  memset(&P, 0, sizeof(P));
  P.L = s.L; P.H = s.H; P.nq = s.nq; P.nkv = s.nkv; P.d = s.d; P.E = s.E; P.k = s.k; P.F = s.F; P.V = s.V;
  P.ps = s.ps; P.G = s.G; P.qkv_rows = s.qkv_rows; P.eps = dims->rms_eps;
  P.B = B; P.bcap = B; P.max_pages = max_pages_per_seq;
  const void* const* dtab = (const void* const*)(base + d_blob + h_tab);
  P.attn_norm = (const uint16_t* const*)(dtab + 0 * L);
  P.wqkv = (const uint16_t* const*)(dtab + 1 * L);
  P.wo = (const uint16_t* const*)(dtab + 2 * L);
  P.ffn_norm = (const uint16_t* const*)(dtab + 3 * L);
  P.router = (const uint16_t* const*)(dtab + 4 * L);
  P.w_gate_up = (const uint16_t* const*)(dtab + 5 * L);
  P.w_down = (const uint16_t* const*)(dtab + 6 * L);
  P.kv_pool = (uint16_t* const*)(dtab + 7 * L);
  P.embed = (const uint16_t*)w->embed;
  P.final_norm = (const uint16_t*)w->final_norm;
  P.lm_head = (const uint16_t*)w->lm_head;
  P.tasks = (const mk::Task*)(base + d_blob + h_tasks);
  P.cta_start = (const int*)(base + d_blob + h_cta);
  P.ctr = (uint32_t*)(base + d_ctr);
  P.status = (int*)(base + d_stat);
  P.epoch = 1;
  P.nsteps = 1;
  P.io_stride = B;
  P.top_p = 1.f;
  P.lg_keep = nullptr;
  P.sdone_cnt = 1;
  P.tm_gu = nullptr;     // the expert gate/up and the projections on CUDA cores here
  P.tm_qkv = P.tm_o = nullptr;
  P.qkv_fx = P.xmid_fx = nullptr;
  P.timeout_ns = 2000000000ull;
  P.strace = nullptr;
  P.cm = cm;
  P.rm = rm;
  P.nstages = sp.nstages;
  P.stage_bytes = sp.stage_bytes;
  P.act_off = sp.act_off;
  P.act_floats = sp.act_floats;
  P.misc_off = sp.misc_off;
  P.psum_off = sp.psum_off;
  P.attn_mrg_floats = sp.attn_mrg_floats;
  P.o_halves = sp.o_halves;
  P.down_rows_max = cnt.down_rows_max;
  P.cf_pairs = mk::cf_floats(s.E, s.k, s.F, C, B) / B > 0 ? mk::cf_floats(s.E, s.k, s.F, C, B) / B : 1;
  P.seq_len = (int*)(base + d_blob + h_seq);
  P.page_table = (const int*)(base + d_blob + h_pt);
  P.rope = (const float2*)(base + d_rope);
  P.rope_npos = npos;
  P.qkv = (float*)(base + d_qkv);
  P.part = (float*)(base + d_part);
  P.part_slots = cnt.slots;
  P.o = (float*)(base + d_o);
  P.x_mid = (float*)(base + d_xm);
  P.x_out = (float*)(base + d_xo);
  P.rlog = (float*)(base + d_rl);
  P.ids = (int*)(base + d_ids);
  P.gates = (float*)(base + d_gt);
  P.route = (int*)(base + d_route);
  P.moe_part = (float*)(base + d_mp);
  P.moe_mask = (uint32_t*)(base + d_mm);
  P.rlsum = (unsigned long long*)(base + d_rp);
  P.lm_val = (float*)(base + d_lmv);
  P.lm_idx = (int*)(base + d_lmi);
  P.lm_tiles = cnt.lm;
  P.tokens = d_tokens;
  P.logits = d_logits;
  P.next_token = d_next_token;
  e = mk::launch_megakernel(P, nb, C, smem, st);
  if (e != cudaSuccess) return fail_cuda(e, "megakernel launch");
  if (d_status) {
    e = cudaMemcpyAsync(d_status, base + d_stat, 4 * sizeof(int), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpyAsync(status)");
  }
  return MK_OK;
}
