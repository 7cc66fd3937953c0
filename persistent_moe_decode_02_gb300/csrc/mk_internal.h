// Internal layout shared by the host planner (plan.cu) and the megakernel
// (megakernel.cu): the task record, the counter map and the kernel parameters.
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace mk {

constexpr int NCW = 8;                     // consumer warps per CTA
constexpr int NTHREADS = (NCW + 1) * 32;   // + one producer warp
constexpr int MAX_STAGES = 16;             // smem ring stages (upper bound)
constexpr int MAX_TOPK = 8;
constexpr int MAX_G = 8;                   // query heads per KV head
constexpr int MAX_BATCH = 8;
constexpr int MAX_EXPERTS = 256;
constexpr int CTR_STRIDE = 8;              // uint32 slots per counter (32 B apart)
constexpr int SMEM_LIMIT = 232448;         // 227 KB opt-in per CTA
// rows per cross-warp partial-sum window of the wide GEMV: 64 at batch <= 2 (a
// projection tile's rows in one window: one flush), fewer for larger batches
// (shared memory)
constexpr int win_rows(int nb) { return nb <= 2 ? 64 : nb <= 4 ? 32 : 16; }
constexpr int RL_COPIES = 8;               // copies of the router-logit sums (O tile i adds to copy i % 8)
// The batch-8 instance uses only the first two: its expert tiles read every
// copy of 8 x E sums, and its O tiles are fewer (interleaved on one box:
// mid_b8 1.384 -> 1.378 ms with two copies, no change with four).
constexpr int RL_COPIES_B8 = 2;
constexpr int TRACE_SLOTS = 12;            // stamps per task in the optional timeline
constexpr int STRACE_CAP = 4096;           // ring stages per CTA in the optional stage timeline
constexpr int STRACE_SLOTS = 6;            // per stage: copy issued, landed, released, task,
                                           // and SM clock64 at landed and released
// timeline slots: consumer fetched / dependency met / activations ready /
// stages consumed / done; producer first copy / last copy / task start;
// consumer warp 0 saw its first / last stage of the task land
enum TraceSlot { TR_FETCH = 0, TR_DEP, TR_ACT, TR_STAGES, TR_DONE, TR_P_FIRST, TR_P_LAST, TR_P_START,
                 TR_S_FIRST, TR_S_LAST, TR_MID1, TR_MID2 };   // MID1/2: steps inside a task's activation part

// Task kinds in per-layer order.  Each kind signals one counter family.
enum TaskType : int32_t {
  T_QKV = 0,     // rows [a0,a1) of the grouped QKV matrix, all requests; a2 = KV group
  T_ATTN = 1,    // request a0, KV group a1, KV pages [a2, a3) (a3 < 0: to the current end);
                 // a4 = partial slot, a5 = first slot of (a0, a1), a6 = chunks of (a0, a1)
  T_OPROJ = 2,   // rows [a0,a1) of Wo, residual add, then the same hidden rows' share of
                 // the router logits (rows [a0,a1) of the transposed router, times the
                 // FFN norm's gain): partial a2 of the layer's router logits
  T_MOE = 3,     // expert tile a0 of a1 over the flattened (distinct expert, ffn unit) space:
                 // router logits from the O tiles' partials, routing (tile 0 publishes it),
                 // the tile's gate/up rows, then the same units' rows of the transposed
                 // down matrix, into a gated partial of the layer output
  T_RED = 4,     // rows [a0,a1) of the hidden dim: residual + the a2 expert tiles' partials
  T_LM = 5,      // rows [a0,a1) of the LM head; a2 = tile index, a3 = tiles (ticket target)
  T_COMB = 6,    // split-KV combine of query heads [a2, a2 + a3) of request a0, KV group a1:
                 // a5 = first partial slot, a6 = chunks (waits for all of them)
  T_SAMPLE = 7,  // nucleus (top-p) draw of request a0 from its logits, once every LM tile is done
};
constexpr int T_LAST = T_SAMPLE;

struct alignas(16) Task {
  int32_t type;
  int32_t layer;
  int32_t a[8];
  int32_t wait_ctr;    // counter index or -1
  uint32_t wait_cnt;   // signals per step that satisfy the wait
};
static_assert(sizeof(Task) == 48, "task record is 48 bytes");

// Counter map.  All counters only grow; a wait for `cnt` signals per step is
// satisfied when counter >= epoch * cnt (epoch = 1, 2, ... since the last reset).
struct CtrMap {
  int L, nkv, bcap;
  int qkv, attn, combine, o, rdone, gu, down, lm, sdone, omt, nomt, total;

  // omt_: 128-row tiles of the O projection that count their tensor-core tasks
  // (a ticket per tile: its last task converts the tile's x_mid rows)
  void init(int L_, int nkv_, int bcap_, int omt_ = 0) {
    L = L_; nkv = nkv_; bcap = bcap_; nomt = omt_;
    int c = 0;
    qkv = c; c += L * nkv;
    attn = c; c += L * bcap * nkv;
    combine = c; c += L;
    o = c; c += L;
    rdone = c; c += L;
    gu = c; c += L;
    down = c; c += L;
    lm = c; c += 1;
    sdone = c; c += 1;   // a step's next tokens are written (one signal per step)
    omt = c; c += L * omt_;
    total = c;
  }
#if defined(__CUDACC__)
  __host__ __device__
#endif
  int attn_idx(int l, int b, int g) const { return attn + (l * bcap + b) * nkv + g; }
};

// Per-layer routing record in global memory (ints):
//   [0] distinct experts U, then expert[umax], count[umax], tok[umax][bcap], rank[umax][bcap]
struct RouteMap {
  int umax, bcap, ints;
  void init(int umax_, int bcap_) { umax = umax_; bcap = bcap_; ints = 1 + 2 * umax + 2 * umax * bcap; }
};

struct Params {
  // shape
  int L, H, nq, nkv, d, E, k, F, V, ps, G;
  int qkv_rows;        // nkv * (G + 2) * d
  float eps;
  int B, bcap, max_pages;
  // weights (device arrays of L device pointers where per layer)
  const uint16_t* embed;
  const uint16_t* final_norm;
  const uint16_t* lm_head;
  const uint16_t* const* attn_norm;
  const uint16_t* const* wqkv;
  const uint16_t* const* wo;
  const uint16_t* const* ffn_norm;
  const uint16_t* const* router;
  const uint16_t* const* w_gate_up;
  const uint16_t* const* w_down;
  uint16_t* const* kv_pool;   // [num_pages][nkv][K, V][d][page_size] per layer
  // plan
  const Task* tasks;
  const int* cta_start;
  uint32_t* ctr;
  int* status;          // [0] code, [1] task, [2] cta, [3] info
  uint32_t epoch;        // epoch of the launch's first step; step s waits for epoch + s
  int nsteps;            // decode steps this launch runs (>= 1), each fed the previous one's tokens
  int io_stride;         // requests between two steps' rows of next_token (and logits): the group's batch
  unsigned long long timeout_ns;
  CtrMap cm;
  RouteMap rm;
  int nstages, stage_bytes;
  int act_off, act_floats, misc_off;
  int psum_off;          // smem offset of the GEMV partial-sum windows (2 * NCW * win_rows(nb) * nb floats)
  int attn_mrg_floats;   // attention page-group states in the activation region (floats)
  int down_rows_max;    // most rows of an H-row tile (O projection, reduce)
  int o_halves;         // 2: the O projection runs over two K halves (its input in shared memory
                        // half at a time, so larger batches keep a deep weight ring), else 1
  int cf_pairs;         // most (expert, unit) pairs of one expert tile
  int* seq_len;         // device [bcap]
  const int* page_table;  // device [bcap * max_pages]
  // prefill chunks: row b belongs to the chunk of one request that starts at
  // row chunk0[b] <= b (rows chunk0[b] .. b hold the request's consecutive
  // prompt positions seq_len[b] - (b - chunk0[b]) .. seq_len[b] and share its
  // page row); null: every row is a request of its own
  const int* chunk0;
  const float2* rope;   // [max_pos][d/2] (cos, sin)
  int rope_npos;
  // per-layer scratch (fp32 unless noted), all strided by bcap
  float* qkv;           // [L][bcap][qkv_rows]
  float* part;          // [L][part_slots][G][d + 2]
  int part_slots;
  float* o;             // [L][bcap][nq*d]
  float* x_mid;         // [L][bcap][H]
  float* x_out;         // [L][bcap][H]
  float* rlog;          // [L][bcap][E]
  int* ids;             // [L][bcap][k]
  float* gates;         // [L][bcap][k]
  int* route;           // [L][rm.ints]
  float* moe_part;      // [expert tiles][bcap][H] gated partial outputs (reused by every layer)
  unsigned long long* rlsum;   // [L][RL_COPIES][bcap][E] router-logit sums in 32.32 fixed point: the O tiles
                               // add their shares (integer adds: exact, any order), the expert
                               // tiles read them, the layer's reduce tasks zero them for the next
                               // step (and every replan zeroes all)
  float* lm_val;        // [bcap][lm_tiles]
  int* lm_idx;          // [bcap][lm_tiles]
  int lm_tiles;
  // optional per-task timeline: TRACE_SLOTS globaltimer stamps per task (nullable)
  unsigned long long* trace;
  // optional per-stage timeline: [cta][STRACE_CAP][STRACE_SLOTS] (nullable)
  unsigned long long* strace;
  // io: step 0 reads tokens[b]; step s >= 1 reads next_token[(s - 1) * io_stride + b];
  // step s writes next_token[s * io_stride + b] and, when logits is set,
  // logits[(s * io_stride + b) * V ...]
  const int* tokens;
  float* logits;        // nullable [nsteps][io_stride][V]
  int* next_token;      // [nsteps][io_stride]
  // temperature sampling (inv_temp = 1 / T; 0: greedy): the next token is the
  // argmax of logit * inv_temp + Gumbel noise drawn by Philox4x32-10 with key
  // (seed_lo, seed_hi) and counter (vocab row, position, slot0 + request, 0)
  float inv_temp;
  uint32_t seed_lo, seed_hi;
  int slot0;
  // nucleus sampling (top_p < 1 with inv_temp > 0): the LM tiles keep every
  // logit in lg_keep and the per-tile maximum logit in lm_val; T_SAMPLE task b
  // draws request b's token from the nucleus and signals sdone (sdone_cnt
  // signals per step: B with nucleus sampling, else 1, the LM finisher's)
  float top_p;
  float* lg_keep;       // [bcap][V] or null
  int sdone_cnt;
  // expert gate/up on the tensor cores (kernel instances of batch 4 and 8):
  // per layer a TMA tensor map (bf16 [E * 2F rows, H columns], 64 x 128 boxes,
  // 128-byte swizzle) of w_gate_up, in device memory; null: CUDA cores
  const void* tm_gu;
  // QKV and O projections on the tensor cores (batch instance 8, with tm_gu):
  // per layer a TMA tensor map of wqkv (bf16 [qkv_rows, H]) and of wo (bf16
  // [H, nq * d]), 64 x 128 boxes, 128-byte swizzle, in device memory.  A task
  // is one 128-row tile of the matrix over a run of its 128-column K stages;
  // the tiles of a row add their parts in 32.32 fixed point (integer adds:
  // exact, so the bits do not depend on the order), the readers convert.
  // null: CUDA cores, fp32 outputs in qkv and x_mid
  const void* tm_qkv;
  const void* tm_o;
  unsigned long long* qkv_fx;    // [L][bcap][qkv_rows]; zeroed after use by the layer's O tiles
  unsigned long long* xmid_fx;   // [L][bcap][H]; the last O task of each 128-row tile converts
                                 // its rows to fp32 x_mid and zeroes them
  // [L][expert tiles]: bit b set when the tile's partial holds request b's
  // row (instances above batch 1; the other rows of a partial are zero, so the
  // reduce tasks skip them)
  uint32_t* moe_mask;
};

// Expert gate/up on the tensor cores: an expert tile's range is a run of whole
// 32-unit halves (64 interleaved gate/up rows of one expert each).  Two halves
// make one 128-row tile, streamed as 128 rows x 64 columns per 16 KB of stage
// (one or two 64-column boxes, each two 64-row copies); a lone last half
// streams its 64 rows x 128 columns per 16 KB instead (two K boxes stacked).
constexpr int TC_HALF = 32;      // ffn units per half tile: the unit of the tiles' cut
constexpr int TC_BOX = 16384;    // bytes of one 128-row x 64-column box
inline bool tc_moe_shape(int H, int F) { return H % 256 == 0 && F % TC_HALF == 0; }
// The projections on the tensor cores: 128-row tiles that never straddle a KV
// group's rows, 128-column K stages, and an O tile's router rows ([128][E]
// bf16) in one stage.  TC_PROJ_UNITS bounds a task's K stages (their B operand
// slots, 4 KB each, share the activation region).
constexpr int TC_PROJ_UNITS = 16;
inline bool tc_proj_shape(int H, int nq, int d, int G, int E, int stage_bytes) {
  return H % 128 == 0 && (nq * d) % 128 == 0 && ((G + 2) * d) % 128 == 0 && E % 4 == 0 &&
         128 * E * 2 <= stage_bytes && stage_bytes == 2 * TC_BOX;
}

// Shared-memory layout of one CTA: [weight ring][activations][misc + down
// sums][GEMV partial-sum windows].  The ring takes what the rest leaves of the
// 227 KB, in 32 KB stages (16 KB when fewer than four would fit).  Returns
// false when the shape leaves no room (fewer than two stages, or an attention
// page split the warps cannot share evenly).
struct SmemPlan {
  int stage_bytes, nstages, act_floats, act_off, misc_off, psum_off, attn_mrg_floats, smem, o_halves;
};

// Per-expert-tile coefficients (gate x silu(gate row) x up row, per token slot)
// kept in shared memory between the tile's gate/up and down parts: at most
// CF_FLOATS, else what one tile per CTA needs at this capacity.
constexpr int CF_FLOATS = 3072;

inline int cf_floats(int E, int k, int F, int C, int bcap) {
  const long long umax = E < bcap * k ? E : (long long)bcap * k;
  const long long pairs = umax * F;
  const long long tiles = pairs < C ? (pairs > 0 ? pairs : 1) : C;
  const long long need = (pairs + tiles - 1) / tiles * bcap;
  return (int)(need < CF_FLOATS ? need : CF_FLOATS);
}

// Expert tiles per layer for umax distinct experts: one per CTA (at most one
// per (expert, unit) pair), but enough that each tile's pairs x capacity
// coefficients fit cf floats.
inline int moe_tiles(int umax, int F, int C, int bcap, int cf) {
  const long long pairs = (long long)umax * F;
  long long cap = cf / bcap;
  if (cap < 1) cap = 1;
  long long t = pairs < C ? pairs : C;
  if (t < 1) t = 1;
  const long long need = (pairs + cap - 1) / cap;
  return (int)(t > need ? t : need);
}

// The router stage of an O tile of nr hidden rows: the rows of the transposed
// router ([nr][E] bf16), then, 16-byte aligned, the 16-byte window of the FFN
// norm's gain that covers the nr entries (at most nr * 2 + 30 bytes).
#if defined(__CUDACC__)
__host__ __device__
#endif
inline int router_stage_gain_off(int nr, int E) { return (nr * E * 2 + 15) / 16 * 16; }
inline int router_stage_bytes(int nr, int E) { return router_stage_gain_off(nr, E) + (nr * 2 + 30 + 15) / 16 * 16; }

// Shared-memory layout: [weight ring][activations][misc struct + scratch][GEMV partial sums].
// The scratch holds an H-row tile's residual rows or an expert tile's coefficients.
inline bool plan_smem(int H, int nq, int d, int G, int E, int F, int ps, int bcap, int nb, int down_rows_max,
                      int cf, size_t misc_struct_bytes, SmemPlan& o) {
  const int nqd = nq * d;
  // above batch 2 the O projection's input (the widest) goes in two K halves
  o.o_halves = nb > 2 && nqd > H && (nqd / 2) % 2048 == 0 ? 2 : 1;
  const int kin = nqd / o.o_halves;
  const int widest = H > kin ? (H > F ? H : F) : (kin > F ? kin : F);
  const long long A1 = (long long)bcap * widest;
  const int RS = d + 4;
  int ppg32 = 32768 / (2 * ps * d * 2);
  if (ppg32 < 1) ppg32 = 1;
  const long long mrg = (long long)NCW * G * RS;   // one softmax state per consumer warp
  const long long A3 = (long long)MAX_G * d + 2 * d + mrg + NCW * 128;  // q (then its mma table), new K/V, states, P
  long long act = A1 > A3 ? A1 : A3;
  o.act_floats = (int)act;
  o.attn_mrg_floats = (int)mrg;
  const size_t act_bytes = ((size_t)act * 4 + 127) / 128 * 128;
  const long long scr = (long long)bcap * down_rows_max > cf ? (long long)bcap * down_rows_max : cf;
  const size_t misc = (misc_struct_bytes + (size_t)scr * 4 + 127) / 128 * 128;
  const size_t psum = ((size_t)2 * NCW * win_rows(nb) * nb * 4 + 127) / 128 * 128;
  const long long avail = (long long)SMEM_LIMIT - (long long)(act_bytes + misc + psum);
  const int need0 = 2 * widest > 4 * H ? 2 * widest : 4 * H;
  const int need = need0 > 2 * ps * d * 2 ? need0 : 2 * ps * d * 2;
  int sb = avail < 4LL * 32768 ? 16384 : 32768;
  while (sb < need) sb *= 2;
  long long nst = avail / sb;
  if (nst > MAX_STAGES) nst = MAX_STAGES;
  if (nst < 2) return false;
  const int ppg = sb / (2 * ps * d * 2) < 1 ? 1 : sb / (2 * ps * d * 2);
  if (ppg > ppg32 || NCW % ppg != 0 || d / 16 > 8) return false;
  if (H > 8 * NCW * 32 || H % 8 != 0) return false;   // the expert tile's down part: 8 columns per thread
  // an O tile's router rows and gain window share one stage; logits are summed four at a time
  if (E % 4 != 0 || router_stage_bytes(down_rows_max, E) > sb) return false;
  o.stage_bytes = sb;
  o.nstages = (int)nst;
  o.act_off = (int)(nst * sb);
  o.misc_off = (int)(nst * sb + act_bytes);
  o.psum_off = (int)(nst * sb + act_bytes + misc);
  o.smem = (int)(nst * sb + act_bytes + misc + psum);
  return true;
}

}  // namespace mk
