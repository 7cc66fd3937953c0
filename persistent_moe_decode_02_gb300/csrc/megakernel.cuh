// The persistent decode megakernel's device code, included by megakernel.cu
// (greedy and temperature-sampled steps) and megakernel_nuc.cu (the same
// kernel with the nucleus-draw tasks compiled in).
#pragma once
// Persistent MoE decode megakernel for GB300 (sm_103a).
//
// One CTA per SM stays resident for the whole decode step and walks its slice
// of a host-prepared task list ("Cohere Publishes One-Kernel Server for North
// Mini Code" — "One resident program, many small tasks"; "Inside the
// Megakernel Serving Engine for North Mini Code" — architecture paragraph).
//
// Inside a CTA:
//   * warp 8 (one lane) is the producer: it walks the CTA's tasks in order and
//     streams each task's weight rows (or cached KV pages) into a ring of
//     shared-memory stages with bulk async copies (cp.async.bulk, completion
//     on an mbarrier).  It never waits for a task's activations, so immutable
//     bytes land while the dependency is still pending ("What the scheduling
//     change is meant to avoid", third bullet).  Only expert tiles wait, for
//     the router's choice, since their addresses depend on it.
//   * warps 0-7 are consumers: per task they wait on a global-memory
//     dependency counter, load the small fp32 activation into shared memory,
//     consume the ring stages (bf16 x fp32 dot products on CUDA cores, or
//     online-softmax attention), write the outputs and bump the task's
//     counter.  A tile starts when its own inputs are ready, not when a whole
//     op is done ("False dependencies" bullet).
// Every spin-wait has a time limit; on expiry the kernel records
// MK_ERR_DEP_TIMEOUT in the status word, all CTAs drain and return.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "mk.h"
#include "mk_internal.h"

namespace mk {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int NCT = NCW * 32;  // consumer threads
// Column-slice GEMV: consume two ring stages per pass, per call site.  It pays
// off in the LM head's long tiles; in the short projection and expert tiles
// waiting for the second stage before any math costs more than it saves.
constexpr bool SP_PROJ = false, SP_MOE = false, SP_LM = true;

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Announce bytes of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx_only(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// n arrivals at once (one warp standing in for n).
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

// Flag handoff between this CTA's consumers and its producer thread.
__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}

// Non-blocking probe: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Global -> shared bulk copy; completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// ---- tensor-core (tcgen05) helpers: 2-D TMA tile loads, shared-memory
// matrix descriptors, TMEM allocation, MMA issue / commit and TMEM loads.

// 2-D tiled bulk tensor copy global -> shared, completion on `bar` in bytes.
// x (the inner, K coordinate) is always a multiple of 64 bf16 (128 bytes).
__device__ __forceinline__ void tma_g2s_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout (8-row groups of 128-byte rows, 1024 bytes apart).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;                  // leading-dimension offset (not used by swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride between 8-row groups
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptors, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = 16 or 32.
constexpr uint32_t UMMA_IDESC_M128_N16 = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t)(16 >> 3) << 17 |
                                         (uint32_t)(128 >> 4) << 24;
constexpr uint32_t UMMA_IDESC_M128_N32 = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t)(32 >> 3) << 17 |
                                         (uint32_t)(128 >> 4) << 24;

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued is complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes
// 32 (w % 4) .. + 31).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Release-ordered add without a returned value: the signalling thread does
// not wait for the atomic's round trip.
__device__ __forceinline__ void red_add_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Explicit shared-memory loads (32-bit shared addresses), so the hot loops
// never go through generic addressing.  Volatile keeps them behind the
// mbarrier waits that publish the data.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
// Tensor-core helpers: 8x8 b16 matrix loads from shared memory and the
// m16n8k16 bf16 MMA with fp32 accumulation (d += a . b).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Task records are read-only during a step: read them through the L1.
__device__ __forceinline__ Task ldg_task(const Task* t) {
  const int4* q = reinterpret_cast<const int4*>(t);
  const int4 a = __ldg(q), b = __ldg(q + 1), c = __ldg(q + 2);
  Task r;
  r.type = a.x; r.layer = a.y; r.a[0] = a.z; r.a[1] = a.w;
  r.a[2] = b.x; r.a[3] = b.y; r.a[4] = b.z; r.a[5] = b.w;
  r.a[6] = c.x; r.a[7] = c.y; r.wait_ctr = c.z; r.wait_cnt = (uint32_t)c.w;
  return r;
}


__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// 32.32 fixed point for the sums that tiles add in any order (router
// logits; on the tensor-core path the projections' outputs): two's
// complement in 64 bits.  Both forms give the same values: v * 2^32 is exact
// (a power-of-two scale), then one rounding to the nearest integer; back, one
// rounding of the integer to fp32 after an exact scale (|q| < 2^53).  FAST
// (the batch-8 instance, whose expert tiles convert 16K values each) keeps
// to fp32 scaling and 64-bit integer conversions: this part runs fp64 at a
// small fraction of its fp32 rate.  The other instances convert a few
// hundred values on the routing's critical path and keep the fp64 form.
template <bool FAST>
__device__ __forceinline__ unsigned long long to_fixed(float v) {
  if constexpr (FAST) return (unsigned long long)__float2ll_rn(v * 4294967296.0f);
  return (unsigned long long)__double2ll_rn((double)v * 4294967296.0);
}
template <bool FAST>
__device__ __forceinline__ float from_fixed(unsigned long long q) {
  if constexpr (FAST) return __ll2float_rn((long long)q) * 2.3283064365386963e-10f;
  return (float)((double)(long long)q * 2.3283064365386963e-10);
}

// Word 0 of Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC 2011): ten rounds of two 32x32 -> 64-bit
// products, the key advanced by the Weyl constants before every round but
// the first.
__device__ __forceinline__ uint32_t philox_w0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                              uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

// Standard Gumbel noise -log(-log(u)) for vocabulary row `row` of the request
// in batch slot `slot` at position `pos`, u = ((x >> 9) + 1/2) * 2^-23 in
// (0, 1) (exact in float32).  Kept out of line: only sampled steps call it.
__device__ __noinline__ float gumbel_noise(uint32_t row, uint32_t pos, uint32_t slot, uint32_t k0, uint32_t k1) {
  const uint32_t x = philox_w0(row, pos, slot, 0u, k0, k1);
  const float u = ((float)(x >> 9) + 0.5f) * 1.1920928955078125e-07f;
  return -logf(-logf(u));
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Barrier over the 256 consumer threads (named barrier 1).
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Same barrier, returning the OR of every consumer thread's predicate.
__device__ __forceinline__ bool cbar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 256, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// Sum of v[h] over the 32 lanes for the head h = (lane >> 2) & 7, by halving
// exchanges (9 shuffles for 8 values instead of 40).
__device__ __forceinline__ float reduce8(const float (&v)[8], int lane) {
  float a[4];
  const bool u16 = lane & 16;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float send = u16 ? v[i] : v[i + 4];
    float keep = u16 ? v[i + 4] : v[i];
    a[i] = keep + __shfl_xor_sync(FULL, send, 16);
  }
  float b[2];
  const bool u8 = lane & 8;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    float send = u8 ? a[i] : a[i + 2];
    float keep = u8 ? a[i + 2] : a[i];
    b[i] = keep + __shfl_xor_sync(FULL, send, 8);
  }
  const bool u4 = lane & 4;
  float c = (u4 ? b[1] : b[0]) + __shfl_xor_sync(FULL, u4 ? b[0] : b[1], 4);
  c += __shfl_xor_sync(FULL, c, 2);
  c += __shfl_xor_sync(FULL, c, 1);
  return c;
}

// Same for 4 values: lane l returns the 32-lane sum of v[(l >> 3) & 3].
__device__ __forceinline__ float reduce4(const float (&v)[4], int lane) {
  float a[2];
  const bool u16 = lane & 16;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = u16 ? v[i] : v[i + 2];
    const float keep = u16 ? v[i + 2] : v[i];
    a[i] = keep + __shfl_xor_sync(FULL, send, 16);
  }
  const bool u8 = lane & 8;
  float c = (u8 ? a[1] : a[0]) + __shfl_xor_sync(FULL, u8 ? a[0] : a[1], 8);
  c += __shfl_xor_sync(FULL, c, 4);
  c += __shfl_xor_sync(FULL, c, 2);
  c += __shfl_xor_sync(FULL, c, 1);
  return c;
}

// ------------------------------------------------------------------ shared state

constexpr int MAX_UNION = MAX_BATCH * MAX_TOPK;   // distinct experts a step can select

// A layer's distinct experts as the producer sees them.
struct RouteCache {
  int layer, U;
  int exp[MAX_UNION];
};

struct Misc {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  int armed[MAX_STAGES];   // round in which the producer last armed a stage, -1 never
  int dead;                // the status word was already set at kernel entry
  int abort_flag;          // a warp of this CTA gave up
  int ticket_last;
  int pad;
  float red[NCW * MAX_BATCH];
  float inv[MAX_BATCH];    // 1 / rms of each activation row of the last norm (its GEMV epilogue scales by it)
  float best_v[NCW * MAX_BATCH];
  int best_i[NCW * MAX_BATCH];
  int sel[MAX_BATCH * MAX_TOPK];
  float selv[MAX_BATCH * MAX_TOPK];
  float gate[MAX_BATCH * MAX_TOPK];
  float rl[MAX_BATCH * MAX_EXPERTS];   // router logits of the layer being routed
  int slot_of[MAX_EXPERTS];
  int cnt_of[MAX_EXPERTS];
  int r_U;                 // distinct experts of the routing in r_exp...
  int r_layer;             // layer whose routing r_exp... holds after a gate/up task computed it (-1: none)
  // routing of the current layer, cached per task
  int r_exp[MAX_UNION];
  int r_cnt[MAX_UNION];
  int r_tok[MAX_UNION * MAX_BATCH];
  int r_rank[MAX_UNION * MAX_BATCH];
  // the producer's copies of a layer's distinct experts, one per cursor
  RouteCache cp_route;
  // tensor-core gate/up: accumulator-ready barrier (one commit per 128-row
  // tile or lone half), final-completion barrier, and the TMEM base address
  uint64_t acc_bar;
  uint64_t tc_fin;
  uint32_t tmem;
  // nucleus draw (T_SAMPLE): target and running mass, key prefix, digit, cut, max logit
  unsigned long long smp_tgt, smp_before;
  uint32_t smp_prefix;
  int smp_digit, smp_cut;
  float smp_max;
};

struct Ring {
  uint8_t* base;
  Misc* m;
  int nst, sb;
  int stage, round;
  __device__ void advance() {
    if (++stage == nst) { stage = 0; ++round; }
  }
};

// ------------------------------------------------------------------ failure handling

__device__ __forceinline__ bool failed(const Params& p) {
  return *(volatile int*)p.status != 0;
}

__device__ void set_error(const Params& p, int code, int task, int info) {
  if (atomicCAS(p.status, 0, code) == 0) {
    p.status[1] = task;
    p.status[2] = blockIdx.x;
    p.status[3] = info;
    __threadfence();
  }
}

// Wait until counter `ctr` holds epoch * cnt signals (bounded).
__device__ bool wait_ctr(const Params& p, int ctr, uint32_t epoch, uint32_t cnt, int task) {
  if (ctr < 0) return true;
  const uint32_t* c = p.ctr + (size_t)ctr * CTR_STRIDE;
  const uint32_t target = epoch * cnt;
  if ((int32_t)(ld_acquire(c) - target) >= 0) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    if ((int32_t)(ld_acquire(c) - target) >= 0) return true;
    if ((it & 31) == 0) {
      if (failed(p)) return false;
      if (gtimer() - t0 > p.timeout_ns) {
        set_error(p, MK_ERR_DEP_TIMEOUT, task, ctr);
        return false;
      }
    }
    if (it > 256) __nanosleep(100);
  }
}

// Bounded mbarrier parity wait; gives up when this CTA or any CTA failed.
__device__ bool mbar_wait(const Params& p, Misc* m, uint64_t* bar, uint32_t parity, int info) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15) == 0) {
      if (*(volatile int*)&m->abort_flag || failed(p)) return false;
      if (gtimer() - t0 > p.timeout_ns) {
        set_error(p, MK_ERR_DEP_TIMEOUT, -1, info);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ stage geometry
// Producer and consumers derive the same stage sequence from the task and the
// same device state, so they agree on what every stage holds.

__device__ __forceinline__ int rows_per_stage(const Params& p, int K) {
  return max(1, p.stage_bytes / (K * 2));
}

__device__ __forceinline__ int pages_per_stage(const Params& p) {
  return max(1, p.stage_bytes / (2 * p.ps * p.d * 2));
}

__device__ __forceinline__ int pairs_per_stage(const Params& p) {
  return max(1, p.stage_bytes / (4 * p.H));
}

// Token range [tok0, tok1) of an attention task at the current lengths.
__device__ __forceinline__ void attn_range(const Params& p, const Task& t, int pos, int& tok0,
                                           int& tok1) {
  tok0 = t.a[2] * p.ps;
  tok1 = (t.a[3] < 0) ? pos + 1 : min(t.a[3] * p.ps, pos + 1);
}

// Flattened (distinct expert, ffn row) range of gate/up tile a0 of a1.
__device__ __forceinline__ void gu_range(const Params& p, const Task& t, int U, long long& q0,
                                         long long& q1) {
  const unsigned tot = (unsigned)U * (unsigned)p.F, i = (unsigned)t.a[0], n = (unsigned)t.a[1];
  if ((unsigned long long)tot * n < (1ull << 32)) {   // 32-bit division: the common case
    q0 = tot * i / n;
    q1 = tot * (i + 1) / n;
  } else {
    q0 = (long long)tot * i / n;
    q1 = (long long)tot * (i + 1) / n;
  }
}

// Above batch 1 the distinct experts serve different numbers of token slots,
// and a unit's work grows with them: the ranges are cut by cost instead, a
// unit of expert u costing GU_UNIT_COST + cnt[u] (its weight rows, then one per
// slot).  When the cut could give some tile more units than its coefficient
// scratch holds (cf_pairs), the plain even cut is kept.  Producer and
// consumers call this with the same routing, so they agree.
constexpr long long GU_UNIT_COST = 1;

__device__ __forceinline__ long long gu_cut(int U, int F, const int* cnt, long long T) {
  long long acc = 0;
  for (int u = 0; u < U; ++u) {
    const long long w = GU_UNIT_COST + cnt[u], span = (long long)F * w;
    if (T <= acc + span) return (long long)u * F + min((long long)F, (T - acc + w - 1) / w);
    acc += span;
  }
  return (long long)U * F;
}

// Whether expert tile t's gate/up runs on the tensor cores: the batch-8
// instance with tensor maps, when the layer's 32-unit halves, cut evenly
// over the tiles, fit the coefficient scratch (the producer and the
// consumers decide alike from the same routing).
__device__ __forceinline__ bool tc_layer(const Params& p, const Task& t, int U) {
  if (!p.tm_gu) return false;
  const long long T = (long long)U * p.F / TC_HALF, n = t.a[1];
  return (T + n - 1) / n * TC_HALF <= p.cf_pairs;
}

// Ring stages of a tensor-core gate/up range of nh halves: kst per pair of
// halves (128-row tiles, 128 columns a stage), kst / 2 for a lone last half
// (64 rows, 256 columns a stage).
__device__ __forceinline__ int tc_gu_stages(const Params& p, int nh) {
  const int kst = p.H / (64 * (p.stage_bytes / TC_BOX));
  return (nh >> 1) * kst + (nh & 1) * (kst >> 1);
}

template <int NB>
__device__ __forceinline__ void gu_range_w(const Params& p, const Task& t, int U, const int* cnt, long long& q0,
                                           long long& q1) {
  if constexpr (NB == 8) {
    if (tc_layer(p, t, U)) {   // tensor-core gate/up: whole 32-unit halves, evenly
      const long long T = (long long)U * p.F / TC_HALF, i = t.a[0], n = t.a[1];
      q0 = T * i / n * TC_HALF;
      q1 = T * (i + 1) / n * TC_HALF;
      return;
    }
  }
  if constexpr (NB > 1) {
    long long tot = 0;
    int cmin = 1 << 30;
    for (int u = 0; u < U; ++u) {
      tot += GU_UNIT_COST + cnt[u];
      cmin = min(cmin, cnt[u]);
    }
    tot *= p.F;
    const long long n = t.a[1], i = t.a[0];
    if (U > 0 && tot / (n * (GU_UNIT_COST + cmin)) + 2 <= p.cf_pairs) {
      q0 = gu_cut(U, p.F, cnt, tot * i / n);
      q1 = gu_cut(U, p.F, cnt, tot * (i + 1) / n);
      return;
    }
  }
  gu_range(p, t, U, q0, q1);
}

__device__ __forceinline__ const int* route_of(const Params& p, int l) {
  return p.route + (size_t)l * p.rm.ints;
}

// ------------------------------------------------------------------ producer

// The producer's view of one task: how many ring stages it fills and where
// each stage's bytes come from.  The consumer walks the same geometry.
struct Geo {
  int type, nst, l;
  // row tasks
  const uint16_t* W;
  const uint16_t* W2;   // expert tile: the layer's down matrix (W: its gate/up matrix)
  int K, r0, r1, rps, halves;
  // attention
  int pg0, pg1, ppg, b, g;
  uint32_t PB;
  // expert tile: the routing cache it reads, its flattened (distinct expert,
  // ffn unit) range, gate/up stages first (pps units each), then down stages
  // (rpw units each, rows of the transposed down matrix)
  const RouteCache* rc;
  int q0, q1;
  int pps, rpw, nst_gu;
  int cs, cu, cf;   // gate/up cursor: stage cs starts at unit cf of distinct expert cu
  int ws, wu, wf;   // down cursor, the same for down stage ws
  bool tc;          // gate/up stages are tensor-core tiles (128 rows x 64 columns per 16 KB)
  int nh, tmt, tks, ty0, ty1;   // tensor-core cursor: halves, tile, its K stage, its halves' first rows
  // projection on the tensor cores: rows [r0, r0 + 128), nw stages of 128
  // columns from K stage ks0 (then, for O, the router stage)
  bool tcp;
  int ks0, nw;
};

// Producer: one thread that walks the CTA's tasks and fills the ring with
// bulk copies, paced by the consumers' releases: a task's weights are in
// flight as soon as ring slots free up, long before its activations exist.
// Kept small: the SM's instruction cache is shared with the consumer warps.
template <int NB>
struct Producer {
  static constexpr bool kSplit = NB > 2;   // the O projection may run in K halves only above batch 2
  const Params& p;
  Ring r;
  uint64_t pol;
  int ti = 0;
  int step = 0;           // step of this launch being walked (0 .. nsteps - 1)
  long long cp_lin = 0;   // ring stages filled so far (stage timeline index)

  __device__ void mark(int k) {
    if (p.trace) p.trace[(size_t)ti * TRACE_SLOTS + k] = gtimer();
  }

  // Routing of layer l into cache c (once per layer and step): this CTA's
  // expert tile computes it and hands it over in shared memory (bounded
  // wait), tagged with the layer's index counted over the launch's steps.
  __device__ bool route_ready(RouteCache* c, int l0, int task) {
    const int l = step * p.L + l0;
    if (c->layer == l) return true;
    Misc* m = r.m;
    if (ld_acquire_cta(&m->r_layer) != l) {
      // poll with plain loads (no fence, no sleep: the table is a few hundred
      // cycles away and the first copies wait on it), acquire once seen
      const uint64_t t0 = gtimer();
      for (uint32_t it = 1; *(volatile int*)&m->r_layer != l; ++it) {
        if ((it & 63) == 0) {
          if (*(volatile int*)&m->abort_flag || failed(p)) return false;
          if (gtimer() - t0 > p.timeout_ns) {
            set_error(p, MK_ERR_DEP_TIMEOUT, task, -5);
            return false;
          }
        }
      }
      if (ld_acquire_cta(&m->r_layer) != l) return false;
    }
    const int U = m->r_U;
    for (int u0 = 0; u0 < U; u0 += 8) {   // eight loads in flight
      int e[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) e[i] = u0 + i < U ? m->r_exp[u0 + i] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (u0 + i < U) c->exp[u0 + i] = e[i];
    }
    c->U = U;
    c->layer = l;
    return true;
  }

  // Stage layout of expert tile t for U distinct experts: its flattened (distinct
  // expert, ffn unit) range, gate/up stages of pps units, then down stages of
  // rpw units, each within one expert; both cursors at their first stage.
  __device__ void moe_layout(const Task& t, Geo& q, int U, const int* cnt) {
    long long g0, g1;
    gu_range_w<NB>(p, t, U, cnt, g0, g1);
    q.q0 = (int)g0;
    q.q1 = (int)g1;
    q.pps = pairs_per_stage(p);
    q.rpw = rows_per_stage(p, p.H);
    const int F = p.F;
    int ngu = 0, nwd = 0;
    for (int u = q.q0 / F; u * F < q.q1; ++u) {
      const int fa = max(q.q0 - u * F, 0), fb = min(F, q.q1 - u * F);
      ngu += (fb - fa + q.pps - 1) / q.pps;
      nwd += (fb - fa + q.rpw - 1) / q.rpw;
    }
    q.tc = NB == 8 && tc_layer(p, t, U);
    if (q.tc) {
      q.nh = (q.q1 - q.q0) / TC_HALF;
      ngu = tc_gu_stages(p, q.nh);
      if (q.nh > 0) tc_tile(q, 0);
    }
    q.nst_gu = ngu;
    q.nst = ngu + nwd;
    q.cs = q.ws = 0;
    q.cu = q.wu = q.q0 / F;
    q.cf = q.wf = q.q0 - q.cu * F;
  }

  // The tensor-core cursor at tile mt of expert range q: K stage 0 and the
  // first gate/up row of each of its halves (a lone last half: both its own).
  __device__ void tc_tile(Geo& q, int mt) const {
    q.tmt = mt;
    q.tks = 0;
    const int F = p.F;
    const int a0 = q.q0 + 2 * mt * TC_HALF, u0 = a0 / F;
    q.ty0 = q.rc->exp[u0] * 2 * F + 2 * (a0 - u0 * F);
    const int a1 = a0 + (2 * mt + 1 < q.nh ? TC_HALF : 0), u1 = a1 / F;
    q.ty1 = q.rc->exp[u1] * 2 * F + 2 * (a1 - u1 * F);
  }

  // Geometry of task t; false on a routing wait that timed out or gave up,
  // or for an unknown task type.
  __device__ bool geo(const Task& t, Geo& q, RouteCache* c, int task) {
    q.type = t.type;
    q.l = t.layer;
    q.tcp = false;
    const int l = t.layer;
    switch (t.type) {
      case T_QKV: case T_OPROJ: case T_LM: {
        if constexpr (NB == 8) {
          if (p.tm_qkv && t.type != T_LM) {
            q.tcp = true;
            q.r0 = t.a[0];
            q.r1 = t.a[1];
            q.ks0 = t.a[3];
            q.nw = t.a[4] - t.a[3];
            q.nst = q.nw + (t.type == T_OPROJ ? 1 : 0);   // + the router stage
            return true;
          }
        }
        q.W = t.type == T_QKV ? p.wqkv[l] : t.type == T_OPROJ ? p.wo[l] : p.lm_head;
        // the O projection's K halves (o_halves = 2) stream one after the other
        q.halves = kSplit && t.type == T_OPROJ ? p.o_halves : 1;
        q.K = t.type == T_OPROJ ? p.nq * p.d / q.halves : p.H;
        q.r0 = t.a[0];
        q.r1 = t.a[1];
        q.rps = rows_per_stage(p, q.K);
        q.nst = q.halves * ((q.r1 - q.r0 + q.rps - 1) / q.rps) + (t.type == T_OPROJ ? 1 : 0);   // + the router stage
        return true;
      }
      case T_ATTN: {
        q.b = t.a[0];
        q.g = t.a[1];
        const int pos = __ldcg(p.seq_len + q.b) + step;
        int tok0, tok1;
        attn_range(p, t, pos, tok0, tok1);
        q.ppg = pages_per_stage(p);
        q.PB = (uint32_t)p.ps * p.d * 2;
        q.pg0 = tok0 / p.ps;
        q.pg1 = (tok1 + p.ps - 1) / p.ps;
        q.nst = (q.pg1 - q.pg0 + q.ppg - 1) / q.ppg;
        return true;
      }
      case T_MOE: {
        // Everything but the expert ids depends on the routing only through U,
        // the number of distinct experts: lay out the stages for the largest U
        // the batch can have (always the U of one request) and load the layer's
        // expert matrices before the wait; redo the layout if U differs.
        q.W = p.w_gate_up[l];
        q.W2 = p.w_down[l];
        asm volatile("" ::"l"(q.W), "l"(q.W2));
        const int Ug = min(p.E, p.B * p.k);
        if constexpr (NB == 1) moe_layout(t, q, Ug, nullptr);
        if (!route_ready(c, l, task)) return false;
        q.rc = c;
        if constexpr (NB == 1) {
          if (c->U != Ug) moe_layout(t, q, c->U, nullptr);
        } else {
          // the cut depends on the token counts: the consumers' table (r_cnt)
          // holds this layer's until this CTA's next expert task routes
          moe_layout(t, q, c->U, r.m->r_cnt);
        }
        return true;
      }
      case T_RED:      // no weights: reads only the expert tiles' partials
      case T_SAMPLE:   // no weights: reads the kept logits
      case T_COMB: {   // no weights: reads only partials
        q.nst = 0;
        return true;
      }
      default: return false;
    }
  }

  // Calls f(src, bytes, dst_offset) for each contiguous piece of stage s.
  // Gate/up stages are walked with a cursor kept in the geometry, so stages
  // visited in order cost O(1) each.
  template <class F>
  __device__ void segs(Geo& q, int s, F f) {
    const int l = q.l;
    switch (q.type) {
      case T_QKV: case T_OPROJ: case T_LM: {
        if (q.type == T_OPROJ && s == q.nst - 1) {
          // the O tile's router stage: rows [r0, r1) of the transposed router,
          // then the 16-byte window of the FFN norm's gain around the same rows
          const int nr = q.r1 - q.r0;
          f(p.router[l] + (size_t)q.r0 * p.E, (uint32_t)nr * p.E * 2, 0u);
          const uint32_t w0 = (uint32_t)q.r0 * 2 / 16 * 16, w1 = ((uint32_t)q.r1 * 2 + 15) / 16 * 16;
          f(reinterpret_cast<const uint8_t*>(p.ffn_norm[l]) + w0, w1 - w0, (uint32_t)router_stage_gain_off(nr, p.E));
          break;
        }
        if (!kSplit || q.halves == 1) {
          const int s0 = q.r0 + s * q.rps;
          const int n = min(q.rps, q.r1 - s0);
          f(q.W + (size_t)s0 * q.K, (uint32_t)n * q.K * 2, 0u);
        } else {   // K half h of rows s0 .. s0 + n: one copy per row
          const int per = (q.r1 - q.r0 + q.rps - 1) / q.rps, h = s / per;
          const int s0 = q.r0 + (s - h * per) * q.rps;
          const int n = min(q.rps, q.r1 - s0);
          for (int i = 0; i < n; ++i)
            f(q.W + (size_t)(s0 + i) * q.K * q.halves + (size_t)h * q.K, (uint32_t)q.K * 2, (uint32_t)i * q.K * 2);
        }
        break;
      }
      case T_ATTN: {
        const int pg = q.pg0 + s * q.ppg;
        const int n = min(q.ppg, q.pg1 - pg);
        const int* pt = p.page_table + (size_t)q.b * p.max_pages;
#pragma unroll 1   // kept rolled: the producer's code shares the SM's instruction cache
        for (int i = 0; i < n; ++i) {   // one copy per page: its K block, then its V block
          const size_t off = ((size_t)pt[pg + i] * p.nkv + q.g) * 2 * p.ps * p.d;
          f(p.kv_pool[l] + off, 2 * q.PB, (uint32_t)i * 2 * q.PB);
        }
        break;
      }
      case T_MOE: {
        const int F = p.F, H = p.H;
        if (s < q.nst_gu) {
          if (s < q.cs) {   // rewind
            q.cs = 0;
            q.cu = q.q0 / F;
            q.cf = q.q0 - q.cu * F;
          }
          while (q.cs < s) {   // advance one stage: pps units, or to the end of this expert's range
            const int fb = min(F, q.q1 - q.cu * F);
            q.cf += q.pps;
            if (q.cf >= fb) {
              ++q.cu;
              q.cf = 0;
            }
            ++q.cs;
          }
          const int fb = min(F, q.q1 - q.cu * F);
          const int n = min(q.pps, fb - q.cf);
          const uint16_t* We = q.W + (size_t)q.rc->exp[q.cu] * 2 * F * H;   // rows 2f, 2f+1
          f(We + (size_t)2 * q.cf * H, (uint32_t)n * 2 * H * 2, 0u);
        } else {
          const int s2 = s - q.nst_gu;
          if (s2 < q.ws) {
            q.ws = 0;
            q.wu = q.q0 / F;
            q.wf = q.q0 - q.wu * F;
          }
          while (q.ws < s2) {
            const int fb = min(F, q.q1 - q.wu * F);
            q.wf += q.rpw;
            if (q.wf >= fb) {
              ++q.wu;
              q.wf = 0;
            }
            ++q.ws;
          }
          const int fb = min(F, q.q1 - q.wu * F);
          const int n = min(q.rpw, fb - q.wf);
          const uint16_t* Wd = q.W2 + ((size_t)q.rc->exp[q.wu] * F + q.wf) * H;   // [E][F][H]
          f(Wd, (uint32_t)n * H * 2, 0u);
        }
        break;
      }
    }
  }

  // Before a later step's first KV page copy: the previous step's K/V appends
  // must be visible to the bulk-copy engine.  Wait (bounded) for that step's
  // done counter, then order the async proxy after it.
  __device__ bool kv_ready(int task) {
    if (!wait_ctr(p, p.cm.sdone, p.epoch + (uint32_t)step - 1u, (uint32_t)p.sdone_cnt, task)) return false;
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
  }

  __device__ void run(int t0, int t1) {
    Misc* m = r.m;
    m->cp_route.layer = -1;
    for (step = 0; step < p.nsteps; ++step) {
      bool kv_seen = step == 0;
      for (ti = t0; ti < t1; ++ti) {
        if (!run_task(ti, kv_seen)) return;
      }
    }
  }

  __device__ bool run_task(int ti_, bool& kv_seen) {
    Misc* m = r.m;
    ti = ti_;
    {
      if (failed(p)) return false;
      const Task t = ldg_task(p.tasks + ti);
      mark(TR_P_START);
      Geo q;
      if (!geo(t, q, &m->cp_route, ti)) {
        if (t.type < T_QKV || t.type > T_LAST) set_error(p, MK_ERR_INVALID, ti, t.type);
        m->abort_flag = 1;
        return false;
      }
      if (t.type == T_ATTN && q.nst > 0 && !kv_seen) {
        if (!kv_ready(ti)) {
          m->abort_flag = 1;
          return false;
        }
        kv_seen = true;
      }
      for (int s = 0; s < q.nst; ++s) {
        // claim the slot once the consumers released it, then for each piece
        // announce its bytes before the copy; the closing arrival completes
        // the phase when the last byte lands
        const uint32_t par = (r.round & 1) ^ 1;
        if (!mbar_wait(p, m, &m->empty[r.stage], par, -3)) {
          m->abort_flag = 1;
          return false;
        }
        if (s == 0) mark(TR_P_FIRST);
        uint64_t* bar = &m->full[r.stage];
        uint8_t* dst = r.base + (size_t)r.stage * r.sb;
        m->armed[r.stage] = r.round;
        if (NB == 8 && q.type == T_MOE && q.tc && s < q.nst_gu) {
          // tensor-core gate/up: per 16 KB box of the stage, two 64-row copies
          // (64 interleaved gate/up rows, 32 units of one expert, by 64
          // columns).  A pair of halves: each half's rows at K box ks * nbox + h.
          // A lone last half: its rows at K boxes 2 (ks * nbox + h) and the next.
          const int nbox = p.stage_bytes / TC_BOX, kst = p.H / (64 * nbox);
          const bool lone = 2 * q.tmt + 1 == q.nh;
          const void* tm = reinterpret_cast<const uint8_t*>(p.tm_gu) + (size_t)q.l * 128;
          mbar_expect_tx_only(bar, (uint32_t)nbox * TC_BOX);
          for (int h = 0; h < nbox; ++h) {
            const int x = lone ? 2 * (q.tks * nbox + h) : q.tks * nbox + h;
            tma_g2s_2d(dst + h * TC_BOX, tm, x * 64, q.ty0, bar, pol);
            tma_g2s_2d(dst + h * TC_BOX + TC_BOX / 2, tm, (x + (lone ? 1 : 0)) * 64, q.ty1, bar, pol);
          }
          if (++q.tks == (lone ? kst >> 1 : kst) && 2 * (q.tmt + 1) < q.nh) tc_tile(q, q.tmt + 1);
        } else if (NB == 8 && q.tcp) {
          if (s < q.nw) {
            // projection tile: 128 rows x 128 columns (two 64-column boxes) of K stage ks0 + s
            const void* tm = reinterpret_cast<const uint8_t*>(q.type == T_QKV ? p.tm_qkv : p.tm_o) + (size_t)q.l * 128;
            mbar_expect_tx_only(bar, 2u * TC_BOX);
            for (int h = 0; h < 2; ++h) tma_g2s_2d(dst + h * TC_BOX, tm, (q.ks0 + s) * 128 + h * 64, q.r0, bar, pol);
          } else {
            // the O tile's router stage: its 128 rows of the transposed router
            const uint32_t nb = 128u * p.E * 2;
            mbar_expect_tx_only(bar, nb);
            bulk_g2s(dst, p.router[q.l] + (size_t)q.r0 * p.E, nb, bar, pol);
          }
        } else {
          // an attention stage's bytes are announced once, not per page
          const bool one_tx = q.type == T_ATTN;
          if (one_tx) mbar_expect_tx_only(bar, (uint32_t)min(q.ppg, q.pg1 - q.pg0 - s * q.ppg) * 2u * q.PB);
          segs(q, s, [&](const void* src, uint32_t b, uint32_t off) {
            if (!one_tx) mbar_expect_tx_only(bar, b);
            bulk_g2s(dst + off, src, b, bar, pol);
          });
        }
        mbar_arrive(bar);
        if (p.strace && cp_lin < STRACE_CAP) {
          unsigned long long* rec = p.strace + ((size_t)blockIdx.x * STRACE_CAP + cp_lin) * STRACE_SLOTS;
          rec[0] = gtimer();
          rec[3] = (unsigned long long)ti;
        }
        r.advance();
        ++cp_lin;
      }
      mark(TR_P_LAST);
    }
    return true;
  }
};

// ------------------------------------------------------------------ consumer pieces

// GEMV epilogue shared by the projection and expert tasks, so that one GEMV
// body (inlined at one call site per row kind) serves all of them.  inv holds
// the RMS-norm scale of each activation row (the GEMV ran on x * gain):
//   STORE:  out[j * ld + row] = inv[j] * s
//   RESID:  out[j * ld + row] = res[j * res_ld + row - res_r0] += s   (no norm; the
//           sum also replaces the residual in res, for the O tile's router share)
//   SWIGLU: (rows are gate/up pairs: row = ffn unit f, s = gate, s2 = up; the
//           token slot j reads activation row toks[j], c = inv[toks[j]])
//           out[(f + base) * ld + j] = gate_w[toks[j] * k + ranks[j]] * silu(c * s) * (c * s2)
struct GemvEpi {
  enum Kind { STORE, RESID, SWIGLU };
  int kind;
  float* out;
  int ld;
  float* res;
  int res_ld, res_r0;
  int base, k;
  const int* toks;
  const int* ranks;
  const float* gate_w;
  const float* inv;
  __device__ __forceinline__ void operator()(int row, int j, float s, float s2) const {
    switch (kind) {
      case STORE: out[(size_t)j * ld + row] = inv[j] * s; break;
      case RESID: {
        float* r = res + j * res_ld + row - res_r0;
        const float v = *r + s;
        *r = v;
        out[(size_t)j * ld + row] = v;
        break;
      }
      default: {
        const int tj = toks[j];
        const float c = inv[tj], g = c * s;
        out[(size_t)(row + base) * ld + j] = gate_w[tj * k + ranks[j]] * (g / (1.0f + expf(-g)) * (c * s2));
      }
    }
  }
};

// A projection task's GEMV: rows [r0, r1) of a K-wide matrix against the activations.
struct ProjGemv {
  int K, r0, r1;
  GemvEpi epi;
};

template <int NB, bool NUC>
struct Consumer {
  // copies of the router-logit sums this instance adds to, reads and clears
  static constexpr int RLC = NB == 8 ? RL_COPIES_B8 : RL_COPIES;
  const Params& p;
  Ring r;
  float* act;
  Misc* m;
  float* scr;      // after the misc struct: an H-row tile's residual rows, or an expert tile's coefficients
  float* psum;   // per-warp partial sums of wide-row GEMVs: [2 windows][NCW][WIN_ROWS][NB]
  static constexpr int WIN_ROWS = win_rows(NB);
  int ct, cw, lane;
  int ti = 0;
  int step = 0;      // step of this launch being run (0 .. nsteps - 1)
  uint32_t epoch = 0;   // its counter epoch: p.epoch + step
  int lm_done = 0;   // LM-head tiles this CTA finished in this step (its last task is the last of them)

  __device__ void mark(int k) {
    if (p.trace && ct == 0) p.trace[(size_t)ti * TRACE_SLOTS + k] = gtimer();
  }

  // ---- ring access (per warp)
  int nstage_seen = 0;   // stages of the current task seen by this warp (timeline only)

  __device__ const uint8_t* wait_stage(bool& ab) {
    if (ab) return nullptr;
    if (!mbar_wait(p, m, &m->full[r.stage], r.round & 1, -4)) {
      ab = true;
      m->abort_flag = 1;
      return nullptr;
    }
    if (p.trace) {
      mark(nstage_seen == 0 ? TR_S_FIRST : TR_S_LAST);
      ++nstage_seen;
    }
    if (p.strace && ct == 0) stage_stamp(1);
    return r.base + (size_t)r.stage * r.sb;
  }
  __device__ void release_stage(bool ab) {
    __syncwarp();
    if (!ab && lane == 0) mbar_arrive(&m->empty[r.stage]);
    if (p.strace && ct == 0) stage_stamp(2);
    r.advance();
  }
  // The same for a stage that only n-th of the warps read: each of them
  // arrives n times, so the slot's count is met without the other warps.
  __device__ void release_stage_n(bool ab, int n) {
    __syncwarp();
    if (!ab && lane == 0) mbar_arrive_n(&m->empty[r.stage], (uint32_t)n);
    if (p.strace && ct == 0) stage_stamp(2);
    r.advance();
  }
  // Release an earlier stage (slot `stage` of round `round`) without moving the ring.
  __device__ void release_at(bool ab, int stage, int round) {
    __syncwarp();
    if (!ab && lane == 0) mbar_arrive(&m->empty[stage]);
    if (p.strace && ct == 0) {
      const long long lin = (long long)round * r.nst + stage;
      if (lin < STRACE_CAP) {
        unsigned long long* rec = p.strace + ((size_t)blockIdx.x * STRACE_CAP + lin) * STRACE_SLOTS;
        rec[2] = gtimer();
        rec[5] = (unsigned long long)clock64();
      }
    }
  }
  __device__ void stage_stamp(int k) {
    const long long lin = (long long)r.round * r.nst + r.stage;
    if (lin < STRACE_CAP) {
      unsigned long long* rec = p.strace + ((size_t)blockIdx.x * STRACE_CAP + lin) * STRACE_SLOTS;
      rec[k] = gtimer();
      rec[3 + k] = (unsigned long long)clock64();
    }
  }

  // ---- activations
  // act[b * H + i] = x_b[i] * gamma[i] for b < B, with x_b read four floats at
  // a time by src(b, i4), and m->inv[b] = 1 / sqrt(mean(x_b^2) + eps): the
  // norm's scale is applied to the GEMV sums (the map is linear), so the gain
  // and x come in one L2 round trip and the activations are written once.
  // m->inv is written after a barrier; every caller passes another barrier
  // before its GEMV reads it.
  template <class Src4>
  __device__ void fill_rmsnorm(const uint16_t* gamma, Src4 src) {
    const int H = p.H, H4 = H >> 2, B = p.B;
    if constexpr (NB == 1) {
      float ss = 0.f;
      float4* dst = reinterpret_cast<float4*>(act);
#pragma unroll 4
      for (int i = ct; i < H4; i += NCT) {
        const float4 v = src(0, i);
        const uint2 gb = __ldg(reinterpret_cast<const uint2*>(gamma) + i);
        dst[i] = make_float4(v.x * bf_lo(gb.x), v.y * bf_hi(gb.x), v.z * bf_lo(gb.y), v.w * bf_hi(gb.y));
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
      }
      ss = warp_sum(ss);
      if (lane == 0) m->red[cw] = ss;
    } else {
      // every request's loads of a column group go out together: one round trip, not B
      float ss[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) ss[b] = 0.f;
      for (int i = ct; i < H4; i += NCT) {
        float4 v[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) v[b] = b < B ? src(b, i) : make_float4(0.f, 0.f, 0.f, 0.f);
        const uint2 gb = __ldg(reinterpret_cast<const uint2*>(gamma) + i);
        const float g0 = bf_lo(gb.x), g1 = bf_hi(gb.x), g2 = bf_lo(gb.y), g3 = bf_hi(gb.y);
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b < B) {
            reinterpret_cast<float4*>(act + (size_t)b * H)[i] =
                make_float4(v[b].x * g0, v[b].y * g1, v[b].z * g2, v[b].w * g3);
            ss[b] = fmaf(v[b].x, v[b].x, fmaf(v[b].y, v[b].y, fmaf(v[b].z, v[b].z, fmaf(v[b].w, v[b].w, ss[b]))));
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < B) {
          const float t = warp_sum(ss[b]);
          if (lane == 0) m->red[b * NCW + cw] = t;
        }
      }
    }
    cbar();
    if (ct < B) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; ++w) tot += m->red[ct * NCW + w];
      m->inv[ct] = 1.0f / sqrtf(tot / (float)H + p.eps);
    }
  }

  // Token id of request b, checked: an id outside [0, vocab) records
  // MK_ERR_INVALID and reads row 0 instead of faulting.
  __device__ int token(int b) const {
    const int tok = step == 0 ? __ldcg(p.tokens + b) : __ldcg(p.next_token + (size_t)(step - 1) * p.io_stride + b);
    if (tok < 0 || tok >= p.V) {
      set_error(p, MK_ERR_INVALID, -1, tok);
      return 0;
    }
    return tok;
  }

  __device__ float4 x_in4(int l, int b, int i4) const {
    if (l == 0) {
      const int tok = token(b);
      const uint2 e = __ldg(reinterpret_cast<const uint2*>(p.embed + (size_t)tok * p.H) + i4);
      return make_float4(bf_lo(e.x), bf_hi(e.x), bf_lo(e.y), bf_hi(e.y));
    }
    return __ldcg(reinterpret_cast<const float4*>(p.x_out + ((size_t)(l - 1) * p.bcap + b) * p.H) + i4);
  }

  __device__ float x_in(int l, int b, int i) const {
    if (l == 0) return bf2f(p.embed[(size_t)token(b) * p.H + i]);
    return __ldcg(p.x_out + ((size_t)(l - 1) * p.bcap + b) * p.H + i);
  }

  // Element `off` of the QKV outputs: fp32, or the tensor-core tiles'
  // fixed-point sums.
  __device__ __forceinline__ float qkv_at(size_t off) const {
    if constexpr (NB == 8) {
      if (p.qkv_fx) return from_fixed<NB == 8>(__ldcg(p.qkv_fx + off));
    }
    return __ldcg(p.qkv + off);
  }

  // x_mid of layer l (after the O projection and residual), request b: four
  // columns from i4 * 4, or column i (fp32; on the tensor-core path the last
  // O task of each 128-row tile converts the tile's fixed-point sums).
  __device__ __forceinline__ float4 xmid4(int l, int b, int i4) const {
    return __ldcg(reinterpret_cast<const float4*>(p.x_mid + ((size_t)l * p.bcap + b) * p.H) + i4);
  }
  __device__ __forceinline__ float xmid1(int l, int b, int i) const {
    return __ldcg(p.x_mid + ((size_t)l * p.bcap + b) * p.H + i);
  }

  // dot of one 16-byte bf16 granule with 8 activations
  __device__ __forceinline__ static float dot8(const uint4 wv, uint32_t a) {
    return dot8r(wv, lds128f(a), lds128f(a + 16));
  }
  __device__ __forceinline__ static float dot8r(const uint4 wv, const float4 x0, const float4 x1) {
    float s0 = bf_lo(wv.x) * x0.x;
    float s1 = bf_hi(wv.x) * x0.y;
    s0 = fmaf(bf_lo(wv.y), x0.z, s0);
    s1 = fmaf(bf_hi(wv.y), x0.w, s1);
    s0 = fmaf(bf_lo(wv.z), x1.x, s0);
    s1 = fmaf(bf_hi(wv.z), x1.y, s1);
    s0 = fmaf(bf_lo(wv.w), x1.z, s0);
    s1 = fmaf(bf_hi(wv.w), x1.w, s1);
    return s0 + s1;
  }

  // ---- GEMV over rows [r0, r1) of a K-wide bf16 matrix streamed through the
  // ring, against nb activation rows (act row map[j], or j when map is null).
  //
  // Wide rows (K a multiple of 2048, the model's hidden and attention widths):
  // warp w owns the 256-column slices w, w+8, ...; per stage it accumulates up
  // to 8 rows at once (independent chains), reduces them across its lanes and
  // parks one partial per (warp, row) in a 32-row smem window.  When a window
  // fills (or the range ends) the consumer threads sum the 8 warp partials in
  // warp order -- the same order every run -- and call the epilogue.
  // Narrow rows (other K): warp w owns rows w, w+8, ..., up to 8 at a time,
  // its lanes span the whole row, and it calls the epilogue itself.
  //
  // PAIRS: rows come as (gate, up) pairs 2f, 2f+1 and the epilogue is
  // epi(f, j, gate_sum, up_sum); otherwise epi(row, j, sum).
  // Window flush of the column-slice GEMV: sum the 8 warps' partials of the
  // window's rows in warp order and hand each (row or pair, batch row) to the epilogue.
  template <class Epi>
  __device__ __forceinline__ void gemv_flush(bool pairs, bool ab, int buf, int wbase, int wrow, int nb, Epi& epi) {
    cbar();
    if (ab) return;
    const float* pb = psum + (size_t)buf * NCW * WIN_ROWS * NB;
    const int units = pairs ? wrow >> 1 : wrow;
    for (int x = ct; x < units * nb; x += NCT) {
      const int u = x / nb, j = x - u * nb;
      if (pairs) {
        float g = 0.f, up = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          g += pb[((size_t)w * WIN_ROWS + 2 * u) * NB + j];
          up += pb[((size_t)w * WIN_ROWS + 2 * u + 1) * NB + j];
        }
        epi((wbase >> 1) + u, j, g, up);
      } else {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) s += pb[((size_t)w * WIN_ROWS + u) * NB + j];
        epi(wbase + u, j, s, 0.f);
      }
    }
  }

  template <bool PAIRS, bool SP, class Epi>
  __device__ bool gemv(int K, int r0, int r1, const float* a, int stride, const int* map, int nb, bool ab,
                       Epi epi) {
    const int rps = PAIRS ? 2 * pairs_per_stage(p) : rows_per_stage(p, K);
    const int ng = K >> 3;
    const uint32_t rowb = (uint32_t)K * 2;
    uint32_t aoff[NB];  // shared address of each activation row
#pragma unroll
    for (int j = 0; j < NB; ++j) aoff[j] = smem_u32(a) + (uint32_t)((j < nb ? (map ? map[j] : j) : 0) * stride * 4);
    if ((K & 2047) == 0) {
      const int spw = K >> 11;  // granules per lane per row
      int wbase = r0, wrow = 0, buf = 0;
      for (int s0 = r0; s0 < r1;) {
        const int n = min(rps, r1 - s0);
        if constexpr (SP && NB <= 2) {
          // two stages per pass when a second one follows and both fit the
          // window: twice the independent work between reductions
          const int n2 = min(rps, r1 - s0 - rps);
          if ((rps == 8 || rps == 4) && n == rps && n2 > 0 && wrow + n + n2 <= WIN_ROWS) {
            const uint8_t* sa = wait_stage(ab);
            const int ga = r.stage, ra = r.round;
            r.advance();
            const uint8_t* sb = wait_stage(ab);
            if (sa && sb) {
              const uint32_t ta = smem_u32(sa), tb = smem_u32(sb);
              float* ps = psum + ((size_t)buf * NCW + cw) * WIN_ROWS * NB;
              if (rps == 8) {
                // 16 rows: 8 from each stage, one granule column per lane (K = 2048)
                float part[16][NB];
#pragma unroll
                for (int q = 0; q < 16; ++q)
#pragma unroll
                  for (int j = 0; j < NB; ++j) part[q][j] = 0.f;
                for (int sw = 0; sw < spw; ++sw) {
                  const int gi = (cw + NCW * sw) * 32 + lane;
                  float4 x0[NB], x1[NB];
#pragma unroll
                  for (int j = 0; j < NB; ++j) {
                    x0[j] = j < nb ? lds128f(aoff[j] + gi * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
                    x1[j] = j < nb ? lds128f(aoff[j] + gi * 32 + 16) : make_float4(0.f, 0.f, 0.f, 0.f);
                  }
                  uint4 wv[16];
#pragma unroll
                  for (int q = 0; q < 8; ++q) wv[q] = lds128(ta + (uint32_t)q * rowb + gi * 16);
#pragma unroll
                  for (int q = 0; q < 8; ++q)
                    wv[8 + q] = q < n2 ? lds128(tb + (uint32_t)q * rowb + gi * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
                  for (int q = 0; q < 16; ++q)
#pragma unroll
                    for (int j = 0; j < NB; ++j) part[q][j] += dot8r(wv[q], x0[j], x1[j]);
                }
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                  if (j < nb) {
                    float v[8], w2[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                      v[q] = part[q][j];
                      w2[q] = part[8 + q][j];
                    }
                    const float sum = reduce8(v, lane), sum2 = reduce8(w2, lane);
                    const int q = (lane >> 2) & 7;
                    if ((lane & 3) == 0) {
                      ps[(wrow + q) * NB + j] = sum;
                      if (q < n2) ps[(wrow + 8 + q) * NB + j] = sum2;
                    }
                  }
                }
              } else {
                // 8 rows: 4 from each stage (K = 4096, two granule columns per lane)
                float part[8][NB];
#pragma unroll
                for (int q = 0; q < 8; ++q)
#pragma unroll
                  for (int j = 0; j < NB; ++j) part[q][j] = 0.f;
                for (int sw = 0; sw < spw; ++sw) {
                  const int gi = (cw + NCW * sw) * 32 + lane;
                  float4 x0[NB], x1[NB];
#pragma unroll
                  for (int j = 0; j < NB; ++j) {
                    x0[j] = j < nb ? lds128f(aoff[j] + gi * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
                    x1[j] = j < nb ? lds128f(aoff[j] + gi * 32 + 16) : make_float4(0.f, 0.f, 0.f, 0.f);
                  }
                  uint4 wv[8];
#pragma unroll
                  for (int q = 0; q < 4; ++q) wv[q] = lds128(ta + (uint32_t)q * rowb + gi * 16);
#pragma unroll
                  for (int q = 0; q < 4; ++q)
                    wv[4 + q] = q < n2 ? lds128(tb + (uint32_t)q * rowb + gi * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
                  for (int q = 0; q < 8; ++q)
#pragma unroll
                    for (int j = 0; j < NB; ++j) part[q][j] += dot8r(wv[q], x0[j], x1[j]);
                }
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                  if (j < nb) {
                    float v[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[q] = part[q][j];
                    const float sum = reduce8(v, lane);
                    const int q = (lane >> 2) & 7;
                    if ((lane & 3) == 0 && q < 4 + n2) ps[(wrow + q) * NB + j] = sum;
                  }
                }
              }
            }
            release_at(ab, ga, ra);
            release_stage(ab);
            wrow += n + n2;
            s0 += n + n2;
            if (wrow + rps > WIN_ROWS || s0 >= r1) {
              gemv_flush(PAIRS, ab, buf, wbase, wrow, nb, epi);
              buf ^= 1;
              wbase = s0;
              wrow = 0;
            }
            continue;
          }
        }
        const uint8_t* st = wait_stage(ab);
        if (st) {
          const uint32_t sts = smem_u32(st);
          bool done4 = false;
          if constexpr (NB <= 2) {
            if (n <= 4) {
              // 4-row stage (K = 4096 at 32 KB): 4 chains, 4-value reduction
              float part4[4][NB];
#pragma unroll
              for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int j = 0; j < NB; ++j) part4[q][j] = 0.f;
              for (int sw = 0; sw < spw; ++sw) {
                const int gi = (cw + NCW * sw) * 32 + lane;
                float4 x0[NB], x1[NB];
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                  x0[j] = j < nb ? lds128f(aoff[j] + gi * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
                  x1[j] = j < nb ? lds128f(aoff[j] + gi * 32 + 16) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                uint4 wv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  wv[q] = q < n ? lds128(sts + (uint32_t)q * rowb + gi * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                  for (int j = 0; j < NB; ++j) part4[q][j] += dot8r(wv[q], x0[j], x1[j]);
              }
              float* ps = psum + ((size_t)buf * NCW + cw) * WIN_ROWS * NB;
#pragma unroll
              for (int j = 0; j < NB; ++j) {
                if (j < nb) {
                  float v[4];
#pragma unroll
                  for (int q = 0; q < 4; ++q) v[q] = part4[q][j];
                  const float sum = reduce4(v, lane);
                  const int q = (lane >> 3) & 3;
                  if ((lane & 7) == 0 && q < n) ps[(wrow + q) * NB + j] = sum;
                }
              }
              done4 = true;
            }
          }
          for (int rb = 0; rb < n && !done4; rb += 8) {
            float part[8][NB];
#pragma unroll
            for (int q = 0; q < 8; ++q)
#pragma unroll
              for (int j = 0; j < NB; ++j) part[q][j] = 0.f;
            for (int sw = 0; sw < spw; ++sw) {
              const int gi = (cw + NCW * sw) * 32 + lane;
              if constexpr (NB <= 4) {
                // this warp's 8 activation columns are the same for every row of the batch
                float4 x0[NB], x1[NB];
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                  x0[j] = j < nb ? lds128f(aoff[j] + gi * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
                  x1[j] = j < nb ? lds128f(aoff[j] + gi * 32 + 16) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if constexpr (NB <= 2) {
                  uint4 wv[8];
#pragma unroll
                  for (int q = 0; q < 8; ++q)
                    wv[q] = rb + q < n ? lds128(sts + (uint32_t)(rb + q) * rowb + gi * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
                  for (int q = 0; q < 8; ++q)
#pragma unroll
                    for (int j = 0; j < NB; ++j) part[q][j] += dot8r(wv[q], x0[j], x1[j]);
                } else {
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    if (rb + q < n) {
                      const uint4 wv = lds128(sts + (uint32_t)(rb + q) * rowb + gi * 16);
#pragma unroll
                      for (int j = 0; j < NB; ++j) part[q][j] += dot8r(wv, x0[j], x1[j]);
                    }
                  }
                }
              } else {
                // rows in two groups of 4 held in registers; each activation
                // row is read once per group instead of once per weight row
#pragma unroll
                for (int h = 0; h < 8; h += 4) {
                  uint4 wv[4];
#pragma unroll
                  for (int q = 0; q < 4; ++q)
                    wv[q] = rb + h + q < n ? lds128(sts + (uint32_t)(rb + h + q) * rowb + gi * 16)
                                           : make_uint4(0, 0, 0, 0);
#pragma unroll
                  for (int j = 0; j < NB; ++j) {
                    if (j < nb) {
                      const float4 x0 = lds128f(aoff[j] + gi * 32), x1 = lds128f(aoff[j] + gi * 32 + 16);
#pragma unroll
                      for (int q = 0; q < 4; ++q) part[h + q][j] += dot8r(wv[q], x0, x1);
                    }
                  }
                }
              }
            }
            float* ps = psum + ((size_t)buf * NCW + cw) * WIN_ROWS * NB;
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              if (j < nb) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = part[q][j];
                const float sum = reduce8(v, lane);
                const int q = (lane >> 2) & 7;
                if ((lane & 3) == 0 && rb + q < n) ps[(wrow + rb + q) * NB + j] = sum;
              }
            }
          }
        }
        release_stage(ab);
        wrow += n;
        s0 += n;
        if (wrow + rps > WIN_ROWS || s0 >= r1) {
          gemv_flush(PAIRS, ab, buf, wbase, wrow, nb, epi);
          buf ^= 1;
          wbase = s0;
          wrow = 0;
        }
      }
    } else {
      for (int s0 = r0; s0 < r1; s0 += rps) {
        const int n = min(rps, r1 - s0);
        const uint8_t* st = wait_stage(ab);
        if constexpr (!PAIRS && NB <= 2) {
          if (st && n <= 2 * NCW) {
            // short stage (the expert down rows of one CTA): warp w takes rows
            // w and w + 8 whole, two independent chains, one warp sum each
            const uint32_t sts = smem_u32(st);
            const bool va = cw < n, vb = cw + NCW < n;
            float pa[NB], pb[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) pa[j] = pb[j] = 0.f;
#pragma unroll 3
            for (int gi = lane; gi < ng; gi += 32) {
              float4 x0[NB], x1[NB];
#pragma unroll
              for (int j = 0; j < NB; ++j) {
                x0[j] = j < nb ? lds128f(aoff[j] + gi * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
                x1[j] = j < nb ? lds128f(aoff[j] + gi * 32 + 16) : make_float4(0.f, 0.f, 0.f, 0.f);
              }
              if (va) {
                const uint4 wv = lds128(sts + (uint32_t)cw * rowb + gi * 16);
#pragma unroll
                for (int j = 0; j < NB; ++j) pa[j] += dot8r(wv, x0[j], x1[j]);
              }
              if (vb) {
                const uint4 wv = lds128(sts + (uint32_t)(cw + NCW) * rowb + gi * 16);
#pragma unroll
                for (int j = 0; j < NB; ++j) pb[j] += dot8r(wv, x0[j], x1[j]);
              }
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              if (j < nb) {
                const float sa = warp_sum(pa[j]), sb = warp_sum(pb[j]);
                if (lane == 0) {
                  if (va) epi(s0 + cw, j, sa, 0.f);
                  if (vb) epi(s0 + cw + NCW, j, sb, 0.f);
                }
              }
            }
            release_stage(ab);
            continue;
          }
        }
        if (st) {
          const uint32_t sts = smem_u32(st);
          // PAIRS: warp w takes pairs w, w+8, ... (rows 2f, 2f+1); else rows w, w+8, ...
          const int unit = PAIRS ? 2 : 1;
          const int per = 8 / unit;  // units per batch of 8 rows
          for (int u0 = cw; u0 * unit < n; u0 += NCW * per) {
            float part[8][NB];
#pragma unroll
            for (int q = 0; q < 8; ++q)
#pragma unroll
              for (int j = 0; j < NB; ++j) part[q][j] = 0.f;
            if constexpr (NB <= 2) {
              for (int gi = lane; gi < ng; gi += 32) {
                float4 x0[NB], x1[NB];
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                  x0[j] = j < nb ? lds128f(aoff[j] + gi * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
                  x1[j] = j < nb ? lds128f(aoff[j] + gi * 32 + 16) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const int row = (u0 + NCW * (q / unit)) * unit + (q % unit);
                  if (row < n) {
                    const uint4 wv = lds128(sts + (uint32_t)row * rowb + gi * 16);
#pragma unroll
                    for (int j = 0; j < NB; ++j) part[q][j] += dot8r(wv, x0[j], x1[j]);
                  }
                }
              }
            } else {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int row = (u0 + NCW * (q / unit)) * unit + (q % unit);
                if (row < n) {
                  for (int gi = lane; gi < ng; gi += 32) {
                    const uint4 wv = lds128(sts + (uint32_t)row * rowb + gi * 16);
#pragma unroll
                    for (int j = 0; j < NB; ++j)
                      if (j < nb) part[q][j] += dot8(wv, aoff[j] + gi * 32);
                  }
                }
              }
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              if (j < nb) {
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) v[q] = part[q][j];
                const float sum = reduce8(v, lane);
                const int q = (lane >> 2) & 7;
                if (PAIRS) {
                  const float other = __shfl_down_sync(FULL, sum, 4);  // group q+1 = the up row
                  const int row = (u0 + NCW * (q / 2)) * 2;
                  if ((lane & 7) == 0 && row < n) epi((s0 + row) >> 1, j, sum, other);
                } else {
                  const int row = u0 + NCW * q;
                  if ((lane & 3) == 0 && row < n) epi(s0 + row, j, sum, 0.f);
                }
              }
            }
          }
        }
        release_stage(ab);
      }
    }
    return ab;
  }

  // End of a task: agree on failure.  The barrier orders every consumer
  // thread's writes before thread 0's release (atom.release.gpu is cumulative),
  // so the signal publishes them without a fence in every thread.
  __device__ bool finish(bool ab) { return cbar_or(ab); }

  __device__ void signal(int ctr) {
    if (ct == 0) red_add_release(p.ctr + (size_t)ctr * CTR_STRIDE, 1u);
  }

  // Uniform "do my add signals complete the n of this step" for counter ctr.
  __device__ bool ticket(int ctr, uint32_t n, uint32_t add) {
    if (ct == 0) {
      const uint32_t old = atom_add_acq_rel(p.ctr + (size_t)ctr * CTR_STRIDE, add);
      m->ticket_last = (old + add == epoch * n) ? 1 : 0;
    }
    cbar();
    return m->ticket_last != 0;
  }

  // ------------------------------------------------------------ tasks

  // ---- projections: QKV, O (+ residual), router logits.  prep_* builds the
  // activations and the GEMV's range and epilogue; the caller runs the GEMV;
  // post_proj signals the task's counter.
  __device__ bool prep_qkv(const Task& t, bool ab, ProjGemv& g) {
    const int l = t.layer;
    if (!ab) fill_rmsnorm(p.attn_norm[l], [&](int b, int i4) { return x_in4(l, b, i4); });
    // the column-slice GEMV (K a multiple of 2048) reads the scale only after its
    // window barrier; the narrow-row path calls the epilogue without one
    if (p.H & 2047) cbar();
    g.K = p.H;
    g.r0 = t.a[0];
    g.r1 = t.a[1];
    g.epi = GemvEpi{};
    g.epi.kind = GemvEpi::STORE;
    g.epi.out = p.qkv + (size_t)l * p.bcap * p.qkv_rows;
    g.epi.ld = p.qkv_rows;
    g.epi.inv = m->inv;
    return ab;
  }

  // K half h of the O projection (h = 0 only, unless o_halves = 2): the
  // attention output's columns of that half as the activations; the residual
  // epilogue accumulates the halves in the scratch rows.
  __device__ bool prep_oproj(const Task& t, bool ab, ProjGemv& g, int h) {
    const int l = t.layer, KF = p.nq * p.d, K = NB > 2 ? KF / p.o_halves : KF, r0 = t.a[0], nr = t.a[1] - r0;
    float* xres = scr;    // residual rows of this tile, [B][nr]
    if (h > 0) cbar();    // the previous half's GEMV is done with the activations
    if (!ab) {
      // the residual rows' loads go out first, with the attention output's
      const bool r1st = h == 0 && ct < p.B * nr;
      const float x1st = r1st ? x_in(l, ct / nr, r0 + ct % nr) : 0.f;
      const float* o = p.o + (size_t)l * p.bcap * KF + (size_t)h * K;
      if (NB <= 2 || K == KF) {   // whole rows: one contiguous copy
        const float4* o4 = reinterpret_cast<const float4*>(o);
        float4* dst = reinterpret_cast<float4*>(act);
#pragma unroll 4
        for (int i = ct; i < (p.B * K) >> 2; i += NCT) dst[i] = __ldcg(o4 + i);
      } else {
        const int K4 = K >> 2;
#pragma unroll 4
        for (int i = ct; i < p.B * K4; i += NCT) {
          const int b = i / K4, c = i - b * K4;
          reinterpret_cast<float4*>(act + (size_t)b * K)[c] =
              __ldcg(reinterpret_cast<const float4*>(o + (size_t)b * KF) + c);
        }
      }
      if (r1st) xres[ct] = x1st;
      if (h == 0)
        for (int i = ct + NCT; i < p.B * nr; i += NCT) xres[i] = x_in(l, i / nr, r0 + i % nr);
    }
    cbar();
    g.K = K;
    g.r0 = r0;
    g.r1 = t.a[1];
    g.epi = GemvEpi{};
    g.epi.kind = GemvEpi::RESID;
    g.epi.out = p.x_mid + (size_t)l * p.bcap * p.H;
    g.epi.ld = p.H;
    g.epi.res = xres;
    g.epi.res_ld = nr;
    g.epi.res_r0 = r0;
    return ab;
  }

  __device__ bool post_proj(const Task& t, bool ab) {
    const int l = t.layer;
    if (t.type == T_OPROJ) ab = router_part(t, ab);
    ab = finish(ab);
    if (!ab) {
      if (t.type == T_QKV) signal(p.cm.qkv + l * p.nkv + t.a[2]);
      else signal(p.cm.o + l);
    }
    return ab;
  }

  // The O tile's share of the router logits over its hidden rows h in [r0, r1):
  //   part[b][e] = sum_h WrT[h][e] * gain[h] * x_mid[b][h]
  // (the logits are inv_rms(x_mid_b) times the sum of every tile's part), from
  // the x_mid rows the residual epilogue left in the scratch and the router
  // stage.  The parts are added as 32.32 fixed-point integers: the sum is
  // exact, so its bits do not depend on the order the tiles arrive in.
  __device__ bool router_part(const Task& t, bool ab) {
    const int r0 = t.a[0], nr = t.a[1] - r0, E = p.E;
    const uint8_t* st = wait_stage(ab);
    cbar();   // every x_mid row of the tile is in the scratch
    if (st) {
      const uint16_t* wr = reinterpret_cast<const uint16_t*>(st);
      const uint16_t* gw = reinterpret_cast<const uint16_t*>(st + router_stage_gain_off(nr, E)) + (r0 & 7);
      // copy t % RLC of the sums: RLC times fewer tiles contend for each address
      unsigned long long* out = p.rlsum + ((size_t)t.layer * RL_COPIES + t.a[2] % RLC) * p.bcap * E;
      // two neighbouring threads per (b, e), each half the rows, then one shuffle
      const int n2 = 2 * p.B * E, hr = (nr + 1) >> 1;
      for (int x0 = 0; x0 < n2; x0 += NCT) {
        const int x = x0 + ct, half = x & 1, be = x >> 1;
        const bool ok = x < n2;
        const int b = ok ? be / E : 0, e = ok ? be - b * E : 0;
        const float* xr = scr + b * nr;
        const int i0 = half ? hr : 0, i1 = half ? nr : hr;
        float acc = 0.f;
        if (ok)
          for (int i = i0; i < i1; ++i) acc = fmaf(bf2f(wr[i * E + e]) * bf2f(gw[i]), xr[i], acc);
        const float other = __shfl_xor_sync(FULL, acc, 1);
        if (ok && half == 0) atomicAdd(out + (size_t)b * E + e, to_fixed<NB == 8>(acc + other));
      }
    }
    release_stage(ab);
    return ab;
  }

  // Order-preserving key of a router logit (never NaN here: moe_act stores
  // NaN as -inf): a larger logit has a larger key, equal logits equal keys,
  // and 0 is below them all.
  __device__ __forceinline__ static uint32_t rkey(float v) {
    const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);   // -0 and +0 compare equal
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  }

  // The top-k of request b's logits (m->rl), by the calling warp: k rounds,
  // each taking the largest logit left, the lowest index on ties, so pick i
  // is the logit of rank i (how many logits are greater, or equal with a
  // lower index).  Lane i < k returns pick i (expert and logit).
  __device__ __forceinline__ void route_pick(int b, int& e_out, float& v_out) const {
    const int E = p.E, k = p.k;
    const float* row = m->rl + b * E;
    constexpr int EPL = MAX_EXPERTS / 32;   // logits per lane: expert lane + 32 j
    uint32_t key[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) key[j] = lane + 32 * j < E ? rkey(row[lane + 32 * j]) : 0u;
    e_out = 0;
    v_out = 0.f;
    for (int r = 0; r < k; ++r) {
      uint32_t bk = 0;
      int bj = 0;
#pragma unroll
      for (int j = EPL - 1; j >= 0; --j)   // this lane's largest key, its lowest j on ties
        if (key[j] >= bk) {
          bk = key[j];
          bj = j;
        }
      const uint32_t top = __reduce_max_sync(FULL, bk);
      const int e = (int)__reduce_min_sync(FULL, bk == top ? (uint32_t)(lane + 32 * bj) : 0xFFFFFFFFu);
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (e == lane + 32 * j) key[j] = 0u;   // taken
      if (lane == r) {
        e_out = e;
        v_out = row[e];
      }
    }
  }

  // Routing of layer l from its router logits (m->rl), computed in every
  // gate/up task the same way, so every CTA gets the same bits:
  //  - per request, the top-k by route_pick, in rank order;
  //  - gates: softmax over the selected logits;
  //  - the distinct experts in ascending order, with their (request, rank)
  //    pairs in request order (r_U, r_exp, r_cnt, r_tok, r_rank).
  // The distinct experts go to this CTA's producer (r_layer) as soon as they
  // are known, before the token lists.  With publish
  // set it also goes to global memory (ids, gates, routing table) and the
  // rdone counter is signalled.
  // Expects m->rl loaded and m->cnt_of zeroed, both behind a barrier.
  __device__ void route_local(int l, bool publish) {
    const int E = p.E, k = p.k, B = p.B;
    const int umax = p.rm.umax, bc = p.rm.bcap;
    if (B == 1) {
      // one request: warp 0 alone.  Its k experts are distinct: the gates
      // (softmax over the picks; the butterfly over all 32 lanes adds only
      // zeros past k), and each pick's place in ascending id order gives the
      // distinct-expert table, one token slot each, handed to the producer
      // before the other warps hear of it.
      if (cw == 0) {
        int e;
        float v;
        route_pick(0, e, v);
        const bool on = lane < k;
        const float v0 = __shfl_sync(FULL, v, 0);   // every lane: the shuffle is warp-wide
        const float ex = on ? expf(v - v0) : 0.f;
        float tot = ex;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) tot += __shfl_xor_sync(FULL, tot, o);
        int pos = 0;
        for (int j = 0; j < k; ++j) pos += __shfl_sync(FULL, e, j) < e;
        if (on) {
          m->sel[lane] = e;
          m->selv[lane] = v;
          m->gate[lane] = ex / tot;
          m->r_exp[pos] = e;
          m->r_cnt[pos] = 1;
          m->r_tok[pos * bc] = 0;
          m->r_rank[pos * bc] = lane;
        }
        if (lane == 0) m->r_U = k;
        __syncwarp();
        if (lane == 0) st_release_cta(&m->r_layer, step * p.L + l);
      }
      cbar();
    } else {
      // warp w picks request w's experts and gates (butterfly sum as above)
      for (int b = cw; b < B; b += NCW) {
        int e;
        float v;
        route_pick(b, e, v);
        const bool on = lane < k;
        const float v0 = __shfl_sync(FULL, v, 0);   // every lane: the shuffle is warp-wide
        const float ex = on ? expf(v - v0) : 0.f;
        float tot = ex;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) tot += __shfl_xor_sync(FULL, tot, o);
        if (on) {
          m->sel[b * k + lane] = e;
          m->selv[b * k + lane] = v;
          m->gate[b * k + lane] = ex / tot;
          atomicAdd(&m->cnt_of[e], 1);
        }
      }
      cbar();
      if (cw == 0) {
        int base = 0;
        for (int c = 0; c < (E + 31) / 32; ++c) {
          const int e = c * 32 + lane;
          const bool pres = e < E && m->cnt_of[e] > 0;
          const unsigned mask = __ballot_sync(FULL, pres);
          if (pres) {
            const int u = base + __popc(mask & ((1u << lane) - 1u));
            m->slot_of[e] = u;
            m->r_exp[u] = e;
            m->r_cnt[u] = m->cnt_of[e];
          }
          base += __popc(mask);
        }
        if (lane == 0) m->r_U = base;
      }
      cbar();
      if (ct == 0) st_release_cta(&m->r_layer, step * p.L + l);   // the producer needs only r_U and r_exp
      if (ct < B * k) {
        const int e = m->sel[ct];
        int rank = 0;
        for (int q = 0; q < ct; ++q) rank += (m->sel[q] == e);
        const int u = m->slot_of[e];
        m->r_tok[u * bc + rank] = ct / k;
        m->r_rank[u * bc + rank] = ct % k;
      }
      cbar();
    }
    if (!publish) return;
    int* rt = const_cast<int*>(route_of(p, l));
    const int U = m->r_U;
    if (ct == 0) rt[0] = U;
    for (int u = ct; u < U; u += NCT) {
      rt[1 + u] = m->r_exp[u];
      rt[1 + umax + u] = m->r_cnt[u];
    }
    for (int i = ct; i < U * bc; i += NCT) {
      rt[1 + 2 * umax + i] = m->r_tok[i];
      rt[1 + 2 * umax + umax * bc + i] = m->r_rank[i];
    }
    if (ct < B * k) {
      p.ids[((size_t)l * p.bcap + ct / k) * k + ct % k] = m->sel[ct];
      p.gates[((size_t)l * p.bcap + ct / k) * k + ct % k] = m->gate[ct];
    }
    for (int i = ct; i < B * E; i += NCT) p.rlog[((size_t)l * p.bcap + i / E) * E + i % E] = m->rl[i];
    cbar();
    signal(p.cm.rdone + l);
  }

  // The expert tile's activations: act = x_mid * FFN gain with m->inv (as
  // fill_rmsnorm), and the layer's router logits m->rl[b * E + e] = inv[b] *
  // (the O tiles' fixed-point sum), NaN ranked as -inf.  The sums' loads go
  // out first and the norm's inputs (at most two float4 per thread: H <= 2048)
  // right after, so both arrive in one round trip.
  __device__ void moe_act(int l) {
    const int H = p.H, H4 = H >> 2, E = p.E, BE = p.B * E;
    const size_t cs = (size_t)p.bcap * E;   // one copy of the sums
    const unsigned long long* rs = p.rlsum + (size_t)l * RL_COPIES * cs;
    auto load_sum = [&](int i) {   // the copies' integer sum: exact in any order
      unsigned long long v[RLC];
#pragma unroll
      for (int c = 0; c < RLC; ++c) v[c] = __ldcg(rs + c * cs + i);
      unsigned long long q = 0;
#pragma unroll
      for (int c = 0; c < RLC; ++c) q += v[c];
      return q;
    };
    unsigned long long v0[RLC];   // this thread's first sum: its loads go out now, the adds come later
#pragma unroll
    for (int c = 0; c < RLC; ++c) v0[c] = ct < BE ? __ldcg(rs + c * cs + ct) : 0ull;
    const uint2* gam = reinterpret_cast<const uint2*>(p.ffn_norm[l]);
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 x0[2];
    uint2 g0[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = ct + h * NCT;
      x0[h] = i < H4 ? xmid4(l, 0, i) : z4;
      g0[h] = i < H4 ? __ldg(gam + i) : make_uint2(0u, 0u);
    }
    for (int i = ct; i < MAX_EXPERTS; i += NCT) m->cnt_of[i] = 0;
    if constexpr (NB == 1) {
      float ss = 0.f;
      float4* dst = reinterpret_cast<float4*>(act);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = ct + h * NCT;
        if (i < H4) {
          const float4 xv = x0[h];
          const uint2 gb = g0[h];
          dst[i] = make_float4(xv.x * bf_lo(gb.x), xv.y * bf_hi(gb.x), xv.z * bf_lo(gb.y), xv.w * bf_hi(gb.y));
          ss = fmaf(xv.x, xv.x, fmaf(xv.y, xv.y, fmaf(xv.z, xv.z, fmaf(xv.w, xv.w, ss))));
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) m->red[cw] = ss;
    } else {
      // the other requests' rows: all loads out together (one round trip, not B - 1)
      float4 xv[2][NB];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = ct + h * NCT;
        xv[h][0] = x0[h];
#pragma unroll
        for (int b = 1; b < NB; ++b)
          xv[h][b] = b < p.B && i < H4 ? xmid4(l, b, i) : z4;
      }
      float ss[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) ss[b] = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = ct + h * NCT;
        if (i < H4) {
          const uint2 gb = g0[h];
          const float ga = bf_lo(gb.x), gc = bf_hi(gb.x), ge = bf_lo(gb.y), gg = bf_hi(gb.y);
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const float4 v = xv[h][b];
            const float4 y = make_float4(v.x * ga, v.y * gc, v.z * ge, v.w * gg);
            if (NB == 8 && p.tm_gu) {
              // the tensor cores' B operand: bf16 hi (row b) and lo (row 8 + b)
              // of x * gain, K-major, 128-byte swizzled (zero rows past the batch)
              store_b_operand(b, 4 * i, b < p.B ? y : z4);
            } else if (b < p.B) {
              reinterpret_cast<float4*>(act + (size_t)b * H)[i] = y;
            }
            if (b < p.B) ss[b] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss[b]))));
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < p.B) {
          const float t = warp_sum(ss[b]);
          if (lane == 0) m->red[b * NCW + cw] = t;
        }
      }
      if (NB == 8 && p.tm_gu) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // read by the tensor cores
    }
    cbar();
    unsigned long long q0 = 0;
#pragma unroll
    for (int c = 0; c < RLC; ++c) q0 += v0[c];
    if constexpr (NB == 1) {
      // one request: every thread forms the scale itself (the same sum in the
      // same order, so the same bits); the routing's barrier orders m->inv[0]
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; ++w) tot += m->red[w];
      const float inv0 = 1.0f / sqrtf(tot / (float)H + p.eps);
      if (ct == 0) m->inv[0] = inv0;
      for (int i = ct; i < BE; i += NCT) {
        const float v = from_fixed<NB == 8>(i == ct ? q0 : load_sum(i)) * inv0;
        m->rl[i] = v == v ? v : -INFINITY;
      }
    } else {
      if (ct < p.B) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) tot += m->red[ct * NCW + w];
        m->inv[ct] = 1.0f / sqrtf(tot / (float)H + p.eps);
      }
      cbar();
      if (ct < BE) {
        const float v = from_fixed<NB == 8>(q0) * m->inv[ct / E];
        m->rl[ct] = v == v ? v : -INFINITY;
      }
      // the rest two sums at a time, both sets of loads in flight together
      for (int i = ct + NCT; i < BE; i += 2 * NCT) {
        const int i2 = i + NCT;
        unsigned long long a[RLC], c2[RLC];
#pragma unroll
        for (int c = 0; c < RLC; ++c) {
          a[c] = __ldcg(rs + c * cs + i);
          c2[c] = i2 < BE ? __ldcg(rs + c * cs + i2) : 0ull;
        }
        unsigned long long qa = 0, qb = 0;
#pragma unroll
        for (int c = 0; c < RLC; ++c) {
          qa += a[c];
          qb += c2[c];
        }
        const float va = from_fixed<NB == 8>(qa) * m->inv[i / E];
        m->rl[i] = va == va ? va : -INFINITY;
        if (i2 < BE) {
          const float vb = from_fixed<NB == 8>(qb) * m->inv[i2 / E];
          m->rl[i2] = vb == vb ? vb : -INFINITY;
        }
      }
    }
  }

  // ---- expert tile: the layer's routing, then for this tile's (distinct
  // expert, ffn unit) pairs the gate/up rows, giving per token slot the
  // coefficient c = gate x silu(gate row . xn) x (up row . xn), then the same
  // units' rows of the transposed down matrix: y_b += c x Wd^T[unit] for the
  // token's request b.  y is this tile's gated partial of the layer output
  // (moe_part); the reduce tasks add the residual and all tiles' partials.
  // No other CTA's gate/up results are needed, so the tile streams its
  // gate/up and down weights back to back.
  // Element k .. k + 3 of B-operand rows `b` (bf16 hi) and 8 + b (bf16 lo) in
  // the K-major 128-byte swizzled layout: 64-column slices of 16 rows x 128
  // bytes (2 KB), rows in two 8-row groups of 1024 bytes, the 16-byte chunk c
  // of row r stored at chunk c ^ r.
  __device__ __forceinline__ void store_b_operand(int b, int k, float4 y) {
    store_b_at(reinterpret_cast<uint8_t*>(act), b, k, y);
  }
  // The same into the slices from `at` (column k counted from there).
  __device__ __forceinline__ static void store_b_at(uint8_t* at, int b, int k, float4 y) {
    const uint16_t h0 = f2bf(y.x), h1 = f2bf(y.y), h2 = f2bf(y.z), h3 = f2bf(y.w);
    const uint16_t l0 = f2bf(y.x - bf2f(h0)), l1 = f2bf(y.y - bf2f(h1)), l2 = f2bf(y.z - bf2f(h2)),
                   l3 = f2bf(y.w - bf2f(h3));
    const int sl = k >> 6, c = (k & 63) >> 3, half = k & 4;
    uint8_t* base = at + sl * 2048 + b * 128 + ((c ^ b) << 4) + half * 2;
    *reinterpret_cast<uint2*>(base) = make_uint2((uint32_t)h0 | ((uint32_t)h1 << 16), (uint32_t)h2 | ((uint32_t)h3 << 16));
    *reinterpret_cast<uint2*>(base + 1024) =
        make_uint2((uint32_t)l0 | ((uint32_t)l1 << 16), (uint32_t)l2 | ((uint32_t)l3 << 16));
  }

  // A QKV or O projection task on the tensor cores (batch instance 8): rows
  // [row0, row0 + 128) of the matrix over its 128-column K stages [ks0, ks1).
  // B operand slot j (4 KB: two 64-column slices of 16 rows, bf16 hi then lo
  // of the 8 requests' activations, K-major, 128-byte swizzled) holds the
  // columns of stage ks0 + j.  One thread issues each stage's M = 128, N = 16,
  // K = 16 MMAs into TMEM and releases the stage by tcgen05.commit; warps 0-3
  // then read the accumulator (one TMEM lane per row), add each request's hi
  // and lo columns and add the part to the rows' 32.32 fixed-point sums:
  //   QKV: the part times the request's RMS-norm scale (the B rows are x * gain);
  //   O:   the part, plus the residual x in the task that holds K stage 0, and
  //        the part's share of the router logits, sum_r WrT[r][e] gain[r] part[b][r]
  //        (linear in x_mid, so the tasks of a row add theirs separately), from
  //        the router stage that follows the weight stages.
  // The O tasks also clear the layer's QKV sums (the attention has read them).
  __device__ bool proj_tc(const Task& t, bool ab) {
    const int l = t.layer, row0 = t.a[0], ks0 = t.a[3], nu = t.a[4] - t.a[3], B = p.B;
    const bool isq = t.type == T_QKV;
    uint8_t* bs = reinterpret_cast<uint8_t*>(act);
    const int c0 = ks0 * 128, nc = nu * 128;   // the B slots' columns
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!ab) {
      if (isq) {
        // the norm needs whole rows; the B slots take columns [c0, c0 + nc)
        const int H4 = p.H >> 2;
        float ss[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) ss[b] = 0.f;
        for (int i = ct; i < H4; i += NCT) {
          float4 v[8];
#pragma unroll
          for (int b = 0; b < 8; ++b) v[b] = b < B ? x_in4(l, b, i) : z4;
          const int c = 4 * i - c0;
          const bool inb = c >= 0 && c < nc;
          const uint2 gb = inb ? __ldg(reinterpret_cast<const uint2*>(p.attn_norm[l]) + i) : make_uint2(0u, 0u);
          const float g0 = bf_lo(gb.x), g1 = bf_hi(gb.x), g2 = bf_lo(gb.y), g3 = bf_hi(gb.y);
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            ss[b] = fmaf(v[b].x, v[b].x, fmaf(v[b].y, v[b].y, fmaf(v[b].z, v[b].z, fmaf(v[b].w, v[b].w, ss[b]))));
            if (inb)
              store_b_at(bs + (c >> 7) * 4096, b, c & 127,
                         make_float4(v[b].x * g0, v[b].y * g1, v[b].z * g2, v[b].w * g3));
          }
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const float tt = warp_sum(ss[b]);
          if (lane == 0) m->red[b * NCW + cw] = tt;
        }
      } else {
        // the attention output's columns [c0, c0 + nc) of every request
        const int KF = p.nq * p.d, n4 = nc >> 2;
        const float* o = p.o + (size_t)l * p.bcap * KF + c0;
        for (int x = ct; x < 8 * n4; x += NCT) {
          const int b = x / n4, i = x - b * n4;
          const float4 y = b < B ? __ldcg(reinterpret_cast<const float4*>(o + (size_t)b * KF) + i) : z4;
          store_b_at(bs + (i >> 5) * 4096, b, (4 * i) & 127, y);
        }
        // every attention task of the layer is done: clear this task's share of the QKV sums
        const long long n = (long long)B * p.qkv_rows;
        unsigned long long* qs = p.qkv_fx + (size_t)l * p.bcap * p.qkv_rows;
        for (long long i = n * t.a[2] / t.a[5] + ct; i < n * (t.a[2] + 1) / t.a[5]; i += NCT) qs[i] = 0ull;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // read by the tensor cores
    }
    cbar();
    if (isq && !ab && ct < B) {
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; ++w) tot += m->red[ct * NCW + w];
      m->inv[ct] = 1.0f / sqrtf(tot / (float)p.H + p.eps);
    }
    mark(TR_ACT);
    const uint32_t bsm = smem_u32(bs), tmem = m->tmem;
    for (int j = 0; j < nu; ++j) {
      const uint8_t* st = wait_stage(ab);
      if (cw == 0) {
        if (lane == 0) {
          if (st) {
            tc_fence_after();
            const uint32_t sa = smem_u32(st);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_f16(tmem, umma_desc_sw128(sa + h * TC_BOX + kk * 32),
                         umma_desc_sw128(bsm + j * 4096 + h * 2048 + kk * 32), UMMA_IDESC_M128_N16,
                         (j | h | kk) != 0);
            umma_commit(&m->empty[r.stage]);   // the stage is free once its MMAs are done
            if (j == nu - 1) umma_commit(&m->acc_bar);
          } else {
            mbar_arrive(&m->empty[r.stage]);
          }
        }
        __syncwarp();
        if (p.strace && ct == 0) stage_stamp(2);
        r.advance();
      } else {
        release_stage(ab);
      }
    }
    const uint8_t* rst = isq ? nullptr : wait_stage(ab);   // the O task's router rows [128][E] bf16
    ab = cbar_or(ab);
    float* vb = psum;   // O: [128 rows][8 requests] part * gain, the router share's input
    if (!ab && cw < 4) {
      const int r = cw * 32 + lane, row = row0 + r;
      float xr[8];   // the residual's loads go out before the accumulator wait
#pragma unroll
      for (int b = 0; b < 8; ++b) xr[b] = !isq && ks0 == 0 && b < B ? x_in(l, b, row) : 0.f;
      if (!mbar_wait(p, m, &m->acc_bar, acc_ph, -7)) ab = true;
      tc_fence_after();
      float v[16];
      tmem_ld16(tmem + ((uint32_t)(cw * 32) << 16), v);
      if (isq) {
        unsigned long long* out = p.qkv_fx + (size_t)l * p.bcap * p.qkv_rows + row;
#pragma unroll
        for (int b = 0; b < 8; ++b)
          if (!ab && b < B) atomicAdd(out + (size_t)b * p.qkv_rows, to_fixed<NB == 8>((v[b] + v[8 + b]) * m->inv[b]));
      } else {
        const float gn = bf2f(p.ffn_norm[l][row]);
        unsigned long long* out = p.xmid_fx + (size_t)l * p.bcap * p.H + row;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const float x = v[b] + v[8 + b] + xr[b];
          if (!ab && b < B) atomicAdd(out + (size_t)b * p.H, to_fixed<NB == 8>(x));
          vb[r * 8 + b] = b < B ? x * gn : 0.f;
        }
      }
    }
    acc_ph ^= 1;
    tc_fence_before();
    ab = cbar_or(ab);   // the accumulator is read before the next task's MMAs overwrite it
    if (!isq) {
      if (!ab && rst) {
        // router share: thread (request half bh, expert e) over the tile's 128 rows
        const uint16_t* wr = reinterpret_cast<const uint16_t*>(rst);
        const int E = p.E;
        unsigned long long* out = p.rlsum + ((size_t)l * RL_COPIES + t.a[2] % RLC) * p.bcap * E;
        for (int x = ct; x < 2 * E; x += NCT) {
          const int bh = x / E, e = x - bh * E;
          if (4 * bh < B) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
            for (int r = 0; r < 128; ++r) {
              const float w = bf2f(wr[r * E + e]);
              const float4 xv = *reinterpret_cast<const float4*>(vb + r * 8 + 4 * bh);
              a0 = fmaf(w, xv.x, a0);
              a1 = fmaf(w, xv.y, a1);
              a2 = fmaf(w, xv.z, a2);
              a3 = fmaf(w, xv.w, a3);
            }
            const float a[4] = {a0, a1, a2, a3};
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (4 * bh + q < B) atomicAdd(out + (size_t)(4 * bh + q) * E + e, to_fixed<NB == 8>(a[q]));
          }
        }
      }
      release_stage(ab);
      // the tile's last task (a ticket over its t.a[6] tasks) turns its rows'
      // sums into fp32 x_mid for the expert tiles and the reduce, and clears them
      ab = cbar_or(ab);
      if (!ab && ticket(p.cm.omt + l * p.cm.nomt + row0 / 128, (uint32_t)t.a[6], 1u)) {
        unsigned long long* fx = p.xmid_fx + (size_t)l * p.bcap * p.H + row0;
        float* xm = p.x_mid + (size_t)l * p.bcap * p.H + row0;
        for (int i = ct; i < B * 128; i += NCT) {
          const size_t off = (size_t)(i >> 7) * p.H + (i & 127);
          xm[off] = from_fixed<NB == 8>(__ldcg(fx + off));
          fx[off] = 0ull;
        }
      }
    }
    return ab;
  }

  // The gate/up part of an expert tile on the tensor cores (batch instance 8):
  // units [q0, q1) are whole 32-unit halves.  Two halves make a 128-row tile
  // (half hh in rows 64 hh ..) that streams through the ring as 128 x 128
  // stages; one thread issues M = 128, N = 16, K = 16 MMAs (A: the weight
  // tile, B: the batch's activations as bf16 hi + lo rows) accumulating in
  // TMEM, and commits each stage's release to the ring's empty barrier.  A
  // lone last half streams 64 x 256 stages, its rows of K box c above those of
  // box c + 1; an N = 32 MMA from B box c reads box c + 1 as B rows 16-31, so
  // TMEM holds the box-c partials in lanes 0-63, columns 0-15, and the box c + 1
  // partials in lanes 64-127, columns 16-31, added in the epilogue.  Warps 0-3
  // then read the accumulator (one TMEM lane per row), add the hi and lo
  // columns of each request, pair gate and up rows and write the SwiGLU
  // coefficients of the expert's token slots, as the CUDA-core epilogue does.
  uint32_t acc_ph = 0;
  __device__ bool gu_tc(int q0, int q1, bool ab, float* cf) {
    const int F = p.F, k = p.k, bc = p.rm.bcap;
    const int nbox = p.stage_bytes / TC_BOX, kst = p.H / (64 * nbox), nh = (q1 - q0) / TC_HALF;
    const int nfull = nh >> 1, nmt = nfull + (nh & 1);
    const uint32_t bsm = smem_u32(act), tmem = m->tmem;
    float* xs = psum;   // the lone half's lanes 64-127, [column][row], between the warps
    for (int mt = 0; mt < nmt; ++mt) {
      const bool lone = mt == nfull;
      const int ksn = lone ? kst >> 1 : kst;
      for (int ks = 0; ks < ksn; ++ks) {
        const uint8_t* st = wait_stage(ab);
        if (cw == 0) {
          if (lane == 0) {
            if (st) {
              tc_fence_after();
              const uint32_t sa = smem_u32(st);
              for (int h = 0; h < nbox; ++h) {
                const uint32_t bb = bsm + (lone ? 2 * (nbox * ks + h) : nbox * ks + h) * 2048;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  umma_f16(tmem, umma_desc_sw128(sa + h * TC_BOX + kk * 32), umma_desc_sw128(bb + kk * 32),
                           lone ? UMMA_IDESC_M128_N32 : UMMA_IDESC_M128_N16, (ks | h | kk) != 0);
              }
              umma_commit(&m->empty[r.stage]);   // the stage is free once its MMAs are done
              if (ks == ksn - 1) umma_commit(&m->acc_bar);
            } else {
              mbar_arrive(&m->empty[r.stage]);
            }
          }
          __syncwarp();
          if (p.strace && ct == 0) stage_stamp(2);
          r.advance();
        } else {
          release_stage(ab);
        }
      }
      ab = cbar_or(ab);
      if (lone) {
        if (!ab && (cw == 2 || cw == 3)) {
          if (!mbar_wait(p, m, &m->acc_bar, acc_ph, -6)) ab = true;
          tc_fence_after();
          float v[16];
          tmem_ld16(tmem + ((uint32_t)(cw * 32) << 16) + 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) xs[i * 64 + (cw - 2) * 32 + lane] = v[i];
        }
        ab = cbar_or(ab);
      }
      if (!ab && cw < (lone ? 2 : 4)) {
        if (!mbar_wait(p, m, &m->acc_bar, acc_ph, -6)) ab = true;
        tc_fence_after();
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(cw * 32) << 16), v);
        if (lone) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] += xs[i * 64 + cw * 32 + lane];
        }
        float gsum[8], usum[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) gsum[j] = v[j] + v[8 + j];   // hi + lo of request j
#pragma unroll
        for (int j = 0; j < 8; ++j) usum[j] = __shfl_down_sync(FULL, gsum[j], 1);   // the up row below
        // this lane's row: half 2 mt + cw / 2 of the range (the lone half: rows 0-63)
        const int qa = q0 + (2 * mt + (cw >> 1)) * TC_HALF, u = qa / F;
        if (!ab && (lane & 1) == 0) {
          const int f = qa - u * F + (((cw & 1) * 32 + lane) >> 1);
          const int nt = m->r_cnt[u];
          const int* toks = m->r_tok + u * bc;
          const int* ranks = m->r_rank + u * bc;
          for (int j = 0; j < nt; ++j) {
            const int tj = toks[j];
            float gs = 0.f, us = 0.f;
#pragma unroll
            for (int b = 0; b < 8; ++b)
              if (b == tj) {
                gs = gsum[b];
                us = usum[b];
              }
            const float c = m->inv[tj], g = c * gs;
            cf[(size_t)(u * F + f - q0) * bc + j] = m->gate[tj * k + ranks[j]] * (g / (1.0f + expf(-g)) * (c * us));
          }
        }
      }
      acc_ph ^= 1;
      tc_fence_before();
      ab = cbar_or(ab);   // the accumulator is read before the next tile's MMAs overwrite it
    }
    return ab;
  }

  __device__ bool moe(const Task& t, bool ab) {
    const int l = t.layer, H = p.H, F = p.F, k = p.k, bc = p.rm.bcap;
    int U = 0;
    if (!ab) {
      // Whether this task routes: read before the barrier below, while no
      // thread can have routed this layer yet, so every consumer thread
      // decides alike (batch-1 routing publishes the layer from warp 0
      // before any barrier, and a thread that skipped route_local would
      // meet its barriers out of step).
      const bool route = m->r_layer != step * p.L + l || t.a[0] == 0;
      moe_act(l);
      cbar();
      mark(TR_MID1);
      if (route) route_local(l, t.a[0] == 0);
      mark(TR_MID2);
      U = m->r_U;
    }
    cbar();
    mark(TR_ACT);
    long long g0, g1;
    gu_range_w<NB>(p, t, U, m->r_cnt, g0, g1);
    const int q0 = (int)g0, q1 = (int)g1;
    float* cf = scr;   // [unit - q0][token slot] coefficients
    bool tc = false;
    if constexpr (NB == 8) {
      tc = tc_layer(p, t, U);
      if (tc) {
        ab = gu_tc(q0, q1, ab, cf);
      } else if (p.tm_gu && !ab) {
        // this layer's blocks do not fit the coefficient scratch: the CUDA
        // cores take it, from fp32 activations in place of the B operand
        const int H4 = H >> 2;
        const uint2* gam = reinterpret_cast<const uint2*>(p.ffn_norm[l]);
        for (int x = ct; x < p.B * H4; x += NCT) {
          const int b = x / H4, i = x - b * H4;
          const float4 v = xmid4(l, b, i);
          const uint2 gb = __ldg(gam + i);
          reinterpret_cast<float4*>(act + (size_t)b * H)[i] =
              make_float4(v.x * bf_lo(gb.x), v.y * bf_hi(gb.x), v.z * bf_lo(gb.y), v.w * bf_hi(gb.y));
        }
        cbar();
      }
    }
    for (int q = tc ? q1 : q0; q < q1;) {
      const int u = q / F, fa = q - u * F, fb = min(F, q1 - u * F);
      const int nt = m->r_cnt[u];
      const int* toks = m->r_tok + u * bc;
      const int* ranks = m->r_rank + u * bc;
      GemvEpi e{};
      e.kind = GemvEpi::SWIGLU;
      e.out = cf;
      e.ld = bc;
      e.base = u * F - q0;
      e.k = k;
      e.toks = toks;
      e.ranks = ranks;
      e.gate_w = m->gate;
      e.inv = m->inv;
      ab = gemv<true, SP_MOE>(H, 2 * fa, 2 * fb, act, H, toks, nt, ab, e);
      q = (u + 1) * F;
    }
    cbar();   // coefficients complete; the activation region is free
    const int rpw = rows_per_stage(p, H);
    const bool col = ct * 8 < H;                 // this thread's 8 output columns
    const uint32_t coff = (uint32_t)ct * 16;
    float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // batch 1: request 0 in registers
    if constexpr (NB > 1) {                      // else: y per request in the activation region,
      if (col) {                                 // each thread owning its 8 columns of every row
        for (int b = 0; b < p.B; ++b) {
          float4* yb = reinterpret_cast<float4*>(act + (size_t)b * H) + 2 * ct;
          yb[0] = make_float4(0.f, 0.f, 0.f, 0.f);
          yb[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    for (int q = q0; q < q1;) {
      const int u = q / F, fa = q - u * F, fb = min(F, q1 - u * F);
      const int nt = m->r_cnt[u];
      const int* toks = m->r_tok + u * bc;
      for (int f0 = fa; f0 < fb; f0 += rpw) {
        const int n = min(rpw, fb - f0);
        const uint8_t* st = wait_stage(ab);
        if (st && col) {
          const uint32_t sts = smem_u32(st) + coff;
          const float* cu = cf + (size_t)(u * F + f0 - q0) * bc;
          if constexpr (NB > 1) {
            // every row of the stage is a unit of expert u, so all share its
            // token slots: up to 8 rows in registers, then each token's 8
            // output columns read and written once for all of them
            for (int i0 = 0; i0 < n; i0 += 8) {
              const int ni = min(8, n - i0);
              uint4 w8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                w8[i] = i < ni ? lds128(sts + (uint32_t)(i0 + i) * H * 2) : make_uint4(0, 0, 0, 0);
              for (int j = 0; j < nt; ++j) {
                float4* yb = reinterpret_cast<float4*>(act + (size_t)toks[j] * H) + 2 * ct;
                float4 a0 = yb[0], a1 = yb[1];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float c = i < ni ? cu[(i0 + i) * bc + j] : 0.f;
                  const uint4 w = w8[i];
                  a0.x = fmaf(c, bf_lo(w.x), a0.x);
                  a0.y = fmaf(c, bf_hi(w.x), a0.y);
                  a0.z = fmaf(c, bf_lo(w.y), a0.z);
                  a0.w = fmaf(c, bf_hi(w.y), a0.w);
                  a1.x = fmaf(c, bf_lo(w.z), a1.x);
                  a1.y = fmaf(c, bf_hi(w.z), a1.y);
                  a1.z = fmaf(c, bf_lo(w.w), a1.z);
                  a1.w = fmaf(c, bf_hi(w.w), a1.w);
                }
                yb[0] = a0;
                yb[1] = a1;
              }
            }
          } else {
            for (int i = 0; i < n; ++i) {
              const uint4 w = lds128(sts + (uint32_t)i * H * 2);
              const float c = cu[i * bc];
              y[0] = fmaf(c, bf_lo(w.x), y[0]);
              y[1] = fmaf(c, bf_hi(w.x), y[1]);
              y[2] = fmaf(c, bf_lo(w.y), y[2]);
              y[3] = fmaf(c, bf_hi(w.y), y[3]);
              y[4] = fmaf(c, bf_lo(w.z), y[4]);
              y[5] = fmaf(c, bf_hi(w.z), y[5]);
              y[6] = fmaf(c, bf_lo(w.w), y[6]);
              y[7] = fmaf(c, bf_hi(w.w), y[7]);
            }
          }
        }
        release_stage(ab);
      }
      q = (u + 1) * F;
    }
    mark(TR_STAGES);
    if (!ab && col) {
      float* part = p.moe_part + (size_t)t.a[0] * p.bcap * H;
      for (int b = 0; b < p.B; ++b) {
        float4* dst = reinterpret_cast<float4*>(part + (size_t)b * H) + 2 * ct;
        if constexpr (NB == 1) {
          dst[0] = make_float4(y[0], y[1], y[2], y[3]);
          dst[1] = make_float4(y[4], y[5], y[6], y[7]);
        } else {
          const float4* src = reinterpret_cast<const float4*>(act + (size_t)b * H) + 2 * ct;
          dst[0] = src[0];
          dst[1] = src[1];
        }
      }
    }
    if constexpr (NB > 1) {
      // the requests whose rows this partial holds (the others stay zero)
      if (!ab && ct == 0) {
        uint32_t rows = 0;
        for (int u = q0 / F; u * F < q1; ++u)
          for (int j = 0; j < m->r_cnt[u]; ++j) rows |= 1u << m->r_tok[u * bc + j];
        p.moe_mask[(size_t)l * t.a[1] + t.a[0]] = rows;
      }
    }
    ab = finish(ab);
    if (!ab) signal(p.cm.gu + l);
    return ab;
  }

  // ---- reduce: rows [a0, a1) of the hidden dim, x_out = x_mid + the a2 expert
  // tiles' partials, summed in tile order (strided chunks, then chunk order)
  __device__ bool red(const Task& t, bool ab) {
    const int l = t.layer, r0 = t.a[0], nr = t.a[1] - r0, ntiles = t.a[2], B = p.B, H = p.H;
    const int no = B * nr;
    const int nch = no > 0 ? max(1, NCT / no) : 1;
    float* rs = act;                                   // [output][chunk] sums
    mark(TR_ACT);
    if (!ab) {   // every expert tile of the layer has read the router sums: zero this task's share
      const long long n = (long long)RLC * p.bcap * p.E;   // the copies in use, at the front
      unsigned long long* rs = p.rlsum + (size_t)l * RL_COPIES * p.bcap * p.E;
      for (long long i = r0 * n / H + ct; i < (long long)t.a[1] * n / H; i += NCT) rs[i] = 0ull;
    }
    // the residual rows first: their load overlaps the partials' (thread o < no keeps row o)
    const float xres = !ab && ct < no ? xmid1(l, ct / nr, r0 + ct % nr) : 0.f;
    if constexpr (NB > 1) {
      // above batch 1 a request's row is nonzero only in the partials of the
      // tiles serving its experts: warp b lists request b's tiles, in tile
      // order, from the tiles' masks, and only those are summed (strided
      // chunks of the list, then chunk order).  When the lists do not fit
      // beside the chunk sums (very few CTAs), every tile is summed.
      int* tl = reinterpret_cast<int*>(rs + no * nch);   // [B][ntiles] tile lists
      int* tn = tl + B * ntiles;                         // [B] their lengths
      uint32_t* msk = reinterpret_cast<uint32_t*>(tn + MAX_BATCH);
      const bool lists = (long long)no * nch + (long long)(B + 1) * ntiles + MAX_BATCH <= p.act_floats;
      if (lists) {
        if (!ab)
          for (int i = ct; i < ntiles; i += NCT) msk[i] = __ldcg(p.moe_mask + (size_t)l * ntiles + i);
        cbar();
        if (!ab && cw < B) {
          int base = 0;
          for (int i0 = 0; i0 < ntiles; i0 += 32) {
            const int i = i0 + lane;
            const bool on = i < ntiles && ((msk[i] >> cw) & 1u);
            const unsigned bal = __ballot_sync(FULL, on);
            if (on) tl[cw * ntiles + base + __popc(bal & ((1u << lane) - 1u))] = i;
            base += __popc(bal);
          }
          if (lane == 0) tn[cw] = base;
        }
        cbar();
      }
      if (!ab) {
        constexpr int BT = 10;
        for (int x = ct; x < no * nch; x += NCT) {
          const int c = x / no, o = x - c * no, b = o / nr, h = r0 + (o - b * nr);
          const float* src = p.moe_part + (size_t)b * H + h;
          const int* lb = lists ? tl + b * ntiles : nullptr;
          const int nb = lists ? tn[b] : ntiles;
          float s = 0.f;
          for (int k0 = c; k0 < nb; k0 += BT * nch) {
            float v[BT];
#pragma unroll
            for (int i = 0; i < BT; ++i) {
              const int kk = k0 + i * nch;
              v[i] = kk < nb ? __ldcg(src + (size_t)(lb ? lb[kk] : kk) * p.bcap * H) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < BT; ++i) s += v[i];
          }
          rs[o * nch + c] = s;
        }
      }
    } else if (!ab) {
      // thread x takes output o = x % no and every nch-th tile from chunk c = x / no,
      // so a warp reads consecutive rows of a tile; up to BT loads in flight
      constexpr int BT = 10;
      for (int x = ct; x < no * nch; x += NCT) {
        const int c = x / no, o = x - c * no, b = o / nr, h = r0 + (o - b * nr);
        const float* src = p.moe_part + (size_t)b * H + h;
        float s = 0.f;
        for (int t0 = c; t0 < ntiles; t0 += BT * nch) {
          float v[BT];
#pragma unroll
          for (int i = 0; i < BT; ++i) {
            const int ti = t0 + i * nch;
            v[i] = ti < ntiles ? __ldcg(src + (size_t)ti * p.bcap * H) : 0.f;
          }
#pragma unroll
          for (int i = 0; i < BT; ++i) s += v[i];
        }
        rs[o * nch + c] = s;
      }
    }
    cbar();
    if (!ab) {
      float* xo = p.x_out + (size_t)l * p.bcap * H;
      for (int o = ct; o < no; o += NCT) {
        const int b = o / nr, h = r0 + (o - b * nr);
        float s = o == ct ? xres : xmid1(l, b, h);
        for (int c = 0; c < nch; ++c) s += rs[o * nch + c];
        xo[(size_t)b * H + h] = s;
      }
    }
    mark(TR_STAGES);
    ab = finish(ab);
    if (!ab) signal(p.cm.down + l);
    return ab;
  }


  // ---- split-KV attention chunk on tensor cores (mma.sync m16n8k16, bf16 in, fp32 acc)
  // Pages hold K and V transposed ([d][16 slots]).  Per page (16 tokens):
  //   S  [16 tok x 8 heads] = K [tok x d] . Q^T            (A = K via ldmatrix.trans, B = q regs)
  //   O^T[16 dim x 8 heads] += V^T [dim x tok] . P^T       (A = V^T via ldmatrix, B = P via smem)
  // q and P enter as bf16 hi + lo pairs (two MMAs each), so the products keep
  // close to fp32 accuracy; K and V are exact bf16.  The warps of a stage take
  // its pages (NCW / pages-per-stage warps per page, splitting the d/16 output
  // row tiles); each page group keeps its own online-softmax state, merged at
  // the end of the chunk into one partial; the combine tasks merge the chunks.
  __device__ bool attn(const Task& t, bool ab) {
    const int l = t.layer, b = t.a[0], g = t.a[1];
    const int G = p.G, d = p.d, half = d >> 1;
    constexpr int PS = 16;                         // page size (tokens)
    const int pos = __ldcg(p.seq_len + b) + step;
    int tok0, tok1;
    attn_range(p, t, pos, tok0, tok1);
    const int RS = d + 4;                          // partial row: acc[d], m, l, pad (16-byte rows)
    float* q_s = act;                              // [MAX_G][d] rotated, scaled q
    float* kn_s = q_s + MAX_G * d;                 // new token's key (bf16 values)
    float* vn_s = kn_s + d;
    float* mrg = vn_s + d;                         // [groups][G][RS]
    uint32_t* pscr = reinterpret_cast<uint32_t*>(mrg + p.attn_mrg_floats);   // [NCW][2][8][8] packed P
    const size_t qo = ((size_t)l * p.bcap + b) * p.qkv_rows + (size_t)g * (G + 2) * d;   // this group's q rows
    const float2* rope = p.rope + (size_t)pos * half;
    const float qscale = 1.4426950408889634f / sqrtf((float)d);  // log2(e)/sqrt(d): exp2 softmax
    const bool has_new = pos >= tok0 && pos < tok1;
    // a prefill row also sees the earlier rows of its chunk: their tokens sit
    // at positions [pos - nprev, pos) of the same pages, written by their own
    // attention tasks of this step, so their K (rotated at its position) and V
    // are patched into the stages here from the QKV outputs, like the row's own
    const int nprev = p.chunk0 ? b - __ldcg(p.chunk0 + b) : 0;
    const int pq0 = max(tok0, pos - nprev), pq1 = min(tok1, pos + 1);   // patched positions
    const size_t qro = (size_t)l * p.bcap * p.qkv_rows + (size_t)g * (G + 2) * d + (size_t)G * d;   // row 0's k
    if (!ab) {
      for (int idx = ct; idx < MAX_G * half; idx += NCT) {
        const int h = idx / half, i = idx - h * half;
        float qa = 0.f, qb = 0.f;
        if (h < G) {
          const float2 cs = rope[i];
          const float a = qkv_at(qo + h * d + i), c = qkv_at(qo + h * d + i + half);
          qa = (a * cs.x - c * cs.y) * qscale;
          qb = (c * cs.x + a * cs.y) * qscale;
        }
        q_s[h * d + i] = qa;
        q_s[h * d + i + half] = qb;
      }
      if (has_new) {
        const size_t kr = qo + (size_t)G * d, vr = kr + d;
        const size_t base =
            ((size_t)p.page_table[(size_t)b * p.max_pages + pos / PS] * p.nkv + g) * 2 * d * PS + pos % PS;
        uint16_t* kd = p.kv_pool[l] + base;
        uint16_t* vd = kd + (size_t)d * PS;
        for (int i = ct; i < half; i += NCT) {
          const float2 cs = rope[i];
          const float a = qkv_at(kr + i), c = qkv_at(kr + i + half);
          const uint16_t k0 = f2bf(a * cs.x - c * cs.y), k1 = f2bf(c * cs.x + a * cs.y);
          kd[(size_t)i * PS] = k0;
          kd[(size_t)(i + half) * PS] = k1;
          kn_s[i] = bf2f(k0);
          kn_s[i + half] = bf2f(k1);
        }
        for (int i = ct; i < d; i += NCT) {
          const uint16_t v0 = f2bf(qkv_at(vr + i));
          vd[(size_t)i * PS] = v0;
          vn_s[i] = bf2f(v0);
        }
      }
    }
    cbar();
    mark(TR_ACT);
    const int gq = lane >> 2, tq = lane & 3;       // mma fragment coordinates
    const int nks = d >> 4;                        // 16-dim k steps (QK) = 16-dim row tiles (PV)
    // B fragments of Q^T per k step and lane (rows (dims) 2tq, 2tq+1 and +8,
    // column (head) gq), as bf16 hi + lo pairs, in a shared table: one
    // 16-byte read per k step instead of 32 registers held across the chunk
    // the table takes the place of q_s (d/16 k steps x 32 lanes x 16 bytes =
    // MAX_G * d floats): every thread reads its entry's q values first, then
    // all write after a barrier
    static_assert(NCT == 8 * 32, "one table entry per consumer thread");
    uint4* qtab = reinterpret_cast<uint4*>(q_s);   // [8 k steps][32 lanes]
    {
      const int ks = ct >> 5, L = ct & 31, gqL = L >> 2, tqL = L & 3;
      uint32_t w[4];
#pragma unroll
      for (int hfi = 0; hfi < 2; ++hfi) {
        float x0 = 0.f, x1 = 0.f;
        if (ks < nks) {
          x0 = q_s[gqL * d + ks * 16 + hfi * 8 + 2 * tqL];
          x1 = q_s[gqL * d + ks * 16 + hfi * 8 + 2 * tqL + 1];
        }
        const uint16_t h0 = f2bf(x0), h1 = f2bf(x1);
        w[hfi] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        w[2 + hfi] = (uint32_t)f2bf(x0 - bf2f(h0)) | ((uint32_t)f2bf(x1 - bf2f(h1)) << 16);
      }
      cbar();
      if (ks < nks) qtab[ct] = make_uint4(w[0], w[1], w[2], w[3]);   // nks * 32 entries = MAX_G * d floats
    }
    cbar();
    const uint32_t qtab_lane = smem_u32(qtab) + (uint32_t)lane * 16;
    const int ppg = pages_per_stage(p);
    const int npar = NCW / ppg;                    // stages in flight: warp (par, grp) takes page
    const int par = cw / ppg, grp = cw - par * ppg;  // grp of every npar-th stage, starting at par
    const int mtw = nks;                           // output row tiles per warp (all of d)
    const uint32_t PB = (uint32_t)d * PS * 2;      // bytes of one page block
    // online-softmax state of heads 2tq, 2tq+1 (identical across gq) and O^T tiles
    float mr0 = -INFINITY, mr1 = -INFINITY, lr0 = 0.f, lr1 = 0.f;
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[i][j] = 0.f;
    uint32_t* myp = pscr + cw * 2 * 64;            // this warp's packed P^T: [hi/lo][head 8][tok/2 8]
    const int pg0 = tok0 / PS, pg1 = (tok1 + PS - 1) / PS;
    int si = 0;                                    // stage index within the chunk
    for (int pg = pg0; pg < pg1; pg += ppg, ++si) {
      const int npg = min(ppg, pg1 - pg);
      const bool own = has_new && pos / PS >= pg && pos / PS < pg + npg;
      const bool patch = own || (nprev > 0 && pq0 < pq1 && pq0 / PS < pg + npg && (pq1 - 1) / PS >= pg);
      // the stage belongs to one warp group (its ppg pages, one per warp): only
      // that group waits for and releases it, each warp arriving npar times;
      // every warp waits for a stage it helps patch
      const bool mine = si % npar == par;
      const uint8_t* st = mine || patch ? wait_stage(ab) : nullptr;
      if (st && patch) {
        // put the new token's K and V into its stage slot before anyone reads the
        // page, and zero the page's later slots: they hold no token yet, and
        // although their scores are masked, their V still enters the P.V product
        // (0 * NaN would poison the output)
        cbar();
        if (own) {
          const int pi = pos / PS - pg, slot = pos % PS;
          uint16_t* kp = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(st) + (size_t)pi * 2 * PB);
          uint16_t* vp = kp + (size_t)d * PS;
          for (int i = ct; i < d * PS; i += NCT) {
            const int dim = i / PS, sl = i - dim * PS;
            if (sl == slot) {
              kp[i] = f2bf(kn_s[dim]);
              vp[i] = f2bf(vn_s[dim]);
            } else if (sl > slot) {
              kp[i] = 0;
              vp[i] = 0;
            }
          }
        }
        if (nprev > 0) {
          // the chunk's earlier rows at positions [pq0, min(pq1, pos)) of this stage's pages
          const int qa = max(pq0, pg * PS), qb = min(min(pq1, pos), (pg + npg) * PS);
          for (int i = ct; i < (qb - qa) * d; i += NCT) {
            const int q = qa + i / d, dim = i - (i / d) * d;
            const int pi = q / PS - pg, sl = q % PS;
            uint16_t* kp = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(st) + (size_t)pi * 2 * PB);
            uint16_t* vp = kp + (size_t)d * PS;
            const size_t kr = qro + (size_t)(b - (pos - q)) * p.qkv_rows;   // row b - (pos - q)
            const int i0 = dim < half ? dim : dim - half;
            const float2 cs = p.rope[(size_t)q * half + i0];
            const float a = qkv_at(kr + i0), c = qkv_at(kr + i0 + half);
            kp[dim * PS + sl] = f2bf(dim < half ? a * cs.x - c * cs.y : c * cs.x + a * cs.y);
            vp[dim * PS + sl] = f2bf(qkv_at(kr + d + dim));
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        cbar();
      } else if (patch) {
        cbar();
        cbar();
      }
      if (st && mine && grp < npg) {
        const int P = pg + grp;                    // global page index of this warp's page
        const int nvalid = min(PS, tok1 - P * PS); // tokens of the page inside the chunk
        const uint32_t kpage = smem_u32(st) + grp * 2 * PB;   // the page's K block, then its V block
        const uint32_t vpage = kpage + PB;
        // S = K . Q^T : A tiles of K^T-stored rows via ldmatrix.trans
        float s[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
        const int li = lane >> 3, lr = lane & 7;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          if (ks < nks) {
            const uint32_t addr = kpage + (uint32_t)((ks * 16 + (li >> 1) * 8 + lr) * PS * 2 + (li & 1) * 16);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(addr, a0, a1, a2, a3);
            const uint4 qf = lds128(qtab_lane + (uint32_t)ks * 512);
            mma_bf16(s, a0, a1, a2, a3, qf.x, qf.y);
            mma_bf16(sl, a0, a1, a2, a3, qf.z, qf.w);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) s[e] += sl[e];
        // s[0]: (tok gq, head 2tq) s[1]: (tok gq, head 2tq+1) s[2]/s[3]: tok gq+8
        if (gq >= nvalid) { s[0] = -INFINITY; s[1] = -INFINITY; }
        if (gq + 8 >= nvalid) { s[2] = -INFINITY; s[3] = -INFINITY; }
        float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(FULL, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(FULL, mx1, off));
        }
        const float mn0 = fmaxf(mr0, mx0), mn1 = fmaxf(mr1, mx1);
        const float sc0 = exp2f(mr0 - mn0), sc1 = exp2f(mr1 - mn1);   // 0 on the first page
        const float p0 = exp2f(s[0] - mn0), p1 = exp2f(s[1] - mn1);
        const float p2 = exp2f(s[2] - mn0), p3 = exp2f(s[3] - mn1);
        float ps0 = p0 + p2, ps1 = p1 + p3;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          ps0 += __shfl_xor_sync(FULL, ps0, off);
          ps1 += __shfl_xor_sync(FULL, ps1, off);
        }
        lr0 = lr0 * sc0 + ps0;
        lr1 = lr1 * sc1 + ps1;
        mr0 = mn0;
        mr1 = mn1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][0] *= sc0; o[mt][1] *= sc1; o[mt][2] *= sc0; o[mt][3] *= sc1;
        }
        // P^T as mma B operand: element (tok k, head n) packed per token pair;
        // store [hi/lo][head][tok/2] as bf16x2 words
        __syncwarp();
        {
          uint16_t* ph = reinterpret_cast<uint16_t*>(myp);
          uint16_t* pl = reinterpret_cast<uint16_t*>(myp + 64);
          const float pv[4] = {p0, p1, p2, p3};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int head = 2 * tq + (e & 1), tok = gq + 8 * (e >> 1);
            const uint16_t hb = f2bf(pv[e]);
            ph[head * 16 + tok] = hb;
            pl[head * 16 + tok] = f2bf(pv[e] - bf2f(hb));
          }
        }
        __syncwarp();
        const uint32_t bh0 = myp[gq * 8 + tq], bh1 = myp[gq * 8 + tq + 4];
        const uint32_t bl0 = myp[64 + gq * 8 + tq], bl1 = myp[64 + gq * 8 + tq + 4];
        // O^T += V^T . P^T over all d/16 row tiles (dims)
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          if (mt < mtw) {
            const int m0 = mt * 16;
            const uint32_t addr = vpage + (uint32_t)((m0 + (li & 1) * 8 + lr) * PS * 2 + (li >> 1) * 16);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(addr, a0, a1, a2, a3);
            mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
            mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
          }
        }
      }
      if (mine)
        release_stage_n(ab, npar);
      else
        r.advance();
    }
    mark(TR_STAGES);
    // merge the warps' partial softmax states of this chunk (a warp that saw
    // no page keeps max -inf and drops out)
    if (!ab) {
      if (gq == 0) {
        if (2 * tq < G) {
          mrg[(cw * G + 2 * tq) * RS + d] = mr0;
          mrg[(cw * G + 2 * tq) * RS + d + 1] = lr0;
        }
        if (2 * tq + 1 < G) {
          mrg[(cw * G + 2 * tq + 1) * RS + d] = mr1;
          mrg[(cw * G + 2 * tq + 1) * RS + d + 1] = lr1;
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        if (mt < mtw) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int head = 2 * tq + (e & 1), dim = mt * 16 + gq + 8 * (e >> 1);
            if (head < G) mrg[(cw * G + head) * RS + dim] = o[mt][e];
          }
        }
      }
    }
    ab = cbar_or(ab);
    if (ab) return ab;
    const int nslots = p.part_slots;
    float* part = p.part + ((size_t)l * nslots + t.a[4]) * G * RS;
    // per head: the chunk max, normaliser and each warp's weight, once
    float* fw = reinterpret_cast<float*>(pscr);    // [NCW][G] weights (P scratch is free now)
    static_assert(NCW == 8 && MAX_G * NCW <= NCT, "eight lanes per head, one per warp state");
    if (ct < MAX_G * NCW) {   // lanes 8h .. 8h + 7: head h, warp state w (butterflies within the 8)
      const int h = ct >> 3, w = ct & 7;
      const bool hv = h < G;
      const float mw = hv ? mrg[(w * G + h) * RS + d] : -INFINITY;
      float M = mw;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
      float Ls = hv ? mrg[(w * G + h) * RS + d + 1] * f : 0.f;
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) Ls += __shfl_xor_sync(FULL, Ls, o);
      if (hv) {
        fw[w * G + h] = f;
        if (w == 0) {
          part[h * RS + d] = M;
          part[h * RS + d + 1] = Ls;
        }
      }
    }
    cbar();
    for (int idx = ct; idx < G * d; idx += NCT) {
      const int h = idx / d, i = idx - h * d;
      float A = 0.f;
#pragma unroll
      for (int w = 0; w < NCW; ++w) A = fmaf(mrg[(w * G + h) * RS + i], fw[w * G + h], A);
      part[h * RS + i] = A;
    }
    ab = finish(ab);
    if (!ab) signal(p.cm.attn_idx(l, b, g));
    return ab;
  }

  // ---- split-KV combine of query heads [a2, a2 + a3) of (request a0, KV group a1)
  // The chunks' partials (max m, normaliser l, accumulator acc[d], in exp2
  // units) merge by log-sum-exp.  Warp w takes chunks w, w + 8, ... in order
  // with an online (max, normaliser, accumulator) state, CB chunks per round
  // trip; the 8 warp states then merge in warp order, so the result does not
  // depend on timing.
  __device__ bool comb(const Task& t, bool ab) {
    constexpr int CB = 8;
    const int l = t.layer, b = t.a[0], g = t.a[1], h0 = t.a[2], nh = t.a[3], nc = t.a[6];
    const int G = p.G, d = p.d, RS = d + 4, d4 = d >> 2;
    const float* part = p.part + ((size_t)l * p.part_slots + t.a[5]) * G * RS;
    float* o = p.o + ((size_t)l * p.bcap + b) * p.nq * d + (size_t)g * G * d;
    float* ws = act;                                   // [NCW][d + 4]: accumulator, max, normaliser
    const bool has = lane < d4;                        // this lane's 4 dims
    mark(TR_ACT);
    for (int hh = 0; hh < nh && !ab; ++hh) {
      const int h = h0 + hh;
      float M = -INFINITY, Ls = 0.f;
      float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c0 = cw; c0 < nc; c0 += NCW * CB) {
        float4 v[CB];
        float2 ml[CB];
#pragma unroll
        for (int q = 0; q < CB; ++q) {
          const int c = c0 + q * NCW;
          if (c < nc) {
            const float* pc = part + ((size_t)c * G + h) * RS;
            ml[q] = __ldcg(reinterpret_cast<const float2*>(pc + d));
            v[q] = has ? __ldcg(reinterpret_cast<const float4*>(pc) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int q = 0; q < CB; ++q) {
          if (c0 + q * NCW < nc) {
            const float mn = fmaxf(M, ml[q].x);
            const float fo = exp2f(M - mn), fn = exp2f(ml[q].x - mn);   // fo = 0 while M = -inf
            A.x = fmaf(v[q].x, fn, A.x * fo);
            A.y = fmaf(v[q].y, fn, A.y * fo);
            A.z = fmaf(v[q].z, fn, A.z * fo);
            A.w = fmaf(v[q].w, fn, A.w * fo);
            Ls = fmaf(ml[q].y, fn, Ls * fo);
            M = mn;
          }
        }
      }
      float* mine = ws + cw * RS;
      if (has) reinterpret_cast<float4*>(mine)[lane] = A;
      if (lane == 0) {
        mine[d] = M;
        mine[d + 1] = Ls;
      }
      cbar();
      for (int i = ct; i < d; i += NCT) {
        float Mt = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) Mt = fmaxf(Mt, ws[w * RS + d]);
        float Lt = 0.f, At = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float mw = ws[w * RS + d];
          if (mw != -INFINITY) {
            const float f = exp2f(mw - Mt);
            Lt = fmaf(ws[w * RS + d + 1], f, Lt);
            At = fmaf(ws[w * RS + i], f, At);
          }
        }
        o[h * d + i] = At / Lt;
      }
      cbar();
    }
    mark(TR_STAGES);
    ab = finish(ab);
    if (!ab) signal(p.cm.combine + l);
    return ab;
  }

  // Nucleus (top-p) draw of request b = t.a[0] from the logits its LM tiles
  // kept.  Rows are ordered by logit, descending, the lower index first among
  // equal logits.  Each row's mass is w = exp((logit - max) / T) in float32,
  // held as the integer round(w * 2^32), so every sum below is exact and does
  // not depend on the order of the adds.  The nucleus is the shortest prefix
  // of the order whose mass reaches ceil(top_p * total).  It is found by a
  // radix search over a 32-bit key that sorts rows the same way (four 8-bit
  // digits, one pass over the logits each), then, for equal logits at the
  // cut, by index.  The token is the Gumbel-max draw of the temperature
  // sampler restricted to the nucleus: the argmax of logit / T + noise over it.
  __device__ static uint32_t desc_key(float l) {
    const uint32_t u = __float_as_uint(l + 0.0f);   // -0 -> +0
    return (u & 0x80000000u) ? u : (~u & 0x7fffffffu);
  }

  __device__ bool sample(const Task& t, bool ab) {
    if (ab) return ab;
    const int b = t.a[0], V = p.V, tiles = p.lm_tiles;
    const float* lg = p.lg_keep + (size_t)b * V;
    unsigned long long* hist = reinterpret_cast<unsigned long long*>(act);   // [256] masses
    unsigned int* hcnt = reinterpret_cast<unsigned int*>(hist + 256);       // [256] row counts
    unsigned long long* red = reinterpret_cast<unsigned long long*>(hcnt + 256);   // [NCT] scan / sums
    unsigned long long& s_tgt = m->smp_tgt;
    unsigned long long& s_before = m->smp_before;
    uint32_t& s_prefix = m->smp_prefix;
    int& s_digit = m->smp_digit;
    int& s_cut = m->smp_cut;
    float& s_max = m->smp_max;
    const int pos = __ldcg(p.seq_len + b) + step;
    const float it = p.inv_temp;
    // the largest logit, from the tiles' maxima
    if (cw == 0) {
      float v = -INFINITY;
      for (int i = lane; i < tiles; i += 32) v = fmaxf(v, __ldcg(p.lm_val + (size_t)b * tiles + i));
#pragma unroll
      for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
      if (lane == 0) s_max = v;
    }
    cbar();
    const float mx = s_max;
    auto mass = [&](float l) -> unsigned long long {
      return __float2ull_rn(expf((l - mx) * it) * 4294967296.0f);
    };
    // the total mass, then the target
    {
      unsigned long long z = 0;
      for (int v = ct; v < V; v += NCT) z += mass(__ldcg(lg + v));
      red[ct] = z;
      cbar();
      if (ct == 0) {
        unsigned long long tot = 0;
        for (int i = 0; i < NCT; ++i) tot += red[i];
        unsigned long long tg = (unsigned long long)ceil((double)p.top_p * (double)tot);
        s_tgt = tg < 1ull ? 1ull : (tg > tot ? tot : tg);
        s_before = 0;
        s_prefix = 0;
      }
      cbar();
    }
    // four digit passes: the digit where the running mass reaches the target
    for (int pass = 0; pass < 4; ++pass) {
      const int sh = 24 - 8 * pass;
      for (int i = ct; i < 256; i += NCT) {
        hist[i] = 0;
        hcnt[i] = 0;
      }
      cbar();
      const uint32_t pre = s_prefix;
      for (int v = ct; v < V; v += NCT) {
        const float l = __ldcg(lg + v);
        const uint32_t k = desc_key(l);
        if (pass > 0 && (k >> (sh + 8)) != pre) continue;
        const int dg = (k >> sh) & 0xff;
        atomicAdd(&hist[dg], mass(l));
        atomicAdd(&hcnt[dg], 1u);
      }
      cbar();
      if (cw == 0) {
        // lane i holds digits 8i .. 8i + 7; an exclusive scan over lanes finds the digit
        unsigned long long loc[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          loc[j] = hist[lane * 8 + j];
          sum += loc[j];
        }
        unsigned long long inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long y = __shfl_up_sync(FULL, inc, o);
          if (lane >= o) inc += y;
        }
        const unsigned long long before = s_before, tgt = s_tgt;
        unsigned long long run = before + inc - sum;   // mass of every digit below this lane's first
        int found = -1;
        unsigned long long found_before = 0;
        for (int j = 0; j < 8; ++j) {
          if (found < 0 && run + loc[j] >= tgt) {
            found = lane * 8 + j;
            found_before = run;
          }
          run += loc[j];
        }
        const unsigned ok = __ballot_sync(FULL, found >= 0);
        const int src = ok ? __ffs(ok) - 1 : 31;
        const int dsel = __shfl_sync(FULL, ok ? found : 255, src);
        const unsigned long long bsel = __shfl_sync(FULL, ok ? found_before : before, src);
        const unsigned long long all = __shfl_sync(FULL, inc, 31);   // this pass's whole mass
        if (lane == 0) {
          // the digits' masses always reach the target (they add up to the
          // digit chosen by the pass before); kept safe regardless: the last
          // occupied digit
          int d = dsel;
          unsigned long long bb = bsel;
          if (!ok) {
            d = 255;
            while (d > 0 && hcnt[d] == 0) --d;
            bb = before + all - hist[d];
          }
          s_digit = d;
          s_before = bb;
          s_prefix = (s_prefix << 8) | (uint32_t)d;
        }
      }
      cbar();
    }
    const uint32_t kcut = s_prefix;
    // equal logits at the cut: rows in index order until the target is reached
    int vcut = V;
    if (hcnt[s_digit] > 1) {
      const int per = (V + NCT - 1) / NCT, v0 = ct * per, v1 = min(V, v0 + per);
      unsigned long long mine = 0;
      for (int v = v0; v < v1; ++v) {
        const float l = __ldcg(lg + v);
        if (desc_key(l) == kcut) mine += mass(l);
      }
      red[ct] = mine;
      cbar();
      if (ct == 0) {
        unsigned long long run = s_before;
        int owner = NCT - 1;
        for (int i = 0; i < NCT; ++i) {
          if (run + red[i] >= s_tgt) { owner = i; break; }
          run += red[i];
        }
        s_cut = owner;
        red[NCT - 1] = run;   // mass before the owner's range (the owner reads it back)
      }
      cbar();
      if (ct == s_cut) {
        unsigned long long run = red[NCT - 1];
        int c = v1 - 1;
        for (int v = v0; v < v1; ++v) {
          const float l = __ldcg(lg + v);
          if (desc_key(l) != kcut) continue;
          run += mass(l);
          if (run >= s_tgt) { c = v; break; }
        }
        s_cut = c;
      }
      cbar();
      vcut = s_cut;
    }
    // the draw: argmax of the temperature keys over the nucleus
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int v = ct; v < V; v += NCT) {
      const float l = __ldcg(lg + v);
      const uint32_t k = desc_key(l);
      if (k > kcut || (k == kcut && v > vcut)) continue;
      const float sv = fmaf(l, it, gumbel_noise((uint32_t)v, (uint32_t)pos, (uint32_t)(p.slot0 + b), p.seed_lo,
                                                p.seed_hi));
      if (sv > bv || (sv == bv && v < bi)) { bv = sv; bi = v; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(FULL, bv, o);
      const int oi = __shfl_xor_sync(FULL, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) {
      m->best_v[cw] = bv;
      m->best_i[cw] = bi;
    }
    cbar();
    if (ct == 0) {
      float v = -INFINITY;
      int ix = 0x7fffffff;
      for (int w = 0; w < NCW; ++w)
        if (m->best_v[w] > v || (m->best_v[w] == v && m->best_i[w] < ix)) { v = m->best_v[w]; ix = m->best_i[w]; }
      p.next_token[(size_t)step * p.io_stride + b] = ix;
      if (step + 1 == p.nsteps) p.seq_len[b] = __ldcg(p.seq_len + b) + p.nsteps;
    }
    ab = finish(false);
    if (!ab) signal(p.cm.sdone);
    return ab;
  }

  // LM-head tile.  A CTA's LM tiles are the last tasks of its list: the first
  // fills the final norm's activations (kept by the later tiles), and only the
  // last takes the ticket, for all of this CTA's tiles at once.
  __device__ bool lm(const Task& t, bool ab, bool last) {
    const int L = p.L, B = p.B;
    if (!ab && lm_done == 0) {
      const float* xo = p.x_out + (size_t)(L - 1) * p.bcap * p.H;
      fill_rmsnorm(p.final_norm, [&](int b, int i4) {
        return __ldcg(reinterpret_cast<const float4*>(xo + (size_t)b * p.H) + i4);
      });
    }
    // nucleus sampling: this tile keeps its logits and finds their plain
    // maximum; the request's T_SAMPLE task draws from them afterwards
    const bool keep = NUC && p.lg_keep != nullptr;
    const bool sampled = p.inv_temp > 0.f && !keep;
    int* pos = reinterpret_cast<int*>(scr);   // each request's position: the noise counter
    if (sampled && ct < B) pos[ct] = __ldcg(p.seq_len + ct) + step;
    cbar();
    ++lm_done;
    mark(TR_ACT);
    // each thread keeps, per activation row, the best (value, lowest index) it saw
    float bv[NB];
    int bi[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      bv[j] = -INFINITY;
      bi[j] = 0x7fffffff;
    }
    float* lg = p.logits ? p.logits + (size_t)step * p.io_stride * p.V : nullptr;
    ab = gemv<false, SP_LM>(p.H, t.a[0], t.a[1], act, p.H, nullptr, B, ab, [&](int row, int j, float s0, float) {
      float s = m->inv[j] * s0;
      if (lg) lg[(size_t)j * p.V + row] = s;
      if (keep) p.lg_keep[(size_t)j * p.V + row] = s;
      if (sampled)   // Gumbel-max: the argmax of the perturbed, scaled logits is a draw from softmax(logits / T)
        s = fmaf(s, p.inv_temp,
                 gumbel_noise((uint32_t)row, (uint32_t)pos[j], (uint32_t)(p.slot0 + j), p.seed_lo, p.seed_hi));
#pragma unroll
      for (int jj = 0; jj < NB; ++jj)
        if (jj == j && (s > bv[jj] || (s == bv[jj] && row < bi[jj]))) {
          bv[jj] = s;
          bi[jj] = row;
        }
    });
    mark(TR_STAGES);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL, bv[j], o);
        const int oi = __shfl_xor_sync(FULL, bi[j], o);
        if (ov > bv[j] || (ov == bv[j] && oi < bi[j])) {
          bv[j] = ov;
          bi[j] = oi;
        }
      }
      if (!ab && lane == 0 && j < B) {
        m->best_v[cw * MAX_BATCH + j] = bv[j];
        m->best_i[cw * MAX_BATCH + j] = bi[j];
      }
    }
    ab = cbar_or(ab);
    if (ab) return ab;
    const int tiles = p.lm_tiles, tile = t.a[2];
    if (ct < B) {
      float v = -INFINITY;
      int ix = 0x7fffffff;
      for (int w = 0; w < NCW; ++w) {
        const float wv = m->best_v[w * MAX_BATCH + ct];
        const int wi = m->best_i[w * MAX_BATCH + ct];
        if (wv > v || (wv == v && wi < ix)) { v = wv; ix = wi; }
      }
      p.lm_val[(size_t)ct * tiles + tile] = v;
      p.lm_idx[(size_t)ct * tiles + tile] = ix;
    }
    if (!last) return ab;   // the last tile's barrier orders these writes before its ticket
    ab = finish(ab);
    if (ab) return ab;
    if (ticket(p.cm.lm, (uint32_t)t.a[3], (uint32_t)lm_done) && !keep) {
      if (cw < B) {
        const int b = cw;
        float v = -INFINITY;
        int ix = 0x7fffffff;
        for (int i = lane; i < tiles; i += 32) {
          const float tv = __ldcg(p.lm_val + (size_t)b * tiles + i);
          const int tix = __ldcg(p.lm_idx + (size_t)b * tiles + i);
          if (tv > v || (tv == v && tix < ix)) { v = tv; ix = tix; }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float ov = __shfl_xor_sync(FULL, v, o);
          const int oi = __shfl_xor_sync(FULL, ix, o);
          if (ov > v || (ov == v && oi < ix)) { v = ov; ix = oi; }
        }
        if (lane == 0) {
          p.next_token[(size_t)step * p.io_stride + b] = ix;
          // positions stay those of the launch's start until its last step is done
          if (step + 1 == p.nsteps) p.seq_len[b] = __ldcg(p.seq_len + b) + p.nsteps;
        }
      }
      ab = finish(false);
      if (!ab) signal(p.cm.sdone);   // the next step's first layer may read these tokens
    }
    return ab;
  }

  __device__ void run(int t0, int t1) {
    for (step = 0; step < p.nsteps; ++step) {
      epoch = p.epoch + (uint32_t)step;
      lm_done = 0;
      if (!run_step(t0, t1)) return;
    }
  }

  // One pass over this CTA's tasks for step `step`; false once a wait gave up.
  __device__ bool run_step(int t0, int t1) {
    for (ti = t0; ti < t1; ++ti) {
      const Task t = ldg_task(p.tasks + ti);
      if (ti + 1 < t1) prefetch_l1(p.tasks + ti + 1);   // the next record arrives while this task runs
      bool ab = false;
      nstage_seen = 0;
      mark(TR_FETCH);
      if (ct == 0) {
        // the first layer of a later step starts from the previous step's tokens
        if (t.wait_ctr < 0 && step > 0)
          ab = !wait_ctr(p, p.cm.sdone, epoch - 1u, (uint32_t)p.sdone_cnt, ti);
        else
          ab = !wait_ctr(p, t.wait_ctr, epoch, t.wait_cnt, ti);
      }
      ab = cbar_or(ab);
      if (ab) return false;
      mark(TR_DEP);
      switch (t.type) {
        case T_QKV:
        case T_OPROJ: {
          if constexpr (NB == 8) {
            if (p.tm_qkv) {   // tensor cores: one 128-row tile over a run of K stages
              ab = proj_tc(t, ab);
              mark(TR_STAGES);
              ab = finish(ab);
              if (!ab) signal(t.type == T_QKV ? p.cm.qkv + t.layer * p.nkv + t.a[2] : p.cm.o + t.layer);
              break;
            }
          }
          ProjGemv g;
          if constexpr (NB > 2) {   // the O projection may run in K halves
            const int parts = t.type == T_OPROJ ? p.o_halves : 1;
            for (int h = 0; h < parts; ++h) {
              ab = t.type == T_QKV ? prep_qkv(t, ab, g) : prep_oproj(t, ab, g, h);
              if (h == 0) mark(TR_ACT);
              ab = gemv<false, SP_PROJ>(g.K, g.r0, g.r1, act, g.K, nullptr, p.B, ab, g.epi);   // the one plain call site
            }
          } else {
            ab = t.type == T_QKV ? prep_qkv(t, ab, g) : prep_oproj(t, ab, g, 0);
            mark(TR_ACT);
            ab = gemv<false, SP_PROJ>(g.K, g.r0, g.r1, act, g.K, nullptr, p.B, ab, g.epi);   // the one plain call site
          }
          mark(TR_STAGES);
          ab = post_proj(t, ab);
          break;
        }
        case T_ATTN: ab = attn(t, ab); break;
        case T_MOE: ab = moe(t, ab); break;
        case T_RED: ab = red(t, ab); break;
        case T_LM:
          if constexpr (NUC)   // the draw tasks follow a CTA's LM tiles
            ab = lm(t, ab, ti + 1 == t1 || ldg_task(p.tasks + ti + 1).type != T_LM);
          else
            ab = lm(t, ab, ti + 1 == t1);
          break;
        case T_COMB: ab = comb(t, ab); break;
        case T_SAMPLE:
          if constexpr (NUC) ab = sample(t, ab);
          else ab = true;
          break;
        default: ab = true;
      }
      if (ab) return false;
      mark(TR_DONE);
    }
    return true;
  }
};

// Wait (bounded) for every bulk copy still in flight before the CTA exits.
__device__ void drain(const Params& p, Misc* m, int nst) {
  for (int s = 0; s < nst; ++s) {
    const int rd = m->armed[s];
    if (rd < 0) continue;
    const uint64_t t0 = gtimer();
    while (!mbar_try_wait(&m->full[s], rd & 1)) {
      if (gtimer() - t0 > p.timeout_ns) {
        set_error(p, MK_ERR_DEP_TIMEOUT, -1, -5);
        break;
      }
    }
  }
}

template <int NB, bool NUC>
__global__ void __launch_bounds__(NTHREADS, 1) mk_megakernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Misc* m = reinterpret_cast<Misc*>(smem + p.misc_off);
  float* act = reinterpret_cast<float*>(smem + p.act_off);
  float* scr = reinterpret_cast<float*>(smem + p.misc_off + sizeof(Misc));
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < p.nstages; ++s) {
      mbar_init(&m->full[s], 1);
      mbar_init(&m->empty[s], NCW);
      m->armed[s] = -1;
    }
    m->abort_flag = 0;
    m->r_layer = -1;
    m->dead = failed(p) ? 1 : 0;
    if constexpr (NB == 8) {
      if (p.tm_gu) {
        mbar_init(&m->acc_bar, 1);
        mbar_init(&m->tc_fin, 1);
      }
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if constexpr (NB == 8) {
    if (p.tm_gu && tid < 32) {   // consumer warp 0 holds 32 TMEM columns for the launch
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" ::"r"(smem_u32(&m->tmem))
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (NB == 8) tc_fence_after();
  if (!m->dead) {
    const int t0 = p.cta_start[blockIdx.x], t1 = p.cta_start[blockIdx.x + 1];
    Ring ring{smem, m, p.nstages, p.stage_bytes, 0, 0};
    if (tid >= NCT) {
      if (tid == NCT) {
        Producer<NB> pr{p, ring, evict_first_policy()};
        pr.run(t0, t1);
      }
    } else {
      Consumer<NB, NUC> c{p, ring, act, m, scr, reinterpret_cast<float*>(smem + p.psum_off), tid, tid >> 5,
                          tid & 31};
      c.run(t0, t1);
    }
  }
  __syncthreads();
  if (tid == 0) drain(p, m, p.nstages);
  if constexpr (NB == 8) {
  if (p.tm_gu && tid < 32) {
    // every MMA of the launch is complete before the TMEM columns go back
    if (tid == 0) {
      umma_commit(&m->tc_fin);
      const uint64_t t0 = gtimer();
      while (!mbar_try_wait(&m->tc_fin, 0))
        if (gtimer() - t0 > p.timeout_ns) {
          set_error(p, MK_ERR_DEP_TIMEOUT, -1, -7);
          break;
        }
    }
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" ::"r"(m->tmem) : "memory");
  }
  }
}

template <int NB, bool NUC>
cudaError_t set_smem_attr() {
  static bool done = false;
  if (done) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(mk_megakernel<NB, NUC>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
  if (e == cudaSuccess) done = true;
  return e;
}

template <int NB, bool NUC>
cudaError_t launch_nb(const Params& p, int grid, int smem, cudaStream_t st) {
  cudaError_t e = set_smem_attr<NB, NUC>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mk_megakernel<NB, NUC>, p);
}

template <int NB, bool NUC>
int occupancy(int smem) {
  if (set_smem_attr<NB, NUC>() != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mk_megakernel<NB, NUC>, NTHREADS, smem) != cudaSuccess) return 0;
  return n;
}

}  // namespace
}  // namespace mk
