/* mk.h — C ABI of the persistent MoE decode megakernel (libmk.so, sm_103a).
 *
 * One decode step of a pre-norm MoE transformer (RMSNorm, QKV projection with
 * RoPE, KV append into a paged cache, split-KV paged GQA attention, O
 * projection, softmax/top-k router, SwiGLU experts, LM head, greedy argmax or
 * a temperature draw)
 * runs as ONE persistent kernel: one CTA per SM walks a host-prepared list of
 * tile tasks, and counters in global memory say when a tile's inputs are
 * ready, so a tile starts as soon as its own inputs land while immutable
 * weights (and already-cached KV pages) stream in ahead of it.
 *   Source of the design: "Cohere Publishes One-Kernel Server for North Mini
 *   Code" — "One resident program, many small tasks" and "What the
 *   scheduling change is meant to avoid"; "Inside the Megakernel Serving
 *   Engine for North Mini Code" — architecture paragraph (task list per SM,
 *   counters in global memory, tile-level scheduling, weight prefetch).
 *
 * Conventions for every function:
 *   - returns MK_OK (0) or a negative MK_ERR_* code; never aborts the process;
 *   - "device" pointers are CUDA device (or managed) memory on the current
 *     device; "host" pointers are ordinary host memory;
 *   - the caller owns all weights, KV pools and input/output buffers; the
 *     plan owns its task lists, counters, per-layer activations and status;
 *   - all matrices are bf16, row-major [out, in]; activations are fp32.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mk_stream; /* a cudaStream_t; NULL = legacy default stream */

enum {
  MK_OK = 0,
  MK_ERR_INVALID = -1,      /* bad argument: dims, pointer, size or page table */
  MK_ERR_CUDA = -2,         /* a CUDA runtime call failed */
  MK_ERR_DEP_TIMEOUT = -3,  /* a bounded device wait on a dependency ran out */
  MK_ERR_CAPACITY = -4,     /* batch, pages or positions beyond what the plan holds */
  MK_ERR_UNSUPPORTED = -5   /* shape this build does not implement */
};

/* Model shape.  Requirements: n_q_heads % n_kv_heads == 0 with at most 8 query
 * heads per KV head; head_dim 64 or 128; hidden, expert_ffn and
 * n_q_heads*head_dim multiples of 8; top_k <= 8; top_k <= n_experts <= 256;
 * page_size == 16; batch <= 8. */
typedef struct mk_model_dims {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim;
  int n_experts, top_k, expert_ffn, vocab, page_size;
  float rms_eps, rope_theta;
} mk_model_dims;

/* Weight pointers (all device, bf16).  Per-layer entries are HOST arrays of
 * n_layers device pointers; the plan copies them at creation.
 *   embed       [vocab, hidden]          lm_head   [vocab, hidden]
 *   final_norm  [hidden]
 *   attn_norm[l], ffn_norm[l]            [hidden]
 *   wqkv[l]     [n_kv_heads * (G + 2) * head_dim, hidden], G = n_q/n_kv,
 *               rows grouped per KV head g: the G query heads of group g
 *               (G*head_dim rows), then key head g, then value head g
 *   wo[l]       [hidden, n_q_heads * head_dim]
 *   router[l]   [hidden, n_experts]: the router stored transposed, row h =
 *               the n_experts weights of hidden unit h (W_router[:, h]), so
 *               an O-projection tile reads the router rows of its own hidden
 *               rows contiguously (n_experts must be a multiple of 4)
 *   w_gate_up[l][n_experts, 2*expert_ffn, hidden]: rows interleaved per ffn
 *               unit f: row 2f = gate row f, row 2f+1 = up row f
 *   w_down[l]   [n_experts, expert_ffn, hidden]: the down projection stored
 *               transposed per expert, row f = the hidden-size column of ffn
 *               unit f (W_down[e][:, f]), so an expert tile reads the down
 *               weights of its ffn units as contiguous rows
 * Every pointer must be 16-byte aligned. */
typedef struct mk_weights {
  const void* embed;
  const void* final_norm;
  const void* lm_head;
  const void* const* attn_norm;
  const void* const* wqkv;
  const void* const* wo;
  const void* const* ffn_norm;
  const void* const* router;
  const void* const* w_gate_up;
  const void* const* w_down;
} mk_weights;

/* Paged KV cache: per layer one pool (a HOST array of n_layers device
 * pointers), bf16 [num_pages, n_kv_heads, 2, head_dim, page_size]: for each
 * page and KV head its K block, then its V block, each holding the page's
 * tokens' vectors transposed (one row of page_size slots per dimension).  A
 * (page, head) is one contiguous 2 * head_dim * page_size * 2-byte copy for
 * the attention tiles, and the transposed blocks keep their tensor-core
 * operand loads nearly free of shared-memory bank conflicts.  Token t of
 * request b lives in page page_table[b][t / page_size], slot t % page_size.
 * 16-byte aligned. */
typedef struct mk_kv {
  void* const* kv_pool;
  int num_pages;
} mk_kv;

/* Plan options; zero-initialise for defaults. */
typedef struct mk_plan_opts {
  int timeout_us;    /* limit of every device spin-wait; 0 -> 2,000,000 us */
  int num_ctas;      /* persistent CTAs; 0 -> one per SM */
  int max_batch;     /* batch capacity for mk_plan_update; 0 -> batch.  Above 8 the plan
                        is a group of sub-plans of at most 8 requests each (requests
                        8i .. 8i + 7 in sub-plan i); a step runs one megakernel launch
                        per sub-plan that holds requests, one after another on the
                        stream, and each launch streams the weights it needs */
  int split_pages;   /* KV pages per attention task; 0 -> balance over the CTAs */
  int debug_drop_task; /* test hook: >0 removes task (value-1) from the list so its
                          counter never fires and the step returns MK_ERR_DEP_TIMEOUT;
                          0 in production */
  int trace;         /* 1: record a per-task timeline every step (MK_DBG_TRACE); 2: also a
                        per-stage timeline (MK_DBG_STAGE_TRACE) */
  float temperature; /* sampling from the first step, as mk_plan_set_sampling; 0 -> greedy */
  unsigned long long seed;
  float top_p;       /* nucleus sampling from the first step, as mk_plan_set_top_p; 0 -> 1 (off) */
  const int* chunk_first; /* prefill chunks of the first batch, as mk_plan_update_rows (host, nullable) */
  int tc_off;        /* 1: plans of capacity 3-8 on the CUDA cores; 0 (default): a capacity of 3 to
                        8 takes the batch-8 kernel instance, whose QKV and O projections and expert
                        gate/up run on the tensor cores (tcgen05, TMEM accumulators, TMA tiles), when
                        hidden, n_q_heads * head_dim and (G + 2) * head_dim are multiples of 128,
                        expert_ffn of 64 and n_experts at most 128 */
} mk_plan_opts;

typedef struct mk_plan mk_plan;

/* Defined by: "Cohere Publishes One-Kernel Server for North Mini Code",
 * "One resident program, many small tasks" (the host prepares a list of small
 * tasks per SM and readiness lives in counters in global memory) and "What
 * the scheduling change is meant to avoid" (tile-level scheduling, no false
 * dependencies); "Inside the Megakernel Serving Engine for North Mini Code",
 * architecture paragraph (a task list per SM).
 *
 * Build the task list and dependency counters for `batch` requests whose
 * caches hold seq_lens[b] tokens (host array), with the host page table
 * page_table[b * max_pages_per_seq + i] (page ids of request b in order).
 * Every page that covers positions [0, seq_lens[b]] must be present and in
 * [0, kv->num_pages).  Allocates the plan's device buffers on the current
 * device.  *out is set only on success. */
int mk_plan_create(const mk_model_dims* dims, const mk_weights* w, const mk_kv* kv, int batch,
                   const int* seq_lens, const int* page_table, int max_pages_per_seq,
                   const mk_plan_opts* opts, mk_plan** out);

/* Defined by: "Cohere Publishes One-Kernel Server for North Mini Code",
 * "The delay is between operations" (one decode step: normalization,
 * projections, attention and expert routing, run without kernel boundaries)
 * and "One resident program, many small tasks" (one resident block per SM
 * walks its tasks); "Inside the Megakernel Serving Engine for North Mini
 * Code", architecture paragraph (QKV, then attention, then the MoE, as one
 * program); "Cohere fuses an entire decode step into one GPU program".
 *
 * One decode step, enqueued on `stream`: request b decodes d_tokens[b] (device
 * int32[batch]) at position seq_len[b], writes its K/V there, and the greedy
 * next token to d_next_token[b] (device int32[batch]); d_logits (device
 * fp32[batch, vocab]) is written when non-NULL.  d_tokens may alias
 * d_next_token.  After the step the plan's lengths are seq_len + 1.  Returns
 * MK_ERR_CAPACITY (nothing enqueued) if a request's next position has no page.
 * Device failures (MK_ERR_DEP_TIMEOUT) are reported by mk_plan_sync; once one
 * is recorded, later steps do no work until mk_plan_update. */
int mk_decode_step(mk_plan* plan, const int* d_tokens, float* d_logits, int* d_next_token,
                   mk_stream stream);

/* Defined by: "Cohere Publishes One-Kernel Server for North Mini Code", "The
 * delay is between operations" (time lost where one kernel ends and the next
 * begins), here at the boundary between decode steps; the pages stop at one
 * step, and running several in one launch is this library's reading of it.
 *
 * n_steps >= 1 decode steps in ONE launch of the persistent kernel, each
 * step's greedy (or sampled) tokens fed to the next on the device: step 0
 * decodes d_tokens[b] (device int32[batch]); step s >= 1 decodes the tokens
 * step s - 1 wrote.  Step s writes request b's next token to
 * d_next_tokens[s * batch + b] (device int32[n_steps, batch]) and, when
 * d_logits is non-NULL, its logits to d_logits[(s * batch + b) * vocab ...]
 * (device fp32[n_steps, batch, vocab]).  Request b's step s runs at position
 * seq_len[b] + s; every one of those positions needs a page (else
 * MK_ERR_CAPACITY, nothing enqueued).  Afterwards the plan's lengths are
 * seq_len + n_steps.  d_tokens may alias the first row of d_next_tokens.
 * The results equal n_steps calls of mk_decode_step.  A group plan (capacity
 * above 8) runs one such launch per sub-plan; the rows stay [n_steps, batch].
 * Errors as mk_decode_step. */
int mk_decode_steps(mk_plan* plan, const int* d_tokens, int n_steps, float* d_logits, int* d_next_tokens,
                    mk_stream stream);

/* The same step with HOST buffers: copies h_tokens in, runs the step, copies
 * the next tokens (and logits when h_logits != NULL) out, and waits for the
 * stream.  Host buffers may be pageable or pinned. */
int mk_decode_step_host(mk_plan* plan, const int* h_tokens, float* h_logits, int* h_next_token,
                        mk_stream stream);

/* Defined by: "Cohere Publishes One-Kernel Server for North Mini Code",
 * introduction (the engine serves with continuous batching, paged attention
 * and ragged sequence lengths) and "A hand-built approach to a specialized
 * server".
 *
 * Continuous batching: replace the batch (requests joining or leaving) with
 * `batch` requests (<= the plan's capacity), their cached lengths and page
 * table (host arrays, same layout as mk_plan_create).  Rebuilds the task list,
 * uploads it with the lengths and page table on `stream`, resets counters and
 * clears a recorded device error.  No kernel is launched. */
int mk_plan_update(mk_plan* plan, int batch, const int* seq_lens, const int* page_table,
                   int max_pages_per_seq, mk_stream stream);

/* Prefill: the same update where some rows are prefill chunks (the pages
 * speak of serving prompts, not of how they enter the cache; here a prompt
 * enters the paged cache through the decode tasks, up to 8 tokens per launch).
 * chunk_first[b] (host int32[batch], NULL = every row its own request) is
 * the first row of the chunk row b belongs to: rows chunk_first[b] .. b are
 * consecutive prompt tokens of ONE request, row b at position seq_lens[b] =
 * seq_lens[b - 1] + 1, with the same page-table row (the request's pages;
 * a page for the last row's position must be there).  Each row appends its
 * token's K/V and attends causally to the request's cache and the chunk's
 * earlier rows; its next token is the model's prediction after it (the last
 * row's is the first output).  Rows of different chunks or requests may not
 * share a page; in a plan with a capacity above 8 a chunk may not cross a
 * multiple of 8 rows (one sub-plan).  A batch with chunks runs exactly one
 * mk_decode_step (MK_ERR_INVALID for a second step or mk_decode_steps with
 * n_steps > 1) before the next update.  MK_ERR_INVALID for a malformed chunk. */
int mk_plan_update_rows(mk_plan* plan, int batch, const int* seq_lens, const int* page_table,
                        int max_pages_per_seq, const int* chunk_first, mk_stream stream);

/* Wait for `stream`, then return the device status (MK_OK or the first error
 * a step recorded). */
int mk_plan_sync(mk_plan* plan, mk_stream stream);

/* Sampling beyond greedy for the following steps (the pages stop at the next
 * token; this is the plainest sampler).  temperature 0 (the default) is
 * greedy; above 0 the next token of request b is a draw from
 * softmax(logits / temperature), made by the Gumbel-max construction: the
 * argmax over rows v of logit_v / temperature - log(-log(u_v)), with u_v =
 * ((x >> 9) + 1/2) * 2^-23 and x word 0 of Philox4x32-10 (Salmon et al.,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC 2011) with key (seed mod
 * 2^32, seed >> 32) and counter (v, the request's position, b, 0); b counts
 * across a group's sub-plans.  Draws are therefore reproducible from (seed,
 * batch slot, position).  Logits written by a step stay unscaled.
 * MK_ERR_INVALID for a negative, NaN or infinite temperature, or a positive
 * one so small that its inverse overflows (below about 2.9e-39); mk_plan_create
 * applies the same rule to opts->temperature.  Takes effect at
 * the next step; mk_decode_step_noalloc is always greedy. */
int mk_plan_set_sampling(mk_plan* plan, float temperature, unsigned long long seed);

/* Nucleus (top-p) sampling for the following sampled steps: with a
 * temperature above 0 and 0 < top_p < 1, the draw of mk_plan_set_sampling is
 * restricted to the nucleus: the rows ordered by logit (descending, the lower
 * index first among equal logits), cut at the shortest prefix whose mass
 * reaches top_p of the total.  A row's mass is w = exp((logit - max logit) /
 * temperature) in float32, held as the integer round(w * 2^32), so the sums
 * are exact and independent of the order of the adds; the cut is the first
 * prefix whose integer mass reaches ceil(top_p * total).  The token is then
 * the argmax of the same keys as mk_plan_set_sampling (logit / temperature
 * plus Gumbel noise keyed by seed, batch slot and position) over the nucleus
 * only.  The pages stop at the next token; this is the standard sampler
 * restricted as its usual definition says.  top_p = 1 (the default) turns it
 * off; temperature 0 stays greedy whatever top_p is.  The first step after
 * the setting changes between on and off rebuilds the task list (one draw
 * task per request after the LM head).  MK_ERR_INVALID outside (0, 1].
 * mk_decode_step_noalloc is always greedy. */
int mk_plan_set_top_p(mk_plan* plan, float top_p);

/* Copy a per-step intermediate of the most recent step into dst (device or
 * host memory, `bytes` long), on `stream`.  A plan with a capacity above 8
 * answers the per-request kinds (HIDDEN, EXPERT_IDS, GATES, ROUTER_LOGITS,
 * SEQ_LENS) and returns MK_ERR_UNSUPPORTED for the others:
 *   MK_DBG_HIDDEN        fp32 [batch, n_layers, hidden]  x after each layer
 *   MK_DBG_EXPERT_IDS    int32 [batch, n_layers, top_k]  rank order
 *   MK_DBG_GATES         fp32 [batch, n_layers, top_k]
 *   MK_DBG_ROUTER_LOGITS fp32 [batch, n_layers, n_experts]
 *   MK_DBG_SEQ_LENS      int32 [batch]                   device lengths
 *   MK_DBG_UNION         int32 [n_layers]                distinct experts per layer
 *   MK_DBG_TASKS         int32 [num_tasks, 12]           the task list in CTA order
 *                        (type, layer, a0..a7, wait counter, wait count)
 *   MK_DBG_TRACE         uint64 [num_tasks, 12]          globaltimer stamps (ns) per task:
 *                        consumer fetched, dependency met, activations ready, stages
 *                        consumed, done; producer first copy, last copy, start;
 *                        first and last stage landed; two steps inside the activation
 *                        part (expert tile: norm and router logits done, routing done);
 *                        0 = not recorded
 *                        (needs opts.trace)
 *   MK_DBG_STAGE_TRACE   uint64 [num_ctas, 4096, 6]      per CTA, its ring stages in order:
 *                        copy issued, landed (seen by the first consumer warp), released
 *                        (globaltimer ns, 0 = not reached), the task index, and the SM's
 *                        clock64 at landed and released (needs opts.trace = 2; stages past
 *                        4096 are not recorded) */
enum { MK_DBG_HIDDEN = 1, MK_DBG_EXPERT_IDS = 2, MK_DBG_GATES = 3, MK_DBG_ROUTER_LOGITS = 4,
       MK_DBG_SEQ_LENS = 5, MK_DBG_UNION = 6, MK_DBG_TASKS = 7, MK_DBG_TRACE = 8,
       MK_DBG_STAGE_TRACE = 9 };
int mk_plan_read_debug(mk_plan* plan, int what, void* dst, size_t bytes, mk_stream stream);

/* Describe the current plan (host-side numbers): writes up to `n` ints:
 * [num_ctas, num_tasks, nstages, stage_bytes, smem_bytes, batch, n_attn_tasks,
 *  n_gu_tasks, n_lm_tiles, replans, expert gate/up on the tensor cores (1/0),
 *  QKV and O projections on the tensor cores (1/0)]. */
int mk_plan_info(const mk_plan* plan, int* out, int n);

void mk_plan_destroy(mk_plan* plan);

const char* mk_status_string(int status);

/* Text of the most recent library failure on the calling thread (for example
 * the CUDA call and error behind an MK_ERR_CUDA); "" when none. */
const char* mk_last_error(void);

/* Host-only planner, for inspection and tests (no CUDA call): builds the task
 * list the plan would run for these lengths on `num_ctas` CTAs.  Writes up to
 * max_tasks tasks as 12 int32 each into `tasks` (type, layer, a0..a7,
 * wait_counter, wait_count) and num_ctas + 1 offsets into `cta_start`;
 * returns the task count (or a negative error). */
int mk_plan_inspect(const mk_model_dims* dims, int batch, const int* seq_lens, int num_ctas,
                    int split_pages, int* tasks, int max_tasks, int* cta_start);

/* One decode step that allocates no memory, for callers that cannot call
 * cudaMalloc where they decode: hosts that reserve all device memory in their
 * own pool and forbid raw allocations inside their enqueue callbacks, custom
 * allocator hooks that would recurse, and latency-critical loops that cannot
 * take the device-wide synchronisation cudaMalloc/cudaFree may cause.  The
 * pages have no counterpart to this call; it is a deployment convenience.
 *
 * Same step as mk_plan_create + mk_decode_step, with no plan: request b
 * decodes d_tokens[b] at position seq_lens[b] (host array; the cache holds
 * seq_lens[b] tokens), writes its K/V there, the greedy next token to
 * d_next_token[b] and, when non-NULL, logits to d_logits [batch, vocab] and
 * the device status (code, task, cta, info) to d_status (device int32[4]).
 * The caller advances seq_lens itself.  Arguments as in mk_plan_create.
 *
 * Scratch lives in one file-scope device array of MK_NOALLOC_SCRATCH_BYTES
 * (64 MiB) that every GPU loading libmk.so holds until the process exits;
 * the task list is staged in a 4 MiB file-scope host array.  A step needing
 * more returns MK_ERR_CAPACITY (mk_last_error() says how much it needed).
 * All calls share both arrays, so calls whose GPU work overlaps, or that run
 * concurrently on several host threads, race: serialise them.  The first call
 * on a device resolves the array's device address (cudaGetSymbolAddress with
 * that device current); make it before any stream capture. */
#define MK_NOALLOC_SCRATCH_BYTES (64ull << 20)
int mk_decode_step_noalloc(const mk_model_dims* dims, const mk_weights* w, const mk_kv* kv, int batch,
                           const int* seq_lens, const int* page_table, int max_pages_per_seq,
                           const int* d_tokens, float* d_logits, int* d_next_token, int* d_status,
                           mk_stream stream);

/* ---- Continuous batching: request scheduler with a KV page allocator ----
 *
 * The pages describe the megakernel as the engine of a server that admits
 * requests continuously into a paged KV cache with ragged lengths ("Cohere
 * Publishes One-Kernel Server for North Mini Code", "A hand-built approach
 * to a specialized server"; "Inside the Megakernel Serving Engine for North
 * Mini Code", architecture paragraph).  mk_sched is the host side of that
 * loop; the pages leave its policy open, and this one is the plainest:
 *   - pages: a free list over the pool's num_pages pages; a request is
 *     admitted only with the pages of its whole sequence (prompt_len +
 *     max_new_tokens - 1 cached positions) reserved, so an admitted request
 *     never waits for a page and nothing is ever preempted;
 *   - admission: first come, first served, while a batch slot (max_batch) is
 *     free and the request at the head of the queue fits in the free pages;
 *   - every step feeds each admitted request one token: its prompt tokens in
 *     order (the prediction of a prompt step is discarded, except after the
 *     last prompt token: that one is the first output), then its own
 *     previous output.  With prefill chunks (mk_sched_set_prefill) a request
 *     still in its prompt may take several rows of the step: after one row
 *     per admitted request, the spare rows go to prompts in batch order, up
 *     to the chunk size and the prompt's remaining tokens each (above 8 rows
 *     a chunk also ends at the next multiple of 8);
 *   - retirement: after max_new_tokens outputs, or right after the request
 *     outputs eos_token (eos_token < 0: none); its pages and slot are freed
 *     at once, and the batch keeps the order of the requests that remain.
 * The mk_sched_* calls are host-only (no CUDA call) and not thread-safe: one
 * thread per scheduler. */
typedef struct mk_sched mk_sched;

/* A scheduler over a KV pool of num_pages pages of page_size tokens, for at
 * most max_batch requests per step, each with a page-table row of
 * max_pages_per_seq entries.  MK_ERR_INVALID for a non-positive argument. */
int mk_sched_create(int num_pages, int page_size, int max_batch, int max_pages_per_seq, mk_sched** out);

/* Queue request `rid` (unique among the requests the scheduler holds) with
 * n_prompt >= 1 prompt tokens (host int32, copied; each >= 0) and
 * max_new_tokens >= 1.  MK_ERR_INVALID for a bad argument or a repeated rid;
 * MK_ERR_CAPACITY when its sequence needs more pages than a page-table row
 * or the whole pool holds (it could never be admitted). */
int mk_sched_submit(mk_sched* s, long long rid, const int* prompt, int n_prompt, int max_new_tokens,
                    int eos_token);

/* Prefill chunks: a request still in its prompt may feed up to max_chunk
 * (1 .. 8) prompt tokens in one step, as consecutive rows (see
 * mk_plan_update_rows).  1, the default, is one token per step.  Set it
 * between steps (MK_ERR_INVALID while a batch is pending). */
int mk_sched_set_prefill(mk_sched* s, int max_chunk);

/* The next step's rows (mk_sched_next with prefill chunks): like
 * mk_sched_next, with rows instead of requests (*rows of them, row arrays
 * sized for max_batch rows) and chunk_first[r] = the first row of row r's
 * request in this batch (r itself for a single row); a request's rows carry
 * its consecutive positions and its page row.  *changed is also 1 whenever
 * this batch or the previous one holds a chunk of several rows. */
int mk_sched_next_rows(mk_sched* s, int* rows, int* seq_lens, int* page_table, int* tokens, long long* rids,
                       int* chunk_first, int* changed);

/* The rows mk_sched_next_rows would hand out next if the pending batch (if
 * any) were committed with outputs that end no request early (no end token).
 * Changes nothing.  A serving loop uses it to prepare the next step (its task
 * list) while the current one runs on the GPU; the prediction misses only
 * when a request outputs its end token. */
int mk_sched_peek_rows(const mk_sched* s, int* rows, int* seq_lens, int* page_table, int* tokens, long long* rids,
                       int* chunk_first);

/* Admit what fits, then describe the next step's batch in host arrays sized
 * for max_batch requests: *batch, seq_lens[b] (tokens cached), page_table[b *
 * max_pages_per_seq + i] (-1 past the request's pages), tokens[b] (the input
 * token) and rids[b]; *changed = 1 when the requests differ from the
 * previous batch (a plan must then be updated), else 0.  *batch = 0: nothing
 * to run.  A non-empty batch must be committed (or abandoned) before the
 * next call, else MK_ERR_INVALID. */
int mk_sched_next(mk_sched* s, int* batch, int* seq_lens, int* page_table, int* tokens, long long* rids,
                  int* changed);   /* MK_ERR_INVALID with prefill chunks above 1 */

/* The step of the last mk_sched_next ran: next_tokens[b] (host int32) is
 * the output of row b (request b without prefill chunks; the prediction
 * after a request's last row is its output).  Advances every request by one position,
 * records outputs and retires finished requests.  MK_ERR_INVALID when no
 * batch is pending. */
int mk_sched_commit(mk_sched* s, const int* next_tokens);

/* The step of the last mk_sched_next did not run: forget the batch (no
 * request advances; the next batch reports changed = 1).  MK_ERR_INVALID
 * when no batch is pending. */
int mk_sched_abandon(mk_sched* s);

/* Outputs of request rid so far: copies min(cap, count) tokens to `tokens`
 * (host, may be NULL when cap == 0), the count to *n_tokens and 1 to *done
 * once it retired.  MK_ERR_INVALID for an unknown rid. */
int mk_sched_result(const mk_sched* s, long long rid, int* tokens, int cap, int* n_tokens, int* done);

/* Drop a retired request's record (its outputs); MK_ERR_INVALID if rid is
 * unknown or not retired. */
int mk_sched_forget(mk_sched* s, long long rid);

/* Counters: out[0] queued, [1] admitted, [2] retired (not forgotten), [3]
 * free pages, [4] steps committed.  Writes min(n, 5) values. */
int mk_sched_stats(const mk_sched* s, int* out, int n);

void mk_sched_destroy(mk_sched* s);

/* One step of the serving loop on `stream`: mk_sched_next_rows; when *plan
 * is NULL, mk_plan_create with that batch (capacity opts->max_batch, or the
 * scheduler's max_batch when 0; a smaller capacity is MK_ERR_INVALID), else
 * mk_plan_update_rows when the rows changed; the step from host buffers
 * (as mk_decode_step_host), during which the host builds the task list of
 * the batch mk_sched_peek_rows predicts, so the next call's update only
 * uploads it when the prediction holds; then
 * mk_sched_commit.  dims, w and kv are read only when the plan is created
 * (kv->num_pages must be at least the scheduler's pool).  Returns the batch
 * size that ran (0: nothing queued or admitted) or an error; on an error the
 * batch is abandoned, so the same requests run again on the next call (after
 * a device error, only once the caller has dealt with it). */
int mk_serve_step(mk_sched* s, mk_plan** plan, const mk_model_dims* dims, const mk_weights* w, const mk_kv* kv,
                  const mk_plan_opts* opts, mk_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
