/*
 * mk.h -- C ABI of the persistent MoE decode megakernel (libmk.so).
 *
 * One call to mk_decode_step() runs one batched decode step of a parallel-block
 * mixture-of-experts transformer as ONE persistent kernel launch: one CTA per SM
 * walks a host-built list of 32-int32 task descriptors, waits on and signals
 * atomic counters in global memory, and claims attention and expert tiles whose
 * number depends on live sequence lengths and routing from atomic work queues.
 *   [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "One kernel for
 *    the full decode step", "The calling convention that makes it hand-writable",
 *    "Scheduling: mostly static, selectively dynamic";
 *    Cohere open-sources fused LLM decode kernel with 1.58x vLLM claim: the 16 task
 *    types and the 32-int32 descriptor.]
 *
 * Conventions for every call:
 *   - Returns an mk_status code; nothing throws across the ABI.  mk_last_error()
 *     gives a message for the last failing call on a handle.
 *   - "device pointer" arguments are CUDA device addresses on the handle's device;
 *     "host pointer" arguments are ordinary host memory.  `stream` is a
 *     cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Errors raised inside the kernel (timeouts of a dependency wait, a page id or
 *     token outside its range, a NaN router logit) are recorded in a device error
 *     word and surface at the next mk_get_status().  Such a step's outputs are not
 *     valid.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mk_status {
  MK_OK = 0,
  MK_ERR_INVALID = 1,      /* bad argument (null pointer, size out of range)        */
  MK_ERR_UNSUPPORTED = 2,  /* shape the kernels do not handle (see mk_create)       */
  MK_ERR_CUDA = 3,         /* a CUDA runtime call failed                           */
  MK_ERR_OOM = 4,          /* device allocation failed                             */
  MK_ERR_TIMEOUT = 5,      /* a dependency wait inside the kernel gave up          */
  MK_ERR_BAD_PAGE = 6,     /* a page-table entry was outside [0, n_pages)          */
  MK_ERR_BAD_TOKEN = 7,    /* a token id was outside [0, vocab)                    */
  MK_ERR_STATE = 8,        /* call out of order (e.g. decode before mk_plan)       */
  MK_ERR_NAN = 9           /* a router logit was NaN: the step's activations are
                              not finite (the route ranks it below every number)  */
} mk_status;

/* Model shape.  The kernels need: head_dim in {32, 64, 128}; d_model, d_ff and
 * (n_q_heads / n_kv_heads) * head_dim multiples of 128; n_q_heads divisible by
 * n_kv_heads (at most 8) with a group of at most 8 query heads and
 * group*head_dim <= 1024;
 * n_experts a multiple of 8 in [8, 256]; top_k <= 8; page_size == 16; max_batch <= 8; n_layers <= 64.
 * swa_layer_mask bit l set = layer l uses a sliding window of sliding_window keys
 * (the window holds the new token and the sliding_window - 1 keys before it).
 * timeout_ms bounds every dependency wait inside the kernel (0 = 2000 ms).
 * dense_layer_mask bit l set = layer l is dense (a mixed dense/MoE stack): one SwiGLU
 * FFN of width dense_ff (a multiple of 128, <= 4096) for every token, no router, in
 * place of the routed experts; 0 = every layer routed (dense_ff ignored).
 * [Cohere open-sources fused LLM decode kernel with 1.58x vLLM claim: the dense GEMM
 * task types FFN_UPGATE_ACT and FFN_DOWN]
 * expert_dtype: MK_EXPERT_BF16 (0) keeps the routed experts' matrices in bf16;
 * MK_EXPERT_FP8 (1) stores them, at mk_create, as E4M3 codes (nearest, ties to even,
 * saturating) with one float32 scale per output channel (row) of gate, up and down
 * (max |w| over the row / 448; 1 for a zero row), and the kernel decodes the codes to
 * fp16 for the MMA and applies the scales to its fp32 results.  It needs d_ff a
 * multiple of 64 (of 32 when max_batch < 4, where the expert items are 32 rows of d_ff
 * instead of 64) (MK_ERR_UNSUPPORTED).  The dense FFNs of a mixed stack stay bf16.
 * MK_WEIGHTS_FP8 (2) stores the QKV, O-proj and LM-head matrices the same way as well
 * (E4M3, one float32 scale per output row, over the whole row); the router, the norms
 * and the embedding stay bf16 (the router's logits decide the top-k; its bytes are
 * under 1% of a step's).
 * [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, Current limitations:
 * FP8 quantization is on the roadmap; the pages fix no format] */
enum { MK_EXPERT_BF16 = 0, MK_EXPERT_FP8 = 1, MK_WEIGHTS_FP8 = 2 };
typedef struct mk_config {
  int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim;
  int32_t n_experts, top_k, d_ff, vocab, page_size, max_batch;
  int32_t sliding_window;
  uint64_t swa_layer_mask;
  float rope_theta, rms_eps;
  int32_t timeout_ms;
  uint64_t dense_layer_mask;
  int32_t dense_ff;
  int32_t expert_dtype;
} mk_config;

/* Model weights, all bf16 DEVICE pointers, row-major [out][in]:
 *   embed, lm_head     [vocab][d_model]
 *   final_norm         [d_model]
 *   attn_norm[l]       [d_model]                      (host array of n_layers ptrs)
 *   wq[l] [Hq*hd][d]   wk[l], wv[l] [Hkv*hd][d]       wo[l] [d][Hq*hd]
 *   router[l]          [n_experts][d]
 *   w_gate[l*E+e], w_up[l*E+e] [d_ff][d];  w_down[l*E+e] [d][d_ff]
 *   ffn_gate[l], ffn_up[l] [dense_ff][d];  ffn_down[l] [d][dense_ff]  (dense layers)
 * The arrays of pointers are HOST arrays.  On a dense layer router[l] and the
 * layer's expert pointers may be NULL; ffn_* may be NULL (the arrays themselves too)
 * when no layer is dense.  mk_create copies everything into a handle-owned packed
 * blob, so the caller may free its tensors afterwards. */
typedef struct mk_weights {
  const void* embed;
  const void* lm_head;
  const void* final_norm;
  const void* const* attn_norm;
  const void* const* wq;
  const void* const* wk;
  const void* const* wv;
  const void* const* wo;
  const void* const* router;
  const void* const* w_gate;
  const void* const* w_up;
  const void* const* w_down;
  const void* const* ffn_gate;
  const void* const* ffn_up;
  const void* const* ffn_down;
} mk_weights;

typedef struct mk_handle mk_handle;

/* Error details read back by mk_get_status(). */
typedef struct mk_error_info {
  int32_t code;      /* mk_status of the first device-side error, MK_OK if none  */
  int32_t task;      /* descriptor index that raised it (-1 if not a task)       */
  int32_t counter;   /* counter index waited on (timeouts)                       */
  int32_t observed;  /* counter value seen at the timeout, or the bad id, or the
                        layer of a NaN router logit                              */
  int32_t target;    /* value waited for; for a NaN router logit its index
                        token * n_experts + expert                               */
  int32_t sm;        /* CTA index                                                */
} mk_error_info;

/* Create a handle on the current CUDA device: validate `cfg`, allocate the packed
 * weight blob and repack every matrix into contiguous per-task tiles whose 16-byte
 * units are the mma.sync A-fragments in the order the consumer warps read them.
 * `stream` orders the packing kernels; the call synchronises it before returning.
 * On error *out is NULL.  Two environment variables, read here, select the tensor-core
 * build of the kernel: MK_LM_UMMA=1 packs the LM head in 64-row tiles in the tcgen05
 * K-major core-matrix layout (bf16 projections, d_model a multiple of 256), and
 * MK_MOE_UMMA=1 beside it does the same for the bf16 expert and dense-FFN items (32-row
 * f-slices); MK_Q_TENSOR_CORES reports what took effect.
 * [Cohere Megakernel, "Getting started": the engine is a shared library
 *  (libmk_release.so) that the serving process loads together with the model's
 *  checkpoint; Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "One
 *  kernel for the full decode step": weights are immutable, so their tiles can be
 *  laid out once, ahead of time, and streamed before a task's inputs are ready.] */
int mk_create(const mk_config* cfg, const mk_weights* w, void* stream, mk_handle** out);

/* Build the task plan for a batch: per-SM descriptor lists, counter targets and
 * the buffers of a step.  Called when the batch composition changes, not per step.
 * [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "Scheduling: mostly
 *  static, selectively dynamic": the host builds named waves per layer, deals task k
 *  to SM k mod #SM, and leaves attention and MoE tiles to claimer tasks on shared
 *  queues; Cohere open-sources fused LLM decode kernel with 1.58x vLLM claim: each
 *  task is a 32-int32 descriptor naming its opcode, layer, output tile, split-K
 *  coordinates, the counter it waits on and the counter it signals.]
 *   batch              1..max_batch
 *   seq_lens_host      HOST int32[batch], cached tokens per sequence (the next
 *                      step writes the new token at this position)
 *   page_table_dev     DEVICE int32[batch][max_pages_per_seq]: physical page of
 *                      logical page j of sequence b; entries past the sequence's
 *                      length may be -1.  Must stay valid while the plan is used.
 *   n_pages            pages in the caller's K/V pools
 * The step reads seq_lens from a device copy that mk_decode_step advances by one
 * after each step (unless mk_set_fixed(h, 1)).  The attention split size (pages per
 * split, MK_Q_SPLIT_PAGES) is fixed here from seq_lens_host and the SM count: about 32
 * splits per (sequence, KV group) at the longest context, or, for long or numerous
 * splits, the size whose splits fill the SMs in one wave with one more per (sequence,
 * group) left for growth; sequences that later outgrow it still run correctly, with
 * more splits (re-plan to re-balance).  MK_SPLIT_PAGES (a multiple of 8) overrides it. */
int mk_plan(mk_handle* h, int batch, const int32_t* seq_lens_host,
            const int32_t* page_table_dev, int max_pages_per_seq, int n_pages);

/* One decode step as ONE kernel launch on `stream` (asynchronous).
 * [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "One kernel for the
 *  full decode step": one persistent launch runs every layer's RMSNorm, QKV with RoPE,
 *  paged attention, router, experts, O-proj and the LM head, one CTA per SM.]
 *   tokens_dev  DEVICE int32[batch]        input token per sequence
 *   k_cache, v_cache  DEVICE bf16 [n_layers][n_pages][n_kv_heads][16][head_dim],
 *               caller-owned; the step writes the new token's K/V into slot
 *               seq_len % 16 of page page_table[b][seq_len / 16] of every layer
 *               and attends over positions 0..seq_len (inclusive).
 *   logits_dev  DEVICE float[batch][vocab] output. */
int mk_decode_step(mk_handle* h, const int32_t* tokens_dev, void* k_cache, void* v_cache,
                   float* logits_dev, void* stream);

/* n_steps greedy decode steps as ONE kernel launch on `stream` (asynchronous): step
 * s feeds its greedy token -- the argmax of its logits, the lowest vocabulary index on
 * ties -- to step s+1 on the device (no host round trip), and the device seq_lens
 * advance after every step (unless mk_set_fixed(h, 1)).  The steps are separated by
 * a grid-wide barrier inside the launch.  This is the step after the path: the
 * serving loop the pages describe runs its decode loop in C++ on the host and
 * samples greedily.  [Fuse decode into one megakernel for 1.58x higher H100
 * throughput -- Persistent decode megakernel, closing section (the C++ decode loop);
 * Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "Current
 * limitations" (greedy sampling)]
 *   tokens_dev      DEVICE int32[batch]             the first step's input tokens
 *   n_steps         1..4096
 *   k_cache, v_cache  as for mk_decode_step; the page table given to mk_plan must
 *                   cover positions seq_len .. seq_len + n_steps - 1 of every
 *                   sequence (a missing page is reported as MK_ERR_BAD_PAGE)
 *   logits_dev      DEVICE float[batch][vocab]      the LAST step's logits
 *   tokens_out_dev  DEVICE int32[n_steps][batch]    every step's greedy token
 * A step that fails (see mk_get_status) stops the launch after that step. */
int mk_decode_steps(mk_handle* h, const int32_t* tokens_dev, int n_steps, void* k_cache,
                    void* v_cache, float* logits_dev, int32_t* tokens_out_dev, void* stream);

/* The same step with HOST token and logit buffers: copies tokens host->device,
 * runs mk_decode_step, copies logits device->host and synchronises `stream`.
 * tokens_host int32[batch]; logits_host float[batch][vocab]. */
int mk_decode_step_host(mk_handle* h, const int32_t* tokens_host, void* k_cache,
                        void* v_cache, float* logits_host, void* stream);

/* The same step as mk_decode_step for callers that cannot allocate device memory
 * while they decode -- e.g. an embedding runtime that owns the whole device heap, or a
 * code path that must not call cudaMalloc (which synchronises the device and may
 * fail under memory pressure).  This call allocates nothing: the step's scratch (the
 * per-layer activations, attention partials, routing tables, MoE accumulators,
 * counters and queues that mk_plan otherwise provides) lives in one file-scope static
 * device array of 64 MiB (kept on every GPU that loads the library until the process
 * exits).  The pages have no counterpart to this entry point.
 *   Arguments, layouts and results are those of mk_decode_step; the handle's packed
 *   weights, plan and seq_lens are used as usual.  mk_read's per-step state (hidden
 *   states, routes, router logits, active lists, counters) follows the handle's last
 *   step: after this call it is read from the static array, as the last
 *   allocation-free call on the device (of any handle) left it.
 *   Plans whose step scratch exceeds 64 MiB are rejected with MK_ERR_UNSUPPORTED and a
 *   message giving the size needed (the pages-scale model needs ~21 MiB at batch 1 with
 *   8K context, ~29 MiB at 128K, ~53 MiB at batch 2 with 32K, ~168 MiB at batch 8).
 *   The first call on a device looks up the array's device address (with that device
 *   current); make that first call before any stream capture.  Every call clears the
 *   counters and queues it needs (an asynchronous memset on `stream`) and overwrites
 *   the rest, but all calls share the one array: calls that overlap on the GPU (other
 *   streams, other handles) race and must be serialised by the caller. */
int mk_decode_step_noalloc(mk_handle* h, const int32_t* tokens_dev, void* k_cache, void* v_cache,
                           float* logits_dev, void* stream);

/* The same step with the same device routines run as one kernel launch per
 * opcode wave per layer (use_graph = 0), or that launch sequence captured once
 * into a CUDA graph and replayed (use_graph = 1).  Measurement baselines. */
int mk_decode_step_perop(mk_handle* h, const int32_t* tokens_dev, void* k_cache,
                         void* v_cache, float* logits_dev, void* stream, int use_graph);

/* Synchronise the handle's last stream and report the device error word; clears
 * it.  Returns info->code.  (The pages describe no error path; every dependency wait
 * of the kernel is bounded and reports here instead of hanging -- the counter waits
 * are the ones of [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "The
 * calling convention that makes it hand-writable"].) */
int mk_get_status(mk_handle* h, mk_error_info* info);

/* Task timeline for profiling.  records_dev: DEVICE uint64 [capacity][16], owned by
 * the caller; every task executed by a later step appends one record
 *   [0] sm | opcode << 8 | layer << 16 | (ran a fan-in follow-up) << 24
 *   [1] claimed item (attention split / expert tile) or 0
 *   [2..7] %globaltimer ns: received, dependency met, operands built / first
 *          weight or KV chunk landed, MMA loop done, fan-in follow-up started (0
 *          if none), done
 *   [8..11] sub-steps of a fan-in follow-up (route step: top-k done, lists
 *          started, lists done, released), 0 where unused; [12..15] zero.
 * capacity 0 (or records_dev NULL with capacity 0) turns tracing off.  Resets the
 * record count.  Synchronising. */
int mk_set_trace(mk_handle* h, void* records_dev, int capacity);

/* Testing hook (host-side fault injection): redirect the completion signal of
 * descriptor `task` (an index into the plan's table, see mk_plan_dry) away from the
 * counter its waiters poll.  The next step's waiters then give up after timeout_ms
 * and the step reports MK_ERR_TIMEOUT (task, counter, observed, target) through
 * mk_get_status; every CTA drains and exits, and the context stays usable.  Undo by
 * calling mk_plan again.  Synchronising. */
int mk_plan_drop_signal(mk_handle* h, int task);

/* Inspection of the schedule's bookkeeping.  on = 1: every later step's last CTA
 * copies the final value of every counter and every queue head and count aside,
 * before it clears them for the next step (read back with MK_READ_FINAL_COUNTERS /
 * MK_READ_FINAL_QUEUES); on = 0 turns it off (the default; the copy costs the last
 * CTA of a step about a microsecond).  Synchronising.  The steps of
 * mk_decode_step_noalloc are not copied.
 * [Cohere open-sources fused LLM decode kernel with 1.58x vLLM claim: the counters a
 *  descriptor waits on and signals; Cohere's Open-Source Megakernel Beats vLLM by
 *  1.58x on H100, "Scheduling: mostly static, selectively dynamic": the claimer
 *  queues] */
int mk_set_inspect(mk_handle* h, int on);

/* fixed = 1: steps do not advance seq_lens (repeated steps move identical bytes). */
int mk_set_fixed(mk_handle* h, int fixed);

/* on = 1: deterministic steps, from the next mk_plan on.  The experts' and O-proj
 * tiles' outputs are added into each layer's accumulator as 64-bit fixed-point
 * integers (32 fraction bits; |value| < 2^31) with integer reductions, whose sum does
 * not depend on the order in which the tiles finish; every other reduction of the step
 * has a fixed order, so two steps on the same inputs give bit-identical hidden states,
 * routing, K/V and logits.  (With on = 0, the default, the accumulators are float32 and
 * the order of the atomic adds changes their last bits from run to run; at a router
 * near-tie that can change the experts chosen.)  Costs twice the accumulator memory and
 * 64-bit scalar reductions in place of 128-bit float ones.  No counterpart in the pages,
 * whose combine is described only as the weighted sum of the experts' outputs
 * [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "One kernel for the full
 * decode step": MOE_COMBINE].  Errors: MK_ERR_INVALID for a NULL handle. */
int mk_set_deterministic(mk_handle* h, int on);

/* Debug/inspection reads into HOST memory (synchronising).  `what`:
 *   MK_READ_HIDDEN   float [n_layers+1][batch][d_model] residual entering each layer
 *                    (index n_layers = input of the final norm)
 *   MK_READ_ROUTES   int32 [n_layers][batch][top_k] selected experts
 *   MK_READ_ROUTE_W  float [n_layers][batch][top_k] their softmax weights
 *   MK_READ_ACTIVE   int32 [n_layers][1 + max_active*(2 + batch)]: per layer
 *                    n_active, then per active slot: expert id, token count, and
 *                    `batch` entries b*16 + j (token b, selection slot j)
 *   MK_READ_SEQ_LENS int32 [batch]
 *   MK_READ_COUNTERS uint32[n_counters] (all zero between steps)
 *   MK_READ_ROUTER_LOGITS float [n_layers][batch][n_experts]
 *   MK_READ_TRACE_COUNT uint32 [1] records appended since mk_set_trace (may exceed
 *                    the capacity; records past it were dropped)
 *   MK_READ_FINAL_COUNTERS uint32[n_counters] every counter's value at the end of the
 *                    last inspected step, before the reset (mk_set_inspect; else
 *                    MK_ERR_STATE).  Counter indices are those of the descriptors'
 *                    wait/signal fields; the bases are listed by mk_plan_dry.
 *   MK_READ_FINAL_QUEUES int32 [2][3 * n_layers] the queue heads, then the queue
 *                    counts, at the end of the last inspected step: queue l is layer
 *                    l's attention items, n_layers + l its expert items (count = items
 *                    routed), 2 n_layers + l its O-proj tiles.  Every claimer takes one
 *                    failing claim when its queue is empty, so a drained queue's head
 *                    is its items + the SMs (MK_Q_NUM_SMS) that ran its drain.
 *   MK_READ_TASKS    int32 [n_tasks][32] the plan's descriptor table
 * `bytes` must equal the size of the requested array. */
enum {
  MK_READ_HIDDEN = 1, MK_READ_ROUTES = 2, MK_READ_ROUTE_W = 3, MK_READ_ACTIVE = 4,
  MK_READ_SEQ_LENS = 5, MK_READ_COUNTERS = 6, MK_READ_ROUTER_LOGITS = 7,
  MK_READ_TRACE_COUNT = 8, MK_READ_FINAL_COUNTERS = 9, MK_READ_FINAL_QUEUES = 10,
  MK_READ_TASKS = 11
};
int mk_read(mk_handle* h, int what, void* host_out, size_t bytes);

/* The stored FP8 form of routed expert `expert` of layer `layer` (expert_dtype
 * MK_EXPERT_FP8), unpacked to row-major arrays in HOST memory, one after another:
 *   gate codes u8 [d_ff][d_model], up codes u8 [d_ff][d_model],
 *   down codes u8 [d_model][d_ff], gate scales f32 [d_ff], up scales f32 [d_ff],
 *   down scales f32 [d_model]
 * (a weight decodes as value(code) * its row's scale).  `bytes` must equal
 * 3 * d_ff * d_model + 4 * (2 * d_ff + d_model).  Synchronises
 * the device; needs no plan.  MK_ERR_STATE if the experts are stored in bf16,
 * MK_ERR_INVALID for a NULL pointer, a layer or expert out of range, a dense layer or
 * a wrong size.
 * [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, Current limitations:
 * FP8 quantization is on the roadmap] */
int mk_read_expert_fp8(mk_handle* h, int layer, int expert, void* host_out, size_t bytes);

/* The stored FP8 form of a projection (expert_dtype MK_WEIGHTS_FP8), unpacked to
 * row-major arrays in HOST memory: codes u8 [rows][cols], then the float32 scale of
 * every row [rows] (a weight decodes as value(code) * its row's scale).  `matrix`:
 *   MK_W_Q [Hq*hd][d_model], MK_W_K / MK_W_V [Hkv*hd][d_model], MK_W_O [d_model][Hq*hd]
 *   of layer `layer`, MK_W_LM [vocab][d_model] (layer ignored).
 * `bytes` must equal rows * cols + 4 * rows.  Synchronises the device; needs no plan.
 * MK_ERR_STATE if the projections are stored in bf16; MK_ERR_INVALID for a NULL
 * pointer, an unknown matrix, a layer out of range or a wrong size.
 * [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, Current limitations:
 * FP8 quantization is on the roadmap] */
enum { MK_W_Q = 0, MK_W_K = 1, MK_W_V = 2, MK_W_O = 3, MK_W_LM = 4 };
int mk_read_weight_fp8(mk_handle* h, int matrix, int layer, void* host_out, size_t bytes);

/* Integer facts about a handle/plan.  `what`: */
enum {
  MK_Q_NUM_SMS = 1, MK_Q_NUM_TASKS = 2, MK_Q_NUM_COUNTERS = 3, MK_Q_PACKED_BYTES = 4,
  MK_Q_MAX_ACTIVE = 5, MK_Q_SPLIT_PAGES = 6, MK_Q_SMEM_BYTES = 7, MK_Q_PEROP_LAUNCHES = 8,
  MK_Q_THREADS = 9, MK_Q_STAGE_BYTES = 10, MK_Q_NUM_STAGES = 11,
  /* which GEMVs of the handle run on the tcgen05 tensor cores (fixed at mk_create by the
   * environment): bit 0 the LM head (MK_LM_UMMA=1), bit 1 the bf16 expert and dense-FFN
   * items (MK_MOE_UMMA=1 beside it); needs no plan */
  MK_Q_TENSOR_CORES = 12
};
int mk_query(mk_handle* h, int what, int64_t* out);

/* Host-only planner run (no device needed): the descriptor table and the per-SM
 * lists that mk_plan would build for `n_sms` SMs (the megakernel segment), for tests
 * of the schedule.  Like mk_plan it takes the per-layer wave order from the
 * environment variable MK_WAVE_ORDER when set (letters r router, q QKV, a attention
 * drain, m MoE drain, o O-proj, x ADD_RMSNORM; default "rqamox"; an order that breaks
 * a dependency is MK_ERR_INVALID).
 *   tasks_out   int32[cap_tasks][32]      sm_off_out int32[n_sms + 1]
 *   sm_list_out int32[cap_list]           info_out int32[32]:
 *     [0] tasks  [1] list length  [2] counters  [3] max active experts  [4] 0
 *     [5] MoE items per expert  [6] MoE item KiB  [7] O-proj tile rows
 *     [8] MoE f-slice rows  [9] QKV tile rows  [10] QKV tiles per KV group
 *     [11] router tiles (per routed layer)  [12] O-proj tiles of a layer (the O-proj-done
 *     target)  [13] done-counter index
 *     [14] plan segments (1 + per-op launches)  [15] LM-head tiles
 *     [16..23] counter bases: layer-ready, QKV-group, router-tiles, route-ready,
 *              attention (layer, seq, group), O-group, MoE-done, row-block
 *     [24] residual row blocks  [25] query heads per KV group
 *     [26] attention-complete counter base  [27] items of a dense layer's FFN
 *     [28], [29] dense-layer mask, low and high 32 bits  [30] expert_dtype
 *     [31] MoE item bytes
 * Returns MK_ERR_INVALID if a cap is too small (info_out[0..1] still hold the sizes
 * needed). */
int mk_plan_dry(const mk_config* cfg, int batch, int n_sms, int32_t* tasks_out,
                int cap_tasks, int32_t* sm_off_out, int32_t* sm_list_out, int cap_list,
                int32_t* info_out);

/* Message for the last failing call on h (or the last global failure if h is
 * NULL).  The string is owned by the library. */
const char* mk_last_error(mk_handle* h);

/* Free everything the handle owns.  Safe on NULL. */
void mk_destroy(mk_handle* h);

/* ABI version (increments on any signature change). */
int mk_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
