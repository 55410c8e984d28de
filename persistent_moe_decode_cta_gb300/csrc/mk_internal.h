// Internal definitions shared by the host planner and the device code of libmk.
//
// Task descriptor: 32 int32 fields per task.  The pages specify the width (32
// int32) and list opcode, layer, output tile, split-K coordinates, and the
// counters a task waits on and signals [Cohere open-sources fused LLM decode
// kernel with 1.58x vLLM claim, descriptor paragraph]; the concrete field order
// below is this library's.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace mk {

// ---- CTA shape -------------------------------------------------------------
// 8 consumer warps (MMA + epilogues), 1 producer warp (descriptor walk, queue
// claims, bulk/TMA copies into the shared-memory ring) and 1 storer warp (publishes
// the consumers' completed outputs to the global counters, so consumers do not wait
// on the release).  One CTA per SM.
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kStorerWarp = kConsumerWarps + 1;
constexpr int kThreads = kConsumerThreads + 64;

// ---- shared memory ---------------------------------------------------------
constexpr int kStageBytes = 32768;            // one ring slot
constexpr int kStages = 6;                    // 192 KB of copies in flight per SM
constexpr int kScratchBytes = 32768;          // cross-warp reductions / merges
constexpr int kSmallBytes = 1024;             // per-warp scalars, flags (256 ints):
// [1, 5) flags; [5] the tensor-memory base address; [16, 144) per-task scratch (route
// step selection, attention combine maxima and sums, residual block list, operand
// partial sums); [192, 224) trace slots; [224, 232) sequence lengths; [240, 248) 1/rms
// per token; [248, 252) epoch, step, grid-barrier generation
constexpr int kMbox = 8;                      // producer -> consumer task mailbox
constexpr int kSq = 8;                        // consumer -> storer signal queue
constexpr int kFragBytes = 512;               // one 16x16 bf16 MMA A-fragment
constexpr int kFragBytes8 = 256;              // the same fragment in E4M3 codes (FP8 experts)
constexpr int kFragsPerStage = kStageBytes / kFragBytes;
constexpr int kMaxNrb = 8;                    // GEMV task rows <= 128
constexpr int kMaxKsw = 16;                   // GEMV task K <= 2048 (16 k16-steps/warp)
constexpr int kBarBytes = (2 * kStages + 2 * kMbox + 2 * kSq + 2) * 8;  // + 2: tensor-core chunk commits
// mailbox entry: {task, item, chunks, n_tok}, {token bytes 0..3, 4..7, -, -}, {weights
// 0..3}, {weights 4..7} (MoE items carry their expert's token list -- byte n = b * 8 + j
// for the n-th token b, rank j -- and the tokens' routing weights as f32 bits)
constexpr int kMboxBytes = kMbox * 64 + kSq * 8;
constexpr int kSmemBytes = 1024 /*align slack*/ + kStages * kStageBytes + kScratchBytes +
                           kSmallBytes + kBarBytes + kMboxBytes;
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-block shared memory limit");

constexpr int kDescInts = 32;
// Size of the static step scratch of mk_decode_step_noalloc (64 MiB).
constexpr size_t kStaticScratchBytes = size_t(64) << 20;
// Counters are padded to one 128-byte line each so that waiters on different
// counters do not poll the same L2 line.
constexpr int kCtrStride = 32;
// Each residual row block's per-token sums of squares sit in their own 128-byte line
// (every consumer of the normed input reads all of them).
constexpr int kSsStride = 32;
constexpr int kMaxBatch = 8;
// Replicas of the per-token greedy-argmax key (multi-step decode): the LM head tiles
// of a step add into replica (SM index mod kAmaxReplicas) so that ~2400 tiles do not
// serialise on one word; the step's last CTA reduces them.
constexpr int kAmaxReplicas = 32;
constexpr int kMaxActive = kMaxBatch * 8;     // active experts per layer <= batch * top_k
constexpr int kRowBlock = 128;                // residual row block (rows of d_model)
// j-groups per ring chunk of a GEMV tile with `nrb` 16-row blocks (chunk = jpc*nrb*4 KB)
constexpr __host__ __device__ int gemv_jpc(int nrb) { return 8 / nrb > 0 ? 8 / nrb : 1; }
// FP8 fragments are half the bytes: twice the j-groups per 32 KB ring chunk
constexpr __host__ __device__ int gemv_jpc8(int nrb) { return 16 / nrb > 0 ? 16 / nrb : 1; }
// FP8 expert item (fs = 32 or 64): [scales: 2*fs gate/up row scales, then the d
// down-row scales of the expert, f32]
// [gate/up E4M3 fragments: 2*fs*d bytes][down E4M3 fragments: d*fs bytes]
constexpr __host__ __device__ int fp8_scale_bytes(int fs, int d) { return (2 * fs + d) * 4; }
// consumer warps whose down-slice regions share one ring chunk (a power of two)
constexpr __host__ __device__ int moe_warps_per_chunk(int region_bytes) {
  return region_bytes * 8 <= 32768 ? 8 : region_bytes * 4 <= 32768 ? 4 : region_bytes * 2 <= 32768 ? 2 : 1;
}

enum Op : int32_t {
  OP_END = 0,
  OP_EMBED = 1,      // x0 = embed[token], row-block sums of squares
  OP_QKV = 2,        // QKV_PROJ tile + RoPE + K/V append
  OP_ROUTER = 3,     // ROUTER_GEMM tile; last tile runs ROUTER_TOPK + ROUTE_FINALIZE
  OP_ATT_DRAIN = 4,  // ATTN_DRAIN: claim (group, seq, split) items; last split of a
                     // (seq, group) runs ATTN_COMBINE
  OP_MOE_DRAIN = 5,  // MOE_UPGATE_ACT + MOE_DOWN + MOE_COMBINE for one (expert, f-slice)
                     // item: gather fused into the operand load, SiLU-mul epilogue kept
                     // in smem, the down slice's routing-weighted partial added into the
                     // layer's MoE accumulator
  OP_OPROJ = 7,      // O_PROJ split-K by KV group
  OP_LMHEAD = 8,     // final RMSNorm + LM_HEAD tile
  OP_RESID = 9,      // ADD_RMSNORM of one residual row block once the layer's O-proj
                     // tiles for it and all MoE items are done
  OP_PREFETCH = 10,  // producer only: L2 prefetch of a weight range (D_WOFF, D_WBYTES)
  OP_PREFETCH_KV = 11  // producer only: L2 prefetch of this SM's share of layer D_LAYER's
                       // cached K/V pages
};

enum DescField : int {
  D_OP = 0, D_LAYER = 1, D_AUX = 2, D_ROW0 = 3, D_NROWS = 4, D_K0 = 5, D_KLEN = 6,
  D_WAIT_CTR = 7, D_WAIT_TARGET = 8, D_SIG_CTR = 9, D_SIG_TARGET = 10,
  D_WOFF_LO = 11, D_WOFF_HI = 12, D_WBYTES = 13, D_QUEUE = 14, D_TASK_ID = 15,
  D_WAVE = 16, D_WAIT2_CTR = 17, D_WAIT2_TARGET = 18
};

// Row-map modes of the weight packer.
enum PackMode : int { PACK_IDENT = 0, PACK_QKV = 1, PACK_GATE_UP = 2 };
// MoE item (expert e, f-slice s = rows [FS s, FS s + FS) of d_ff, FS in {16, 32})
// packed as one contiguous tile: the 2 FS interleaved gate/up rows x d_model (GEMV
// fragment order, FS/8 row blocks), then the down slice W_down[:, FS s : FS s + FS]
// row-block-major (fragment order [16-row block of d_model][k16-step]).

// Device error word layout (int32[16]).
enum ErrField : int { E_CODE = 0, E_TASK = 1, E_CTR = 2, E_OBS = 3, E_TARGET = 4,
                      E_SM = 5, E_ABORT = 8 };

struct Params {
  // shape
  int L, d, Hq, Hkv, hd, E, topk, f, V, gs, nrb_d, B, maxa;
  int max_pages, n_pages, window;
  unsigned long long swa_mask;
  float theta, eps, scale_log2;
  int split_pages, max_items_bg;
  int moe_fs, t_moe, qkv_tpg, n_router_tasks;  // MoE item = moe_fs rows of d_ff; t_moe = d_ff / moe_fs
  long long timeout_ns;
  int fixed, do_reset;
  int inflight;             // max issued-but-not-landed ring chunks per CTA (1..kStages-1)
  int inflight_moe;         // the same for the chunks of expert items
  // the tail of a layer's expert phase: the last tail_items expert items of the queue
  // and the O-proj tiles claimed by the MoE drains keep inflight_tail chunks in flight
  // (fewer SMs stream then; each needs more bytes in flight); tail_items 0 = off
  int tail_items, inflight_tail;
  // at the route step (batch 1), L2 prefetch of the first route_pf_bytes of every item
  // of the selected experts (0 = off)
  int route_pf_bytes;
  // batch 1: the route step on one warp (route_step_b1) instead of the block-wide one
  int route_warp;
  // LM head on the 5th-generation tensor cores: 128-row tiles whose weight chunks are in
  // the K-major core-matrix layout, accumulated in tensor memory (tcgen05.mma); selects
  // the kernel build compiled with MK_UMMA
  int lm_umma;
  int moe_umma;  // (in that build) the bf16 expert and dense-FFN items on tcgen05 too
  // deterministic accumulation: the layer accumulators `moe` hold 64-bit fixed-point
  // integers (32 fraction bits) added with integer reductions, so that their sums, and
  // everything downstream, do not depend on the order of the expert and O-proj adds
  int det;
  int fp8;                  // expert weights as E4M3 codes with f32 scales (items: see fp8_scale_bytes)
  int dense_fs;             // f-slice rows of a dense layer's FFN items (bf16; = moe_fs without FP8)
  // FP8 projections: the QKV, O-proj and LM-head tiles hold E4M3 codes (8 bytes a lane
  // per fragment) and their rows' float32 scales sit in these arrays (packed-row order)
  int fp8d;
  int qkv_rows_group;       // packed QKV rows of a KV group
  const float* qkv_scale;   // [L][Hkv][qkv_rows_group]
  const float* o_scale;     // [L][d]
  const float* lm_scale;    // [v_pad]
  long long dense_item_bytes;
  // mixed dense/MoE stacks: bit l set = layer l is dense, its FFN is t_dense items (one
  // per moe_fs rows of dense_ff) at off_dense + (r * t_dense + t) * moe_item_bytes, r =
  // the number of dense layers below l
  unsigned long long dense_mask;
  int t_dense;
  long long off_dense;
  // multi-step decode: n_steps steps per launch, each step's greedy token (argmax of its
  // logits, lowest index on ties) written to tok_out[step][B] and fed to the next step
  int n_steps;
  int32_t* tok_out;               // [n_steps][B] or null (then no argmax)
  unsigned long long* amax;       // [kAmaxReplicas][B] (value key << 32 | ~row), zero between steps
  unsigned* gen;                  // step generation word of the grid barrier between steps
  // weights
  const uint8_t* wblob;
  long long off_moe, moe_item_bytes;  // item (l, e, s) at off_moe + ((l*E + e)*t_moe + s) * item_bytes
  const unsigned long long* rope_turns;  // [hd/2] inv_freq_i / (2 pi) as 0.64 fixed point
  const float* attn_norm;   // [L][d]
  const float* final_norm;  // [d]
  const uint16_t* embed;    // [V][d] bf16
  // step inputs / outputs
  const int* tokens;
  const int* page_table;    // [B][max_pages]
  int* seq_lens;            // [B]
  uint16_t* kc;             // [L][n_pages][Hkv][16][hd] bf16
  uint16_t* vc;
  float* logits;            // [B][V]
  // activations (per layer)
  float* X;                 // [L+1][B][d]
  float* SS;                // [L+1][nrb_d][kSsStride]: token b's sum of squares at [.][.][b]
  uint16_t* XG;             // [L+1][B][d] bf16(x_l * gain_l), gain_L = final norm
  uint16_t* XGL;            // [L+1][B][d] bf16 of the rounding residue x_l*gain_l - XG
  uint16_t* Q;              // [L][B][Hq*hd]
  float* attp;              // [L][Hkv][B][max_items_bg][gs*(hd+2)]
  uint16_t* atto;           // [L][B][Hq*hd]
  uint64_t* rlog;           // [L][B][E] router logits as (step epoch << 32 | f32 bits)
  uint64_t* rword;          // [L][rw_stride] route words (epoch << 32 | value): n_active,
                            // active ids [maxa], token counts [maxa], tokens [maxa][B]
                            // (b * 16 + j), token weights [maxa][B] (f32 bits)
  unsigned* epoch;          // step epoch (device word; the step's last launch advances it)
  int rw_stride;
  int* ridx;                // [L][B][topk]
  float* rw;                // [L][B][topk]
  int* active;              // [L][maxa]
  int* nact;                // [L]
  int* act_cnt;             // [L][maxa]
  int* act_tok;             // [L][maxa][B]  (b*16 + j)
  float* moe;               // [L][B][d] layer accumulator: the routing-weighted expert outputs
                            // plus the O-proj outputs of every KV group
  // synchronisation
  unsigned* ctr;
  int* qhead;               // [3L]
  int* qcount;              // [3L]
  int* err;                 // [16]
  int c_lr, c_qkvg, c_rt, c_rr, c_att, c_og, c_md, c_od, c_oa, c_done, n_ctr, n_queues;
  int od_target;
  // inspection (null = off): the step's last CTA copies the final counter values
  // [n_ctr], then the queue heads [n_queues] and counts [n_queues], before the reset
  unsigned* snap;
  // optional task timeline (see trace_emit)
  unsigned long long* trace;
  unsigned* trace_n;
  int trace_cap;
  // plan (one segment)
  const int* tasks;
  const int* sm_off;
  const int* sm_list;
};

}  // namespace mk
