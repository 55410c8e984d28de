// Host side of libmk: the C ABI (include/mk.h), shape validation, the weight
// packer driver, the task planner (static per-SM wave lists + claimer drains),
// step launches (megakernel, per-op launches, CUDA graph of the per-op launches)
// and status/debug reads.
//
// Planner: per layer the host emits named waves of tasks and deals the static
// ones round-robin, task k of the step to SM k mod #SM; attention and expert
// work is left to claimer ("drain") tasks that every SM runs, pulling items from
// per-layer atomic queues [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on
// H100, "Scheduling: mostly static, selectively dynamic"; Fuse decode into one
// megakernel for 1.58x higher H100 throughput: the layer's wave order QKV, router,
// attention, MoE projections, O-proj].
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "mk.h"
#include "mk_internal.h"

namespace mk {
cudaError_t launch_pack(uint8_t* dst, const void* src_a, const void* src_b, const void* src_c,
                        int n_rows_packed, int n_src_rows, int K, long long ld, int col0, int mode, int hd,
                        int gs, int grp, int tile_rows, cudaStream_t st);
cudaError_t launch_convert(float* dst, const void* src, long long n, cudaStream_t st);
cudaError_t launch_pack_moe(uint8_t* dst, const void* gate, const void* up, const void* down, int d, int f, int fs,
                            cudaStream_t st);
cudaError_t launch_pack_moe_fp8(uint8_t* dst, const void* gate, const void* up, const void* down, int d, int f,
                                int fs, long long item_bytes, cudaStream_t st);
cudaError_t launch_pack_rowscale(float* dst, const void* src_a, const void* src_b, const void* src_c,
                                 int n_rows_packed, int n_src_rows, int k_full, long long ld, int mode, int hd,
                                 int gs, int grp, cudaStream_t st);
cudaError_t launch_pack_fp8(uint8_t* dst, const float* scales, const void* src_a, const void* src_b,
                            const void* src_c, int n_rows_packed, int n_src_rows, int K, long long ld, int col0,
                            int mode, int hd, int gs, int grp, int tile_rows, cudaStream_t st);
cudaError_t prepare_megakernel();
int megakernel_occupancy(int* blocks);
cudaError_t launch_megakernel(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                              bool cooperative, cudaStream_t st);
cudaError_t static_scratch_address(void** ptr);
cudaError_t launch_pack_umma(uint8_t* dst, const void* src, int n_rows_packed, int n_src_rows, int K, cudaStream_t st);
cudaError_t launch_pack_moe_umma(uint8_t* dst, const void* gate, const void* up, const void* down, int d, int f,
                                 cudaStream_t st);
}  // namespace mk
// the same megakernel with deterministic (64-bit fixed-point) layer accumulators
namespace mk_det {
cudaError_t prepare_megakernel();
int megakernel_occupancy(int* blocks);
cudaError_t launch_megakernel(const mk::Params& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                              bool cooperative, cudaStream_t st);
}  // namespace mk_det
// ... and with the LM head on the tcgen05 tensor cores
namespace mk_umma {
cudaError_t prepare_megakernel();
int megakernel_occupancy(int* blocks);
cudaError_t launch_megakernel(const mk::Params& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                              bool cooperative, cudaStream_t st);
}  // namespace mk_umma
// ... and with the bf16 expert and dense-FFN items on them too
namespace mk_umma_ffn {
cudaError_t prepare_megakernel();
int megakernel_occupancy(int* blocks);
cudaError_t launch_megakernel(const mk::Params& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                              bool cooperative, cudaStream_t st);
}  // namespace mk_umma_ffn

namespace {
// the kernel build a plan runs: deterministic accumulators, the tensor-core LM head (and
// FFN items), or the default
cudaError_t launch_variant(const mk::Params& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                           bool cooperative, cudaStream_t st) {
  if (p.det) return mk_det::launch_megakernel(p, tk, tv, grid, cooperative, st);
  if (p.moe_umma) return mk_umma_ffn::launch_megakernel(p, tk, tv, grid, cooperative, st);
  if (p.lm_umma) return mk_umma::launch_megakernel(p, tk, tv, grid, cooperative, st);
  return mk::launch_megakernel(p, tk, tv, grid, cooperative, st);
}
}  // namespace

using namespace mk;

namespace {

thread_local std::string g_err;

// ------------------------------------------------------------------ shapes
struct Shape {
  int L, d, Hq, Hkv, hd, E, topk, f, V, gs, nrb_d, max_batch;
  int r_qkv, qkv_rows_group, qkv_tpg;
  int r_router, n_router_tasks, e_pad;
  int r_o, t_o, k_o;
  int moe_fs, t_moe;
  uint64_t dense_mask;  // mixed stacks: dense layers
  int f_dense, t_dense, dense_fs;  // dense FFN items: bf16, f-slices of dense_fs rows
  bool fp8;             // routed experts as E4M3 codes + f32 scales
  bool fp8d;            // QKV, O-proj and LM head as E4M3 codes + per-row f32 scales
  int esz;              // bytes of a QKV / O-proj / LM-head weight (2 bf16, 1 E4M3)
  int r_lm, v_pad, n_lm_tasks;
  int lm_umma;   // LM head on the tensor cores (64-row tiles in the core-matrix layout)
  int moe_umma;  // ... and the bf16 expert / dense-FFN items (32-row f-slices)
  size_t qkv_layer_bytes, o_layer_bytes, router_layer_bytes, moe_item_bytes, moe_bytes_e, lm_bytes, embed_bytes;
  size_t dense_item_bytes;
  size_t off_qkv, off_o, off_router, off_moe, off_dense, off_lm, off_embed, total;
  size_t off_qkv_scale, off_o_scale, off_lm_scale;  // FP8 projections' row scales (f32)
  bool dense(int l) const { return (dense_mask >> l) & 1ull; }
};

int fail(std::string* dst, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  if (dst) *dst = buf;
  return code;
}

int derive_shape(const mk_config* c, Shape& s, std::string* err) {
  if (!c) return fail(err, MK_ERR_INVALID, "config is NULL");
  s.L = c->n_layers; s.d = c->d_model; s.Hq = c->n_q_heads; s.Hkv = c->n_kv_heads; s.hd = c->head_dim;
  s.E = c->n_experts; s.topk = c->top_k; s.f = c->d_ff; s.V = c->vocab; s.max_batch = c->max_batch;
  if (s.L < 1 || s.L > 64) return fail(err, MK_ERR_UNSUPPORTED, "n_layers %d not in [1, 64]", s.L);
  if (s.hd != 32 && s.hd != 64 && s.hd != 128) return fail(err, MK_ERR_UNSUPPORTED, "head_dim %d not in {32,64,128}", s.hd);
  if (s.d < 256 || s.d % 256 || s.d > 2048) return fail(err, MK_ERR_UNSUPPORTED, "d_model %d must be a multiple of 256 <= 2048", s.d);
  if (s.f < 128 || s.f % 128 || s.f > 2048) return fail(err, MK_ERR_UNSUPPORTED, "d_ff %d must be a multiple of 128 <= 2048", s.f);
  if (s.Hkv < 1 || s.Hq < 1 || s.Hq % s.Hkv) return fail(err, MK_ERR_UNSUPPORTED, "n_q_heads %d not divisible by n_kv_heads %d", s.Hq, s.Hkv);
  s.gs = s.Hq / s.Hkv;
  if (s.gs > 8) return fail(err, MK_ERR_UNSUPPORTED, "query group %d > 8", s.gs);
  if (s.Hkv > 8) return fail(err, MK_ERR_UNSUPPORTED, "n_kv_heads %d > 8", s.Hkv);
  if ((s.gs * s.hd) % 128 || s.gs * s.hd > 1024) return fail(err, MK_ERR_UNSUPPORTED, "group*head_dim %d must be a multiple of 128 <= 1024", s.gs * s.hd);
  if (s.E < 8 || s.E > 256 || s.E % 8)
    return fail(err, MK_ERR_UNSUPPORTED, "n_experts %d: need a multiple of 8 in [8, 256]", s.E);
  if (s.topk < 1 || s.topk > 8 || s.topk > s.E) return fail(err, MK_ERR_UNSUPPORTED, "top_k %d not in [1, min(8, E)]", s.topk);
  if (c->page_size != 16) return fail(err, MK_ERR_UNSUPPORTED, "page_size %d != 16", c->page_size);
  if (s.max_batch < 1 || s.max_batch > kMaxBatch) return fail(err, MK_ERR_UNSUPPORTED, "max_batch %d not in [1, 8]", s.max_batch);
  if (s.V < 1) return fail(err, MK_ERR_INVALID, "vocab %d", s.V);
  if (c->sliding_window < 0) return fail(err, MK_ERR_INVALID, "sliding_window %d < 0", c->sliding_window);
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return fail(err, MK_ERR_INVALID, "bad rms_eps / rope_theta");
  s.nrb_d = s.d / kRowBlock;
  s.qkv_rows_group = (s.gs + 2) * s.hd;
  s.r_qkv = (s.qkv_rows_group % 32 == 0) ? 32 : 16;  // 128 KB tiles at d 2048: one fits the ring
  if (const char* e = getenv("MK_QKV_ROWS")) { const int v = atoi(e); if ((v == 16 || v == 32 || v == 64) && s.qkv_rows_group % v == 0) s.r_qkv = v; }
  s.qkv_tpg = s.qkv_rows_group / s.r_qkv;
  s.r_router = 16;
  if (const char* e = getenv("MK_ROUTER_ROWS")) { const int v = atoi(e); if (v == 16 || v == 32) s.r_router = v; }
  s.e_pad = (s.E + s.r_router - 1) / s.r_router * s.r_router;
  s.n_router_tasks = s.e_pad / s.r_router;
  // O-proj tiles of 128 rows x one KV group (256 KB at the pages scale): 64 tiles a
  // layer, each started by a free SM in the tail of the MoE phase (64-row tiles: -2.8%
  // at batch 1, the tail ran two deep on a third of the SMs)
  s.r_o = 128;
  if (const char* e = getenv("MK_OPROJ_ROWS")) { const int v = atoi(e); if (v == 32 || v == 64 || v == 128) s.r_o = v; }
  s.t_o = s.d / s.r_o; s.k_o = s.gs * s.hd;
  // MoE f-slice width: 32 rows of d_ff (measured best at the pages-scale shape against
  // 16/48/64: wider items start late on SMs still busy with attention items)
  s.moe_fs = (s.f % 32 == 0) ? 32 : 16;
  if (const char* e = getenv("MK_MOE_FS")) {
    const int v = atoi(e);
    if ((v == 16 || v == 32) && s.f % v == 0) s.moe_fs = v;
  }
  // FP8 experts: f-slices of 64 rows for handles of max_batch >= 4 (fewer, longer items:
  // +16% over 32-row items at batch 8 ragged), of 32 rows below (at batch 1 the 64-row
  // items occupy only 96 SMs: -4% against 32-row ones)
  if (c->expert_dtype != MK_EXPERT_BF16 && c->expert_dtype != MK_EXPERT_FP8 && c->expert_dtype != MK_WEIGHTS_FP8)
    return fail(err, MK_ERR_INVALID, "expert_dtype %d unknown", c->expert_dtype);
  s.fp8d = c->expert_dtype == MK_WEIGHTS_FP8;
  s.fp8 = c->expert_dtype == MK_EXPERT_FP8 || s.fp8d;
  s.esz = s.fp8d ? 1 : 2;
  if (s.fp8) {
    s.moe_fs = s.max_batch >= 4 ? 64 : 32;
    if (const char* e = getenv("MK_FP8_FS")) { const int v = atoi(e); if (v == 32 || v == 64) s.moe_fs = v; }
    if (s.f % s.moe_fs)
      return fail(err, MK_ERR_UNSUPPORTED, "FP8 experts need d_ff a multiple of %d (f-slices of %d)", s.moe_fs,
                  s.moe_fs);
  }
  s.t_moe = s.f / s.moe_fs;
  s.dense_mask = s.L < 64 ? c->dense_layer_mask & ((1ull << s.L) - 1) : c->dense_layer_mask;
  s.f_dense = s.dense_mask ? c->dense_ff : 0;
  if (s.dense_mask && (s.f_dense < 128 || s.f_dense % 128 || s.f_dense > 4096))
    return fail(err, MK_ERR_UNSUPPORTED, "dense_ff %d must be a multiple of 128 <= 4096", s.f_dense);
  // the dense FFN items keep the bf16 slice width (FP8 applies to the routed experts)
  s.dense_fs = s.fp8 ? 32 : s.moe_fs;
  s.t_dense = s.f_dense / s.dense_fs;
  s.r_lm = 64;
  if (const char* e = getenv("MK_LM_ROWS")) { const int v = atoi(e); if (v == 32 || v == 64 || v == 128) s.r_lm = v; }
  // MK_LM_UMMA=1 (read at mk_create): the LM head's tiles on the tcgen05 tensor cores,
  // 64 rows each (bf16 weights; d a multiple of 256, at most 2048)
  s.lm_umma = 0;
  if (const char* e = getenv("MK_LM_UMMA"))
    if (atoi(e) && !s.fp8d && s.d % 256 == 0 && s.d / 128 <= kMaxKsw) { s.lm_umma = 1; s.r_lm = 64; }
  // MK_MOE_UMMA=1 beside it: the bf16 expert and dense-FFN items (32-row f-slices) too
  s.moe_umma = 0;
  if (const char* e = getenv("MK_MOE_UMMA"))
    if (atoi(e) && s.lm_umma && !s.fp8 && s.moe_fs == 32 && s.dense_fs == 32) s.moe_umma = 1;
  s.v_pad = (s.V + s.r_lm - 1) / s.r_lm * s.r_lm; s.n_lm_tasks = s.v_pad / s.r_lm;
  s.qkv_layer_bytes = (size_t)s.Hkv * s.qkv_rows_group * s.d * s.esz;
  s.o_layer_bytes = (size_t)s.Hkv * s.d * s.k_o * s.esz;
  s.router_layer_bytes = (size_t)s.e_pad * s.d * 2;
  s.moe_item_bytes = s.fp8 ? (size_t)fp8_scale_bytes(s.moe_fs, s.d) + (size_t)3 * s.moe_fs * s.d
                           : (size_t)3 * s.moe_fs * s.d * 2;
  s.moe_bytes_e = s.moe_item_bytes * s.t_moe;
  s.dense_item_bytes = (size_t)3 * s.dense_fs * s.d * 2;
  s.lm_bytes = (size_t)s.v_pad * s.d * s.esz;
  s.embed_bytes = (size_t)s.V * s.d * 2;
  size_t o = 0;
  auto take = [&](size_t n) { size_t r = o; o += (n + 255) / 256 * 256; return r; };
  s.off_qkv = take(s.qkv_layer_bytes * s.L);
  s.off_o = take(s.o_layer_bytes * s.L);
  s.off_router = take(s.router_layer_bytes * s.L);
  s.off_moe = take(s.moe_bytes_e * s.E * s.L);
  s.off_dense = take((size_t)__builtin_popcountll(s.dense_mask) * s.t_dense * s.dense_item_bytes);
  s.off_lm = take(s.lm_bytes);
  s.off_embed = take(s.embed_bytes);
  s.off_qkv_scale = take(s.fp8d ? (size_t)s.L * s.Hkv * s.qkv_rows_group * 4 : 0);
  s.off_o_scale = take(s.fp8d ? (size_t)s.L * s.d * 4 : 0);
  s.off_lm_scale = take(s.fp8d ? (size_t)s.v_pad * 4 : 0);
  s.total = o;
  return MK_OK;
}

// ------------------------------------------------------------------ planner
enum Wave { W_QKV = 0, W_ROUTER, W_ATT, W_MOE, W_OPROJ, W_RESID, W_COUNT };

struct PlanOut {
  int B = 0, maxa = 0, n_sm = 0;
  int c_lr, c_qkvg, c_rt, c_rr, c_att, c_og, c_md, c_od, c_oa, c_done, n_ctr;
  int od_target;
  std::vector<int32_t> tasks;     // n_tasks * 32
  std::vector<int32_t> sm_off;    // n_segs * (n_sm + 1), absolute offsets into sm_list
  std::vector<int32_t> sm_list;
  int n_segs = 0;
  int n_tasks() const { return (int)(tasks.size() / kDescInts); }
};

bool parse_wave_order(const char* s, std::vector<int>& order) {
  // letters: q=QKV r=router a=attention m=MoE items o=O-proj x=ADD_RMSNORM
  order.clear();
  for (const char* c = s; *c; ++c) {
    switch (*c) {
      case 'q': order.push_back(W_QKV); break;
      case 'r': order.push_back(W_ROUTER); break;
      case 'a': order.push_back(W_ATT); break;
      case 'm': order.push_back(W_MOE); break;
      case 'x': order.push_back(W_RESID); break;
      case 'o': order.push_back(W_OPROJ); break;
      default: return false;
    }
  }
  if (order.size() != W_COUNT) return false;
  auto pos = [&](int w) { return (int)(std::find(order.begin(), order.end(), w) - order.begin()); };
  for (int w = 0; w < W_COUNT; ++w) if (pos(w) >= W_COUNT) return false;
  // every order that respects the dependencies is deadlock-free with in-order lists
  return pos(W_QKV) < pos(W_ATT) && pos(W_ATT) < pos(W_OPROJ) && pos(W_ROUTER) < pos(W_MOE) &&
         pos(W_MOE) < pos(W_RESID) && pos(W_OPROJ) < pos(W_RESID);
}

int build_plan(const Shape& s, int B, int n_sm, const std::vector<int>& order, PlanOut& P, std::string* err,
               int prefetch = 0, int router_sms = 0) {
  if (B < 1 || B > s.max_batch) return fail(err, MK_ERR_INVALID, "batch %d not in [1, %d]", B, s.max_batch);
  if (n_sm < 1) return fail(err, MK_ERR_INVALID, "n_sms %d", n_sm);
  P = PlanOut();
  P.B = B; P.n_sm = n_sm;
  P.maxa = std::min(s.E, B * s.topk);
  const int L = s.L;
  int c = 0;
  P.c_lr = c; c += L + 1;
  P.c_qkvg = c; c += L * s.Hkv;
  P.c_rt = c; c += L;
  P.c_rr = c; c += L;
  P.c_att = c; c += L * B * s.Hkv;
  P.c_og = c; c += L * s.Hkv;
  P.c_md = c; c += L;
  P.c_od = c; c += L;  // O-proj tiles done per layer (target od_target)
  P.c_oa = c; c += L;  // attention outputs complete per layer (target Hkv * B)
  P.c_done = c; c += 1;
  P.n_ctr = c;
  P.od_target = s.Hkv * s.t_o;  // O-proj tiles of a layer

  auto add = [&](int op, int layer, int aux, int row0, int nrows, int k0, int klen, int wc, int wt, int sc,
                 int st, size_t woff, int wbytes, int wave) {
    const int id = P.n_tasks();
    P.tasks.resize(P.tasks.size() + kDescInts, 0);
    int32_t* T = &P.tasks[(size_t)id * kDescInts];
    T[D_OP] = op; T[D_LAYER] = layer; T[D_AUX] = aux; T[D_ROW0] = row0; T[D_NROWS] = nrows;
    T[D_K0] = k0; T[D_KLEN] = klen; T[D_WAIT_CTR] = wc; T[D_WAIT_TARGET] = wt; T[D_SIG_CTR] = sc;
    T[D_SIG_TARGET] = st; T[D_WOFF_LO] = (int32_t)(uint32_t)(woff & 0xffffffffull);
    T[D_WOFF_HI] = (int32_t)(uint32_t)(woff >> 32); T[D_WBYTES] = wbytes; T[D_QUEUE] = -1;
    T[D_TASK_ID] = id; T[D_WAVE] = wave; T[D_WAIT2_CTR] = -1;
    return id;
  };

  // items a layer's MoE-done counter counts: every slot of the routed experts (the
  // route step pads the inactive ones), or the dense FFN's items
  auto md_target = [&](int l) { return s.dense(l) ? s.t_dense : P.maxa * s.t_moe; };
  // ---- descriptors
  const int t_embed = add(OP_EMBED, 0, 0, 0, 0, 0, 0, -1, 0, P.c_lr + 0, s.nrb_d, 0, 0, -1);
  std::vector<std::vector<int>> waves((size_t)L * W_COUNT);
  std::vector<int> drains((size_t)L * W_COUNT, -1);
  std::vector<int> moe_oq(L, -1);  // megakernel MoE drains that also serve the O-proj queue
  for (int l = 0; l < L; ++l) {
    // layer 0's QKV and router tiles wait for the embedding (its operand); the later
    // layers' wait for the previous layer's experts and O-proj tiles and build their
    // operand from its parts
    const int w1 = l == 0 ? P.c_lr : P.c_md + l - 1;
    const int t1 = l == 0 ? s.nrb_d : md_target(l - 1);
    auto wait2 = [&](int t) {
      if (l == 0) return t;
      P.tasks[(size_t)t * kDescInts + D_WAIT2_CTR] = P.c_od + l - 1;
      P.tasks[(size_t)t * kDescInts + D_WAIT2_TARGET] = P.od_target;
      return t;
    };
    auto& wq = waves[(size_t)l * W_COUNT + W_QKV];
    for (int g = 0; g < s.Hkv; ++g)
      for (int t = 0; t < s.qkv_tpg; ++t)
        wq.push_back(wait2(add(OP_QKV, l, g, t * s.r_qkv, s.r_qkv, 0, s.d, w1, t1, P.c_qkvg + l * s.Hkv + g,
                               s.qkv_tpg,
                               s.off_qkv + l * s.qkv_layer_bytes + (size_t)g * s.qkv_rows_group * s.d * s.esz +
                                   (size_t)t * s.r_qkv * s.d * s.esz,
                               s.r_qkv * s.d * s.esz, W_QKV)));
    auto& wr = waves[(size_t)l * W_COUNT + W_ROUTER];
    // the last tile (dealt last on its SM) collects all tiles' logits and routes (a
    // dense layer has no router)
    for (int t = 0; t < (s.dense(l) ? 0 : s.n_router_tasks); ++t)
      wr.push_back(wait2(add(OP_ROUTER, l, t == s.n_router_tasks - 1 ? 1 : 0, t * s.r_router, s.r_router, 0, s.d,
                             w1, t1, P.c_rt + l, s.n_router_tasks,
                             s.off_router + l * s.router_layer_bytes + (size_t)t * s.r_router * s.d * 2,
                             s.r_router * s.d * 2, W_ROUTER)));
    drains[(size_t)l * W_COUNT + W_ATT] = add(OP_ATT_DRAIN, l, 0, 0, 0, 0, 0, -1, 0, -1, 0, 0, 0, W_ATT);
    // D_AUX = 1: the dense FFN's items (every token, weight 1) instead of routed experts
    const int dz = s.dense(l) ? 1 : 0;
    // (a routed layer's items wait for its route, published once by the route step; a
    // dense layer's need no route; both count on the MoE-done counter)
    const int rr = s.dense(l) ? -1 : P.c_rr + l;
    drains[(size_t)l * W_COUNT + W_MOE] =
        add(OP_MOE_DRAIN, l, dz, 0, 0, 0, 0, rr, 1, P.c_md + l, md_target(l), 0, 0, W_MOE);
    moe_oq[l] = add(OP_MOE_DRAIN, l, dz, 0, 0, 0, 0, rr, 1, P.c_md + l, md_target(l), 0, 0, W_MOE);
    auto& wo = waves[(size_t)l * W_COUNT + W_OPROJ];
    for (int g = 0; g < s.Hkv; ++g)
      for (int t = 0; t < s.t_o; ++t)
        wo.push_back(add(OP_OPROJ, l, g, t * s.r_o, s.r_o, g * s.k_o, s.k_o, P.c_og + l * s.Hkv + g, B,
                         P.c_od + l, P.od_target,
                         s.off_o + l * s.o_layer_bytes + (size_t)g * s.d * s.k_o * s.esz +
                             (size_t)t * s.r_o * s.k_o * s.esz,
                         s.r_o * s.k_o * s.esz, W_OPROJ));
  }
  for (int l = 0; l < L; ++l) {
    auto& wx = waves[(size_t)l * W_COUNT + W_RESID];
    for (int r = 0; r < s.nrb_d; ++r) {
      const int t = add(OP_RESID, l, r, r * kRowBlock, kRowBlock, 0, 0, P.c_od + l, P.od_target,
                        P.c_lr + l + 1, s.nrb_d, 0, 0, W_RESID);
      P.tasks[(size_t)t * kDescInts + D_WAIT2_CTR] = P.c_md + l;
      P.tasks[(size_t)t * kDescInts + D_WAIT2_TARGET] = md_target(l);
      wx.push_back(t);
    }
  }
  std::vector<int> lm;
  for (int t = 0; t < s.n_lm_tasks; ++t)
    lm.push_back(add(OP_LMHEAD, L, 0, t * s.r_lm, s.r_lm, 0, s.d, P.c_lr + L, s.nrb_d, -1, 0,
                     s.off_lm + (size_t)t * s.r_lm * s.d * s.esz, s.r_lm * s.d * s.esz, -1));

  // ---- segments
  auto emit_segment = [&](const std::vector<std::vector<int>>& lists) {
    int o = (int)P.sm_list.size();
    for (int sm = 0; sm < n_sm; ++sm) {
      P.sm_off.push_back(o);
      for (int t : lists[sm]) P.sm_list.push_back(t);
      o += (int)lists[sm].size();
    }
    P.sm_off.push_back(o);
    P.n_segs++;
  };
  auto is_drain = [](int w) { return w == W_ATT || w == W_MOE; };
  // segment 0: the whole step for the megakernel
  {
    std::vector<std::vector<int>> lists(n_sm);
    lists[0].push_back(t_embed);
    long long cursor = 0;
    std::vector<char> has_router(n_sm);
    // router_sms > 0: every layer's router tiles on the last router_sms SMs, which take
    // no other work until the LM head; the other waves and the drains on the rest
    const int nrs = (router_sms > 0 && router_sms < n_sm && s.n_router_tasks > 0) ? router_sms : 0;
    const int nw = n_sm - nrs;
    auto pos = [&](int w) { return (int)(std::find(order.begin(), order.end(), w) - order.begin()); };
    // With O-proj after the MoE drain, the O-proj tiles are not dealt: the MoE drain
    // claims them from a queue, ahead of expert items once the layer's attention is
    // complete and all remaining ones after the expert queue is empty, so that they
    // run on whichever SMs are free instead of behind each SM's own expert items.
    // Not when the attention drain follows the MoE drain: a drain that holds an O-proj
    // tile waits for the layer's attention, which its own SM would only run later (with
    // as many O-proj tiles as SMs every SM could be holding one); those orders deal the
    // O-proj tiles statically, after the attention drain.
    const bool oq = pos(W_OPROJ) > pos(W_MOE) && pos(W_ATT) < pos(W_MOE);
    for (int l = 0; l < L && oq; ++l) {
      const auto& wo = waves[(size_t)l * W_COUNT + W_OPROJ];
      int32_t* D = &P.tasks[(size_t)moe_oq[l] * kDescInts];
      D[D_K0] = wo.empty() ? 0 : wo.front();
      D[D_KLEN] = (int)wo.size();
      for (size_t i = 1; i < wo.size(); ++i)
        if (wo[i] != wo[0] + (int)i) return fail(err, MK_ERR_INVALID, "O-proj descriptors not contiguous");
    }
    for (int l = 0; l < L; ++l) {
      std::fill(has_router.begin(), has_router.end(), 0);
      for (int w : order) {
        if (oq && w == W_OPROJ) continue;
        if (oq && w == W_MOE) {
          for (int sm = 0; sm < nw; ++sm) lists[sm].push_back(moe_oq[l]);
        } else if (is_drain(w)) {
          for (int sm = 0; sm < nw; ++sm) lists[sm].push_back(drains[(size_t)l * W_COUNT + w]);
        } else if (nrs > 0) {
          int k = 0;
          for (int t : waves[(size_t)l * W_COUNT + w]) {
            if (w == W_ROUTER) lists[nw + (k++ % nrs)].push_back(t);
            else lists[cursor++ % nw].push_back(t);
          }
        } else if (w == W_QKV && pos(W_ROUTER) < pos(W_QKV) && n_sm > s.n_router_tasks) {
          // the router tiles head the MoE's critical path and the QKV tiles the
          // attention's: keep the QKV tiles off the SMs that run this layer's router
          for (int t : waves[(size_t)l * W_COUNT + w]) {
            while (has_router[cursor % n_sm]) ++cursor;
            lists[cursor++ % n_sm].push_back(t);
          }
        } else {
          for (int t : waves[(size_t)l * W_COUNT + w]) {
            if (w == W_ROUTER) has_router[cursor % n_sm] = 1;
            lists[cursor++ % n_sm].push_back(t);
          }
        }
      }
    }
    for (int t : lm) lists[cursor++ % n_sm].push_back(t);
    if (prefetch) {
      // L2 prefetch entries around each layer's attention drain: before it, this
      // layer's K/V pages (each SM a share) and the weights of this SM's own O-proj
      // tiles of the layer; after it, the weights of its QKV and router tiles of the
      // next layer.  The producer reaches the drain about when the layer's QKV tiles
      // start, and the attention queue empties about when its MoE items start.
      auto field = [&](int t, int f) { return P.tasks[(size_t)t * kDescInts + f]; };
      auto pf_of = [&](int t) {
        const size_t off = ((size_t)(uint32_t)field(t, D_WOFF_HI) << 32) | (uint32_t)field(t, D_WOFF_LO);
        return add(OP_PREFETCH, field(t, D_LAYER), field(t, D_TASK_ID), 0, 0, 0, 0, -1, 0, -1, 0, off,
                   field(t, D_WBYTES), -1);
      };
      std::vector<int> pf_kv(L);
      for (int l = 0; l < L; ++l) pf_kv[l] = add(OP_PREFETCH_KV, l, 0, 0, 0, 0, 0, -1, 0, -1, 0, 0, 0, -1);
      for (int sm = 0; sm < n_sm; ++sm) {
        const std::vector<int> in = lists[sm];
        std::vector<int>& out = lists[sm];
        out.clear();
        for (size_t i = 0; i < in.size(); ++i) {
          const int t = in[i];
          if (field(t, D_OP) != OP_ATT_DRAIN) { out.push_back(t); continue; }
          const int l = field(t, D_LAYER);
          if (prefetch & 1) out.push_back(pf_kv[l]);
          if (prefetch & 4) {  // this SM's share of the layer's O-proj weights (512-byte units)
            const size_t units = s.o_layer_bytes / 512;
            const size_t u0 = units * sm / n_sm, u1 = units * (sm + 1) / n_sm;
            if (u1 > u0)
              out.push_back(add(OP_PREFETCH, l, 0, 0, 0, 0, 0, -1, 0, -1, 0,
                                s.off_o + l * s.o_layer_bytes + u0 * 512, (int)((u1 - u0) * 512), -1));
          }
          if (prefetch & 2)
            for (size_t j = i + 1; j < in.size() && field(in[j], D_LAYER) <= l; ++j)
              if (field(in[j], D_OP) == OP_OPROJ) out.push_back(pf_of(in[j]));
          out.push_back(t);
          if (prefetch & 2)
            for (size_t j = i + 1; j < in.size() && field(in[j], D_LAYER) <= l + 1; ++j) {
              const int op = field(in[j], D_OP);
              if (field(in[j], D_LAYER) == l + 1 && (op == OP_QKV || op == OP_ROUTER)) out.push_back(pf_of(in[j]));
            }
        }
      }
    }
    emit_segment(lists);
  }
  // segments 1..: one launch per wave per layer (embed first, LM head last)
  {
    std::vector<std::vector<int>> lists(n_sm);
    lists[0].push_back(t_embed);
    emit_segment(lists);
    for (int l = 0; l < L; ++l)
      for (int w : order) {
        std::vector<std::vector<int>> ls(n_sm);
        if (is_drain(w)) {
          for (int sm = 0; sm < n_sm; ++sm) ls[sm].push_back(drains[(size_t)l * W_COUNT + w]);
        } else {
          long long cur = 0;
          for (int t : waves[(size_t)l * W_COUNT + w]) ls[cur++ % n_sm].push_back(t);
        }
        emit_segment(ls);
      }
    std::vector<std::vector<int>> ll(n_sm);
    long long cur = 0;
    for (int t : lm) ll[cur++ % n_sm].push_back(t);
    emit_segment(ll);
  }
  return MK_OK;
}

// Pages per attention split, in whole 8-page ring stages.  The base size gives about 32
// splits per (sequence, group) at the longest context.  Every SM claims splits and a
// split is one long serial stream of pages, so a layer's attention ends with its longest
// run of splits on one SM.  Where the base size's splits of a full-attention layer do
// not fit the SMs in one wave, or fit with long splits (128 pages or more) and SMs to
// spare, the size becomes the smallest for which they fit, with one more split per
// (sequence, group) for the sequences to grow into before the next plan.  (Same-box
// A/Bs: 128K, 37 splits of 224 pages per group on 152 SMs against 32 of 256: +5.7%;
// batch 8 ragged up to 32K, 120 splits of 296 pages against 508 of 64: +1.5%; at 8K,
// 32 splits of 16 pages per group against the base 22 of 24: -9%, so short splits keep
// the base size.)
int choose_split_pages(const int32_t* lens, int B, int Hkv, int n_sm, int max_pages) {
  int base = (max_pages + 31) / 32;
  base = std::max(8, (base + 7) / 8 * 8);
  std::vector<int> npg(B);
  int longest = 0;
  for (int b = 0; b < B; ++b) {
    npg[b] = lens[b] > 0 ? (lens[b] - 1) / 16 + 1 : 0;  // pages of the cached keys
    longest = std::max(longest, npg[b]);
  }
  auto splits = [&](int sp) {
    long long n = 0;
    for (int b = 0; b < B; ++b) n += (npg[b] + sp - 1) / sp;
    return n * Hkv;
  };
  const long long budget = (long long)n_sm - (long long)B * Hkv;
  if (budget <= 0 || (splits(base) <= budget && base < 128)) return base;
  for (int sp = 8; sp < longest + 8; sp += 8)
    if (splits(sp) <= budget) return sp;
  return base;
}

constexpr int kDefaultPrefetch = 0;

// L2 prefetch entries in the megakernel's lists, as a bit mask (MK_PREFETCH): 1 = each
// SM's share of the layer's cached K/V pages, 2 = the weights of the SM's own later
// static tiles (next layer's QKV and router), 4 = each SM's share of the layer's O-proj
// weights (the O-proj tiles are claimed later, from a queue).
int prefetch_mask() {
  const char* e = getenv("MK_PREFETCH");
  return e ? atoi(e) : kDefaultPrefetch;
}

// SMs reserved for the router tiles (MK_ROUTER_SMS; 0 = none): see build_plan.
int router_sms() {
  const char* e = getenv("MK_ROUTER_SMS");
  return e ? atoi(e) : 0;
}

// Router first: its weights are then prefetched behind the previous layer's tasks
// rather than behind this layer's QKV tiles.
const char* default_order() { return "rqamox"; }

}  // namespace

// ------------------------------------------------------------------ handle
struct mk_handle {
  mk_config cfg;
  Shape s;
  int dev = 0, n_sm = 0;
  std::string err;
  uint8_t* wblob = nullptr;
  float* norms = nullptr;  // attn [L][d] then final [d]
  unsigned long long* rope_turns = nullptr;  // [hd/2]
  // plan
  bool planned = false;
  PlanOut P;
  int B = 0, max_pages = 0, n_pages = 0, split_pages = 0, max_items_bg = 0;
  const int32_t* page_table = nullptr;
  std::vector<void*> bufs;  // plan allocations
  int32_t *d_tasks = nullptr, *d_sm_off = nullptr, *d_sm_list = nullptr;
  Params prm{};
  int32_t* d_tokens = nullptr;
  float* d_logits = nullptr;
  unsigned* d_trace_n = nullptr;
  unsigned* d_snap = nullptr;  // inspection copy: counters, queue heads, queue counts
  bool last_noalloc = false;   // the last step ran in the static scratch (mk_read follows it)
  int inspect = 0;
  int fixed = 0;
  int det = 0;     // deterministic accumulation, from the next mk_plan (mk_set_deterministic)
  cudaStream_t last_stream = nullptr;
  // tensor maps
  CUtensorMap tmK{}, tmV{};
  void *tm_k = nullptr, *tm_v = nullptr;
  // graph of the per-op launches
  cudaGraphExec_t graph = nullptr;
  const void* g_key[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  int g_fixed = -1;
};

namespace {

int cuda_fail(mk_handle* h, cudaError_t e, const char* what) {
  return fail(h ? &h->err : nullptr, MK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(h, call)                                              \
  do {                                                           \
    cudaError_t _e = (call);                                     \
    if (_e != cudaSuccess) return cuda_fail((h), _e, #call);     \
  } while (0)

void free_plan(mk_handle* h) {
  for (void* p : h->bufs) cudaFree(p);
  h->bufs.clear();
  if (h->graph) { cudaGraphExecDestroy(h->graph); h->graph = nullptr; }
  h->planned = false;
  h->tm_k = h->tm_v = nullptr;
}

template <class T>
int alloc(mk_handle* h, T** p, size_t count) {
  void* q = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 16);
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) return fail(&h->err, MK_ERR_OOM, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
  e = cudaMemset(q, 0, bytes);
  if (e != cudaSuccess) { cudaFree(q); return cuda_fail(h, e, "cudaMemset"); }
  h->bufs.push_back(q);
  *p = static_cast<T*>(q);
  return MK_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 2-D view of a K or V pool: rows = (layer, page, kv head, token), columns = head dim.
int encode_kv_map(mk_handle* h, CUtensorMap* tm, void* base) {
  auto fn = get_encode();
  if (!fn) return fail(&h->err, MK_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const Shape& s = h->s;
  const cuuint64_t rows = (cuuint64_t)s.L * h->n_pages * s.Hkv * 16;
  // One box per (page, KV head): all 16 keys x head_dim.  A 128-byte swizzle span
  // holds 64 bf16, so a 128-wide row is addressed as two 64-column halves (a 3-D map:
  // column, half, row) and the box lands as 32 swizzled 128-byte lines, row-major.
  CUresult r;
  if (s.hd == 128) {
    cuuint64_t dims[3] = {64, 2, rows};
    cuuint64_t strides[2] = {128, (cuuint64_t)s.hd * 2};
    cuuint32_t box[3] = {64, 2, 16};
    cuuint32_t estr[3] = {1, 1, 1};
    r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[2] = {(cuuint64_t)s.hd, rows};
    cuuint64_t strides[1] = {(cuuint64_t)s.hd * 2};
    cuuint32_t box[2] = {(cuuint32_t)s.hd, 16};
    cuuint32_t estr[2] = {1, 1};
    r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, s.hd == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return fail(&h->err, MK_ERR_INVALID, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MK_OK;
}

int prepare_step(mk_handle* h, const int32_t* tokens, void* k, void* v, float* logits) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  if (!h->planned) return fail(&h->err, MK_ERR_STATE, "mk_plan has not been called");
  if (!tokens || !k || !v || !logits) return fail(&h->err, MK_ERR_INVALID, "NULL step pointer");
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15)
    return fail(&h->err, MK_ERR_INVALID, "K/V pools must be 16-byte aligned");
  CK(h, cudaSetDevice(h->dev));
  if (k != h->tm_k) { int r = encode_kv_map(h, &h->tmK, k); if (r) return r; h->tm_k = k; }
  if (v != h->tm_v) { int r = encode_kv_map(h, &h->tmV, v); if (r) return r; h->tm_v = v; }
  Params& p = h->prm;
  p.tokens = tokens;
  p.kc = static_cast<uint16_t*>(k);
  p.vc = static_cast<uint16_t*>(v);
  p.logits = logits;
  p.fixed = h->fixed;
  return MK_OK;
}

int launch_segment(mk_handle* h, int seg, bool cooperative, bool reset, cudaStream_t st) {
  Params p = h->prm;
  p.sm_off = h->d_sm_off + (size_t)seg * (h->n_sm + 1);
  p.do_reset = reset ? 1 : 0;
  cudaError_t e = launch_variant(p, h->tmK, h->tmV, h->n_sm, cooperative, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "megakernel launch");
  return MK_OK;
}

}  // namespace

// ================================================================== C ABI
extern "C" {

int mk_version(void) { return 1; }

const char* mk_last_error(mk_handle* h) { return h ? h->err.c_str() : g_err.c_str(); }

int mk_create(const mk_config* cfg, const mk_weights* w, void* stream, mk_handle** out) {
  if (!out) return fail(nullptr, MK_ERR_INVALID, "out is NULL");
  *out = nullptr;
  Shape s;
  int r = derive_shape(cfg, s, nullptr);
  if (r) return r;
  if (!w || !w->embed || !w->lm_head || !w->final_norm || !w->attn_norm || !w->wq || !w->wk || !w->wv ||
      !w->wo || !w->router || !w->w_gate || !w->w_up || !w->w_down)
    return fail(nullptr, MK_ERR_INVALID, "weights struct has a NULL member");
  for (int l = 0; l < s.L; ++l) {
    if (!w->attn_norm[l] || !w->wq[l] || !w->wk[l] || !w->wv[l] || !w->wo[l] || (!s.dense(l) && !w->router[l]))
      return fail(nullptr, MK_ERR_INVALID, "NULL weight pointer at layer %d", l);
    if (s.dense(l)) {
      if (!w->ffn_gate || !w->ffn_up || !w->ffn_down || !w->ffn_gate[l] || !w->ffn_up[l] || !w->ffn_down[l])
        return fail(nullptr, MK_ERR_INVALID, "NULL dense FFN pointer at layer %d", l);
      continue;
    }
    for (int e = 0; e < s.E; ++e) {
      const int i = l * s.E + e;
      if (!w->w_gate[i] || !w->w_up[i] || !w->w_down[i])
        return fail(nullptr, MK_ERR_INVALID, "NULL expert pointer at index %d", i);
    }
  }

  mk_handle* h = new mk_handle();
  h->cfg = *cfg;
  if (h->cfg.timeout_ms <= 0) h->cfg.timeout_ms = 2000;
  h->s = s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto bail = [&](int code) { *out = nullptr; mk_destroy(h); return code; };
  cudaError_t e = cudaGetDevice(&h->dev);
  if (e != cudaSuccess) { cuda_fail(h, e, "cudaGetDevice"); return bail(MK_ERR_CUDA); }
  e = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->dev);
  if (e != cudaSuccess) { cuda_fail(h, e, "cudaDeviceGetAttribute"); return bail(MK_ERR_CUDA); }
  int smem_optin = 0;
  cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev);
  if (smem_optin < kSmemBytes) {
    fail(&h->err, MK_ERR_UNSUPPORTED, "device allows %d B shared memory per block, kernel needs %d", smem_optin, kSmemBytes);
    return bail(MK_ERR_UNSUPPORTED);
  }
  e = prepare_megakernel();
  if (e == cudaSuccess) e = mk_det::prepare_megakernel();
  if (e == cudaSuccess) e = mk_umma::prepare_megakernel();
  if (e == cudaSuccess) e = mk_umma_ffn::prepare_megakernel();
  if (e != cudaSuccess) { cuda_fail(h, e, "cudaFuncSetAttribute"); return bail(MK_ERR_CUDA); }
  e = cudaMalloc(&h->wblob, s.total);
  if (e != cudaSuccess) { fail(&h->err, MK_ERR_OOM, "packed weights (%zu B): %s", s.total, cudaGetErrorString(e)); return bail(MK_ERR_OOM); }
  e = cudaMalloc(&h->norms, sizeof(float) * ((size_t)s.L * s.d + s.d));
  if (e != cudaSuccess) { fail(&h->err, MK_ERR_OOM, "norms: %s", cudaGetErrorString(e)); return bail(MK_ERR_OOM); }
  {
    // RoPE inverse frequencies theta^(-2i/hd) as exact 0.64 fixed-point turns per position
    std::vector<unsigned long long> turns(s.hd / 2);
    for (int i = 0; i < s.hd / 2; ++i) {
      const long double inv = powl((long double)cfg->rope_theta, -2.0L * i / s.hd);
      const long double t = inv / (2.0L * 3.14159265358979323846264338327950288L);
      turns[i] = (unsigned long long)(t * 18446744073709551616.0L);
    }
    e = cudaMalloc(&h->rope_turns, turns.size() * sizeof(unsigned long long));
    if (e != cudaSuccess) { fail(&h->err, MK_ERR_OOM, "rope table: %s", cudaGetErrorString(e)); return bail(MK_ERR_OOM); }
    e = cudaMemcpy(h->rope_turns, turns.data(), turns.size() * sizeof(unsigned long long), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) { cuda_fail(h, e, "rope table copy"); return bail(MK_ERR_CUDA); }
  }

  // ---- pack
  const int L = s.L, d = s.d, hd = s.hd, gs = s.gs, f = s.f, E = s.E;
#define PK(...)                                                          \
  do {                                                                   \
    cudaError_t _e = launch_pack(__VA_ARGS__, st);                       \
    if (_e != cudaSuccess) { cuda_fail(h, _e, "pack"); return bail(MK_ERR_CUDA); } \
  } while (0)
  // FP8 projections: each packed row's scale (over the whole source row), then the codes
#define PK8(dst, scales, a, b, c, rows, srows, K, ld, col0, mode, grp, tile)                                    \
  do {                                                                                                    \
    cudaError_t _e = launch_pack_fp8(dst, scales, a, b, c, rows, srows, K, ld, col0, mode, hd, gs, grp, tile, st); \
    if (_e != cudaSuccess) { cuda_fail(h, _e, "pack fp8"); return bail(MK_ERR_CUDA); }                    \
  } while (0)
#define PKS(scales, a, b, c, rows, srows, kfull, ld, mode, grp)                                               \
  do {                                                                                                    \
    cudaError_t _e = launch_pack_rowscale(scales, a, b, c, rows, srows, kfull, ld, mode, hd, gs, grp, st);      \
    if (_e != cudaSuccess) { cuda_fail(h, _e, "pack fp8 scales"); return bail(MK_ERR_CUDA); }             \
  } while (0)
  float* qkv_sc = reinterpret_cast<float*>(h->wblob + s.off_qkv_scale);
  float* o_sc = reinterpret_cast<float*>(h->wblob + s.off_o_scale);
  float* lm_sc = reinterpret_cast<float*>(h->wblob + s.off_lm_scale);
  for (int l = 0; l < L; ++l) {
    uint8_t* q = h->wblob + s.off_qkv + l * s.qkv_layer_bytes;
    for (int g = 0; g < s.Hkv; ++g) {
      if (s.fp8d) {
        float* sc = qkv_sc + ((size_t)l * s.Hkv + g) * s.qkv_rows_group;
        PKS(sc, w->wq[l], w->wk[l], w->wv[l], s.qkv_rows_group, 0, d, d, PACK_QKV, g);
        PK8(q + (size_t)g * s.qkv_rows_group * d, sc, w->wq[l], w->wk[l], w->wv[l], s.qkv_rows_group, 0, d, d, 0,
            PACK_QKV, g, s.r_qkv);
      } else {
        PK(q + (size_t)g * s.qkv_rows_group * d * 2, w->wq[l], w->wk[l], w->wv[l], s.qkv_rows_group, 0, d, d, 0,
           PACK_QKV, hd, gs, g, s.r_qkv);
      }
    }
    uint8_t* o = h->wblob + s.off_o + l * s.o_layer_bytes;
    if (s.fp8d)  // one scale per row of Wo, over all its Hq * hd columns (every KV group's slice)
      PKS(o_sc + (size_t)l * d, w->wo[l], nullptr, nullptr, d, d, s.Hq * hd, (long long)s.Hq * hd, PACK_IDENT, 0);
    for (int g = 0; g < s.Hkv; ++g) {
      if (s.fp8d)
        PK8(o + (size_t)g * d * s.k_o, o_sc + (size_t)l * d, w->wo[l], nullptr, nullptr, d, d, s.k_o,
            (long long)s.Hq * hd, g * s.k_o, PACK_IDENT, 0, s.r_o);
      else
        PK(o + (size_t)g * d * s.k_o * 2, w->wo[l], nullptr, nullptr, d, d, s.k_o, (long long)s.Hq * hd, g * s.k_o,
           PACK_IDENT, hd, gs, 0, s.r_o);
    }
    if (s.dense(l)) {  // mixed stack: the layer's FFN in the dense region, no router or experts
      const int rank = __builtin_popcountll(s.dense_mask & ((1ull << l) - 1ull));  // dense layers before l
      uint8_t* dd = h->wblob + s.off_dense + (size_t)rank * s.t_dense * s.dense_item_bytes;
      e = s.moe_umma ? launch_pack_moe_umma(dd, w->ffn_gate[l], w->ffn_up[l], w->ffn_down[l], d, s.f_dense, st)
                     : launch_pack_moe(dd, w->ffn_gate[l], w->ffn_up[l], w->ffn_down[l], d, s.f_dense, s.dense_fs, st);
      if (e != cudaSuccess) { cuda_fail(h, e, "pack dense FFN"); return bail(MK_ERR_CUDA); }
      e = launch_convert(h->norms + (size_t)l * d, w->attn_norm[l], d, st);
      if (e != cudaSuccess) { cuda_fail(h, e, "convert"); return bail(MK_ERR_CUDA); }
      continue;
    }
    PK(h->wblob + s.off_router + l * s.router_layer_bytes, w->router[l], nullptr, nullptr, s.e_pad, E, d, d, 0,
       PACK_IDENT, hd, gs, 0, s.r_router);
    for (int e2 = 0; e2 < E; ++e2) {
      const int i = l * E + e2;
      e = s.fp8 ? launch_pack_moe_fp8(h->wblob + s.off_moe + (size_t)i * s.moe_bytes_e, w->w_gate[i], w->w_up[i],
                                      w->w_down[i], d, f, s.moe_fs, (long long)s.moe_item_bytes, st)
                : s.moe_umma ? launch_pack_moe_umma(h->wblob + s.off_moe + (size_t)i * s.moe_bytes_e, w->w_gate[i],
                                                    w->w_up[i], w->w_down[i], d, f, st)
                : launch_pack_moe(h->wblob + s.off_moe + (size_t)i * s.moe_bytes_e, w->w_gate[i], w->w_up[i],
                                  w->w_down[i], d, f, s.moe_fs, st);
      if (e != cudaSuccess) { cuda_fail(h, e, "pack moe"); return bail(MK_ERR_CUDA); }
    }
    e = launch_convert(h->norms + (size_t)l * d, w->attn_norm[l], d, st);
    if (e != cudaSuccess) { cuda_fail(h, e, "convert"); return bail(MK_ERR_CUDA); }
  }
  if (s.fp8d) {
    PKS(lm_sc, w->lm_head, nullptr, nullptr, s.v_pad, s.V, d, d, PACK_IDENT, 0);
    PK8(h->wblob + s.off_lm, lm_sc, w->lm_head, nullptr, nullptr, s.v_pad, s.V, d, d, 0, PACK_IDENT, 0, s.r_lm);
  } else if (s.lm_umma) {
    e = launch_pack_umma(h->wblob + s.off_lm, w->lm_head, s.v_pad, s.V, d, st);
    if (e != cudaSuccess) { cuda_fail(h, e, "pack"); return bail(MK_ERR_CUDA); }
  } else {
    PK(h->wblob + s.off_lm, w->lm_head, nullptr, nullptr, s.v_pad, s.V, d, d, 0, PACK_IDENT, hd, gs, 0, s.r_lm);
  }
#undef PK
#undef PK8
#undef PKS
  e = launch_convert(h->norms + (size_t)L * d, w->final_norm, d, st);
  if (e != cudaSuccess) { cuda_fail(h, e, "convert"); return bail(MK_ERR_CUDA); }
  e = cudaMemcpyAsync(h->wblob + s.off_embed, w->embed, s.embed_bytes, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) { cuda_fail(h, e, "embed copy"); return bail(MK_ERR_CUDA); }
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) { cuda_fail(h, e, "pack sync"); return bail(MK_ERR_CUDA); }
  *out = h;
  return MK_OK;
}

int mk_plan_dry(const mk_config* cfg, int batch, int n_sms, int32_t* tasks_out, int cap_tasks,
                int32_t* sm_off_out, int32_t* sm_list_out, int cap_list, int32_t* info_out) {
  Shape s;
  int r = derive_shape(cfg, s, nullptr);
  if (r) return r;
  std::vector<int> order;
  const char* env = getenv("MK_WAVE_ORDER");
  if (!parse_wave_order(env && *env ? env : default_order(), order))
    return fail(nullptr, MK_ERR_INVALID, "bad wave order '%s'", env ? env : "");
  PlanOut P;
  r = build_plan(s, batch, n_sms, order, P, nullptr, prefetch_mask(), router_sms());
  if (r) return r;
  const int list_len = P.sm_off[n_sms];  // segment 0 only
  if (info_out) {
    int32_t* I = info_out;
    I[0] = P.n_tasks(); I[1] = list_len; I[2] = P.n_ctr; I[3] = P.maxa; I[4] = 0;
    I[5] = s.t_moe; I[6] = (int)(s.moe_item_bytes / 1024); I[7] = s.r_o; I[8] = s.moe_fs; I[9] = s.r_qkv; I[10] = s.qkv_tpg;
    I[11] = s.n_router_tasks; I[12] = P.od_target; I[13] = P.c_done; I[14] = P.n_segs; I[15] = s.n_lm_tasks;
    I[16] = P.c_lr; I[17] = P.c_qkvg; I[18] = P.c_rt; I[19] = P.c_rr; I[20] = P.c_att; I[21] = P.c_og;
    I[22] = P.c_md; I[23] = P.c_od; I[24] = s.nrb_d; I[25] = s.gs; I[26] = P.c_oa;
    I[27] = s.t_dense; I[28] = (int32_t)(uint32_t)(s.dense_mask & 0xffffffffull);
    I[29] = (int32_t)(uint32_t)(s.dense_mask >> 32);
    I[30] = s.fp8d ? MK_WEIGHTS_FP8 : s.fp8 ? MK_EXPERT_FP8 : MK_EXPERT_BF16; I[31] = (int32_t)s.moe_item_bytes;
  }
  if (!tasks_out || !sm_off_out || !sm_list_out || cap_tasks < P.n_tasks() || cap_list < list_len)
    return fail(nullptr, MK_ERR_INVALID, "output capacity too small (tasks %d, list %d)", P.n_tasks(), list_len);
  std::memcpy(tasks_out, P.tasks.data(), P.tasks.size() * sizeof(int32_t));
  std::memcpy(sm_off_out, P.sm_off.data(), (n_sms + 1) * sizeof(int32_t));
  std::memcpy(sm_list_out, P.sm_list.data(), list_len * sizeof(int32_t));
  return MK_OK;
}

int mk_plan(mk_handle* h, int batch, const int32_t* seq_lens_host, const int32_t* page_table_dev,
            int max_pages_per_seq, int n_pages) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  if (!seq_lens_host || !page_table_dev) return fail(&h->err, MK_ERR_INVALID, "NULL seq_lens or page table");
  if (max_pages_per_seq < 1 || n_pages < 1) return fail(&h->err, MK_ERR_INVALID, "max_pages_per_seq/n_pages < 1");
  const Shape& s = h->s;
  if (batch < 1 || batch > s.max_batch) return fail(&h->err, MK_ERR_INVALID, "batch %d not in [1, %d]", batch, s.max_batch);
  for (int b = 0; b < batch; ++b)
    if (seq_lens_host[b] < 0 || seq_lens_host[b] >= max_pages_per_seq * 16)
      return fail(&h->err, MK_ERR_INVALID, "seq_len[%d] = %d does not fit %d pages", b, seq_lens_host[b], max_pages_per_seq);
  if ((long long)s.L * n_pages * s.Hkv * 16 >= (1ll << 31))
    return fail(&h->err, MK_ERR_UNSUPPORTED, "K/V pool too large for 32-bit row coordinates");
  CK(h, cudaSetDevice(h->dev));
  CK(h, cudaDeviceSynchronize());
  free_plan(h);
  std::vector<int> order;
  const char* env = getenv("MK_WAVE_ORDER");
  if (!parse_wave_order(env && *env ? env : default_order(), order))
    return fail(&h->err, MK_ERR_INVALID, "bad wave order '%s'", env ? env : "");
  int r = build_plan(s, batch, h->n_sm, order, h->P, &h->err, prefetch_mask(), router_sms());
  if (r) return r;
  int occ = 0;
  if (h->det) mk_det::megakernel_occupancy(&occ);
  else if (h->s.moe_umma) mk_umma_ffn::megakernel_occupancy(&occ);
  else if (h->s.lm_umma) mk_umma::megakernel_occupancy(&occ);
  else megakernel_occupancy(&occ);
  if (occ < 1) return fail(&h->err, MK_ERR_UNSUPPORTED, "megakernel cannot be resident (occupancy %d)", occ);
  PlanOut& P = h->P;
  h->B = batch;
  h->max_pages = max_pages_per_seq;
  h->n_pages = n_pages;
  h->page_table = page_table_dev;
  h->split_pages = choose_split_pages(seq_lens_host, batch, s.Hkv, h->n_sm, max_pages_per_seq);
  if (const char* sp = getenv("MK_SPLIT_PAGES")) { int v = atoi(sp); if (v >= 8 && v % 8 == 0) h->split_pages = v; }
  h->max_items_bg = (max_pages_per_seq + h->split_pages - 1) / h->split_pages + 1;

  Params& p = h->prm;
  p = Params{};
  const int L = s.L, B = batch;
  p.L = L; p.d = s.d; p.Hq = s.Hq; p.Hkv = s.Hkv; p.hd = s.hd; p.E = s.E; p.topk = s.topk; p.f = s.f;
  p.V = s.V; p.gs = s.gs; p.nrb_d = s.nrb_d; p.B = B; p.maxa = P.maxa;
  p.max_pages = max_pages_per_seq; p.n_pages = n_pages; p.window = h->cfg.sliding_window;
  p.swa_mask = h->cfg.swa_layer_mask; p.theta = h->cfg.rope_theta; p.eps = h->cfg.rms_eps;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)s.hd));
  p.split_pages = h->split_pages; p.max_items_bg = h->max_items_bg;
  p.moe_fs = s.moe_fs; p.t_moe = s.t_moe; p.qkv_tpg = s.qkv_tpg;
  p.n_router_tasks = s.n_router_tasks;
  p.timeout_ns = (long long)h->cfg.timeout_ms * 1000000ll;
  p.n_steps = 1; p.tok_out = nullptr;  // one step, no greedy tokens (mk_decode_steps sets both)
  p.inflight = 2;
  if (const char* fl = getenv("MK_INFLIGHT")) { int v = atoi(fl); if (v >= 1 && v < kStages) p.inflight = v; }
  // expert items: 3 chunks in flight per SM from batch 4 up (the MoE phase streams
  // ~1200 items a layer at batch 8 and is bandwidth-bound: +3%), 2 below (at batch 1
  // it is latency-bound and a deeper window measured 2.6% slower)
  p.inflight_moe = B >= 4 ? std::min(3, kStages - 1) : p.inflight;
  if (const char* fl = getenv("MK_INFLIGHT_MOE")) { int v = atoi(fl); if (v >= 1 && v < kStages) p.inflight_moe = v; }
  p.tail_items = 0;
  p.inflight_tail = 4;
  if (const char* e = getenv("MK_TAIL_ITEMS")) { int v = atoi(e); if (v >= 0) p.tail_items = v; }
  if (const char* e = getenv("MK_INFLIGHT_TAIL")) { int v = atoi(e); if (v >= 1 && v < kStages) p.inflight_tail = v; }
  p.route_warp = 0;
  if (const char* e = getenv("MK_ROUTE_WARP")) p.route_warp = atoi(e) ? 1 : 0;
  p.route_pf_bytes = 0;
  if (const char* e = getenv("MK_ROUTE_PF")) {
    int v = atoi(e);
    if (v >= 0 && v % 16 == 0 && v <= (int)s.moe_item_bytes) p.route_pf_bytes = v;
  }
  p.wblob = h->wblob; p.off_moe = (long long)s.off_moe; p.moe_item_bytes = (long long)s.moe_item_bytes;
  p.dense_mask = s.dense_mask; p.t_dense = s.t_dense; p.off_dense = (long long)s.off_dense;
  p.dense_fs = s.dense_fs; p.dense_item_bytes = (long long)s.dense_item_bytes;
  p.fp8 = s.fp8 ? 1 : 0;
  p.fp8d = s.fp8d ? 1 : 0;
  p.lm_umma = s.lm_umma;
  p.moe_umma = s.moe_umma;
  p.qkv_rows_group = s.qkv_rows_group;
  p.qkv_scale = reinterpret_cast<const float*>(h->wblob + s.off_qkv_scale);
  p.o_scale = reinterpret_cast<const float*>(h->wblob + s.off_o_scale);
  p.lm_scale = reinterpret_cast<const float*>(h->wblob + s.off_lm_scale);
  p.attn_norm = h->norms; p.final_norm = h->norms + (size_t)L * s.d;
  p.rope_turns = h->rope_turns;
  p.embed = reinterpret_cast<const uint16_t*>(h->wblob + s.off_embed);
  p.page_table = page_table_dev;
  const size_t maxa = (size_t)P.maxa;
#define AL(ptr, n) do { int _r = alloc(h, &(ptr), (n)); if (_r) { free_plan(h); return _r; } } while (0)
  AL(p.seq_lens, B);
  AL(p.X, (size_t)(L + 1) * B * s.d);
  AL(p.SS, (size_t)(L + 1) * s.nrb_d * kSsStride);
  AL(p.XG, (size_t)(L + 1) * B * s.d);
  AL(p.XGL, (size_t)(L + 1) * B * s.d);
  AL(p.Q, (size_t)L * B * s.Hq * s.hd);
  AL(p.attp, (size_t)L * s.Hkv * B * h->max_items_bg * s.gs * (s.hd + 2));
  AL(p.atto, (size_t)L * B * s.Hq * s.hd);
  AL(p.rlog, (size_t)L * B * s.E);
  p.rw_stride = (int)(1 + 2 * maxa + 2 * maxa * B);
  AL(p.rword, (size_t)L * p.rw_stride);
  AL(p.epoch, 1);
  AL(p.ridx, (size_t)L * B * s.topk);
  AL(p.rw, (size_t)L * B * s.topk);
  AL(p.active, (size_t)L * maxa);
  AL(p.nact, (size_t)L);
  AL(p.act_cnt, (size_t)L * maxa);
  AL(p.act_tok, (size_t)L * maxa * B);
  p.det = h->det;
  AL(p.moe, (size_t)L * B * s.d * (h->det ? 2 : 1));  // 64-bit fixed point when deterministic
  AL(p.ctr, (size_t)P.n_ctr * kCtrStride);
  AL(p.qhead, (size_t)3 * L);
  AL(p.qcount, (size_t)3 * L);
  AL(p.err, 16);
  AL(p.amax, (size_t)kAmaxReplicas * B);
  AL(p.gen, 2);
  AL(h->d_tasks, P.tasks.size());
  AL(h->d_sm_off, P.sm_off.size());
  AL(h->d_sm_list, P.sm_list.size());
  AL(h->d_tokens, B);
  AL(h->d_logits, (size_t)B * s.V);
  AL(h->d_trace_n, 1);
  AL(h->d_snap, (size_t)P.n_ctr + 6 * L);
#undef AL
  p.c_lr = P.c_lr; p.c_qkvg = P.c_qkvg; p.c_rt = P.c_rt; p.c_rr = P.c_rr; p.c_att = P.c_att; p.c_og = P.c_og;
  p.c_md = P.c_md; p.c_od = P.c_od; p.c_oa = P.c_oa; p.c_done = P.c_done; p.n_ctr = P.n_ctr;
  p.n_queues = 3 * L;
  p.od_target = P.od_target;
  p.tasks = h->d_tasks; p.sm_off = h->d_sm_off; p.sm_list = h->d_sm_list;
  p.trace = nullptr; p.trace_n = h->d_trace_n; p.trace_cap = 0;
  p.snap = h->inspect ? h->d_snap : nullptr;
  CK(h, cudaMemcpy(h->d_tasks, P.tasks.data(), P.tasks.size() * 4, cudaMemcpyHostToDevice));
  CK(h, cudaMemcpy(h->d_sm_off, P.sm_off.data(), P.sm_off.size() * 4, cudaMemcpyHostToDevice));
  CK(h, cudaMemcpy(h->d_sm_list, P.sm_list.data(), P.sm_list.size() * 4, cudaMemcpyHostToDevice));
  CK(h, cudaMemcpy(p.seq_lens, seq_lens_host, (size_t)B * 4, cudaMemcpyHostToDevice));
  const unsigned first_epoch = 1;  // the cleared tagged words carry epoch 0
  CK(h, cudaMemcpy(p.epoch, &first_epoch, 4, cudaMemcpyHostToDevice));
  h->last_noalloc = false;
  h->planned = true;
  return MK_OK;
}

int mk_decode_step(mk_handle* h, const int32_t* tokens_dev, void* k_cache, void* v_cache, float* logits_dev,
                   void* stream) {
  int r = prepare_step(h, tokens_dev, k_cache, v_cache, logits_dev);
  if (r) return r;
  h->last_noalloc = false;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  return launch_segment(h, 0, true, true, st);
}

int mk_decode_steps(mk_handle* h, const int32_t* tokens_dev, int n_steps, void* k_cache, void* v_cache,
                    float* logits_dev, int32_t* tokens_out_dev, void* stream) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  if (n_steps < 1 || n_steps > 4096) return fail(&h->err, MK_ERR_INVALID, "n_steps %d not in [1, 4096]", n_steps);
  if (!tokens_out_dev) return fail(&h->err, MK_ERR_INVALID, "tokens_out is NULL");
  int r = prepare_step(h, tokens_dev, k_cache, v_cache, logits_dev);
  if (r) return r;
  h->last_noalloc = false;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  Params p = h->prm;
  p.sm_off = h->d_sm_off;  // the megakernel segment
  p.do_reset = 1;
  p.n_steps = n_steps;
  p.tok_out = tokens_out_dev;
  cudaError_t e = launch_variant(p, h->tmK, h->tmV, h->n_sm, true, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "megakernel launch (multi-step)");
  return MK_OK;
}

// The step's scratch buffers (everything mk_plan allocates per step except the plan
// state: seq_lens, error word, task lists, trace count, host-step staging) laid out in
// one byte range, 256-byte aligned pieces.  Returns the bytes needed; with `base`
// non-null also points the Params fields at it and reports the counter/queue span.
static size_t step_scratch_layout(const mk_handle* h, uint8_t* base, Params* p, size_t* zero_off,
                                  size_t* zero_bytes) {
  const Shape& s = h->s;
  const size_t L = s.L, B = h->B, maxa = h->P.maxa;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += (bytes + 255) / 256 * 256; return base ? base + r : nullptr; };
  uint8_t* q;
  q = take((L + 1) * B * s.d * 4);                              if (p) p->X = (float*)q;
  q = take((L + 1) * s.nrb_d * kSsStride * 4);                  if (p) p->SS = (float*)q;
  q = take((L + 1) * B * s.d * 2);                              if (p) p->XG = (uint16_t*)q;
  q = take((L + 1) * B * s.d * 2);                              if (p) p->XGL = (uint16_t*)q;
  q = take(L * B * s.Hq * s.hd * 2);                            if (p) p->Q = (uint16_t*)q;
  q = take(L * s.Hkv * B * (size_t)h->max_items_bg * s.gs * (s.hd + 2) * 4); if (p) p->attp = (float*)q;
  q = take(L * B * s.Hq * s.hd * 2);                            if (p) p->atto = (uint16_t*)q;
  // cleared each call: the routing arrays read back by mk_read (a dense layer of a
  // mixed stack never writes its own: they must read as "no experts"), the layer
  // accumulators, the counters and queues, and the epoch-tagged words (other handles'
  // calls share this array and may have used the same epochs)
  const size_t z0 = o;
  q = take(L * B * s.topk * 4);                                 if (p) p->ridx = (int*)q;
  q = take(L * B * s.topk * 4);                                 if (p) p->rw = (float*)q;
  q = take(L * maxa * 4);                                       if (p) p->active = (int*)q;
  q = take(L * 4);                                              if (p) p->nact = (int*)q;
  q = take(L * maxa * 4);                                       if (p) p->act_cnt = (int*)q;
  q = take(L * maxa * B * 4);                                   if (p) p->act_tok = (int*)q;
  q = take(L * B * s.d * 4 * (h->prm.det ? 2 : 1));             if (p) p->moe = (float*)q;
  q = take(L * B * s.E * 8);                                    if (p) p->rlog = (uint64_t*)q;
  q = take(L * (1 + 2 * maxa + 2 * maxa * B) * 8);              if (p) { p->rword = (uint64_t*)q; p->rw_stride = (int)(1 + 2 * maxa + 2 * maxa * B); }
  q = take((size_t)h->P.n_ctr * kCtrStride * 4);                if (p) p->ctr = (unsigned*)q;
  q = take(3 * L * 4);                                          if (p) p->qhead = (int*)q;
  q = take(3 * L * 4);                                          if (p) p->qcount = (int*)q;
  if (zero_off) *zero_off = z0;
  if (zero_bytes) *zero_bytes = o - z0;
  return o;
}

int mk_decode_step_noalloc(mk_handle* h, const int32_t* tokens_dev, void* k_cache, void* v_cache,
                           float* logits_dev, void* stream) {
  int r = prepare_step(h, tokens_dev, k_cache, v_cache, logits_dev);
  if (r) return r;
  const size_t need = step_scratch_layout(h, nullptr, nullptr, nullptr, nullptr);
  if (need > kStaticScratchBytes)
    return fail(&h->err, MK_ERR_UNSUPPORTED,
                "mk_decode_step_noalloc: this plan needs %zu bytes of step scratch, the static buffer holds %zu "
                "(reduce batch or context, or use mk_decode_step)", need, kStaticScratchBytes);
  void* base = nullptr;
  CK(h, static_scratch_address(&base));
  Params p = h->prm;
  p.snap = nullptr;  // the inspection reads describe the handle's own step buffers
  size_t z_off = 0, z_bytes = 0;
  step_scratch_layout(h, static_cast<uint8_t*>(base), &p, &z_off, &z_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // counters, queues and tagged words must start at zero; the rest is written before it is read
  CK(h, cudaMemsetAsync(static_cast<uint8_t*>(base) + z_off, 0, z_bytes, st));
  h->last_noalloc = true;
  h->last_stream = st;
  p.sm_off = h->d_sm_off;
  p.do_reset = 1;
  cudaError_t e = launch_variant(p, h->tmK, h->tmV, h->n_sm, true, st);
  if (e != cudaSuccess) return cuda_fail(h, e, "megakernel launch (static scratch)");
  return MK_OK;
}

int mk_decode_step_host(mk_handle* h, const int32_t* tokens_host, void* k_cache, void* v_cache,
                        float* logits_host, void* stream) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  if (!h->planned) return fail(&h->err, MK_ERR_STATE, "mk_plan has not been called");
  if (!tokens_host || !logits_host) return fail(&h->err, MK_ERR_INVALID, "NULL host buffer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(h, cudaMemcpyAsync(h->d_tokens, tokens_host, (size_t)h->B * 4, cudaMemcpyHostToDevice, st));
  int r = mk_decode_step(h, h->d_tokens, k_cache, v_cache, h->d_logits, stream);
  if (r) return r;
  CK(h, cudaMemcpyAsync(logits_host, h->d_logits, (size_t)h->B * h->s.V * 4, cudaMemcpyDeviceToHost, st));
  CK(h, cudaStreamSynchronize(st));
  return MK_OK;
}

int mk_decode_step_perop(mk_handle* h, const int32_t* tokens_dev, void* k_cache, void* v_cache,
                         float* logits_dev, void* stream, int use_graph) {
  int r = prepare_step(h, tokens_dev, k_cache, v_cache, logits_dev);
  if (r) return r;
  h->last_noalloc = false;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  const int first = 1, last = h->P.n_segs - 1;
  if (!use_graph) {
    for (int seg = first; seg <= last; ++seg) {
      r = launch_segment(h, seg, false, seg == last, st);
      if (r) return r;
    }
    return MK_OK;
  }
  const void* key[5] = {tokens_dev, k_cache, v_cache, logits_dev, stream};
  if (!h->graph || std::memcmp(key, h->g_key, sizeof key) != 0 || h->g_fixed != h->fixed) {
    if (h->graph) { cudaGraphExecDestroy(h->graph); h->graph = nullptr; }
    cudaStream_t cap = nullptr;
    CK(h, cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking));
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) { cudaStreamDestroy(cap); return cuda_fail(h, e, "begin capture"); }
    for (int seg = first; seg <= last && r == MK_OK; ++seg) r = launch_segment(h, seg, false, seg == last, cap);
    e = cudaStreamEndCapture(cap, &g);
    cudaStreamDestroy(cap);
    if (r) { if (g) cudaGraphDestroy(g); return r; }
    if (e != cudaSuccess) return cuda_fail(h, e, "end capture");
    e = cudaGraphInstantiate(&h->graph, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) { h->graph = nullptr; return cuda_fail(h, e, "graph instantiate"); }
    std::memcpy(h->g_key, key, sizeof key);
    h->g_fixed = h->fixed;
  }
  CK(h, cudaGraphLaunch(h->graph, st));
  return MK_OK;
}

int mk_get_status(mk_handle* h, mk_error_info* info) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  mk_error_info tmp;
  mk_error_info* o = info ? info : &tmp;
  std::memset(o, 0, sizeof *o);
  if (!h->planned) return MK_OK;
  CK(h, cudaSetDevice(h->dev));
  CK(h, cudaStreamSynchronize(h->last_stream));
  int32_t e[16];
  CK(h, cudaMemcpy(e, h->prm.err, sizeof e, cudaMemcpyDeviceToHost));
  o->code = e[E_CODE]; o->task = e[E_TASK]; o->counter = e[E_CTR]; o->observed = e[E_OBS];
  o->target = e[E_TARGET]; o->sm = e[E_SM];
  if (o->code) {
    CK(h, cudaMemset(h->prm.err, 0, sizeof e));
    fail(&h->err, o->code, "device error %d (task %d, counter %d, observed %d, target %d, sm %d)", o->code,
         o->task, o->counter, o->observed, o->target, o->sm);
  }
  return o->code;
}

int mk_set_trace(mk_handle* h, void* records_dev, int capacity) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  if (!h->planned) return fail(&h->err, MK_ERR_STATE, "mk_plan has not been called");
  if (capacity < 0 || (capacity > 0 && !records_dev)) return fail(&h->err, MK_ERR_INVALID, "bad trace buffer");
  CK(h, cudaSetDevice(h->dev));
  CK(h, cudaDeviceSynchronize());
  CK(h, cudaMemset(h->d_trace_n, 0, sizeof(unsigned)));
  h->prm.trace = capacity > 0 ? static_cast<unsigned long long*>(records_dev) : nullptr;
  h->prm.trace_cap = capacity;
  if (h->graph) { cudaGraphExecDestroy(h->graph); h->graph = nullptr; }
  return MK_OK;
}

int mk_plan_drop_signal(mk_handle* h, int task) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  if (!h->planned) return fail(&h->err, MK_ERR_STATE, "mk_plan has not been called");
  if (task < 0 || task >= h->P.n_tasks()) return fail(&h->err, MK_ERR_INVALID, "task %d out of range", task);
  int32_t* T = &h->P.tasks[(size_t)task * kDescInts];
  if (T[D_SIG_CTR] < 0) return fail(&h->err, MK_ERR_INVALID, "task %d signals no counter", task);
  T[D_SIG_CTR] = h->P.c_done;  // the launch-completion counter: never waited on by a task
  CK(h, cudaSetDevice(h->dev));
  CK(h, cudaDeviceSynchronize());
  CK(h, cudaMemcpy(h->d_tasks + (size_t)task * kDescInts, T, kDescInts * 4, cudaMemcpyHostToDevice));
  if (h->graph) { cudaGraphExecDestroy(h->graph); h->graph = nullptr; }
  return MK_OK;
}

int mk_set_inspect(mk_handle* h, int on) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  h->inspect = on ? 1 : 0;
  if (h->planned) {
    CK(h, cudaSetDevice(h->dev));
    CK(h, cudaDeviceSynchronize());
    h->prm.snap = h->inspect ? h->d_snap : nullptr;
    if (h->graph) { cudaGraphExecDestroy(h->graph); h->graph = nullptr; }
  }
  return MK_OK;
}

int mk_set_fixed(mk_handle* h, int fixed) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  h->fixed = fixed ? 1 : 0;
  return MK_OK;
}

int mk_set_deterministic(mk_handle* h, int on) {
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  if (on && h->s.lm_umma)
    return fail(&h->err, MK_ERR_UNSUPPORTED, "deterministic steps with the tensor-core LM head (MK_LM_UMMA)");
  h->det = on ? 1 : 0;
  return MK_OK;
}

int mk_read(mk_handle* h, int what, void* host_out, size_t bytes) {
  if (!h || !host_out) return fail(h ? &h->err : nullptr, MK_ERR_INVALID, "NULL argument");
  if (!h->planned) return fail(&h->err, MK_ERR_STATE, "mk_plan has not been called");
  const Shape& s = h->s;
  Params p = h->prm;
  const size_t L = s.L, B = h->B;
  CK(h, cudaSetDevice(h->dev));
  CK(h, cudaDeviceSynchronize());
  if (h->last_noalloc) {  // the step buffers of the last step are in the static scratch
    void* base = nullptr;
    CK(h, static_scratch_address(&base));
    step_scratch_layout(h, static_cast<uint8_t*>(base), &p, nullptr, nullptr);
  }
  auto copy = [&](const void* src, size_t n) -> int {
    if (n != bytes) return fail(&h->err, MK_ERR_INVALID, "mk_read(%d): need %zu bytes, got %zu", what, n, bytes);
    CK(h, cudaMemcpy(host_out, src, n, cudaMemcpyDeviceToHost));
    return MK_OK;
  };
  switch (what) {
    case MK_READ_HIDDEN: return copy(p.X, (L + 1) * B * s.d * 4);
    case MK_READ_ROUTES: return copy(p.ridx, L * B * s.topk * 4);
    case MK_READ_ROUTE_W: return copy(p.rw, L * B * s.topk * 4);
    case MK_READ_SEQ_LENS: return copy(p.seq_lens, B * 4);
    case MK_READ_COUNTERS: {
      if (bytes != (size_t)p.n_ctr * 4) return fail(&h->err, MK_ERR_INVALID, "mk_read(COUNTERS): need %zu bytes", (size_t)p.n_ctr * 4);
      std::vector<unsigned> raw((size_t)p.n_ctr * kCtrStride);
      CK(h, cudaMemcpy(raw.data(), p.ctr, raw.size() * 4, cudaMemcpyDeviceToHost));
      unsigned* o = static_cast<unsigned*>(host_out);
      for (int i = 0; i < p.n_ctr; ++i) o[i] = raw[(size_t)i * kCtrStride];
      return MK_OK;
    }
    case MK_READ_ROUTER_LOGITS: {  // stored tagged with the step epoch: return the values
      if (bytes != L * B * s.E * 4) return fail(&h->err, MK_ERR_INVALID, "mk_read(ROUTER_LOGITS): need %zu bytes", L * B * s.E * 4);
      std::vector<uint64_t> raw(L * B * s.E);
      CK(h, cudaMemcpy(raw.data(), p.rlog, raw.size() * 8, cudaMemcpyDeviceToHost));
      uint32_t* o = static_cast<uint32_t*>(host_out);
      for (size_t i = 0; i < raw.size(); ++i) o[i] = (uint32_t)raw[i];
      return MK_OK;
    }
    case MK_READ_TRACE_COUNT: return copy(h->d_trace_n, 4);
    case MK_READ_FINAL_COUNTERS:
      if (!h->inspect) return fail(&h->err, MK_ERR_STATE, "mk_read(FINAL_COUNTERS): inspection is off");
      return copy(h->d_snap, (size_t)p.n_ctr * 4);
    case MK_READ_FINAL_QUEUES:
      if (!h->inspect) return fail(&h->err, MK_ERR_STATE, "mk_read(FINAL_QUEUES): inspection is off");
      return copy(h->d_snap + p.n_ctr, (size_t)2 * p.n_queues * 4);
    case MK_READ_TASKS: {
      const size_t n = h->P.tasks.size() * 4;
      if (bytes != n) return fail(&h->err, MK_ERR_INVALID, "mk_read(TASKS): need %zu bytes, got %zu", n, bytes);
      std::memcpy(host_out, h->P.tasks.data(), n);
      return MK_OK;
    }
    case MK_READ_ACTIVE: {
      const size_t maxa = p.maxa, per = 1 + maxa * (2 + B);
      if (bytes != L * per * 4) return fail(&h->err, MK_ERR_INVALID, "mk_read(ACTIVE): need %zu bytes", L * per * 4);
      std::vector<int32_t> nact(L), act(L * maxa), cnt(L * maxa), tok(L * maxa * B);
      CK(h, cudaMemcpy(nact.data(), p.nact, L * 4, cudaMemcpyDeviceToHost));
      CK(h, cudaMemcpy(act.data(), p.active, L * maxa * 4, cudaMemcpyDeviceToHost));
      CK(h, cudaMemcpy(cnt.data(), p.act_cnt, L * maxa * 4, cudaMemcpyDeviceToHost));
      CK(h, cudaMemcpy(tok.data(), p.act_tok, L * maxa * B * 4, cudaMemcpyDeviceToHost));
      int32_t* o = static_cast<int32_t*>(host_out);
      for (size_t l = 0; l < L; ++l) {
        int32_t* r = o + l * per;
        r[0] = nact[l];
        for (size_t a = 0; a < maxa; ++a) {
          int32_t* q = r + 1 + a * (2 + B);
          q[0] = act[l * maxa + a];
          q[1] = cnt[l * maxa + a];
          for (size_t b = 0; b < B; ++b) q[2 + b] = tok[(l * maxa + a) * B + b];
        }
      }
      return MK_OK;
    }
    default:
      return fail(&h->err, MK_ERR_INVALID, "mk_read: unknown item %d", what);
  }
}

int mk_read_expert_fp8(mk_handle* h, int layer, int expert, void* host_out, size_t bytes) {
  if (!h || !host_out) return fail(h ? &h->err : nullptr, MK_ERR_INVALID, "NULL argument");
  const Shape& s = h->s;
  if (!s.fp8) return fail(&h->err, MK_ERR_STATE, "experts are stored in bf16");
  if (layer < 0 || layer >= s.L || expert < 0 || expert >= s.E)
    return fail(&h->err, MK_ERR_INVALID, "layer %d / expert %d out of range", layer, expert);
  if (s.dense(layer)) return fail(&h->err, MK_ERR_INVALID, "layer %d is dense (no routed experts)", layer);
  const int d = s.d, f = s.f, fs = s.moe_fs, nrb1 = fs / 8, k2 = fs / 16;
  const size_t need = (size_t)3 * f * d + 4 * ((size_t)2 * f + (size_t)d);
  if (bytes != need) return fail(&h->err, MK_ERR_INVALID, "mk_read_expert_fp8: need %zu bytes, got %zu", need, bytes);
  std::vector<uint8_t> raw(s.moe_bytes_e);
  CK(h, cudaSetDevice(h->dev));
  CK(h, cudaDeviceSynchronize());
  CK(h, cudaMemcpy(raw.data(), h->wblob + s.off_moe + ((size_t)layer * s.E + expert) * s.moe_bytes_e, raw.size(),
                   cudaMemcpyDeviceToHost));
  uint8_t* gc = static_cast<uint8_t*>(host_out);
  uint8_t* uc = gc + (size_t)f * d;
  uint8_t* dc = uc + (size_t)f * d;
  float* gsc = reinterpret_cast<float*>(dc + (size_t)d * f);
  float* usc = gsc + f;
  float* dsc = usc + f;
  const int sb = fp8_scale_bytes(fs, d);
  // the inverse of the item packing: scales, then gate/up and down fragments whose
  // lane holds rows g and g + 8, columns 2c, 2c + 1, 2c + 8, 2c + 9 of a 16x16 block
  for (int t = 0; t < s.t_moe; ++t) {
    const uint8_t* item = raw.data() + (size_t)t * s.moe_item_bytes;
    float scl[2 * 64 + 2048];
    memcpy(scl, item, (size_t)sb);
    for (int rb = 0; rb < nrb1; ++rb)
      for (int i = 0; i < 16; ++i) (i < 8 ? gsc : usc)[t * fs + 8 * rb + (i & 7)] = scl[rb * 16 + i];
    if (t == 0)  // (every item holds the expert's down-row scales)
      for (int r = 0; r < d; ++r) dsc[r] = scl[2 * fs + r];
    const uint8_t* gu = item + sb;
    for (int fi = 0; fi < nrb1 * (d / 16); ++fi) {
      const int j = fi / (nrb1 * 8), rem = fi % (nrb1 * 8), rb = rem / 8, ks = rem % 8 + 8 * j;
      for (int lane = 0; lane < 32; ++lane)
        for (int q = 0; q < 4; ++q)
          for (int e = 0; e < 2; ++e) {
            const int i = (lane >> 2) + ((q & 1) ? 8 : 0);
            const int k = 16 * ks + 2 * (lane & 3) + ((q & 2) ? 8 : 0) + e;
            (i < 8 ? gc : uc)[(size_t)(t * fs + 8 * rb + (i & 7)) * d + k] = gu[((size_t)fi * 32 + lane) * 8 + 2 * q + e];
          }
    }
    const uint8_t* dn = gu + (size_t)2 * fs * d;
    for (int fi = 0; fi < (d / 16) * k2; ++fi) {
      const int rb = fi / k2, ks = fi % k2;
      for (int lane = 0; lane < 32; ++lane)
        for (int q = 0; q < 4; ++q)
          for (int e = 0; e < 2; ++e) {
            const int row = rb * 16 + (lane >> 2) + ((q & 1) ? 8 : 0);
            const int col = t * fs + 16 * ks + 2 * (lane & 3) + ((q & 2) ? 8 : 0) + e;
            dc[(size_t)row * f + col] = dn[((size_t)fi * 32 + lane) * 8 + 2 * q + e];
          }
    }
  }
  return MK_OK;
}

// Source row of packed row r (host twin of the packer's mapping): matrix 0/1/2 and row.
static void host_pack_source_row(int mode, int r, int n_src_rows, int hd, int gs, int grp, int& which,
                                 long long& srow) {
  which = 0;
  srow = r;
  if (mode == PACK_QKV) {
    const int head = r / hd, jj = r % hd, m = jj / 16, i = jj % 16;
    const int dim = (i < 8) ? 8 * m + i : hd / 2 + 8 * m + (i - 8);
    if (head < gs) { which = 0; srow = (long long)(grp * gs + head) * hd + dim; }
    else { which = head == gs ? 1 : 2; srow = (long long)grp * hd + dim; }
  } else if (srow >= n_src_rows) {
    srow = -1;
  }
}

// The E4M3 codes of packed row r of a region of FP8 GEMV tiles (tile_rows rows each, K
// columns, fragment order of the packer, 8 bytes a lane).
static void unpack_fp8_row(const uint8_t* region, int r, int K, int tile_rows, uint8_t* out) {
  const int nrb_t = tile_rows / 16, t = r / tile_rows, rb = (r % tile_rows) / 16, i = r % 16;
  const size_t per_tile = (size_t)nrb_t * (K / 16);
  for (int ks = 0; ks < K / 16; ++ks) {
    const int j = ks / 8, w = ks % 8;
    const uint8_t* frag = region + (t * per_tile + (size_t)(j * nrb_t + rb) * 8 + w) * kFragBytes8;
    for (int c = 0; c < 4; ++c)
      for (int half = 0; half < 2; ++half)
        for (int e = 0; e < 2; ++e) {
          const int q = (i >= 8 ? 1 : 0) + 2 * half;
          out[16 * ks + 2 * c + 8 * half + e] = frag[((i & 7) * 4 + c) * 8 + 2 * q + e];
        }
  }
}

int mk_read_weight_fp8(mk_handle* h, int matrix, int layer, void* host_out, size_t bytes) {
  if (!h || !host_out) return fail(h ? &h->err : nullptr, MK_ERR_INVALID, "NULL argument");
  const Shape& s = h->s;
  if (!s.fp8d) return fail(&h->err, MK_ERR_STATE, "the projections are stored in bf16");
  if (matrix < MK_W_Q || matrix > MK_W_LM) return fail(&h->err, MK_ERR_INVALID, "matrix %d unknown", matrix);
  if (matrix != MK_W_LM && (layer < 0 || layer >= s.L))
    return fail(&h->err, MK_ERR_INVALID, "layer %d out of range", layer);
  const int d = s.d, hd = s.hd, gs = s.gs;
  const int rows = matrix == MK_W_Q ? s.Hq * hd : matrix == MK_W_K || matrix == MK_W_V ? s.Hkv * hd
                 : matrix == MK_W_O ? d : s.V;
  const int cols = matrix == MK_W_O ? s.Hq * hd : d;
  const size_t need = (size_t)rows * cols + 4 * (size_t)rows;
  if (bytes != need) return fail(&h->err, MK_ERR_INVALID, "mk_read_weight_fp8: need %zu bytes, got %zu", need, bytes);
  uint8_t* codes = static_cast<uint8_t*>(host_out);
  float* scales = reinterpret_cast<float*>(codes + (size_t)rows * cols);
  CK(h, cudaSetDevice(h->dev));
  CK(h, cudaDeviceSynchronize());
  std::vector<uint8_t> row((size_t)std::max(d, s.Hq * hd));
  if (matrix <= MK_W_V) {  // QKV: per KV group, packed rows [q heads | k | v], RoPE-paired
    std::vector<uint8_t> reg((size_t)s.qkv_rows_group * d);
    std::vector<float> sc(s.qkv_rows_group);
    for (int g = 0; g < s.Hkv; ++g) {
      CK(h, cudaMemcpy(reg.data(), h->wblob + s.off_qkv + layer * s.qkv_layer_bytes + (size_t)g * reg.size(),
                       reg.size(), cudaMemcpyDeviceToHost));
      CK(h, cudaMemcpy(sc.data(), h->wblob + s.off_qkv_scale + (((size_t)layer * s.Hkv + g) * s.qkv_rows_group) * 4,
                       sc.size() * 4, cudaMemcpyDeviceToHost));
      for (int r = 0; r < s.qkv_rows_group; ++r) {
        int which;
        long long srow;
        host_pack_source_row(PACK_QKV, r, 0, hd, gs, g, which, srow);
        if (which != matrix) continue;
        unpack_fp8_row(reg.data(), r, d, s.r_qkv, codes + (size_t)srow * cols);
        scales[srow] = sc[r];
      }
    }
  } else if (matrix == MK_W_O) {  // per KV group: the group's k_o columns of every row
    std::vector<uint8_t> reg((size_t)d * s.k_o);
    for (int g = 0; g < s.Hkv; ++g) {
      CK(h, cudaMemcpy(reg.data(), h->wblob + s.off_o + layer * s.o_layer_bytes + (size_t)g * reg.size(),
                       reg.size(), cudaMemcpyDeviceToHost));
      for (int r = 0; r < d; ++r) {
        unpack_fp8_row(reg.data(), r, s.k_o, s.r_o, row.data());
        std::memcpy(codes + (size_t)r * cols + (size_t)g * s.k_o, row.data(), s.k_o);
      }
    }
    CK(h, cudaMemcpy(scales, h->wblob + s.off_o_scale + (size_t)layer * d * 4, (size_t)d * 4, cudaMemcpyDeviceToHost));
  } else {
    std::vector<uint8_t> reg((size_t)s.v_pad * d);
    CK(h, cudaMemcpy(reg.data(), h->wblob + s.off_lm, reg.size(), cudaMemcpyDeviceToHost));
    for (int r = 0; r < s.V; ++r) unpack_fp8_row(reg.data(), r, d, s.r_lm, codes + (size_t)r * cols);
    CK(h, cudaMemcpy(scales, h->wblob + s.off_lm_scale, (size_t)s.V * 4, cudaMemcpyDeviceToHost));
  }
  return MK_OK;
}

int mk_query(mk_handle* h, int what, int64_t* out) {
  if (!out) return fail(h ? &h->err : nullptr, MK_ERR_INVALID, "out is NULL");
  switch (what) {
    case MK_Q_SMEM_BYTES: *out = kSmemBytes; return MK_OK;
    case MK_Q_THREADS: *out = kThreads; return MK_OK;
    case MK_Q_STAGE_BYTES: *out = kStageBytes; return MK_OK;
    case MK_Q_NUM_STAGES: *out = kStages; return MK_OK;
    default: break;
  }
  if (!h) return fail(nullptr, MK_ERR_INVALID, "handle is NULL");
  switch (what) {
    case MK_Q_NUM_SMS: *out = h->n_sm; return MK_OK;
    case MK_Q_PACKED_BYTES: *out = (int64_t)h->s.total; return MK_OK;
    case MK_Q_TENSOR_CORES: *out = (h->s.lm_umma ? 1 : 0) | (h->s.moe_umma ? 2 : 0); return MK_OK;
    default: break;
  }
  if (!h->planned) return fail(&h->err, MK_ERR_STATE, "mk_plan has not been called");
  switch (what) {
    case MK_Q_NUM_TASKS: *out = h->P.n_tasks(); return MK_OK;
    case MK_Q_NUM_COUNTERS: *out = h->P.n_ctr; return MK_OK;
    case MK_Q_MAX_ACTIVE: *out = h->P.maxa; return MK_OK;
    case MK_Q_SPLIT_PAGES: *out = h->split_pages; return MK_OK;
    case MK_Q_PEROP_LAUNCHES: *out = h->P.n_segs - 1; return MK_OK;
    default: return fail(&h->err, MK_ERR_INVALID, "mk_query: unknown item %d", what);
  }
}

void mk_destroy(mk_handle* h) {
  if (!h) return;
  cudaSetDevice(h->dev);
  cudaDeviceSynchronize();
  free_plan(h);
  if (h->wblob) cudaFree(h->wblob);
  if (h->norms) cudaFree(h->norms);
  if (h->rope_turns) cudaFree(h->rope_turns);
  delete h;
}

}  // extern "C"
