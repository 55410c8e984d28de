// The persistent decode megakernel and the weight packer.
//
// One CTA per SM.  Warp 8 is the producer: it walks this CTA's host-built list of
// task descriptors, claims attention / expert items from per-layer atomic queues,
// and streams each task's immutable weight tiles (1-D bulk copies of pre-packed
// tiles) or KV pages (2-D tensor-map copies) into a 6-stage shared-memory ring
// ahead of the consumers -- before the task's activation dependency resolves.
// Warps 0-7 are consumers: per task they wait on one counter, build their MMA
// operands from the activations, run mma.sync over the ring stages, reduce across
// warps and write the task's output, then signal one counter.  Where a counter
// completes a fan-in (router tiles, attention splits, residual row blocks), the
// last arriving CTA runs the follow-up step itself (top-k/route, LSE combine,
// residual add + sums of squares).
//   [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "One kernel for
//    the full decode step", "The calling convention that makes it hand-writable",
//    "Scheduling: mostly static, selectively dynamic"; Fuse decode into one
//    megakernel for 1.58x higher H100 throughput (the kitchen ticket rail, the
//    three stalls); Cohere open-sources fused LLM decode kernel with 1.58x vLLM
//    claim (16 task types, 32-int32 descriptor, warp roles).]
#include <atomic>

#include "mk_device.cuh"

// This file is compiled four times: as is (float32 layer accumulators, every GEMV on
// mma.sync), by mk_kernel_det.cu with MK_DET = 1 (deterministic steps: 64-bit
// fixed-point accumulators; namespace mk_det), by mk_kernel_umma.cu with MK_UMMA = 1
// (the LM head on tcgen05 tensor cores with a tensor-memory accumulator; namespace
// mk_umma) and by mk_kernel_umma_ffn.cu with MK_UMMA = 2 (the bf16 expert and dense-FFN
// items on them too; namespace mk_umma_ffn).  The weight packers and the static step
// scratch exist in the first build only.
#ifndef MK_DET
#define MK_DET 0
#endif
#ifndef MK_UMMA
#define MK_UMMA 0
#endif
#if MK_DET && MK_UMMA
#error "one kernel variant per build"
#endif
#if MK_DET
#define MK_KNS mk_det
#elif MK_UMMA == 2
#define MK_KNS mk_umma_ffn
#elif MK_UMMA
#define MK_KNS mk_umma
#else
#define MK_KNS mk
#endif

namespace MK_KNS {
using namespace ::mk;

// ============================================================== errors / waits
__device__ void raise_err(const Params& p, int code, int task, int ctr, int obs, int target) {
  if (atomicCAS(&p.err[E_CODE], 0, code) == 0) {
    p.err[E_TASK] = task;
    p.err[E_CTR] = ctr;
    p.err[E_OBS] = obs;
    p.err[E_TARGET] = target;
    p.err[E_SM] = blockIdx.x;
  }
  if (code == MK_ERR_TIMEOUT) atomicExch(&p.err[E_ABORT], 1);
}

__device__ __forceinline__ bool aborted(const Params& p) { return ld_volatile(&p.err[E_ABORT]) != 0; }

// Optional per-task timeline (Params::trace != nullptr): thread 0 stamps the
// moments of a task into shared memory and appends one record when it ends.
//   record (16 x u64): [0] sm | op << 8 | layer << 16 | fan-in << 24, [1] item,
//   [2] received, [3] dependency met (activation loads start), [4] first weight/KV
//   chunk landed (activations built), [5] MMA loop done, [6] fan-in follow-up
//   started (0 if none), [7] task done, [8..11] sub-steps of a fan-in follow-up,
//   [12..15] sub-steps of the task's own epilogue (per opcode, see the marks).
__device__ __forceinline__ unsigned long long* trace_slots(const Smem& S) {
  return reinterpret_cast<unsigned long long*>(S.small + 192);
}
__device__ __forceinline__ void trace_mark(const Params& p, const Smem& S, int slot) {
  if (p.trace && threadIdx.x == 0) trace_slots(S)[slot] = gtime();
}
__device__ void trace_emit(const Params& p, const Smem& S, int op, int layer, int item) {
  if (!p.trace || threadIdx.x != 0) return;
  const unsigned idx = atomicAdd(p.trace_n, 1u);
  if (idx >= (unsigned)p.trace_cap) return;
  unsigned long long* r = p.trace + (size_t)idx * 16;
  unsigned long long* t = trace_slots(S);
  r[0] = (unsigned long long)blockIdx.x | ((unsigned long long)op << 8) |
         ((unsigned long long)(layer & 0xff) << 16) | ((unsigned long long)(t[6] != 0) << 24);
  r[1] = (unsigned long long)(unsigned)item;
  r[2] = t[0]; r[3] = t[1]; r[4] = t[2]; r[5] = t[3]; r[6] = t[6]; r[7] = gtime();
  r[8] = t[8]; r[9] = t[9]; r[10] = t[10]; r[11] = t[11];
  r[12] = t[12]; r[13] = t[13]; r[14] = t[14]; r[15] = t[15];
}

// Spin until ctr >= target, bounded by the timeout and the abort flag.  Polls are
// acquire loads with a growing back-off (32 ns .. 256 ns) so that the many waiters
// of a layer boundary do not saturate the counter's L2 line.  The load that sees the
// target is itself the acquire: no trailing fence, which would also wait for this
// thread's unrelated earlier stores (the previous task's outputs) to drain.
__device__ bool wait_ge(const Params& p, int ci, unsigned target, int task) {
  const unsigned* c = p.ctr + (size_t)ci * kCtrStride;
  if (ld_acquire(c) >= target) return true;
  const uint64_t t0 = gtime();
  unsigned ns = 32;
  for (int it = 0;; ++it) {
    __nanosleep(ns);
    ns = ns < 256 ? ns * 2 : 256;
    const unsigned v = ld_acquire(c);
    if (v >= target) return true;
    if ((it & 7) == 7) {
      if (aborted(p)) return false;
      if ((long long)(gtime() - t0) > p.timeout_ns) {
        raise_err(p, MK_ERR_TIMEOUT, task, ci, (int)v, (int)target);
        return false;
      }
    }
  }
}

__device__ __forceinline__ unsigned* ctr_ptr(const Params& p, int ci) { return p.ctr + (size_t)ci * kCtrStride; }

// The layer accumulators [L][B][d] (expert and O-proj outputs), float or, in the
// deterministic build, 64-bit fixed point: element i (4 consecutive from a multiple of
// 4 for the vector forms)
__device__ __forceinline__ float acc_ld1(const Params& p, size_t i) {
  if (MK_DET) return fx_to_f(__ldcg(reinterpret_cast<const long long*>(p.moe) + i));
  return __ldcg(p.moe + i);
}
__device__ __forceinline__ float4 acc_ld4(const Params& p, size_t i) {
  if (MK_DET) {
    const longlong2* q = reinterpret_cast<const longlong2*>(reinterpret_cast<const long long*>(p.moe) + i);
    const longlong2 a = __ldcg(q), b = __ldcg(q + 1);
    return make_float4(fx_to_f(a.x), fx_to_f(a.y), fx_to_f(b.x), fx_to_f(b.y));
  }
  return __ldcg(reinterpret_cast<const float4*>(p.moe + i));
}
__device__ __forceinline__ void acc_add1(const Params& p, size_t i, float v) {
  if (MK_DET) red_add_fx(reinterpret_cast<long long*>(p.moe) + i, v);
  else red_add_f32(p.moe + i, v);
}
__device__ __forceinline__ void acc_add4(const Params& p, size_t i, float4 v) {
  if (MK_DET) {
    long long* q = reinterpret_cast<long long*>(p.moe) + i;
    red_add_fx(q, v.x); red_add_fx(q + 1, v.y); red_add_fx(q + 2, v.z); red_add_fx(q + 3, v.w);
  } else {
    red_add_v4(p.moe + i, v);
  }
}
// float4 words of the accumulators (twice as many with 64-bit entries)
__device__ __forceinline__ size_t acc_words4(const Params& p) {
  return (size_t)p.L * p.B * p.d / 4 * (MK_DET ? 2 : 1);
}

// Greedy-token key: larger for a larger logit, then for a lower row (ties go to the
// lowest index); -0 and +0 compare equal; 0 is below every key of a real logit.
__device__ __forceinline__ unsigned long long argmax_key(float v, int row) {
  const unsigned u = __float_as_uint(v + 0.f);
  const unsigned k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)k << 32) | (unsigned)~(unsigned)row;
}

// Two counters polled in the same loop (one detection instead of two in sequence).
__device__ bool wait_ge2(const Params& p, int c1, unsigned t1, int c2, unsigned t2, int task) {
  if (c2 < 0) return wait_ge(p, c1, t1, task);
  const unsigned* a = ctr_ptr(p, c1);
  const unsigned* b = ctr_ptr(p, c2);
  const uint64_t t0 = gtime();
  unsigned ns = 32;
  for (int it = 0;; ++it) {
    const unsigned va = ld_acquire(a), vb = ld_acquire(b);
    if (va >= t1 && vb >= t2) return true;
    __nanosleep(ns);
    ns = ns < 256 ? ns * 2 : 256;
    if ((it & 7) == 7) {
      if (aborted(p)) return false;
      if ((long long)(gtime() - t0) > p.timeout_ns) {
        if (va < t1) raise_err(p, MK_ERR_TIMEOUT, task, c1, (int)va, (int)t1);
        else raise_err(p, MK_ERR_TIMEOUT, task, c2, (int)vb, (int)t2);
        return false;
      }
    }
  }
}

// Consumer-side wait: thread 0 polls, the others learn the result at a barrier.
__device__ bool consumer_wait(const Params& p, const Smem& S, int ci, unsigned target, int task, int ci2 = -1,
                              unsigned target2 = 0) {
  if (ci < 0) {
    trace_mark(p, S, 1);
    return true;
  }
  // thread 0 polls; one OR-reduction barrier hands its result (and, as a barrier, the
  // order of its acquire) to the other consumer threads
  bool ok = false;
  if (threadIdx.x == 0) {
    ok = wait_ge2(p, ci, target, ci2, target2, task);
    if (p.trace) trace_slots(S)[1] = gtime();
  }
  return bar_or_consumers(ok);
}

// Hand a counter release to the storer warp and carry on: each consumer warp orders
// its own output stores before its lane 0 arrives on the request's mbarrier (CTA-scope
// release); the storer waits for all eight warps (acquire) and then performs the
// GPU-scope release-add, which covers the stores it has synchronised with.
__device__ __forceinline__ void signal_async(const Params& p, const Smem& S, uint32_t& sseq, int ci, unsigned v) {
  const uint32_t slot = sseq % kSq, use = sseq / kSq;
  const int lane = threadIdx.x & 31;
  if (use > 0 && lane == 0) mbar_wait(S.sempty(slot), (use - 1) & 1u, 8 * p.timeout_ns);
  __syncwarp();
  if (threadIdx.x == 0) S.sq[slot] = make_int2(ci, (int)v);
  __syncwarp();
  if (lane == 0) mbar_arrive(S.sfull(slot));
  ++sseq;
}

__device__ void storer(const Params& p, const Smem& S) {
  for (uint32_t q = 0;; ++q) {
    const uint32_t slot = q % kSq;
    if (!mbar_wait(S.sfull(slot), (q / kSq) & 1u, 8 * p.timeout_ns)) {
      raise_err(p, MK_ERR_TIMEOUT, -8, -1, (int)q, 0);
      break;
    }
    const int2 r = S.sq[slot];
    mbar_arrive(S.sempty(slot));
    if (r.x < 0) break;
    red_release(ctr_ptr(p, r.x), (unsigned)r.y);
  }
}

__device__ __forceinline__ bool wait_full(const Params& p, const Smem& S, uint32_t seq) {
  if (mbar_wait(S.full(seq % kStages), (seq / kStages) & 1u, 4 * p.timeout_ns)) return true;
  if ((threadIdx.x & 31) == 0) raise_err(p, MK_ERR_TIMEOUT, -2, -1, (int)seq, 0);
  return false;
}
__device__ __forceinline__ void release_stage(const Smem& S, uint32_t seq) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive_relaxed(S.empty(seq % kStages));
}
// Consume n chunks without computing (error / abort path).
__device__ bool drain_chunks(const Params& p, const Smem& S, uint32_t& cseq, int n) {
  for (int i = 0; i < n; ++i) {
    if (!wait_full(p, S, cseq)) return false;
    release_stage(S, cseq);
    ++cseq;
  }
  return true;
}

// ============================================================== counters / items
__device__ __forceinline__ int C_LR(const Params& p, int l) { return p.c_lr + l; }
__device__ __forceinline__ int C_QKVG(const Params& p, int l, int g) { return p.c_qkvg + l * p.Hkv + g; }
__device__ __forceinline__ int C_RT(const Params& p, int l) { return p.c_rt + l; }
__device__ __forceinline__ int C_RR(const Params& p, int l) { return p.c_rr + l; }
__device__ __forceinline__ int C_ATT(const Params& p, int l, int b, int g) {
  return p.c_att + (l * p.B + b) * p.Hkv + g;
}
__device__ __forceinline__ int C_OG(const Params& p, int l, int g) { return p.c_og + l * p.Hkv + g; }
__device__ __forceinline__ int C_MD(const Params& p, int l) { return p.c_md + l; }
__device__ __forceinline__ int C_OA(const Params& p, int l) { return p.c_oa + l; }
__device__ __forceinline__ int C_OD(const Params& p, int l) { return p.c_od + l; }

struct AttItem {
  int b, g, s, ns;      // sequence, KV group, split (s == ns: the new token itself)
  int pos;              // position of the new token
  int pg0, np;          // logical pages of the split
  int klo, khi;         // key positions [klo, khi) of the split
  int part;             // partial slot: ((g*B + b) * max_items_bg + s)
};

// seq_lens are constant during a step: the kernel prologue copies them to smem.
__device__ __forceinline__ const int* seq_lens_s(const Smem& S) { return S.small + 224; }
// The step's epoch (read from device memory at launch): tags the router logits and the
// route words of this step, so that a reader can tell them from the previous step's.
__device__ __forceinline__ unsigned step_epoch(const Smem& S) { return (unsigned)S.small[248]; }
__device__ __forceinline__ uint64_t tagged(unsigned ep, unsigned v) { return ((uint64_t)ep << 32) | v; }

__device__ __forceinline__ int layer_window(const Params& p, int l) {
  return ((p.swa_mask >> l) & 1ull) ? p.window : 0;
}

// Splits of the cached keys in the window of sequence b at layer l.
__device__ __forceinline__ void att_range(const Params& p, const Smem& S, int l, int b, int& pos, int& lo,
                                          int& first_pg, int& npg, int& ns) {
  pos = seq_lens_s(S)[b];
  const int w = layer_window(p, l);
  lo = (w > 0) ? max(0, pos - w + 1) : 0;
  if (pos > lo) {
    first_pg = lo / 16;
    npg = (pos - 1) / 16 - first_pg + 1;
    ns = (npg + p.split_pages - 1) / p.split_pages;
  } else {
    first_pg = 0;
    npg = 0;
    ns = 0;
  }
}

__device__ int att_item_count(const Params& p, const Smem& S, int l) {
  int per_g = 0;
  for (int b = 0; b < p.B; ++b) {
    int pos, lo, fp, npg, ns;
    att_range(p, S, l, b, pos, lo, fp, npg, ns);
    per_g += ns + 1;
  }
  return per_g * p.Hkv;
}

// Items are ordered by (group, sequence, split): group 0's items come first, in
// step with the QKV tiles, which are dealt group by group.
// Queue order: the KV groups interleaved (item = rem * Hkv + g), so that all groups'
// splits are claimed, and their combines finish, at about the same time (the O-proj
// tiles go ahead of expert items once every group is complete).
__device__ AttItem att_decode(const Params& p, const Smem& S, int l, int item) {
  AttItem it;
  it.g = item % p.Hkv;
  int rem = item / p.Hkv;
  for (int b = 0; b < p.B; ++b) {
    int pos, lo, fp, npg, ns;
    att_range(p, S, l, b, pos, lo, fp, npg, ns);
    if (rem <= ns) {
      it.b = b;
      it.s = rem;
      it.ns = ns;
      it.pos = pos;
      if (rem < ns) {
        it.pg0 = fp + rem * p.split_pages;
        it.np = min(p.split_pages, npg - rem * p.split_pages);
        it.klo = max(lo, it.pg0 * 16);
        it.khi = min(pos, (it.pg0 + it.np) * 16);
      } else {
        it.pg0 = 0;
        it.np = 0;
        it.klo = pos;
        it.khi = pos + 1;
      }
      it.part = (it.g * p.B + b) * p.max_items_bg + rem;
      return it;
    }
    rem -= ns + 1;
  }
  it.b = -1;
  return it;
}

__device__ __forceinline__ int checked_page(const Params& p, int b, int logical, int task) {
  int pg = -1;
  if (logical >= 0 && logical < p.max_pages) pg = p.page_table[b * p.max_pages + logical];
  if (pg < 0 || pg >= p.n_pages) {
    raise_err(p, MK_ERR_BAD_PAGE, task, -1, pg, logical);
    return -1;
  }
  return pg;
}

// ============================================================== producer
// The entry's op word: the task's op, layer and whether its aux field is 1 (a dense
// FFN layer, the last router tile), so that the consumer dispatches, and starts an
// expert item, without reading the descriptor from global memory.
__device__ __forceinline__ int op_word(const int* T) {
  return (T[D_OP] & 0xff) | ((T[D_LAYER] & 0xffff) << 8) | ((T[D_AUX] == 1 ? 1 : 0) << 24);
}

__device__ bool mbox_push(const Params& p, const Smem& S, uint32_t& mseq, int task, int item, int nch,
                          int word, int4 extra = make_int4(0, 0, 0, 0), int4 w_lo = make_int4(0, 0, 0, 0),
                          int4 w_hi = make_int4(0, 0, 0, 0), uint64_t stamp = 0) {
  const uint32_t slot = mseq % kMbox, use = mseq / kMbox;
  if (use > 0 && !mbar_wait(S.mempty(slot), (use - 1) & 1u, 8 * p.timeout_ns)) {
    raise_err(p, MK_ERR_TIMEOUT, task, -3, (int)mseq, 0);
    return false;
  }
  S.mbox[4 * slot] = make_int4(task, item, nch, extra.x);
  S.mbox[4 * slot + 1] = make_int4(extra.y, extra.z, (int)(unsigned)stamp, word);
  S.mbox[4 * slot + 2] = w_lo;
  S.mbox[4 * slot + 3] = w_hi;
  mbar_arrive(S.mfull(slot));
  ++mseq;
  return true;
}

// Before chunk `seq` is issued: its stage must be free (consumed), and at most
// p.inflight older chunks may still be in flight.  The ring can hold up to kStages
// landed chunks ahead of the consumers, but only a few are requested at a time:
// that is enough to keep HBM busy, and keeps the memory queues -- which every
// other load of the step also waits in -- short.
__device__ __forceinline__ bool acquire_stage(const Params& p, const Smem& S, uint32_t seq, int task,
                                              int inflight) {
  const uint32_t use = seq / kStages;
  if (use > 0 && !mbar_wait(S.empty(seq % kStages), (use - 1) & 1u, 8 * p.timeout_ns)) {
    raise_err(p, MK_ERR_TIMEOUT, task, -4, (int)seq, 0);
    return false;
  }
  if (seq >= (uint32_t)inflight) {
    const uint32_t q = seq - inflight;
    if (!mbar_wait(S.full(q % kStages), (q / kStages) & 1u, 8 * p.timeout_ns)) {
      raise_err(p, MK_ERR_TIMEOUT, task, -6, (int)q, 0);
      return false;
    }
  }
  return true;
}

// Claim just in time: a queue item is taken only when this CTA's consumers have
// picked up every earlier mailbox entry but the last one, so an SM busy with a long
// task does not hold items that idle SMs could start at once.  (No deadlock: a
// consumer only waits on work that is already claimed -- expert-down items are
// claimed after the expert-up queue is empty -- or on static tasks.)
__device__ __forceinline__ bool claim_gate(const Params& p, const Smem& S, uint32_t mseq, int task) {
  if (mseq < 2) return true;
  const uint32_t q = mseq - 2;
  if (mbar_wait(S.mempty(q % kMbox), (q / kMbox) & 1u, 8 * p.timeout_ns)) return true;
  raise_err(p, MK_ERR_TIMEOUT, task, -7, (int)q, 0);
  return false;
}

__device__ bool issue_linear(const Params& p, const Smem& S, uint32_t& cseq, const uint8_t* src,
                             int bytes, uint64_t pol, int task, int chunk, int inflight) {
  for (int off = 0; off < bytes; off += chunk) {
    const int n = min(chunk, bytes - off);
    if (!acquire_stage(p, S, cseq, task, inflight)) return false;
    const uint32_t s = cseq % kStages;
    mbar_expect_tx(S.full(s), (uint32_t)n);
    bulk_g2s(S.stage(cseq), src + off, (uint32_t)n, S.full(s), pol);
    ++cseq;
  }
  return true;
}

// L2 prefetches (no completion to wait for): they move HBM reads of data that a later
// task on this SM will load -- its own O-proj, QKV and router tiles -- and this SM's
// share of the layer's cached K/V pages into the periods when the layer's dependency
// chain leaves HBM idle, so that the tasks later find their operands in L2.
__device__ __forceinline__ void prefetch_range(const uint8_t* src, int bytes) {
  constexpr int kPiece = 65536;
  for (int off = 0; off < bytes; off += kPiece) prefetch_l2(src + off, (uint32_t)min(kPiece, bytes - off));
}
// This SM's share of layer l's cached pages (the pages attention reads this step,
// counted over all sequences): per page id, the K and the V rows of all KV groups are
// each one contiguous range (Hkv * 16 * hd bf16).
__device__ void prefetch_kv_share(const Params& p, const Smem& S, int l) {
  int total = 0;
  for (int b = 0; b < p.B; ++b) {
    int pos, lo, fp, npg, ns;
    att_range(p, S, l, b, pos, lo, fp, npg, ns);
    total += npg;
  }
  const int beg = (int)((long long)total * blockIdx.x / gridDim.x);
  const int end = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  const uint32_t span = (uint32_t)p.Hkv * 16u * (uint32_t)p.hd * 2u;
  int base = 0;
  for (int b = 0; b < p.B && base < end; ++b) {
    int pos, lo, fp, npg, ns;
    att_range(p, S, l, b, pos, lo, fp, npg, ns);
    for (int i = max(beg - base, 0); i < npg && base + i < end; ++i) {
      const int logical = fp + i;
      if (logical >= p.max_pages) break;
      const int pg = p.page_table[b * p.max_pages + logical];
      if (pg < 0 || pg >= p.n_pages) continue;  // reported by the tasks that use it
      const size_t o = (((size_t)l * p.n_pages + pg) * p.Hkv) * 16 * p.hd;
      prefetch_l2(p.kc + o, span);
      prefetch_l2(p.vc + o, span);
    }
    base += npg;
  }
}

// K pages then V pages of a split, 8 pages per ring stage, one tensor-map copy per page.
__device__ bool issue_kv(const Params& p, const Smem& S, uint32_t& cseq, const CUtensorMap* tmK,
                         const CUtensorMap* tmV, int l, const AttItem& it, uint64_t pol, int task) {
  const int page_bytes = 16 * p.hd * 2;
  // page ids of the first chunk, then each chunk's ids are loaded (all 8 at once)
  // while the previous chunk's copies are issued
  int ids[8];
  auto load_ids = [&](int c0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int logical = it.pg0 + c0 + i;
      ids[i] = -1;
      ldg_cg_pred_i(ids[i], p.page_table + it.b * p.max_pages + logical,
                    c0 + i < it.np && logical >= 0 && logical < p.max_pages);
    }
  };
  load_ids(0);
  for (int c0 = 0; c0 < it.np; c0 += 8) {
    const int n = min(8, it.np - c0);
    int rows[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int pg = ids[i];
      if (i < n && (pg < 0 || pg >= p.n_pages)) {
        raise_err(p, MK_ERR_BAD_PAGE, task, -1, pg, it.pg0 + c0 + i);
        pg = 0;
      }
      rows[i] = ((l * p.n_pages + max(pg, 0)) * p.Hkv + it.g) * 16;
    }
    if (c0 + 8 < it.np) load_ids(c0 + 8);
    for (int kv = 0; kv < 2; ++kv) {
      if (!acquire_stage(p, S, cseq, task, p.inflight)) return false;
      const uint32_t s = cseq % kStages;
      mbar_expect_tx(S.full(s), (uint32_t)(n * page_bytes));
      const uint32_t dst = S.stage(cseq);
      const CUtensorMap* tm = kv ? tmV : tmK;
      for (int i = 0; i < n; ++i) {  // one box per page
        if (p.hd == 128)
          tma_load_3d(dst + i * page_bytes, tm, 0, 0, rows[i], S.full(s), pol);
        else
          tma_load_2d(dst + i * page_bytes, tm, 0, rows[i], S.full(s), pol);
      }
      ++cseq;
    }
  }
  return true;
}

// A GEMV tile task: mailbox entry, then its weight chunks.
__device__ __forceinline__ bool push_gemv(const Params& p, const Smem& S, uint32_t& mseq, uint32_t& cseq, int ti,
                                          uint64_t pol, int inflight) {
  const int* T = p.tasks + ti * kDescInts;
  const long long off = (long long)(((unsigned long long)(unsigned)T[D_WOFF_HI] << 32) | (unsigned)T[D_WOFF_LO]);
  const int bytes = T[D_WBYTES];
  const int nrb = T[D_NROWS] / 16;
  const bool f8 = p.fp8d && T[D_OP] != OP_ROUTER;  // (FP8 projections: QKV, O-proj, LM head)
  const int cs = f8 ? gemv_jpc8(nrb) * nrb * 8 * kFragBytes8 : gemv_jpc(nrb) * nrb * 8 * kFragBytes;
  const int nch = (bytes + cs - 1) / cs;
  return mbox_push(p, S, mseq, ti, 0, nch, op_word(T)) &&
         issue_linear(p, S, cseq, p.wblob + off, bytes, pol, ti, cs, inflight);
}

__device__ void producer(const Params& p, const Smem& S, const CUtensorMap* tmK, const CUtensorMap* tmV) {
  const uint64_t pol = policy_evict_first();
  uint32_t cseq = 0, mseq = 0;
  const int beg = p.sm_off[blockIdx.x], end = p.sm_off[blockIdx.x + 1];
  bool ok = true;
  for (int li = beg; li < end && ok; ++li) {
    if (aborted(p)) break;
    const int ti = p.sm_list[li];
    const int* T = p.tasks + ti * kDescInts;
    const int op = T[D_OP];
    const int l = T[D_LAYER];
    switch (op) {
      case OP_EMBED:
      case OP_RESID:
        ok = mbox_push(p, S, mseq, ti, 0, 0, op_word(T));
        break;
      case OP_PREFETCH: {
        const long long off = (long long)(((unsigned long long)(unsigned)T[D_WOFF_HI] << 32) |
                                          (unsigned)T[D_WOFF_LO]);
        prefetch_range(p.wblob + off, T[D_WBYTES]);
        break;
      }
      case OP_PREFETCH_KV:
        prefetch_kv_share(p, S, l);
        break;
      case OP_QKV:
      case OP_ROUTER:
      case OP_OPROJ:
      case OP_LMHEAD:
        ok = push_gemv(p, S, mseq, cseq, ti, pol, p.inflight);
        break;
      case OP_ATT_DRAIN: {
        const int count = att_item_count(p, S, l);
        int* head = p.qhead + l;
        while (ok) {
          if (!(ok = claim_gate(p, S, mseq, ti))) break;
          const int item = atomicAdd(head, 1);
          if (item >= count) break;
          const AttItem it = att_decode(p, S, l, item);
          const int nch = 2 * ((it.np + 7) / 8);
          ok = mbox_push(p, S, mseq, ti, item, nch, op_word(T)) && issue_kv(p, S, cseq, tmK, tmV, l, it, pol, ti);
        }
        break;
      }
      case OP_MOE_DRAIN: {
        // The first claim is taken before the layer's route is known (its round trip
        // overlaps the wait).  The route words an item needs -- n_active, the expert of
        // its slot, the slot's tokens and their weights -- are polled until they carry
        // this step's epoch: the detection and the data come with the same loads, and
        // the consumers get tokens and weights in the mailbox entry.
        const int q = p.L + l;
        if (!(ok = claim_gate(p, S, mseq, ti))) break;
        int item = atomicAdd(p.qhead + q, 1);
        const uint64_t* rw = p.rword + (size_t)l * p.rw_stride;
        const unsigned ep = step_epoch(S);
        const int maxa = p.maxa;
        int nact = -1, tl_slot = -1, tl_e = 0, tl_cnt = 0, tl_tok[kMaxBatch], tl_w[kMaxBatch];
        // the items' operand (bf16(x_l * gain), 1/rms) is written by the previous layer's
        // ADD_RMSNORM tasks: their counter is read (and acquired) in the same batch
        bool lr_done = false;
        const unsigned* lr_ctr = ctr_ptr(p, C_LR(p, l));
        const unsigned lr_target = (unsigned)p.nrb_d;
        // a dense layer of a mixed stack: one FFN for every token with weight 1 (no route
        // words; only the items' operand is waited for)
        const bool dense = T[D_AUX] == 1;
        auto fetch = [&](int a) -> bool {  // slot a's words (and n_active while unknown)
          const uint64_t t0 = gtime();
          unsigned ns = 32;
          if (dense) {
            for (int it = 0; ld_acquire(lr_ctr) < lr_target; ++it) {  // acquire: the ADD_RMSNORM outputs
              __nanosleep(64);
              if ((it & 15) == 15 && (aborted(p) || (long long)(gtime() - t0) > p.timeout_ns)) {
                if (!aborted(p)) raise_err(p, MK_ERR_TIMEOUT, ti, C_LR(p, l), -1, (int)lr_target);
                return false;
              }
            }
            lr_done = true;
            nact = 1;
            tl_slot = 0;
            tl_e = 0;
            tl_cnt = p.B;
#pragma unroll
            for (int n = 0; n < kMaxBatch; ++n) {
              tl_tok[n] = n < p.B ? n * 16 : 0;
              tl_w[n] = n < p.B ? __float_as_int(1.f) : 0;
            }
            return true;
          }
          for (int it = 0;; ++it) {
            const bool sl = a >= 0 && a < maxa;
            const int as = sl ? a : 0;
            const unsigned lr = lr_done ? lr_target : ld_acquire(lr_ctr);  // acquire: the ADD_RMSNORM outputs
            uint64_t wn = 0, we = 0, wc = 0, wt[kMaxBatch], ww[kMaxBatch];
            ld_relaxed_u64_pred(wn, rw, nact < 0);
            ld_relaxed_u64_pred(we, rw + 1 + as, sl);
            ld_relaxed_u64_pred(wc, rw + 1 + maxa + as, sl);
#pragma unroll
            for (int n = 0; n < kMaxBatch; ++n) {
              wt[n] = ww[n] = 0;
              ld_relaxed_u64_pred(wt[n], rw + 1 + 2 * maxa + as * p.B + n, sl && n < p.B);
              ld_relaxed_u64_pred(ww[n], rw + 1 + 2 * maxa + maxa * p.B + as * p.B + n, sl && n < p.B);
            }
            if (nact < 0 && (unsigned)(wn >> 32) == ep) nact = (int)(unsigned)wn;
            if (!lr_done && lr >= lr_target) lr_done = true;
            if (nact >= 0 && lr_done) {
              if (!sl || a >= nact) return true;  // no such item
              const int c2 = (int)(unsigned)wc;
              bool good = (unsigned)(we >> 32) == ep && (unsigned)(wc >> 32) == ep;
#pragma unroll
              for (int n = 0; n < kMaxBatch; ++n)
                if (n < c2 && ((unsigned)(wt[n] >> 32) != ep || (unsigned)(ww[n] >> 32) != ep)) good = false;
              if (good) {
                tl_slot = a;
                tl_e = (int)(unsigned)we;
                tl_cnt = c2;
#pragma unroll
                for (int n = 0; n < kMaxBatch; ++n) {
                  tl_tok[n] = (n < c2) ? (int)(unsigned)wt[n] : 0;
                  tl_w[n] = (n < c2) ? (int)(unsigned)ww[n] : 0;
                }
                return true;
              }
            }
            __nanosleep(ns);
            ns = ns < 64 ? ns * 2 : 64;
            if ((it & 15) == 15) {
              if (aborted(p)) return false;
              if ((long long)(gtime() - t0) > p.timeout_ns) {
                raise_err(p, MK_ERR_TIMEOUT, ti, -12, a, (int)ep);
                return false;
              }
            }
          }
        };
        if (!fetch(dense ? 0 : item / p.t_moe)) { ok = false; break; }
        const int count = dense ? p.t_dense : nact * p.t_moe;
        // part 1 (gate/up tile) in whole k16-groups, part 2 (down slice) in warp regions
        // (FP8 experts: a chunk of the item's scales first, fragments of half the bytes;
        // a dense layer's FFN items stay bf16)
        const bool f8 = p.fp8 && !dense;
        const int fs = dense ? p.dense_fs : p.moe_fs;
        const long long ib = dense ? p.dense_item_bytes : p.moe_item_bytes;
        const int nrb1 = fs / 8;
        const int fb = f8 ? kFragBytes8 : kFragBytes;
        const int sb = f8 ? fp8_scale_bytes(fs, p.d) : 0;
        const int cs1 = (f8 ? gemv_jpc8(nrb1) : gemv_jpc(nrb1)) * nrb1 * 8 * fb;
        const int gu_bytes = 2 * fs * p.d * fb / 256;
        const int region = (p.d / 128) * (fs / 16) * fb;
        const int cs2 = moe_warps_per_chunk(region) * region;
        const int dn_bytes = (int)ib - sb - gu_bytes;
        const int nch = (sb > 0) + (gu_bytes + cs1 - 1) / cs1 + (dn_bytes + cs2 - 1) / cs2;
        // O-proj tiles of the layer as a queue (D_KLEN tiles from task D_K0; none when
        // they are dealt statically): taken before expert items once all attention
        // outputs of the layer are complete, and after the expert queue empties
        const int qo = 2 * p.L + l, o_base = T[D_K0], n_o = T[D_KLEN];
        bool o_left = n_o > 0;
        auto claim_oproj = [&]() {
          const int o = atomicAdd(p.qhead + qo, 1);
          if (o >= n_o) { o_left = false; return false; }
          ok = push_gemv(p, S, mseq, cseq, o_base + o, pol, p.tail_items > 0 ? p.inflight_tail : p.inflight);
          return true;
        };
        for (bool first = true; ok; first = false) {
          if (!first) {
            // read ahead: the count arrives while the claim gate waits for the consumers
            const unsigned oa = o_left ? ld_relaxed(ctr_ptr(p, C_OA(p, l))) : 0u;
            if (!(ok = claim_gate(p, S, mseq, ti))) break;
            if (o_left && oa >= (unsigned)(p.Hkv * p.B) && claim_oproj()) continue;
            item = atomicAdd(p.qhead + q, 1);
          }
          if (item >= count) break;
          const int a = dense ? 0 : item / p.t_moe, t = dense ? item : item % p.t_moe;
          if (a != tl_slot && !fetch(a)) { ok = false; break; }
          const int e = tl_e;
          int4 extra = make_int4(tl_cnt, 0, 0, 0);
#pragma unroll
          for (int n = 0; n < kMaxBatch; ++n) {
            const int byte = ((tl_tok[n] >> 4) << 3) | (tl_tok[n] & 7);
            if (n < 4) extra.y |= byte << (8 * n);
            else extra.z |= byte << (8 * (n - 4));
          }
          const uint8_t* src =
              dense ? p.wblob + p.off_dense +
                          ((long long)__popcll(p.dense_mask & ((1ull << l) - 1ull)) * p.t_dense + t) * ib
                    : p.wblob + p.off_moe + ((long long)(l * p.E + e) * p.t_moe + t) * p.moe_item_bytes;
          const int fl = (p.tail_items > 0 && item >= count - p.tail_items) ? p.inflight_tail : p.inflight_moe;
          ok = mbox_push(p, S, mseq, ti, item, nch, op_word(T), extra, make_int4(tl_w[0], tl_w[1], tl_w[2], tl_w[3]),
                         make_int4(tl_w[4], tl_w[5], tl_w[6], tl_w[7]), p.trace ? gtime() : 0ull) &&
               (sb == 0 || issue_linear(p, S, cseq, src, sb, pol, ti, sb, fl)) &&
               issue_linear(p, S, cseq, src + sb, gu_bytes, pol, ti, cs1, fl) &&
               issue_linear(p, S, cseq, src + sb + gu_bytes, dn_bytes, pol, ti, cs2, fl);
        }
        // after the expert queue empties: while the layer's attention outputs are
        // incomplete a producer holds at most one O-proj tile (its weights land while
        // it waits); the rest go to whichever SMs are free once they are complete,
        // instead of queueing behind the first on the SMs that emptied the queue
        bool held = false;
        while (ok && o_left) {
          if (!(ok = claim_gate(p, S, mseq, ti))) break;
          if (held && !(ok = wait_ge(p, C_OA(p, l), (unsigned)(p.Hkv * p.B), ti))) break;
          held = ld_relaxed(ctr_ptr(p, C_OA(p, l))) < (unsigned)(p.Hkv * p.B);
          claim_oproj();
        }
        break;
      }
      default:
        break;
    }
  }
  mbox_push(p, S, mseq, -1, 0, 0, 0);
  // make sure no copy is still landing in shared memory when the CTA retires
  const uint32_t first = cseq > (uint32_t)kStages ? cseq - kStages : 0;
  for (uint32_t q = first; q < cseq; ++q) mbar_wait(S.full(q % kStages), (q / kStages) & 1u, 8 * p.timeout_ns);
}

// ============================================================== GEMV machinery
struct BFrag {
  uint32_t b0[kMaxKsw], b1[kMaxKsw];
};

// B operand (activations) for this warp's k16-steps ks = warp + 8 j: row n = lane/4
// of the operand is one token's activation row `row` (bf16, nullptr for a zero row);
// the lane holds the pairs at k = 16 ks + 2 (lane%4) and k + 8.  All loads are
// issued before any is used.
__device__ __forceinline__ void load_bfrag(BFrag& fr, int ksw, const uint16_t* row) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane & 3;
  const bool on = row != nullptr;
  const uint16_t* base = on ? row + 16 * warp + 2 * c : nullptr;
#pragma unroll
  for (int j = 0; j < kMaxKsw; ++j) {
    fr.b0[j] = 0u;
    fr.b1[j] = 0u;
    const bool pj = on && j < ksw;
    ldg_cg_pred(fr.b0[j], base + 128 * j, pj);
    ldg_cg_pred(fr.b1[j], base + 128 * j + 8, pj);
  }
}

// acc[rb] += W_tile[rb] * act over this warp's k16-steps ks = warp + 8 j, consuming the
// task's ring chunks.  Tiles are packed so that fragment (rb, ks) sits at index
// (j * NRB + rb) * 8 + warp: every ring chunk holds JPC = floor(8 / NRB) consecutive j
// for all row blocks (JPC * NRB * 4 KB <= 32 KB), so chunk, register and smem indices
// are compile-time constants.
// With `lo` non-null the operand is the exact-ish sum hi + lo of two bf16 parts and
// every fragment is multiplied twice (router logits: top-k decisions need them to
// ~1e-5; the tensor-core work is negligible against the weight bytes).
template <int NRB>
__device__ __forceinline__ bool gemv_mainloop(const Params& p, const Smem& S, uint32_t& cseq, int nch,
                                              int ksw, const BFrag& fr, float (&acc)[NRB][4],
                                              const BFrag* lo = nullptr) {
  constexpr int JPC = gemv_jpc(NRB);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int r = 0; r < NRB; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
  if (nch <= 0) return true;
#pragma unroll
  for (int j = 0; j < kMaxKsw; ++j) {
    if (j < ksw) {
      const int c = j / JPC;
      if (j % JPC == 0) {
        if (c > 0) release_stage(S, cseq + c - 1);
        if (!wait_full(p, S, cseq + c)) return false;
        if (c == 0) trace_mark(p, S, 2);
      }
      const uint32_t base = S.stage(cseq + c) + ((j % JPC) * NRB * 8 + warp) * kFragBytes + lane * 16;
#pragma unroll
      for (int rb = 0; rb < NRB; ++rb) {
        const uint4 a = lds128(base + rb * 8 * kFragBytes);
        mma_bf16(acc[rb], a.x, a.y, a.z, a.w, fr.b0[j], fr.b1[j]);
        if (lo) mma_bf16(acc[rb], a.x, a.y, a.z, a.w, lo->b0[j], lo->b1[j]);
      }
    }
  }
  release_stage(S, cseq + (ksw - 1) / JPC);
  cseq += nch;
  return true;
}

// Cross-warp sum.  Afterwards thread (warp w, lane) holds out[] for row block w:
// out[0] = (row 16w+g, token 2c), out[1] = (16w+g, 2c+1), out[2] = (16w+g+8, 2c),
// out[3] = (16w+g+8, 2c+1), g = lane/4, c = lane%4.
template <int NRB>
__device__ __forceinline__ void gemv_reduce(const Smem& S, const float (&acc)[NRB][4], float (&out)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float4* scr = reinterpret_cast<float4*>(S.scratch);
#pragma unroll
  for (int rb = 0; rb < NRB; ++rb)
    scr[(warp * NRB + rb) * 32 + lane] = make_float4(acc[rb][0], acc[rb][1], acc[rb][2], acc[rb][3]);
  bar_sync_consumers();
  out[0] = out[1] = out[2] = out[3] = 0.f;
  if (warp < NRB) {
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float4 v = scr[(w * NRB + warp) * 32 + lane];
      out[0] += v.x; out[1] += v.y; out[2] += v.z; out[3] += v.w;
    }
  }
}

// The same reduction through at most 16 KB of scratch (4 row blocks at a time): the
// FP8 expert items keep their scales in the scratch above that.
template <int NRB>
__device__ __forceinline__ void gemv_reduce16k(const Smem& S, const float (&acc)[NRB][4], float (&out)[4]) {
  if (NRB <= 4) {
    gemv_reduce<NRB>(S, acc, out);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float4* scr = reinterpret_cast<float4*>(S.scratch);
  out[0] = out[1] = out[2] = out[3] = 0.f;
#pragma unroll
  for (int h = 0; h < NRB; h += 4) {
    if (h > 0) bar_sync_consumers();  // every warp has read the previous half
#pragma unroll
    for (int rb = 0; rb < 4; ++rb)
      scr[(warp * 4 + rb) * 32 + lane] =
          make_float4(acc[h + rb][0], acc[h + rb][1], acc[h + rb][2], acc[h + rb][3]);
    bar_sync_consumers();
    if (warp >= h && warp < h + 4) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float4 v = scr[(w * 4 + warp - h) * 32 + lane];
        out[0] += v.x; out[1] += v.y; out[2] += v.z; out[3] += v.w;
      }
    }
  }
}

template <int NRB>
__device__ __forceinline__ bool gemv_run(const Params& p, const Smem& S, uint32_t& cseq, int nch, int ksw,
                                         const BFrag& fr, float (&v)[4], const BFrag* lo = nullptr) {
  float acc[NRB][4];
  if (!gemv_mainloop<NRB>(p, S, cseq, nch, ksw, fr, acc, lo)) return false;
  trace_mark(p, S, 3);
  gemv_reduce<NRB>(S, acc, v);
  return true;
}

// One E4M3 A-fragment (8 codes a lane) decoded on the integer pipe to f16 values
// scaled by 2^-8 (undone with the f32 scales) and multiplied in.  (The conversion
// instruction was measured slower here: -1.5% at batch 1 with the whole decode on it,
// -1.3% with half.)
__device__ __forceinline__ void fp8_mma(float (&acc)[4], uint2 a, uint32_t b0, uint32_t b1) {
  uint32_t r0, r1, r2, r3;
  e4m3x4_to_f16x2_scaled(a.x, r0, r1);
  e4m3x4_to_f16x2_scaled(a.y, r2, r3);
  mma_f16(acc, r0, r1, r2, r3, b0, b1);
}

// The GEMV on E4M3 weight fragments (FP8 experts): 8 bytes a lane per fragment,
// widened exactly to f16 (x 2^-8) and multiplied with the f16 operand `fr` (f32
// accumulation); twice the j-groups per ring chunk.  The row scales are applied by
// the caller.
template <int NRB, bool CVT = false>
__device__ __forceinline__ bool gemv_run8(const Params& p, const Smem& S, uint32_t& cseq, int nch, int ksw,
                                          const BFrag& fr, float (&v)[4]) {
  constexpr int JPC = gemv_jpc8(NRB);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[NRB][4];
#pragma unroll
  for (int r = 0; r < NRB; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;
  if (nch > 0) {
#pragma unroll
    for (int j = 0; j < kMaxKsw; ++j) {
      if (j < ksw) {
        const int c = j / JPC;
        if (j % JPC == 0) {
          if (c > 0) release_stage(S, cseq + c - 1);
          if (!wait_full(p, S, cseq + c)) return false;
          if (c == 0) trace_mark(p, S, 2);
        }
        const uint32_t base = S.stage(cseq + c) + ((j % JPC) * NRB * 8 + warp) * kFragBytes8 + lane * 8;
        // CVT: the operand is bf16 (shared with the bf16 tiles), widened to f16 here
        const uint32_t b0 = CVT ? bf16x2_to_f16x2(fr.b0[j]) : fr.b0[j];
        const uint32_t b1 = CVT ? bf16x2_to_f16x2(fr.b1[j]) : fr.b1[j];
#pragma unroll
        for (int rb = 0; rb < NRB; ++rb) {
          const uint2 a = lds64(base + rb * 8 * kFragBytes8);
          fp8_mma(acc[rb], a, b0, b1);
        }
      }
    }
    release_stage(S, cseq + (ksw - 1) / JPC);
    cseq += nch;
  }
  trace_mark(p, S, 3);
  gemv_reduce16k<NRB>(S, acc, v);
  return true;
}

// 1 / rms of x_b (layer input) from the per-row-block sums of squares.
// 1/rms of token b entering `layer`, from the per-row-block sums of squares; all
// partials are loaded before any is summed (one L2 round trip).
__device__ __forceinline__ float rstd_of(const Params& p, int layer, int b) {
  const float* ss = p.SS + (size_t)layer * p.nrb_d * kSsStride + b;
  constexpr int kMaxRb = 2048 / kRowBlock;
  float v[kMaxRb];
#pragma unroll
  for (int r = 0; r < kMaxRb; ++r) {
    v[r] = 0.f;
    ldg_cg_pred(v[r], ss + r * kSsStride, r < p.nrb_d);
  }
  float s = 0.f;
#pragma unroll
  for (int r = 0; r < kMaxRb; ++r) s += v[r];
  return rsqrtf(s / (float)p.d + p.eps);
}

// 1/rms of every token, computed once per CTA (threads 0..B-1) into shared memory.
__device__ __forceinline__ float* rstd_smem(const Smem& S) { return reinterpret_cast<float*>(S.small + 240); }
__device__ __forceinline__ void rstd_all(const Params& p, const Smem& S, int layer) {
  if (threadIdx.x < p.B) rstd_smem(S)[threadIdx.x] = rstd_of(p, layer, threadIdx.x);
  bar_sync_consumers();
}

// B operand of the normed input: bf16(x_layer * gain) pairs written by the residual
// step (or the embedding), loaded as-is; the per-token 1/rms is applied to the GEMV
// output in the epilogue.  `b` is the token of this lane's operand row (lane/4), or
// -1 for a zero row.  Returns this lane's token's 1/rms (0 for a zero row).
__device__ __forceinline__ float build_norm_bfrag(const Params& p, const Smem& S, BFrag& fr, int ksw, int layer,
                                                 int b) {
  load_bfrag(fr, ksw, b < 0 ? nullptr : p.XG + ((size_t)layer * p.B + b) * p.d);
  rstd_all(p, S, layer);
  return b < 0 ? 0.f : rstd_smem(S)[b];
}

// Normed operand of layer l >= 1 straight from its parts, without waiting for the
// ADD_RMSNORM step: x_l = x_{l-1} + the accumulator of layer l-1 (expert and O-proj
// outputs).  The B fragments get bf16(x_l * gain) (and, with `lo`, the bf16 residue of
// the product); the returned value is 1/rms of this lane's token row (lane / 4).  The
// products are staged in scratch as bf16 rows [token][d] whose 16-byte chunks are
// XOR-swizzled by the token index (conflict-free fragment reads); with `lo`, hi rows
// sit at 0 and lo rows at 16 KB, four tokens per pass.
__device__ float build_operand_parts(const Params& p, const Smem& S, BFrag& fr, BFrag* lo, int ksw, int l) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = lane & 3, nl = lane >> 2;
  const int d = p.d, B = p.B, d4 = d / 4;
  const float* xa = p.X + (size_t)(l - 1) * B * d;
  const size_t ma = (size_t)(l - 1) * B * d;  // accumulator of layer l - 1
  const float4* gain4 = reinterpret_cast<const float4*>(p.attn_norm + (size_t)l * d);
  uint8_t* st = reinterpret_cast<uint8_t*>(S.scratch);
  float* ssw = reinterpret_cast<float*>(S.small + 16);  // [8 warps][8 tokens] partial sums
  const int row_bytes = 2 * d;
  const int per_pass = lo ? 4 : 8;
#pragma unroll
  for (int j = 0; j < kMaxKsw; ++j) {
    fr.b0[j] = fr.b1[j] = 0u;
    if (lo) lo->b0[j] = lo->b1[j] = 0u;
  }
  constexpr int kG = 2048 / 4 / kConsumerThreads;  // float4 groups per thread (d <= 2048)
  constexpr int kU = 2;                             // tokens whose loads are in flight together
  float4 gv[kG];
#pragma unroll
  for (int q = 0; q < kG; ++q) {
    const int g = tid + q * kConsumerThreads;
    gv[q] = g < d4 ? gain4[g] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int t0 = 0; t0 < B; t0 += per_pass) {
    const int t1 = min(B, t0 + per_pass);
    for (int u0 = t0; u0 < t1; u0 += kU) {
      // loads of kU tokens in flight together
      float4 av[kU][kG], mv[kU][kG];
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int q = 0; q < kG; ++q) {
          const int n = u0 + u, g = tid + q * kConsumerThreads;
          av[u][q] = mv[u][q] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (n < t1 && g < d4) {
            av[u][q] = __ldcg(reinterpret_cast<const float4*>(xa + (size_t)n * d) + g);
            mv[u][q] = acc_ld4(p, ma + (size_t)n * d + 4 * (size_t)g);
          }
        }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int n = u0 + u;
        float s2 = 0.f;
#pragma unroll
        for (int q = 0; q < kG; ++q) {
          const int g = tid + q * kConsumerThreads;
          if (n < t1 && g < d4) {
            const float x0 = av[u][q].x + mv[u][q].x, x1 = av[u][q].y + mv[u][q].y;
            const float x2 = av[u][q].z + mv[u][q].z, x3 = av[u][q].w + mv[u][q].w;
            s2 += x0 * x0 + x1 * x1 + x2 * x2 + x3 * x3;
            const float y0 = x0 * gv[q].x, y1 = x1 * gv[q].y, y2 = x2 * gv[q].z, y3 = x3 * gv[q].w;
            const uint16_t h0 = to_bf16(y0), h1 = to_bf16(y1), h2 = to_bf16(y2), h3 = to_bf16(y3);
            const int off = (n - t0) * row_bytes + ((((g >> 1) ^ (n & 7))) << 4) + (g & 1) * 8;
            *reinterpret_cast<uint2*>(st + off) =
                make_uint2((uint32_t)h0 | ((uint32_t)h1 << 16), (uint32_t)h2 | ((uint32_t)h3 << 16));
            if (lo) {
              const uint16_t l0 = to_bf16(y0 - bf16_to_f(h0)), l1 = to_bf16(y1 - bf16_to_f(h1));
              const uint16_t l2 = to_bf16(y2 - bf16_to_f(h2)), l3 = to_bf16(y3 - bf16_to_f(h3));
              *reinterpret_cast<uint2*>(st + 16384 + off) =
                  make_uint2((uint32_t)l0 | ((uint32_t)l1 << 16), (uint32_t)l2 | ((uint32_t)l3 << 16));
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        if (lane == 0 && n < t1) ssw[warp * 8 + n] = s2;
      }
    }
    if (t0 == 0) trace_mark(p, S, 15);
    bar_sync_consumers();
    if (tid >= t0 && tid < t1) {
      float s2 = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) s2 += ssw[w * 8 + tid];
      rstd_smem(S)[tid] = rsqrtf(s2 / (float)d + p.eps);
    }
    if (nl >= t0 && nl < t1) {
      const uint8_t* row = st + (nl - t0) * row_bytes;
#pragma unroll
      for (int j = 0; j < kMaxKsw; ++j) {
        if (j < ksw) {
          const int ks = warp + 8 * j;
          const int o0 = (((2 * ks) ^ (nl & 7)) << 4) + 4 * c, o1 = (((2 * ks + 1) ^ (nl & 7)) << 4) + 4 * c;
          fr.b0[j] = *reinterpret_cast<const uint32_t*>(row + o0);
          fr.b1[j] = *reinterpret_cast<const uint32_t*>(row + o1);
          if (lo) {
            lo->b0[j] = *reinterpret_cast<const uint32_t*>(row + 16384 + o0);
            lo->b1[j] = *reinterpret_cast<const uint32_t*>(row + 16384 + o1);
          }
        }
      }
    }
    bar_sync_consumers();
  }
  return nl < B ? rstd_smem(S)[nl] : 0.f;
}

// ============================================================== epilogues / fan-in steps

// Route step of a batch of one token, on one warp (warp 0; the other consumer warps
// do not take part): the 128-or-fewer tagged logits are polled four to a lane until they
// all carry this step's epoch, the top_k are taken in K rounds of a warp-wide argmax (the
// larger logit wins, then the lower expert id; a NaN ranks below every number and reports
// MK_ERR_NAN), the softmax over them runs in registers, and each selected expert is placed
// in its slot (the number of selected ids below it) and published in the route words.
// Returns nothing: a timeout raises the error word (every wait then drains).
__device__ void route_step_b1(const Params& p, const Smem& S, int l, int ti) {
  const int lane = threadIdx.x & 31;
  const int E = p.E, K = p.topk;
  constexpr int kPer = 8;  // logits a lane holds (E <= 256)
  const unsigned ep = step_epoch(S);
  const uint64_t* src = p.rlog + (size_t)l * E;
  float v[kPer];
  const uint64_t t0 = gtime();
  for (int it = 0;; ++it) {
    bool ok = true;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = lane + 32 * j;
      uint64_t w = tagged(ep, 0xff800000u);  // -inf for lanes past E
      ld_relaxed_u64_pred(w, src + e, e < E);
      if ((unsigned)(w >> 32) != ep) ok = false;
      v[j] = __uint_as_float((unsigned)w);
    }
    if (__all_sync(0xffffffffu, ok)) break;
    __nanosleep(32);
    if ((it & 15) == 15 && (aborted(p) || (long long)(gtime() - t0) > p.timeout_ns)) {
      if (lane == 0 && !aborted(p)) raise_err(p, MK_ERR_TIMEOUT, ti, -11, l, 0);
      return;
    }
  }
  if (p.trace && lane == 0) trace_slots(S)[6] = gtime();
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if (v[j] != v[j]) {
      raise_err(p, MK_ERR_NAN, ti, -1, l, lane + 32 * j);
      v[j] = -INFINITY;
    }
  // K rounds: this lane's best (value, lowest id), then the warp's; the winner's lane
  // takes it out of its list
  float sv = -INFINITY;   // lane j < K: the j-th selected logit
  int se = 0x7fffffff;    //             and its expert id
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = lane + 32 * j;
      if (e < E && (v[j] > bv || (v[j] == bv && e < be))) { bv = v[j]; be = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
    }
    if (lane == k) { sv = bv; se = be; }
    // the winner is taken: NaN never compares larger or equal, so it is not chosen again
    // (not even among ties at -inf)
#pragma unroll
    for (int j = 0; j < kPer; ++j)
      if (lane + 32 * j == be) v[j] = __int_as_float(0x7fc00000u);
  }
  if (p.trace && lane == 0) trace_slots(S)[13] = gtime();
  // softmax over the selected logits (lane 0 holds the largest)
  const float mx = __shfl_sync(0xffffffffu, sv, 0);
  const float w = (lane < K) ? __expf(sv - mx) : 0.f;
  float sum = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float wk = w / sum;
  trace_mark(p, S, 8);
  const int maxa = p.maxa;
  int slot = 0;
  for (int j = 0; j < K; ++j) slot += __shfl_sync(0xffffffffu, se, j) < se ? 1 : 0;
  uint64_t* rw = p.rword + (size_t)l * p.rw_stride;
  if (lane < K) {
    rw[1 + 2 * maxa + slot] = tagged(ep, (unsigned)lane);  // token 0, selection rank
    rw[1 + 2 * maxa + maxa + slot] = tagged(ep, __float_as_uint(wk));
    rw[1 + slot] = tagged(ep, (unsigned)se);
    rw[1 + maxa + slot] = tagged(ep, 1u);
  }
  __syncwarp();
  if (lane == 0) {
    rw[0] = tagged(ep, (unsigned)K);
    if (p.trace) trace_slots(S)[10] = gtime();
  }
  // the routing in plain arrays (host-side readers), and the MoE-done padding
  if (lane < K) {
    p.ridx[(size_t)l * K + lane] = se;
    p.rw[(size_t)l * K + lane] = wk;
    p.active[l * maxa + slot] = se;
    p.act_cnt[l * maxa + slot] = 1;
    p.act_tok[(size_t)l * maxa + slot] = lane;
  }
  if (lane == 0) {
    p.nact[l] = K;
    p.qcount[p.L + l] = K * p.t_moe;
    const unsigned pad = (unsigned)((maxa - K) * p.t_moe);
    if (pad > 0) atomicAdd(ctr_ptr(p, C_MD(p, l)), pad);
    if (p.trace) trace_slots(S)[11] = gtime();
  }
}

// Route step: top-k of the router logits per token (ties to the lower expert id),
// softmax over the selected logits, the active-expert list in ascending expert id,
// per-expert token lists in (token, slot) order, and the layer's MoE queue sizes.
// Top-k by counting: thread (b, e) finds the rank of logit e = how many logits of
// token b beat it; ranks below top_k are the selection, in descending order.
__device__ bool route_step(const Params& p, const Smem& S, int l, int ti) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* sel = S.small + 16;                               // [B][topk] expert ids (<= 64)
  float* lg = S.scratch;                                 // [B][E] logits
  int* slot_of = reinterpret_cast<int*>(S.scratch) + kMaxBatch * 256;  // [E]
  int* act_s = slot_of + 256;                            // [maxa] active expert ids
  int* cnt_s = act_s + kMaxActive;                       // [maxa] tokens per active expert
  int* tok_s = cnt_s + kMaxActive;                       // [maxa][B] b * 16 + j
  const int BE = p.B * p.E;
  const unsigned ep = step_epoch(S);
  // the logits of every router tile, polled until all carry this step's epoch (the
  // poll's loads are the data: no separate fan-in counter and reload)
  const uint64_t* src = p.rlog + (size_t)l * BE;
  const uint64_t t0 = gtime();
  unsigned ns = 32;
  for (int it = 0;; ++it) {
    bool stale = false;
    for (int i = tid; i < BE; i += kConsumerThreads) {
      const uint64_t w = ld_relaxed_u64(src + i);
      if ((unsigned)(w >> 32) != ep) {
        stale = true;
      } else {
        // a NaN logit (non-finite activations) ranks below every number, so that all
        // top_k slots are filled; the step reports MK_ERR_NAN
        const float v = __uint_as_float((unsigned)w);
        if (v != v) raise_err(p, MK_ERR_NAN, ti, -1, l, i);
        lg[i] = (v != v) ? -INFINITY : v;
      }
    }
    if (!bar_or_consumers(stale)) break;
    if (tid == 0) __nanosleep(ns);
    ns = ns < 64 ? ns * 2 : 64;
    if ((it & 7) == 7 && bar_or_consumers(tid == 0 && (aborted(p) || (long long)(gtime() - t0) > p.timeout_ns))) {
      if (tid == 0 && !aborted(p)) raise_err(p, MK_ERR_TIMEOUT, ti, -11, l, 0);
      return false;
    }
  }
  if (p.trace && tid == 0) trace_slots(S)[6] = gtime();
  const long long c_rank0 = clock64();
  float* wsel = reinterpret_cast<float*>(tok_s + kMaxActive * kMaxBatch);  // [B][topk] weights
  int* prk = reinterpret_cast<int*>(wsel + kMaxActive);                    // [2][B*E] partial ranks
  int* tot_s = prk + 256;                                                 // n_active
  const int E = p.E, K = p.topk, B = p.B;
  for (int e = tid; e < E; e += kConsumerThreads) slot_of[e] = 0;
  // rank of logit (b, e) = how many logits of token b beat it (ties to the lower id),
  // by 128-bit shared-memory reads; with few logits two threads split the range
  const int H = (2 * BE <= kConsumerThreads) ? 2 : 1;
  for (int t = tid; t < H * BE; t += kConsumerThreads) {
    const int h = t >= BE ? 1 : 0, i = t - h * BE;
    const int b = i / E, e = i - b * E;
    const float* r = lg + b * E;
    const float ve = r[e];
    const int f0 = h * (E / H), f1 = f0 + E / H;
    int r0 = 0, r1 = 0, r2 = 0, r3 = 0;  // independent counts (no serial add chain)
#pragma unroll 4
    for (int f = f0; f < f1; f += 4) {
      const float4 q = *reinterpret_cast<const float4*>(r + f);
      r0 += (q.x > ve || (q.x == ve && f < e)) ? 1 : 0;
      r1 += (q.y > ve || (q.y == ve && f + 1 < e)) ? 1 : 0;
      r2 += (q.z > ve || (q.z == ve && f + 2 < e)) ? 1 : 0;
      r3 += (q.w > ve || (q.w == ve && f + 3 < e)) ? 1 : 0;
    }
    const int rank = (r0 + r1) + (r2 + r3);
    if (H == 1) {
      if (rank < K) sel[b * K + rank] = e;
    } else {
      prk[t] = rank;
    }
  }
  trace_mark(p, S, 13);
  if (p.trace && tid == 0) trace_slots(S)[9] = (unsigned long long)(clock64() - c_rank0);
  if (H == 2) {
    bar_sync_consumers();
    for (int i = tid; i < BE; i += kConsumerThreads) {
      const int rank = prk[i] + prk[BE + i];
      if (rank < K) sel[(i / E) * K + rank] = i % E;
    }
  }
  bar_sync_consumers();
  trace_mark(p, S, 14);
  if (warp < B) {  // softmax over the selected logits of token `warp`
    const int b = warp;
    const float* r = lg + b * E;
    const int ej = (lane < K) ? sel[b * K + lane] : 0;
    const float mx = r[sel[b * K]];
    const float w = (lane < K) ? __expf(r[ej] - mx) : 0.f;
    float sum = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < K) wsel[b * K + lane] = w / sum;
  }
  trace_mark(p, S, 8);
  if (B == 1 && p.route_pf_bytes > 0 && warp >= 1) {
    // warps 1..7: the first route_pf_bytes of every item of the selected experts into
    // L2, while warp 0 publishes the route (the claimers' copies then start from L2)
    const int n = K * p.t_moe;
    for (int i = tid - 32; i < n; i += kConsumerThreads - 32) {
      const int e = sel[i / p.t_moe], t = i % p.t_moe;
      prefetch_l2(p.wblob + p.off_moe + ((long long)(l * p.E + e) * p.t_moe + t) * p.moe_item_bytes,
                  (uint32_t)p.route_pf_bytes);
    }
  }
  if (B == 1) {
    // one token: the active experts are its selection (maxa = top_k); warp 0 places
    // each in its slot (the number of selected ids below it) and writes everything
    if (warp == 0) {
      __syncwarp();
      const int maxa = p.maxa;
      const int e = lane < K ? sel[lane] : 0x7fffffff;
      int slot = 0;
      for (int j = 0; j < K; ++j) slot += __shfl_sync(0xffffffffu, e, j) < e ? 1 : 0;
      uint64_t* rw = p.rword + (size_t)l * p.rw_stride;
      if (lane < K) {
        const float w = wsel[lane];
        rw[1 + 2 * maxa + slot] = tagged(ep, (unsigned)lane);  // token 0, selection rank
        rw[1 + 2 * maxa + maxa + slot] = tagged(ep, __float_as_uint(w));
        rw[1 + slot] = tagged(ep, (unsigned)e);
        rw[1 + maxa + slot] = tagged(ep, 1u);
        p.ridx[(size_t)l * K + lane] = e;
        p.rw[(size_t)l * K + lane] = w;
        p.active[l * maxa + slot] = e;
        p.act_cnt[l * maxa + slot] = 1;
        p.act_tok[(size_t)l * maxa + slot] = lane;
      }
      if (lane == 0) {
        rw[0] = tagged(ep, (unsigned)K);
        if (p.trace) trace_slots(S)[10] = gtime();
        p.nact[l] = K;
        p.qcount[p.L + l] = K * p.t_moe;
        const unsigned pad = (unsigned)((maxa - K) * p.t_moe);
        if (pad > 0) atomicAdd(ctr_ptr(p, C_MD(p, l)), pad);
        if (p.trace) trace_slots(S)[11] = gtime();
      }
    }
    return true;
  }
  // active experts (ascending id) and per active expert its tokens in ascending b, in
  // parallel: a bitmap of the selected experts and per expert a mask of its tokens
  const int nsel = B * K;  // <= 64
  unsigned* emask = reinterpret_cast<unsigned*>(slot_of);  // [E / 32] selected experts
  unsigned* tmask = reinterpret_cast<unsigned*>(prk);      // [E] tokens per expert (ranks done)
  if (tid < 8) emask[tid] = 0u;
  for (int e = tid; e < E; e += kConsumerThreads) tmask[e] = 0u;
  bar_sync_consumers();
  if (tid < nsel) {
    const int e = sel[tid];
    atomicOr(&emask[e >> 5], 1u << (e & 31));
    atomicOr(&tmask[e], 1u << (tid / K));
  }
  bar_sync_consumers();
  if (tid < nsel) {
    const int e = sel[tid], b = tid / K;
    int slot = __popc(emask[e >> 5] & ((1u << (e & 31)) - 1u));
    for (int w = 0; w < (e >> 5); ++w) slot += __popc(emask[w]);
    const unsigned tm = tmask[e];
    tok_s[slot * B + __popc(tm & ((1u << b) - 1u))] = b * 16 + (tid % K);
    if ((tm & ((1u << b) - 1u)) == 0u) {  // the expert's first token fills its slot
      act_s[slot] = e;
      cnt_s[slot] = __popc(tm);
    }
  }
  if (tid == 0) {
    int total = 0;
    for (int w = 0; w < (E + 31) / 32; ++w) total += __popc(emask[w]);
    *tot_s = total;
  }
  bar_sync_consumers();
  trace_mark(p, S, 9);
  // route words for the expert-item claimers (each carries the epoch: no ordering needed)
  const int total = *tot_s, maxa = p.maxa;
  uint64_t* rw = p.rword + (size_t)l * p.rw_stride;
  for (int a = tid; a < total; a += kConsumerThreads) {
    const int c2 = cnt_s[a];
    for (int n = 0; n < c2; ++n) {
      const int tk = tok_s[a * B + n];
      rw[1 + 2 * maxa + a * B + n] = tagged(ep, (unsigned)tk);
      rw[1 + 2 * maxa + maxa * B + a * B + n] = tagged(ep, __float_as_uint(wsel[(tk >> 4) * K + (tk & 15)]));
    }
    rw[1 + a] = tagged(ep, (unsigned)act_s[a]);
    rw[1 + maxa + a] = tagged(ep, (unsigned)c2);
  }
  if (tid == 0) rw[0] = tagged(ep, (unsigned)total);
  if (p.trace && tid == 0) trace_slots(S)[10] = gtime();
  // the routing in plain arrays (host-side readers), and the MoE-done padding: the
  // inactive slots' share of the maxa * t_moe arrivals the ADD_RMSNORM tasks wait for
  for (int i = tid; i < nsel; i += kConsumerThreads) {
    p.ridx[(size_t)l * nsel + i] = sel[i];
    p.rw[(size_t)l * nsel + i] = wsel[i];
  }
  for (int a = tid; a < total; a += kConsumerThreads) {
    p.active[l * maxa + a] = act_s[a];
    p.act_cnt[l * maxa + a] = cnt_s[a];
    for (int n = 0; n < cnt_s[a]; ++n) p.act_tok[((size_t)l * maxa + a) * B + n] = tok_s[a * B + n];
  }
  if (tid == 0) {
    p.nact[l] = total;
    p.qcount[p.L + l] = total * p.t_moe;
    const unsigned pad = (unsigned)((maxa - total) * p.t_moe);
    if (pad > 0) atomicAdd(ctr_ptr(p, C_MD(p, l)), pad);
    if (p.trace) trace_slots(S)[11] = gtime();
  }
  return true;
}

// ADD_RMSNORM for the residual row blocks in `mask` (bit r = rows [128 r, 128 r + 128))
// of layer l, in one pass over the CTA: x_{l+1} = x_l + the layer accumulator (expert and
// O-proj outputs); the next layer's operand bf16(x_{l+1} * gain_{l+1}) as hi/lo parts (for
// the expert items and the LM head) and the blocks' per-token sums of squares.  Then
// LR(l+1) += number of blocks.  (The next layer's router and QKV tiles do not wait for
// this: they build their operand from x_l and the accumulator themselves.)
__device__ void residual_blocks(const Params& p, const Smem& S, uint32_t& sseq, int l, unsigned mask) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* rbl = S.small + 16;  // list of the blocks (<= 16)
  if (tid == 0) {
    int n = 0;
    for (int r = 0; r < p.nrb_d; ++r)
      if ((mask >> r) & 1u) rbl[n++] = r;
    rbl[16] = n;
  }
  bar_sync_consumers();
  const int nblk = rbl[16];
  const int nchunks = nblk * p.B * (kRowBlock / 32);  // warp-sized chunks of 32 rows
  float* ssp = S.scratch;                             // [nblk * B][4] partial sums
  const float* gain_next = (l + 1 < p.L) ? p.attn_norm + (size_t)(l + 1) * p.d : p.final_norm;
#pragma unroll 4
  for (int q = warp; q < nchunks; q += kConsumerWarps) {
    const int blk = q >> 2;                      // (block index, token)
    const int r = rbl[blk / p.B], b = blk % p.B;
    const int row = r * kRowBlock + (q & 3) * 32 + lane;
    const float x = ldg_cg(p.X + ((size_t)l * p.B + b) * p.d + row) + acc_ld1(p, ((size_t)l * p.B + b) * p.d + row);
    const size_t o = ((size_t)(l + 1) * p.B + b) * p.d + row;
    p.X[o] = x;
    const float xg = x * gain_next[row];
    const uint16_t hi = to_bf16(xg);
    p.XG[o] = hi;
    p.XGL[o] = to_bf16(xg - bf16_to_f(hi));
    float sq = x * x;
#pragma unroll
    for (int s2 = 16; s2 > 0; s2 >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, s2);
    if (lane == 0) ssp[q] = sq;
  }
  bar_sync_consumers();
  for (int blk = tid; blk < nblk * p.B; blk += kConsumerThreads) {
    const int r = rbl[blk / p.B], b = blk % p.B;
    const float s4 = ssp[4 * blk] + ssp[4 * blk + 1] + ssp[4 * blk + 2] + ssp[4 * blk + 3];
    p.SS[((size_t)(l + 1) * p.nrb_d + r) * kSsStride + b] = s4;
  }
  signal_async(p, S, sseq, C_LR(p, l + 1), (unsigned)nblk);
}

// Signal a fan-in counter; returns true (to all consumer threads) if this CTA was last.
__device__ bool signal_fanin(const Params& p, const Smem& S, int ci, unsigned target) {
  bar_sync_consumers();
  if (threadIdx.x == 0) {
    const unsigned old = atom_add_acq_rel(ctr_ptr(p, ci), 1u);
    S.small[1] = (old + 1 == target) ? 1 : 0;
    if (p.trace && old + 1 == target) trace_slots(S)[6] = gtime();
  }
  bar_sync_consumers();
  return S.small[1] != 0;
}
// Publish this task's output: the barrier orders every consumer thread's stores
// before thread 0's release-add at GPU scope; waiters acquire the counter.
__device__ void signal_plain(const Params& p, int ci, unsigned v) {
  bar_sync_consumers();
  if (threadIdx.x == 0) red_release(ctr_ptr(p, ci), v);
}


// ============================================================== GEMV tasks
// The B operand of consecutive tasks that read the same activation (same layer and
// source: the layer's normed input, one expert's gathered rows or gated block, one
// KV group's attention output) is built once: the later tasks skip both the
// dependency wait (already met) and the loads.
struct OperandKey {
  int kind, layer, sub;
  __device__ __forceinline__ bool operator==(const OperandKey& o) const {
    return kind == o.kind && layer == o.layer && sub == o.sub;
  }
};


// ---------------------------------------------------------------- LM head on tcgen05
// Completion of the tensor-core MMAs committed as chunk number u of this step (two
// mbarriers, alternating; every consumer thread waits).
__device__ __forceinline__ bool wait_mma(const Params& p, const Smem& S, uint32_t u) {
  if (mbar_wait(S.mmadone(u & 1u), (u >> 1) & 1u, 4 * p.timeout_ns)) return true;
  if ((threadIdx.x & 31) == 0) raise_err(p, MK_ERR_TIMEOUT, -15, -1, (int)u, 0);
  return false;
}

// A ring chunk consumed by tcgen05 MMAs: every consumer thread waits for it to land;
// thread 0 issues the MMAs (issue(stage address)) and commits them to the stage's empty
// barrier, which then completes once they have read it; warps 1-7 arrive there at once
// (their share of the release).  Nothing waits for the MMAs here.
template <class Issue>
__device__ __forceinline__ bool umma_chunk(const Params& p, const Smem& S, uint32_t seq, Issue issue) {
  const bool ok = wait_full(p, S, seq);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    if (ok) {
      tc_fence_after();
      issue(S.stage(seq));
    }
    umma_commit(S.empty(seq % kStages));
  } else if (warp > 0) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_relaxed(S.empty(seq % kStages));
  }
  return ok;
}

// Thread 0 commits every MMA issued so far to the phase-end mbarrier number u (two,
// alternating); every consumer thread waits for it.
__device__ __forceinline__ bool umma_phase_end(const Params& p, const Smem& S, uint32_t& u) {
  if (threadIdx.x == 0) umma_commit(S.mmadone(u & 1u));
  const bool ok = wait_mma(p, S, u);
  ++u;
  tc_fence_after();
  return ok;
}

// LM_HEAD tile of 64 rows on the 5th-generation tensor cores (the MK_UMMA build).  Every
// 32 KB weight chunk holds the tile's 64 rows x 256 columns in the K-major core-matrix
// layout with the second 128 columns stacked under the first as rows 64..127 (core
// matrix (kc, mg): rows 8 mg .. 8 mg + 7 of that stacking, columns 8 kc .. 8 kc + 7 of
// its half, 16 bytes a row, at (kc * 16 + mg) * 128 bytes), so that every MMA has
// M = 128: an MMA costs about the same time for any N up to 64.  The tokens' operand is
// staged once per tile from the warps' fragments into shared memory (core matrix kc of
// the K columns at kc * 128 bytes, rows beyond the batch zero) and read as N = 16 rows:
// rows 0-7 the chunk's first-half columns, rows 8-15 its second-half ones (2048 bytes
// on).  One thread issues each chunk's 8 MMAs (K = 16) into a 128 x 16 f32 accumulator
// in tensor memory as soon as the chunk lands, committing them to the stage's release;
// row m of the tile is D[m][n] + D[64 + m][8 + n].  Warps 2-3 hand the second-half sums
// to warps 0-1 through shared memory, whose lanes then hold one row each.  useq counts
// the phase-end commits of this step (the mbarriers' phases).
__device__ bool lm_umma_tile(const Params& p, const Smem& S, uint32_t& cseq, uint32_t& useq, int nch, int ksw,
                             const BFrag& fr, float rs_have, const int* T) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = lane >> 2, c = lane & 3;
  uint8_t* bsm = reinterpret_cast<uint8_t*>(S.scratch);  // [K / 8][8 rows][16 bytes]
  const uint32_t taddr = (uint32_t)S.small[5];
  constexpr uint32_t kIdesc = umma_idesc_bf16(128, 16);
  // the operand: warp w holds k16-steps ks = w + 8 j, columns 16 ks + 2 c (+1) and + 8 of
  // token n, i.e. core matrices 2 ks and 2 ks + 1, row n, bytes 4 c
#pragma unroll
  for (int j = 0; j < kMaxKsw; ++j) {
    if (j < ksw) {
      const int ks = warp + 8 * j;
      *reinterpret_cast<uint32_t*>(bsm + (2 * ks) * 128 + n * 16 + 4 * c) = fr.b0[j];
      *reinterpret_cast<uint32_t*>(bsm + (2 * ks + 1) * 128 + n * 16 + 4 * c) = fr.b1[j];
    }
  }
  fence_proxy_async_smem();
  bar_sync_consumers();
  bool ok = true;
  for (int j = 0; j < nch; ++j) {
    const uint32_t b0 = S.scratch_s + (uint32_t)j * 4096;
    ok = umma_chunk(p, S, cseq + j, [&](uint32_t a0) {
      if (j == 0) trace_mark(p, S, 2);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        umma_bf16(taddr, umma_sdesc(a0 + s * 4096, 2048, 128), umma_sdesc(b0 + s * 256, 128, 2048), kIdesc,
                  j > 0 || s > 0);
    }) && ok;
  }
  cseq += (uint32_t)nch;
  ok = umma_phase_end(p, S, useq) && ok;
  trace_mark(p, S, 3);
  // epilogue (the operand is no longer read: its first 2 KB take the second-half sums)
  float rs[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) rs[b] = __shfl_sync(0xffffffffu, rs_have, 4 * b);  // 1/rms of token b
  float* xch = S.scratch;  // [8 tokens][64 rows]
  if (warp == 2 || warp == 3) {
    float v[8];
    tmem_ld8(taddr + 8 + ((uint32_t)(32 * warp) << 16), v);
#pragma unroll
    for (int b = 0; b < 8; ++b) xch[b * 64 + 32 * (warp - 2) + lane] = v[b];
  }
  bar_sync_consumers();
  if (warp < 2) {
    float v[8];
    tmem_ld8(taddr + ((uint32_t)(32 * warp) << 16), v);
    const int r0 = T[D_ROW0] + 32 * warp + lane;
    const bool mine = r0 < p.V;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (b < p.B) {
        const float x = (v[b] + xch[b * 64 + 32 * warp + lane]) * rs[b];
        if (mine) p.logits[(size_t)b * p.V + r0] = x;
        if (p.tok_out) {
          unsigned long long best = mine ? argmax_key(x, r0) : 0ull;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
            best = y > best ? y : best;
          }
          if (lane == 0) atomicMax(p.amax + (size_t)(blockIdx.x % kAmaxReplicas) * p.B + b, best);
        }
      }
    }
  }
  tc_fence_before();  // (the next tile's MMAs overwrite the accumulator after the caller's barrier)
  return ok;
}

__device__ __forceinline__ bool task_gemv(const Params& p, const Smem& S, uint32_t& cseq, uint32_t& sseq,
                                          uint32_t& useq, const int* T, int ti, int nch, BFrag& fr,
                                          OperandKey& have, float& rs_have) {
  const int op = T[D_OP];
  const int l = T[D_LAYER];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g8 = lane >> 2, c = lane & 3;

  const int nrows = T[D_NROWS];
  const int klen = T[D_KLEN];
  OperandKey key;
  switch (op) {
    case OP_OPROJ: key = {5, l, T[D_AUX]}; break;
    case OP_LMHEAD: key = {2, p.L, 0}; break;
    default: key = {1, l, 0}; break;  // QKV and ROUTER share the layer's normed input
  }
  const bool reuse = key == have;
  // The QKV epilogue's inputs that do not depend on the wait -- this lane's RoPE rate
  // and, for K/V rows, the page of each token's new slot -- are loaded first, so that
  // their L2 round trips overlap the wait and the GEMV instead of following them.
  unsigned long long fturn = 0ull;
  int kv_pg[2] = {-1, -1};
  // FP8 projections: this lane's two epilogue rows' scales (x 256: the integer-pipe
  // decode yields the codes' values x 2^-8), loaded before the wait as well
  const bool f8 = p.fp8d && op != OP_ROUTER;
  float rsc0 = 1.f, rsc1 = 1.f;
  if (f8 && warp < nrows / 16) {
    const int r0 = T[D_ROW0] + warp * 16 + g8;
    const float* sp = op == OP_QKV ? p.qkv_scale + ((size_t)l * p.Hkv + T[D_AUX]) * p.qkv_rows_group
                    : op == OP_OPROJ ? p.o_scale + (size_t)l * p.d
                                     : p.lm_scale;
    rsc0 = __ldg(sp + r0) * 256.f;
    rsc1 = __ldg(sp + r0 + 8) * 256.f;
  }
  if (op == OP_QKV && warp < nrows / 16) {
    const int pr = T[D_ROW0] + warp * 16 + g8;
    const int seg = pr / p.hd, j = pr % p.hd;
    if (seg <= p.gs) fturn = __ldg(p.rope_turns + 8 * (j / 16) + g8);
    if (seg >= p.gs)
      for (int e = 0; e < 2; ++e) {
        const int n = 2 * c + e;
        if (n < p.B) kv_pg[e] = checked_page(p, n, seq_lens_s(S)[n] / 16, ti);
      }
  }
  if (reuse) {
    trace_mark(p, S, 1);
  } else if (!consumer_wait(p, S, T[D_WAIT_CTR], (unsigned)T[D_WAIT_TARGET], ti, T[D_WAIT2_CTR],
                            (unsigned)T[D_WAIT2_TARGET])) {
    drain_chunks(p, S, cseq, nch);
    return false;
  }
  // QKV and router tiles of layers >= 1 build their operand from the previous layer's
  // residual stream and accumulator (they wait for the layer's experts and O-proj, not
  // for its ADD_RMSNORM step)
  const bool from_parts = (op == OP_QKV || op == OP_ROUTER) && l >= 1;
  const int nrb = nrows / 16;
  const int ksw = klen / 16 / kConsumerWarps;

  float v[4];
  bool ran;
  if (op == OP_ROUTER) {
    // the router's operand is hi + lo bf16 parts (hi is shared with the layer's QKV
    // tiles; the residue lo is loaded for the router only)
    const int n = lane >> 2;
    BFrag lo;
    if (from_parts) {
      // the hi part is rebuilt as well (it is the shared QKV operand)
      rs_have = build_operand_parts(p, S, fr, &lo, ksw, l);
    } else {
      // issued first: its loads share the round trip of the hi part and 1/rms
      load_bfrag(lo, ksw, n < p.B ? p.XGL + ((size_t)l * p.B + n) * p.d : nullptr);
      if (!reuse) rs_have = build_norm_bfrag(p, S, fr, ksw, l, n < p.B ? n : -1);
    }
    have = key;
    ran = (nrb == 1) ? gemv_run<1>(p, S, cseq, nch, ksw, fr, v, &lo) : gemv_run<2>(p, S, cseq, nch, ksw, fr, v, &lo);
  } else {
    if (!reuse) {
      const int n = lane >> 2;
      if (op == OP_OPROJ) {
        load_bfrag(fr, ksw, n < p.B ? p.atto + ((size_t)l * p.B + n) * p.Hq * p.hd + T[D_K0] : nullptr);
      } else if (from_parts) {
        rs_have = build_operand_parts(p, S, fr, nullptr, ksw, l);
      } else {
        // RMSNorm operand of QKV (layer input) and LM_HEAD (final norm)
        rs_have = build_norm_bfrag(p, S, fr, ksw, op == OP_LMHEAD ? p.L : l, n < p.B ? n : -1);
      }
    }
    have = key;
    if (MK_UMMA && op == OP_LMHEAD) {
      const bool done = lm_umma_tile(p, S, cseq, useq, nch, ksw, fr, rs_have, T);
      trace_mark(p, S, 12);
      bar_sync_consumers();
      return done;
    }
    if (f8) {
      switch (nrb) {
        case 1: ran = gemv_run8<1, true>(p, S, cseq, nch, ksw, fr, v); break;
        case 2: ran = gemv_run8<2, true>(p, S, cseq, nch, ksw, fr, v); break;
        case 4: ran = gemv_run8<4, true>(p, S, cseq, nch, ksw, fr, v); break;
        default: ran = gemv_run8<8, true>(p, S, cseq, nch, ksw, fr, v); break;
      }
      v[0] *= rsc0; v[1] *= rsc0;   // row 16w + g8, tokens 2c, 2c + 1
      v[2] *= rsc1; v[3] *= rsc1;   // row 16w + g8 + 8
    } else {
      switch (nrb) {
        case 1: ran = gemv_run<1>(p, S, cseq, nch, ksw, fr, v); break;
        case 2: ran = gemv_run<2>(p, S, cseq, nch, ksw, fr, v); break;
        case 4: ran = gemv_run<4>(p, S, cseq, nch, ksw, fr, v); break;
        default: ran = gemv_run<8>(p, S, cseq, nch, ksw, fr, v); break;
      }
    }
  }
  if (!ran) return false;

  // ---- epilogue: thread (warp = row block, lane) owns rows 16w+g8, 16w+g8+8, tokens 2c, 2c+1
  if (op == OP_QKV || op == OP_ROUTER || op == OP_LMHEAD) {
    // 1/rms of tokens 2c and 2c+1 lives in lanes 8c and 8c+4 (operand row n = lane/4)
    const float rs0 = __shfl_sync(0xffffffffu, rs_have, 8 * c);
    const float rs1 = __shfl_sync(0xffffffffu, rs_have, 8 * c + 4);
    v[0] *= rs0; v[2] *= rs0;
    v[1] *= rs1; v[3] *= rs1;
  }
  if (warp < nrb) {
    const int rlo = warp * 16 + g8;  // row within the task tile (row 'rlo + 8' is the pair)
    switch (op) {
      case OP_QKV: {
        const int g = T[D_AUX];
        const int pr = T[D_ROW0] + rlo;  // packed row inside the group's [q heads | k | v]
        const int seg = pr / p.hd;
        const int j = pr % p.hd;
        const int d1 = 8 * (j / 16) + g8, d2 = d1 + p.hd / 2;
        const bool rot = seg <= p.gs;
        // angle = pos * inv_freq[d1]; turns = frac(pos * inv_freq / 2pi) computed exactly
        // in 64-bit fixed point (fturn = rope_turns[d1] = inv_freq / 2pi * 2^64, loaded
        // before the wait), then sin/cos of 2*pi*turns in fp32.
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          if (n >= p.B) continue;
          const float x1 = v[e], x2 = v[2 + e];
          const int pos = seq_lens_s(S)[n];
          float y1 = x1, y2 = x2;
          if (rot) {
            const unsigned long long u = (unsigned long long)(unsigned)pos * fturn;
            const float t = (float)(u >> 40) * 5.9604644775390625e-08f;  // 2^-24
            float fs, fc;
            sincospif(2.f * t, &fs, &fc);
            y1 = x1 * fc - x2 * fs;
            y2 = x2 * fc + x1 * fs;
          }
          if (seg < p.gs) {
            uint16_t* q = p.Q + ((size_t)l * p.B + n) * p.Hq * p.hd + (size_t)(p.gs * g + seg) * p.hd;
            q[d1] = to_bf16(y1);
            q[d2] = to_bf16(y2);
          } else {
            const int pg = kv_pg[e];  // (checked before the wait)
            if (pg >= 0) {
              uint16_t* dst = (seg == p.gs ? p.kc : p.vc) +
                              ((((size_t)l * p.n_pages + pg) * p.Hkv + g) * 16 + (pos % 16)) * p.hd;
              dst[d1] = to_bf16(y1);
              dst[d2] = to_bf16(y2);
            }
          }
        }
        break;
      }
      case OP_ROUTER: {
        const int r0 = T[D_ROW0] + rlo;
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          if (n >= p.B) continue;
          uint64_t* out = p.rlog + ((size_t)l * p.B + n) * p.E;
          const unsigned ep = step_epoch(S);
          if (r0 < p.E) out[r0] = tagged(ep, __float_as_uint(v[e]));
          if (r0 + 8 < p.E) out[r0 + 8] = tagged(ep, __float_as_uint(v[2 + e]));
        }
        break;
      }
      case OP_OPROJ: {  // added into the layer accumulator (with the expert outputs)
        const int r0 = T[D_ROW0] + rlo;
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          if (n >= p.B) continue;
          const size_t out = ((size_t)l * p.B + n) * p.d;
          acc_add1(p, out + r0, v[e]);
          acc_add1(p, out + r0 + 8, v[2 + e]);
        }
        break;
      }
      case OP_LMHEAD: {
        const int r0 = T[D_ROW0] + rlo;
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          if (n >= p.B) continue;
          float* out = p.logits + (size_t)n * p.V;
          if (r0 < p.V) out[r0] = v[e];
          if (r0 + 8 < p.V) out[r0 + 8] = v[2 + e];
        }
        if (p.tok_out) {
          // greedy token: the tile's best (value, lowest row) per token over the 8 lanes
          // of a row group, then one max into this SM's replica of the step's key
          unsigned long long best[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const unsigned long long k0 = r0 < p.V ? argmax_key(v[e], r0) : 0ull;
            const unsigned long long k1 = r0 + 8 < p.V ? argmax_key(v[2 + e], r0 + 8) : 0ull;
            best[e] = k0 > k1 ? k0 : k1;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
              const unsigned long long x = __shfl_xor_sync(0xffffffffu, best[e], o);
              best[e] = x > best[e] ? x : best[e];
            }
          }
          if (g8 == 0)
            for (int e = 0; e < 2; ++e)
              if (2 * c + e < p.B)
                atomicMax(p.amax + (size_t)(blockIdx.x % kAmaxReplicas) * p.B + 2 * c + e, best[e]);
        }
        break;
      }
      default:
        break;
    }
  }

  trace_mark(p, S, 12);
  // ---- signal
  switch (op) {
    case OP_QKV:
    case OP_OPROJ:
      signal_async(p, S, sseq, T[D_SIG_CTR], 1u);
      trace_mark(p, S, 13);
      break;
    case OP_ROUTER:
      // no fan-in: the layer's last router tile (D_AUX = 1) collects every tile's
      // tagged logits itself and runs the route step.  The router-tiles and route-ready
      // counters are counted for the bookkeeping only (no task waits on them: the
      // tagged logits and route words carry the readiness themselves).
      if (T[D_AUX] == 1) {
        if (p.B == 1 && p.route_warp) {
          if (warp == 0) route_step_b1(p, S, l, ti);
        } else if (!route_step(p, S, l, ti)) {
          return false;
        }
        signal_async(p, S, sseq, C_RR(p, l), 1u);
      }
      signal_async(p, S, sseq, T[D_SIG_CTR], 1u);
      break;
    default:
      break;
  }
  bar_sync_consumers();
  return true;
}

// ADD_RMSNORM task of residual row block r: waits for all MoE items of the layer and
// the block's O-proj tiles.
__device__ bool task_resid(const Params& p, const Smem& S, uint32_t& sseq, const int* T, int ti) {
  const int l = T[D_LAYER], r = T[D_AUX];
  if (!consumer_wait(p, S, T[D_WAIT2_CTR], (unsigned)T[D_WAIT2_TARGET], ti)) return false;
  if (!consumer_wait(p, S, T[D_WAIT_CTR], (unsigned)T[D_WAIT_TARGET], ti)) return false;
  residual_blocks(p, S, sseq, l, 1u << r);
  bar_sync_consumers();
  return true;
}

// One MoE item: expert slot a = item / t_moe, f-slice s = item % t_moe.
//   phase 1: [gate; up] rows of the slice times the expert's gathered normed tokens
//            -> a = silu(gate) * up for 32 f-rows x n_tok, bf16 in shared memory;
//   phase 2: W_down[:, slice] * a -> per-token partial of the expert output, times the
//            token's routing weight, added into the layer's MoE accumulator.
// Completion is counted on the layer's MoE-done counter (padded to max_active * t_moe
// by the route step).
// F8: the expert's weights are E4M3 codes (FP8 experts): the item's first chunk holds
// its f32 row scales (copied to shared memory), the operand and the SiLU product are
// f16, and each GEMV output is scaled by its row's scale.
template <int FS, bool F8 = false>
__device__ __forceinline__ bool task_moe(const Params& p, const Smem& S, uint32_t& cseq, uint32_t& sseq, int l,
                                         bool dense, int ti, int item, int nch, int ntok, int tok_lo, int tok_hi,
                                         int4 w_lo, int4 w_hi, BFrag& fr, OperandKey& have, float& rs_have) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g8 = lane >> 2, c = lane & 3;
  const int a_slot = dense ? 0 : item / p.t_moe;  // a dense layer: one token set
  const OperandKey key = {3, l, a_slot};
  // The producer claimed this item from the layer's route words and passed the
  // expert's token list and weights in the mailbox entry: no dependency wait here.
  const bool reuse = key == have;
  trace_mark(p, S, 1);
  auto tok_byte = [&](int n) { return ((n < 4 ? tok_lo : tok_hi) >> (8 * (n & 3))) & 0xff; };
  // this lane's two epilogue tokens (2c, 2c+1): batch index and routing weight (both
  // from the mailbox entry)
  const int wbits[8] = {w_lo.x, w_lo.y, w_lo.z, w_lo.w, w_hi.x, w_hi.y, w_hi.z, w_hi.w};
  int bt[2];
  float wt[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int n = 2 * c + e;
    int wb = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) wb = (k == n) ? wbits[k] : wb;
    bt[e] = (n < ntok) ? (tok_byte(n) >> 3) : -1;
    wt[e] = (n < ntok) ? __int_as_float(wb) : 0.f;
  }
  const int ksw1 = p.d / 128;
  if (!reuse) {
    const int n = lane >> 2;
    rs_have = build_norm_bfrag(p, S, fr, ksw1, l, (n < ntok) ? (tok_byte(n) >> 3) : -1);
    if (F8) {  // the operand in f16 (kept so for the next items of this token set)
#pragma unroll
      for (int j = 0; j < kMaxKsw; ++j) {
        fr.b0[j] = bf16x2_to_f16x2(fr.b0[j]);
        fr.b1[j] = bf16x2_to_f16x2(fr.b1[j]);
      }
    }
    have = key;
  }
  // FP8: the scales chunk -> shared memory [2*fs gate/up rows][d down rows] (f32)
  // scratch: [0, 17408) phase-2 staging / [0, 16384) phase-1 reduction; [18432, ...) the
  // scales; [28672, ...) the SwiGLU activations
  static_assert(kConsumerWarps * kMaxBatch * 68 * 4 <= 18432 && 18432 + (2 * 64 + 2048) * 4 <= 28672 &&
                    28672 + kMaxBatch * 64 * 2 <= kScratchBytes,
                "MoE item scratch layout");
  const float* scl = reinterpret_cast<const float*>(reinterpret_cast<uint8_t*>(S.scratch) + 18432);
  if (F8) {
    if (!wait_full(p, S, cseq)) return false;
    const int n16 = fp8_scale_bytes(FS, p.d) / 16;
    const uint4* src = reinterpret_cast<const uint4*>(S.ring_g + (cseq % kStages) * kStageBytes);
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(S.scratch) + 18432);
    for (int i = threadIdx.x; i < n16; i += kConsumerThreads) dst[i] = src[i];
    release_stage(S, cseq);
    ++cseq;
    bar_sync_consumers();
  }
  // ---- phase 1: 2*FS interleaved gate/up rows = FS/8 row blocks
  constexpr int fs = FS, nrb1 = FS / 8;
  const int jpc1 = F8 ? gemv_jpc8(nrb1) : gemv_jpc(nrb1);
  const int nch1 = (ksw1 + jpc1 - 1) / jpc1;
  float v[4];
  if (F8) {
    if (!gemv_run8<nrb1>(p, S, cseq, nch1, ksw1, fr, v)) return false;
  } else {
    if (!gemv_run<nrb1>(p, S, cseq, nch1, ksw1, fr, v)) return false;
  }
  trace_mark(p, S, 12);
  uint16_t* a_s = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(S.scratch) + 28672);  // [8][fs]
  {
    const float rs0 = __shfl_sync(0xffffffffu, rs_have, 8 * c);
    const float rs1 = __shfl_sync(0xffffffffu, rs_have, 8 * c + 4);
    if (warp < nrb1) {  // row block w = gate rows 8w..8w+7 (row g8) paired with up rows (g8 + 8)
      const int frow = warp * 8 + g8;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int n = 2 * c + e;
        const float rs = e ? rs1 : rs0;
        // FP8: packed row 16w + g8 is gate row 8w + g8, row 16w + 8 + g8 its up row
        // (x 256: the integer-pipe decode yields the codes' values x 2^-8)
        const float sg = F8 ? scl[warp * 16 + g8] * 256.f : 1.f, su = F8 ? scl[warp * 16 + 8 + g8] * 256.f : 1.f;
        const float gt = v[e] * rs * sg, up = v[2 + e] * rs * su;
        const float a = (n < ntok) ? gt / (1.f + __expf(-gt)) * up : 0.f;
        // (FP8: fp16 range; a SwiGLU output beyond it saturates instead of becoming inf)
        a_s[n * fs + frow] = F8 ? __half_as_ushort(__float2half_rn(fminf(fmaxf(a, -65504.f), 65504.f))) : to_bf16(a);
      }
    }
  }
  bar_sync_consumers();
  trace_mark(p, S, 13);
  // ---- phase 2: warp w owns output rows [w * rpw * 16, (w + 1) * rpw * 16), K = fs
  constexpr int k2 = FS / 16;
  uint32_t b2[k2][2];
#pragma unroll
  for (int ks = 0; ks < k2; ++ks) {
    b2[ks][0] = *reinterpret_cast<const uint32_t*>(a_s + g8 * fs + 16 * ks + 2 * c);
    b2[ks][1] = *reinterpret_cast<const uint32_t*>(a_s + g8 * fs + 16 * ks + 8 + 2 * c);
  }
  // The down slice is packed row-block-major (fragment (rb, ks) at (rb * k2 + ks) * 512 B),
  // so every ring chunk holds rbc consecutive row blocks; all 8 warps share each chunk,
  // rbw = rbc / 8 row blocks apiece, with independent accumulators for 4 at a time.
  // The weighted outputs of those (up to 64 rows) are staged per warp as [token slot]
  // [64 rows] (stride 68 floats: conflict-free stores) and added into the accumulator
  // with 128-bit reductions, 16 lanes x 4 rows per token.
  const int rpw = p.d / 128;
  const int rbc = moe_warps_per_chunk(rpw * k2 * (F8 ? kFragBytes8 : kFragBytes)) * rpw;
  const int rbw = rbc / kConsumerWarps;
  const int nch2 = nch - nch1 - (F8 ? 1 : 0);
  const float* sd = scl + 2 * fs;  // FP8: down-row scales of this slice
  constexpr int kStg = 68;
  float* stg = S.scratch + warp * (kMaxBatch * kStg);
  const int fq = (lane & 15) * 4;  // flush: this lane's 4 rows
  for (int ch = 0; ch < nch2; ++ch) {
    if (!wait_full(p, S, cseq)) return false;
    if (ch == 0) trace_mark(p, S, 8);
    if (ch == nch2 - 1) trace_mark(p, S, 10);
    const uint32_t base = S.stage(cseq) + lane * (F8 ? 8 : 16);
    for (int i0 = 0; i0 < rbw; i0 += 4) {
      float acc[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
        if (i0 + u < rbw) {
          const int rbl = warp * rbw + i0 + u;
#pragma unroll
          for (int ks = 0; ks < k2; ++ks) {
            if (F8) {
              const uint2 a = lds64(base + (rbl * k2 + ks) * kFragBytes8);
              fp8_mma(acc[u], a, b2[ks][0], b2[ks][1]);
            } else {
              const uint4 a = lds128(base + (rbl * k2 + ks) * kFragBytes);
              mma_bf16(acc[u], a.x, a.y, a.z, a.w, b2[ks][0], b2[ks][1]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int rl = u * 16 + g8;
        float s0 = 1.f, s1 = 1.f;
        if (F8) {  // this slice's scales of output rows rg and rg + 8
          const int rg = (ch * rbc + warp * rbw + i0 + u) * 16 + g8;
          s0 = (i0 + u < rbw) ? sd[rg] * 256.f : 0.f;  // (x 256: see phase 1)
          s1 = (i0 + u < rbw) ? sd[rg + 8] * 256.f : 0.f;
        }
        stg[(2 * c) * kStg + rl] = wt[0] * s0 * acc[u][0];
        stg[(2 * c) * kStg + rl + 8] = wt[0] * s1 * acc[u][2];
        stg[(2 * c + 1) * kStg + rl] = wt[1] * s0 * acc[u][1];
        stg[(2 * c + 1) * kStg + rl + 8] = wt[1] * s1 * acc[u][3];
      }
      __syncwarp();
      const int nrow = min(4, rbw - i0) * 16;
      const int row0 = (ch * rbc + warp * rbw + i0) * 16;
      for (int n0 = 0; n0 < ntok; n0 += 2) {
        const int n = n0 + (lane >> 4);
        // batch index of token slot n: held as bt[n & 1] by lane n / 2
        const int x0 = __shfl_sync(0xffffffffu, bt[0], (n >> 1) & 3);
        const int x1 = __shfl_sync(0xffffffffu, bt[1], (n >> 1) & 3);
        const int b = (n & 1) ? x1 : x0;
        if (n < ntok && fq < nrow)
          acc_add4(p, ((size_t)l * p.B + b) * p.d + row0 + fq, *reinterpret_cast<const float4*>(stg + n * kStg + fq));
      }
      __syncwarp();
    }
    if (ch == 0) trace_mark(p, S, 9);
    release_stage(S, cseq);
    ++cseq;
  }
  trace_mark(p, S, 3);
  // ---- signal the layer's MoE-done counter (waited on by the ADD_RMSNORM tasks)
  signal_async(p, S, sseq, C_MD(p, l), 1u);
  trace_mark(p, S, 14);
  bar_sync_consumers();
  trace_mark(p, S, 15);
  return true;
}

// One MoE item (bf16, 32-row f-slice) on the 5th-generation tensor cores (the MK_UMMA = 2
// build, with items packed by mk_pack_moe_umma_kernel).  An MMA costs about the same
// time for any N up to 64, so every MMA here has M = 128 (twice the weight bytes of
// M = 64 per instruction).  Phase 1: each 32 KB gate/up chunk holds 64 packed rows x 256
// columns with the second 128 columns stacked under the first as rows 64..127; the
// operand (N = 16) pairs them block-diagonally -- rows 0-7 the tokens' first-half
// columns, rows 8-15 their second-half columns -- so that 8 MMAs a chunk accumulate
// D[m][n] (first half, m < 64, n < 8) and D[64 + m][8 + n] (second half) into tensor
// memory columns 256..271 as soon as the chunk lands.  SwiGLU: warps 2-3 hand the
// second-half sums to warps 0-1 through shared memory; lane l of warp w holds packed row
// 32 w + l (gate rows at l % 16 < 8, their up rows 8 lanes above) and writes
// silu(gate) * up (bf16) as the phase-2 operand (K = 32; rows 8-15 zero).  Phase 2:
// every 128-row block of the down slice (8 KB; a chunk holds several) gets 2 MMAs into
// its own 128 x 16 accumulator (block j: columns 16 j; columns 8-15 unused).  Epilogue:
// warp w reads quadrant w % 4 of the blocks j = w / 4 mod 2, scales by the tokens'
// routing weights and adds them into the layer accumulator with 128-bit reductions.
// Stages go back to the producer once the MMAs that read them completed.
__device__ bool task_moe_umma(const Params& p, const Smem& S, uint32_t& cseq, uint32_t& sseq, uint32_t& useq, int l,
                              bool dense, int item, int nch, int ntok, int tok_lo, int tok_hi, int4 w_lo, int4 w_hi,
                              BFrag& fr, OperandKey& have, float& rs_have) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n8 = lane >> 2, c = lane & 3;
  const int a_slot = dense ? 0 : item / p.t_moe;
  const OperandKey key = {3, l, a_slot};
  trace_mark(p, S, 1);
  auto tok_byte = [&](int n) { return ((n < 4 ? tok_lo : tok_hi) >> (8 * (n & 3))) & 0xff; };
  const int ksw1 = p.d / 128;
  if (!(key == have)) {
    rs_have = build_norm_bfrag(p, S, fr, ksw1, l, (n8 < ntok) ? (tok_byte(n8) >> 3) : -1);
    have = key;
  }
  uint8_t* sm = reinterpret_cast<uint8_t*>(S.scratch);
  const uint32_t taddr = (uint32_t)S.small[5];
  constexpr uint32_t kIdesc = umma_idesc_bf16(128, 16);
  // ---- phase 1 operand: warp w's k16-steps ks = w + 8 j -> core matrices 2 ks, 2 ks + 1
  //      (core kc of the K columns at kc * 128 bytes, 8 token rows of 16 bytes)
#pragma unroll
  for (int j = 0; j < kMaxKsw; ++j) {
    if (j < ksw1) {
      const int ks = warp + 8 * j;
      *reinterpret_cast<uint32_t*>(sm + (2 * ks) * 128 + n8 * 16 + 4 * c) = fr.b0[j];
      *reinterpret_cast<uint32_t*>(sm + (2 * ks + 1) * 128 + n8 * 16 + 4 * c) = fr.b1[j];
    }
  }
  fence_proxy_async_smem();
  bar_sync_consumers();
  bool ok = true;
  const int nch1 = p.d / 256;
  for (int j = 0; j < nch1; ++j) {
    // k-step s: weight cores (kc, mg) at s * 4096 (K-adjacent 2048 apart, row groups 128);
    // operand: first-half cores 32 j + 2 s (+1), second-half ones 16 cores (2048 B) on
    const uint32_t b0 = S.scratch_s + (uint32_t)j * 4096;
    ok = umma_chunk(p, S, cseq + j, [&](uint32_t a0) {
      if (j == 0) trace_mark(p, S, 2);
      if (j == nch1 - 1) trace_mark(p, S, 11);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        umma_bf16(taddr + 256, umma_sdesc(a0 + k * 4096, 2048, 128), umma_sdesc(b0 + k * 256, 128, 2048), kIdesc,
                  j > 0 || k > 0);
    }) && ok;
  }
  cseq += (uint32_t)nch1;
  ok = umma_phase_end(p, S, useq) && ok;
  trace_mark(p, S, 12);
  // ---- SwiGLU into the phase-2 operand: element (token n, f) at (f / 8) * 128 + n * 16 +
  //      (f % 8) * 2; rows 8-15 (512 bytes on) zero
  float rs[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) rs[b] = __shfl_sync(0xffffffffu, rs_have, 4 * b);  // 1/rms of token slot b
  float* xch = reinterpret_cast<float*>(sm + 4096);  // [8 tokens][64 rows]: second-half sums
  if (warp == 2 || warp == 3) {
    float v[8];
    tmem_ld8(taddr + 256 + 8 + ((uint32_t)(32 * warp) << 16), v);
#pragma unroll
    for (int n = 0; n < 8; ++n) xch[n * 64 + 32 * (warp - 2) + lane] = v[n];
  } else if (warp == 4) {
    for (int i = lane; i < 128; i += 32) reinterpret_cast<uint32_t*>(sm + 512)[i] = 0u;
  }
  bar_sync_consumers();
  if (warp < 2) {
    float v[8];
    tmem_ld8(taddr + 256 + ((uint32_t)(32 * warp) << 16), v);
    const int f = 16 * warp + 8 * (lane >> 4) + (lane & 7);  // gate row of this lane's pair
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float x = v[n] + xch[n * 64 + 32 * warp + lane];
      const float upv = __shfl_down_sync(0xffffffffu, x, 8);
      if ((lane & 8) == 0) {
        const float gt = x * rs[n], upr = upv * rs[n];
        const float a = (n < ntok) ? gt / (1.f + __expf(-gt)) * upr : 0.f;
        *reinterpret_cast<uint16_t*>(sm + (f >> 3) * 128 + n * 16 + (f & 7) * 2) = to_bf16(a);
      }
    }
  }
  tc_fence_before();
  fence_proxy_async_smem();
  bar_sync_consumers();
  trace_mark(p, S, 13);
  // ---- phase 2: 128-row blocks of the down slice, each into its own accumulator
  const int region = (p.d / 128) * 2 * kFragBytes;
  const int bpc = moe_warps_per_chunk(region) * region / 8192;  // blocks a chunk
  const int nblk = p.d / 128;
  const int nch2 = nch - nch1;
  for (int j = 0; j < nch2; ++j) {
    ok = umma_chunk(p, S, cseq + j, [&](uint32_t a0) {
      if (j == 0) trace_mark(p, S, 8);
      if (j == nch2 - 1) trace_mark(p, S, 10);
      for (int bb = 0; bb < bpc; ++bb) {
        const int blk = j * bpc + bb;
        if (blk < nblk) {
#pragma unroll
          for (int k = 0; k < 2; ++k)
            umma_bf16(taddr + 16 * blk, umma_sdesc(a0 + bb * 8192 + k * 4096, 2048, 128),
                      umma_sdesc(S.scratch_s + k * 256, 128, 512), kIdesc, k > 0);
        }
      }
    }) && ok;
  }
  cseq += (uint32_t)nch2;
  ok = umma_phase_end(p, S, useq) && ok;
  trace_mark(p, S, 9);
  // ---- epilogue: weighted block outputs into the layer accumulator
  const int wbits[8] = {w_lo.x, w_lo.y, w_lo.z, w_lo.w, w_hi.x, w_hi.y, w_hi.z, w_hi.w};
  constexpr int kStg = 36;                                              // row stride of a token
  float* stg = reinterpret_cast<float*>(sm + 4096) + warp * 8 * kStg;  // [8 tokens][32 rows]
  const int q = warp & 3;
  const int r4 = (lane & 7) * 4;  // flush: 4 rows of tokens lane / 8 and lane / 8 + 4
  float wn[2];
  int bn[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int nt = (lane >> 3) + 4 * h;
    int wb = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) wb = (k == nt) ? wbits[k] : wb;
    wn[h] = nt < ntok ? __int_as_float(wb) : 0.f;
    bn[h] = nt < ntok ? (tok_byte(nt) >> 3) : 0;
  }
  for (int b4 = warp >> 2; b4 < nblk; b4 += 8) {
    uint32_t v[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (b4 + 2 * i < nblk) tmem_ld8_async(taddr + 16 * (b4 + 2 * i) + ((uint32_t)(32 * q) << 16), v[i]);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int blk = b4 + 2 * i;
      if (blk < nblk) {
#pragma unroll
        for (int n = 0; n < 8; ++n) stg[n * kStg + lane] = __uint_as_float(v[i][n]);
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int nt = (lane >> 3) + 4 * h;
          if (nt < ntok) {
            const float4 x = *reinterpret_cast<const float4*>(stg + nt * kStg + r4);
            acc_add4(p, ((size_t)l * p.B + bn[h]) * p.d + 128 * blk + 32 * q + r4,
                     make_float4(wn[h] * x.x, wn[h] * x.y, wn[h] * x.z, wn[h] * x.w));
          }
        }
        __syncwarp();
      }
    }
  }
  tc_fence_before();
  trace_mark(p, S, 3);
  signal_async(p, S, sseq, C_MD(p, l), 1u);
  trace_mark(p, S, 14);
  bar_sync_consumers();
  trace_mark(p, S, 15);
  return ok;
}

// ============================================================== attention
// Address of the 16-byte chunk `ch` (8 dims) of key row `key` inside a page of the
// stage, as the tensor-map copy lays it out: 16 keys x hd dims, row-major, cut into
// lines of min(hd, 64) dims (two lines a key at hd = 128), with the 128-byte swizzle
// (hd >= 64: chunk ^= line % 8) or the 64-byte one (hd = 32: chunk ^= (line / 2) % 4).
template <int HD>
__device__ __forceinline__ uint32_t kv_addr(uint32_t page_base, int key, int ch) {
  constexpr int kLineB = (HD < 64 ? HD : 64) * 2;
  constexpr int kCpl = kLineB / 16;
  const int line = key * (HD * 2 / kLineB) + ch / kCpl;
  const int swz = (kLineB == 128) ? (line & 7) : ((line >> 1) & 3);
  return page_base + line * kLineB + (((ch % kCpl) ^ swz) << 4);
}

template <int HD>
__device__ bool attention_split(const Params& p, const Smem& S, uint32_t& cseq, int l, const AttItem& it) {
  constexpr int KS = HD / 16;
  constexpr int NT = HD / 8;
  constexpr int kPageB = 16 * HD * 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g8 = lane >> 2, c = lane & 3;
  const int gs = p.gs;
  // Q A-fragments: rows = the group's query heads (rows >= gs are zero)
  uint32_t qa[KS][2];
  {
    const uint16_t* q = p.Q + ((size_t)l * p.B + it.b) * p.Hq * HD + (size_t)gs * it.g * HD;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = qa[ks][1] = 0u;
      ldg_cg_pred(qa[ks][0], q + g8 * HD + 16 * ks + 2 * c, g8 < gs);
      ldg_cg_pred(qa[ks][1], q + g8 * HD + 16 * ks + 8 + 2 * c, g8 < gs);
    }
  }
  float m_run = -INFINITY, l_run = 0.f;
  float oacc[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) oacc[t][0] = oacc[t][1] = 0.f;
  trace_mark(p, S, 11);  // (the Q loads are issued, not necessarily complete)

  for (int c0 = 0; c0 < it.np; c0 += 8) {
    const int n = min(8, it.np - c0);
    const bool have = warp < n;
    if (!wait_full(p, S, cseq)) return false;
    if (c0 == 0) trace_mark(p, S, 2);
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (have) {
      const uint32_t pbase = S.stage(cseq) + warp * kPageB;
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(kv_addr<HD>(pbase, (mi >> 1) * 8 + rr, 2 * ks + (mi & 1)), r0, r1, r2, r3);
        mma_bf16(sc[0], qa[ks][0], 0u, qa[ks][1], 0u, r0, r1);
        mma_bf16(sc[1], qa[ks][0], 0u, qa[ks][1], 0u, r2, r3);
      }
    }
    release_stage(S, cseq);  // the K page is in registers: its stage goes back now
    if (!wait_full(p, S, cseq + 1)) return false;
    if (have) {
      const int kbase = (it.pg0 + c0 + warp) * 16;
      float pr[2][2];
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kp = kbase + nt * 8 + 2 * c + e;
          const float s = (kp >= it.klo && kp < it.khi) ? sc[nt][e] * p.scale_log2 : -INFINITY;
          pr[nt][e] = s;
          mx = fmaxf(mx, s);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float corr = exp2f(m_run - m_use);
      float psum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) { pr[nt][e] = exp2f(pr[nt][e] - m_use); psum += pr[nt][e]; }
      l_run = l_run * corr + psum;
      m_run = m_new;
#pragma unroll
      for (int t = 0; t < NT; ++t) { oacc[t][0] *= corr; oacc[t][1] *= corr; }
      const uint32_t a0 = pack_bf16(pr[0][0], pr[0][1]);
      const uint32_t a2 = pack_bf16(pr[1][0], pr[1][1]);
      const uint32_t vbase = S.stage(cseq + 1) + warp * kPageB;
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int t2 = 0; t2 < NT / 2; ++t2) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(kv_addr<HD>(vbase, (mi & 1) * 8 + rr, 2 * t2 + (mi >> 1)), r0, r1, r2, r3);
        float d0[4] = {oacc[2 * t2][0], oacc[2 * t2][1], 0.f, 0.f};
        float d1[4] = {oacc[2 * t2 + 1][0], oacc[2 * t2 + 1][1], 0.f, 0.f};
        mma_bf16(d0, a0, 0u, a2, 0u, r0, r1);
        mma_bf16(d1, a0, 0u, a2, 0u, r2, r3);
        oacc[2 * t2][0] = d0[0]; oacc[2 * t2][1] = d0[1];
        oacc[2 * t2 + 1][0] = d1[0]; oacc[2 * t2 + 1][1] = d1[1];
      }
    }
    release_stage(S, cseq + 1);
    cseq += 2;
  }
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  trace_mark(p, S, 3);

  // ---- merge the 8 warps' (m, l, o)
  float* sm_m = reinterpret_cast<float*>(S.small + 16);  // [8][8]
  float* sm_l = sm_m + 64;                                 // [8][8]
  float* so = S.scratch;                                   // [8][gs][HD]
  if (c == 0) sm_m[warp * 8 + g8] = m_run;
  bar_sync_consumers();
  trace_mark(p, S, 8);
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * 8 + g8]);
  const float sc = (m_run == -INFINITY) ? 0.f : exp2f(m_run - M);
  if (g8 < gs) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float2 v2 = make_float2(oacc[t][0] * sc, oacc[t][1] * sc);
      *reinterpret_cast<float2*>(so + ((size_t)warp * gs + g8) * HD + 8 * t + 2 * c) = v2;
    }
    if (c == 0) sm_l[warp * 8 + g8] = l_run * sc;
  }
  bar_sync_consumers();
  trace_mark(p, S, 9);
  float* dst = p.attp + ((size_t)l * p.Hkv * p.B * p.max_items_bg + it.part) * (size_t)(gs * (HD + 2));
  for (int o = threadIdx.x; o < gs * HD; o += kConsumerThreads) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) s += so[(size_t)w * gs * HD + o];
    dst[o] = s;
  }
  if (threadIdx.x < gs) {
    const int h = threadIdx.x;
    float mm = -INFINITY, ll = 0.f;
    for (int w = 0; w < kConsumerWarps; ++w) mm = fmaxf(mm, sm_m[w * 8 + h]);
    for (int w = 0; w < kConsumerWarps; ++w) ll += sm_l[w * 8 + h];
    dst[gs * HD + h] = mm;
    dst[gs * HD + gs + h] = ll;
  }
  trace_mark(p, S, 10);
  return true;
}

// The new token's own key: partial with m = s, l = 1, o = v_new.
template <int HD>
__device__ void attention_self(const Params& p, int l, const AttItem& it, int task) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gs = p.gs;
  float* dst = p.attp + ((size_t)l * p.Hkv * p.B * p.max_items_bg + it.part) * (size_t)(gs * (HD + 2));
  int pg = (it.pos / 16 < p.max_pages) ? p.page_table[it.b * p.max_pages + it.pos / 16] : -1;
  if (pg < 0 || pg >= p.n_pages) pg = 0;  // the QKV epilogue has already raised MK_ERR_BAD_PAGE
  const size_t slot = ((((size_t)l * p.n_pages + pg) * p.Hkv + it.g) * 16 + (it.pos % 16)) * HD;
  for (int h = warp; h < gs; h += kConsumerWarps) {
    const uint16_t* q = p.Q + ((size_t)l * p.B + it.b) * p.Hq * HD + (size_t)(gs * it.g + h) * HD;
    float s = 0.f;
    for (int dd = lane; dd < HD; dd += 32) {
      const float kv = bf16_to_f(__ldcg(p.kc + slot + dd));
      s += bf16_to_f(__ldcg(q + dd)) * kv;
      dst[h * HD + dd] = bf16_to_f(__ldcg(p.vc + slot + dd));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      dst[gs * HD + h] = s * p.scale_log2;
      dst[gs * HD + gs + h] = 1.f;
    }
  }
}

// ATTN_COMBINE: log-sum-exp merge of the (ns + 1) partials of (b, g) -> o (bf16).
// Warp h merges head h over batches of KB partials: lane t < KB loads partial t's
// (m, l) and every lane its HD/32 dims of all KB partials' o, all loads of a batch in
// flight together (one L2 round trip per batch); the running sums are rescaled to the
// running maximum between batches (the split-softmax merge applied batch by batch).
template <int HD>
__device__ void attention_combine(const Params& p, int l, int b, int g, int ns) {
  constexpr int V = HD / 32;  // dims per lane: 4 (128), 2 (64), 1 (32)
  constexpr int KB = 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gs = p.gs;
  const size_t stride = (size_t)gs * (HD + 2);
  const float* base = p.attp + ((size_t)l * p.Hkv * p.B * p.max_items_bg + (size_t)(g * p.B + b) * p.max_items_bg) * stride;
  const int n = ns + 1;
  for (int h = warp; h < gs; h += kConsumerWarps) {
    float M = -INFINITY, Ls = 0.f;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    for (int s0 = 0; s0 < n; s0 += KB) {
      const int cnt = min(KB, n - s0);
      const float* bs = base + (size_t)s0 * stride;
      float mt = -INFINITY, lt = 0.f;
      if (lane < cnt) {
        mt = ldg_cg(bs + lane * stride + gs * HD + h);
        lt = ldg_cg(bs + lane * stride + gs * HD + gs + h);
      }
      float x[KB][V];
#pragma unroll
      for (int t = 0; t < KB; ++t) {
        const float* o = bs + t * stride + h * HD + lane * V;
        if (t < cnt) {
          if (V == 4) {
            const float4 q = __ldcg(reinterpret_cast<const float4*>(o));
            x[t][0] = q.x; x[t][V > 1 ? 1 : 0] = q.y; x[t][V > 2 ? 2 : 0] = q.z; x[t][V > 3 ? 3 : 0] = q.w;
          } else if (V == 2) {
            const float2 q = __ldcg(reinterpret_cast<const float2*>(o));
            x[t][0] = q.x; x[t][V > 1 ? 1 : 0] = q.y;
          } else {
            x[t][0] = __ldcg(o);
          }
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) x[t][i] = 0.f;
        }
      }
      float mb = mt;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      const float Mn = fmaxf(M, mb);
      const float sc = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
      const float w = (mt == -INFINITY) ? 0.f : exp2f(mt - Mn);
      Ls = Ls * sc + w * lt;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] *= sc;
#pragma unroll
      for (int t = 0; t < KB; ++t) {
        const float wt = __shfl_sync(0xffffffffu, w, t);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += wt * x[t][i];
      }
      M = Mn;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    const float inv = 1.f / Ls;
    uint16_t* out = p.atto + ((size_t)l * p.B + b) * p.Hq * HD + (size_t)(gs * g + h) * HD + lane * V;
#pragma unroll
    for (int i = 0; i < V; ++i) out[i] = to_bf16(acc[i] * inv);
  }
}

template <int HD>
__device__ bool task_attention(const Params& p, const Smem& S, uint32_t& cseq, uint32_t& sseq, int l, int item, int nch,
                               int ti) {
  const AttItem it = att_decode(p, S, l, item);
  if (!consumer_wait(p, S, C_QKVG(p, l, it.g), (unsigned)p.qkv_tpg, ti)) {
    drain_chunks(p, S, cseq, nch);
    return false;
  }
  if (it.s < it.ns) {
    if (!attention_split<HD>(p, S, cseq, l, it)) return false;
  } else {
    attention_self<HD>(p, l, it, ti);
  }
  trace_mark(p, S, 12);
  if (signal_fanin(p, S, C_ATT(p, l, it.b, it.g), (unsigned)(it.ns + 1))) {
    attention_combine<HD>(p, l, it.b, it.g, it.ns);
    trace_mark(p, S, 14);
    signal_async(p, S, sseq, C_OG(p, l, it.g), 1u);
    signal_async(p, S, sseq, C_OA(p, l), 1u);
  }
  trace_mark(p, S, 13);
  bar_sync_consumers();
  return true;
}

// ============================================================== embed
// x0 = Embed[token] for every token.  The rows are read as 16-byte chunks of 8 values,
// four chunks a thread in flight together (the loads of a serial per-element loop each
// paid a full HBM round trip); 16 consecutive chunks are one 128-row block of one
// token, so each block's sum of squares is a reduction over 16 lanes.
__device__ void task_embed(const Params& p, const Smem& S, uint32_t& sseq, int ti) {
  const int tid = threadIdx.x, lane = tid & 31;
  int* tok = reinterpret_cast<int*>(S.scratch);
  // step 0 reads the caller's tokens, later steps (multi-step decode) the previous
  // step's greedy tokens
  const int step = S.small[249];
  if (tid < p.B) {
    int t = step == 0 ? p.tokens[tid] : ld_volatile(p.tok_out + (size_t)(step - 1) * p.B + tid);
    if (t < 0 || t >= p.V) {
      raise_err(p, MK_ERR_BAD_TOKEN, ti, -1, t, tid);
      t = 0;
    }
    tok[tid] = t;
  }
  bar_sync_consumers();
  const int cpr = p.d / 8, n = p.B * cpr;  // chunks a row, in all
  const float4* gain = reinterpret_cast<const float4*>(p.attn_norm);
  constexpr int kU = 4;
  for (int c0 = 0; c0 < n; c0 += kU * kConsumerThreads) {
    uint4 e[kU];
    float4 g0[kU], g1[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c0 + u * kConsumerThreads + tid;
      e[u] = make_uint4(0u, 0u, 0u, 0u);
      g0[u] = g1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < n) {
        const int b = c / cpr, k8 = c - b * cpr;
        e[u] = __ldg(reinterpret_cast<const uint4*>(p.embed + (size_t)tok[b] * p.d) + k8);
        g0[u] = __ldg(gain + 2 * k8);
        g1[u] = __ldg(gain + 2 * k8 + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c0 + u * kConsumerThreads + tid;
      const bool on = c < n;
      const int b = on ? c / cpr : 0, k8 = on ? c - b * cpr : 0;
      const uint32_t ew[4] = {e[u].x, e[u].y, e[u].z, e[u].w};
      const float gw[8] = {g0[u].x, g0[u].y, g0[u].z, g0[u].w, g1[u].x, g1[u].y, g1[u].z, g1[u].w};
      float x[8];
      uint32_t hw[4], lw[4];
      float sq = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        x[j] = bf16_to_f((uint16_t)(ew[j / 2] >> (16 * (j & 1))));
        sq += x[j] * x[j];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float y0 = x[2 * j] * gw[2 * j], y1 = x[2 * j + 1] * gw[2 * j + 1];
        const uint16_t h0 = to_bf16(y0), h1 = to_bf16(y1);
        hw[j] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        lw[j] = (uint32_t)to_bf16(y0 - bf16_to_f(h0)) | ((uint32_t)to_bf16(y1 - bf16_to_f(h1)) << 16);
      }
      if (on) {
        const size_t o = (size_t)b * p.d + 8 * k8;
        reinterpret_cast<float4*>(p.X + o)[0] = make_float4(x[0], x[1], x[2], x[3]);
        reinterpret_cast<float4*>(p.X + o)[1] = make_float4(x[4], x[5], x[6], x[7]);
        *reinterpret_cast<uint4*>(p.XG + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(p.XGL + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (on && (lane & 15) == 0) p.SS[(size_t)(k8 >> 4) * kSsStride + b] = sq;
    }
  }
  bar_sync_consumers();
  signal_async(p, S, sseq, C_LR(p, 0), (unsigned)p.nrb_d);
  bar_sync_consumers();
}

// ============================================================== consumer loop
__device__ void consumer(const Params& p, const Smem& S) {
  uint32_t cseq = 0, mseq = 0, sseq = 0;
  uint32_t useq = 0;  // tensor-core chunk commits of this step (LM head on tcgen05)
  bool skip = false;
  BFrag fr;
  OperandKey have = {-1, -1, -1};
  float rs_have = 0.f;
  // thread 0: the abort flag as loaded one entry earlier (the load's round trip then
  // overlaps the task instead of delaying the start of the next one)
  int abort_seen = threadIdx.x == 0 ? ld_volatile(&p.err[E_ABORT]) : 0;
  while (true) {
    // Thread 0 takes the mailbox entry and the abort flag; every consumer thread
    // then follows the same path, so the named barriers stay matched.
    const uint32_t slot = mseq % kMbox;
    if (threadIdx.x == 0) {
      const bool got = mbar_wait(S.mfull(slot), (mseq / kMbox) & 1u, 16 * p.timeout_ns);
      if (!got) raise_err(p, MK_ERR_TIMEOUT, -5, -1, (int)mseq, 0);
      S.small[3] = got ? 1 : 0;
      S.small[4] = abort_seen != 0 ? 1 : 0;
      abort_seen = ld_volatile(&p.err[E_ABORT]);
    }
    bar_sync_consumers();
    const bool got = S.small[3] != 0;
    const bool abort_now = S.small[4] != 0;
    const int4 ent = got ? S.mbox[4 * slot] : make_int4(-1, 0, 0, 0);
    const int4 ent2 = got ? S.mbox[4 * slot + 1] : make_int4(0, 0, 0, 0);
    const int4 ew_lo = got ? S.mbox[4 * slot + 2] : make_int4(0, 0, 0, 0);
    const int4 ew_hi = got ? S.mbox[4 * slot + 3] : make_int4(0, 0, 0, 0);
    bar_sync_consumers();
    if (got && threadIdx.x == 0) mbar_arrive(S.mempty(slot));
    ++mseq;
    if (ent.x < 0) break;
    const int* T = p.tasks + ent.x * kDescInts;
    const int nch = ent.z;
    const int op = ent2.w & 0xff, wl = (ent2.w >> 8) & 0xffff;
    const bool aux1 = ((ent2.w >> 24) & 1) != 0;
    if (p.trace && threadIdx.x == 0) {
      unsigned long long* t = trace_slots(S);
      t[0] = gtime(); t[1] = t[2] = t[3] = t[6] = t[8] = t[9] = t[10] = 0ull;
      t[12] = t[13] = t[14] = t[15] = 0ull;
      // (expert items: when the producer pushed the entry, route words in hand)
      t[11] = ent2.z ? t[0] - (unsigned)((unsigned)t[0] - (unsigned)ent2.z) : 0ull;
    }
    if (abort_now) skip = true;
    if (skip) {
      if (!drain_chunks(p, S, cseq, nch)) break;
      continue;
    }
    bool ok = true;
    switch (op) {
      case OP_EMBED:
        task_embed(p, S, sseq, ent.x);
        break;
      case OP_RESID:
        ok = task_resid(p, S, sseq, T, ent.x);
        break;
      case OP_ATT_DRAIN:
        // the cached GEMV operand is dropped here (re-defined below), so its
        // registers are free while the attention routine runs
        if (p.hd == 128) ok = task_attention<128>(p, S, cseq, sseq, T[D_LAYER], ent.y, nch, ent.x);
        else if (p.hd == 64) ok = task_attention<64>(p, S, cseq, sseq, T[D_LAYER], ent.y, nch, ent.x);
        else ok = task_attention<32>(p, S, cseq, sseq, T[D_LAYER], ent.y, nch, ent.x);
        have = {-1, -1, -1};
#pragma unroll
        for (int j = 0; j < kMaxKsw; ++j) fr.b0[j] = fr.b1[j] = 0u;
        break;
      case OP_MOE_DRAIN: {
        // (a dense layer's FFN items: bf16 f-slices of dense_fs rows)
        const int fsi = aux1 ? p.dense_fs : p.moe_fs;
        if (MK_UMMA == 2 && p.moe_umma) {
          ok = task_moe_umma(p, S, cseq, sseq, useq, wl, aux1, ent.y, nch, ent.w, ent2.x, ent2.y, ew_lo, ew_hi, fr,
                             have, rs_have);
          break;
        }
        ok = (p.fp8 && !aux1)
                 ? (p.moe_fs == 64 ? task_moe<64, true>(p, S, cseq, sseq, wl, aux1, ent.x, ent.y, nch, ent.w, ent2.x,
                                                           ent2.y, ew_lo, ew_hi, fr, have, rs_have)
                                     : task_moe<32, true>(p, S, cseq, sseq, wl, aux1, ent.x, ent.y, nch, ent.w, ent2.x,
                                                           ent2.y, ew_lo, ew_hi, fr, have, rs_have))
             : (fsi == 32)
                 ? task_moe<32>(p, S, cseq, sseq, wl, aux1, ent.x, ent.y, nch, ent.w, ent2.x, ent2.y, ew_lo, ew_hi, fr,
                                have, rs_have)
                 : task_moe<16>(p, S, cseq, sseq, wl, aux1, ent.x, ent.y, nch, ent.w, ent2.x, ent2.y, ew_lo, ew_hi, fr,
                                have, rs_have);
        break;
      }
      default:
        ok = task_gemv(p, S, cseq, sseq, useq, T, ent.x, nch, fr, have, rs_have);
        break;
    }
    if (!ok) skip = true;
    trace_emit(p, S, op, wl, ent.y);
  }
  signal_async(p, S, sseq, -1, 0u);  // tells the storer to finish
}

// ============================================================== the kernel
__global__ void __launch_bounds__(kThreads, 1)
    mk_megakernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  const Smem S = carve_smem(smem_raw);
  // multi-step decode: the generation word of the grid barrier between steps, read
  // before any CTA can advance it (the first advance waits for every CTA's arrival)
  if (threadIdx.x == 0 && p.n_steps > 1) S.small[250] = (int)ld_volatile(reinterpret_cast<const int*>(p.gen));
  // tensor memory for the LM head's and the expert items' accumulators (all 512
  // columns; one CTA per SM)
  if (MK_UMMA) {
    if ((threadIdx.x >> 5) == 0) tmem_alloc(smem_u32(S.small + 5), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  for (int step = 0; step < p.n_steps; ++step) {
    if (threadIdx.x == 0) {  // (re)initialised per step: no copy or arrival is pending here
      for (int s = 0; s < kStages; ++s) {
        mbar_init(S.full(s), 1);
        mbar_init(S.empty(s), kConsumerWarps);
      }
      for (int m = 0; m < kMbox; ++m) {
        mbar_init(S.mfull(m), 1);
        mbar_init(S.mempty(m), 1);
      }
      for (int q = 0; q < kSq; ++q) {
        mbar_init(S.sfull(q), kConsumerWarps);
        mbar_init(S.sempty(q), 1);
      }
      if (MK_UMMA) {
        mbar_init(S.mmadone(0), 1);
        mbar_init(S.mmadone(1), 1);
      }
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (threadIdx.x < p.B) S.small[224 + threadIdx.x] = ld_volatile(p.seq_lens + threadIdx.x);
    if (threadIdx.x == 0) {
      S.small[248] = (int)ld_volatile(reinterpret_cast<const int*>(p.epoch));
      S.small[249] = step;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if (warp == kProducerWarp) {
      if ((threadIdx.x & 31) == 0) producer(p, S, &tmK, &tmV);
    } else if (warp == kStorerWarp) {
      if ((threadIdx.x & 31) == 0) storer(p, S);
    } else {
      consumer(p, S);
    }
    __syncthreads();
    // every CTA clears its slice of the layer accumulators for the next step, once the
    // last layer's input is complete (every read of them is then done: each layer's
    // accumulator is read by its ADD_RMSNORM tasks and the next layer's router and QKV
    // tiles, all before the last layer-ready count completes)
    // (after an error the last CTA clears them all instead)
    if (p.do_reset) {
      if (threadIdx.x == 0)
        S.small[2] = (!aborted(p) && wait_ge(p, C_LR(p, p.L), (unsigned)p.nrb_d, -1)) ? 1 : 0;
      __syncthreads();
      if (S.small[2]) {
        float4* acc = reinterpret_cast<float4*>(p.moe);
        const size_t n4 = acc_words4(p);
        const size_t i0 = n4 * blockIdx.x / gridDim.x, i1 = n4 * (blockIdx.x + 1) / gridDim.x;
        for (size_t i = i0 + threadIdx.x; i < i1; i += blockDim.x) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __syncthreads();
    }
    // last CTA out resets the counters and queues for the next step or launch
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned old = atom_add_acq_rel(ctr_ptr(p, p.c_done), 1u);
      S.small[2] = (old == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    const bool more = step + 1 < p.n_steps;
    if (S.small[2]) {
      __threadfence();
      if (p.tok_out && threadIdx.x < p.B) {
        // the step's greedy tokens from the replicas of the argmax key
        const int b = threadIdx.x;
        unsigned long long best = 0ull;
        for (int r = 0; r < kAmaxReplicas; ++r) {
          const unsigned long long k = p.amax[(size_t)r * p.B + b];
          best = k > best ? k : best;
          p.amax[(size_t)r * p.B + b] = 0ull;
        }
        p.tok_out[(size_t)step * p.B + b] = best ? (int)~(unsigned)best : 0;
      }
      if (p.do_reset && p.snap) {
        // inspection: the step's final counters and queues, before they are cleared
        for (int i = threadIdx.x; i < p.n_ctr; i += blockDim.x) p.snap[i] = *ctr_ptr(p, i);
        for (int i = threadIdx.x; i < p.n_queues; i += blockDim.x) {
          p.snap[p.n_ctr + i] = (unsigned)p.qhead[i];
          p.snap[p.n_ctr + p.n_queues + i] = (unsigned)p.qcount[i];
        }
        __syncthreads();
      }
      if (p.do_reset) {
        for (int i = threadIdx.x; i < p.n_ctr; i += blockDim.x)
          if (i != p.c_done) *ctr_ptr(p, i) = 0u;
        for (int i = threadIdx.x; i < p.n_queues; i += blockDim.x) { p.qhead[i] = 0; p.qcount[i] = 0; }
        if (aborted(p)) {
          float4* acc = reinterpret_cast<float4*>(p.moe);
          const size_t n4 = acc_words4(p);
          for (size_t i = threadIdx.x; i < n4; i += blockDim.x) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!p.fixed)
          for (int b = threadIdx.x; b < p.B; b += blockDim.x) p.seq_lens[b] += 1;
        // the next step's epoch (never 0: freshly cleared words must not look current)
        if (threadIdx.x == 0) {
          const unsigned ep = step_epoch(S) + 1u;
          *p.epoch = ep ? ep : 1u;
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        *ctr_ptr(p, p.c_done) = 0u;
        __threadfence();
        if (more) {  // release the next step (and say whether to stop)
          p.gen[1] = aborted(p) ? 1u : 0u;
          __threadfence();
          st_release(p.gen, (unsigned)S.small[250] + (unsigned)step + 1u);
        }
      }
    }
    if (!more) break;
    if (threadIdx.x == 0) {
      // grid barrier: wait (bounded) for the last CTA of this step
      const unsigned target = (unsigned)S.small[250] + (unsigned)step + 1u;
      const uint64_t t0 = gtime();
      bool stop = false;
      while ((int)(ld_acquire(p.gen) - target) < 0) {
        __nanosleep(256);
        if ((long long)(gtime() - t0) > p.timeout_ns) {
          raise_err(p, MK_ERR_TIMEOUT, -20, -1, (int)ld_acquire(p.gen), (int)target);
          stop = true;
          break;
        }
      }
      S.small[251] = (stop || ld_volatile(reinterpret_cast<const int*>(p.gen + 1)) != 0) ? 1 : 0;
    }
    __syncthreads();
    if (S.small[251]) break;
  }
  // every MMA and tensor-memory read of the launch has completed (waited in its task)
  if (MK_UMMA) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
      tc_fence_after();
      tmem_dealloc((uint32_t)S.small[5], 512);
    }
  }
}

#if !MK_DET && !MK_UMMA
// ============================================================== weight packer
// Source of packed row r (see mk_pack_kernel): the matrix (0 = a, 1 = b, 2 = c) and its
// row, or row -1 for a zero padding row.
__device__ __forceinline__ void pack_source_row(int mode, int r, int n_src_rows, int hd, int gs, int grp,
                                                int& which, long long& srow) {
  which = 0;
  srow = r;
  if (mode == PACK_QKV) {
    const int head = r / hd, jj = r % hd, m = jj / 16, i = jj % 16;
    const int dim = (i < 8) ? 8 * m + i : hd / 2 + 8 * m + (i - 8);
    if (head < gs) { which = 0; srow = (long long)(grp * gs + head) * hd + dim; }
    else { which = head == gs ? 1 : 2; srow = (long long)grp * hd + dim; }
  } else if (mode == PACK_GATE_UP) {
    const int blk = r / 16, i = r % 16;
    which = i < 8 ? 0 : 1;
    srow = 8LL * blk + (i & 7);
    if (srow >= n_src_rows) srow = -1;
  } else if (srow >= n_src_rows) {
    srow = -1;
  }
}

// FP8 projections, setup (1): the float32 scale of every packed row -- max|w| over the
// source row's first k_full columns / 448, 1 for an all-zero or padding row.
__global__ void mk_pack_rowscale_kernel(float* __restrict__ dst, const uint16_t* __restrict__ src_a,
                                        const uint16_t* __restrict__ src_b, const uint16_t* __restrict__ src_c,
                                        int n_rows_packed, int n_src_rows, int k_full, long long ld, int mode,
                                        int hd, int gs, int grp) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows_packed) return;
  int which;
  long long srow;
  pack_source_row(mode, r, n_src_rows, hd, gs, grp, which, srow);
  float amax = 0.f;
  if (srow >= 0) {
    const uint16_t* src = (which == 0 ? src_a : which == 1 ? src_b : src_c) + srow * ld;
    for (int k = 0; k < k_full; ++k) amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)src[k] << 16)));
  }
  dst[r] = amax > 0.f ? amax / 448.f : 1.f;
}

// FP8 projections, setup (2): the E4M3 codes of the packed tiles, in the bf16 fragment
// order of mk_pack_kernel with 8 bytes a lane: each element divided by its packed row's
// scale and rounded to the nearest code (ties to even, saturating at 448).
__global__ void mk_pack_fp8_kernel(uint8_t* __restrict__ dst, const float* __restrict__ scales,
                                   const uint16_t* __restrict__ src_a, const uint16_t* __restrict__ src_b,
                                   const uint16_t* __restrict__ src_c, int n_rows_packed, int n_src_rows, int K,
                                   long long ld, int col0, int mode, int hd, int gs, int grp, int tile_rows) {
  const long long total = (long long)(n_rows_packed / 16) * (K / 16) * 32;
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= total) return;
  const int lane = (int)(u & 31);
  const long long fr = u >> 5;
  const int nrb_t = tile_rows / 16;
  const int ks_n = K / 16;
  const long long per_tile = (long long)nrb_t * ks_n;
  const int t = (int)(fr / per_tile);
  const int fi = (int)(fr % per_tile);
  const int j = fi / (nrb_t * 8), rem = fi % (nrb_t * 8);
  const int rb = t * nrb_t + rem / 8;
  const int ks = rem % 8 + 8 * j;
  const int g8 = lane >> 2, c = lane & 3;
  uint8_t out[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = rb * 16 + g8 + ((q & 1) ? 8 : 0);
    const int k = 16 * ks + 2 * c + ((q & 2) ? 8 : 0);
    int which;
    long long srow;
    pack_source_row(mode, r, n_src_rows, hd, gs, grp, which, srow);
    const uint16_t* src = which == 0 ? src_a : which == 1 ? src_b : src_c;
    const float sc = scales[r];
    for (int e = 0; e < 2; ++e) {
      const float x = srow >= 0 ? __uint_as_float((uint32_t)src[srow * ld + col0 + k + e] << 16) : 0.f;
      out[2 * q + e] = (uint8_t)__nv_cvt_float_to_fp8(x / sc, __NV_SATFINITE, __NV_E4M3);
    }
  }
  reinterpret_cast<uint2*>(dst)[u] =
      make_uint2((uint32_t)out[0] | ((uint32_t)out[1] << 8) | ((uint32_t)out[2] << 16) | ((uint32_t)out[3] << 24),
                 (uint32_t)out[4] | ((uint32_t)out[5] << 8) | ((uint32_t)out[6] << 16) | ((uint32_t)out[7] << 24));
}


// Packs a row-major bf16 matrix into 16x16 MMA A-fragments (16 bytes per lane):
//   lane -> (g, 2c..2c+1) (g+8, 2c..2c+1) (g, 2c+8..2c+9) (g+8, 2c+8..2c+9), g = lane/4, c = lane%4.
// Packed rows are cut into tiles of `tile_rows`; inside a tile of NRB row blocks,
// fragment (row block rb, k16-step ks = w + 8 j) is stored at index (j*NRB + rb)*8 + w,
// the order in which consumer warp w walks the tile.  Packed row r maps to a source
// row by `mode`: identity; QKV (a KV group's query heads, then its K head and V head,
// each head's rows permuted so rows g and g+8 of a 16-row block are the RoPE pair
// (i, i + hd/2)); or GATE_UP (8 gate rows then the 8 matching up rows per block).
__global__ void mk_pack_kernel(uint8_t* __restrict__ dst, const uint16_t* __restrict__ src_a,
                               const uint16_t* __restrict__ src_b, const uint16_t* __restrict__ src_c,
                               int n_rows_packed, int n_src_rows, int K, long long ld, int col0, int mode,
                               int hd, int gs, int grp, int tile_rows) {
  const long long total = (long long)(n_rows_packed / 16) * (K / 16) * 32;
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= total) return;
  const int lane = (int)(u & 31);
  const long long fr = u >> 5;
  const int nrb_t = tile_rows / 16;
  const int ks_n = K / 16;
  const long long per_tile = (long long)nrb_t * ks_n;
  const int t = (int)(fr / per_tile);
  const int fi = (int)(fr % per_tile);
  const int j = fi / (nrb_t * 8), rem = fi % (nrb_t * 8);
  const int rb = t * nrb_t + rem / 8;
  const int ks = rem % 8 + 8 * j;
  const int g8 = lane >> 2, c = lane & 3;
  uint16_t out[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = rb * 16 + g8 + ((q & 1) ? 8 : 0);
    const int k = 16 * ks + 2 * c + ((q & 2) ? 8 : 0);
    const uint16_t* src = src_a;
    long long srow = r;
    long long nsrc = n_src_rows;
    if (mode == PACK_QKV) {
      const int head = r / hd, jj = r % hd, m = jj / 16, i = jj % 16;
      const int dim = (i < 8) ? 8 * m + i : hd / 2 + 8 * m + (i - 8);
      if (head < gs) { src = src_a; srow = (long long)(grp * gs + head) * hd + dim; }
      else { src = (head == gs) ? src_b : src_c; srow = (long long)grp * hd + dim; }
      nsrc = 1ll << 40;
    } else if (mode == PACK_GATE_UP) {
      const int blk = r / 16, i = r % 16;
      src = (i < 8) ? src_a : src_b;
      srow = 8LL * blk + (i & 7);
    }
    for (int e = 0; e < 2; ++e)
      out[2 * q + e] = (srow < nsrc) ? src[srow * ld + col0 + k + e] : (uint16_t)0;
  }
  uint4 v;
  v.x = out[0] | ((uint32_t)out[1] << 16);
  v.y = out[2] | ((uint32_t)out[3] << 16);
  v.z = out[4] | ((uint32_t)out[5] << 16);
  v.w = out[6] | ((uint32_t)out[7] << 16);
  reinterpret_cast<uint4*>(dst)[u] = v;
}

// All t = d_ff / 32 items of one expert (see the MoE item layout in mk_internal.h).
__global__ void mk_pack_moe_kernel(uint8_t* __restrict__ dst, const uint16_t* __restrict__ gate,
                                   const uint16_t* __restrict__ up, const uint16_t* __restrict__ down, int d,
                                   int f, int fs) {
  const int t_n = f / fs;
  const int nrb1 = fs / 8, k2 = fs / 16;
  const long long gu_units = (long long)nrb1 * (d / 16) * 32;
  const long long dn_units = (long long)(d / 16) * k2 * 32;
  const long long item_units = gu_units + dn_units;
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= item_units * t_n) return;
  const int s = (int)(u / item_units);
  long long r = u % item_units;
  const int lane = (int)(r & 31);
  const int g8 = lane >> 2, c = lane & 3;
  uint16_t out[8];
  if (r < gu_units) {
    // gate/up tile: fs/8 row blocks (8 gate + 8 up rows each), GEMV order (j*nrb1 + rb)*8 + w
    const long long fi = r >> 5;
    const int j = (int)(fi / (nrb1 * 8)), rem = (int)(fi % (nrb1 * 8));
    const int rb = rem / 8, ks = rem % 8 + 8 * j;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = g8 + ((q & 1) ? 8 : 0);                 // row within the block
      const int k = 16 * ks + 2 * c + ((q & 2) ? 8 : 0);
      const uint16_t* src = (i < 8) ? gate : up;
      const long long srow = (long long)s * fs + 8 * rb + (i & 7);
      out[2 * q] = src[srow * d + k];
      out[2 * q + 1] = src[srow * d + k + 1];
    }
  } else {
    // down slice: warp w owns rows [w d/8, (w+1) d/8); order [w][row block][ks]
    const long long fi = (r - gu_units) >> 5;
    const int rpw = d / 128;
    const int w = (int)(fi / (rpw * k2)), rem = (int)(fi % (rpw * k2));
    const int rb = w * rpw + rem / k2, ks = rem % k2;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const long long row = (long long)rb * 16 + g8 + ((q & 1) ? 8 : 0);
      const int col = s * fs + 16 * ks + 2 * c + ((q & 2) ? 8 : 0);
      out[2 * q] = down[row * f + col];
      out[2 * q + 1] = down[row * f + col + 1];
    }
  }
  uint4 v;
  v.x = out[0] | ((uint32_t)out[1] << 16);
  v.y = out[2] | ((uint32_t)out[3] << 16);
  v.z = out[4] | ((uint32_t)out[5] << 16);
  v.w = out[6] | ((uint32_t)out[7] << 16);
  reinterpret_cast<uint4*>(dst)[u] = v;
}

// FP8 experts, setup (1): the f32 scales of each item of one expert, one per output
// channel -- its gate/up rows in packed-row order (block rb: 8 gate rows then their 8
// up rows), then every down row (the same in each item of the expert): max|w| over
// the whole row / 448, 1 for an all-zero row.
__global__ void mk_pack_moe_fp8_scales(uint8_t* __restrict__ dst, const uint16_t* __restrict__ gate,
                                       const uint16_t* __restrict__ up, const uint16_t* __restrict__ down, int d,
                                       int f, int fs, long long item_bytes) {
  const int per = 2 * fs + d;
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= (long long)per * (f / fs)) return;
  const int s = (int)(u / per), r = (int)(u % per);
  float amax = 0.f;
  if (r < 2 * fs) {
    const int rb = r / 16, i = r % 16;
    const uint16_t* src = (i < 8 ? gate : up) + ((size_t)s * fs + 8 * rb + (i & 7)) * d;
    for (int k = 0; k < d; ++k) amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)src[k] << 16)));
  } else {
    const uint16_t* src = down + (size_t)(r - 2 * fs) * f;
    for (int k = 0; k < f; ++k) amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)src[k] << 16)));
  }
  reinterpret_cast<float*>(dst + (size_t)s * item_bytes)[r] = amax > 0.f ? amax / 448.f : 1.f;
}

// FP8 experts, setup (2): the E4M3 codes, in the bf16 fragment order (8 bytes a lane),
// each element divided by its row's scale and rounded to the nearest code (ties to
// even, saturating at 448).
__global__ void mk_pack_moe_fp8_codes(uint8_t* __restrict__ dst, const uint16_t* __restrict__ gate,
                                      const uint16_t* __restrict__ up, const uint16_t* __restrict__ down, int d,
                                      int f, int fs, long long item_bytes) {
  const int t_n = f / fs;
  const int nrb1 = fs / 8, k2 = fs / 16;
  const long long gu_units = (long long)nrb1 * (d / 16) * 32;
  const long long dn_units = (long long)(d / 16) * k2 * 32;
  const long long item_units = gu_units + dn_units;
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= item_units * t_n) return;
  const int s = (int)(u / item_units);
  const long long r = u % item_units;
  const int lane = (int)(r & 31);
  const int g8 = lane >> 2, c = lane & 3;
  uint8_t* item = dst + (size_t)s * item_bytes;
  const float* scl = reinterpret_cast<const float*>(item);
  const int sb = fp8_scale_bytes(fs, d);
  uint8_t out[8];
  if (r < gu_units) {
    const long long fi = r >> 5;
    const int j = (int)(fi / (nrb1 * 8)), rem = (int)(fi % (nrb1 * 8));
    const int rb = rem / 8, ks = rem % 8 + 8 * j;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = g8 + ((q & 1) ? 8 : 0);
      const int k = 16 * ks + 2 * c + ((q & 2) ? 8 : 0);
      const uint16_t* src = (i < 8) ? gate : up;
      const long long srow = (long long)s * fs + 8 * rb + (i & 7);
      const float sc = scl[rb * 16 + i];
      for (int e = 0; e < 2; ++e)
        out[2 * q + e] = (uint8_t)__nv_cvt_float_to_fp8(__uint_as_float((uint32_t)src[srow * d + k + e] << 16) / sc,
                                                        __NV_SATFINITE, __NV_E4M3);
    }
    *reinterpret_cast<uint2*>(item + sb + r * 8) =
        make_uint2((uint32_t)out[0] | ((uint32_t)out[1] << 8) | ((uint32_t)out[2] << 16) | ((uint32_t)out[3] << 24),
                   (uint32_t)out[4] | ((uint32_t)out[5] << 8) | ((uint32_t)out[6] << 16) | ((uint32_t)out[7] << 24));
  } else {
    const long long fi = (r - gu_units) >> 5;
    const int rb = (int)(fi / k2), ks = (int)(fi % k2);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const long long row = (long long)rb * 16 + g8 + ((q & 1) ? 8 : 0);
      const int col = s * fs + 16 * ks + 2 * c + ((q & 2) ? 8 : 0);
      const float sc = scl[2 * fs + row];
      for (int e = 0; e < 2; ++e)
        out[2 * q + e] = (uint8_t)__nv_cvt_float_to_fp8(__uint_as_float((uint32_t)down[row * f + col + e] << 16) / sc,
                                                        __NV_SATFINITE, __NV_E4M3);
    }
    *reinterpret_cast<uint2*>(item + sb + gu_units / 32 * kFragBytes8 + (r - gu_units) * 8) =
        make_uint2((uint32_t)out[0] | ((uint32_t)out[1] << 8) | ((uint32_t)out[2] << 16) | ((uint32_t)out[3] << 24),
                   (uint32_t)out[4] | ((uint32_t)out[5] << 8) | ((uint32_t)out[6] << 16) | ((uint32_t)out[7] << 24));
  }
}

cudaError_t launch_pack_moe_fp8(uint8_t* dst, const void* gate, const void* up, const void* down, int d, int f,
                                int fs, long long item_bytes, cudaStream_t st) {
  const long long nsc = (long long)(2 * fs + d) * (f / fs);
  mk_pack_moe_fp8_scales<<<(unsigned)((nsc + 255) / 256), 256, 0, st>>>(
      dst, (const uint16_t*)gate, (const uint16_t*)up, (const uint16_t*)down, d, f, fs, item_bytes);
  const long long units = ((long long)(fs / 8) * (d / 16) * 32 + (long long)(d / 16) * (fs / 16) * 32) * (f / fs);
  mk_pack_moe_fp8_codes<<<(unsigned)((units + 255) / 256), 256, 0, st>>>(
      dst, (const uint16_t*)gate, (const uint16_t*)up, (const uint16_t*)down, d, f, fs, item_bytes);
  return cudaGetLastError();
}

// LM-head tiles for the tensor-core path: 64-row tiles, each cut into chunks of 256
// columns (32 KB, one ring stage), each chunk in the K-major core-matrix layout with its
// second 128 columns stacked under the first as rows 64..127: core matrix (kc, mg) --
// rows 8 mg .. 8 mg + 7 of the stacking, columns 8 kc .. 8 kc + 7 of its half, 16 bytes
// a row -- at (kc * 16 + mg) * 128 bytes.  One thread per 16-byte core-matrix row; rows
// past n_src_rows are zero.  K is a multiple of 256.
__global__ void mk_pack_umma_kernel(uint8_t* __restrict__ dst, const uint16_t* __restrict__ src, int n_rows_packed,
                                    int n_src_rows, int K) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int g8 = K / 8;
  if (u >= (long long)n_rows_packed * g8) return;
  const int r = (int)(u / g8), kk = (int)(u % g8);
  const int tile = r / 64, m = r % 64, chunk = kk / 32, kc = kk % 16, mg = m / 8 + 8 * ((kk % 32) / 16);
  uint16_t e[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) e[i] = r < n_src_rows ? src[(size_t)r * K + 8 * kk + i] : (uint16_t)0;
  const size_t off = ((size_t)tile * (K / 256) + chunk) * 32768 + ((size_t)kc * 16 + mg) * 128 + (m % 8) * 16;
  *reinterpret_cast<uint4*>(dst + off) =
      make_uint4((uint32_t)e[0] | ((uint32_t)e[1] << 16), (uint32_t)e[2] | ((uint32_t)e[3] << 16),
                 (uint32_t)e[4] | ((uint32_t)e[5] << 16), (uint32_t)e[6] | ((uint32_t)e[7] << 16));
}

// Expert items (bf16, 32-row f-slices) for the tensor-core path, item s of an expert:
// [gate/up: 64 packed rows x d] then [down: d rows x 32].  Packed row 16 rb + i is gate
// row 32 s + 8 rb + i (i < 8) or its up row (i >= 8), so that the pair sits 8 lanes apart
// in one warp's lane quadrant of the accumulator.  The gate/up rows come in chunks of
// 256 columns (32 KB) laid out like the LM-head chunks (the second 128 columns stacked
// under the first as rows 64..127; core (kc, mg) at (kc * 16 + mg) * 128 bytes), the down
// rows in blocks of 128 rows (8 KB, core (kc, mg) at (kc * 16 + mg) * 128 bytes).  One
// thread per 16-byte core row.
__global__ void mk_pack_moe_umma_kernel(uint8_t* __restrict__ dst, const uint16_t* __restrict__ gate,
                                        const uint16_t* __restrict__ up, const uint16_t* __restrict__ down, int d,
                                        int f) {
  constexpr int FS = 32;
  const long long per_item = 12LL * d;  // 64 rows x d/8 + d rows x 4 core rows
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= per_item * (f / FS)) return;
  const int s = (int)(u / per_item);
  const long long r = u % per_item;
  const uint16_t* src;
  size_t off = (size_t)s * 192 * d;  // item bytes
  if (r < 8LL * d) {
    const int m = (int)(r / (d / 8)), kk = (int)(r % (d / 8));
    const int rb = m / 16, i = m % 16;
    const int frow = FS * s + 8 * rb + (i & 7);
    src = (i < 8 ? gate : up) + (size_t)frow * d + 8 * kk;
    off += (size_t)(kk / 32) * 32768 + ((size_t)(kk % 16) * 16 + m / 8 + 8 * ((kk % 32) / 16)) * 128 + (m % 8) * 16;
  } else {
    const long long q = r - 8LL * d;
    const int row = (int)(q / 4), kk = (int)(q % 4);
    src = down + (size_t)row * f + FS * s + 8 * kk;
    off += (size_t)128 * d + (size_t)(row / 128) * 8192 + ((size_t)kk * 16 + (row % 128) / 8) * 128 + (row % 8) * 16;
  }
  uint16_t e[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) e[i] = src[i];
  *reinterpret_cast<uint4*>(dst + off) =
      make_uint4((uint32_t)e[0] | ((uint32_t)e[1] << 16), (uint32_t)e[2] | ((uint32_t)e[3] << 16),
                 (uint32_t)e[4] | ((uint32_t)e[5] << 16), (uint32_t)e[6] | ((uint32_t)e[7] << 16));
}

__global__ void mk_convert_kernel(float* __restrict__ dst, const uint16_t* __restrict__ src, long long n) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = __uint_as_float((uint32_t)src[i] << 16);
}

}  // namespace mk

// ============================================================== static step scratch
// Scratch for mk_decode_step_noalloc, for callers that cannot allocate device memory.
// A file-scope device array: every GPU that loads the library holds it until exit.
static __device__ __align__(256) uint8_t g_mk_static_scratch[mk::kStaticScratchBytes];

// ============================================================== host-side launchers
namespace MK_KNS {

// Device address of the static scratch array on the current device, looked up once
// per device (with that device current) and cached.  The host-side name of the array
// is only a stand-in and must never be passed to a kernel.
cudaError_t static_scratch_address(void** ptr) {
  constexpr int kMaxDevices = 64;
  // atomic entries: host threads may make their first call on a device concurrently
  // (each looks the address up itself; they store the same value)
  static std::atomic<void*> addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* a = addr[dev].load(std::memory_order_acquire);
  if (!a) {
    e = cudaGetSymbolAddress(&a, g_mk_static_scratch);
    if (e != cudaSuccess) return e;
    addr[dev].store(a, std::memory_order_release);
  }
  *ptr = a;
  return cudaSuccess;
}

cudaError_t launch_pack(uint8_t* dst, const void* src_a, const void* src_b, const void* src_c,
                        int n_rows_packed, int n_src_rows, int K, long long ld, int col0, int mode, int hd,
                        int gs, int grp, int tile_rows, cudaStream_t st) {
  const long long total = (long long)(n_rows_packed / 16) * (K / 16) * 32;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  mk_pack_kernel<<<(unsigned)blocks, threads, 0, st>>>(dst, (const uint16_t*)src_a, (const uint16_t*)src_b,
                                                     (const uint16_t*)src_c, n_rows_packed, n_src_rows, K, ld,
                                                     col0, mode, hd, gs, grp, tile_rows);
  return cudaGetLastError();
}

cudaError_t launch_pack_rowscale(float* dst, const void* src_a, const void* src_b, const void* src_c,
                                 int n_rows_packed, int n_src_rows, int k_full, long long ld, int mode, int hd,
                                 int gs, int grp, cudaStream_t st) {
  if (n_rows_packed == 0) return cudaSuccess;
  mk_pack_rowscale_kernel<<<(unsigned)((n_rows_packed + 127) / 128), 128, 0, st>>>(
      dst, (const uint16_t*)src_a, (const uint16_t*)src_b, (const uint16_t*)src_c, n_rows_packed, n_src_rows, k_full,
      ld, mode, hd, gs, grp);
  return cudaGetLastError();
}

cudaError_t launch_pack_fp8(uint8_t* dst, const float* scales, const void* src_a, const void* src_b,
                            const void* src_c, int n_rows_packed, int n_src_rows, int K, long long ld, int col0,
                            int mode, int hd, int gs, int grp, int tile_rows, cudaStream_t st) {
  const long long total = (long long)(n_rows_packed / 16) * (K / 16) * 32;
  if (total == 0) return cudaSuccess;
  mk_pack_fp8_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
      dst, scales, (const uint16_t*)src_a, (const uint16_t*)src_b, (const uint16_t*)src_c, n_rows_packed, n_src_rows,
      K, ld, col0, mode, hd, gs, grp, tile_rows);
  return cudaGetLastError();
}

cudaError_t launch_pack_moe(uint8_t* dst, const void* gate, const void* up, const void* down, int d, int f, int fs,
                            cudaStream_t st) {
  const long long units = ((long long)(fs / 8) * (d / 16) * 32 + (long long)(d / 16) * (fs / 16) * 32) * (f / fs);
  mk_pack_moe_kernel<<<(unsigned)((units + 255) / 256), 256, 0, st>>>(dst, (const uint16_t*)gate,
                                                                     (const uint16_t*)up, (const uint16_t*)down, d, f,
                                                                     fs);
  return cudaGetLastError();
}

cudaError_t launch_pack_umma(uint8_t* dst, const void* src, int n_rows_packed, int n_src_rows, int K, cudaStream_t st) {
  const long long units = (long long)n_rows_packed * (K / 8);
  if (units == 0) return cudaSuccess;
  mk_pack_umma_kernel<<<(unsigned)((units + 255) / 256), 256, 0, st>>>(dst, (const uint16_t*)src, n_rows_packed,
                                                                      n_src_rows, K);
  return cudaGetLastError();
}

cudaError_t launch_pack_moe_umma(uint8_t* dst, const void* gate, const void* up, const void* down, int d, int f,
                                 cudaStream_t st) {
  const long long units = 12LL * d * (f / 32);
  mk_pack_moe_umma_kernel<<<(unsigned)((units + 255) / 256), 256, 0, st>>>(
      dst, (const uint16_t*)gate, (const uint16_t*)up, (const uint16_t*)down, d, f);
  return cudaGetLastError();
}

cudaError_t launch_convert(float* dst, const void* src, long long n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  mk_convert_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(dst, (const uint16_t*)src, n);
  return cudaGetLastError();
}

#endif  // !MK_DET && !MK_UMMA

cudaError_t prepare_megakernel() {
  return cudaFuncSetAttribute(mk_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

int megakernel_occupancy(int* blocks) {
  return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, mk_megakernel, kThreads, kSmemBytes);
}

cudaError_t launch_megakernel(const Params& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                              bool cooperative, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mk_megakernel, p, tk, tv);
}

}  // namespace mk
