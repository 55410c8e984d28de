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
#include "mk_device.cuh"

namespace mk {

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
//   record (8 x u64): [0] sm | op << 8 | layer << 16 | fan-in << 24, [1] item,
//   [2] received, [3] dependency met, [4] first weight/KV chunk landed,
//   [5] MMA loop done, [6] fan-in follow-up started (0 if none), [7] task done.
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
  unsigned long long* r = p.trace + (size_t)idx * 8;
  unsigned long long* t = trace_slots(S);
  r[0] = (unsigned long long)blockIdx.x | ((unsigned long long)op << 8) |
         ((unsigned long long)(layer & 0xff) << 16) | ((unsigned long long)(t[6] != 0) << 24);
  r[1] = (unsigned long long)(unsigned)item;
  r[2] = t[0]; r[3] = t[1]; r[4] = t[2]; r[5] = t[3]; r[6] = t[6]; r[7] = gtime();
}

// Spin until ctr >= target (acquire), bounded by the timeout and the abort flag.
__device__ bool wait_ge(const Params& p, int ci, unsigned target, int task) {
  const unsigned* c = p.ctr + ci;
  if (ld_acquire(c) >= target) return true;
  const uint64_t t0 = gtime();
  for (int it = 0;; ++it) {
    __nanosleep(32);
    const unsigned v = ld_acquire(c);
    if (v >= target) return true;
    if ((it & 15) == 15) {
      if (aborted(p)) return false;
      if ((long long)(gtime() - t0) > p.timeout_ns) {
        raise_err(p, MK_ERR_TIMEOUT, task, ci, (int)v, (int)target);
        return false;
      }
    }
  }
}

// Consumer-side wait: thread 0 polls, the others learn the result at a barrier.
__device__ bool consumer_wait(const Params& p, const Smem& S, int ci, unsigned target, int task) {
  if (ci < 0) {
    trace_mark(p, S, 1);
    return true;
  }
  if (threadIdx.x == 0) {
    S.small[0] = wait_ge(p, ci, target, task) ? 1 : 0;
    if (p.trace) trace_slots(S)[1] = gtime();
  }
  bar_sync_consumers();
  const int ok = S.small[0];
  bar_sync_consumers();
  return ok != 0;
}

__device__ __forceinline__ bool wait_full(const Params& p, const Smem& S, uint32_t seq) {
  if (mbar_wait(S.full(seq % kStages), (seq / kStages) & 1u, 4 * p.timeout_ns)) return true;
  if ((threadIdx.x & 31) == 0) raise_err(p, MK_ERR_TIMEOUT, -2, -1, (int)seq, 0);
  return false;
}
__device__ __forceinline__ void release_stage(const Smem& S, uint32_t seq) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(S.empty(seq % kStages));
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
__device__ __forceinline__ int C_UP(const Params& p, int l, int a) { return p.c_up + l * p.maxa + a; }
__device__ __forceinline__ int C_RB(const Params& p, int l, int r) { return p.c_rb + l * p.nrb_d + r; }

struct AttItem {
  int b, g, s, ns;      // sequence, KV group, split (s == ns: the new token itself)
  int pos;              // position of the new token
  int pg0, np;          // logical pages of the split
  int klo, khi;         // key positions [klo, khi) of the split
  int part;             // partial slot: ((g*B + b) * max_items_bg + s)
};

__device__ __forceinline__ int layer_window(const Params& p, int l) {
  return ((p.swa_mask >> l) & 1ull) ? p.window : 0;
}

// Splits of the cached keys in the window of sequence b at layer l.
__device__ __forceinline__ void att_range(const Params& p, int l, int b, int& pos, int& lo,
                                          int& first_pg, int& npg, int& ns) {
  pos = p.seq_lens[b];
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

__device__ int att_item_count(const Params& p, int l) {
  int per_g = 0;
  for (int b = 0; b < p.B; ++b) {
    int pos, lo, fp, npg, ns;
    att_range(p, l, b, pos, lo, fp, npg, ns);
    per_g += ns + 1;
  }
  return per_g * p.Hkv;
}

// Items are ordered by (group, sequence, split): group 0's items come first, in
// step with the QKV tiles, which are dealt group by group.
__device__ AttItem att_decode(const Params& p, int l, int item) {
  int per_g = 0;
  for (int b = 0; b < p.B; ++b) {
    int pos, lo, fp, npg, ns;
    att_range(p, l, b, pos, lo, fp, npg, ns);
    per_g += ns + 1;
  }
  AttItem it;
  it.g = item / per_g;
  int rem = item % per_g;
  for (int b = 0; b < p.B; ++b) {
    int pos, lo, fp, npg, ns;
    att_range(p, l, b, pos, lo, fp, npg, ns);
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
__device__ bool mbox_push(const Params& p, const Smem& S, uint32_t& mseq, int task, int item, int nch) {
  const uint32_t slot = mseq % kMbox, use = mseq / kMbox;
  if (use > 0 && !mbar_wait(S.mempty(slot), (use - 1) & 1u, 8 * p.timeout_ns)) {
    raise_err(p, MK_ERR_TIMEOUT, task, -3, (int)mseq, 0);
    return false;
  }
  S.mbox[slot] = make_int4(task, item, nch, 0);
  mbar_arrive(S.mfull(slot));
  ++mseq;
  return true;
}

__device__ __forceinline__ bool acquire_stage(const Params& p, const Smem& S, uint32_t seq, int task) {
  const uint32_t use = seq / kStages;
  if (use == 0) return true;
  if (mbar_wait(S.empty(seq % kStages), (use - 1) & 1u, 8 * p.timeout_ns)) return true;
  raise_err(p, MK_ERR_TIMEOUT, task, -4, (int)seq, 0);
  return false;
}

__device__ bool issue_linear(const Params& p, const Smem& S, uint32_t& cseq, const uint8_t* src,
                             int bytes, uint64_t pol, int task) {
  for (int off = 0; off < bytes; off += kStageBytes) {
    const int n = min(kStageBytes, bytes - off);
    if (!acquire_stage(p, S, cseq, task)) return false;
    const uint32_t s = cseq % kStages;
    mbar_expect_tx(S.full(s), (uint32_t)n);
    bulk_g2s(S.stage(cseq), src + off, (uint32_t)n, S.full(s), pol);
    ++cseq;
  }
  return true;
}

// K pages then V pages of a split, 8 pages per ring stage.
__device__ bool issue_kv(const Params& p, const Smem& S, uint32_t& cseq, const CUtensorMap* tmK,
                         const CUtensorMap* tmV, int l, const AttItem& it, uint64_t pol, int task) {
  const int inner = p.hd < 64 ? p.hd : 64;
  const int nbox = p.hd / inner;
  const int box_bytes = 16 * inner * 2;
  const int page_bytes = 16 * p.hd * 2;
  for (int c0 = 0; c0 < it.np; c0 += 8) {
    const int n = min(8, it.np - c0);
    int rows[8];
    for (int i = 0; i < n; ++i) {
      int pg = checked_page(p, it.b, it.pg0 + c0 + i, task);
      if (pg < 0) pg = 0;
      rows[i] = ((l * p.n_pages + pg) * p.Hkv + it.g) * 16;
    }
    for (int kv = 0; kv < 2; ++kv) {
      if (!acquire_stage(p, S, cseq, task)) return false;
      const uint32_t s = cseq % kStages;
      mbar_expect_tx(S.full(s), (uint32_t)(n * page_bytes));
      const uint32_t dst = S.stage(cseq);
      const CUtensorMap* tm = kv ? tmV : tmK;
      for (int i = 0; i < n; ++i)
        for (int j = 0; j < nbox; ++j)
          tma_load_2d(dst + i * page_bytes + j * box_bytes, tm, j * inner, rows[i], S.full(s), pol);
      ++cseq;
    }
  }
  return true;
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
        ok = mbox_push(p, S, mseq, ti, 0, 0);
        break;
      case OP_QKV:
      case OP_ROUTER:
      case OP_OPROJ:
      case OP_LMHEAD: {
        const long long off = (long long)(((unsigned long long)(unsigned)T[D_WOFF_HI] << 32) |
                                          (unsigned)T[D_WOFF_LO]);
        const int bytes = T[D_WBYTES];
        const int nch = (bytes + kStageBytes - 1) / kStageBytes;
        ok = mbox_push(p, S, mseq, ti, 0, nch) && issue_linear(p, S, cseq, p.wblob + off, bytes, pol, ti);
        break;
      }
      case OP_ATT_DRAIN: {
        const int count = att_item_count(p, l);
        int* head = p.qhead + l;
        while (ok) {
          const int item = atomicAdd(head, 1);
          if (item >= count) break;
          const AttItem it = att_decode(p, l, item);
          const int nch = 2 * ((it.np + 7) / 8);
          ok = mbox_push(p, S, mseq, ti, item, nch) && issue_kv(p, S, cseq, tmK, tmV, l, it, pol, ti);
        }
        break;
      }
      case OP_UP_DRAIN:
      case OP_DN_DRAIN: {
        if (!wait_ge(p, C_RR(p, l), 1u, ti)) { ok = false; break; }
        const bool up = op == OP_UP_DRAIN;
        const int q = (up ? p.L : 2 * p.L) + l;
        const int count = ldg_cg(p.qcount + q);
        const int per = up ? p.t_up : p.t_dn;
        const long long tile_bytes = up ? (long long)p.r_up * p.d * 2 : (long long)p.r_dn * p.f * 2;
        const int nch = (int)((tile_bytes + kStageBytes - 1) / kStageBytes);
        while (ok) {
          const int item = atomicAdd(p.qhead + q, 1);
          if (item >= count) break;
          const int a = item / per, t = item % per;
          const int e = ldg_cg(p.active + l * p.maxa + a);
          const long long base = up ? p.off_up + (long long)(l * p.E + e) * p.up_bytes_e
                                    : p.off_dn + (long long)(l * p.E + e) * p.dn_bytes_e;
          ok = mbox_push(p, S, mseq, ti, item, nch) &&
               issue_linear(p, S, cseq, p.wblob + base + t * tile_bytes, (int)tile_bytes, pol, ti);
        }
        break;
      }
      default:
        break;
    }
  }
  mbox_push(p, S, mseq, -1, 0, 0);
  // make sure no copy is still landing in shared memory when the CTA retires
  const uint32_t first = cseq > (uint32_t)kStages ? cseq - kStages : 0;
  for (uint32_t q = first; q < cseq; ++q) mbar_wait(S.full(q % kStages), (q / kStages) & 1u, 8 * p.timeout_ns);
}

// ============================================================== GEMV machinery
struct BFrag {
  uint32_t b0[kMaxKsw], b1[kMaxKsw];
};

// B operand (activations) for this warp's k16-steps ks = warp + 8 j: rows n = lane/4 are
// tokens, k pairs at 2*(lane%4) and +8.  `pair(n, k)` returns bf16x2 of act[n][k..k+1].
template <class F>
__device__ __forceinline__ void build_bfrag(BFrag& fr, int ksw, F&& pair) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = lane >> 2, c = lane & 3;
#pragma unroll
  for (int j = 0; j < kMaxKsw; ++j) {
    if (j < ksw) {
      const int k = 16 * (warp + 8 * j) + 2 * c;
      fr.b0[j] = pair(n, k);
      fr.b1[j] = pair(n, k + 8);
    } else {
      fr.b0[j] = 0u;
      fr.b1[j] = 0u;
    }
  }
}

// acc[rb] += W_tile[rb] * act over this warp's k16-steps ks = warp + 8 j, consuming the
// task's ring chunks.  Tiles are packed so that fragment (rb, ks) sits at index
// (j * NRB + rb) * 8 + warp: every 32 KB chunk holds 8 / NRB consecutive j for all
// row blocks, so chunk, register and smem indices are compile-time constants.
template <int NRB>
__device__ __forceinline__ bool gemv_mainloop(const Params& p, const Smem& S, uint32_t& cseq, int nch,
                                              int ksw, const BFrag& fr, float (&acc)[NRB][4]) {
  constexpr int JPC = 8 / NRB;
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

template <int NRB>
__device__ __forceinline__ bool gemv_run(const Params& p, const Smem& S, uint32_t& cseq, int nch, int ksw,
                                         const BFrag& fr, float (&v)[4]) {
  float acc[NRB][4];
  if (!gemv_mainloop<NRB>(p, S, cseq, nch, ksw, fr, acc)) return false;
  trace_mark(p, S, 3);
  gemv_reduce<NRB>(S, acc, v);
  return true;
}

// 1 / rms of x_b (layer input) from the per-row-block sums of squares.
__device__ __forceinline__ float rstd_of(const Params& p, int layer, int b) {
  const float* ss = p.SS + (size_t)layer * p.nrb_d * p.B;
  float s = 0.f;
  for (int r = 0; r < p.nrb_d; ++r) s += ldg_cg(ss + r * p.B + b);
  return rsqrtf(s / (float)p.d + p.eps);
}

// B operand from h = RMSNorm(x_layer) * gain; `b` is the token of this lane's
// operand row (lane/4), or -1 for a zero row.
__device__ __forceinline__ void build_norm_bfrag(const Params& p, BFrag& fr, int ksw, int layer,
                                                 const float* gain, int b) {
  float rs = 0.f;
  const float* x = nullptr;
  if (b >= 0) {
    rs = rstd_of(p, layer, b);
    x = p.X + ((size_t)layer * p.B + b) * p.d;
  }
  build_bfrag(fr, ksw, [&](int, int k) -> uint32_t {
    if (b < 0) return 0u;
    const float2 xv = ldg_cg_f2(x + k);
    const float2 gv = *reinterpret_cast<const float2*>(gain + k);
    return pack_bf16(xv.x * rs * gv.x, xv.y * rs * gv.y);
  });
}

// ============================================================== epilogues / fan-in steps

// Route step: top-k of the router logits per token, softmax over the selected,
// active-expert list (ascending expert id), per-expert token lists, MoE queue sizes.
__device__ void route_step(const Params& p, const Smem& S, int l) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int* sel = S.small + 16;  // [B][topk] <= 64 ints
  if (warp < p.B) {
    const int b = warp;
    const float* r = p.rlog + ((size_t)l * p.B + b) * p.E;
    float v[8];
    int used = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < p.E) ? ldg_cg(r + e) : -INFINITY;
    }
    float selv[8];
    int sele[8];
    for (int j = 0; j < p.topk; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        if (e < p.E && !((used >> i) & 1) && (v[i] > bv || (v[i] == bv && e < be))) { bv = v[i]; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
      }
      if ((be & 31) == lane) used |= 1 << (be >> 5);
      selv[j] = bv;
      sele[j] = be;
    }
    float sum = 0.f, w[8];
    for (int j = 0; j < p.topk; ++j) { w[j] = __expf(selv[j] - selv[0]); sum += w[j]; }
    if (lane < p.topk) {
      float wj = 0.f; int ej = 0;
      for (int j = 0; j < p.topk; ++j) if (j == lane) { wj = w[j] / sum; ej = sele[j]; }
      p.ridx[((size_t)l * p.B + b) * p.topk + lane] = ej;
      p.rw[((size_t)l * p.B + b) * p.topk + lane] = wj;
      sel[b * p.topk + lane] = ej;
    }
  }
  bar_sync_consumers();
  if (warp == 0) {
    int* used = reinterpret_cast<int*>(S.scratch);  // [E]
    for (int e = lane; e < p.E; e += 32) used[e] = 0;
    __syncwarp();
    for (int i = lane; i < p.B * p.topk; i += 32) used[sel[i]] = 1;
    __syncwarp();
    const int per = (p.E + 31) / 32;
    int cnt = 0;
    for (int i = 0; i < per; ++i) { const int e = lane * per + i; if (e < p.E && used[e]) ++cnt; }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) { const int t = __shfl_up_sync(0xffffffffu, incl, o); if (lane >= o) incl += t; }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    int slot = incl - cnt;
    for (int i = 0; i < per; ++i) {
      const int e = lane * per + i;
      if (e < p.E && used[e]) { p.active[l * p.maxa + slot] = e; ++slot; }
    }
    __syncwarp();
    __threadfence_block();
    for (int a = lane; a < total; a += 32) {
      const int e = p.active[l * p.maxa + a];
      int c = 0;
      for (int b = 0; b < p.B; ++b)
        for (int j = 0; j < p.topk; ++j)
          if (sel[b * p.topk + j] == e) { p.act_tok[((size_t)l * p.maxa + a) * p.B + c] = b * 16 + j; ++c; }
      p.act_cnt[l * p.maxa + a] = c;
    }
    if (lane == 0) {
      p.nact[l] = total;
      p.qcount[p.L + l] = total * p.t_up;
      p.qcount[2 * p.L + l] = total * p.t_dn;
    }
    const unsigned pad = (unsigned)((p.maxa - total) * (kRowBlock / p.r_dn));
    if (pad > 0)
      for (int r = lane; r < p.nrb_d; r += 32) atomicAdd(p.ctr + C_RB(p, l, r), pad);
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      red_release(p.ctr + C_RR(p, l), 1u);
    }
  }
}

// Residual row block r of layer l: x_{l+1} = x_l + sum_g O-proj partial + sum_j w_j y_j,
// and the block's sums of squares for the next RMSNorm.
__device__ void residual_step(const Params& p, const Smem& S, int l, int r) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = r * kRowBlock + (tid & 127);
  const int half = tid >> 7;
  float* red = reinterpret_cast<float*>(S.small + 16);  // [8 warps][4]
  for (int i = 0; i < 4; ++i) {
    const int b = half + 2 * i;
    float sq = 0.f;
    if (b < p.B) {
      float x = ldg_cg(p.X + ((size_t)l * p.B + b) * p.d + row);
      for (int g = 0; g < p.Hkv; ++g) x += ldg_cg(p.opart + (((size_t)l * p.Hkv + g) * p.B + b) * p.d + row);
      for (int j = 0; j < p.topk; ++j) x += ldg_cg(p.Y + (((size_t)l * p.B + b) * p.topk + j) * p.d + row);
      p.X[((size_t)(l + 1) * p.B + b) * p.d + row] = x;
      sq = x * x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if (lane == 0) red[warp * 4 + i] = sq;
  }
  bar_sync_consumers();
  if (tid < p.B) {
    const int b = tid, hf = b & 1, i = b >> 1;
    float s = 0.f;
    for (int w = 0; w < 4; ++w) s += red[(hf * 4 + w) * 4 + i];
    p.SS[((size_t)(l + 1) * p.nrb_d + r) * p.B + b] = s;
  }
  bar_sync_consumers();
  if (tid == 0) {
    __threadfence();
    red_release(p.ctr + C_LR(p, l + 1), 1u);
  }
}

// Signal a fan-in counter; returns true (to all consumer threads) if this CTA was last.
__device__ bool signal_fanin(const Params& p, const Smem& S, int ci, unsigned target) {
  bar_sync_consumers();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atom_add_acq_rel(p.ctr + ci, 1u);
    S.small[1] = (old + 1 == target) ? 1 : 0;
    if (p.trace && old + 1 == target) trace_slots(S)[6] = gtime();
  }
  bar_sync_consumers();
  const bool last = S.small[1] != 0;
  if (last) __threadfence();
  return last;
}
__device__ void signal_plain(const Params& p, int ci, unsigned v) {
  bar_sync_consumers();
  if (threadIdx.x == 0) {
    __threadfence();
    red_release(p.ctr + ci, v);
  }
}

// ============================================================== GEMV tasks
__device__ bool task_gemv(const Params& p, const Smem& S, uint32_t& cseq, const int* T, int ti, int item, int nch) {
  const int op = T[D_OP];
  const int l = T[D_LAYER];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g8 = lane >> 2, c = lane & 3;

  int nrows, klen, wait_ci;
  unsigned wait_t;
  int a_slot = 0, t_idx = 0, ntok = p.B;
  const int* tok_list = nullptr;  // expert path: act_tok row of this active slot (b*16 + j)
  if (op == OP_UP_DRAIN || op == OP_DN_DRAIN) {
    const bool up = op == OP_UP_DRAIN;
    const int per = up ? p.t_up : p.t_dn;
    a_slot = item / per;
    t_idx = item % per;
    nrows = up ? p.r_up : p.r_dn;
    klen = up ? p.d : p.f;
    wait_ci = up ? C_RR(p, l) : C_UP(p, l, a_slot);
    wait_t = up ? 1u : (unsigned)p.t_up;
  } else {
    nrows = T[D_NROWS];
    klen = T[D_KLEN];
    wait_ci = T[D_WAIT_CTR];
    wait_t = (unsigned)T[D_WAIT_TARGET];
  }
  if (!consumer_wait(p, S, wait_ci, wait_t, ti)) {
    drain_chunks(p, S, cseq, nch);
    return false;
  }
  if (op == OP_UP_DRAIN || op == OP_DN_DRAIN) {
    ntok = ldg_cg(p.act_cnt + l * p.maxa + a_slot);
    tok_list = p.act_tok + ((size_t)l * p.maxa + a_slot) * p.B;
  }
  const int nrb = nrows / 16;
  const int ksw = klen / 16 / kConsumerWarps;

  BFrag fr;
  if (op == OP_OPROJ) {
    const int k0 = T[D_K0];
    const uint16_t* o = p.atto + (size_t)l * p.B * p.Hq * p.hd;
    const int HQD = p.Hq * p.hd;
    build_bfrag(fr, ksw, [&](int n, int k) -> uint32_t {
      return n < p.B ? ldg_cg_u32(o + (size_t)n * HQD + k0 + k) : 0u;
    });
  } else if (op == OP_DN_DRAIN) {
    const uint16_t* a = p.aup + ((size_t)l * p.maxa + a_slot) * p.B * p.f;
    build_bfrag(fr, ksw, [&](int n, int k) -> uint32_t {
      return n < ntok ? ldg_cg_u32(a + (size_t)n * p.f + k) : 0u;
    });
  } else {
    // RMSNorm operand: QKV / ROUTER over the batch, UP over the expert's gathered
    // tokens (MOE_GATHER folded into the operand load), LM_HEAD with the final norm
    const int n = lane >> 2;
    int b = -1;
    if (op == OP_UP_DRAIN) {
      if (n < ntok) b = ldg_cg(tok_list + n) >> 4;
    } else if (n < p.B) {
      b = n;
    }
    const bool last = op == OP_LMHEAD;
    build_norm_bfrag(p, fr, ksw, last ? p.L : l, last ? p.final_norm : p.attn_norm + (size_t)l * p.d, b);
  }

  float v[4];
  bool ran;
  switch (nrb) {
    case 1: ran = gemv_run<1>(p, S, cseq, nch, ksw, fr, v); break;
    case 2: ran = gemv_run<2>(p, S, cseq, nch, ksw, fr, v); break;
    case 4: ran = gemv_run<4>(p, S, cseq, nch, ksw, fr, v); break;
    default: ran = gemv_run<8>(p, S, cseq, nch, ksw, fr, v); break;
  }
  if (!ran) return false;

  // ---- epilogue: thread (warp = row block, lane) owns rows 16w+g8, 16w+g8+8, tokens 2c, 2c+1
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
        const double inv = rot ? exp(-2.0 * (double)d1 / (double)p.hd * log((double)p.theta)) : 0.0;
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          if (n >= p.B) continue;
          const float x1 = v[e], x2 = v[2 + e];
          const int pos = p.seq_lens[n];
          float y1 = x1, y2 = x2;
          if (rot) {
            double sn, cs;
            sincos((double)pos * inv, &sn, &cs);
            const float fc = (float)cs, fs = (float)sn;
            y1 = x1 * fc - x2 * fs;
            y2 = x2 * fc + x1 * fs;
          }
          if (seg < p.gs) {
            uint16_t* q = p.Q + ((size_t)l * p.B + n) * p.Hq * p.hd + (size_t)(p.gs * g + seg) * p.hd;
            q[d1] = to_bf16(y1);
            q[d2] = to_bf16(y2);
          } else {
            const int pg = checked_page(p, n, pos / 16, ti);
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
          float* out = p.rlog + ((size_t)l * p.B + n) * p.E;
          if (r0 < p.E) out[r0] = v[e];
          if (r0 + 8 < p.E) out[r0 + 8] = v[2 + e];
        }
        break;
      }
      case OP_OPROJ: {
        const int g = T[D_AUX];
        const int r0 = T[D_ROW0] + rlo;
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          if (n >= p.B) continue;
          float* out = p.opart + (((size_t)l * p.Hkv + g) * p.B + n) * p.d;
          out[r0] = v[e];
          out[r0 + 8] = v[2 + e];
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
        break;
      }
      case OP_UP_DRAIN: {
        const int frow = t_idx * (p.r_up / 2) + warp * 8 + g8;
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          if (n >= ntok) continue;
          const float gt = v[e], u = v[2 + e];
          const float a = gt / (1.f + __expf(-gt)) * u;
          p.aup[(((size_t)l * p.maxa + a_slot) * p.B + n) * p.f + frow] = to_bf16(a);
        }
        break;
      }
      case OP_DN_DRAIN: {
        const int r0 = t_idx * p.r_dn + rlo;
        for (int e = 0; e < 2; ++e) {
          const int n = 2 * c + e;
          if (n >= ntok) continue;
          const int pk = ldg_cg(tok_list + n);
          const int b = pk >> 4, jj = pk & 15;
          const float w = ldg_cg(p.rw + ((size_t)l * p.B + b) * p.topk + jj);
          float* out = p.Y + (((size_t)l * p.B + b) * p.topk + jj) * p.d;
          out[r0] = w * v[e];
          out[r0 + 8] = w * v[2 + e];
        }
        break;
      }
      default:
        break;
    }
  }

  // ---- signal
  switch (op) {
    case OP_QKV:
      signal_plain(p, T[D_SIG_CTR], 1u);
      break;
    case OP_ROUTER:
      if (signal_fanin(p, S, T[D_SIG_CTR], (unsigned)T[D_SIG_TARGET])) route_step(p, S, l);
      break;
    case OP_UP_DRAIN:
      signal_plain(p, C_UP(p, l, a_slot), 1u);
      break;
    case OP_OPROJ: {
      const int r = T[D_ROW0] / kRowBlock;
      if (signal_fanin(p, S, C_RB(p, l, r), (unsigned)p.rb_target)) residual_step(p, S, l, r);
      break;
    }
    case OP_DN_DRAIN: {
      const int r = (t_idx * p.r_dn) / kRowBlock;
      if (signal_fanin(p, S, C_RB(p, l, r), (unsigned)p.rb_target)) residual_step(p, S, l, r);
      break;
    }
    default:
      break;
  }
  bar_sync_consumers();
  return true;
}

// ============================================================== attention
// Address of the 16-byte chunk `ch` (8 dims) of key row `key` inside a page of the
// stage, laid out by the tensor-map copy with 128-byte (hd >= 64) or 64-byte (hd = 32)
// swizzle: boxes of 16 keys x min(hd, 64) dims.
template <int HD>
__device__ __forceinline__ uint32_t kv_addr(uint32_t page_base, int key, int ch) {
  constexpr int kInner = HD < 64 ? HD : 64;
  constexpr int kRowB = kInner * 2;
  constexpr int kCpr = kRowB / 16;
  constexpr int kBoxB = 16 * kRowB;
  const int box = ch / kCpr, q = ch % kCpr;
  const int swz = (kRowB == 128) ? (key & 7) : ((key >> 1) & 3);
  return page_base + box * kBoxB + key * kRowB + ((q ^ swz) << 4);
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
      qa[ks][0] = (g8 < gs) ? ldg_cg_u32(q + g8 * HD + 16 * ks + 2 * c) : 0u;
      qa[ks][1] = (g8 < gs) ? ldg_cg_u32(q + g8 * HD + 16 * ks + 8 + 2 * c) : 0u;
    }
  }
  float m_run = -INFINITY, l_run = 0.f;
  float oacc[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t) oacc[t][0] = oacc[t][1] = 0.f;

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
    release_stage(S, cseq);
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
template <int HD>
__device__ void attention_combine(const Params& p, int l, int b, int g, int ns) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gs = p.gs;
  const size_t stride = (size_t)gs * (HD + 2);
  const float* base = p.attp + ((size_t)l * p.Hkv * p.B * p.max_items_bg + (size_t)(g * p.B + b) * p.max_items_bg) * stride;
  for (int h = warp; h < gs; h += kConsumerWarps) {
    float M = -INFINITY;
    for (int s = lane; s <= ns; s += 32) M = fmaxf(M, ldg_cg(base + s * stride + gs * HD + h));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Ls = 0.f;
    for (int s = lane; s <= ns; s += 32) {
      const float m = ldg_cg(base + s * stride + gs * HD + h);
      Ls += ldg_cg(base + s * stride + gs * HD + gs + h) * exp2f(m - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    float acc[HD / 32];
#pragma unroll
    for (int i = 0; i < HD / 32; ++i) acc[i] = 0.f;
#pragma unroll 4
    for (int s = 0; s <= ns; ++s) {
      const float wgt = exp2f(ldg_cg(base + s * stride + gs * HD + h) - M);
#pragma unroll
      for (int i = 0; i < HD / 32; ++i) acc[i] += wgt * ldg_cg(base + s * stride + h * HD + lane + 32 * i);
    }
    const float inv = 1.f / Ls;
    uint16_t* o = p.atto + ((size_t)l * p.B + b) * p.Hq * HD + (size_t)(gs * g + h) * HD;
#pragma unroll
    for (int i = 0; i < HD / 32; ++i) o[lane + 32 * i] = to_bf16(acc[i] * inv);
  }
}

template <int HD>
__device__ bool task_attention(const Params& p, const Smem& S, uint32_t& cseq, int l, int item, int nch, int ti) {
  const AttItem it = att_decode(p, l, item);
  if (!consumer_wait(p, S, C_QKVG(p, l, it.g), (unsigned)p.qkv_tpg, ti)) {
    drain_chunks(p, S, cseq, nch);
    return false;
  }
  if (it.s < it.ns) {
    if (!attention_split<HD>(p, S, cseq, l, it)) return false;
  } else {
    attention_self<HD>(p, l, it, ti);
  }
  if (signal_fanin(p, S, C_ATT(p, l, it.b, it.g), (unsigned)(it.ns + 1))) {
    attention_combine<HD>(p, l, it.b, it.g, it.ns);
    signal_plain(p, C_OG(p, l, it.g), 1u);
  }
  bar_sync_consumers();
  return true;
}

// ============================================================== embed
__device__ void task_embed(const Params& p, const Smem& S, int ti) {
  const int tid = threadIdx.x;
  for (int i = tid; i < p.B * p.d; i += kConsumerThreads) {
    const int b = i / p.d, k = i % p.d;
    int t = p.tokens[b];
    if (t < 0 || t >= p.V) {
      if (k == 0) raise_err(p, MK_ERR_BAD_TOKEN, ti, -1, t, b);
      t = 0;
    }
    p.X[(size_t)b * p.d + k] = bf16_to_f(p.embed[(size_t)t * p.d + k]);
  }
  bar_sync_consumers();
  for (int i = tid; i < p.B * p.nrb_d; i += kConsumerThreads) {
    const int b = i / p.nrb_d, r = i % p.nrb_d;
    const float* x = p.X + (size_t)b * p.d + r * kRowBlock;
    float s = 0.f;
    for (int k = 0; k < kRowBlock; ++k) s += x[k] * x[k];
    p.SS[(size_t)r * p.B + b] = s;
  }
  signal_plain(p, C_LR(p, 0), (unsigned)p.nrb_d);
  bar_sync_consumers();
}

// ============================================================== consumer loop
__device__ void consumer(const Params& p, const Smem& S) {
  uint32_t cseq = 0, mseq = 0;
  bool skip = false;
  while (true) {
    // Thread 0 takes the mailbox entry and the abort flag; every consumer thread
    // then follows the same path, so the named barriers stay matched.
    const uint32_t slot = mseq % kMbox;
    if (threadIdx.x == 0) {
      const bool got = mbar_wait(S.mfull(slot), (mseq / kMbox) & 1u, 16 * p.timeout_ns);
      if (!got) raise_err(p, MK_ERR_TIMEOUT, -5, -1, (int)mseq, 0);
      S.small[3] = got ? 1 : 0;
      S.small[4] = aborted(p) ? 1 : 0;
    }
    bar_sync_consumers();
    const bool got = S.small[3] != 0;
    const bool abort_now = S.small[4] != 0;
    const int4 ent = got ? S.mbox[slot] : make_int4(-1, 0, 0, 0);
    bar_sync_consumers();
    if (got && threadIdx.x == 0) mbar_arrive(S.mempty(slot));
    ++mseq;
    if (ent.x < 0) break;
    const int* T = p.tasks + ent.x * kDescInts;
    const int nch = ent.z;
    if (p.trace && threadIdx.x == 0) {
      unsigned long long* t = trace_slots(S);
      t[0] = gtime(); t[1] = t[2] = t[3] = t[6] = 0ull;
    }
    if (abort_now) skip = true;
    if (skip) {
      if (!drain_chunks(p, S, cseq, nch)) break;
      continue;
    }
    bool ok = true;
    switch (T[D_OP]) {
      case OP_EMBED:
        task_embed(p, S, ent.x);
        break;
      case OP_ATT_DRAIN:
        if (p.hd == 128) ok = task_attention<128>(p, S, cseq, T[D_LAYER], ent.y, nch, ent.x);
        else if (p.hd == 64) ok = task_attention<64>(p, S, cseq, T[D_LAYER], ent.y, nch, ent.x);
        else ok = task_attention<32>(p, S, cseq, T[D_LAYER], ent.y, nch, ent.x);
        break;
      default:
        ok = task_gemv(p, S, cseq, T, ent.x, ent.y, nch);
        break;
    }
    if (!ok) skip = true;
    trace_emit(p, S, T[D_OP], T[D_LAYER], ent.y);
  }
}

// ============================================================== the kernel
__global__ void __launch_bounds__(kThreads, 1)
    mk_megakernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  const Smem S = carve_smem(smem_raw);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(S.full(s), 1);
      mbar_init(S.empty(s), kConsumerWarps);
    }
    for (int m = 0; m < kMbox; ++m) {
      mbar_init(S.mfull(m), 1);
      mbar_init(S.mempty(m), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if (warp == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) producer(p, S, &tmK, &tmV);
  } else {
    consumer(p, S);
  }
  __syncthreads();
  // last CTA out resets the counters and queues for the next launch
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atom_add_acq_rel(p.ctr + p.c_done, 1u);
    S.small[2] = (old == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (S.small[2]) {
    __threadfence();
    if (p.do_reset) {
      for (int i = threadIdx.x; i < p.n_ctr; i += blockDim.x)
        if (i != p.c_done) p.ctr[i] = 0u;
      for (int i = threadIdx.x; i < p.n_queues; i += blockDim.x) { p.qhead[i] = 0; p.qcount[i] = 0; }
      if (!p.fixed)
        for (int b = threadIdx.x; b < p.B; b += blockDim.x) p.seq_lens[b] += 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      p.ctr[p.c_done] = 0u;
      __threadfence();
    }
  }
}

// ============================================================== weight packer
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

__global__ void mk_convert_kernel(float* __restrict__ dst, const uint16_t* __restrict__ src, long long n) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = __uint_as_float((uint32_t)src[i] << 16);
}

}  // namespace mk

// ============================================================== host-side launchers
namespace mk {

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

cudaError_t launch_convert(float* dst, const void* src, long long n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  mk_convert_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(dst, (const uint16_t*)src, n);
  return cudaGetLastError();
}

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
