// Device primitives for the megakernel: shared-memory carving, mbarriers, bulk and
// tensor-map copies, global acquire/release counters, MMA and ldmatrix wrappers.
// Written for sm_103a; only documented PTX forms are used.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "mk.h"
#include "mk_internal.h"

namespace mk {

// ---------------------------------------------------------------- smem layout
struct Smem {
  uint32_t ring;      // shared address of stage 0 (1024-aligned)
  uint8_t* ring_g;    // generic pointer of stage 0
  float* scratch;     // kScratchBytes
  uint32_t scratch_s;
  int* small;         // kSmallBytes
  uint32_t bars;      // full[kStages], empty[kStages], mfull[kMbox], mempty[kMbox], sfull[kSq], sempty[kSq]
  int4* mbox;        // [kMbox][4] task entries
  int2* sq;           // signal requests [kSq]

  __device__ __forceinline__ uint32_t full(uint32_t s) const { return bars + 8u * s; }
  __device__ __forceinline__ uint32_t empty(uint32_t s) const { return bars + 8u * (kStages + s); }
  __device__ __forceinline__ uint32_t mfull(uint32_t m) const { return bars + 8u * (2 * kStages + m); }
  __device__ __forceinline__ uint32_t mempty(uint32_t m) const {
    return bars + 8u * (2 * kStages + kMbox + m);
  }
  __device__ __forceinline__ uint32_t sfull(uint32_t q) const { return bars + 8u * (2 * kStages + 2 * kMbox + q); }
  __device__ __forceinline__ uint32_t sempty(uint32_t q) const {
    return bars + 8u * (2 * kStages + 2 * kMbox + kSq + q);
  }
  // completion of the tensor-core MMAs of a weight chunk (two, alternating)
  __device__ __forceinline__ uint32_t mmadone(uint32_t i) const {
    return bars + 8u * (2 * kStages + 2 * kMbox + 2 * kSq + i);
  }
  __device__ __forceinline__ uint32_t stage(uint32_t seq) const {
    return ring + (seq % kStages) * (uint32_t)kStageBytes;
  }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ Smem carve_smem(uint8_t* raw) {
  Smem S;
  uint32_t base = smem_u32(raw);
  uint32_t aligned = (base + 1023u) & ~1023u;
  uint8_t* g = raw + (aligned - base);
  S.ring = aligned;
  S.ring_g = g;
  S.scratch = reinterpret_cast<float*>(g + kStages * kStageBytes);
  S.scratch_s = aligned + kStages * kStageBytes;
  S.small = reinterpret_cast<int*>(g + kStages * kStageBytes + kScratchBytes);
  S.bars = aligned + kStages * kStageBytes + kScratchBytes + kSmallBytes;
  S.mbox = reinterpret_cast<int4*>(g + kStages * kStageBytes + kScratchBytes + kSmallBytes +
                                   kBarBytes);
  S.sq = reinterpret_cast<int2*>(S.mbox + 4 * kMbox);
  return S;
}

// ---------------------------------------------------------------- timers
__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive without release semantics: for a consumer handing a ring stage back to the
// producer.  The stage's shared-memory reads have all returned by then (their values
// fed instructions issued earlier), so nothing needs ordering, and the arrive does not
// wait for the warp's outstanding global writes or reductions to be acknowledged.
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// One fp32 atomic add whose old value is not needed (a reduction, no round trip).
__device__ __forceinline__ void red_add_f32(float* dst, float v) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(dst), "f"(v) : "memory");
}
// Deterministic accumulation: x as a 64-bit fixed-point integer with 32 fraction bits
// (|x| < 2^31; x * 2^32 is exact in float, then rounded to the nearest integer), added
// with an integer reduction: the sum of such adds does not depend on their order.
__device__ __forceinline__ void red_add_fx(long long* dst, float v) {
  const long long q = __float2ll_rn(v * 4294967296.f);
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(dst), "l"(q) : "memory");
}
__device__ __forceinline__ float fx_to_f(long long q) { return __ll2float_rn(q) * 2.3283064365386963e-10f; }
// Four consecutive fp32 atomic adds in one 128-bit reduction (16-byte aligned).
__device__ __forceinline__ void red_add_v4(float* dst, float4 v) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false after `limit_ns` without completion.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtime();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(gtime() - t0) > limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- async copies
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}
// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y, int z,
                                            uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}

// ---------------------------------------------------------------- global sync
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Predicated relaxed 64-bit load: `v` keeps its value when `pred` is false.
__device__ __forceinline__ void ld_relaxed_u64_pred(uint64_t& v, const uint64_t* ptr, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q ld.relaxed.gpu.global.u64 %0, [%1];\n\t}"
      : "+l"(v)
      : "l"(ptr), "r"((int)pred)
      : "memory");
}
// OR-reduction barrier of the 256 consumer threads (named barrier 1).
__device__ __forceinline__ bool bar_or_consumers(bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((int)pred)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}
// ---------------------------------------------------------------- tcgen05 (sm_100+)
// Shared-memory matrix descriptor: start address, leading-dimension byte offset (between
// core matrices adjacent in K for a K-major operand) and stride-dimension byte offset
// (between 8-row groups), all >> 4; bits 46-48 = 0b001; no swizzle.
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, both K-major, N, M.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// (whole warp) allocate / free `cols` columns of tensor memory; the base address is
// written to shared memory at `dst`
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(cols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
               ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u) : "memory");
}
// arrive on the mbarrier once every tcgen05.mma issued so far by this thread has completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 lanes x 8 columns of 32 bits (this warp's lane quadrant), without the wait
__device__ __forceinline__ void tmem_ld8_async(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 8 columns of 32 bits (this warp's lane quadrant), then the wait for them
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_volatile(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

__device__ __forceinline__ void bar_sync_consumers() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ float ldg_cg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ int ldg_cg(const int* p) { return __ldcg(p); }
__device__ __forceinline__ uint32_t ldg_cg_u32(const void* p) {
  return __ldcg(reinterpret_cast<const unsigned*>(p));
}
__device__ __forceinline__ float2 ldg_cg_f2(const float* p) {
  return __ldcg(reinterpret_cast<const float2*>(p));
}
// Predicated L2 loads: `v` keeps its value when `pred` is false.  Written as one
// straight run of asm loads so that a whole operand's loads are in flight together.
__device__ __forceinline__ void ldg_cg_pred(uint32_t& v, const void* ptr, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q ld.global.cg.u32 %0, [%1];\n\t}"
      : "+r"(v)
      : "l"(ptr), "r"((int)pred));
}
__device__ __forceinline__ void ldg_cg_pred_i(int& v, const int* ptr, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q ld.global.cg.s32 %0, [%1];\n\t}"
      : "+r"(v)
      : "l"(ptr), "r"((int)pred));
}
__device__ __forceinline__ void ldg_cg_pred(float& v, const float* ptr, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q ld.global.cg.f32 %0, [%1];\n\t}"
      : "+f"(v)
      : "l"(ptr), "r"((int)pred));
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- bf16
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint16_t to_bf16(float x) {
  __nv_bfloat16 v = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&v);
}
__device__ __forceinline__ float bf16_to_f(uint16_t u) {
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// ---------------------------------------------------------------- tensor cores
// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
// FP8 expert weights: fragments of E4M3 codes (one byte per element, in the order of
// the bf16 fragment) widen exactly to f16 and multiply f16 activations.
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
// Four E4M3 codes -> two f16x2 of value * 2^-8, on the integer pipe: each code is
// sign-extended to 16 bits (prmt's sign-replicate selectors), shifted left by 7 so
// that its 4 exponent and 3 mantissa bits land in the f16 exponent and top mantissa
// bits (bias 15 against 7: a factor 2^-8, subnormals included), and masked to keep
// the sign in bit 15.  lo holds codes 0 and 1, hi codes 2 and 3.
__device__ __forceinline__ void e4m3x4_to_f16x2_scaled(uint32_t x, uint32_t& lo, uint32_t& hi) {
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x9180;" : "=r"(a) : "r"(x), "r"(0u));
  asm("prmt.b32 %0, %1, %2, 0xB3A2;" : "=r"(b) : "r"(x), "r"(0u));
  lo = (a << 7) & 0xBF80BF80u;
  hi = (b << 7) & 0xBF80BF80u;
}
// bf16x2 -> f16x2 (round to nearest; exact in f16's normal range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u) {
  const __half2 h = __floats2half2_rn(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

}  // namespace mk
