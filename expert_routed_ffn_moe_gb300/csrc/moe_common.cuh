// Shared device helpers of the sm_103a MoE kernels: status word, bounded
// waits, bf16 packing, warp reductions, and inline-PTX wrappers for mbarrier,
// TMA (cp.async.bulk.tensor) and the 5th-generation tensor core (tcgen05).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "moe.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

// ---------------------------------------------------------------- status word
// Kernels never trap.  A kernel that detects a problem ORs a bit into the
// context's status word and abandons its work; the host reads it back with
// moe_status().
enum : unsigned { kStatusTimeout = 1u, kStatusBounds = 2u };

struct DevCtl {
  unsigned* status;        // device status word
  long long spin_limit;    // nanoseconds a bounded wait polls before giving up
  int stall;               // test hook: 1 = wait once on a barrier nothing signals (see moe_inject_stall)
};

MOE_DEV void raise_status(const DevCtl& c, unsigned bit) { atomicOr(c.status, bit); }

// Bounds checks of the grouping tables' entries where kernels read them (the
// grouped GEMMs' tile list, the combine's slots, the scatter's positions, the
// fused decode kernel's active experts), compiled in with -DMOE_DEBUG_CHECKS:
// a bad entry latches kStatusBounds and is replaced by a valid one, so no
// access leaves its array (the output is then wrong and the status says so).
#ifdef MOE_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// ---------------------------------------------------------------- small math
MOE_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
// The 8 bf16 of a 16-byte chunk (columns 0..7) reordered as 0, 4, 1, 5, 2,
// 6, 3, 7: the column order in which the 4-bit GEMM expands a code word (its
// nibbles i and i + 4 come out as one bf16 pair), so that the A operands of
// that GEMM are stored in the same order and no reordering is needed when the
// weights are expanded (the k-sum does not depend on the order).
MOE_DEV uint4 q4_chunk_order(uint4 v) {
  uint4 r;
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(r.x) : "r"(v.x), "r"(v.z));
  asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(r.y) : "r"(v.x), "r"(v.z));
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(r.z) : "r"(v.y), "r"(v.w));
  asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(r.w) : "r"(v.y), "r"(v.w));
  return r;
}
MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// silu(g) = g / (1 + exp(-g)) and sigmoid(z) = 1 / (1 + exp(-z)) with the
// fast exponential and the fast division (each a few instructions; the IEEE
// division made the gate/up GEMM's epilogue take ~7 us per tile, which small
// batches see in full).  The exponent is clamped so the divisor stays below
// 2^126, where the fast division is defined; errors are ~2^-21 relative, far
// below the bf16 rounding of the results.
MOE_DEV float silu(float g) { return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))); }
MOE_DEV float sigmoid(float z) { return __fdividef(1.0f, 1.0f + __expf(fminf(-z, 80.0f))); }

// ---------------------------------------------------------------- top-k selection
// Order-preserving map of an fp32 value to u32 (NaN taken as -inf).
MOE_DEV uint32_t ordered_key(float v) {
  if (v != v) v = -INFINITY;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
MOE_DEV float key_value(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }

// Compare-exchange of (key, id) pairs into descending key, ascending id.
MOE_DEV void key_cx(uint32_t& ka, int& ea, uint32_t& kb, int& eb) {
  const bool swap = (kb > ka) || (kb == ka && eb < ea);
  const uint32_t k0 = swap ? kb : ka, k1 = swap ? ka : kb;
  const int e0 = swap ? eb : ea, e1 = swap ? ea : eb;
  ka = k0;
  kb = k1;
  ea = e0;
  eb = e1;
}

// The logit of expert e in the warp layout of warp_top_k (lane l holds experts
// l, l + 32, ..., in u[0..7]); every lane may ask for its own e.
MOE_DEV float warp_logit_of(const float (&u)[8], int e) {
  const int src = e & 31, slot = e >> 5;
  float r = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float x = __shfl_sync(0xffffffffu, u[i], src);
    if (i == slot) r = x;
  }
  return r;
}

// Warp-wide top-k of one token's E <= 256 logits, lane l holding the logits of
// experts l, l+32, ..., l+224 in v[0..7] (-inf past E).  Every lane sorts its
// 8 experts; each of the k rounds takes the warp's largest head with one warp
// reduction on a word that packs the value's order key with the expert id, and
// the winning lane pops it.  When that key's truncation leaves the boundary
// between the k-th and (k+1)-th values undecided, the k rounds are redone with
// two warp reductions each on the exact values (value, then the lowest expert
// id among equal values).  Ties always go to the lower expert id.  On return lane j < k holds pick j:
// its expert id, its weight exp(l_j - l_max) / sum over the picks (the softmax
// over all E renormalised over the picks, common denominator cancelled) and its
// rank in ascending expert id.  Returns false if some pick was not a number.
MOE_DEV bool warp_top_k(const float (&v)[8], int E, int k, int lane, int& pick_e, float& pick_w, int& pick_rank) {
  unsigned taken = 0u;  // bit i: this lane's expert lane + 32 i was picked
  int my_e = 0;
  float my_v = 0.f;
  bool done = false;
  if (E <= 256) {
    // One reduction per pick: a 32-bit word packs the order key's top 24 bits
    // with 255 - expert id, so the largest word is the largest value and,
    // among equal words, the lower id.  The picks are the exact top k when the
    // k-th pick's 24-bit key is above every other expert's (the truncation is
    // monotone); otherwise (a near-tie at the boundary, ~3e-4 of tokens) the
    // exact rounds below decide.
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      pk[i] = e < E ? ((ordered_key(v[i]) & 0xFFFFFF00u) | (uint32_t)(255 - e)) : 0u;
    }
#define MOE_PK_CX(a, b)                  \
  {                                      \
    const uint32_t hi = max(pk[a], pk[b]); \
    pk[b] = min(pk[a], pk[b]);           \
    pk[a] = hi;                          \
  }
    MOE_PK_CX(0, 1) MOE_PK_CX(2, 3) MOE_PK_CX(4, 5) MOE_PK_CX(6, 7)
    MOE_PK_CX(0, 2) MOE_PK_CX(1, 3) MOE_PK_CX(4, 6) MOE_PK_CX(5, 7)
    MOE_PK_CX(1, 2) MOE_PK_CX(5, 6)
    MOE_PK_CX(0, 4) MOE_PK_CX(1, 5) MOE_PK_CX(2, 6) MOE_PK_CX(3, 7)
    MOE_PK_CX(2, 4) MOE_PK_CX(3, 5)
    MOE_PK_CX(1, 2) MOE_PK_CX(3, 4) MOE_PK_CX(5, 6)
#undef MOE_PK_CX
    uint32_t mk = 0u;
    for (int r = 0; r < k; ++r) {
      const uint32_t m = __reduce_max_sync(0xffffffffu, pk[0]);
      const int e = 255 - (int)(m & 0xFFu);
      if ((e & 31) == lane) {
        taken |= 1u << (e >> 5);
#pragma unroll
        for (int i = 0; i < 7; ++i) pk[i] = pk[i + 1];
        pk[7] = 0u;
      }
      if (lane == r) my_e = e;
      mk = m;
    }
    const uint32_t mn = k < E ? __reduce_max_sync(0xffffffffu, pk[0]) : 0u;
    done = k >= E || (mk >> 8) > (mn >> 8);
    if (done) {
      my_v = warp_logit_of(v, my_e);
    } else {
      taken = 0u;
      my_e = 0;
    }
  }
  if (!done) {
    uint32_t kk[8];
    int ee[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      ee[i] = e < E ? e : 0x7fffffff;
      kk[i] = e < E ? ordered_key(v[i]) : 0u;
    }
    key_cx(kk[0], ee[0], kk[1], ee[1]); key_cx(kk[2], ee[2], kk[3], ee[3]);
    key_cx(kk[4], ee[4], kk[5], ee[5]); key_cx(kk[6], ee[6], kk[7], ee[7]);
    key_cx(kk[0], ee[0], kk[2], ee[2]); key_cx(kk[1], ee[1], kk[3], ee[3]);
    key_cx(kk[4], ee[4], kk[6], ee[6]); key_cx(kk[5], ee[5], kk[7], ee[7]);
    key_cx(kk[1], ee[1], kk[2], ee[2]); key_cx(kk[5], ee[5], kk[6], ee[6]);
    key_cx(kk[0], ee[0], kk[4], ee[4]); key_cx(kk[1], ee[1], kk[5], ee[5]);
    key_cx(kk[2], ee[2], kk[6], ee[6]); key_cx(kk[3], ee[3], kk[7], ee[7]);
    key_cx(kk[2], ee[2], kk[4], ee[4]); key_cx(kk[3], ee[3], kk[5], ee[5]);
    key_cx(kk[1], ee[1], kk[2], ee[2]); key_cx(kk[3], ee[3], kk[4], ee[4]); key_cx(kk[5], ee[5], kk[6], ee[6]);
    for (int r = 0; r < k; ++r) {
      const uint32_t m = __reduce_max_sync(0xffffffffu, kk[0]);
      const int emin = (int)__reduce_min_sync(0xffffffffu, (unsigned)(kk[0] == m ? ee[0] : 0x7fffffff));
      if (ee[0] == emin) {
        taken |= 1u << (emin >> 5);
#pragma unroll
        for (int i = 0; i < 7; ++i) {
          kk[i] = kk[i + 1];
          ee[i] = ee[i + 1];
        }
        kk[7] = 0u;
        ee[7] = 0x7fffffff;
      }
      if (lane == r) {
        my_e = emin < E ? emin : r;
        my_v = key_value(m);
      }
    }
  }
  const bool finite = !(lane < k && !(my_v == my_v && my_v > -INFINITY));
  // weights: exp(l_j - l_max) / sum over the picks.  The fast exp2-based
  // exponential and reciprocal are accurate to a few 1e-7 relative (the weight
  // check allows 1e-5); with k <= 8 the picks sit in lanes 0..7, so three
  // butterfly steps sum them (measured on one warp: the accurate expf, divide
  // and 5-step sum took ~590 of the ~1800 cycles of a top-8 selection)
  float vmax = lane < k ? my_v : -INFINITY;
  for (int o = k <= 8 ? 4 : 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
  const float ex = lane < k ? __expf(my_v - vmax) : 0.f;
  float den = ex;
  for (int o = k <= 8 ? 4 : 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  // rank by expert id: word[i] bit l <=> expert 32 i + l picked
  unsigned word[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) word[i] = __ballot_sync(0xffffffffu, (taken >> i) & 1u);
  const int wi = my_e >> 5, bi = my_e & 31;
  int rank = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    rank += (i < wi) ? __popc(word[i]) : ((i == wi) ? __popc(word[i] & ((1u << bi) - 1u)) : 0);
  pick_e = my_e;
  pick_w = __fdividef(ex, den);
  pick_rank = rank;
  return __all_sync(0xffffffffu, finite);
}

// Weights of the picks from other logits than the ones that chose them (a
// router bias used only for selection): lane j < k holds pick j's unbiased
// logit lu; returns exp(lu - max) / sum over the k picks.
MOE_DEV float warp_pick_weight(float lu, int k, int lane) {
  float m = lane < k ? lu : -INFINITY;
  for (int o = k <= 8 ? 4 : 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float ex = lane < k ? __expf(lu - m) : 0.f;
  float den = ex;
  for (int o = k <= 8 ? 4 : 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  return __fdividef(ex, den);
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy accesses (TMA, tcgen05.mma) that a barrier hands them to.
MOE_DEV void fence_proxy_async_shared_cta() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

MOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
MOE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
MOE_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
MOE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
MOE_DEV void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
MOE_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Deadline of a bounded wait in SM clock cycles.  The limit is given in
// nanoseconds; 2 cycles per ns matches the 2.07 GHz top clock, so at lower
// clocks a wait may last somewhat longer than the limit, never shorter.
MOE_DEV long long wait_cycles(const DevCtl& c) { return c.spin_limit * 2; }

// Bounded wait: false (and the timeout bit raised) once the barrier has not
// completed within the limit.  The cycle counter is read only every 256 polls
// so that checking the deadline never delays noticing a completed phase.
MOE_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, const DevCtl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64(), lim = wait_cycles(c);
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > lim) break;
  }
  raise_status(c, kStatusTimeout);
  return false;
}

// ---------------------------------------------------------------- TMA
MOE_DEV void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
MOE_DEV void tma_load_2d(void* dst, const CUtensorMap* m, int c0, int c1, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
MOE_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEV uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MOE_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor for a K-major bf16 tile stored with the
// 128-byte swizzle: rows of 128 B (64 elements), 8-row groups 1024 B apart.
MOE_DEV uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3ffffu) >> 4);       // start address
  d |= static_cast<uint64_t>(1) << 16;                       // leading byte offset (unused for SW128 K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                       // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;                       // 128-byte swizzle
  return d;
}
// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B (both K-major),
// fp32 accumulator, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4)                               // D format: f32
         | (1u << 7)                             // A format: bf16
         | (1u << 10)                            // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17) // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);// M / 16
}
MOE_DEV void umma_bf16(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once all previously issued tcgen05.mma of this thread finish.
MOE_DEV void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
MOE_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
MOE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive fp32 columns of this thread's TMEM lane, without waiting:
// the registers are valid only after tmem_ld_wait().
MOE_DEV void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
MOE_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 consecutive fp32 columns of this thread's TMEM lane.
MOE_DEV void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace moe
