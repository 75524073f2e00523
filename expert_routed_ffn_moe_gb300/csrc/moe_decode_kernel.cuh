// Fused decode layer: the whole MoE layer for a handful of tokens in ONE
// cooperative persistent kernel (one block per SM), three phases separated by
// two grid-wide data dependencies.
//
// "Optimizing on-device inference for Apple Silicon", section "Decoding:
// minimize bytes moved per token": at batch 1 throughput is set by the bytes
// read per token; section "Optimizing the single-row weight path": a SIMD group
// cooperates on one output while reading different parts of the weight matrix
// in parallel; section "Reducing intermediate and state traffic": the expert
// input projections are fused with the gated activation and the output
// projection with the routing score and the shared expert; section "Overlapping
// independent GPU work": a barrier only where later work needs an earlier
// result.  Section "Keeping each decode step on the GPU": no host round trip.
//
//   phase A  router logits l[t, e] (fp32 FMA, four experts per pass, each row
//            split over 4 warps and summed in a fixed order), and the shared
//            expert's gate/up GEMV + SwiGLU, which needs no routing (on the
//            last warps, so the selection warps go on to phase B).
//   -- every block waits for all logits --
//   phase B  every block selects the top-k of every token from the logits
//            (one warp per token; same result in every block); groups tokens
//            by expert in shared memory (at batch 1 the selection warp writes
//            the active list itself); streams and runs the routed gate/up
//            GEMV + SwiGLU for its (expert, neuron) units.  Weight rows of
//            phases A-C move through a ring of shared-memory slots filled by
//            TMA bulk copies; the down rows of phase C enter it behind the
//            last gate/up units.
//   -- every block waits for all of h --
//   phase C  one warp per output feature: for the active experts in ascending
//            id (shared expert last) the down-projection row, dotted with each
//            routed token's h, scaled by its routing weight, summed per token
//            in fp32 and written to y.  The shared expert's weight is one,
//            or sigmoid(x_t . g) for a sigmoid-gated shared expert (g = router
//            row E; each block computes it beside its selection).
// h is written in several copies and block b reads copy b mod copies, so that
// no L2 line is read by every SM at once.
//
// The two waits are not barriers: every logit and every h value is published
// as a 64-bit word holding the value and the launch's epoch, and a reader
// polls the words it needs until all carry the current epoch (bounded spin,
// MOE_ERR_TIMEOUT).  Data and readiness travel in one access, so a block
// starts on the logits one L2 round trip after the last of them lands, instead
// of after a barrier's arrive, poll and release and then a separate load.
// (Per-block "h written" flags behind a fence measured slower: the fence waits
// out the block's in-flight traffic.)  Every block publishes the launch's
// epoch (an atomic maximum on a 64-bit counter) as it leaves; the next launch,
// a graph replay included, tags with the one after it.
#pragma once
#include <math.h>

#include <mutex>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kWarps = 16;
constexpr int kRowChunks = 4;                    // warps sharing one router row
constexpr int kSlots = kWarps / kRowChunks;      // router rows per pass
constexpr int kThreads = kWarps * 32;
constexpr int kMaxSlots = 48;                    // TMA ring slots (array bound)
// Ring depth used: measured at batch 1 (d = 2048, 9 active experts), 14 slots
// of 9 KB beat both 12 (too little in flight) and 16..22 (more bytes queued per
// SM only spread the blocks' finishing times further apart).
constexpr int kRingSlots = 14;

MOE_DEV void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}
MOE_DEV unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Values that one block produces and every other block consumes (the router
// logits, the SwiGLU activations h) carry the launch's epoch in the high half
// of the same 64-bit word.  A reader polls the word itself until the tag
// matches, so no separate barrier or flag is needed: the payload and its
// readiness arrive in one single-copy-atomic access.
MOE_DEV void st_tagged(unsigned long long* p, float v, unsigned ep) {
  const unsigned long long w = ((unsigned long long)ep << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// (volatile, so every poll re-reads; no memory clobber, so independent polls
// issue back to back)
MOE_DEV unsigned long long ld_tagged(const unsigned long long* p) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p));
  return w;
}
MOE_DEV void ld_tagged2(const unsigned long long* p, unsigned long long& a, unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p));
}
MOE_DEV unsigned tag_of(unsigned long long w) { return (unsigned)(w >> 32); }
MOE_DEV float value_of(unsigned long long w) { return __uint_as_float((unsigned)w); }

// Dot products over 4 consecutive elements: an 8-byte chunk of bf16 weights
// against one float4 of activations.  A lane takes chunk lane + 32 c, so a
// warp reads 256 contiguous weight bytes and 512 contiguous activation bytes
// per step: no shared-memory bank conflicts on either side.
// Packed fp32 pairs (fma.rn.f32x2: two independent FMAs in one instruction).
MOE_DEV unsigned long long pk2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
MOE_DEV unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
MOE_DEV float sum2(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
MOE_DEV void dot4x2(const uint2 g, const uint2 u, const float4 a, float& gs, float& us) {
  gs = fmaf(bf16_lo(g.x), a.x, gs);
  us = fmaf(bf16_lo(u.x), a.x, us);
  gs = fmaf(bf16_hi(g.x), a.y, gs);
  us = fmaf(bf16_hi(u.x), a.y, us);
  gs = fmaf(bf16_lo(g.y), a.z, gs);
  us = fmaf(bf16_lo(u.y), a.z, us);
  gs = fmaf(bf16_hi(g.y), a.w, gs);
  us = fmaf(bf16_hi(u.y), a.w, us);
}
MOE_DEV float dot4(const uint2 w, const float4 a, float s) {
  s = fmaf(bf16_lo(w.x), a.x, s);
  s = fmaf(bf16_hi(w.x), a.y, s);
  s = fmaf(bf16_lo(w.y), a.z, s);
  return fmaf(bf16_hi(w.y), a.w, s);
}

}  // namespace

struct DecodeArgs {
  Shapes s;
  const void* x;
  const float* wr;
  const float* rb;
  const uint16_t* gate_up;
  const uint16_t* down;
  const uint16_t* shared_w;
  void* y;
  Scratch sc;
  DevCtl ctl;
  unsigned* bar;   // control words: [2..3] the largest epoch published so far (64-bit), [0..1] unused
  // optional prefetch hint: weights the next layer reads first (may be null)
  const float* next_wr;
  const uint16_t* next_shared;
  int ring_slots;     // S: slots of the weight ring in shared memory (2..kMaxSlots)
  int slot_bytes;     // bytes per slot: max(gate + up row, chunk_experts down rows)
  int chunk_experts;  // down-projection rows (one per active expert) per slot
  // 4-bit group-affine weights (s.q4): every row of K weights is 9 K / 16
  // bytes, its code words (8 codes per word, lowest nibble first), then its
  // K / 64 bf16 scales, then its K / 64 bf16 biases
  const uint8_t* sh_down_q4;  // the shared expert's down rows (behind its gate_up rows)
};

// The 64-bit epoch counter of the fused decode kernel inside its control
// words (bytes 8..15; the block of words is 256-byte aligned).
MOE_DEV unsigned long long* epoch_word(unsigned* bar) { return reinterpret_cast<unsigned long long*>(bar + 2); }

MOE_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
MOE_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// An active expert id before its rows are copied: a routed expert (and, for
// down rows, the shared expert E); with MOE_DEBUG_CHECKS anything else latches
// kStatusBounds and reads expert 0 instead.
MOE_DEV int checked_expert(const DecodeArgs& A, int e, bool shared_ok) {
  if (kDebugChecks && (e < 0 || e > A.s.E || (e == A.s.E && !(shared_ok && A.s.has_shared)))) {
    raise_status(A.ctl, kStatusBounds);
    return 0;
  }
  return e;
}

// Start the bulk copies of item q of this block's weight stream into `slot`
// (one thread).  Items q < n_sh are the shared expert's gate/up units
// i = b + q G: its gate row i and up row i, back to back.  The next nu items
// are routed gate/up units u = b + q' G (q' = q - n_sh): the gate and up rows
// of neuron i of active expert a.  Later items are chunks of phase-C rows: for
// output row r = b + j G, the down-projection rows r of active experts
// a0 .. a0 + na - 1, back to back.
MOE_DEV void issue_item(const DecodeArgs& A, int q, int slot, int n_sh, int nu, int nch, int b, int G, int n_act,
                        const int* act_e, uint8_t* ring, uint64_t* full, int* slot_issued) {
  const Shapes& s = A.s;
  uint8_t* dst = ring + (size_t)slot * A.slot_bytes;
  const uint64_t pol = policy_evict_first();
  if (s.q4) {
    // 4-bit items: a gate/up unit is [gate row | up row], a phase-C chunk the
    // rows r of its experts, back to back; each row carries its own scales and
    // biases behind its codes, so one copy moves it
    if (q < n_sh || q - n_sh < nu) {
      const uint32_t row = (uint32_t)s.d / 16 * 9;
      const uint8_t* W;
      int i;
      if (q < n_sh) {
        i = b + q * G;
        W = reinterpret_cast<const uint8_t*>(A.shared_w);
      } else {
        const int u = b + (q - n_sh) * G, a = u / s.I;
        i = u - a * s.I;
        W = reinterpret_cast<const uint8_t*>(A.gate_up) + (size_t)checked_expert(A, act_e[a], false) * 2 * s.I * row;
      }
      mbar_expect_tx(&full[slot], 2 * row);
      bulk_g2s(dst, W + (size_t)i * row, row, &full[slot], pol);
      bulk_g2s(dst + row, W + (size_t)(s.I + i) * row, row, &full[slot], pol);
    } else {
      const int m = q - n_sh - nu, j = m / nch, c = m - j * nch;
      const int r = b + j * G, a0 = c * A.chunk_experts, na = min(A.chunk_experts, n_act - a0);
      const uint32_t row = (uint32_t)s.I / 16 * 9;
      mbar_expect_tx(&full[slot], (uint32_t)na * row);
      for (int qa = 0; qa < na; ++qa) {
        const int e = checked_expert(A, act_e[a0 + qa], true);
        const uint8_t* Wd = (e < s.E) ? reinterpret_cast<const uint8_t*>(A.down) + (size_t)e * s.d * row : A.sh_down_q4;
        bulk_g2s(dst + (size_t)qa * row, Wd + (size_t)r * row, row, &full[slot], pol);
      }
    }
  } else if (q < n_sh) {
    const int i = b + q * G;
    const uint32_t row = (uint32_t)s.d * 2;
    mbar_expect_tx(&full[slot], 2 * row);
    bulk_g2s(dst, A.shared_w + (size_t)i * s.d, row, &full[slot], pol);
    bulk_g2s(dst + row, A.shared_w + (size_t)(s.I + i) * s.d, row, &full[slot], pol);
  } else if ((q -= n_sh) < nu) {
    const int u = b + q * G, a = u / s.I, i = u - a * s.I;
    const uint16_t* W = A.gate_up + (size_t)checked_expert(A, act_e[a], false) * 2 * s.I * s.d;
    const uint32_t row = (uint32_t)s.d * 2;
    mbar_expect_tx(&full[slot], 2 * row);
    bulk_g2s(dst, W + (size_t)i * s.d, row, &full[slot], pol);
    bulk_g2s(dst + row, W + (size_t)(s.I + i) * s.d, row, &full[slot], pol);
  } else {
    const int m = q - nu, j = m / nch, c = m - j * nch;
    const int r = b + j * G, a0 = c * A.chunk_experts, na = min(A.chunk_experts, n_act - a0);
    const uint32_t row = (uint32_t)s.I * 2;
    mbar_expect_tx(&full[slot], (uint32_t)na * row);
    for (int qa = 0; qa < na; ++qa) {
      const int e = checked_expert(A, act_e[a0 + qa], true);
      const uint16_t* Wd = (e < s.E) ? A.down + (size_t)e * s.d * s.I : A.shared_w + (size_t)2 * s.I * s.d;
      bulk_g2s(dst + (size_t)qa * row, Wd + (size_t)r * s.I, row, &full[slot], pol);
    }
  }
  __threadfence_block();
  volatile int* issued = slot_issued + slot;
  *issued = *issued + 1;  // read by other warps' wait_item
}

// Wait until item q of the weight stream has landed in its slot q mod S.  An
// mbarrier's parity names a phase only up to two: a consumer that reached
// item q while the slot still held item q - S in flight would see the parity
// it waits for already flipped.  So the consumer first waits until item q has
// been issued (slot_issued[slot] > q / S); items are issued into a slot only
// after the previous one there was consumed, so from then on the parity is
// unambiguous.  Bounded like every wait (false and MOE_ERR_TIMEOUT latched).
MOE_DEV bool wait_item(uint64_t* full, const int* slot_issued, int q, int S, const DevCtl& c) {
  const int slot = q % S, use = q / S;
  const volatile int* issued = slot_issued + slot;
  if (*issued <= use) {
    const long long t0 = clock64(), lim = wait_cycles(c);
    for (int polls = 1; *issued <= use; ++polls) {
      if (polls >= 256 && clock64() - t0 > lim) {
        raise_status(c, kStatusTimeout);
        return false;
      }
    }
  }
  return mbar_wait(&full[slot], (uint32_t)use & 1u, c);
}

// A slot holds at most one item in flight (the next is issued only after the
// previous one was waited for), so waiting for the parity of the last issued
// item of the slot waits for everything still in flight there.
MOE_DEV void drain_slot(uint64_t* full, const int* slot_issued, int slot, const DevCtl& c) {
  const int m = slot_issued[slot];
  if (m > 0) mbar_wait(&full[slot], (uint32_t)(m - 1) & 1u, c);
}

// Shared-memory layout (bytes from the dynamic base).
struct DecodeSmem {
  size_t big;      // x as fp32 [T][d] in phases A/B, then h as fp32 [pairs][I] in phase C
  size_t total;
};

// With 4-bit weights the region also holds, behind x (or h), the sums of each
// run of 8 consecutive values (one per 32-bit code word): d / 8 floats per
// token (I / 8 per grouped h row).
__host__ __device__ inline size_t decode_big_bytes(const Shapes& s) {
  const size_t pairs = (size_t)s.T * s.k + (s.has_shared ? s.T : 0);
  size_t a = (size_t)s.T * s.d * 4, b = pairs * s.I * 4;
  if (s.q4) {
    a += a / 8;
    b += b / 8;
  }
  return a > b ? a : b;
}

// 1 + q / 16 for the 4-bit code q in bits [4 NIB, 4 NIB + 3] of w, built as an
// fp32 bit pattern (q lands in mantissa bits 19..22): exact, one shift and
// one bitwise operation.
template <int NIB>
MOE_DEV float q4_one_plus(uint32_t w) {
  constexpr int sh = 19 - 4 * NIB;
  const uint32_t v = sh >= 0 ? (w << sh) : (w >> (-sh));
  return __uint_as_float((v & 0x00780000u) | 0x3F800000u);
}
// sum_i (1 + q_i / 16) a_i over the 8 codes of word w and a[0..7] (two
// independent chains, so consecutive FMAs do not wait on each other)
MOE_DEV float q4_dot8(uint32_t w, const float4 a0, const float4 a1) {
  // codes 0..7 against a0.xyzw, a1.xyzw as (even, odd) pairs: two chains of
  // two packed FMAs
  unsigned long long r = ffma2(pk2(q4_one_plus<0>(w), q4_one_plus<1>(w)), pk2(a0.x, a0.y), 0ull);
  unsigned long long t = ffma2(pk2(q4_one_plus<4>(w), q4_one_plus<5>(w)), pk2(a1.x, a1.y), 0ull);
  r = ffma2(pk2(q4_one_plus<2>(w), q4_one_plus<3>(w)), pk2(a0.z, a0.w), r);
  t = ffma2(pk2(q4_one_plus<6>(w), q4_one_plus<7>(w)), pk2(a1.z, a1.w), t);
  return sum2(r) + sum2(t);
}
// One word's share of a 4-bit row dot product: with sum_i (1 + q_i/16) a_i =
// raw and sum_i a_i = as, sum_i (s q_i + b) a_i = 16 s raw + (b - 16 s) as.
MOE_DEV float q4_word(float raw, float as, uint16_t s_bits, uint16_t b_bits, float acc) {
  const float sc = __uint_as_float((uint32_t)s_bits << 16), bi = __uint_as_float((uint32_t)b_bits << 16);
  return fmaf(16.f * sc, raw, fmaf(bi - 16.f * sc, as, acc));
}
// Gate and up dot products of one 4-bit unit (gate row, then up row, each
// [codes | scales | biases]) against one token row: lane takes code words
// lane + 32 c (NW per lane); x fp32 [d] and its 8-sums xs [d / 8].
template <int NW>
MOE_DEV void q4_unit_dot(const uint8_t* slot, int d, const float* x, const float* xs, int lane, float& g, float& u) {
  const uint32_t* gc = reinterpret_cast<const uint32_t*>(slot);
  const uint32_t* uc = reinterpret_cast<const uint32_t*>(slot + d / 16 * 9);
  const uint16_t* gp = reinterpret_cast<const uint16_t*>(slot + d / 2);
  const uint16_t* up = reinterpret_cast<const uint16_t*>(slot + d / 16 * 9 + d / 2);
  const int ng = d / 64;
  // two words per step, not fully unrolled: the fully unrolled dot of two
  // phases made the kernel stall on instruction fetch
#pragma unroll 2
  for (int c = 0; c < NW; ++c) {
    const int w = lane + 32 * c, grp = w >> 3;
    const float4 a0 = reinterpret_cast<const float4*>(x)[2 * w], a1 = reinterpret_cast<const float4*>(x)[2 * w + 1];
    const float as = xs[w];
    g = q4_word(q4_dot8(gc[w], a0, a1), as, gp[grp], gp[ng + grp], g);
    u = q4_word(q4_dot8(uc[w], a0, a1), as, up[grp], up[ng + grp], u);
  }
}
// One 4-bit down row (I codes, NW words per lane) against one h row and its 8-sums.
template <int NW>
MOE_DEV float q4_row_dot(const uint32_t* codes, const uint16_t* params, int I, const float* h, const float* hs,
                         int lane) {
  const int ng = I / 64;
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < NW; ++c) {
    const int w = lane + 32 * c, grp = w >> 3;
    const float4 a0 = reinterpret_cast<const float4*>(h)[2 * w], a1 = reinterpret_cast<const float4*>(h)[2 * w + 1];
    acc = q4_word(q4_dot8(codes[w], a0, a1), hs[w], params[grp], params[ng + grp], acc);
  }
  return acc;
}
// The 8-sums of n consecutive runs of 8 floats (block-wide).
MOE_DEV void sums_of_8(const float* v, float* out, int n, int tid, int nthreads) {
  for (int i = tid; i < n; i += nthreads) {
    const float4 a = reinterpret_cast<const float4*>(v)[2 * i], b = reinterpret_cast<const float4*>(v)[2 * i + 1];
    out[i] = ((a.x + a.y) + (a.z + a.w)) + ((b.x + b.y) + (b.z + b.w));
  }
}

// MAXT: compile-time bound on T (1, 2, 4, 8 or 16): the per-token loops unroll over it, and the
// batch-1 kernel keeps one accumulator per lane.
template <int NCH, int NCI, bool XBF16, int MAXT, bool Q4>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(const DecodeArgs A) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const Shapes& s = A.s;
  const Scratch& sc = A.sc;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int G = gridDim.x, b = blockIdx.x;
  const int tk = s.T * s.k;
  const size_t pairs = (size_t)tk + (s.has_shared ? s.T : 0);
  const size_t hrep = pairs * s.I;  // floats per copy of h

  float* big = reinterpret_cast<float*>(dsm);  // x as fp32 [T][d] (phases A, B), then h [pairs][I] (phase C)
  __shared__ float rpart[kSlots][kRowChunks][MAXT];  // router partial sums [slot][chunk][token]
  __shared__ int sel_e[MAXT][kMaxTopK];         // picks per token, ascending expert id
  __shared__ float sel_w[MAXT][kMaxTopK];       // their weights
  __shared__ int act_e[kMaxExperts + 1];        // active experts ascending, shared last
  __shared__ unsigned act_m[kMaxExperts + 1];
  __shared__ int act_row[kMaxExperts + 1];      // first grouped h row of each active expert
  __shared__ float act_w[kMaxExperts + 1][MAXT];
  __shared__ float sgate_s[MAXT];               // the shared expert's weight per token
  // grouped h row p -> (active expert, token): phase C walks a chunk's rows (MAXT > 1)
  __shared__ uint16_t pair_a[MAXT > 1 ? MAXT * (kMaxTopK + 1) : 1];
  __shared__ uint8_t pair_t[MAXT > 1 ? MAXT * (kMaxTopK + 1) : 1];
  __shared__ int n_act_s, flag_s;
  __shared__ unsigned ep_s;  // this launch's epoch: the tag of every value it publishes
  __shared__ unsigned long long ep64_s;  // the same epoch as a 64-bit count (never wraps)
  __shared__ int warp_tot[kWarps];
  __shared__ __align__(8) uint64_t full[kMaxSlots];  // ring slot filled (TMA transaction count)
  __shared__ int slot_issued[kMaxSlots];             // items issued into each slot so far
  uint8_t* const ring = dsm + decode_big_bytes(s);   // A.ring_slots x A.slot_bytes
  int n_items = 0;                                   // this block's weight items (phases B and C)
  const int n_sh = s.has_shared ? ((s.I > b) ? (s.I - b + G - 1) / G : 0) : 0;  // shared-expert units

  if (tid == 0) {
    flag_s = 1;
    for (int i = 0; i < A.ring_slots; ++i) {
      mbar_init(&full[i], 1);
      slot_issued[i] = 0;
    }
    fence_mbar_init();
  }
  unsigned long long* const dlog = reinterpret_cast<unsigned long long*>(sc.dec_logits);
  unsigned long long* const dh = reinterpret_cast<unsigned long long*>(sc.dec_h);
  bool ok = true;
  // ---------------------------------------------------------------- phase A
  // router logits, and the shared expert's gate/up GEMV (it needs no routing)
  {
    // a warp covers a d/4-wide quarter of a router row; its lane takes the
    // float4 columns lane + 32 i of that quarter (coalesced weight loads,
    // conflict-free x reads)
    constexpr int kPer4 = NCH / 2;  // = d / 512: float4 per lane
    const int chunk = s.d / kRowChunks;
    const int slot = warp / kRowChunks, cw = warp % kRowChunks;
    const int col0 = cw * chunk;
    float4 rw[kPer4];
    {
      const int e = b + slot * G;
      if (e < s.E) {
        const float4* wrow = reinterpret_cast<const float4*>(A.wr + (size_t)e * s.d + col0) + lane;
#pragma unroll
        for (int i = 0; i < kPer4; ++i) rw[i] = __ldg(wrow + 32 * i);
      }
    }
    // this block's shared-expert neurons i = b + q G (items q < n_sh of the
    // weight stream) start streaming into the ring now: they need no routing
    if (tid == 0) {
      for (int q = 0; q < n_sh && q < A.ring_slots; ++q)
        issue_item(A, q, q, n_sh, 0, 1, b, G, 0, nullptr, ring, full, slot_issued);
      if (s.shared_gate) prefetch_l2(A.wr + (size_t)s.E * s.d, (uint32_t)s.d * 4u);  // the gate row, for phase B
    }
    // Everything above reads weights only.  Launched with programmatic stream
    // serialization, this block may have started while the previous kernel
    // on the stream is still running: wait for it before touching x or any
    // scratch (a no-op for a normal launch).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
      // the largest epoch any earlier launch used, + 1; the tag is its low 32
      // bits, skipping 0 (zeroed scratch must never look ready)
      unsigned long long e = ld_relaxed64(epoch_word(A.bar)) + 1ull;
      if ((unsigned)e == 0u) ++e;
      ep64_s = e;
      ep_s = (unsigned)e;
    }
    const int nx = s.T * s.d;
    if (XBF16) {
      const uint32_t* xb = static_cast<const uint32_t*>(A.x);
      for (int i = tid; i < nx / 2; i += kThreads) {
        const uint32_t v = __ldg(xb + i);
        big[2 * i] = bf16_lo(v);
        big[2 * i + 1] = bf16_hi(v);
      }
    } else {
      const float2* xf = static_cast<const float2*>(A.x);
      for (int i = tid; i < nx / 2; i += kThreads) reinterpret_cast<float2*>(big)[i] = __ldg(xf + i);
    }
    __syncthreads();
    if (Q4) {  // the 8-sums of x for the 4-bit dot products (behind x)
      sums_of_8(big, big + nx, nx / 8, tid, kThreads);
      __syncthreads();
    }
    int n_e0 = 0;
    for (int e0 = b; e0 < s.E; e0 += kSlots * G) ++n_e0;
    for (int rep = 0; rep < n_e0; ++rep) {
      const int e = b + rep * kSlots * G + slot * G;
      if (rep > 0 && e < s.E) {
        const float4* wrow = reinterpret_cast<const float4*>(A.wr + (size_t)e * s.d + col0) + lane;
#pragma unroll
        for (int i = 0; i < kPer4; ++i) rw[i] = __ldg(wrow + 32 * i);
      }
      if (e < s.E) {
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
          if (t < s.T) {
            const float4* xr = reinterpret_cast<const float4*>(big + (size_t)t * s.d + col0) + lane;
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kPer4; ++i) {
              const float4 xv = xr[32 * i];
              acc = fmaf(rw[i].x, xv.x, acc);
              acc = fmaf(rw[i].y, xv.y, acc);
              acc = fmaf(rw[i].z, xv.z, acc);
              acc = fmaf(rw[i].w, xv.w, acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) rpart[slot][cw][t] = acc;
          }
        }
      }
      __syncthreads();
      // every block reads all logits in phase B: write dec_reps copies so
      // that the reads spread over several L2 lines instead of one hot set
      for (int q = tid; q < kSlots * MAXT * sc.dec_reps; q += kThreads) {
        const int sl = q % kSlots, t = (q / kSlots) % MAXT, r = q / (kSlots * MAXT);
        const int ee = b + rep * kSlots * G + sl * G;
        if (ee < s.E && t < s.T) {
          float l = 0.f;
#pragma unroll
          for (int c = 0; c < kRowChunks; ++c) l += rpart[sl][c][t];
          st_tagged(dlog + ((size_t)r * s.T + t) * s.E + ee, l, ep_s);
        }
      }
      __syncthreads();
    }
  }

  // ---------------------------------------------------------------- phase B
  // selection, identical in every block (same logits, same arithmetic); the
  // logits are polled until every one carries this launch's tag
  {
    const unsigned long long* logits = dlog + (size_t)(b % sc.dec_reps) * s.T * s.E;
    // test hook: wait for a tag that no block writes
    const unsigned want = ep_s + (A.ctl.stall ? 1u : 0u);
    for (int t = warp; t < s.T; t += kWarps) {
      // the shared expert's weight: one, or sigmoid(x_t . g) for the gate
      // vector g in router row E (computed while other blocks finish routing)
      float sg = 1.f;
      if (s.shared_gate) {
        const float4* g4 = reinterpret_cast<const float4*>(A.wr + (size_t)s.E * s.d);
        const float4* xr = reinterpret_cast<const float4*>(big + (size_t)t * s.d);
        float acc = 0.f;
        for (int c = lane; c < s.d / 4; c += 32) {
          const float4 gv = __ldg(g4 + c), xv = xr[c];
          acc = fmaf(xv.x, gv.x, acc);
          acc = fmaf(xv.y, gv.y, acc);
          acc = fmaf(xv.z, gv.z, acc);
          acc = fmaf(xv.w, gv.w, acc);
        }
        sg = sigmoid(warp_sum(acc));
      }
      if (lane == 0) sgate_s[t] = sg;
      float v[8], u[8];  // logits with and without the router bias
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (A.rb && lane + 32 * i < s.E) ? __ldg(A.rb + lane + 32 * i) : 0.f;
      const long long t0 = clock64(), lim = wait_cycles(A.ctl);
      bool late = false;
      for (int polls = 1;; ++polls) {
        // all eight words are loaded before any is tested: a load that waited
        // on the previous one's tag would make the poll eight round trips long
        unsigned long long w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = (lane + 32 * i < s.E) ? ld_tagged(logits + (size_t)t * s.E + lane + 32 * i) : 0ull;
        bool ready = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) ready = ready && (lane + 32 * i >= s.E || tag_of(w[i]) == want);
        if (__all_sync(0xffffffffu, ready)) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            u[i] = (lane + 32 * i < s.E) ? value_of(w[i]) : -INFINITY;
            v[i] = (lane + 32 * i < s.E) ? u[i] + v[i] : -INFINITY;
          }
          break;
        }
        if (polls >= 256 && __any_sync(0xffffffffu, clock64() - t0 > lim)) {
          late = true;
          break;
        }
      }
      if (late) {
        if (lane == 0) {
          raise_status(A.ctl, kStatusTimeout);
          flag_s = 0;
        }
        continue;
      }
      int pe, rank;
      float pw;
      if (!warp_top_k(v, s.E, s.k, lane, pe, pw, rank) && lane == 0) raise_status(A.ctl, kStatusBounds);
      if (s.bias_sel) pw = warp_pick_weight(warp_logit_of(u, pe), s.k, lane);
      if (lane < s.k) {
        sel_e[t][rank] = pe;
        sel_w[t][rank] = pw;
        if (b == 0) {
          sc.idx[(size_t)t * s.k + rank] = pe;
          sc.w[(size_t)t * s.k + rank] = pw;
        }
        if (MAXT == 1) {
          // batch 1: the active experts are the picks in ascending id (rank
          // order), grouped h row = rank, then the shared expert (row k)
          act_e[rank] = pe;
          act_m[rank] = 1u;
          act_row[rank] = rank;
          act_w[rank][0] = pw;
        }
      }
      if (MAXT == 1 && lane == 0) {
        if (s.has_shared) {
          act_e[s.k] = s.E;
          act_m[s.k] = 1u;
          act_row[s.k] = s.k;
          act_w[s.k][0] = sg;
        }
        n_act_s = s.k + (s.has_shared ? 1 : 0);
      }
    }
  }
  __syncthreads();
  ok = flag_s != 0;
  if (ok) {
    if (MAXT > 1) {
    // group tokens by expert: masks, active list (ascending), grouped h rows
    unsigned m = 0u;
    if (tid < s.E) {
      for (int t = 0; t < s.T; ++t)
        for (int j = 0; j < s.k; ++j)
          if (sel_e[t][j] == tid) m |= 1u << t;
    }
    {
      const int flag = (tid < s.E && m) ? 1 : 0, cnt = (tid < s.E) ? __popc(m) : 0;
      int v = (flag << 16) | cnt, incl = v;  // flag count in the high half, rows in the low half
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (lane == 31) warp_tot[warp] = incl;
      __syncthreads();
      int base = 0;
      for (int i = 0; i < warp; ++i) base += warp_tot[i];
      const int excl = base + incl - v;
      if (b == 0 && sc.counts != nullptr && tid < s.E) {
        // the layer's grouping tables, for moe_last_routing: block 0 writes its
        // in-shared-memory grouping out once (counts, exclusive offsets, the
        // stable permutation and each pick's position in it)
        sc.counts[tid] = cnt;
        sc.offsets[tid] = excl & 0xffff;
        for (int t = 0, i = 0; t < s.T; ++t)
          if ((m >> t) & 1u) {
            const int p = (excl & 0xffff) + i++;
            sc.perm[p] = t;
            for (int j = 0; j < s.k; ++j)
              if (sel_e[t][j] == tid) sc.slot[(size_t)t * s.k + j] = p;
          }
        if (tid == 0) sc.offsets[s.E] = tk;
      }
      if (flag) {
        const int pos = excl >> 16;
        act_e[pos] = tid;
        act_m[pos] = m;
        act_row[pos] = excl & 0xffff;
        for (int t = 0, i = 0; t < MAXT; ++t)
          if ((m >> t) & 1u) {
            pair_a[(excl & 0xffff) + i] = (uint16_t)pos;
            pair_t[(excl & 0xffff) + i] = (uint8_t)t;
            ++i;
          }
        for (int t = 0; t < MAXT; ++t) {
          float wt = 0.f;
          if (t < s.T)
            for (int j = 0; j < s.k; ++j)
              if (sel_e[t][j] == tid) wt = sel_w[t][j];
          act_w[pos][t] = wt;
        }
      }
      if (tid == kThreads - 1) {
        int all = 0;
        for (int i = 0; i < kWarps; ++i) all += warp_tot[i];
        const int n_routed = all >> 16;
        if (s.has_shared) {
          act_e[n_routed] = s.E;
          act_m[n_routed] = (s.T >= 32) ? 0xffffffffu : ((1u << s.T) - 1u);
          act_row[n_routed] = tk;
          for (int t = 0; t < MAXT; ++t) act_w[n_routed][t] = t < s.T ? sgate_s[t] : 0.f;
          for (int t = 0; t < s.T; ++t) {
            pair_a[tk + t] = (uint16_t)n_routed;
            pair_t[tk + t] = (uint8_t)t;
          }
        }
        n_act_s = n_routed + (s.has_shared ? 1 : 0);
      }
    }
    __syncthreads();
    }
    const int n_act = n_act_s;
    const int n_routed = n_act - (s.has_shared ? 1 : 0);
    const int units = n_routed * s.I;
    // This block's stream of weight items, all moved by TMA bulk copies into a
    // ring of A.ring_slots shared-memory slots: first its gate/up units
    // (u = b + j G: the gate and up rows of one routed neuron), then, per
    // phase-C output row r = b + j G, the down-projection rows of the active
    // experts in chunks of A.chunk_experts.  Slots 0..S-1 are filled now; the
    // warp that consumes item q refills its slot with item q + S, so the
    // copies of phase C's rows start as soon as phase B frees slots.
    const int S = A.ring_slots;
    const int nu = (units > b) ? (units - b + G - 1) / G : 0;
    const int nr = (s.d > b) ? (s.d - b + G - 1) / G : 0;
    const int nch = (n_act + A.chunk_experts - 1) / A.chunk_experts;
    n_items = n_sh + nu + nr * nch;
    // the slots past the shared expert's items are free: fill them (each
    // shared item's slot is refilled by the warp that consumes it, below)
    if (warp == 0) {
      for (int q = n_sh + lane; q < S && q < n_items; q += 32)
        issue_item(A, q, q, n_sh, nu, nch, b, G, n_act, act_e, ring, full, slot_issued);
    }
    // shared-expert gate/up + SwiGLU, from rows that landed during the
    // selection: item q < n_sh goes to warp kWarps - 1 - (q mod kWarps), the
    // last warps, which have one routed unit fewer.  Computed beside the
    // selection, their shared-memory loads took the issue slots of the pipe
    // the selection's warp reductions use, and the selection ran 1.5 us.
    for (int q = kWarps - 1 - warp; q < n_sh; q += kWarps) {
      const int slot = q % S;
      if (!wait_item(full, slot_issued, q, S, A.ctl)) {
        flag_s = 0;
        break;
      }
      const int i = b + q * G;
      const uint2* grow = reinterpret_cast<const uint2*>(ring + (size_t)slot * A.slot_bytes) + lane;
      const uint2* urow = grow + s.d / 4;
      for (int t = 0; t < s.T; ++t) {
        float g = 0.f, up = 0.f;
        if (Q4) {
          q4_unit_dot<NCH>(ring + (size_t)slot * A.slot_bytes, s.d, big + (size_t)t * s.d,
                           big + (size_t)s.T * s.d + (size_t)t * (s.d / 8), lane, g, up);
        } else {
          const float4* xr = reinterpret_cast<const float4*>(big + (size_t)t * s.d) + lane;
#pragma unroll
          for (int c = 0; c < 2 * NCH; ++c) dot4x2(grow[32 * c], urow[32 * c], xr[32 * c], g, up);
        }
        g = warp_sum(g);
        up = warp_sum(up);
        if (lane < sc.dec_hreps) st_tagged(dh + (size_t)lane * hrep + ((size_t)tk + t) * s.I + i, silu(g) * up, ep_s);
      }
      __syncwarp();  // every lane has read the slot
      if (lane == 0 && q + S < n_items) {
        fence_proxy_async_smem();
        issue_item(A, q + S, slot, n_sh, nu, nch, b, G, n_act, act_e, ring, full, slot_issued);
      }
    }
    if (MAXT == 1 && b == 0 && sc.counts != nullptr && tid >= 32 && tid < 32 + s.E) {
      // batch 1: the layer's grouping tables, for moe_last_routing (one row per
      // pick, in ascending expert id); warps 1.. write them while warp 0 issues
      const int e = tid - 32;
      int c = 0, o = 0;
      for (int j = 0; j < s.k; ++j) {
        c += sel_e[0][j] == e;
        o += sel_e[0][j] < e;
      }
      sc.counts[e] = c;
      sc.offsets[e] = o;
      if (e < s.k) {
        sc.perm[e] = 0;
        sc.slot[e] = e;
      }
      if (e == 0) sc.offsets[s.E] = s.k;
    }
    // routed gate/up GEMV + SwiGLU: routed unit j (item n_sh + j) goes to warp j mod kWarps
    for (int j = warp; j < nu; j += kWarps) {
      const int q = n_sh + j, slot = q % S;
      if (!wait_item(full, slot_issued, q, S, A.ctl)) {
        flag_s = 0;
        break;
      }
      const int u = b + j * G;
      const int a = u / s.I, i = u - a * s.I;
      const uint2* grow = reinterpret_cast<const uint2*>(ring + (size_t)slot * A.slot_bytes) + lane;
      const uint2* urow = grow + s.d / 4;
      unsigned mm = act_m[a];
      int row = act_row[a];
      while (mm) {
        const int t = __ffs(mm) - 1;
        mm &= mm - 1u;
        float g = 0.f, up = 0.f;
        if (Q4) {
          q4_unit_dot<NCH>(ring + (size_t)slot * A.slot_bytes, s.d, big + (size_t)t * s.d,
                           big + (size_t)s.T * s.d + (size_t)t * (s.d / 8), lane, g, up);
        } else {
          const float4* xr = reinterpret_cast<const float4*>(big + (size_t)t * s.d) + lane;
#pragma unroll
          for (int c = 0; c < 2 * NCH; ++c) dot4x2(grow[32 * c], urow[32 * c], xr[32 * c], g, up);
        }
        g = warp_sum(g);
        up = warp_sum(up);
        if (lane < sc.dec_hreps) st_tagged(dh + (size_t)lane * hrep + (size_t)row * s.I + i, silu(g) * up, ep_s);
        ++row;
      }
      __syncwarp();  // every lane has read the slot
      if (lane == 0 && q + S < n_items) {
        fence_proxy_async_smem();
        issue_item(A, q + S, slot, n_sh, nu, nch, b, G, n_act, act_e, ring, full, slot_issued);
      }
    }
  }
  __syncthreads();  // every warp is done with x in shared memory
  ok = ok && flag_s != 0;

  // ---------------------------------------------------------------- phase C
  // a dependent launch (the next layer) may be scheduled now; its blocks take
  // an SM as ours leave
  asm volatile("griddepcontrol.launch_dependents;");
  if (ok) {
    {
      // stage this block's copy of h, polling each pair of values until both
      // carry this launch's tag (the last ones land when the slowest block
      // finishes phase B)
      const unsigned long long* src = dh + (size_t)(b % sc.dec_hreps) * hrep;
      float2* dst = reinterpret_cast<float2*>(big);
      const int n2 = (int)(hrep >> 1);
      const unsigned ep = ep_s;
      const long long t0 = clock64(), lim = wait_cycles(A.ctl);
      bool late = false;
      for (int i0 = tid; i0 < n2 && !late; i0 += 8 * kThreads) {
        unsigned long long lo[8], hi[8];
        for (int polls = 1;; ++polls) {
          // the batch is re-read whole until every pair in it is ready, so that
          // the loads stay independent of each other
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (i0 + u * kThreads < n2) ld_tagged2(src + 2 * (i0 + u * kThreads), lo[u], hi[u]);
          bool ready = true;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            ready = ready && (i0 + u * kThreads >= n2 || (tag_of(lo[u]) == ep && tag_of(hi[u]) == ep));
          if (ready) break;
          if (polls >= 256 && clock64() - t0 > lim) {
            late = true;
            break;
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (i0 + u * kThreads < n2) dst[i0 + u * kThreads] = make_float2(value_of(lo[u]), value_of(hi[u]));
      }
      if (late) {
        raise_status(A.ctl, kStatusTimeout);
        flag_s = 0;
      }
    }
    __syncthreads();
    if (Q4) {  // the 8-sums of h for the 4-bit dot products (behind h)
      sums_of_8(big, big + hrep, (int)(hrep / 8), tid, kThreads);
      __syncthreads();
    }
    ok = flag_s != 0;
  }
  if (ok) {
    const int n_act = n_act_s;
    const int n_routed = n_act - (s.has_shared ? 1 : 0);
    const int S = A.ring_slots;
    const int units = n_routed * s.I;
    const int nu = (units > b) ? (units - b + G - 1) / G : 0;
    const int nch = (n_act + A.chunk_experts - 1) / A.chunk_experts;
    // the next layer's router rows and shared expert, if the caller named them:
    // pull them into L2 while this phase is bound by latency, not bandwidth
    // (the last warp: it has no output row when d < kWarps G)
    if (warp == kWarps - 1) {
      // the shared expert's bytes: 3 I d bf16 weights, or 4-bit codes and parameters (27/16 I d bytes)
      const size_t rbytes = (size_t)(s.E + s.shared_gate) * s.d * 4,
                   sbytes = Q4 ? (size_t)27 * s.I * s.d / 16 : (size_t)3 * s.I * s.d * 2;
      const size_t rper = ((rbytes / G) + 4095) & ~size_t(4095), sper = ((sbytes / G) + 4095) & ~size_t(4095);
      if (A.next_wr)
        for (size_t off = rper * b + (size_t)lane * 4096; off < min(rbytes, rper * (b + 1)); off += 32 * 4096)
          prefetch_l2(reinterpret_cast<const uint8_t*>(A.next_wr) + off, (uint32_t)min((size_t)4096, rbytes - off));
      if (A.next_shared)
        for (size_t off = sper * b + (size_t)lane * 4096; off < min(sbytes, sper * (b + 1)); off += 32 * 4096)
          prefetch_l2(reinterpret_cast<const uint8_t*>(A.next_shared) + off,
                      (uint32_t)min((size_t)4096, sbytes - off));
    }
    for (int j = warp;; j += kWarps) {
      const int r = b + j * G;
      if (r >= s.d) break;
      // per-lane partial sums of every token, reduced across the warp once at the end
      float part[MAXT];
#pragma unroll
      for (int t = 0; t < MAXT; ++t) part[t] = 0.f;
      bool fail = false;
      for (int c = 0; c < nch; ++c) {
        const int q = n_sh + nu + j * nch + c, slot = q % S;
        if (!wait_item(full, slot_issued, q, S, A.ctl)) {
          fail = true;
          break;
        }
        const int a0 = c * A.chunk_experts;
        const int na = min(A.chunk_experts, n_act - a0);
        const uint2* base = reinterpret_cast<const uint2*>(ring + (size_t)slot * A.slot_bytes) + lane;
        if (MAXT == 1) {
          // batch 1 (one token per expert, h row act_row[a]): three experts per
          // step with independent partial sums, so the shared-memory loads and
          // FMA chains of different experts overlap (one expert at a time, the
          // loop was latency-bound: ~430 cycles per expert)
          float ps[3] = {0.f, 0.f, 0.f};
          for (int qa0 = 0; qa0 < na; qa0 += 3) {
#pragma unroll
            for (int u = 0; u < 3; ++u) {
              const int qa = qa0 + u;
              if (qa < na) {
                const int a = a0 + qa;
                float d0 = 0.f, d1 = 0.f;
                if (Q4) {
                  const uint8_t* rw = ring + (size_t)slot * A.slot_bytes + (size_t)qa * (s.I / 16 * 9);
                  d0 = q4_row_dot<NCI>(reinterpret_cast<const uint32_t*>(rw),
                                       reinterpret_cast<const uint16_t*>(rw + s.I / 2), s.I,
                                       big + (size_t)act_row[a] * s.I, big + hrep + (size_t)act_row[a] * (s.I / 8),
                                       lane);
                } else {
                  const float4* hr = reinterpret_cast<const float4*>(big + (size_t)act_row[a] * s.I) + lane;
                  const uint2* wr = base + (size_t)qa * (s.I / 4);
#pragma unroll
                  for (int cc = 0; cc < 2 * NCI; cc += 2) {
                    d0 = dot4(wr[32 * cc], hr[32 * cc], d0);
                    d1 = dot4(wr[32 * (cc + 1)], hr[32 * (cc + 1)], d1);
                  }
                }
                ps[u] = fmaf(act_w[a][0], d0 + d1, ps[u]);
              }
            }
          }
          part[0] += (ps[0] + ps[1]) + ps[2];
        }
        if (MAXT > 1) {
          // the chunk's (expert, token) pairs are the contiguous grouped h rows
          // p0 .. p1 - 1 (experts ascending, tokens ascending within one);
          // three pairs per step with independent dot products, so that their
          // shared-memory loads and FMA chains overlap (one expert at a time,
          // token by token, the loop was a chain of dependent latencies)
          const int p0 = act_row[a0];
          const int p1 = (a0 + na < n_act) ? act_row[a0 + na] : (int)pairs;
          for (int p = p0; p < p1; p += 3) {
            float dd[3], ww[3];
            int tt[3];
#pragma unroll
            for (int u = 0; u < 3; ++u) {
              dd[u] = 0.f;
              ww[u] = 0.f;
              tt[u] = -1;
              const int pu = p + u;
              if (pu < p1) {
                const int a = pair_a[pu];
                tt[u] = pair_t[pu];
                ww[u] = act_w[a][tt[u]];
                float d0 = 0.f, d1 = 0.f;
                if (Q4) {
                  const uint8_t* rw = ring + (size_t)slot * A.slot_bytes + (size_t)(a - a0) * (s.I / 16 * 9);
                  d0 = q4_row_dot<NCI>(reinterpret_cast<const uint32_t*>(rw),
                                       reinterpret_cast<const uint16_t*>(rw + s.I / 2), s.I, big + (size_t)pu * s.I,
                                       big + hrep + (size_t)pu * (s.I / 8), lane);
                } else {
                  const uint2* wr = base + (size_t)(a - a0) * (s.I / 4);
                  const float4* hr = reinterpret_cast<const float4*>(big + (size_t)pu * s.I) + lane;
#pragma unroll
                  for (int cc = 0; cc < 2 * NCI; cc += 2) {
                    d0 = dot4(wr[32 * cc], hr[32 * cc], d0);
                    d1 = dot4(wr[32 * (cc + 1)], hr[32 * (cc + 1)], d1);
                  }
                }
                dd[u] = d0 + d1;
              }
            }
            // every token's sum takes a term (zero unless the pair is its own):
            // a conditional update indexed by the pair's token would move
            // part[] to local memory
#pragma unroll
            for (int u = 0; u < 3; ++u) {
              const float v = ww[u] * dd[u];
#pragma unroll
              for (int t = 0; t < MAXT; ++t) part[t] += (tt[u] == t) ? v : 0.f;
            }
          }
        }
        __syncwarp();
        if (lane == 0 && q + S < n_items) {
          fence_proxy_async_smem();
          issue_item(A, q + S, slot, n_sh, nu, nch, b, G, n_act, act_e, ring, full, slot_issued);
        }
      }
      if (fail) {
        flag_s = 0;
        break;
      }
      float mine = 0.f;
#pragma unroll
      for (int t = 0; t < MAXT; ++t) {
        if (t < s.T) {
          const float v = warp_sum(part[t]);
          if (lane == t) mine = v;
        }
      }
      if (lane < s.T) {
        if (XBF16) {
          const __nv_bfloat16 v = __float2bfloat16_rn(mine);
          static_cast<uint16_t*>(A.y)[(size_t)lane * s.d + r] = *reinterpret_cast<const uint16_t*>(&v);
        } else {
          static_cast<float*>(A.y)[(size_t)lane * s.d + r] = mine;
        }
      }
    }
  }
  // a block that gave up may still have bulk copies in flight into its ring:
  // wait (bounded) for every issued item before the shared memory is released
  __syncthreads();
  if (flag_s == 0 && tid < A.ring_slots) drain_slot(full, slot_issued, tid, A.ctl);
  // leave: publish this launch's epoch (the next launch, which starts after
  // this grid completes, tags with one more than the largest epoch published).
  // Every block publishes, with no exit counter: in a run without timeouts no
  // block can leave before every block has read the old epoch, since each
  // first waits for every block's logits, which carry it.  A block that gave
  // up may have left before a late block read the word (which then took
  // epoch + 1); so a block that gave up publishes with an atomic maximum,
  // which no other store can lower.  A block that finished normally saw every
  // block's logits tagged with its own epoch, so in its launch all blocks
  // share one epoch and its plain store writes that same value (and costs no
  // atomic round trip on the common path).  Either way the next launch's
  // epoch exceeds every tag written so far.
  if (tid == 0) {
    if (flag_s == 0)
      atomicMax(epoch_word(A.bar), ep64_s);
    else
      *reinterpret_cast<volatile unsigned long long*>(epoch_word(A.bar)) = ep64_s;
  }
}


template <int NCH, int NCI, int MAXT, bool Q4>
static const void* pick(bool xbf16) {
  return xbf16 ? (const void*)decode_fused_kernel<NCH, NCI, true, MAXT, Q4>
               : (const void*)decode_fused_kernel<NCH, NCI, false, MAXT, Q4>;
}

// The instantiation for a shape (d / 256 = NCH, I / 256 = NCI); Q4 selects
// the 4-bit weight kernels (compiled in their own translation units).
template <int MAXT, bool Q4>
static const void* pick_shape(const Shapes& s) {
  const int nch = s.d / 256, nci = s.I / 256;
  if (nci == 2) {
    if (nch == 2) return pick<2, 2, MAXT, Q4>(s.x_bf16);
    if (nch == 4) return pick<4, 2, MAXT, Q4>(s.x_bf16);
    if (nch == 8) return pick<8, 2, MAXT, Q4>(s.x_bf16);
  } else if (nci == 1) {
    if (nch == 2) return pick<2, 1, MAXT, Q4>(s.x_bf16);
    if (nch == 4) return pick<4, 1, MAXT, Q4>(s.x_bf16);
    if (nch == 8) return pick<8, 1, MAXT, Q4>(s.x_bf16);
  } else if (nci == 4) {
    if (nch == 4) return pick<4, 4, MAXT, Q4>(s.x_bf16);
    if (nch == 8) return pick<8, 4, MAXT, Q4>(s.x_bf16);
  }
  return nullptr;
}

}  // namespace moe
