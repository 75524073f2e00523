// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, for the prefill (many-token) path.
//
// "Optimizing on-device inference for Apple Silicon", sections "Keeping expert
// routing on the GPU" and "Matching tile size to expert load": a grouped GEMM
// multiplies each expert's routed activation rows by that expert's weights,
// tile by tile, from a block map built on the GPU; section "Dequantizing
// weights during matrix multiplication": fp32 accumulation, bf16 output.
// "LLM in a flash", section 3.2 "Bundling columns and rows": the projections
// of one intermediate neuron are used together -- here the gate and up rows of
// the same neurons are loaded into one B tile so SwiGLU completes in the
// epilogue.
//
// One persistent kernel per GEMM, one CTA per SM, 6 warps:
//   warp 0     TMA producer: A tiles (expert-grouped token rows, h rows or x
//              rows -- always contiguous rows) and B tiles (weights) into a
//              4-stage shared-memory ring with the 128-byte swizzle;
//   warp 1     allocates 512 TMEM columns; lane 0 issues tcgen05.mma
//              (M = 128, N = 256, K = 16 per instruction) into one of two TMEM
//              accumulators;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (one TMEM lane = one
//              output row per thread), then SwiGLU -> bf16 h, bf16 expert
//              outputs, or fp32 router logits;
// The gate/up GEMM reads its token rows from a copy of x already permuted
// into expert groups (moe_route.cu, group_scatter_rows_kernel): gathering 128-byte
// row pieces inside the main loop, by TMA tile::gather4 or by cp.async from
// helper warps, measured several times slower than streaming contiguous tiles.
// Two accumulators let the epilogue of tile i overlap the main loop of tile
// i + 1.  Every wait is bounded (MOE_ERR_TIMEOUT on expiry); on expiry the
// kernel drains what it has in flight, frees TMEM and returns.
//
// 4-bit weights ("Optimizing on-device inference for Apple Silicon", section
// "Dequantizing weights during matrix multiplication": the codes are expanded
// one tile at a time inside the GEMM and never written out): the producer
// loads each k block's raw codes (256 rows x 32 bytes) and, every 8 k blocks,
// the rows' scales and biases of those 8 groups; 8 more warps expand the codes
// to bf16, w = s q + b rounded once (bf16x2 fma), straight into the 128-byte
// swizzled B tile the MMA reads, then release it to the MMA issuer.  A work
// item is a pair of m-tiles of one expert, so each expanded tile serves two
// tiles' MMAs.  The loads run in a 3-stage ring of (two A tiles 32 KB + codes
// 8 KB) and the expanded B tiles in a 2-stage ring of 32 KB, so that the
// copies in flight cover the memory latency while expansion and MMA overlap;
// plus two 8 KB parameter buffers.
//
// bf16 gate/up at large batches (T k >= 512 E) also runs pairs: a 3-stage ring
// of (two A tiles + one B tile), see grouped_gemm_kernel.
#include "moe_internal.h"

namespace moe {

namespace {

enum Mode { kGateUp = 0, kDown = 1, kRouter = 2 };

constexpr int kStages = 4;
constexpr int kBK = 64;                          // bf16 elements per 128-byte row of a k slice
constexpr int kABytes = kBM * kBK * 2;           // 16 KB
constexpr int kBRows = 256;                      // MMA N
constexpr int kBBytes = kBRows * kBK * 2;        // 32 KB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
// 4-bit weights
constexpr int kStagesQ4 = 3;                     // loads (two A tiles + codes) in flight
constexpr int kBStagesQ4 = 2;                    // expanded B tiles
constexpr int kRawBytes = kBRows * 32;           // one k block of codes: 256 rows x 8 words
constexpr int kParGroups = 8;                    // groups (k blocks) per parameter load
constexpr int kParBytes = kBRows * kParGroups * 2;  // scales (or biases) of 8 groups for 256 rows: 4 KB
constexpr int kConvWarps = 8;                    // warps expanding codes (one B row per thread)
constexpr int kThreadsQ4 = kThreads + kConvWarps * 32;

constexpr int kMaxStages = 6;  // the deepest load ring (small-batch layout with 16-row A slots)

struct __align__(8) Barriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t conv[kBStagesQ4];    // 4-bit: the B stage's tile has been expanded
  uint64_t bempty[kBStagesQ4];  // 4-bit: the MMA is done with the B stage
  uint64_t pfull[2];         // 4-bit: parameter buffer loaded
  uint64_t pempty[2];        // 4-bit: parameter buffer consumed
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kSmemBytes = 1024 /*align slack*/ + (size_t)kStages * (kABytes + kBBytes) + sizeof(Barriers);
// bf16 pairs (gate/up at large batches): a load stage holds both A tiles of a
// pair and one B tile, 64 KB instead of 48 KB for twice the MMA work
constexpr int kStagesPairs = 3;
constexpr size_t kSmemBytesPairs = 1024 + (size_t)kStagesPairs * (2 * kABytes + kBBytes) + sizeof(Barriers);
// Small batches (every expert group, the shared one included, has at most
// AROWS <= T rows): an A slot holds only AROWS rows (2 or 4 KB), which frees
// shared memory for more weight stages in flight.  The MMA still reads 128 rows
// from the slot's start; past the AROWS real rows it reads whatever shared
// memory follows (later A slots, then B tiles) -- finite values whose output
// rows the epilogue drops -- and the slots are laid out first so those reads
// stay inside the CTA's shared memory.
constexpr int small_a_stages(int arows) { return arows == 16 ? 6 : 5; }
constexpr size_t small_a_smem(int arows) {
  return 1024 + (size_t)small_a_stages(arows) * (arows * kBK * 2 + kBBytes) + sizeof(Barriers);
}
constexpr size_t kSmemBytesQ4 = 1024 + (size_t)kStagesQ4 * (2 * kABytes + kRawBytes) + (size_t)kBStagesQ4 * kBBytes +
                                2 * 2 * kParBytes + sizeof(Barriers);
static_assert(kSmemBytesQ4 <= 227 * 1024 && kSmemBytes <= 227 * 1024 && kSmemBytesPairs <= 227 * 1024,
              "shared memory of one CTA");
static_assert(small_a_stages(16) <= kMaxStages && small_a_stages(32) <= kMaxStages && kStagesQ4 <= kMaxStages,
              "barrier arrays");
static_assert(small_a_smem(16) <= 227 * 1024 && small_a_smem(32) <= 227 * 1024, "shared memory of one CTA");
// the MMA reads 128 rows (16 KB) from any small A slot: the last slot's read must end inside the ring
static_assert((small_a_stages(16) - 1) * 16 * 128 + kABytes <= small_a_stages(16) * (16 * 128 + kBBytes), "A reads");
static_assert((small_a_stages(32) - 1) * 32 * 128 + kABytes <= small_a_stages(32) * (32 * 128 + kBBytes), "A reads");

// fma.rn.bf16x2: a * b + c per half, computed exactly and rounded once
MOE_DEV uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// The 8 weights of one code word (columns 8 c .. 8 c + 7 of the k block) as
// bf16 s q + b, in the column order 0, 4, 1, 5, 2, 6, 3, 7 (q4_chunk_order):
// nibbles i and i + 4 come out as one bf16 pair, and the A operands (x_perm,
// h) are stored in the same order, so no reordering is needed.  A code q is
// made exact in bf16 as (128 + q) - 128: the bits 0x4300 | q are the bf16
// value 128 + q.
MOE_DEV uint4 expand_q4_word(uint32_t w, uint32_t s2, uint32_t b2) {
  constexpr uint32_t kMagic = 0x43004300u, kOne = 0x3F803F80u, kMinus128 = 0xC300C300u;
  const uint32_t v0 = fma_bf16x2(fma_bf16x2((w & 0x000F000Fu) | kMagic, kOne, kMinus128), s2, b2);          // cols 0, 4
  const uint32_t v1 = fma_bf16x2(fma_bf16x2(((w >> 4) & 0x000F000Fu) | kMagic, kOne, kMinus128), s2, b2);   // 1, 5
  const uint32_t v2 = fma_bf16x2(fma_bf16x2(((w >> 8) & 0x000F000Fu) | kMagic, kOne, kMinus128), s2, b2);   // 2, 6
  const uint32_t v3 = fma_bf16x2(fma_bf16x2(((w >> 12) & 0x000F000Fu) | kMagic, kOne, kMinus128), s2, b2);  // 3, 7
  return make_uint4(v0, v1, v2, v3);
}
MOE_DEV void tma_load_2d_nohint(void* dst, const CUtensorMap* m, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

struct Work {
  int e, row0, rows;   // expert (E = shared), first grouped row, valid rows
  int rows2;           // pairs: valid rows of the pair's second tile (rows row0 + 128 ...; 0: none)
  int n0;              // first output column of the tile (B row offset inside the expert)
  int part;            // router: 0 / 1 / 2 = hi / mid / lo weight term
};

template <int MODE, bool PAIRS = false>
MOE_DEV int work_count(const Shapes& s, const Scratch& sc) {
  if (MODE == kRouter) return ((s.T + kBM - 1) / kBM) * 3;
  int n = sc.meta[PAIRS ? 2 : 0];
  if (kDebugChecks && (n < 0 || n > sc.max_mtiles)) {
    atomicOr(sc.status, kStatusBounds);
    n = 0;
  }
  return n * (MODE == kGateUp ? s.I / 128 : s.d / 256);
}

template <int MODE, bool PAIRS = false>
MOE_DEV Work work_item(const Shapes& s, const Scratch& sc, int w) {
  Work r{};
  if (MODE == kRouter) {
    const int mt = w / 3;
    r.e = 0;
    r.row0 = mt * kBM;
    r.rows = min(kBM, s.T - r.row0);
    r.n0 = 0;
    r.part = w - mt * 3;
    return r;
  }
  const int nnt = (MODE == kGateUp) ? s.I / 128 : s.d / 256;
  const int mt = w / nnt, nt = w - mt * nnt;
  MTile m = PAIRS ? sc.mpairs[mt] : sc.mtiles[mt];
  if (!PAIRS) m.pad = 0;
  if (kDebugChecks) {
    const int total = s.T * s.k + (s.has_shared ? s.T : 0);  // grouped rows
    if (m.e < 0 || m.e > s.E || (m.e == s.E && !s.has_shared) || m.rows < 1 || m.rows > kBM || m.row0 < 0 ||
        m.pad < 0 || m.pad > kBM || (m.pad > 0 && m.rows != kBM) || m.row0 + m.rows + m.pad > total) {
      atomicOr(sc.status, kStatusBounds);
      m = MTile{0, 0, 1, 0};  // every role of the kernel reads the same entry and replaces it alike
    }
  }
  r.e = m.e;
  r.row0 = m.row0;
  r.rows = m.rows;
  r.rows2 = m.pad;
  r.n0 = nt * ((MODE == kGateUp) ? 128 : 256);
  r.part = 0;
  return r;
}

MOE_DEV bool aborted(const Barriers* b) { return *reinterpret_cast<const volatile int*>(&b->abort_flag) != 0; }
MOE_DEV void set_abort(Barriers* b) { *reinterpret_cast<volatile int*>(&b->abort_flag) = 1; }

}  // namespace

// Q4: the B operand (weights) is expanded from 4-bit codes by the converter
// warps 6 .. 6 + kConvWarps - 1 (gate/up and down modes only).
// AROWS (bf16 only): 0 = full 128-row A slots; 16 or 32 = the small-batch
// layout above (valid only when T <= AROWS).
// PAIRED: a work item is a pair of m-tiles of one expert, both multiplied by
// each B tile the item loads (always for 4-bit; for bf16 an option of the
// full-slot layout).  Each SM then takes in 64 KB per k block for two tiles'
// MMAs instead of 2 x 48 KB, which pays where groups are long (pairs_for).
template <int MODE, bool Q4, int AROWS = 0, bool PAIRED = Q4>
__global__ void __launch_bounds__(Q4 ? kThreadsQ4 : kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmMaps maps, Shapes s, Scratch sc, DevCtl ctl, DevCtl drain) {
  static_assert(!(PAIRED && AROWS), "pairs use full A slots");
  constexpr bool PAIRS = PAIRED && MODE != kRouter;
  // load ring (A, and B or codes)
  constexpr int S = Q4 ? kStagesQ4 : (AROWS ? small_a_stages(AROWS) : (PAIRS ? kStagesPairs : kStages));
  constexpr int SB = Q4 ? kBStagesQ4 : S;          // B tiles the MMA reads (bf16: part of the load ring)
  constexpr int kASlot = PAIRS ? 2 * kABytes : (AROWS ? AROWS * kBK * 2 : kABytes);  // bytes per A slot
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_buf = base;
  uint8_t* b_buf = base + S * kASlot;
  uint8_t* raw_buf = b_buf + SB * kBBytes;                 // Q4: codes of each load stage
  uint8_t* par_buf = raw_buf + (Q4 ? S * kRawBytes : 0);   // Q4: [2 buffers][scales | biases]
  Barriers* bar = reinterpret_cast<Barriers*>(par_buf + (Q4 ? 2 * 2 * kParBytes : 0));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_work = work_count<MODE, PAIRS>(s, sc);
  if ((int)blockIdx.x >= n_work) return;
  const int K = (MODE == kDown) ? s.I : s.d;   // reduction length
  const int KB = K / kBK;
  const int G = K / 64;                        // Q4: groups (of 64 columns) per weight row

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&bar->full[i], 1);
      mbar_init(&bar->empty[i], 1);
    }
    for (int i = 0; i < kBStagesQ4; ++i) {
      mbar_init(&bar->conv[i], kConvWarps * 32);
      mbar_init(&bar->bempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->tfull[i], 1);
      mbar_init(&bar->tempty[i], 128);
      mbar_init(&bar->pfull[i], 1);
      mbar_init(&bar->pempty[i], kConvWarps * 32);
    }
    mbar_init(&bar->mma_done, 1);
    bar->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&bar->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) tma_prefetch_desc(MODE == kGateUp ? &maps.x_perm : (MODE == kDown ? &maps.h : &maps.x_tile));
    const uint64_t pol_reuse = policy_evict_normal();  // several m-tiles of one expert reuse its weights
    const uint64_t pol_once = policy_evict_first();    // ... or are read by one item only
    const uint64_t pol_a = policy_evict_last();
    constexpr uint32_t tx_b = Q4 ? kRawBytes : kBBytes;
    int it = 0, pc = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
      const Work wk = work_item<MODE, PAIRS>(s, sc, w);
      // bf16 weight tiles of a group that fits one item (one m-tile, or a
      // pair) are read once: stream them, so that they do not push the token
      // rows, which every n-tile of the group reads, out of L2 (T = 32 layer
      // 197 -> 190 us, T = 128 292 -> 285 us, skewed T = 4096 371 -> 366 us).
      // A group of more tiles reads them again from later items (balanced
      // T = 4096, where half the groups spill a few rows into a second tile:
      // 435 -> 464 us per layer when those were streamed too), and a 4-bit
      // k block reads 32 bytes of each code row, so four k blocks share a line
      // (gate/up 253 -> 259 us when streamed)
      const int group_rows = MODE == kRouter ? 0 : (wk.e < s.E ? sc.counts[wk.e] : s.T);
      const uint64_t pol_w = (!Q4 && MODE != kRouter && group_rows <= (PAIRS ? 2 : 1) * kBM) ? pol_once : pol_reuse;
      const CUtensorMap* mb;
      const CUtensorMap* mp = nullptr;  // Q4: parameter view of the same rows
      int brow0, brow1 = 0;
      if (MODE == kGateUp) {
        mb = Q4 ? ((wk.e < s.E) ? &maps.gu_codes : &maps.sgu_codes) : ((wk.e < s.E) ? &maps.gate_up : &maps.shared_gu);
        mp = (wk.e < s.E) ? &maps.gu_params : &maps.sgu_params;
        const int eb = (wk.e < s.E) ? wk.e * 2 * s.I : 0;
        brow0 = eb + wk.n0;
        brow1 = eb + s.I + wk.n0;
      } else if (MODE == kDown) {
        mb = Q4 ? ((wk.e < s.E) ? &maps.dn_codes : &maps.sdn_codes) : ((wk.e < s.E) ? &maps.down : &maps.shared_down);
        mp = (wk.e < s.E) ? &maps.dn_params : &maps.sdn_params;
        brow0 = ((wk.e < s.E) ? wk.e * s.d : 0) + wk.n0;
      } else {
        mb = &maps.wr_split;
        brow0 = wk.part * s.E;
      }
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int st = it % S;
        if (lane == 0) {
          bool good = true;
          if (Q4 && kb % kParGroups == 0) {
            // scales and biases of groups kb .. kb + 7 of this tile's rows: each
            // row's K / 8 code words are followed by its G scales, then G biases
            // (bf16 columns K / 4 + g and K / 4 + G + g); with G = 4 one 8-wide
            // box holds both
            const int pb = pc & 1;
            good = mbar_wait(&bar->pempty[pb], ((pc >> 1) & 1) ^ 1, ctl);
            if (!good) set_abort(bar);
            else if (aborted(bar)) good = false;
            if (good) {
              uint8_t* ps = par_buf + pb * 2 * kParBytes;
              uint8_t* pbb = ps + kParBytes;
              const int xs = K / 4 + kb, xb = K / 4 + G + kb;
              const bool two = G >= kParGroups;
              mbar_expect_tx(&bar->pfull[pb], (two ? 2 : 1) * kParBytes);
              if (MODE == kGateUp) {
                tma_load_2d_nohint(ps, mp, xs, brow0, &bar->pfull[pb]);
                tma_load_2d_nohint(ps + kParBytes / 2, mp, xs, brow1, &bar->pfull[pb]);
                if (two) {
                  tma_load_2d_nohint(pbb, mp, xb, brow0, &bar->pfull[pb]);
                  tma_load_2d_nohint(pbb + kParBytes / 2, mp, xb, brow1, &bar->pfull[pb]);
                }
              } else {
                tma_load_2d_nohint(ps, mp, xs, brow0, &bar->pfull[pb]);
                if (two) tma_load_2d_nohint(pbb, mp, xb, brow0, &bar->pfull[pb]);
              }
            }
            ++pc;
          }
          if (good) {
            good = mbar_wait(&bar->empty[st], ((it / S) & 1) ^ 1, ctl);
            if (!good) set_abort(bar);
            else if (aborted(bar)) good = false;
          }
          if (good) {
            // A: the whole 128-row tile, or, for a group of at most 64 rows,
            // only the 16-row boxes that cover them (the MMA still multiplies
            // 128 rows; the rows not loaded hold stale finite values of an
            // earlier tile, and the epilogue drops their outputs).  Above 64
            // rows the extra box loads cost the producer more than the bytes
            // they save (the balanced T = 4096 gate/up GEMM: 229 -> 236 us
            // with boxes up to 112 rows)
            const int a_boxes = (wk.rows + 15) / 16, a2_boxes = (wk.rows2 + 15) / 16;
            const bool whole = AROWS == 0 && a_boxes > 4, whole2 = a2_boxes > 4;
            const uint32_t a_bytes = whole ? kABytes : a_boxes * 16 * kBK * 2;
            const uint32_t a2_bytes = PAIRS ? (whole2 ? kABytes : a2_boxes * 16 * kBK * 2) : 0u;
            mbar_expect_tx(&bar->full[st], a_bytes + a2_bytes + tx_b);
            uint8_t* a_dst = a_buf + st * kASlot;
            uint8_t* b_dst = Q4 ? raw_buf + st * kRawBytes : b_buf + st * kBBytes;
            const int kc = kb * kBK;
            const CUtensorMap* ma = MODE == kGateUp ? &maps.x_perm : (MODE == kDown ? &maps.h : &maps.x_tile);
            const CUtensorMap* ma16 = MODE == kGateUp ? &maps.x_perm16 : (MODE == kDown ? &maps.h16 : &maps.x_tile16);
            if (whole) {
              tma_load_2d(a_dst, ma, kc, wk.row0, &bar->full[st], pol_a);
            } else {
              for (int i = 0; i < a_boxes; ++i)
                tma_load_2d(a_dst + i * 16 * kBK * 2, ma16, kc, wk.row0 + 16 * i, &bar->full[st], pol_a);
            }
            if (PAIRS && wk.rows2 > 0) {  // the pair's second tile, rows row0 + 128 ...
              if (whole2) {
                tma_load_2d(a_dst + kABytes, ma, kc, wk.row0 + kBM, &bar->full[st], pol_a);
              } else {
                for (int i = 0; i < a2_boxes; ++i)
                  tma_load_2d(a_dst + kABytes + i * 16 * kBK * 2, ma16, kc, wk.row0 + kBM + 16 * i, &bar->full[st],
                              pol_a);
              }
            }
            if (Q4) {  // the k block's code words: 8 per row
              if (MODE == kGateUp) {
                tma_load_2d(b_dst, mb, kb * 8, brow0, &bar->full[st], pol_w);
                tma_load_2d(b_dst + kRawBytes / 2, mb, kb * 8, brow1, &bar->full[st], pol_w);
              } else {
                tma_load_2d(b_dst, mb, kb * 8, brow0, &bar->full[st], pol_w);
              }
            } else if (MODE == kGateUp) {  // gate rows, then the up rows of the same neurons
              tma_load_2d(b_dst, mb, kc, brow0, &bar->full[st], pol_w);
              tma_load_2d(b_dst + 128 * 128, mb, kc, brow1, &bar->full[st], pol_w);
            } else {
              tma_load_2d(b_dst, mb, kc, brow0, &bar->full[st], pol_w);
            }
          } else {
            ok = false;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
    }
    // drain: the copies into the last stages must land before the CTA exits
    if (lane == 0) {
      const int n = min(it, S);
      for (int j = it - n; j < it; ++j) mbar_wait(&bar->full[j % S], (j / S) & 1, drain);
      if (Q4)
        for (int j = max(0, pc - 2); j < pc; ++j) mbar_wait(&bar->pfull[j & 1], (j >> 1) & 1, drain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kBM, kBRows);
      int it = 0, lt = 0;
      bool ok = true;
      if (ctl.stall) {  // test hook: a barrier nothing arrives at; the bounded wait must give up
        // mma_done completes its phase 0 only at the final commit below
        if (!mbar_wait(&bar->mma_done, 0, ctl)) {
          set_abort(bar);
          ok = false;
        }
      }
      for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x, ++lt) {
        // single tiles alternate between the two accumulators; pairs use both
        // (tile 1 in columns 0..255, tile 2 in 256..511)
        const int acc = PAIRS ? 0 : (lt & 1);
        const uint32_t use = PAIRS ? lt : (lt >> 1);
        if (!mbar_wait(&bar->tempty[acc], (use & 1) ^ 1, ctl) || aborted(bar)) {
          set_abort(bar);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * kAccCols;
        const bool second = PAIRS && work_item<MODE, PAIRS>(s, sc, w).rows2 > 0;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = it % S, sb = it % SB;
          // bf16: the stage's copies landed; 4-bit: the converters expanded the
          // B tile (after the stage's copies landed)
          if (!mbar_wait(Q4 ? &bar->conv[sb] : &bar->full[st], Q4 ? (it / SB) & 1 : (it / S) & 1, ctl) ||
              aborted(bar)) {
            set_abort(bar);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = umma_desc_sw128(smem_u32(a_buf + st * kASlot));
          const uint64_t bd = umma_desc_sw128(smem_u32(b_buf + sb * kBBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // +32 bytes per 16-element k step inside the 128-byte swizzled row
            umma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
          }
          if (PAIRS && kb == 0 && !mbar_wait(&bar->tempty[1], (use & 1) ^ 1, ctl)) {
            // accumulator 1 is drained only now: the epilogue's second half
            // overlaps this item's first k block on accumulator 0
            set_abort(bar);
            ok = false;
            break;
          }
          if (second) {
            tc_fence_after();
            const uint64_t ad2 = umma_desc_sw128(smem_u32(a_buf + st * kASlot + kABytes));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_bf16(tmem + kAccCols, ad2 + 2 * kk, bd + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
          }
          umma_commit(&bar->empty[st]);
          if (Q4) umma_commit(&bar->bempty[sb]);
        }
        if (!ok) break;
        umma_commit(&bar->tfull[acc]);
        if (PAIRS) umma_commit(&bar->tfull[1]);
      }
      umma_commit(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, drain);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int row_local = q * 32 + lane;
    int lt = 0;
    bool stop = false;
    for (int w = blockIdx.x; w < n_work && !stop; w += gridDim.x, ++lt) {
      const Work wk = work_item<MODE, PAIRS>(s, sc, w);
      // single tiles: the item's accumulator; pairs: tile 1 in accumulator 0,
      // tile 2 (rows row0 + 128 ..., maybe none) in accumulator 1
      for (int tt = 0; tt < (PAIRS ? 2 : 1); ++tt) {
        const int acc = PAIRS ? tt : (lt & 1);
        const uint32_t use = PAIRS ? lt : (lt >> 1);
        if (!mbar_wait(&bar->tfull[acc], use & 1, ctl) || aborted(bar)) {
          set_abort(bar);
          stop = true;
          break;
        }
        tc_fence_after();
        const int row0 = wk.row0 + tt * kBM, rows = tt ? wk.rows2 : wk.rows;
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
        const bool live = row_local < rows;
        if (rows > 0) {
          if (MODE == kGateUp) {
            uint16_t* dst = sc.h + (size_t)(row0 + row_local) * s.I + wk.n0;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              // the gate and up columns of the chunk: both loads, then one wait
              uint32_t gr[32], ur[32];
              tmem_ld32_async(taddr + c * 32, gr);
              tmem_ld32_async(taddr + 128 + c * 32, ur);
              tmem_ld_wait();
              uint32_t pk[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float g0 = __uint_as_float(gr[2 * j]), g1 = __uint_as_float(gr[2 * j + 1]);
                pk[j] = pack_bf16x2(silu(g0) * __uint_as_float(ur[2 * j]), silu(g1) * __uint_as_float(ur[2 * j + 1]));
              }
              if (live) {
                uint4* o = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint4 v = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                  o[j] = Q4 ? q4_chunk_order(v) : v;  // 4-bit: h is the down GEMM's A, in the expansion order
                }
              }
            }
          } else if (MODE == kDown) {
            uint16_t* dst = sc.out + (size_t)(row0 + row_local) * s.d + wk.n0;
#pragma unroll 1
            for (int c = 0; c < 8; c += 2) {
              // two 32-column chunks per wait
              uint32_t v0[32], v1[32];
              tmem_ld32_async(taddr + c * 32, v0);
              tmem_ld32_async(taddr + (c + 1) * 32, v1);
              tmem_ld_wait();
              uint32_t pk[32];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                pk[j] = pack_bf16x2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1]));
                pk[16 + j] = pack_bf16x2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1]));
              }
              if (live) {
                uint4* o = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
              }
            }
          } else {
            float* dst = sc.logits + (size_t)wk.part * s.T * s.E + (size_t)(row0 + row_local) * s.E;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              float v[32];
              tmem_ld32(taddr + c * 32, v);
              if (live) {
                float4* o = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&bar->tempty[acc]);
      }
    }
  } else if (Q4) {
    // ------------------------------------------------------------ code expansion (4-bit)
    // thread r expands B row r of every stage: its 8 code words (32 bytes of
    // the raw tile) into 8 swizzled 16-byte chunks of bf16 weights
    const int r = threadIdx.x - 6 * 32;
    int it = 0, pc = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int st = it % S, sb = it % SB, pb = pc & 1;  // pc: this k block's parameter load
        if (kb % kParGroups == 0) {
          if (!mbar_wait(&bar->pfull[pb], (pc >> 1) & 1, ctl) || aborted(bar)) {
            set_abort(bar);
            ok = false;
            break;
          }
        }
        if (!mbar_wait(&bar->full[st], (it / S) & 1, ctl) || !mbar_wait(&bar->bempty[sb], ((it / SB) & 1) ^ 1, ctl) ||
            aborted(bar)) {
          set_abort(bar);
          ok = false;
          break;
        }
        const uint16_t* ps = reinterpret_cast<const uint16_t*>(par_buf + pb * 2 * kParBytes);
        const int g = kb % kParGroups;
        const uint32_t sbits = ps[r * kParGroups + (G >= kParGroups ? g : kb)];
        const uint32_t bbits = G >= kParGroups ? ps[kParBytes / 2 + r * kParGroups + g] : ps[r * kParGroups + G + kb];
        const uint32_t s2 = sbits | (sbits << 16), b2 = bbits | (bbits << 16);
        const uint4* raw = reinterpret_cast<const uint4*>(raw_buf + st * kRawBytes + r * 32);
        const uint4 c0 = raw[0], c1 = raw[1];
        uint8_t* row = b_buf + sb * kBBytes + r * 128;
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) = expand_q4_word(words[c], s2, b2);
        // the MMA reads the tile through the async proxy
        fence_proxy_async_shared_cta();
        mbar_arrive(&bar->conv[sb]);
        if (kb % kParGroups == kParGroups - 1 || kb == KB - 1) {
          mbar_arrive(&bar->pempty[pb]);
          ++pc;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// bf16 pairs for the gate/up GEMM once the mean group (T k / E rows) spans 4
// tiles.  Measured per launch at d = 2048, 256 experts of 512, top-8 + shared:
// T = 32768 (8 tiles a group) 868 -> 782 us with pairs; T = 4096 (1 tile a
// group) balanced 219 -> 238 us and skewed (3.5 tiles per active expert)
// 166 -> 170 us.  There the mean CTA finishes its loop sooner with pairs
// (skewed: 136 vs 144 us), but the items are twice as long, so the slowest
// CTA ends later than with single tiles, and a pair's two accumulators both
// wait for the epilogue before the next item starts.
static bool pairs_for(int mode, const Shapes& s) {
  return mode == kGateUp && (long long)s.T * s.k >= 4LL * s.E * kBM;
}

template <int MODE>
static cudaError_t launch_mode(const Shapes& s, const GemmMaps& m, const Scratch& sc, const DevCtl& ctl,
                               int num_sms, cudaStream_t st) {
  DevCtl drain = ctl;
  drain.spin_limit = 2000000000LL;  // 2 s: copies and MMAs already issued always finish
  drain.stall = 0;
  if (MODE != kRouter && s.q4)
    grouped_gemm_kernel<MODE, true><<<num_sms, kThreadsQ4, kSmemBytesQ4, st>>>(m, s, sc, ctl, drain);
  else if (MODE != kRouter && s.T <= 16)  // every group has at most T rows
    grouped_gemm_kernel<MODE, false, 16><<<num_sms, kThreads, small_a_smem(16), st>>>(m, s, sc, ctl, drain);
  else if (MODE != kRouter && s.T <= 32)
    grouped_gemm_kernel<MODE, false, 32><<<num_sms, kThreads, small_a_smem(32), st>>>(m, s, sc, ctl, drain);
  else if (pairs_for(MODE, s))
    grouped_gemm_kernel<kGateUp, false, 0, true><<<num_sms, kThreads, kSmemBytesPairs, st>>>(m, s, sc, ctl, drain);
  else
    grouped_gemm_kernel<MODE, false><<<num_sms, kThreads, kSmemBytes, st>>>(m, s, sc, ctl, drain);
  return cudaGetLastError();
}

cudaError_t prepare_gemm_kernels() {
  const void* ks[] = {(const void*)grouped_gemm_kernel<kGateUp, false>, (const void*)grouped_gemm_kernel<kDown, false>,
                      (const void*)grouped_gemm_kernel<kRouter, false>};
  for (const void* k : ks) {
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
  }
  {
    cudaError_t err = cudaFuncSetAttribute((const void*)grouped_gemm_kernel<kGateUp, false, 0, true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesPairs);
    if (err != cudaSuccess) return err;
  }
  const void* kq[] = {(const void*)grouped_gemm_kernel<kGateUp, true>, (const void*)grouped_gemm_kernel<kDown, true>};
  for (const void* k : kq) {
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytesQ4);
    if (err != cudaSuccess) return err;
  }
  const void* k16[] = {(const void*)grouped_gemm_kernel<kGateUp, false, 16>,
                       (const void*)grouped_gemm_kernel<kDown, false, 16>};
  for (const void* k : k16) {
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)small_a_smem(16));
    if (err != cudaSuccess) return err;
  }
  const void* k32[] = {(const void*)grouped_gemm_kernel<kGateUp, false, 32>,
                       (const void*)grouped_gemm_kernel<kDown, false, 32>};
  for (const void* k : k32) {
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)small_a_smem(32));
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

// The 4-bit kernels' parameter loads need every weight row's K / 64 groups to
// split into whole boxes of 8 (or to be exactly 4): K = 256 or K % 512 == 0.
bool gemm_q4_supported(int d, int inter) {
  auto ok = [](int K) { return K == 256 || K % 512 == 0; };
  return ok(d) && ok(inter);
}

cudaError_t launch_gemm_gate_up(const Shapes& s, const GemmMaps& m, const Scratch& sc, const DevCtl& ctl,
                                int num_sms, cudaStream_t st) {
  return launch_mode<kGateUp>(s, m, sc, ctl, num_sms, st);
}
cudaError_t launch_gemm_down(const Shapes& s, const GemmMaps& m, const Scratch& sc, const DevCtl& ctl, int num_sms,
                             cudaStream_t st) {
  return launch_mode<kDown>(s, m, sc, ctl, num_sms, st);
}
cudaError_t launch_gemm_router(const Shapes& s, const GemmMaps& m, const Scratch& sc, const DevCtl& ctl,
                               int num_sms, cudaStream_t st) {
  return launch_mode<kRouter>(s, m, sc, ctl, num_sms, st);
}

}  // namespace moe
