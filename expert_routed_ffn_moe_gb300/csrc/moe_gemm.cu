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

struct __align__(8) Barriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kSmemBytes = 1024 /*align slack*/ + (size_t)kStages * (kABytes + kBBytes) + sizeof(Barriers);

struct Work {
  int e, row0, rows;   // expert (E = shared), first grouped row, valid rows
  int n0;              // first output column of the tile (B row offset inside the expert)
  int part;            // router: 0 / 1 / 2 = hi / mid / lo weight term
};

template <int MODE>
MOE_DEV int work_count(const Shapes& s, const Scratch& sc) {
  if (MODE == kGateUp) return sc.meta[0] * (s.I / 128);
  if (MODE == kDown) return sc.meta[0] * (s.d / 256);
  return ((s.T + kBM - 1) / kBM) * 3;
}

template <int MODE>
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
  const MTile m = sc.mtiles[mt];
  r.e = m.e;
  r.row0 = m.row0;
  r.rows = m.rows;
  r.n0 = nt * ((MODE == kGateUp) ? 128 : 256);
  r.part = 0;
  return r;
}

MOE_DEV bool aborted(const Barriers* b) { return *reinterpret_cast<const volatile int*>(&b->abort_flag) != 0; }
MOE_DEV void set_abort(Barriers* b) { *reinterpret_cast<volatile int*>(&b->abort_flag) = 1; }

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmMaps maps, Shapes s,
                                                                   Scratch sc, DevCtl ctl, DevCtl drain) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_buf = base;
  uint8_t* b_buf = base + kStages * kABytes;
  Barriers* bar = reinterpret_cast<Barriers*>(b_buf + kStages * kBBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_work = work_count<MODE>(s, sc);
  if ((int)blockIdx.x >= n_work) return;
  const int KB = ((MODE == kDown) ? s.I : s.d) / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar->full[i], 1);
      mbar_init(&bar->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->tfull[i], 1);
      mbar_init(&bar->tempty[i], 128);
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
    const uint64_t pol_w = policy_evict_normal();  // several m-tiles of one expert reuse its weights
    const uint64_t pol_a = policy_evict_last();
    constexpr uint32_t tx = kABytes + kBBytes;
    int it = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_work && ok; w += gridDim.x) {
      const Work wk = work_item<MODE>(s, sc, w);
      const CUtensorMap* mb;
      int brow0, brow1 = 0;
      if (MODE == kGateUp) {
        mb = (wk.e < s.E) ? &maps.gate_up : &maps.shared_gu;
        const int eb = (wk.e < s.E) ? wk.e * 2 * s.I : 0;
        brow0 = eb + wk.n0;
        brow1 = eb + s.I + wk.n0;
      } else if (MODE == kDown) {
        mb = (wk.e < s.E) ? &maps.down : &maps.shared_down;
        brow0 = ((wk.e < s.E) ? wk.e * s.d : 0) + wk.n0;
      } else {
        mb = &maps.wr_split;
        brow0 = wk.part * s.E;
      }
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int st = it % kStages;
        if (lane == 0) {
          bool good = mbar_wait(&bar->empty[st], ((it / kStages) & 1) ^ 1, ctl);
          if (!good) set_abort(bar);
          else if (aborted(bar)) good = false;
          if (good) {
            mbar_expect_tx(&bar->full[st], tx);
            uint8_t* a_dst = a_buf + st * kABytes;
            uint8_t* b_dst = b_buf + st * kBBytes;
            const int kc = kb * kBK;
            const CUtensorMap* ma = MODE == kGateUp ? &maps.x_perm : (MODE == kDown ? &maps.h : &maps.x_tile);
            tma_load_2d(a_dst, ma, kc, wk.row0, &bar->full[st], pol_a);
            if (MODE == kGateUp) {  // gate rows, then the up rows of the same neurons
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
      const int n = min(it, kStages);
      for (int j = it - n; j < it; ++j) mbar_wait(&bar->full[j % kStages], (j / kStages) & 1, drain);
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
        const int acc = lt & 1;
        const uint32_t use = lt >> 1;
        if (!mbar_wait(&bar->tempty[acc], (use & 1) ^ 1, ctl) || aborted(bar)) {
          set_abort(bar);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * kAccCols;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = it % kStages;
          if (!mbar_wait(&bar->full[st], (it / kStages) & 1, ctl) || aborted(bar)) {
            set_abort(bar);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = umma_desc_sw128(smem_u32(a_buf + st * kABytes));
          const uint64_t bd = umma_desc_sw128(smem_u32(b_buf + st * kBBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // +32 bytes per 16-element k step inside the 128-byte swizzled row
            umma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) ? 1u : 0u);
          }
          umma_commit(&bar->empty[st]);
        }
        if (!ok) break;
        umma_commit(&bar->tfull[acc]);
      }
      umma_commit(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, drain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int row_local = q * 32 + lane;
    int lt = 0;
    for (int w = blockIdx.x; w < n_work; w += gridDim.x, ++lt) {
      const int acc = lt & 1;
      const uint32_t use = lt >> 1;
      if (!mbar_wait(&bar->tfull[acc], use & 1, ctl) || aborted(bar)) {
        set_abort(bar);
        break;
      }
      tc_fence_after();
      const Work wk = work_item<MODE>(s, sc, w);
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
      const bool live = row_local < wk.rows;
      if (MODE == kGateUp) {
        uint16_t* dst = sc.h + (size_t)(wk.row0 + row_local) * s.I + wk.n0;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float g[32], u[32];
          tmem_ld32(taddr + c * 32, g);
          tmem_ld32(taddr + 128 + c * 32, u);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(silu(g[2 * j]) * u[2 * j], silu(g[2 * j + 1]) * u[2 * j + 1]);
          if (live) {
            uint4* o = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      } else if (MODE == kDown) {
        uint16_t* dst = sc.out + (size_t)(wk.row0 + row_local) * s.d + wk.n0;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
          if (live) {
            uint4* o = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      } else {
        float* dst = sc.logits + (size_t)wk.part * s.T * s.E + (size_t)(wk.row0 + row_local) * s.E;
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
      tc_fence_before();
      mbar_arrive(&bar->tempty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int MODE>
static cudaError_t launch_mode(const Shapes& s, const GemmMaps& m, const Scratch& sc, const DevCtl& ctl,
                               int num_sms, cudaStream_t st) {
  DevCtl drain = ctl;
  drain.spin_limit = 2000000000LL;  // 2 s: copies and MMAs already issued always finish
  drain.stall = 0;
  grouped_gemm_kernel<MODE><<<num_sms, kThreads, kSmemBytes, st>>>(m, s, sc, ctl, drain);
  return cudaGetLastError();
}

cudaError_t prepare_gemm_kernels() {
  const void* ks[] = {(const void*)grouped_gemm_kernel<kGateUp>, (const void*)grouped_gemm_kernel<kDown>,
                      (const void*)grouped_gemm_kernel<kRouter>};
  for (const void* k : ks) {
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
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
