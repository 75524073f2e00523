// Fused decode layer: the whole MoE layer for a handful of tokens in ONE
// cooperative persistent kernel (one block per SM), three phases separated by
// two grid barriers.
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
//   phase A  router logits l[t, e] (fp32 FMA, one block per expert pair, the
//            row split over 8 warps and summed in a fixed order); meanwhile the
//            shared expert's weights (routing-independent) are prefetched into L2.
//   -- grid barrier --
//   phase B  every block selects the top-k of every token from the logits (same
//            result in every block), groups tokens by expert in shared memory,
//            prefetches into L2 every weight row it will read in phases B and C,
//            then runs the gate/up GEMV + SwiGLU for its (expert, neuron) units.
//   -- grid barrier --
//   phase C  one warp per output feature: for the active experts in ascending
//            id (shared expert last) the down-projection row from L2, dotted
//            with each routed token's h, scaled by its routing weight, summed
//            per token in fp32 and written to y.
//
// Barriers are counter barriers with a bounded spin (MOE_ERR_TIMEOUT); the last
// block to leave resets the counters, so graph replays start from zero.
#include <math.h>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;

MOE_DEV void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}
MOE_DEV unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Arrive at grid barrier `n` (1-based) and wait for every block; false on timeout.
MOE_DEV bool grid_sync(unsigned* count, unsigned n, const DevCtl& c, int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(count, 1u);
    // test hook: wait for one arrival more than there are blocks (never happens)
    const unsigned target = n * gridDim.x + (c.stall ? 1u : 0u);
    const long long t0 = clock64(), lim = wait_cycles(c);
    while (ld_acquire(count) < target) {
      if (clock64() - t0 > lim) {
        raise_status(c, kStatusTimeout);
        ok = 0;
        break;
      }
    }
    __threadfence();
    *flag = ok;
  }
  __syncthreads();
  return *flag != 0;
}

MOE_DEV float dot8(const uint4 w, const float* x) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  const float4 b = *reinterpret_cast<const float4*>(x + 4);
  float s = bf16_lo(w.x) * a.x;
  s = fmaf(bf16_hi(w.x), a.y, s);
  s = fmaf(bf16_lo(w.y), a.z, s);
  s = fmaf(bf16_hi(w.y), a.w, s);
  s = fmaf(bf16_lo(w.z), b.x, s);
  s = fmaf(bf16_hi(w.z), b.y, s);
  s = fmaf(bf16_lo(w.w), b.z, s);
  s = fmaf(bf16_hi(w.w), b.w, s);
  return s;
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
  unsigned* bar;   // [0] arrivals, [1] departures
};

// Shared-memory layout (bytes from the dynamic base).
struct DecodeSmem {
  size_t big;      // x as fp32 [T][d] in phases A/B, then h as fp32 [pairs][I] in phase C
  size_t total;
};

__host__ __device__ inline size_t decode_big_bytes(const Shapes& s) {
  const size_t pairs = (size_t)s.T * s.k + (s.has_shared ? s.T : 0);
  const size_t a = (size_t)s.T * s.d * 4, b = pairs * s.I * 4;
  return a > b ? a : b;
}

// MAXT: compile-time bound on T (1 or 16), so the batch-1 kernel keeps one accumulator per lane.
template <int NCH, int NCI, bool XBF16, int MAXT>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(const DecodeArgs A) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const Shapes& s = A.s;
  const Scratch& sc = A.sc;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int G = gridDim.x, b = blockIdx.x;

  float* big = reinterpret_cast<float*>(dsm);
  __shared__ float rpart[2][8][16];        // router partial sums [slot][chunk][token]
  __shared__ int sel_e[16][kMaxTopK];      // chosen experts per token, ascending
  __shared__ float sel_w[16][kMaxTopK];
  __shared__ int act_e[kMaxExperts + 1];   // active experts ascending, shared last
  __shared__ unsigned act_m[kMaxExperts + 1];
  __shared__ int act_row[kMaxExperts + 1]; // first grouped h row of each active expert
  __shared__ float act_w[kMaxExperts + 1][16];  // routing weight of each token for the expert
  __shared__ int n_act_s, flag_s;
  __shared__ int warp_tot[kWarps];

  bool ok = true;
  // ---------------------------------------------------------------- phase A
  {
    // router rows first (they need nothing), then x; lane owns NCH consecutive
    // columns of its warp's d/8-wide chunk
    constexpr int kPer = NCH;  // = d / 256
    const int chunk = s.d / 8;
    const int slot = warp >> 3, cw = warp & 7;
    const int col0 = cw * chunk + lane * kPer;
    float wv[1][kPer];
    int n_e0 = 0;
    for (int e0 = b; e0 < s.E; e0 += 2 * G) ++n_e0;
    {
      const int e = b + slot * G;
      if (e < s.E) {
        const float2* wrow = reinterpret_cast<const float2*>(A.wr + (size_t)e * s.d + col0);
#pragma unroll
        for (int i = 0; i < kPer / 2; ++i) {
          const float2 v = __ldg(wrow + i);
          wv[0][2 * i] = v.x;
          wv[0][2 * i + 1] = v.y;
        }
      }
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
    // the shared expert does not depend on routing: pull its weights into L2 now
    if (s.has_shared) {
      const size_t bytes = (size_t)3 * s.I * s.d * 2;
      const size_t per = ((bytes / G) + 4095) & ~size_t(4095);
      const size_t lo = per * b, hi = min(bytes, lo + per);
      const uint8_t* base = reinterpret_cast<const uint8_t*>(A.shared_w);
      for (size_t off = lo + (size_t)tid * 4096; off < hi; off += (size_t)kThreads * 4096)
        prefetch_l2(base + off, (uint32_t)min((size_t)4096, hi - off));
    }
    __syncthreads();
    for (int rep = 0; rep < n_e0; ++rep) {
      const int e = b + rep * 2 * G + slot * G;
      if (rep > 0 && e < s.E) {
        const float2* wrow = reinterpret_cast<const float2*>(A.wr + (size_t)e * s.d + col0);
#pragma unroll
        for (int i = 0; i < kPer / 2; ++i) {
          const float2 v = __ldg(wrow + i);
          wv[0][2 * i] = v.x;
          wv[0][2 * i + 1] = v.y;
        }
      }
      if (e < s.E) {
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
          if (t < s.T) {
            const float* xr = big + (size_t)t * s.d + col0;
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kPer; ++i) acc = fmaf(wv[0][i], xr[i], acc);
            acc = warp_sum(acc);
            if (lane == 0) rpart[slot][cw][t] = acc;
          }
        }
      }
      __syncthreads();
      if (tid < 2 * 16) {
        const int sl = tid >> 4, t = tid & 15;
        const int ee = b + rep * 2 * G + sl * G;
        if (ee < s.E && t < s.T) {
          float l = 0.f;
#pragma unroll
          for (int c = 0; c < 8; ++c) l += rpart[sl][c][t];
          sc.logits[(size_t)t * s.E + ee] = l;
        }
      }
      __syncthreads();
    }
  }
  ok = grid_sync(A.bar, 1, A.ctl, &flag_s);

  // ---------------------------------------------------------------- phase B
  if (ok) {
    // selection, identical in every block (same logits, same arithmetic)
    if (warp < s.T) {
      const int t = warp;
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < s.E) ? __ldcg(sc.logits + (size_t)t * s.E + e) + (A.rb ? A.rb[e] : 0.f) : -INFINITY;
      }
      int pe, rank;
      float pw;
      if (!warp_top_k(v, s.E, s.k, lane, pe, pw, rank) && lane == 0) raise_status(A.ctl, kStatusBounds);
      if (lane < s.k) {
        sel_e[t][rank] = pe;
        sel_w[t][rank] = pw;
        if (b == 0) {
          sc.idx[(size_t)t * s.k + rank] = pe;
          sc.w[(size_t)t * s.k + rank] = pw;
        }
      }
    }
    __syncthreads();
    // group tokens by expert: masks, active list (ascending), grouped h rows
    unsigned m = 0u;
    if (tid < s.E) {
      for (int t = 0; t < s.T; ++t)
        for (int j = 0; j < s.k; ++j)
          if (sel_e[t][j] == tid) m |= 1u << t;
    }
    {
      const int flag = (tid < s.E && m) ? 1 : 0, cnt = (tid < s.E) ? __popc(m) : 0;
      // block scan of (flag, cnt) packed: flag in the high half, count in the low half
      int v = (flag << 16) | cnt, incl = v;
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
      if (flag) {
        const int pos = excl >> 16;
        act_e[pos] = tid;
        act_m[pos] = m;
        act_row[pos] = excl & 0xffff;
        for (int t = 0; t < s.T; ++t) {
          float wt = 0.f;
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
          act_row[n_routed] = s.T * s.k;
          for (int t = 0; t < s.T; ++t) act_w[n_routed][t] = 1.f;
        }
        n_act_s = n_routed + (s.has_shared ? 1 : 0);
      }
    }
    __syncthreads();
    const int n_act = n_act_s;
    const int units = n_act * s.I;
    const size_t row_bytes = (size_t)s.d * 2, drow_bytes = (size_t)s.I * 2;
    // L2 prefetch of everything this block reads in phases B and C, so the
    // memory system sees all of it at once
    {
      const int my_units = (units > b) ? (units - b + G - 1) / G : 0;
      for (int q = tid; q < 2 * my_units; q += kThreads) {
        const int u = b + (q >> 1) * G;
        const int a = u / s.I, i = u - a * s.I;
        const int e = act_e[a];
        const uint16_t* W = (e < s.E) ? A.gate_up + (size_t)e * 2 * s.I * s.d : A.shared_w;
        prefetch_l2(W + (size_t)((q & 1) ? s.I + i : i) * s.d, (uint32_t)row_bytes);
      }
      const int my_rows = (s.d > b) ? (s.d - b + G - 1) / G : 0;
      for (int q = tid; q < my_rows * n_act; q += kThreads) {
        const int r = b + (q / n_act) * G, a = q % n_act;
        const int e = act_e[a];
        const uint16_t* Wd = (e < s.E) ? A.down + (size_t)e * s.d * s.I : A.shared_w + (size_t)2 * s.I * s.d;
        prefetch_l2(Wd + (size_t)r * s.I, (uint32_t)drow_bytes);
      }
    }
    // gate/up GEMV + SwiGLU; units dealt to blocks first (u = b + j * G)
    for (int j = warp;; j += kWarps) {
      const int u = b + j * G;
      if (u >= units) break;
      const int a = u / s.I, i = u - a * s.I;
      const int e = act_e[a];
      const uint16_t* W = (e < s.E) ? A.gate_up + (size_t)e * 2 * s.I * s.d : A.shared_w;
      const uint4* grow = reinterpret_cast<const uint4*>(W + (size_t)i * s.d) + lane;
      const uint4* urow = reinterpret_cast<const uint4*>(W + (size_t)(s.I + i) * s.d) + lane;
      uint4 gv[NCH], uv[NCH];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        gv[c] = __ldcg(grow + 32 * c);
        uv[c] = __ldcg(urow + 32 * c);
      }
      unsigned mm = act_m[a];
      int row = act_row[a];
      while (mm) {
        const int t = __ffs(mm) - 1;
        mm &= mm - 1u;
        const float* xr = big + (size_t)t * s.d + lane * 8;
        float g = 0.f, up = 0.f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          g += dot8(gv[c], xr + 256 * c);
          up += dot8(uv[c], xr + 256 * c);
        }
        g = warp_sum(g);
        up = warp_sum(up);
        if (lane == 0) sc.h_gemv[(size_t)row * s.I + i] = silu(g) * up;
        ++row;
      }
    }
  }
  ok = grid_sync(A.bar, 2, A.ctl, &flag_s) && ok;

  // ---------------------------------------------------------------- phase C
  if (ok) {
    const int n_act = n_act_s;
    const int pairs = s.T * s.k + (s.has_shared ? s.T : 0);
    constexpr int kBatch = (18 / NCI) > 0 ? (18 / NCI) : 1;  // experts whose rows are loaded together
    // this warp's first output row: its down rows need nothing from phase B,
    // so they are requested before h is staged
    const int r0 = b + warp * G;
    uint4 wv[kBatch][NCI];
    if (r0 < s.d) {
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        if (q < n_act) {
          const int e = act_e[q];
          const uint16_t* Wd = (e < s.E) ? A.down + (size_t)e * s.d * s.I : A.shared_w + (size_t)2 * s.I * s.d;
          const uint4* row = reinterpret_cast<const uint4*>(Wd + (size_t)r0 * s.I) + lane;
#pragma unroll
          for (int c = 0; c < NCI; ++c) wv[q][c] = __ldcg(row + 32 * c);
        }
      }
    }
    {
      const float4* src = reinterpret_cast<const float4*>(sc.h_gemv);
      float4* dst = reinterpret_cast<float4*>(big);
      const int n4 = (pairs * s.I) >> 2;
      for (int i = tid; i < n4; i += kThreads) dst[i] = __ldcg(src + i);
    }
    __syncthreads();
    for (int j = warp;; j += kWarps) {
      const int r = b + j * G;
      if (r >= s.d) break;
      // per-lane partial sums of every token, reduced across the warp once at the end
      float part[MAXT];
#pragma unroll
      for (int t = 0; t < MAXT; ++t) part[t] = 0.f;
      for (int a0 = 0; a0 < n_act; a0 += kBatch) {
        if (j != warp || a0 > 0) {
#pragma unroll
          for (int q = 0; q < kBatch; ++q) {
            if (a0 + q < n_act) {
              const int e = act_e[a0 + q];
              const uint16_t* Wd =
                  (e < s.E) ? A.down + (size_t)e * s.d * s.I : A.shared_w + (size_t)2 * s.I * s.d;
              const uint4* row = reinterpret_cast<const uint4*>(Wd + (size_t)r * s.I) + lane;
#pragma unroll
              for (int c = 0; c < NCI; ++c) wv[q][c] = __ldcg(row + 32 * c);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          if (a0 + q >= n_act) break;
          const unsigned mm = act_m[a0 + q];
          const int row0 = act_row[a0 + q];
#pragma unroll
          for (int t = 0; t < MAXT; ++t) {
            if ((mm >> t) & 1u) {
              const int row = row0 + __popc(mm & ((1u << t) - 1u));
              const float* hr = big + (size_t)row * s.I + lane * 8;
              float dsum = 0.f;
#pragma unroll
              for (int c = 0; c < NCI; ++c) dsum += dot8(wv[q][c], hr + 256 * c);
              part[t] = fmaf(act_w[a0 + q][t], dsum, part[t]);
            }
          }
        }
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
  // leave: the last block out resets the barrier counters for the next launch
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(A.bar + 1, 1u) == (unsigned)G - 1) {
      A.bar[0] = 0u;
      A.bar[1] = 0u;
      __threadfence();
    }
  }
}

size_t decode_smem_bytes(const Shapes& s) { return decode_big_bytes(s); }

template <int NCH, int NCI, int MAXT>
static const void* pick(bool xbf16) {
  return xbf16 ? (const void*)decode_fused_kernel<NCH, NCI, true, MAXT>
               : (const void*)decode_fused_kernel<NCH, NCI, false, MAXT>;
}

template <int MAXT>
static const void* pick_shape(const Shapes& s) {
  const int nch = s.d / 256, nci = s.I / 256;
  if (nci == 2) {
    if (nch == 2) return pick<2, 2, MAXT>(s.x_bf16);
    if (nch == 4) return pick<4, 2, MAXT>(s.x_bf16);
    if (nch == 8) return pick<8, 2, MAXT>(s.x_bf16);
  } else if (nci == 1) {
    if (nch == 2) return pick<2, 1, MAXT>(s.x_bf16);
    if (nch == 4) return pick<4, 1, MAXT>(s.x_bf16);
    if (nch == 8) return pick<8, 1, MAXT>(s.x_bf16);
  } else if (nci == 4) {
    if (nch == 4) return pick<4, 4, MAXT>(s.x_bf16);
    if (nch == 8) return pick<8, 4, MAXT>(s.x_bf16);
  }
  return nullptr;
}

static const void* decode_kernel_for(const Shapes& s) {
  if (s.T <= 1) return pick_shape<1>(s);
  if (s.T <= 16) return pick_shape<16>(s);
  return nullptr;
}

bool decode_supported(const Shapes& s, int max_smem) {
  return s.T <= 16 && s.d % 256 == 0 && s.I % 256 == 0 && decode_kernel_for(s) != nullptr &&
         decode_smem_bytes(s) <= (size_t)max_smem;
}

cudaError_t prepare_decode_kernels(int max_smem) {
  for (int T : {1, 16})
    for (int d : {512, 1024, 2048})
      for (int I : {256, 512, 1024})
        for (int xb = 0; xb < 2; ++xb) {
          Shapes s{};
          s.T = T;
          s.d = d;
          s.I = I;
          s.x_bf16 = xb;
          const void* k = decode_kernel_for(s);
          if (!k) continue;
          cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
          if (err != cudaSuccess) return err;
        }
  return cudaSuccess;
}

int decode_blocks_per_sm(const Shapes& s) {
  int n = 0;
  const void* k = decode_kernel_for(s);
  if (!k || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, decode_smem_bytes(s)) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t launch_decode_fused(const Shapes& s, const void* x, const float* wr, const float* rb,
                                const uint16_t* gate_up, const uint16_t* down, const uint16_t* shared_w, void* y,
                                const Scratch& sc, const DevCtl& ctl, unsigned* bar, int num_sms, cudaStream_t st) {
  DecodeArgs a;
  a.s = s;
  a.x = x;
  a.wr = wr;
  a.rb = rb;
  a.gate_up = gate_up;
  a.down = down;
  a.shared_w = shared_w;
  a.y = y;
  a.sc = sc;
  a.ctl = ctl;
  a.bar = bar;
  const void* k = decode_kernel_for(s);
  if (!k) return cudaErrorInvalidValue;
  void* params[] = {&a};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = decode_smem_bytes(s);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, k, params);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free variant of the fused decode layer (moe_decode_noalloc).
//
// Some callers cannot call cudaMalloc, so they cannot create a context with
// moe_init: code that builds its GPU work inside an ongoing CUDA stream capture
// (allocation is not allowed there), and processes that run under a strict
// no-allocation policy (real-time serving loops, or hosts whose device memory
// is owned by another allocator).  For them the same kernel runs on scratch
// memory that is part of the library image: one file-scope device array, sized
// for the limits below, that every GPU loading the library holds until exit.
// The host learns its device address once per device with
// cudaGetSymbolAddress; the array's name in host code is only a host-side
// stand-in, never a device address.
// ---------------------------------------------------------------------------
#include <mutex>

using namespace moe;

namespace {

constexpr int kNoAllocMaxT = 16;
constexpr int kNoAllocMaxTopK = 8;
constexpr int kNoAllocMaxInter = 1024;
constexpr size_t kNoAllocH = (size_t)kNoAllocMaxT * (kNoAllocMaxTopK + 1) * kNoAllocMaxInter * 4;  // fp32 h rows
constexpr size_t kNoAllocLogits = (size_t)kNoAllocMaxT * kMaxExperts * 4;
constexpr size_t kNoAllocPicks = (size_t)kNoAllocMaxT * kNoAllocMaxTopK * 4;
constexpr size_t kNoAllocOffLogits = kNoAllocH;
constexpr size_t kNoAllocOffIdx = kNoAllocOffLogits + kNoAllocLogits;
constexpr size_t kNoAllocOffW = kNoAllocOffIdx + kNoAllocPicks;
constexpr size_t kNoAllocOffWords = kNoAllocOffW + kNoAllocPicks;  // [0] status, [2..3] barrier counters
constexpr size_t kNoAllocBytes = kNoAllocOffWords + 256;

struct NoAllocDevice {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of the array on this device
  int sms = 0;
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

}  // namespace

// The scratch array (about 600 KB).  Every call shares it and it keeps the
// last call's contents; the barrier counters, which must start at zero, are
// cleared at the start of every call.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

extern "C" int moe_decode_noalloc(const void* x, int T, int x_dtype, int d, int n_experts, int inter, int top_k,
                                  const float* router_w, const float* router_b, const void* experts_gate_up,
                                  const void* experts_down, const void* shared_w, void* y, unsigned* status,
                                  void* stream) {
  if (T < 0 || d <= 0 || n_experts <= 0 || inter <= 0 || top_k <= 0) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !experts_gate_up || !experts_down || !y) return MOE_ERR_ARG;
  if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_ARG;
  if (top_k > n_experts) return MOE_ERR_ARG;
  // the fixed size of the scratch array
  if (T > kNoAllocMaxT || top_k > kNoAllocMaxTopK || inter > kNoAllocMaxInter || n_experts > kMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  const void* ptrs[] = {x, router_w, router_b, experts_gate_up, experts_down, shared_w, y, status};
  for (const void* p : ptrs)
    if (p && (reinterpret_cast<uintptr_t>(p) & 15u)) return MOE_ERR_ALIGN;
  Shapes s{};
  s.T = T;
  s.d = d;
  s.E = n_experts;
  s.I = inter;
  s.k = top_k;
  s.has_shared = shared_w != nullptr;
  s.x_bf16 = x_dtype == MOE_BF16;
  const int smem_limit = 200 * 1024;
  if (!decode_supported(s, smem_limit)) return MOE_ERR_UNSUPPORTED;

  // set-up, once per device, with that device current
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_CUDA;
  NoAllocDevice nd;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocDevice& slot = g_noalloc_dev[dev];
    if (!slot.ready) {
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MOE_ERR_CUDA;
      if (!(prop.major == 10 && prop.minor == 3)) return MOE_ERR_UNSUPPORTED;
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      if (prepare_decode_kernels(smem_limit) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      slot.base = static_cast<unsigned char*>(p);
      slot.sms = prop.multiProcessorCount;
      slot.ready = true;
    }
    nd = slot;
  }
  if (decode_blocks_per_sm(s) < 1) return MOE_ERR_UNSUPPORTED;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* words = reinterpret_cast<unsigned*>(nd.base + kNoAllocOffWords);
  unsigned* bar = words + 2;
  if (cudaMemsetAsync(bar, 0, 2 * sizeof(unsigned), st) != cudaSuccess) return MOE_ERR_CUDA;
  Scratch sc{};
  sc.h_gemv = reinterpret_cast<float*>(nd.base);
  sc.logits = reinterpret_cast<float*>(nd.base + kNoAllocOffLogits);
  sc.idx = reinterpret_cast<int*>(nd.base + kNoAllocOffIdx);
  sc.w = reinterpret_cast<float*>(nd.base + kNoAllocOffW);
  sc.status = status ? status : words;
  sc.gridbar = bar;
  DevCtl ctl;
  ctl.status = sc.status;
  ctl.spin_limit = 1000000000LL;
  ctl.stall = 0;
  const cudaError_t err =
      launch_decode_fused(s, x, router_w, router_b, static_cast<const uint16_t*>(experts_gate_up),
                          static_cast<const uint16_t*>(experts_down), static_cast<const uint16_t*>(shared_w), y, sc,
                          ctl, bar, nd.sms, st);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
