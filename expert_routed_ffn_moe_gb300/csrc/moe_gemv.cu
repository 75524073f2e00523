// Small-T expert FFN path: bandwidth-bound GEMV over the selected experts only.
//
// "Optimizing on-device inference for Apple Silicon", section "Optimizing the
// single-row weight path": with one activation row per step a GEMV is limited
// by weight reads, so a group of 32 threads cooperates on one output while
// reading different parts of the weight matrix in parallel.  Section "Reducing
// intermediate and state traffic": the two expert input projections are fused
// with the gated activation, and the output projection with the routing score
// and the shared expert's result, so temporaries stay in registers.
//
// Kernel 1 (gate_up + SwiGLU): one warp per (active expert, inner neuron i).
// The warp streams gate row i and up row i of that expert once, with 16-byte
// loads, and dots them with every token routed to the expert (x staged in
// shared memory).  h[i] = silu(g) * u goes to an fp32 buffer, grouped rows.
//
// Kernel 2 (down + weighted combine + shared): one warp per output feature r.
// For each active expert in ascending id (the shared expert last) the warp
// streams row r of that expert's down projection once and dots it with the
// staged h of each token routed there; the routing weight scales the result
// and each token accumulates its own sum in fp32.  y is written directly.
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kGemvWarps = 16;

MOE_DEV uint4 ld_stream(const uint4* p) { return __ldcs(p); }

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

// MAXCH: largest number of 16-byte chunks per lane per weight row (d / 256).
template <int MAXCH, bool XBF16>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_gate_up_kernel(Shapes s, const void* __restrict__ x,
                                                                       const uint16_t* __restrict__ gate_up,
                                                                       const uint16_t* __restrict__ shared_w,
                                                                       Scratch sc, DevCtl ctl) {
  extern __shared__ __align__(16) float xs[];  // [T][d] fp32
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nx = s.T * s.d;
  if (XBF16) {
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    for (int i = threadIdx.x; i < nx; i += blockDim.x) xs[i] = __uint_as_float(uint32_t(xb[i]) << 16);
  } else {
    const float* xf = static_cast<const float*>(x);
    for (int i = threadIdx.x; i < nx; i += blockDim.x) xs[i] = xf[i];
  }
  __syncthreads();
  const int nch = s.d >> 8;
  const int n_active = sc.meta[1];
  const int units = n_active * s.I;
  // units are dealt to blocks first (u = block + j * grid), so every SM streams
  // the same number of weight bytes to within one unit
  for (int j = warp;; j += kGemvWarps) {
    const int u = blockIdx.x + j * gridDim.x;
    if (u >= units) break;
    const int a = u / s.I, i = u - a * s.I;
    const int e = sc.active[a];
    if (e < 0 || e > s.E || (e == s.E && !s.has_shared)) {
      if (lane == 0) raise_status(ctl, kStatusBounds);
      continue;
    }
    const uint16_t* W = (e < s.E) ? gate_up + (size_t)e * 2 * s.I * s.d : shared_w;
    const uint4* grow = reinterpret_cast<const uint4*>(W + (size_t)i * s.d) + lane;
    const uint4* urow = reinterpret_cast<const uint4*>(W + (size_t)(s.I + i) * s.d) + lane;
    uint4 gv[MAXCH], uv[MAXCH];
#pragma unroll
    for (int c = 0; c < MAXCH; ++c) {
      if (c < nch) {
        gv[c] = ld_stream(grow + 32 * c);
        uv[c] = ld_stream(urow + 32 * c);
      }
    }
    const int beg = sc.offsets[e], cnt = sc.counts[e];
    for (int p = 0; p < cnt; ++p) {
      const int t = sc.perm[beg + p];
      if (t < 0 || t >= s.T) {
        if (lane == 0) raise_status(ctl, kStatusBounds);
        continue;
      }
      const float* xr = xs + (size_t)t * s.d + lane * 8;
      float g = 0.f, up = 0.f;
#pragma unroll
      for (int c = 0; c < MAXCH; ++c) {
        if (c < nch) {
          g += dot8(gv[c], xr + 256 * c);
          up += dot8(uv[c], xr + 256 * c);
        }
      }
      g = warp_sum(g);
      up = warp_sum(up);
      if (lane == 0) sc.h_gemv[(size_t)(beg + p) * s.I + i] = silu(g) * up;
    }
  }
}

// MAXCI: largest number of 16-byte chunks per lane per down row (I / 256).
template <int MAXCI, bool YBF16>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_down_kernel(Shapes s, const uint16_t* __restrict__ down,
                                                                    const uint16_t* __restrict__ shared_w,
                                                                    void* __restrict__ y, Scratch sc,
                                                                    DevCtl ctl) {
  extern __shared__ __align__(16) float hs[];  // [n_pairs][I] fp32, then pair weight, then pair token
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tk = s.T * s.k;
  const int n_pairs = tk + (s.has_shared ? s.T : 0);
  float* pw = hs + (size_t)n_pairs * s.I;
  int* pt = reinterpret_cast<int*>(pw + n_pairs);
  {
    const float4* src = reinterpret_cast<const float4*>(sc.h_gemv);
    float4* dst = reinterpret_cast<float4*>(hs);
    const int n4 = (n_pairs * s.I) >> 2;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = __ldcg(src + i);
  }
  for (int q = threadIdx.x; q < tk; q += blockDim.x) {
    const int p = sc.slot[q];
    if (p < 0 || p >= tk) {
      raise_status(ctl, kStatusBounds);
      continue;
    }
    pw[p] = sc.w[q];
    pt[p] = q / s.k;
  }
  for (int t = threadIdx.x; t < n_pairs - tk; t += blockDim.x) {
    pw[tk + t] = s.shared_gate ? sc.sgate[t] : 1.f;
    pt[tk + t] = t;
  }
  __syncthreads();
  const int nci = s.I >> 8;
  const int n_active = sc.meta[1];
  for (int j = warp;; j += kGemvWarps) {
    const int r = blockIdx.x + j * gridDim.x;
    if (r >= s.d) break;
    float acc = 0.f;  // lane t accumulates token t
    constexpr int kBatch = (16 / MAXCI) > 0 ? (16 / MAXCI) : 1;  // experts whose rows are in flight together
    for (int a0 = 0; a0 < n_active; a0 += kBatch) {
      uint4 wv[kBatch][MAXCI];
      int ev[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        ev[b] = (a0 + b < n_active) ? sc.active[a0 + b] : -1;
        const int e = ev[b];
        if (e >= 0 && e <= s.E) {
          const uint16_t* Wd = (e < s.E) ? down + (size_t)e * s.d * s.I : shared_w + (size_t)2 * s.I * s.d;
          const uint4* row = reinterpret_cast<const uint4*>(Wd + (size_t)r * s.I) + lane;
#pragma unroll
          for (int c = 0; c < MAXCI; ++c)
            if (c < nci) wv[b][c] = ld_stream(row + 32 * c);
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int e = ev[b];
        if (e < 0) continue;
        if (e > s.E) {
          if (lane == 0) raise_status(ctl, kStatusBounds);
          continue;
        }
        const int beg = sc.offsets[e], cnt = sc.counts[e];
        for (int p = beg; p < beg + cnt; ++p) {
          const float* hr = hs + (size_t)p * s.I + lane * 8;
          float dsum = 0.f;
#pragma unroll
          for (int c = 0; c < MAXCI; ++c)
            if (c < nci) dsum += dot8(wv[b][c], hr + 256 * c);
          dsum = warp_sum(dsum);
          if (lane == pt[p]) acc = fmaf(pw[p], dsum, acc);
        }
      }
    }
    if (lane < s.T) {
      if (YBF16) {
        const __nv_bfloat16 v = __float2bfloat16_rn(acc);
        static_cast<uint16_t*>(y)[(size_t)lane * s.d + r] = *reinterpret_cast<const uint16_t*>(&v);
      } else {
        static_cast<float*>(y)[(size_t)lane * s.d + r] = acc;
      }
    }
  }
}

size_t gemv_gate_up_smem(const Shapes& s) { return (size_t)s.T * s.d * sizeof(float); }
size_t gemv_down_smem(const Shapes& s) {
  const size_t n_pairs = (size_t)s.T * s.k + (s.has_shared ? s.T : 0);
  return n_pairs * s.I * sizeof(float) + n_pairs * 8;
}

template <int MAXCH>
static cudaError_t gate_up_dispatch(const Shapes& s, const void* x, const uint16_t* gu, const uint16_t* sw,
                                    const Scratch& sc, const DevCtl& ctl, int num_sms, cudaStream_t st) {
  const size_t smem = gemv_gate_up_smem(s);
  if (s.x_bf16)
    gemv_gate_up_kernel<MAXCH, true><<<num_sms, kGemvWarps * 32, smem, st>>>(s, x, gu, sw, sc, ctl);
  else
    gemv_gate_up_kernel<MAXCH, false><<<num_sms, kGemvWarps * 32, smem, st>>>(s, x, gu, sw, sc, ctl);
  return cudaGetLastError();
}

cudaError_t launch_gemv_gate_up(const Shapes& s, const void* x, const uint16_t* gate_up, const uint16_t* shared_w,
                                const Scratch& sc, const DevCtl& ctl, int num_sms, cudaStream_t st) {
  const int nch = s.d / 256;
  if (nch <= 2) return gate_up_dispatch<2>(s, x, gate_up, shared_w, sc, ctl, num_sms, st);
  if (nch <= 4) return gate_up_dispatch<4>(s, x, gate_up, shared_w, sc, ctl, num_sms, st);
  if (nch <= 8) return gate_up_dispatch<8>(s, x, gate_up, shared_w, sc, ctl, num_sms, st);
  return gate_up_dispatch<16>(s, x, gate_up, shared_w, sc, ctl, num_sms, st);
}

template <int MAXCI>
static cudaError_t down_dispatch(const Shapes& s, const uint16_t* dn, const uint16_t* sw, void* y,
                                 const Scratch& sc, const DevCtl& ctl, int num_sms, cudaStream_t st) {
  const size_t smem = gemv_down_smem(s);
  if (s.x_bf16)
    gemv_down_kernel<MAXCI, true><<<num_sms, kGemvWarps * 32, smem, st>>>(s, dn, sw, y, sc, ctl);
  else
    gemv_down_kernel<MAXCI, false><<<num_sms, kGemvWarps * 32, smem, st>>>(s, dn, sw, y, sc, ctl);
  return cudaGetLastError();
}

// Shared-memory opt-in of every GEMV instantiation, done once at context
// creation (never inside a launch sequence that may be under stream capture).
cudaError_t prepare_gemv_kernels(int max_smem) {
  const void* ks[] = {
      (const void*)gemv_gate_up_kernel<2, true>,  (const void*)gemv_gate_up_kernel<2, false>,
      (const void*)gemv_gate_up_kernel<4, true>,  (const void*)gemv_gate_up_kernel<4, false>,
      (const void*)gemv_gate_up_kernel<8, true>,  (const void*)gemv_gate_up_kernel<8, false>,
      (const void*)gemv_gate_up_kernel<16, true>, (const void*)gemv_gate_up_kernel<16, false>,
      (const void*)gemv_down_kernel<1, true>,     (const void*)gemv_down_kernel<1, false>,
      (const void*)gemv_down_kernel<2, true>,     (const void*)gemv_down_kernel<2, false>,
      (const void*)gemv_down_kernel<4, true>,     (const void*)gemv_down_kernel<4, false>,
      (const void*)gemv_down_kernel<8, true>,     (const void*)gemv_down_kernel<8, false>};
  for (const void* k : ks) {
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_gemv_down(const Shapes& s, const uint16_t* down, const uint16_t* shared_w, void* y,
                             const Scratch& sc, const DevCtl& ctl, int num_sms, cudaStream_t st) {
  const int nci = s.I / 256;
  if (nci <= 1) return down_dispatch<1>(s, down, shared_w, y, sc, ctl, num_sms, st);
  if (nci <= 2) return down_dispatch<2>(s, down, shared_w, y, sc, ctl, num_sms, st);
  if (nci <= 4) return down_dispatch<4>(s, down, shared_w, y, sc, ctl, num_sms, st);
  return down_dispatch<8>(s, down, shared_w, y, sc, ctl, num_sms, st);
}

}  // namespace moe
