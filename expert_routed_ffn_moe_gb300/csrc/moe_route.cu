// Routing: router logits, top-k selection with renormalised weights, and the
// GPU-resident grouping of tokens by expert (histogram, exclusive prefix,
// stable scatter, and the list of grouped-GEMM tiles).
//
// "Optimizing on-device inference for Apple Silicon", section "Qwen creates
// three different workload shapes": the router scores 256 experts per token
// and keeps eight.  Section "Keeping expert routing on the GPU": a histogram
// counts the assignments of each expert, a prefix pass turns the counts into
// start offsets, a scatter places the rows into their expert groups, and a
// block map lists the fixed-size tiles the grouped GEMM must process -- all
// inside one command stream, without a CPU round trip.
//
// Grouping here is deterministic: tokens are cut into chunks of 32; each chunk
// records, per expert, a 32-bit mask of the tokens that chose it.  The rank of
// token t inside its expert group is then (offset of the expert) + (tokens of
// the expert in earlier chunks) + popc(mask & bits below t), which yields the
// stable (expert asc, token asc) order without atomics deciding any position.
#include <float.h>
#include <math.h>

#include "moe_internal.h"

namespace moe {

// ----------------------------------------------------------- router logits
// Small T: one warp per (expert, group of up to 16 tokens); the expert's row
// of router_w is streamed once per group with 16-byte loads.
template <bool XBF16>
__global__ void __launch_bounds__(256) router_logits_small_kernel(Shapes s, const void* __restrict__ x,
                                                                   const float* __restrict__ wr,
                                                                   float* __restrict__ logits) {
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int e = gw % s.E;
  const int g = gw / s.E;
  const int t0 = g * 16;
  if (t0 >= s.T) return;
  const int nt = min(16, s.T - t0);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  const float4* wrow = reinterpret_cast<const float4*>(wr + (size_t)e * s.d);
  const int n4 = s.d >> 2;
#pragma unroll 4
  for (int c = lane; c < n4; c += 32) {
    const float4 wv = __ldg(wrow + c);
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      if (tt < nt) {
        float4 xv;
        if (XBF16) {
          const uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) +
                                                                 (size_t)(t0 + tt) * s.d) + c);
          xv = make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
        } else {
          xv = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)(t0 + tt) * s.d) + c);
        }
        acc[tt] = fmaf(xv.x, wv.x, acc[tt]);
        acc[tt] = fmaf(xv.y, wv.y, acc[tt]);
        acc[tt] = fmaf(xv.z, wv.z, acc[tt]);
        acc[tt] = fmaf(xv.w, wv.w, acc[tt]);
      }
    }
  }
#pragma unroll
  for (int tt = 0; tt < 16; ++tt) {
    if (tt < nt) {
      const float r = warp_sum(acc[tt]);
      if (lane == 0) logits[(size_t)(t0 + tt) * s.E + e] = r;
    }
  }
}

// Larger T: a 64-token x 64-expert tile per block, 16-deep k slices staged in
// shared memory, 4 x 4 outputs per thread, fp32 FMA.
template <bool XBF16>
__global__ void __launch_bounds__(256) router_logits_tiled_kernel(Shapes s, const void* __restrict__ x,
                                                                   const float* __restrict__ wr,
                                                                   float* __restrict__ logits) {
  __shared__ float xs[16][64 + 4];
  __shared__ float ws[16][64 + 4];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
  const int ty = tid >> 4, tx = tid & 15;
  float acc[4][4] = {};
  // loader mapping: row r = tid / 4 (0..63), k quad q = tid % 4 (4 values each)
  const int lr = tid >> 2, lq = (tid & 3) * 4;
  for (int k0 = 0; k0 < s.d; k0 += 16) {
    {
      const int t = t0 + lr;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < s.T) {
        if (XBF16) {
          const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + (size_t)t * s.d + k0 + lq);
          v = make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
        } else {
          v = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)t * s.d + k0 + lq);
        }
      }
      xs[lq + 0][lr] = v.x;
      xs[lq + 1][lr] = v.y;
      xs[lq + 2][lr] = v.z;
      xs[lq + 3][lr] = v.w;
      const int e = e0 + lr;
      float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < s.E) u = *reinterpret_cast<const float4*>(wr + (size_t)e * s.d + k0 + lq);
      ws[lq + 0][lr] = u.x;
      ws[lq + 1][lr] = u.y;
      ws[lq + 2][lr] = u.z;
      ws[lq + 3][lr] = u.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= s.T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < s.E) logits[(size_t)t * s.E + e] = acc[i][j];
    }
  }
}

cudaError_t launch_router_logits_simt(const Shapes& s, const void* x, const float* wr, const float*,
                                      const Scratch& sc, cudaStream_t st) {
  if (s.T <= 64) {
    const int warps = s.E * ((s.T + 15) / 16);
    const dim3 grid((warps + 7) / 8);
    if (s.x_bf16)
      router_logits_small_kernel<true><<<grid, 256, 0, st>>>(s, x, wr, sc.logits);
    else
      router_logits_small_kernel<false><<<grid, 256, 0, st>>>(s, x, wr, sc.logits);
  } else {
    const dim3 grid((s.T + 63) / 64, (s.E + 63) / 64);
    if (s.x_bf16)
      router_logits_tiled_kernel<true><<<grid, 256, 0, st>>>(s, x, wr, sc.logits);
    else
      router_logits_tiled_kernel<false><<<grid, 256, 0, st>>>(s, x, wr, sc.logits);
  }
  return cudaGetLastError();
}

// Router weights split into three bf16 terms, hi = bf16(w), mid = bf16(w - hi),
// lo = bf16(w - hi - mid), stacked as [3E, d].  hi + mid + lo equals w to about
// 2^-25 relative, and every bf16 x bf16 product is exact in fp32, so bf16 x
// times the three terms on the tensor cores (fp32 accumulation) reproduces the
// fp32 logits.
__global__ void router_split_kernel(int n, const float* __restrict__ wr, uint16_t* __restrict__ out) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float v = wr[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    out[i] = *reinterpret_cast<const uint16_t*>(&hi);
    out[n + i] = *reinterpret_cast<const uint16_t*>(&mid);
    out[2 * n + i] = *reinterpret_cast<const uint16_t*>(&lo);
  }
}

cudaError_t launch_router_split_weights(const Shapes& s, const float* wr, const Scratch& sc, cudaStream_t st) {
  const int n = s.E * s.d;
  router_split_kernel<<<(n + 1023) / 1024, 256, 0, st>>>(n, wr, sc.wr_split);
  return cudaGetLastError();
}

// ----------------------------------------------------------- selection
// One block per chunk of 32 tokens, one warp per token (warp_top_k: each
// lane holds 8 logits; k rounds of warp reductions, ties to the lower expert
// id).  The weights are the softmax over all E experts renormalised over the
// picks; the picks are written in ascending expert id, and the chunk's
// per-expert token masks feed the grouping.  For a sigmoid-gated shared
// expert the warp also writes the token's gate, sigmoid(x_t . gate_w).
__global__ void __launch_bounds__(1024) select_kernel(Shapes s, const float* __restrict__ rb, int parts, Scratch sc,
                                                      DevCtl ctl, const void* __restrict__ x,
                                                      const float* __restrict__ gate_w) {
  __shared__ unsigned mask[kMaxExperts];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x, t0 = c * kChunk;
  const int nchunk = (s.T + kChunk - 1) / kChunk;
  for (int e = tid; e < s.E; e += blockDim.x) mask[e] = 0u;
  __syncthreads();
  const int t = t0 + warp;
  if (t < s.T) {
    float v[8], u[8];  // logits with and without the router bias
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      float l = -INFINITY;
      if (e < s.E) {
        const size_t te = (size_t)t * s.E + e;
        if (parts == 3) {  // tensor-core partial logits of the lo, mid and hi weight terms, small first
          const size_t part = (size_t)s.T * s.E;
          l = (sc.logits[2 * part + te] + sc.logits[part + te]) + sc.logits[te];
        } else {
          l = sc.logits[te];
        }
        u[i] = l;
        if (rb) l += rb[e];
      }
      v[i] = l;
      if (e >= s.E) u[i] = -INFINITY;
    }
    int pe, rank;
    float pw;
    if (!warp_top_k(v, s.E, s.k, lane, pe, pw, rank) && lane == 0) raise_status(ctl, kStatusBounds);
    if (s.bias_sel) pw = warp_pick_weight(warp_logit_of(u, pe), s.k, lane);
    if (lane < s.k) {
      sc.idx[(size_t)t * s.k + rank] = pe;
      sc.w[(size_t)t * s.k + rank] = pw;
      atomicOr(&mask[pe], 1u << warp);
    }
    if (s.shared_gate) {
      const float4* g4 = reinterpret_cast<const float4*>(gate_w);
      float acc = 0.f;
      for (int c = lane; c < s.d / 4; c += 32) {
        float4 xv;
        if (s.x_bf16) {
          const uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + (size_t)t * s.d) + c);
          xv = make_float4(bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y));
        } else {
          xv = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)t * s.d) + c);
        }
        const float4 gv = __ldg(g4 + c);
        acc = fmaf(xv.x, gv.x, acc);
        acc = fmaf(xv.y, gv.y, acc);
        acc = fmaf(xv.z, gv.z, acc);
        acc = fmaf(xv.w, gv.w, acc);
      }
      acc = warp_sum(acc);
      if (lane == 0) sc.sgate[t] = sigmoid(acc);
    }
  }
  __syncthreads();
  for (int e = tid; e < s.E; e += blockDim.x) {
    const unsigned m = mask[e];
    sc.chunk_mask[(size_t)c * s.E + e] = m;
    sc.chunk_base[(size_t)e * nchunk + c] = __popc(m);
  }
}

cudaError_t launch_select(const Shapes& s, const float* rb, int parts, const Scratch& sc, const DevCtl& ctl,
                          cudaStream_t st, const void* x, const float* gate_w) {
  if (s.shared_gate && (!x || !gate_w)) return cudaErrorInvalidValue;
  const int nchunk = (s.T + kChunk - 1) / kChunk;
  select_kernel<<<nchunk, kChunk * 32, 0, st>>>(s, rb, parts, sc, ctl, x, gate_w);
  return cudaGetLastError();
}

// ----------------------------------------------------------- grouping
// Block-wide exclusive scan of one int per thread (256 threads).
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_tot[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, all = 0;
  for (int i = 0; i < 8; ++i) {
    base += (i < warp) ? warp_tot[i] : 0;
    all += warp_tot[i];
  }
  __syncthreads();
  *total = all;
  return base + incl - v;
}

// Phase 1 (every block): one warp per expert turns the per-chunk counts into
// exclusive prefixes over chunks and writes the expert's total.
// Phase 2 (the last block to finish): expert offsets, the shared expert's
// group, the grouped-GEMM m-tiles and the list of active experts.
__global__ void __launch_bounds__(256) group_scan_kernel(Shapes s, Scratch sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nchunk = (s.T + kChunk - 1) / kChunk;
  const int e = blockIdx.x * 8 + warp;
  if (e < s.E) {
    int* col = sc.chunk_base + (size_t)e * nchunk;
    int carry = 0;
    for (int c0 = 0; c0 < nchunk; c0 += 32) {
      const int c = c0 + lane;
      const int v = c < nchunk ? col[c] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (c < nchunk) col[c] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sc.counts[e] = carry;
  }
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (threadIdx.x == 0) is_last = (atomicAdd(&sc.tickets[0], 1u) == gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  const int tid = threadIdx.x;
  const int cnt = tid < s.E ? __ldcg(sc.counts + tid) : 0;
  int total;
  const int off = block_exclusive_scan(cnt, &total);
  if (tid < s.E) sc.offsets[tid] = off;
  const int shared_cnt = s.has_shared ? s.T : 0;
  if (tid == 0) {
    sc.offsets[s.E] = total;  // == T * k
    sc.offsets[s.E + 1] = total + shared_cnt;
    sc.counts[s.E] = shared_cnt;
  }
  const int nm = (cnt + kBM - 1) / kBM;
  int mt_total;
  const int mt_off = block_exclusive_scan(nm, &mt_total);
  for (int i = 0; i < nm; ++i) {
    MTile m;
    m.e = tid;
    m.row0 = off + i * kBM;
    m.rows = min(kBM, cnt - i * kBM);
    m.pad = 0;
    sc.mtiles[mt_off + i] = m;
  }
  const int snm = (shared_cnt + kBM - 1) / kBM;
  for (int i = tid; i < snm; i += blockDim.x) {
    MTile m;
    m.e = s.E;
    m.row0 = total + i * kBM;
    m.rows = min(kBM, shared_cnt - i * kBM);
    m.pad = 0;
    sc.mtiles[mt_total + i] = m;
  }
  // the same tiles two by two within each group (the paired GEMMs load or
  // expand each weight tile once for both tiles of a pair).  The shared
  // expert's pairs, all full but the last, come first: the persistent GEMMs
  // take items in list order, so the heaviest are not left for the end.
  const int snp = (snm + 1) / 2;
  for (int i = tid; i < snp; i += blockDim.x) {
    MTile m;
    m.e = s.E;
    m.row0 = total + 2 * i * kBM;
    m.rows = min(kBM, shared_cnt - 2 * i * kBM);
    m.pad = max(0, min(kBM, shared_cnt - (2 * i + 1) * kBM));
    sc.mpairs[i] = m;
  }
  const int np = (nm + 1) / 2;
  int np_total;
  const int np_off = block_exclusive_scan(np, &np_total);
  for (int i = 0; i < np; ++i) {
    MTile m;
    m.e = tid;
    m.row0 = off + 2 * i * kBM;
    m.rows = min(kBM, cnt - 2 * i * kBM);
    m.pad = max(0, min(kBM, cnt - (2 * i + 1) * kBM));
    sc.mpairs[snp + np_off + i] = m;
  }
  int n_act;
  const int apos = block_exclusive_scan(cnt > 0 ? 1 : 0, &n_act);
  if (cnt > 0) sc.active[apos] = tid;
  if (tid == 0) {
    if (s.has_shared) sc.active[n_act] = s.E;
    sc.meta[2] = np_total + snp;
    sc.meta[0] = mt_total + snm;
    sc.meta[1] = n_act + (s.has_shared ? 1 : 0);
    sc.tickets[0] = 0u;  // ready for the next launch
  }
}

// One block per chunk: the grouped row of every (token, pick), and the shared
// expert's identity rows.
__global__ void __launch_bounds__(256) group_scatter_kernel(Shapes s, Scratch sc, DevCtl ctl) {
  const int c = blockIdx.x, t0 = c * kChunk;
  const int nchunk = (s.T + kChunk - 1) / kChunk;
  for (int p = threadIdx.x; p < kChunk * s.k; p += blockDim.x) {
    const int tl = p / s.k, j = p - tl * s.k;
    const int t = t0 + tl;
    if (t >= s.T) continue;
    const int e = sc.idx[(size_t)t * s.k + j];
    if (e < 0 || e >= s.E) {
      raise_status(ctl, kStatusBounds);
      continue;
    }
    const unsigned m = sc.chunk_mask[(size_t)c * s.E + e];
    const int pos = sc.offsets[e] + sc.chunk_base[(size_t)e * nchunk + c] + __popc(m & ((1u << tl) - 1u));
    if (kDebugChecks && (pos < 0 || pos >= s.T * s.k)) {
      raise_status(ctl, kStatusBounds);
      continue;
    }
    sc.perm[pos] = t;
    sc.slot[(size_t)t * s.k + j] = pos;
  }
  if (s.has_shared) {
    const int tl = threadIdx.x;
    if (tl < kChunk && t0 + tl < s.T) sc.perm[(size_t)s.T * s.k + t0 + tl] = t0 + tl;
  }
}

// The scatter fused with the row permutation of the grouped GEMM path: one
// warp per token computes the grouped positions of its k picks (as above),
// reads the token's x row once, and writes it, in bf16, to each of those rows
// of x_perm and to its shared-expert row -- instead of a scatter kernel that
// writes perm and a second pass that gathers x by perm.  With 4-bit weights
// each 8-column chunk is stored in the 4-bit GEMM's column order
// (q4_chunk_order).
template <bool XBF16>
__global__ void __launch_bounds__(256) group_scatter_rows_kernel(Shapes s, const void* __restrict__ x, Scratch sc,
                                                                 DevCtl ctl) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= s.T) return;
  const int c = t / kChunk, tl = t - c * kChunk;
  const int nchunk = (s.T + kChunk - 1) / kChunk;
  int pos = -1;
  if (lane < s.k) {
    const int e = sc.idx[(size_t)t * s.k + lane];
    if (e < 0 || e >= s.E) {
      raise_status(ctl, kStatusBounds);
    } else {
      const unsigned m = sc.chunk_mask[(size_t)c * s.E + e];
      pos = sc.offsets[e] + sc.chunk_base[(size_t)e * nchunk + c] + __popc(m & ((1u << tl) - 1u));
      if (kDebugChecks && (pos < 0 || pos >= s.T * s.k)) {
        raise_status(ctl, kStatusBounds);
        pos = -1;
      } else {
        sc.perm[pos] = t;
        sc.slot[(size_t)t * s.k + lane] = pos;
      }
    }
  }
  const long long shared_row = s.has_shared ? (long long)s.T * s.k + t : -1;
  if (lane == 0 && shared_row >= 0) sc.perm[shared_row] = t;
  // the row in 16-byte pieces of 8 bf16: lane takes pieces lane + 32 i
  const int pieces = s.d / 8;
  for (int p0 = 0; p0 < pieces; p0 += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int pc = p0 + lane + 32 * i;
      if (pc < pieces) {
        if (XBF16) {
          v[i] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)t * s.d) + pc);
        } else {
          const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(x) + (size_t)t * s.d);
          const float4 a = __ldg(src + 2 * pc), b = __ldg(src + 2 * pc + 1);
          v[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
        }
        if (s.q4) v[i] = q4_chunk_order(v[i]);  // the 4-bit GEMM's expansion order
      }
    }
    for (int j = -1; j < s.k; ++j) {
      const long long row = (j < 0) ? shared_row : (long long)__shfl_sync(0xffffffffu, pos, j);
      if (row < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(sc.x_perm + (size_t)row * s.d);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int pc = p0 + lane + 32 * i;
        if (pc < pieces) __stcs(dst + pc, v[i]);
      }
    }
  }
}

cudaError_t launch_group(const Shapes& s, const Scratch& sc, const DevCtl& ctl, cudaStream_t st,
                         const void* x_rows) {
  const int nchunk = (s.T + kChunk - 1) / kChunk;
  group_scan_kernel<<<(s.E + 7) / 8, 256, 0, st>>>(s, sc);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (!x_rows)
    group_scatter_kernel<<<nchunk, 256, 0, st>>>(s, sc, ctl);
  else if (s.x_bf16)
    group_scatter_rows_kernel<true><<<(s.T + 7) / 8, 256, 0, st>>>(s, x_rows, sc, ctl);
  else
    group_scatter_rows_kernel<false><<<(s.T + 7) / 8, 256, 0, st>>>(s, x_rows, sc, ctl);
  return cudaGetLastError();
}

cudaError_t launch_export_route(const Shapes& s, const Scratch& sc, int32_t* idx, float* w, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* slot, cudaStream_t st) {
  const size_t tk = (size_t)s.T * s.k;
  cudaError_t err = cudaSuccess;
  if (idx && err == cudaSuccess) err = cudaMemcpyAsync(idx, sc.idx, tk * 4, cudaMemcpyDeviceToDevice, st);
  if (w && err == cudaSuccess) err = cudaMemcpyAsync(w, sc.w, tk * 4, cudaMemcpyDeviceToDevice, st);
  if (counts && err == cudaSuccess)
    err = cudaMemcpyAsync(counts, sc.counts, (size_t)s.E * 4, cudaMemcpyDeviceToDevice, st);
  if (offsets && err == cudaSuccess)
    err = cudaMemcpyAsync(offsets, sc.offsets, (size_t)(s.E + 1) * 4, cudaMemcpyDeviceToDevice, st);
  if (perm && err == cudaSuccess) err = cudaMemcpyAsync(perm, sc.perm, tk * 4, cudaMemcpyDeviceToDevice, st);
  if (slot && err == cudaSuccess) err = cudaMemcpyAsync(slot, sc.slot, tk * 4, cudaMemcpyDeviceToDevice, st);
  return err;
}

}  // namespace moe
