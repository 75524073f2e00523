// The weighted combine of the grouped-GEMM path.
//
// "Optimizing on-device inference for Apple Silicon", section "Reducing
// intermediate and state traffic": the experts' output projections are
// combined with their routing scores and the shared expert's result.  Here,
// per token t: y_t = sum_j w[t, j] * out[slot[t, j]] + g_t * out[T*k + t],
// summed in fp32 over j in ascending expert order, then stored in x's dtype;
// g_t is one, or sigmoid(x_t . g) for a sigmoid-gated shared expert.
#include "moe_internal.h"

namespace moe {

MOE_DEV void fma8(float (&acc)[8], float w, const uint4 v) {
  acc[0] = fmaf(w, bf16_lo(v.x), acc[0]);
  acc[1] = fmaf(w, bf16_hi(v.x), acc[1]);
  acc[2] = fmaf(w, bf16_lo(v.y), acc[2]);
  acc[3] = fmaf(w, bf16_hi(v.y), acc[3]);
  acc[4] = fmaf(w, bf16_lo(v.z), acc[4]);
  acc[5] = fmaf(w, bf16_hi(v.z), acc[5]);
  acc[6] = fmaf(w, bf16_lo(v.w), acc[6]);
  acc[7] = fmaf(w, bf16_hi(v.w), acc[7]);
}

// One warp per (token, 256-column slice); each lane owns 8 consecutive columns
// and reads them with one 16-byte load per contributing row.  The rows' slots
// and weights are read first and the rows' loads (8 at a time, and the shared
// expert's row) are all in flight before the first is used: with each slot
// read just before its row, every row cost two dependent memory round trips
// and the kernel stalled on them with DRAM 62 % busy.
template <bool YBF16>
__global__ void __launch_bounds__(256) combine_kernel(Shapes s, void* __restrict__ y, Scratch sc) {
  constexpr int kRows = 8;  // routed rows in flight per step
  const int lane = threadIdx.x & 31;
  const int slices = s.d >> 8;
  const long long gw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (gw >= (long long)s.T * slices) return;
  const int t = (int)(gw / slices);
  const int col = (int)(gw - (long long)t * slices) * 256 + lane * 8;
  uint4 vs = make_uint4(0u, 0u, 0u, 0u);
  if (s.has_shared) vs = __ldcs(reinterpret_cast<const uint4*>(sc.out + ((size_t)s.T * s.k + t) * s.d + col));
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < s.k; j0 += kRows) {
    int p[kRows];
    float wj[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const bool in = j0 + u < s.k;
      p[u] = in ? sc.slot[(size_t)t * s.k + j0 + u] : 0;
      if (kDebugChecks && (p[u] < 0 || p[u] >= s.T * s.k)) {
        atomicOr(sc.status, kStatusBounds);
        p[u] = 0;
      }
      wj[u] = in ? sc.w[(size_t)t * s.k + j0 + u] : 0.f;
    }
    uint4 v[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u)
      v[u] = (j0 + u < s.k) ? __ldcs(reinterpret_cast<const uint4*>(sc.out + (size_t)p[u] * s.d + col))
                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < kRows; ++u)
      if (j0 + u < s.k) fma8(acc, wj[u], v[u]);
  }
  if (s.has_shared) {
    // fmaf with a gate of exactly one adds v exactly as a plain sum would
    const float gs = s.shared_gate ? sc.sgate[t] : 1.f;
    fma8(acc, gs, vs);
  }
  if (YBF16) {
    uint4 o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                         pack_bf16x2(acc[6], acc[7]));
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(y) + (size_t)t * s.d + col) = o;
  } else {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(y) + (size_t)t * s.d + col);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

cudaError_t launch_combine(const Shapes& s, void* y, const Scratch& sc, cudaStream_t st) {
  const long long warps = (long long)s.T * (s.d >> 8);
  const int blocks = (int)((warps + 7) / 8);
  if (s.x_bf16)
    combine_kernel<true><<<blocks, 256, 0, st>>>(s, y, sc);
  else
    combine_kernel<false><<<blocks, 256, 0, st>>>(s, y, sc);
  return cudaGetLastError();
}

}  // namespace moe
