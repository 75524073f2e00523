// Internal declarations shared by the translation units of the MoE library:
// the layout of a context's scratch memory and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"
#include "moe_common.cuh"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
constexpr int kChunk = 32;       // tokens per grouping chunk (one bit each in a 32-bit mask)
constexpr int kBM = 128;         // rows (tokens) per grouped-GEMM tile

// m-tile of the grouped GEMM: rows [row0, row0 + rows) of the expert-grouped
// buffers belong to expert `e` (e == E is the shared expert).
struct MTile {
  int e, row0, rows, pad;
};

// Device scratch memory of one context (all sized for max_tokens).
struct Scratch {
  float* logits;          // [T, E] fp32 router logits (SIMT router) / [3, T, E] partials (tensor router)
  int* idx;               // [T, k]
  float* w;               // [T, k]
  unsigned* chunk_mask;   // [nchunk, E]: bit i = token chunk*32+i chose expert e
  int* chunk_base;        // [E, nchunk]: per-chunk count, then the exclusive prefix within expert
  int* counts;            // [E + 1]; counts[E] = T for the shared expert
  int* offsets;           // [E + 2]; offsets[E] = T*k, offsets[E+1] = T*k + T
  int* perm;              // [T*k + T]: token of each grouped row; rows T*k.. are the shared expert's
  int* slot;              // [T, k]: grouped row of (t, idx[t][j])
  MTile* mtiles;          // grouped-GEMM m-tiles
  MTile* mpairs;          // the m-tiles two by two within each expert group (pad = rows of the second, 0: none)
  int* meta;              // [0] = number of m-tiles, [1] = number of active experts, [2] = number of m-tile pairs
  int* active;            // [E + 1]: experts with count > 0, ascending, then the shared expert
  unsigned* tickets;      // last-block counters (self-resetting)
  uint16_t* x_perm;       // [T*k + T, d] bf16 token rows in grouped order (GEMM path)
  uint16_t* wr_split;     // [3E, d] router weights as bf16 hi + mid + lo terms
  uint16_t* h;            // [T*k + T, I] bf16 SwiGLU activations, grouped rows (GEMM path)
  float* h_gemv;          // [Tg*k + Tg, I] fp32 SwiGLU activations (GEMV path)
  uint16_t* out;          // [T*k + T, d] bf16 expert outputs, grouped rows (GEMM path)
  unsigned* status;       // device status word
  unsigned* gridbar;      // fused decode kernel: control words, [2..3] = 64-bit epoch counter
  float* dec_logits;      // fused decode kernel: [dec_reps][T][E] router logits as (fp32, epoch) 64-bit words
  float* dec_h;           // fused decode kernel: [dec_hreps][T*k + T][I] SwiGLU activations as (fp32, epoch) words
  float* sgate;           // [T] sigmoid(x_t . g), the shared expert's gate (GEMV and GEMM paths)
  int dec_reps;           // copies of the logits (blocks read copy b % reps)
  int dec_hreps;          // copies of h
  int max_mtiles;
};

struct Shapes {
  int T, d, E, I, k;
  int has_shared;
  int x_bf16;             // 1: x is bf16, 0: fp32
  int bias_sel;           // 1: the router bias picks the experts but does not enter their weights
  int shared_gate;        // 1: the shared expert's output is scaled by sigmoid(x . g), g = router row E
  int q4;                 // 1: expert weights are 4-bit group-affine (MOE_W_Q4G64 planes), 0: bf16
};

// moe_route.cu
cudaError_t launch_router_logits_simt(const Shapes& s, const void* x, const float* wr, const float* rb,
                                      const Scratch& sc, cudaStream_t st);
cudaError_t launch_router_split_weights(const Shapes& s, const float* wr, const Scratch& sc, cudaStream_t st);
// with s.shared_gate, also sc.sgate[t] = sigmoid(x_t . gate_w)
cudaError_t launch_select(const Shapes& s, const float* rb, int logit_parts, const Scratch& sc,
                          const DevCtl& ctl, cudaStream_t st, const void* x = nullptr,
                          const float* gate_w = nullptr);
// x_rows non-null: also write every token's row, in bf16, to its grouped rows of sc.x_perm
cudaError_t launch_group(const Shapes& s, const Scratch& sc, const DevCtl& ctl, cudaStream_t st,
                         const void* x_rows = nullptr);
cudaError_t launch_export_route(const Shapes& s, const Scratch& sc, int32_t* idx, float* w, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* slot, cudaStream_t st);

// moe_gemv.cu
size_t gemv_gate_up_smem(const Shapes& s);
size_t gemv_down_smem(const Shapes& s);
cudaError_t launch_gemv_gate_up(const Shapes& s, const void* x, const uint16_t* gate_up, const uint16_t* shared_w,
                                const Scratch& sc, const DevCtl& ctl, int num_sms, cudaStream_t st);
cudaError_t prepare_gemv_kernels(int max_smem);
cudaError_t launch_gemv_down(const Shapes& s, const uint16_t* down, const uint16_t* shared_w, void* y,
                             const Scratch& sc, const DevCtl& ctl, int num_sms, cudaStream_t st);

// moe_gemm.cu
struct GemmMaps {
  CUtensorMap x_tile;       // x (bf16) [T, d], box 64 x 128
  CUtensorMap x_perm;       // grouped token rows [T*k + T, d], box 64 x 128
  CUtensorMap gate_up;      // experts [E*2I, d], box 64 x 128 (gate half and up half of one B tile)
  CUtensorMap shared_gu;    // shared gate_up [2I, d], box 64 x 128
  CUtensorMap h;            // h [T*k + T, I], box 64 x 128
  CUtensorMap down;         // experts [E*d, I], box 64 x 256
  CUtensorMap shared_down;  // shared down [d, I], box 64 x 256
  CUtensorMap wr_split;     // router weights hi/mid/lo [3E, d], box 64 x 256
  // the same A operands in boxes of 16 rows: a tile whose group has at most
  // 64 rows loads only the boxes that cover its rows
  CUtensorMap x_tile16, x_perm16, h16;
  // 4-bit weights (MOE_W_Q4G64 rows of 9 K / 16 bytes): each matrix seen twice,
  // as uint32 words (the codes of a 64-column k block: box 8 x rows) and as
  // bf16 (the scales / biases of 8 groups: box 8 x rows); no swizzle
  CUtensorMap gu_codes, gu_params;      // routed gate_up [E 2I rows]
  CUtensorMap sgu_codes, sgu_params;    // shared gate_up [2I rows]
  CUtensorMap dn_codes, dn_params;      // routed down [E d rows]
  CUtensorMap sdn_codes, sdn_params;    // shared down [d rows]
};
cudaError_t prepare_gemm_kernels();
bool gemm_q4_supported(int d, int inter);
cudaError_t launch_gemm_gate_up(const Shapes& s, const GemmMaps& m, const Scratch& sc, const DevCtl& ctl,
                                int num_sms, cudaStream_t st);
cudaError_t launch_gemm_down(const Shapes& s, const GemmMaps& m, const Scratch& sc, const DevCtl& ctl,
                             int num_sms, cudaStream_t st);
cudaError_t launch_gemm_router(const Shapes& s, const GemmMaps& m, const Scratch& sc, const DevCtl& ctl,
                               int num_sms, cudaStream_t st);

// moe_decode.cu
// Shared memory the fused decode kernel may use (clamped to what the device
// allows a block next to the kernel's static shared memory).
constexpr int kDecodeSmemLimit = 227 * 1024;
size_t decode_smem_bytes(const Shapes& s, int max_smem);
bool decode_supported(const Shapes& s, int max_smem);
int decode_blocks_per_sm(const Shapes& s, int max_smem);
cudaError_t prepare_decode_kernels(int max_smem);
cudaError_t launch_decode_fused(const Shapes& s, const void* x, const float* wr, const float* rb,
                                const uint16_t* gate_up, const uint16_t* down, const uint16_t* shared_w, void* y,
                                const Scratch& sc, const DevCtl& ctl, unsigned* bar, int num_sms, cudaStream_t st,
                                const float* next_wr, const uint16_t* next_shared, int max_smem,
                                bool overlap = false);

// moe_combine.cu
cudaError_t launch_combine(const Shapes& s, void* y, const Scratch& sc, cudaStream_t st);

}  // namespace moe
