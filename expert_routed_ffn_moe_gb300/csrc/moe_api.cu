// C ABI of the MoE layer: argument checking, the context and its scratch
// memory, TMA tensor maps, and the per-call kernel sequence.  Declarations and
// the full contract are in include/moe.h.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "moe_internal.h"

using namespace moe;

// signature of the driver's cuTensorMapEncodeTiled (fetched at run time, so the
// library needs no link-time dependency on libcuda)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct moe_ctx {
  moe_config cfg;
  int device = 0;
  int num_sms = 0;
  int path = MOE_PATH_AUTO;
  int router = MOE_ROUTER_AUTO;
  long long spin_ns = 0;
  int stall = 0;            // test hook (moe_inject_stall)
  const float* next_wr = nullptr;         // prefetch hint for the next call (moe_set_prefetch)
  bool overlap = false;                   // programmatic launch overlap (moe_set_overlap)
  int chunk = 0;                          // chunked prefill: tokens per slice (moe_set_chunk_tokens), 0 = off
  const uint16_t* next_shared = nullptr;
  int gemv_max_t = 0;       // largest T the GEMV kernels accept for this shape (0: none)
  int decode_max_t = 0;     // largest T the fused decode kernel accepts (0: none)
  void* block = nullptr;    // the single device allocation holding all scratch
  Scratch sc{};
  EncodeTiledFn encode = nullptr;
  // profiling hook (moe_time_kernel) and launch counter
  int timed_kernel = -1;
  cudaEvent_t ev_start = nullptr, ev_stop = nullptr;
  long long launches = 0;
  // T and top_k of the last moe_forward call (or slice) whose routing tables the scratch holds
  int last_T = 0, last_k = 0;
};

namespace {

constexpr long long kDefaultSpinNs = 1000000000LL;  // 1 s
// Largest T the automatic path sends to the small-T kernels.  Measured per layer (d = 2048, 256
// experts, inter 512, top-8 + shared, bf16; fused kernel vs grouped GEMMs, us): T = 1: 19.2 vs 46.8,
// 2: 31.5 vs 52.5, 3: 45.5 vs 58.9, 4: 62.1 vs 65.5, 5: 79.4 vs 78.6, 6: 98.3 vs 86.2, 7: 129.1 vs
// 89.2 -- the GEMMs tie at T = 5 and win beyond.
constexpr int kGemvMaxT = 4;
constexpr int kGemvSmemLimit = 200 * 1024;           // dynamic shared memory of the GEMV kernels
constexpr int kDecodeReps = 8;                       // copies of the decode kernel's broadcast data

int cuda_fail(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// GEMV path limits: x of all T tokens and h of all T*(k+1) rows live in shared memory.
int gemv_limit(const moe_config& c) {
  if (c.d % 256 != 0 || c.inter % 256 != 0) return 0;
  const size_t kSmem = kGemvSmemLimit;
  int best = 0;
  for (int T = 1; T <= 32 && T <= c.max_tokens; ++T) {
    const size_t pairs = (size_t)T * c.top_k + (c.has_shared ? T : 0);
    const size_t xs = (size_t)T * c.d * 4;
    const size_t hs = pairs * c.inter * 4 + pairs * 8;
    if (xs <= kSmem && hs <= kSmem) best = T;
  }
  return best;
}

int make_map(moe_ctx* ctx, CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
             uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = ctx->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                                 estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// A 2-D map over 4-bit weight rows (9 K / 16 bytes each, `rows` of them): as
// uint32 words (codes; box 8 words) or as bf16 (scales / biases; box 8 values),
// `box_rows` rows per box, no swizzle.
int make_q4_map(moe_ctx* ctx, CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, uint32_t box_rows,
                bool codes) {
  const uint64_t row_bytes = K / 16 * 9;
  const cuuint64_t dims[2] = {codes ? row_bytes / 4 : row_bytes / 2, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {8, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = ctx->encode(m, codes ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                 const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                 CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

int check_route_args(moe_ctx* ctx, const void* x, int T, const float* wr, const float* rb, int top_k) {
  if (!ctx || T < 0) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  const moe_config& c = ctx->cfg;
  if (!x || !wr) return MOE_ERR_ARG;
  if (T > c.max_tokens || top_k < 1 || top_k > c.top_k) return MOE_ERR_ARG;
  if (c.has_router_bias && !rb) return MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(wr) || (rb && !aligned16(rb))) return MOE_ERR_ALIGN;
  return MOE_OK;
}

Shapes shapes(const moe_ctx* ctx, int T, int top_k) {
  const moe_config& c = ctx->cfg;
  Shapes s;
  s.T = T;
  s.d = c.d;
  s.E = c.n_experts;
  s.I = c.inter;
  s.k = top_k;
  s.has_shared = c.has_shared;
  s.x_bf16 = c.x_dtype == MOE_BF16;
  s.bias_sel = c.has_router_bias && c.bias_select_only;
  s.shared_gate = c.has_shared && c.shared_gate;
  s.q4 = c.weight_format == MOE_W_Q4G64;
  return s;
}

DevCtl devctl(const moe_ctx* ctx) {
  DevCtl d;
  d.status = ctx->sc.status;
  d.spin_limit = ctx->spin_ns;
  d.stall = ctx->stall;
  return d;
}

bool use_tensor_router(const moe_ctx* ctx, const Shapes& s) {
  if (ctx->router == MOE_ROUTER_SIMT) return false;
  const bool able = s.x_bf16 && s.E == 256 && s.d % 64 == 0;
  if (ctx->router == MOE_ROUTER_TENSOR) return able;
  return able && s.T > 64;
}

// Every kernel launch goes through `launch`: it counts the launch and, when
// the profiling hook is armed for this kernel id, records the caller's events
// around it.
// Under stream capture an event record must be marked external to become a
// timeable event-record node of the graph.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  return cudaEventRecordWithFlags(ev, st, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0u);
}

// An NVTX range over a scope.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

// NVTX range names of the launches (a profiler shows each launch's host call
// under its step of the layer; header-only NVTX costs nothing without a tool)
const char* range_name(int id) {
  switch (id) {
    case -2: return "moe.router_split";
    case MOE_K_ROUTER: return "moe.router";
    case MOE_K_SELECT: return "moe.select";
    case MOE_K_GROUP: return "moe.group";
    case MOE_K_GEMV_GATE_UP: return "moe.gemv_gate_up";
    case MOE_K_GEMV_DOWN: return "moe.gemv_down";
    case MOE_K_GEMM_GATE_UP: return "moe.gemm_gate_up";
    case MOE_K_GEMM_DOWN: return "moe.gemm_down";
    case MOE_K_COMBINE: return "moe.combine";
    case MOE_K_DECODE_FUSED: return "moe.decode_fused";
    default: return "moe.kernel";
  }
}

template <typename F>
cudaError_t launch_timed(moe_ctx* ctx, int id, cudaStream_t st, F&& f) {
  const bool timed = ctx->timed_kernel == id;
  if (timed) {
    cudaError_t e = record_event(ctx->ev_start, st);
    if (e != cudaSuccess) return e;
  }
  cudaError_t err = f();
  ++ctx->launches;
  if (timed && err == cudaSuccess) {
    err = record_event(ctx->ev_stop, st);
    ctx->timed_kernel = -1;
  }
  return err;
}

template <typename F>
cudaError_t launch(moe_ctx* ctx, int id, cudaStream_t st, F&& f) {
  const NvtxRange range(range_name(id));
  return launch_timed(ctx, id, st, f);
}

// Steps 1-4 on the device: logits, selection, grouping.
int run_route(moe_ctx* ctx, const Shapes& s, const void* x, const float* wr, const float* rb, bool tensor,
              const GemmMaps* maps, cudaStream_t st, bool permute_rows = false) {
  const DevCtl ctl = devctl(ctx);
  cudaError_t err;
  int parts = 1;
  const Scratch& sc = ctx->sc;
  const int sms = ctx->num_sms;
  if (tensor) {
    err = launch(ctx, -2, st, [&] { return launch_router_split_weights(s, wr, sc, st); });
    if (err != cudaSuccess) return cuda_fail(err);
    err = launch(ctx, MOE_K_ROUTER, st, [&] { return launch_gemm_router(s, *maps, sc, ctl, sms, st); });
    if (err != cudaSuccess) return cuda_fail(err);
    parts = 3;
  } else {
    err = launch(ctx, MOE_K_ROUTER, st, [&] { return launch_router_logits_simt(s, x, wr, rb, sc, st); });
    if (err != cudaSuccess) return cuda_fail(err);
  }
  const float* gate_w = s.shared_gate ? wr + (size_t)s.E * s.d : nullptr;  // router row E
  err = launch(ctx, MOE_K_SELECT, st, [&] { return launch_select(s, rb, parts, sc, ctl, st, x, gate_w); });
  if (err != cudaSuccess) return cuda_fail(err);
  err = launch(ctx, MOE_K_GROUP, st, [&] { return launch_group(s, sc, ctl, st, permute_rows ? x : nullptr); });
  ctx->launches += 1;  // the group step is two kernels
  return cuda_fail(err);
}

}  // namespace

extern "C" {

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case MOE_ERR_UNSUPPORTED: return "shape or device not supported";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case MOE_ERR_BOUNDS: return "an index read by a kernel was out of range";
    case MOE_ERR_NOMEM: return "out of device memory";
    default: return "unknown error";
  }
}

int moe_init(const moe_config* cfg, moe_ctx** out) {
  if (!cfg || !out) return MOE_ERR_ARG;
  *out = nullptr;
  const moe_config c = *cfg;
  if (c.d <= 0 || c.n_experts <= 0 || c.inter <= 0 || c.top_k <= 0 || c.max_tokens <= 0) return MOE_ERR_ARG;
  if (c.x_dtype != MOE_F32 && c.x_dtype != MOE_BF16) return MOE_ERR_ARG;
  if (c.top_k > c.n_experts || c.top_k > kMaxTopK) return MOE_ERR_ARG;
  if (c.n_experts > kMaxExperts || c.d % 256 != 0 || c.inter % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (c.has_shared && c.shared_inter != c.inter) return MOE_ERR_UNSUPPORTED;
  if (c.bias_select_only != 0 && c.bias_select_only != 1) return MOE_ERR_ARG;
  if (c.shared_gate != 0 && c.shared_gate != 1) return MOE_ERR_ARG;
  if (c.shared_gate && !c.has_shared) return MOE_ERR_ARG;
  if (c.weight_format != MOE_W_BF16 && c.weight_format != MOE_W_Q4G64) return MOE_ERR_ARG;
  if (c.weight_format == MOE_W_Q4G64 && c.inter % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if ((long long)c.max_tokens * (c.top_k + 1) >= (1LL << 31) / 2) return MOE_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (!(prop.major == 10 && prop.minor == 3)) return MOE_ERR_UNSUPPORTED;

  if (prepare_gemm_kernels() != cudaSuccess || prepare_gemv_kernels(kGemvSmemLimit) != cudaSuccess ||
      prepare_decode_kernels(kDecodeSmemLimit) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }

  moe_ctx* ctx = new moe_ctx();
  ctx->cfg = c;
  if (!c.has_shared) ctx->cfg.shared_inter = 0;
  ctx->device = dev;
  ctx->num_sms = prop.multiProcessorCount;
  ctx->spin_ns = kDefaultSpinNs;
  ctx->gemv_max_t = c.weight_format == MOE_W_BF16 ? gemv_limit(ctx->cfg) : 0;  // the modular GEMV kernels read bf16
  for (int t = 1; t <= 16 && t <= c.max_tokens; ++t) {
    Shapes s1{};
    s1.T = t;
    s1.d = c.d;
    s1.E = c.n_experts;
    s1.I = c.inter;
    s1.k = c.top_k;
    s1.has_shared = c.has_shared;
    s1.x_bf16 = c.x_dtype == MOE_BF16;
    s1.shared_gate = c.has_shared && c.shared_gate;
    s1.q4 = c.weight_format == MOE_W_Q4G64;
    if (decode_supported(s1, kDecodeSmemLimit) && decode_blocks_per_sm(s1, kDecodeSmemLimit) >= 1) ctx->decode_max_t = t;
  }

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    delete ctx;
    return MOE_ERR_CUDA;
  }
  ctx->encode = reinterpret_cast<EncodeTiledFn>(fn);

  // carve the scratch memory out of one allocation
  const size_t T = c.max_tokens, k = c.top_k, E = c.n_experts, d = c.d, I = c.inter;
  const size_t nchunk = (T + kChunk - 1) / kChunk;
  const size_t rows = T * k + T;
  const size_t tg = ctx->gemv_max_t > ctx->decode_max_t ? ctx->gemv_max_t : ctx->decode_max_t;
  const int max_mtiles = (int)(T * k / kBM + E + T / kBM + 2);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = round_up(off + bytes, 256);
    return o;
  };
  const size_t o_logits = take(3 * T * E * 4);
  const size_t o_idx = take(T * k * 4);
  const size_t o_w = take(T * k * 4);
  const size_t o_cmask = take(nchunk * E * 4);
  const size_t o_cbase = take(E * nchunk * 4);
  const size_t o_counts = take((E + 1) * 4);
  const size_t o_offsets = take((E + 2) * 4);
  const size_t o_perm = take(rows * 4);
  const size_t o_slot = take(T * k * 4);
  const size_t o_mtiles = take((size_t)max_mtiles * sizeof(MTile));
  const size_t o_mpairs = take((size_t)max_mtiles * sizeof(MTile));
  const size_t o_meta = take(4 * 4);
  const size_t o_active = take((E + 1) * 4);
  const size_t o_tickets = take(4 * 4);
  const size_t o_xperm = take(rows * d * 2);
  const size_t o_wrs = take(3 * E * d * 2);
  const size_t o_h = take(rows * I * 2);
  const size_t o_hg = take(tg ? (tg * k + tg) * I * 4 : 16);
  const size_t o_out = take(rows * d * 2);
  const size_t o_status = take(16);
  const size_t o_gridbar = take(64);
  const size_t o_dlog = take(ctx->decode_max_t ? (size_t)kDecodeReps * ctx->decode_max_t * E * 8 : 16);
  const size_t dpairs = (size_t)ctx->decode_max_t * (k + 1);
  const size_t o_dh = take(ctx->decode_max_t ? (size_t)kDecodeReps * dpairs * I * 8 : 16);
  const size_t o_sgate = take(T * 4);
  if (cudaMalloc(&ctx->block, off) != cudaSuccess) {
    cudaGetLastError();
    delete ctx;
    return MOE_ERR_NOMEM;
  }
  if (cudaMemset(ctx->block, 0, off) != cudaSuccess) {
    cudaFree(ctx->block);
    delete ctx;
    return MOE_ERR_CUDA;
  }
  char* b = static_cast<char*>(ctx->block);
  Scratch& sc = ctx->sc;
  sc.logits = reinterpret_cast<float*>(b + o_logits);
  sc.idx = reinterpret_cast<int*>(b + o_idx);
  sc.w = reinterpret_cast<float*>(b + o_w);
  sc.chunk_mask = reinterpret_cast<unsigned*>(b + o_cmask);
  sc.chunk_base = reinterpret_cast<int*>(b + o_cbase);
  sc.counts = reinterpret_cast<int*>(b + o_counts);
  sc.offsets = reinterpret_cast<int*>(b + o_offsets);
  sc.perm = reinterpret_cast<int*>(b + o_perm);
  sc.slot = reinterpret_cast<int*>(b + o_slot);
  sc.mtiles = reinterpret_cast<MTile*>(b + o_mtiles);
  sc.mpairs = reinterpret_cast<MTile*>(b + o_mpairs);
  sc.meta = reinterpret_cast<int*>(b + o_meta);
  sc.active = reinterpret_cast<int*>(b + o_active);
  sc.tickets = reinterpret_cast<unsigned*>(b + o_tickets);
  sc.x_perm = reinterpret_cast<uint16_t*>(b + o_xperm);
  sc.wr_split = reinterpret_cast<uint16_t*>(b + o_wrs);
  sc.h = reinterpret_cast<uint16_t*>(b + o_h);
  sc.h_gemv = reinterpret_cast<float*>(b + o_hg);
  sc.out = reinterpret_cast<uint16_t*>(b + o_out);
  sc.status = reinterpret_cast<unsigned*>(b + o_status);
  sc.gridbar = reinterpret_cast<unsigned*>(b + o_gridbar);
  sc.dec_logits = reinterpret_cast<float*>(b + o_dlog);
  sc.dec_h = reinterpret_cast<float*>(b + o_dh);
  sc.sgate = reinterpret_cast<float*>(b + o_sgate);
  sc.dec_reps = kDecodeReps;
  sc.dec_hreps = kDecodeReps;
  sc.max_mtiles = max_mtiles;
  *out = ctx;
  return MOE_OK;
}

int moe_set_path(moe_ctx* ctx, int path) {
  if (!ctx || path < MOE_PATH_AUTO || path > MOE_PATH_GEMM) return MOE_ERR_ARG;
  ctx->path = path;
  return MOE_OK;
}

int moe_set_router(moe_ctx* ctx, int router) {
  if (!ctx || router < MOE_ROUTER_AUTO || router > MOE_ROUTER_TENSOR) return MOE_ERR_ARG;
  ctx->router = router;
  return MOE_OK;
}

int moe_set_spin_limit(moe_ctx* ctx, long long limit) {
  if (!ctx || limit < 0) return MOE_ERR_ARG;
  ctx->spin_ns = limit == 0 ? kDefaultSpinNs : limit;
  return MOE_OK;
}

int moe_record_event(void* event, void* stream) {
  if (!event) return MOE_ERR_ARG;
  return cuda_fail(record_event(static_cast<cudaEvent_t>(event), static_cast<cudaStream_t>(stream)));
}

int moe_set_overlap(moe_ctx* ctx, int on) {
  if (!ctx || (on != 0 && on != 1)) return MOE_ERR_ARG;
  ctx->overlap = on == 1;
  return MOE_OK;
}

int moe_set_prefetch(moe_ctx* ctx, const float* next_router_w, const void* next_shared_w) {
  if (!ctx) return MOE_ERR_ARG;
  if ((next_router_w && !aligned16(next_router_w)) || (next_shared_w && !aligned16(next_shared_w)))
    return MOE_ERR_ALIGN;
  ctx->next_wr = next_router_w;
  ctx->next_shared = static_cast<const uint16_t*>(next_shared_w);
  return MOE_OK;
}

int moe_inject_stall(moe_ctx* ctx, int on) {
  if (!ctx || (on != 0 && on != 1)) return MOE_ERR_ARG;
  ctx->stall = on;
  return MOE_OK;
}

int moe_time_kernel(moe_ctx* ctx, int kernel_id, void* ev_start, void* ev_stop) {
  if (!ctx || kernel_id < MOE_K_ROUTER || kernel_id > MOE_K_DECODE_FUSED || !ev_start || !ev_stop) return MOE_ERR_ARG;
  ctx->timed_kernel = kernel_id;
  ctx->ev_start = static_cast<cudaEvent_t>(ev_start);
  ctx->ev_stop = static_cast<cudaEvent_t>(ev_stop);
  return MOE_OK;
}

long long moe_launch_count(moe_ctx* ctx) { return ctx ? ctx->launches : 0; }

int moe_route(moe_ctx* ctx, const void* x, int T, const float* router_w, const float* router_b, int top_k,
              int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm, void* stream) {
  int rc = check_route_args(ctx, x, T, router_w, router_b, top_k);
  if (rc != MOE_OK || T == 0) return rc;
  if (!ctx->cfg.has_router_bias) router_b = nullptr;
  if ((idx && !aligned16(idx)) || (w && !aligned16(w)) || (counts && !aligned16(counts)) ||
      (offsets && !aligned16(offsets)) || (perm && !aligned16(perm)))
    return MOE_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Shapes s = shapes(ctx, T, top_k);
  s.shared_gate = 0;  // routing only: router_w may hold just the E expert rows
  const bool tensor = use_tensor_router(ctx, s);
  GemmMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (tensor) {
    if ((rc = make_map(ctx, &maps.x_tile, x, s.d, s.T, 64, 128)) != MOE_OK) return rc;
    if ((rc = make_map(ctx, &maps.x_tile16, x, s.d, s.T, 64, 16)) != MOE_OK) return rc;
    if ((rc = make_map(ctx, &maps.wr_split, ctx->sc.wr_split, s.d, 3 * s.E, 64, 256)) != MOE_OK) return rc;
  }
  if ((rc = run_route(ctx, s, x, router_w, router_b, tensor, &maps, st)) != MOE_OK) return rc;
  ctx->last_T = 0;  // the scratch tables now hold this call's routing, not a forward's
  return cuda_fail(launch_export_route(s, ctx->sc, idx, w, counts, offsets, perm, nullptr, st));
}

int moe_last_routing(moe_ctx* ctx, int32_t* idx, float* w, int32_t* counts, int32_t* offsets, int32_t* perm,
                     int32_t* slot, int* T_out, int* k_out, void* stream) {
  if (!ctx || ctx->last_T <= 0) return MOE_ERR_ARG;
  if ((idx && !aligned16(idx)) || (w && !aligned16(w)) || (counts && !aligned16(counts)) ||
      (offsets && !aligned16(offsets)) || (perm && !aligned16(perm)) || (slot && !aligned16(slot)))
    return MOE_ERR_ALIGN;
  if (T_out) *T_out = ctx->last_T;
  if (k_out) *k_out = ctx->last_k;
  const Shapes s = shapes(ctx, ctx->last_T, ctx->last_k);
  return cuda_fail(launch_export_route(s, ctx->sc, idx, w, counts, offsets, perm, slot,
                                       static_cast<cudaStream_t>(stream)));
}

static int forward_one(moe_ctx* ctx, const void* x, int T, const float* router_w, const float* router_b,
                       const void* experts_gate_up, const void* experts_down, const void* shared_w, int top_k,
                       void* y, void* stream);

// After a forward call: the scratch routing tables are that call's (for
// moe_last_routing) if it launched its kernels.
static int remember_routing(moe_ctx* ctx, int T, int top_k, int rc) {
  ctx->last_T = rc == MOE_OK ? T : 0;
  ctx->last_k = rc == MOE_OK ? top_k : 0;
  return rc;
}

int moe_set_chunk_tokens(moe_ctx* ctx, int chunk) {
  if (!ctx || chunk < 0 || chunk > ctx->cfg.max_tokens) return MOE_ERR_ARG;
  ctx->chunk = chunk;
  return MOE_OK;
}

int moe_forward(moe_ctx* ctx, const void* x, int T, const float* router_w, const float* router_b,
                const void* experts_gate_up, const void* experts_down, const void* shared_w, int top_k, void* y,
                void* stream) {
  if (!ctx || T < 0) return MOE_ERR_ARG;
  const NvtxRange range("moe_forward");
  const int chunk = ctx->chunk;
  if (chunk == 0 || T <= chunk)
    return forward_one(ctx, x, T, router_w, router_b, experts_gate_up, experts_down, shared_w, top_k, y, stream);
  // Chunked prefill: tokens are independent, so the layer over T tokens is the
  // layer over consecutive slices of at most `chunk` tokens, each through the
  // context's workspace (sized for max_tokens) -- exact, at the price of
  // reading the selected experts' weights once per slice.
  if (!x || !y) return MOE_ERR_ARG;
  const size_t row = (size_t)ctx->cfg.d * (ctx->cfg.x_dtype == MOE_BF16 ? 2 : 4);
  for (int t0 = 0; t0 < T; t0 += chunk) {
    const int n = T - t0 < chunk ? T - t0 : chunk;
    const int rc = forward_one(ctx, static_cast<const char*>(x) + (size_t)t0 * row, n, router_w, router_b,
                               experts_gate_up, experts_down, shared_w, top_k, static_cast<char*>(y) + (size_t)t0 * row,
                               stream);
    if (rc != MOE_OK) return rc;
  }
  return MOE_OK;
}

static int forward_one(moe_ctx* ctx, const void* x, int T, const float* router_w, const float* router_b,
                       const void* experts_gate_up, const void* experts_down, const void* shared_w, int top_k,
                       void* y, void* stream) {
  int rc = check_route_args(ctx, x, T, router_w, router_b, top_k);
  if (rc != MOE_OK || T == 0) return rc;
  const moe_config& c = ctx->cfg;
  if (!experts_gate_up || !experts_down || !y || (c.has_shared && !shared_w)) return MOE_ERR_ARG;
  if (!aligned16(experts_gate_up) || !aligned16(experts_down) || !aligned16(y) ||
      (shared_w && !aligned16(shared_w)))
    return MOE_ERR_ALIGN;
  if (!c.has_router_bias) router_b = nullptr;
  if (!c.has_shared) shared_w = nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Shapes s = shapes(ctx, T, top_k);
  int path = ctx->path;
  const int small_max = ctx->gemv_max_t > ctx->decode_max_t ? ctx->gemv_max_t : ctx->decode_max_t;
  if (path == MOE_PATH_AUTO) path = (T <= kGemvMaxT && T <= small_max) ? MOE_PATH_GEMV : MOE_PATH_GEMM;
  if (path == MOE_PATH_GEMV && T > small_max) return MOE_ERR_UNSUPPORTED;
  const DevCtl ctl = devctl(ctx);
  const uint16_t* gu = static_cast<const uint16_t*>(experts_gate_up);
  const uint16_t* dn = static_cast<const uint16_t*>(experts_down);
  const uint16_t* sw = static_cast<const uint16_t*>(shared_w);

  if (path == MOE_PATH_GEMV && T <= ctx->decode_max_t) {
    // the whole layer in one cooperative launch
    const cudaError_t err = launch(ctx, MOE_K_DECODE_FUSED, st, [&] {
      return launch_decode_fused(s, x, router_w, router_b, gu, dn, sw, y, ctx->sc, ctl, ctx->sc.gridbar,
                                 ctx->num_sms, st, ctx->next_wr, ctx->next_shared, kDecodeSmemLimit, ctx->overlap);
    });
    ctx->next_wr = nullptr;  // a hint serves one call
    ctx->next_shared = nullptr;
    return remember_routing(ctx, T, top_k, cuda_fail(err));
  }
  if (path == MOE_PATH_GEMV) {
    if ((rc = run_route(ctx, s, x, router_w, router_b, false, nullptr, st)) != MOE_OK) return rc;
    const Scratch& sc = ctx->sc;
    const int sms = ctx->num_sms;
    cudaError_t err =
        launch(ctx, MOE_K_GEMV_GATE_UP, st, [&] { return launch_gemv_gate_up(s, x, gu, sw, sc, ctl, sms, st); });
    if (err == cudaSuccess)
      err = launch(ctx, MOE_K_GEMV_DOWN, st, [&] { return launch_gemv_down(s, dn, sw, y, sc, ctl, sms, st); });
    return remember_routing(ctx, T, top_k, cuda_fail(err));
  }

  // grouped-GEMM path
  if (s.q4 && !gemm_q4_supported(s.d, s.I)) return MOE_ERR_UNSUPPORTED;
  const bool tensor = use_tensor_router(ctx, s);
  GemmMaps maps;
  memset(&maps, 0, sizeof(maps));
  const uint64_t rows = (uint64_t)s.T * s.k + (s.has_shared ? s.T : 0);
  if (s.x_bf16 && (rc = make_map(ctx, &maps.x_tile, x, s.d, s.T, 64, 128)) != MOE_OK) return rc;
  if (s.x_bf16 && (rc = make_map(ctx, &maps.x_tile16, x, s.d, s.T, 64, 16)) != MOE_OK) return rc;
  if ((rc = make_map(ctx, &maps.x_perm, ctx->sc.x_perm, s.d, rows, 64, 128)) != MOE_OK) return rc;
  if ((rc = make_map(ctx, &maps.x_perm16, ctx->sc.x_perm, s.d, rows, 64, 16)) != MOE_OK) return rc;
  if ((rc = make_map(ctx, &maps.h, ctx->sc.h, s.I, rows, 64, 128)) != MOE_OK) return rc;
  if ((rc = make_map(ctx, &maps.h16, ctx->sc.h, s.I, rows, 64, 16)) != MOE_OK) return rc;
  if ((rc = make_map(ctx, &maps.wr_split, ctx->sc.wr_split, s.d, 3 * s.E, 64, 256)) != MOE_OK) return rc;
  if (s.q4) {
    // 4-bit rows: the routed experts, and the shared expert's gate_up rows followed by its down rows
    const uint8_t* gq = static_cast<const uint8_t*>(experts_gate_up);
    const uint8_t* dq = static_cast<const uint8_t*>(experts_down);
    const uint8_t* sgq = sw ? reinterpret_cast<const uint8_t*>(sw) : gq;
    const uint8_t* sdq = sw ? sgq + (size_t)2 * s.I * (s.d / 16 * 9) : dq;
    const uint64_t egu = (uint64_t)s.E * 2 * s.I, edn = (uint64_t)s.E * s.d;
    if ((rc = make_q4_map(ctx, &maps.gu_codes, gq, s.d, egu, 128, true)) != MOE_OK) return rc;
    if ((rc = make_q4_map(ctx, &maps.gu_params, gq, s.d, egu, 128, false)) != MOE_OK) return rc;
    if ((rc = make_q4_map(ctx, &maps.dn_codes, dq, s.I, edn, 256, true)) != MOE_OK) return rc;
    if ((rc = make_q4_map(ctx, &maps.dn_params, dq, s.I, edn, 256, false)) != MOE_OK) return rc;
    if ((rc = make_q4_map(ctx, &maps.sgu_codes, sgq, s.d, 2 * s.I, 128, true)) != MOE_OK) return rc;
    if ((rc = make_q4_map(ctx, &maps.sgu_params, sgq, s.d, 2 * s.I, 128, false)) != MOE_OK) return rc;
    if ((rc = make_q4_map(ctx, &maps.sdn_codes, sdq, s.I, s.d, 256, true)) != MOE_OK) return rc;
    if ((rc = make_q4_map(ctx, &maps.sdn_params, sdq, s.I, s.d, 256, false)) != MOE_OK) return rc;
  } else {
    if ((rc = make_map(ctx, &maps.gate_up, gu, s.d, (uint64_t)s.E * 2 * s.I, 64, 128)) != MOE_OK) return rc;
    if ((rc = make_map(ctx, &maps.down, dn, s.I, (uint64_t)s.E * s.d, 64, 256)) != MOE_OK) return rc;
    // without a shared expert these maps are never read; point them at routed weights
    const uint16_t* sgu = sw ? sw : gu;
    const uint16_t* sdn = sw ? sw + (size_t)2 * s.I * s.d : dn;
    if ((rc = make_map(ctx, &maps.shared_gu, sgu, s.d, 2 * s.I, 64, 128)) != MOE_OK) return rc;
    if ((rc = make_map(ctx, &maps.shared_down, sdn, s.I, s.d, 64, 256)) != MOE_OK) return rc;
  }

  // routing, grouping, and the token rows written in grouped order (x_perm)
  if ((rc = run_route(ctx, s, x, router_w, router_b, tensor, &maps, st, true)) != MOE_OK) return rc;
  const Scratch& sc = ctx->sc;
  const int sms = ctx->num_sms;
  cudaError_t err = launch(ctx, MOE_K_GEMM_GATE_UP, st, [&] { return launch_gemm_gate_up(s, maps, sc, ctl, sms, st); });
  if (err == cudaSuccess)
    err = launch(ctx, MOE_K_GEMM_DOWN, st, [&] { return launch_gemm_down(s, maps, sc, ctl, sms, st); });
  if (err == cudaSuccess) err = launch(ctx, MOE_K_COMBINE, st, [&] { return launch_combine(s, y, sc, st); });
  return remember_routing(ctx, T, top_k, cuda_fail(err));
}

int moe_status(moe_ctx* ctx) {
  if (!ctx) return MOE_ERR_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, ctx->sc.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v && cudaMemset(ctx->sc.status, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
  // nothing to repair after a timeout: every block of a decode launch that gave
  // up still publishes the launch's epoch, and the next launch tags its values
  // with a new one, so nothing the failed launch wrote is taken as ready
  if (v & kStatusTimeout) return MOE_ERR_TIMEOUT;
  if (v & kStatusBounds) return MOE_ERR_BOUNDS;
  return MOE_OK;
}

void moe_destroy(moe_ctx* ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  if (ctx->block) cudaFree(ctx->block);
  delete ctx;
}

}  // extern "C"
