// Host side of the fused decode layer: kernel choice by token count, the
// shared-memory ring sizing, the cooperative launch, and the allocation-free
// entry point.  The kernel itself is in moe_decode_kernel.cuh; each token
// bound MAXT is instantiated in its own translation unit (moe_decode_k*.cu)
// so that the instantiations compile in parallel.
#include <mutex>

#include "moe_decode_kernel.cuh"

namespace moe {

// defined in moe_decode_k<MAXT>.cu
const void* decode_kernel_maxt1(const Shapes& s);
const void* decode_kernel_maxt2(const Shapes& s);
const void* decode_kernel_maxt4(const Shapes& s);
const void* decode_kernel_maxt8(const Shapes& s);
const void* decode_kernel_maxt16(const Shapes& s);
// defined in moe_decode_q4_k<MAXT>.cu (4-bit weights)
const void* decode_kernel_q4_maxt1(const Shapes& s);
const void* decode_kernel_q4_maxt2(const Shapes& s);
const void* decode_kernel_q4_maxt4(const Shapes& s);
const void* decode_kernel_q4_maxt8(const Shapes& s);
const void* decode_kernel_q4_maxt16(const Shapes& s);

// The smallest instantiated token bound MAXT >= T: the per-token loops of
// phases B and C are unrolled over MAXT, so a tight bound saves issue slots
// (measured at d = 2048, I = 512: T = 4 took 101 us per layer with MAXT = 16,
// 66 us with MAXT = 4).
static const void* decode_kernel_for(const Shapes& s) {
  if (s.q4) {
    if (s.T <= 1) return decode_kernel_q4_maxt1(s);
    if (s.T <= 2) return decode_kernel_q4_maxt2(s);
    if (s.T <= 4) return decode_kernel_q4_maxt4(s);
    if (s.T <= 8) return decode_kernel_q4_maxt8(s);
    if (s.T <= 16) return decode_kernel_q4_maxt16(s);
    return nullptr;
  }
  if (s.T <= 1) return decode_kernel_maxt1(s);
  if (s.T <= 2) return decode_kernel_maxt2(s);
  if (s.T <= 4) return decode_kernel_maxt4(s);
  if (s.T <= 8) return decode_kernel_maxt8(s);
  if (s.T <= 16) return decode_kernel_maxt16(s);
  return nullptr;
}

// Dynamic shared memory a kernel instantiation may use: the per-block opt-in
// maximum less its static shared memory (looked up once per kernel and device).
static int decode_dyn_limit(const void* k) {
  struct Entry {
    const void* k;
    int dev, lim;
  };
  static Entry cache[128];
  static int n_cache = 0;
  static std::mutex mu;
  int dev = 0;
  if (!k || cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].k == k && cache[i].dev == dev) return cache[i].lim;
  int optin = 0;
  cudaFuncAttributes fa;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, k) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int lim = optin - (int)fa.sharedSizeBytes;
  if (n_cache < 128) cache[n_cache++] = {k, dev, lim};
  return lim;
}

// The weight ring: slots hold one gate/up unit (2 d bf16, or the two 4-bit
// code rows and their parameters) or the down rows of top_k + 1 experts (a
// whole phase-C row at batch 1), whichever is larger; as many slots as the
// shared memory left after x / h holds, up to kRingSlots (bf16) or
// kRingSlotsQ4 (4-bit items are 3.7 times smaller, so more of them must be in
// flight to cover the same memory latency).
constexpr int kRingSlotsQ4 = kMaxSlots;
struct DecodeRing {
  int slots, slot_bytes, chunk;
};
static DecodeRing decode_ring(const Shapes& s, int max_smem) {
  DecodeRing r{0, 0, 0};
  const void* k = decode_kernel_for(s);
  if (!k) return r;
  const int lim = decode_dyn_limit(k);
  const long long budget = (long long)(max_smem < lim ? max_smem : lim) - (long long)decode_big_bytes(s);
  // bytes of one gate/up unit and of one expert's down row
  const int unit = s.q4 ? s.d + s.d / 8 : 4 * s.d;
  const int drow1 = s.q4 ? s.I / 2 + s.I / 16 : 2 * s.I;
  const int drow = drow1 * (s.k + 1);
  const int widest = unit > drow ? unit : drow;
  r.slot_bytes = (widest + 15) / 16 * 16;
  r.chunk = r.slot_bytes / drow1;
  const long long n = budget > 0 ? budget / r.slot_bytes : 0;
  const int cap = s.q4 ? kRingSlotsQ4 : kRingSlots;
  r.slots = (int)(n < cap ? n : cap);
  return r;
}

size_t decode_smem_bytes(const Shapes& s, int max_smem) {
  const DecodeRing r = decode_ring(s, max_smem);
  return decode_big_bytes(s) + (size_t)r.slots * r.slot_bytes;
}

// Below this ring depth every refill wave adds a memory round trip and the
// kernel falls off a cliff (d = 2048, I = 512: T = 10 leaves a few slots and
// took 480-800 us per layer, against ~110 us on the grouped GEMMs); such calls
// go to the modular GEMV kernels instead.
constexpr int kMinRingSlots = 6;

bool decode_supported(const Shapes& s, int max_smem) {
  const void* k = decode_kernel_for(s);
  if (!(s.T <= 16 && s.d % 256 == 0 && s.I % 256 == 0 && k != nullptr)) return false;
  return decode_ring(s, max_smem).slots >= kMinRingSlots;
}

cudaError_t prepare_decode_kernels(int max_smem) {
  for (int T : {1, 2, 4, 8, 16})
    for (int d : {512, 1024, 2048})
      for (int I : {256, 512, 1024})
        for (int xb = 0; xb < 4; ++xb) {
          Shapes s{};
          s.T = T;
          s.d = d;
          s.I = I;
          s.x_bf16 = xb & 1;
          s.q4 = xb >> 1;
          const void* k = decode_kernel_for(s);
          if (!k) continue;
          const int lim = decode_dyn_limit(k);
          cudaError_t err =
              cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem < lim ? max_smem : lim);
          if (err != cudaSuccess) return err;
        }
  return cudaSuccess;
}

int decode_blocks_per_sm(const Shapes& s, int max_smem) {
  int n = 0;
  const void* k = decode_kernel_for(s);
  if (!k ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, decode_smem_bytes(s, max_smem)) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t launch_decode_fused(const Shapes& s, const void* x, const float* wr, const float* rb,
                                const uint16_t* gate_up, const uint16_t* down, const uint16_t* shared_w, void* y,
                                const Scratch& sc, const DevCtl& ctl, unsigned* bar, int num_sms, cudaStream_t st,
                                const float* next_wr, const uint16_t* next_shared, int max_smem, bool overlap) {
  const DecodeRing ring = decode_ring(s, max_smem);
  if (ring.slots < 2) return cudaErrorInvalidValue;
  DecodeArgs a;
  a.ring_slots = ring.slots;
  a.slot_bytes = ring.slot_bytes;
  a.chunk_experts = ring.chunk;
  a.next_wr = next_wr;
  a.next_shared = next_shared;
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
  // 4-bit weights: the shared expert's down rows follow its 2I gate_up rows (9 d / 16 bytes each)
  a.sh_down_q4 = (s.q4 && shared_w) ? reinterpret_cast<const uint8_t*>(shared_w) + (size_t)2 * s.I * (s.d / 16 * 9)
                                     : nullptr;
  const void* k = decode_kernel_for(s);
  if (!k) return cudaErrorInvalidValue;
  void* params[] = {&a};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = decode_big_bytes(s) + (size_t)ring.slots * ring.slot_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 2 : 1;
  return cudaLaunchKernelExC(&cfg, k, params);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free variant of the fused decode layer (moe_decode_noalloc).
//
// Some callers cannot call cudaMalloc, so they cannot create a context with
// moe_init: a plugin running inside a host application whose device memory
// belongs to the host's own allocator (the host hands out every buffer and
// forbids allocations outside its pool), and serving loops with a fixed
// latency budget, where an allocation may synchronise the device and stall
// every stream.  For them the same kernel runs on scratch memory that is part
// of the library image: one file-scope device array, sized for the limits
// below, that every GPU loading the library holds until exit.  The host
// learns its device address once per device with cudaGetSymbolAddress; the
// array's name in host code is only a host-side stand-in, never a device
// address.
// ---------------------------------------------------------------------------

using namespace moe;

namespace {

constexpr int kNoAllocMaxT = 16;
constexpr int kNoAllocMaxTopK = 8;
constexpr int kNoAllocMaxInter = 1024;
constexpr size_t kNoAllocH = (size_t)kNoAllocMaxT * (kNoAllocMaxTopK + 1) * kNoAllocMaxInter * 8;  // tagged h rows
constexpr int kNoAllocReps = 4;  // copies of the logits
constexpr size_t kNoAllocLogits = (size_t)kNoAllocReps * kNoAllocMaxT * kMaxExperts * 8;  // tagged logits
constexpr size_t kNoAllocPicks = (size_t)kNoAllocMaxT * kNoAllocMaxTopK * 4;
constexpr size_t kNoAllocOffLogits = kNoAllocH;
constexpr size_t kNoAllocOffIdx = kNoAllocOffLogits + kNoAllocLogits;
constexpr size_t kNoAllocOffW = kNoAllocOffIdx + kNoAllocPicks;
constexpr size_t kNoAllocOffStatus = kNoAllocOffW + kNoAllocPicks;
constexpr size_t kNoAllocOffBar = kNoAllocOffStatus + 256;  // control words: the 64-bit epoch counter
constexpr size_t kNoAllocBarBytes = 256;
constexpr size_t kNoAllocBytes = kNoAllocOffBar + kNoAllocBarBytes;

struct NoAllocDevice {
  bool ready = false;
  unsigned char* base = nullptr;  // device address of the array on this device
  int sms = 0;
};
constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

}  // namespace

// The scratch array (1,312,256 bytes, about 1.3 MB: tagged h rows 1.18 MB,
// tagged logits 128 KB, picks, status and control words).  Every call shares
// it and it keeps the last call's contents.  Its zero initial contents are a
// valid start: tag 0 is never a launch's epoch, and nothing must be cleared
// between calls (the epoch counter is kept, since a tag left by an earlier
// call must never match a later one).
static_assert(kNoAllocBytes == 1312256, "the documented size of the allocation-free scratch array");
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
  const int smem_limit = kDecodeSmemLimit;
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
  if (decode_blocks_per_sm(s, smem_limit) < 1) return MOE_ERR_UNSUPPORTED;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* words = reinterpret_cast<unsigned*>(nd.base + kNoAllocOffStatus);
  unsigned* bar = reinterpret_cast<unsigned*>(nd.base + kNoAllocOffBar);
  Scratch sc{};
  sc.dec_h = reinterpret_cast<float*>(nd.base);
  sc.dec_hreps = 1;
  sc.dec_logits = reinterpret_cast<float*>(nd.base + kNoAllocOffLogits);
  sc.dec_reps = kNoAllocReps;
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
                          ctl, bar, nd.sms, st, nullptr, nullptr, smem_limit);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
