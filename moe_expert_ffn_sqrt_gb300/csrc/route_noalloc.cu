// moe_route_noalloc: the routing call without a workspace and without any allocation.
//
// Some callers cannot hand this library a workspace and cannot allocate one either: for
// example an inference engine that plans every device buffer before it starts and forbids
// cudaMalloc afterwards, a plugin interface that passes in only its inputs and outputs, or code
// running where an allocation would stall or fail.  For them this entry point keeps the
// routing scratch in a fixed array in device memory that is part of the library image, so the
// call needs nothing beyond its inputs and outputs.
//
// Properties of the array:
//   * 4 MiB (kNoAllocScratchBytes), held on every GPU that loads the library until the process
//     exits.  Layout: [0, 256) a word that records whether this call's tensor-core gate GEMM
//     (T > 16) gave up on a wait; [256, ...) the routing scratch of route.cu: a 256-byte ticket
//     slot at a fixed place, the split-over-H partial gate sums (nsplit * T * E * 4 bytes, rounded
//     up to 256; nsplit = 4 for T <= 16), and for T > 16 the three bf16 parts of the gate weight
//     (3 * E * H * 2 bytes).  Problems whose scratch does not fit are rejected with
//     MOE_ERR_UNSUPPORTED before anything is launched.
//   * Shared by every call on a device and left holding the last call's partial sums.  A call
//     reads only partial sums and gate parts that it wrote itself.  The ticket counter is zero when
//     the library loads and every call that uses it leaves it at zero, and it sits at the same
//     address for every problem size, so a call never sees another call's count.  The failure word
//     is cleared (cudaMemsetAsync, no allocation) at the start of every call above 16 tokens.
//     Calls that can overlap on the GPU (different streams without ordering) race on the array.
//   * There is no workspace to hold a device-side status, so a wait timeout inside the gate GEMM
//     is reported in the outputs: every topk_ids entry is -1 and every weight (and logit) NaN.
//   * Host code cannot pass the array's name to a kernel (on the host it is only a stand-in for
//     the device symbol), so the first call on each device looks up its device address with
//     cudaGetSymbolAddress while that device is current and caches it.  That first call is a
//     host-side query: make it before any stream capture begins.
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
constexpr size_t kFailSlot = 256;          // [0, 256): the gate-failure word; routing scratch after it
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint32_t g_route_scratch[kNoAllocScratchBytes / sizeof(uint32_t)];

char* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_route_scratch on the current device (looked up once per device).
moe_status scratch_on_current_device(char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<char*>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" moe_status moe_route_noalloc(const uint16_t* hidden, const float* w_gate, const float* gate_bias,
                                        const float* e_score_bias, int T, int H, int E, int K, moe_score_fn fn,
                                        int renormalize, float* logits_out, int32_t* topk_ids, float* topk_w,
                                        uint8_t* x_q, uint8_t* x_sf, void* stream) {
  if (T < 0 || H <= 0 || H % 128 || E <= 0 || E > 1024 || K <= 0 || K > E || K > 32) return MOE_ERR_INVALID_ARG;
  if (!hidden || !w_gate || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (fn != MOE_SCORE_SOFTMAX && fn != MOE_SCORE_SQRT_SOFTPLUS) return MOE_ERR_INVALID_ARG;
  if ((x_q == nullptr) != (x_sf == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(w_gate)) return MOE_ERR_INVALID_ARG;
  if (x_q && (reinterpret_cast<uintptr_t>(x_q) & 3)) return MOE_ERR_INVALID_ARG;
  if (kFailSlot + moe::route_scratch_bytes(T, H, E) > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  char* base = nullptr;
  const moe_status st = scratch_on_current_device(&base);
  if (st != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* fail = reinterpret_cast<uint32_t*>(base);
  if (T > 16 && cudaMemsetAsync(fail, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  const cudaError_t err = moe::launch_route(hidden, w_gate, gate_bias, e_score_bias, T, H, E, K, static_cast<int>(fn),
                                            renormalize, logits_out, topk_ids, topk_w, x_q, x_sf, base + kFailSlot,
                                            fail, s, nullptr, fail);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
