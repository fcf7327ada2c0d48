// layout_static.cu -- ep_get_dispatch_layout_no_alloc: get_dispatch_layout
// for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocator) at all: code inside
// a custom memory pool or allocator callback, and runtimes that hand the
// library fixed buffers and forbid it from touching the device heap.  They still need the
// layout kernel, whose decoupled look-back keeps per-chunk words and ticket
// counters in scratch memory.  This entry point keeps that scratch in a
// file-scope __device__ array of kStaticScratchBytes, so the caller passes
// only its inputs and outputs.
//
// Costs and rules of the static scratch:
//  - every GPU that loads libep holds the 4 MiB array until the process exits;
//  - problems whose look-back state exceeds it are rejected (EP_ERR_TOO_LARGE);
//  - all calls share the one array: calls that overlap on the GPU race, so
//    they must be ordered on one stream (or otherwise serialised);
//  - the array keeps the last call's contents, so each call first clears the
//    part it uses (a stream-ordered memset, no allocation);
//  - the first call on a device looks the array's device address up with
//    cudaGetSymbolAddress (with that device current).  The address is kept
//    for the life of the process, so the library must not be used on a device after
//    cudaDeviceReset on it;
//  - the stream must belong to the current device (the array looked up is
//    the current device's); a stream of another device is refused with
//    EP_ERR_INVALID_ARG before anything is launched.

#include <mutex>

#include "ep_common.cuh"
#include "layout.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kMaxDevices = 64;

// Host code must not use this name as an address: it is a host-side stand-in
// for the device array.  The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_layout_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_layout_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return EP_ERR_CUDA;
    }
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return EP_OK;
}

}  // namespace

extern "C" int ep_get_dispatch_layout_no_alloc(const int64_t* topk_idx, int R, int T_r, int k,
                                               int E, int32_t* num_tokens_per_rank,
                                               int32_t* num_tokens_per_expert,
                                               uint8_t* is_token_in_rank, int32_t* slot_rank,
                                               int32_t* status, void* stream) {
  if (R <= 0 || R > ep::kMaxR || E <= 0 || E > ep::kMaxE || E % R != 0 || k <= 0 ||
      k > ep::kMaxK || T_r < 0)
    return EP_ERR_INVALID_ARG;
  const size_t bytes = ep::layout_geometry(R, T_r, k, E, ep::kNormalChunkIds).bytes;
  if (bytes > kStaticScratchBytes) return EP_ERR_TOO_LARGE;
  if (!num_tokens_per_rank || !num_tokens_per_expert ||
      (T_r > 0 && (!topk_idx || !is_token_in_rank || !slot_rank)))
    return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread) {
    int cur = -1, sdev = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess) {
      cudaGetLastError();
      return EP_ERR_INVALID_ARG;
    }
    if (sdev != cur) return EP_ERR_INVALID_ARG;   // scratch of one device, work on another
  }
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != EP_OK) return rc;
  // start from a clean scratch: ticket / epoch words and look-back words
  if (cudaMemsetAsync(scratch, 0, bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  ep::LayoutParams p{};
  p.topk_idx = topk_idx;
  p.R = R;
  p.T_r = T_r;
  p.k = k;
  p.E = E;
  p.E_l = E / R;
  p.num_tokens_per_rank = num_tokens_per_rank;
  p.num_tokens_per_expert = num_tokens_per_expert;
  p.is_token_in_rank = is_token_in_rank;
  p.slot_rank = slot_rank;
  p.status = status;
  return ep::launch_layout(p, false, scratch, s);
}
