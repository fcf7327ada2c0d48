// api.cu -- host-side helpers and the small entry points of libep.

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "ep_common.cuh"

namespace ep_host {

static std::atomic<uint64_t> g_launches{0};

int num_sms() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 1;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 1;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

int64_t l2_bytes() {
  static std::mutex mu;
  static int64_t cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 1;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

static std::atomic<int> g_sm_budget{0};   // 0: every SM

int grid_cap(int ctas_per_sm) {
  const int sms = num_sms();
  const int budget = g_sm_budget.load(std::memory_order_relaxed);
  return budget > 0 ? std::min(budget, sms) : sms * ctas_per_sm;
}

int device_view(void* p, void** dev) {
  *dev = p;
  if (p == nullptr) return EP_OK;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_INVALID_ARG;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return EP_OK;
    case cudaMemoryTypeHost:
      if (a.devicePointer == nullptr) return EP_ERR_INVALID_ARG;
      *dev = a.devicePointer;
      return EP_OK;
    default:
      return EP_ERR_INVALID_ARG;
  }
}

bool sm_budget_set() { return g_sm_budget.load(std::memory_order_relaxed) > 0; }

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int check_launch() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

int ensure_max_smem(const void* func, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;   // largest limit set per (kernel, device)
  std::lock_guard<std::mutex> lock(mu);
  const auto it = done.find({func, dev});
  if (it != done.end() && it->second >= bytes) return EP_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  done[{func, dev}] = bytes;
  return EP_OK;
}

}  // namespace ep_host

extern "C" int ep_clean_ll_buffer(int32_t* recv_count, int R, int E, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (R <= 0 || E <= 0 || E % R != 0) return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (recv_count != nullptr &&
      cudaMemsetAsync(recv_count, 0, sizeof(int32_t) * (size_t)E, s) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  if (workspace != nullptr && workspace_bytes > 0 &&
      cudaMemsetAsync(workspace, 0, workspace_bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  return EP_OK;
}

extern "C" int ep_read_status(const int32_t* status, int32_t* host_value, void* stream) {
  if (status == nullptr || host_value == nullptr) return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_value, status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  return EP_OK;
}

extern "C" int ep_set_num_sms(int num_sms) {
  if (num_sms < 0) return EP_ERR_INVALID_ARG;
  ep_host::g_sm_budget.store(num_sms, std::memory_order_relaxed);
  return EP_OK;
}

extern "C" int ep_get_num_sms(void) { return ep_host::grid_cap(1); }

extern "C" uint64_t ep_launch_count(void) {
  return ep_host::g_launches.load(std::memory_order_relaxed);
}

extern "C" const char* ep_error_string(int code) {
  switch (code) {
    case EP_OK: return "ok";
    case EP_ERR_INVALID_ARG: return "invalid argument";
    case EP_ERR_CAPACITY: return "receive buffer capacity exceeded";
    case EP_ERR_TIMEOUT: return "wait timed out";
    case EP_ERR_CUDA: return "CUDA error";
    case EP_ERR_STATE: return "workspace not initialised (call ep_clean_ll_buffer)";
    case EP_ERR_TOO_LARGE: return "problem exceeds the no-allocation entry point's static scratch";
    default: return "unknown error";
  }
}
