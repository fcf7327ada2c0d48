// notify.cu -- notify_dispatch: exchange of the [R, R] / [R, E] count
// matrices and the prefix sums the receivers need (llm-infra-atlas DeepEP
// article §2.1, §2.3, §4.3).
//
// In DeepEP every rank writes its counts into its peers' buffers over NVLink
// and then scans along the source-rank dimension.  With the ranks emulated
// as partitions of one HBM, the stacked [R, R] / [R, E] count matrices are
// already "all-to-all'ed"; one CTA computes every rank's prefixes:
//   rank_prefix_matrix (inclusive over source ranks, token level),
//   expert_prefix      (exclusive over source ranks, plus the totals row),
//   num_recv_tokens_per_expert (totals aligned to expert_alignment),
//   psum               (exclusive prefix of the aligned totals = segment
//                       starts, V2's psum_num_recv_tokens_per_expert),
// and optionally publishes each rank's receive row count to host-mapped
// memory for the CPU handshake of §2.1.

#include <chrono>
#include <thread>

#include "notify.cuh"

namespace ep {

constexpr int kNotifyThreads = 1024;

// staged: the count tables are loaded into dynamic shared memory first
// (notify_stage_words(R, E) words), see notify_tables.
__global__ void __launch_bounds__(kNotifyThreads) k_notify(NotifyParams p, int staged) {
  __shared__ int32_t s_recv[kMaxE];
  extern __shared__ __align__(16) int32_t s_stage[];
  notify_tables<false>(p, threadIdx.x, kNotifyThreads, s_recv, staged ? s_stage : nullptr);
}

}  // namespace ep

extern "C" int ep_host_wait_counters(const volatile int64_t* counters, int n, int timeout_ms) {
  if (counters == nullptr || n < 0) return EP_ERR_INVALID_ARG;
  const auto t0 = std::chrono::steady_clock::now();
  int spins = 0;
  while (true) {
    bool ready = true;
    for (int r = 0; r < n; ++r) {
      if (counters[r] < 0) {
        ready = false;
        break;
      }
    }
    if (ready) return EP_OK;
    const auto dt = std::chrono::steady_clock::now() - t0;
    if (std::chrono::duration_cast<std::chrono::milliseconds>(dt).count() >= timeout_ms)
      return EP_ERR_TIMEOUT;
    if (++spins > 1024) std::this_thread::yield();
  }
}

extern "C" int ep_notify_dispatch(const int32_t* num_tokens_per_rank,
                                  const int32_t* num_tokens_per_expert, int R, int E,
                                  int expert_alignment, int64_t num_worst_tokens,
                                  int32_t* rank_prefix_matrix, int32_t* expert_prefix,
                                  int32_t* num_recv_tokens_per_expert, int64_t* psum,
                                  int64_t* host_recv_rows, int timeout_ms, int32_t* status,
                                  void* stream) {
  if (R <= 0 || R > ep::kMaxR || E <= 0 || E > ep::kMaxE || E % R != 0 || expert_alignment <= 0)
    return EP_ERR_INVALID_ARG;
  if (!num_tokens_per_rank || !num_tokens_per_expert || !rank_prefix_matrix || !expert_prefix ||
      !num_recv_tokens_per_expert || !psum)
    return EP_ERR_INVALID_ARG;
  ep::NotifyParams p{};
  p.num_tokens_per_rank = num_tokens_per_rank;
  p.num_tokens_per_expert = num_tokens_per_expert;
  p.R = R;
  p.E = E;
  p.E_l = E / R;
  p.expert_alignment = expert_alignment;
  p.num_worst_tokens = num_worst_tokens;
  p.rank_prefix_matrix = rank_prefix_matrix;
  p.expert_prefix = expert_prefix;
  p.num_recv_tokens_per_expert = num_recv_tokens_per_expert;
  p.psum = psum;
  p.status = status;
  const bool wait = host_recv_rows != nullptr && num_worst_tokens < 0;
  if (host_recv_rows != nullptr) {
    void* dev = nullptr;
    if (cudaHostGetDevicePointer(&dev, host_recv_rows, 0) != cudaSuccess) {
      cudaGetLastError();
      return EP_ERR_INVALID_ARG;
    }
    volatile int64_t* h = host_recv_rows;
    for (int r = 0; r < R; ++r) h[r] = -1;
    p.host_recv_rows = static_cast<int64_t*>(dev);
  }
  const int64_t words = ep::notify_stage_words(R, E);
  const bool staged = words <= ep::kNotifyStageMaxWords;
  {
    const int rc = ep_host::ensure_max_smem(reinterpret_cast<const void*>(ep::k_notify),
                                            ep::kNotifyStageMaxWords * (int)sizeof(int32_t));
    if (rc != EP_OK) return rc;
  }
  ep::k_notify<<<1, ep::kNotifyThreads, staged ? (size_t)words * sizeof(int32_t) : 0,
                 static_cast<cudaStream_t>(stream)>>>(p, staged ? 1 : 0);
  ep_host::count_launch();
  int rc = ep_host::check_launch();
  if (rc != EP_OK || !wait) return rc;
  return ep_host_wait_counters(host_recv_rows, R, timeout_ms);
}
