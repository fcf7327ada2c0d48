// notify.cuh -- the body of notify_dispatch (llm-infra-atlas DeepEP article
// §2.1, §2.3, §4.3) as a device function of one CTA, shared by the notify
// kernel and by the layout kernel's last CTA (layout and notify in one
// launch).
#pragma once

#include "ep_common.cuh"

namespace ep {

struct NotifyParams {
  const int32_t* num_tokens_per_rank;
  const int32_t* num_tokens_per_expert;
  int R, E, E_l, expert_alignment;
  int64_t num_worst_tokens;
  int32_t* rank_prefix_matrix;
  int32_t* expert_prefix;
  int32_t* num_recv_tokens_per_expert;
  int64_t* psum;
  int64_t* host_recv_rows;   // device view of host-mapped memory, or null
  int32_t* status;
};

// Every column walks R source ranks; its loads go out kNotifyBatch at a time
// (ahead of the stores), so a column costs R / kNotifyBatch memory round
// trips instead of R.  The aligned totals are kept in shared memory (s_recv,
// E words) for the per-rank segment starts.
constexpr int kNotifyBatch = 16;

// The prefix tables, computed by the nt threads of one CTA (tid < nt).
// kCoherent: the count tables were written by other CTAs of the running
// kernel, so they are read through L2, not the read-only path.
template <bool kCoherent>
__device__ __forceinline__ void notify_tables(const NotifyParams& p, int tid, int nt,
                                              int32_t* s_recv) {
  auto ld = [](const int32_t* q) { return kCoherent ? ld_cg_i32(q) : __ldg(q); };
  // expert totals: exclusive prefix over source ranks, then aligned totals
  for (int e = tid; e < p.E; e += nt) {
    int32_t run = 0;
    for (int i0 = 0; i0 < p.R; i0 += kNotifyBatch) {
      int32_t c[kNotifyBatch];
#pragma unroll
      for (int u = 0; u < kNotifyBatch; ++u)
        c[u] = i0 + u < p.R ? ld(&p.num_tokens_per_expert[(size_t)(i0 + u) * p.E + e]) : 0;
#pragma unroll
      for (int u = 0; u < kNotifyBatch; ++u) {
        if (i0 + u < p.R) {
          p.expert_prefix[(size_t)(i0 + u) * p.E + e] = run;
          run += c[u];
        }
      }
    }
    p.expert_prefix[(size_t)p.R * p.E + e] = run;
    const int32_t a = p.expert_alignment;
    const int32_t aligned = (run + a - 1) / a * a;
    p.num_recv_tokens_per_expert[e] = aligned;
    s_recv[e] = aligned;
  }
  // token-level prefix matrix, inclusive over source ranks
  for (int j = tid; j < p.R; j += nt) {
    int32_t run = 0;
    for (int i0 = 0; i0 < p.R; i0 += kNotifyBatch) {
      int32_t c[kNotifyBatch];
#pragma unroll
      for (int u = 0; u < kNotifyBatch; ++u)
        c[u] = i0 + u < p.R ? ld(&p.num_tokens_per_rank[(size_t)(i0 + u) * p.R + j]) : 0;
#pragma unroll
      for (int u = 0; u < kNotifyBatch; ++u) {
        if (i0 + u < p.R) {
          run += c[u];
          p.rank_prefix_matrix[(size_t)(i0 + u) * p.R + j] = run;
        }
      }
    }
    if (p.num_worst_tokens >= 0 && run > p.num_worst_tokens) set_status(p.status, EP_ERR_CAPACITY);
  }
  __syncthreads();
  // segment starts per destination rank
  for (int r = tid; r < p.R; r += nt) {
    int64_t s = 0;
    int64_t* ps = p.psum + (size_t)r * (p.E_l + 1);
    ps[0] = 0;
    for (int l = 0; l < p.E_l; ++l) {
      s += s_recv[r * p.E_l + l];
      ps[l + 1] = s;
    }
    if (p.host_recv_rows != nullptr) {
      *reinterpret_cast<volatile int64_t*>(&p.host_recv_rows[r]) = s;
    }
  }
  if (p.host_recv_rows != nullptr) __threadfence_system();
}

}  // namespace ep
