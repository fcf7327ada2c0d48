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

// Every column walks R source ranks.  When the two count tables fit in
// shared memory (notify_stage_words(R, E) <= kNotifyStageMaxWords) they are
// first loaded there by every thread at once -- one memory round trip --
// and the prefixes run from shared memory.  Otherwise each column's loads
// go out kNotifyBatch at a time (ahead of the stores), so a column costs
// R / kNotifyBatch memory round trips instead of R.  The aligned totals are
// kept in shared memory (s_recv, E words) for the per-rank segment starts.
constexpr int kNotifyBatch = 16;
constexpr int kNotifyStageMaxWords = 24 * 1024;   // 96 KB of staged counts

__host__ __device__ inline int64_t notify_stage_words(int R, int E) {
  return (int64_t)R * E + (int64_t)R * R;
}

// Copy n int32 words from global (src) to shared memory (dst), every
// thread's loads in flight before its stores; 16-byte loads when src is
// 16-byte aligned.
template <bool kCoherent>
__device__ __forceinline__ void stage_words(int32_t* dst, const int32_t* src, int n, int tid, int nt) {
  constexpr int kUnroll = 4;
  if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    const int n4 = n / 4;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int q0 = tid; q0 < n4; q0 += nt * kUnroll) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int q = q0 + u * nt;
        if (q < n4) v[u] = kCoherent ? ld_cg_v4(s4 + q) : __ldg(s4 + q);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (q0 + u * nt < n4) d4[q0 + u * nt] = v[u];
    }
    for (int q = n4 * 4 + tid; q < n; q += nt) dst[q] = kCoherent ? ld_cg_i32(src + q) : __ldg(src + q);
  } else {
    for (int q0 = tid; q0 < n; q0 += nt * kUnroll) {
      int32_t v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int q = q0 + u * nt;
        if (q < n) v[u] = kCoherent ? ld_cg_i32(src + q) : __ldg(src + q);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (q0 + u * nt < n) dst[q0 + u * nt] = v[u];
    }
  }
}

// The prefix tables, computed by the nt threads of one CTA (tid < nt).
// kCoherent: the count tables were written by other CTAs of the running
// kernel, so they are read through L2, not the read-only path.  s_recv: E
// words of shared memory; s_stage: notify_stage_words(R, E) words of shared
// memory (16-byte aligned), or null for the column-walking form.
template <bool kCoherent>
__device__ __forceinline__ void notify_tables(const NotifyParams& p, int tid, int nt,
                                              int32_t* s_recv, int32_t* s_stage) {
  auto ld = [](const int32_t* q) { return kCoherent ? ld_cg_i32(q) : __ldg(q); };
  const int32_t* cnt_e = p.num_tokens_per_expert;   // [R][E]
  const int32_t* cnt_r = p.num_tokens_per_rank;     // [R][R]
  const bool staged = s_stage != nullptr;
  if (staged) {
    stage_words<kCoherent>(s_stage, cnt_e, p.R * p.E, tid, nt);
    stage_words<kCoherent>(s_stage + p.R * p.E, cnt_r, p.R * p.R, tid, nt);
    __syncthreads();
  }
  // expert totals: exclusive prefix over source ranks, then aligned totals
  for (int e = tid; e < p.E; e += nt) {
    int32_t run = 0;
    if (staged) {
      for (int i = 0; i < p.R; ++i) {
        p.expert_prefix[(size_t)i * p.E + e] = run;
        run += s_stage[i * p.E + e];
      }
    } else {
      for (int i0 = 0; i0 < p.R; i0 += kNotifyBatch) {
        int32_t c[kNotifyBatch];
#pragma unroll
        for (int u = 0; u < kNotifyBatch; ++u)
          c[u] = i0 + u < p.R ? ld(&cnt_e[(size_t)(i0 + u) * p.E + e]) : 0;
#pragma unroll
        for (int u = 0; u < kNotifyBatch; ++u) {
          if (i0 + u < p.R) {
            p.expert_prefix[(size_t)(i0 + u) * p.E + e] = run;
            run += c[u];
          }
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
    if (staged) {
      const int32_t* sr = s_stage + p.R * p.E;
      for (int i = 0; i < p.R; ++i) {
        run += sr[i * p.R + j];
        p.rank_prefix_matrix[(size_t)i * p.R + j] = run;
      }
    } else {
      for (int i0 = 0; i0 < p.R; i0 += kNotifyBatch) {
        int32_t c[kNotifyBatch];
#pragma unroll
        for (int u = 0; u < kNotifyBatch; ++u)
          c[u] = i0 + u < p.R ? ld(&cnt_r[(size_t)(i0 + u) * p.R + j]) : 0;
#pragma unroll
        for (int u = 0; u < kNotifyBatch; ++u) {
          if (i0 + u < p.R) {
            run += c[u];
            p.rank_prefix_matrix[(size_t)(i0 + u) * p.R + j] = run;
          }
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
