// rank.cu -- the once-per-rank receive layout of DeepEP V1's normal mode
// (llm-infra-atlas DeepEP article §2.1, §2.3): a token goes ONCE to every
// rank that holds one of its experts, source rank i's tokens landing at
// rank_prefix_matrix[i-1][r] in token order, and the combine sums the rows
// the ranks return.
//
// The layout is the per-expert pipeline run on derived ids: slot j of a
// token carries its destination rank r = e / E_l if j is the token's first
// slot on r, else -1 (ep_rank_ids).  With those ids and "experts" = ranks
// (E' = R, one per rank), get_dispatch_layout counts tokens per (source,
// destination) and ranks each token among source rank i's tokens for r;
// notify's expert_prefix becomes the exclusive rank prefix (the row start
// of source rank i in rank r's buffer) and psum[r] = [0, total]; dispatch
// then writes exactly the V1 rows.  ep_rank_recv_topk adds each received
// row's local top-k ids and weights; ep_rank_combine sums the returned rows.

#include "ep_common.cuh"

namespace ep {

constexpr int kRankThreads = 256;

__global__ void __launch_bounds__(kRankThreads) k_rank_ids(const int64_t* __restrict__ idx, int64_t T,
                                                           int k, int E, int E_l, int64_t* rank_ids,
                                                           int32_t* status) {
  const int64_t t = (int64_t)blockIdx.x * kRankThreads + threadIdx.x;
  if (t >= T) return;
  int r_seen[kMaxK];
  int n_seen = 0;
  bool bad = false;
  for (int j = 0; j < k; ++j) {
    const int64_t e = __ldg(&idx[t * k + j]);
    int64_t out = -1;
    if (e >= 0 && e < E) {
      const int r = (int)(e / E_l);
      bool first = true;
      for (int q = 0; q < n_seen; ++q) first &= (r_seen[q] != r);
      if (first) {
        r_seen[n_seen++] = r;
        out = r;
      }
    } else if (e != -1) {
      bad = true;
    }
    rank_ids[t * k + j] = out;
  }
  if (bad) set_status(status, EP_ERR_INVALID_ARG);
}

// One thread per (token, slot): a slot pointing at a received row (the
// token's first slot on that rank) fills the row's k local ids / weights.
__global__ void __launch_bounds__(kRankThreads) k_rank_recv_topk(
    const int64_t* __restrict__ idx, const float* __restrict__ w, const int32_t* __restrict__ cidx,
    int64_t T, int k, int E, int E_l, int64_t cap_rows, int64_t n_rows, int64_t* recv_topk_idx,
    float* recv_topk_weights, int32_t* status) {
  const int64_t s = (int64_t)blockIdx.x * kRankThreads + threadIdx.x;
  if (s >= T * k) return;
  const int32_t f = __ldg(&cidx[s]);
  if (f < 0) return;
  if ((int64_t)f >= n_rows) {
    set_status(status, EP_ERR_INVALID_ARG);
    return;
  }
  const int64_t t = s / k;
  const int64_t r = f / cap_rows;
  for (int j = 0; j < k; ++j) {
    const int64_t e = __ldg(&idx[t * k + j]);
    const bool on_r = e >= 0 && e < E && e / E_l == r;
    recv_topk_idx[(int64_t)f * k + j] = on_r ? e - r * E_l : -1;
    recv_topk_weights[(int64_t)f * k + j] = on_r ? __ldg(&w[t * k + j]) : 0.0f;
  }
}

}  // namespace ep

extern "C" int ep_rank_ids(const int64_t* topk_idx, int R, int T_r, int k, int E, int64_t* rank_ids,
                           int32_t* status, void* stream) {
  if (R <= 0 || R > ep::kMaxR || E <= 0 || E > ep::kMaxE || E % R != 0 || k <= 0 ||
      k > ep::kMaxK || T_r < 0)
    return EP_ERR_INVALID_ARG;
  const int64_t T = (int64_t)R * T_r;
  if (T == 0) return EP_OK;
  if (!topk_idx || !rank_ids) return EP_ERR_INVALID_ARG;
  const int64_t blocks = (T + ep::kRankThreads - 1) / ep::kRankThreads;
  ep::k_rank_ids<<<(unsigned)blocks, ep::kRankThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      topk_idx, T, k, E, E / R, rank_ids, status);
  ep_host::count_launch();
  return ep_host::check_launch();
}

extern "C" int ep_rank_recv_topk(const int64_t* topk_idx, const float* topk_weights,
                                 const int32_t* combine_idx, int R, int T_r, int k, int E,
                                 int64_t cap_rows, int64_t* recv_topk_idx, float* recv_topk_weights,
                                 int32_t* status, void* stream) {
  if (R <= 0 || R > ep::kMaxR || E <= 0 || E > ep::kMaxE || E % R != 0 || k <= 0 ||
      k > ep::kMaxK || T_r < 0 || cap_rows < 0)
    return EP_ERR_INVALID_ARG;
  const int64_t T = (int64_t)R * T_r;
  if (T == 0 || cap_rows == 0) return EP_OK;
  if (!topk_idx || !topk_weights || !combine_idx || !recv_topk_idx || !recv_topk_weights)
    return EP_ERR_INVALID_ARG;
  const int64_t blocks = (T * k + ep::kRankThreads - 1) / ep::kRankThreads;
  ep::k_rank_recv_topk<<<(unsigned)blocks, ep::kRankThreads, 0,
                         static_cast<cudaStream_t>(stream)>>>(
      topk_idx, topk_weights, combine_idx, T, k, E, E / R, cap_rows, (int64_t)R * cap_rows,
      recv_topk_idx, recv_topk_weights, status);
  ep_host::count_launch();
  return ep_host::check_launch();
}
