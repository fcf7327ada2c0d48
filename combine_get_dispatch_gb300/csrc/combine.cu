// combine.cu -- top-k weighted combine back to token order (llm-infra-atlas
// DeepEP article §1.1 "FP8 dispatch, BF16 combine", §2.3 / §4.3: combine
// walks the dispatch handle backwards).
//
//   out[t][:] = bf16_rn( fp32 fma chain over j = 0..k-1 of w[t][j] * y[f_j][:] )
//
// with f_j = combine_idx[t][j] (flat receive row; -1 = skip), accumulated
// from +0 in slot order with __fmaf_rn and rounded once with
// __floats2bfloat162_rn.  The same kernel serves the contiguous layout
// (rows of [R, cap_rows]) and the packed layout (rows of [E, R*max]).
//
// Launched with programmatic dependent launch: it waits (griddepcontrol)
// for the kernel before it -- the dispatch that wrote combine_idx -- to
// complete.  The library's kernels before it do not trigger it early: its
// CTAs would then be placed on whichever SMs free up first, several to an
// SM, and the static split of the items over them would run unevenly.
//
// One warp handles one (token, 512-channel segment) item: every lane issues
// all k row loads of its 2 x 16 bytes before the first fma (k*2 independent
// 16-byte streaming loads in flight per lane), then reduces in registers and
// stores 2 x 16 bytes of bf16.  The row loads carry an L2 evict-first hint
// (each row is read once, and the dispatch's rows still dirty in L2 are then
// not the lines evicted) unless the combine reads many times the L2
// (kNoHintL2Multiple): decode combine 49.1-49.4 us with the hint against
// 52.3-52.9 without, skewed 81.4-81.7 against 85.1-86.0, but the large
// combine (15 GB of rows) 2.462-2.466 ms with it against 2.408-2.435 without.  Rows are read whole
// and in order, so every warp load instruction moves 512 contiguous bytes.

#include "ep_common.cuh"

namespace ep {

constexpr int kCombineThreads = 256;   // two CTAs per SM; one CTA of twice that
                                       // per SM under an SM budget

struct CombineParams {
  const uint8_t* y;
  const float* w;
  const int32_t* cidx;
  int64_t n_rows;
  int64_t T;
  int H, k, nseg;
  uint8_t* out;
  int32_t* status;
};

constexpr int64_t kNoHintL2Multiple = 32;   // rows read beyond this many L2 sizes: no hint

template <int kU, int kK, bool kHint>
__global__ void __launch_bounds__(2 * kCombineThreads, 1) k_combine(CombineParams p) {
  constexpr int kSegC = kU * kWarp * 8;
  // launched as a programmatic dependent: the CTAs may be resident before
  // the kernel that wrote combine_idx (the dispatch) has finished
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const uint64_t pol = l2_policy_evict_first();   // every expert-output row is read once
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t row_bytes = (int64_t)p.H * 2;

  for (int64_t it = warp0; it < (int64_t)p.T * p.nseg; it += nwarps) {
    const int64_t g = it / p.nseg;
    const int s = (int)(it - g * p.nseg);
    const int ch0 = s * kSegC;

    int32_t my_f = -1;
    float my_w = 0.0f;
    if (lane < p.k) {
      my_f = p.cidx[g * p.k + lane];
      my_w = p.w != nullptr ? p.w[g * p.k + lane] : 1.0f;   // no weights: a plain sum
      if (my_f < -1 || (int64_t)my_f >= p.n_rows) {
        if (s == 0) set_status(p.status, EP_ERR_INVALID_ARG);
        my_f = -1;
      }
    }
    int32_t f[kK];
    float wt[kK];
#pragma unroll
    for (int j = 0; j < kK; ++j) {
      f[j] = __shfl_sync(0xffffffffu, my_f, j);
      wt[j] = __shfl_sync(0xffffffffu, my_w, j);
    }

    uint4 v[kU][kK];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int ch = ch0 + u * 256 + lane * 8;
#pragma unroll
      for (int j = 0; j < kK; ++j) {
        if (j < p.k && f[j] >= 0 && ch < p.H)
          v[u][j] = kHint ? ld_stream_v4(p.y + (int64_t)f[j] * row_bytes + (int64_t)ch * 2, pol)
                          : __ldg(reinterpret_cast<const uint4*>(p.y + (int64_t)f[j] * row_bytes + (int64_t)ch * 2));
        else
          v[u][j] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int ch = ch0 + u * 256 + lane * 8;
      float acc[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
      for (int j = 0; j < kK; ++j) {
        if (j < p.k && f[j] >= 0) {
          const uint4 a = v[u][j];
          acc[0] = __fmaf_rn(wt[j], bf16_lo(a.x), acc[0]);
          acc[1] = __fmaf_rn(wt[j], bf16_hi(a.x), acc[1]);
          acc[2] = __fmaf_rn(wt[j], bf16_lo(a.y), acc[2]);
          acc[3] = __fmaf_rn(wt[j], bf16_hi(a.y), acc[3]);
          acc[4] = __fmaf_rn(wt[j], bf16_lo(a.z), acc[4]);
          acc[5] = __fmaf_rn(wt[j], bf16_hi(a.z), acc[5]);
          acc[6] = __fmaf_rn(wt[j], bf16_lo(a.w), acc[6]);
          acc[7] = __fmaf_rn(wt[j], bf16_hi(a.w), acc[7]);
        }
      }
      if (ch < p.H) {
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        st_v4(p.out + g * row_bytes + (int64_t)ch * 2, o);
      }
    }
  }
}

template <int kU, int kK, bool kHint>
static int launch_combine_t(const CombineParams& p, cudaStream_t stream) {
  constexpr int kSegC = kU * kWarp * 8;
  CombineParams q = p;
  q.nseg = (p.H + kSegC - 1) / kSegC;
  const int64_t items = q.T * q.nseg;
  if (items == 0) return EP_OK;
  // two CTAs per SM; under an SM budget one CTA of twice the threads on
  // each budgeted SM (the same warps per SM, on fewer SMs)
  const int threads = ep_host::sm_budget_set() ? 2 * kCombineThreads : kCombineThreads;
  const int64_t want = (items + (threads / kWarp) - 1) / (threads / kWarp);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)ep_host::grid_cap(2)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k_combine<kU, kK, kHint>, q) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  ep_host::count_launch();
  return ep_host::check_launch();
}

static int launch_combine(const CombineParams& p, cudaStream_t stream) {
  // rows read at most: every slot of every token, H bf16 channels each
  const bool hint = p.T * p.k * (int64_t)p.H * 2 <= kNoHintL2Multiple * ep_host::l2_bytes();
  if (p.k <= 8)
    return hint ? launch_combine_t<2, 8, true>(p, stream) : launch_combine_t<2, 8, false>(p, stream);
  return hint ? launch_combine_t<1, 16, true>(p, stream) : launch_combine_t<1, 16, false>(p, stream);
}

static int check_combine(const void* y, const float* w, const int32_t* cidx, int R, int T_r, int H,
                         int k, const void* out) {
  if (R <= 0 || R > kMaxR || T_r < 0 || H <= 0 || H % 8 != 0 || k <= 0 || k > kMaxK)
    return EP_ERR_INVALID_ARG;
  if (T_r > 0 && (!y || !w || !cidx || !out)) return EP_ERR_INVALID_ARG;
  if (!ep_host::aligned16(y) || !ep_host::aligned16(out)) return EP_ERR_INVALID_ARG;
  return EP_OK;
}

}  // namespace ep

extern "C" int ep_combine(const void* y, const float* topk_weights, const int32_t* combine_idx,
                          int R, int T_r, int H, int k, int64_t cap_rows, void* out,
                          int32_t* status, void* stream) {
  int rc = ep::check_combine(y, topk_weights, combine_idx, R, T_r, H, k, out);
  if (rc != EP_OK) return rc;
  if (cap_rows < 0) return EP_ERR_INVALID_ARG;
  ep::CombineParams p{};
  p.y = static_cast<const uint8_t*>(y);
  p.w = topk_weights;
  p.cidx = combine_idx;
  p.n_rows = (int64_t)R * cap_rows;
  p.T = (int64_t)R * T_r;
  p.H = H;
  p.k = k;
  void* out_dev = nullptr;   // device memory, or pinned host memory written across the link
  if (ep_host::device_view(out, &out_dev) != EP_OK) return EP_ERR_INVALID_ARG;
  p.out = static_cast<uint8_t*>(out_dev);
  p.status = status;
  return ep::launch_combine(p, static_cast<cudaStream_t>(stream));
}

extern "C" int ep_ll_combine(const void* y, const float* topk_weights, const int32_t* combine_idx,
                             int R, int T_r, int H, int E, int k, int max_tokens_per_rank,
                             void* out, int32_t* status, void* stream) {
  int rc = ep::check_combine(y, topk_weights, combine_idx, R, T_r, H, k, out);
  if (rc != EP_OK) return rc;
  if (E <= 0 || E % R != 0 || max_tokens_per_rank <= 0) return EP_ERR_INVALID_ARG;
  ep::CombineParams p{};
  p.y = static_cast<const uint8_t*>(y);
  p.w = topk_weights;
  p.cidx = combine_idx;
  p.n_rows = (int64_t)E * R * max_tokens_per_rank;
  p.T = (int64_t)R * T_r;
  p.H = H;
  p.k = k;
  void* out_dev = nullptr;   // device memory, or pinned host memory written across the link
  if (ep_host::device_view(out, &out_dev) != EP_OK) return EP_ERR_INVALID_ARG;
  p.out = static_cast<uint8_t*>(out_dev);
  p.status = status;
  return ep::launch_combine(p, static_cast<cudaStream_t>(stream));
}

extern "C" int ep_rank_combine(const void* y, const int32_t* combine_idx, int R, int T_r, int H,
                               int k, int64_t cap_rows, void* out, int32_t* status, void* stream) {
  // the rows are summed as they are: weight 1 (fma(1, y, acc) is acc + y, rounded once)
  if (R <= 0 || R > ep::kMaxR || T_r < 0 || H <= 0 || H % 8 != 0 || k <= 0 || k > ep::kMaxK ||
      cap_rows < 0)
    return EP_ERR_INVALID_ARG;
  if (T_r > 0 && (!y || !combine_idx || !out)) return EP_ERR_INVALID_ARG;
  if (!ep_host::aligned16(y) || !ep_host::aligned16(out)) return EP_ERR_INVALID_ARG;
  ep::CombineParams p{};
  p.y = static_cast<const uint8_t*>(y);
  p.w = nullptr;
  p.cidx = combine_idx;
  p.n_rows = (int64_t)R * cap_rows;
  p.T = (int64_t)R * T_r;
  p.H = H;
  p.k = k;
  void* out_dev = nullptr;   // device memory, or pinned host memory written across the link
  if (ep_host::device_view(out, &out_dev) != EP_OK) return EP_ERR_INVALID_ARG;
  p.out = static_cast<uint8_t*>(out_dev);
  p.status = status;
  return ep::launch_combine(p, static_cast<cudaStream_t>(stream));
}
