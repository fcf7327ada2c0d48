// dispatch.cu -- token scatter into the receive layouts, with optional fused
// FP8 E4M3 quantisation (llm-infra-atlas DeepEP article §1.1, §1.2, §2.3,
// §3.2, §4.3).
//
// Every emulated rank's receive buffer is a partition of this GPU's HBM, so
// the "put" of a token to expert e's rank is a plain store into that
// partition.  One warp handles one (token, 1024-channel segment) item: it
// reads the segment of x once with 16-byte streaming loads (512 contiguous
// bytes per warp instruction), quantises it once when FP8 is requested
// (amax over each 128-channel block by a 16-lane shuffle reduction), and
// stores it to the k destination rows.  The destinations come from
//   normal mode:       psum[r][l] + expert_prefix[i][e] + slot_rank[i][t][j]
//                      (segment start + source-rank offset + position, the
//                      receiver address of §2.3 with V2's psum, §4.3)
//   low-latency mode:  combine_idx written by the layout kernel just before
//                      (packed row in (rank, token, slot) order, §1.2/§3.2).
// The low-latency scatter is a programmatic dependent launch: it loads its
// first segment of x while the layout kernel is still running and only then
// waits for the layout (griddepcontrol.wait).
//
// FP8 arithmetic is exact IEEE: amax is floored at 1e-4, the scale and its
// inverse use correctly rounded division (__fdiv_rn), x * inv one rounded
// multiply (__fmul_rn), and the E4M3 conversion is CUDA's satfinite RNE
// intrinsic; ue8m0 scales are amax/448 rounded up to a power of two through
// the exponent bits, so x * 2^-p is exact.

#include "ep_common.cuh"
#include "layout.cuh"

namespace ep {

constexpr int kScatterThreads = 256;
constexpr int kScatterU = 4;                          // 16-byte vectors per lane per item
constexpr int kScatterSegC = kScatterU * kWarp * 8;   // 1024 channels per item
constexpr int kPadChunkRows = 1024;

struct ScatterParams {
  const uint8_t* x;
  int R, T_r, H, E, E_l, k;
  int64_t T;
  int nseg;
  const int64_t* topk_idx;
  const int32_t* slot_rank;
  const int32_t* expert_prefix;
  const int64_t* psum;
  int64_t seg_rows;
  int64_t n_rows;          // rows of the whole receive buffer
  uint8_t* recv_x;
  void* recv_scales;
  int32_t* recv_src_idx;
  int32_t* combine_idx;
  int32_t* status;
  int64_t n_items;
  int64_t n_pad_items;
  int tail_chunks;
};

// Quantise 8 channels held by this lane; amax is reduced over the 16 lanes
// that share the 128-channel block.  Returns the 8 E4M3 bytes; the block's
// scale goes to *scale_f32 / *scale_u8.
template <int kMode>
__device__ __forceinline__ uint2 quantize8(const uint4 v, float* scale_f32, uint32_t* scale_u8) {
  float f[8];
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
  float amax = 0.0f;
#pragma unroll
  for (int c = 0; c < 8; ++c) amax = fmaxf(amax, fabsf(f[c]));
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  amax = fmaxf(amax, 1e-4f);
  float mul;
  if (kMode == EP_FP8_E4M3_F32_SCALE) {
    *scale_f32 = __fdiv_rn(amax, 448.0f);
    mul = __fdiv_rn(448.0f, amax);
  } else {
    const uint32_t bits = __float_as_uint(__fdiv_rn(amax, 448.0f));
    uint32_t biased = (bits >> 23) & 0xffu;
    if (bits & 0x7fffffu) biased += 1u;
    *scale_u8 = biased;
    mul = __uint_as_float((254u - biased) << 23);   // 2^(127 - biased), exact
  }
  uint2 q;
  q.x = cvt_e4m3x2(__fmul_rn(f[0], mul), __fmul_rn(f[1], mul)) |
        (cvt_e4m3x2(__fmul_rn(f[2], mul), __fmul_rn(f[3], mul)) << 16);
  q.y = cvt_e4m3x2(__fmul_rn(f[4], mul), __fmul_rn(f[5], mul)) |
        (cvt_e4m3x2(__fmul_rn(f[6], mul), __fmul_rn(f[7], mul)) << 16);
  return q;
}

template <int kMode, bool kLL>
__global__ void __launch_bounds__(kScatterThreads, 4) k_scatter(ScatterParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kScatterThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kScatterThreads) >> 5;
  const int nb = p.H / kFp8Block;
  const int64_t row_bytes = kMode == EP_FP8_NONE ? (int64_t)p.H * 2 : (int64_t)p.H;
  bool waited = false;

  for (int64_t it = warp0; it < p.n_items; it += nwarps) {
    const int64_t g = it / p.nseg;
    const int s = (int)(it - g * p.nseg);
    const int ch0 = s * kScatterSegC;
    const uint8_t* xrow = p.x + g * (int64_t)p.H * 2;

    uint4 v[kScatterU];
#pragma unroll
    for (int u = 0; u < kScatterU; ++u) {
      const int ch = ch0 + u * 256 + lane * 8;
      v[u] = ch < p.H ? ld_stream_v4(xrow + (int64_t)ch * 2) : make_uint4(0, 0, 0, 0);
    }
    if (kLL && !waited) {
      pdl_wait();
      waited = true;
    }

    // destination of slot j = lane (flat row, scale base)
    int64_t my_f = -1, my_sb = 0;
    if (lane < p.k) {
      const int64_t pos = g * p.k + lane;
      if (kLL) {
        my_f = p.combine_idx[pos];
        if (my_f < -1 || my_f >= p.n_rows) {   // never write outside the buffer
          set_status(p.status, EP_ERR_INVALID_ARG);
          my_f = -1;
        }
      } else {
        const int64_t e = p.topk_idx[pos];
        if (e >= 0 && e < p.E) {
          const int r = (int)(e / p.E_l);
          const int l = (int)(e - (int64_t)r * p.E_l);
          const int i = (int)(g / p.T_r);
          const int64_t row = p.psum[(int64_t)r * (p.E_l + 1) + l] +
                              p.expert_prefix[(int64_t)i * p.E + e] + p.slot_rank[pos];
          if (row >= 0 && row < p.seg_rows) my_f = (int64_t)r * p.seg_rows + row;
          else set_status(p.status, EP_ERR_CAPACITY);
        } else if (e != -1) {
          set_status(p.status, EP_ERR_INVALID_ARG);
        }
        if (s == 0) {
          p.combine_idx[pos] = (int32_t)my_f;
          if (my_f >= 0) p.recv_src_idx[my_f] = (int32_t)g;
        }
      }
      if (my_f >= 0 && kMode != EP_FP8_NONE) {
        const int64_t seg = my_f / p.seg_rows;
        my_sb = seg * nb * p.seg_rows + (my_f - seg * p.seg_rows);
      }
    }

    if (kMode == EP_FP8_NONE) {
      for (int j = 0; j < p.k; ++j) {
        const int64_t f = __shfl_sync(0xffffffffu, my_f, j);
        if (f < 0) continue;
        uint8_t* dst = p.recv_x + f * row_bytes;
#pragma unroll
        for (int u = 0; u < kScatterU; ++u) {
          const int ch = ch0 + u * 256 + lane * 8;
          if (ch < p.H) st_v4(dst + (int64_t)ch * 2, v[u]);
        }
      }
    } else {
      uint2 q[kScatterU];
      float sf[kScatterU];
      uint32_t su[kScatterU];
#pragma unroll
      for (int u = 0; u < kScatterU; ++u) q[u] = quantize8<kMode>(v[u], &sf[u], &su[u]);
      for (int j = 0; j < p.k; ++j) {
        const int64_t f = __shfl_sync(0xffffffffu, my_f, j);
        if (f < 0) continue;
        const int64_t sb = __shfl_sync(0xffffffffu, my_sb, j);
        uint8_t* dst = p.recv_x + f * row_bytes;
#pragma unroll
        for (int u = 0; u < kScatterU; ++u) {
          const int ch = ch0 + u * 256 + lane * 8;
          if (ch < p.H) {
            st_v2(dst + ch, q[u]);
            if ((lane & 15) == 0) {
              const int64_t sidx = sb + (int64_t)(ch / kFp8Block) * p.seg_rows;
              if (kMode == EP_FP8_E4M3_F32_SCALE)
                static_cast<float*>(p.recv_scales)[sidx] = sf[u];
              else
                static_cast<uint8_t*>(p.recv_scales)[sidx] = (uint8_t)su[u];
            }
          }
        }
      }
    }
  }

  if (kLL) return;
  // normal mode: recv_src_idx = -1 on alignment padding and past the last row
  const int n_seg_items = p.R * p.E_l;
  for (int64_t it = warp0; it < p.n_pad_items; it += nwarps) {
    int r;
    int64_t lo, hi;
    if (it < n_seg_items) {
      r = (int)(it / p.E_l);
      const int l = (int)(it - (int64_t)r * p.E_l);
      const int e = r * p.E_l + l;
      lo = p.psum[(int64_t)r * (p.E_l + 1) + l] + p.expert_prefix[(int64_t)p.R * p.E + e];
      hi = p.psum[(int64_t)r * (p.E_l + 1) + l + 1];
    } else {
      const int64_t q = it - n_seg_items;
      r = (int)(q / p.tail_chunks);
      const int64_t c = q - (int64_t)r * p.tail_chunks;
      lo = max(p.psum[(int64_t)r * (p.E_l + 1) + p.E_l], c * kPadChunkRows);
      hi = (c + 1) * kPadChunkRows;
    }
    hi = min(hi, p.seg_rows);
    lo = max(lo, (int64_t)0);
    for (int64_t row = lo + lane; row < hi; row += 32) p.recv_src_idx[(int64_t)r * p.seg_rows + row] = -1;
  }
}

template <int kMode, bool kLL>
static int launch_scatter_t(const ScatterParams& p, cudaStream_t stream, bool pdl) {
  const int64_t total = p.n_items + p.n_pad_items;
  const int64_t want = (total + (kScatterThreads / kWarp) - 1) / (kScatterThreads / kWarp);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)ep_host::num_sms() * 4));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kScatterThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, k_scatter<kMode, kLL>, p) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  ep_host::count_launch();
  return ep_host::check_launch();
}

static int launch_scatter(const ScatterParams& p, int fp8_mode, bool ll, cudaStream_t stream) {
  switch (fp8_mode * 2 + (ll ? 1 : 0)) {
    case 0: return launch_scatter_t<EP_FP8_NONE, false>(p, stream, false);
    case 1: return launch_scatter_t<EP_FP8_NONE, true>(p, stream, true);
    case 2: return launch_scatter_t<EP_FP8_E4M3_F32_SCALE, false>(p, stream, false);
    case 3: return launch_scatter_t<EP_FP8_E4M3_F32_SCALE, true>(p, stream, true);
    case 4: return launch_scatter_t<EP_FP8_E4M3_UE8M0, false>(p, stream, false);
    case 5: return launch_scatter_t<EP_FP8_E4M3_UE8M0, true>(p, stream, true);
  }
  return EP_ERR_INVALID_ARG;
}

static int check_common(int R, int T_r, int H, int E, int k, int fp8_mode) {
  if (R <= 0 || R > kMaxR || E <= 0 || E > kMaxE || E % R != 0 || k <= 0 || k > kMaxK ||
      T_r < 0 || H <= 0 || H % 8 != 0)
    return EP_ERR_INVALID_ARG;
  if (fp8_mode < EP_FP8_NONE || fp8_mode > EP_FP8_E4M3_UE8M0) return EP_ERR_INVALID_ARG;
  if (fp8_mode != EP_FP8_NONE && H % kFp8Block != 0) return EP_ERR_INVALID_ARG;
  return EP_OK;
}

}  // namespace ep

extern "C" int ep_dispatch(const void* x, const int64_t* topk_idx, const int32_t* slot_rank,
                           const int32_t* expert_prefix, const int64_t* psum, int R, int T_r,
                           int H, int E, int k, int fp8_mode, int64_t cap_rows, void* recv_x,
                           void* recv_scales, int32_t* recv_src_idx, int32_t* combine_idx,
                           int32_t* status, void* stream) {
  int rc = ep::check_common(R, T_r, H, E, k, fp8_mode);
  if (rc != EP_OK) return rc;
  if (cap_rows < 0 || (int64_t)R * cap_rows > INT32_MAX) return EP_ERR_INVALID_ARG;
  if (!expert_prefix || !psum || !recv_src_idx ||
      (T_r > 0 && (!x || !topk_idx || !slot_rank || !combine_idx)) ||
      (cap_rows > 0 && !recv_x) || (fp8_mode != EP_FP8_NONE && cap_rows > 0 && !recv_scales))
    return EP_ERR_INVALID_ARG;
  if (!ep_host::aligned16(x) || !ep_host::aligned16(recv_x)) return EP_ERR_INVALID_ARG;
  ep::ScatterParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.R = R;
  p.T_r = T_r;
  p.H = H;
  p.E = E;
  p.E_l = E / R;
  p.k = k;
  p.T = (int64_t)R * T_r;
  p.nseg = (H + ep::kScatterSegC - 1) / ep::kScatterSegC;
  p.topk_idx = topk_idx;
  p.slot_rank = slot_rank;
  p.expert_prefix = expert_prefix;
  p.psum = psum;
  p.seg_rows = cap_rows;
  p.n_rows = (int64_t)R * cap_rows;
  p.recv_x = static_cast<uint8_t*>(recv_x);
  p.recv_scales = recv_scales;
  p.recv_src_idx = recv_src_idx;
  p.combine_idx = combine_idx;
  p.status = status;
  p.n_items = p.T * p.nseg;
  p.tail_chunks = (int)((cap_rows + ep::kPadChunkRows - 1) / ep::kPadChunkRows);
  p.n_pad_items = (int64_t)R * p.E_l + (int64_t)R * p.tail_chunks;
  return ep::launch_scatter(p, fp8_mode, false, static_cast<cudaStream_t>(stream));
}

extern "C" int ep_ll_dispatch(const void* x, const int64_t* topk_idx, int R, int T_r, int H, int E,
                              int k, int max_tokens_per_rank, int fp8_mode, void* packed_recv_x,
                              void* packed_recv_scales, int32_t* packed_recv_src_info,
                              int64_t* layout_range, int32_t* recv_count, int32_t* combine_idx,
                              void* workspace, size_t workspace_bytes, int32_t* status,
                              void* stream) {
  int rc = ep::check_common(R, T_r, H, E, k, fp8_mode);
  if (rc != EP_OK) return rc;
  if (max_tokens_per_rank <= 0 || T_r > max_tokens_per_rank) return EP_ERR_INVALID_ARG;
  const int64_t seg_rows = (int64_t)R * max_tokens_per_rank;
  if ((int64_t)E * seg_rows > INT32_MAX) return EP_ERR_INVALID_ARG;
  if (!packed_recv_x || !packed_recv_src_info || !layout_range || !recv_count || !workspace ||
      (T_r > 0 && (!x || !topk_idx || !combine_idx)) ||
      (fp8_mode != EP_FP8_NONE && !packed_recv_scales))
    return EP_ERR_INVALID_ARG;
  if (!ep_host::aligned16(x) || !ep_host::aligned16(packed_recv_x)) return EP_ERR_INVALID_ARG;
  if (workspace_bytes < ep_workspace_size(R, T_r, k, E)) return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  ep::LayoutParams lp{};
  lp.topk_idx = topk_idx;
  lp.R = R;
  lp.T_r = T_r;
  lp.k = k;
  lp.E = E;
  lp.E_l = E / R;
  lp.combine_idx = combine_idx;
  lp.src_info = packed_recv_src_info;
  lp.recv_count = recv_count;
  lp.layout_range = layout_range;
  lp.seg_rows = seg_rows;
  lp.status = status;
  rc = ep::launch_layout(lp, true, workspace, s);
  if (rc != EP_OK) return rc;

  ep::ScatterParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.R = R;
  p.T_r = T_r;
  p.H = H;
  p.E = E;
  p.E_l = E / R;
  p.k = k;
  p.T = (int64_t)R * T_r;
  p.nseg = (H + ep::kScatterSegC - 1) / ep::kScatterSegC;
  p.seg_rows = seg_rows;
  p.n_rows = (int64_t)E * seg_rows;
  p.recv_x = static_cast<uint8_t*>(packed_recv_x);
  p.recv_scales = packed_recv_scales;
  p.combine_idx = combine_idx;
  p.status = status;
  p.n_items = p.T * p.nseg;
  p.n_pad_items = 0;
  if (p.n_items == 0) return EP_OK;
  return ep::launch_scatter(p, fp8_mode, true, s);
}
