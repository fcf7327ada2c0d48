// formats.cu -- the two number-format conversions of the path, as the
// kernels perform them, applied elementwise: fp32 -> E4M3 (round to nearest
// even, saturating to +-448; the FP8 dispatch, llm-infra-atlas DeepEP
// article §1.1, §1.2) and fp32 -> bf16 (round to nearest even; the combine's
// output).  They use the same device helpers as the dispatch and combine
// kernels, so a test can hold them against an independent encoder on every
// input that matters.

#include "ep_common.cuh"

namespace ep {

constexpr int kFmtThreads = 256;

__global__ void __launch_bounds__(kFmtThreads) k_format_e4m3(const float2* __restrict__ in,
                                                             uint16_t* __restrict__ out, int64_t pairs) {
  for (int64_t i = (int64_t)blockIdx.x * kFmtThreads + threadIdx.x; i < pairs;
       i += (int64_t)gridDim.x * kFmtThreads) {
    const float2 v = in[i];
    out[i] = (uint16_t)cvt_e4m3x2(v.x, v.y);
  }
}

__global__ void __launch_bounds__(kFmtThreads) k_format_bf16(const float2* __restrict__ in,
                                                             uint32_t* __restrict__ out, int64_t pairs) {
  for (int64_t i = (int64_t)blockIdx.x * kFmtThreads + threadIdx.x; i < pairs;
       i += (int64_t)gridDim.x * kFmtThreads) {
    const float2 v = in[i];
    out[i] = pack_bf16x2(v.x, v.y);
  }
}

template <class K, class O>
static int launch_format(K kernel, const float* in, O* out, int64_t n, void* stream) {
  if (n < 0 || (n & 1)) return EP_ERR_INVALID_ARG;
  if (n == 0) return EP_OK;
  if (!in || !out || (reinterpret_cast<uintptr_t>(in) & 7) || (reinterpret_cast<uintptr_t>(out) & 3))
    return EP_ERR_INVALID_ARG;
  const int64_t pairs = n / 2;
  const int64_t want = (pairs + kFmtThreads - 1) / kFmtThreads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)ep_host::num_sms() * 8));
  kernel<<<grid, kFmtThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const float2*>(in), out, pairs);
  ep_host::count_launch();
  return ep_host::check_launch();
}

}  // namespace ep

extern "C" int ep_format_e4m3(const float* in, uint8_t* out, int64_t n, void* stream) {
  return ep::launch_format(ep::k_format_e4m3, in, reinterpret_cast<uint16_t*>(out), n, stream);
}

extern "C" int ep_format_bf16(const float* in, uint16_t* out, int64_t n, void* stream) {
  return ep::launch_format(ep::k_format_bf16, in, reinterpret_cast<uint32_t*>(out), n, stream);
}
