// dispatch.cuh -- shared by the two dispatch translation units: the
// normal-mode / multi-kernel scatter (dispatch.cu) and the single-launch
// low-latency kernel (ll_fused.cu).
#pragma once

#include "ep_common.cuh"
#include "layout.cuh"

namespace ep {

constexpr int kScatterMaxWarps = 16;
constexpr int kBf16Warps = 16;     // target warps per CTA, bf16 path (1792-channel pieces at H = 7168)
constexpr int kFp8Warps = 16;      // target warps per CTA, FP8 path
constexpr int kBf16Stages = 3;     // staged source pieces per warp (bf16 path)
constexpr int kFp8InStages = 2;    // staged source pieces per warp (FP8 path)
constexpr int kFp8OutStages = 2;   // staged E4M3 pieces per warp
constexpr size_t kScatterSmemBudget = 200 * 1024;
// Workspace control words (uint32 at the start of the workspace): 0-3 the
// layout kernel's ticket / done / epoch / abort, 8-9 the single-launch
// low-latency kernel's grid barrier, 10-11 the scatter's unit claims.
constexpr int kCtlClaim = 10;
constexpr int kPadChunkRows = 1024;
constexpr int kScaleColThreads = 256;

struct ScatterParams {
  const uint8_t* x;
  int R, T_r, H, E, E_l, k;
  int64_t T;
  const int64_t* topk_idx;
  const int32_t* slot_rank;
  const int32_t* expert_prefix;
  const int64_t* psum;
  int64_t seg_rows;        // rows per segment (cap_rows, or R*max per expert)
  int64_t n_rows;          // rows of the whole receive buffer
  uint8_t* recv_x;
  int32_t* recv_src_idx;
  int32_t* combine_idx;
  uint8_t* scale_rows;     // [T][scale_row_bytes] per-token scales (FP8)
  int scale_row_bytes;
  int32_t* status;
  // pipeline geometry
  int Hp;                  // channels per row piece
  int P;                   // pieces per row
  int warps_per_cta;
  uint32_t warp_smem;      // bytes of shared memory per warp
  uint32_t in_bytes, out_bytes;   // per-stage sizes (128-byte multiples)
  int64_t n_units;         // T * P
  int64_t n_pad_items;
  int tail_chunks;
  uint32_t* claim;         // [2] workspace words: unit claim counter, CTAs done; null: static split
};

__host__ __device__ inline uint32_t round128(uint32_t v) { return (v + 127u) / 128u * 128u; }

// Bytes of one token's staged scales (16-byte rows).
__host__ __device__ inline int scale_row_bytes(int H, int elem) {
  return ((H / kFp8Block) * elem + 15) / 16 * 16;
}

constexpr float kFloatMax = 3.40282346638528859812e+38f;   // largest finite float

// Quantise 16 channels (two 16-byte bf16 vectors) of this lane; amax is
// reduced over the 8 lanes sharing the 128-channel block (NaN entries do not
// raise it), floored at 1e-4 and capped at the largest finite float, so a
// block holding an infinity still gets a finite scale and the infinity
// saturates to +-448.  Returns 16 E4M3
// bytes; the block's scale goes to *sf (fp32 mode) or *su (ue8m0 mode).
template <int kMode>
__device__ __forceinline__ uint4 quantize16(const uint4 a, const uint4 b, float* sf, uint32_t* su) {
  float f[16];
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    f[2 * c] = bf16_lo(w[c]);
    f[2 * c + 1] = bf16_hi(w[c]);
  }
  float amax = 0.0f;
#pragma unroll
  for (int c = 0; c < 16; ++c) amax = fmaxf(amax, fabsf(f[c]));
#pragma unroll
  for (int off = 4; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  amax = fminf(fmaxf(amax, 1e-4f), kFloatMax);   // floor; an infinity saturates
  float mul;
  if (kMode == EP_FP8_E4M3_F32_SCALE) {
    *sf = __fdiv_rn(amax, 448.0f);
    mul = __fdiv_rn(448.0f, amax);
  } else {
    const uint32_t bits = __float_as_uint(__fdiv_rn(amax, 448.0f));
    uint32_t biased = (bits >> 23) & 0xffu;
    if (bits & 0x7fffffu) biased += 1u;
    *su = biased;
    mul = __uint_as_float((254u - biased) << 23);   // 2^(127 - biased), exact
  }
  uint32_t q[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    q[c] = cvt_e4m3x2(__fmul_rn(f[4 * c], mul), __fmul_rn(f[4 * c + 1], mul)) |
           (cvt_e4m3x2(__fmul_rn(f[4 * c + 2], mul), __fmul_rn(f[4 * c + 3], mul)) << 16);
  }
  return make_uint4(q[0], q[1], q[2], q[3]);
}

// ------------------------------------------------------------------ scale columns

struct ScaleColParams {
  const uint8_t* scale_rows;   // [T][row_bytes] per-token scales
  int row_bytes, nb;
  int64_t T;
  int64_t seg_rows;
  int64_t n_rows;              // rows of the receive buffer (segments * seg_rows)
  int64_t max_items;           // normal mode: bound on the flat loop's items (valid rows,
                               // or 4-row quads), which sizes the grid
  const int32_t* src_idx;      // token of every receive row, -1 = none (normal mode)
  const int32_t* recv_count;   // low-latency mode: rows per expert segment (src_idx
                               // is only defined below it)
  const int64_t* psum;         // normal mode: [R][E_l + 1] segment starts
  const int32_t* expert_total; // normal mode: [E] rows of every expert (unaligned)
  int E, E_l;
  bool quad;                   // ue8m0 with seg_rows % 4 == 0 and out 4-byte aligned: a
                               // thread writes 4 consecutive rows (one word per block)
  bool tables_after_wait;      // normal mode: the segment tables may still be in the making
                               // when this kernel starts (the scatter itself was a dependent
                               // launch of layout + notify): read them after the wait
  void* out;                   // column-major scales [segment][block][row]
};

// Host launchers and helpers defined in dispatch.cu.
int launch_scatter(const ScatterParams& p, int fp8_mode, bool ll, cudaStream_t stream,
                   bool pdl_normal = false);
int launch_scale_columns(const ScaleColParams& p, bool ll, int fp8_mode, cudaStream_t s);
int check_common(int R, int T_r, int H, int E, int k, int fp8_mode);
size_t staging_bytes(int R, int T_r, int H);
uint8_t* scale_staging(void* ws, int R, int T_r, int k, int E);

}  // namespace ep
