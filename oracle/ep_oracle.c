/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for MoE token
 * dispatch / combine (DeepEP-style), used ONLY as test infrastructure.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * reference leg may load this library.  The product path (the CUDA library
 * under combine_get_dispatch_gb300/csrc) shares no code, header, table or
 * constant with this file.
 *
 * Source of the definitions (cited as [06_deepep §n]): the llm-infra-atlas
 * article on DeepEP at llm-infra-atlas.github.io/moe/06_deepep/ --
 *   §1.1 normal mode (contiguous layout, FP8 dispatch with BF16 combine),
 *   §1.2 low-latency mode (packed masked layout, recv_count = masked_m,
 *        FP8 options round_scale / use_ue8m0, column-major scales),
 *   §2.1 notify_dispatch (count all-to-all, prefix over source ranks,
 *        per-local-expert receive totals aligned to expert_alignment,
 *        num_worst_tokens),
 *   §2.3 prefix matrix (rank_prefix_matrix[i][j] = tokens for rank j from
 *        ranks <= i; receiver offset = rank offset + finer offset),
 *   §3.2 low-latency routing (dst_rank = expert / num_local_experts),
 *   §4.3 EPHandle (psum_num_recv_tokens_per_expert = aligned prefix sum =
 *        segment start of each expert in the receive buffer; combine is
 *        dispatch walked backwards);
 *   V1's once-per-rank receive layout (§2.1, §2.3): a token goes once to
 *        every rank holding one of its experts, at rank_prefix_matrix[i-1][r]
 *        plus its position among source rank i's tokens for r, and the
 *        combine sums the rows the ranks return.
 * Number formats: OCP 8-bit floating point specification (E4M3: bias 7,
 * max 448, no infinities, NaN = S.1111.111) and the bfloat16 format (top 16
 * bits of IEEE-754 binary32), both rounded to nearest, ties to even.
 *
 * Readings where the article is silent (each also listed in the design
 * notes): rows of a segment are ordered by (source rank, token, slot);
 * topk id -1 means "no expert"; FP8 blocks are 128 channels; amax is floored
 * at 1e-4 and capped at the largest finite float (an infinity in x gives a
 * finite scale; the infinity itself saturates to +-448); fp32 mode stores scale = amax/448 and quantises x * (448/amax);
 * ue8m0 mode rounds amax/448 up to a power of two and stores its biased
 * exponent byte; combine accumulates w*y in fp32 with fma in slot order and
 * rounds once to bf16.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math, no
 * contraction: every float operation below is one IEEE-754 rounding).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes returned by the oracle (same numeric meaning as the
 * library's, written out here on purpose rather than shared). */
#define ORACLE_OK 0
#define ORACLE_ERR_INVALID_ARG 1
#define ORACLE_ERR_CAPACITY 2

#define FP8_NONE 0
#define FP8_E4M3_F32_SCALE 1
#define FP8_E4M3_UE8M0 2

#define BLOCK_CHANNELS 128

/* ------------------------------------------------------------------ */
/* Number formats                                                       */
/* ------------------------------------------------------------------ */

/* bfloat16 -> float: the 16 bits are the top half of a binary32. */
float ep_oracle_bf16_to_f32(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* float -> bfloat16, round to nearest even: keep the top 16 bits and round
 * on the 16 discarded bits (above half: up; exactly half: to even).  A carry
 * runs into the exponent, so the largest finite values round to infinity as
 * RNE requires.  NaN maps to the quiet NaN 0x7FFF. */
uint16_t ep_oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fff;
  uint32_t hi = u >> 16;
  uint32_t lo = u & 0xffffu;
  if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
  return (uint16_t)hi;
}

/* E4M3 byte -> float (OCP FP8): normal values 2^(E-7) * (1 + M/8),
 * subnormals 2^-6 * (M/8), S.1111.111 is NaN. */
float ep_oracle_e4m3_to_f32(uint8_t b) {
  int s = b >> 7;
  int E = (b >> 3) & 15;
  int M = b & 7;
  if (E == 15 && M == 7) return NAN;
  double v = (E == 0) ? ldexp((double)M, -9) : ldexp((double)(8 + M), E - 10);
  return (float)(s ? -v : v);
}

/* float -> E4M3, round to nearest even, saturating to +-448 (finite
 * saturation: anything above the largest normal, infinity included, becomes
 * 448; NaN stays NaN).  The value is snapped to the E4M3 grid in exact
 * double arithmetic: step 2^-9 below 2^-6 (subnormals), 2^(e-3) in the
 * binade [2^e, 2^(e+1)).  nearbyint() rounds ties to even in the default
 * rounding mode. */
uint8_t ep_oracle_f32_to_e4m3(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint8_t sign = (u >> 31) ? 0x80 : 0x00;
  if (isnan(f)) return (uint8_t)(sign | 0x7f);
  double a = fabs((double)f);
  if (a >= 448.0) return (uint8_t)(sign | 0x7e);
  const double min_normal = ldexp(1.0, -6);
  double step = (a < min_normal) ? ldexp(1.0, -9) : ldexp(1.0, ilogb(a) - 3);
  double q = nearbyint(a / step) * step;
  if (q > 448.0) q = 448.0;
  if (q < min_normal) {
    int m = (int)(q / ldexp(1.0, -9));
    return (uint8_t)(sign | m);
  }
  int e = ilogb(q);
  int m = (int)(q / ldexp(1.0, e - 3)) - 8;
  return (uint8_t)(sign | ((e + 7) << 3) | m);
}

void ep_oracle_f32_to_e4m3_batch(const float* in, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_f32_to_e4m3(in[i]);
}

void ep_oracle_f32_to_bf16_batch(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_f32_to_bf16(in[i]);
}

void ep_oracle_e4m3_to_f32_batch(const uint8_t* in, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ep_oracle_e4m3_to_f32(in[i]);
}

/* ------------------------------------------------------------------ */
/* FP8 quantisation of one row ([06_deepep §1.1, §1.2]; block size 128)  */
/* ------------------------------------------------------------------ */

/* Quantise one bf16 row of H channels (H % 128 == 0) block by block.
 *   amax  = min(max(max |x| over the block, 1e-4), FLT_MAX)
 *           (NaN entries do not raise amax; an infinity saturates it to the
 *           largest finite float, so every scale stays finite)
 *   mode 1 (fp32 scale): scale = amax / 448, q = E4M3(x * (448 / amax))
 *   mode 2 (ue8m0):      s = amax / 448 rounded UP to a power of two 2^p
 *                        (biased exponent + 1 when any mantissa bit is set),
 *                        byte = biased exponent of 2^p, q = E4M3(x * 2^-p)
 * Scales go to scale_f32[b * scale_stride] or scale_ue8m0[b * scale_stride]
 * (column-major: consecutive rows of the same block are adjacent). */
void ep_oracle_quantize_row(const uint16_t* x, int H, int mode, uint8_t* q,
                            float* scale_f32, uint8_t* scale_ue8m0,
                            int64_t scale_stride) {
  int nb = H / BLOCK_CHANNELS;
  for (int b = 0; b < nb; ++b) {
    const uint16_t* xb = x + (int64_t)b * BLOCK_CHANNELS;
    uint8_t* qb = q + (int64_t)b * BLOCK_CHANNELS;
    float amax = 0.0f;
    for (int c = 0; c < BLOCK_CHANNELS; ++c) {
      float a = fabsf(ep_oracle_bf16_to_f32(xb[c]));
      if (a > amax) amax = a;
    }
    if (amax < 1e-4f) amax = 1e-4f;
    if (amax > FLT_MAX) amax = FLT_MAX;   /* an infinity in the block saturates */
    if (mode == FP8_E4M3_F32_SCALE) {
      float scale = amax / 448.0f;
      float inv = 448.0f / amax;
      for (int c = 0; c < BLOCK_CHANNELS; ++c) {
        float v = ep_oracle_bf16_to_f32(xb[c]) * inv;
        qb[c] = ep_oracle_f32_to_e4m3(v);
      }
      scale_f32[(int64_t)b * scale_stride] = scale;
    } else {
      float s = amax / 448.0f;
      uint32_t bits;
      memcpy(&bits, &s, 4);
      uint32_t biased = (bits >> 23) & 0xffu;
      if (bits & 0x7fffffu) biased += 1u;
      float mult = ldexpf(1.0f, 127 - (int)biased);
      for (int c = 0; c < BLOCK_CHANNELS; ++c) {
        float v = ep_oracle_bf16_to_f32(xb[c]) * mult;
        qb[c] = ep_oracle_f32_to_e4m3(v);
      }
      scale_ue8m0[(int64_t)b * scale_stride] = (uint8_t)biased;
    }
  }
}

/* ------------------------------------------------------------------ */
/* get_dispatch_layout ([06_deepep §2.1, §2.3]; handle fields §2.3)      */
/* ------------------------------------------------------------------ */

/* Per source rank i, from topk_idx [R, T_r, k] (expert ids, -1 = none):
 *   num_tokens_per_expert[i][e] = #{(t, j) : idx[i][t][j] == e}
 *   is_token_in_rank[i][t][r]   = 1 iff some j has idx[i][t][j] / E_l == r
 *   num_tokens_per_rank[i][r]   = sum_t is_token_in_rank[i][t][r]
 *   slot_rank[i][t][j]          = #{(t', j') before (t, j) in (token, slot)
 *                                   order within rank i with the same expert}
 *                                 (-1 for a masked slot)
 * Returns ORACLE_ERR_INVALID_ARG for an id outside [-1, E). */
int ep_oracle_layout(const int64_t* topk_idx, int R, int T_r, int k, int E,
                     int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                     uint8_t* is_token_in_rank, int32_t* slot_rank) {
  if (R <= 0 || E <= 0 || E % R != 0 || T_r < 0 || k <= 0) return ORACLE_ERR_INVALID_ARG;
  int E_l = E / R;
  memset(num_tokens_per_rank, 0, sizeof(int32_t) * (size_t)R * R);
  memset(num_tokens_per_expert, 0, sizeof(int32_t) * (size_t)R * E);
  memset(is_token_in_rank, 0, (size_t)R * T_r * R);
  for (int i = 0; i < R; ++i) {
    for (int t = 0; t < T_r; ++t) {
      for (int j = 0; j < k; ++j) {
        int64_t p = ((int64_t)i * T_r + t) * k + j;
        int64_t e = topk_idx[p];
        if (e == -1) {
          slot_rank[p] = -1;
          continue;
        }
        if (e < -1 || e >= E) return ORACLE_ERR_INVALID_ARG;
        slot_rank[p] = num_tokens_per_expert[(int64_t)i * E + e];
        num_tokens_per_expert[(int64_t)i * E + e] += 1;
        is_token_in_rank[((int64_t)i * T_r + t) * R + e / E_l] = 1;
      }
    }
    for (int t = 0; t < T_r; ++t)
      for (int r = 0; r < R; ++r)
        num_tokens_per_rank[(int64_t)i * R + r] += is_token_in_rank[((int64_t)i * T_r + t) * R + r];
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* notify_dispatch ([06_deepep §2.1, §2.3, §4.3])                        */
/* ------------------------------------------------------------------ */

/* From the per-rank counts of every rank:
 *   rank_prefix_matrix[i][j]        = sum_{i' <= i} num_tokens_per_rank[i'][j]
 *   expert_prefix[i][e] (i < R)     = sum_{i' < i} num_tokens_per_expert[i'][e]
 *   expert_prefix[R][e]             = sum_{i'} num_tokens_per_expert[i'][e]
 *   num_recv_tokens_per_expert[r][l]= align_up(expert_prefix[R][r*E_l + l], A)
 *   psum[r][0] = 0, psum[r][l+1]    = psum[r][l] + num_recv_tokens_per_expert[r][l]
 * With num_worst_tokens >= 0, a rank that receives more tokens than that
 * (last row of rank_prefix_matrix) is ORACLE_ERR_CAPACITY. */
int ep_oracle_notify(const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_expert,
                     int R, int E, int expert_alignment, int64_t num_worst_tokens,
                     int32_t* rank_prefix_matrix, int32_t* expert_prefix,
                     int32_t* num_recv_tokens_per_expert, int64_t* psum) {
  if (R <= 0 || E <= 0 || E % R != 0 || expert_alignment <= 0) return ORACLE_ERR_INVALID_ARG;
  int E_l = E / R;
  int rc = ORACLE_OK;
  for (int j = 0; j < R; ++j) {
    int32_t run = 0;
    for (int i = 0; i < R; ++i) {
      run += num_tokens_per_rank[(int64_t)i * R + j];
      rank_prefix_matrix[(int64_t)i * R + j] = run;
    }
    if (num_worst_tokens >= 0 && run > num_worst_tokens) rc = ORACLE_ERR_CAPACITY;
  }
  for (int e = 0; e < E; ++e) {
    int32_t run = 0;
    for (int i = 0; i < R; ++i) {
      expert_prefix[(int64_t)i * E + e] = run;
      run += num_tokens_per_expert[(int64_t)i * E + e];
    }
    expert_prefix[(int64_t)R * E + e] = run;
    int32_t a = expert_alignment;
    num_recv_tokens_per_expert[e] = ((run + a - 1) / a) * a;
  }
  for (int r = 0; r < R; ++r) {
    int64_t s = 0;
    psum[(int64_t)r * (E_l + 1)] = 0;
    for (int l = 0; l < E_l; ++l) {
      s += num_recv_tokens_per_expert[(int64_t)r * E_l + l];
      psum[(int64_t)r * (E_l + 1) + l + 1] = s;
    }
  }
  return rc;
}

/* ------------------------------------------------------------------ */
/* Row copy (bf16) or quantise (FP8) into a destination row             */
/* ------------------------------------------------------------------ */

static void put_row(const uint16_t* xrow, int H, int fp8_mode, void* recv_x, int64_t flat_row,
                    void* recv_scales, int64_t scale_base, int64_t scale_stride) {
  if (fp8_mode == FP8_NONE) {
    uint16_t* dst = (uint16_t*)recv_x + flat_row * H;
    for (int h = 0; h < H; ++h) dst[h] = xrow[h];
  } else {
    uint8_t* dst = (uint8_t*)recv_x + flat_row * H;
    float* sf = NULL;
    uint8_t* su = NULL;
    if (fp8_mode == FP8_E4M3_F32_SCALE) sf = (float*)recv_scales + scale_base;
    else su = (uint8_t*)recv_scales + scale_base;
    ep_oracle_quantize_row(xrow, H, fp8_mode, dst, sf, su, scale_stride);
  }
}

/* ------------------------------------------------------------------ */
/* Normal-mode dispatch ([06_deepep §1.1, §2.3, §4.3])                   */
/* ------------------------------------------------------------------ */

/* Contiguous per-expert receive layout.  Rank r's buffer is [cap_rows, H];
 * local expert l owns rows [psum[r][l], psum[r][l+1]).  Slot (i, t, j) with
 * expert e = r*E_l + l lands in row
 *     psum[r][l] + expert_prefix[i][e] + slot_rank[i][t][j]
 * (segment start + offset of source rank i + position within rank i), i.e.
 * the receiver-side "rank offset + finer offset" address of §2.3.
 *   recv_x      [R, cap_rows, H]  bf16, or E4M3 bytes when fp8_mode > 0
 *   recv_scales [R, H/128, cap_rows] fp32 (mode 1) or uint8 (mode 2)
 *   recv_src_idx[R, cap_rows]     i*T_r + t of the row's token, -1 elsewhere
 *   combine_idx [R, T_r, k]       r*cap_rows + row, -1 for a masked slot
 * A row at or past cap_rows is not written; its slot gets -1 and the call
 * returns ORACLE_ERR_CAPACITY. */
int ep_oracle_dispatch(const uint16_t* x, const int64_t* topk_idx, const int32_t* slot_rank,
                       const int32_t* expert_prefix, const int64_t* psum,
                       int R, int T_r, int H, int E, int k, int fp8_mode, int64_t cap_rows,
                       void* recv_x, void* recv_scales, int32_t* recv_src_idx,
                       int32_t* combine_idx) {
  if (R <= 0 || E % R != 0 || (fp8_mode != FP8_NONE && H % BLOCK_CHANNELS != 0))
    return ORACLE_ERR_INVALID_ARG;
  int E_l = E / R;
  int nb = H / BLOCK_CHANNELS;
  int rc = ORACLE_OK;
  for (int64_t p = 0; p < (int64_t)R * cap_rows; ++p) recv_src_idx[p] = -1;
  for (int i = 0; i < R; ++i) {
    for (int t = 0; t < T_r; ++t) {
      for (int j = 0; j < k; ++j) {
        int64_t p = ((int64_t)i * T_r + t) * k + j;
        int64_t e = topk_idx[p];
        if (e == -1) {
          combine_idx[p] = -1;
          continue;
        }
        if (e < -1 || e >= E) return ORACLE_ERR_INVALID_ARG;
        int r = (int)(e / E_l);
        int l = (int)(e % E_l);
        int64_t row = psum[(int64_t)r * (E_l + 1) + l] + expert_prefix[(int64_t)i * E + e] + slot_rank[p];
        if (row >= cap_rows) {
          combine_idx[p] = -1;
          rc = ORACLE_ERR_CAPACITY;
          continue;
        }
        int64_t flat = (int64_t)r * cap_rows + row;
        put_row(x + ((int64_t)i * T_r + t) * H, H, fp8_mode, recv_x, flat, recv_scales,
                (int64_t)r * nb * cap_rows + row, cap_rows);
        recv_src_idx[flat] = i * T_r + t;
        combine_idx[p] = (int32_t)flat;
      }
    }
  }
  return rc;
}

/* ------------------------------------------------------------------ */
/* Low-latency dispatch ([06_deepep §1.2, §3.2])                         */
/* ------------------------------------------------------------------ */

/* Packed masked layout.  Expert e lives on rank r = e / E_l (§3.2) as local
 * expert l = e % E_l; its rows are packed_recv_x[r][l][0 .. recv_count[r][l])
 * out of R*max_tokens_per_rank, ordered by (source rank, token, slot):
 *     row = expert_prefix[i][e] + slot_rank[i][t][j]
 * where both terms come from this oracle's own layout / notify definitions.
 *   packed_recv_x      [R, E_l, R*max, H] bf16 or E4M3
 *   packed_recv_scales [R, E_l, H/128, R*max] fp32 / uint8 (column-major)
 *   packed_recv_src_info [R, E_l, R*max] i*T_r + t (rows past recv_count untouched)
 *   layout_range       [R, E_l, R] (expert_prefix[i][e] << 32) | count[i][e]
 *   recv_count         [R, E_l] unaligned received rows (= masked_m)
 *   combine_idx        [R, T_r, k] e*(R*max) + row, -1 for a masked slot
 * T_r > max_tokens_per_rank is ORACLE_ERR_INVALID_ARG; a row past R*max
 * (only possible with a repeated expert in one token) is skipped and
 * reported as ORACLE_ERR_CAPACITY. */
int ep_oracle_ll_dispatch(const uint16_t* x, const int64_t* topk_idx, int R, int T_r, int H,
                          int E, int k, int max_tokens_per_rank, int fp8_mode,
                          void* packed_recv_x, void* packed_recv_scales,
                          int32_t* packed_recv_src_info, int64_t* layout_range,
                          int32_t* recv_count, int32_t* combine_idx) {
  if (R <= 0 || E % R != 0 || T_r > max_tokens_per_rank ||
      (fp8_mode != FP8_NONE && H % BLOCK_CHANNELS != 0))
    return ORACLE_ERR_INVALID_ARG;
  int E_l = E / R;
  int nb = H / BLOCK_CHANNELS;
  int64_t seg_rows = (int64_t)R * max_tokens_per_rank;
  int32_t* ntpr = (int32_t*)calloc((size_t)R * R, sizeof(int32_t));
  int32_t* ntpe = (int32_t*)calloc((size_t)R * E, sizeof(int32_t));
  uint8_t* in_rank = (uint8_t*)calloc((size_t)R * T_r * R + 1, 1);
  int32_t* slot_rank = (int32_t*)calloc((size_t)R * T_r * k + 1, sizeof(int32_t));
  int32_t* rpm = (int32_t*)calloc((size_t)R * R, sizeof(int32_t));
  int32_t* eprefix = (int32_t*)calloc((size_t)(R + 1) * E, sizeof(int32_t));
  int32_t* nrecv = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  int64_t* psum = (int64_t*)calloc((size_t)R * (E_l + 1), sizeof(int64_t));
  int rc = ep_oracle_layout(topk_idx, R, T_r, k, E, ntpr, ntpe, in_rank, slot_rank);
  if (rc == ORACLE_OK)
    rc = ep_oracle_notify(ntpr, ntpe, R, E, 1, -1, rpm, eprefix, nrecv, psum);
  if (rc == ORACLE_OK) {
    for (int e = 0; e < E; ++e) {
      recv_count[e] = eprefix[(int64_t)R * E + e];
      for (int i = 0; i < R; ++i)
        layout_range[(int64_t)e * R + i] =
            ((int64_t)eprefix[(int64_t)i * E + e] << 32) | (int64_t)ntpe[(int64_t)i * E + e];
    }
    for (int i = 0; i < R; ++i) {
      for (int t = 0; t < T_r; ++t) {
        for (int j = 0; j < k; ++j) {
          int64_t p = ((int64_t)i * T_r + t) * k + j;
          int64_t e = topk_idx[p];
          if (e < 0) {
            combine_idx[p] = -1;
            continue;
          }
          int64_t row = (int64_t)eprefix[(int64_t)i * E + e] + slot_rank[p];
          if (row >= seg_rows) {
            combine_idx[p] = -1;
            rc = ORACLE_ERR_CAPACITY;
            continue;
          }
          int64_t flat = e * seg_rows + row;
          put_row(x + ((int64_t)i * T_r + t) * H, H, fp8_mode, packed_recv_x, flat,
                  packed_recv_scales, e * nb * seg_rows + row, seg_rows);
          packed_recv_src_info[flat] = i * T_r + t;
          combine_idx[p] = (int32_t)flat;
        }
      }
    }
  }
  free(ntpr); free(ntpe); free(in_rank); free(slot_rank);
  free(rpm); free(eprefix); free(nrecv); free(psum);
  return rc;
}

/* ------------------------------------------------------------------ */
/* Combine ([06_deepep §1.1, §4.3, §5: combine is dispatch reversed])    */
/* ------------------------------------------------------------------ */

/* out[t][h] = bf16( fma chain over j = 0..k-1 of w[t][j] * y[combine_idx[t][j]][h] )
 * in fp32, starting from +0, skipping slots whose combine_idx is -1.  y is
 * any receive buffer viewed as [n_rows, H] (contiguous or packed layout), so
 * the same definition serves normal and low-latency combine. */
int ep_oracle_combine(const uint16_t* y, const float* topk_weights, const int32_t* combine_idx,
                      int64_t n_rows, int64_t n_tokens, int H, int k, uint16_t* out) {
  for (int64_t t = 0; t < n_tokens; ++t) {
    for (int j = 0; j < k; ++j) {
      int32_t f = combine_idx[t * k + j];
      if (f < -1 || f >= n_rows) return ORACLE_ERR_INVALID_ARG;
    }
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        int32_t f = combine_idx[t * k + j];
        if (f < 0) continue;
        acc = fmaf(topk_weights[t * k + j], ep_oracle_bf16_to_f32(y[(int64_t)f * H + h]), acc);
      }
      out[t * H + h] = ep_oracle_f32_to_bf16(acc);
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Once-per-rank receive layout ([06_deepep §2.1, §2.3]: V1 normal mode) */
/* ------------------------------------------------------------------ */

/* Token t of source rank i goes ONCE to every rank r that holds one of its
 * experts (is_token_in_rank[i][t][r]).  Rank r's buffer [cap_rows, H] holds
 * source rank i's tokens in rows [rpm[i-1][r], rpm[i][r]) -- rpm the
 * rank_prefix_matrix, inclusive over source ranks, rpm[-1] = 0 -- in token
 * order:
 *     row(i, t, r) = rpm[i-1][r] + #{ t' < t : is_token_in_rank[i][t'][r] }.
 *   recv_x, recv_scales  as in dispatch, one row per (token, rank)
 *   recv_src_idx     [R, cap_rows]    i*T_r + t, -1 where no token sits
 *   recv_topk_idx    [R, cap_rows, k] per slot j of the row's token: its
 *                    expert's local index e - r*E_l when that expert is on
 *                    r, else -1 (rows holding no token are left untouched)
 *   recv_topk_weights[R, cap_rows, k] the slot's weight when its expert is
 *                    on r, else 0
 *   combine_idx      [R, T_r, k]     r*cap_rows + row(i, t, r) at the token's
 *                    FIRST slot whose expert is on r, -1 at every other slot
 * rpm is computed here from the definition (count, then prefix), not taken
 * from the caller.  A row at or past cap_rows is not written (its slot gets
 * -1) and the call returns ORACLE_ERR_CAPACITY. */
int ep_oracle_rank_dispatch(const uint16_t* x, const int64_t* topk_idx, const float* topk_weights,
                            int R, int T_r, int H, int E, int k, int fp8_mode, int64_t cap_rows,
                            void* recv_x, void* recv_scales, int32_t* recv_src_idx,
                            int64_t* recv_topk_idx, float* recv_topk_weights,
                            int32_t* combine_idx) {
  if (R <= 0 || E % R != 0 || (fp8_mode != FP8_NONE && H % BLOCK_CHANNELS != 0))
    return ORACLE_ERR_INVALID_ARG;
  int E_l = E / R;
  int nb = H / BLOCK_CHANNELS;
  int rc = ORACLE_OK;
  for (int64_t p = 0; p < (int64_t)R * T_r * k; ++p)
    if (topk_idx[p] < -1 || topk_idx[p] >= E) return ORACLE_ERR_INVALID_ARG;
  /* tokens of source rank i that go to rank r, and the inclusive prefix */
  int64_t* cnt = (int64_t*)calloc((size_t)R * R, sizeof(int64_t));
  for (int i = 0; i < R; ++i)
    for (int t = 0; t < T_r; ++t)
      for (int r = 0; r < R; ++r) {
        int hit = 0;
        for (int j = 0; j < k; ++j) {
          int64_t e = topk_idx[((int64_t)i * T_r + t) * k + j];
          if (e >= 0 && e / E_l == r) hit = 1;
        }
        cnt[(int64_t)i * R + r] += hit;
      }
  for (int64_t q = 0; q < (int64_t)R * cap_rows; ++q) recv_src_idx[q] = -1;
  for (int r = 0; r < R; ++r) {
    int64_t before = 0; /* rpm[i-1][r] */
    for (int i = 0; i < R; ++i) {
      int64_t pos = 0; /* tokens of rank i before t that go to r */
      for (int t = 0; t < T_r; ++t) {
        int64_t base = ((int64_t)i * T_r + t) * k;
        int first = -1;
        for (int j = 0; j < k; ++j) {
          int64_t e = topk_idx[base + j];
          if (e >= 0 && e / E_l == r) {
            first = j;
            break;
          }
        }
        if (first < 0) continue;
        int64_t row = before + pos;
        pos += 1;
        if (row >= cap_rows) {
          combine_idx[base + first] = -1;
          rc = ORACLE_ERR_CAPACITY;
          continue;
        }
        int64_t flat = (int64_t)r * cap_rows + row;
        put_row(x + ((int64_t)i * T_r + t) * H, H, fp8_mode, recv_x, flat, recv_scales,
                (int64_t)r * nb * cap_rows + row, cap_rows);
        recv_src_idx[flat] = i * T_r + t;
        for (int j = 0; j < k; ++j) {
          int64_t e = topk_idx[base + j];
          int on_r = e >= 0 && e / E_l == r;
          recv_topk_idx[flat * k + j] = on_r ? e - (int64_t)r * E_l : -1;
          recv_topk_weights[flat * k + j] = on_r ? topk_weights[base + j] : 0.0f;
        }
        combine_idx[base + first] = (int32_t)flat;
      }
      before += cnt[(int64_t)i * R + r];
    }
  }
  /* slots that are not a token's first slot on their rank */
  for (int i = 0; i < R; ++i)
    for (int t = 0; t < T_r; ++t) {
      int64_t base = ((int64_t)i * T_r + t) * k;
      for (int j = 0; j < k; ++j) {
        int64_t e = topk_idx[base + j];
        int first = e >= 0;
        for (int jj = 0; jj < j && first; ++jj) {
          int64_t ee = topk_idx[base + jj];
          if (ee >= 0 && ee / E_l == e / E_l) first = 0;
        }
        if (!first) combine_idx[base + j] = -1;
      }
    }
  free(cnt);
  return rc;
}

/* Rank-level combine ([06_deepep §2.3]: dispatch walked backwards): every
 * rank returns one row per token it received, already weighted by the
 * experts that rank holds, and the rows are summed:
 *     out[t][h] = bf16( sum in slot order over the slots j with
 *                       combine_idx[t][j] >= 0 of y[combine_idx[t][j]][h] )
 * in fp32 from +0 (one row per destination rank, at the token's first slot
 * on that rank), rounded once. */
int ep_oracle_rank_combine(const uint16_t* y, const int32_t* combine_idx, int64_t n_rows,
                           int64_t n_tokens, int H, int k, uint16_t* out) {
  for (int64_t t = 0; t < n_tokens; ++t) {
    for (int j = 0; j < k; ++j) {
      int32_t f = combine_idx[t * k + j];
      if (f < -1 || f >= n_rows) return ORACLE_ERR_INVALID_ARG;
    }
    for (int h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        int32_t f = combine_idx[t * k + j];
        if (f < 0) continue;
        acc = acc + ep_oracle_bf16_to_f32(y[(int64_t)f * H + h]);
      }
      out[t * H + h] = ep_oracle_f32_to_bf16(acc);
    }
  }
  return ORACLE_OK;
}
