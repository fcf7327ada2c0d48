/* abi_check.c -- libep driven from plain C through include/ep.h (device
 * buffers from cudaMalloc, no Python, no torch), each result held against
 * the C oracle linked beside it.  Inputs come from a small LCG here: they
 * hold none of the method's arithmetic.  Checks, on a small batch:
 *   low-latency path: ep_clean_ll_buffer, ep_ll_dispatch (E4M3 + ue8m0),
 *                     ep_ll_combine;
 *   normal path:      ep_layout_notify, ep_dispatch (bf16), ep_combine;
 * and ep_read_status after each.  Prints "abi check ok" and exits 0, or
 * names the first mismatch and exits 1. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ep.h"

/* the oracle's entry points (oracle/ep_oracle.c) */
int ep_oracle_ll_dispatch(const uint16_t* x, const int64_t* topk_idx, int R, int T_r, int H, int E,
                          int k, int max_tokens_per_rank, int fp8_mode, void* packed_recv_x,
                          void* packed_recv_scales, int32_t* packed_recv_src_info,
                          int64_t* layout_range, int32_t* recv_count, int32_t* combine_idx);
int ep_oracle_layout(const int64_t* topk_idx, int R, int T_r, int k, int E,
                     int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                     uint8_t* is_token_in_rank, int32_t* slot_rank);
int ep_oracle_notify(const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_expert,
                     int R, int E, int expert_alignment, int64_t num_worst_tokens,
                     int32_t* rank_prefix_matrix, int32_t* expert_prefix,
                     int32_t* num_recv_tokens_per_expert, int64_t* psum);
int ep_oracle_dispatch(const uint16_t* x, const int64_t* topk_idx, const int32_t* slot_rank,
                       const int32_t* expert_prefix, const int64_t* psum, int R, int T_r, int H,
                       int E, int k, int fp8_mode, int64_t cap_rows, void* recv_x,
                       void* recv_scales, int32_t* recv_src_idx, int32_t* combine_idx);
int ep_oracle_combine(const uint16_t* y, const float* topk_weights, const int32_t* combine_idx,
                      int64_t n_rows, int64_t n_tokens, int H, int k, uint16_t* out);

enum { R = 4, T_R = 16, H = 256, E = 16, K = 2, MAXT = 16 };
enum { T = R * T_R, EL = E / R, S = R * MAXT, NB = H / 128 };

static uint64_t lcg = 0x9E3779B97F4A7C15ull;
static uint32_t rnd(void) {
  lcg = lcg * 6364136223846793005ull + 1442695040888963407ull;
  return (uint32_t)(lcg >> 33);
}

#define CK(call)                                                          \
  do {                                                                    \
    cudaError_t e_ = (call);                                              \
    if (e_ != cudaSuccess) {                                              \
      printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, \
             __LINE__);                                                   \
      return 1;                                                           \
    }                                                                     \
  } while (0)
#define EPK(call)                                            \
  do {                                                       \
    int rc_ = (call);                                        \
    if (rc_ != EP_OK) {                                      \
      printf("%s failed: %s\n", #call, ep_error_string(rc_)); \
      return 1;                                              \
    }                                                        \
  } while (0)
#define SAME(a, b, bytes, what)                       \
  do {                                                \
    if (memcmp((a), (b), (bytes)) != 0) {             \
      printf("mismatch: %s\n", what);                 \
      return 1;                                       \
    }                                                 \
  } while (0)

static void* dalloc(size_t bytes) {
  void* p = NULL;
  if (cudaMalloc(&p, bytes ? bytes : 16) != cudaSuccess) return NULL;
  cudaMemset(p, 0x5A, bytes ? bytes : 16);
  return p;
}

int main(void) {
  static uint16_t x[T * H];
  static int64_t idx[T * K];
  static float w[T * K];
  for (int i = 0; i < T * H; ++i) x[i] = (uint16_t)(0x3C00u + (rnd() & 0x7FFu) - 0x400u) ^ (uint16_t)((rnd() & 1u) << 15);
  for (int t = 0; t < T; ++t) {
    int e0 = (int)(rnd() % E), e1 = (int)(rnd() % (E - 1));
    if (e1 >= e0) e1 += 1;
    idx[t * K] = e0;
    idx[t * K + 1] = (rnd() % 8 == 0) ? -1 : e1;   /* some slots unused */
    w[t * K] = (float)(rnd() % 1000) / 1000.0f;
    w[t * K + 1] = (float)(rnd() % 1000) / 1000.0f;
  }
  cudaStream_t st;
  CK(cudaStreamCreate(&st));
  void *dx = dalloc(sizeof x), *didx = dalloc(sizeof idx), *dw = dalloc(sizeof w);
  int32_t* dstatus = (int32_t*)dalloc(4);
  CK(cudaMemcpy(dx, x, sizeof x, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(didx, idx, sizeof idx, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dw, w, sizeof w, cudaMemcpyHostToDevice));
  CK(cudaMemset(dstatus, 0, 4));
  const size_t ws_bytes = ep_workspace_size(R, T_R, K, E, H);
  void* dws = dalloc(ws_bytes);
  int32_t status = 0;

  /* ---- low-latency path, E4M3 + ue8m0 */
  {
    const size_t rx = (size_t)E * S * H, rs = (size_t)E * NB * S;
    void *dpx = dalloc(rx), *dps = dalloc(rs), *dsrc = dalloc((size_t)E * S * 4),
         *dlr = dalloc((size_t)E * R * 8), *dcnt = dalloc((size_t)E * 4), *dcidx = dalloc((size_t)T * K * 4);
    EPK(ep_clean_ll_buffer((int32_t*)dcnt, R, E, dws, ws_bytes, st));
    EPK(ep_ll_dispatch(dx, (const int64_t*)didx, R, T_R, H, E, K, MAXT, EP_FP8_E4M3_UE8M0, dpx, dps,
                       (int32_t*)dsrc, (int64_t*)dlr, (int32_t*)dcnt, (int32_t*)dcidx, dws, ws_bytes,
                       dstatus, st));
    EPK(ep_read_status(dstatus, &status, st));
    if (status != EP_OK) { printf("ll dispatch status %d\n", status); return 1; }
    uint8_t* gx = (uint8_t*)malloc(rx); uint8_t* ox = (uint8_t*)calloc(rx, 1);
    uint8_t* gs = (uint8_t*)malloc(rs); uint8_t* os = (uint8_t*)calloc(rs, 1);
    int32_t *gsrc = (int32_t*)malloc((size_t)E * S * 4), *osrc = (int32_t*)calloc((size_t)E * S, 4);
    int64_t glr[E * R], olr[E * R];
    int32_t gcnt[E], ocnt[E], gcidx[T * K], ocidx[T * K];
    CK(cudaMemcpy(gx, dpx, rx, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gs, dps, rs, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gsrc, dsrc, (size_t)E * S * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(glr, dlr, sizeof glr, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gcnt, dcnt, sizeof gcnt, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gcidx, dcidx, sizeof gcidx, cudaMemcpyDeviceToHost));
    if (ep_oracle_ll_dispatch(x, idx, R, T_R, H, E, K, MAXT, EP_FP8_E4M3_UE8M0, ox, os, osrc, olr,
                              ocnt, ocidx) != 0) { printf("oracle ll dispatch failed\n"); return 1; }
    SAME(gcnt, ocnt, sizeof gcnt, "recv_count");
    SAME(glr, olr, sizeof glr, "layout_range");
    SAME(gcidx, ocidx, sizeof gcidx, "combine_idx (low latency)");
    for (int e = 0; e < E; ++e) {
      for (int r = 0; r < ocnt[e]; ++r) {
        const size_t f = (size_t)e * S + r;
        SAME(gx + f * H, ox + f * H, H, "packed_recv_x row");
        SAME(gsrc + f, osrc + f, 4, "packed_recv_src_info");
        for (int b = 0; b < NB; ++b) {
          const size_t o = ((size_t)e * NB + b) * S + r;
          SAME(gs + o, os + o, 1, "packed_recv_scales");
        }
      }
    }
    /* combine: y = the packed rows widened back to bf16 would need the
     * dequantiser; any bf16 rows do, so y holds fresh values */
    const size_t ny = (size_t)E * S * H;
    uint16_t* y = (uint16_t*)malloc(ny * 2);
    for (size_t i = 0; i < ny; ++i) y[i] = (uint16_t)(0x3C00u + (rnd() & 0x3FFu) - 0x200u);
    void *dy = dalloc(ny * 2), *dout = dalloc((size_t)T * H * 2);
    CK(cudaMemcpy(dy, y, ny * 2, cudaMemcpyHostToDevice));
    EPK(ep_ll_combine(dy, (const float*)dw, (const int32_t*)dcidx, R, T_R, H, E, K, MAXT, dout, dstatus, st));
    EPK(ep_read_status(dstatus, &status, st));
    if (status != EP_OK) { printf("ll combine status %d\n", status); return 1; }
    static uint16_t gout[T * H], oout[T * H];
    CK(cudaMemcpy(gout, dout, sizeof gout, cudaMemcpyDeviceToHost));
    if (ep_oracle_combine(y, w, ocidx, (int64_t)E * S, T, H, K, oout) != 0) { printf("oracle combine failed\n"); return 1; }
    SAME(gout, oout, sizeof gout, "low-latency combine output");
  }

  /* ---- normal path, bf16: layout + notify in one launch, dispatch, combine */
  {
    int32_t *dntpr = (int32_t*)dalloc(R * R * 4), *dntpe = (int32_t*)dalloc(R * E * 4),
            *dslot = (int32_t*)dalloc(T * K * 4), *drpm = (int32_t*)dalloc(R * R * 4),
            *dep = (int32_t*)dalloc((R + 1) * E * 4), *dnr = (int32_t*)dalloc(R * EL * 4);
    uint8_t* ditr = (uint8_t*)dalloc(T * R);
    int64_t* dps = (int64_t*)dalloc(R * (EL + 1) * 8);
    EPK(ep_layout_notify((const int64_t*)didx, R, T_R, K, E, 4, -1, dntpr, dntpe, ditr, dslot, drpm, dep,
                         dnr, dps, NULL, 10000, dws, ws_bytes, dstatus, st));
    int32_t ontpr[R * R], ontpe[R * E], oslot[T * K], orpm[R * R], oep[(R + 1) * E], onr[R * EL];
    uint8_t oitr[T * R];
    int64_t ops[R * (EL + 1)], gps[R * (EL + 1)];
    ep_oracle_layout(idx, R, T_R, K, E, ontpr, ontpe, oitr, oslot);
    ep_oracle_notify(ontpr, ontpe, R, E, 4, -1, orpm, oep, onr, ops);
    CK(cudaMemcpy(gps, dps, sizeof gps, cudaMemcpyDeviceToHost));
    SAME(gps, ops, sizeof gps, "psum");
    int64_t cap = 1;
    for (int r = 0; r < R; ++r) if (ops[r * (EL + 1) + EL] > cap) cap = ops[r * (EL + 1) + EL];
    const size_t rx = (size_t)R * cap * H * 2;
    void *drx = dalloc(rx), *dsrc = dalloc((size_t)R * cap * 4), *dcidx = dalloc((size_t)T * K * 4);
    EPK(ep_dispatch(dx, (const int64_t*)didx, dslot, dep, dps, R, T_R, H, E, K, EP_FP8_NONE, cap, drx,
                    NULL, (int32_t*)dsrc, (int32_t*)dcidx, dws, ws_bytes, dstatus, st));
    EPK(ep_read_status(dstatus, &status, st));
    if (status != EP_OK) { printf("dispatch status %d\n", status); return 1; }
    uint16_t* grx = (uint16_t*)malloc(rx); uint16_t* orx = (uint16_t*)calloc(rx, 1);
    int32_t* gsrc = (int32_t*)malloc((size_t)R * cap * 4); int32_t* osrc = (int32_t*)calloc((size_t)R * cap, 4);
    int32_t gcidx[T * K], ocidx[T * K];
    CK(cudaMemcpy(grx, drx, rx, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gsrc, dsrc, (size_t)R * cap * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(gcidx, dcidx, sizeof gcidx, cudaMemcpyDeviceToHost));
    ep_oracle_dispatch(x, idx, oslot, oep, ops, R, T_R, H, E, K, EP_FP8_NONE, cap, orx, NULL, osrc, ocidx);
    SAME(gcidx, ocidx, sizeof gcidx, "combine_idx (normal)");
    SAME(gsrc, osrc, (size_t)R * cap * 4, "recv_src_idx");
    for (int64_t f = 0; f < R * cap; ++f)
      if (osrc[f] >= 0) SAME(grx + f * H, orx + f * H, H * 2, "recv_x row");
    void* dout = dalloc((size_t)T * H * 2);
    EPK(ep_combine(drx, (const float*)dw, (const int32_t*)dcidx, R, T_R, H, K, cap, dout, dstatus, st));
    EPK(ep_read_status(dstatus, &status, st));
    if (status != EP_OK) { printf("combine status %d\n", status); return 1; }
    static uint16_t gout[T * H], oout[T * H];
    CK(cudaMemcpy(gout, dout, sizeof gout, cudaMemcpyDeviceToHost));
    ep_oracle_combine(orx, w, ocidx, (int64_t)R * cap, T, H, K, oout);   /* identity experts */
    SAME(gout, oout, sizeof gout, "normal combine output");
  }
  printf("abi check ok (%llu libep launches)\n", (unsigned long long)ep_launch_count());
  return 0;
}
