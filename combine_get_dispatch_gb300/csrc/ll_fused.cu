// ll_fused.cu -- the single-launch low-latency dispatch (k_ll_fused) and
// the ep_ll_dispatch entry point, which takes it for decode-size batches and
// the layout + scatter + scale-column kernels of dispatch.cu otherwise
// (llm-infra-atlas DeepEP article §1.2, §3.2, §4.6).

#include <mutex>

#include "dispatch.cuh"

namespace ep {

// ------------------------------------------------------------------ fused low latency

// Low-latency dispatch of a decode-size batch in ONE launch: routing layout,
// scatter, FP8 quantisation and the column-major scales.  One CTA per SM;
// the batch's (token, 1024-channel piece) units are split evenly over the
// CTAs (a CTA's "own" tokens are those it holds a piece of), and every CTA
//   0. loads every id from the first up to its last own id (in (rank,
//      token, slot) order), then bulk-loads all of its x pieces behind them;
//   1. counts, per expert, the ids before its own range -- the slots that
//      precede its own range in the packed order -- and keeps its own ids,
//      so it needs nothing from any other CTA to place its rows;
//   2. its 4 rank warps rank the own slots in order (equal-key lane masks),
//      which gives each slot's packed row -- the global exclusive count of
//      its expert (§1.2, §3.2) -- and write combine_idx and src_info for the
//      tokens whose first piece the CTA holds (the CTA holding the last token
//      has seen every id and writes recv_count);
//   3. bf16: as each piece lands, its k bulk stores go out.  FP8: warps 0..11
//      own the units, quantise each in place as it lands (staging the token's
//      block scales row-major) and mark it on a per-unit mbarrier; warps
//      12..15 (the rank warps) issue each unit's k bulk stores the moment it
//      is marked and its rows are known;
//   4. the unit warps (bf16: all warps) arrive at a grid barrier (workspace
//      counter), wait for every CTA, and write the per-expert outputs of
//      the experts e = cta + n * grid while the stores drain: layout_range
//      from the sources of their rows (sorted by token, so each rank is one
//      run) and (FP8) the column-major scales, coalesced along rows.
// The id scan is redundant across CTAs (CTA j reads ~j/grid of the ids, from
// L2 after the first touch) but takes no round trip through another CTA: an
// exchange of per-chunk counts, read while the x pieces are queued, made
// every CTA wait for the slowest and for the x queue.
// All CTAs are resident at once (one per SM, grid at most the SM count,
// launched cooperatively, so the runtime starts the grid only when every
// CTA has an SM), so the wait at the grid barrier ends; every wait is
// bounded anyway and gives up with EP_ERR_TIMEOUT.

constexpr int kFusedWarps = 16;
constexpr int kQuantWarps = 12;          // FP8: warps owning (loading, quantising) units; the
                                         // other 4 issue the bulk stores as units are quantised
constexpr int kFusedMaxPerWarp = 8;      // units per warp
constexpr int kFusedPiece = 1024;        // channels per unit
constexpr int kEarlyUnits = 1;           // units per warp loaded with the ids; the rest right
                                         // after every thread's id loads are out
constexpr int kRankWarps = 4;            // the last warps: rank the CTA's own slots (FP8: the
                                         // store warps)
constexpr int kRankIdsPerLane = 8;
constexpr int kMaxOwnIds = kRankWarps * kWarp * kRankIdsPerLane;
constexpr int kScanIdsPerThread = 32;    // ids a thread has in flight per pass of the id scan
constexpr int kFusedMaxIds = 4 * kFusedWarps * kWarp * kScanIdsPerThread;   // at most 4 passes
constexpr int kFusedBarBytes = 2 * kFusedWarps * kFusedMaxPerWarp * 8;   // load + quantised barriers
constexpr size_t kFusedSmemCap = 225 * 1024;
static_assert(kRankWarps == kFusedWarps - kQuantWarps, "FP8: the rank warps are the store warps");
static_assert(kFusedMaxPerWarp <= kWarp, "a warp issues its pieces one per lane");
constexpr int kCtlArrive = 8;            // workspace control words of this kernel (see kCtlClaim)
constexpr int kCtlExit = 9;

// Wait (bounded, kWaitNs) until a grid counter reaches n; false on timeout.
__device__ __forceinline__ bool wait_count(const uint32_t* ctr, uint32_t n) {
  if (ld_acquire_u32(ctr) >= n) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_u32(ctr) < n) {
    __nanosleep(64);
    if (globaltimer_ns() - t0 > kWaitNs) return false;
  }
  return true;
}

struct FusedParams {
  const uint8_t* x;
  const int64_t* topk_idx;
  int R, T_r, H, E, k;
  int32_t T;
  int32_t n_ids;             // T * k
  int64_t seg_rows;          // R * max_tokens_per_rank (rows per expert)
  uint8_t* recv_x;           // packed [E][seg_rows][row bytes]
  void* scales;              // packed column-major [E][H/128][seg_rows]
  int32_t* src_info;         // [E][seg_rows]
  int64_t* layout_range;     // [E][R]
  int32_t* recv_count;       // [E]
  int32_t* combine_idx;      // [T][k]
  uint8_t* scale_rows;       // [T][scale_row_bytes] staged per-token scales
  int scale_row_bytes;
  uint32_t* ctl;             // workspace control words
  int32_t* status;
  // geometry
  int Hp, P;
  int32_t n_units;
  uint32_t slot_bytes;       // one bf16 piece, 128-byte multiple
  uint32_t slot_area;        // bytes of the CTA's slots
  int own_cap;               // own-id capacity (multiple of 32)
  int nA;                    // experts per CTA (ceil(E / grid))
  int nbits;
  bool fp8;                  // FP8 modes: units owned by kQuantWarps warps
};

// Per-expert outputs of the fused path for this CTA's experts e = cta + a * grid
// (a < nA), by threads t < nt of a group that `sync` synchronises:
// layout_range from the sources of their rows (sorted by token, so each
// rank is one run) and (FP8) their column-major scales from the staged rows.
// One item per (row, 16-byte scale group); a thread keeps kColBatch items'
// loads in flight at once -- the bulk stores are draining and every round
// trip is slow.
template <bool kFp8, int kEs, class Sync>
__device__ __forceinline__ void fused_expert_outputs(const FusedParams& p, int cta, int grid, int t,
                                                     int nt, int32_t* s_rows, int32_t* s_lo, Sync sync) {
  constexpr int kColBatch = 4;
  if (t < p.nA) {
    const int e = cta + t * grid;
    s_rows[t] = e < p.E ? (int32_t)min((int64_t)max(ld_cg_i32(&p.recv_count[e]), 0), p.seg_rows) : 0;
  }
  sync();
  int32_t total = 0;
  for (int a = 0; a < p.nA; ++a) total += s_rows[a];
  const int R1 = p.R + 1;
  for (int a = 0; a < p.nA; ++a)   // experts without rows: every rank starts at 0
    if (s_rows[a] == 0)
      for (int i = t; i < R1; i += nt) s_lo[a * R1 + i] = 0;
  const int ngrp = kFp8 ? p.scale_row_bytes / 16 : 1;
  const int nb = p.H / kFp8Block;
  const int32_t items = total * ngrp;
  for (int32_t i0 = 0; i0 < items; i0 += nt * kColBatch) {
    int a_of[kColBatch], grp[kColBatch];
    int32_t row[kColBatch], s[kColBatch], s_prev[kColBatch];
#pragma unroll
    for (int u = 0; u < kColBatch; ++u) {
      const int32_t it = i0 + u * nt + t;
      a_of[u] = -1;
      grp[u] = 0;
      row[u] = 0;
      s[u] = -1;
      s_prev[u] = -1;
      if (it < items) {
        grp[u] = it % ngrp;
        int32_t f = it / ngrp;
        int a = 0;
        while (a < p.nA - 1 && f >= s_rows[a]) f -= s_rows[a++];
        a_of[u] = a;
        row[u] = f;
        const int32_t* src = p.src_info + (int64_t)(cta + a * grid) * p.seg_rows;
        s[u] = ld_cg_i32(&src[f]);
        if (grp[u] == 0 && f > 0) s_prev[u] = ld_cg_i32(&src[f - 1]);
      }
    }
    uint4 w4[kColBatch];
#pragma unroll
    for (int u = 0; u < kColBatch; ++u) {
      w4[u] = make_uint4(0, 0, 0, 0);
      if (kFp8 && a_of[u] >= 0 && s[u] >= 0 && s[u] < p.T)
        w4[u] = ld_cg_v4(p.scale_rows + (int64_t)s[u] * p.scale_row_bytes + grp[u] * 16);
    }
#pragma unroll
    for (int u = 0; u < kColBatch; ++u) {
      if (a_of[u] < 0) continue;
      const int a = a_of[u];
      const int e = cta + a * grid;
      if (grp[u] == 0) {
        // ranks (rank of row - 1, rank of row] start at this row; the last
        // row also closes the ranks after its own
        int32_t* lo = s_lo + a * R1;
        const int cnt = s_rows[a];
        const int lo_rank = row[u] == 0 ? 0 : max(s_prev[u], 0) / p.T_r + 1;
        const int cur_rank = max(s[u], 0) / p.T_r;
        for (int i = max(lo_rank, 0); i <= min(cur_rank, p.R); ++i) lo[i] = row[u];
        if (row[u] == cnt - 1)
          for (int i = max(cur_rank + 1, 0); i <= p.R; ++i) lo[i] = cnt;
      }
      if (kFp8 && s[u] >= 0 && s[u] < p.T) {
        constexpr int kPer16 = 16 / kEs;
        const uint32_t w[4] = {w4[u].x, w4[u].y, w4[u].z, w4[u].w};
#pragma unroll
        for (int q = 0; q < kPer16; ++q) {
          const int b = grp[u] * kPer16 + q;
          if (b < nb) {
            const int64_t o = ((int64_t)e * nb + b) * p.seg_rows + row[u];
            if (kEs == 4) static_cast<uint32_t*>(p.scales)[o] = w[q];
            else static_cast<uint8_t*>(p.scales)[o] = (uint8_t)(w[q >> 2] >> (8 * (q & 3)));
          }
        }
      }
    }
  }
  sync();
  for (int i = t; i < p.nA * p.R; i += nt) {
    const int a = i / p.R;
    const int r = i - a * p.R;
    const int e = cta + a * grid;
    if (e < p.E)
      p.layout_range[(size_t)e * p.R + r] =
          ((int64_t)s_lo[a * R1 + r] << 32) | (int64_t)(s_lo[a * R1 + r + 1] - s_lo[a * R1 + r]);
  }
}

template <int kMode>
__global__ void __launch_bounds__(kFusedWarps * kWarp, 1) k_ll_fused(FusedParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr bool kFp8 = kMode != EP_FP8_NONE;
  constexpr int kEs = kMode == EP_FP8_E4M3_F32_SCALE ? 4 : 1;
  constexpr int kThreads = kFusedWarps * kWarp;
  __shared__ int s_units_ok, s_passed;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int grid = (int)gridDim.x;
  const int cta = (int)blockIdx.x;

  // U * grid < 2^32 (checked on the host): 32-bit unit range arithmetic
  const uint32_t U = (uint32_t)p.n_units;
  const int32_t u0 = (int32_t)(U * (uint32_t)cta / (uint32_t)grid);
  const int32_t u1 = (int32_t)(U * (uint32_t)(cta + 1) / (uint32_t)grid);
  // FP8: warps 0..kQuantWarps-1 own (load, quantise) the units, the rest
  // issue their bulk stores; bf16: every warp owns units and stores them
  constexpr int kOwnWarps = kFp8 ? kQuantWarps : kFusedWarps;
  const int32_t nm = (warp < kOwnWarps && warp < u1 - u0)
                         ? (u1 - u0 - warp + kOwnWarps - 1) / kOwnWarps : 0;
  uint8_t* slots = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.slot_area) + warp * kFusedMaxPerWarp;
  // FP8: one "quantised" barrier per unit of the CTA (slot index q = u - u0)
  uint64_t* qbars = reinterpret_cast<uint64_t*>(smem + p.slot_area) + kFusedWarps * kFusedMaxPerWarp;
  int32_t* s_P = reinterpret_cast<int32_t*>(smem + p.slot_area + kFusedBarBytes);   // [E]
  int32_t* s_cnt = s_P + p.E;                    // [kRankWarps][E]
  int32_t* s_own = s_cnt + kRankWarps * p.E;     // [own_cap] own ids
  int32_t* s_f = s_own + p.own_cap;              // [own_cap] their packed rows
  int32_t* s_lo = s_f + p.own_cap;               // [nA][R + 1] first row of every rank
  auto unit_slot = [&](int32_t m) { return slots + (size_t)(warp + m * kOwnWarps) * p.slot_bytes; };
  auto unit_of = [&](int32_t m, int32_t* g, int* pc) {
    const int32_t u = u0 + warp + m * kOwnWarps;
    *g = u / p.P;
    *pc = u - *g * p.P;
  };

  // own token range [ga, gb) and its ids [own_lo, own_hi)
  const int32_t ga = u0 / p.P;
  const int32_t gb = u1 > u0 ? (u1 - 1) / p.P + 1 : ga;
  const int32_t own_lo = ga * p.k;
  const int32_t own_hi = gb * p.k;
  const int32_t own_n = own_hi - own_lo;
  const int64_t last_first = (int64_t)(p.T - 1) * p.P;
  const bool totals = last_first >= u0 && last_first < u1;   // sees every id: writes recv_count
  const int32_t scan_hi = own_n > 0 ? own_hi : 0;   // a CTA without units reads no ids

  // ---- 0. kEarlyUnits x pieces per warp go out first, then every id up to
  //      the end of the own range: the CTA counts the ids before its range
  //      itself (their per-expert counts are its prefix), so it waits for no
  //      other CTA.  The rest of the pieces follow after the block barrier
  //      below, when every thread's id loads are out ahead of them.  (The
  //      early pieces ahead of the ids rather than behind them: decode
  //      dispatch 31.2-31.3 us mean instead of 31.8-31.9.)
  constexpr int kScanPairs = kScanIdsPerThread / 2;   // 16-byte id loads per thread per pass
  constexpr int kPassIds = 2 * kThreads * kScanPairs;
  longlong2 vs[kScanPairs];
  auto load_scan = [&](int32_t base) {
#pragma unroll
    for (int u = 0; u < kScanPairs; ++u) {
      const int32_t q = base + 2 * (tid + u * kThreads);
      vs[u] = make_longlong2(-1, -1);
      if (q + 1 < scan_hi) vs[u] = ld_nc_i64x2(p.topk_idx + q);
      else if (q < scan_hi) vs[u].x = __ldg(p.topk_idx + q);
    }
  };
  auto load_unit = [&](int32_t m) {
    int32_t g;
    int pc;
    unit_of(m, &g, &pc);
    const uint32_t bytes = (uint32_t)min(p.Hp, p.H - pc * p.Hp) * 2u;
    mbar_arrive_expect_tx(&bars[m], bytes);
    tma_load_1d_hint(unit_slot(m), p.x + (int64_t)g * p.H * 2 + (int64_t)pc * p.Hp * 2, bytes, &bars[m],
                     l2_policy_evict_first());   // every token is read once
  };
  if (nm > 0 && lane == 0) {
    for (int32_t m = 0; m < nm; ++m) mbar_init(&bars[m], 1);
    fence_barrier_init();
    for (int32_t m = 0; m < min(nm, kEarlyUnits); ++m) load_unit(m);
  }
  load_scan(0);
  if (kFp8 && warp == kFusedWarps - 1) {   // the quantised-unit barriers, a lane each
    for (int32_t q = lane; q < u1 - u0; q += kWarp) mbar_init(&qbars[q], 1);
    fence_barrier_init();
  }
  for (int i = tid; i < (1 + kRankWarps) * p.E; i += kThreads) s_P[i] = 0;   // s_P, s_cnt
  if (tid == 0) s_units_ok = 1;
  __syncthreads();
  // every thread's id loads are issued now: the rest of the pieces queue
  // behind them (issued any earlier, a piece could go out ahead of another
  // thread's ids and hold them back), landing while the ids are counted.
  // Lane m issues the warp's piece m: one thread's bulk copies are issued
  // one after another.
  if (lane >= min(nm, kEarlyUnits) && lane < nm) load_unit(lane);

  // ---- 1. per-expert counts of the ids before the own range, and the own ids
  {
    bool bad = false;
    auto count = [&](int32_t q, int64_t id) {
      int e = -1;
      if (id >= 0 && id < p.E) e = (int)id;
      else bad |= (id != -1);
      if (q < own_lo) {
        if (e >= 0) atomicAdd(&s_P[e], 1);
      } else {
        s_own[q - own_lo] = e;
      }
    };
    for (int32_t base = 0; base < scan_hi; base += kPassIds) {
      if (base > 0) load_scan(base);
#pragma unroll
      for (int u = 0; u < kScanPairs; ++u) {
        const int32_t q = base + 2 * (tid + u * kThreads);
        if (q < scan_hi) count(q, vs[u].x);
        if (q + 1 < scan_hi) count(q + 1, vs[u].y);
      }
    }
    if (bad) set_status(p.status, EP_ERR_INVALID_ARG);
  }
  __syncthreads();

  // ---- 2. the rank warps rank the own slots among themselves (ballots), turn
  //      the per-warp counts into warp starts after the prefix and write the
  //      own rows; the FP8 unit warps meanwhile quantise (step 3)
  const int rw = warp - (kFusedWarps - kRankWarps);   // rank warp index (< 0: not one)
  if (rw >= 0) {
    constexpr int kRankThreads = kRankWarps * kWarp;
    const int rt = tid - (kFusedWarps - kRankWarps) * kWarp;
    const int per = ((own_n + kRankThreads - 1) / kRankThreads) * kWarp;
    int my_rank[kRankIdsPerLane];
#pragma unroll
    for (int u = 0; u < kRankIdsPerLane; ++u) {
      my_rank[u] = 0;
      if (u * kWarp < per) {
        const int q = rw * per + u * kWarp + lane;
        const int e = q < own_n ? s_own[q] : -1;
        const uint32_t peers = peers_mask(e, p.nbits);
        int r = 0;
        if (e >= 0) r = s_cnt[rw * p.E + e] + __popc(peers & lanemask_lt());
        __syncwarp();
        if (e >= 0 && (__ffs(peers) - 1) == lane) s_cnt[rw * p.E + e] += __popc(peers);
        __syncwarp();
        my_rank[u] = r;
      }
    }
    named_barrier_sync(2, kRankThreads);
    for (int e = rt; e < p.E; e += kRankThreads) {   // per-warp counts -> warp starts
      int run = s_P[e];
#pragma unroll
      for (int w = 0; w < kRankWarps; ++w) {
        const int c = s_cnt[w * p.E + e];
        s_cnt[w * p.E + e] = run;
        run += c;
      }
      if (totals) p.recv_count[e] = run;
    }
    named_barrier_sync(2, kRankThreads);
#pragma unroll
    for (int u = 0; u < kRankIdsPerLane; ++u) {
      if (u * kWarp < per) {
        const int q = rw * per + u * kWarp + lane;
        if (q < own_n) {
          const int e = s_own[q];
          int32_t f = -1;
          if (e >= 0) {
            const int64_t row = (int64_t)s_cnt[rw * p.E + e] + my_rank[u];
            if (row < p.seg_rows) f = (int32_t)((int64_t)e * p.seg_rows + row);
            else set_status(p.status, EP_ERR_CAPACITY);
          }
          s_f[q] = f;
          const int32_t g = ga + q / p.k;
          if ((int64_t)g * p.P >= u0) {   // this CTA holds the token's first piece
            p.combine_idx[own_lo + q] = f;
            if (f >= 0) p.src_info[f] = g;
          }
        }
      }
    }
    // FP8: the src_info writes are released to the unit warps' grid-barrier
    // arrival (barrier 3); the rows are complete for the store warps (barrier 2)
    if (kFp8) named_barrier_arrive(3, kThreads);
    named_barrier_sync(2, kRankThreads);
  }
  if (!kFp8) __syncthreads();   // bf16: every warp stores, with the rows

  // ---- 3. FP8: the unit warps quantise their units in place as they land
  //      (staging each token's scales row-major) and mark each one; the store
  //      warps issue each unit's k bulk stores as soon as it is marked.  bf16:
  //      every warp stores its units as they land.
  // A unit that never landed: report it, wait (bounded) for the loads still
  // in flight and release the store warps from unit m on.
  auto fail_from = [&](int32_t m) {
    set_status(p.status, EP_ERR_TIMEOUT);
    s_units_ok = 0;
    __syncwarp();
    if (lane == 0)
      for (int32_t r = m; r < nm; ++r) {
        mbar_wait_bounded(&bars[r], 0);
        if (kFp8) mbar_arrive(&qbars[warp + r * kOwnWarps]);
      }
  };
  const int64_t row_bytes = kFp8 ? (int64_t)p.H : (int64_t)p.H * 2;
  const int32_t n_own_units = u1 - u0;
  if (!kFp8 || warp < kQuantWarps) {
    for (int32_t m = 0; m < nm; ++m) {
      const bool landed = mbar_wait_bounded(&bars[m], 0);
      if (!__all_sync(0xffffffffu, landed)) {
        fail_from(m);
        break;
      }
      int32_t g;
      int pc;
      unit_of(m, &g, &pc);
      const int hc = min(p.Hp, p.H - pc * p.Hp);
      uint8_t* sl = unit_slot(m);
      if (kFp8) {
        uint8_t* srow = p.scale_rows + (int64_t)g * p.scale_row_bytes;
        constexpr int kSegs = kFusedPiece / 512;
        uint4 a[kSegs], b[kSegs];
#pragma unroll
        for (int sg = 0; sg < kSegs; ++sg) {
          const int c0 = sg * 512 + lane * 16;
          a[sg] = make_uint4(0, 0, 0, 0);
          b[sg] = a[sg];
          if (c0 < hc) {
            a[sg] = ld_shared_v4(sl + (size_t)c0 * 2);
            b[sg] = ld_shared_v4(sl + (size_t)c0 * 2 + 16);
          }
        }
        __syncwarp();   // every lane has read its bf16 before any E4M3 lands on top
#pragma unroll
        for (int sg = 0; sg < kSegs; ++sg) {
          const int c0 = sg * 512 + lane * 16;
          float sf;
          uint32_t su;
          const uint4 qv = quantize16<kMode>(a[sg], b[sg], &sf, &su);
          if (c0 < hc) {
            st_shared_v4(sl + c0, qv);
            if ((lane & 7) == 0) {
              const int blk = (pc * p.Hp + c0) >> 7;
              if (kEs == 4) reinterpret_cast<float*>(srow)[blk] = sf;
              else srow[blk] = (uint8_t)su;
            }
          }
        }
        fence_proxy_async_smem();   // the E4M3 piece is read by bulk stores
        __syncwarp();
        if (lane == 0) mbar_arrive(&qbars[warp + m * kOwnWarps]);
      } else if (lane < p.k) {
        const int32_t f = s_f[(g - ga) * p.k + lane];
        if (f >= 0)
          tma_store_1d(p.recv_x + f * row_bytes + (int64_t)pc * p.Hp * 2, sl, (uint32_t)hc * 2u);
        tma_commit();
      }
    }
  } else {
    // FP8 store warps: units in slot order, each once it is quantised.  A
    // warp takes G = 32 / k units at a time, one lane per (unit, slot): a
    // thread's bulk copies go out one after another, so the number of
    // issuing threads, not the warps, sets how many 1 KB pieces are in flight.
    const int G = kWarp / p.k;
    const int32_t gq = lane / p.k;   // this lane's unit within the group
    const int j = lane - gq * p.k;   // and its slot
    constexpr int kStoreWarps = kFusedWarps - kQuantWarps;
    for (int32_t qb = (warp - kQuantWarps) * G; qb < n_own_units; qb += kStoreWarps * G) {
      const int32_t q = qb + gq;
      const bool mine = gq < G && q < n_own_units;
      const bool ready = mine ? mbar_wait_bounded(&qbars[q], 0) : true;
      if (!__all_sync(0xffffffffu, ready)) {
        set_status(p.status, EP_ERR_TIMEOUT);
        break;
      }
      if (!s_units_ok) continue;
      if (mine) {
        const int32_t u = u0 + q;
        const int32_t g = u / p.P;
        const int pc = u - g * p.P;
        const int hc = min(p.Hp, p.H - pc * p.Hp);
        const int32_t f = s_f[(g - ga) * p.k + j];
        if (f >= 0)
          tma_store_1d(p.recv_x + f * row_bytes + (int64_t)pc * p.Hp,
                       slots + (size_t)q * p.slot_bytes, (uint32_t)hc);
        tma_commit();
      }
    }
  }

  // ---- 4. grid barrier, then the per-expert outputs of this CTA's experts
  //      e = cta + a * grid: layout_range and (FP8) the column-major scales.
  //      FP8: the unit warps do it while the store warps keep issuing;
  //      bf16: every warp, once its stores are issued.
  if (!kFp8 || warp < kQuantWarps) {
    constexpr int kGroup = kFp8 ? kQuantWarps * kWarp : kThreads;
    auto sync = [&]() {
      if (kFp8) named_barrier_sync(1, kGroup);
      else __syncthreads();
    };
    // the group's staged scales and (FP8: the rank warps arrive at barrier 3
    // once their src_info is written) every row source are out
    if (kFp8) named_barrier_sync(3, kThreads);
    else sync();
    if (tid == 0) {   // the group leader alone writes s_passed
      __threadfence();
      int passed = 1;
      if (atomicAdd(&p.ctl[kCtlArrive], 1u) >= (uint32_t)grid) {   // workspace not cleaned
        set_status(p.status, EP_ERR_STATE);
        passed = 0;
      }
      if (passed && !wait_count(&p.ctl[kCtlArrive], (uint32_t)grid)) {
        set_status(p.status, EP_ERR_TIMEOUT);
        passed = 0;
      }
      __threadfence();
      s_passed = passed;
    }
    sync();   // s_passed is read by the whole group
    if (s_passed) fused_expert_outputs<kFp8, kEs>(p, cta, grid, tid, kGroup, s_P, s_lo, sync);
  }
  // No early trigger of the dependent combine: its CTAs would be placed on
  // the SMs this kernel frees first, several to an SM, and its static split
  // of the tokens over them then runs unevenly (measured: decode step 89.4-
  // 90.3 us with the trigger here, 76.3-76.6 without).
  if (tid == 0) {   // the last CTA out resets the barrier
    const uint32_t d = atomicAdd(&p.ctl[kCtlExit], 1u);
    if (d == (uint32_t)grid - 1) {
      p.ctl[kCtlArrive] = 0;
      p.ctl[kCtlExit] = 0;
    }
  }
  tma_wait_all();   // the bulk stores have read their slots before the CTA leaves
}

static size_t fused_smem(const FusedParams& p) {
  const size_t tables = (size_t)p.E * (1 + kRankWarps) + 2 * (size_t)p.own_cap +
                        (size_t)p.nA * (p.R + 1);
  return (size_t)p.slot_area + kFusedBarBytes + tables * sizeof(int32_t);
}

// Geometry of the fused path, or false when the batch does not fit it.
static bool plan_fused(FusedParams& p, int grid) {
  if ((int64_t)p.T * p.k > kFusedMaxIds || p.T == 0) return false;
  if ((int64_t)p.T * ((p.H + kFusedPiece - 1) / kFusedPiece) * grid >= ((int64_t)1 << 32))
    return false;   // the kernel's unit-range arithmetic is 32-bit
  const int hp = std::min(p.H, kFusedPiece);
  p.Hp = hp;
  p.P = (p.H + hp - 1) / hp;
  const int64_t units = (int64_t)p.T * p.P;
  const int64_t per_cta = (units + grid - 1) / grid;
  // units per CTA: at most kFusedMaxPerWarp per unit-owning warp
  if (per_cta > (int64_t)(p.fp8 ? kQuantWarps : kFusedWarps) * kFusedMaxPerWarp) return false;
  p.n_units = (int32_t)units;
  p.slot_bytes = round128((uint32_t)hp * 2u);
  p.slot_area = (uint32_t)(per_cta * p.slot_bytes);
  const int64_t own_tokens = (per_cta + p.P - 1) / p.P + 1;
  const int64_t own = (own_tokens * p.k + kWarp - 1) / kWarp * kWarp;
  if (own > kMaxOwnIds) return false;
  p.own_cap = (int)own;
  p.nA = (p.E + grid - 1) / grid;
  if (p.nA > kFusedWarps * kWarp) return false;
  p.nbits = key_bits(p.E);
  return fused_smem(p) <= kFusedSmemCap;
}

// Returned by launch_fused when the grid cannot be co-resident (the caller
// then takes the multi-kernel path); never returned to a user.
constexpr int kFusedNotLaunched = -1;

// Whether one CTA of k_ll_fused<kMode> with the largest shared-memory size
// it is planned for fits on an SM of the current device (then any grid of at
// most one CTA per SM can be co-resident).  Cached per device.
template <int kMode>
static bool fused_fits_one_per_sm() {
  static std::mutex mu;
  static signed char cached[64] = {0};   // 0 unknown, 1 fits, -1 does not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_ll_fused<kMode>, kFusedWarps * kWarp,
                                                      kFusedSmemCap) != cudaSuccess) {
      cudaGetLastError();
      per_sm = 0;
    }
    cached[dev] = per_sm >= 1 ? 1 : -1;
  }
  return cached[dev] > 0;
}

// The kernel waits at a grid barrier, so it is launched cooperatively: the
// runtime starts it only with every CTA resident (while kernels on other
// streams hold SMs it waits for them instead of starting part of the grid),
// and refuses a grid that could never be co-resident; that refusal, or an
// occupancy check that fails, sends the call to the multi-kernel path.
template <int kMode>
static int launch_fused_t(const FusedParams& p, int grid, cudaStream_t stream) {
  {
    const int rc = ep_host::ensure_max_smem(reinterpret_cast<const void*>(k_ll_fused<kMode>), (int)kFusedSmemCap);
    if (rc != EP_OK) return rc;
  }
  if (grid > ep_host::num_sms() || !fused_fits_one_per_sm<kMode>()) return kFusedNotLaunched;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kFusedWarps * kWarp);
  cfg.dynamicSmemBytes = fused_smem(p);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_ll_fused<kMode>, p);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return kFusedNotLaunched;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  ep_host::count_launch();
  return EP_OK;
}

static int launch_fused(const FusedParams& p, int fp8_mode, int grid, cudaStream_t stream) {
  switch (fp8_mode) {
    case EP_FP8_NONE: return launch_fused_t<EP_FP8_NONE>(p, grid, stream);
    case EP_FP8_E4M3_F32_SCALE: return launch_fused_t<EP_FP8_E4M3_F32_SCALE>(p, grid, stream);
    case EP_FP8_E4M3_UE8M0: return launch_fused_t<EP_FP8_E4M3_UE8M0>(p, grid, stream);
  }
  return EP_ERR_INVALID_ARG;
}

}  // namespace ep

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
  const bool fp8 = fp8_mode != EP_FP8_NONE;
  if (!packed_recv_x || !packed_recv_src_info || !layout_range || !recv_count || !workspace ||
      (T_r > 0 && (!x || !topk_idx || !combine_idx)) || (fp8 && !packed_recv_scales))
    return EP_ERR_INVALID_ARG;
  if (!ep_host::aligned16(x) || !ep_host::aligned16(packed_recv_x) ||
      !ep_host::aligned16(workspace))
    return EP_ERR_INVALID_ARG;
  if (fp8_mode == EP_FP8_E4M3_F32_SCALE && reinterpret_cast<uintptr_t>(packed_recv_scales) % 4 != 0)
    return EP_ERR_INVALID_ARG;   // fp32 scales are stored as 4-byte words
  if (workspace_bytes < ep_workspace_size(R, T_r, k, E, H)) return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int es = fp8_mode == EP_FP8_E4M3_F32_SCALE ? 4 : 1;
  uint8_t* scale_rows = fp8 ? ep::scale_staging(workspace, R, T_r, k, E) : nullptr;

  // decode-size batches: one fused launch (layout + scatter + scales)
  const int grid = ep_host::grid_cap(1);   // one CTA per SM, all resident
  if (ep_host::aligned16(topk_idx) && (int64_t)R * T_r * k < INT32_MAX) {
    ep::FusedParams fp{};
    fp.x = static_cast<const uint8_t*>(x);
    fp.topk_idx = topk_idx;
    fp.R = R;
    fp.T_r = T_r;
    fp.H = H;
    fp.E = E;
    fp.k = k;
    fp.T = R * T_r;
    fp.n_ids = fp.T * k;
    fp.seg_rows = seg_rows;
    fp.recv_x = static_cast<uint8_t*>(packed_recv_x);
    fp.scales = packed_recv_scales;
    fp.src_info = packed_recv_src_info;
    fp.layout_range = layout_range;
    fp.recv_count = recv_count;
    fp.combine_idx = combine_idx;
    fp.scale_rows = scale_rows;
    fp.scale_row_bytes = fp8 ? ep::scale_row_bytes(H, es) : 0;
    fp.ctl = static_cast<uint32_t*>(workspace);
    fp.status = status;
    fp.fp8 = fp8;
    if (ep::plan_fused(fp, grid)) {
      rc = ep::launch_fused(fp, fp8_mode, grid, s);
      if (rc != ep::kFusedNotLaunched) return rc;
    }
  }

  // larger batches: multi-CTA look-back layout; the scatter follows as its
  // programmatic dependent launch, the scale columns as the scatter's.
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
  p.seg_rows = seg_rows;
  p.n_rows = (int64_t)E * seg_rows;
  p.recv_x = static_cast<uint8_t*>(packed_recv_x);
  p.combine_idx = combine_idx;
  if (fp8) {
    p.scale_rows = scale_rows;
    p.scale_row_bytes = ep::scale_row_bytes(H, es);
  }
  p.status = status;
  p.claim = static_cast<uint32_t*>(workspace) + ep::kCtlClaim;
  p.n_pad_items = 0;
  if (p.T == 0) return EP_OK;
  rc = ep::launch_scatter(p, fp8_mode, true, s);
  if (rc != EP_OK || !fp8) return rc;
  ep::ScaleColParams sp{};
  sp.scale_rows = p.scale_rows;
  sp.row_bytes = p.scale_row_bytes;
  sp.nb = H / ep::kFp8Block;
  sp.T = p.T;
  sp.seg_rows = seg_rows;
  sp.n_rows = (int64_t)E * seg_rows;
  sp.src_idx = packed_recv_src_info;
  sp.recv_count = recv_count;
  sp.out = packed_recv_scales;
  sp.quad = fp8_mode == EP_FP8_E4M3_UE8M0 && seg_rows % 4 == 0 &&
            (reinterpret_cast<uintptr_t>(packed_recv_scales) & 3) == 0;
  return ep::launch_scale_columns(sp, true, fp8_mode, s);
}
