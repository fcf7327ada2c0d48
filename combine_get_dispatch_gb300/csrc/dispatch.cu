// dispatch.cu -- token scatter into the receive layouts, with optional fused
// FP8 E4M3 quantisation (llm-infra-atlas DeepEP article §1.1, §1.2, §2.3,
// §3.2, §4.3).
//
// Every emulated rank's receive buffer is a partition of this GPU's HBM, so
// the "put" of a token to expert e's rank is a store into that partition.
// The scatter is built on TMA bulk copies (cp.async.bulk): every warp runs
// its own pipeline over (token, row piece) units --
//   * lane 0 streams the source pieces global -> shared with bulk copies
//     that complete on per-stage mbarriers, units ahead of the one being
//     consumed (deep memory-level parallelism from one thread);
//   * bf16: the staged piece is written to its k destination rows straight
//     from shared memory by k bulk stores (no register traffic at all);
//   * FP8: the 32 lanes quantise the staged piece once (each lane owns 16
//     channels, a 128-channel scale block is 8 lanes, amax by a 3-step
//     shuffle reduction) into a staged E4M3 piece, which k bulk stores write.
// The destinations come from
//   normal mode:       psum[r][l] + expert_prefix[i][e] + slot_rank[i][t][j]
//                      (segment start + source-rank offset + position, the
//                      receiver address of §2.3 with V2's psum of §4.3)
//   low-latency mode:  combine_idx written by the layout kernel just before
//                      (packed row in (rank, token, slot) order, §1.2/§3.2)
// and are fetched one / two units ahead of their use.  The low-latency
// scatter is a programmatic dependent launch of the layout kernel: its first
// bulk loads of x are issued before it waits for the layout.  Decode-size
// low-latency batches skip all of this: k_ll_fused does layout, scatter and
// scales in one launch (see its comment).
//
// Scales.  The receive layout keeps them column-major ([segment][block][row],
// §1.2): one value per row and block at a stride of a whole column.  Stored
// from the token side that is one scattered 1- or 4-byte store per
// (destination row, block) -- measured ~20% of the FP8 dispatch time.  So
// the scatter writes each token's scales once, row-major, into the
// workspace, and k_scale_columns (a programmatic dependent of the scatter)
// gathers them into the column layout with stores coalesced along rows.
//
// FP8 arithmetic is exact IEEE: amax is floored at 1e-4, the scale and its
// inverse use correctly rounded division (__fdiv_rn), x * inv one rounded
// multiply (__fmul_rn), and the E4M3 conversion is CUDA's satfinite RNE
// intrinsic; ue8m0 scales are amax/448 rounded up to a power of two through
// the exponent bits, so x * 2^-p is exact.
//
// Every mbarrier wait is bounded (kWaitNs); on expiry the warp records
// EP_ERR_TIMEOUT, stops issuing work, waits (bounded) for its copies in
// flight and leaves.

#include "ep_common.cuh"
#include "layout.cuh"

namespace ep {

constexpr int kScatterMaxWarps = 16;
constexpr int kBf16Warps = 8;      // target warps per CTA, bf16 path
constexpr int kFp8Warps = 16;      // target warps per CTA, FP8 path
constexpr int kBf16Stages = 3;     // staged source pieces per warp (bf16 path)
constexpr int kFp8InStages = 2;    // staged source pieces per warp (FP8 path)
constexpr int kFp8OutStages = 2;   // staged E4M3 pieces per warp
constexpr size_t kScatterSmemBudget = 200 * 1024;
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
};

__host__ __device__ inline uint32_t round128(uint32_t v) { return (v + 127u) / 128u * 128u; }

// Bytes of one token's staged scales (16-byte rows).
__host__ __device__ inline int scale_row_bytes(int H, int elem) {
  return ((H / kFp8Block) * elem + 15) / 16 * 16;
}

// Quantise 16 channels (two 16-byte bf16 vectors) of this lane; amax is
// reduced over the 8 lanes sharing the 128-channel block.  Returns 16 E4M3
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
  amax = fmaxf(amax, 1e-4f);
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

// ------------------------------------------------------------------ warp pipeline

// One warp's TMA pipeline over its units u = first + i * stride (i < count);
// unit u is piece u % P of token u / P.  Units are walked with incremental
// (token, piece) cursors, so the loop does no integer division.
struct Pipe {
  uint8_t* s_in;            // [NS][in_bytes] staged bf16 source pieces
  uint8_t* s_out;           // [NO][out_bytes] staged E4M3 pieces
  uint64_t* bar;            // [NS] mbarriers of the source stages
  uint32_t in_bytes, out_bytes;
  int H, Hp, P, k;
  const uint8_t* x;
  uint8_t* recv_x;
  uint8_t* scale_rows;
  int scale_row_bytes;
  int32_t* status;
  int32_t first, stride, count;
  int32_t stride_g, stride_pc;   // stride / P, stride % P
};

struct Cursor {
  int32_t g, pc;
};

__device__ __forceinline__ Cursor cursor_at(const Pipe& q, int32_t u) {
  Cursor c;
  c.g = u / q.P;
  c.pc = u - c.g * q.P;
  return c;
}

__device__ __forceinline__ void cursor_next(const Pipe& q, Cursor& c) {
  c.g += q.stride_g;
  c.pc += q.stride_pc;
  if (c.pc >= q.P) {
    c.pc -= q.P;
    c.g += 1;
  }
}

template <int kMode>
struct PipeDepth {
  static constexpr bool kFp8 = kMode != EP_FP8_NONE;
  static constexpr int NS = kFp8 ? kFp8InStages : kBf16Stages;
  static constexpr int NO = kFp8 ? kFp8OutStages : 1;
  static constexpr int kPrologue = kFp8 ? NS : NS - 1;   // loads issued before the loop
};

// Lane 0: bulk-load unit i (at cursor c) into stage i % NS.
template <int kMode>
__device__ __forceinline__ void pipe_issue_load(const Pipe& q, int32_t i, const Cursor& c) {
  constexpr int NS = PipeDepth<kMode>::NS;
  const uint32_t bytes = (uint32_t)min(q.Hp, q.H - c.pc * q.Hp) * 2u;
  uint64_t* b = &q.bar[i % NS];
  mbar_arrive_expect_tx(b, bytes);
  tma_load_1d(q.s_in + (size_t)(i % NS) * q.in_bytes,
              q.x + (int64_t)c.g * q.H * 2 + (int64_t)c.pc * q.Hp * 2, bytes, b);
}

// Barrier set-up and the first source loads (they depend on nothing but x).
// Returns the cursor of the next unit to load.
template <int kMode>
__device__ __forceinline__ Cursor pipe_prologue(const Pipe& q, int lane) {
  Cursor c = cursor_at(q, q.first);
  if (q.count <= 0) return c;
  const int32_t pro = min((int32_t)PipeDepth<kMode>::kPrologue, q.count);
  if (lane == 0) {
    for (int s = 0; s < PipeDepth<kMode>::NS; ++s) mbar_init(&q.bar[s], 1);
    fence_barrier_init();
  }
  for (int32_t i = 0; i < pro; ++i) {
    if (lane == 0) pipe_issue_load<kMode>(q, i, c);
    cursor_next(q, c);
  }
  __syncwarp();
  return c;
}

// Run the pipeline.  D supplies each unit's destinations in two stages so
// that their global loads are issued one / two units ahead of their use:
//   d.pre(g, lane)              first-level value for slot lane (lane < k)
//   d.fin(g, pc, lane, pre)     flat receive row of slot lane, or -1
template <int kMode, class D>
__device__ __forceinline__ void pipe_run(const Pipe& q, const D& d, int lane, Cursor ld) {
  constexpr bool kFp8 = PipeDepth<kMode>::kFp8;
  constexpr int NS = PipeDepth<kMode>::NS;
  constexpr int NO = PipeDepth<kMode>::NO;
  constexpr int kEs = kMode == EP_FP8_E4M3_F32_SCALE ? 4 : 1;
  const int32_t n = q.count;
  if (n <= 0) return;
  const int64_t row_bytes = kFp8 ? (int64_t)q.H : (int64_t)q.H * 2;
  Cursor cur = cursor_at(q, q.first);
  Cursor c1 = cur, c2 = cur;
  cursor_next(q, c1);
  cursor_next(q, c2);
  cursor_next(q, c2);
  int64_t pre_a = d.pre(cur.g, lane);
  int64_t pre_b = n > 1 ? d.pre(c1.g, lane) : -1;
  int32_t ld_i = min((int32_t)PipeDepth<kMode>::kPrologue, n);   // next unit to load

  bool failed = false;
  int32_t i = 0;
  for (; i < n; ++i) {
    const int hc = min(q.Hp, q.H - cur.pc * q.Hp);
    const int s = i % NS;
    const int32_t my_f = d.fin(cur.g, cur.pc, lane, pre_a);
    pre_a = pre_b;
    if (i + 2 < n) pre_b = d.pre(c2.g, lane);
    const bool landed = mbar_wait_bounded(&q.bar[s], (uint32_t)((i / NS) & 1));
    if (!__all_sync(0xffffffffu, landed)) {   // warp-uniform decision
      set_status(q.status, EP_ERR_TIMEOUT);
      failed = true;
      break;
    }
    const int64_t col = (int64_t)cur.pc * q.Hp * (kFp8 ? 1 : 2);   // byte offset of the piece
    if (!kFp8) {
      const uint8_t* src = q.s_in + (size_t)s * q.in_bytes;
      for (int j = 0; j < q.k; ++j) {
        const int32_t f = __shfl_sync(0xffffffffu, my_f, j);
        if (lane == 0 && f >= 0) tma_store_1d(q.recv_x + f * row_bytes + col, src, (uint32_t)hc * 2u);
      }
      // unit i-1's stores have read their stage: refill it with unit i+NS-1
      if (lane == 0) {
        tma_commit();
        tma_wait_read<1>();
        if (ld_i < n) pipe_issue_load<kMode>(q, ld_i, ld);
      }
      if (ld_i < n) {
        ++ld_i;
        cursor_next(q, ld);
      }
      __syncwarp();
    } else {
      const int o = i % NO;
      if (lane == 0 && i >= NO) tma_wait_read<NO - 1>();   // out stage o is free again
      __syncwarp();
      const uint8_t* src = q.s_in + (size_t)s * q.in_bytes;
      uint8_t* dst = q.s_out + (size_t)o * q.out_bytes;
      uint8_t* srow = q.scale_rows + (int64_t)cur.g * q.scale_row_bytes;
      for (int c0 = lane * 16; c0 < ((hc + 511) / 512) * 512; c0 += 512) {
        const bool ok = c0 < hc;
        uint4 a = make_uint4(0, 0, 0, 0), b = a;
        if (ok) {
          a = ld_shared_v4(src + (size_t)c0 * 2);
          b = ld_shared_v4(src + (size_t)c0 * 2 + 16);
        }
        float sf;
        uint32_t su;
        const uint4 qv = quantize16<kMode>(a, b, &sf, &su);
        if (ok) {
          st_shared_v4(dst + c0, qv);
          if ((lane & 7) == 0) {   // the token's scale of this block, row-major staging
            const int blk = (cur.pc * q.Hp + c0) >> 7;
            if (kEs == 4) reinterpret_cast<float*>(srow)[blk] = sf;
            else srow[blk] = (uint8_t)su;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      // source stage s was fully read: refill it with unit i+NS
      if (lane == 0 && ld_i < n) pipe_issue_load<kMode>(q, ld_i, ld);
      if (ld_i < n) {
        ++ld_i;
        cursor_next(q, ld);
      }
      for (int j = 0; j < q.k; ++j) {
        const int32_t f = __shfl_sync(0xffffffffu, my_f, j);
        if (lane == 0 && f >= 0) tma_store_1d(q.recv_x + f * row_bytes + col, dst, (uint32_t)hc);
      }
      if (lane == 0) tma_commit();
    }
    cur = c1;
    c1 = c2;
    cursor_next(q, c2);
  }
  if (failed && lane == 0) {
    // drain (bounded) the loads this warp still has in flight
    for (int32_t r = i; r < ld_i; ++r) mbar_wait_bounded(&q.bar[r % NS], (uint32_t)((r / NS) & 1));
  }
  if (lane == 0) tma_wait_all();
}

// Carve this warp's pipeline out of the CTA's shared memory; units
// first, first + stride, ... (count of them).
template <int kMode>
__device__ __forceinline__ Pipe make_pipe(uint8_t* smem, const ScatterParams& p, int warp,
                                          int32_t first, int32_t stride, int32_t count) {
  Pipe q;
  uint8_t* ws = smem + (size_t)warp * p.warp_smem;
  q.s_in = ws;
  q.s_out = q.s_in + (size_t)PipeDepth<kMode>::NS * p.in_bytes;
  q.bar = reinterpret_cast<uint64_t*>(q.s_out + (size_t)PipeDepth<kMode>::NO * p.out_bytes);
  q.in_bytes = p.in_bytes;
  q.out_bytes = p.out_bytes;
  q.H = p.H;
  q.Hp = p.Hp;
  q.P = p.P;
  q.k = p.k;
  q.x = p.x;
  q.recv_x = p.recv_x;
  q.scale_rows = p.scale_rows;
  q.scale_row_bytes = p.scale_row_bytes;
  q.status = p.status;
  q.first = first;
  q.stride = stride;
  q.count = count;
  q.stride_g = stride / p.P;
  q.stride_pc = stride - q.stride_g * p.P;
  return q;
}

// ------------------------------------------------------------------ destinations

// Normal mode: e = topk_idx (first level), then segment start + source-rank
// offset + slot rank (second level); records combine_idx / recv_src_idx on
// the token's first piece.
struct NormalDest {
  const ScatterParams* p;
  __device__ __forceinline__ int64_t pre(int32_t g, int lane) const {
    return lane < p->k ? __ldg(&p->topk_idx[(int64_t)g * p->k + lane]) : -1;
  }
  __device__ __forceinline__ int32_t fin(int32_t g, int pc, int lane, int64_t e64) const {
    if (lane >= p->k) return -1;
    const int64_t pos = (int64_t)g * p->k + lane;
    int32_t f = -1;
    if (e64 >= 0 && e64 < p->E) {
      const int e = (int)e64;
      const int r = e / p->E_l;
      const int l = e - r * p->E_l;
      const int i = g / p->T_r;
      const int64_t row = __ldg(&p->psum[(int64_t)r * (p->E_l + 1) + l]) +
                          __ldg(&p->expert_prefix[(int64_t)i * p->E + e]) + __ldg(&p->slot_rank[pos]);
      if (row >= 0 && row < p->seg_rows) f = (int32_t)((int64_t)r * p->seg_rows + row);
      else set_status(p->status, EP_ERR_CAPACITY);
    } else if (e64 != -1) {
      set_status(p->status, EP_ERR_INVALID_ARG);
    }
    if (pc == 0) {
      p->combine_idx[pos] = f;
      if (f >= 0) p->recv_src_idx[f] = g;
    }
    return f;
  }
};

// Low-latency mode after the layout kernel: the packed row is combine_idx.
struct PackedDest {
  const ScatterParams* p;
  __device__ __forceinline__ int64_t pre(int32_t g, int lane) const {
    return lane < p->k ? (int64_t)p->combine_idx[(int64_t)g * p->k + lane] : -1;
  }
  __device__ __forceinline__ int32_t fin(int32_t, int, int lane, int64_t f) const {
    if (lane >= p->k) return -1;
    if (f < -1 || f >= p->n_rows) {   // never write outside the buffer
      set_status(p->status, EP_ERR_INVALID_ARG);
      return -1;
    }
    return (int32_t)f;
  }
};

// Normal mode: recv_src_idx = -1 on alignment padding and past the last row
// of every rank (work items spread over the warps gw, gw + W, ...).
__device__ __forceinline__ void pad_fill(const ScatterParams& p, int32_t gw, int32_t W, int lane) {
  const int n_seg_items = p.R * p.E_l;
  for (int64_t it = gw; it < p.n_pad_items; it += W) {
    int r;
    int64_t lo, hi;
    if (it < n_seg_items) {
      r = (int)(it / p.E_l);
      const int l = (int)(it - (int64_t)r * p.E_l);
      const int e = r * p.E_l + l;
      lo = p.psum[(int64_t)r * (p.E_l + 1) + l] + p.expert_prefix[(int64_t)p.R * p.E + e];
      hi = p.psum[(int64_t)r * (p.E_l + 1) + l + 1];
    } else {
      const int64_t c4 = it - n_seg_items;
      r = (int)(c4 / p.tail_chunks);
      const int64_t c = c4 - (int64_t)r * p.tail_chunks;
      lo = max(p.psum[(int64_t)r * (p.E_l + 1) + p.E_l], c * kPadChunkRows);
      hi = (c + 1) * kPadChunkRows;
    }
    hi = min(hi, p.seg_rows);
    lo = max(lo, (int64_t)0);
    for (int64_t row = lo + lane; row < hi; row += 32) p.recv_src_idx[(int64_t)r * p.seg_rows + row] = -1;
  }
}

template <int kMode, bool kLL>
__global__ void __launch_bounds__(kScatterMaxWarps * kWarp) k_scatter(ScatterParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (kMode != EP_FP8_NONE) pdl_launch_dependents();   // the scale-column pass may launch
  const int32_t gw = blockIdx.x * p.warps_per_cta + warp;
  const int32_t W = gridDim.x * p.warps_per_cta;
  const int32_t n_units = (int32_t)p.n_units;
  const int32_t count = gw < n_units ? (n_units - gw + W - 1) / W : 0;
  Pipe q = make_pipe<kMode>(smem, p, warp, gw, W, count);
  const Cursor ld = pipe_prologue<kMode>(q, lane);
  if (kLL) {
    pdl_wait();   // combine_idx of the layout kernel is read from here on
    pipe_run<kMode>(q, PackedDest{&p}, lane, ld);
    return;
  }
  // launched as a programmatic dependent of the layout + notify kernel, the
  // first x pieces went out above; the prefix tables are read from here on
  // (a no-op after an ordinary launch)
  pdl_wait();
  pipe_run<kMode>(q, NormalDest{&p}, lane, ld);
  pad_fill(p, gw, W, lane);
}

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
// All CTAs are resident at once (one per SM, grid = SM count), so the wait
// at the grid barrier ends; every wait is bounded anyway and gives up with
// EP_ERR_TIMEOUT.

constexpr int kFusedWarps = 16;
constexpr int kQuantWarps = 12;          // FP8: warps owning (loading, quantising) units; the
                                         // other 4 issue the bulk stores as units are quantised
constexpr int kFusedMaxPerWarp = 8;      // units per warp
constexpr int kFusedPiece = 1024;        // channels per unit
constexpr int kEarlyUnits = 1;           // units per warp loaded with the ids; the rest once
                                         // the ids have landed
constexpr int kRankWarps = 4;            // the last warps: rank the CTA's own slots (FP8: the
                                         // store warps)
constexpr int kRankIdsPerLane = 8;
constexpr int kMaxOwnIds = kRankWarps * kWarp * kRankIdsPerLane;
constexpr int kScanIdsPerThread = 32;    // ids a thread has in flight per pass of the id scan
constexpr int kFusedMaxIds = 4 * kFusedWarps * kWarp * kScanIdsPerThread;   // at most 4 passes
constexpr int kFusedBarBytes = 2 * kFusedWarps * kFusedMaxPerWarp * 8;   // load + quantised barriers
constexpr size_t kFusedSmemCap = 225 * 1024;
static_assert(kRankWarps == kFusedWarps - kQuantWarps, "FP8: the rank warps are the store warps");
constexpr int kCtlArrive = 8;            // workspace control words of this kernel
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

  const int32_t U = p.n_units;
  const int32_t u0 = (int32_t)((int64_t)U * cta / grid);
  const int32_t u1 = (int32_t)((int64_t)U * (cta + 1) / grid);
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

  // ---- 0. every id up to the end of the own range goes out first: the CTA
  //      counts the ids before its range itself (their per-expert counts are
  //      its prefix), so it waits for no other CTA.  Only kEarlyUnits pieces
  //      per warp follow them now: ~30 MB of reads in flight grid-wide would
  //      hold the ids back by microseconds.
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
  load_scan(0);
  auto load_unit = [&](int32_t m) {
    int32_t g;
    int pc;
    unit_of(m, &g, &pc);
    const uint32_t bytes = (uint32_t)min(p.Hp, p.H - pc * p.Hp) * 2u;
    mbar_arrive_expect_tx(&bars[m], bytes);
    tma_load_1d_hint(unit_slot(m), p.x + (int64_t)g * p.H * 2 + (int64_t)pc * p.Hp * 2, bytes, &bars[m],
                     l2_policy_evict_first());   // every token is read once
  };
  if (kFp8 && tid == kThreads - 1) {
    for (int32_t q = 0; q < u1 - u0; ++q) mbar_init(&qbars[q], 1);
    fence_barrier_init();
  }
  if (nm > 0 && lane == 0) {
    for (int32_t m = 0; m < nm; ++m) mbar_init(&bars[m], 1);
    fence_barrier_init();
    for (int32_t m = 0; m < min(nm, kEarlyUnits); ++m) load_unit(m);
  }
  for (int i = tid; i < (1 + kRankWarps) * p.E; i += kThreads) s_P[i] = 0;   // s_P, s_cnt
  if (tid == 0) s_units_ok = 1;
  __syncthreads();

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
  if (nm > 0 && lane == 0)   // the ids are in: the rest of the pieces may queue now
    for (int32_t m = min(nm, kEarlyUnits); m < nm; ++m) load_unit(m);

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
  __syncthreads();
  pdl_launch_dependents();   // a dependent combine may take its place as this drains
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

template <int kMode>
static int launch_fused_t(const FusedParams& p, int grid, cudaStream_t stream) {
  {
    const int rc = ep_host::ensure_max_smem(reinterpret_cast<const void*>(k_ll_fused<kMode>), (int)kFusedSmemCap);
    if (rc != EP_OK) return rc;
  }
  k_ll_fused<kMode><<<grid, kFusedWarps * kWarp, fused_smem(p), stream>>>(p);
  ep_host::count_launch();
  return ep_host::check_launch();
}

static int launch_fused(const FusedParams& p, int fp8_mode, int grid, cudaStream_t stream) {
  switch (fp8_mode) {
    case EP_FP8_NONE: return launch_fused_t<EP_FP8_NONE>(p, grid, stream);
    case EP_FP8_E4M3_F32_SCALE: return launch_fused_t<EP_FP8_E4M3_F32_SCALE>(p, grid, stream);
    case EP_FP8_E4M3_UE8M0: return launch_fused_t<EP_FP8_E4M3_UE8M0>(p, grid, stream);
  }
  return EP_ERR_INVALID_ARG;
}

// ------------------------------------------------------------------ scale columns

struct ScaleColParams {
  const uint8_t* scale_rows;   // [T][row_bytes] per-token scales
  int row_bytes, nb;
  int64_t T;
  int64_t seg_rows;
  int64_t n_rows;              // rows of the receive buffer (segments * seg_rows)
  const int32_t* src_idx;      // token of every receive row, -1 = none (normal mode)
  const int32_t* recv_count;   // low-latency mode: rows per expert segment (src_idx
                               // is only defined below it)
  const int64_t* psum;         // normal mode: [R][E_l + 1] segment starts
  const int32_t* expert_total; // normal mode: [E] rows of every expert (unaligned)
  int E, E_l;
  bool tables_after_wait;      // normal mode: the segment tables may still be in the making
                               // when this kernel starts (the scatter itself was a dependent
                               // launch of layout + notify): read them after the wait
  void* out;                   // column-major scales [segment][block][row]
};

constexpr int kScaleMaxGroups = 8;   // 16-byte groups of a staged scale row held at once

// One lane per receive row holding a token: it gathers that token's staged
// scales (16-byte loads, all issued before any store) and writes them down
// its column entries -- consecutive lanes write consecutive rows, so every
// store instruction is coalesced.
//   low-latency: one CTA per expert over its rows below recv_count;
//   normal: a flat index over the valid rows of all expert segments (a
//   segment's valid rows are its first expert_total[e] rows; the aligned
//   rest and the capacity tail hold no token), mapped to (segment, row) by
//   a binary search over the per-CTA prefix of the segment sizes, so skewed
//   routing (one expert with most rows) spreads over all CTAs and padding
//   rows cost nothing.
template <int kEs>
__device__ __forceinline__ void scale_row_to_columns(const ScaleColParams& p, int64_t seg,
                                                     int64_t row, int64_t src) {
  constexpr int kPer16 = 16 / kEs;   // scale values per 16-byte group
  const int ngrp = p.row_bytes / 16;
  const uint8_t* srow = p.scale_rows + src * p.row_bytes;
  for (int g0 = 0; g0 < ngrp; g0 += kScaleMaxGroups) {
    uint4 v[kScaleMaxGroups];
#pragma unroll
    for (int u = 0; u < kScaleMaxGroups; ++u)
      v[u] = g0 + u < ngrp ? __ldg(reinterpret_cast<const uint4*>(srow) + g0 + u)
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < kScaleMaxGroups; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int t = 0; t < kPer16; ++t) {
        const int b = (g0 + u) * kPer16 + t;
        if (b < p.nb) {
          const int64_t o = (seg * p.nb + b) * p.seg_rows + row;
          if (kEs == 4) static_cast<uint32_t*>(p.out)[o] = w[t];
          else static_cast<uint8_t*>(p.out)[o] = (uint8_t)(w[t >> 2] >> (8 * (t & 3)));
        }
      }
    }
  }
}

template <bool kLL, int kEs>
__global__ void __launch_bounds__(kScaleColThreads) k_scale_columns(ScaleColParams p) {
  if (kLL) {
    pdl_wait();   // the scatter's staged scales and row sources
    const int64_t n_seg = p.n_rows / p.seg_rows;
    for (int64_t e = blockIdx.x; e < n_seg; e += gridDim.x) {   // one expert per CTA pass
      const int64_t lim = min((int64_t)max(__ldg(&p.recv_count[e]), 0), p.seg_rows);
      for (int64_t row = threadIdx.x; row < lim; row += kScaleColThreads) {
        const int64_t f = e * p.seg_rows + row;
        const int64_t src = __ldg(&p.src_idx[f]);
        if (src >= 0 && src < p.T) scale_row_to_columns<kEs>(p, e, row, src);
      }
    }
    return;
  }
  if (p.tables_after_wait) pdl_wait();
  __shared__ int32_t s_base[kMaxE + 1];   // exclusive prefix of the valid rows per segment
  __shared__ int32_t s_start[kMaxE];      // first row of every segment in its rank
  __shared__ int32_t s_warp[kScaleColThreads / kWarp];
  constexpr int kPer = (kMaxE + kScaleColThreads - 1) / kScaleColThreads;
  const int tid = threadIdx.x;
  int32_t cnt[kPer];
  int32_t sum = 0;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid * kPer + u;
    cnt[u] = 0;
    if (e < p.E) {
      const int r = e / p.E_l;
      const int64_t start = __ldg(&p.psum[(size_t)r * (p.E_l + 1) + (e - r * p.E_l)]);
      const int64_t room = max((int64_t)0, p.seg_rows - start);
      cnt[u] = (int32_t)min((int64_t)max(__ldg(&p.expert_total[e]), 0), room);
      s_start[e] = (int32_t)min(start, p.seg_rows);
    }
    sum += cnt[u];
  }
  // block-wide exclusive scan of the per-thread sums
  const int lane = tid & 31, warp = tid >> 5;
  int32_t incl = sum;
#pragma unroll
  for (int off = 1; off < kWarp; off <<= 1) {
    const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == kWarp - 1) s_warp[warp] = incl;
  __syncthreads();
  int32_t before = 0;
  for (int w = 0; w < warp; ++w) before += s_warp[w];
  int32_t run = before + incl - sum;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = tid * kPer + u;
    if (e < p.E) s_base[e] = run;
    run += cnt[u];
  }
  if (tid == kScaleColThreads - 1) s_base[p.E] = run;   // the last thread holds the total
  __syncthreads();
  // the segment tables come from notify, complete before the scatter began
  // (unless tables_after_wait); the staged scales and row sources need the
  // scatter itself
  if (!p.tables_after_wait) pdl_wait();
  const int32_t total = s_base[p.E];
  for (int32_t f = blockIdx.x * kScaleColThreads + tid; f < total;
       f += gridDim.x * kScaleColThreads) {
    int lo = 0, hi = p.E;   // the segment e with s_base[e] <= f < s_base[e + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_base[mid] <= f) lo = mid;
      else hi = mid;
    }
    const int r = lo / p.E_l;
    const int64_t row = (int64_t)s_start[lo] + (f - s_base[lo]);
    const int64_t src = __ldg(&p.src_idx[(int64_t)r * p.seg_rows + row]);
    if (src >= 0 && src < p.T) scale_row_to_columns<kEs>(p, r, row, src);
  }
}

template <bool kLL, int kEs>
static int launch_scale_columns_t(const ScaleColParams& p, cudaStream_t stream) {
  dim3 grid;
  if (kLL) {
    grid = dim3((unsigned)std::min<int64_t>(p.n_rows / p.seg_rows, ep_host::grid_cap(8)));
  } else {   // the valid rows are known only on the device: at most T * k
    const int64_t want = (p.T * 16 + kScaleColThreads - 1) / kScaleColThreads;
    grid = dim3((unsigned)std::max<int64_t>(
        1, std::min<int64_t>(want, (int64_t)ep_host::grid_cap(8))));
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kScaleColThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k_scale_columns<kLL, kEs>, p) != cudaSuccess) {
    cudaGetLastError();
    return EP_ERR_CUDA;
  }
  ep_host::count_launch();
  return ep_host::check_launch();
}

static int launch_scale_columns(const ScaleColParams& p, bool ll, int fp8_mode, cudaStream_t s) {
  const bool f32 = fp8_mode == EP_FP8_E4M3_F32_SCALE;
  if (ll) return f32 ? launch_scale_columns_t<true, 4>(p, s) : launch_scale_columns_t<true, 1>(p, s);
  return f32 ? launch_scale_columns_t<false, 4>(p, s) : launch_scale_columns_t<false, 1>(p, s);
}

// ------------------------------------------------------------------ launch

// Piece size, per-warp shared memory and warps per CTA: the largest piece
// (a multiple of the 16-byte / 128-channel granule) whose stages fit the
// per-warp share of `budget` for `target_warps` warps.
static void plan_pipeline(ScatterParams& p, int fp8_mode, int target_warps, size_t budget) {
  const bool fp8 = fp8_mode != EP_FP8_NONE;
  const int gran = fp8 ? kFp8Block : 8;
  const int ns = fp8 ? kFp8InStages : kBf16Stages;
  const int no = fp8 ? kFp8OutStages : 1;
  auto warp_bytes = [&](int hp, uint32_t* in_b, uint32_t* out_b) {
    *in_b = round128((uint32_t)hp * 2u);
    *out_b = fp8 ? round128((uint32_t)hp) : 0u;
    return (size_t)ns * *in_b + (size_t)no * *out_b + 128;
  };
  const size_t per_warp = budget / (size_t)target_warps;
  uint32_t in_b, out_b;
  int P = 1;
  int hp = p.H;
  while (hp > gran && warp_bytes(hp, &in_b, &out_b) > per_warp) {
    ++P;
    hp = ((p.H + P - 1) / P + gran - 1) / gran * gran;
  }
  P = (p.H + hp - 1) / hp;
  const size_t wb = warp_bytes(hp, &in_b, &out_b);
  p.Hp = hp;
  p.P = P;
  p.in_bytes = in_b;
  p.out_bytes = out_b;
  p.warp_smem = (uint32_t)wb;
  p.warps_per_cta = (int)std::max<size_t>(1, std::min<size_t>((size_t)kScatterMaxWarps, budget / wb));
}

template <int kMode, bool kLL>
static int launch_scatter_t(ScatterParams p, cudaStream_t stream, bool pdl) {
  plan_pipeline(p, kMode, kMode == EP_FP8_NONE ? kBf16Warps : kFp8Warps, kScatterSmemBudget);
  p.n_units = p.T * p.P;
  if (p.n_units > INT32_MAX) return EP_ERR_INVALID_ARG;
  const size_t smem = (size_t)p.warps_per_cta * p.warp_smem;
  {
    const int rc = ep_host::ensure_max_smem(reinterpret_cast<const void*>(k_scatter<kMode, kLL>), (int)kScatterSmemBudget + 1024);
    if (rc != EP_OK) return rc;
  }
  const int64_t work = std::max<int64_t>(p.n_units, p.n_pad_items);
  const int64_t want = (work + p.warps_per_cta - 1) / p.warps_per_cta;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)ep_host::grid_cap(1)));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(p.warps_per_cta * kWarp);
  cfg.dynamicSmemBytes = smem;
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

// Normal mode: pdl when the previous kernel on the stream is this library's
// layout + notify kernel launched to trigger it (its x loads then overlap
// the layout); low-latency mode always follows its layout kernel that way.
static int launch_scatter(const ScatterParams& p, int fp8_mode, bool ll, cudaStream_t stream,
                          bool pdl_normal = false) {
  switch (fp8_mode * 2 + (ll ? 1 : 0)) {
    case 0: return launch_scatter_t<EP_FP8_NONE, false>(p, stream, pdl_normal);
    case 1: return launch_scatter_t<EP_FP8_NONE, true>(p, stream, true);
    case 2: return launch_scatter_t<EP_FP8_E4M3_F32_SCALE, false>(p, stream, pdl_normal);
    case 3: return launch_scatter_t<EP_FP8_E4M3_F32_SCALE, true>(p, stream, true);
    case 4: return launch_scatter_t<EP_FP8_E4M3_UE8M0, false>(p, stream, pdl_normal);
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

// Workspace: [layout kernel region][staged per-token FP8 scales][fused-path
// chunk flags and histograms]; the three never alias.
static size_t staging_bytes(int R, int T_r, int H) {
  return ((size_t)R * T_r * scale_row_bytes(H, 4) + 255) / 256 * 256;
}

static uint8_t* scale_staging(void* ws, int R, int T_r, int k, int E) {
  return static_cast<uint8_t*>(ws) + layout_region_bytes(R, T_r, k, E);
}

}  // namespace ep

extern "C" size_t ep_workspace_size(int R, int T_r, int k, int E, int H) {
  if (R <= 0 || k <= 0 || k > ep::kMaxK || E <= 0 || T_r < 0 || H <= 0) return 0;
  return ep::layout_region_bytes(R, T_r, k, E) + ep::staging_bytes(R, T_r, H);
}

static int dispatch_normal(const void* x, const int64_t* topk_idx, const int32_t* slot_rank,
                           const int32_t* expert_prefix, const int64_t* psum, int R, int T_r,
                           int H, int E, int k, int fp8_mode, int64_t cap_rows, void* recv_x,
                           void* recv_scales, int32_t* recv_src_idx, int32_t* combine_idx,
                           void* workspace, size_t workspace_bytes, int32_t* status,
                           void* stream, bool pdl) {
  int rc = ep::check_common(R, T_r, H, E, k, fp8_mode);
  if (rc != EP_OK) return rc;
  if (cap_rows < 0 || (int64_t)R * cap_rows > INT32_MAX) return EP_ERR_INVALID_ARG;
  const bool fp8 = fp8_mode != EP_FP8_NONE;
  if (!expert_prefix || !psum || !recv_src_idx ||
      (T_r > 0 && (!x || !topk_idx || !slot_rank || !combine_idx)) ||
      (cap_rows > 0 && !recv_x) || (fp8 && cap_rows > 0 && !recv_scales))
    return EP_ERR_INVALID_ARG;
  if (fp8 && (!workspace || workspace_bytes < ep_workspace_size(R, T_r, k, E, H)))
    return EP_ERR_INVALID_ARG;
  if (!ep_host::aligned16(x) || !ep_host::aligned16(recv_x) || !ep_host::aligned16(workspace))
    return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ep::ScatterParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.R = R;
  p.T_r = T_r;
  p.H = H;
  p.E = E;
  p.E_l = E / R;
  p.k = k;
  p.T = (int64_t)R * T_r;
  p.topk_idx = topk_idx;
  p.slot_rank = slot_rank;
  p.expert_prefix = expert_prefix;
  p.psum = psum;
  p.seg_rows = cap_rows;
  p.n_rows = (int64_t)R * cap_rows;
  p.recv_x = static_cast<uint8_t*>(recv_x);
  p.recv_src_idx = recv_src_idx;
  p.combine_idx = combine_idx;
  const int es = fp8_mode == EP_FP8_E4M3_F32_SCALE ? 4 : 1;
  if (fp8) {
    p.scale_rows = ep::scale_staging(workspace, R, T_r, k, E);
    p.scale_row_bytes = ep::scale_row_bytes(H, es);
  }
  p.status = status;
  p.tail_chunks = (int)((cap_rows + ep::kPadChunkRows - 1) / ep::kPadChunkRows);
  p.n_pad_items = (int64_t)R * p.E_l + (int64_t)R * p.tail_chunks;
  rc = ep::launch_scatter(p, fp8_mode, false, s, pdl);
  if (rc != EP_OK || !fp8 || cap_rows == 0) return rc;
  ep::ScaleColParams sp{};
  sp.scale_rows = p.scale_rows;
  sp.row_bytes = p.scale_row_bytes;
  sp.nb = H / ep::kFp8Block;
  sp.T = p.T;
  sp.seg_rows = cap_rows;
  sp.n_rows = (int64_t)R * cap_rows;
  sp.src_idx = recv_src_idx;
  sp.psum = psum;
  sp.expert_total = expert_prefix + (size_t)R * E;
  sp.E = E;
  sp.E_l = E / R;
  sp.out = recv_scales;
  sp.tables_after_wait = pdl;
  return ep::launch_scale_columns(sp, false, fp8_mode, s);
}

extern "C" int ep_dispatch(const void* x, const int64_t* topk_idx, const int32_t* slot_rank,
                           const int32_t* expert_prefix, const int64_t* psum, int R, int T_r,
                           int H, int E, int k, int fp8_mode, int64_t cap_rows, void* recv_x,
                           void* recv_scales, int32_t* recv_src_idx, int32_t* combine_idx,
                           void* workspace, size_t workspace_bytes, int32_t* status,
                           void* stream) {
  return dispatch_normal(x, topk_idx, slot_rank, expert_prefix, psum, R, T_r, H, E, k, fp8_mode,
                         cap_rows, recv_x, recv_scales, recv_src_idx, combine_idx, workspace,
                         workspace_bytes, status, stream, false);
}

extern "C" int ep_layout_notify_dispatch(
    const void* x, const int64_t* topk_idx, int R, int T_r, int H, int E, int k, int fp8_mode,
    int expert_alignment, int64_t num_worst_tokens, int64_t cap_rows, int32_t* num_tokens_per_rank,
    int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank, int32_t* slot_rank,
    int32_t* rank_prefix_matrix, int32_t* expert_prefix, int32_t* num_recv_tokens_per_expert,
    int64_t* psum, void* recv_x, void* recv_scales, int32_t* recv_src_idx, int32_t* combine_idx,
    void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  // fixed shape only: the receive buffers exist before the counts do
  if (num_worst_tokens < 0) return EP_ERR_INVALID_ARG;
  int rc = ep::check_common(R, T_r, H, E, k, fp8_mode);
  if (rc != EP_OK) return rc;
  if (workspace_bytes < ep_workspace_size(R, T_r, k, E, H)) return EP_ERR_INVALID_ARG;
  rc = ep::layout_notify(topk_idx, R, T_r, k, E, expert_alignment, num_worst_tokens,
                         num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank, slot_rank,
                         rank_prefix_matrix, expert_prefix, num_recv_tokens_per_expert, psum,
                         nullptr, 0, workspace, workspace_bytes, status,
                         static_cast<cudaStream_t>(stream), true);
  if (rc != EP_OK) return rc;
  return dispatch_normal(x, topk_idx, slot_rank, expert_prefix, psum, R, T_r, H, E, k, fp8_mode,
                         cap_rows, recv_x, recv_scales, recv_src_idx, combine_idx, workspace,
                         workspace_bytes, status, stream, true);
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
  const bool fp8 = fp8_mode != EP_FP8_NONE;
  if (!packed_recv_x || !packed_recv_src_info || !layout_range || !recv_count || !workspace ||
      (T_r > 0 && (!x || !topk_idx || !combine_idx)) || (fp8 && !packed_recv_scales))
    return EP_ERR_INVALID_ARG;
  if (!ep_host::aligned16(x) || !ep_host::aligned16(packed_recv_x) ||
      !ep_host::aligned16(workspace))
    return EP_ERR_INVALID_ARG;
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
    if (ep::plan_fused(fp, grid))
      return ep::launch_fused(fp, fp8_mode, grid, s);
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
  return ep::launch_scale_columns(sp, true, fp8_mode, s);
}
