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
// low-latency batches skip all of this: k_ll_fused (ll_fused.cu) does layout,
// scatter and scales in one launch.
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

#include "dispatch.cuh"

namespace ep {

// ------------------------------------------------------------------ warp pipeline

// One warp's TMA pipeline over a sequence of units; unit u is piece u % P of
// token u / P.  The sequence (UnitSeq below) starts with kSeqStatic units
// first + j * stride, and continues either the same way or, with a
// workspace counter, with units claimed in batches as the warp goes: SMs
// of a GB300 do not all stream at the same rate (a static split of the
// 152 SMs' work measured CTAs finishing between 0.62x and 1.0x of the
// slowest one's time), so a warp on a faster SM takes more units.
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
  int32_t first, stride, n_units;
  uint32_t* claim;   // workspace counter of dynamically claimed units, or null (static sequence)
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

constexpr int kSeqStatic = 4;    // units per warp assigned by index before any claim
constexpr int kClaimMax = 4;     // units per claim at most (with 1024-channel pieces: large
                                 // dispatch 1456-1457 us against 1464-1465 with 8, 1480
                                 // with 16; 2 overloads the counter, 1.80 ms)

// A warp's units at positions i, i + 1, i + 2 (warp-uniform; -1 = the
// sequence has ended) and where the later ones come from: the static units
// first + j * stride for j < kSeqStatic, then batches claimed from the
// workspace counter (unit = kSeqStatic * stride + counter value).  Claims
// are guided: a batch holds max(1, min(kClaimMax, remaining / (4 * stride)))
// units, so early claims are few and large and the last ones single units
// (the counter is not contended and the warps end together).  The next
// batch's claim goes out as soon as the current batch is taken, a whole
// batch ahead of its use.  Once a position is past the end every later one
// is too.
struct UnitSeq {
  int32_t u0, u1, u2;
  int32_t next;       // position of the next unit to bring in
  int32_t nb, ne;     // dynamic units [nb, ne) taken but not yet handed out
  uint32_t pend;      // lane 0: counter value returned by the claim in flight
  int32_t pend_n;     // size of that claim (0: none in flight)
  bool ended;

  __device__ __forceinline__ int32_t static_unit(const Pipe& q, int32_t j) const {
    const int64_t u = (int64_t)q.first + (int64_t)j * q.stride;
    return u < q.n_units ? (int32_t)u : -1;
  }
  __device__ __forceinline__ int64_t dyn_base(const Pipe& q) const {
    return (int64_t)kSeqStatic * q.stride;
  }
  // Issue a claim sized for `remaining` units left after the counter value seen.
  __device__ __forceinline__ void claim(const Pipe& q, int64_t remaining, int lane) {
    int64_t b = remaining / (4 * (int64_t)q.stride);
    b = b < 1 ? 1 : (b > kClaimMax ? kClaimMax : b);
    pend_n = (int32_t)b;
    if (lane == 0) pend = atomicAdd(q.claim, (uint32_t)b);
  }
  __device__ __forceinline__ int32_t take(const Pipe& q, int lane) {
    if (ended) return -1;
    if (next < kSeqStatic || q.claim == nullptr) {
      const int32_t u = static_unit(q, next++);
      if (u < 0) ended = true;
      return u;
    }
    ++next;
    if (nb >= ne) {   // the claimed batch: wait for it, and claim the following one
      const uint32_t c = __shfl_sync(0xffffffffu, pend, 0);
      const int64_t lo = dyn_base(q) + c;
      const int64_t hi = lo + pend_n;
      pend_n = 0;
      if (lo >= q.n_units) {
        ended = true;
        return -1;
      }
      nb = (int32_t)lo;
      ne = (int32_t)(hi < q.n_units ? hi : q.n_units);
      claim(q, q.n_units - hi, lane);
    }
    return nb++;
  }
  __device__ __forceinline__ void init(const Pipe& q, int lane) {
    next = 0;
    nb = ne = 0;
    pend = 0u;
    pend_n = 0;
    ended = false;
    u0 = take(q, lane);
    u1 = take(q, lane);
    u2 = take(q, lane);
    // the first batch is claimed now, kSeqStatic positions ahead of its use
    // (only if the static units are not already past the end)
    if (q.claim != nullptr && !ended) claim(q, q.n_units - dyn_base(q), lane);
  }
  // Lane 0 waits for a claim still in flight (the counter must have taken
  // every claim before the launch's last CTA resets it).
  __device__ __forceinline__ void settle(int lane) const {
    if (lane == 0 && pend_n > 0) asm volatile("" ::"r"(pend) : "memory");
  }
  // Move to the next position.
  __device__ __forceinline__ void shift(const Pipe& q, int lane) {
    u0 = u1;
    u1 = u2;
    u2 = take(q, lane);
  }
};

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

// Barrier set-up and the source loads of positions 0 and 1 (static units:
// they depend on nothing but x).
template <int kMode>
__device__ __forceinline__ void pipe_prologue(const Pipe& q, const UnitSeq& seq, int lane) {
  static_assert(PipeDepth<kMode>::kPrologue == 2, "loads run two positions ahead (UnitSeq holds three)");
  if (seq.u0 < 0) return;
  if (lane == 0) {
    for (int s = 0; s < PipeDepth<kMode>::NS; ++s) mbar_init(&q.bar[s], 1);
    fence_barrier_init();
    pipe_issue_load<kMode>(q, 0, cursor_at(q, seq.u0));
    if (seq.u1 >= 0) pipe_issue_load<kMode>(q, 1, cursor_at(q, seq.u1));
  }
  __syncwarp();
}

// Run the pipeline.  D supplies each unit's destinations in two stages so
// that their global loads are issued one / two units ahead of their use:
//   d.pre(g, lane)              first-level value for slot lane (lane < k)
//   d.fin(g, pc, lane, pre)     flat receive row of slot lane, or -1
template <int kMode, class D>
__device__ __forceinline__ void pipe_run(const Pipe& q, const D& d, int lane, UnitSeq& seq) {
  constexpr bool kFp8 = PipeDepth<kMode>::kFp8;
  constexpr int NS = PipeDepth<kMode>::NS;
  constexpr int NO = PipeDepth<kMode>::NO;
  constexpr int kEs = kMode == EP_FP8_E4M3_F32_SCALE ? 4 : 1;
  if (seq.u0 < 0) return;
  const int64_t row_bytes = kFp8 ? (int64_t)q.H : (int64_t)q.H * 2;
  int64_t pre_a = d.pre(seq.u0 / q.P, lane);
  int64_t pre_b = seq.u1 >= 0 ? d.pre(seq.u1 / q.P, lane) : -1;
  int32_t ld_i = seq.u1 >= 0 ? 2 : 1;   // positions whose loads are out (the prologue's)

  bool failed = false;
  int32_t i = 0;
  for (; seq.u0 >= 0; ++i) {
    const Cursor cur = cursor_at(q, seq.u0);
    const int hc = min(q.Hp, q.H - cur.pc * q.Hp);
    const int s = i % NS;
    const int32_t my_f = d.fin(cur.g, cur.pc, lane, pre_a);
    pre_a = pre_b;
    if (seq.u2 >= 0) pre_b = d.pre(seq.u2 / q.P, lane);
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
      // position i-1's stores have read their stage: refill it with position i+2
      if (lane == 0) {
        tma_commit();
        tma_wait_read<1>();
        if (seq.u2 >= 0) pipe_issue_load<kMode>(q, i + 2, cursor_at(q, seq.u2));
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
      // source stage s was fully read: refill it with position i+2
      if (lane == 0 && seq.u2 >= 0) pipe_issue_load<kMode>(q, i + 2, cursor_at(q, seq.u2));
      for (int j = 0; j < q.k; ++j) {
        const int32_t f = __shfl_sync(0xffffffffu, my_f, j);
        if (lane == 0 && f >= 0) tma_store_1d(q.recv_x + f * row_bytes + col, dst, (uint32_t)hc);
      }
      if (lane == 0) tma_commit();
    }
    if (seq.u2 >= 0) ld_i = i + 3;
    seq.shift(q, lane);
  }
  if (failed && lane == 0) {
    // drain (bounded) the loads this warp still has in flight
    for (int32_t r = i; r < ld_i; ++r) mbar_wait_bounded(&q.bar[r % NS], (uint32_t)((r / NS) & 1));
  }
  seq.settle(lane);
  if (lane == 0) tma_wait_all();
}

// Carve this warp's pipeline out of the CTA's shared memory; its units
// start with first, first + stride, ... (UnitSeq).
template <int kMode>
__device__ __forceinline__ Pipe make_pipe(uint8_t* smem, const ScatterParams& p, int warp,
                                          int32_t first, int32_t stride) {
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
  q.n_units = (int32_t)p.n_units;
  q.claim = p.claim;
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
  Pipe q = make_pipe<kMode>(smem, p, warp, gw, W);
  UnitSeq seq;
  seq.init(q, lane);
  pipe_prologue<kMode>(q, seq, lane);
  // low latency: combine_idx of the layout kernel is read from here on;
  // normal mode launched as a programmatic dependent of the layout + notify
  // kernel: the first x pieces went out above, the prefix tables are read
  // from here on (a no-op after an ordinary launch)
  pdl_wait();
  if (kLL) {
    pipe_run<kMode>(q, PackedDest{&p}, lane, seq);
  } else {
    pipe_run<kMode>(q, NormalDest{&p}, lane, seq);
    pad_fill(p, gw, W, lane);
  }
  if (p.claim != nullptr) {   // the last CTA out resets the claim counter for the next launch
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();   // every claim of this CTA is performed before its arrival
      const uint32_t d = atomicAdd(&p.claim[1], 1u);
      if (d >= gridDim.x) set_status(p.status, EP_ERR_STATE);   // workspace not cleaned
      if (d == gridDim.x - 1) {
        __threadfence();
        p.claim[0] = 0u;
        p.claim[1] = 0u;
      }
    }
  }
}

// ------------------------------------------------------------------ scale columns

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

// ue8m0, rows [row0, row0 + 4) of segment seg (row0 % 4 == 0), of which
// rows row0 + [lo, hi) hold tokens: the four rows' scale bytes of a block
// are adjacent in its column, so a full quad is one 4-byte store per block
// (a warp writes 128 consecutive bytes per instruction instead of 32); a
// partial quad at a segment edge writes its bytes one by one.
__device__ __forceinline__ void scale_quad_to_columns(const ScaleColParams& p, int64_t seg,
                                                      int64_t row0, int lo, int hi) {
  int64_t src[4];
  bool ok[4];
  bool full = lo == 0 && hi == 4;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    src[u] = (u >= lo && u < hi) ? __ldg(&p.src_idx[seg * p.seg_rows + row0 + u]) : -1;
    ok[u] = src[u] >= 0 && src[u] < p.T;
    full &= ok[u];
  }
  const int ngrp = p.row_bytes / 16;
  for (int g0 = 0; g0 < ngrp; g0 += 2) {
    uint4 v[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int gg = 0; gg < 2; ++gg)
        v[u][gg] = (ok[u] && g0 + gg < ngrp)
                       ? __ldg(reinterpret_cast<const uint4*>(p.scale_rows + src[u] * p.row_bytes) +
                               g0 + gg)
                       : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int gg = 0; gg < 2; ++gg) {
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int b = (g0 + gg) * 16 + t;
        if (b >= p.nb) break;
        uint32_t c[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t w = t < 4 ? v[u][gg].x : t < 8 ? v[u][gg].y : t < 12 ? v[u][gg].z : v[u][gg].w;
          c[u] = (w >> (8 * (t & 3))) & 0xffu;
        }
        const int64_t o = (seg * p.nb + b) * p.seg_rows + row0;
        uint8_t* out = static_cast<uint8_t*>(p.out);
        if (full) {
          *reinterpret_cast<uint32_t*>(out + o) = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (ok[u]) out[o + u] = (uint8_t)c[u];
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
      if (kEs == 1 && p.quad) {
        for (int64_t q = threadIdx.x; q * 4 < lim; q += kScaleColThreads)
          scale_quad_to_columns(p, e, q * 4, 0, (int)min((int64_t)4, lim - q * 4));
        continue;
      }
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
  __shared__ int32_t s_valid[kMaxE];      // quad mode: valid rows of every segment
  __shared__ int32_t s_warp[kScaleColThreads / kWarp];
  const bool quad = kEs == 1 && p.quad;   // s_base then counts 4-row quads
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
      if (quad) {
        s_valid[e] = cnt[u];
        const int64_t a = s_start[e];
        cnt[u] = cnt[u] > 0 ? (int32_t)(((a + cnt[u] + 3) >> 2) - (a >> 2)) : 0;
      }
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
    if (quad) {   // quad f - s_base[lo] of the segment's quads
      const int64_t a = s_start[lo];
      const int64_t row0 = ((a >> 2) + (f - s_base[lo])) * 4;
      const int64_t b = a + s_valid[lo];
      scale_quad_to_columns(p, r, row0, (int)(max(a, row0) - row0), (int)(min(b, row0 + 4) - row0));
      continue;
    }
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
  } else {   // the valid rows are known only on the device: bounded by max_items
    const int64_t want = (p.max_items + kScaleColThreads - 1) / kScaleColThreads;
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

int launch_scale_columns(const ScaleColParams& p, bool ll, int fp8_mode, cudaStream_t s) {
  const bool f32 = fp8_mode == EP_FP8_E4M3_F32_SCALE;
  if (ll) return f32 ? launch_scale_columns_t<true, 4>(p, s) : launch_scale_columns_t<true, 1>(p, s);
  return f32 ? launch_scale_columns_t<false, 4>(p, s) : launch_scale_columns_t<false, 1>(p, s);
}

// ------------------------------------------------------------------ launch

// Small FP8 batches: pieces shrink (to kMinFp8Piece channels at the least)
// until every warp of the launch has about kMinUnitsPerWarp units.  The
// skewed workload (8192 tokens, H = 4096) gets 6.7 units per warp with the
// 2048-channel pieces that fit; measured in the timed step (L2 dirty after
// the flush): 1024-channel pieces (13.5 units per warp) made its dispatch
// 58.9 us instead of 61.4 (the scatter alone 52.2 instead of 53.3, the
// column pass behind it 6.7 instead of 8.1), 1408-channel ones (3 pieces,
// 10.1 units per warp: this rule) 57.5-58.0 against 59.2-59.5 for 1024 on
// another box, 768-channel ones were slower again.  Cold and serialised
// under ncu the smaller pieces are the slower ones: the gain is in the
// conditions of the step.
constexpr int kMinFp8Piece = 1024;
constexpr int kMinUnitsPerWarp = 10;
// Every other batch: pieces of at most kMaxPiece channels (1 KB E4M3 or 2 KB
// bf16 rows per bulk store): large dispatch 1464-1466 us against 1480-1483
// with the 1792-channel pieces that fit, prefill 644-646 against 653-655;
// 768-channel pieces were slower than either (interleaved A/B, three runs).
constexpr int kMaxPiece = 1024;

// Piece size, per-warp shared memory and warps per CTA: the largest piece
// (a multiple of the 16-byte / 128-channel granule) whose stages fit the
// per-warp share of `budget` for `target_warps` warps, then shrunk by the
// rules above (a small FP8 batch toward kMinUnitsPerWarp units per warp,
// any other batch to kMaxPiece channels).
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
  const int64_t warps = (int64_t)ep_host::grid_cap(1) * target_warps;
  if (fp8 && p.T * (int64_t)P < kMinUnitsPerWarp * warps) {
    while (hp > kMinFp8Piece && p.T * (int64_t)P < kMinUnitsPerWarp * warps) {
      ++P;
      hp = std::max(kMinFp8Piece, ((p.H + P - 1) / P + gran - 1) / gran * gran);
    }
  } else {
    while (hp > kMaxPiece) {
      ++P;
      hp = ((p.H + P - 1) / P + gran - 1) / gran * gran;
    }
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

// The scatter is persistent: one CTA per SM.  Launched as a programmatic
// dependent of the layout kernel, its shared-memory request is at least
// kScatterMinSmem, over half of an SM's, so that no SM holds two of its CTAs
// -- which the early launch would otherwise do while the layout's CTAs still
// hold other SMs (a small FP8 batch needs only ~100 KB; measured with two
// CTAs to an SM: the skewed single-call step 158.7 us instead of 152.6).  An
// ordinary launch starts on free SMs and is not padded (padded, the skewed
// dispatch took 60.1 us instead of 58.3).
constexpr size_t kScatterMinSmem = 120 * 1024;
static_assert(kScatterMinSmem <= kScatterSmemBudget, "the pad stays within the planned budget");

template <int kMode, bool kLL>
static int launch_scatter_t(ScatterParams p, cudaStream_t stream, bool pdl) {
  plan_pipeline(p, kMode, kMode == EP_FP8_NONE ? kBf16Warps : kFp8Warps, kScatterSmemBudget);
  p.n_units = p.T * p.P;
  if (p.n_units > INT32_MAX) return EP_ERR_INVALID_ARG;
  const size_t smem = std::max((size_t)p.warps_per_cta * p.warp_smem, pdl ? kScatterMinSmem : (size_t)0);
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
int launch_scatter(const ScatterParams& p, int fp8_mode, bool ll, cudaStream_t stream,
                   bool pdl_normal) {
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

int check_common(int R, int T_r, int H, int E, int k, int fp8_mode) {
  if (R <= 0 || R > kMaxR || E <= 0 || E > kMaxE || E % R != 0 || k <= 0 || k > kMaxK ||
      T_r < 0 || H <= 0 || H % 8 != 0)
    return EP_ERR_INVALID_ARG;
  if (fp8_mode < EP_FP8_NONE || fp8_mode > EP_FP8_E4M3_UE8M0) return EP_ERR_INVALID_ARG;
  if (fp8_mode != EP_FP8_NONE && H % kFp8Block != 0) return EP_ERR_INVALID_ARG;
  return EP_OK;
}

// Workspace: [layout kernel region][staged per-token FP8 scales][fused-path
// chunk flags and histograms]; the three never alias.
size_t staging_bytes(int R, int T_r, int H) {
  return ((size_t)R * T_r * scale_row_bytes(H, 4) + 255) / 256 * 256;
}

uint8_t* scale_staging(void* ws, int R, int T_r, int k, int E) {
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
  if (fp8_mode == EP_FP8_E4M3_F32_SCALE && reinterpret_cast<uintptr_t>(recv_scales) % 4 != 0)
    return EP_ERR_INVALID_ARG;   // fp32 scales are stored as 4-byte words
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
  p.claim = workspace != nullptr ? static_cast<uint32_t*>(workspace) + ep::kCtlClaim : nullptr;
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
  sp.quad = fp8_mode == EP_FP8_E4M3_UE8M0 && cap_rows % 4 == 0 &&
            (reinterpret_cast<uintptr_t>(recv_scales) & 3) == 0;
  sp.tables_after_wait = pdl;
  // at most T * k valid rows; a segment's quads cover its rows plus at most
  // one partial quad at each end
  sp.max_items = sp.quad ? (p.T * k + 3) / 4 + 2 * (int64_t)E : p.T * k;
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
  // the dispatch's own argument checks, before anything is launched
  const bool fp8 = fp8_mode != EP_FP8_NONE;
  if (cap_rows < 0 || (int64_t)R * cap_rows > INT32_MAX || !recv_src_idx ||
      (T_r > 0 && (!x || !combine_idx)) || (cap_rows > 0 && !recv_x) ||
      (fp8 && cap_rows > 0 && !recv_scales) || !ep_host::aligned16(x) ||
      !ep_host::aligned16(recv_x) || !ep_host::aligned16(workspace) ||
      (fp8_mode == EP_FP8_E4M3_F32_SCALE && reinterpret_cast<uintptr_t>(recv_scales) % 4 != 0))
    return EP_ERR_INVALID_ARG;
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

