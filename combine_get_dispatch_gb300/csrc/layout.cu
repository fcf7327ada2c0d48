// layout.cu -- routing layout: per-rank / per-expert counts, is_token_in_rank
// and the deterministic slot ranks, in ONE pass over topk_idx.
//
// get_dispatch_layout (llm-infra-atlas DeepEP article, §2.1) counts, per
// source rank, the tokens for every rank and the slots for every expert.
// The contiguous and packed layouts (§1.1, §1.2, §2.3) additionally need, for
// each slot, its position among the slots routed to the same expert -- the
// row offset the receiver uses.  That is a segmented exclusive scan over
// T*k ids with E buckets, done here as one kernel:
//   1. a CTA takes a chunk of tokens (claimed through an atomic ticket, so
//      chunks start in order and every wait below is on an earlier,
//      already-running CTA; in normal mode a rank that is a single chunk
//      waits for nobody, so its CTA index names it and its ids load at
//      once), ranks its ids per warp with equal-key lane masks built from
//      ballots (peers_mask) and reduces the per-warp counts in shared
//      memory; in normal mode (R <= 64) it also forms each token's
//      destination-rank mask, counts tokens per rank by a warp bit transpose
//      and writes the chunk's is_token_in_rank rows as 16-byte stores;
//   2. it publishes the chunk aggregate and looks back over the previous
//      chunks' published (aggregate | inclusive) words, kLookbackWindow at
//      a time, to get its exclusive prefix per expert (decoupled look-back);
//   3. it writes the per-slot results.
// Chunks hold 2048 ids, or 8192 in normal mode once 2048-id chunks would
// need more than one wave of a CTA per SM.
// Normal mode scans within each source rank (get_dispatch_layout is a
// per-rank operation).  Low-latency mode scans across all ranks in
// (rank, token, slot) order, which directly yields the packed row
// expert_prefix[i][e] + slot_rank (§1.2, §3.2), so ep_ll_dispatch needs no
// separate notify step -- the V2 design of §4.6 (counting fused into the
// dispatch launch, no CPU round trip).
//
// Every wait is bounded by kWaitNs of %globaltimer; on expiry the CTA
// records EP_ERR_TIMEOUT, treats the missing value as 0 and carries on, so
// no CTA can hang.  Look-back words carry a launch epoch, so the workspace
// needs no clearing between launches.

#include "ep_common.cuh"
#include "layout.cuh"

namespace ep {

constexpr int kIdsPerLane = 4;            // ids per thread per chunk (low latency; normal mode up
                                          // to one wave of chunks, see launch_layout)
constexpr int kMaxIdsPerLane = 16;        // normal mode, batches of more than a wave of chunks
constexpr int kLookbackWindow = 16;
constexpr int kSmallLLThreads = 256;       // low-latency batches up to kSmallLLMaxIds
constexpr int64_t kSmallLLMaxIds = 32768;

enum : uint32_t { kFlagAggregate = 1, kFlagInclusive = 2 };

__device__ __forceinline__ uint64_t pack_flag(uint32_t epoch, uint32_t kind, uint32_t value) {
  return ((uint64_t)((epoch << 2) | kind) << 32) | value;
}

// Wait (bounded) until a look-back word of this launch is published.  A wait
// gives up after kWaitNs, or at once when another CTA already gave up (the
// workspace's abort word), so a broken launch ends after one bound rather
// than one bound per predecessor.  Giving up records EP_ERR_TIMEOUT and
// counts the missing value as 0.
__device__ __forceinline__ uint64_t wait_flag(const uint64_t* addr, uint64_t f, uint32_t epoch,
                                              uint32_t* abort_word, int32_t* status) {
  const uint32_t tag_a = (epoch << 2) | kFlagAggregate;
  const uint32_t tag_i = (epoch << 2) | kFlagInclusive;
  uint32_t tag = (uint32_t)(f >> 32);
  if (tag == tag_a || tag == tag_i) return f;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (ld_relaxed_u32(abort_word) != 0u) break;
    __nanosleep(40);
    f = ld_relaxed_u64(addr);
    tag = (uint32_t)(f >> 32);
    if (tag == tag_a || tag == tag_i) return f;
    if (globaltimer_ns() - t0 > kWaitNs) {
      atomicExch(abort_word, 1u);
      break;
    }
  }
  set_status(status, EP_ERR_TIMEOUT);
  return pack_flag(epoch, kFlagAggregate, 0);
}

// The rank of expert e (e / E_l) by a multiply with el_magic = floor(2^32 /
// E_l) + 1, exact for 0 <= e < 2^32 / E_l (E_l <= 1024, e < 1024 here).
__device__ __forceinline__ int rank_of(int e, const LayoutParams& p) {
  return (int)(((uint64_t)(uint32_t)e * p.el_magic) >> 32);
}

// Transpose of a 32 x 32 bit matrix held one row per lane (lane i, bit j =
// entry (i, j)): on return lane j holds column j (bit i = entry (i, j)).
// Five exchange rounds, swapping the off-diagonal blocks of 16, 8, 4, 2 and
// 1 bits with the partner lane.
__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
  constexpr uint32_t kLeft[5] = {0x0000ffffu, 0x00ff00ffu, 0x0f0f0f0fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int r = 0; r < 5; ++r) {
    const int j = 16 >> r;
    const uint32_t m = kLeft[r];   // columns whose index has bit j clear
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
    x = (lane & j) ? ((x & ~m) | ((y & ~m) >> j)) : ((x & m) | ((y & m) << j));
  }
  return x;
}

template <bool kLL, int kLayoutThreads, int kIds>
__global__ void __launch_bounds__(kLayoutThreads, 1) k_layout(LayoutParams p) {
  constexpr int kLayoutWarps = kLayoutThreads / kWarp;
  constexpr int kMaxChunkIds = kLayoutThreads * kIds;
  static_assert(kMaxChunkIds % 2 == 0 && kLayoutWarps % 2 == 0, "s_mask must stay 8-byte aligned");
  extern __shared__ __align__(16) int32_t smem[];
  int32_t* s_ids = smem;                                  // [kMaxChunkIds]
  int32_t* s_cnt = s_ids + kMaxChunkIds;                  // [warps][E]
  int32_t* s_agg = s_cnt + kLayoutWarps * p.E;            // [V]
  int32_t* s_excl = s_agg + p.V;                          // [V]
  uint64_t* s_mask = reinterpret_cast<uint64_t*>(s_excl + p.V);   // [chunk_tokens] (8-byte aligned:
                                                                   // every count above is even)
  __shared__ uint32_t s_ticket, s_epoch;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nbits = key_bits(p.E);
  // normal mode with one chunk per rank: no chunk waits for another, so the
  // CTA index is the chunk (no ticket) and no look-back word is published
  const bool solo = !kLL && p.chunks_per_rank == 1;

  if (kLL || p.trigger_dependents) pdl_launch_dependents();   // the scatter may start loading x
  if (tid == 0 && !solo) {
    s_ticket = atomicAdd(&p.ctl[0], 1u);
    s_epoch = ld_relaxed_u32(&p.ctl[2]);
  }
  for (int v = tid; v < kLayoutWarps * p.E; v += kLayoutThreads) s_cnt[v] = 0;
  for (int v = p.E + tid; v < p.V; v += kLayoutThreads) s_agg[v] = 0;

  // chunk b: source rank i, tokens [t0, t0 + nt), ids [id_base, id_base + n)
  int i = 0, c = 0, t0 = 0, nt = 0, n = 0;
  int64_t id_base = 0;
  auto chunk_of = [&](uint32_t bb) {
    i = (int)bb / p.chunks_per_rank;
    c = (int)bb % p.chunks_per_rank;
    t0 = c * p.chunk_tokens;
    nt = max(0, min(p.chunk_tokens, p.T_r - t0));
    n = nt * p.k;
    id_base = ((int64_t)i * p.T_r + t0) * p.k;
  };
  // ---- 1. load the chunk's ids (validated) into shared memory; all loads
  //      of a thread are issued before the first is used
  auto load_ids = [&]() {
    int64_t ev[kIds];
#pragma unroll
    for (int u = 0; u < kIds; ++u) {
      const int q = tid + u * kLayoutThreads;
      ev[u] = q < n ? __ldg(&p.topk_idx[id_base + q]) : -1;
    }
    bool bad = false;
#pragma unroll
    for (int u = 0; u < kIds; ++u) {
      const int q = tid + u * kLayoutThreads;
      if (q < n) {
        const int64_t e = ev[u];
        int v = -1;
        if (e >= 0 && e < p.E) v = (int)e;
        else bad |= (e != -1);
        s_ids[q] = v;
      }
    }
    if (bad) set_status(p.status, EP_ERR_INVALID_ARG);
  };

  uint32_t b = blockIdx.x;
  uint32_t epoch = 0;
  if (solo) {   // the ids go out at once, ahead of the barrier
    chunk_of(b);
    load_ids();
    __syncthreads();
  } else {
    __syncthreads();
    b = s_ticket;
    epoch = s_epoch & 0x3fffffffu;
    if (b >= (uint32_t)p.num_chunks) {   // workspace not cleaned: give up loudly
      if (tid == 0) {
        atomicExch(&p.ctl[3], 1u);
        set_status(p.status, EP_ERR_STATE);
      }
      return;
    }
    chunk_of(b);
    load_ids();
    __syncthreads();
  }

  // ---- per-warp ranks: warp w owns a contiguous run of the chunk's ids
  const int per_warp = ((n + kLayoutThreads - 1) / kLayoutThreads) * kWarp;
  const int wbase = warp * per_warp;
  int my_rank[kIds];
#pragma unroll
  for (int u = 0; u < kIds; ++u) {
    my_rank[u] = 0;
    if (u * kWarp < per_warp) {
      const int q = wbase + u * kWarp + lane;
      const int e = (q < n) ? s_ids[q] : -1;
      const uint32_t peers = peers_mask(e, nbits);
      int r = 0;
      if (e >= 0) r = s_cnt[warp * p.E + e] + __popc(peers & lanemask_lt());
      __syncwarp();
      if (e >= 0 && (__ffs(peers) - 1) == lane) s_cnt[warp * p.E + e] += __popc(peers);
      __syncwarp();
      my_rank[u] = r;
    }
  }
  __syncthreads();

  // ---- chunk aggregate per expert; per-warp counts become warp offsets
  for (int e = tid; e < p.E; e += kLayoutThreads) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kLayoutWarps; ++w) {
      const int tmp = s_cnt[w * p.E + e];
      s_cnt[w * p.E + e] = run;
      run += tmp;
    }
    s_agg[e] = run;
  }
  // ---- normal mode: is_token_in_rank and tokens per destination rank
  if (!kLL && p.R <= 64) {
    // each token's destination ranks as a bit mask; the tokens per rank from
    // a bit transpose over 32 tokens at a time (a hot rank gets one shared
    // atomic per warp, not one per token); the chunk's is_token_in_rank rows
    // are one contiguous byte range, written with 16-byte stores below
    for (int base = warp * kWarp; base < nt; base += kLayoutThreads) {
      const int tt = base + lane;
      uint64_t m = 0;
      if (tt < nt) {
        for (int j = 0; j < p.k; ++j) {
          const int e = s_ids[tt * p.k + j];
          if (e >= 0) m |= 1ull << rank_of(e, p);
        }
        s_mask[tt] = m;
      }
      // lane r's column of the warp's 32 x R bit matrix: its tokens for rank r
      const uint32_t lo = transpose32((uint32_t)m, lane);
      if (lane < p.R && lo != 0u) atomicAdd(&s_agg[p.E + lane], __popc(lo));
      if (p.R > 32) {
        const uint32_t hi = transpose32((uint32_t)(m >> 32), lane);
        if (lane + 32 < p.R && hi != 0u) atomicAdd(&s_agg[p.E + 32 + lane], __popc(hi));
      }
    }
  } else if (!kLL) {
    for (int tt = tid; tt < nt; tt += kLayoutThreads) {
      const int32_t* te = s_ids + tt * p.k;
      uint8_t* row = p.is_token_in_rank + ((int64_t)i * p.T_r + t0 + tt) * p.R;
      int dst[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) dst[j] = (j < p.k && te[j] >= 0) ? rank_of(te[j], p) : -1;
      for (int r = 0; r < p.R; ++r) {
        bool hit = false;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) hit |= (dst[j] == r);
        row[r] = hit ? 1 : 0;
        if (hit) atomicAdd(&s_agg[p.E + r], 1);
      }
    }
  }
  __syncthreads();

  if (!kLL && p.R <= 64) {
    // is_token_in_rank rows [i][t0, t0 + nt): byte q is token q / R, rank q % R
    uint8_t* out = p.is_token_in_rank + ((int64_t)i * p.T_r + t0) * p.R;
    const int nbytes = nt * p.R;
    const int head = min(nbytes, (int)((16u - (uint32_t)(reinterpret_cast<uintptr_t>(out) & 15u)) & 15u));
    const int nbody = (nbytes - head) / 16;
    auto byte_at = [&](int q) -> uint32_t {
      const int tq = q / p.R;
      return (uint32_t)((s_mask[tq] >> (q - tq * p.R)) & 1ull);
    };
    if (tid < head) out[tid] = (uint8_t)byte_at(tid);
    for (int g = tid; g < nbody; g += kLayoutThreads) {
      const int q0 = head + g * 16;
      int tq = q0 / p.R;
      int r = q0 - tq * p.R;
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        w[u >> 2] |= (uint32_t)((s_mask[tq] >> r) & 1ull) << (8 * (u & 3));
        if (++r == p.R) {
          r = 0;
          ++tq;
        }
      }
      st_v4(out + q0, make_uint4(w[0], w[1], w[2], w[3]));
    }
    for (int q = head + nbody * 16 + tid; q < nbytes; q += kLayoutThreads) out[q] = (uint8_t)byte_at(q);
  }

  // ---- 2. publish the aggregate, look back for the exclusive prefix
  const int seq_first = kLL ? 0 : i * p.chunks_per_rank;
  uint64_t* F = p.flags;
  if (solo) {   // a chunk per rank: its prefix within the rank is 0, nobody reads its words
    for (int v = tid; v < p.V; v += kLayoutThreads) s_excl[v] = 0;
  } else if ((int)b == seq_first) {
    for (int v = tid; v < p.V; v += kLayoutThreads) {
      s_excl[v] = 0;
      st_relaxed_u64(&F[(size_t)b * p.V + v], pack_flag(epoch, kFlagInclusive, (uint32_t)s_agg[v]));
    }
  } else {
    for (int v = tid; v < p.V; v += kLayoutThreads)
      st_relaxed_u64(&F[(size_t)b * p.V + v], pack_flag(epoch, kFlagAggregate, (uint32_t)s_agg[v]));
    for (int v = tid; v < p.V; v += kLayoutThreads) {
      uint32_t excl = 0;
      int pp = (int)b - 1;
      bool done = false;
      while (!done && pp >= seq_first) {
        const int nw = min(kLookbackWindow, pp - seq_first + 1);
        uint64_t wv[kLookbackWindow];
#pragma unroll
        for (int q = 0; q < kLookbackWindow; ++q)
          if (q < nw) wv[q] = ld_relaxed_u64(&F[(size_t)(pp - q) * p.V + v]);
#pragma unroll
        for (int q = 0; q < kLookbackWindow; ++q) {
          if (q < nw && !done) {
            const uint64_t f =
                wait_flag(&F[(size_t)(pp - q) * p.V + v], wv[q], epoch, &p.ctl[3], p.status);
            excl += (uint32_t)f;
            if ((uint32_t)(f >> 32) == ((epoch << 2) | kFlagInclusive)) done = true;
          }
        }
        pp -= nw;
      }
      s_excl[v] = (int32_t)excl;
      st_relaxed_u64(&F[(size_t)b * p.V + v],
                     pack_flag(epoch, kFlagInclusive, excl + (uint32_t)s_agg[v]));
    }
  }
  __syncthreads();

  // ---- 3. per-slot outputs
#pragma unroll
  for (int u = 0; u < kIds; ++u) {
    if (u * kWarp < per_warp) {
      const int q = wbase + u * kWarp + lane;
      if (q < n) {
        const int e = s_ids[q];
        const int64_t pos = id_base + q;
        if (kLL) {
          int32_t out = -1;
          if (e >= 0) {
            const int64_t row = (int64_t)s_excl[e] + s_cnt[warp * p.E + e] + my_rank[u];
            if (row >= 0 && row < p.seg_rows) {
              const int64_t f = (int64_t)e * p.seg_rows + row;
              out = (int32_t)f;
              p.src_info[f] = i * p.T_r + t0 + q / p.k;
            } else {
              set_status(p.status, EP_ERR_CAPACITY);
            }
          }
          p.combine_idx[pos] = out;
        } else {
          p.slot_rank[pos] = (e >= 0) ? s_excl[e] + s_cnt[warp * p.E + e] + my_rank[u] : -1;
        }
      }
    }
  }
  if (kLL && p.chunks_per_rank == 1) {
    // the chunk is the whole rank: both ends of its range are known here
    for (int e = tid; e < p.E; e += kLayoutThreads) {
      const uint32_t lo = (uint32_t)s_excl[e];
      const uint32_t hi = lo + (uint32_t)s_agg[e];
      p.layout_range[(size_t)e * p.R + i] = ((int64_t)lo << 32) | (int64_t)(hi - lo);
      if (i == p.R - 1) p.recv_count[e] = (int32_t)hi;
    }
  } else if (kLL) {
    // rank boundaries for layout_range: the first chunk of rank i publishes
    // expert_prefix[i][e] (its exclusive prefix) as a tagged word; the last
    // chunk of rank i pairs it with its inclusive prefix.
    if (c == 0) {
      for (int e = tid; e < p.E; e += kLayoutThreads)
        st_relaxed_u64(&p.rank_start[(size_t)i * p.E + e],
                       pack_flag(epoch, kFlagInclusive, (uint32_t)s_excl[e]));
    }
    if (c == p.chunks_per_rank - 1) {
      for (int e = tid; e < p.E; e += kLayoutThreads) {
        const uint64_t* a = &p.rank_start[(size_t)i * p.E + e];
        const uint32_t lo =
            (uint32_t)wait_flag(a, ld_relaxed_u64(a), epoch, &p.ctl[3], p.status);
        const uint32_t hi = (uint32_t)(s_excl[e] + s_agg[e]);
        p.layout_range[(size_t)e * p.R + i] = ((int64_t)lo << 32) | (int64_t)(hi - lo);
        if (i == p.R - 1) p.recv_count[e] = (int32_t)hi;
      }
    }
  } else if (c == p.chunks_per_rank - 1) {     // last chunk of rank i: rank totals
    for (int e = tid; e < p.E; e += kLayoutThreads)
      p.num_tokens_per_expert[(size_t)i * p.E + e] = s_excl[e] + s_agg[e];
    for (int r = tid; r < p.R; r += kLayoutThreads)
      p.num_tokens_per_rank[(size_t)i * p.R + r] = s_excl[p.E + r] + s_agg[p.E + r];
  }

  // ---- the last CTA to finish resets the ticket state for the next launch
  //      (and, layout and notify fused, computes the notify tables: every
  //      other CTA's count rows are out before its arrival)
  __shared__ int s_last;
  __syncthreads();
  if (tid == 0) {
    // fused notify: the arrival releases this CTA's count rows (its threads
    // wrote them before the barrier above) and, for the last CTA, acquires
    // everyone else's before the reads below
    const uint32_t d = p.fuse_notify ? atom_add_acq_rel_u32(&p.ctl[1], 1u) : atomicAdd(&p.ctl[1], 1u);
    if (d >= (uint32_t)p.num_chunks) set_status(p.status, EP_ERR_STATE);   // not cleaned
    const bool last = d == (uint32_t)p.num_chunks - 1;
    if (last) {
      p.ctl[0] = 0;
      p.ctl[1] = 0;
      p.ctl[2] = ld_relaxed_u32(&p.ctl[2]) + 1;   // the next launch's epoch
      p.ctl[3] = 0;
    }
    s_last = last;
  }
  if (!kLL && p.fuse_notify) {
    __syncthreads();
    if (s_last) {   // smem is free now: aligned totals, then (if they fit) the staged counts
      const int e4 = (p.E + 3) & ~3;
      const bool staged = notify_stage_words(p.R, p.E) <= kNotifyStageMaxWords;
      notify_tables<true>(p.nt, tid, kLayoutThreads, smem, staged ? smem + e4 : nullptr);
    }
  }
}

// ------------------------------------------------------------------ host side

LayoutGeometry layout_geometry(int R, int T_r, int k, int E, int chunk_ids) {
  LayoutGeometry g;
  g.chunk_tokens = chunk_ids / k;
  g.chunks_per_rank = T_r > 0 ? (T_r + g.chunk_tokens - 1) / g.chunk_tokens : 1;
  g.num_chunks = (int64_t)R * g.chunks_per_rank;
  g.V = E + R;
  g.flags_offset = 256;
  g.rank_start_offset = g.flags_offset + (size_t)g.num_chunks * g.V * sizeof(uint64_t);
  g.bytes = (g.rank_start_offset + (size_t)R * E * sizeof(uint64_t) + 255) / 256 * 256;
  return g;
}

static bool small_ll(int R, int T_r, int k) {
  return (int64_t)R * T_r * k <= kSmallLLMaxIds;
}

size_t layout_region_bytes(int R, int T_r, int k, int E) {
  size_t b = layout_geometry(R, T_r, k, E, kNormalChunkIds).bytes;
  if (small_ll(R, T_r, k))
    b = std::max(b, layout_geometry(R, T_r, k, E, kSmallLLThreads * kIdsPerLane).bytes);
  return b;
}

template <bool kLL, int kThreads, int kIds>
static int launch_layout_t(LayoutParams p, void* ws, cudaStream_t stream) {
  char* base = static_cast<char*>(ws);
  const LayoutGeometry g = layout_geometry(p.R, p.T_r, p.k, p.E, kThreads * kIds);
  p.el_magic = (uint64_t)((1ull << 32) / (uint64_t)p.E_l) + 1;
  p.ctl = reinterpret_cast<uint32_t*>(base);
  p.flags = reinterpret_cast<uint64_t*>(base + g.flags_offset);
  p.rank_start = reinterpret_cast<uint64_t*>(base + g.rank_start_offset);
  p.chunk_tokens = g.chunk_tokens;
  p.chunks_per_rank = g.chunks_per_rank;
  p.num_chunks = (int)g.num_chunks;
  p.V = kLL ? p.E : p.E + p.R;
  // ids, per-warp counts, aggregates and prefixes, the token masks (normal
  // mode); the last CTA reuses it for the notify tables (normal mode, fused)
  auto smem_bytes = [](int E, int V, int chunk_tokens, int R, bool notify) {
    const size_t words = (size_t)kThreads * kIds + (size_t)(kThreads / kWarp) * E + 2 * (size_t)V;
    size_t b = sizeof(int32_t) * words + (kLL ? 0 : sizeof(uint64_t) * (size_t)chunk_tokens);
    const int64_t stage = notify_stage_words(R, E);
    if (notify && stage <= kNotifyStageMaxWords)
      b = std::max(b, sizeof(int32_t) * ((size_t)((E + 3) & ~3) + (size_t)stage));
    return b;
  };
  {
    const size_t cap = std::max(smem_bytes(kMaxE, kMaxE + kMaxR, kThreads * kIds, 1, false),
                                sizeof(int32_t) * ((size_t)kMaxE + kNotifyStageMaxWords));
    const int rc = ep_host::ensure_max_smem(reinterpret_cast<const void*>(k_layout<kLL, kThreads, kIds>), (int)cap);
    if (rc != EP_OK) return rc;
  }
  k_layout<kLL, kThreads, kIds><<<p.num_chunks, kThreads,
                            smem_bytes(p.E, p.V, p.chunk_tokens, p.R, !kLL && p.fuse_notify), stream>>>(p);
  ep_host::count_launch();
  return ep_host::check_launch();
}

int launch_layout(const LayoutParams& p, bool ll, void* ws, cudaStream_t stream) {
  constexpr int kThreads = kNormalChunkIds / kIdsPerLane;
  if (!ll) {
    // normal mode: chunks of 2048 ids while they fit in one wave (a CTA per
    // SM), else 8192 ids per chunk -- fewer, longer CTAs and a shorter
    // look-back chain instead of several waves of latency-bound ones
    const int64_t ids = (int64_t)p.R * p.T_r * p.k;
    if (ids <= (int64_t)ep_host::num_sms() * kNormalChunkIds)
      return launch_layout_t<false, kThreads, kIdsPerLane>(p, ws, stream);
    return launch_layout_t<false, kThreads, kMaxIdsPerLane>(p, ws, stream);
  }
  // decode-sized batches: smaller CTAs (they fit beside the scatter CTAs
  // that follow as a programmatic dependent launch), 1024 ids per chunk
  if (small_ll(p.R, p.T_r, p.k)) return launch_layout_t<true, kSmallLLThreads, kIdsPerLane>(p, ws, stream);
  return launch_layout_t<true, kThreads, kIdsPerLane>(p, ws, stream);
}

}  // namespace ep

int ep::layout_notify(const int64_t* topk_idx, int R, int T_r, int k, int E, int expert_alignment,
                      int64_t num_worst_tokens, int32_t* num_tokens_per_rank,
                      int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank, int32_t* slot_rank,
                      int32_t* rank_prefix_matrix, int32_t* expert_prefix,
                      int32_t* num_recv_tokens_per_expert, int64_t* psum, int64_t* host_recv_rows,
                      int timeout_ms, void* workspace, size_t workspace_bytes, int32_t* status,
                      cudaStream_t stream, bool trigger_dependents) {
  if (R <= 0 || R > ep::kMaxR || E <= 0 || E > ep::kMaxE || E % R != 0 || k <= 0 ||
      k > ep::kMaxK || T_r < 0 || expert_alignment <= 0)
    return EP_ERR_INVALID_ARG;
  if (!num_tokens_per_rank || !num_tokens_per_expert || !workspace || !rank_prefix_matrix ||
      !expert_prefix || !num_recv_tokens_per_expert || !psum ||
      (T_r > 0 && (!topk_idx || !is_token_in_rank || !slot_rank)))
    return EP_ERR_INVALID_ARG;
  if (workspace_bytes < ep::layout_geometry(R, T_r, k, E, ep::kNormalChunkIds).bytes)
    return EP_ERR_INVALID_ARG;
  ep::LayoutParams p{};
  p.topk_idx = topk_idx;
  p.R = R;
  p.T_r = T_r;
  p.k = k;
  p.E = E;
  p.E_l = E / R;
  p.num_tokens_per_rank = num_tokens_per_rank;
  p.num_tokens_per_expert = num_tokens_per_expert;
  p.is_token_in_rank = is_token_in_rank;
  p.slot_rank = slot_rank;
  p.status = status;
  p.fuse_notify = true;
  p.trigger_dependents = trigger_dependents;
  ep::NotifyParams& n = p.nt;
  n.num_tokens_per_rank = num_tokens_per_rank;
  n.num_tokens_per_expert = num_tokens_per_expert;
  n.R = R;
  n.E = E;
  n.E_l = E / R;
  n.expert_alignment = expert_alignment;
  n.num_worst_tokens = num_worst_tokens;
  n.rank_prefix_matrix = rank_prefix_matrix;
  n.expert_prefix = expert_prefix;
  n.num_recv_tokens_per_expert = num_recv_tokens_per_expert;
  n.psum = psum;
  n.status = status;
  const bool wait = host_recv_rows != nullptr && num_worst_tokens < 0;
  if (host_recv_rows != nullptr) {
    void* dev = nullptr;
    if (cudaHostGetDevicePointer(&dev, host_recv_rows, 0) != cudaSuccess) {
      cudaGetLastError();
      return EP_ERR_INVALID_ARG;
    }
    volatile int64_t* h = host_recv_rows;
    for (int r = 0; r < R; ++r) h[r] = -1;
    n.host_recv_rows = static_cast<int64_t*>(dev);
  }
  const int rc = ep::launch_layout(p, false, workspace, stream);
  if (rc != EP_OK || !wait) return rc;
  return ep_host_wait_counters(host_recv_rows, R, timeout_ms);
}

extern "C" int ep_layout_notify(const int64_t* topk_idx, int R, int T_r, int k, int E,
                                int expert_alignment, int64_t num_worst_tokens,
                                int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                                uint8_t* is_token_in_rank, int32_t* slot_rank,
                                int32_t* rank_prefix_matrix, int32_t* expert_prefix,
                                int32_t* num_recv_tokens_per_expert, int64_t* psum,
                                int64_t* host_recv_rows, int timeout_ms, void* workspace,
                                size_t workspace_bytes, int32_t* status, void* stream) {
  return ep::layout_notify(topk_idx, R, T_r, k, E, expert_alignment, num_worst_tokens,
                           num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
                           slot_rank, rank_prefix_matrix, expert_prefix,
                           num_recv_tokens_per_expert, psum, host_recv_rows, timeout_ms,
                           workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream),
                           false);
}

extern "C" int ep_get_dispatch_layout(const int64_t* topk_idx, int R, int T_r, int k, int E,
                                      int32_t* num_tokens_per_rank,
                                      int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                                      int32_t* slot_rank, void* workspace, size_t workspace_bytes,
                                      int32_t* status, void* stream) {
  if (R <= 0 || R > ep::kMaxR || E <= 0 || E > ep::kMaxE || E % R != 0 || k <= 0 ||
      k > ep::kMaxK || T_r < 0)
    return EP_ERR_INVALID_ARG;
  if (!num_tokens_per_rank || !num_tokens_per_expert || !workspace ||
      (T_r > 0 && (!topk_idx || !is_token_in_rank || !slot_rank)))
    return EP_ERR_INVALID_ARG;
  if (workspace_bytes < ep::layout_geometry(R, T_r, k, E, ep::kNormalChunkIds).bytes)
    return EP_ERR_INVALID_ARG;
  ep::LayoutParams p{};
  p.topk_idx = topk_idx;
  p.R = R;
  p.T_r = T_r;
  p.k = k;
  p.E = E;
  p.E_l = E / R;
  p.num_tokens_per_rank = num_tokens_per_rank;
  p.num_tokens_per_expert = num_tokens_per_expert;
  p.is_token_in_rank = is_token_in_rank;
  p.slot_rank = slot_rank;
  p.status = status;
  return ep::launch_layout(p, false, workspace, static_cast<cudaStream_t>(stream));
}
