// layout.cuh -- parameters of the layout kernel (see layout.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "notify.cuh"

namespace ep {

struct LayoutParams {
  const int64_t* topk_idx;
  int R, T_r, k, E, E_l;
  uint64_t el_magic;   // floor(2^32 / E_l) + 1: rank of an expert by a multiply
  int chunk_tokens, chunks_per_rank, num_chunks, V;
  // normal-mode outputs (get_dispatch_layout)
  int32_t* num_tokens_per_rank;
  int32_t* num_tokens_per_expert;
  uint8_t* is_token_in_rank;
  int32_t* slot_rank;
  // low-latency outputs (packed rows)
  int32_t* combine_idx;
  int32_t* src_info;
  int32_t* recv_count;
  int64_t* layout_range;
  int64_t seg_rows;
  // workspace views
  uint32_t* ctl;        // [0] ticket, [1] finished CTAs, [2] launch epoch, [3] abort
  uint64_t* flags;      // [num_chunks][V] look-back words
  uint64_t* rank_start;  // [R][E] low-latency: tagged prefix at the start of each rank
  int32_t* status;
  // normal mode, layout and notify in one launch: the last CTA to finish
  // computes the notify tables from the count tables the CTAs wrote
  bool fuse_notify;
  NotifyParams nt;
  bool trigger_dependents;   // normal mode: a programmatic dependent scatter may launch early
};

struct LayoutGeometry {
  int chunk_tokens;
  int chunks_per_rank;
  int64_t num_chunks;
  int V;
  size_t flags_offset, rank_start_offset, bytes;
};

constexpr int kNormalChunkIds = 2048;   // ids per chunk (512 threads x 4); the layout's workspace
                                        // is sized for it (larger chunks need less)

LayoutGeometry layout_geometry(int R, int T_r, int k, int E, int chunk_ids);

// Workspace bytes the layout kernels use (the largest of their geometries).
size_t layout_region_bytes(int R, int T_r, int k, int E);





// Launch the layout kernel on workspace `ws` (normal: per-rank scan into
// p's normal outputs; ll: global scan into p's low-latency outputs).
int launch_layout(const LayoutParams& p, bool ll, void* ws, cudaStream_t stream);

// Layout and notify in one launch (ep_layout_notify); with
// trigger_dependents the next kernel, launched as a programmatic dependent,
// may start before this one ends (it must wait before reading the tables).
int layout_notify(const int64_t* topk_idx, int R, int T_r, int k, int E, int expert_alignment,
                  int64_t num_worst_tokens, int32_t* num_tokens_per_rank,
                  int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank, int32_t* slot_rank,
                  int32_t* rank_prefix_matrix, int32_t* expert_prefix,
                  int32_t* num_recv_tokens_per_expert, int64_t* psum, int64_t* host_recv_rows,
                  int timeout_ms, void* workspace, size_t workspace_bytes, int32_t* status,
                  cudaStream_t stream, bool trigger_dependents);

}  // namespace ep
