/*
 * ep.h -- C ABI of libep: DeepEP-style MoE token dispatch and combine on one
 * GB300 (sm_103a), with R expert-parallel ranks emulated as partitions of the
 * GPU's own HBM (a "remote put" is a store into another partition).
 *
 * Citations name the llm-infra-atlas article on DeepEP
 * (llm-infra-atlas.github.io/moe/06_deepep/) and its sections:
 *   §1.1 normal mode, §1.2 low-latency mode, §2.1 get_dispatch_layout /
 *   notify_dispatch, §2.3 prefix matrix and handle, §3.2 low-latency routing,
 *   §4.3 EPHandle (psum_num_recv_tokens_per_expert), §4.6 V2 fused notify.
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers unless stated otherwise (the combines'
 *    `out` may be pinned host memory); the caller owns and allocates every
 *    buffer.  No entry point allocates memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is stream-ordered and asynchronous, except
 *    ep_notify_dispatch / ep_layout_notify when given host counters (they
 *    then wait on the host, bounded by timeout_ms), ep_read_status and
 *    ep_host_wait_counters.
 *  - Entry points: layout (ep_get_dispatch_layout, ..._no_alloc), notify
 *    (ep_notify_dispatch), both in one launch (ep_layout_notify), normal
 *    dispatch (ep_dispatch; fixed shape with layout + notify in one call:
 *    ep_layout_notify_dispatch) and combine (ep_combine), low-latency
 *    dispatch / combine (ep_ll_dispatch, ep_ll_combine, ep_clean_ll_buffer),
 *    the once-per-rank layout (ep_rank_ids, ep_rank_recv_topk,
 *    ep_rank_combine), the SM budget (ep_set_num_sms, ep_get_num_sms), the
 *    kernels' number formats (ep_format_e4m3, ep_format_bf16) and plumbing
 *    (ep_workspace_size, ep_read_status, ep_host_wait_counters,
 *    ep_launch_count, ep_error_string).
 *  - Return value: EP_OK, or the first argument / launch error found on the
 *    host (nothing was launched when a validation error is returned).
 *  - `status` (int32 device word, may be NULL): kernels record the first
 *    error they detect there (EP_ERR_INVALID_ARG for an expert id outside
 *    [-1, E), EP_ERR_CAPACITY for a row past the buffer, EP_ERR_TIMEOUT for a
 *    device wait that expired).  Kernels never trap; a bad slot is skipped.
 *    The caller zeroes the word and reads it back (ep_read_status).
 *  - Layouts are row-major, C-contiguous.  bf16 is IEEE bfloat16, FP8 is
 *    OCP E4M3 ("e4m3fn": max 448, no infinities).
 *  - Stacked rank dimension: x [R, T_r, H], topk_idx / topk_weights
 *    [R, T_r, k]; expert e lives on rank e / E_l as local expert e % E_l,
 *    E_l = E / R (§3.2).  Expert id -1 marks an unused slot.
 *  - Limits: 1 <= R <= 1024, E % R == 0, E <= 1024, 1 <= k <= 16,
 *    0 <= T_r, H % 8 == 0 (16-byte rows), H % 128 == 0 with FP8, x / recv /
 *    y / out 16-byte aligned.
 *  - Row order inside every expert segment is (source rank, token, slot)
 *    ascending, so every output is deterministic.
 */
#ifndef EP_H_
#define EP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return / status codes. */
#define EP_OK 0
#define EP_ERR_INVALID_ARG 1
#define EP_ERR_CAPACITY 2
#define EP_ERR_TIMEOUT 3
#define EP_ERR_CUDA 4
#define EP_ERR_STATE 5 /* workspace not cleaned (ep_clean_ll_buffer) */
#define EP_ERR_TOO_LARGE 6 /* problem exceeds ep_get_dispatch_layout_no_alloc's scratch */

/* FP8 modes of dispatch (§1.1 "FP8 dispatch, BF16 combine"; §1.2
 * round_scale / use_ue8m0).  Scales cover blocks of 128 channels and are
 * stored column-major (rows of one block adjacent), the layout §1.2 says
 * DeepEP uses to suit TMA.
 *   EP_FP8_E4M3_F32_SCALE: amax = max(max|x|, 1e-4), scale = amax/448
 *     stored as fp32 (x ~ q * scale), q = E4M3_satfinite(x * (448/amax)).
 *   EP_FP8_E4M3_UE8M0: amax/448 rounded up to a power of two 2^p, one uint8
 *     per block holding the biased exponent p + 127, q = E4M3(x * 2^-p). */
#define EP_FP8_NONE 0
#define EP_FP8_E4M3_F32_SCALE 1
#define EP_FP8_E4M3_UE8M0 2

/* Bytes of device workspace that ep_get_dispatch_layout, ep_dispatch and
 * ep_ll_dispatch need for problems up to (R, T_r, k, E, H); 0 for invalid
 * sizes.  The workspace holds the cross-block prefix (decoupled look-back)
 * state of the layout kernels, the per-token FP8 scales staged between the
 * scatter and the column-major scale pass, the grid-barrier words of the
 * single-launch low-latency path and the work counter that spreads the
 * scatter's (token, piece) units over the SMs as they finish.  It must be zeroed once with
 * ep_clean_ll_buffer before its first use, after which every call leaves it
 * ready for the next.  Calls that share one workspace must be ordered on
 * one stream (overlapping calls race).  16-byte aligned. */
size_t ep_workspace_size(int R, int T_r, int k, int E, int H);

/* get_dispatch_layout (§2.1; handle fields §2.3).  For every source rank i:
 *   num_tokens_per_rank   [R, R] int32: [i][r] = tokens of rank i that go to
 *                         rank r (counted once per token)
 *   num_tokens_per_expert [R, E] int32: [i][e] = slots of rank i routed to e
 *   is_token_in_rank      [R, T_r, R] uint8 (0/1)
 *   slot_rank             [R, T_r, k] int32: position of slot (t, j) among
 *                         rank i's slots routed to the same expert, in
 *                         (token, slot) order; -1 for an unused slot.
 * Invalid ids set EP_ERR_INVALID_ARG in *status and count as unused. */
int ep_get_dispatch_layout(const int64_t* topk_idx, int R, int T_r, int k, int E,
                           int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                           uint8_t* is_token_in_rank, int32_t* slot_rank,
                           void* workspace, size_t workspace_bytes, int32_t* status,
                           void* stream);

/* ep_get_dispatch_layout for callers that cannot allocate device memory
 * (allocator callbacks, runtimes that forbid the library any allocation).  No counterpart in the article: it is the same
 * layout computation, same arguments and outputs as ep_get_dispatch_layout
 * minus the workspace, which is replaced by a 4 MiB array inside libep
 * (held on every GPU that loads the library, until the process exits).
 *  - Returns EP_ERR_TOO_LARGE, launching nothing, when the problem's
 *    look-back state (the layout part of ep_workspace_size) exceeds the
 *    array: e.g. R=8, T_r=16384, k=8, E=256 fits.
 *  - Allocates nothing: no cudaMalloc / cudaFree, no allocating library call.
 *  - Every call shares the one array and clears the part it uses first
 *    (stream-ordered); calls that overlap on the GPU race, so order them on
 *    one stream.
 *  - The first call on a device looks up the array's address with that
 *    device current.  The address is kept until the process exits: do not use the library on a device
 *    after cudaDeviceReset on it.
 *  - `stream` must belong to the current device (NULL: the current
 *    device's default stream); a stream of another device returns
 *    EP_ERR_INVALID_ARG, launching nothing. */
int ep_get_dispatch_layout_no_alloc(const int64_t* topk_idx, int R, int T_r, int k, int E,
                                    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                                    uint8_t* is_token_in_rank, int32_t* slot_rank,
                                    int32_t* status, void* stream);

/* notify_dispatch (§2.1, §2.3, §4.3): the count exchange and prefix sums.
 *   rank_prefix_matrix [R, R] int32: [i][j] = sum_{i' <= i} num_tokens_per_rank[i'][j]
 *   expert_prefix [R + 1, E] int32: [i][e] = sum_{i' < i} num_tokens_per_expert[i'][e];
 *                 row R holds the totals (rows each expert receives)
 *   num_recv_tokens_per_expert [R, E_l] int32: totals aligned up to
 *                 expert_alignment (>= 1)
 *   psum [R, E_l + 1] int64: exclusive prefix of the aligned totals per
 *                 rank = start row of each local expert's segment; psum[r][E_l]
 *                 is rank r's receive row count.
 * num_worst_tokens >= 0 selects the fixed-shape mode (§2.1): a rank
 * receiving more tokens than that sets EP_ERR_CAPACITY, and no host wait is
 * done.  Otherwise, when host_recv_rows (HOST pointer to R int64 in pinned,
 * mapped memory, e.g. cudaHostAlloc(..., cudaHostAllocMapped)) is not NULL,
 * the call sets them to -1, launches, and spins on the host until the
 * kernel has written psum[r][E_l] into every one of them (the CPU handshake
 * of §2.1), returning EP_ERR_TIMEOUT after timeout_ms. */
int ep_notify_dispatch(const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_expert,
                       int R, int E, int expert_alignment, int64_t num_worst_tokens,
                       int32_t* rank_prefix_matrix, int32_t* expert_prefix,
                       int32_t* num_recv_tokens_per_expert, int64_t* psum,
                       int64_t* host_recv_rows, int timeout_ms, int32_t* status, void* stream);

/* get_dispatch_layout and notify_dispatch in ONE launch (the V2 design of
 * §4.6 folds notify into the dispatch-side grid): the layout kernel's last
 * CTA to finish computes the notify tables from the count tables the other
 * CTAs wrote.  Arguments, outputs, host handshake and errors are those of
 * ep_get_dispatch_layout followed by ep_notify_dispatch on the same
 * stream; the outputs are identical. */
int ep_layout_notify(const int64_t* topk_idx, int R, int T_r, int k, int E, int expert_alignment,
                     int64_t num_worst_tokens, int32_t* num_tokens_per_rank,
                     int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                     int32_t* slot_rank, int32_t* rank_prefix_matrix, int32_t* expert_prefix,
                     int32_t* num_recv_tokens_per_expert, int64_t* psum,
                     int64_t* host_recv_rows, int timeout_ms, void* workspace,
                     size_t workspace_bytes, int32_t* status, void* stream);

/* Fixed-shape normal mode (num_worst_tokens >= 0, cap_rows given) in ONE
 * call: ep_layout_notify, then ep_dispatch launched as its programmatic
 * dependent (the dispatch kernel's first token loads overlap the layout;
 * it waits for the prefix tables before placing any row).  Arguments and
 * outputs are those of the two calls; the results are identical.
 * EP_ERR_INVALID_ARG for num_worst_tokens < 0 (no host handshake here). */
int ep_layout_notify_dispatch(const void* x, const int64_t* topk_idx, int R, int T_r, int H, int E,
                              int k, int fp8_mode, int expert_alignment, int64_t num_worst_tokens,
                              int64_t cap_rows, int32_t* num_tokens_per_rank,
                              int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                              int32_t* slot_rank, int32_t* rank_prefix_matrix,
                              int32_t* expert_prefix, int32_t* num_recv_tokens_per_expert,
                              int64_t* psum, void* recv_x, void* recv_scales,
                              int32_t* recv_src_idx, int32_t* combine_idx, void* workspace,
                              size_t workspace_bytes, int32_t* status, void* stream);

/* Normal-mode dispatch into the contiguous per-expert layout (§1.1, §2.3,
 * §4.3).  Slot (i, t, j) with expert e = r*E_l + l is copied (or quantised)
 * into rank r's row psum[r][l] + expert_prefix[i][e] + slot_rank[i][t][j].
 *   x            [R, T_r, H] bf16
 *   recv_x       [R, cap_rows, H] bf16 (fp8_mode 0) or E4M3 bytes
 *   recv_scales  [R, H/128, cap_rows] fp32 (mode 1, 4-byte aligned) / uint8 (mode 2);
 *                NULL in mode 0
 *   recv_src_idx [R, cap_rows] int32: i*T_r + t for every filled row, -1 on
 *                alignment padding and past the last row
 *   combine_idx  [R, T_r, k] int32: r*cap_rows + row, -1 for an unused slot
 *   workspace    ep_workspace_size bytes (required when fp8_mode > 0, may be
 *                NULL for bf16: the scatter then splits its units statically
 *                over the CTAs, which is slower when SMs run at different
 *                speeds)
 * A row at or past cap_rows is not written (EP_ERR_CAPACITY, slot -1).
 * Rows of recv_x that no slot fills are left untouched; scale entries of
 * rows that hold no token are unspecified. */
int ep_dispatch(const void* x, const int64_t* topk_idx, const int32_t* slot_rank,
                const int32_t* expert_prefix, const int64_t* psum, int R, int T_r, int H,
                int E, int k, int fp8_mode, int64_t cap_rows, void* recv_x, void* recv_scales,
                int32_t* recv_src_idx, int32_t* combine_idx, void* workspace,
                size_t workspace_bytes, int32_t* status, void* stream);

/* Output of the combines (ep_combine, ep_ll_combine, ep_rank_combine): `out`
 * is device memory or pinned host memory (cudaHostAlloc, cudaHostRegister):
 * the kernel then writes the result straight across the host link, with no
 * separate copy.  Pageable host memory is refused (EP_ERR_INVALID_ARG,
 * nothing launched).  Every other buffer of every call is device memory. */

/* Normal-mode combine (§1.1, §2.3: dispatch walked backwards):
 *   out[i][t][:] = bf16_rn( fp32 fma chain over j = 0..k-1 of
 *                           topk_weights[i][t][j] * y[combine_idx[i][t][j]][:] )
 * starting from +0 and skipping slots with combine_idx -1.
 *   y [R, cap_rows, H] bf16 (expert outputs in the dispatch layout),
 *   topk_weights [R, T_r, k] fp32, combine_idx as returned by ep_dispatch,
 *   out [R, T_r, H] bf16. */
int ep_combine(const void* y, const float* topk_weights, const int32_t* combine_idx, int R,
               int T_r, int H, int k, int64_t cap_rows, void* out, int32_t* status,
               void* stream);

/* Low-latency dispatch into the packed masked layout (§1.2, §3.2), layout
 * computed inside the call (no host round trip; graph-capturable).  Expert
 * e = r*E_l + l owns rows [0, recv_count[r][l]) of packed_recv_x[r][l],
 * ordered by (source rank, token, slot); T_r <= max_tokens_per_rank.
 *   packed_recv_x        [R, E_l, R*max_tokens_per_rank, H] bf16 or E4M3
 *   packed_recv_scales   [R, E_l, H/128, R*max_tokens_per_rank] fp32 (4-byte
 *                        aligned) / uint8
 *   packed_recv_src_info [R, E_l, R*max_tokens_per_rank] int32: i*T_r + t
 *   layout_range         [R, E_l, R] int64: (offset << 32) | count of source
 *                        rank i's rows inside the segment
 *   recv_count           [R, E_l] int32 (the masked GEMM's masked_m)
 *   combine_idx          [R, T_r, k] int32: e*(R*max) + row, -1 if unused
 * Rows past recv_count are left untouched.  workspace: ep_workspace_size. */
int ep_ll_dispatch(const void* x, const int64_t* topk_idx, int R, int T_r, int H, int E, int k,
                   int max_tokens_per_rank, int fp8_mode, void* packed_recv_x,
                   void* packed_recv_scales, int32_t* packed_recv_src_info,
                   int64_t* layout_range, int32_t* recv_count, int32_t* combine_idx,
                   void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* Low-latency combine (§1.2): as ep_combine with y the packed layout
 * [R, E_l, R*max_tokens_per_rank, H] bf16 and combine_idx from
 * ep_ll_dispatch. */
int ep_ll_combine(const void* y, const float* topk_weights, const int32_t* combine_idx, int R,
                  int T_r, int H, int E, int k, int max_tokens_per_rank, void* out,
                  int32_t* status, void* stream);

/* ---- once-per-rank receive layout (V1 normal mode, §2.1, §2.3) ----------
 * A token goes ONCE to every rank holding one of its experts; rank r's
 * buffer holds source rank i's tokens from rank_prefix_matrix[i-1][r] on,
 * in token order, and the combine sums the rows the ranks return (the
 * experts of a rank weight their outputs before returning them).  It is the
 * per-expert pipeline run on per-slot destination-rank ids, with "experts"
 * = ranks (E' = R, one per rank):
 *   1. ep_rank_ids(topk_idx, ...)             -> rank_ids [R, T_r, k]
 *   2. ep_get_dispatch_layout(rank_ids, R, T_r, k, E' = R, ...)
 *        num_tokens_per_expert' = num_tokens_per_rank, slot_rank' = each
 *        token's position among source rank i's tokens for r
 *   3. ep_notify_dispatch(..., E' = R, expert_alignment 1, ...)
 *        rank_prefix_matrix as for the per-expert layout; expert_prefix'
 *        [i][r] = rank_prefix_matrix[i-1][r]; psum'[r] = {0, total};
 *        num_worst_tokens caps received TOKENS per rank (cap_rows = it)
 *   4. ep_dispatch(x, rank_ids, slot_rank', expert_prefix', psum', E' = R,
 *        fp8_mode, cap_rows, ...) -> recv_x [R, cap_rows, H] (+ scales),
 *        recv_src_idx, combine_idx [R, T_r, k]: r*cap_rows + row at the
 *        token's first slot on r, -1 at its other slots
 *   5. ep_rank_recv_topk(...)  -> each received row's local top-k ids/weights
 *   6. ep_rank_combine(y, combine_idx, ...) -> out [R, T_r, H] bf16 */

/* Per-slot destination rank: rank_ids[i][t][j] = topk_idx[i][t][j] / E_l
 * when slot j is token t's first slot whose expert is on that rank, else -1
 * (unused slot, or a rank the token already reached at an earlier slot).
 * Invalid ids (outside [-1, E)) set EP_ERR_INVALID_ARG in *status and give -1.
 * rank_ids: int64 [R, T_r, k], caller-owned device memory. */
int ep_rank_ids(const int64_t* topk_idx, int R, int T_r, int k, int E, int64_t* rank_ids,
                int32_t* status, void* stream);

/* For every received row of the once-per-rank layout, the local view of
 * its token's top-k: recv_topk_idx[r][row][j] = topk_idx[t][j] - r*E_l when
 * that expert is on rank r, else -1; recv_topk_weights[r][row][j] = its
 * weight, else 0.  combine_idx as returned by step 4 above.  Rows holding
 * no token are left untouched.
 *   recv_topk_idx     int64 [R, cap_rows, k]
 *   recv_topk_weights fp32  [R, cap_rows, k] */
int ep_rank_recv_topk(const int64_t* topk_idx, const float* topk_weights,
                      const int32_t* combine_idx, int R, int T_r, int k, int E, int64_t cap_rows,
                      int64_t* recv_topk_idx, float* recv_topk_weights, int32_t* status,
                      void* stream);

/* Rank-level combine (§2.3, dispatch walked backwards):
 *   out[t][:] = bf16_rn( fp32 sum, from +0 in slot order, of y[f_j][:] over
 *               the slots with f_j = combine_idx[t][j] >= 0 )
 * one row per destination rank the token reached, each already weighted by
 * that rank's experts.  y [R, cap_rows, H] bf16, out [R, T_r, H] bf16. */
int ep_rank_combine(const void* y, const int32_t* combine_idx, int R, int T_r, int H, int k,
                    int64_t cap_rows, void* out, int32_t* status, void* stream);

/* clean_low_latency_buffer (§1.2): zero recv_count [R, E_l] (may be NULL)
 * and the workspace (may be NULL), stream-ordered.  Required once before a
 * workspace's first use and after any call that reported EP_ERR_TIMEOUT or
 * EP_ERR_STATE. */
int ep_clean_ll_buffer(int32_t* recv_count, int R, int E, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Copy the device status word to *host_value and wait for the stream. */
int ep_read_status(const int32_t* status, int32_t* host_value, void* stream);

/* Host-side bounded wait: spin until all n HOST counters are >= 0
 * (EP_OK) or timeout_ms passes (EP_ERR_TIMEOUT).  Used by
 * ep_notify_dispatch; pure host code. */
int ep_host_wait_counters(const volatile int64_t* counters, int n, int timeout_ms);

/* Number formats, as the kernels convert (elementwise over n floats, n
 * even; in 8-byte and out 4-byte aligned device memory):
 *   ep_format_e4m3: fp32 -> OCP E4M3 byte, round to nearest even, finite
 *     values saturate to +-448 (the FP8 dispatch's cast, §1.1, §1.2);
 *   ep_format_bf16: fp32 -> bfloat16 bits, round to nearest even (the
 *     combine's output rounding).
 * EP_ERR_INVALID_ARG for odd n, null or misaligned pointers. */
int ep_format_e4m3(const float* in, uint8_t* out, int64_t n, void* stream);
int ep_format_bf16(const float* in, uint16_t* out, int64_t n, void* stream);

/* SM budget (Buffer.num_sms, §2.2; the per-SM bandwidth model of §4.6):
 * caps the SMs that the data kernels of ep_dispatch, ep_ll_dispatch,
 * ep_combine, ep_ll_combine and ep_rank_combine occupy, so the rest of the
 * GPU stays free for work that overlaps them.  num_sms = 0 lifts the cap
 * (every SM; the default); num_sms > 0 launches those kernels with at most
 * min(num_sms, SM count) CTAs of one per SM.  The single-launch low-latency
 * path then runs on that many SMs if the batch still fits them, else the
 * multi-kernel path is taken.  The layout and notify kernels (a few
 * microseconds, one CTA per id chunk / one CTA) are not capped.  Process-
 * wide, read at every launch; returns EP_ERR_INVALID_ARG for num_sms < 0.
 * ep_get_num_sms: the CTA count one-per-SM kernels get now (the SM count of
 * the current device, or the budget). */
int ep_set_num_sms(int num_sms);
int ep_get_num_sms(void);

/* Number of kernels this library has launched in the process. */
uint64_t ep_launch_count(void);

/* Static text for a return / status code. */
const char* ep_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* EP_H_ */
