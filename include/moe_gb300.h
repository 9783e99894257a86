/*
 * moe_gb300.h - C ABI of libmoe_gb300.so: the MoE expert layer on one
 * NVIDIA GB300 (sm_103a).
 *
 * The layer is the one expert parallelism wraps in its two all-to-alls:
 *   route    logits = x . W_r (+ bias), FP32 softmax, top-k, renormalised
 *            weights             ("InternVL3.5 接入 pure FSDP2 后端开发实践",
 *                                 MindSpeed-MM issue 625, §8.2)
 *   permute  per-expert counts, exclusive scan, stable scatter
 *                                ("Awesome-ML-SYS-Tutorial" MoE/EP guide,
 *                                 gsyq.cn, "Expert Parallelism"; same MindSpeed
 *                                 page §8.3)
 *   experts  grouped gate_up GEMM + SwiGLU, grouped down GEMM over the fused
 *            expert layout gate_up_proj [E*H, 2I], down_proj [E*I, H]
 *                                (MindSpeed page §2 and §8.3)
 *   combine  unpermute with the gate-weighted sum ("Awesome-ML-SYS-Tutorial"
 *            guide: experts' outputs summed with the gate weights)
 * plus the backward of each step (dX, d_router_logits, d_gate_up, d_down).
 *
 * Conventions (every entry point):
 *   - Every pointer argument is a DEVICE pointer, allocated and owned by the
 *     caller; the library never allocates or frees memory and keeps no
 *     pointer after the call returns (work is enqueued on `stream`).
 *   - Matrices are row-major and contiguous.  bf16 values are passed as
 *     uint16_t bit patterns (layout-compatible with __nv_bfloat16).
 *   - `stream` is a cudaStream_t (NULL: the legacy default stream).  Calls are
 *     asynchronous: a MOE_OK return means the work was validated and enqueued.
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid call enqueues nothing and returns a MOE_ERR_* code.
 *   - Errors found on the device (an expert id out of range, a bounded wait
 *     that ran out) set a device status word that moe_sync_status() reads.
 *   - Sizes are int64_t.  R = T*k is the number of permuted rows.
 *   - An empty batch (T == 0, or R == 0) is a valid call.  It writes only
 *     the outputs whose size does not depend on the rows: zero counts and
 *     offsets (moe_permute), zero weight gradients (the backward GEMMs,
 *     moe_route_bwd_weight).  Its row pointers may be NULL, including the
 *     optional ones, so an empty tensor's NULL data pointer is accepted.
 *   - Alignment: every base pointer must be 16-byte aligned; H and I must be
 *     multiples of 64 for the grouped GEMMs and of 8 elsewhere.
 *   - Per-device state: on its first call on a device the library looks up
 *     and keeps, for that device ordinal, the device addresses of its own
 *     __device__ arrays (the status word, moe_permute_noalloc's scratch) and
 *     the kernels' launch attributes.  They belong to the device's primary
 *     context.  A process that destroys that context (cudaDeviceReset) must
 *     not call the library on that device again: the kept addresses would
 *     then point into a context that no longer exists.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1 /* null pointer, negative size, k > E, bad alignment */
#define MOE_ERR_UNSUPPORTED 2 /* a shape outside the kernels' limits (e.g. H % 64) */
#define MOE_ERR_CUDA 3        /* a CUDA runtime/driver call failed */
#define MOE_ERR_TIMEOUT 4     /* a bounded device-side wait ran out */
#define MOE_ERR_WORKSPACE 5   /* workspace missing or smaller than required */
#define MOE_ERR_DEVICE 6      /* a device-side check failed (e.g. id out of range) */
#define MOE_ERR_SCRATCH_LIMIT 7 /* beyond the fixed scratch of moe_permute_noalloc */

/* Version of this ABI (major*10000 + minor*100 + patch). */
int moe_version(void);

/* Static string describing a status code. */
const char* moe_error_string(int status);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device.  Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE, or
 * MOE_ERR_CUDA when the synchronisation itself failed.  `detail` (nullable)
 * receives the raw device status word (0 when clean). */
int moe_sync_status(void* stream, uint32_t* detail);

/* Upper bound, in nanoseconds, of every device-side spin wait (mbarrier
 * waits in the grouped GEMMs) launched after this call.  A wait that runs out
 * records MOE_ERR_TIMEOUT in the status word and its kernel returns early
 * (the outputs are then undefined).  Default 2e9 (2 s).  0 restores the
 * default.  Not thread-safe against concurrent launches. */
int moe_set_wait_limit_ns(uint64_t ns);

/* Where the grouped GEMMs run: on single CTAs (128- or 256-row tiles) or on
 * CTA pairs (clusters of two CTAs issuing 2-SM tcgen05 MMAs on 256-row
 * tiles, 128-row tails as M = 128 pair MMAs; each CTA holds half of every
 * operand tile).  mode 0: single CTAs everywhere; 1: pairs for every forward
 * and dgrad grouped GEMM; 2 (default): pairs for the forward gate_up GEMM
 * only; 3: pairs for the forward gate_up GEMM and the two weight-gradient
 * GEMMs (whose expert K tails rank 0 of each pair zeroes in both CTAs'
 * shared memory).  Results are bit-identical in every mode.  Mode 2 is the
 * fastest measured on GB300 at the Qwen3-MoE shapes (the pairs' gate_up tile
 * count fills whole waves there; down and the backward GEMMs measured slower
 * on pairs).  Another mode returns MOE_ERR_INVALID_ARG.  Applies to launches
 * after the call; not thread-safe against them. */
int moe_set_gemm_pairs(int mode);

/* Programmatic dependent launch: 1 (default) launches every kernel so that it
 * may start while the kernel before it on the same stream finishes (its
 * set-up overlaps that kernel's tail; it waits for it before touching
 * memory), 0 launches them the plain way.  Results are identical either
 * way.  Faster for one stream (a training step: 2.12 -> 2.09 ms on GB300 at
 * the Qwen3-MoE shape, T = 8192); slower when two streams of this library's
 * kernels run side by side, where the early-resident kernels take the SMs
 * that the other stream would fill.  Applies to launches (and stream
 * captures) after the call; not thread-safe against them. */
int moe_set_pdl(int on);

/* Test hook of the failure-detection path: while on (1), the grouped GEMMs
 * launched afterwards issue no operand loads, so their MMA warp's bounded
 * wait runs out; the kernel then records MOE_ERR_TIMEOUT, stops its other
 * warps, frees its tensor memory and returns (outputs undefined), leaving
 * the context usable.  Off (0) by default; not for production use. */
int moe_test_stall_gemm_producer(int on);

/* ------------------------------------------------------------------ route */

/* Bytes of workspace moe_route needs.  With E % 8 == 0 and H % 64 == 0 the
 * logits run on the tensor cores and the workspace holds the exact
 * three-term bf16 split of W_r (3*H*E*2 bytes); when E is not also a
 * multiple of 16 in [16, 256] it adds the fp32 partial logits of a split-K
 * GEMM (parts*T*E*4 bytes).  Other shapes: the fp32 logits (T*E*4). */
int moe_route_workspace_size(int64_t T, int64_t H, int64_t E, size_t* bytes);

/* Router (MindSpeed page §8.2: gate -> FP32 softmax -> top-k -> renormalise).
 *   x        [T, H] bf16         tokens
 *   w_router [H, E] fp32         router weight
 *   bias     [E] fp32 or NULL    added to the logits before the softmax
 *   ids      [T, k] int32 (out)  chosen experts, largest probability first;
 *                                equal fp32 logits go to the lower index
 *   w        [T, k] fp32 (out)   p_j / sum of the chosen p (sums to 1)
 *   logits   [T, E] fp32 (out, nullable) x . W_r + bias
 *   workspace                    device scratch, moe_route_workspace_size bytes
 * Limits: 1 <= k <= min(E, 32), E <= 1024, H % 8 == 0.  The logits are the
 * fp32-accumulated dot products of the exact bf16 x with the fp32 W_r (on
 * the tensor cores through an exact three-term bf16 split of W_r, or on the
 * CUDA cores); the softmax is fp32. */
int moe_route(const uint16_t* x, const float* w_router, const float* bias, int64_t T, int64_t H,
              int64_t E, int64_t k, int32_t* ids, float* w, float* logits, void* workspace,
              size_t workspace_bytes, void* stream);

/* The router with W_r's bf16 split prepared once.  On the tensor-core path
 * moe_route first splits W_r exactly into three bf16 terms, W = W0 + W1 + W2
 * (24 = 3 x 8 significant bits: Henry, Tang & Heinecke, ARITH 2019), then
 * multiplies the exact bf16 x with all three, accumulating in fp32.  While
 * W_r does not change (inference; a training step changes it once per
 * optimizer step) the split can be made once and reused:
 *   moe_route_split_weight   w_split [3, H, E] bf16 (out: W0 rows, then W1,
 *                            then W2; 3*H*E*2 bytes, caller-owned, 16-byte
 *                            aligned) from w_router [H, E] fp32
 *   moe_route_presplit       moe_route's arguments with w_split in place of
 *                            w_router and its own (smaller) workspace; ids, w
 *                            and logits are bit for bit those of moe_route
 * Both need the tensor-core path (E % 8 == 0, H % 64 == 0, E <= 1024); other
 * shapes return MOE_ERR_UNSUPPORTED (use moe_route).  The presplit workspace
 * is 0 bytes when 16 <= E <= 256 and E % 16 == 0 (the fused cluster router;
 * workspace may then be NULL), else the split-K partial logits. */
int moe_route_split_weight(const float* w_router, int64_t H, int64_t E, uint16_t* w_split, void* stream);
int moe_route_presplit_workspace_size(int64_t T, int64_t H, int64_t E, size_t* bytes);
int moe_route_presplit(const uint16_t* x, const uint16_t* w_split, const float* bias, int64_t T, int64_t H,
                       int64_t E, int64_t k, int32_t* ids, float* w, float* logits, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- permute */

/* Bytes of workspace moe_permute needs: per-block expert histograms, the
 * expert totals and two grid-barrier counters (the workspace must be 16-byte
 * aligned; nothing in it needs clearing). */
int moe_permute_workspace_size(int64_t T, int64_t k, int64_t E, size_t* bytes);

/* Group the R = T*k assignments by expert ("Awesome-ML-SYS-Tutorial" guide:
 * per-expert token counts, then permute by expert; MindSpeed page §8.3).
 *   ids      [T, k] int32  expert of each (token, slot); i = t*k + j
 *   w        [T, k] fp32 or NULL   gate weights to carry along (with w_perm)
 *   counts   [E] int32 (out)     rows per expert (empty experts give 0)
 *   offsets  [E+1] int32 (out)   exclusive scan of counts, offsets[E] = R
 *   row_map  [R] int32 (out)     permuted row of assignment i; stable: the
 *                                rows of one expert keep increasing i
 *   src_row  [R] int32 (out)     token of each permuted row (= i / k)
 *   w_perm   [R] fp32 (out) or NULL   w_perm[row_map[i]] = w[i]
 * Deterministic (no order-dependent atomics).  Up to 2^18 assignments and
 * E <= 256 it is one launch of clusters of 8 CTAs that share their counts
 * through distributed shared memory (no waits beyond the hardware cluster
 * barrier; the workspace is not used).  Otherwise, when all of its blocks
 * fit on the device at once (R up to about 300k assignments on a GB300), one
 * cooperative launch whose two grid barriers are bounded waits
 * (MOE_ERR_TIMEOUT in the status word if one runs out); else three
 * launches.  An id outside [0, E) sets MOE_ERR_DEVICE in the status word;
 * the outputs are then undefined.  A misaligned workspace returns
 * MOE_ERR_INVALID_ARG.  Limits: E <= 1024, R < 2^31. */
int moe_permute(const int32_t* ids, const float* w, int64_t T, int64_t k, int64_t E, int32_t* counts,
                int32_t* offsets, int32_t* row_map, int32_t* src_row, float* w_perm, void* workspace,
                size_t workspace_bytes, void* stream);

/* moe_permute without a workspace, for callers that cannot allocate device
 * memory when they route: e.g. a plugin running inside an inference engine's
 * enqueue step (which must not allocate), a runtime that has reserved all
 * device memory for its own pool, or a latency-critical path that cannot pay
 * for cudaMalloc's implicit device synchronisation.  The pages have no
 * counterpart to this entry point; it computes exactly what moe_permute
 * computes, with the same arguments minus the workspace.
 *   Scratch: a fixed 4 MiB array in device memory inside this library
 *   (every GPU that loads the library holds it until the process exits).
 *   Limit: ceil(T*k / 2048) * E <= 2^20; larger sizes return
 *   MOE_ERR_SCRATCH_LIMIT and enqueue nothing.
 *   Allocation: none (no cudaMalloc, cudaFree or allocating library call).
 *   Set-up: the first call on each device looks up the array's device
 *   address (with that device current); make that first call before any
 *   stream capture.
 *   Concurrency: all calls share the one array; calls that overlap on the GPU
 *   (different streams, or devices sharing a context) race.  Each call
 *   overwrites the scratch it reads, so nothing carries over between calls. */
int moe_permute_noalloc(const int32_t* ids, const float* w, int64_t T, int64_t k, int64_t E,
                        int32_t* counts, int32_t* offsets, int32_t* row_map, int32_t* src_row,
                        float* w_perm, void* stream);

/* The materialised permute: x_perm[row] = x[src_row[row]] for R rows of H
 * bf16 (the grouped GEMMs gather rows themselves and do not need it).  The
 * source rows are not range-checked here (the token count is not passed). */
int moe_permute_rows(const uint16_t* x, const int32_t* src_row, int64_t R, int64_t H,
                     uint16_t* x_perm, void* stream);

/* The same rows moved token by token (MindSpeed page §8.3 permute, the
 * materialised form): x_perm[row_map[t*k + j]] = x[t] for t < T, j < k.
 * Each token row is read once and written to its k permuted rows, so x is
 * read from memory once whatever its size (moe_permute_rows reads each token
 * row k times, in permuted order).  With row_map from moe_permute (a
 * permutation of [0, T*k)) every row of x_perm is written exactly once and
 * the result equals moe_permute_rows with its src_row bit for bit.
 *   x        [T, H] bf16;  row_map [T*k] int32;  x_perm [T*k, H] bf16
 * H % 8 == 0, 1 <= k <= 32, x and x_perm 16-byte aligned.  A row_map entry
 * outside [0, T*k) sets MOE_ERR_DEVICE in the status word and that copy is
 * not written. */
int moe_permute_rows_scatter(const uint16_t* x, const int32_t* row_map, int64_t T, int64_t k, int64_t H,
                             uint16_t* x_perm, void* stream);

/* ----------------------------------------------------------- grouped GEMMs */

/* Every grouped GEMM checks its offsets on the device (offsets[0] = 0,
 * non-decreasing, offsets[E] = R); other values set MOE_ERR_DEVICE in the
 * status word and the call computes nothing (its outputs are undefined). */

/* Grouped gate_up GEMM with the SwiGLU fused into its epilogue (MindSpeed
 * page §2 layout, §8.3 "grouped_matmul -> SwiGLU").  For each expert e and
 * each permuted row r in [offsets[e], offsets[e+1]):
 *   a = x[src_row[r]]  (or x[r] when src_row is NULL)
 *   g = a . gate_up[e*H:(e+1)*H, 0:I],   u = a . gate_up[e*H:(e+1)*H, I:2I]
 *   h[r] = silu(g) * u                          (fp32, stored bf16)
 *   gu_pre[r] = [g | u]                          (fp32, when not NULL)
 *   h_w[r] = w_perm[r] * silu(g) * u             (bf16, when not NULL)
 *   x        [T, H] bf16 (or [R, H] already permuted, src_row NULL)
 *   gate_up  [E*H, 2I] bf16;  h, h_w [R, I] bf16;  gu_pre [R, 2I] fp32
 *   src_row  [R] int32: the permute is fused into the A-operand load (TMA
 *            row gather); NULL: rows are read in order
 *   offsets  [E+1] int32 on the device (never read back to the host), or
 *            NULL for one group of all R rows (E must be 1): the dense mode
 *            used for the shared expert
 *   w_perm   [R] fp32 (from moe_permute), needed only for h_w
 * The training forward saves gu_pre and h_w for the backward.
 * bf16 inputs, fp32 accumulation (tcgen05 tensor cores). */
int moe_grouped_gemm_gate_up_swiglu(const uint16_t* x, const int32_t* src_row,
                                    const int32_t* offsets, const uint16_t* gate_up, int64_t T,
                                    int64_t R, int64_t H, int64_t E, int64_t I, uint16_t* h,
                                    const float* w_perm, float* gu_pre, uint16_t* h_w, void* stream);

/* Grouped down GEMM (MindSpeed page §2 layout, §8.3):
 *   y_perm[r] = h[r] . down[e*I:(e+1)*I, :]   for r in expert e's rows
 *   h [R, I] bf16;  down [E*I, H] bf16;  y_perm [R, H] bf16
 *   offsets as above (NULL: one group, E == 1). */
int moe_grouped_gemm_down(const uint16_t* h, const int32_t* offsets, const uint16_t* down, int64_t R,
                          int64_t H, int64_t E, int64_t I, uint16_t* y_perm, void* stream);

/* ---------------------------------------------------------------- combine */

/* Unpermute with the gate-weighted combine ("Awesome-ML-SYS-Tutorial" guide:
 * the experts' outputs summed with the gate weights; MindSpeed page §8.3
 * "unpermute"):
 *   y[t] = sum_{j<k} w[t,j] * y_perm[row_map[t*k+j]]  (+ y_shared[t])
 * accumulated in fp32 in increasing j, stored bf16.  Deterministic.
 *   y_perm [R, H] bf16; row_map [R] int32; w [T, k] fp32;
 *   y_shared [T, H] bf16 or NULL (the always-active shared expert, weight 1);
 *   y [T, H] bf16 (out).  Limits: k <= 32.  A row_map entry outside [0, T*k)
 * sets MOE_ERR_DEVICE in the status word (row 0 is read in its place). */
int moe_unpermute_combine(const uint16_t* y_perm, const int32_t* row_map, const float* w,
                          const uint16_t* y_shared, int64_t T, int64_t H, int64_t k, uint16_t* y,
                          void* stream);

/* --------------------------------------------------------------- backward */
/* The backward of L with upstream gradient dY, the chosen experts held fixed
 * (the gradient reaches the router only through the renormalised weights).
 * Call order: combine_bwd -> down_bwd -> route_bwd -> gate_up_bwd -> gather_dx. */

/* Backward of the combine with respect to the expert outputs, before the
 * gate weights (which the grouped GEMMs apply in fp32):
 *   dy_perm[row] = dY[src_row[row]]         (an exact bf16 copy; R = T*k rows)
 * The gate-weight gradient dw[t,j] = <dY[t], y_perm[row_map[t*k+j]]> is
 * produced by moe_grouped_gemm_down_bwd (as <dY . Wd^T, h>) and summed by
 * moe_route_bwd.  dy [T, H] bf16; src_row [R] int32; dy_perm [R, H] bf16.
 * A src_row entry outside [0, T) sets MOE_ERR_DEVICE (row 0 is read).
 * moe_permute_rows_scatter(dy, row_map, ...) computes the same dy_perm bit
 * for bit, reading each dY row once. */
int moe_unpermute_combine_bwd(const uint16_t* dy, const int32_t* src_row, int64_t T, int64_t H,
                              int64_t k, uint16_t* dy_perm, void* stream);

/* Number of partial sums per permuted row that moe_grouped_gemm_down_bwd
 * writes into dw_part (one per 64 columns of I: I / 64). */
int moe_grouped_gemm_down_bwd_parts(int64_t I, int64_t* nparts);

/* Backward of the down GEMM and of the SwiGLU, per expert e:
 *   a = dy_perm[r] . down_e^T                         (fp32)
 *   dh = w_perm[r] * a;  g, u = gu_pre[r];  s = sigmoid(g)
 *   dgu[r] = [ dh * u * s * (1 + g*(1-s))  |  dh * g * s ]   (bf16)
 *   dw_part[r, n] = sum over column block n of a * silu(g) * u    (fp32;
 *                   summed over n this is <dY[t], y_perm[r]>, the gradient
 *                   of the gate weight of row r)
 *   d_down_e = h_w_e^T . dy_perm_e                    (fp32 accumulate, bf16;
 *                                                      0 for an empty expert)
 *   dy_perm [R, H] bf16 (unweighted); h_w [R, I] bf16 (w * h, saved forward);
 *   gu_pre [R, 2I] fp32; w_perm [R] fp32; down [E*I, H] bf16;
 *   dgu [R, 2I] bf16 (out); d_down [E*I, H] bf16 (out);
 *   dw_part [R, nparts] fp32 (out), nparts from moe_grouped_gemm_down_bwd_parts. */
int moe_grouped_gemm_down_bwd(const uint16_t* dy_perm, const uint16_t* h_w, const float* gu_pre,
                              const float* w_perm, const int32_t* offsets, const uint16_t* down,
                              int64_t R, int64_t H, int64_t E, int64_t I, uint16_t* dgu,
                              uint16_t* d_down, float* dw_part, void* stream);

/* Backward of the renormalised softmax (w = softmax over the chosen logits):
 *   dw[t,j] = sum_n dw_part[row_map[t*k+j], n]          (fixed order)
 *   d_logits[t, ids[t,j]] = w[t,j] * (dw[t,j] - sum_i w[t,i] dw[t,i])
 *   d_logits[t, e] = 0 for every expert not chosen by t
 *   d_logits [T, E] fp32 (out); dw [T, k] fp32 (out, nullable).
 * A row_map entry outside [0, T*k) sets MOE_ERR_DEVICE (row 0 is read). */
int moe_route_bwd(const float* dw_part, int64_t nparts, const int32_t* row_map, const float* w,
                  const int32_t* ids, int64_t T, int64_t E, int64_t k, float* d_logits, float* dw,
                  void* stream);

/* Backward of the gate_up GEMM, per expert e:
 *   dx_perm[r] = dgu[r] . gate_up_e^T                (bf16)
 *   d_gate_up_e = x[src_rows of e]^T . dgu_e         (fp32 accumulate, bf16;
 *                                                     0 for an empty expert)
 *   dgu [R, 2I]; x [T, H]; src_row [R] (NULL: x is already permuted, [R, H]);
 *   gate_up [E*H, 2I]; dx_perm [R, H] (out); d_gate_up [E*H, 2I] (out). */
int moe_grouped_gemm_gate_up_bwd(const uint16_t* dgu, const uint16_t* x, const int32_t* src_row,
                                 const int32_t* offsets, const uint16_t* gate_up, int64_t T,
                                 int64_t R, int64_t H, int64_t E, int64_t I, uint16_t* dx_perm,
                                 uint16_t* d_gate_up, void* stream);

/* Bytes of workspace moe_gather_dx needs (a transposed copy of W_r, H*E*4). */
int moe_gather_dx_workspace_size(int64_t H, int64_t E, size_t* bytes);

/* The input gradient, summed per token in increasing j (deterministic):
 *   dX[t] = sum_j dx_perm[row_map[t*k+j]] + sum_j d_logits[t, ids[t,j]] * W_r[:, ids[t,j]]
 * (the second sum is the router's contribution d_logits . W_r^T, whose only
 * nonzero terms are the chosen experts).  d_logits/w_router may both be NULL
 * to leave the router term out (no workspace needed then).  dX [T, H] bf16
 * (out), fp32 accumulation, one bf16 rounding.  A row_map entry outside
 * [0, T*k) or an id outside [0, E) sets MOE_ERR_DEVICE (row / expert 0 is
 * read in its place). */
int moe_gather_dx(const uint16_t* dx_perm, const int32_t* row_map, const float* d_logits,
                  const int32_t* ids, const float* w_router, int64_t T, int64_t H, int64_t E,
                  int64_t k, uint16_t* dx, void* workspace, size_t workspace_bytes, void* stream);

/* The router weight gradient d_w_router[h, e] = sum_t x[t,h] * d_logits[t,e]
 * (fp32, summed in increasing t).  x [T, H] bf16; d_logits [T, E] fp32;
 * d_w_router [H, E] fp32 (out). */
int moe_route_bwd_weight(const uint16_t* x, const float* d_logits, int64_t T, int64_t H, int64_t E,
                         float* d_w_router, void* stream);

/* ---------------------------------------------------- expert parallelism */

/* The single-device pieces of expert-parallel dispatch and combine
 * ("Awesome-ML-SYS-Tutorial" MoE/EP guide, "Expert Parallelism": dispatch
 * and combine by all-to-all, split sizes from per-expert token counts, the
 * receiver's re-sort of its chunks by local expert `sort_chunks_by_idxs`;
 * hotspot experts and EPLB-style replication).  Experts are split over the
 * EP ranks on dim 0, so a rank's permuted rows are already grouped by the
 * rank that owns their expert.  The transport between ranks (an all-to-all-v
 * of NCCL or another library) is not part of this library. */

/* Bytes of workspace moe_sort_chunks needs: (2*A*B + 1) int32. */
int moe_sort_chunks_workspace_size(int64_t A, int64_t B, size_t* bytes);

/* Rows that arrive as an A x B matrix of chunks in row-major (a, b) order
 * (chunk (a, b) holds counts[a*B + b] rows) are reordered to (b, a) order:
 * the transpose of the chunk matrix, each chunk's rows kept in order.  It is
 * what an all-to-all does to the order of the rows of every sender (a =
 * source rank, b = destination rank) and what the receiver's re-sort does to
 * its chunks (a = source rank, b = local expert), after which each local
 * expert's rows are contiguous.
 *   counts        [A*B] int32 (device)   chunk sizes, >= 0, summing to N
 *   src_of        [N] int32 (out)        input row at each output position
 *   pos_of        [N] int32 (out)        output position of each input row
 *   group_offsets [B+1] int32 (out)      first output row of each b, then N
 *                                        (the receiver's local expert offsets)
 * The rows themselves move with moe_permute_rows (x_out = x_in[src_of]; back
 * again with pos_of).  Counts that are negative or do not sum to N are
 * reported as MOE_ERR_DEVICE (outputs undefined, nothing written out of
 * bounds).  Limits: A*B <= 2^24, N < 2^31. */
int moe_sort_chunks(const int32_t* counts, int64_t A, int64_t B, int64_t N, int32_t* src_of, int32_t* pos_of,
                    int32_t* group_offsets, void* workspace, size_t workspace_bytes, void* stream);

/* EPLB-style expert replication, on the host (no GPU).  From each logical
 * expert's load (e.g. the rows it received in recent steps) and n_phys >= E
 * physical expert slots over G ranks (n_phys % G == 0):
 *   1. each of the n_phys - E extra replicas goes to the expert with the
 *      largest load per replica (ties to the lower index);
 *   2. a replica's load is its share under the round-robin by token of
 *      moe_ep_map_replicas (load / replicas, the first load % replicas
 *      replicas one more);
 *   3. replicas, heaviest first, each go to the least-loaded rank with a free
 *      slot (n_phys / G slots per rank; ties to the lower rank);
 *   4. physical ids are rank-major (rank g owns ids g*n_phys/G ...), within a
 *      rank ordered by (expert, replica).
 * Outputs (host arrays): phys_to_log [n_phys], rep_first [E] and rep_count
 * [E] (replica r of expert e is physical expert rep_list[rep_first[e] + r]),
 * rep_list [n_phys], rank_load [G] (nullable).  The pages name the method
 * (hotspot experts, EPLB) without its steps; this is the plain greedy reading. */
int moe_eplb_plan(const int64_t* expert_load, int64_t E, int64_t G, int64_t n_phys, int32_t* phys_to_log,
                  int32_t* rep_first, int32_t* rep_count, int32_t* rep_list, int64_t* rank_load);

/* Logical expert ids -> physical replica ids (device): assignment i = t*k + j
 * of logical expert e goes to replica t mod rep_count[e], i.e. physical expert
 * rep_list[rep_first[e] + t % rep_count[e]].  The replicas carry copies of
 * the expert's weights, so the layer's output is unchanged; a replicated
 * expert's rows are shared by its replicas.  ids out of [0, E) or a plan
 * that points outside [0, n_phys) are reported as MOE_ERR_DEVICE (physical
 * expert 0 is written instead). */
int moe_ep_map_replicas(const int32_t* ids, int64_t T, int64_t k, int64_t E, const int32_t* rep_first,
                        const int32_t* rep_count, const int32_t* rep_list, int64_t n_phys, int32_t* phys_ids,
                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
