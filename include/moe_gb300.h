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
 *   - Alignment: every base pointer must be 16-byte aligned; H and I must be
 *     multiples of 64 for the grouped GEMMs and of 8 elsewhere.
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

/* ------------------------------------------------------------------ route */

/* Bytes of workspace moe_route needs: T*E*4 when `logits` is NULL (the logits
 * are staged there), else 0. */
int moe_route_workspace_size(int64_t T, int64_t E, int has_logits_out, size_t* bytes);

/* Router (MindSpeed page §8.2: gate -> FP32 softmax -> top-k -> renormalise).
 *   x        [T, H] bf16         tokens
 *   w_router [H, E] fp32         router weight
 *   bias     [E] fp32 or NULL    added to the logits before the softmax
 *   ids      [T, k] int32 (out)  chosen experts, largest probability first;
 *                                equal fp32 logits go to the lower index
 *   w        [T, k] fp32 (out)   p_j / sum of the chosen p (sums to 1)
 *   logits   [T, E] fp32 (out, nullable) x . W_r + bias
 * Limits: 1 <= k <= min(E, 32), E <= 1024, H % 8 == 0.  The dot products
 * accumulate in fp32 from the exact bf16 x; the softmax is fp32. */
int moe_route(const uint16_t* x, const float* w_router, const float* bias, int64_t T, int64_t H,
              int64_t E, int64_t k, int32_t* ids, float* w, float* logits, void* workspace,
              size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- permute */

/* Bytes of workspace moe_permute needs (per-block expert histograms). */
int moe_permute_workspace_size(int64_t T, int64_t k, int64_t E, size_t* bytes);

/* Group the R = T*k assignments by expert ("Awesome-ML-SYS-Tutorial" guide:
 * per-expert token counts, then permute by expert; MindSpeed page §8.3).
 *   ids      [T, k] int32  expert of each (token, slot); i = t*k + j
 *   counts   [E] int32 (out)     rows per expert (empty experts give 0)
 *   offsets  [E+1] int32 (out)   exclusive scan of counts, offsets[E] = R
 *   row_map  [R] int32 (out)     permuted row of assignment i; stable: the
 *                                rows of one expert keep increasing i
 *   src_row  [R] int32 (out)     token of each permuted row (= i / k)
 * Deterministic (no order-dependent atomics).  An id outside [0, E) sets
 * MOE_ERR_DEVICE in the status word; the outputs are then undefined.
 * Limits: E <= 1024, R < 2^31. */
int moe_permute(const int32_t* ids, int64_t T, int64_t k, int64_t E, int32_t* counts,
                int32_t* offsets, int32_t* row_map, int32_t* src_row, void* workspace,
                size_t workspace_bytes, void* stream);

/* The materialised permute: x_perm[row] = x[src_row[row]] for R rows of H
 * bf16 (the grouped GEMMs gather rows themselves and do not need it). */
int moe_permute_rows(const uint16_t* x, const int32_t* src_row, int64_t R, int64_t H,
                     uint16_t* x_perm, void* stream);

/* ----------------------------------------------------------- grouped GEMMs */

/* Grouped gate_up GEMM with the SwiGLU fused into its epilogue (MindSpeed
 * page §2 layout, §8.3 "grouped_matmul -> SwiGLU").  For each expert e and
 * each permuted row r in [offsets[e], offsets[e+1]):
 *   g = x[src_row[r]] . gate_up[e*H:(e+1)*H, 0:I]
 *   u = x[src_row[r]] . gate_up[e*H:(e+1)*H, I:2I]
 *   h[r] = silu(g) * u                        (fp32, stored bf16)
 *   gu_pre[r] = [g | u]                        (bf16, when not NULL)
 *   x        [T, H] bf16;  gate_up [E*H, 2I] bf16;  h [R, I] bf16
 *   src_row  [R] int32, or NULL for rows taken in order (x has R rows)
 *   offsets  [E+1] int32 on the device (never read back to the host), or
 *            NULL for one group of all R rows (E must be 1): the dense mode
 *            used for the shared expert
 * bf16 inputs, fp32 accumulation (tcgen05 tensor cores), bf16 outputs. */
int moe_grouped_gemm_gate_up_swiglu(const uint16_t* x, const int32_t* src_row,
                                    const int32_t* offsets, const uint16_t* gate_up, int64_t T,
                                    int64_t R, int64_t H, int64_t E, int64_t I, uint16_t* h,
                                    uint16_t* gu_pre, void* stream);

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
 *   y [T, H] bf16 (out).  Limits: k <= 32. */
int moe_unpermute_combine(const uint16_t* y_perm, const int32_t* row_map, const float* w,
                          const uint16_t* y_shared, int64_t T, int64_t H, int64_t k, uint16_t* y,
                          void* stream);

/* --------------------------------------------------------------- backward */
/* The backward of L with upstream gradient dY, the chosen experts held fixed
 * (the gradient reaches the router only through the renormalised weights).
 * Call order: combine_bwd -> route_bwd -> down_bwd -> gate_up_bwd -> gather_dx. */

/* Backward of the combine:
 *   dy_perm[row_map[t*k+j]] = w[t,j] * dY[t]            (bf16)
 *   dw[t,j] = <dY[t], y_perm[row_map[t*k+j]]>           (fp32)
 *   dy [T, H] bf16; y_perm [R, H] bf16 (saved forward output). */
int moe_unpermute_combine_bwd(const uint16_t* dy, const uint16_t* y_perm, const int32_t* row_map,
                              const float* w, int64_t T, int64_t H, int64_t k, uint16_t* dy_perm,
                              float* dw, void* stream);

/* Backward of the renormalised softmax (w = softmax over the chosen logits):
 *   d_logits[t, ids[t,j]] = w[t,j] * (dw[t,j] - sum_i w[t,i] dw[t,i])
 *   d_logits[t, e] = 0 for every expert not chosen by t
 *   d_logits [T, E] fp32 (out). */
int moe_route_bwd(const float* dw, const float* w, const int32_t* ids, int64_t T, int64_t E,
                  int64_t k, float* d_logits, void* stream);

/* Backward of the down GEMM and of the SwiGLU, per expert e:
 *   dh = dy_perm[r] . down_e^T                       (fp32)
 *   g, u = gu_pre[r];  s = sigmoid(g)
 *   dgu[r] = [ dh * u * s * (1 + g*(1-s))  |  dh * g * s ]   (bf16)
 *   d_down_e = h_e^T . dy_perm_e                     (fp32 accumulate, bf16;
 *                                                     0 for an empty expert)
 *   dy_perm [R, H]; h [R, I]; gu_pre [R, 2I]; down [E*I, H];
 *   dgu [R, 2I] (out); d_down [E*I, H] (out). */
int moe_grouped_gemm_down_bwd(const uint16_t* dy_perm, const uint16_t* h, const uint16_t* gu_pre,
                              const int32_t* offsets, const uint16_t* down, int64_t R, int64_t H,
                              int64_t E, int64_t I, uint16_t* dgu, uint16_t* d_down, void* stream);

/* Backward of the gate_up GEMM, per expert e:
 *   dx_perm[r] = dgu[r] . gate_up_e^T                (bf16)
 *   d_gate_up_e = x[src_rows of e]^T . dgu_e         (fp32 accumulate, bf16;
 *                                                     0 for an empty expert)
 *   dgu [R, 2I]; x [T, H]; src_row [R] (NULL: rows in order, T == R);
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
 * (out), fp32 accumulation, one bf16 rounding. */
int moe_gather_dx(const uint16_t* dx_perm, const int32_t* row_map, const float* d_logits,
                  const int32_t* ids, const float* w_router, int64_t T, int64_t H, int64_t E,
                  int64_t k, uint16_t* dx, void* workspace, size_t workspace_bytes, void* stream);

/* The router weight gradient d_w_router[h, e] = sum_t x[t,h] * d_logits[t,e]
 * (fp32, summed in increasing t).  x [T, H] bf16; d_logits [T, E] fp32;
 * d_w_router [H, E] fp32 (out). */
int moe_route_bwd_weight(const uint16_t* x, const float* d_logits, int64_t T, int64_t H, int64_t E,
                         float* d_w_router, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
