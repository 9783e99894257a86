// Unpermute with the gate-weighted combine and the token-side backward steps.
//
// Forward ("Awesome-ML-SYS-Tutorial" MoE/EP guide, gsyq.cn, "Expert
// Parallelism": the experts' outputs summed with the gate weights;
// "InternVL3.5 接入 pure FSDP2 后端开发实践" §8.3: unpermute):
//   y[t] = sum_{j<k} w[t,j] * y_perm[row_map[t*k+j]]  (+ y_shared[t])
// One warp per (token, 1024-column slice); each lane owns 16-byte (8 x bf16)
// column chunks and accumulates in fp32 in increasing j, so the result does
// not depend on the launch shape (a gather, not a scatter-add: deterministic).
//
// Backward (the gradient of the same expression, experts held fixed):
//   combine_bwd   dy_perm[row] = dY[src_row[row]]: an exact copy (the rows
//                 permute of dY); the gate weight w[t,j] is applied in fp32
//                 by the GEMM epilogues, so it is never rounded into a bf16
//                 operand.  dw[t,j] = <dY[t], y_perm[row]> is computed by the
//                 down GEMM's backward as <dY . Wd^T, h> in fp32.
//   route_bwd     dw[t,j] = sum of its per-tile partials (fixed order);
//                 d_logits[t, ids_j] = w_j (dw_j - sum_i w_i dw_i), 0 elsewhere
//   gather_dx     dX[t] = sum_j dx_perm[row_map[t*k+j]]
//                         + sum_j d_logits[t, ids_j] * W_r[:, ids_j]
//                 (W_r read through a transposed copy [E, H] so the router
//                 term streams contiguous rows)
//   route_bwd_weight  d_W_r = x^T . d_logits (fp32 register-tiled GEMM)
#include "kernels.h"

namespace moe {

namespace {

constexpr int kWarpsPerBlock = 8;

// Rows are split into slices of kSliceChunks 16-byte chunks (1024 bf16), one
// warp per (token, slice), so that a launch has enough warps in flight to
// keep HBM busy even when T is small.
constexpr int kSliceChunks = 128;

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y_perm,
                                                      const int32_t* __restrict__ row_map,
                                                      const float* __restrict__ w,
                                                      const uint16_t* __restrict__ y_shared,
                                                      int T, int H, int k,
                                                      uint16_t* __restrict__ y, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nch = H / 8;
  const int slices = (nch + kSliceChunks - 1) / kSliceChunks;
  const int gw = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int t = gw / slices;
  const int c_begin = (gw - t * slices) * kSliceChunks;
  const int c_end = min(nch, c_begin + kSliceChunks);
  if (t >= T) return;
  int my_row = 0;
  float my_w = 0.f;
  if (lane < k) {
    my_row = row_map[(int64_t)t * k + lane];
    my_w = w[(int64_t)t * k + lane];
    if (my_row < 0 || (int64_t)my_row >= (int64_t)T * k) {   // not a permuted row: report, read row 0
      report_status(status, kStatusDevice, kKernCombine, 1);
      my_row = 0;
    }
  }
  // The chunk loop stays warp-uniform (lanes past the slice only predicate
  // their loads and stores) because every lane takes part in the shuffles
  // that hand out the k rows and weights.  Each lane takes two chunks per
  // pass (c and c + 32), so 2k independent 16-byte loads are in flight.
  for (int base = c_begin; base < c_end; base += 64) {
    const int c0 = base + lane, c1 = c0 + 32;
    const bool act0 = c0 < c_end, act1 = c1 < c_end;
    float acc0[8], acc1[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      acc0[q] = 0.f;
      acc1[q] = 0.f;
    }
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      const float wj = __shfl_sync(0xffffffffu, my_w, j);
      const uint4* src = reinterpret_cast<const uint4*>(y_perm + (int64_t)row * H);
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
      if (act0) v0 = ld_stream16(src + c0);
      if (act1) v1 = ld_stream16(src + c1);
      float f[8];
      unpack8(v0, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc0[q] = fmaf(wj, f[q], acc0[q]);
      unpack8(v1, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc1[q] = fmaf(wj, f[q], acc1[q]);
    }
    uint4* dst = reinterpret_cast<uint4*>(y + (int64_t)t * H);
    if (act0) {
      if (y_shared) {
        float f[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(y_shared + (int64_t)t * H) + c0), f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc0[q] += f[q];
      }
      dst[c0] = pack8(acc0);
    }
    if (act1) {
      if (y_shared) {
        float f[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(y_shared + (int64_t)t * H) + c1), f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc1[q] += f[q];
      }
      dst[c1] = pack8(acc1);
    }
  }
}

__global__ void __launch_bounds__(256) route_bwd_kernel(const float* __restrict__ dw_part, int nparts,
                                                        const int32_t* __restrict__ row_map,
                                                        const float* __restrict__ w,
                                                        const int32_t* __restrict__ ids, int T,
                                                        int E, int k,
                                                        float* __restrict__ d_logits,
                                                        float* __restrict__ dw, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (t >= T) return;
  float my_w = 0.f, my_dw = 0.f;
  int my_id = -1;
  if (lane < k) {
    my_w = w[(int64_t)t * k + lane];
    my_id = ids[(int64_t)t * k + lane];
    int64_t row = row_map[(int64_t)t * k + lane];
    if (row < 0 || row >= (int64_t)T * k) {   // not a permuted row: report, read row 0
      report_status(status, kStatusDevice, kKernCombine, 4);
      row = 0;
    }
    for (int n = 0; n < nparts; ++n) my_dw += dw_part[row * nparts + n];   // fixed order
    if (dw) dw[(int64_t)t * k + lane] = my_dw;
  }
  const float mean = warp_sum(my_w * my_dw);   // sum_i w_i dw_i
  const float my_dz = my_w * (my_dw - mean);
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    float v = 0.f;
    for (int j = 0; j < k; ++j) {
      const int idj = __shfl_sync(0xffffffffu, my_id, j);
      const float dzj = __shfl_sync(0xffffffffu, my_dz, j);
      if (idj == e) v = dzj;
    }
    if (e < E) d_logits[(int64_t)t * E + e] = v;
  }
}

__global__ void transpose_f32_kernel(const float* __restrict__ in, int rows, int cols,
                                     float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int q = threadIdx.y; q < 32; q += blockDim.y) {
    const int r = r0 + q, c = c0 + threadIdx.x;
    if (r < rows && c < cols) tile[q][threadIdx.x] = in[(int64_t)r * cols + c];
  }
  __syncthreads();
  for (int q = threadIdx.y; q < 32; q += blockDim.y) {
    const int c = c0 + q, r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[(int64_t)c * rows + r] = tile[threadIdx.x][q];
  }
}

__global__ void __launch_bounds__(256) gather_dx_kernel(const uint16_t* __restrict__ dx_perm,
                                                        const int32_t* __restrict__ row_map,
                                                        const float* __restrict__ d_logits,
                                                        const int32_t* __restrict__ ids,
                                                        const float* __restrict__ wr_t, int T,
                                                        int H, int E, int k,
                                                        uint16_t* __restrict__ dx, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nch = H / 8;
  const int slices = (nch + kSliceChunks - 1) / kSliceChunks;
  const int gw = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int t = gw / slices;
  const int c_begin = (gw - t * slices) * kSliceChunks;
  const int c_end = min(nch, c_begin + kSliceChunks);
  if (t >= T) return;
  int my_row = 0, my_id = 0;
  float my_dz = 0.f;
  if (lane < k) {
    my_row = row_map[(int64_t)t * k + lane];
    if (my_row < 0 || (int64_t)my_row >= (int64_t)T * k) {   // not a permuted row: report, read row 0
      report_status(status, kStatusDevice, kKernCombine, 2);
      my_row = 0;
    }
    if (d_logits) {
      my_id = ids[(int64_t)t * k + lane];
      if (my_id < 0 || my_id >= E) {   // not an expert id: report, use expert 0
        report_status(status, kStatusDevice, kKernCombine, 3);
        my_id = 0;
      }
      my_dz = d_logits[(int64_t)t * E + my_id];
    }
  }
  // warp-uniform, two chunks per lane per pass, as in combine_kernel
  for (int base = c_begin; base < c_end; base += 64) {
    const int c0 = base + lane, c1 = c0 + 32;
    const bool act0 = c0 < c_end, act1 = c1 < c_end;
    float acc0[8], acc1[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      acc0[q] = 0.f;
      acc1[q] = 0.f;
    }
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
      const int row = __shfl_sync(0xffffffffu, my_row, j);
      const uint4* src = reinterpret_cast<const uint4*>(dx_perm + (int64_t)row * H);
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
      if (act0) v0 = ld_stream16(src + c0);
      if (act1) v1 = ld_stream16(src + c1);
      float f[8];
      unpack8(v0, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc0[q] += f[q];
      unpack8(v1, f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc1[q] += f[q];
    }
    if (d_logits) {
#pragma unroll 4
      for (int j = 0; j < k; ++j) {
        const int e = __shfl_sync(0xffffffffu, my_id, j);
        const float dz = __shfl_sync(0xffffffffu, my_dz, j);
        const float4* wr = reinterpret_cast<const float4*>(wr_t + (int64_t)e * H);
        if (act0) {
          const float4 a = __ldg(wr + 2 * c0), b = __ldg(wr + 2 * c0 + 1);
          acc0[0] = fmaf(dz, a.x, acc0[0]); acc0[1] = fmaf(dz, a.y, acc0[1]);
          acc0[2] = fmaf(dz, a.z, acc0[2]); acc0[3] = fmaf(dz, a.w, acc0[3]);
          acc0[4] = fmaf(dz, b.x, acc0[4]); acc0[5] = fmaf(dz, b.y, acc0[5]);
          acc0[6] = fmaf(dz, b.z, acc0[6]); acc0[7] = fmaf(dz, b.w, acc0[7]);
        }
        if (act1) {
          const float4 a = __ldg(wr + 2 * c1), b = __ldg(wr + 2 * c1 + 1);
          acc1[0] = fmaf(dz, a.x, acc1[0]); acc1[1] = fmaf(dz, a.y, acc1[1]);
          acc1[2] = fmaf(dz, a.z, acc1[2]); acc1[3] = fmaf(dz, a.w, acc1[3]);
          acc1[4] = fmaf(dz, b.x, acc1[4]); acc1[5] = fmaf(dz, b.y, acc1[5]);
          acc1[6] = fmaf(dz, b.z, acc1[6]); acc1[7] = fmaf(dz, b.w, acc1[7]);
        }
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(dx + (int64_t)t * H);
    if (act0) dst[c0] = pack8(acc0);
    if (act1) dst[c1] = pack8(acc1);
  }
}

// d_w_r[h, e] = sum_t x[t, h] * d_logits[t, e]; block tile 32 h x 64 e,
// each thread 2 x 4, T staged 32 at a time (summed in increasing t).
__global__ void __launch_bounds__(256) route_bwd_weight_kernel(const uint16_t* __restrict__ x,
                                                               const float* __restrict__ dl, int T,
                                                               int H, int E,
                                                               float* __restrict__ dwr) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) float xs[32][32];  // [t][h]
  __shared__ __align__(16) float ds[32][64];  // [t][e]
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int h0 = blockIdx.x * 32, e0 = blockIdx.y * 64;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  for (int t0 = 0; t0 < T; t0 += 32) {
    for (int q = tid; q < 32 * 32; q += 256) {
      const int tl = q / 32, hl = q % 32;
      const int t = t0 + tl, h = h0 + hl;
      xs[tl][hl] = (t < T && h < H) ? __uint_as_float((uint32_t)x[(int64_t)t * H + h] << 16) : 0.f;
    }
    for (int q = tid; q < 32 * 64; q += 256) {
      const int tl = q / 64, el = q % 64;
      const int t = t0 + tl, e = e0 + el;
      ds[tl][el] = (t < T && e < E) ? dl[(int64_t)t * E + e] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int tl = 0; tl < 32; ++tl) {
      const float2 xv = *reinterpret_cast<const float2*>(&xs[tl][ty * 2]);
      const float4 dv = *reinterpret_cast<const float4*>(&ds[tl][tx * 4]);
      acc[0][0] = fmaf(xv.x, dv.x, acc[0][0]); acc[0][1] = fmaf(xv.x, dv.y, acc[0][1]);
      acc[0][2] = fmaf(xv.x, dv.z, acc[0][2]); acc[0][3] = fmaf(xv.x, dv.w, acc[0][3]);
      acc[1][0] = fmaf(xv.y, dv.x, acc[1][0]); acc[1][1] = fmaf(xv.y, dv.y, acc[1][1]);
      acc[1][2] = fmaf(xv.y, dv.z, acc[1][2]); acc[1][3] = fmaf(xv.y, dv.w, acc[1][3]);
    }
    __syncthreads();
  }
  for (int a = 0; a < 2; ++a) {
    const int h = h0 + ty * 2 + a;
    if (h >= H) continue;
    for (int b = 0; b < 4; ++b) {
      const int e = e0 + tx * 4 + b;
      if (e < E) dwr[(int64_t)h * E + e] = acc[a][b];
    }
  }
}

}  // namespace

cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* row_map, const float* w,
                           const uint16_t* y_shared, int64_t T, int64_t H, int64_t k, uint16_t* y,
                           uint32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int64_t warps = T * ((H / 8 + kSliceChunks - 1) / kSliceChunks);
  return launch_pdl(combine_kernel, dim3((unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock)), dim3(256), 0,
                    stream, 1, y_perm, row_map, w, y_shared, (int)T, (int)H, (int)k, y, status);
}

cudaError_t launch_route_bwd(const float* dw_part, int nparts, const int32_t* row_map, const float* w,
                             const int32_t* ids, int64_t T, int64_t E, int64_t k, float* d_logits,
                             float* dw, uint32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(route_bwd_kernel, dim3((unsigned)((T + kWarpsPerBlock - 1) / kWarpsPerBlock)), dim3(256), 0,
                    stream, 1, dw_part, nparts, row_map, w, ids, (int)T, (int)E, (int)k, d_logits, dw, status);
}

size_t gather_dx_workspace_bytes(int64_t H, int64_t E) { return (size_t)(H * E * sizeof(float)); }

cudaError_t launch_gather_dx(const uint16_t* dx_perm, const int32_t* row_map, const float* d_logits,
                             const int32_t* ids, const float* w_router, int64_t T, int64_t H,
                             int64_t E, int64_t k, uint16_t* dx, void* ws, uint32_t* status,
                             cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  float* wr_t = nullptr;
  if (d_logits) {
    wr_t = static_cast<float*>(ws);
    dim3 g((unsigned)((E + 31) / 32), (unsigned)((H + 31) / 32));
    const cudaError_t err = launch_pdl(transpose_f32_kernel, g, dim3(32, 8), 0, stream, 1, w_router, (int)H,
                                       (int)E, wr_t);
    if (err != cudaSuccess) return err;
  }
  const int64_t warps = T * ((H / 8 + kSliceChunks - 1) / kSliceChunks);
  return launch_pdl(gather_dx_kernel, dim3((unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock)), dim3(256),
                    0, stream, 1, dx_perm, row_map, d_logits, ids, wr_t, (int)T, (int)H, (int)E, (int)k, dx,
                    status);
}

cudaError_t launch_route_bwd_weight(const uint16_t* x, const float* d_logits, int64_t T, int64_t H,
                                    int64_t E, float* d_w_router, cudaStream_t stream) {
  dim3 g((unsigned)((H + 31) / 32), (unsigned)((E + 63) / 64));
  return launch_pdl(route_bwd_weight_kernel, g, dim3(256), 0, stream, 1, x, d_logits, (int)T, (int)H, (int)E,
                    d_w_router);
}

}  // namespace moe
