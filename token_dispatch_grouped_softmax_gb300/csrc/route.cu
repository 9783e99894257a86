// Router: logits = x . W_r (+ bias) in fp32, then FP32 softmax, top-k and
// renormalised weights ("InternVL3.5 接入 pure FSDP2 后端开发实践",
// MindSpeed-MM issue 625, §8.2: gate -> FP32 softmax -> top-k -> 权重归一化).
//
// Kernel 1 (route_logits_kernel): a register-tiled fp32 GEMM on the CUDA
// cores.  A 256-thread block owns 32 tokens x 64 experts; each thread 2 x 4
// outputs; K (= H) is staged through shared memory 32 at a time, x widened
// exactly from bf16.  The router is < 1% of the layer's FLOPs at the
// Qwen3-MoE shape, and its fp32 precision decides the top-k, so it stays off
// the bf16 tensor cores.
//
// Kernel 2 (route_topk_kernel): one warp per token.  The k largest logits are
// picked by k rounds of a warp arg-max on (value desc, index asc), so equal
// fp32 logits go to the lower expert index; picking on the logits orders the
// experts exactly as their softmax probabilities.  With m the largest logit,
// w_j = exp(z_j - m) / sum_{i chosen} exp(z_i - m), which is p_j / sum of
// the chosen p (the softmax denominator cancels).
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRT = 32;   // tokens per block
constexpr int kRE = 64;   // experts per block
constexpr int kRK = 32;   // K chunk

__global__ void __launch_bounds__(256) route_logits_kernel(const uint16_t* __restrict__ x,
                                                           const float* __restrict__ wr,
                                                           const float* __restrict__ bias, int T,
                                                           int H, int E,
                                                           float* __restrict__ logits) {
  __shared__ __align__(16) float xs[kRK][kRT];   // [k][token]
  __shared__ __align__(16) float ws[kRK][kRE];   // [k][expert]
  const int tid = threadIdx.x;
  const int ty = tid / 16;          // token pair
  const int tx = tid % 16;          // expert quad
  const int t0 = blockIdx.x * kRT;
  const int e0 = blockIdx.y * kRE;

  float acc[2][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

  for (int k0 = 0; k0 < H; k0 += kRK) {
    {  // x tile: 32 tokens x 32 k, 4 bf16 per thread
      const int tl = tid / 8, kk = (tid % 8) * 4;
      const int t = t0 + tl;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < T) {
        if (k0 + kk + 3 < H) {
          const uint2 u = *reinterpret_cast<const uint2*>(x + (int64_t)t * H + k0 + kk);
          v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        } else {
          for (int q = 0; q < 4; ++q)
            if (k0 + kk + q < H) v[q] = __uint_as_float((uint32_t)x[(int64_t)t * H + k0 + kk + q] << 16);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) xs[kk + q][tl] = v[q];
    }
    // W_r tile: 32 k x 64 experts, 8 floats per thread
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int idx = tid + rep * 256;       // 0..511 float4 slots
      const int kk = idx / 16, eq = (idx % 16) * 4;
      const int kr = k0 + kk;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kr < H) {
        const float* src = wr + (int64_t)kr * E + e0 + eq;
        if (e0 + eq + 3 < E && (E % 4) == 0) {
          v = *reinterpret_cast<const float4*>(src);
        } else {
          float tmp[4] = {0.f, 0.f, 0.f, 0.f};
          for (int q = 0; q < 4; ++q)
            if (e0 + eq + q < E) tmp[q] = src[q];
          v = make_float4(tmp[0], tmp[1], tmp[2], tmp[3]);
        }
      }
      *reinterpret_cast<float4*>(&ws[kk][eq]) = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRK; ++kk) {
      const float2 xv = *reinterpret_cast<const float2*>(&xs[kk][ty * 2]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[kk][tx * 4]);
      acc[0][0] = fmaf(xv.x, wv.x, acc[0][0]);
      acc[0][1] = fmaf(xv.x, wv.y, acc[0][1]);
      acc[0][2] = fmaf(xv.x, wv.z, acc[0][2]);
      acc[0][3] = fmaf(xv.x, wv.w, acc[0][3]);
      acc[1][0] = fmaf(xv.y, wv.x, acc[1][0]);
      acc[1][1] = fmaf(xv.y, wv.y, acc[1][1]);
      acc[1][2] = fmaf(xv.y, wv.z, acc[1][2]);
      acc[1][3] = fmaf(xv.y, wv.w, acc[1][3]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int t = t0 + ty * 2 + a;
    if (t >= T) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int e = e0 + tx * 4 + b;
      if (e < E) logits[(int64_t)t * E + e] = acc[a][b] + (bias ? bias[e] : 0.f);
    }
  }
}

// (value, index) with larger value first, lower index first on equal values
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* z = logits + (int64_t)t * E;
  float v[32];
  const float NEG = -INFINITY;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? z[e] : NEG;
  }
  uint32_t taken = 0;
  float zmax = 0.f, esum = 0.f;
  int my_id = 0;
  float my_e = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = NEG;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == 0) zmax = bv;
    const float ez = expf(bv - zmax);
    esum += ez;
    if (lane == j) {
      my_id = bi;
      my_e = ez;
    }
  }
  if (lane < k) {
    ids[(int64_t)t * k + lane] = my_id;
    w[(int64_t)t * k + lane] = my_e / esum;
  }
}

}  // namespace

cudaError_t launch_route(const uint16_t* x, const float* w_router, const float* bias, int64_t T,
                         int64_t H, int64_t E, int64_t k, int32_t* ids, float* w, float* logits,
                         cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  dim3 g1((unsigned)((T + kRT - 1) / kRT), (unsigned)((E + kRE - 1) / kRE));
  route_logits_kernel<<<g1, 256, 0, stream>>>(x, w_router, bias, (int)T, (int)H, (int)E, logits);
  route_topk_kernel<<<(unsigned)((T + 7) / 8), 256, 0, stream>>>(logits, (int)T, (int)E, (int)k,
                                                                  ids, w);
  return cudaGetLastError();
}

}  // namespace moe
