// Router: logits = x . W_r (+ bias) in fp32, then FP32 softmax, top-k and
// renormalised weights ("InternVL3.5 接入 pure FSDP2 后端开发实践",
// MindSpeed-MM issue 625, §8.2: gate -> FP32 softmax -> top-k -> 权重归一化).
//
// Logits on the tensor cores (E % 8 == 0, H % 64 == 0): W_r is split exactly
// into three bf16 matrices, W_r = W0 + W1 + W2 (W0 = bf16(W_r), W1 =
// bf16(W_r - W0), W2 = W_r - W0 - W1, which fits bf16 exactly: 24 = 3 x 8
// significant bits; the split of an fp32 value into bf16 terms follows
// Henry, Tang & Heinecke, "Leveraging the bfloat16 artificial intelligence
// datatype for higher-precision computations", ARITH 2019).  x is exact in
// bf16, so x . W_r = x . W0 + x . W1 + x . W2 with exact products and fp32
// accumulation: the tcgen05 GEMM runs over the stacked [W0; W1; W2] (K = 3H)
// with x repeated along K, split into `parts` K ranges (one CTA tile each)
// whose fp32 partials the top-k kernel adds in a fixed order.
//
// Other shapes use route_logits_kernel: a register-tiled fp32 GEMM on the
// CUDA cores (32 tokens x 64 experts per 256-thread block).
//
// route_topk_kernel: one warp per token, NV logits per lane.  The k largest
// logits are picked by k rounds of a warp arg-max on (value desc, index
// asc), so equal fp32 logits go to the lower expert index; the logits order
// the experts exactly as their softmax probabilities.  With m the largest
// logit, w_j = exp(z_j - m) / sum_{i chosen} exp(z_i - m), which equals
// p_j / sum of the chosen p (the softmax denominator cancels).
#include <algorithm>

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

// W_r [H, E] fp32 -> [3, H, E] bf16 with W_r = W0 + W1 + W2 exactly.
__global__ void split_router_weight_kernel(const float* __restrict__ wr, int64_t n,
                                           uint16_t* __restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float w = wr[i];
    const __nv_bfloat16 w0 = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(w0);
    const __nv_bfloat16 w1 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(w1);
    const __nv_bfloat16 w2 = __float2bfloat16_rn(r2);
    out[i] = __bfloat16_as_ushort(w0);
    out[n + i] = __bfloat16_as_ushort(w1);
    out[2 * n + i] = __bfloat16_as_ushort(w2);
  }
}

// One warp per token.  z[e] = sum_p part[p][t][e] (+ bias[e]), p in
// increasing order; NV = logits per lane (E <= 32 * NV).
template <int NV>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ part, int nparts,
                                                         const float* __restrict__ bias, int T, int E,
                                                         int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w,
                                                         float* __restrict__ logits_out) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const float NEG = -INFINITY;
  float v[NV];
  // partials added in increasing part order; the NV loads of one part are
  // independent, and the part loop is unrolled so the loads overlap
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(part + (int64_t)t * E + e) : 0.f;
  }
#pragma unroll 4
  for (int q = 1; q < nparts; ++q) {
    const float* pq = part + ((int64_t)q * T + t) * E;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      if (e < E) v[i] += __ldg(pq + e);
    }
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      if (bias) v[i] += bias[e];
      if (logits_out) logits_out[(int64_t)t * E + e] = v[i];
    } else {
      v[i] = NEG;
    }
  }
  float zmax = 0.f, esum = 0.f;
  int my_id = 0;
  float my_e = 0.f;
  uint32_t taken = 0;               // bit i: expert lane + 32 i already chosen
  for (int j = 0; j < k; ++j) {
    float bv = NEG;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
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

template <int NV>
void launch_topk(const float* part, int nparts, const float* bias, int64_t T, int64_t E, int64_t k,
                 int32_t* ids, float* w, float* logits_out, cudaStream_t stream) {
  route_topk_kernel<NV><<<(unsigned)((T + 7) / 8), 256, 0, stream>>>(part, nparts, bias, (int)T, (int)E,
                                                                     (int)k, ids, w, logits_out);
}

void topk_dispatch(const float* part, int nparts, const float* bias, int64_t T, int64_t E, int64_t k,
                   int32_t* ids, float* w, float* logits_out, cudaStream_t stream) {
  if (E <= 32) launch_topk<1>(part, nparts, bias, T, E, k, ids, w, logits_out, stream);
  else if (E <= 64) launch_topk<2>(part, nparts, bias, T, E, k, ids, w, logits_out, stream);
  else if (E <= 128) launch_topk<4>(part, nparts, bias, T, E, k, ids, w, logits_out, stream);
  else if (E <= 256) launch_topk<8>(part, nparts, bias, T, E, k, ids, w, logits_out, stream);
  else if (E <= 512) launch_topk<16>(part, nparts, bias, T, E, k, ids, w, logits_out, stream);
  else launch_topk<32>(part, nparts, bias, T, E, k, ids, w, logits_out, stream);
}

}  // namespace

bool route_on_tensor_cores(int64_t H, int64_t E) { return E % 8 == 0 && H % 64 == 0; }

size_t route_workspace_bytes(int64_t T, int64_t H, int64_t E) {
  auto align = [](size_t b) { return (b + 255) & ~size_t(255); };
  if (route_on_tensor_cores(H, E)) {
    const int parts = router_parts(T, H, E);
    return align((size_t)(3 * H * E * 2)) + align((size_t)(parts * T * E * 4));
  }
  return align((size_t)(T * E * 4));
}

cudaError_t launch_route(const uint16_t* x, const float* w_router, const float* bias, int64_t T,
                         int64_t H, int64_t E, int64_t k, int32_t* ids, float* w, float* logits,
                         void* ws, const DeviceInfo& dev, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  auto align = [](size_t b) { return (b + 255) & ~size_t(255); };
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  if (route_on_tensor_cores(H, E)) {
    const int parts = router_parts(T, H, E);
    uint16_t* w_split = reinterpret_cast<uint16_t*>(wsb);
    float* part = reinterpret_cast<float*>(wsb + align((size_t)(3 * H * E * 2)));
    const int64_t n = H * E;
    split_router_weight_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, stream>>>(
        w_router, n, w_split);
    if (launch_router_logits(x, w_split, T, H, E, parts, part, dev, stream) != 0) return cudaErrorInvalidValue;
    topk_dispatch(part, parts, bias, T, E, k, ids, w, logits, stream);
  } else {
    float* lg = reinterpret_cast<float*>(wsb);
    dim3 g1((unsigned)((T + kRT - 1) / kRT), (unsigned)((E + kRE - 1) / kRE));
    route_logits_kernel<<<g1, 256, 0, stream>>>(x, w_router, nullptr, (int)T, (int)H, (int)E, lg);
    topk_dispatch(lg, 1, bias, T, E, k, ids, w, logits, stream);
  }
  return cudaGetLastError();
}

}  // namespace moe
