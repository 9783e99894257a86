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
// With 16 <= E <= 256 and E % 16 == 0 one fused kernel also picks the top
// k: a cluster of CTAs per 128-token tile splits K and sums its fp32
// partials over distributed shared memory (fused_router_kernel below).
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
  pdl_wait();
  pdl_trigger();
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

// W_r [H, E] fp32 -> [3, H, E] bf16 with W_r = W0 + W1 + W2 exactly.
__global__ void split_router_weight_kernel(const float* __restrict__ wr, int64_t n,
                                           uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
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

// Order-preserving 64-bit key of (logit v, expert e): larger v gives a
// larger key, and on equal v the lower expert index does (the float's bits
// are mapped to an unsigned order, the index is stored complemented).
__device__ __forceinline__ uint64_t topk_key(float v, int e) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
}
__device__ __forceinline__ float topk_key_value(uint64_t key) {
  uint32_t u = (uint32_t)(key >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}
__device__ __forceinline__ int topk_key_index(uint64_t key) { return (int)(0xFFFFFFFFu - (uint32_t)key); }

// Expert held in v[i] by lane `lane`: l + 32 i, or with QUAD 128 (i / 4) +
// 4 l + i % 4 (four consecutive experts per lane, read as one vector).
template <bool QUAD>
__device__ __forceinline__ int topk_expert(int lane, int i) {
  return QUAD ? 128 * (i / 4) + 4 * lane + (i % 4) : lane + 32 * i;
}

// Top k of one token's logits, warp-wide: lane l holds z[topk_expert(l, i)]
// in v[i] (the partial sums, before the bias).  Adds the bias, writes the logits
// when asked, and writes the ids and renormalised weights.  Each lane sorts
// its NV keys; round j takes the warp maximum of the lanes' leading keys
// (warp reductions) and the lane that held it drops it.  The keys
// are distinct (they carry the index), so the order is the (value desc,
// index asc) order; w_j = exp(z_j - z_0) / sum_j exp(z_j - z_0), summed in
// increasing j.
template <int NV, bool QUAD = false>
__device__ __forceinline__ void topk_row(float (&v)[NV], int64_t t, int E, int k, int lane,
                                         const float* __restrict__ bias, int32_t* __restrict__ ids,
                                         float* __restrict__ w, float* __restrict__ logits_out) {
  uint64_t key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = topk_expert<QUAD>(lane, i);
    key[i] = 0;   // below every logit's key
    if (e < E) {
      if (bias) v[i] += bias[e];
      if (logits_out) logits_out[t * E + e] = v[i];
      key[i] = topk_key(v[i], e);
    }
  }
#pragma unroll
  for (int a = 0; a < NV - 1; ++a)     // descending, by adjacent compare-exchanges
#pragma unroll
    for (int b = NV - 1; b > a; --b)
      if (key[b] > key[b - 1]) {
        const uint64_t tmp = key[b];
        key[b] = key[b - 1];
        key[b - 1] = tmp;
      }
  uint64_t mine = 0;   // lane j < k: the j-th chosen key
  for (int j = 0; j < k; ++j) {
    // warp maximum of the leading keys: of the value bits, then of the
    // index bits among the lanes holding that value (two warp reductions)
    const uint32_t hi = (uint32_t)(key[0] >> 32), lo = (uint32_t)key[0];
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
    const uint64_t m = ((uint64_t)mhi << 32) | mlo;
    if (key[0] == m) {   // this lane held it
#pragma unroll
      for (int i = 0; i < NV - 1; ++i) key[i] = key[i + 1];
      key[NV - 1] = 0;
    }
    if (lane == j) mine = m;
  }
  const float zmax = topk_key_value(__shfl_sync(0xffffffffu, mine, 0));
  const float ez = lane < k ? expf(topk_key_value(mine) - zmax) : 0.f;
  float esum = 0.f;
  for (int j = 0; j < k; ++j) esum += __shfl_sync(0xffffffffu, ez, j);
  if (lane < k) {
    ids[t * k + lane] = topk_key_index(mine);
    w[t * k + lane] = ez / esum;
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
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
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
  topk_row<NV>(v, t, E, k, lane, bias, ids, w, logits_out);
}

// ---------------------------------------------------------------------------
// Fused router (E % 16 == 0, 16 <= E <= 256, H % 64 == 0).  One cluster of P
// CTAs per 128-token tile splits K into P equal ranges.  CTA c accumulates
// its range in TMEM (tcgen05.mma, M = 128, N = E, bf16 x bf16 -> fp32; warp
// 0 loads x and W tiles by TMA, warp 1 issues the MMAs), warps 2..5 copy the
// fp32 partial tile into shared memory (over the emptied operand ring), and
// after a cluster barrier each CTA sums, for its share of the tile's rows,
// the P partials over distributed shared memory in increasing CTA rank and
// picks the top k of each row.  No partial logits reach HBM.
//   E <= 128: a stage holds one 64-wide K block of x and of all three terms
//             W0, W1, W2 (x loaded once for the three); K = H is split.
//   E > 128:  a stage holds one K block of the stacked K = 3H of [W0; W1; W2]
//             and the x block it multiplies.
// Waits are bounded (MOE_ERR_TIMEOUT in the status word).
// Threads per CTA: warps 0..5 take the roles above; then every warp picks
// the top k of rows of the tile, one row at a time.  With E <= 128 a CTA has
// 32 warps, so a cluster of 4 has one warp per row of its 128-token tile;
// with E > 128 (more registers per lane) 12.
template <int NV>
__host__ __device__ constexpr int fr_threads() { return NV <= 4 ? 1024 : 384; }
// Ring stages: three of 64 KB with three terms per stage (E <= 128, NV = 4);
// four of 48 KB with one (E > 128, NV = 8).  Either ring is 192 KB.  At the
// DeepSeek-V3 shape four stages measured 217.7 us against 221.9 with three.
template <int NV>
__host__ __device__ constexpr int fr_stages() { return NV <= 4 ? 3 : 4; }
constexpr int kFrMaxStages = 4;
constexpr int kFrMaxCluster = 4;   // fused_router_cluster returns 1 to 4
constexpr int kFrABytes = 128 * 64 * 2;     // 128 tokens x 64 K
constexpr int kFrChunkBytes = 64 * 64 * 2;  // 64 K x 64 experts

struct FusedRouterParams {
  CUtensorMap tmA;   // x [T, H] bf16, boxes of 64 K x 128 tokens, 128-byte swizzle
  CUtensorMap tmB;   // [W0; W1; W2] [3H, E] bf16, boxes of 64 experts x 64 K
  const float* bias;
  int32_t* ids;
  float* w;
  float* logits;
  uint32_t* status;
  uint64_t wait_limit_ns;
  int T, H, E, k;
  int kblocks;       // 64-wide K blocks per CTA
  int nchunks;       // 64-expert chunks of a B tile: ceil(E / 64)
  int terms;         // W terms per stage: 3 (K = H split), or 1 (K = 3H split)
  uint32_t tmem_cols;
};

__host__ __device__ inline int fr_stage_bytes(int nchunks, int terms) {
  return kFrABytes + terms * nchunks * kFrChunkBytes;
}

template <int NV>
__global__ void __launch_bounds__(fr_threads<NV>(), 1) fused_router_kernel(const __grid_constant__ FusedRouterParams p) {
  constexpr int kWarps = fr_threads<NV>() / 32;
  extern __shared__ uint8_t fr_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fr_raw) + 1023) & ~uintptr_t(1023));
  const int stage_bytes = fr_stage_bytes(p.nchunks, p.terms);
  uint8_t* ring = smem;
  constexpr int kFrStages = fr_stages<NV>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFrStages * stage_bytes);   // full[S], empty[S], accf, drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kFrStages + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // the partial tile [128][E + 4] (16-byte aligned rows) over the ring, once
  // the MMAs are done
  float* part = reinterpret_cast<float*>(smem);
  const int ldp = p.E + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = (int)cluster_nctas();
  const int crank = (int)cluster_ctarank();
  const int row0 = (blockIdx.x / P) * 128;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kFrStages + s); };
  const uint32_t accf_bar = bar0 + 8u * (2 * kFrStages);
  const uint32_t drain_bar = bar0 + 8u * (2 * kFrStages + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFrStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(accf_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  pdl_wait();      // the set-up above overlaps the kernel before this one
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int kb0 = crank * p.kblocks;   // first K block of this CTA (of H, or of the stacked 3H)

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, last_par = 0;
    bool ok = true;
    for (int kb = 0; kb < p.kblocks; ++kb) {
      ok = mbar_wait_warp(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit_ns, p.status, 1, kKernRoute);
      if (!ok) break;
      if (lane == 0) {
        const uint32_t fb = full_bar(stage);
        const uint32_t sA = smem_u32(ring + stage * stage_bytes);
        const int kg = (kb0 + kb) * 64;   // K row: of H (three terms), or of the stacked 3H
        mbar_arrive_expect_tx(fb, (uint32_t)stage_bytes);
        tma_load_2d(sA, &p.tmA, kg % p.H, row0, fb);   // x repeats along the stacked K
        for (int q = 0; q < p.terms; ++q)              // term q: rows q*H + kg of [W0; W1; W2]
          for (int c = 0; c < p.nchunks; ++c)
            tma_load_2d(sA + kFrABytes + (q * p.nchunks + c) * kFrChunkBytes, &p.tmB, 64 * c, q * p.H + kg, fb);
      }
      __syncwarp();
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == kFrStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {   // stopped early: wait (bounded) for the copies in flight
      for (int s = 0; s < kFrStages; ++s)
        if (issued & (1u << s)) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(full_bar(s), (last_par >> s) & 1u) && globaltimer_ns() - t0 < p.wait_limit_ns) {
          }
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    // D fp32, A bf16 K-major, B bf16 MN-major, M = 128.  One term (K = 3H
    // stacked): N = E.  Three terms: the stage holds the terms' 64-expert
    // chunks side by side (term q, chunk c at q * nchunks + c), so each MMA
    // takes up to four chunks (N = 256) into the TMEM columns of the same
    // index; term q's partial logits are then at columns 64 q nchunks + e
    // and the drain adds them.  Two MMAs per K step at E = 128, not three.
    auto idesc_n = [](int n) {
      return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    };
    const int nch = p.terms * p.nchunks;                   // chunks in a stage's B
    const int per_mma = p.terms == 3 ? 4 : p.nchunks;      // chunks per MMA
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true, issued_any = false;
    for (int kb = 0; kb < p.kblocks; ++kb) {
      ok = mbar_wait_warp(full_bar(stage), phase, abort_flag, p.wait_limit_ns, p.status, 2, kKernRoute);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sA = smem_u32(ring + stage * stage_bytes);
        for (int j0 = 0; j0 < nch; j0 += per_mma) {
          const int nj = nch - j0 < per_mma ? nch - j0 : per_mma;
          const uint32_t idesc = idesc_n(p.terms == 3 ? 64 * nj : p.E);
          const uint32_t sB = sA + kFrABytes + j0 * kFrChunkBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(tmem_base + 64u * (uint32_t)j0, umma_desc(sA + kk * 32, 16, 1024),
                        umma_desc(sB + kk * 2048, kFrChunkBytes, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        tc_commit(empty_bar(stage));
      }
      issued_any = true;
      __syncwarp();
      if (++stage == kFrStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (lane == 0) {
      if (ok) {
        tc_commit(accf_bar);
      } else if (issued_any) {   // make sure every MMA issued has finished before TMEM is freed
        tc_commit(drain_bar);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain_bar, 0) && globaltimer_ns() - t0 < p.wait_limit_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------- partial tile: TMEM -> shared
    // every lane acquires the accumulator itself before the warp reads it
    if (mbar_wait_warp(accf_bar, 0, abort_flag, p.wait_limit_ns, p.status, 3, kKernRoute)) {
      tc_fence_after();
      const int quarter = warp & 3;              // TMEM lanes 32 quarter .. +31
      const int r = quarter * 32 + lane;         // tile row of this thread
      float* prow = part + r * ldp;
      const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
      if (p.terms == 3) {
        // (term 0 + term 1) + term 2, 16 columns at a time
        const uint32_t cs = 64u * (uint32_t)p.nchunks;
        for (int c0 = 0; c0 < p.E; c0 += 16) {   // E % 16 == 0
          float v[16], u[16];
          tmem_ld16(lane_base + (uint32_t)c0, v);
          tmem_ld16(lane_base + cs + (uint32_t)c0, u);
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] += u[q];
          tmem_ld16(lane_base + 2u * cs + (uint32_t)c0, u);
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] += u[q];
#pragma unroll
          for (int q = 0; q < 16; q += 4)
            *reinterpret_cast<float4*>(prow + c0 + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
        }
      } else {
        for (int c0 = 0; c0 < p.E; c0 += 32) {   // E % 16 == 0: 4-column groups are whole
          float v[32];
          tmem_ld32(lane_base + (uint32_t)c0, v);
#pragma unroll
          for (int q = 0; q < 32; q += 4)
            if (c0 + q < p.E) *reinterpret_cast<float4*>(prow + c0 + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
        }
      }
    }
  }

  // every CTA's partial tile is in its shared memory
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  // ------------------------------------------------ reduce and pick top k
  // rows crank, crank + P, ... of the tile, one warp per row
  const uint32_t part_u32 = smem_u32(part);
  for (int r = crank + P * warp; r < 128; r += P * kWarps) {
    const int64_t t = row0 + r;
    if (t >= p.T) break;
    // all remote loads first (they overlap), four consecutive experts per
    // lane and load; then the sums in increasing CTA rank
    float4 xs[kFrMaxCluster][NV / 4];
    const uint32_t row_addr = part_u32 + (uint32_t)(r * ldp) * 4u;
#pragma unroll
    for (int c = 0; c < kFrMaxCluster; ++c) {
      if (c < P) {
        const uint32_t base = mapa_shared(row_addr, (uint32_t)c);
#pragma unroll
        for (int q = 0; q < NV / 4; ++q) {
          const int e = topk_expert<true>(lane, 4 * q);
          xs[c][q] = e < p.E ? ld_shared_cluster_f32x4(base + 4u * (uint32_t)e) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    float v[NV];
#pragma unroll
    for (int q = 0; q < NV / 4; ++q) {
      float4 a = xs[0][q];
#pragma unroll
      for (int c = 1; c < kFrMaxCluster; ++c)
        if (c < P) {
          a.x += xs[c][q].x;
          a.y += xs[c][q].y;
          a.z += xs[c][q].z;
          a.w += xs[c][q].w;
        }
      v[4 * q] = a.x;
      v[4 * q + 1] = a.y;
      v[4 * q + 2] = a.z;
      v[4 * q + 3] = a.w;
    }
    topk_row<NV, true>(v, t, p.E, p.k, lane, p.bias, p.ids, p.w, p.logits);
  }
  // no CTA leaves (or frees its TMEM) while another may still read its partials
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

int fused_router_terms(int64_t E) { return E <= 128 ? 3 : 1; }

// The cluster size, which is how K is split and so the order in which each
// logit's fp32 partial sums add up: a function of H and E alone, so that a
// token's logits, weights and experts do not depend on how many tokens are
// routed with it (the same bits for a batch of 512 tokens as for 4096; an
// expert-parallel rank routing its share of a batch gets what routing the
// whole batch gives).  With three terms per stage: the largest divisor of the
// K blocks up to 4 (4: one wave of 128 clusters at 4096 tokens, the largest
// count a single wave of 152 SMs takes at that size).  With one term per
// stage (the stacked K = 3H): 3, so that each CTA of a cluster takes one of
// W_r's three terms over the whole of H.  Measured at the DeepSeek-V3 shape
// (T = 16384, H = 7168, E = 256), router alone, L2 flushed: 313.5 us with
// clusters of 8, 250.5 with 6, 234.1 with 4, 221.9 with 3, 230.0 with 2.
int fused_router_cluster(int64_t H, int64_t E) {
  const int terms = fused_router_terms(E);
  if (terms == 1) return 3;   // 3H / 64 K blocks: three parts of H / 64
  const int64_t kb = H / 64;
  for (int d = 4; d > 1; --d)
    if (kb % d == 0) return d;
  return 1;
}

bool fused_router_ok(int64_t H, int64_t E) { return H % 64 == 0 && E % 16 == 0 && E >= 16 && E <= 256; }

size_t fused_router_smem(int64_t E) {
  const int stages = E <= 128 ? fr_stages<4>() : fr_stages<8>();
  return 1024 + (size_t)stages * fr_stage_bytes((int)((E + 63) / 64), fused_router_terms(E)) +
         8 * (2 * kFrMaxStages + 2) + 16;
}

template <int NV>
cudaError_t launch_fused_router_nv(const FusedRouterParams& p, int P, int64_t T, const DeviceInfo& dev,
                                   cudaStream_t stream) {
  static std::atomic<int> configured[kMaxDevices] = {};   // per device (a race only repeats the set-up)
  if (!configured[dev.ordinal].load()) {
    const cudaError_t err = cudaFuncSetAttribute(fused_router_kernel<NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)std::max(fused_router_smem(128), fused_router_smem(256)));
    if (err != cudaSuccess) return err;
    configured[dev.ordinal].store(1);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned)(((T + 127) / 128) * P));
  cfg.blockDim = dim3(fr_threads<NV>());
  cfg.dynamicSmemBytes = fused_router_smem(p.E);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = g_pdl.load(std::memory_order_relaxed) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fused_router_kernel<NV>, p);
}

cudaError_t launch_fused_router(const uint16_t* x, const uint16_t* w_split, const float* bias, int64_t T, int64_t H,
                                int64_t E, int64_t k, int32_t* ids, float* w, float* logits, const DeviceInfo& dev,
                                cudaStream_t stream) {
  FusedRouterParams p;
  const cuuint32_t estr[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)(H * 2)};
    const cuuint32_t box[2] = {64, 128};
    if (!encode_tensor_map_2d_bf16(&p.tmA, x, dims, strides, box, estr)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)(3 * H)};
    const cuuint64_t strides[1] = {(cuuint64_t)(E * 2)};
    const cuuint32_t box[2] = {64, 64};
    if (!encode_tensor_map_2d_bf16(&p.tmB, w_split, dims, strides, box, estr)) return cudaErrorInvalidValue;
  }
  const int P = fused_router_cluster(H, E);
  p.bias = bias;
  p.ids = ids;
  p.w = w;
  p.logits = logits;
  p.status = dev.status;
  p.wait_limit_ns = dev.wait_limit_ns;
  p.T = (int)T;
  p.H = (int)H;
  p.E = (int)E;
  p.k = (int)k;
  p.terms = fused_router_terms(E);
  p.kblocks = (int)((p.terms == 3 ? 1 : 3) * H / 64 / P);
  p.nchunks = (int)((E + 63) / 64);
  // three terms: 3 x 64 nchunks columns (192 or 384); one term: E
  const int64_t cols = p.terms == 3 ? 3 * 64 * p.nchunks : E;
  p.tmem_cols = cols <= 32 ? 32u : cols <= 64 ? 64u : cols <= 128 ? 128u : cols <= 256 ? 256u : 512u;
  // NV: logits per lane, four consecutive experts per vector
  if (E <= 128) return launch_fused_router_nv<4>(p, P, T, dev, stream);
  return launch_fused_router_nv<8>(p, P, T, dev, stream);
}

template <int NV>
void launch_topk(const float* part, int nparts, const float* bias, int64_t T, int64_t E, int64_t k,
                 int32_t* ids, float* w, float* logits_out, cudaStream_t stream) {
  launch_pdl(route_topk_kernel<NV>, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, stream, 1, part, nparts, bias,
             (int)T, (int)E, (int)k, ids, w, logits_out);
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
  if (fused_router_ok(H, E)) return align((size_t)(3 * H * E * 2));
  if (route_on_tensor_cores(H, E)) {
    const int parts = router_parts(T, H, E);
    return align((size_t)(3 * H * E * 2)) + align((size_t)(parts * T * E * 4));
  }
  return align((size_t)(T * E * 4));
}

size_t route_presplit_workspace_bytes(int64_t T, int64_t H, int64_t E) {
  auto align = [](size_t b) { return (b + 255) & ~size_t(255); };
  if (fused_router_ok(H, E)) return 0;
  return align((size_t)(router_parts(T, H, E) * T * E * 4));
}

cudaError_t launch_route_split(const float* w_router, int64_t H, int64_t E, uint16_t* w_split,
                               cudaStream_t stream) {
  const int64_t n = H * E;
  if (n == 0) return cudaSuccess;
  return launch_pdl(split_router_weight_kernel, dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4096)), dim3(256),
                    0, stream, 1, w_router, n, w_split);
}

// The router on a split of W_r prepared once (launch_route_split): the same
// kernels as launch_route on the tensor-core path, without the split.
cudaError_t launch_route_presplit(const uint16_t* x, const uint16_t* w_split, const float* bias, int64_t T,
                                  int64_t H, int64_t E, int64_t k, int32_t* ids, float* w, float* logits,
                                  void* ws, const DeviceInfo& dev, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (fused_router_ok(H, E)) return launch_fused_router(x, w_split, bias, T, H, E, k, ids, w, logits, dev, stream);
  const int parts = router_parts(T, H, E);
  float* part = static_cast<float*>(ws);
  if (launch_router_logits(x, w_split, T, H, E, parts, part, dev, stream) != 0) return cudaErrorInvalidValue;
  topk_dispatch(part, parts, bias, T, E, k, ids, w, logits, stream);
  return cudaGetLastError();
}

cudaError_t launch_route(const uint16_t* x, const float* w_router, const float* bias, int64_t T,
                         int64_t H, int64_t E, int64_t k, int32_t* ids, float* w, float* logits,
                         void* ws, const DeviceInfo& dev, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  auto align = [](size_t b) { return (b + 255) & ~size_t(255); };
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  if (fused_router_ok(H, E)) {
    uint16_t* w_split = reinterpret_cast<uint16_t*>(wsb);
    const int64_t n = H * E;
    cudaError_t err = launch_pdl(split_router_weight_kernel, dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4096)),
                                 dim3(256), 0, stream, 1, w_router, n, w_split);
    if (err == cudaSuccess) err = launch_fused_router(x, w_split, bias, T, H, E, k, ids, w, logits, dev, stream);
    if (err != cudaSuccess) return err;
  } else if (route_on_tensor_cores(H, E)) {
    const int parts = router_parts(T, H, E);
    uint16_t* w_split = reinterpret_cast<uint16_t*>(wsb);
    float* part = reinterpret_cast<float*>(wsb + align((size_t)(3 * H * E * 2)));
    const int64_t n = H * E;
    const cudaError_t err = launch_pdl(split_router_weight_kernel,
                                       dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4096)), dim3(256), 0,
                                       stream, 1, w_router, n, w_split);
    if (err != cudaSuccess) return err;
    if (launch_router_logits(x, w_split, T, H, E, parts, part, dev, stream) != 0) return cudaErrorInvalidValue;
    topk_dispatch(part, parts, bias, T, E, k, ids, w, logits, stream);
  } else {
    float* lg = reinterpret_cast<float*>(wsb);
    dim3 g1((unsigned)((T + kRT - 1) / kRT), (unsigned)((E + kRE - 1) / kRE));
    const cudaError_t err = launch_pdl(route_logits_kernel, g1, dim3(256), 0, stream, 1, x, w_router,
                                       (const float*)nullptr, (int)T, (int)H, (int)E, lg);
    if (err != cudaSuccess) return err;
    topk_dispatch(lg, 1, bias, T, E, k, ids, w, logits, stream);
  }
  return cudaGetLastError();
}

}  // namespace moe
