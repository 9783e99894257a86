// Permute: group the R = T*k (token, slot) assignments by expert
// ("Awesome-ML-SYS-Tutorial" MoE/EP guide, gsyq.cn, "Expert Parallelism":
// per-expert token counts, then permute so each expert's tokens are
// contiguous; "InternVL3.5 接入 pure FSDP2 后端开发实践" §8.3: permute).
//
// Deterministic three-pass counting sort, no order-dependent atomics:
//   1. permute_hist_kernel   block b counts the ids of its chunk of
//                            CHUNK assignments -> hist[b][e]
//   2. permute_scan_kernel   one block: counts[e] = sum_b hist[b][e];
//                            offsets = exclusive scan; hist[b][e] becomes
//                            offsets[e] + sum_{b'<b} hist[b'][e] (each
//                            expert's blocks split over G threads)
//   3. permute_scatter_kernel block b ranks its chunk stably: warp w owns a
//                            contiguous slice, warp bases come from a scan of
//                            per-warp counts, and inside a warp step the
//                            lanes holding the same expert rank themselves
//                            with __match_any_sync (lower lane = lower i).
// Outputs: counts, offsets, row_map[i] (permuted row of assignment i),
// src_row[row] = i / k, and optionally w_perm[row] = w[i] (the gate weight
// travelling with its row).  Workspace: hist, nblocks * E int32.
#include <mutex>

#include "../../include/moe_gb300.h"
#include "kernels.h"

namespace moe {

namespace {

// Assignments per block: 256 (one 32-wide step per warp) fill the GPU at a
// few thousand tokens; moe_permute_noalloc keeps 2048, which its fixed
// scratch limit is stated in.
constexpr int kChunk = 256;
constexpr int kChunkNoAlloc = 2048;
constexpr int kPermThreads = 256;
constexpr int kPermWarps = kPermThreads / 32;

template <int CHUNK>
__global__ void __launch_bounds__(kPermThreads) permute_hist_kernel(const int32_t* __restrict__ ids,
                                                                    int64_t R, int E,
                                                                    int32_t* __restrict__ hist,
                                                                    uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int32_t sh[];  // [E]
  for (int e = threadIdx.x; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * CHUNK;
  for (int q = threadIdx.x; q < CHUNK; q += blockDim.x) {
    const int64_t i = base + q;
    if (i < R) {
      const int e = ids[i];
      if (e < 0 || e >= E) {
        report_status(status, kStatusDevice, kKernPermute, 1);
      } else {
        atomicAdd(&sh[e], 1);   // counts only: the order of increments is irrelevant
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(int64_t)blockIdx.x * E + e] = sh[e];
}

// One block of 1024 threads.  Each expert's block histograms are split into
// G = 1024 / E contiguous ranges of blocks, one thread per (range, expert):
// range sums, then per expert the total and the exclusive scan over
// experts, then each thread rewrites its range with running bases.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int32_t* __restrict__ hist, int nblocks,
                                                            int E, int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t part[1024];     // [G][E] range sums, then exclusive range prefixes
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t ex[1024];       // offsets[e]
  const int tid = threadIdx.x;
  const int G = 1024 / E;            // E <= 1024
  const int g = tid / E, e = tid - (tid / E) * E;
  const bool act = g < G;
  const int per = (nblocks + G - 1) / G;
  const int b0 = min(nblocks, g * per), b1 = min(nblocks, b0 + per);
  if (act) {
    int32_t sum = 0;
#pragma unroll 8
    for (int b = b0; b < b1; ++b) sum += hist[(int64_t)b * E + e];
    part[g * E + e] = sum;
  }
  __syncthreads();
  // per expert (thread tid = e < E): the total, and the ranges' exclusive prefixes
  int32_t c = 0;
  if (tid < E) {
    for (int gg = 0; gg < G; ++gg) {
      const int32_t v = part[gg * E + tid];
      part[gg * E + tid] = c;
      c += v;
    }
  }
  // exclusive scan of c over e (block of 1024 threads = 32 warps)
  const int lane = tid & 31, wid = tid >> 5;
  int32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int32_t v = warp_tot[lane];
    int32_t s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    warp_tot[lane] = s - v;   // exclusive prefix of warp totals
  }
  __syncthreads();
  if (tid < E) {
    const int32_t excl = incl - c + warp_tot[wid];
    counts[tid] = c;
    offsets[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + c;
    ex[tid] = excl;
  }
  __syncthreads();
  if (act) {
    // eight reads in flight before the writes (the array is read and written)
    int32_t run = ex[e] + part[g * E + e];
    for (int b = b0; b < b1; b += 8) {
      int32_t h[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) h[q] = (b + q < b1) ? hist[(int64_t)(b + q) * E + e] : 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (b + q < b1) hist[(int64_t)(b + q) * E + e] = run;
        run += h[q];
      }
    }
  }
}

template <int CHUNK>
__global__ void __launch_bounds__(kPermThreads) permute_scatter_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int64_t R, int k, int E,
    const int32_t* __restrict__ base_be, int32_t* __restrict__ row_map, int32_t* __restrict__ src_row,
    float* __restrict__ w_perm) {
  pdl_wait();
  pdl_trigger();
  constexpr int kPerWarp = CHUNK / kPermWarps;  // assignments per warp, in steps of 32
  extern __shared__ int32_t sh[];              // [kPermWarps][E] counts, then bases
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t chunk0 = (int64_t)blockIdx.x * CHUNK;
  const int64_t slice0 = chunk0 + (int64_t)wid * kPerWarp;
  for (int q = threadIdx.x; q < kPermWarps * E; q += blockDim.x) sh[q] = 0;
  __syncthreads();
  // per-warp counts of its slice
  for (int s = 0; s < kPerWarp; s += 32) {
    const int64_t i = slice0 + s + lane;
    if (i < R) {
      const int e = ids[i];
      if (e >= 0 && e < E) atomicAdd(&sh[wid * E + e], 1);
    }
  }
  __syncthreads();
  // per expert: exclusive scan over warps, plus the block's global base
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = base_be[(int64_t)blockIdx.x * E + e];
    for (int w = 0; w < kPermWarps; ++w) {
      const int32_t c = sh[w * E + e];
      sh[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // stable ranking inside the warp's slice, 32 assignments per step
  int32_t* my = sh + wid * E;
  for (int s = 0; s < kPerWarp; s += 32) {
    const int64_t i = slice0 + s + lane;
    const bool valid = i < R;
    int e = valid ? ids[i] : -1;
    if (e < 0 || e >= E) e = E + lane;        // unique key: matches no other lane
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const uint32_t lower = peers & ((1u << lane) - 1u);
    if (e < E) {
      const int32_t row = my[e] + __popc(lower);
      row_map[i] = row;
      src_row[row] = (int32_t)(i / k);
      if (w_perm) w_perm[row] = w[i];
    }
    __syncwarp();
    // the highest lane of each group advances that expert's running base
    if (e < E && (peers >> lane) == 1u) my[e] += __popc(peers);
    __syncwarp();
  }
}

// ------------------------------------------------------------------------
// The same counting sort in one cooperative launch (every block resident at
// once), its three passes separated by two grid barriers:
//   1. block b counts its chunk per warp (kept in shared memory) and writes
//      its block histogram hist[b][e];
//   2. warp g of the grid scans expert column e = g, g + G, ...: hist[b][e]
//      becomes sum_{b' < b} hist[b'][e], totals[e] the column sum;
//   3. every block scans the totals over experts (offsets; block 0 writes
//      counts and offsets), forms its warps' bases offsets[e] + hist[b][e] +
//      the counts of its lower warps, and ranks its chunk stably.
// Each barrier is an arrival counter (zeroed by the host before the launch)
// that a block's thread 0 waits on with a bounded spin; a wait that runs out
// records MOE_ERR_TIMEOUT and ends the block.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ bool grid_barrier(uint32_t* count, uint32_t nblocks, uint64_t limit_ns,
                                             uint32_t* status, uint32_t site, int* ok_sh) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(count, 1u);
    bool ok = true;
    if (ld_acquire_gpu(count) < nblocks) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(count) < nblocks) {
        if (globaltimer_ns() - t0 > limit_ns) {
          report_status(status, kStatusTimeout, kKernPermute, site);
          ok = false;
          break;
        }
      }
    }
    __threadfence();
    *ok_sh = ok ? 1 : 0;
  }
  __syncthreads();
  return *ok_sh != 0;
}

template <int CHUNK>
__global__ void __launch_bounds__(kPermThreads) permute_fused_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int64_t R, int k, int E,
    int32_t* __restrict__ hist, int32_t* __restrict__ totals, uint32_t* __restrict__ bar,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ row_map,
    int32_t* __restrict__ src_row, float* __restrict__ w_perm, uint32_t* status, uint64_t wait_limit_ns) {
  pdl_wait();
  pdl_trigger();
  constexpr int kPerWarp = CHUNK / kPermWarps;
  extern __shared__ int32_t sh[];   // [kPermWarps][E] warp counts, then bases; [E] offsets; [32] scan
  int32_t* off = sh + kPermWarps * E;
  int32_t* wtot = off + E;
  __shared__ int ok_sh;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nb = gridDim.x;
  const int64_t slice0 = (int64_t)blockIdx.x * CHUNK + (int64_t)wid * kPerWarp;

  // 1. per-warp counts and the block histogram
  for (int q = threadIdx.x; q < kPermWarps * E; q += blockDim.x) sh[q] = 0;
  __syncthreads();
  for (int s = 0; s < kPerWarp; s += 32) {
    const int64_t i = slice0 + s + lane;
    if (i < R) {
      const int e = ids[i];
      if (e < 0 || e >= E) report_status(status, kStatusDevice, kKernPermute, 1);
      else atomicAdd(&sh[wid * E + e], 1);   // counts only: the order of increments is irrelevant
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t c = 0;
    for (int w2 = 0; w2 < kPermWarps; ++w2) c += sh[w2 * E + e];
    hist[(int64_t)blockIdx.x * E + e] = c;
  }
  if (!grid_barrier(bar, (uint32_t)nb, wait_limit_ns, status, 3, &ok_sh)) return;

  // 2. column scans over the blocks, one warp per expert column
  const int G = nb * kPermWarps;
  for (int e = blockIdx.x * kPermWarps + wid; e < E; e += G) {
    int32_t carry = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int b = b0 + lane;
      const int32_t v = b < nb ? __ldcg(hist + (int64_t)b * E + e) : 0;
      int32_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (b < nb) hist[(int64_t)b * E + e] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) totals[e] = carry;
  }
  if (!grid_barrier(bar + 1, (uint32_t)nb, wait_limit_ns, status, 4, &ok_sh)) return;

  // 3a. offsets: exclusive scan of the totals over experts (every block)
  for (int e0 = 0; e0 < E; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    const int32_t v = e < E ? __ldcg(totals + e) : 0;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) wtot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int32_t t = lane < kPermWarps ? wtot[lane] : 0;
      int32_t s2 = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, s2, o);
        if (lane >= o) s2 += n;
      }
      if (lane < kPermWarps) wtot[lane] = s2 - t;           // exclusive prefix of the warp sums
      if (lane == kPermWarps - 1) wtot[kPermWarps] = s2;    // this chunk's total
    }
    __syncthreads();
    const int32_t base = e0 == 0 ? 0 : off[e0 - 1] + __ldcg(totals + e0 - 1);
    if (e < E) off[e] = base + wtot[wid] + incl - v;
    __syncthreads();
  }
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const int32_t c = __ldcg(totals + e);
      counts[e] = c;
      offsets[e] = off[e];
      if (e == E - 1) offsets[E] = off[e] + c;
    }
  }
  // 3b. warp bases: offsets[e] + the block's prefix + the counts of lower warps
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = off[e] + __ldcg(hist + (int64_t)blockIdx.x * E + e);
    for (int w2 = 0; w2 < kPermWarps; ++w2) {
      const int32_t c = sh[w2 * E + e];
      sh[w2 * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // 3c. stable ranking inside each warp's slice (as permute_scatter_kernel)
  int32_t* my = sh + wid * E;
  for (int s = 0; s < kPerWarp; s += 32) {
    const int64_t i = slice0 + s + lane;
    const bool valid = i < R;
    int e = valid ? ids[i] : -1;
    if (e < 0 || e >= E) e = E + lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const uint32_t lower = peers & ((1u << lane) - 1u);
    if (e < E) {
      const int32_t row = my[e] + __popc(lower);
      row_map[i] = row;
      src_row[row] = (int32_t)(i / k);
      if (w_perm) w_perm[row] = w[i];
    }
    __syncwarp();
    if (e < E && (peers >> lane) == 1u) my[e] += __popc(peers);
    __syncwarp();
  }
}

// One launch without a grid-wide barrier, for up to kClusterPermuteMaxR
// assignments and E <= kPermThreads: clusters of kPermCluster CTAs.  CTA b
// ranks chunk b (`chunk` assignments); the chunks of cluster c form group c.
// Every cluster counts every group, its CTA r taking groups r, r + 8, ...
// (one histogram each, in its shared memory), so after one cluster barrier
// each CTA reads from its cluster's shared memory the per-expert totals and
// the counts before its chunk: the groups before its cluster's, then the
// chunks of the lower CTAs of its own cluster.  Each CTA thus counts R / 8
// ids plus its chunk, and no CTA waits for one outside its cluster.
constexpr int kPermCluster = 8;
constexpr int kPermMaxSlots = 2;   // groups counted per CTA, so at most 16 clusters
constexpr int64_t kClusterPermuteMaxR = int64_t(1) << 18;

__global__ void __launch_bounds__(kPermThreads) permute_cluster_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int64_t R, int k, int E, int chunk,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ row_map,
    int32_t* __restrict__ src_row, float* __restrict__ w_perm, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  // [kPermMaxSlots][E] group counts | [kPermWarps][E] warp counts, then bases |
  // [E] chunk counts | [E] totals, then offsets | [E] counts before the chunk | [40] scan
  extern __shared__ int32_t sh[];
  int32_t* ghist = sh;
  int32_t* wcnt = ghist + kPermMaxSlots * E;
  int32_t* chist = wcnt + kPermWarps * E;
  int32_t* off = chist + E;
  int32_t* pre = off + E;
  int32_t* wtot = pre + E;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int r = (int)cluster_ctarank();
  const int c = (int)(blockIdx.x / kPermCluster);
  const int nclus = (int)(gridDim.x / kPermCluster);
  const int per_warp = chunk / kPermWarps;
  const int64_t slice0 = (int64_t)blockIdx.x * chunk + (int64_t)wid * per_warp;
  const int64_t group_len = (int64_t)kPermCluster * chunk;

  for (int q = threadIdx.x; q < (kPermMaxSlots + kPermWarps) * E; q += kPermThreads) sh[q] = 0;
  __syncthreads();
  // 1. this chunk, per warp; the ids are checked here
  for (int s = 0; s < per_warp; s += 32) {
    const int64_t i = slice0 + s + lane;
    if (i < R) {
      const int e = ids[i];
      if (e < 0 || e >= E) report_status(status, kStatusDevice, kKernPermute, 1);
      else atomicAdd(&wcnt[wid * E + e], 1);   // counts only: the order of increments is irrelevant
    }
  }
  // 2. this CTA's groups, eight loads in flight per thread
  for (int j = 0; j < kPermMaxSlots; ++j) {
    const int g = r + kPermCluster * j;
    if (g >= nclus) break;
    const int64_t g0 = (int64_t)g * group_len;
    const int64_t g1 = g0 + group_len < R ? g0 + group_len : R;
    int32_t* hj = ghist + j * E;
    int64_t i = g0 + threadIdx.x;
    for (; i + 7 * kPermThreads < g1; i += 8 * kPermThreads) {
      int e[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) e[u] = ids[i + u * kPermThreads];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if ((unsigned)e[u] < (unsigned)E) atomicAdd(&hj[e[u]], 1);
    }
    for (; i < g1; i += kPermThreads) {
      const int e = ids[i];
      if ((unsigned)e < (unsigned)E) atomicAdd(&hj[e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPermThreads) {
    int32_t s = 0;
    for (int w2 = 0; w2 < kPermWarps; ++w2) s += wcnt[w2 * E + e];
    chist[e] = s;
  }
  // 3. every histogram of the cluster is complete: totals, and the counts
  //    before this chunk, summed in a fixed order from the cluster's CTAs
  cluster_sync_all();
  const uint32_t ghist_u32 = smem_u32(ghist), chist_u32 = smem_u32(chist);
  for (int q = threadIdx.x; q < 2 * E; q += kPermThreads) {
    const int e = q < E ? q : q - E;
    const int ng = q < E ? nclus : c;
    int32_t s = 0;
    for (int g = 0; g < ng; ++g)
      s += ld_shared_cluster_s32(
          mapa_shared(ghist_u32 + 4u * (uint32_t)((g / kPermCluster) * E + e), (uint32_t)(g % kPermCluster)));
    if (q < E) {
      off[e] = s;
    } else {
      for (int r2 = 0; r2 < r; ++r2) s += ld_shared_cluster_s32(mapa_shared(chist_u32 + 4u * (uint32_t)e, (uint32_t)r2));
      pre[e] = s;
    }
  }
  // this CTA's reads of the others' memory are done; it waits for theirs
  // before it leaves (the wait at the end)
  cluster_arrive_release();
  __syncthreads();
  // 4. offsets: exclusive scan of the totals (E <= kPermThreads, one per thread)
  {
    const int e = threadIdx.x;
    const int32_t v = e < E ? off[e] : 0;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) wtot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int32_t t = lane < kPermWarps ? wtot[lane] : 0;
      int32_t s2 = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, s2, o);
        if (lane >= o) s2 += n;
      }
      if (lane < kPermWarps) wtot[lane] = s2 - t;
    }
    __syncthreads();
    const int32_t ex = wtot[wid] + incl - v;
    if (e < E) {
      off[e] = ex;
      if (blockIdx.x == 0) {
        counts[e] = v;
        offsets[e] = ex;
        if (e == E - 1) offsets[E] = ex + v;
      }
    }
    __syncthreads();
  }
  // 5. warp bases: offsets[e] + the counts before the chunk + lower warps'
  for (int e = threadIdx.x; e < E; e += kPermThreads) {
    int32_t run = off[e] + pre[e];
    for (int w2 = 0; w2 < kPermWarps; ++w2) {
      const int32_t n = wcnt[w2 * E + e];
      wcnt[w2 * E + e] = run;
      run += n;
    }
  }
  __syncthreads();
  // 6. stable ranking inside each warp's slice (as permute_scatter_kernel)
  int32_t* my = wcnt + wid * E;
  for (int s = 0; s < per_warp; s += 32) {
    const int64_t i = slice0 + s + lane;
    const bool valid = i < R;
    int e = valid ? ids[i] : -1;
    if (e < 0 || e >= E) e = E + lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const uint32_t lower = peers & ((1u << lane) - 1u);
    if (e < E) {
      const int32_t row = my[e] + __popc(lower);
      row_map[i] = row;
      src_row[row] = (int32_t)(i / k);
      if (w_perm) w_perm[row] = w[i];
    }
    __syncwarp();
    if (e < E && (peers >> lane) == 1u) my[e] += __popc(peers);
    __syncwarp();
  }
  cluster_wait_acquire();
}

// src_rows: rows of x (a source row outside [0, src_rows) is reported and
// row 0 read instead), or 0: unchecked.
__global__ void permute_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ src_row,
                                    int64_t R, int H, uint16_t* __restrict__ x_perm, int64_t src_rows,
                                    uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= R) return;
  int64_t s = src_row[row];
  if (src_rows > 0 && (s < 0 || s >= src_rows)) {
    if (lane == 0) report_status(status, kStatusDevice, kKernPermute, 3);
    s = 0;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + s * H);
  uint4* dst = reinterpret_cast<uint4*>(x_perm + row * H);
  const int nch = H / 8;
  for (int c0 = lane; c0 < nch; c0 += 128) {   // four 16-byte loads in flight per lane
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (c0 + 32 * q < nch) v[q] = __ldg(src + c0 + 32 * q);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (c0 + 32 * q < nch) dst[c0 + 32 * q] = v[q];
  }
}

// The same rows moved token by token: x_perm[row_map[t*k + j]] = x[t] for
// j < k.  One warp per (token, slice of kScatterChunks 16-byte chunks) reads its slice
// of x[t] once (kScatterPerLane 16-byte chunks per lane) and writes it to the token's
// k rows.  Where x is larger than L2 this reads it from DRAM once, where the
// gather above reads each token row k times in permuted (scattered) order.
// A destination outside [0, T*k) is reported and not written.
// 16-byte chunks per warp: 64 (512 bf16).  Measured in the layer at the
// Qwen3-MoE shape / the DeepSeek-V3 shape: 32 chunks 26.2 / 313 us, 64
// 26.3 / 313, 128 27.2 / 318, 256 28.2 / 318.
constexpr int kScatterChunks = 64;
constexpr int kScatterPerLane = kScatterChunks / 32;

__global__ void scatter_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ row_map, int64_t T,
                                    int k, int H, uint16_t* __restrict__ x_perm, uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int nch = H / 8;
  const int slices = (nch + kScatterChunks - 1) / kScatterChunks;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t t = gw / slices;
  if (t >= T) return;
  const int c0 = (int)(gw - t * slices) * kScatterChunks;
  const int lane = threadIdx.x & 31;
  const int64_t R = T * k;
  int my_row = -1;
  if (lane < k) {
    my_row = row_map[t * k + lane];
    if (my_row < 0 || (int64_t)my_row >= R) {
      report_status(status, kStatusDevice, kKernPermute, 4);
      my_row = -1;
    }
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
  uint4 v[kScatterPerLane];
#pragma unroll
  for (int q = 0; q < kScatterPerLane; ++q) {
    const int c = c0 + lane + 32 * q;
    v[q] = c < nch ? ld_stream16(src + c) : make_uint4(0, 0, 0, 0);
  }
  for (int j = 0; j < k; ++j) {
    const int row = __shfl_sync(0xffffffffu, my_row, j);
    if (row < 0) continue;   // warp-uniform
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (int64_t)row * H);
#pragma unroll
    for (int q = 0; q < kScatterPerLane; ++q) {
      const int c = c0 + lane + 32 * q;
      if (c < nch) dst[c] = v[q];
    }
  }
}

}  // namespace

// Workspace: hist [nblocks][E]; with the one-launch path also totals [E]
// and the two barrier counters (256-byte aligned after hist).
size_t permute_workspace_bytes(int64_t R, int64_t E, bool noalloc) {
  const int64_t chunk = noalloc ? kChunkNoAlloc : kChunk;
  const int64_t nb = (R + chunk - 1) / chunk;
  const size_t hist = (size_t)((nb > 0 ? nb : 1) * E * sizeof(int32_t));
  if (noalloc) return hist;
  return ((hist + 255) & ~size_t(255)) + (((size_t)E * sizeof(int32_t) + 255) & ~size_t(255)) + 256;
}

// Blocks of permute_fused_kernel that can be resident at once on `dev`.
int64_t permute_fused_capacity(const DeviceInfo& dev, int64_t E) {
  static std::atomic<int> per_sm[kMaxDevices][2] = {};   // cached per device (a race only repeats the query)
  const int slot = E <= 256 ? 0 : 1;   // shared memory grows with E; size the query for the larger E
  if (!per_sm[dev.ordinal][slot].load()) {
    const size_t smem = ((size_t)(kPermWarps + 1) * (slot ? kMaxExperts : 256) + 40) * sizeof(int32_t);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, permute_fused_kernel<kChunk>, kPermThreads, smem) !=
        cudaSuccess)
      return 0;
    per_sm[dev.ordinal][slot].store(n > 0 ? n : -1);
  }
  const int ps = per_sm[dev.ordinal][slot].load();
  return ps > 0 ? (int64_t)ps * dev.num_sms : 0;
}

template <int CHUNK>
cudaError_t enqueue_permute(const int32_t* ids, const float* w, int64_t R, int64_t k, int64_t E,
                            int32_t* counts, int32_t* offsets, int32_t* row_map, int32_t* src_row,
                            float* w_perm, int32_t* hist, uint32_t* status, cudaStream_t stream) {
  const int nb = (int)((R + CHUNK - 1) / CHUNK);
  cudaError_t err = cudaSuccess;
  if (nb > 0)
    err = launch_pdl(permute_hist_kernel<CHUNK>, dim3(nb), dim3(kPermThreads), E * sizeof(int32_t), stream, 1, ids,
                     R, (int)E, hist, status);
  if (err == cudaSuccess)
    err = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), 0, stream, 1, hist, nb, (int)E, counts, offsets);
  if (err == cudaSuccess && nb > 0)
    err = launch_pdl(permute_scatter_kernel<CHUNK>, dim3(nb), dim3(kPermThreads), kPermWarps * E * sizeof(int32_t),
                     stream, 1, ids, w, R, (int)k, (int)E, (const int32_t*)hist, row_map, src_row, w_perm);
  return err;
}

cudaError_t launch_permute(const int32_t* ids, const float* w, int64_t T, int64_t k, int64_t E,
                           int32_t* counts, int32_t* offsets, int32_t* row_map, int32_t* src_row,
                           float* w_perm, void* ws, const DeviceInfo& dev, cudaStream_t stream, bool noalloc) {
  int32_t* hist = static_cast<int32_t*>(ws);
  const int64_t R = T * k;
  const int64_t nb = (R + kChunk - 1) / kChunk;
  if (!noalloc && R > 0 && R <= kClusterPermuteMaxR && E <= kPermThreads) {
    // one cluster launch: chunks of 256 x m assignments, at most 128 of them
    constexpr int64_t kMaxChunks = (int64_t)kPermCluster * kPermCluster * kPermMaxSlots;
    const int64_t chunk = kChunk * ((nb + kMaxChunks - 1) / kMaxChunks);
    const int64_t nbc = (R + chunk - 1) / chunk;
    const int64_t grid = (nbc + kPermCluster - 1) / kPermCluster * kPermCluster;
    const size_t smem = ((size_t)(kPermMaxSlots + kPermWarps + 3) * E + 40) * sizeof(int32_t);
    return launch_pdl(permute_cluster_kernel, dim3((unsigned)grid), dim3(kPermThreads), smem, stream, kPermCluster,
                      ids, w, R, (int)k, (int)E, (int)chunk, counts, offsets, row_map, src_row, w_perm, dev.status);
  }
  if (!noalloc && nb > 0 && nb <= permute_fused_capacity(dev, E)) {
    // one cooperative launch (every block resident), after zeroing its barrier counters
    const size_t hist_bytes = ((size_t)(nb * E * sizeof(int32_t)) + 255) & ~size_t(255);
    int32_t* totals = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + hist_bytes);
    uint32_t* bar = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(totals) +
                                                ((E * sizeof(int32_t) + 255) & ~size_t(255)));
    cudaError_t err = cudaMemsetAsync(bar, 0, 2 * sizeof(uint32_t), stream);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3((unsigned)nb);
    cfg.blockDim = dim3(kPermThreads);
    cfg.dynamicSmemBytes = ((size_t)(kPermWarps + 1) * E + 40) * sizeof(int32_t);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, permute_fused_kernel<kChunk>, ids, w, R, (int)k, (int)E, hist, totals, bar,
                              counts, offsets, row_map, src_row, w_perm, dev.status, dev.wait_limit_ns);
  }
  uint32_t* status = dev.status;
  if (noalloc)
    return enqueue_permute<kChunkNoAlloc>(ids, w, T * k, k, E, counts, offsets, row_map, src_row, w_perm, hist,
                                          status, stream);
  return enqueue_permute<kChunk>(ids, w, T * k, k, E, counts, offsets, row_map, src_row, w_perm, hist, status,
                                 stream);
}

cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* row_map, int64_t T, int64_t k, int64_t H,
                                uint16_t* x_perm, uint32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int64_t slices = (H / 8 + kScatterChunks - 1) / kScatterChunks;
  const int64_t warps = T * slices;
  return launch_pdl(scatter_rows_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, stream, 1, x, row_map, T,
                    (int)k, (int)H, x_perm, status);
}

cudaError_t launch_permute_rows(const uint16_t* x, const int32_t* src_row, int64_t R, int64_t H,
                                uint16_t* x_perm, int64_t src_rows, uint32_t* status, cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  return launch_pdl(permute_rows_kernel, dim3((unsigned)((R + 7) / 8)), dim3(256), 0, stream, 1, x, src_row, R,
                    (int)H, x_perm, src_rows, status);
}

}  // namespace moe

// ------------------------------------------------------------------------
// moe_permute_noalloc: the same permutation without a caller workspace.
//
// Some callers cannot allocate device memory at the moment they route
// tokens: a plugin called from an inference engine's enqueue step, which
// must not allocate; a runtime that has already reserved all device memory
// for its own pool; or a latency-critical path that cannot afford
// cudaMalloc's implicit device synchronisation.  For them the per-block
// histograms live in a fixed array in device memory, declared here; every
// GPU that loads this library keeps it until the process exits.
namespace moe {

constexpr int64_t kNoAllocScratchInts = int64_t(1) << 20;   // 4 MiB
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

static std::mutex g_noalloc_mu;
static int32_t* g_noalloc_scratch[kMaxDevices] = {nullptr};

}  // namespace moe

extern "C" int moe_permute_noalloc(const int32_t* ids, const float* w, int64_t T, int64_t k, int64_t E,
                                   int32_t* counts, int32_t* offsets, int32_t* row_map,
                                   int32_t* src_row, float* w_perm, void* stream) {
  if (T < 0 || k < 1 || E < 1 || T * k > 2147483647) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || (T > 0 && (!ids || !row_map || !src_row))) return MOE_ERR_INVALID_ARG;
  if ((w == nullptr) != (w_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (E > moe::kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (moe::permute_workspace_bytes(T * k, E, true) > sizeof(moe::g_permute_scratch))
    return MOE_ERR_SCRATCH_LIMIT;
  moe::DeviceInfo dev;
  int rc = moe::device_info(&dev);
  if (rc != MOE_OK) return rc;
  int32_t* scratch = nullptr;
  {
    // Set-up, once per device, with that device current: the device
    // address of the array (in host code its name is only a host-side
    // stand-in, which a kernel must never be given).
    std::lock_guard<std::mutex> lock(moe::g_noalloc_mu);
    if (!moe::g_noalloc_scratch[dev.ordinal]) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, moe::g_permute_scratch) != cudaSuccess || !addr) return MOE_ERR_CUDA;
      moe::g_noalloc_scratch[dev.ordinal] = static_cast<int32_t*>(addr);
    }
    scratch = moe::g_noalloc_scratch[dev.ordinal];
  }
  // Every call fully overwrites the histogram entries it reads (the count
  // pass writes all nblocks x E of them first), so nothing has to be cleared.
  return moe::launch_permute(ids, w, T, k, E, counts, offsets, row_map, src_row, w_perm, scratch,
                             dev, static_cast<cudaStream_t>(stream), true) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
