// Expert-parallel dispatch and combine, the pieces that run on one device
// ("Awesome-ML-SYS-Tutorial" MoE/EP guide, gsyq.cn, "Expert Parallelism":
// dispatch by all-to-all, expert compute, combine by all-to-all; the split
// sizes from per-expert token counts (`preprocess`), the receiver's re-sort
// of its chunks by local expert (`sort_chunks_by_idxs`); hotspot experts and
// EPLB-style replication).
//
// Experts are split over G ranks on dim 0: rank d owns the experts
// [d E/G, (d+1) E/G).  A rank's permuted rows (moe_permute) are then already
// grouped by destination rank, in chunks of its per-expert counts.  The
// all-to-all turns the (source, destination) chunk order into (destination,
// source) order, and the receiver turns its (source, local expert) chunks
// into (local expert, source) order so that each local expert's rows are
// contiguous for the grouped GEMMs.  Both are the same row permutation, a
// transpose of a matrix of chunks, computed here by moe_sort_chunks.  The
// collective itself (NCCL all-to-all-v, or any other transport) is not part
// of this library.
//
// EPLB-style replication: a plan (moe_eplb_plan, on the host) gives hot
// experts extra physical replicas and places the physical experts on the
// ranks; moe_ep_map_replicas sends each (token, slot) of a replicated expert
// to replica (token mod replicas), so the replicas share its rows.
#include <algorithm>
#include <vector>

#include "../../include/moe_gb300.h"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kScanThreads = 1024;

// Exclusive scans of the A x B chunk counts in (a, b) order (in_off[a B + b],
// in_off[A B] = total) and in (b, a) order (out_off[b A + a]); group_off[b]
// = first row of group b in (b, a) order, group_off[B] = total.  One block.
__global__ void __launch_bounds__(kScanThreads) chunk_scan_kernel(const int32_t* __restrict__ counts, int A, int B,
                                                                  int64_t N, int32_t* __restrict__ in_off,
                                                                  int32_t* __restrict__ out_off,
                                                                  int32_t* __restrict__ group_off,
                                                                  uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ long long warp_tot[kScanThreads / 32];
  __shared__ long long carry_sh;
  const int n = A * B;
  const int per = (n + kScanThreads - 1) / kScanThreads;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int order = 0; order < 2; ++order) {
    // element q of this order: (a, b) order q = a B + b; (b, a) order q = b A + a
    auto value = [&](int q) -> int {
      const int a = order == 0 ? q / B : q % A;
      const int b = order == 0 ? q % B : q / A;
      const int c = counts[a * B + b];
      if (c < 0) report_status(status, kStatusDevice, kKernPermute, 7);
      return c < 0 ? 0 : c;
    };
    const int q0 = threadIdx.x * per;
    long long sum = 0;
    for (int q = q0; q < min(q0 + per, n); ++q) sum += value(q);
    long long incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      long long t = lane < kScanThreads / 32 ? warp_tot[lane] : 0;
      long long ti = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, ti, o);
        if (lane >= o) ti += v;
      }
      if (lane < kScanThreads / 32) warp_tot[lane] = ti - t;   // exclusive over warps
      if (lane == 31) carry_sh = ti;                         // the total
    }
    __syncthreads();
    long long run = warp_tot[wid] + incl - sum;
    for (int q = q0; q < min(q0 + per, n); ++q) {
      const int c = value(q);
      const int v = (int)min(run, (long long)0x7fffffff);
      if (order == 0) {
        in_off[q] = v;
      } else {
        out_off[q] = v;
        if (q % A == 0) group_off[q / A] = v;
      }
      run += c;
    }
    if (threadIdx.x == 0) {
      const long long total = carry_sh;
      if (order == 0) in_off[n] = (int)min(total, (long long)0x7fffffff);
      else group_off[B] = (int)min(total, (long long)0x7fffffff);
      if (total != N) report_status(status, kStatusDevice, kKernPermute, 8);
    }
    __syncthreads();
  }
}

// For every input row i (in (a, b) chunk order): its output position o in
// (b, a) order; pos_of[i] = o, src_of[o] = i.  Rows past the counts' total
// (a count total that is not N, reported by the scan) are not written.
__global__ void chunk_rows_kernel(const int32_t* __restrict__ in_off, const int32_t* __restrict__ out_off, int A,
                                  int B, int64_t N, int32_t* __restrict__ src_of, int32_t* __restrict__ pos_of) {
  pdl_wait();
  pdl_trigger();
  const int n = A * B;
  const int64_t total = in_off[n];
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += (int64_t)gridDim.x * blockDim.x) {
    if (i >= total) continue;
    int lo = 0, hi = n - 1;   // the last chunk q with in_off[q] <= i (a non-empty one)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (in_off[mid] <= i) lo = mid; else hi = mid - 1;
    }
    const int a = lo / B, b = lo % B;
    const int64_t o = (int64_t)out_off[b * A + a] + (i - in_off[lo]);
    if (o < 0 || o >= N) continue;
    pos_of[i] = (int32_t)o;
    src_of[o] = (int32_t)i;
  }
}

// phys_ids[i] = the replica of logical expert ids[i] that token i / k goes to:
// rep_list[rep_first[e] + (i / k) % rep_count[e]].
__global__ void map_replicas_kernel(const int32_t* __restrict__ ids, int64_t R, int k, int E,
                                    const int32_t* __restrict__ rep_first, const int32_t* __restrict__ rep_count,
                                    const int32_t* __restrict__ rep_list, int n_phys, int32_t* __restrict__ phys_ids,
                                    uint32_t* status) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < R; i += (int64_t)gridDim.x * blockDim.x) {
    const int e = ids[i];
    int p = 0;
    if (e < 0 || e >= E) {
      report_status(status, kStatusDevice, kKernPermute, 9);
    } else {
      const int c = rep_count[e];
      const int f = rep_first[e];
      const int64_t slot = (int64_t)f + (c > 0 ? (i / k) % c : 0);
      if (c < 1 || slot >= n_phys || f < 0) {
        report_status(status, kStatusDevice, kKernPermute, 9);
      } else {
        p = rep_list[slot];
        if (p < 0 || p >= n_phys) {
          report_status(status, kStatusDevice, kKernPermute, 9);
          p = 0;
        }
      }
    }
    phys_ids[i] = p;
  }
}

}  // namespace

size_t sort_chunks_workspace_bytes(int64_t A, int64_t B) { return (size_t)(2 * A * B + 1) * 4; }

cudaError_t launch_sort_chunks(const int32_t* counts, int64_t A, int64_t B, int64_t N, int32_t* src_of,
                               int32_t* pos_of, int32_t* group_off, void* ws, uint32_t* status,
                               cudaStream_t stream) {
  int32_t* in_off = static_cast<int32_t*>(ws);
  int32_t* out_off = in_off + A * B + 1;
  cudaError_t err = launch_pdl(chunk_scan_kernel, dim3(1), dim3(kScanThreads), 0, stream, 1, counts, (int)A,
                               (int)B, N, in_off, out_off, group_off, status);
  if (err != cudaSuccess || N == 0) return err;
  const int64_t blocks = std::min<int64_t>((N + 255) / 256, 4096);
  return launch_pdl(chunk_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 1, (const int32_t*)in_off,
                    (const int32_t*)out_off, (int)A, (int)B, N, src_of, pos_of);
}

cudaError_t launch_map_replicas(const int32_t* ids, int64_t R, int64_t k, int64_t E, const int32_t* rep_first,
                                const int32_t* rep_count, const int32_t* rep_list, int64_t n_phys,
                                int32_t* phys_ids, uint32_t* status, cudaStream_t stream) {
  if (R == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((R + 255) / 256, 4096);
  return launch_pdl(map_replicas_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 1, ids, R, (int)k, (int)E,
                    rep_first, rep_count, rep_list, (int)n_phys, phys_ids, status);
}

// EPLB-style plan on the host.  1. Replication: every expert starts with one
// replica; each of the n_phys - E extra replicas goes to the expert with the
// largest load per replica (ties to the lower index).  2. A replica's load
// is its share of the expert's rows under the round-robin by token (load /
// replicas, the first load % replicas replicas one more).  3. Placement: the
// replicas, heaviest first (ties: lower expert, then lower replica), each go
// to the rank with the least load so far among those with a free slot
// (n_phys / G slots each; ties to the lower rank).  4. Physical ids are rank
// major; within a rank, by (expert, replica).
void eplb_plan(const int64_t* load, int64_t E, int64_t G, int64_t n_phys, int32_t* phys_to_log,
               int32_t* rep_first, int32_t* rep_count, int32_t* rep_list, int64_t* rank_load) {
  std::vector<int64_t> rep(E, 1);
  for (int64_t extra = 0; extra < n_phys - E; ++extra) {
    int64_t best = 0;
    for (int64_t e = 1; e < E; ++e)   // load[e] / rep[e] > load[best] / rep[best], exactly
      if ((__int128)load[e] * rep[best] > (__int128)load[best] * rep[e]) best = e;
    ++rep[best];
  }
  struct Rep { int64_t load, e, r; };
  std::vector<Rep> reps;
  for (int64_t e = 0; e < E; ++e)
    for (int64_t r = 0; r < rep[e]; ++r) reps.push_back({load[e] / rep[e] + (r < load[e] % rep[e] ? 1 : 0), e, r});
  std::stable_sort(reps.begin(), reps.end(), [](const Rep& x, const Rep& y) {
    if (x.load != y.load) return x.load > y.load;
    if (x.e != y.e) return x.e < y.e;
    return x.r < y.r;
  });
  const int64_t slots = n_phys / G;
  std::vector<int64_t> rl(G, 0), used(G, 0);
  std::vector<std::vector<std::pair<int64_t, int64_t>>> on(G);   // (expert, replica) per rank
  for (const Rep& x : reps) {
    int64_t g = -1;
    for (int64_t c = 0; c < G; ++c)
      if (used[c] < slots && (g < 0 || rl[c] < rl[g])) g = c;
    rl[g] += x.load;
    ++used[g];
    on[g].push_back({x.e, x.r});
  }
  int64_t first = 0;
  for (int64_t e = 0; e < E; ++e) {
    rep_first[e] = (int32_t)first;
    rep_count[e] = (int32_t)rep[e];
    first += rep[e];
  }
  for (int64_t g = 0; g < G; ++g) {
    std::sort(on[g].begin(), on[g].end());
    for (int64_t i = 0; i < slots; ++i) {
      const int64_t p = g * slots + i;
      const int64_t e = on[g][i].first, r = on[g][i].second;
      phys_to_log[p] = (int32_t)e;
      rep_list[rep_first[e] + r] = (int32_t)p;
    }
    if (rank_load) rank_load[g] = rl[g];
  }
}

}  // namespace moe
