// Internal launchers of libmoe_gb300 (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "common.cuh"

namespace moe {

// Programmatic dependent launch on (1) or off (0), moe_set_pdl.
extern std::atomic<int> g_pdl;

// Launches `kernel` with programmatic stream serialization while g_pdl is on
// (see pdl_wait in common.cuh) and, when cluster_x > 1, in clusters of
// cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (g_pdl.load(std::memory_order_relaxed)) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kMaxDevices = 64;
constexpr int kMaxExperts = 1024;

struct DeviceInfo {
  int ordinal;
  int num_sms;
  uint32_t* status;        // device address of the status word
  uint64_t wait_limit_ns;  // bound of every device-side spin wait
  int test_stall_producer; // test hook of the bounded-wait path (grouped GEMMs)
  int gemm_pairs;          // CTA pairs: 0 none, 1 every forward / dgrad grouped GEMM, 2 forward gate_up only,
                           // 3 forward gate_up and the weight-gradient GEMMs
};

// Device information of the current device (status word address, SM count).
int device_info(DeviceInfo* out);

// Encodes a 2-D bf16 tensor map with 128-byte swizzle (driver entry point
// looked up at run time); false when the driver rejects it.
bool encode_tensor_map_2d_bf16(CUtensorMap* map, const void* base, const cuuint64_t* dims,
                               const cuuint64_t* strides, const cuuint32_t* box,
                               const cuuint32_t* estr);

size_t route_workspace_bytes(int64_t T, int64_t H, int64_t E);
bool route_on_tensor_cores(int64_t H, int64_t E);
size_t route_presplit_workspace_bytes(int64_t T, int64_t H, int64_t E);
cudaError_t launch_route_split(const float* w_router, int64_t H, int64_t E, uint16_t* w_split,
                               cudaStream_t stream);
cudaError_t launch_route_presplit(const uint16_t* x, const uint16_t* w_split, const float* bias, int64_t T,
                                  int64_t H, int64_t E, int64_t k, int32_t* ids, float* w, float* logits,
                                  void* ws, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_route(const uint16_t* x, const float* w_router, const float* bias, int64_t T,
                         int64_t H, int64_t E, int64_t k, int32_t* ids, float* w, float* logits,
                         void* ws, const DeviceInfo& dev, cudaStream_t stream);

size_t permute_workspace_bytes(int64_t R, int64_t E, bool noalloc = false);
cudaError_t launch_permute(const int32_t* ids, const float* w, int64_t T, int64_t k, int64_t E,
                           int32_t* counts, int32_t* offsets, int32_t* row_map, int32_t* src_row,
                           float* w_perm, void* ws, const DeviceInfo& dev, cudaStream_t stream,
                           bool noalloc = false);
// src_rows: rows of x, checked on the device (0: unchecked)
cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* row_map, int64_t T, int64_t k, int64_t H,
                                uint16_t* x_perm, uint32_t* status, cudaStream_t stream);
cudaError_t launch_permute_rows(const uint16_t* x, const int32_t* src_row, int64_t R, int64_t H,
                                uint16_t* x_perm, int64_t src_rows, uint32_t* status, cudaStream_t stream);

cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* row_map, const float* w,
                           const uint16_t* y_shared, int64_t T, int64_t H, int64_t k, uint16_t* y,
                           uint32_t* status, cudaStream_t stream);
cudaError_t launch_route_bwd(const float* dw_part, int nparts, const int32_t* row_map, const float* w,
                             const int32_t* ids, int64_t T, int64_t E, int64_t k, float* d_logits,
                             float* dw, uint32_t* status, cudaStream_t stream);
size_t gather_dx_workspace_bytes(int64_t H, int64_t E);
cudaError_t launch_gather_dx(const uint16_t* dx_perm, const int32_t* row_map, const float* d_logits,
                             const int32_t* ids, const float* w_router, int64_t T, int64_t H,
                             int64_t E, int64_t k, uint16_t* dx, void* ws, uint32_t* status,
                             cudaStream_t stream);
cudaError_t launch_route_bwd_weight(const uint16_t* x, const float* d_logits, int64_t T, int64_t H,
                                    int64_t E, float* d_w_router, cudaStream_t stream);

// Expert-parallel dispatch pieces (ep.cu).
size_t sort_chunks_workspace_bytes(int64_t A, int64_t B);
cudaError_t launch_sort_chunks(const int32_t* counts, int64_t A, int64_t B, int64_t N, int32_t* src_of,
                               int32_t* pos_of, int32_t* group_off, void* ws, uint32_t* status,
                               cudaStream_t stream);
cudaError_t launch_map_replicas(const int32_t* ids, int64_t R, int64_t k, int64_t E, const int32_t* rep_first,
                                const int32_t* rep_count, const int32_t* rep_list, int64_t n_phys,
                                int32_t* phys_ids, uint32_t* status, cudaStream_t stream);
void eplb_plan(const int64_t* load, int64_t E, int64_t G, int64_t n_phys, int32_t* phys_to_log,
               int32_t* rep_first, int32_t* rep_count, int32_t* rep_list, int64_t* rank_load);

// Grouped GEMMs: 0 = enqueued, -1 = tensor map rejected, 1 = launch failed.
int router_parts(int64_t T, int64_t H, int64_t E);
int launch_router_logits(const uint16_t* x, const uint16_t* w_split, int64_t T, int64_t H, int64_t E,
                         int parts, float* part_out, const DeviceInfo& dev, cudaStream_t stream);
int launch_gemm_gate_up(const uint16_t* x, const int32_t* src_row, const int32_t* offsets,
                        const uint16_t* gate_up, int64_t T, int64_t R, int64_t H, int64_t E,
                        int64_t I, uint16_t* h, const float* w_perm, float* gu_pre, uint16_t* h_w,
                        const DeviceInfo& dev, cudaStream_t stream);
int launch_gemm_down(const uint16_t* h, const int32_t* offsets, const uint16_t* down, int64_t R,
                     int64_t H, int64_t E, int64_t I, uint16_t* y_perm, const DeviceInfo& dev,
                     cudaStream_t stream);
int down_bwd_parts(int64_t I);   // n tiles of the dgrad: partial dot products per row
int launch_gemm_down_bwd(const uint16_t* dy_perm, const uint16_t* h_w, const float* gu_pre,
                         const float* w_perm, const int32_t* offsets, const uint16_t* down, int64_t R,
                         int64_t H, int64_t E, int64_t I, uint16_t* dgu, uint16_t* d_down,
                         float* dw_part, const DeviceInfo& dev, cudaStream_t stream);
int launch_gemm_gate_up_bwd(const uint16_t* dgu, const uint16_t* x, const int32_t* src_row,
                            const int32_t* offsets, const uint16_t* gate_up, int64_t T, int64_t R,
                            int64_t H, int64_t E, int64_t I, uint16_t* dx_perm,
                            uint16_t* d_gate_up, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace moe
