// C ABI of libmoe_gb300.so (declared in include/moe_gb300.h): argument
// validation on the host, then the launches.  Nothing here allocates device
// memory; every buffer is the caller's.
#include <mutex>

#include "../../include/moe_gb300.h"
#include "kernels.h"

namespace moe {

__device__ uint32_t g_status_word;   // first device-side error (see common.cuh)

std::atomic<int> g_pdl{1};           // programmatic dependent launch (moe_set_pdl)

namespace {

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {false};
uint64_t g_wait_limit_ns = 2000000000ull;
int g_test_stall_producer = 0;
int g_gemm_pairs = 2;   // CTA pairs for the forward gate_up GEMM only

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Device information of the current device, set up on first use.
int current_device(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_ready[dev]) {
    DeviceInfo d;
    d.ordinal = dev;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) return MOE_ERR_CUDA;
    d.status = static_cast<uint32_t*>(addr);
    g_dev[dev] = d;
    g_dev_ready[dev] = true;
  }
  *out = g_dev[dev];
  out->wait_limit_ns = g_wait_limit_ns;
  out->test_stall_producer = g_test_stall_producer;
  out->gemm_pairs = g_gemm_pairs;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int gemm_status(int rc) { return rc == 0 ? MOE_OK : (rc < 0 ? MOE_ERR_UNSUPPORTED : MOE_ERR_CUDA); }

constexpr int64_t kMaxI32 = 2147483647;

}  // namespace

int device_info(DeviceInfo* out) { return current_device(out); }

bool encode_tensor_map_2d_bf16(CUtensorMap* map, const void* base, const cuuint64_t* dims,
                               const cuuint64_t* strides, const cuuint32_t* box,
                               const cuuint32_t* estr) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return false;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace moe

using moe::aligned16;
using moe::cuda_status;
using moe::kMaxI32;

extern "C" {

int moe_version(void) { return 10000; }

const char* moe_error_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_DEVICE: return "device-side check failed";
    case MOE_ERR_SCRATCH_LIMIT: return "size exceeds the fixed scratch of moe_permute_noalloc";
    default: return "unknown status";
  }
}

int moe_set_wait_limit_ns(uint64_t ns) {
  moe::g_wait_limit_ns = ns ? ns : 2000000000ull;
  return MOE_OK;
}

int moe_set_gemm_pairs(int mode) {
  if (mode < 0 || mode > 3) return MOE_ERR_INVALID_ARG;
  moe::g_gemm_pairs = mode;
  return MOE_OK;
}

int moe_set_pdl(int on) {
  moe::g_pdl.store(on ? 1 : 0);
  return MOE_OK;
}

int moe_test_stall_gemm_producer(int on) {
  moe::g_test_stall_producer = on ? 1 : 0;
  return MOE_OK;
}

int moe_sync_status(void* stream, uint32_t* detail) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, moe::g_status_word, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(moe::g_status_word, &zero, sizeof(zero)) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (detail) *detail = v;
  if (v == 0) return MOE_OK;
  return (v & 0xFFu) == moe::kStatusTimeout ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE;
}

/* ------------------------------------------------------------------ route */

int moe_route_workspace_size(int64_t T, int64_t H, int64_t E, size_t* bytes) {
  if (!bytes || T < 0 || H < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  *bytes = moe::route_workspace_bytes(T, H, E);
  return MOE_OK;
}

int moe_route(const uint16_t* x, const float* w_router, const float* bias, int64_t T, int64_t H,
              int64_t E, int64_t k, int32_t* ids, float* w, float* logits, void* workspace,
              size_t workspace_bytes, void* stream) {
  if (T < 0 || H < 1 || E < 1 || k < 1 || k > E || T > kMaxI32 || T * k > kMaxI32)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !w_router || !ids || !w)) return MOE_ERR_INVALID_ARG;
  if (E > moe::kMaxExperts || k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if ((x && !aligned16(x)) || (w_router && !aligned16(w_router))) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!workspace || !aligned16(workspace) ||
                workspace_bytes < moe::route_workspace_bytes(T, H, E)))
    return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  moe::DeviceInfo dev;
  int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_route(x, w_router, bias, T, H, E, k, ids, w, logits, workspace, dev,
                                       static_cast<cudaStream_t>(stream)));
}

int moe_route_split_weight(const float* w_router, int64_t H, int64_t E, uint16_t* w_split, void* stream) {
  if (H < 1 || E < 1 || !w_router || !w_split) return MOE_ERR_INVALID_ARG;
  if (E > moe::kMaxExperts || !moe::route_on_tensor_cores(H, E)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(w_router) || !aligned16(w_split)) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_route_split(w_router, H, E, w_split, static_cast<cudaStream_t>(stream)));
}

int moe_route_presplit_workspace_size(int64_t T, int64_t H, int64_t E, size_t* bytes) {
  if (!bytes || T < 0 || H < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (!moe::route_on_tensor_cores(H, E)) return MOE_ERR_UNSUPPORTED;
  *bytes = moe::route_presplit_workspace_bytes(T, H, E);
  return MOE_OK;
}

int moe_route_presplit(const uint16_t* x, const uint16_t* w_split, const float* bias, int64_t T, int64_t H,
                       int64_t E, int64_t k, int32_t* ids, float* w, float* logits, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (T < 0 || H < 1 || E < 1 || k < 1 || k > E || T > kMaxI32 || T * k > kMaxI32)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !w_split || !ids || !w)) return MOE_ERR_INVALID_ARG;
  if (E > moe::kMaxExperts || k > 32 || !moe::route_on_tensor_cores(H, E)) return MOE_ERR_UNSUPPORTED;
  if ((x && !aligned16(x)) || (w_split && !aligned16(w_split))) return MOE_ERR_INVALID_ARG;
  const size_t need = moe::route_presplit_workspace_bytes(T, H, E);
  if (T > 0 && need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need))
    return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  moe::DeviceInfo dev;
  int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_route_presplit(x, w_split, bias, T, H, E, k, ids, w, logits, workspace, dev,
                                                static_cast<cudaStream_t>(stream)));
}

/* ---------------------------------------------------------------- permute */

int moe_permute_workspace_size(int64_t T, int64_t k, int64_t E, size_t* bytes) {
  if (!bytes || T < 0 || k < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  *bytes = moe::permute_workspace_bytes(T * k, E);
  return MOE_OK;
}

int moe_permute(const int32_t* ids, const float* w, int64_t T, int64_t k, int64_t E, int32_t* counts,
                int32_t* offsets, int32_t* row_map, int32_t* src_row, float* w_perm, void* workspace,
                size_t workspace_bytes, void* stream) {
  if (T < 0 || k < 1 || E < 1 || T * k > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || (T > 0 && (!ids || !row_map || !src_row))) return MOE_ERR_INVALID_ARG;
  if ((w == nullptr) != (w_perm == nullptr)) return MOE_ERR_INVALID_ARG;
  if (E > moe::kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < moe::permute_workspace_bytes(T * k, E)) return MOE_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MOE_ERR_INVALID_ARG;
  moe::DeviceInfo dev;
  int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_permute(ids, w, T, k, E, counts, offsets, row_map, src_row, w_perm,
                                         workspace, dev, static_cast<cudaStream_t>(stream)));
}

int moe_permute_rows(const uint16_t* x, const int32_t* src_row, int64_t R, int64_t H,
                     uint16_t* x_perm, void* stream) {
  if (R < 0 || H < 1 || R > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (R > 0 && (!x || !src_row || !x_perm)) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (R > 0 && (!aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  moe::DeviceInfo dev;
  const int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_permute_rows(x, src_row, R, H, x_perm, 0, dev.status,
                                              static_cast<cudaStream_t>(stream)));
}

int moe_permute_rows_scatter(const uint16_t* x, const int32_t* row_map, int64_t T, int64_t k, int64_t H,
                             uint16_t* x_perm, void* stream) {
  if (T < 0 || H < 1 || k < 1 || T > kMaxI32 || T * k > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !row_map || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
  moe::DeviceInfo dev;
  const int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_scatter_rows(x, row_map, T, k, H, x_perm, dev.status,
                                              static_cast<cudaStream_t>(stream)));
}

/* ----------------------------------------------------------- grouped GEMMs */

static int gemm_shape_check(int64_t R, int64_t H, int64_t E, int64_t I) {
  if (R < 0 || H < 1 || E < 1 || I < 1 || R > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (H % 64 != 0 || I % 64 != 0 || E > moe::kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (E * H > kMaxI32 || E * I > kMaxI32) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int moe_grouped_gemm_gate_up_swiglu(const uint16_t* x, const int32_t* src_row,
                                    const int32_t* offsets, const uint16_t* gate_up, int64_t T,
                                    int64_t R, int64_t H, int64_t E, int64_t I, uint16_t* h,
                                    const float* w_perm, float* gu_pre, uint16_t* h_w, void* stream) {
  int rc = gemm_shape_check(R, H, E, I);
  if (rc != MOE_OK) return rc;
  if (T < 0 || T > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (!offsets && E != 1) return MOE_ERR_INVALID_ARG;
  if (!src_row && T < R) return MOE_ERR_INVALID_ARG;
  if (h_w && !w_perm) return MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  if (!x || !gate_up || !h || T < 1) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(gate_up) || !aligned16(h) || (gu_pre && !aligned16(gu_pre)) ||
      (h_w && !aligned16(h_w)))
    return MOE_ERR_INVALID_ARG;
  moe::DeviceInfo dev;
  if ((rc = moe::current_device(&dev)) != MOE_OK) return rc;
  return moe::gemm_status(moe::launch_gemm_gate_up(x, src_row, offsets, gate_up, T, R, H, E, I, h,
                                                   w_perm, gu_pre, h_w, dev,
                                                   static_cast<cudaStream_t>(stream)));
}

int moe_grouped_gemm_down(const uint16_t* h, const int32_t* offsets, const uint16_t* down, int64_t R,
                          int64_t H, int64_t E, int64_t I, uint16_t* y_perm, void* stream) {
  int rc = gemm_shape_check(R, H, E, I);
  if (rc != MOE_OK) return rc;
  if (!offsets && E != 1) return MOE_ERR_INVALID_ARG;
  if (R == 0) return MOE_OK;
  if (!h || !down || !y_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(down) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  moe::DeviceInfo dev;
  if ((rc = moe::current_device(&dev)) != MOE_OK) return rc;
  return moe::gemm_status(moe::launch_gemm_down(h, offsets, down, R, H, E, I, y_perm, dev,
                                                static_cast<cudaStream_t>(stream)));
}

/* ---------------------------------------------------------------- combine */

int moe_unpermute_combine(const uint16_t* y_perm, const int32_t* row_map, const float* w,
                          const uint16_t* y_shared, int64_t T, int64_t H, int64_t k, uint16_t* y,
                          void* stream) {
  if (T < 0 || H < 1 || k < 1 || T > kMaxI32 || T * k > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_perm || !row_map || !w || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y) || (y_shared && !aligned16(y_shared))) return MOE_ERR_INVALID_ARG;
  moe::DeviceInfo dev;
  const int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_combine(y_perm, row_map, w, y_shared, T, H, k, y, dev.status,
                                         static_cast<cudaStream_t>(stream)));
}

/* --------------------------------------------------------------- backward */

int moe_unpermute_combine_bwd(const uint16_t* dy, const int32_t* src_row, int64_t T, int64_t H,
                              int64_t k, uint16_t* dy_perm, void* stream) {
  if (T < 0 || H < 1 || k < 1 || T > kMaxI32 || T * k > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!dy || !src_row || !dy_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dy) || !aligned16(dy_perm)) return MOE_ERR_INVALID_ARG;
  moe::DeviceInfo dev;
  const int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_permute_rows(dy, src_row, T * k, H, dy_perm, T, dev.status,
                                              static_cast<cudaStream_t>(stream)));
}

int moe_route_bwd(const float* dw_part, int64_t nparts, const int32_t* row_map, const float* w,
                  const int32_t* ids, int64_t T, int64_t E, int64_t k, float* d_logits, float* dw,
                  void* stream) {
  if (T < 0 || E < 1 || k < 1 || k > E || nparts < 1 || T > kMaxI32 || T * k > kMaxI32)
    return MOE_ERR_INVALID_ARG;
  if (k > 32 || nparts > 64) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!dw_part || !row_map || !w || !ids || !d_logits) return MOE_ERR_INVALID_ARG;
  moe::DeviceInfo dev;
  const int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_route_bwd(dw_part, (int)nparts, row_map, w, ids, T, E, k, d_logits, dw,
                                           dev.status, static_cast<cudaStream_t>(stream)));
}

int moe_grouped_gemm_down_bwd_parts(int64_t I, int64_t* nparts) {
  if (!nparts || I < 1) return MOE_ERR_INVALID_ARG;
  *nparts = moe::down_bwd_parts(I);
  return MOE_OK;
}

int moe_grouped_gemm_down_bwd(const uint16_t* dy_perm, const uint16_t* h_w, const float* gu_pre,
                              const float* w_perm, const int32_t* offsets, const uint16_t* down,
                              int64_t R, int64_t H, int64_t E, int64_t I, uint16_t* dgu,
                              uint16_t* d_down, float* dw_part, void* stream) {
  int rc = gemm_shape_check(R, H, E, I);
  if (rc != MOE_OK) return rc;
  if (!offsets && E != 1) return MOE_ERR_INVALID_ARG;
  if (!down || !d_down || (R > 0 && (!dy_perm || !h_w || !gu_pre || !w_perm || !dgu || !dw_part)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(down) || !aligned16(d_down) ||
      (R > 0 && (!aligned16(dy_perm) || !aligned16(h_w) || !aligned16(gu_pre) || !aligned16(dgu))))
    return MOE_ERR_INVALID_ARG;
  if (R == 0) return cuda_status(cudaMemsetAsync(d_down, 0, (size_t)(E * I * H * 2), static_cast<cudaStream_t>(stream)));
  moe::DeviceInfo dev;
  if ((rc = moe::current_device(&dev)) != MOE_OK) return rc;
  return moe::gemm_status(moe::launch_gemm_down_bwd(dy_perm, h_w, gu_pre, w_perm, offsets, down, R, H,
                                                    E, I, dgu, d_down, dw_part, dev,
                                                    static_cast<cudaStream_t>(stream)));
}

int moe_grouped_gemm_gate_up_bwd(const uint16_t* dgu, const uint16_t* x, const int32_t* src_row,
                                 const int32_t* offsets, const uint16_t* gate_up, int64_t T,
                                 int64_t R, int64_t H, int64_t E, int64_t I, uint16_t* dx_perm,
                                 uint16_t* d_gate_up, void* stream) {
  int rc = gemm_shape_check(R, H, E, I);
  if (rc != MOE_OK) return rc;
  if (T < 0 || T > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (!offsets && E != 1) return MOE_ERR_INVALID_ARG;
  if (!src_row && T < R) return MOE_ERR_INVALID_ARG;
  if (!gate_up || !d_gate_up || (R > 0 && (!dgu || !x || !dx_perm))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(gate_up) || !aligned16(d_gate_up) ||
      (R > 0 && (!aligned16(dgu) || !aligned16(x) || !aligned16(dx_perm))))
    return MOE_ERR_INVALID_ARG;
  if (R == 0)
    return cuda_status(cudaMemsetAsync(d_gate_up, 0, (size_t)(E * H * 2 * I * 2), static_cast<cudaStream_t>(stream)));
  moe::DeviceInfo dev;
  if ((rc = moe::current_device(&dev)) != MOE_OK) return rc;
  return moe::gemm_status(moe::launch_gemm_gate_up_bwd(dgu, x, src_row, offsets, gate_up, T, R, H, E,
                                                       I, dx_perm, d_gate_up, dev,
                                                       static_cast<cudaStream_t>(stream)));
}

int moe_gather_dx_workspace_size(int64_t H, int64_t E, size_t* bytes) {
  if (!bytes || H < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  *bytes = moe::gather_dx_workspace_bytes(H, E);
  return MOE_OK;
}

int moe_gather_dx(const uint16_t* dx_perm, const int32_t* row_map, const float* d_logits,
                  const int32_t* ids, const float* w_router, int64_t T, int64_t H, int64_t E,
                  int64_t k, uint16_t* dx, void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || H < 1 || E < 1 || k < 1 || k > E || T > kMaxI32 || T * k > kMaxI32)
    return MOE_ERR_INVALID_ARG;
  if (k > 32 || H % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;   // no rows: the optional router term's pointers may be NULL too
  if ((d_logits == nullptr) != (w_router == nullptr)) return MOE_ERR_INVALID_ARG;
  if (!dx_perm || !row_map || !dx || (d_logits && !ids)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(dx_perm) || !aligned16(dx)) return MOE_ERR_INVALID_ARG;
  if (d_logits && (!workspace || !aligned16(workspace) ||
                   workspace_bytes < moe::gather_dx_workspace_bytes(H, E)))
    return MOE_ERR_WORKSPACE;
  moe::DeviceInfo dev;
  const int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_gather_dx(dx_perm, row_map, d_logits, ids, w_router, T, H, E, k, dx,
                                           workspace, dev.status, static_cast<cudaStream_t>(stream)));
}

int moe_route_bwd_weight(const uint16_t* x, const float* d_logits, int64_t T, int64_t H, int64_t E,
                         float* d_w_router, void* stream) {
  if (T < 0 || H < 1 || E < 1 || T > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (!d_w_router || (T > 0 && (!x || !d_logits))) return MOE_ERR_INVALID_ARG;
  return cuda_status(moe::launch_route_bwd_weight(x, d_logits, T, H, E, d_w_router,
                                                  static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

/* ---------------------------------------------------- expert parallelism */

int moe_sort_chunks_workspace_size(int64_t A, int64_t B, size_t* bytes) {
  if (!bytes || A < 1 || B < 1 || A * B > (int64_t)1 << 24) return MOE_ERR_INVALID_ARG;
  *bytes = moe::sort_chunks_workspace_bytes(A, B);
  return MOE_OK;
}

int moe_sort_chunks(const int32_t* counts, int64_t A, int64_t B, int64_t N, int32_t* src_of, int32_t* pos_of,
                    int32_t* group_offsets, void* workspace, size_t workspace_bytes, void* stream) {
  if (A < 1 || B < 1 || A * B > (int64_t)1 << 24 || N < 0 || N > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (!counts || !group_offsets || (N > 0 && (!src_of || !pos_of))) return MOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < moe::sort_chunks_workspace_bytes(A, B))
    return MOE_ERR_WORKSPACE;
  moe::DeviceInfo dev;
  int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_sort_chunks(counts, A, B, N, src_of, pos_of, group_offsets, workspace, dev.status,
                                             static_cast<cudaStream_t>(stream)));
}

int moe_ep_map_replicas(const int32_t* ids, int64_t T, int64_t k, int64_t E, const int32_t* rep_first,
                        const int32_t* rep_count, const int32_t* rep_list, int64_t n_phys, int32_t* phys_ids,
                        void* stream) {
  if (T < 0 || k < 1 || E < 1 || n_phys < E || T * k > kMaxI32 || n_phys > kMaxI32) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !phys_ids)) return MOE_ERR_INVALID_ARG;
  if (!rep_first || !rep_count || !rep_list) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  moe::DeviceInfo dev;
  int rc = moe::current_device(&dev);
  if (rc != MOE_OK) return rc;
  return cuda_status(moe::launch_map_replicas(ids, T * k, k, E, rep_first, rep_count, rep_list, n_phys, phys_ids,
                                              dev.status, static_cast<cudaStream_t>(stream)));
}

int moe_eplb_plan(const int64_t* expert_load, int64_t E, int64_t G, int64_t n_phys, int32_t* phys_to_log,
                  int32_t* rep_first, int32_t* rep_count, int32_t* rep_list, int64_t* rank_load) {
  if (!expert_load || !phys_to_log || !rep_first || !rep_count || !rep_list) return MOE_ERR_INVALID_ARG;
  if (E < 1 || G < 1 || n_phys < E || n_phys % G != 0 || n_phys > (int64_t)1 << 20) return MOE_ERR_INVALID_ARG;
  for (int64_t e = 0; e < E; ++e)
    if (expert_load[e] < 0) return MOE_ERR_INVALID_ARG;
  moe::eplb_plan(expert_load, E, G, n_phys, phys_to_log, rep_first, rep_count, rep_list, rank_load);
  return MOE_OK;
}
