// ffn_noalloc.cu -- moe_expert_ffn_noalloc: the expert FFN for callers that
// cannot allocate device memory.
//
// moe_expert_ffn needs a caller workspace for two scratch buffers: the batch
// rows gathered into expert order and the SwiGLU intermediate.  Some callers
// have no way to provide one: code embedded in a host application that owns
// every byte of device memory through its own allocator and gives plugins no
// call to obtain more, or latency-critical code that must never call
// cudaMalloc (which may synchronize the whole device).  This variant keeps
// that scratch in a fixed array compiled into the library instead, so the
// caller passes only inputs and outputs and nothing is allocated per call.
//
// Limits and sharing:
//   * the array holds kNoAllocScratchBytes (64 MiB); a layer whose scratch
//     (256 B of flags + gathered rows + intermediate, each with
//     round32(T*(k+S)) + 256 rows) does not fit is rejected with
//     MOE_ERR_UNSUPPORTED before anything is launched;
//   * every GPU on which the library's device code is loaded holds the array
//     until the process exits;
//   * all calls share the one array per device and it keeps the last call's
//     contents, so calls that overlap on the GPU (different streams, or
//     different host threads on the same device) race with each other; they
//     must be ordered by the caller;
//   * the first call on each device looks up the array's device address with
//     that device current (cudaGetSymbolAddress) and keeps it for the life of
//     the process; that first call should come before any stream capture;
//   * after a device reset (cudaDeviceReset) the library's device code may be
//     reloaded at another address, so the kept address is stale: do not call
//     this entry point on a device after resetting it;
//   * the kernels' error word lives in the array and is cleared at every
//     call; device-detected problems are not reported by this entry point.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;
constexpr int kMaxDevices = 64;

}  // namespace

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, not a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).
cudaError_t scratch_on_current_device(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_expert_ffn_noalloc(const moe_layer_desc* desc, const void* x,
                                             const int32_t* expert_offsets,
                                             const int32_t* token_indices, const float* slot_w,
                                             const void* Wg, const void* Wu, const void* Wd,
                                             void* y_perm, void* stream) {
  size_t ws_bytes = 0;
  const moe_status st = moe_workspace_size(desc, &ws_bytes);  // validates the layer record
  if (st != MOE_OK) return st;
  if (desc->T == 0) return MOE_OK;
  if (!x || !expert_offsets || !token_indices || !Wg || !Wu || !Wd || !y_perm)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) || !aligned16(y_perm))
    return MOE_ERR_INVALID_ARG;

  const int P = desc->T * (desc->k + desc->S);
  const int nE = desc->E + desc->S;
  const size_t es = moe::dtype_size(desc->dtype);
  const size_t cap = (size_t)moe::tc_row_capacity(P);
  const size_t rows_bytes = round256(cap * (size_t)desc->d * es);
  const size_t h_bytes = round256(cap * (size_t)desc->I * es);
  if (256 + rows_bytes + h_bytes > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;

  unsigned char* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  int* flags = reinterpret_cast<int*>(scratch);
  void* x_perm = scratch + 256;
  void* h = scratch + 256 + rows_bytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (cudaMemsetAsync(flags, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_gather_rows(desc->dtype, x, token_indices, expert_offsets + nE, P, desc->T,
                              desc->d, x_perm, flags, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaError_t e;
  if (desc->dtype == MOE_F32) {
    e = moe::launch_ffn_simt(static_cast<const float*>(x_perm), expert_offsets, nE, P, desc->d,
                             desc->I, static_cast<const float*>(Wg), static_cast<const float*>(Wu),
                             static_cast<const float*>(Wd), slot_w, static_cast<float*>(h),
                             static_cast<float*>(y_perm), s);
  } else {
    e = moe::launch_ffn_tc(x_perm, expert_offsets, nE, P, desc->d, desc->I, (double)P / nE, Wg,
                           Wu, Wd, slot_w, h, y_perm, flags, s);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
