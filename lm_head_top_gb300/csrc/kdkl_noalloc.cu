// Allocation-free forward: kd_kl_forward with its scratch taken from a fixed
// array compiled into this library instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory for a workspace.
// A host framework that manages the whole GPU through its own memory pool
// typically reserves all free HBM up front, so a side cudaMalloc fails or
// fragments the pool, and such frameworks often forbid libraries from
// allocating behind their back. A training loop with a hard latency budget
// also avoids cudaMalloc, which can synchronise the device. These callers
// still pass their inputs and outputs, but have nothing to pass as scratch.
//
// The scratch is a file-scope __device__ array of KDKL_NOALLOC_SCRATCH_BYTES.
// Every GPU on which this library's device code is loaded holds that memory
// until the process exits. In host code the array's name is only a host-side
// stand-in, so its device address is looked up with cudaGetSymbolAddress, once
// per device, with that device current, on the first call made on it.
#include <cuda_runtime.h>

#include <mutex>

#include "kdkl.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KDKL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
kd_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return KD_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KD_OK;
}

}  // namespace

extern "C" kd_status kd_kl_forward_noalloc(const kd_kl_problem* prob, const uint16_t* H,
                                           const uint16_t* W, const int32_t* topk_idx,
                                           const float* topk_logit, const uint8_t* mask,
                                           float* loss, float* lse, float* token_kl,
                                           void* stream) {
  void* scratch = nullptr;
  const kd_status st = scratch_on_current_device(&scratch);
  if (st != KD_OK) return st;
  // An invalid problem sizes to 0 and is rejected by kd_kl_forward below with
  // its usual code; a valid one that needs more scratch than the array holds
  // is rejected here, before anything is queued.
  if (kd_kl_workspace_size(prob, 0) > (size_t)KDKL_NOALLOC_SCRATCH_BYTES) return KD_ERR_WORKSPACE;
  // kd_kl_forward clears the scratch header (status word, token count) at the
  // start of every call, so nothing is left over from the previous call.
  return kd_kl_forward(prob, H, W, topk_idx, topk_logit, mask, loss, lse, token_kl, scratch,
                       (size_t)KDKL_NOALLOC_SCRATCH_BYTES, stream);
}
