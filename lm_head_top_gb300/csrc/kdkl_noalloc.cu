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
// per device and context, with that device current, on the first call made on
// it (and again on the first call after a device reset).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kdkl.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[KDKL_NOALLOC_SCRATCH_BYTES];

// The array's device address belongs to a CUDA context: after a device reset
// the device's next primary context places it anew. So the cached address is
// kept with the id of the context it was looked up in (cuCtxGetId, reached
// through the runtime's driver entry point) and looked up again when the
// current context's id differs.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_once;

struct ScratchAddr {
  unsigned long long ctx_id = 0;  // 0: not looked up yet
  void* addr = nullptr;
};
constexpr int kMaxDevices = 64;
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

kd_status current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return KD_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return KD_ERR_CUDA;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS ? KD_OK : KD_ERR_CUDA;
}

// Device address of the scratch array in the current device's context,
// looked up with cudaGetSymbolAddress the first time it is needed there (a
// runtime call, which also makes the device's primary context current when
// no call has done so yet).
kd_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KD_ERR_UNSUPPORTED;
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx) == KD_OK;  // false before the first runtime call
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& a = g_scratch[dev];
  if (!have_ctx || a.addr == nullptr || a.ctx_id != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return KD_ERR_CUDA;
    if (!have_ctx && current_context_id(&ctx) != KD_OK) return KD_ERR_CUDA;
    a.addr = p;
    a.ctx_id = ctx;
  }
  *out = a.addr;
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

// Reads back the device-detected status of the latest allocation-free call on
// the current device (the status word sits at the start of the scratch array).
extern "C" kd_status kd_kl_noalloc_check_status(void* stream) {
  void* scratch = nullptr;
  const kd_status st = scratch_on_current_device(&scratch);
  if (st != KD_OK) return st;
  return kd_kl_check_status(scratch, stream);
}
