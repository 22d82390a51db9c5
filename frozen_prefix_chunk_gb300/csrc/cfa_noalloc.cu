// cfa_forward_noalloc: the forward pass for callers that cannot allocate.
//
// cfa_forward needs a caller-provided workspace for its split partials.  Some
// callers cannot call cudaMalloc (or any allocator) to make one: a trainer
// that runs beside an inference server which reserved the GPU's memory up
// front, or a plain C program whose device memory is handed out by someone
// else's pool.  This entry point runs the same forward with its scratch in a
// fixed-size array that lives in this file's device module instead, so the
// caller only passes inputs and outputs.
//
// The array is kScratchBytes long.  It is reserved on a device when this
// module is loaded there: with lazy module loading (the CUDA default) that is
// the first use of the array on that device, with eager loading
// (CUDA_MODULE_LOADING=EAGER) every device on which the process uses this
// library holds it, whether or not the entry point is ever called.  It stays
// reserved until the process exits.  All calls share it and it keeps the last
// call's contents; the status word at its start is cleared at the start of
// every call and the split partials are fully rewritten before they are read,
// so nothing else needs clearing.  Calls that overlap on the GPU (different
// streams, or different host threads on one device) race on the array and
// must be serialised by the caller.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "cfa.h"

namespace {

constexpr size_t kScratchBytes = size_t(48) << 20;  // 48 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  In host code the name
// g_scratch is only a host-side stand-in, so the address is looked up once
// per device (this loads the module that holds the array) and cached.  A
// cudaDeviceReset destroys the context and the array with it; the cached
// address is then stale, so this entry point must not be used across a
// device reset in one process.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CFA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return CFA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CFA_OK;
}

}  // namespace

extern "C" {

size_t cfa_noalloc_scratch_bytes(void) { return kScratchBytes; }

int cfa_forward_noalloc(const cfa_args* a, void* o, float* lse, void* stream) {
  const size_t need = cfa_workspace_size(a, CFA_WS_FORWARD);
  if (need == 0) {
    // the arguments are rejected: cfa_forward reports why before it would
    // touch the (absent) workspace, and enqueues nothing
    const int st = cfa_forward(a, o, lse, nullptr, 0, stream);
    return st ? st : CFA_ERR_INVALID_ARG;
  }
  if (need > kScratchBytes) return CFA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st) return st;
  return cfa_forward(a, o, lse, scratch, kScratchBytes, stream);
}

int cfa_noalloc_read_status(void* stream) {
  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st) return st;
  return cfa_read_status(scratch, stream);
}

}  // extern "C"
