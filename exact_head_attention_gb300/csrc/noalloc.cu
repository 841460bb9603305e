// attn_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory, with its scratch space in a fixed array built into this library.
//
// Who needs it: code that runs where device allocation is not allowed or not
// affordable -- for example a plugin inside an inference or training engine
// that owns all device memory and forbids allocation while it executes, or a
// latency-bound loop that cannot risk an allocator call (or its failure) on
// every step.  Such callers still pass every input and output; only the
// backward's scratch (the fp32 dQ accumulator and two fp32 row vectors) comes
// from the array below instead of a caller-supplied workspace.
#include <cstddef>
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/exattn.h"
#include "kernels.h"

namespace exattn {
namespace {

constexpr size_t kScratchBytes = ATTN_BWD_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The scratch array.  A GPU reserves it when this file's module is loaded there
// (with CUDA's default lazy module loading: at the first attn_bwd_noalloc call
// on that device; with eager loading: when the library's code is loaded) and
// keeps it until the process exits.  In host code `g_bwd_scratch` only names a
// host-side stand-in: its device address comes from cudaGetSymbolAddress.  The
// address is looked up once per device and kept, so a device must not be
// reset (cudaDeviceReset) while the library is in use: a new context may place
// the array elsewhere.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_dev[kMaxDevices];  // device address of g_bwd_scratch, per device (null until set up)

}  // namespace
}  // namespace exattn

using namespace exattn;

extern "C" attn_status attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                        const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk,
                                        int d, int causal, float scale, attn_dtype dtype, void* stream) {
  const size_t need = attn_bwd_workspace_size(B, H, Nq, d);
  if (need == 0)  // invalid sizes: let the regular entry point report which argument is wrong
    return attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, nullptr, 0, stream);
  if (need > kScratchBytes) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "attn_bwd_noalloc: this shape needs %zu bytes of scratch; the built-in maximum is %zu",
                  need, kScratchBytes);
    set_last_error(msg);
    return ATTN_ERR_WORKSPACE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "attn_bwd_noalloc: cudaGetDevice: %s", cudaGetErrorName(e));
    set_last_error(msg);
    return ATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "attn_bwd_noalloc: device index %d is beyond the %d devices this library tracks",
                  dev, kMaxDevices);
    set_last_error(msg);
    return ATTN_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  {
    // One-time set-up per device, with that device current: look up the array's device address.
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_dev[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_bwd_scratch);
      if (e != cudaSuccess || !p) {
        char msg[160];
        std::snprintf(msg, sizeof(msg), "attn_bwd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorName(e));
        set_last_error(msg);
        return ATTN_ERR_CUDA;
      }
      g_scratch_dev[dev] = p;
    }
    scratch = g_scratch_dev[dev];
  }
  // The regular backward clears the part of the scratch that must start at zero (the dQ
  // accumulator) and overwrites the rest on every call.
  return attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, scratch, kScratchBytes,
                  stream);
}
