// C-ABI entry points declared in include/exattn.h: argument validation,
// TMA tensor-map encoding, the per-device error word and kernel dispatch.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/exattn.h"
#include "kernels.h"

namespace exattn {
namespace {

// Error word written by kernels whose bounded waits expired (0 = no error).
__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  uint32_t* err_word = nullptr;  // device address of g_error_word on this device
};

std::mutex g_mutex;
thread_local char g_last_error[256] = "";

// Records a failing CUDA runtime call for attn_last_error and returns ATTN_ERR_CUDA.
attn_status cuda_fail(const char* what, cudaError_t e) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return ATTN_ERR_CUDA;
}

attn_status driver_fail(const char* what, int code) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: CUresult %d", what, code);
  return ATTN_ERR_CUDA;
}
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

uint64_t wait_timeout_ns() {
  static const uint64_t v = [] {
    const char* s = std::getenv("EXATTN_WAIT_TIMEOUT_MS");
    const long ms = s ? std::strtol(s, nullptr, 10) : 0;
    return static_cast<uint64_t>(ms > 0 ? ms : 4000) * 1000000ull;
  }();
  return v;
}

bool checked_mode() {
  static const bool v = [] {
    const char* s = std::getenv("EXATTN_CHECKED");
    return s && s[0] && s[0] != '0';
  }();
  return v;
}

// Per-device one-time set-up: capability check, error-word address, encoder.
attn_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail("cudaDeviceGetAttribute", e);
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_error_word)) != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
      st.err_word = static_cast<uint32_t*>(p);
      if ((e = cudaMemset(st.err_word, 0, sizeof(uint32_t))) != cudaSuccess) return cuda_fail("cudaMemset", e);
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return cuda_fail("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", e);
        if (q != cudaDriverEntryPointSuccess || !fn) return driver_fail("cuTensorMapEncodeTiled lookup", q);
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
    st.ready = true;
  }
  if (!st.supported) return ATTN_ERR_UNSUPPORTED;
  *out = &st;
  return ATTN_OK;
}

// 3-D map over a contiguous [BH][N][d] 16-bit tensor; box = 64 columns x 128 rows x 1,
// 128-byte swizzle (matches the kernels' shared-memory operand layout); rows
// past N read as zero and are dropped on store.
CUresult encode_map(CUtensorMap* map, const void* ptr, bool bf16, int bh, int n, int d) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(bh)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(n) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kTileRows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                              const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status check_common(int B, int H, int Nq, int Nk, int d, float scale, attn_dtype dtype) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  // grid.y limit of the forward (256 query rows per block) and of the backward (128 key rows per block)
  if ((Nq + 255) / 256 > 65535 || (Nk + 127) / 128 > 65535) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

int padded_rows(int Nq) { return (Nq + kTileRows - 1) / kTileRows * kTileRows; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

attn_status finish(cudaError_t e, cudaStream_t stream) {
  if (e != cudaSuccess) return cuda_fail("kernel launch", e);
  if (checked_mode()) return attn_check_device_error(stream);
  return ATTN_OK;
}

}  // namespace
}  // namespace exattn

using namespace exattn;

extern "C" attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                                int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype, void* stream) {
  attn_status st = check_common(B, H, Nq, Nk, d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != ATTN_OK) return st;
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const bool bf16 = dtype == ATTN_BF16;
  const int bh = B * H;
  CUresult r;
  if ((r = encode_map(&a.tm_q, Q, bf16, bh, Nq, d)) != CUDA_SUCCESS || (r = encode_map(&a.tm_k, K, bf16, bh, Nk, d)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_v, V, bf16, bh, Nk, d)) != CUDA_SUCCESS || (r = encode_map(&a.tm_o, O, bf16, bh, Nq, d)) != CUDA_SUCCESS)
    return driver_fail("cuTensorMapEncodeTiled", r);
  a.lse = LSE;
  a.err_word = ds->err_word;
  a.bh_count = bh;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal != 0;
  a.bf16 = bf16;
  a.scale = scale;
  a.timeout_ns = wait_timeout_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_fwd(a, s), s);
}

extern "C" size_t attn_bwd_workspace_size(int B, int H, int Nq, int d) {
  if (B <= 0 || H <= 0 || Nq <= 0 || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * padded_rows(Nq);
  return align256(rows * d * sizeof(float)) + 2 * align256(rows * sizeof(float));
}

namespace {

attn_status bwd_steps(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                      void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                      attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream, int steps) {
  attn_status st = check_common(B, H, Nq, Nk, d, scale, dtype);
  if (st != ATTN_OK) return st;
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return ATTN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < attn_bwd_workspace_size(B, H, Nq, d)) return ATTN_ERR_WORKSPACE;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(LSE) ||
      !aligned16(dQ) || !aligned16(dK) || !aligned16(dV) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != ATTN_OK) return st;
  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const bool bf16 = dtype == ATTN_BF16;
  const int bh = B * H;
  CUresult r;
  if ((r = encode_map(&a.tm_q, Q, bf16, bh, Nq, d)) != CUDA_SUCCESS || (r = encode_map(&a.tm_k, K, bf16, bh, Nk, d)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_v, V, bf16, bh, Nk, d)) != CUDA_SUCCESS || (r = encode_map(&a.tm_do, dO, bf16, bh, Nq, d)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_dk, dK, bf16, bh, Nk, d)) != CUDA_SUCCESS || (r = encode_map(&a.tm_dv, dV, bf16, bh, Nk, d)) != CUDA_SUCCESS)
    return driver_fail("cuTensorMapEncodeTiled", r);
  const int nq_pad = padded_rows(Nq);
  const size_t rows = static_cast<size_t>(bh) * nq_pad;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o = O;
  a.dout = dO;
  a.lse = LSE;
  a.dq = dQ;
  a.dq_acc = reinterpret_cast<float*>(ws);
  a.lse2 = reinterpret_cast<float*>(ws + align256(rows * d * sizeof(float)));
  a.dsum = reinterpret_cast<float*>(ws + align256(rows * d * sizeof(float)) + align256(rows * sizeof(float)));
  a.err_word = ds->err_word;
  a.bh_count = bh;
  a.Nq = Nq;
  a.Nq_pad = nq_pad;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal != 0;
  a.bf16 = bf16;
  a.scale = scale;
  a.timeout_ns = wait_timeout_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_bwd(a, steps, s), s);
}

}  // namespace

extern "C" attn_status attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk, int d,
                                int causal, float scale, attn_dtype dtype, void* workspace, size_t workspace_bytes,
                                void* stream) {
  return bwd_steps(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                   workspace_bytes, stream, kBwdAll);
}

extern "C" attn_status attn_bwd_preprocess(const void* Q, const void* K, const void* V, const void* O,
                                           const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                                           int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_steps(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                   workspace_bytes, stream, kBwdPre);
}

extern "C" attn_status attn_bwd_kv_blocks(const void* Q, const void* K, const void* V, const void* O,
                                          const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                                          int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_steps(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                   workspace_bytes, stream, kBwdMain);
}

extern "C" attn_status attn_bwd_dq_convert(const void* Q, const void* K, const void* V, const void* O,
                                           const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                                           int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_steps(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                   workspace_bytes, stream, kBwdConvert);
}

extern "C" const char* attn_status_string(attn_status status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported (head dim must be 64 or 128; device must be sm_103)";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case ATTN_ERR_CUDA: return "CUDA runtime or launch error";
    case ATTN_ERR_TIMEOUT: return "a bounded device wait expired";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_NOT_IMPLEMENTED: return "not implemented";
  }
  return "unknown status";
}

extern "C" attn_status attn_check_device_error(void* stream) {
  DeviceState* ds = nullptr;
  attn_status st = device_state(&ds);
  if (st != ATTN_OK) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
  uint32_t code = 0;
  if ((e = cudaMemcpy(&code, ds->err_word, sizeof(code), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail("cudaMemcpy(error word)", e);
  if (code != 0) {
    const uint32_t zero = 0;
    if ((e = cudaMemcpy(ds->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail("cudaMemcpy(error word)", e);
    if (code == 8) {
      std::snprintf(g_last_error, sizeof(g_last_error), "device error word 8: dynamic shared memory not 1024-byte aligned");
      return ATTN_ERR_CUDA;
    }
    std::snprintf(g_last_error, sizeof(g_last_error), "device error word %u (a bounded wait expired)", code);
    return ATTN_ERR_TIMEOUT;
  }
  return ATTN_OK;
}

extern "C" const char* attn_last_error(void) { return g_last_error; }

void exattn::set_last_error(const char* msg) { std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }
