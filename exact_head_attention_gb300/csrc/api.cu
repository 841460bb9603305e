// C-ABI entry points declared in include/exattn.h: argument validation,
// TMA tensor-map encoding, the per-device error word and kernel dispatch.
#include <algorithm>
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
#include "fwd_schedule.h"
#include "kernels.h"
#include "ptx.cuh"

namespace exattn {
namespace {

// Error word written by kernels whose bounded waits expired (0 = no error).
__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  uint32_t* err_word = nullptr;  // device address of g_error_word on this device
  size_t l2_bytes = 0;
  int sm_count = 0;
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
      int l2 = 0, sms = 0;
      if ((e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_fail("cudaDeviceGetAttribute", e);
      st.l2_bytes = static_cast<size_t>(l2);
      st.sm_count = sms;
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

// 4-D map {d, N, H, B} over a 16-bit tensor with element strides `st` (d contiguous); box = 64
// columns x 128 rows x 1 x 1, 128-byte swizzle (the kernels' shared-memory operand layout); rows
// past N read as zero and are dropped on store.
CUresult encode_map(CUtensorMap* map, const void* ptr, bool bf16, int B, int H, int n, int d, const RowStrides& st) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n) * 2, static_cast<cuuint64_t>(st.h) * 2,
                                 static_cast<cuuint64_t>(st.b) * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kTileRows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                              const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r;
}

// 2-D fp32 map over the backward's dQ accumulator [rows][d]: box = 32 columns (128 bytes) x 128 rows,
// 128-byte swizzle; the d = 64 kernel reduce-adds [128 query][32 d] boxes into it.
CUresult encode_acc_map(CUtensorMap* map, float* acc, size_t rows, int d) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(kTileRows)};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, acc, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

RowStrides contiguous(int H, int n, int d) {
  return RowStrides{static_cast<long long>(H) * n * d, static_cast<long long>(n) * d, d};
}

// Checks a caller's strides and replaces the stride of a dimension of extent 1 (never used to
// address anything) by the row stride, so that the tensor map accepts it.
bool normalise_strides(const attn_strides& in, int B, int H, int d, RowStrides* out) {
  constexpr long long kMax = (1ll << 39) - 1;  // byte strides below 2^40
  RowStrides st{in.batch, in.head, in.row};
  if (st.n < d || st.n % 8 != 0 || st.n > kMax) return false;
  if (H == 1) st.h = st.n;
  if (B == 1) st.b = st.n;
  if (st.h <= 0 || st.h % 8 != 0 || st.h > kMax) return false;
  if (st.b <= 0 || st.b % 8 != 0 || st.b > kMax) return false;
  *out = st;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status check_common(int B, int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return ATTN_ERR_INVALID_ARG;
  if (causal != ATTN_MASK_NONE && causal != ATTN_MASK_CAUSAL && causal != ATTN_MASK_CAUSAL_BOTTOM_RIGHT)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  if (bh > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  // grid.y limit of the forward (256 query rows per block) and of the backward (128 key rows per block)
  if ((Nq + 255) / 256 > 65535 || (Nk + 127) / 128 > 65535) return ATTN_ERR_INVALID_ARG;
  // the key/value-block kernels number their B*H*ceil(Nk/128) blocks along grid.x in an int
  if (bh * ((Nk + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

int padded_rows(int Nq) { return (Nq + kTileRows - 1) / kTileRows * kTileRows; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Diagonal offset of the causal mask: query q sees keys k <= q + offset.
int causal_offset(int causal, int Nq, int Nk) { return causal == ATTN_MASK_CAUSAL_BOTTOM_RIGHT ? Nk - Nq : 0; }

// Heads per launch group of the key/value-block kernels (kv_order.cuh) when they add dQ into an fp32
// accumulator of acc_per_head bytes per head.  All heads in one group (heads fastest) while the whole
// accumulator fits in a quarter of L2 with no mask, or in half of it under a causal mask (key block j
// adds only into the rows at or after its own, and the heavy blocks of every head start first); the rest
// of L2 holds the Q, dO, K and V tiles in flight.  Past that, groups whose accumulator rows take about a
// sixteenth of L2, so each head's key blocks find its rows still in L2 (swept over 1 to 64 heads per
// group on GB300, that size was within a few per cent of the best group on every shape).  Under a causal
// mask the first key block of a head is the heaviest (it sees every query tile), and a group's first
// blocks start only when that group does; a group of at least 2 * SMs / nkb heads has enough lighter
// blocks to run beside them.
int head_group_for(bool causal, long long bh, int Nk, size_t acc_per_head, size_t l2_bytes, int sm_count) {
  if (static_cast<size_t>(bh) * acc_per_head <= (causal ? l2_bytes / 2 : l2_bytes / 4)) return static_cast<int>(bh);
  long long g = std::max<long long>(1, static_cast<long long>(l2_bytes / 16 / acc_per_head));
  if (causal) {
    const long long nkb = (Nk + kTileRows - 1) / kTileRows;
    g = std::max(g, (2LL * sm_count + nkb - 1) / nkb);
  }
  return static_cast<int>(std::min(g, bh));
}

int head_group(bool causal, long long bh, int Nk, size_t acc_per_head, const DeviceState* ds) {
  return head_group_for(causal, bh, Nk, acc_per_head, ds->l2_bytes, ds->sm_count);
}

attn_status finish(cudaError_t e, cudaStream_t stream) {
  if (e != cudaSuccess) return cuda_fail("kernel launch", e);
  if (checked_mode()) return attn_check_device_error(stream);
  return ATTN_OK;
}

}  // namespace
}  // namespace exattn

using namespace exattn;

namespace {

attn_status fwd_impl(const void* Q, const RowStrides& qs, const void* K, const RowStrides& ks, const void* V,
                     const RowStrides& vs, void* O, const RowStrides& os, float* LSE, int B, int H, int Nq, int Nk,
                     int d, int causal, float scale, attn_dtype dtype, void* stream) {
  DeviceState* ds = nullptr;
  attn_status st = device_state(&ds);
  if (st != ATTN_OK) return st;
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const bool bf16 = dtype == ATTN_BF16;
  CUresult r;
  if ((r = encode_map(&a.tm_q, Q, bf16, B, H, Nq, d, qs)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_k, K, bf16, B, H, Nk, d, ks)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_v, V, bf16, B, H, Nk, d, vs)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_o, O, bf16, B, H, Nq, d, os)) != CUDA_SUCCESS)
    return driver_fail("cuTensorMapEncodeTiled", r);
  a.lse = LSE;
  a.err_word = ds->err_word;
  a.sm_count = ds->sm_count;
  a.bh_count = B * H;
  a.heads = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal != ATTN_MASK_NONE;
  a.causal_off = causal_offset(causal, Nq, Nk);
  a.bf16 = bf16;
  a.scale = scale;
  a.timeout_ns = wait_timeout_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_fwd(a, s), s);
}

}  // namespace

extern "C" attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                                int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype, void* stream) {
  attn_status st = check_common(B, H, Nq, Nk, d, causal, scale, dtype);
  if (st != ATTN_OK) return st;
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return ATTN_ERR_MISALIGNED;
  const RowStrides qs = contiguous(H, Nq, d), ks = contiguous(H, Nk, d);
  return fwd_impl(Q, qs, K, ks, V, ks, O, qs, LSE, B, H, Nq, Nk, d, causal, scale, dtype, stream);
}

extern "C" attn_status attn_fwd_strided(const void* Q, attn_strides q_strides, const void* K, attn_strides k_strides,
                                        const void* V, attn_strides v_strides, void* O, attn_strides o_strides,
                                        float* LSE, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                        attn_dtype dtype, void* stream) {
  attn_status st = check_common(B, H, Nq, Nk, d, causal, scale, dtype);
  if (st != ATTN_OK) return st;
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  RowStrides qs, ks, vs, os;
  if (!normalise_strides(q_strides, B, H, d, &qs) || !normalise_strides(k_strides, B, H, d, &ks) ||
      !normalise_strides(v_strides, B, H, d, &vs) || !normalise_strides(o_strides, B, H, d, &os))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return ATTN_ERR_MISALIGNED;
  return fwd_impl(Q, qs, K, ks, V, vs, O, os, LSE, B, H, Nq, Nk, d, causal, scale, dtype, stream);
}

extern "C" size_t attn_bwd_workspace_size(int B, int H, int Nq, int d) {
  if (B <= 0 || H <= 0 || Nq <= 0 || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * padded_rows(Nq);
  return align256(rows * d * sizeof(float)) + 2 * align256(rows * sizeof(float));
}

// The forward's packed lists of query blocks (persistent_schedule), for callers and tests.
extern "C" int attn_fwd_schedule(int B, int H, int Nq, int Nk, int d, int causal, int sm_count, uint32_t* blocks,
                                 int blocks_cap, int* begin, int begin_cap) {
  if (check_common(B, H, Nq, Nk, d, causal, 1.0f, ATTN_BF16) != ATTN_OK) return -1;
  if (sm_count <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return -1;
  }
  if (causal == ATTN_MASK_NONE || fwd_uses_tile_kernel(d, true, Nk)) return 0;
  const int nqb = (Nq + kFwdSubTiles * kTileRows - 1) / (kFwdSubTiles * kTileRows);
  const FwdSchedule* sch = persistent_schedule(B * H, nqb, Nq, Nk, causal_offset(causal, Nq, Nk), sm_count);
  if (!sch) return 0;
  const int n = sch->begin[sch->ctas];
  if (!blocks || !begin || blocks_cap < n || begin_cap < sch->ctas + 1) return -1;
  for (int i = 0; i < n; ++i) blocks[i] = sch->unit[i];
  for (int c = 0; c <= sch->ctas; ++c) begin[c] = sch->begin[c];
  return sch->ctas;
}

// The launch grouping head_group picks, for callers and tests (sm_count / l2_bytes 0: this device's).
extern "C" int attn_bwd_head_group(int B, int H, int Nq, int Nk, int d, int causal, int sm_count, size_t l2_bytes) {
  if (check_common(B, H, Nq, Nk, d, causal, 1.0f, ATTN_BF16) != ATTN_OK) return -1;
  if (sm_count <= 0 || l2_bytes == 0) {
    int dev = 0, sms = 0, l2 = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return -1;
    if (sm_count <= 0) sm_count = sms;
    if (l2_bytes == 0) l2_bytes = static_cast<size_t>(l2);
  }
  const size_t acc_per_head = static_cast<size_t>(padded_rows(Nq)) * d * sizeof(float);
  return head_group_for(causal != ATTN_MASK_NONE, static_cast<long long>(B) * H, Nk, acc_per_head, l2_bytes, sm_count);
}

// ATTN_DQ_AUTO.  The StreamKL summary (backward, kernel fusion) adds dQ atomically while the buffer fits
// in L2 and uses separate kernels when contention grows.  What decides on GB300 is whether the key
// blocks that add into the same head's rows find them still in L2, and the launch order
// (head_group) sees to that: a head's blocks run close together whenever the accumulator as a whole
// would not stay in L2.  The reductions then measured faster than the query-tile kernel on every
// shape tried, by 1.3x to 1.6x, so the rule takes them for every shape; the mask is not needed.
extern "C" int attn_bwd_auto_dq_mode(int B, int H, int Nq, int Nk, int d, int /*causal*/) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return -1;
  return ATTN_DQ_ATOMIC;
}

namespace {

// Tensor views of one backward call (element strides; d contiguous).
struct BwdViews {
  RowStrides q, k, v, o, dout, dq, dk, dv;
};

attn_status bwd_steps(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                      void* dQ, void* dK, void* dV, const BwdViews& vw, int B, int H, int Nq, int Nk, int d,
                      int causal, float scale, attn_dtype dtype, void* workspace, size_t workspace_bytes,
                      void* stream, int steps, int dq_mode = ATTN_DQ_ATOMIC) {
  if (dq_mode != ATTN_DQ_ATOMIC && dq_mode != ATTN_DQ_DETERMINISTIC && dq_mode != ATTN_DQ_AUTO)
    return ATTN_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return ATTN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < attn_bwd_workspace_size(B, H, Nq, d)) return ATTN_ERR_WORKSPACE;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(LSE) ||
      !aligned16(dQ) || !aligned16(dK) || !aligned16(dV) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  attn_status st = device_state(&ds);
  if (st != ATTN_OK) return st;
  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  const bool bf16 = dtype == ATTN_BF16;
  const int bh = B * H;
  CUresult r;
  if ((r = encode_map(&a.tm_q, Q, bf16, B, H, Nq, d, vw.q)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_k, K, bf16, B, H, Nk, d, vw.k)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_v, V, bf16, B, H, Nk, d, vw.v)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_do, dO, bf16, B, H, Nq, d, vw.dout)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_dk, dK, bf16, B, H, Nk, d, vw.dk)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_dv, dV, bf16, B, H, Nk, d, vw.dv)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_dq, dQ, bf16, B, H, Nq, d, vw.dq)) != CUDA_SUCCESS)
    return driver_fail("cuTensorMapEncodeTiled", r);
  if (dq_mode == ATTN_DQ_AUTO) dq_mode = attn_bwd_auto_dq_mode(B, H, Nq, Nk, d, causal);
  const int nq_pad = padded_rows(Nq);
  const size_t rows = static_cast<size_t>(bh) * nq_pad;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o = O;
  a.dout = dO;
  a.lse = LSE;
  a.dq = dQ;
  a.so = vw.o;
  a.sdo = vw.dout;
  a.sdq = vw.dq;
  a.dq_acc = reinterpret_cast<float*>(ws);
  a.nlse2 = reinterpret_cast<float*>(ws + align256(rows * d * sizeof(float)));
  a.dsum = reinterpret_cast<float*>(ws + align256(rows * d * sizeof(float)) + align256(rows * sizeof(float)));
  a.err_word = ds->err_word;
  a.bh_count = bh;
  a.heads = H;
  a.Nq = Nq;
  a.Nq_pad = nq_pad;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal != ATTN_MASK_NONE;
  a.causal_off = causal_offset(causal, Nq, Nk);
  a.bf16 = bf16;
  a.scale = scale;
  a.timeout_ns = wait_timeout_ns();
  // deterministic mode: no accumulator, heads fastest
  a.head_group = dq_mode == ATTN_DQ_DETERMINISTIC ? static_cast<int>(bh)
                                                  : head_group(a.causal, bh, Nk, static_cast<size_t>(nq_pad) * d * sizeof(float), ds);
  if (dq_mode == ATTN_DQ_DETERMINISTIC) {
    a.dq_acc = nullptr;  // no accumulator: dK, dV from the key/value blocks, dQ from the query-tile kernel
    steps = kBwdDeterministic;
  } else if (d == 64 && rows > 0x7fffffffull) {
    return ATTN_ERR_INVALID_ARG;  // the accumulator map's row coordinate is a 32-bit integer
  } else if (d == 64 && (r = encode_acc_map(&a.tm_dqacc, a.dq_acc, rows, d)) != CUDA_SUCCESS) {
    return driver_fail("cuTensorMapEncodeTiled(dQ accumulator)", r);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_bwd(a, steps, s), s);
}

// Contiguous [B][H][N][d] tensors.
attn_status bwd_contiguous(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                           const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk, int d,
                           int causal, float scale, attn_dtype dtype, void* workspace, size_t workspace_bytes,
                           void* stream, int steps, int dq_mode = ATTN_DQ_ATOMIC) {
  attn_status st = check_common(B, H, Nq, Nk, d, causal, scale, dtype);
  if (st != ATTN_OK) return st;
  const RowStrides qs = contiguous(H, Nq, d), ks = contiguous(H, Nk, d);
  const BwdViews vw{qs, ks, ks, qs, qs, qs, ks, ks};
  return bwd_steps(Q, K, V, O, dO, LSE, dQ, dK, dV, vw, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                   workspace_bytes, stream, steps, dq_mode);
}

}  // namespace

extern "C" attn_status attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk, int d,
                                int causal, float scale, attn_dtype dtype, void* workspace, size_t workspace_bytes,
                                void* stream) {
  return bwd_contiguous(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                        workspace_bytes, stream, kBwdAll);
}

extern "C" attn_status attn_bwd_strided_ex(const void* Q, attn_strides q_strides, const void* K,
                                           attn_strides k_strides, const void* V, attn_strides v_strides,
                                           const void* O, attn_strides o_strides, const void* dO,
                                           attn_strides do_strides, const float* LSE, void* dQ,
                                           attn_strides dq_strides, void* dK, attn_strides dk_strides, void* dV,
                                           attn_strides dv_strides, int B, int H, int Nq, int Nk, int d, int causal,
                                           float scale, attn_dtype dtype, int dq_mode, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  attn_status st = check_common(B, H, Nq, Nk, d, causal, scale, dtype);
  if (st != ATTN_OK) return st;
  BwdViews vw;
  if (!normalise_strides(q_strides, B, H, d, &vw.q) || !normalise_strides(k_strides, B, H, d, &vw.k) ||
      !normalise_strides(v_strides, B, H, d, &vw.v) || !normalise_strides(o_strides, B, H, d, &vw.o) ||
      !normalise_strides(do_strides, B, H, d, &vw.dout) || !normalise_strides(dq_strides, B, H, d, &vw.dq) ||
      !normalise_strides(dk_strides, B, H, d, &vw.dk) || !normalise_strides(dv_strides, B, H, d, &vw.dv))
    return ATTN_ERR_INVALID_ARG;
  return bwd_steps(Q, K, V, O, dO, LSE, dQ, dK, dV, vw, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                   workspace_bytes, stream, kBwdAll, dq_mode);
}

extern "C" attn_status attn_bwd_strided(const void* Q, attn_strides q_strides, const void* K, attn_strides k_strides,
                                        const void* V, attn_strides v_strides, const void* O, attn_strides o_strides,
                                        const void* dO, attn_strides do_strides, const float* LSE, void* dQ,
                                        attn_strides dq_strides, void* dK, attn_strides dk_strides, void* dV,
                                        attn_strides dv_strides, int B, int H, int Nq, int Nk, int d, int causal,
                                        float scale, attn_dtype dtype, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  return attn_bwd_strided_ex(Q, q_strides, K, k_strides, V, v_strides, O, o_strides, dO, do_strides, LSE, dQ,
                             dq_strides, dK, dk_strides, dV, dv_strides, B, H, Nq, Nk, d, causal, scale, dtype,
                             ATTN_DQ_ATOMIC, workspace, workspace_bytes, stream);
}

extern "C" attn_status attn_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                   const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nk,
                                   int d, int causal, float scale, attn_dtype dtype, int dq_mode, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  return bwd_contiguous(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                        workspace_bytes, stream, kBwdAll, dq_mode);
}

extern "C" attn_status attn_bwd_preprocess(const void* Q, const void* K, const void* V, const void* O,
                                           const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                                           int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_contiguous(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                        workspace_bytes, stream, kBwdPre);
}

extern "C" attn_status attn_bwd_kv_blocks(const void* Q, const void* K, const void* V, const void* O,
                                          const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                                          int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_contiguous(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
                        workspace_bytes, stream, kBwdMain);
}

extern "C" attn_status attn_bwd_dq_convert(const void* Q, const void* K, const void* V, const void* O,
                                           const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                                           int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_contiguous(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, dtype, workspace,
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

// ----------------------------------------------------------------- split-KV forward

namespace {

constexpr int kMaxSplits = 256;

// Slices per query tile that minimise (waves of CTAs) x (key tiles per CTA + one tile of fixed cost),
// with `per_sm` slice CTAs resident per SM.  1 means the plain forward is the better launch, which is
// always the case once the query tiles alone fill the SMs.
int choose_splits(long long bh, int Nq, int Nk, int sm_count, int per_sm) {
  const long long base = bh * ((Nq + kTileRows - 1) / kTileRows);
  const int nkv = (Nk + kTileRows - 1) / kTileRows;
  if (base >= sm_count) return 1;
  const long long slots = static_cast<long long>(sm_count) * per_sm;
  int best = 1;
  double best_cost = 0.0;
  for (int s = 1; s <= std::min(nkv, kMaxSplits); ++s) {
    const long long waves = (base * s + slots - 1) / slots;
    const double cost = static_cast<double>(waves) * ((nkv + s - 1) / s + 1);
    if (s == 1 || cost < best_cost * 0.98) {  // a split must win clearly: it adds a merge pass
      best = s;
      best_cost = cost;
    }
  }
  return best;
}

// Slice CTAs of the split-KV attention forward resident per SM: two at d = 64 (the one-tile kernel of
// fwd_tile.cuh), one at d = 128.
int split_blocks_per_sm(int d) { return d == 64 ? 2 : 1; }

int device_sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return sms;
}

size_t split_workspace(int B, int H, int Nq, int d, int splits) {
  const size_t rows = static_cast<size_t>(splits) * B * H * Nq;
  return align256(rows * d * sizeof(float)) + align256(rows * sizeof(float));
}

attn_status fwd_split_impl(const void* Q, const RowStrides& qs, const void* K, const RowStrides& ks, const void* V,
                           const RowStrides& vs, void* O, const RowStrides& os, float* LSE, int B, int H, int Nq,
                           int Nk, int d, int causal, float scale, attn_dtype dtype, int num_splits,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  if ((Nq + kTileRows - 1) / kTileRows > 65535 || static_cast<long long>(B) * H * Nq / 8 >= 0x7fffffffLL)
    return ATTN_ERR_INVALID_ARG;
  if (num_splits == 0) {
    int sms = device_sm_count();
    num_splits = choose_splits(static_cast<long long>(B) * H, Nq, Nk, sms > 0 ? sms : 1, split_blocks_per_sm(d));
    if (num_splits == 1) return fwd_impl(Q, qs, K, ks, V, vs, O, os, LSE, B, H, Nq, Nk, d, causal, scale, dtype, stream);
  }
  if (!workspace || workspace_bytes < split_workspace(B, H, Nq, d, num_splits)) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  attn_status st = device_state(&ds);
  if (st != ATTN_OK) return st;
  SplitArgs a;
  std::memset(&a, 0, sizeof(a));
  const bool bf16 = dtype == ATTN_BF16;
  CUresult r;
  if ((r = encode_map(&a.tm_q, Q, bf16, B, H, Nq, d, qs)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_k, K, bf16, B, H, Nk, d, ks)) != CUDA_SUCCESS ||
      (r = encode_map(&a.tm_v, V, bf16, B, H, Nk, d, vs)) != CUDA_SUCCESS)
    return driver_fail("cuTensorMapEncodeTiled", r);
  const size_t rows = static_cast<size_t>(num_splits) * B * H * Nq;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.o_part = reinterpret_cast<float*>(ws);
  a.l_part = reinterpret_cast<float*>(ws + align256(rows * d * sizeof(float)));
  a.o = O;
  a.so = os;
  a.lse = LSE;
  a.err_word = ds->err_word;
  a.bh_count = B * H;
  a.heads = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.splits = num_splits;
  a.causal = causal != ATTN_MASK_NONE;
  a.causal_off = causal_offset(causal, Nq, Nk);
  a.bf16 = bf16;
  a.scale = scale;
  a.timeout_ns = wait_timeout_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_fwd_split(a, s), s);
}

}  // namespace

extern "C" int attn_fwd_splitkv_num_splits(int B, int H, int Nq, int Nk, int d, int sm_count) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128)) return 0;
  if (sm_count <= 0) sm_count = device_sm_count();
  if (sm_count <= 0) return 0;
  return choose_splits(static_cast<long long>(B) * H, Nq, Nk, sm_count, split_blocks_per_sm(d));
}

extern "C" size_t attn_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128) || num_splits < 0 || num_splits > kMaxSplits)
    return 0;
  if (num_splits == 0) {
    num_splits = attn_fwd_splitkv_num_splits(B, H, Nq, Nk, d, 0);
    if (num_splits <= 1) return 0;
  }
  return split_workspace(B, H, Nq, d, num_splits);
}

extern "C" attn_status attn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                                        int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype,
                                        int num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  attn_status st = check_common(B, H, Nq, Nk, d, causal, scale, dtype);
  if (st != ATTN_OK) return st;
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return ATTN_ERR_MISALIGNED;
  const RowStrides qs = contiguous(H, Nq, d), ks = contiguous(H, Nk, d);
  return fwd_split_impl(Q, qs, K, ks, V, ks, O, qs, LSE, B, H, Nq, Nk, d, causal, scale, dtype, num_splits,
                        workspace, workspace_bytes, stream);
}

extern "C" attn_status attn_fwd_splitkv_strided(const void* Q, attn_strides q_strides, const void* K,
                                                attn_strides k_strides, const void* V, attn_strides v_strides,
                                                void* O, attn_strides o_strides, float* LSE, int B, int H, int Nq,
                                                int Nk, int d, int causal, float scale, attn_dtype dtype,
                                                int num_splits, void* workspace, size_t workspace_bytes,
                                                void* stream) {
  attn_status st = check_common(B, H, Nq, Nk, d, causal, scale, dtype);
  if (st != ATTN_OK) return st;
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  RowStrides qs, ks, vs, os;
  if (!normalise_strides(q_strides, B, H, d, &qs) || !normalise_strides(k_strides, B, H, d, &ks) ||
      !normalise_strides(v_strides, B, H, d, &vs) || !normalise_strides(o_strides, B, H, d, &os))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return ATTN_ERR_MISALIGNED;
  return fwd_split_impl(Q, qs, K, ks, V, vs, O, os, LSE, B, H, Nq, Nk, d, causal, scale, dtype, num_splits,
                        workspace, workspace_bytes, stream);
}

// ----------------------------------------------------------------- attention KL divergence

namespace {

attn_status kl_common(const void* Q1, const void* K1, const void* Q2, const void* K2, int B, int H, int Nq, int Nk,
                      int d, int causal, float scale, attn_dtype dtype, KlArgs* a, DeviceState** ds) {
  attn_status st = check_common(B, H, Nq, Nk, d, causal, scale, dtype);
  if (st != ATTN_OK) return st;
  if ((Nq + kTileRows - 1) / kTileRows > 65535) return ATTN_ERR_INVALID_ARG;
  if (!Q1 || !K1 || !Q2 || !K2) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(Q1) || !aligned16(K1) || !aligned16(Q2) || !aligned16(K2)) return ATTN_ERR_MISALIGNED;
  if ((st = device_state(ds)) != ATTN_OK) return st;
  std::memset(a, 0, sizeof(*a));
  const bool bf16 = dtype == ATTN_BF16;
  const RowStrides qs = contiguous(H, Nq, d), ks = contiguous(H, Nk, d);
  CUresult r;
  if ((r = encode_map(&a->tm_qa, Q1, bf16, B, H, Nq, d, qs)) != CUDA_SUCCESS ||
      (r = encode_map(&a->tm_ka, K1, bf16, B, H, Nk, d, ks)) != CUDA_SUCCESS ||
      (r = encode_map(&a->tm_qb, Q2, bf16, B, H, Nq, d, qs)) != CUDA_SUCCESS ||
      (r = encode_map(&a->tm_kb, K2, bf16, B, H, Nk, d, ks)) != CUDA_SUCCESS)
    return driver_fail("cuTensorMapEncodeTiled", r);
  a->err_word = (*ds)->err_word;
  a->bh_count = B * H;
  a->heads = H;
  a->Nq = Nq;
  a->Nk = Nk;
  a->d = d;
  a->causal = causal != ATTN_MASK_NONE;
  a->causal_off = causal_offset(causal, Nq, Nk);
  a->bf16 = bf16;
  a->scale = scale;
  a->timeout_ns = wait_timeout_ns();
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_kl_fwd(const void* Q1, const void* K1, const void* Q2, const void* K2, float* KL,
                                   float* LSE1, float* LSE2, int B, int H, int Nq, int Nk, int d, int causal,
                                   float scale, attn_dtype dtype, void* stream) {
  if (!KL || !LSE1 || !LSE2) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(KL) || !aligned16(LSE1) || !aligned16(LSE2)) return ATTN_ERR_MISALIGNED;
  KlArgs a;
  DeviceState* ds = nullptr;
  attn_status st = kl_common(Q1, K1, Q2, K2, B, H, Nq, Nk, d, causal, scale, dtype, &a, &ds);
  if (st != ATTN_OK) return st;
  a.kl = KL;
  a.lse1 = LSE1;
  a.lse2 = LSE2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_kl_fwd(a, s), s);
}

extern "C" size_t attn_kl_bwd_workspace_size(int B, int H, int Nq, int d) {
  if (B <= 0 || H <= 0 || Nq <= 0 || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * padded_rows(Nq);
  return align256(rows * d * sizeof(float)) + align256(3 * rows * sizeof(float));
}

namespace {

attn_status kl_bwd_impl(const void* Q1, const void* K1, const void* Q2, const void* K2, const float* KL,
                        const float* LSE1, const float* LSE2, const float* G, int setting, void* dQ, void* dK, int B,
                        int H, int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype, int dq_mode,
                        void* workspace, size_t workspace_bytes, void* stream) {
  if (setting != 1 && setting != 2) return ATTN_ERR_INVALID_ARG;
  if (dq_mode != ATTN_DQ_ATOMIC && dq_mode != ATTN_DQ_DETERMINISTIC && dq_mode != ATTN_DQ_AUTO)
    return ATTN_ERR_INVALID_ARG;
  if (!KL || !LSE1 || !LSE2 || !G || !dQ || !dK) return ATTN_ERR_INVALID_ARG;
  const bool fused = dq_mode != ATTN_DQ_DETERMINISTIC;  // AUTO: the one-pass kernel, as for attention
  if (fused && (!workspace || workspace_bytes < attn_kl_bwd_workspace_size(B, H, Nq, d))) return ATTN_ERR_WORKSPACE;
  if (!aligned16(KL) || !aligned16(LSE1) || !aligned16(LSE2) || !aligned16(G) || !aligned16(dQ) || !aligned16(dK))
    return ATTN_ERR_MISALIGNED;
  if (fused && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_MISALIGNED;
  KlArgs a;
  DeviceState* ds = nullptr;
  attn_status st = kl_common(Q1, K1, Q2, K2, B, H, Nq, Nk, d, causal, scale, dtype, &a, &ds);
  if (st != ATTN_OK) return st;
  const bool bf16 = dtype == ATTN_BF16;
  CUresult r;
  if ((r = encode_map(&a.tm_dk, dK, bf16, B, H, Nk, d, contiguous(H, Nk, d))) != CUDA_SUCCESS)
    return driver_fail("cuTensorMapEncodeTiled", r);
  a.kl = const_cast<float*>(KL);
  a.lse1 = const_cast<float*>(LSE1);
  a.lse2 = const_cast<float*>(LSE2);
  a.g = G;
  a.op = setting == 1 ? kPairKlStudent : kPairKlTeacher;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fused) {
    // One pass over key tiles: dK, and dQ added into the fp32 accumulator; then dQ = scale * accumulator.
    const size_t rows = static_cast<size_t>(B) * H * padded_rows(Nq);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.dq_acc = reinterpret_cast<float*>(ws);
    a.rowv = reinterpret_cast<float*>(ws + align256(rows * d * sizeof(float)));
    a.Nq_pad = padded_rows(Nq);
    a.head_group = head_group(a.causal, a.bh_count, Nk, static_cast<size_t>(a.Nq_pad) * d * sizeof(float), ds);
    if (d == 64 && rows > 0x7fffffffull) return ATTN_ERR_INVALID_ARG;  // 32-bit row coordinate of the map
    if (d == 64 && (r = encode_acc_map(&a.tm_dqacc, a.dq_acc, rows, d)) != CUDA_SUCCESS)
      return driver_fail("cuTensorMapEncodeTiled (accumulator)", r);
    cudaError_t e = launch_kl_bwd_fused(a, s);
    if (e == cudaSuccess) {
      BwdArgs c;
      std::memset(&c, 0, sizeof(c));
      c.dq = dQ;
      c.sdq = contiguous(H, Nq, d);
      c.dq_acc = a.dq_acc;
      c.err_word = a.err_word;
      c.bh_count = a.bh_count;
      c.heads = H;
      c.Nq = Nq;
      c.Nq_pad = a.Nq_pad;
      c.Nk = Nk;
      c.d = d;
      c.causal = a.causal;
      c.bf16 = bf16;
      c.scale = scale;
      c.timeout_ns = a.timeout_ns;
      e = launch_bwd(c, kBwdConvert, s);
    }
    return finish(e, s);
  }
  // dQ over query tiles (teacher a, student b), then dK over key tiles: no atomics, the same bits on
  // every run.
  PairDqArgs p;
  std::memset(&p, 0, sizeof(p));
  p.tm_qa = a.tm_qa;
  p.tm_ka = a.tm_ka;
  p.tm_qb = a.tm_qb;
  p.tm_kb = a.tm_kb;
  if ((r = encode_map(&p.tm_dq, dQ, bf16, B, H, Nq, d, contiguous(H, Nq, d))) != CUDA_SUCCESS)
    return driver_fail("cuTensorMapEncodeTiled", r);
  p.rv[0] = LSE1;
  p.rv[1] = LSE2;
  p.rv[2] = KL;
  p.rv[3] = G;
  p.rv_stride = Nq;
  p.err_word = a.err_word;
  p.bh_count = a.bh_count;
  p.heads = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.d = d;
  p.causal = a.causal;
  p.bf16 = bf16;
  p.causal_off = a.causal_off;
  p.scale = scale;
  p.op = a.op;
  p.timeout_ns = a.timeout_ns;
  cudaError_t e = launch_pair_dq(p, s);
  if (e == cudaSuccess) e = launch_kl_dk(a, s);
  return finish(e, s);
}

}  // namespace

extern "C" attn_status attn_kl_bwd(const void* Q1, const void* K1, const void* Q2, const void* K2, const float* KL,
                                   const float* LSE1, const float* LSE2, const float* G, int setting, void* dQ,
                                   void* dK, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                   attn_dtype dtype, void* stream) {
  return kl_bwd_impl(Q1, K1, Q2, K2, KL, LSE1, LSE2, G, setting, dQ, dK, B, H, Nq, Nk, d, causal, scale, dtype,
                     ATTN_DQ_DETERMINISTIC, nullptr, 0, stream);
}

extern "C" attn_status attn_kl_bwd_ex(const void* Q1, const void* K1, const void* Q2, const void* K2, const float* KL,
                                      const float* LSE1, const float* LSE2, const float* G, int setting, void* dQ,
                                      void* dK, int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                      attn_dtype dtype, int dq_mode, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  return kl_bwd_impl(Q1, K1, Q2, K2, KL, LSE1, LSE2, G, setting, dQ, dK, B, H, Nq, Nk, d, causal, scale, dtype,
                     dq_mode, workspace, workspace_bytes, stream);
}

// ----------------------------------------------------------------- bounded-wait self-test

namespace exattn {
namespace {

// One block; its first thread waits on an mbarrier that nothing arrives at, through the same bounded
// wait the attention kernels use.  The wait gives up after timeout_ns, records the timeout in the error
// word and the kernel returns normally.
__global__ void selftest_wait_kernel(uint32_t* err_word, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_word;
  if (threadIdx.x == 0) {
    abort_word = 0u;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&abort_word, err_word, timeout_ns};
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, wc);
  __syncthreads();
}

}  // namespace
}  // namespace exattn

extern "C" attn_status attn_selftest_wait_timeout(int timeout_ms, void* stream) {
  if (timeout_ms < 1 || timeout_ms > 10000) return ATTN_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  attn_status st = device_state(&ds);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selftest_wait_kernel<<<1, 32, 0, s>>>(ds->err_word, static_cast<uint64_t>(timeout_ms) * 1000000ull);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail("kernel launch", e);
  return attn_check_device_error(stream);
}

// ----------------------------------------------------------------- attention KL: split-K forward

namespace {

size_t kl_split_workspace(int B, int H, int Nq, int splits) {
  return align256(static_cast<size_t>(5) * splits * B * H * Nq * sizeof(float));
}

}  // namespace

extern "C" size_t attn_kl_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || (d != 64 && d != 128) || num_splits < 0 || num_splits > kMaxSplits)
    return 0;
  if (num_splits == 0) {
    const int sms = device_sm_count();
    num_splits = choose_splits(static_cast<long long>(B) * H, Nq, Nk, sms > 0 ? sms : 1, 1);
    if (num_splits <= 1) return 0;
  }
  return kl_split_workspace(B, H, Nq, num_splits);
}

extern "C" attn_status attn_kl_fwd_splitkv(const void* Q1, const void* K1, const void* Q2, const void* K2, float* KL,
                                           float* LSE1, float* LSE2, int B, int H, int Nq, int Nk, int d, int causal,
                                           float scale, attn_dtype dtype, int num_splits, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  if (num_splits < 0 || num_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  if (!KL || !LSE1 || !LSE2) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(KL) || !aligned16(LSE1) || !aligned16(LSE2)) return ATTN_ERR_MISALIGNED;
  if (num_splits == 0) {
    attn_status st = check_common(B, H, Nq, Nk, d, causal, scale, dtype);
    if (st != ATTN_OK) return st;
    const int sms = device_sm_count();
    num_splits = choose_splits(static_cast<long long>(B) * H, Nq, Nk, sms > 0 ? sms : 1, 1);
    if (num_splits == 1)
      return attn_kl_fwd(Q1, K1, Q2, K2, KL, LSE1, LSE2, B, H, Nq, Nk, d, causal, scale, dtype, stream);
  }
  if (!workspace || workspace_bytes < kl_split_workspace(B, H, Nq, num_splits)) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_MISALIGNED;
  KlArgs a;
  DeviceState* ds = nullptr;
  attn_status st = kl_common(Q1, K1, Q2, K2, B, H, Nq, Nk, d, causal, scale, dtype, &a, &ds);
  if (st != ATTN_OK) return st;
  if (static_cast<long long>(B) * H * Nq > 0x7fffffffLL * 255LL) return ATTN_ERR_INVALID_ARG;
  a.kl = KL;
  a.lse1 = LSE1;
  a.lse2 = LSE2;
  a.part = static_cast<float*>(workspace);
  a.splits = num_splits;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return finish(launch_kl_fwd(a, s), s);
}
