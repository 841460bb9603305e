/*
 * A plain C99 caller of the exattn C ABI (include/exattn.h), built and run by
 * tests/test_c_abi.py.  It uses nothing but the header, the shared library
 * and, in the GPU mode, the CUDA runtime for device memory.
 *
 *   consumer cpu                 argument validation and the host-side helpers;
 *                                needs no GPU (fake device pointers are never
 *                                dereferenced: validation happens first)
 *   consumer gpu IN OUT          (built with -DWITH_CUDART) reads a problem from
 *                                IN, runs attn_fwd then attn_bwd on the GPU
 *                                and writes O, LSE, dQ, dK, dV to OUT
 *
 * IN: int32 B, H, Nq, Nk, d, causal, dtype; float32 scale; then Q [B,H,Nq,d],
 * K, V [B,H,Nk,d] and dO [B,H,Nq,d] as raw 16-bit values.
 * OUT: O (16-bit), LSE (fp32 [B,H,Nq]), dQ, dK, dV (16-bit), in that order.
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "exattn.h"

#ifdef WITH_CUDART
#include <cuda_runtime_api.h>
#endif

static int failures = 0;

#define EXPECT(cond, what)                                          \
  do {                                                              \
    if (!(cond)) {                                                  \
      fprintf(stderr, "FAILED: %s (line %d)\n", what, __LINE__);    \
      ++failures;                                                   \
    }                                                               \
  } while (0)

static int cpu_checks(void) {
  /* fake device pointers: 16-byte aligned, never dereferenced */
  void* p = (void*)(uintptr_t)0x10000;
  void* odd = (void*)(uintptr_t)0x10008;
  float* lse = (float*)p;
  const size_t ws = attn_bwd_workspace_size(1, 12, 8192, 128);
  int code;
  uint32_t blocks[2048];
  int begin[257];
  int n, i, j;
  unsigned char seen[384];

  EXPECT(ws == (size_t)12 * 8192 * 128 * 4 + (size_t)2 * 12 * 8192 * 4, "attn_bwd_workspace_size of 1x12x8192, d=128");
  EXPECT(attn_bwd_workspace_size(1, 1, 1, 96) == 0, "attn_bwd_workspace_size rejects d=96");

  for (code = 0; code <= 7; ++code) {
    const char* s = attn_status_string((attn_status)code);
    EXPECT(s != NULL && s[0] != '\0', "attn_status_string names every status");
  }
  EXPECT(strcmp(attn_status_string((attn_status)99), "unknown status") == 0, "attn_status_string of an unknown code");

  EXPECT(attn_fwd(p, p, p, p, lse, 0, 1, 128, 128, 64, ATTN_MASK_NONE, 0.125f, ATTN_BF16, NULL) == ATTN_ERR_INVALID_ARG,
         "attn_fwd rejects B = 0");
  EXPECT(attn_fwd(p, p, p, p, lse, 1, 1, 128, 128, 96, ATTN_MASK_NONE, 0.125f, ATTN_BF16, NULL) == ATTN_ERR_UNSUPPORTED,
         "attn_fwd rejects d = 96");
  EXPECT(attn_fwd(p, p, odd, p, lse, 1, 1, 128, 128, 64, ATTN_MASK_CAUSAL, 0.125f, ATTN_FP16, NULL) == ATTN_ERR_MISALIGNED,
         "attn_fwd rejects a misaligned V");
  EXPECT(attn_fwd(p, NULL, p, p, lse, 1, 1, 128, 128, 64, ATTN_MASK_NONE, 0.125f, ATTN_BF16, NULL) == ATTN_ERR_INVALID_ARG,
         "attn_fwd rejects a null K");
  EXPECT(attn_fwd(p, p, p, p, lse, 1, 1, 128, 128, 64, 3, 0.125f, ATTN_BF16, NULL) == ATTN_ERR_INVALID_ARG,
         "attn_fwd rejects an unknown mask");
  EXPECT(attn_last_error() != NULL, "attn_last_error is never NULL");

  EXPECT(attn_bwd(p, p, p, p, p, lse, p, p, p, 1, 1, 128, 128, 64, ATTN_MASK_NONE, 0.125f, ATTN_BF16, NULL, 0, NULL) ==
             ATTN_ERR_WORKSPACE,
         "attn_bwd rejects a missing workspace");
  EXPECT(attn_bwd(p, p, p, p, p, lse, p, p, p, 1, 1, 128, 128, 64, ATTN_MASK_NONE, -1.0f, ATTN_BF16, p,
                  attn_bwd_workspace_size(1, 1, 128, 64), NULL) == ATTN_ERR_INVALID_ARG,
         "attn_bwd rejects a negative scale");
  EXPECT(attn_bwd_ex(p, p, p, p, p, lse, p, p, p, 1, 1, 128, 128, 64, ATTN_MASK_NONE, 0.125f, ATTN_BF16, 9, p,
                     attn_bwd_workspace_size(1, 1, 128, 64), NULL) == ATTN_ERR_INVALID_ARG,
         "attn_bwd_ex rejects an unknown dQ mode");

  EXPECT(attn_bwd_auto_dq_mode(1, 12, 8192, 8192, 128, ATTN_MASK_CAUSAL) == ATTN_DQ_ATOMIC, "attn_bwd_auto_dq_mode");
  EXPECT(attn_bwd_head_group(1, 12, 8192, 8192, 128, ATTN_MASK_CAUSAL, 152, (size_t)126 << 20) == 12,
         "attn_bwd_head_group keeps 12 heads together when the accumulator fits");

  /* the 8k causal forward on 152 SMs runs from packed lists: every 256-row block on exactly one list */
  n = attn_fwd_schedule(1, 12, 8192, 8192, 128, ATTN_MASK_CAUSAL, 152, blocks, 2048, begin, 257);
  EXPECT(n > 0 && n <= 152, "attn_fwd_schedule packs the 8k causal forward");
  if (n > 0) {
    memset(seen, 0, sizeof(seen));
    EXPECT(begin[0] == 0 && begin[n] == 12 * 32, "attn_fwd_schedule lists 384 blocks");
    for (i = 0; i < n; ++i)
      for (j = begin[i]; j < begin[i + 1]; ++j)
        if (blocks[j] < 384) ++seen[blocks[j]];
    for (i = 0; i < 384; ++i) EXPECT(seen[i] == 1, "every block on exactly one list");
  }
  EXPECT(attn_fwd_schedule(1, 12, 8192, 8192, 128, ATTN_MASK_NONE, 152, blocks, 2048, begin, 257) == 0,
         "no lists without a mask");
  return failures;
}

#ifdef WITH_CUDART
static size_t read_exact(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes ? bytes : 0; }

static int gpu_run(const char* in_path, const char* out_path) {
  int32_t hdr[7];
  float scale;
  FILE* f = fopen(in_path, "rb");
  size_t nq, nk, nl, ws_bytes;
  void *hq, *hk, *hv, *hdo, *ho, *hdq, *hdk, *hdv;
  float* hlse;
  void *q, *k, *v, *dout, *o, *dq, *dk, *dv, *ws;
  float* lse;
  attn_status st;
  if (!f) {
    fprintf(stderr, "cannot open %s\n", in_path);
    return 2;
  }
  if (!read_exact(f, hdr, sizeof(hdr)) || !read_exact(f, &scale, sizeof(scale))) {
    fprintf(stderr, "short header\n");
    fclose(f);
    return 2;
  }
  nq = (size_t)hdr[0] * hdr[1] * hdr[2] * hdr[4] * 2; /* bytes of a [B,H,Nq,d] 16-bit tensor */
  nk = (size_t)hdr[0] * hdr[1] * hdr[3] * hdr[4] * 2;
  nl = (size_t)hdr[0] * hdr[1] * hdr[2] * 4;
  hq = malloc(nq), hk = malloc(nk), hv = malloc(nk), hdo = malloc(nq);
  ho = malloc(nq), hdq = malloc(nq), hdk = malloc(nk), hdv = malloc(nk);
  hlse = (float*)malloc(nl);
  if (!hq || !hk || !hv || !hdo || !ho || !hdq || !hdk || !hdv || !hlse) return 2;
  if (!read_exact(f, hq, nq) || !read_exact(f, hk, nk) || !read_exact(f, hv, nk) || !read_exact(f, hdo, nq)) {
    fprintf(stderr, "short input\n");
    fclose(f);
    return 2;
  }
  fclose(f);

  ws_bytes = attn_bwd_workspace_size(hdr[0], hdr[1], hdr[2], hdr[4]);
  if (cudaMalloc(&q, nq) || cudaMalloc(&k, nk) || cudaMalloc(&v, nk) || cudaMalloc(&dout, nq) ||
      cudaMalloc(&o, nq) || cudaMalloc(&dq, nq) || cudaMalloc(&dk, nk) || cudaMalloc(&dv, nk) ||
      cudaMalloc((void**)&lse, nl) || cudaMalloc(&ws, ws_bytes)) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 3;
  }
  cudaMemcpy(q, hq, nq, cudaMemcpyHostToDevice);
  cudaMemcpy(k, hk, nk, cudaMemcpyHostToDevice);
  cudaMemcpy(v, hv, nk, cudaMemcpyHostToDevice);
  cudaMemcpy(dout, hdo, nq, cudaMemcpyHostToDevice);

  st = attn_fwd(q, k, v, o, lse, hdr[0], hdr[1], hdr[2], hdr[3], hdr[4], hdr[5], scale, (attn_dtype)hdr[6], NULL);
  if (st != ATTN_OK) {
    fprintf(stderr, "attn_fwd: %s (%s)\n", attn_status_string(st), attn_last_error());
    return 4;
  }
  st = attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, hdr[0], hdr[1], hdr[2], hdr[3], hdr[4], hdr[5], scale,
                (attn_dtype)hdr[6], ws, ws_bytes, NULL);
  if (st != ATTN_OK) {
    fprintf(stderr, "attn_bwd: %s (%s)\n", attn_status_string(st), attn_last_error());
    return 4;
  }
  st = attn_check_device_error(NULL);
  if (st != ATTN_OK) {
    fprintf(stderr, "attn_check_device_error: %s\n", attn_status_string(st));
    return 4;
  }
  if (cudaMemcpy(ho, o, nq, cudaMemcpyDeviceToHost) || cudaMemcpy(hlse, lse, nl, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(hdq, dq, nq, cudaMemcpyDeviceToHost) || cudaMemcpy(hdk, dk, nk, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(hdv, dv, nk, cudaMemcpyDeviceToHost)) {
    fprintf(stderr, "cudaMemcpy back failed\n");
    return 3;
  }
  f = fopen(out_path, "wb");
  if (!f) return 2;
  fwrite(ho, 1, nq, f);
  fwrite(hlse, 1, nl, f);
  fwrite(hdq, 1, nq, f);
  fwrite(hdk, 1, nk, f);
  fwrite(hdv, 1, nk, f);
  fclose(f);
  cudaFree(q), cudaFree(k), cudaFree(v), cudaFree(dout), cudaFree(o);
  cudaFree(dq), cudaFree(dk), cudaFree(dv), cudaFree(lse), cudaFree(ws);
  free(hq), free(hk), free(hv), free(hdo), free(ho), free(hdq), free(hdk), free(hdv), free(hlse);
  return 0;
}
#endif

int main(int argc, char** argv) {
  if (argc >= 2 && strcmp(argv[1], "cpu") == 0) {
    int bad = cpu_checks();
    if (bad) return 1;
    printf("ok\n");
    return 0;
  }
#ifdef WITH_CUDART
  if (argc >= 4 && strcmp(argv[1], "gpu") == 0) return gpu_run(argv[2], argv[3]);
#endif
  fprintf(stderr, "usage: consumer cpu | consumer gpu IN OUT\n");
  return 2;
}
