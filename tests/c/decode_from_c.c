/* decode_from_c.c -- the C ABI driven from plain C99 and the CUDA runtime, no Python.
 * Reads a small bf16 problem from a file, writes the step's new K/V with
 * pa_reshape_and_cache, then decodes it four ways and writes the four outputs and the
 * device error flag to a file:
 *   1. pa_decode_splitkv (num_splits slots per head) + pa_merge_lse;
 *   2. pa_decode given a workspace of num_segments segments (split decode + merge);
 *   3. pa_decode without a workspace;
 *   4. pa_merge_lse of partials read from the file (made elsewhere).
 *
 * Input file: int32 B, Hq, Hkv, D, block_size, nblocks, max_blocks, num_splits,
 * num_segments, ext_splits; float sm_scale; then q [B,Hq,D] bf16, k_pool and v_pool
 * [nblocks,block_size,Hkv,D] bf16, k_new and v_new [B,Hkv,D] bf16, block_tables
 * [B,max_blocks] int32, seq_lens [B] int32, slot_mapping [B] int64, and the external
 * partials o_part [B,Hq,ext_splits,D] and lse [B,Hq,ext_splits] fp32.
 * Output file: the four outputs ([B,Hq,D] fp32 each), then the int32 error flag.
 * Exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "pa.h"

#define CHECK_CUDA(x)                                                             \
  do {                                                                            \
    cudaError_t e_ = (x);                                                         \
    if (e_ != cudaSuccess) {                                                      \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                    \
      return 2;                                                                   \
    }                                                                             \
  } while (0)
#define CHECK_PA(x)                                                               \
  do {                                                                            \
    pa_status s_ = (x);                                                           \
    if (s_ != PA_OK) {                                                            \
      fprintf(stderr, "%s: %s\n", #x, pa_status_string(s_));                      \
      return 3;                                                                   \
    }                                                                             \
  } while (0)

/* n bytes from f into a new device buffer (16 bytes at least, so never NULL) */
static int upload(FILE *f, size_t n, void **dev) {
  void *host = malloc(n ? n : 1);
  int ok = host && fread(host, 1, n, f) == n && cudaMalloc(dev, n ? n : 16) == cudaSuccess &&
           cudaMemcpy(*dev, host, n, cudaMemcpyHostToDevice) == cudaSuccess;
  free(host);
  return ok;
}

int main(int argc, char **argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s input output\n", argv[0]);
    return 1;
  }
  FILE *in = fopen(argv[1], "rb");
  if (!in) return 1;
  int32_t h[10];
  float sm_scale;
  if (fread(h, 4, 10, in) != 10 || fread(&sm_scale, 4, 1, in) != 1) return 1;
  pa_shape s;
  s.B = h[0];
  s.Hq = h[1];
  s.Hkv = h[2];
  s.D = h[3];
  s.block_size = h[4];
  s.nblocks = h[5];
  s.max_blocks = h[6];
  s.kv_dtype = PA_KV_BF16;
  const int32_t num_splits = h[7], num_segments = h[8], ext_splits = h[9];
  const size_t nq = (size_t)s.B * s.Hq * s.D, npool = (size_t)s.nblocks * s.block_size * s.Hkv * s.D;
  const size_t nnew = (size_t)s.B * s.Hkv * s.D;
  void *q, *kp, *vp, *kn, *vn, *bt, *sl, *slot, *ext_o, *ext_l;
  if (!upload(in, nq * 2, &q) || !upload(in, npool * 2, &kp) || !upload(in, npool * 2, &vp) ||
      !upload(in, nnew * 2, &kn) || !upload(in, nnew * 2, &vn) ||
      !upload(in, (size_t)s.B * s.max_blocks * 4, &bt) || !upload(in, (size_t)s.B * 4, &sl) ||
      !upload(in, (size_t)s.B * 8, &slot) || !upload(in, nq * ext_splits * 4, &ext_o) ||
      !upload(in, (size_t)s.B * s.Hq * ext_splits * 4, &ext_l))
    return 1;
  fclose(in);

  float *out[4], *o_part, *lse;
  int32_t *err;
  void *ws;
  const size_t parts_bytes = pa_splitkv_workspace_bytes(&s, num_splits);
  const size_t ws_bytes = pa_decode_workspace_bytes(&s, num_segments);
  if (parts_bytes == 0 || ws_bytes == 0) return 3;
  for (int i = 0; i < 4; ++i) CHECK_CUDA(cudaMalloc((void **)&out[i], nq * 4));
  /* o_part and lse carved from one allocation, o_part first */
  CHECK_CUDA(cudaMalloc((void **)&o_part, parts_bytes));
  lse = o_part + nq * num_splits;
  CHECK_CUDA(cudaMalloc((void **)&err, 4));
  CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_CUDA(cudaMemset(err, 0, 4));

  CHECK_PA(pa_reshape_and_cache(&s, kn, vn, kp, vp, NULL, NULL, (const int64_t *)slot, err, NULL));
  CHECK_PA(pa_decode_splitkv(&s, o_part, lse, num_splits, q, kp, vp, NULL, NULL,
                             (const int32_t *)bt, (const int32_t *)sl, NULL, sm_scale, err, NULL));
  CHECK_PA(pa_merge_lse(&s, out[0], o_part, lse, num_splits, NULL));
  pa_decode_opts opts = {0};
  opts.workspace = ws;
  opts.workspace_bytes = ws_bytes;
  opts.num_segments = num_segments;
  CHECK_PA(pa_decode(&s, out[1], q, kp, vp, NULL, NULL, (const int32_t *)bt, (const int32_t *)sl,
                     &opts, sm_scale, err, NULL));
  CHECK_PA(pa_decode(&s, out[2], q, kp, vp, NULL, NULL, (const int32_t *)bt, (const int32_t *)sl,
                     NULL, sm_scale, err, NULL));
  CHECK_PA(pa_merge_lse(&s, out[3], (const float *)ext_o, (const float *)ext_l, ext_splits, NULL));
  CHECK_CUDA(cudaDeviceSynchronize());
  int32_t err_host = -1;
  CHECK_PA(pa_read_error_flag(err, &err_host, NULL));

  float *host = (float *)malloc(nq * 4 * 4);
  if (!host) return 1;
  for (int i = 0; i < 4; ++i)
    CHECK_CUDA(cudaMemcpy(host + nq * i, out[i], nq * 4, cudaMemcpyDeviceToHost));
  FILE *fo = fopen(argv[2], "wb");
  if (!fo || fwrite(host, 4, nq * 4, fo) != nq * 4 || fwrite(&err_host, 4, 1, fo) != 1) return 1;
  fclose(fo);
  free(host);
  return 0;
}
