/*
 * A plain C program that uses libnormrope through include/nr.h alone: device
 * buffers from the CUDA runtime, one stream, no Python and no torch in the
 * process.  Test infrastructure: tests/test_c_consumer.py compiles it, writes
 * the seeded inputs as raw files, runs it and checks the files it writes
 * against the oracle.
 *
 * usage: nr_consumer <dir> <rows> <hidden> <tokens> <hq> <hk> <head_dim>
 *                    <ln_rows> <ln_hidden> <act_rows> <inter>
 *   add + RMSNorm (bf16, gemma):  x.bin, res.bin, w.bin   -> rms_out.bin, rms_res.bin
 *   Q/K norm + RoPE (bf16, f32 weights, in place on q):
 *                                 q.bin, k.bin, wq.bin, wk.bin, pos.bin -> q_out.bin, k_out.bin
 *   LN + modulation (bf16):       lx.bin, shift.bin, scale.bin -> ln_out.bin
 *   silu_and_mul (bf16):          ax.bin                 -> silu_out.bin
 * Exit status 0 when every call returned the expected status.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "nr.h"

static int failures = 0;

static void expect(const char* what, nr_status got, nr_status want) {
  if (got != want) {
    fprintf(stderr, "%s: got %s (%s), want %s\n", what, nr_status_string(got),
            nr_last_error_message(), nr_status_string(want));
    failures++;
  }
}

static void cuda_ok(const char* what, cudaError_t e) {
  if (e != cudaSuccess) {
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    exit(2);
  }
}

/* Read <dir>/<name> (exactly `bytes` bytes) into a new device buffer. */
static void* upload(const char* dir, const char* name, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (f == NULL) {
    fprintf(stderr, "cannot open %s\n", path);
    exit(2);
  }
  void* host = malloc(bytes);
  if (host == NULL || fread(host, 1, bytes, f) != bytes) {
    fprintf(stderr, "short read: %s\n", path);
    exit(2);
  }
  fclose(f);
  void* dev = NULL;
  cuda_ok("cudaMalloc", cudaMalloc(&dev, bytes));
  cuda_ok("cudaMemcpy H2D", cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice));
  free(host);
  return dev;
}

static void* device_buffer(size_t bytes) {
  void* dev = NULL;
  cuda_ok("cudaMalloc", cudaMalloc(&dev, bytes));
  return dev;
}

/* Copy `bytes` of a device buffer to <dir>/<name>. */
static void download(const char* dir, const char* name, const void* dev, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  void* host = malloc(bytes);
  if (host == NULL) exit(2);
  cuda_ok("cudaMemcpy D2H", cudaMemcpy(host, dev, bytes, cudaMemcpyDeviceToHost));
  FILE* f = fopen(path, "wb");
  if (f == NULL || fwrite(host, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot write %s\n", path);
    exit(2);
  }
  fclose(f);
  free(host);
}

int main(int argc, char** argv) {
  if (argc != 12) {
    fprintf(stderr, "usage: %s dir rows hidden tokens hq hk head_dim ln_rows ln_hidden "
                    "act_rows inter\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  const int64_t rows = atoll(argv[2]), hidden = atoll(argv[3]);
  const int64_t tokens = atoll(argv[4]), hq = atoll(argv[5]), hk = atoll(argv[6]);
  const int64_t D = atoll(argv[7]);
  const int64_t ln_rows = atoll(argv[8]), ln_hidden = atoll(argv[9]);
  const int64_t act_rows = atoll(argv[10]), inter = atoll(argv[11]);
  const size_t b2 = 2; /* bytes per bf16 */

  cudaStream_t stream;
  cuda_ok("cudaStreamCreate", cudaStreamCreate(&stream));
  if (nr_version() <= 0) failures++;

  /* add + RMSNorm, residual in place, gemma */
  void* x = upload(dir, "x.bin", rows * hidden * b2);
  void* res = upload(dir, "res.bin", rows * hidden * b2);
  void* w = upload(dir, "w.bin", hidden * b2);
  void* out = device_buffer(rows * hidden * b2);
  expect("nr_rmsnorm", nr_rmsnorm(out, x, w, res, rows, hidden, NR_BF16, 1e-6f, 1, stream), NR_OK);

  /* Q/K: q in place, k out of place */
  const size_t qb = tokens * hq * D * b2, kb = tokens * hk * D * b2;
  void* q = upload(dir, "q.bin", qb);
  void* k = upload(dir, "k.bin", kb);
  void* wq = upload(dir, "wq.bin", D * 4);
  void* wk = upload(dir, "wk.bin", D * 4);
  void* pos = upload(dir, "pos.bin", tokens * 4);
  void* k_out = device_buffer(kb);
  expect("nr_qk_norm_rope",
         nr_qk_norm_rope(q, k_out, q, k, wq, wk, NR_F32, (const int32_t*)pos, tokens, hq, hk, D,
                         hq * D, hk * D, 1e-6f, 10000.0, 0, NR_BF16, stream),
         NR_OK);

  /* LayerNorm + modulation, one sample */
  void* lx = upload(dir, "lx.bin", ln_rows * ln_hidden * b2);
  void* shift = upload(dir, "shift.bin", ln_hidden * b2);
  void* scale = upload(dir, "scale.bin", ln_hidden * b2);
  void* ln_out = device_buffer(ln_rows * ln_hidden * b2);
  expect("nr_ln_modulate",
         nr_ln_modulate(ln_out, lx, shift, scale, ln_rows, ln_hidden, ln_rows, 1e-6f, NR_BF16,
                        stream),
         NR_OK);

  /* silu_and_mul */
  void* ax = upload(dir, "ax.bin", act_rows * 2 * inter * b2);
  void* silu_out = device_buffer(act_rows * inter * b2);
  expect("nr_silu_and_mul", nr_silu_and_mul(silu_out, ax, act_rows, inter, NR_BF16, stream), NR_OK);

  /* host-side refusals: nothing is launched for these */
  expect("null x", nr_rmsnorm(out, NULL, w, NULL, rows, hidden, NR_BF16, 1e-6f, 0, stream),
         NR_ERR_NULL);
  expect("out aliases the residual",
         nr_rmsnorm(res, x, w, res, rows, hidden, NR_BF16, 1e-6f, 0, stream), NR_ERR_ALIAS);
  expect("hidden not a multiple of 8",
         nr_rmsnorm(out, x, w, NULL, rows, 4, NR_BF16, 1e-6f, 0, stream), NR_ERR_UNSUPPORTED);
  expect("zero rows", nr_rmsnorm(out, x, w, NULL, 0, hidden, NR_BF16, 1e-6f, 0, stream), NR_OK);

  expect("nr_device_status", nr_device_status(stream), NR_OK);
  cuda_ok("cudaStreamSynchronize", cudaStreamSynchronize(stream));

  download(dir, "rms_out.bin", out, rows * hidden * b2);
  download(dir, "rms_res.bin", res, rows * hidden * b2);
  download(dir, "q_out.bin", q, qb);
  download(dir, "k_out.bin", k_out, kb);
  download(dir, "ln_out.bin", ln_out, ln_rows * ln_hidden * b2);
  download(dir, "silu_out.bin", silu_out, act_rows * inter * b2);

  void* bufs[] = {x, res, w, out, q, k, wq, wk, pos, k_out, lx, shift, scale, ln_out, ax,
                  silu_out};
  for (size_t i = 0; i < sizeof bufs / sizeof bufs[0]; i++) cudaFree(bufs[i]);
  cudaStreamDestroy(stream);
  printf("nr_consumer: %d failure(s)\n", failures);
  return failures == 0 ? 0 : 1;
}
