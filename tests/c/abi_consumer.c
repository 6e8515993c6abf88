/*
 * A plain C consumer of libdiffattn.so: no PyTorch, no C++, only the C ABI in
 * diffattn.h and the CUDA runtime for device memory.  It reads seeded inputs
 * from a file, runs lambda_reparam, the bf16 forward and the bf16 decode step
 * on the device, reads the device status word, and writes the results to a
 * second file for the test that compares them with the oracle.
 *
 * Input file (little-endian): int32 B, H, n, d, n_cache, causal; float
 * lambda_init; then bf16 (raw 16-bit) q1, q2, k1, k2 [B, n, H, d], v
 * [B, n, H, 2d]; float lq1, lk1, lq2, lk2 [d], gamma [2d]; bf16 decode
 * queries q1, q2 [B, H, d], caches k1, k2 [B, n_cache, H, d], v
 * [B, n_cache, H, 2d]; int32 lens [B].
 * Output file: float lambda; bf16 out [B, n, H, 2d]; bf16 decode out [B, H, 2d].
 * Usage: abi_consumer IN OUT
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "diffattn.h"

#define CK(x)                                                                   \
  do {                                                                          \
    cudaError_t e_ = (x);                                                       \
    if (e_ != cudaSuccess) {                                                    \
      fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));           \
      return 2;                                                                 \
    }                                                                           \
  } while (0)
#define DA(x)                                                                   \
  do {                                                                          \
    diffattn_status s_ = (x);                                                   \
    if (s_ != DIFFATTN_OK) {                                                    \
      fprintf(stderr, "%s returned %d: %s\n", #x, (int)s_, diffattn_last_error()); \
      return 3;                                                                 \
    }                                                                           \
  } while (0)

/* Reads `bytes` from the input buffer into a new device allocation. */
static int to_device(const unsigned char** cur, const unsigned char* end, size_t bytes, void** dev) {
  if ((size_t)(end - *cur) < bytes) {
    fprintf(stderr, "input file too short\n");
    return 1;
  }
  CK(cudaMalloc(dev, bytes > 0 ? bytes : 1));
  CK(cudaMemcpy(*dev, *cur, bytes, cudaMemcpyHostToDevice));
  *cur += bytes;
  return 0;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s IN OUT\n", argv[0]);
    return 1;
  }
  FILE* f = fopen(argv[1], "rb");
  if (!f) {
    perror(argv[1]);
    return 1;
  }
  fseek(f, 0, SEEK_END);
  const long size = ftell(f);
  fseek(f, 0, SEEK_SET);
  unsigned char* buf = (unsigned char*)malloc((size_t)size);
  if (!buf || fread(buf, 1, (size_t)size, f) != (size_t)size) {
    fprintf(stderr, "cannot read %s\n", argv[1]);
    return 1;
  }
  fclose(f);
  const unsigned char* cur = buf;
  const unsigned char* end = buf + size;

  int32_t hdr[6];
  float lambda_init;
  memcpy(hdr, cur, sizeof(hdr));
  cur += sizeof(hdr);
  memcpy(&lambda_init, cur, sizeof(float));
  cur += sizeof(float);
  const int B = hdr[0], H = hdr[1], n = hdr[2], d = hdr[3], nc = hdr[4], causal = hdr[5];
  const size_t qk = (size_t)B * n * H * d * 2, vo = 2 * qk;
  const size_t dq = (size_t)B * H * d * 2, dk = (size_t)B * nc * H * d * 2, dvb = 2 * dk;

  void *q1, *q2, *k1, *k2, *v, *lq1, *lk1, *lq2, *lk2, *gamma;
  void *tq1, *tq2, *tk1, *tk2, *tv, *lens;
  int rc = 0;
  rc |= to_device(&cur, end, qk, &q1);
  rc |= to_device(&cur, end, qk, &q2);
  rc |= to_device(&cur, end, qk, &k1);
  rc |= to_device(&cur, end, qk, &k2);
  rc |= to_device(&cur, end, vo, &v);
  rc |= to_device(&cur, end, (size_t)d * 4, &lq1);
  rc |= to_device(&cur, end, (size_t)d * 4, &lk1);
  rc |= to_device(&cur, end, (size_t)d * 4, &lq2);
  rc |= to_device(&cur, end, (size_t)d * 4, &lk2);
  rc |= to_device(&cur, end, (size_t)2 * d * 4, &gamma);
  rc |= to_device(&cur, end, dq, &tq1);
  rc |= to_device(&cur, end, dq, &tq2);
  rc |= to_device(&cur, end, dk, &tk1);
  rc |= to_device(&cur, end, dk, &tk2);
  rc |= to_device(&cur, end, dvb, &tv);
  rc |= to_device(&cur, end, (size_t)B * 4, &lens);
  if (rc) return rc;

  void *lambda, *out, *dec_out;
  CK(cudaMalloc(&lambda, sizeof(float)));
  CK(cudaMalloc(&out, vo));
  CK(cudaMalloc(&dec_out, (size_t)B * H * 2 * d * 2));
  cudaStream_t s;
  CK(cudaStreamCreate(&s));

  /* lambda on the device, then the forward and the decode step that read it, all on one stream */
  DA(lambda_reparam((const float*)lq1, (const float*)lk1, (const float*)lq2, (const float*)lk2, d, lambda_init,
                    (float*)lambda, s));
  DA(diffattn_forward(DIFFATTN_BF16, B, H, n, d, q1, q2, k1, k2, v, (const float*)lambda, lambda_init,
                      (const float*)gamma, 1e-5f, causal, out, s));
  DA(diffattn_decode(DIFFATTN_BF16, B, H, nc, d, tq1, tq2, tk1, tk2, tv, (const int*)lens, (const float*)lambda,
                     lambda_init, (const float*)gamma, 1e-5f, dec_out, NULL, 0, s));
  DA(diffattn_device_status(s));

  const size_t obytes = sizeof(float) + vo + (size_t)B * H * 2 * d * 2;
  unsigned char* res = (unsigned char*)malloc(obytes);
  if (!res) return 1;
  CK(cudaMemcpy(res, lambda, sizeof(float), cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(res + sizeof(float), out, vo, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(res + sizeof(float) + vo, dec_out, (size_t)B * H * 2 * d * 2, cudaMemcpyDeviceToHost));
  FILE* o = fopen(argv[2], "wb");
  if (!o || fwrite(res, 1, obytes, o) != obytes) {
    fprintf(stderr, "cannot write %s\n", argv[2]);
    return 1;
  }
  fclose(o);
  printf("ok: B=%d H=%d n=%d d=%d n_cache=%d\n", B, H, n, d, nc);
  return 0;
}
