/*
 * One paged decode step through the C ABI alone, no Python: plan
 * (paged_decode_plan), run (paged_decode_run) on device buffers, read the
 * device status word (paged_decode_plan_check).  The inputs are uniform
 * random values drawn here; the inputs and the outputs are written under
 * <out dir> as raw little-endian arrays, for tests/test_c_abi_gpu.py to
 * compare with the fp64 oracle.
 *
 * usage: decode_step <out dir> <num_qo_heads> [mma_min_rows]
 *   3 requests of 37, 100 and 300 keys, 2 KV heads, head_dim 128, 16-token
 *   pages drawn from a pool of 48 in a random order, one query row each, LSE.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "pka.h"

#define CHECK_CUDA(x)                                                        \
  do {                                                                       \
    cudaError_t e_ = (x);                                                    \
    if (e_ != cudaSuccess) {                                                 \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));              \
      return 1;                                                              \
    }                                                                        \
  } while (0)
#define CHECK_PKA(x)                                                         \
  do {                                                                       \
    int r_ = (x);                                                            \
    if (r_ != PKA_OK) {                                                      \
      fprintf(stderr, "%s: %d %s\n", #x, r_, pka_last_error());             \
      return 1;                                                              \
    }                                                                        \
  } while (0)

/* xorshift64* */
static uint64_t rng = 0x2545F4914F6CDD1Dull;
static uint32_t next_u32(void) {
  rng ^= rng >> 12;
  rng ^= rng << 25;
  rng ^= rng >> 27;
  return (uint32_t)((rng * 2685821657736338717ull) >> 32);
}
static float next_unit(void) { return (float)next_u32() * (2.0f / 4294967296.0f) - 1.0f; }

/* float -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static int save(const char* dir, const char* name, const void* p, size_t n) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  const size_t w = fwrite(p, 1, n, f);
  fclose(f);
  return w != n;
}

int main(int argc, char** argv) {
  if (argc != 3 && argc != 4) {
    fprintf(stderr, "usage: %s <out dir> <num_qo_heads> [mma_min_rows]\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  const int B = 3, Hq = atoi(argv[2]), Hkv = 2, D = 128, ps = 16, C = 19, P = 48;
  const int32_t lens[3] = {37, 100, 300};
  if (Hq < Hkv || Hq % Hkv != 0) return 2;

  const size_t nq = (size_t)B * Hq * D, npool = (size_t)P * Hkv * ps * D, nt = (size_t)B * C;
  uint16_t* q = malloc(nq * 2);
  uint16_t* k = malloc(npool * 2);
  uint16_t* v = malloc(npool * 2);
  int32_t* tables = malloc(nt * 4);
  int32_t perm[48];
  uint16_t* out = malloc(nq * 2);
  float* lse = malloc((size_t)B * Hq * 4);
  if (!q || !k || !v || !tables || !out || !lse) return 1;
  for (size_t i = 0; i < nq; ++i) q[i] = to_bf16(next_unit());
  for (size_t i = 0; i < npool; ++i) k[i] = to_bf16(next_unit());
  for (size_t i = 0; i < npool; ++i) v[i] = to_bf16(next_unit());
  for (int i = 0; i < P; ++i) perm[i] = i;
  for (int i = P - 1; i > 0; --i) {   /* Fisher-Yates */
    const int j = (int)(next_u32() % (uint32_t)(i + 1));
    const int t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  int used = 0;
  for (int b = 0; b < B; ++b)
    for (int c = 0; c < C; ++c)
      tables[b * C + c] = c < (lens[b] + ps - 1) / ps ? perm[used++] : -1;   /* -1: never read */

  void *q_d, *k_d, *v_d, *out_d;
  int32_t* bt_d;
  float* lse_d;
  CHECK_CUDA(cudaMalloc(&q_d, nq * 2));
  CHECK_CUDA(cudaMalloc(&k_d, npool * 2));
  CHECK_CUDA(cudaMalloc(&v_d, npool * 2));
  CHECK_CUDA(cudaMalloc((void**)&bt_d, nt * 4));
  CHECK_CUDA(cudaMalloc(&out_d, nq * 2));
  CHECK_CUDA(cudaMalloc((void**)&lse_d, (size_t)B * Hq * 4));
  CHECK_CUDA(cudaMemcpy(q_d, q, nq * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(k_d, k, npool * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(v_d, v, npool * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(bt_d, tables, nt * 4, cudaMemcpyHostToDevice));

  pka_decode_desc d;
  memset(&d, 0, sizeof d);
  d.batch_size = B;
  d.num_qo_heads = Hq;
  d.num_kv_heads = Hkv;
  d.head_dim = D;
  d.page_size = ps;
  d.max_pages_per_seq = C;
  d.num_pages = P;
  d.dtype = PKA_DTYPE_BF16;
  d.q_len = 1;
  d.mask = PKA_MASK_DENSE;
  d.window_left = -1;
  d.scale = NAN;   /* 1 / sqrt(head_dim) */
  d.bmm2_scale = 1.0f;
  d.return_lse = 1;
  d.freeze_seq_lens = 1;
  d.out_dtype = PKA_DTYPE_BF16;
  d.mma_min_rows = argc == 4 ? atoi(argv[3]) : 0;   /* 0: the library's default */

  pka_plan* plan = NULL;
  size_t ws_bytes = 0;
  CHECK_PKA(paged_decode_plan(&plan, &d, lens, NULL, &ws_bytes, NULL));
  void* ws = NULL;
  if (ws_bytes > 0) CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
  CHECK_PKA(paged_decode_run(plan, q_d, (int64_t)Hq * D, D, k_d, v_d, (int64_t)Hkv * ps * D,
                             (int64_t)ps * D, bt_d, C, NULL, NULL, out_d, lse_d, ws, ws_bytes,
                             NULL));
  CHECK_PKA(paged_decode_plan_check(plan, NULL));
  pka_plan_info info;
  CHECK_PKA(paged_decode_plan_info(plan, &info));
  CHECK_CUDA(cudaMemcpy(out, out_d, nq * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(lse, lse_d, (size_t)B * Hq * 4, cudaMemcpyDeviceToHost));

  int bad = save(dir, "q.bin", q, nq * 2) || save(dir, "k.bin", k, npool * 2) ||
            save(dir, "v.bin", v, npool * 2) || save(dir, "tables.bin", tables, nt * 4) ||
            save(dir, "lens.bin", lens, sizeof lens) || save(dir, "out.bin", out, nq * 2) ||
            save(dir, "lse.bin", lse, (size_t)B * Hq * 4);
  if (bad) return 1;
  printf("B=%d Hq=%d Hkv=%d D=%d ps=%d C=%d P=%d kernel=%d num_split=%d\n", B, Hq, Hkv, D, ps,
         C, P, info.kernel, info.num_split);

  paged_decode_plan_destroy(plan);
  cudaFree(ws);
  cudaFree(q_d);
  cudaFree(k_d);
  cudaFree(v_d);
  cudaFree(bt_d);
  cudaFree(out_d);
  cudaFree(lse_d);
  free(q);
  free(k);
  free(v);
  free(tables);
  free(out);
  free(lse);
  return 0;
}
