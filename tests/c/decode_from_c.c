/* pa_cache_append + pa_decode driven from plain C (C11) with the CUDA runtime only (no
 * torch): device buffers from cudaMalloc, descriptors filled by hand.  Checked against
 * closed forms of softmax attention ("Solving the LLM Memory Wall", "1. The
 * Mathematical Foundation"): a one-token context returns that token's value row, and
 * tokens with equal keys get equal weights, so the output is the mean of their value
 * rows.  Values are small multiples of 1/4, so every expected element is exact in fp16.
 * Exit status 0 = every element as expected and no device status bit set. */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "pa.h"

enum { NB = 4, B = 16, H = 2, D = 128, S = 2 };

/* fp16 bits of small multiples of 1/4 (|x| < 2048): exact */
static uint16_t h16(float x) {
  uint32_t f;
  uint16_t sign, exp16, man16;
  int e;
  memcpy(&f, &x, 4);
  sign = (uint16_t)((f >> 16) & 0x8000u);
  if ((f & 0x7fffffffu) == 0) return sign;
  e = (int)((f >> 23) & 0xff) - 127 + 15;
  exp16 = (uint16_t)(e << 10);
  man16 = (uint16_t)((f >> 13) & 0x3ffu);
  return (uint16_t)(sign | exp16 | man16);
}

static pa_tensor desc(void* p, int32_t dtype, int ndim, const int64_t* shape) {
  pa_tensor t;
  int i;
  int64_t st = 1;
  memset(&t, 0, sizeof(t));
  t.data = p;
  t.dtype = dtype;
  t.ndim = ndim;
  for (i = ndim - 1; i >= 0; --i) {
    t.shape[i] = shape[i];
    t.stride[i] = st;
    st *= shape[i];
  }
  return t;
}

#define CU(x)                                                     \
  do {                                                            \
    if ((x) != cudaSuccess) {                                     \
      printf("cuda error at %s\n", #x);                           \
      return 1;                                                   \
    }                                                             \
  } while (0)
#define PA(x)                                                     \
  do {                                                            \
    int rc_ = (x);                                                \
    if (rc_ < 0) {                                                \
      printf("error %d (%s) at %s\n", rc_, pa_strerror(rc_), #x); \
      return 1;                                                   \
    }                                                             \
  } while (0)

int main(void) {
  static uint16_t k_rows[4][H][D], v_rows[4][H][D], q[S][H][D], out[S][H][D];
  /* sequence 0: one token in frame 2 (slot 32); sequence 1: three tokens in frame 1 */
  const int32_t slots[4] = {32, 16, 17, 18};
  const int32_t tables[S][2] = {{2, -1}, {1, -1}};
  const int32_t lens[S] = {1, 3};
  const int64_t cache_shape[4] = {NB, B, H, D}, rows_shape[3] = {4, H, D}, q_shape[3] = {S, H, D};
  const int64_t slot_shape[1] = {4}, table_shape[2] = {S, 2}, len_shape[1] = {S};
  void *kc, *vc, *kn, *vn, *sl, *qd, *od, *td, *ld;
  pa_tensor tkc, tvc, tkn, tvn, tsl, tq, tout, ttab, tlen;
  int r, h, d, s, bad = 0;
  int32_t status = 0;

  for (r = 0; r < 4; ++r)
    for (h = 0; h < H; ++h)
      for (d = 0; d < D; ++d) {
        k_rows[r][h][d] = h16(r == 0 ? 0.25f * (float)((d % 7) - 3) : 0.5f); /* rows 1-3: equal keys */
        v_rows[r][h][d] = h16(0.25f * (float)((d + 3 * h + 5 * r) % 9) - 1.0f);
      }
  for (s = 0; s < S; ++s)
    for (h = 0; h < H; ++h)
      for (d = 0; d < D; ++d) q[s][h][d] = h16(0.25f * (float)((d * (s + 1) + h) % 5) - 0.5f);

  CU(cudaMalloc(&kc, sizeof(uint16_t) * NB * B * H * D));
  CU(cudaMalloc(&vc, sizeof(uint16_t) * NB * B * H * D));
  CU(cudaMemset(kc, 0, sizeof(uint16_t) * NB * B * H * D));
  CU(cudaMemset(vc, 0, sizeof(uint16_t) * NB * B * H * D));
  CU(cudaMalloc(&kn, sizeof(k_rows)));
  CU(cudaMalloc(&vn, sizeof(v_rows)));
  CU(cudaMalloc(&sl, sizeof(slots)));
  CU(cudaMalloc(&qd, sizeof(q)));
  CU(cudaMalloc(&od, sizeof(out)));
  CU(cudaMalloc(&td, sizeof(tables)));
  CU(cudaMalloc(&ld, sizeof(lens)));
  CU(cudaMemcpy(kn, k_rows, sizeof(k_rows), cudaMemcpyHostToDevice));
  CU(cudaMemcpy(vn, v_rows, sizeof(v_rows), cudaMemcpyHostToDevice));
  CU(cudaMemcpy(sl, slots, sizeof(slots), cudaMemcpyHostToDevice));
  CU(cudaMemcpy(qd, q, sizeof(q), cudaMemcpyHostToDevice));
  CU(cudaMemcpy(td, tables, sizeof(tables), cudaMemcpyHostToDevice));
  CU(cudaMemcpy(ld, lens, sizeof(lens), cudaMemcpyHostToDevice));

  tkc = desc(kc, PA_F16, 4, cache_shape);
  tvc = desc(vc, PA_F16, 4, cache_shape);
  tkn = desc(kn, PA_F16, 3, rows_shape);
  tvn = desc(vn, PA_F16, 3, rows_shape);
  tsl = desc(sl, PA_I32, 1, slot_shape);
  tq = desc(qd, PA_F16, 3, q_shape);
  tout = desc(od, PA_F16, 3, q_shape);
  ttab = desc(td, PA_I32, 2, table_shape);
  tlen = desc(ld, PA_I32, 1, len_shape);

  PA(pa_cache_append(&tkn, &tvn, &tsl, &tkc, &tvc, NULL));
  PA(pa_decode(&tq, &tkc, &tvc, &ttab, &tlen, 0.08838834764f, &tout, NULL));
  CU(cudaMemcpy(out, od, sizeof(out), cudaMemcpyDeviceToHost));
  PA(pa_get_device_status(NULL, &status));

  for (h = 0; h < H; ++h)
    for (d = 0; d < D; ++d) {
      /* sequence 0: its only value row */
      const uint16_t want0 = v_rows[0][h][d];
      /* sequence 1: mean of value rows 1..3 (a multiple of 1/12; exact when it is a multiple of 1/4) */
      const float m = (0.25f * (float)((d + 3 * h + 5) % 9) + 0.25f * (float)((d + 3 * h + 10) % 9) +
                       0.25f * (float)((d + 3 * h + 15) % 9)) / 3.0f - 1.0f;
      const float m4 = m * 4.0f;
      if (out[0][h][d] != want0) {
        if (bad < 5) printf("seq 0 h %d d %d: got %04x want %04x\n", h, d, out[0][h][d], want0);
        ++bad;
      }
      if (m4 == (float)(int)m4 && out[1][h][d] != h16(m)) {
        if (bad < 5) printf("seq 1 h %d d %d: got %04x want %04x\n", h, d, out[1][h][d], h16(m));
        ++bad;
      }
    }
  printf("mismatches %d status %d\n", bad, (int)status);
  cudaFree(kc);
  cudaFree(vc);
  cudaFree(kn);
  cudaFree(vn);
  cudaFree(sl);
  cudaFree(qd);
  cudaFree(od);
  cudaFree(td);
  cudaFree(ld);
  pa_shutdown();
  return bad != 0 || status != 0;
}
