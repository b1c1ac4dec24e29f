/* A decode step driven from plain C through include/decattn.h: write each
 * sequence's new token into the paged caches, then attend (GQA with and
 * without splits, absorbed MLA), and check results that have closed forms:
 *   - every cached V row of KV head j equals the constant c_j, so any
 *     softmax-weighted sum of them is c_j (up to the rounding of the 16-bit
 *     probabilities, far inside the 1/128 relative bound checked here; the
 *     two KV heads' constants differ by a factor of -2, so a wrong head
 *     mapping fails);
 *   - MLA with a latent whose first 512 entries are the constant c returns c.
 * Exit status 0 and "c abi ok" on success. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "decattn.h"

#define CHECK(x)                                                        \
  do {                                                                  \
    int st_ = (x);                                                      \
    if (st_ != 0) {                                                     \
      fprintf(stderr, "%s:%d: %s -> %d\n", __FILE__, __LINE__, #x, st_); \
      return 1;                                                         \
    }                                                                   \
  } while (0)

static uint16_t bf16_of(float f) { /* exact for the small dyadic values used here */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

static float float_of_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static int near(float got, float want) { return fabsf(got - want) <= fabsf(want) / 128.f; }

static void* dev_copy(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
  if (cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return d;
}

int main(void) {
  enum { B = 3, HQ = 8, HKV = 2, D = 128, BS = 16, MAXB = 8, NB = B * MAXB };
  const int lens[B] = {1, 50, 128}; /* lengths after this step's append */
  int32_t seq_lens[B], positions[B], table[B * MAXB];
  for (int b = 0; b < B; ++b) {
    seq_lens[b] = lens[b];
    positions[b] = lens[b] - 1;
    for (int k = 0; k < MAXB; ++k) table[b * MAXB + k] = (b * MAXB + k * 5) % NB; /* a permutation */
  }
  /* caches: K arbitrary, V constant c_j per KV head; new rows follow the same rule */
  const size_t cache_elems = (size_t)NB * BS * HKV * D;
  uint16_t* k = malloc(cache_elems * 2);
  uint16_t* v = malloc(cache_elems * 2);
  for (size_t i = 0; i < cache_elems; ++i) {
    const int j = (int)((i / D) % HKV);
    k[i] = bf16_of((float)((int)(i % 7) - 3) * 0.125f);
    v[i] = bf16_of(j == 0 ? 0.75f : -1.5f);
  }
  uint16_t kn[B * HKV * D], vn[B * HKV * D], q[B * HQ * D];
  for (int i = 0; i < B * HKV * D; ++i) {
    kn[i] = bf16_of(0.25f);
    vn[i] = bf16_of(((i / D) % HKV) == 0 ? 0.75f : -1.5f);
  }
  for (int i = 0; i < B * HQ * D; ++i) q[i] = bf16_of((float)((i % 5) - 2) * 0.0625f);

  void *dk = dev_copy(k, cache_elems * 2), *dv = dev_copy(v, cache_elems * 2);
  void *dkn = dev_copy(kn, sizeof kn), *dvn = dev_copy(vn, sizeof vn), *dq = dev_copy(q, sizeof q);
  void *dsl = dev_copy(seq_lens, sizeof seq_lens), *dpos = dev_copy(positions, sizeof positions);
  void* dbt = dev_copy(table, sizeof table);
  void *dout = NULL, *dflag = NULL, *dws = NULL;
  int zero = 0;
  dflag = dev_copy(&zero, sizeof zero);
  if (!dk || !dv || !dkn || !dvn || !dq || !dsl || !dpos || !dbt || !dflag ||
      cudaMalloc(&dout, sizeof q) != cudaSuccess) {
    fprintf(stderr, "allocation failed\n");
    return 1;
  }

  decattn_launch L;
  memset(&L, 0, sizeof L);
  L.batch = B;
  L.num_blocks = NB;
  L.block_size = BS;
  L.max_blocks_per_seq = MAXB;
  L.max_seq_len = 128;
  L.dtype = DECATTN_BF16;
  L.err_flag = (int*)dflag;
  CHECK(gqa_kv_append(dkn, dvn, (const int32_t*)dpos, (const int32_t*)dbt, dk, dv, HKV, D, &L));

  uint16_t out[B * HQ * D];
  for (int ns = 1; ns <= 3; ns += 2) {
    L.num_splits = ns;
    const size_t ws = gqa_decode_workspace_size(B, HQ, D, ns);
    if (ws && cudaMalloc(&dws, ws) != cudaSuccess) return 1;
    L.workspace = dws;
    L.workspace_bytes = ws;
    CHECK(gqa_decode(dq, dk, dv, (const int32_t*)dbt, (const int32_t*)dsl, dout, HQ, HKV, D,
                     1.0f / sqrtf((float)D), &L));
    if (cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
    for (int i = 0; i < B * HQ * D; ++i) {
      const int head = (i / D) % HQ, j = head / (HQ / HKV);
      const float want = j == 0 ? 0.75f : -1.5f;
      if (!near(float_of_bf16(out[i]), want)) {
        fprintf(stderr, "gqa splits=%d: element %d = %g, want %g\n", ns, i,
                float_of_bf16(out[i]), want);
        return 1;
      }
    }
    if (dws) cudaFree(dws);
    dws = NULL;
  }

  /* MLA: 128 heads over a latent cache whose first 512 entries are 0.5 */
  enum { H = 128, W = 576 };
  const size_t lat_elems = (size_t)NB * BS * W;
  uint16_t* lat = malloc(lat_elems * 2);
  for (size_t i = 0; i < lat_elems; ++i)
    lat[i] = bf16_of((i % W) < 512 ? 0.5f : (float)((int)(i % 3) - 1) * 0.25f);
  uint16_t* qa = malloc((size_t)B * H * 512 * 2);
  uint16_t* qr = malloc((size_t)B * H * 64 * 2);
  for (size_t i = 0; i < (size_t)B * H * 512; ++i) qa[i] = bf16_of((float)((int)(i % 9) - 4) * 0.03125f);
  for (size_t i = 0; i < (size_t)B * H * 64; ++i) qr[i] = bf16_of(0.125f);
  void *dlat = dev_copy(lat, lat_elems * 2), *dqa = dev_copy(qa, (size_t)B * H * 512 * 2);
  void* dqr = dev_copy(qr, (size_t)B * H * 64 * 2);
  void* dmo = NULL;
  if (!dlat || !dqa || !dqr || cudaMalloc(&dmo, (size_t)B * H * 512 * 2) != cudaSuccess) return 1;
  L.num_splits = 2; /* two CTA pairs share the batch's tiles */
  const size_t mws = mla_decode_workspace_size(B, 2);
  if (cudaMalloc(&dws, mws) != cudaSuccess) return 1;
  L.workspace = dws;
  L.workspace_bytes = mws;
  CHECK(mla_decode(dqa, dqr, dlat, (const int32_t*)dbt, (const int32_t*)dsl, dmo,
                   1.0f / sqrtf(192.0f), &L));
  uint16_t* mo = malloc((size_t)B * H * 512 * 2);
  if (cudaMemcpy(mo, dmo, (size_t)B * H * 512 * 2, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
  for (size_t i = 0; i < (size_t)B * H * 512; ++i) {
    if (!near(float_of_bf16(mo[i]), 0.5f)) {
      fprintf(stderr, "mla: element %zu = %g, want 0.5\n", i, float_of_bf16(mo[i]));
      return 1;
    }
  }
  int flag = -1;
  if (cudaMemcpy(&flag, dflag, sizeof flag, cudaMemcpyDeviceToHost) != cudaSuccess) return 1;
  if (flag != 0) {
    fprintf(stderr, "error flag %d\n", flag);
    return 1;
  }
  void* dev[] = {dk, dv, dkn, dvn, dq, dsl, dpos, dbt, dout, dflag, dws, dlat, dqa, dqr, dmo};
  for (size_t i = 0; i < sizeof dev / sizeof dev[0]; ++i) cudaFree(dev[i]);
  free(k);
  free(v);
  free(lat);
  free(qa);
  free(qr);
  free(mo);
  printf("c abi ok (%s, version %d)\n", decattn_status_string(DECATTN_OK), decattn_version());
  return 0;
}
