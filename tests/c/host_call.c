/*
 * host_call.c -- a C program that uses the library through include/sa.h
 * alone: it reads q, k, v (raw [B,H,N,D] arrays of the given dtype) from a
 * file, runs sa_forward_host on them with the global prefix 0..n_global-1 and
 * scale 1/sqrt(D), and writes out ([B,H,N,D], same dtype) and lse ([B,H,N]
 * float32) to a second file.
 *
 *   host_call IN OUT B H N D WINDOW N_GLOBAL DTYPE HEADS_PER_GROUP
 *
 * Exit status: 0 on success, 1 on a usage or file error, 2 with the library's
 * status and message on stderr when the call fails.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "sa.h"

static int read_all(const char *path, void *dst, size_t bytes) {
  FILE *f = fopen(path, "rb");
  if (!f) return 0;
  size_t got = fread(dst, 1, bytes, f);
  fclose(f);
  return got == bytes;
}

int main(int argc, char **argv) {
  if (argc != 11) {
    fprintf(stderr, "usage: %s IN OUT B H N D WINDOW N_GLOBAL DTYPE HEADS_PER_GROUP\n", argv[0]);
    return 1;
  }
  const int B = atoi(argv[3]), H = atoi(argv[4]), N = atoi(argv[5]), D = atoi(argv[6]);
  const int window = atoi(argv[7]), n_global = atoi(argv[8]), hpg = atoi(argv[10]);
  const sa_dtype dtype = (sa_dtype)atoi(argv[9]);
  const size_t es = dtype == SA_BF16 ? 2 : 4;
  const size_t n = (size_t)B * H * N * D, bytes = n * es;
  char *in = (char *)malloc(3 * bytes), *out = (char *)malloc(bytes);
  float *lse = (float *)malloc((size_t)B * H * N * sizeof(float));
  int32_t *g = (int32_t *)malloc(sizeof(int32_t) * (n_global > 0 ? n_global : 1));
  if (!in || !out || !lse || !g) return 1;
  if (!read_all(argv[1], in, 3 * bytes)) {
    fprintf(stderr, "cannot read %zu bytes from %s\n", 3 * bytes, argv[1]);
    return 1;
  }
  for (int i = 0; i < n_global; ++i) g[i] = i;
  const sa_status s = sa_forward_host(in, in + bytes, in + 2 * bytes, out, lse, B, H, N, D, window,
                                      NULL, g, n_global, 1.0f / sqrtf((float)D), dtype, hpg);
  if (s != SA_OK) {
    fprintf(stderr, "sa_forward_host: status %d: %s\n", (int)s, sa_last_error());
    return 2;
  }
  FILE *f = fopen(argv[2], "wb");
  if (!f) return 1;
  int ok = fwrite(out, 1, bytes, f) == bytes &&
           fwrite(lse, sizeof(float), (size_t)B * H * N, f) == (size_t)B * H * N;
  fclose(f);
  free(in);
  free(out);
  free(lse);
  free(g);
  printf("%s: %s\n", sa_version(), ok ? "written" : "write failed");
  return ok ? 0 : 1;
}
