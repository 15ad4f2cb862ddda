// sa_kernels.h -- device-side view of one call, and the kernel launchers.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "sa_internal.h"

namespace sa {

// Error bits OR-ed into the per-device error word by kernels.
enum : int {
  kErrWaitTimeout = 1,  // an mbarrier wait gave up (bounded spin ran out)
  kErrBadWork = 2,      // a work item failed a device-side range check
};

struct DevProblem {
  const void *q, *k, *v;
  // What the global-row pass reads: queries (gathered at the global
  // positions), keys and values.  q, k, v themselves, or separate global
  // projections of the same shape.
  const void *gq_src, *gk_src, *gv_src;
  void *out;
  float *lse;       // [B*H*N] or null
  int N, D, H;
  int half;         // floor(window / 2)
  int chunk, memory;  // chunked pattern (chunk > 0): chunk length, memory tokens
  float scale_log2; // scale * log2(e): scores are kept in base-2 units
  const int32_t *globals;  // device, sorted unique, n_g entries
  int n_g, g_pad;
  // >= 0: the globals are the contiguous positions [g_first, g_first + n_g), and
  // the tensor-core kernels read their rows through views of q (or the global
  // queries' source), k and v instead of gathered copies; -1 otherwise
  int g_first;
  const Slot *slots;
  int n_slots;
  const BandItem *band;
  int n_band;
  int BH;  // batch x heads
  const GlobalItem *gitems;
  int n_gitems;
  int n_chunks, chunk_len;
  // Partials of the global-row pass: part_sets sets per head, each g_pad rows.
  // Global g's partials are rows g + 64 s (s < part_sub) of every set.  With
  // g_alt the two query tiles of a CTA take alternate key tiles of chunk c and
  // leave sets 2c and 2c + 1 (a chunk of a single key tile leaves only 2c);
  // with g_packed the (at most 64) global rows fill a query tile twice, rows
  // r and r + 64 taking the first and second 64 keys of each key tile.
  int part_sets, part_sub;
  int g_alt, g_packed;
  // scratch
  void *qg, *kg, *vg;  // [B*H][g_pad][D] gathered global rows, input dtype
  // fp32 inputs on the tensor cores (tf32): values transposed so that the P V
  // product reads them K-major (tf32 operands must be K-major)
  float *vT_slots;  // per residue-class slot s, back to back: [B*H][D][len_pad(s)]
  float *vT_plain;  // [B*H][D][round_up(N, 4)] of the global-row pass's values
  float *vgT;       // [B*H][D][g_pad] of the gathered global values
  float *part_o;       // [B*H][part_sets][g_pad][D]  unnormalised partial outputs
  float *part_ml;      // [B*H][part_sets][g_pad][2]  partial (max, sum), base 2
  int *err;
};

// Attention over per-query key lists (sa_gather.cu).
struct GatherProblem {
  const void *q, *k, *v;  // [B*H][Nq][D], [B*H][Nk][D], [B*H][Nk][D]
  const int32_t *idx;     // [B*H][Nq][K]; entries outside [0, Nk) are padding
  void *out;              // [B*H][Nq][D]
  float *lse;             // [B*H][Nq] or null
  int64_t rows;           // B*H*Nq
  int Nq, Nk, K, D;
  float scale_log2;
};
cudaError_t launch_gather_attention(const GatherProblem &p, sa_dtype dt, cudaStream_t s);

// SIMT path (fp32 inputs): CUDA-core arithmetic, fp32 throughout.
constexpr Tiling kSimtTiling{64, 1, 64, 64, 64, 608, 1 << 30};
cudaError_t launch_gather(const DevProblem &p, int BH, sa_dtype dt, cudaStream_t s);
cudaError_t launch_band_simt(const DevProblem &p, sa_dtype dt, cudaStream_t s);
cudaError_t launch_global_simt(const DevProblem &p, sa_dtype dt, cudaStream_t s);
cudaError_t launch_merge(const DevProblem &p, int BH, sa_dtype dt, cudaStream_t s);
// dst[bh][d][t] = src[bh][r + step t][d] for t < len, 0 for len <= t < len_pad
// (src: [BH][n_src][D] fp32); len_pad a multiple of 4.
cudaError_t launch_transpose_values(const float *src, float *dst, int n_src, int D, int r,
                                    int step, int len, int len_pad, int BH, cudaStream_t s);
inline int values_len_pad(int len) { return (len + 3) & ~3; }

}  // namespace sa
