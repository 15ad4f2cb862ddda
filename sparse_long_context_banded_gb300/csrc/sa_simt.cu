// sa_simt.cu -- CUDA-core kernels of the sparse attention path:
//   gather of the global rows, the fp32 band-tile kernel, the fp32 global-row
//   split-K kernel, and the merge of partial softmax statistics.
//
// Attention per row (Unlimiformer section 2.3 Eq. (1) with GMAT's additive
// {0,-inf} mask): o_i = sum_{j in S_i} exp(s_j - m) v_j / sum_{j in S_i} exp(s_j - m),
// s_j = scale * q_i.k_j.  Rows are processed one key tile at a time with a
// running maximum and sum (the tiled exact softmax that the Longformer
// glossary's "Flash Attention" entry describes: tiles held on chip).  Scores
// are kept in base-2 units (s * log2 e) so that exp2 can be used throughout.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "sa_kernels.h"

namespace sa {
namespace {

template <typename T>
__device__ __forceinline__ float ld(const void *p, int64_t i);
template <>
__device__ __forceinline__ float ld<float>(const void *p, int64_t i) {
  return static_cast<const float *>(p)[i];
}
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const void *p, int64_t i) {
  return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
}
template <typename T>
__device__ __forceinline__ void st(void *p, int64_t i, float x);
template <>
__device__ __forceinline__ void st<float>(void *p, int64_t i, float x) {
  static_cast<float *>(p)[i] = x;
}
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(void *p, int64_t i, float x) {
  static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------------------
// gather: q/k/v rows of the global positions -> [bh][g_pad][D]; pad rows zero.
template <typename T>
__global__ void gather_kernel(DevProblem p) {
  const int g = blockIdx.x, bh = blockIdx.y;
  const int64_t dst = ((int64_t)bh * p.g_pad + g) * p.D;
  if (g < p.n_g) {
    const int64_t src = ((int64_t)bh * p.N + p.globals[g]) * p.D;
    for (int c = threadIdx.x; c < p.D; c += blockDim.x) {
      static_cast<T *>(p.qg)[dst + c] = static_cast<const T *>(p.gq_src)[src + c];
      static_cast<T *>(p.kg)[dst + c] = static_cast<const T *>(p.k)[src + c];
      static_cast<T *>(p.vg)[dst + c] = static_cast<const T *>(p.v)[src + c];
    }
  } else {
    for (int c = threadIdx.x; c < p.D; c += blockDim.x) {
      static_cast<T *>(p.qg)[dst + c] = T(0.f);
      static_cast<T *>(p.kg)[dst + c] = T(0.f);
      static_cast<T *>(p.vg)[dst + c] = T(0.f);
    }
  }
}

// ---------------------------------------------------------------------------
// One 64-row query tile against one 64-key tile, 256 threads: thread (row,
// quarter) scores keys quarter, quarter+4, ... and owns D/4 output columns.
constexpr int QT = 64, KT = 64, NT = 256;

template <int D>
struct SimtState {
  float m, l;
  float acc[D / 4];
};

template <int D, typename Valid>
__device__ __forceinline__ void simt_tile(const float *Qs, const float *Ks,
                                          const float *Vs, float *Ps, int row,
                                          int qd, float scale_log2, Valid valid,
                                          SimtState<D> &st_) {
  constexpr int LD = D + 1;
  float s[KT / 4];
  float tmax = -INFINITY;
#pragma unroll
  for (int mm = 0; mm < KT / 4; ++mm) {
    const int c = qd + 4 * mm;
    float x = -INFINITY;
    if (valid(c)) {
      float dot = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) dot = fmaf(Qs[row * LD + d], Ks[c * LD + d], dot);
      x = dot * scale_log2;
    }
    s[mm] = x;
    tmax = fmaxf(tmax, x);
  }
  tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
  tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
  const float m_new = fmaxf(st_.m, tmax);
  const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // no valid key yet
  const float alpha = exp2f(st_.m - m_use);
  float psum = 0.f;
#pragma unroll
  for (int mm = 0; mm < KT / 4; ++mm) {
    const float pr = exp2f(s[mm] - m_use);
    Ps[row * (KT + 1) + qd + 4 * mm] = pr;
    psum += pr;
  }
  psum += __shfl_xor_sync(0xffffffffu, psum, 1);
  psum += __shfl_xor_sync(0xffffffffu, psum, 2);
  st_.l = st_.l * alpha + psum;
  st_.m = m_new;
#pragma unroll
  for (int j = 0; j < D / 4; ++j) st_.acc[j] *= alpha;
  __syncwarp();
  for (int c = 0; c < KT; ++c) {
    const float pr = Ps[row * (KT + 1) + c];
    const float *vr = Vs + c * LD + qd * (D / 4);
#pragma unroll
    for (int j = 0; j < D / 4; ++j) st_.acc[j] = fmaf(pr, vr[j], st_.acc[j]);
  }
  __syncwarp();
}

template <typename T, int D>
__device__ __forceinline__ void load_rows(float *dst, const void *src, int64_t row0_elem,
                                          int64_t row_stride_elems, int n_rows_valid) {
  constexpr int LD = D + 1;
  for (int e = threadIdx.x; e < KT * D; e += NT) {
    const int rr = e / D, c = e % D;
    dst[rr * LD + c] = rr < n_rows_valid ? ld<T>(src, row0_elem + rr * row_stride_elems + c) : 0.f;
  }
}

template <int D>
__host__ __device__ constexpr size_t simt_smem_bytes() {
  return sizeof(float) * (size_t)(QT * (D + 1) + 2 * KT * (D + 1) + QT * (KT + 1)) +
         sizeof(int32_t) * SA_MAX_GLOBALS;
}

// Band tiles of one query tile of one residue class, then the global tile(s).
template <typename T, int D>
__global__ void __launch_bounds__(NT) band_simt_kernel(DevProblem p) {
  extern __shared__ float smem[];
  constexpr int LD = D + 1;
  float *Qs = smem;
  float *Ks = Qs + QT * LD;
  float *Vs = Ks + KT * LD;
  float *Ps = Vs + KT * LD;
  int32_t *Gs = reinterpret_cast<int32_t *>(Ps + QT * (KT + 1));

  const BandItem it = p.band[blockIdx.x];
  const Slot sl = p.slots[it.slot];
  const int64_t base = (int64_t)it.bh * p.N * D;
  const int64_t cls_stride = (int64_t)sl.d * D;          // elements between class rows
  const int64_t cls_base = base + (int64_t)sl.r * D;      // element of class row 0
  const int tid = threadIdx.x, row = tid >> 2, qd = tid & 3;
  const int t_row = it.q_tile * QT + row;
  const bool row_ok = t_row < sl.len;
  const int64_t pos_row = sl.r + (int64_t)sl.d * t_row;
  const int half = p.half;
  int key_lo, key_hi;  // the row's non-global keys (band or chunk), class coordinates
  row_keys(half, p.chunk, p.memory, sl.len, t_row, key_lo, key_hi);

  for (int g = tid; g < p.n_g; g += NT) Gs[g] = p.globals[g];
  load_rows<T, D>(Qs, p.q, cls_base + (int64_t)it.q_tile * QT * cls_stride, cls_stride,
                  min(QT, sl.len - it.q_tile * QT));

  SimtState<D> st_;
  st_.m = -INFINITY;
  st_.l = 0.f;
#pragma unroll
  for (int j = 0; j < D / 4; ++j) st_.acc[j] = 0.f;

  for (int kt = it.k_lo[0]; kt <= it.k_hi[0]; ++kt) {
    __syncthreads();
    const int t0 = kt * KT;
    load_rows<T, D>(Ks, p.k, cls_base + (int64_t)t0 * cls_stride, cls_stride, min(KT, sl.len - t0));
    load_rows<T, D>(Vs, p.v, cls_base + (int64_t)t0 * cls_stride, cls_stride, min(KT, sl.len - t0));
    __syncthreads();
    simt_tile<D>(Qs, Ks, Vs, Ps, row, qd, p.scale_log2,
                 [&](int c) {
                   const int tk = t0 + c;
                   return row_ok && tk < sl.len && tk >= key_lo && tk <= key_hi;
                 },
                 st_);
  }
  for (int g0 = 0; g0 < p.n_g; g0 += KT) {
    __syncthreads();
    const int64_t gbase = ((int64_t)it.bh * p.g_pad + g0) * D;
    load_rows<T, D>(Ks, p.kg, gbase, D, min(KT, p.n_g - g0));
    load_rows<T, D>(Vs, p.vg, gbase, D, min(KT, p.n_g - g0));
    __syncthreads();
    simt_tile<D>(Qs, Ks, Vs, Ps, row, qd, p.scale_log2,
                 [&](int c) {
                   const int gi = g0 + c;
                   if (!row_ok || gi >= p.n_g) return false;
                   // a global key already among this row's band keys is not counted
                   // twice (the chunked pattern's memory never is)
                   if (p.chunk > 0) return true;
                   const int64_t diff = pos_row - Gs[gi];
                   const int64_t reach = (int64_t)half * sl.d;
                   const bool in_band = diff <= reach && -diff <= reach && diff % sl.d == 0;
                   return !in_band;
                 },
                 st_);
  }
  if (row_ok) {
    const float inv = 1.f / st_.l;
    const int64_t o = base + pos_row * D + qd * (D / 4);
#pragma unroll
    for (int j = 0; j < D / 4; ++j) st<T>(p.out, o + j, st_.acc[j] * inv);
    if (p.lse && qd == 0)
      p.lse[(int64_t)it.bh * p.N + pos_row] = (st_.m + log2f(st_.l)) * 0.6931471805599453f;
  }
}

// Global rows: gathered global queries against one key chunk, all keys valid.
template <typename T, int D>
__global__ void __launch_bounds__(NT) global_simt_kernel(DevProblem p) {
  extern __shared__ float smem[];
  constexpr int LD = D + 1;
  float *Qs = smem;
  float *Ks = Qs + QT * LD;
  float *Vs = Ks + KT * LD;
  float *Ps = Vs + KT * LD;

  const GlobalItem it = p.gitems[blockIdx.x];
  const int64_t base = (int64_t)it.bh * p.N * D;
  const int tid = threadIdx.x, row = tid >> 2, qd = tid & 3;
  const int g = it.g_tile * QT + row;
  const bool row_ok = g < p.n_g;
  const int key_lo = it.chunk * p.chunk_len;
  const int key_hi = min(p.N, key_lo + p.chunk_len);

  load_rows<T, D>(Qs, p.qg, ((int64_t)it.bh * p.g_pad + it.g_tile * QT) * D, D, QT);

  SimtState<D> st_;
  st_.m = -INFINITY;
  st_.l = 0.f;
#pragma unroll
  for (int j = 0; j < D / 4; ++j) st_.acc[j] = 0.f;

  for (int t0 = key_lo; t0 < key_hi; t0 += KT) {
    __syncthreads();
    load_rows<T, D>(Ks, p.gk_src, base + (int64_t)t0 * D, D, min(KT, key_hi - t0));
    load_rows<T, D>(Vs, p.gv_src, base + (int64_t)t0 * D, D, min(KT, key_hi - t0));
    __syncthreads();
    simt_tile<D>(Qs, Ks, Vs, Ps, row, qd, p.scale_log2,
                 [&](int c) { return row_ok && t0 + c < key_hi; }, st_);
  }
  if (row_ok) {
    const int64_t slot = ((int64_t)it.bh * p.part_sets + it.chunk) * p.g_pad + g;
#pragma unroll
    for (int j = 0; j < D / 4; ++j) p.part_o[slot * D + qd * (D / 4) + j] = st_.acc[j];
    if (qd == 0) {
      p.part_ml[slot * 2 + 0] = st_.m;
      p.part_ml[slot * 2 + 1] = st_.l;
    }
  }
}

// ---------------------------------------------------------------------------
// merge: m = max_c m_c, l = sum_c l_c 2^(m_c - m), o = sum_c o_c 2^(m_c - m) / l.
// One block per (global row, head); writes that global row of `out` (and lse).
// Upper bound of the key chunks of the global-row pass (the schedule asks for
// at most a few hundred CTAs).
constexpr int kMaxMergeChunks = 1024;  // a multiple of the merge block

constexpr int kMergeThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(DevProblem p) {
  // One block per (global row, head).  Partial x is row g + 64 (x % part_sub)
  // of set x / part_sub.  The odd set of a chunk holding a single key tile was
  // never written (g_alt: the chunk's second query tile had no key tile to
  // take), and a partial that saw no key has max -inf and sum 0: both get
  // weight 0.  Each partial's (max, sum) pair is read once, as one 8-byte
  // load.  Then the block sums the partials column by column: thread t takes
  // four consecutive columns (one 16-byte load per partial) of the partials
  // x = g, g + G, g + 2G, ... (g = t / (D/4), G = 128 / (D/4) groups), eight
  // loads in flight at a time, and the G group sums of each column are added
  // in a fixed order, so the result is the same for every call.  The partials
  // are read in full only after the kernels that write them are done (launched
  // as a programmatic dependent: the launch itself overlaps them).
  __shared__ float w_part[kMaxMergeChunks];
  __shared__ int64_t row_part[kMaxMergeChunks];
  __shared__ float red[kMergeThreads / 32];
  __shared__ __align__(16) float colsum[kMergeThreads * 4];  // [group][D]
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int g = blockIdx.x, bh = blockIdx.y, t = threadIdx.x;
  constexpr int nt = kMergeThreads, nw = kMergeThreads / 32;
  const int np = p.part_sets * p.part_sub;
  const int64_t row0 = (int64_t)bh * p.part_sets * p.g_pad + g;  // set 0, first sub-row: written
  float m = -INFINITY;
  float2 ml[kMaxMergeChunks / nt];  // this thread's partials x = t, t + nt, ...
#pragma unroll
  for (int k = 0; k < kMaxMergeChunks / nt; ++k) {
    const int x = t + k * nt;
    ml[k] = make_float2(-INFINITY, 0.f);
    if (x < np) {
      const int set = x / p.part_sub, sub = x - set * p.part_sub;
      bool written = true;
      if (p.g_alt && (set & 1)) {
        const int c = set >> 1;
        written = min(p.N, (c + 1) * p.chunk_len) - c * p.chunk_len > 128;
      }
      const int64_t r = row0 + (int64_t)set * p.g_pad + 64 * sub;
      row_part[x] = written ? r : row0;
      if (written) ml[k] = reinterpret_cast<const float2 *>(p.part_ml)[r];
      m = fmaxf(m, ml[k].x);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((t & 31) == 0) red[t >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < nw; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  float l = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxMergeChunks / nt; ++k) {
    const int x = t + k * nt;
    if (x < np) {
      const float wc = ml[k].x == -INFINITY ? 0.f : exp2f(ml[k].x - m);
      l += wc != 0.f ? ml[k].y * wc : 0.f;
      w_part[x] = wc;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if ((t & 31) == 0) red[t >> 5] = l;
  __syncthreads();  // (also: w_part and row_part complete)
  l = red[0];
#pragma unroll
  for (int i = 1; i < nw; ++i) l += red[i];
  // column sums: thread t, columns 4 (t % q) .. + 3 of the partials x = grp, grp + G, ...
  const int q = p.D / 4, G = nt / q, grp = t / q, c4 = t - grp * q;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int x = grp;
  for (; x + 7 * G < np; x += 8 * G) {
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[k] = reinterpret_cast<const float4 *>(p.part_o + row_part[x + k * G] * p.D)[c4];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float wk = w_part[x + k * G];
      if (wk != 0.f) {
        acc.x += v[k].x * wk;
        acc.y += v[k].y * wk;
        acc.z += v[k].z * wk;
        acc.w += v[k].w * wk;
      }
    }
  }
  for (; x < np; x += G) {
    const float wk = w_part[x];
    const float4 vk = reinterpret_cast<const float4 *>(p.part_o + row_part[x] * p.D)[c4];
    if (wk != 0.f) {
      acc.x += vk.x * wk;
      acc.y += vk.y * wk;
      acc.z += vk.z * wk;
      acc.w += vk.w * wk;
    }
  }
  reinterpret_cast<float4 *>(colsum)[grp * q + c4] = acc;
  __syncthreads();
  const float inv = 1.f / l;
  const int64_t orow = ((int64_t)bh * p.N + p.globals[g]) * p.D;
  for (int d = t; d < p.D; d += nt) {
    float sum = 0.f;
    for (int k = 0; k < G; ++k) sum += colsum[k * p.D + d];
    st<T>(p.out, orow + d, sum * inv);
  }
  if (p.lse && t == 0)
    p.lse[(int64_t)bh * p.N + p.globals[g]] = (m + log2f(l)) * 0.6931471805599453f;
}

template <typename T, int D>
cudaError_t band_simt_launch(const DevProblem &p, cudaStream_t s) {
  constexpr size_t smem = simt_smem_bytes<D>();
  cudaError_t e = cudaFuncSetAttribute(band_simt_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  band_simt_kernel<T, D><<<p.n_band, NT, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t global_simt_launch(const DevProblem &p, cudaStream_t s) {
  constexpr size_t smem = simt_smem_bytes<D>();
  cudaError_t e = cudaFuncSetAttribute(global_simt_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  global_simt_kernel<T, D><<<p.n_gitems, NT, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

// 32 x 32 tiles through shared memory: coalesced reads of value rows,
// coalesced writes of the transposed rows.
__global__ void transpose_values_kernel(const float *src, float *dst, int n_src, int D, int r,
                                        int step, int len, int len_pad) {
  __shared__ float tile[32][33];
  const int t0 = blockIdx.x * 32, d0 = blockIdx.y * 32, bh = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int i = ty; i < 32; i += 8) {
    const int t = t0 + i;
    tile[i][tx] = (t < len && d0 + tx < D)
                      ? src[((int64_t)bh * n_src + r + (int64_t)step * t) * D + d0 + tx]
                      : 0.f;
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int d = d0 + i, t = t0 + tx;
    if (d < D && t < len_pad) dst[((int64_t)bh * D + d) * len_pad + t] = tile[tx][i];
  }
}

cudaError_t launch_transpose_values(const float *src, float *dst, int n_src, int D, int r,
                                    int step, int len, int len_pad, int BH, cudaStream_t s) {
  dim3 grid((len_pad + 31) / 32, (D + 31) / 32, BH), block(32, 8);
  transpose_values_kernel<<<grid, block, 0, s>>>(src, dst, n_src, D, r, step, len, len_pad);
  return cudaGetLastError();
}

cudaError_t launch_gather(const DevProblem &p, int BH, sa_dtype dt, cudaStream_t s) {
  dim3 grid(p.g_pad, BH);
  if (dt == SA_BF16)
    gather_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(p);
  else
    gather_kernel<float><<<grid, 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_band_simt(const DevProblem &p, sa_dtype dt, cudaStream_t s) {
  if (dt == SA_BF16)
    return p.D == 64 ? band_simt_launch<__nv_bfloat16, 64>(p, s)
                     : band_simt_launch<__nv_bfloat16, 128>(p, s);
  return p.D == 64 ? band_simt_launch<float, 64>(p, s) : band_simt_launch<float, 128>(p, s);
}

cudaError_t launch_global_simt(const DevProblem &p, sa_dtype dt, cudaStream_t s) {
  if (dt == SA_BF16)
    return p.D == 64 ? global_simt_launch<__nv_bfloat16, 64>(p, s)
                     : global_simt_launch<__nv_bfloat16, 128>(p, s);
  return p.D == 64 ? global_simt_launch<float, 64>(p, s) : global_simt_launch<float, 128>(p, s);
}

cudaError_t launch_merge(const DevProblem &p, int BH, sa_dtype dt, cudaStream_t s) {
  if (p.part_sets * p.part_sub > kMaxMergeChunks) return cudaErrorInvalidValue;
  // 128 threads per (global row, head); a programmatic dependent launch, so
  // that the launch overlaps the kernels before it (the kernel waits for them
  // with griddepcontrol.wait before it reads anything)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.n_g, BH);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (dt == SA_BF16) return cudaLaunchKernelEx(&cfg, merge_kernel<__nv_bfloat16>, p);
  return cudaLaunchKernelEx(&cfg, merge_kernel<float>, p);
}

}  // namespace sa
