// sa_gather.cu -- attention over per-query key lists: each query row attends
// only to the keys its list names ("Unlimiformer", section 2.2
// "Retrieval-augmented Cross-Attention": every head retrieves its top-k keys
// and attends only to them; section 2.3 Eq. (1): standard dot-product
// attention over that set).  The retrieval itself (a kNN index) is the
// caller's; this kernel takes its output, the lists.
//
// Each query has its own key set, so there is no tile of keys shared by many
// queries to put on the tensor cores: the work is a gather of key and value
// rows (2 * D * element size bytes per listed entry) with a handful of flops per
// byte, bound by memory.  The layout follows from that:
//
//  * one warp per query row, split into lane groups of LPR lanes, each group
//    on a key of its own: a key or value row is read by the LPR lanes of a
//    group in one coalesced load (lane l of the group holds elements
//    [E l, E l + E), E = D / LPR; 32 bytes per lane for bf16 rows of 128), so
//    one warp-wide load fetches 32 / LPR rows and the per-row cost of index
//    broadcasts, addresses and loads shrinks by that factor;
//  * keys are taken 32 at a time (one list entry per lane) in LPR rounds of
//    32 / LPR keys, their rows loaded four rounds at a time with all loads in
//    flight before the first use;
//  * the LPR per-lane partial dot products of a group are summed by a
//    reduce-scatter butterfly within the group (LPR - 1 shuffles), after
//    which lane (g, l) holds the score of the key of round l in group g -- no
//    per-key reduction;
//  * online softmax in base 2 with fp32 state: the running maximum is a warp
//    maximum per 32 keys, each lane keeps a partial row sum, the value rows
//    are weighted with each key's probability fetched from its lane, each
//    group accumulating its own keys; the groups are added at the end.
//
// Rows are numbered head-major, so the warps running at one time read the keys
// and values of one or two heads, which stay in L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sa_kernels.h"

namespace sa {
namespace {

constexpr int kWarpsPerBlock = 8;

// A lane's slice of a row: E elements of T in NV 16-byte words, loaded with
// 16-byte loads and kept packed until used (bf16 pairs stay packed, so that a
// batch of loads in flight costs half the registers).
template <typename T, int E>
struct Slice {
  static constexpr int NV = E * (int)sizeof(T) / 16;
  static_assert(NV * 16 == E * (int)sizeof(T), "a lane's slice is a whole number of 16-byte words");
  uint4 w[NV];
  static __device__ __forceinline__ Slice load(const void *base, int64_t elem) {
    const uint4 *r = reinterpret_cast<const uint4 *>(static_cast<const T *>(base) + elem);
    Slice x;
#pragma unroll
    for (int i = 0; i < NV; ++i) x.w[i] = __ldg(r + i);
    return x;
  }
  static __device__ __forceinline__ Slice zero() {
    Slice x;
#pragma unroll
    for (int i = 0; i < NV; ++i) x.w[i] = make_uint4(0u, 0u, 0u, 0u);
    return x;
  }
  __device__ __forceinline__ void unpack(float (&f)[E]) const {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const uint32_t u[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if constexpr (sizeof(T) == 2) {
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u[k]));
          f[8 * i + 2 * k] = a.x;
          f[8 * i + 2 * k + 1] = a.y;
        } else {
          f[4 * i + k] = __uint_as_float(u[k]);
        }
      }
    }
  }
  // writes f (rounded to T) as the lane's slice of the row at `elem`
  static __device__ __forceinline__ void store(void *base, int64_t elem, const float (&f)[E]) {
    uint4 *o = reinterpret_cast<uint4 *>(static_cast<T *>(base) + elem);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      uint32_t u[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if constexpr (sizeof(T) == 2) {
          __nv_bfloat162 h = __floats2bfloat162_rn(f[8 * i + 2 * k], f[8 * i + 2 * k + 1]);
          u[k] = *reinterpret_cast<uint32_t *>(&h);
        } else {
          u[k] = __float_as_uint(f[4 * i + k]);
        }
      }
      o[i] = make_uint4(u[0], u[1], u[2], u[3]);
    }
  }
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Lanes per row: a lane takes 16 bytes of a key or value row, 32 for bf16
// rows of 128 (8 lanes per row, four rows per warp-wide load: 1.5% faster
// than 16 lanes on the retrieval workload); bf16 D=64: 8 lanes; fp32: 16 / 32.
template <typename T, int D>
constexpr int kLanesPerRow = (sizeof(T) == 2 && D == 128) ? 8 : D * (int)sizeof(T) / 16;
// Rounds (one row per lane group each) whose loads one batch keeps in flight.
constexpr int kRoundBatch = 4;
// Blocks per SM the registers are sized for: three where a lane holds 32
// bytes of a row or 32 partial scores, four otherwise.
template <typename T, int D, int LPR>
constexpr int kMinBlocks = ((D / LPR) * (int)sizeof(T) >= 32 || LPR == 32) ? 3 : 4;

template <typename T, int D, int LPR>
__global__ void __launch_bounds__(32 * kWarpsPerBlock, kMinBlocks<T, D, LPR>)
    gather_attention_kernel(GatherProblem p) {
  constexpr int E = D / LPR;    // row elements per lane
  constexpr int G = 32 / LPR;   // lane groups: rows per warp-wide load
  constexpr int R = LPR;        // rounds per 32 keys
  constexpr int NB = kRoundBatch < R ? kRoundBatch : R;
  using SL = Slice<T, E>;
  const int lane = threadIdx.x & 31, grp = lane / LPR, gl = lane % LPR;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= p.rows) return;  // whole warps only: the warp's lanes share `row`
  const int64_t bh = row / p.Nq;
  const int64_t kv_head = bh * (int64_t)p.Nk * D;  // first element of this head's keys / values
  const int32_t *list = p.idx + row * (int64_t)p.K;

  float qf[E];  // every lane group holds the same elements of the query row
  SL::load(p.q, row * D + gl * E).unpack(qf);
#pragma unroll
  for (int e = 0; e < E; ++e) qf[e] *= p.scale_log2;  // scores in base-2 units

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float m_run = -INFINITY, l_lane = 0.f;

  for (int t0 = 0; t0 < p.K; t0 += 32) {
    // this lane's list entry; padding and out-of-range entries become -1
    int j_mine = -1;
    if (t0 + lane < p.K) {
      const int j = __ldg(list + t0 + lane);
      j_mine = (j >= 0 && j < p.Nk) ? j : -1;
    }
    // partial dot products of this lane's elements with its group's key of
    // each round x (the group of 32's key G x + grp)
    float part[R];
#pragma unroll
    for (int h = 0; h < R / NB; ++h) {
      SL kr[NB];
#pragma unroll
      for (int x = 0; x < NB; ++x) {
        const int j = __shfl_sync(0xffffffffu, j_mine, G * (h * NB + x) + grp);
        kr[x] = j >= 0 ? SL::load(p.k, kv_head + (int64_t)j * D + gl * E) : SL::zero();
      }
#pragma unroll
      for (int x = 0; x < NB; ++x) {
        float kf[E];
        kr[x].unpack(kf);
        float s = qf[0] * kf[0];
#pragma unroll
        for (int e = 1; e < E; ++e) s = fmaf(qf[e], kf[e], s);
        part[h * NB + x] = s;
      }
    }
    // reduce-scatter over the LPR lanes of each group: after the step with
    // offset o, a lane keeps the half of its values selected by bit o of gl,
    // summed with its partner's copy of that half; lane (grp, gl) ends with
    // the full score of round gl, i.e. of the key G gl + grp
#pragma unroll
    for (int o = R / 2; o > 0; o >>= 1) {
      const bool upper = (gl & o) != 0;
#pragma unroll
      for (int i = 0; i < o; ++i) {
        const float send = upper ? part[i] : part[i + o];
        const float keep = upper ? part[i + o] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    const int j_key = __shfl_sync(0xffffffffu, j_mine, G * gl + grp);
    const float s = j_key >= 0 ? part[0] : -INFINITY;
    // online softmax: the reference maximum moves only upwards, with the
    // accumulator and the partial sum rescaled when it does
    const float m_grp = warp_max(s);
    if (m_grp > m_run) {
      const float alpha = exp2f(m_run - m_grp);  // 0 while nothing was accumulated
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= alpha;
      l_lane *= alpha;
      m_run = m_grp;
    }
    const float pw = (m_run == -INFINITY) ? 0.f : exp2f(s - m_run);
    l_lane += pw;
    // weighted value rows: the group's key of round x, whose probability sits
    // in lane grp LPR + x
#pragma unroll
    for (int h = 0; h < R / NB; ++h) {
      SL vr[NB];
#pragma unroll
      for (int x = 0; x < NB; ++x) {
        const int j = __shfl_sync(0xffffffffu, j_mine, G * (h * NB + x) + grp);
        vr[x] = j >= 0 ? SL::load(p.v, kv_head + (int64_t)j * D + gl * E) : SL::zero();
      }
#pragma unroll
      for (int x = 0; x < NB; ++x) {
        const float pj = __shfl_sync(0xffffffffu, pw, grp * LPR + h * NB + x);
        float vf[E];
        vr[x].unpack(vf);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(pj, vf[e], acc[e]);
      }
    }
  }
  // the groups hold the weighted sums of different keys
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  const float l = warp_sum(l_lane);
  const float inv = l > 0.f ? 1.f / l : 0.f;  // a row with no valid entry gives 0
  if (grp == 0) {
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = acc[e] * inv;
    SL::store(p.out, row * D + gl * E, o);
  }
  if (p.lse && lane == 0)
    p.lse[row] = l > 0.f ? (m_run + log2f(l)) * 0.6931471805599453f : -INFINITY;
}

template <typename T>
cudaError_t launch_typed(const GatherProblem &p, cudaStream_t s) {
  const int64_t blocks = (p.rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  if (p.D == 64)
    gather_attention_kernel<T, 64, kLanesPerRow<T, 64>><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, s>>>(p);
  else
    gather_attention_kernel<T, 128, kLanesPerRow<T, 128>><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_attention(const GatherProblem &p, sa_dtype dt, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  return dt == SA_BF16 ? launch_typed<__nv_bfloat16>(p, s) : launch_typed<float>(p, s);
}

}  // namespace sa
