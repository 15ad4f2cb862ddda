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
//  * one warp per query row; a key or value row is read by the whole warp in
//    one coalesced load (lane l holds elements [E l, E l + E), E = D / 32);
//  * keys are taken 32 at a time (one list entry per lane), their rows loaded
//    16 at a time with all loads in flight before the first use, kept packed
//    so that four blocks of eight warps fit on an SM (enough loads in flight
//    to keep the memory system busy);
//  * the 32 per-lane partial dot products of a group are summed by a
//    reduce-scatter butterfly (31 shuffles), after which lane l holds the score
//    of the group's key l -- no per-key warp reduction;
//  * online softmax in base 2 with fp32 state: the running maximum is a warp
//    maximum per group, each lane keeps a partial row sum, the value rows are
//    weighted with each key's probability broadcast from its lane.
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

// Output row chunks (lane l writes elements [E l, E l + E) of its row).
template <typename T, int E>
struct OutChunk;
template <>
struct OutChunk<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void store(void *base, int64_t elem, const float (&x)[4]) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(base) + elem) = u;
  }
};
template <>
struct OutChunk<__nv_bfloat16, 2> {
  static __device__ __forceinline__ void store(void *base, int64_t elem, const float (&x)[2]) {
    *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(base) + elem) =
        __floats2bfloat162_rn(x[0], x[1]);
  }
};
template <>
struct OutChunk<float, 4> {
  static __device__ __forceinline__ void store(void *base, int64_t elem, const float (&x)[4]) {
    *reinterpret_cast<float4 *>(static_cast<float *>(base) + elem) = make_float4(x[0], x[1], x[2], x[3]);
  }
};
template <>
struct OutChunk<float, 2> {
  static __device__ __forceinline__ void store(void *base, int64_t elem, const float (&x)[2]) {
    *reinterpret_cast<float2 *>(static_cast<float *>(base) + elem) = make_float2(x[0], x[1]);
  }
};

// Row chunks as loaded (packed: bf16 pairs stay packed until used, so that a
// batch of loads in flight costs half the registers).
template <typename T, int E>
struct Raw;
template <>
struct Raw<__nv_bfloat16, 4> {
  using type = uint2;
  static __device__ __forceinline__ type load(const void *b, int64_t e) {
    return __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(b) + e));
  }
  static __device__ __forceinline__ type zero() { return make_uint2(0u, 0u); }
  static __device__ __forceinline__ void unpack(type u, float (&x)[4]) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    x[0] = a.x;
    x[1] = a.y;
    x[2] = c.x;
    x[3] = c.y;
  }
};
template <>
struct Raw<__nv_bfloat16, 2> {
  using type = uint32_t;
  static __device__ __forceinline__ type load(const void *b, int64_t e) {
    return __ldg(reinterpret_cast<const unsigned int *>(static_cast<const __nv_bfloat16 *>(b) + e));
  }
  static __device__ __forceinline__ type zero() { return 0u; }
  static __device__ __forceinline__ void unpack(type u, float (&x)[2]) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
    x[0] = a.x;
    x[1] = a.y;
  }
};
template <>
struct Raw<float, 4> {
  using type = float4;
  static __device__ __forceinline__ type load(const void *b, int64_t e) {
    return __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(b) + e));
  }
  static __device__ __forceinline__ type zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  static __device__ __forceinline__ void unpack(type u, float (&x)[4]) {
    x[0] = u.x;
    x[1] = u.y;
    x[2] = u.z;
    x[3] = u.w;
  }
};
template <>
struct Raw<float, 2> {
  using type = float2;
  static __device__ __forceinline__ type load(const void *b, int64_t e) {
    return __ldg(reinterpret_cast<const float2 *>(static_cast<const float *>(b) + e));
  }
  static __device__ __forceinline__ type zero() { return make_float2(0.f, 0.f); }
  static __device__ __forceinline__ void unpack(type u, float (&x)[2]) {
    x[0] = u.x;
    x[1] = u.y;
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

template <typename T, int D>
__global__ void __launch_bounds__(32 * kWarpsPerBlock, 4) gather_attention_kernel(GatherProblem p) {
  constexpr int E = D / 32;  // row elements per lane
  using RW = Raw<T, E>;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= p.rows) return;  // whole warps only: the warp's lanes share `row`
  const int64_t bh = row / p.Nq;
  const int64_t kv_head = bh * (int64_t)p.Nk * D;  // first element of this head's keys / values
  const int32_t *list = p.idx + row * (int64_t)p.K;

  float qf[E];
  RW::unpack(RW::load(p.q, row * D + lane * E), qf);
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
    // partial dot products of this lane's elements with the group's 32 keys
    float part[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      typename RW::type kr[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const int j = __shfl_sync(0xffffffffu, j_mine, h * 16 + x);
        kr[x] = j >= 0 ? RW::load(p.k, kv_head + (int64_t)j * D + lane * E) : RW::zero();
      }
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        float kf[E];
        RW::unpack(kr[x], kf);
        float s = qf[0] * kf[0];
#pragma unroll
        for (int e = 1; e < E; ++e) s = fmaf(qf[e], kf[e], s);
        part[h * 16 + x] = s;
      }
    }
    // reduce-scatter over the lanes: after the step with offset o, a lane keeps
    // the half of its values selected by bit o of its lane id, summed with its
    // partner's copy of that half; lane l ends with key l's full sum
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < o; ++i) {
        const float send = upper ? part[i] : part[i + o];
        const float keep = upper ? part[i + o] : part[i];
        part[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    const float s = j_mine >= 0 ? part[0] : -INFINITY;
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
    // weighted value rows
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      typename RW::type vr[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const int j = __shfl_sync(0xffffffffu, j_mine, h * 16 + x);
        vr[x] = j >= 0 ? RW::load(p.v, kv_head + (int64_t)j * D + lane * E) : RW::zero();
      }
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const float pj = __shfl_sync(0xffffffffu, pw, h * 16 + x);
        float vf[E];
        RW::unpack(vr[x], vf);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(pj, vf[e], acc[e]);
      }
    }
  }
  const float l = warp_sum(l_lane);
  const float inv = l > 0.f ? 1.f / l : 0.f;  // a row with no valid entry gives 0
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = acc[e] * inv;
  OutChunk<T, E>::store(p.out, row * D + lane * E, o);
  if (p.lse && lane == 0)
    p.lse[row] = l > 0.f ? (m_run + log2f(l)) * 0.6931471805599453f : -INFINITY;
}

template <typename T>
cudaError_t launch_typed(const GatherProblem &p, cudaStream_t s) {
  const int64_t blocks = (p.rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  if (p.D == 64)
    gather_attention_kernel<T, 64><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, s>>>(p);
  else
    gather_attention_kernel<T, 128><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_attention(const GatherProblem &p, sa_dtype dt, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  return dt == SA_BF16 ? launch_typed<__nv_bfloat16>(p, s) : launch_typed<float>(p, s);
}

}  // namespace sa
