// sa_tc.cu -- tensor-core kernels (sm_103a: TMA, mbarrier, tcgen05 + TMEM):
// the band-tile kernel and the global-row split-K kernel, for bf16 inputs
// (kind::f16) and for fp32 inputs with tf32 products (kind::tf32, D = 64).
//
// What one CTA computes (Unlimiformer section 2.3 Eq. (1) under the additive
// {0,-inf} mask of GMAT's "Global-Memory Augmented Transformers" section):
// two 128-row query tiles Q_0, Q_1, each against its own list of key tiles --
// the band tiles that intersect its rows' windows (Longformer glossary, "How
// the Longformer attention works": sliding / dilated window) followed by the
// global keys (the same section's global attention; GMAT "Global Memory") --
// with an exact online softmax in fp32.  The two query tiles are neighbours, so
// their band lists overlap and each key/value tile is loaded once for both.
// The global rows are read from gathered copies, or in place through views of
// q, k, v when they are contiguous.
//
//   S = Q_u K_j^T (fp32 in TMEM; Q negated for a negative scale) -> mask (edge
//   tiles only), running max / sum per row -> P = exp2(scale S - m) written
//   back over S (bf16 pairs, or fp32 for tf32) -> O_u += P V_j (A operand from
//   TMEM).  Band CTAs take each key tile as two 64-key sub-tiles whose S
//   products alternate between the two halves of S_u's columns: the S of the
//   next sub-tile is computed while the softmax works on the current one
//   (its P sits in the other half), so a query tile's softmax does not wait
//   for its own P V before the next scores exist.  Global-row CTAs take
//   whole 128-key tiles, P written over S in two halves, the first half of
//   P V starting once the first half of P is in place.  tf32 operands must be
//   K-major, so for fp32 inputs the values arrive transposed (32-key chunks
//   of D rows).
//
// In global mode the two query tiles are the gathered global rows and the key
// tiles one chunk of all N keys; the CTA writes unnormalised partial outputs
// and their (max, sum) for the merge kernel.
//
// The kernel is persistent: one CTA per SM walks the launch's work items with
// a grid stride, keeping its barriers, TMEM and key/value ring across items,
// so the next item's Q load and first MMAs overlap the current item's tail.
//
// Warp roles (352 threads): warps 0-3 softmax of Q_0 (one thread per row; they
// also normalise and stage the finished rows), warps 4-7 softmax of Q_1, warp 8
// TMA producers (lane 0 keys/values; lane 1 queries, and the TMA store of each
// staged output tile), warp 9 MMA issuer of Q_0 (and TMEM allocator), warp 10
// MMA issuer of Q_1.  TMEM: S_0 cols [0,128), S_1 [128,256), O_0 [256,256+D),
// O_1 [384,384+D).  Shared memory: three query-tile buffers (used in rotation,
// so the next item's first query tile can land while both current ones are in
// use; a finished output tile is staged in its query tile's buffer), then a
// ring of key/value slots (one K or V tile each), then barriers.  All tiles use
// the 128-byte swizzle that TMA writes and the UMMA descriptors read.
//
// Every wait on an mbarrier is bounded: after kWaitLimitNs the waiting thread
// sets the CTA's abort flag and the device error word, and every role winds
// down (no trap, no endless spin).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "sa_tc.h"
#include "sa_tmem_ops.h"

#ifndef SA_DEBUG
#define SA_DEBUG 0
#endif
#if SA_DEBUG
#include "sa_debug.h"
#endif

namespace sa {
namespace tc {

constexpr int kThreads = 352;     // eleven warps (three on some sub-partitions): 168 registers
constexpr int kRows = 128;         // query rows per tile (TMEM lanes)
constexpr int kKeys = 128;         // keys per band tile
constexpr int kGKeys = 64;         // keys per global tile
constexpr int kMaxSlotsPerLaunch = 16;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kTmemCols = 512;
constexpr int kFarAway = -(1 << 30);  // class coordinate of a global outside the class
constexpr bool kGlobalsFirst = false;  // global key tiles before (or after) the band tiles

struct Maps {
  CUtensorMap q[kMaxSlotsPerLaunch], k[kMaxSlotsPerLaunch], v[kMaxSlotsPerLaunch],
      o[kMaxSlotsPerLaunch];
  CUtensorMap kg, vg;  // gathered global keys / values, 64-row boxes
  CUtensorMap qg;      // gathered global queries, 128-row boxes
  CUtensorMap qg64;    // the same, 64-row boxes (a query tile packed with two copies)
  CUtensorMap kp, vp;  // plain (undilated) keys / values, 128-row boxes
};

struct Params {
  Maps maps;
  DevProblem p;
  int slot_base;    // slot index held in maps.q[0]
  int item_offset;  // first band work item of this launch
  int n_items;      // band work items of this launch (band CTAs stride over them)
  int n_gctas;      // CTAs 0 .. n_gctas-1 run the global-row items instead
  int n_gitems;     // global-row work items (those CTAs stride over them)
};

// TF: fp32 inputs on the tensor cores as tf32 (kind::tf32), else bf16 (kind::f16).
template <int D, bool TF>
struct Cfg {
  static constexpr int kElem = TF ? 4 : 2;             // bytes per input element
  static constexpr int kQBytes = kRows * D * kElem;    // one query tile
  static constexpr int kSlotBytes = kKeys * D * kElem; // one key or value tile
  static constexpr int kHalfCols = 128 / kElem;        // elements per 128-byte row
  static constexpr int kHalves = D / kHalfCols;
  static constexpr int kMmaK = 32 / kElem;             // K of one MMA (32 bytes of a row)
  static constexpr int kAux = 3072;  // barriers, flags, global positions (class coordinates)
  static constexpr int kSmemMax = 232448;
  static constexpr int kQBufs = 3;   // query tiles rotate through three buffers
  static constexpr int kSlots0 = (kSmemMax - kQBufs * kQBytes - kAux) / kSlotBytes;
  static constexpr int kSlots = kSlots0 > 12 ? 12 : kSlots0;
  static constexpr int kSmemBytes = kQBufs * kQBytes + kSlots * kSlotBytes + kAux;
  static_assert(kSlots >= 4, "the key/value ring needs at least four slots");
  // query buffers and ring together; a global-row CTA with one query buffer
  // fits (kRegion - kQBytes) / kSlotBytes slots, at most kMaxSlots
  static constexpr int kRegion = kQBufs * kQBytes + kSlots * kSlotBytes;
  static constexpr int kMaxSlots0 = (kRegion - kQBytes) / kSlotBytes;
  static constexpr int kMaxSlots = kMaxSlots0 > 12 ? 12 : kMaxSlots0;
};

// ---------------------------------------------------------------------------
// PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking check of a barrier phase.  Several polls issued back to back
// overlap their latency (~80 cycles each), unlike a chain of waits.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait.  Returns false (and leaves the abort flag set) if the CTA is
// aborting or the limit ran out.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      int *err, bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (honour_abort && err && (*(volatile int *)err & kErrWaitTimeout)) {
        *abort_flag = 1;
        return false;
      }
      if (global_timer() - start > kWaitLimitNs) {
        *abort_flag = 1;
        if (err) atomicOr(err, kErrWaitTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y,
                                             int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// AND of `v` over the `threads` threads that reach named barrier `id`.
__device__ __forceinline__ bool named_bar_and(int id, int threads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n"
      ".reg .pred p, q;\n"
      "setp.ne.u32 p, %1, 0;\n"
      "bar.red.and.pred q, %2, %3, p;\n"
      "selp.u32 %0, 1, 0, q;\n"
      "}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Issue forms for a converged warp: elect.sync picks one lane, which issues the
// tcgen05 operation (a converged warp with warp-uniform operands issues MMAs at
// about twice the rate of a single diverged lane).
template <bool TF>
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  if constexpr (TF)
    asm volatile(
        "{\n"
        ".reg .pred p, e;\n"
        ".reg .b32 r;\n"
        "elect.sync r|e, 0xffffffff;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n"
        ".reg .pred p, e;\n"
        ".reg .b32 r;\n"
        "elect.sync r|e, 0xffffffff;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
template <bool TF>
__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  if constexpr (TF)
    asm volatile(
        "{\n"
        ".reg .pred p, e;\n"
        ".reg .b32 r;\n"
        "elect.sync r|e, 0xffffffff;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n"
        ".reg .pred p, e;\n"
        ".reg .b32 r;\n"
        "elect.sync r|e, 0xffffffff;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n"
      ".reg .pred e;\n"
      ".reg .b32 r;\n"
      "elect.sync r|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
      "}\n" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
  asm volatile(
      "{\n"
      ".reg .pred e;\n"
      ".reg .b32 r;\n"
      "elect.sync r|e, 0xffffffff;\n"
      "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n"
      "}\n" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// Residual of a bf16 pair: (lo - bf16(lo), hi - bf16(hi)) rounded to bf16
// pairs again, where `packed` = pack_bf16(lo, hi).  bf16(x) + residual carries
// 16 significant bits of x.
__device__ __forceinline__ uint32_t pack_bf16_residual(float lo, float hi, uint32_t packed) {
  return pack_bf16(lo - __uint_as_float(packed << 16), hi - __uint_as_float(packed & 0xffff0000u));
}

// UMMA shared-memory descriptor, 128-byte swizzle (SM100 layout, version 1).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor: bf16 x bf16 (kind::f16, type 1) or tf32 x tf32
// (kind::tf32, type 2) -> fp32, M x N, A K-major, B K- or MN-major.
__host__ __device__ constexpr uint32_t idesc_mma(int M, int N, bool b_mn_major, bool tf32) {
  return (1u << 4) | ((tf32 ? 2u : 1u) << 7) | ((tf32 ? 2u : 1u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Key tiles a global-row item keeps in flight to L2 ahead of its loads.
constexpr int kGlobalAhead = 6;

// L2 prefetch of the key and value tile starting at row y (128 rows).
template <typename C>
__device__ __forceinline__ void prefetch_kv(const CUtensorMap *mk, const CUtensorMap *mv, int y,
                                            int bh) {
  for (int h = 0; h < C::kHalves; ++h) tma_prefetch_3d(mk, C::kHalfCols * h, y, bh);
  if (C::kElem == 4) {
    // transposed values (tf32): boxes of 32 keys
    for (int c = 0; c < kKeys / 32; ++c) tma_prefetch_3d(mv, y + 32 * c, 0, bh);
  } else {
    for (int h = 0; h < C::kHalves; ++h) tma_prefetch_3d(mv, C::kHalfCols * h, y, bh);
  }
}

// ---------------------------------------------------------------------------
// work description shared by all roles of one CTA

struct Work {
  int bh;
  int slot;      // residue-class slot (band mode)
  int d, r, len; // residue class: positions r + d*t, t < len (band mode)
  int q_tile;    // first query tile (band mode)
  int flags;     // bit u: global tile of query tile u needs the in-band test
  int lo;        // first band tile of the CTA's list
  int nb;        // band tiles in the list
  int ng;        // global tiles in the list
  int n_lo[2], n_cnt[2];  // per query tile: first band tile, band tile count
  int active[2];
  int key0;      // global mode: first key of the chunk
  int key_end;   // global mode: one past the chunk's last key
  int chunk;
  int g_tile;    // global mode: pair of 128-row tiles of the gathered global rows
};

#if SA_DEBUG
// Range checks of the work descriptions (SA_DEBUG builds): a band item's
// residue class lies in the problem's classes and in this launch's window of
// kMaxSlotsPerLaunch tensor maps, its head in [0, BH), its query tile and
// every key-tile range it lists inside the class; a global-row item's head,
// key chunk and tile of global rows inside the problem.
__device__ __forceinline__ bool band_item_in_range(const BandItem &it, const Slot *slots, int n_slots,
                                                   int slot_base, int BH) {
  const int ls = it.slot - slot_base;
  if (it.slot < 0 || it.slot >= n_slots || ls < 0 || ls >= kMaxSlotsPerLaunch) return false;
  if (it.bh < 0 || it.bh >= BH) return false;
  const Slot sl = slots[it.slot];
  if (it.q_tile < 0 || (int64_t)it.q_tile * kRows >= sl.len) return false;
  for (int u = 0; u < 2; ++u)
    if (it.k_hi[u] >= it.k_lo[u] && (it.k_lo[u] < 0 || (int64_t)it.k_hi[u] * kKeys >= sl.len)) return false;
  return true;
}
__device__ __forceinline__ bool global_item_in_range(const GlobalItem &it, const DevProblem &p) {
  return it.bh >= 0 && it.bh < p.BH && it.chunk >= 0 && it.chunk < p.n_chunks && it.g_tile >= 0 &&
         (int64_t)it.g_tile * 2 * kRows < p.g_pad;
}
#endif

template <bool GLOBAL>
__device__ __forceinline__ Work make_work(const Params &P, int item) {
  Work w{};
  const DevProblem &p = P.p;
  if (!GLOBAL) {
    const BandItem it = p.band[P.item_offset + item];
#if SA_DEBUG
    if (!band_item_in_range(it, p.slots, p.n_slots, P.slot_base, p.BH)) {
      // no tiles and no rows: every role skips the item
      if (p.err) atomicOr(p.err, kErrBadWork);
      return w;
    }
#endif
    const Slot sl = p.slots[it.slot];
    w.bh = it.bh;
    w.slot = it.slot;
    w.d = sl.d;
    w.r = sl.r;
    w.len = sl.len;
    w.q_tile = it.q_tile;
    w.flags = it.flags;
    int lo = 0x7fffffff, hi = -1;
    for (int u = 0; u < 2; ++u) {
      w.active[u] = it.k_hi[u] >= it.k_lo[u];
      w.n_lo[u] = it.k_lo[u];
      w.n_cnt[u] = w.active[u] ? it.k_hi[u] - it.k_lo[u] + 1 : 0;
      if (w.active[u]) {
        lo = min(lo, it.k_lo[u]);
        hi = max(hi, it.k_hi[u]);
      }
    }
    w.lo = hi >= 0 ? lo : 0;
    w.nb = hi - w.lo + 1;
    w.ng = (p.n_g + kGKeys - 1) / kGKeys;
  } else {
    const GlobalItem it = p.gitems[item];
#if SA_DEBUG
    if (!global_item_in_range(it, p)) {
      if (p.err) atomicOr(p.err, kErrBadWork);
      return w;
    }
#endif
    w.bh = it.bh;
    w.chunk = it.chunk;
    w.g_tile = it.g_tile;
    w.key0 = it.chunk * p.chunk_len;
    w.key_end = min(p.N, w.key0 + p.chunk_len);
    w.lo = 0;
    w.nb = (w.key_end - w.key0 + kKeys - 1) / kKeys;
    w.ng = 0;
    for (int u = 0; u < 2; ++u) {
      w.n_lo[u] = 0;
      if (p.g_alt) {
        // one tile of global rows; query tile u takes the key tiles u, u+2, ...
        w.active[u] = w.nb > u;
        w.n_cnt[u] = (w.nb - u + 1) / 2;
      } else {
        w.active[u] = (it.g_tile * 2 + u) * kRows < p.n_g;
        w.n_cnt[u] = w.active[u] ? w.nb : 0;
      }
    }
  }
  return w;
}

// First row of query tile u in its tensor map (class coordinate, or row of the
// gathered global rows).
template <bool GLOBAL>
__device__ __forceinline__ int q_row_of(const Params &P, const Work &w, int u) {
  if (GLOBAL) return (w.g_tile * 2 + (P.p.g_alt ? 0 : u)) * kRows;
  return (w.q_tile + u) * kRows;
}
template <bool GLOBAL>
__device__ __forceinline__ const CUtensorMap *map_q_of(const Params &P, const Work &w) {
  return GLOBAL ? &P.maps.qg : &P.maps.q[w.slot - P.slot_base];
}

// Position in the CTA's tile list of the i-th tile of a query tile whose band
// tiles start at n_lo (n_cnt of them).
__device__ __forceinline__ int seq_pos_s(const Work &w, int n_lo, int n_cnt, int i) {
  if (kGlobalsFirst) return i < w.ng ? i : w.ng + (n_lo - w.lo) + (i - w.ng);
  return i < n_cnt ? (n_lo - w.lo + i) : (w.nb + (i - n_cnt));
}
// Is position pos of the item's tile list a global tile, and which band tile
// (or global tile) is it?
__device__ __forceinline__ bool is_global_pos(const Work &w, int pos) {
  return kGlobalsFirst ? pos < w.ng : pos >= w.nb;
}
__device__ __forceinline__ int band_index(const Work &w, int pos) {
  return kGlobalsFirst ? pos - w.ng : pos;
}
__device__ __forceinline__ int global_index(const Work &w, int pos) {
  return kGlobalsFirst ? pos : pos - w.nb;
}
__device__ __forceinline__ int seq_len(const Work &w, int u) {
  return w.active[u] ? w.n_cnt[u] + w.ng : 0;
}
struct Bars {
  uint32_t slot_full, slot_empty;  // arrays of kSlots
  uint32_t q_full, q_empty;  // arrays of kQBufs
  uint32_t s_full, p_half, p_full, o_final, mma_done, s_issued, pv_done;  // arrays of 2
  // band sub-tiles: S complete and P written, per chain and S half ([2 u + half])
  uint32_t s_sub, p_sub;
};

// ---------------------------------------------------------------------------
// softmax: one key tile of W columns for one row

// Masking of one key tile's scores (base-2 units; the scale's sign is applied
// by the S product itself, which negates Q when the scale is negative, so the
// softmax only ever sees a positive scale):
//   every column is kept, or, when `interval` is set, columns [c_lo, c_hi]
//   only (the window's edge tiles; a global tile keeps columns [0, c_hi], the
//   globals it holds).  With `dedup`, a global tile also drops the globals
//   already in the row's band (globals[g0 + x] is the global's class
//   coordinate t_g, or kFarAway; the row is class position t_q; the global is
//   in the row's band when |t_q - t_g| <= half, and is then counted once, as a
//   band key).  One code path serves band and global tiles alike: the kernel's
//   code has to stay small enough for the instruction caches of warps that
//   run different roles on one sub-partition.

// W (128 or 64) scores of this thread's row from TMEM, masked to -inf.
template <int W>
__device__ __forceinline__ void load_scores(uint32_t t_s, bool interval, int c_lo, int c_hi,
                                            const int32_t *globals, int g0, int t_q, int half,
                                            bool dedup, float (&s)[W]) {
  {
    uint32_t r[W];
    if constexpr (W == 128)
      tmem_ld128(t_s, r);
    else
      tmem_ld64(t_s, r);
#pragma unroll
    for (int x = 0; x < W; ++x) s[x] = __uint_as_float(r[x]);
  }
  // branch-free: a compare and a select per column (the bounds differ per row)
  if (interval) {
    const uint32_t span = (uint32_t)(c_hi - c_lo);
#pragma unroll
    for (int x = 0; x < W; ++x) {
      const bool keep = (uint32_t)(x - c_lo) <= span;  // c_lo <= x <= c_hi
      s[x] = keep ? s[x] : -INFINITY;
    }
  }
  if (dedup) {
    const uint32_t band = 2u * (uint32_t)half;
#pragma unroll
    for (int x = 0; x < kGKeys; ++x) {
      // |t_q - t_g| > half, i.e. t_q - t_g + half outside [0, 2 half]; kFarAway
      // (a global outside the class) is never in band
      const bool out_of_band = (uint32_t)(t_q - globals[g0 + x] + half) > band;
      s[x] = out_of_band ? s[x] : -INFINITY;
    }
  }
}

// One key tile for one query row (this thread's TMEM lane): P =
// 2^(scale*S - m) as bf16 written over S, running maximum m and row sum l
// updated, O in TMEM rescaled when the reference maximum moves.  The reference
// maximum is raised only when the tile maximum exceeds it by more than 2^8, so
// O is rescaled rarely; the same reference is used for P and for the running
// sum, so the result is exact either way.  P (bf16 pairs, or fp32 for fp32
// inputs) is written over S in two halves of 64 keys and the first is announced
// on bar_half, so that the first half of P V
// can start while the second half of P is computed; a global tile has 64 keys
// (`narrow`) and only its first half is computed.
template <int D, bool TF, bool PRECISE>
__device__ __forceinline__ void softmax_tile(uint32_t t_s, uint32_t t_o, float scale, bool interval,
                                             int c_lo, int c_hi, const int32_t *globals, int g0,
                                             int t_q, int half, bool dedup, bool narrow,
                                             uint32_t bar_half, int lane, float &m_run,
                                             float &l_run) {
  constexpr int W = kKeys;
  const float scl = scale;
  float s[W];
  load_scores<W>(t_s, interval, c_lo, c_hi, globals, g0, t_q, half, dedup, s);
  // row maximum: eight chains of three-input max
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
  for (int x = 16; x < W; x += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i) mx[i] = max3(mx[i], s[x + 2 * i], s[x + 2 * i + 1]);
  const float mt =
      max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * scl;
  const bool need = mt > m_run + 8.f;
  const float m_new = need ? mt : m_run;
  const float alpha = need ? ex2(m_run - m_new) : 1.f;
  const bool rescale = need && m_run != -INFINITY;  // O holds earlier tiles of this row
  if (__any_sync(0xffffffffu, rescale)) {
    // O holds the previous tiles (their PV was issued before this tile's S,
    // whose completion has been observed); bring it to the new reference
    // before any of this tile's P can be multiplied into it
    const float a = rescale ? alpha : 1.f;
#pragma unroll 1
    for (int c = 0; c < D / 16; ++c) {
      uint32_t r[16];
      tmem_ld16(t_o + c * 16, r);
#pragma unroll
      for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * a);
      tmem_st16(t_o + c * 16, r);
    }
  }
  // P: the argument two columns at a time (packed fp32x2 FMA), the exponential
  // on the SFU, row sums in four packed accumulators
  const float neg = (m_new == -INFINITY) ? 0.f : -m_new;
  const float2 scl2 = make_float2(scl, scl), neg2 = make_float2(neg, neg);
  float2 sum2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) sum2[i] = make_float2(0.f, 0.f);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    if (hh == 1 && narrow) break;
    // bf16 P: two keys per TMEM column; tf32 P (fp32 inputs): one
    constexpr int kWords = TF ? W / 2 : W / 4;
    if constexpr (PRECISE) {
      // P = P_hi + P_lo, both bf16 (P_lo in the columns 64 on, free once S
      // has been read): the P V product runs over both parts, so the weights
      // it multiplies carry 16 bits, as the row sum does
      static_assert(!TF, "split P is for bf16 inputs");
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int i = hh * (W / 4) + qq * 16 + j;
          const float2 arg = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), scl2, neg2);
          const float2 e = make_float2(ex2(arg.x), ex2(arg.y));
          sum2[i & 3] = __fadd2_rn(sum2[i & 3], e);
          ph[j] = pack_bf16(e.x, e.y);
          pl[j] = pack_bf16_residual(e.x, e.y, ph[j]);
        }
        tmem_st16(t_s + hh * kWords + qq * 16, ph);
        tmem_st16(t_s + 64 + hh * kWords + qq * 16, pl);
      }
    } else {
      uint32_t pr[kWords];
#pragma unroll
      for (int j = 0; j < W / 4; ++j) {
        const int i = hh * (W / 4) + j;
        const float2 arg = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), scl2, neg2);
        const float2 e = make_float2(ex2(arg.x), ex2(arg.y));
        sum2[i & 3] = __fadd2_rn(sum2[i & 3], e);
        if constexpr (TF) {
          pr[2 * j] = __float_as_uint(e.x);
          pr[2 * j + 1] = __float_as_uint(e.y);
        } else {
          pr[j] = pack_bf16(e.x, e.y);
        }
      }
      if constexpr (TF)
        tmem_st64(t_s + hh * kWords, pr);
      else
        tmem_st32(t_s + hh * kWords, pr);
    }
    if (hh == 0) {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_half);
    }
  }
  const float2 s01 = __fadd2_rn(sum2[0], sum2[1]), s23 = __fadd2_rn(sum2[2], sum2[3]);
  const float2 s4 = __fadd2_rn(s01, s23);
  l_run = (need ? l_run * alpha : l_run) + (s4.x + s4.y);
  m_run = m_new;
}

// P of a 64-key sub-tile that this thread's row does not score: zeros, so
// that the sub-tile's P V product adds nothing to the row.
template <bool TF, bool PRECISE>
__device__ __forceinline__ void zero_p_sub(uint32_t t_s) {
  if constexpr (TF) {
    uint32_t z[64];
#pragma unroll
    for (int x = 0; x < 64; ++x) z[x] = 0u;
    tmem_st64(t_s, z);
  } else {
    uint32_t z[32];
#pragma unroll
    for (int x = 0; x < 32; ++x) z[x] = 0u;
    tmem_st32(t_s, z);
    if constexpr (PRECISE) tmem_st32(t_s + 32, z);
  }
}

// One 64-key sub-tile of a band item for one query row (this thread's TMEM
// lane).  The scores sit in one half of the tile's S columns (t_s .. t_s+63);
// P = 2^(scale*S - m) is written over the first columns of that half (bf16
// pairs in 32 columns, the low parts of split P in the next 32; tf32 in all
// 64), where only this sub-tile's P V reads it, so the S product of the
// sub-tile after next -- the other half holds the next one -- can run while
// this P is computed.  Running maximum and sum as in softmax_tile.  O is
// rescaled when the reference maximum moves, after the previous sub-tile's
// P V has completed: its commit is phase `pv_parity` of `pv_done` (the P V
// before that one completed before this sub-tile's S, which follows it in
// issue order, so the barrier is at most one phase behind).  Returns false
// if that wait gave up.
template <int D, bool TF, bool PRECISE>
__device__ __forceinline__ bool softmax_sub(uint32_t t_s, uint32_t t_o, float scale, bool interval,
                                            int c_lo, int c_hi, const int32_t *globals, int g0,
                                            int t_q, int half, bool dedup, uint32_t pv_done,
                                            uint32_t pv_parity, volatile int *abort_flag,
                                            int *err, float &m_run, float &l_run) {
  constexpr int W = kKeys / 2;
  const float scl = scale;
  float s[W];
  load_scores<W>(t_s, interval, c_lo, c_hi, globals, g0, t_q, half, dedup, s);
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
  for (int x = 16; x < W; x += 16)
#pragma unroll
    for (int i = 0; i < 8; ++i) mx[i] = max3(mx[i], s[x + 2 * i], s[x + 2 * i + 1]);
  const float mt =
      max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * scl;
  const bool need = mt > m_run + 8.f;
  const float m_new = need ? mt : m_run;
  const float alpha = need ? ex2(m_run - m_new) : 1.f;
  const bool rescale = need && m_run != -INFINITY;  // O holds earlier sub-tiles of this row
  const float neg = (m_new == -INFINITY) ? 0.f : -m_new;
  const float2 scl2 = make_float2(scl, scl), neg2 = make_float2(neg, neg);
  float2 sum2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) sum2[i] = make_float2(0.f, 0.f);
  if constexpr (PRECISE) {
    static_assert(!TF, "split P is for bf16 inputs");
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      uint32_t ph[16], pl[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int i = qq * 16 + j;
        const float2 arg = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), scl2, neg2);
        const float2 e = make_float2(ex2(arg.x), ex2(arg.y));
        sum2[i & 3] = __fadd2_rn(sum2[i & 3], e);
        ph[j] = pack_bf16(e.x, e.y);
        pl[j] = pack_bf16_residual(e.x, e.y, ph[j]);
      }
      tmem_st16(t_s + qq * 16, ph);
      tmem_st16(t_s + 32 + qq * 16, pl);
    }
  } else {
    constexpr int kWords = TF ? W : W / 2;
    uint32_t pr[kWords];
#pragma unroll
    for (int i = 0; i < W / 2; ++i) {
      const float2 arg = __ffma2_rn(make_float2(s[2 * i], s[2 * i + 1]), scl2, neg2);
      const float2 e = make_float2(ex2(arg.x), ex2(arg.y));
      sum2[i & 3] = __fadd2_rn(sum2[i & 3], e);
      if constexpr (TF) {
        pr[2 * i] = __float_as_uint(e.x);
        pr[2 * i + 1] = __float_as_uint(e.y);
      } else {
        pr[i] = pack_bf16(e.x, e.y);
      }
    }
    if constexpr (TF)
      tmem_st64(t_s, pr);
    else
      tmem_st32(t_s, pr);
  }
  bool ok = true;
  if (__any_sync(0xffffffffu, rescale)) {
    ok = __all_sync(0xffffffffu, wait_bar(pv_done, pv_parity, abort_flag, err));
    if (ok) {
      tc_fence_after();
      const float a = rescale ? alpha : 1.f;
#pragma unroll 1
      for (int c = 0; c < D / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(t_o + c * 16, r);
#pragma unroll
        for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * a);
        tmem_st16(t_o + c * 16, r);
      }
    }
  }
  const float2 s01 = __fadd2_rn(sum2[0], sum2[1]), s23 = __fadd2_rn(sum2[2], sum2[3]);
  const float2 s4 = __fadd2_rn(s01, s23);
  l_run = (need ? l_run * alpha : l_run) + (s4.x + s4.y);
  m_run = m_new;
  return ok;
}

template <int D, bool GLOBAL, bool TF, bool PRECISE>
__device__ __forceinline__ void cta_body(const Params &P, const int item0, const int stride,
                                         const int n_items) {
  using C = Cfg<D, TF>;
  const DevProblem &p = P.p;
  // Global-row CTAs whose global rows fit one query tile (g_alt) load that
  // tile once per item for both chains, and give the space of the other query
  // buffers to the key/value ring: their chains take alternate key tiles, so
  // they drain the ring twice as fast as band CTAs and need it deeper.
  const bool shared_q = GLOBAL && p.g_alt;
  const int NQ = GLOBAL ? (shared_q ? 1 : 2) : C::kQBufs;
  const int NS = GLOBAL ? min(C::kMaxSlots, (C::kRegion - NQ * C::kQBytes) / C::kSlotBytes) : C::kSlots;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw;
  const uint32_t s_q0 = smem_u32(smem);
  const uint32_t s_slots = s_q0 + NQ * C::kQBytes;
  uint8_t *aux = smem + C::kRegion;
  constexpr int kBars = 2 * C::kMaxSlots + 2 * C::kQBufs + 22;
  uint64_t *bar_mem = reinterpret_cast<uint64_t *>(aux);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(aux + 8 * kBars);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(aux + 8 * kBars + 4);
  int32_t *g_lists = reinterpret_cast<int32_t *>(aux + 1024);  // [2][SA_MAX_GLOBALS]
  static_assert(8 * kBars + 16 <= 1024 && 1024 + 8 * SA_MAX_GLOBALS <= C::kAux, "aux layout");
  Bars B;
  B.slot_full = smem_u32(bar_mem);
  B.slot_empty = B.slot_full + 8 * C::kMaxSlots;
  B.q_full = B.slot_empty + 8 * C::kMaxSlots;  // [NQ]
  B.q_empty = B.q_full + 8 * C::kQBufs;        // [NQ]
  B.s_full = B.q_empty + 8 * C::kQBufs;        // [2]
  B.p_half = B.s_full + 16;          // [2]
  B.p_full = B.p_half + 16;          // [2]
  B.o_final = B.p_full + 16;         // [2]
  B.mma_done = B.o_final + 16;       // [2]
  B.s_issued = B.mma_done + 16;      // [2]
  B.pv_done = B.s_issued + 16;       // [2]
  B.s_sub = B.pv_done + 16;          // [4]
  B.p_sub = B.s_sub + 32;            // [4]

  const int tid = threadIdx.x;
  if (s_q0 & 1023u) {  // 128-byte-swizzled tiles need 1024-byte alignment
    if (tid == 0 && p.err) atomicOr(p.err, kErrBadWork);
    return;
  }
  const int warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(B.slot_full + 8 * i, 1);
      // one arrival per MMA issuer; per reading issuer with alternating tiles
      mbar_init(B.slot_empty + 8 * i, shared_q ? 1 : 2);
    }
    for (int b = 0; b < NQ; ++b) {
      mbar_init(B.q_full + 8 * b, 1);
      // a shared query tile is released by both softmax warpgroups
      mbar_init(B.q_empty + 8 * b, shared_q ? 2 : 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(B.s_full + 8 * u, 1);
      mbar_init(B.p_half + 8 * u, 4);  // one arrival per softmax warp of the tile's warpgroup
      mbar_init(B.p_full + 8 * u, 4);
      mbar_init(B.o_final + 8 * u, 1);
      mbar_init(B.mma_done + 8 * u, 1);
      mbar_init(B.s_issued + 8 * u, 1);
      mbar_init(B.pv_done + 8 * u, 1);
      for (int h = 0; h < 2; ++h) {
        mbar_init(B.s_sub + 8 * (2 * u + h), 1);
        mbar_init(B.p_sub + 8 * (2 * u + h), 4);
      }
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 8 && lane == 1) {
    // ------------------------------------------------------------- Q producer
    // Query tiles are loaded in order (item by item, tile 0 then tile 1) into
    // the buffers 0, 1, 2, 0, ...; the next item's first query tile lands in
    // the spare buffer while the current item is still running, and the
    // following item's query rows are prefetched into L2.  The softmax
    // warpgroup stages each finished output tile in its query buffer; this
    // thread stores it with TMA when the buffer comes round again (or at the
    // end), so that no softmax warp waits for a store to read shared memory.
    {
      uint32_t j = 0;  // query tiles loaded so far
      bool ok = true;
      // output tile staged in each buffer: map index, first row, head
      int out_ls[C::kQBufs], out_row[C::kQBufs], out_bh[C::kQBufs];
      auto store_staged = [&](uint32_t b) {
        for (int h = 0; h < C::kHalves; ++h)
          tma_store_3d(&P.maps.o[out_ls[b]], s_q0 + b * C::kQBytes + h * (kRows * 128),
                       C::kHalfCols * h, out_row[b], out_bh[b]);  // rows past the class end are clipped
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      };
      for (int item = item0; item < n_items && ok; item += stride) {
        const Work w = make_work<GLOBAL>(P, item);
        if (item + stride < n_items) {
          const Work wn = make_work<GLOBAL>(P, item + stride);
          const CUtensorMap *mq = map_q_of<GLOBAL>(P, wn);
          for (int u = 0; u < 2; ++u)
            if (wn.active[u])
              for (int h = 0; h < C::kHalves; ++h)
                tma_prefetch_3d(mq, C::kHalfCols * h, q_row_of<GLOBAL>(P, wn, u), wn.bh);
        }
        const CUtensorMap *mq = map_q_of<GLOBAL>(P, w);
        if (shared_q) {
          // one tile of global rows for both chains
          const uint32_t b = j % NQ, use = j / NQ;
          if (!wait_bar(B.q_empty + 8 * b, (use & 1u) ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(B.q_full + 8 * b, C::kQBytes);
          if (p.g_packed) {
            for (int h = 0; h < C::kHalves; ++h)
              for (int c = 0; c < 2; ++c)
                tma_load_3d(s_q0 + b * C::kQBytes + h * (kRows * 128) + c * (kRows / 2) * 128,
                            &P.maps.qg64, B.q_full + 8 * b, C::kHalfCols * h, 0, w.bh);
          } else {
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_3d(s_q0 + b * C::kQBytes + h * (kRows * 128), mq, B.q_full + 8 * b,
                          C::kHalfCols * h, q_row_of<GLOBAL>(P, w, 0), w.bh);
          }
          ++j;
          continue;
        }
        for (int u = 0; u < 2 && ok; ++u) {
          if (!w.active[u]) continue;
          const uint32_t b = j % NQ, use = j / NQ;
          if (!wait_bar(B.q_empty + 8 * b, (use & 1u) ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          if (!GLOBAL && use > 0) {
            // the previous occupant's output tile is staged: store it, and
            // reload the buffer once the store has read it
            store_staged(b);
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          }
          if (!GLOBAL) {
            out_ls[b] = w.slot - P.slot_base;
            out_row[b] = (w.q_tile + u) * kRows;
            out_bh[b] = w.bh;
          }
          mbar_expect_tx(B.q_full + 8 * b, C::kQBytes);
          if (GLOBAL && p.g_packed) {
            // the (at most 64) global rows twice: rows 0-63 and 64-127 of the tile
            for (int h = 0; h < C::kHalves; ++h)
              for (int c = 0; c < 2; ++c)
                tma_load_3d(s_q0 + b * C::kQBytes + h * (kRows * 128) + c * (kRows / 2) * 128,
                            &P.maps.qg64, B.q_full + 8 * b, C::kHalfCols * h, 0, w.bh);
          } else {
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_3d(s_q0 + b * C::kQBytes + h * (kRows * 128), mq, B.q_full + 8 * b,
                          C::kHalfCols * h, q_row_of<GLOBAL>(P, w, u), w.bh);
          }
          ++j;
        }
      }
      if (!ok) {
        // the last loads may still be in flight: let them land
        for (uint32_t x = j > (uint32_t)NQ ? j - NQ : 0u; x < j; ++x)
          wait_bar(B.q_full + 8 * (x % NQ), (x / NQ) & 1u, abort_flag, nullptr, false);
      } else if (!GLOBAL) {
        // the last output tiles: store each once it is staged
        for (uint32_t x = j > (uint32_t)NQ ? j - NQ : 0u; x < j; ++x) {
          if (!wait_bar(B.q_empty + 8 * (x % NQ), (x / NQ) & 1u, abort_flag, p.err)) break;
          store_staged(x % NQ);
        }
      }
      // every store issued has finished reading shared memory and writing
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------- K/V producer
    // (lane 0; lane 1 of this warp is the Q producer, waiting independently).
    // Alternating chains (global rows in one query tile) get a producer each:
    // lane 0 loads the even key tiles (chain 0), lane 2 the odd ones (chain 1),
    // each into its own half of the ring [c NS/2, (c+1) NS/2), so that every
    // use of a slot belongs to the chain that waits on it (a barrier's waiter
    // may never fall two phases behind it) and neither chain's loads queue
    // behind the other's.
    const bool split = GLOBAL && shared_q;
    if (lane == 0 || (split && lane == 2)) {
      const int chain = lane == 2 ? 1 : 0;
      const int nsc = NS / 2;
      int n = 0;  // loads issued by this thread
      bool ok = true;
      for (int item = item0; item < n_items && ok; item += stride) {
        const Work w = make_work<GLOBAL>(P, item);
        const CUtensorMap *map_k = GLOBAL ? &P.maps.kp : &P.maps.k[w.slot - P.slot_base];
        const CUtensorMap *map_v = GLOBAL ? &P.maps.vp : &P.maps.v[w.slot - P.slot_base];
        const int n_tiles = w.nb + w.ng;
        const int first_pos = split ? chain : 0, step = split ? 2 : 1;
        if (GLOBAL)  // the first key tiles of the item into L2 ahead of their loads
          for (int a = first_pos; a < kGlobalAhead && a < n_tiles; a += step)
            prefetch_kv<C>(map_k, map_v, w.key0 + a * kKeys, w.bh);
        for (int pos = first_pos; pos < n_tiles && ok; pos += step) {
          // global rows: each key tile serves one query tile, so tiles are
          // consumed twice as fast as band tiles, and the ring alone cannot
          // cover the memory latency; keep kGlobalAhead tiles on their way to L2
          if (GLOBAL && pos + kGlobalAhead < n_tiles)
            prefetch_kv<C>(map_k, map_v, w.key0 + (pos + kGlobalAhead) * kKeys, w.bh);
          const bool gt = is_global_pos(w, pos);
          const int bp = band_index(w, pos);
          const int rows = gt ? kGKeys : kKeys;
          const int y = gt ? global_index(w, pos) * kGKeys : (GLOBAL ? w.key0 + bp * kKeys : (w.lo + bp) * kKeys);
          const CUtensorMap *mk = gt ? &P.maps.kg : map_k;
          const CUtensorMap *mv = gt ? &P.maps.vg : map_v;
          for (int which = 0; which < 2; ++which, ++n) {
            const int s = split ? chain * nsc + n % nsc : n % NS;
            const int use = split ? n / nsc : n / NS;
            if (!wait_bar(B.slot_empty + 8 * s, (use & 1) ^ 1, abort_flag, p.err)) {
              ok = false;
              break;
            }
            const uint32_t dst = s_slots + s * C::kSlotBytes;
            mbar_expect_tx(B.slot_full + 8 * s, rows * D * C::kElem);
            if (TF && which) {
              // transposed values: chunks of 32 keys x D rows (K-major for P V)
              for (int c = 0; c < rows / 32; ++c)
                tma_load_3d(dst + c * (D * 128), mv, B.slot_full + 8 * s, y + 32 * c, 0, w.bh);
            } else {
              for (int h = 0; h < C::kHalves; ++h)
                tma_load_3d(dst + h * (rows * 128), which ? mv : mk, B.slot_full + 8 * s,
                            C::kHalfCols * h, y, w.bh);
            }
          }
        }
      }
      if (!ok) {
        // drain the loads still in flight before the CTA's memory is released
        const int depth = split ? nsc : NS;
        for (int k = max(0, n - depth); k < n; ++k) {
          const int s = split ? chain * nsc + k % nsc : k % NS;
          wait_bar(B.slot_full + 8 * s, (k / depth) & 1, abort_flag, nullptr, false);
        }
      }
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------- MMA issuers
    // Warp 9 issues the MMAs of query tile 0, warp 10 those of query tile 1.
    // Both walk every item's tile list in order; for position i an issuer does
    //   PV_u(i-1) [needs P_u(i-1), V_{i-1}], then S_u(i) [needs K_i]
    // S_u(i) overwrites the TMEM columns P_u(i-1) was read from; MMAs of one
    // thread execute in order, so issuing it after PV_u(i-1) is enough.  Each
    // issuer releases every K and V slot once: by a commit after its MMAs that
    // read the slot, or -- for a tile its query tile does not reach, or an
    // item whose query tile u is empty -- by a plain arrive after the tile has
    // landed (so no issuer can run a lap of the ring ahead of the other).
    // The two query tiles are kept half a period apart (ping-pong): S_0(g) is
    // issued after S_1(g-1), and S_1(g) after S_0(g), counting positions g over
    // all items of the CTA, so the tensor core runs S_0(g), PV_1(g-1), S_1(g),
    // PV_0(g), ... and each softmax warpgroup works while the other tile's MMAs
    // execute.
    const int u = warp - 9;
    {
      // a negative scale negates Q in the S products (bit 13: negate A)
      const uint32_t neg_a = p.scale_log2 < 0.f ? (1u << 13) : 0u;
      const uint32_t kIdescS = idesc_mma(kRows, kKeys, false, TF) | neg_a;
      const uint32_t kIdescSg = idesc_mma(kRows, kGKeys, false, TF) | neg_a;
      // B = V: MN-major bf16 tiles as loaded, or K-major transposed fp32 tiles
      // (tf32 operands must be K-major)
      constexpr uint32_t kIdescPV = idesc_mma(kRows, D, !TF, TF);
      // P V: K steps of C::kMmaK keys.  P in TMEM is bf16 pairs (16 keys in 8
      // columns) or tf32 (8 keys in 8 columns): either way a step advances 8
      // TMEM columns, and C::kMmaK 128-byte rows of V
      constexpr int kPvHalf = kKeys / 2 / C::kMmaK;  // steps per half of a band tile
      constexpr uint64_t kVStep = (uint64_t)C::kMmaK * 128 / 16;
      // descriptor offset (16-byte units) of P V step kk in a value tile
      auto v_step = [](int kk) -> uint64_t {
        if constexpr (TF)
          return (uint64_t)(((kk >> 2) * (D * 128) + (kk & 3) * 32) >> 4);  // 32-key chunks
        else
          return (uint64_t)kk * kVStep;
      };
      const uint64_t dk_base = sw128_desc(s_slots, 16, 1024);
      const uint64_t dv_band = TF ? sw128_desc(s_slots, 16, 1024)                // K-major
                                  : sw128_desc(s_slots, kKeys * 128, 1024);  // LBO: next 64 columns of V
      const uint64_t dv_glob = TF ? sw128_desc(s_slots, 16, 1024) : sw128_desc(s_slots, kGKeys * 128, 1024);
      const uint32_t d_s = tmem + u * 128, d_o = tmem + 256 + u * 128;
      const uint32_t s_full = B.s_full + 8 * u, p_full = B.p_full + 8 * u;
      if (GLOBAL && p.g_alt) {
        // Global rows in one query tile: chain u reads only the key tiles u,
        // u+2, ... of each item, so this issuer visits only those -- no
        // hand-off, as the chains share no tile.  Chain u's loads cycle
        // through its half of the ring (slots u NS/2 ..): the keys of its i-th
        // tile are its load base + 2 i (values: + 1), and it alone waits on and
        // releases those slots.  Each key tile is taken as two 64-key
        // sub-tiles in the order of the band items (S of sub-tile j in the half
        // j & 1 of S_u's columns, S(j + 1) issued right after PV(j - 1)).
        const int nsc = NS / 2;
        const uint32_t kIdescSh = idesc_mma(kRows, kKeys / 2, false, TF) | neg_a;
        uint32_t pv = 0, jq = 0, base = 0, sc = 0;
        bool ok = true;
        for (int item = item0; item < n_items && ok; item += stride) {
          const Work w = make_work<GLOBAL>(P, item);
          const bool act = u ? w.active[1] : w.active[0];
          const uint32_t jt = jq++;  // one shared query tile per item
          const uint32_t qb = jt % NQ;
          const uint64_t dq = sw128_desc(s_q0 + qb * C::kQBytes, 16, 1024);
          const int n_u = act ? (u ? w.n_cnt[1] : w.n_cnt[0]) : 0;
          // every item's tile is waited for, used or not: the barrier's phases
          // are then followed one by one
          ok = __all_sync(0xffffffffu, wait_bar(B.q_full + 8 * qb, (jt / NQ) & 1u, abort_flag, p.err));
          if (!ok) break;
          tc_fence_after();
          bool pd = false;
          int pd_h = 0, pd_vslot = 0;
          uint32_t pd_vpar = 0, pd_col = 0;
          int pv_item = 0;
          auto issue_pv = [&]() -> bool {
            bool good = __all_sync(0xffffffffu, wait_bar(B.p_sub + 8 * (2 * u + (pv & 1u)), (pv >> 1) & 1u,
                                                         abort_flag, p.err));
            if (good && pd_h == 0)
              good = __all_sync(0xffffffffu, wait_bar(B.slot_full + 8 * pd_vslot, pd_vpar, abort_flag, p.err));
            if (!good) return false;
            tc_fence_after();
            const uint64_t off = (uint64_t)((pd_vslot * C::kSlotBytes) >> 4);
            const uint32_t first = pv_item == 0 ? 0u : 1u;
            const uint32_t a = d_s + pd_col;
#pragma unroll
            for (int kk = 0; kk < kPvHalf; ++kk)
              mma_ts_warp<TF>(d_o, a + kk * 8, dv_band + off + v_step(pd_h * kPvHalf + kk), kIdescPV,
                              kk > 0 ? 1u : first);
            if constexpr (PRECISE) {
#pragma unroll
              for (int kk = 0; kk < kPvHalf; ++kk)
                mma_ts_warp<TF>(d_o, a + 32 + kk * 8, dv_band + off + v_step(pd_h * kPvHalf + kk), kIdescPV, 1u);
            }
            ++pv;
            ++pv_item;
            mma_commit_warp(B.pv_done + 8 * u);
            if (pd_h == 1) mma_commit_warp(B.slot_empty + 8 * pd_vslot);
            pd = false;
            return true;
          };
          for (int i = 0; i < n_u && ok; ++i) {
            const uint32_t nk = base + 2u * (uint32_t)i;
            const int k_slot = u * nsc + (int)(nk % (uint32_t)nsc);
            const uint32_t k_par = (nk / (uint32_t)nsc) & 1u;
            const uint32_t nv = nk + 1u;
            const int v_slot = u * nsc + (int)(nv % (uint32_t)nsc);
            const uint32_t v_par = (nv / (uint32_t)nsc) & 1u;
            ok = __all_sync(0xffffffffu, wait_bar(B.slot_full + 8 * k_slot, k_par, abort_flag, p.err));
            if (!ok) break;
            tc_fence_after();
            const uint64_t dk = dk_base + (uint64_t)((k_slot * C::kSlotBytes) >> 4);
            for (int h = 0; h < 2 && ok; ++h) {
              const uint32_t col = (sc & 1u) * 64u;
#pragma unroll
              for (int kk = 0; kk < D / C::kMmaK; ++kk)
                mma_ss_warp<TF>(d_s + col, dq + (((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4),
                                dk + (((kk >> 2) * (kKeys * 128) + (kk & 3) * 32 + h * (kKeys / 2) * 128) >> 4),
                                kIdescSh, kk > 0);
              mma_commit_warp(B.s_sub + 8 * (2 * u + (sc & 1u)));
              if (h == 1) mma_commit_warp(B.slot_empty + 8 * k_slot);
              ++sc;
              if (pd) ok = issue_pv();
              pd = true;
              pd_h = h;
              pd_col = col;
              pd_vslot = v_slot;
              pd_vpar = v_par;
            }
          }
          if (ok && pd) ok = issue_pv();
          if (ok && pv_item > 0) mma_commit_warp(B.o_final + 8 * u);
          base += 2u * (uint32_t)(u ? w.n_cnt[1] : w.n_cnt[0]);
        }
      }
      if constexpr (!GLOBAL) {
        // Band items in 64-key sub-tiles.  Sub-tile j of this chain (counted
        // over all its items) has its S in the half (j & 1) of S_u's columns
        // and its P over the first columns of that half, so the issue order
        //   S(0), S(1), PV(0), S(2), PV(1), S(3), ...
        // lets S(j + 1) overwrite the half of sub-tile j - 1 right after
        // PV(j - 1) in issue order (MMAs of one thread execute in order),
        // without waiting for P(j): the S product of the next sub-tile runs
        // while the softmax works on this one.  The key tile of a position is
        // read by its two sub-tiles (a global tile: one), the value tile by
        // their P V products; both slots are released by a commit after the
        // last MMA that reads them, or by a plain arrive, after the tile has
        // landed, at a position this query tile does not reach.  At the end of
        // an item, and before a position the tile does not reach, the pending
        // P V is issued at once.
        const uint32_t kIdescSh = idesc_mma(kRows, kKeys / 2, false, TF) | neg_a;
        uint32_t pv = 0, jq = 0, sc = 0;  // sc: S products issued (sub-tiles)
        int k_slot = 0, k_par = 0;
        bool ok = true;
        for (int item = item0; item < n_items && ok; item += stride) {
          const Work w = make_work<GLOBAL>(P, item);
          const bool act = u ? w.active[1] : w.active[0];
          const uint32_t jt = jq + ((u == 1 && w.active[0]) ? 1u : 0u);
          jq += (uint32_t)w.active[0] + (uint32_t)w.active[1];
          const uint32_t qb = jt % NQ;
          const uint64_t dq = sw128_desc(s_q0 + qb * C::kQBytes, 16, 1024);
          if (act) {
            ok = __all_sync(0xffffffffu, wait_bar(B.q_full + 8 * qb, (jt / NQ) & 1u, abort_flag, p.err));
            if (!ok) break;
            tc_fence_after();
          }
          const int n_tiles = w.nb + w.ng;
          const int a_u = (u ? w.n_lo[1] : w.n_lo[0]) - w.lo;
          const int b_u = a_u + (u ? w.n_cnt[1] : w.n_cnt[0]);
          // the sub-tile whose P V is still to be issued
          bool pd = false, pd_glob = false, pd_last = false;
          int pd_h = 0, pd_vslot = 0, pd_vpar = 0;
          uint32_t pd_col = 0;
          int pv_item = 0;
          // Sub-tile j's barriers are those of its S half (j & 1), in their
          // use (j >> 1): a waiter is never two phases behind, as sub-tile
          // j + 2 cannot start before this sub-tile's P V is issued.
          auto issue_pv = [&]() -> bool {
            bool good = __all_sync(0xffffffffu, wait_bar(B.p_sub + 8 * (2 * u + (pv & 1u)), (pv >> 1) & 1u,
                                                         abort_flag, p.err));
            // the value tile: waited for by its first P V
            if (good && pd_h == 0)
              good = __all_sync(0xffffffffu, wait_bar(B.slot_full + 8 * pd_vslot, pd_vpar, abort_flag, p.err));
            if (!good) return false;
            tc_fence_after();
            const uint64_t off = (uint64_t)((pd_vslot * C::kSlotBytes) >> 4);
            const uint32_t first = pv_item == 0 ? 0u : 1u;
            const uint32_t a = d_s + pd_col;
            const uint64_t dv = pd_glob ? dv_glob : dv_band;
            const int k0 = pd_glob ? 0 : pd_h * kPvHalf;  // first K step in the value tile
#pragma unroll
            for (int kk = 0; kk < kPvHalf; ++kk)
              mma_ts_warp<TF>(d_o, a + kk * 8, dv + off + v_step(k0 + kk), kIdescPV, kk > 0 ? 1u : first);
            if constexpr (PRECISE) {
              // the low parts of split P, 32 columns after the high parts
#pragma unroll
              for (int kk = 0; kk < kPvHalf; ++kk)
                mma_ts_warp<TF>(d_o, a + 32 + kk * 8, dv + off + v_step(k0 + kk), kIdescPV, 1u);
            }
            ++pv;
            ++pv_item;
            mma_commit_warp(B.pv_done + 8 * u);
            if (pd_last) mma_commit_warp(B.slot_empty + 8 * pd_vslot);
            pd = false;
            return true;
          };
          for (int i = 0; i < n_tiles && ok; ++i) {
            const bool gc = is_global_pos(w, i);
            const int ib = band_index(w, i);
            const bool reads = act && (gc || (ib >= a_u && ib < b_u));
            int v_slot = k_slot + 1, v_par = k_par;  // the value tile follows the key tile
            if (v_slot == NS) {
              v_slot = 0;
              v_par ^= 1;
            }
            ok = __all_sync(0xffffffffu, wait_bar(B.slot_full + 8 * k_slot, k_par, abort_flag, p.err));
            if (!ok) break;
            if (reads) {
              tc_fence_after();
              const uint64_t dk = dk_base + (uint64_t)((k_slot * C::kSlotBytes) >> 4);
              const int n_sub = gc ? 1 : 2;
              for (int h = 0; h < n_sub && ok; ++h) {
                const uint32_t col = (sc & 1u) * 64u;
                // K steps of 32 bytes of a row: four per 128-byte swizzled row
                // chunk, then on to the next chunk; sub-tile h starts 64 key
                // rows into each chunk of a band tile
                if (!gc) {
#pragma unroll
                  for (int kk = 0; kk < D / C::kMmaK; ++kk)
                    mma_ss_warp<TF>(d_s + col, dq + (((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4),
                                    dk + (((kk >> 2) * (kKeys * 128) + (kk & 3) * 32 + h * (kKeys / 2) * 128) >> 4),
                                    kIdescSh, kk > 0);
                } else {
#pragma unroll
                  for (int kk = 0; kk < D / C::kMmaK; ++kk)
                    mma_ss_warp<TF>(d_s + col, dq + (((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4),
                                    dk + (((kk >> 2) * (kGKeys * 128) + (kk & 3) * 32) >> 4), kIdescSg, kk > 0);
                }
                mma_commit_warp(B.s_sub + 8 * (2 * u + (sc & 1u)));
                if (h == n_sub - 1) mma_commit_warp(B.slot_empty + 8 * k_slot);
                ++sc;
                if (pd) ok = issue_pv();
                pd = true;
                pd_glob = gc;
                pd_last = h == n_sub - 1;
                pd_h = h;
                pd_col = col;
                pd_vslot = v_slot;
                pd_vpar = v_par;
              }
            } else {
              mbar_arrive_warp(B.slot_empty + 8 * k_slot);
              if (pd) ok = issue_pv();
              if (ok) ok = __all_sync(0xffffffffu, wait_bar(B.slot_full + 8 * v_slot, v_par, abort_flag, p.err));
              if (!ok) break;
              mbar_arrive_warp(B.slot_empty + 8 * v_slot);
            }
            k_slot += 2;  // advance by two loads (K_i, V_i)
            if (k_slot >= NS) {
              k_slot -= NS;
              k_par ^= 1;
            }
          }
          if (ok && pd) ok = issue_pv();
          // O_u is final once every P V of the item has completed (the last
          // one may have been issued before a position this tile does not
          // reach)
          if (ok && pv_item > 0) mma_commit_warp(B.o_final + 8 * u);
        }
      } else {
        // More global rows than one query tile holds: two query tiles of
        // different global rows, each over every key tile of the item's chunk,
        // taken whole.  For position i an issuer does
        //   PV_u(i-1) [needs P_u(i-1), V_{i-1}], then S_u(i) [needs K_i];
        // S_u(i) overwrites the TMEM columns P_u(i-1) was read from, and MMAs
        // of one thread execute in order, so issuing it after PV_u(i-1) is
        // enough.  P arrives in two halves (keys 0-63, then 64-127), so the
        // first half of P V starts while the second half of P is computed.  The
        // two query tiles are kept half a period apart: S_0(g) is issued after
        // S_1(g-1), and S_1(g) after S_0(g), counting positions g over all
        // items of the CTA.  An issuer whose query tile is empty releases each
        // key and value slot by a plain arrive after the tile has landed.
        uint32_t pv = 0, jq = 0, g = 0;  // jq: query tiles of earlier items
        int k_slot = 0, k_par = 0;  // ring position and phase of the next K load
        bool ok = !p.g_alt;  // (the alternating issuer above has run instead)
        for (int item = item0; item < n_items && ok; item += stride) {
          const Work w = make_work<GLOBAL>(P, item);
          const bool act = u ? w.active[1] : w.active[0];
          const uint32_t jt = jq + ((u == 1 && w.active[0]) ? 1u : 0u);
          jq += (uint32_t)w.active[0] + (uint32_t)w.active[1];
          const uint32_t qb = jt % NQ;
          const uint64_t dq = sw128_desc(s_q0 + qb * C::kQBytes, 16, 1024);
          if (act) {
            ok = __all_sync(0xffffffffu, wait_bar(B.q_full + 8 * qb, (jt / NQ) & 1u, abort_flag, p.err));
            if (!ok) break;
            tc_fence_after();
          }
          const int n_tiles = w.nb;
          int pv_item = 0;
          for (int i = 0; i <= n_tiles && ok; ++i) {
            const int v_slot = k_slot == 0 ? NS - 1 : k_slot - 1;
            const int v_par = k_slot == 0 ? k_par ^ 1 : k_par;
            const bool do_pv = i > 0, do_s = i < n_tiles;
            // ping-pong hand-off (position g of tile 1 follows position g of tile 0)
            const bool hs = do_s && (u == 1 || g > 0);
            const uint32_t hs_bar = u == 1 ? B.s_issued : B.s_issued + 8;
            const uint32_t hs_par = u == 1 ? (g & 1u) : ((g - 1) & 1u);
            // the slot and hand-off conditions are usually met already: poll
            // them together, block only on P, and wait for what was not met
            uint32_t pend = 0;
            if (do_pv && !mbar_test(B.slot_full + 8 * v_slot, v_par)) pend |= 1u;
            if (do_s && !mbar_test(B.slot_full + 8 * k_slot, k_par)) pend |= 2u;
            if (hs && !mbar_test(hs_bar, hs_par)) pend |= 4u;
            pend = __reduce_or_sync(0xffffffffu, pend);
            if (do_pv) {
              if (act) ok = __all_sync(0xffffffffu, wait_bar(B.p_half + 8 * u, pv & 1u, abort_flag, p.err));
              if (ok && (pend & 1u))
                ok = __all_sync(0xffffffffu, wait_bar(B.slot_full + 8 * v_slot, v_par, abort_flag, p.err));
              if (!ok) break;
              if (act) {
                tc_fence_after();
                const uint64_t off = (uint64_t)((v_slot * C::kSlotBytes) >> 4);
                const uint32_t first = pv_item == 0 ? 0u : 1u;
                // split P (PRECISE): the low parts sit 64 columns after the high
                // parts and multiply the same value rows
#pragma unroll
                for (int kk = 0; kk < kPvHalf; ++kk)
                  mma_ts_warp<TF>(d_o, d_s + kk * 8, dv_band + off + v_step(kk), kIdescPV,
                                  kk > 0 ? 1u : first);
                if constexpr (PRECISE) {
#pragma unroll
                  for (int kk = 0; kk < kPvHalf; ++kk)
                    mma_ts_warp<TF>(d_o, d_s + 64 + kk * 8, dv_band + off + v_step(kk), kIdescPV, 1u);
                }
                ok = __all_sync(0xffffffffu, wait_bar(p_full, pv & 1u, abort_flag, p.err));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = kPvHalf; kk < 2 * kPvHalf; ++kk)
                  mma_ts_warp<TF>(d_o, d_s + kk * 8, dv_band + off + v_step(kk), kIdescPV, 1u);
                if constexpr (PRECISE) {
#pragma unroll
                  for (int kk = kPvHalf; kk < 2 * kPvHalf; ++kk)
                    mma_ts_warp<TF>(d_o, d_s + 64 + kk * 8, dv_band + off + v_step(kk), kIdescPV, 1u);
                }
                ++pv;
                ++pv_item;
                mma_commit_warp(B.slot_empty + 8 * v_slot);
                if (i == n_tiles) mma_commit_warp(B.o_final + 8 * u);
              } else {
                mbar_arrive_warp(B.slot_empty + 8 * v_slot);
              }
            }
            if (do_s) {
              if (pend & 2u)
                ok = __all_sync(0xffffffffu, wait_bar(B.slot_full + 8 * k_slot, k_par, abort_flag, p.err));
              if (ok && (pend & 4u)) ok = __all_sync(0xffffffffu, wait_bar(hs_bar, hs_par, abort_flag, p.err));
              if (!ok) break;
              if (act) {
                tc_fence_after();
                const uint64_t dk = dk_base + (uint64_t)((k_slot * C::kSlotBytes) >> 4);
                // K steps of 32 bytes of a row: four per 128-byte swizzled row
                // chunk, then on to the next chunk of the tile
#pragma unroll
                for (int kk = 0; kk < D / C::kMmaK; ++kk)
                  mma_ss_warp<TF>(d_s, dq + (((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4),
                                  dk + (((kk >> 2) * (kKeys * 128) + (kk & 3) * 32) >> 4), kIdescS, kk > 0);
                mma_commit_warp(s_full);
                mma_commit_warp(B.slot_empty + 8 * k_slot);
              } else {
                mbar_arrive_warp(B.slot_empty + 8 * k_slot);
              }
              mbar_arrive_warp(B.s_issued + 8 * u);  // S_u(g) issued (or not needed)
              ++g;
              k_slot += 2;  // advance by two loads (K_i, V_i)
              if (k_slot >= NS) {
                k_slot -= NS;
                k_par ^= 1;
              }
            }
          }
        }
      }
      // everything this thread issued has completed before TMEM is released
      mma_commit_warp(B.mma_done + 8 * u);
      __syncwarp();
      wait_bar(B.mma_done + 8 * u, 0, abort_flag, nullptr, false);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------- softmax
    // warpgroup u: one thread per row of query tile u
    const int u = warp >> 2;
    const int row = tid & 127;
    const uint32_t lane_addr = (uint32_t)((row >> 5) * 32) << 16;
    const uint32_t t_s = tmem + lane_addr + u * 128;
    const uint32_t t_o = tmem + lane_addr + 256 + u * 128;
    // the S product carries the sign; a zero scale becomes a tiny one (every
    // finite score then gives exactly 2^0, and a masked -inf stays -inf
    // instead of turning into NaN)
    const float sl = fmaxf(fabsf(p.scale_log2), 1e-30f);
    const int half = p.half;
    const int bar_id = 1 + u;
    int32_t *g_list = g_lists + u * SA_MAX_GLOBALS;
    uint32_t scnt = 0, ocnt = 0, jq = 0;  // jq: query tiles of earlier items
    bool ok = true;
    for (int item = item0; item < n_items && ok; item += stride) {
      const Work w = make_work<GLOBAL>(P, item);
      const bool act_u = u ? w.active[1] : w.active[0];
      // this tile's load index (a shared tile: one load per item)
      const uint32_t jt = shared_q ? jq : jq + ((u == 1 && w.active[0]) ? 1u : 0u);
      jq += shared_q ? 1u : (uint32_t)w.active[0] + (uint32_t)w.active[1];
      const uint32_t qb = jt % NQ;  // buffer holding Q_u; the output is staged there
      if (!act_u) {
        // A shared tile is released by both warpgroups, working or not.  An
        // idle warpgroup first waits for the item's tile to be loaded: it may
        // not release a later use of the buffer before the current one has
        // been released (the barrier would run a phase ahead of its waiter).
        if (shared_q) {
          ok = named_bar_and(bar_id, 128, wait_bar(B.q_full + 8 * qb, (jt / NQ) & 1u, abort_flag, p.err));
          if (!ok) break;
          if (row == 0) mbar_arrive(B.q_empty + 8 * qb);
        }
        continue;
      }
      const int nlo_u = u ? w.n_lo[1] : w.n_lo[0];
      const int ncnt_u = u ? w.n_cnt[1] : w.n_cnt[0];
      const int n = ncnt_u + w.ng;
      const int t_q = GLOBAL ? 0 : (w.q_tile + u) * kRows + row;  // class coordinate
      if (!GLOBAL && w.ng > 0 && ((w.flags >> u) & 1)) {
        // (only read by the in-band test of the global tile)
        // global positions in this item's residue-class coordinates: g = r + d*t
        // gives t; a global outside the class can never lie in a row's band.
        // (The previous item's readers of this list passed the warpgroup's
        // epilogue barrier before this point.)
        for (int i = row; i < p.n_g; i += 128) {
          const int gg = p.globals[i] - w.r;
          g_list[i] = (gg >= 0 && gg % w.d == 0) ? gg / w.d : kFarAway;
        }
        named_bar_sync(bar_id, 128);
      }
      // this row's key interval and the tile's extreme rows (band mode); a
      // band tile is full when every row's interval covers it -- the intervals
      // only move forward with the row, so the first row has the earliest end
      // and the last row the latest start
      int r_lo = 0, r_hi = 0, lo_last = 0, hi_first = 0;
      if (!GLOBAL) {
        const int q0 = (w.q_tile + u) * kRows;
        int unused;
        row_keys(half, p.chunk, p.memory, w.len, q0 + kRows - 1, lo_last, unused);
        row_keys(half, p.chunk, p.memory, w.len, q0, unused, hi_first);
        row_keys(half, p.chunk, p.memory, w.len, t_q, r_lo, r_hi);
      }
      // packed global rows: this copy of the row scores the key half `sub`
      const bool packed = GLOBAL && p.g_packed;
      const int sub = row >> 6;
      float m_run = -INFINITY, l_run = 0.f;
      if constexpr (!GLOBAL) {
        // 64-key sub-tiles (a global tile is one), S in alternate halves of
        // S_u's columns, as the issuer computes them
        for (int i = 0; i < n && ok; ++i) {
          const int pos = seq_pos_s(w, nlo_u, ncnt_u, i);
          const bool gt = is_global_pos(w, pos);
          const int n_sub = gt ? 1 : 2;
          for (int h = 0; h < n_sub; ++h) {
            bool interval = true;
            int c_lo = 0, c_hi, g0 = 0;
            if (!gt) {
              const int kb = (w.lo + band_index(w, pos)) * kKeys + h * (kKeys / 2);
              interval = !(lo_last <= kb && hi_first >= kb + kKeys / 2 - 1);
              c_lo = r_lo - kb;
              c_hi = r_hi - kb;
            } else {
              g0 = global_index(w, pos) * kGKeys;
              c_hi = min(p.n_g - 1 - g0, kGKeys - 1);
            }
            const bool dedup = gt && ((w.flags >> u) & 1);
            const uint32_t col = (scnt & 1u) * 64u;
            const uint32_t sb = 2 * u + (scnt & 1u);  // this sub-tile's S half
            ok = __all_sync(0xffffffffu, wait_bar(B.s_sub + 8 * sb, (scnt >> 1) & 1u, abort_flag, p.err));
            if (!ok) break;
            tc_fence_after();
            ok = softmax_sub<D, TF, PRECISE>(t_s + col, t_o, sl, interval, c_lo, c_hi, g_list, g0, t_q,
                                             half, dedup, B.pv_done + 8 * u, (scnt - 1u) & 1u,
                                             abort_flag, p.err, m_run, l_run);
            ++scnt;
            if (!ok) break;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.p_sub + 8 * sb);
          }
        }
      } else if (p.g_alt) {
        // Global rows in one query tile: chain u takes the key tiles u, u+2,
        // ... as 64-key sub-tiles, as the issuer computes them.  A packed row
        // scores only the sub-tiles of its key half (the other copy of the row
        // scores the other half); for the other sub-tiles, and for keys past
        // the end of the chunk, its P is zero.
        for (int i = 0; i < n && ok; ++i) {
          const int kb = w.key0 + (2 * i + u) * kKeys;
          const int c_hi = w.key_end - 1 - kb;  // last key of the chunk, as a column of the tile
          for (int h = 0; h < 2; ++h) {
            const int c_hi_h = c_hi - h * (kKeys / 2);
            const bool scores = (!packed || sub == h) && c_hi_h >= 0;  // warp-uniform
            const uint32_t col = (scnt & 1u) * 64u;
            const uint32_t sb = 2 * u + (scnt & 1u);
            ok = __all_sync(0xffffffffu, wait_bar(B.s_sub + 8 * sb, (scnt >> 1) & 1u, abort_flag, p.err));
            if (!ok) break;
            tc_fence_after();
            if (scores)
              ok = softmax_sub<D, TF, PRECISE>(t_s + col, t_o, sl, c_hi_h < kKeys / 2 - 1, 0, c_hi_h, g_list,
                                               0, 0, half, false, B.pv_done + 8 * u, (scnt - 1u) & 1u,
                                               abort_flag, p.err, m_run, l_run);
            else
              zero_p_sub<TF, PRECISE>(t_s + col);
            ++scnt;
            if (!ok) break;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.p_sub + 8 * sb);
          }
        }
      } else {
        // more global rows than one query tile holds: each query tile takes
        // every key tile of the chunk, whole (P in two halves)
        for (int i = 0; i < n && ok; ++i) {
          const int kb = w.key0 + i * kKeys;
          const bool interval = kb + kKeys > w.key_end;
          const int c_hi = w.key_end - 1 - kb;
          ok = __all_sync(0xffffffffu, wait_bar(B.s_full + 8 * u, scnt & 1u, abort_flag, p.err));
          ++scnt;
          if (!ok) break;
          tc_fence_after();
          softmax_tile<D, TF, PRECISE>(t_s, t_o, sl, interval, 0, c_hi, g_list, 0, t_q, half, false,
                                       false, B.p_half + 8 * u, lane, m_run, l_run);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(B.p_full + 8 * u);
        }
      }

      // every thread of the warpgroup takes part in the same barriers, so the
      // decision to write the tile is made jointly
      bool fin = ok && wait_bar(B.o_final + 8 * u, ocnt & 1u, abort_flag, p.err);
      ++ocnt;
      fin = named_bar_and(bar_id, 128, fin);
      ok = fin;
      if (!fin) break;
      tc_fence_after();
      if (!GLOBAL) {
        // normalise, stage the tile (bf16, or fp32 for fp32 inputs) in this
        // tile's query buffer (its last S MMA has completed) in the TMA
        // 128-byte-swizzle layout, and store it with TMA; the buffer is handed
        // back to the Q producer once the store has read it
        uint8_t *stage = smem + qb * C::kQBytes;
        const float inv = rcp_approx(l_run);
        // O read out of TMEM in one load (one wait)
        uint32_t rall[D];
        if constexpr (D == 128)
          tmem_ld128(t_o, rall);
        else
          tmem_ld64(t_o, rall);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint32_t *r = rall + 32 * c;
          // 32 output columns: a quarter of a 128-byte row chunk in bf16, a
          // whole one in fp32
          const int h = (c * 32) / C::kHalfCols;
          const int chunk0 = ((c * 32) % C::kHalfCols) * C::kElem / 16;  // first 16-byte chunk
          uint8_t *rowp = stage + h * (kRows * 128) + row * 128;
          if constexpr (TF) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 v = make_float4(
                  __uint_as_float(r[q4 * 4 + 0]) * inv, __uint_as_float(r[q4 * 4 + 1]) * inv,
                  __uint_as_float(r[q4 * 4 + 2]) * inv, __uint_as_float(r[q4 * 4 + 3]) * inv);
              const int phys = (chunk0 + q4) ^ (row & 7);
              *reinterpret_cast<float4 *>(rowp + phys * 16) = v;
            }
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(r[q4 * 8 + 0]) * inv, __uint_as_float(r[q4 * 8 + 1]) * inv);
              v.y = pack_bf16(__uint_as_float(r[q4 * 8 + 2]) * inv, __uint_as_float(r[q4 * 8 + 3]) * inv);
              v.z = pack_bf16(__uint_as_float(r[q4 * 8 + 4]) * inv, __uint_as_float(r[q4 * 8 + 5]) * inv);
              v.w = pack_bf16(__uint_as_float(r[q4 * 8 + 6]) * inv, __uint_as_float(r[q4 * 8 + 7]) * inv);
              const int phys = (chunk0 + q4) ^ (row & 7);
              *reinterpret_cast<uint4 *>(rowp + phys * 16) = v;
            }
          }
        }
        if (p.lse && t_q < w.len) {
          const int64_t pos_q = (int64_t)w.r + (int64_t)w.d * t_q;
          p.lse[(int64_t)w.bh * p.N + pos_q] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
        }
        // the staged tile is handed to the Q producer, which stores it
        fence_proxy_async_smem();
        named_bar_sync(bar_id, 128);
        if (row == 0) mbar_arrive(B.q_empty + 8 * qb);
      } else {
        // partial set of this query tile and its row there; the global row it
        // belongs to (a packed tile holds each global row twice, rows g and
        // g + 64, one partial per key half)
        const int set = p.g_alt ? 2 * w.chunk + u : w.chunk;
        const int prow = q_row_of<GLOBAL>(P, w, u) + row;
        const int gr = packed ? (row & 63) : prow;
        const int64_t slot = ((int64_t)w.bh * p.part_sets + set) * p.g_pad + prow;
        float4 *dst = reinterpret_cast<float4 *>(p.part_o + slot * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(t_o + c * 32, r);  // collective: every lane loads
          if (gr < p.n_g) {
#pragma unroll
            for (int x = 0; x < 8; ++x)
              dst[c * 8 + x] = make_float4(__uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                                           __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
          }
        }
        if (gr < p.n_g) {
          p.part_ml[slot * 2 + 0] = m_run;
          p.part_ml[slot * 2 + 1] = l_run;
        }
        if (row == 0) mbar_arrive(B.q_empty + 8 * qb);  // every S MMA has completed
      }
      // O_u has been read out (tcgen05.ld waits): the next item's first PV_u,
      // issued only after this warpgroup's next P arrival, may overwrite it
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One launch runs both kinds of work on CTAs of their own: CTAs [0, n_gctas)
// the global-row items (the global rows against every key, split over key
// chunks), the others the band items.  Every CTA occupies one SM for the whole
// launch, so the two kinds run side by side and the global rows' keys and
// values are read while the band tiles run, not in a pass of their own.
template <int D, bool TF, bool PRECISE>
__global__ void __launch_bounds__(kThreads, 1) tc_attention_kernel(const __grid_constant__ Params P) {
  const int b = blockIdx.x;
  if (b < P.n_gctas)
    cta_body<D, true, TF, PRECISE>(P, b, P.n_gctas, P.n_gitems);
  else
    cta_body<D, false, TF, PRECISE>(P, b - P.n_gctas, gridDim.x - P.n_gctas, P.n_items);
}

// ---------------------------------------------------------------------------
// host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

cudaError_t get_encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// 3-D map {D, rows, bh} of bf16 (or fp32 when tf32), 128-byte swizzle, boxes
// of {one 128-byte row chunk, box_rows, 1}.
cudaError_t make_map(CUtensorMap *m, const void *base, int D, uint64_t rows, uint64_t bh,
                     uint64_t row_stride_bytes, uint64_t bh_stride_bytes, uint32_t box_rows,
                     bool tf32) {
  cuuint64_t dims[3] = {(cuuint64_t)D, rows, bh};
  cuuint64_t strides[2] = {row_stride_bytes, bh_stride_bytes};
  cuuint32_t box[3] = {tf32 ? 32u : 64u, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D fp32 map of transposed values {len_pad (keys), D, bh}, 128-byte swizzle,
// boxes of {32 keys, D, 1}: one box is the K-major operand chunk of 32 keys.
cudaError_t make_map_values_t(CUtensorMap *m, const float *base, int D, uint64_t len_pad,
                              uint64_t bh) {
  cuuint64_t dims[3] = {len_pad, (cuuint64_t)D, bh};
  cuuint64_t strides[2] = {len_pad * 4, (cuuint64_t)D * len_pad * 4};
  cuuint32_t box[3] = {32, (cuuint32_t)D, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Persistent launch: one CTA per SM.  The first g_ctas CTAs stride over the
// P.n_gitems global-row items, the other band_ctas CTAs over the P.n_items band
// items.
template <int D, bool TF, bool PRECISE>
cudaError_t launch(Params &P, int band_ctas, int g_ctas, cudaStream_t s) {
  const int grid = band_ctas + g_ctas;
  if (grid <= 0) return cudaSuccess;
  constexpr int smem = Cfg<D, TF>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(tc_attention_kernel<D, TF, PRECISE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  P.n_gctas = g_ctas;
  tc_attention_kernel<D, TF, PRECISE><<<grid, kThreads, smem, s>>>(P);
  return cudaGetLastError();
}

}  // namespace tc

Tiling tc_tiling(int, int sms) {
  Tiling t{tc::kRows, 2, tc::kKeys, 128, 256, 2 * sms, tc::kMaxSlotsPerLaunch};
  t.sms = sms;
  t.fuse_global = true;
  return t;
}

namespace {

cudaError_t fill_common(tc::Params &P, const DevProblem &p, int BH, bool tf) {
  cudaError_t e = tc::get_encoder();
  if (e != cudaSuccess) return e;
  std::memset(&P.maps, 0, sizeof P.maps);
  P.p = p;
  P.p.half = std::min(p.half, p.N);  // a wider window changes nothing
  P.n_items = 0;
  P.n_gitems = p.n_gitems;
  P.n_gctas = 0;
  const int D = p.D;
  const uint64_t es = tf ? 4 : 2;
  const uint64_t head = (uint64_t)p.N * D * es;
  if (p.n_g > 0 && p.g_first >= 0) {
    // contiguous globals: views of the rows [g_first, N) of the inputs (rows past
    // the globals are read but masked; rows past N read as zeros)
    const uint64_t off = (uint64_t)p.g_first * D * es, rows = (uint64_t)(p.N - p.g_first);
    const char *kv = static_cast<const char *>(p.k) + off;
    const char *vv = static_cast<const char *>(p.v) + off;
    const char *qv = static_cast<const char *>(p.gq_src) + off;
    if ((e = tc::make_map(&P.maps.kg, kv, D, rows, BH, D * es, head, tc::kGKeys, tf)) ||
        (e = tf ? tc::make_map_values_t(&P.maps.vg, p.vgT, D, p.g_pad, BH)
                : tc::make_map(&P.maps.vg, vv, D, rows, BH, D * es, head, tc::kGKeys, tf)) ||
        (e = tc::make_map(&P.maps.qg, qv, D, rows, BH, D * es, head, tc::kRows, tf)) ||
        (e = tc::make_map(&P.maps.qg64, qv, D, rows, BH, D * es, head, tc::kRows / 2, tf)))
      return e;
  } else if (p.n_g > 0) {
    const uint64_t ghead = (uint64_t)p.g_pad * D * es;
    if ((e = tc::make_map(&P.maps.kg, p.kg, D, p.g_pad, BH, D * es, ghead, tc::kGKeys, tf)) ||
        (e = tf ? tc::make_map_values_t(&P.maps.vg, p.vgT, D, p.g_pad, BH)
                : tc::make_map(&P.maps.vg, p.vg, D, p.g_pad, BH, D * es, ghead, tc::kGKeys, tf)) ||
        (e = tc::make_map(&P.maps.qg, p.qg, D, p.g_pad, BH, D * es, ghead, tc::kRows, tf)) ||
        (e = tc::make_map(&P.maps.qg64, p.qg, D, p.g_pad, BH, D * es, ghead, tc::kRows / 2, tf)))
      return e;
  }
  if (p.n_g > 0) {
    // keys and values of the global-row pass
    if ((e = tc::make_map(&P.maps.kp, p.gk_src, D, p.N, BH, D * es, head, tc::kKeys, tf)) ||
        (e = tf ? tc::make_map_values_t(&P.maps.vp, p.vT_plain, D, values_len_pad(p.N), BH)
                : tc::make_map(&P.maps.vp, p.gv_src, D, p.N, BH, D * es, head, tc::kKeys, tf)))
      return e;
  }
  return cudaSuccess;
}

cudaError_t launch_any(tc::Params &P, int D, bool tf, bool precise, int band_ctas, int g_ctas,
                       cudaStream_t s) {
  if (tf) return tc::launch<64, true, false>(P, band_ctas, g_ctas, s);  // fp32 inputs: D = 64 only
  if (D == 64)
    return precise ? tc::launch<64, false, true>(P, band_ctas, g_ctas, s)
                   : tc::launch<64, false, false>(P, band_ctas, g_ctas, s);
  return precise ? tc::launch<128, false, true>(P, band_ctas, g_ctas, s)
                 : tc::launch<128, false, false>(P, band_ctas, g_ctas, s);
}

}  // namespace

bool tc_supports(sa_dtype dt, int D) {
  return dt == SA_BF16 ? (D == 64 || D == 128) : dt == SA_TF32 && D == 64;
}

cudaError_t launch_band_tc(const DevProblem &p, sa_dtype dt, bool precise, const Slot *host_slots,
                           int n_slots, const std::vector<int32_t> &group_begin, int BH, int sms,
                           int g_ctas, int band_ctas, cudaStream_t s) {
  static thread_local tc::Params P;  // ~9 KB of tensor maps: keep it off the stack
  const bool tf = dt == SA_TF32;
  cudaError_t e = fill_common(P, p, BH, tf);
  if (e != cudaSuccess) return e;
  const int D = p.D;
  const uint64_t es = tf ? 4 : 2;
  const uint64_t head = (uint64_t)p.N * D * es;
  // transposed values of each slot (tf32), back to back in slot order
  std::vector<size_t> vt_off(n_slots + 1, 0);
  for (int i = 0; i < n_slots; ++i)
    vt_off[i + 1] = vt_off[i] + (size_t)BH * D * values_len_pad(host_slots[i].len);
  const int n_groups = (int)group_begin.size() - 1;
  for (int g = 0; g < n_groups; ++g) {
    const int first = g * tc::kMaxSlotsPerLaunch;
    const int count = std::min(tc::kMaxSlotsPerLaunch, n_slots - first);
    for (int i = 0; i < count; ++i) {
      const Slot &sl = host_slots[first + i];
      const uint64_t off = (uint64_t)sl.r * D * es;
      const uint64_t stride = (uint64_t)sl.d * D * es;
      const char *q = static_cast<const char *>(p.q) + off;
      const char *k = static_cast<const char *>(p.k) + off;
      const char *v = static_cast<const char *>(p.v) + off;
      char *o = static_cast<char *>(p.out) + off;
      if ((e = tc::make_map(&P.maps.q[i], q, D, sl.len, BH, stride, head, tc::kRows, tf)) ||
          (e = tc::make_map(&P.maps.k[i], k, D, sl.len, BH, stride, head, tc::kKeys, tf)) ||
          (e = tf ? tc::make_map_values_t(&P.maps.v[i], p.vT_slots + vt_off[first + i], D,
                                          values_len_pad(sl.len), BH)
                  : tc::make_map(&P.maps.v[i], v, D, sl.len, BH, stride, head, tc::kKeys, tf)) ||
          (e = tc::make_map(&P.maps.o[i], o, D, sl.len, BH, stride, head, tc::kRows, tf)))
        return e;
    }
    P.slot_base = first;
    P.item_offset = group_begin[g];
    P.n_items = group_begin[g + 1] - group_begin[g];
    // the global-row CTAs run beside the first group's band CTAs
    const int gc = g == 0 ? g_ctas : 0;
    const int bc = gc > 0 ? std::min(band_ctas, P.n_items) : std::min(P.n_items, std::max(sms, 1));
    e = launch_any(P, D, tf, precise, bc, gc, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {
// Failure-detection check: one warp waits on an mbarrier that nothing arrives
// on, through the same bounded wait the attention kernels use but with a
// short limit, then records the timeout in the error word and returns.
__global__ void stalled_wait_kernel(int *err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = tc::smem_u32(&bar);
  if (threadIdx.x == 0) {
    tc::mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  const uint64_t start = tc::global_timer();
  while (!tc::mbar_try_wait(b, 0)) {
    if (tc::global_timer() - start > limit_ns) {
      if (threadIdx.x == 0) atomicOr(err, kErrWaitTimeout);
      break;
    }
  }
}
}  // namespace

cudaError_t launch_stalled_wait_check(int *err, uint32_t limit_us, cudaStream_t s) {
  stalled_wait_kernel<<<1, 32, 0, s>>>(err, (uint64_t)limit_us * 1000ull);
  return cudaGetLastError();
}

cudaError_t launch_global_tc(const DevProblem &p, sa_dtype dt, bool precise, int BH, int sms,
                             cudaStream_t s) {
  static thread_local tc::Params P;
  const bool tf = dt == SA_TF32;
  cudaError_t e = fill_common(P, p, BH, tf);
  if (e != cudaSuccess) return e;
  P.slot_base = 0;
  P.item_offset = 0;
  P.n_items = 0;
  return launch_any(P, p.D, tf, precise, 0, std::min(p.n_gitems, std::max(sms, 1)), s);
}

}  // namespace sa

#if SA_DEBUG
namespace sa {
namespace tc {
namespace {
__global__ void check_band_items_kernel(const BandItem *items, int n, const Slot *slots, int n_slots,
                                        int slot_base, int BH, int *n_bad) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && !band_item_in_range(items[i], slots, n_slots, slot_base, BH)) atomicAdd(n_bad, 1);
}
}  // namespace
}  // namespace tc
}  // namespace sa

// The band-item range check of the SA_DEBUG kernels, run by itself on a
// list of items (include/sa_debug.h).
extern "C" sa_status sa_debug_check_band_items(const void *items, int n_items, const void *slots,
                                               int n_slots, int slot_base, int BH, int *n_bad) {
  using namespace sa;
  if (!items || !slots || !n_bad || n_items < 0 || n_slots <= 0)
    return record_error(SA_ERR_INVALID_ARG, "sa_debug_check_band_items: null pointer or bad count");
  BandItem *d_items = nullptr;
  Slot *d_slots = nullptr;
  int *d_bad = nullptr;
  cudaError_t e = cudaMalloc(&d_items, sizeof(BandItem) * (size_t)(n_items > 0 ? n_items : 1));
  if (e == cudaSuccess) e = cudaMalloc(&d_slots, sizeof(Slot) * (size_t)n_slots);
  if (e == cudaSuccess) e = cudaMalloc(&d_bad, sizeof(int));
  if (e == cudaSuccess && n_items > 0)
    e = cudaMemcpy(d_items, items, sizeof(BandItem) * (size_t)n_items, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(d_slots, slots, sizeof(Slot) * (size_t)n_slots, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(d_bad, 0, sizeof(int));
  if (e == cudaSuccess && n_items > 0) {
    tc::check_band_items_kernel<<<(n_items + 127) / 128, 128>>>(d_items, n_items, d_slots, n_slots,
                                                                slot_base, BH, d_bad);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(n_bad, d_bad, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(d_items);
  cudaFree(d_slots);
  cudaFree(d_bad);
  if (e != cudaSuccess) return record_error(SA_ERR_CUDA, cudaGetErrorString(e));
  return SA_OK;
}
#endif
