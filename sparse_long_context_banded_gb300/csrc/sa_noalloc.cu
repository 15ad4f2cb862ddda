// sa_noalloc.cu -- sa_forward_noalloc: the forward pass without any device
// memory allocation.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run attention: code that runs under a memory budget owned by someone
// else, an allocator-free runtime or plug-in host, or a process whose device
// memory is already fully handed out to another framework's pool.  For them
// this entry point takes every scratch buffer the pass needs -- the band-tile
// work list, the residue-class table, the global index list, the gathered
// global rows and the split-K partial softmax statistics -- from one static
// __device__ array of fixed size that is part of the library image.  Every GPU
// that loads the library holds that array until the process exits.
//
// The pass runs on the CUDA-core kernels (gather, band, global rows, merge),
// which compute in fp32 for either input type.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <tuple>
#include <mutex>
#include <string>

#include "sa.h"
#include "sa_internal.h"
#include "sa_kernels.h"

namespace sa {
namespace {

// Size of the static scratch array.  A call that needs more is rejected.
constexpr size_t kStaticScratchBytes = SA_NOALLOC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch, resolved per device with that device
// current and kept with the CUDA context it was resolved in: the set-up is
// repeated when the device's context is a new one (after a device reset).  In
// host code the symbol itself is only a host stand-in; kernels must be given
// this address instead.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchAddr {
  char *ptr = nullptr;
  unsigned long long ctx_id = 0;
};
ScratchAddr g_scratch_addr[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Identity of the current context (0 if it cannot be had).
unsigned long long current_context_id() {
  std::call_once(g_ctx_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current && g_ctx_id && g_ctx_current(&ctx) == CUDA_SUCCESS && ctx &&
      g_ctx_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

sa_status static_scratch_address(int dev, char **out) {
  if (dev < 0 || dev >= kMaxDevices)
    return record_error(SA_ERR_UNSUPPORTED, "device ordinal beyond the static-scratch table");
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchAddr &a = g_scratch_addr[dev];
  if (!a.ptr || ctx == 0 || a.ctx_id != ctx) {
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || !ptr) {
      std::string m = std::string("cudaGetSymbolAddress(static scratch): ") + cudaGetErrorString(e);
      cudaGetLastError();  // consumed: a later launch check must not see it
      return record_error(SA_ERR_CUDA, m.c_str());
    }
    a.ptr = static_cast<char *>(ptr);
    a.ctx_id = ctx;
  }
  *out = a.ptr;
  return SA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// The work lists of the CUDA-core kernels (64-row query tiles, 64-key tiles;
// one query tile per band item) are written into the static array by a
// kernel on the caller's stream, from values passed as kernel parameters: no
// host buffer is copied.  Band items come in (batch, head, residue class,
// query tile) order and each (head, residue class) has a slot of its own.
constexpr int kTile = 64;
constexpr int kBuildHeads = 256;  // heads described by one building launch

struct BuildParams {
  int N, half, H, B;
  int h0, nh;                     // the heads [h0, h0 + nh) of this launch
  int64_t items_per_batch;        // band items of one batch element (all heads)
  int32_t dil[kBuildHeads];       // dilation of head h0 + i
  int32_t item_off[kBuildHeads];  // first band item of head h0 + i (batch element 0)
  int32_t slot_off[kBuildHeads];  // first slot of head h0 + i
  int32_t n_slots_here, n_items_here;  // slots and band items (per batch element) of these heads
  // written by the first launch only
  int first;
  int n_g, n_chunks, g_items, bh;
  int32_t globals[SA_MAX_GLOBALS];
  Slot *slots;
  BandItem *band;
  GlobalItem *gitems;
  int32_t *glist;
};

__device__ int head_of(const BuildParams &bp, int32_t x, const int32_t *off) {
  int h = 0;  // last head whose offset is <= x
  for (int i = 1; i < bp.nh; ++i) h = off[i] <= x ? i : h;
  return h;
}

__global__ void build_work_lists_kernel(const __grid_constant__ BuildParams bp) {
  const int64_t n_band = (int64_t)bp.B * bp.n_items_here;
  const int64_t n_gi = bp.first ? (int64_t)bp.bh * bp.n_chunks * bp.g_items : 0;
  const int64_t total = max(max(n_band, (int64_t)bp.n_slots_here), max(n_gi, (int64_t)(bp.first ? bp.n_g : 0)));
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    if (x < bp.n_slots_here) {
      const int i = head_of(bp, (int32_t)x, bp.slot_off);
      const int d = bp.dil[i], r = (int)x - (bp.slot_off[i] - bp.slot_off[0]);
      bp.slots[bp.slot_off[i] + r] = Slot{d, r, (bp.N - r + d - 1) / d, 0};
    }
    if (x < n_band) {
      const int b = (int)(x / bp.n_items_here);
      const int32_t local = (int32_t)(x % bp.n_items_here) + bp.item_off[0];
      const int i = head_of(bp, local, bp.item_off);
      const int d = bp.dil[i];
      int32_t k = local - bp.item_off[i];
      int r = 0, len = 0, tiles = 0;
      for (r = 0; r < d && r < bp.N; ++r) {  // the residue class holding tile k
        len = (bp.N - r + d - 1) / d;
        tiles = (len + kTile - 1) / kTile;
        if (k < tiles) break;
        k -= tiles;
      }
      BandItem it{};
      it.bh = b * bp.H + bp.h0 + i;
      it.slot = bp.slot_off[i] + r;
      it.q_tile = k;
      const int row_lo = k * kTile, row_hi = min(len - 1, row_lo + kTile - 1);
      int lo, hi, unused;
      row_keys(bp.half, 0, 0, len, row_lo, lo, unused);
      row_keys(bp.half, 0, 0, len, row_hi, unused, hi);
      it.k_lo[0] = max(0, lo) / kTile;
      it.k_hi[0] = min(len - 1, hi) / kTile;
      it.k_lo[1] = 0;
      it.k_hi[1] = -1;
      bp.band[(int64_t)b * bp.items_per_batch + local] = it;
    }
    if (x < n_gi) {
      const int gt = (int)(x % bp.g_items);
      const int c = (int)((x / bp.g_items) % bp.n_chunks);
      const int bh = (int)(x / ((int64_t)bp.g_items * bp.n_chunks));
      bp.gitems[x] = GlobalItem{bh, c, gt, 0};
    }
    if (bp.first && x < bp.n_g) bp.glist[x] = bp.globals[x];
  }
}

struct Plan {
  // global-row pass
  int g_pad = 0, g_items = 0, n_chunks = 0, chunk_len = 0;
  // band work
  std::vector<int32_t> item_off, slot_off;  // per head, H + 1 entries
  // layout
  size_t slots, band, global, globals, qg, kg, vg, part_o, part_ml, total;
};

void layout(const Problem &p, Plan &L) {
  size_t at = 0;
  auto take = [&at](size_t bytes) {
    size_t here = at;
    at += round256(bytes);
    return here;
  };
  const size_t BH = (size_t)p.B * p.H;
  const size_t es = p.dtype == SA_BF16 ? 2 : 4;
  L.slots = take(sizeof(Slot) * (size_t)L.slot_off[p.H]);
  L.band = take(sizeof(BandItem) * (size_t)p.B * L.item_off[p.H]);
  L.global = take(sizeof(GlobalItem) * BH * L.n_chunks * L.g_items);
  L.globals = take(sizeof(int32_t) * p.globals.size());
  const size_t g_rows = BH * L.g_pad * p.D;
  L.qg = take(g_rows * es);
  L.kg = take(g_rows * es);
  L.vg = take(g_rows * es);
  const size_t part_rows = BH * (size_t)L.n_chunks * L.g_pad;
  L.part_o = take(part_rows * p.D * sizeof(float));
  L.part_ml = take(part_rows * 2 * sizeof(float));
  L.total = at;
}

sa_status fail_fmt(sa_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
sa_status fail_fmt(sa_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  // the failed runtime call's error would otherwise linger as the thread's
  // last error and be reported by a later launch check as its own
  if (s == SA_ERR_CUDA) cudaGetLastError();
  return record_error(s, buf);
}

}  // namespace
}  // namespace sa

using namespace sa;

extern "C" sa_status sa_forward_noalloc(const void *q, const void *k, const void *v, void *out,
                                        float *lse, int B, int H, int N, int D, int window,
                                        const int32_t *dilation, const int32_t *global_idx,
                                        int n_global, float scale, sa_dtype dtype,
                                        sa_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!q || !k || !v || !out) return fail_fmt(SA_ERR_INVALID_ARG, "q, k, v and out must be non-null");
  if (n_global < 0) return fail_fmt(SA_ERR_INVALID_ARG, "n_global must be >= 0");
  if (n_global > 0 && !global_idx)
    return fail_fmt(SA_ERR_INVALID_ARG, "global_idx is null but n_global = %d", n_global);
  if (H < 1) return fail_fmt(SA_ERR_INVALID_ARG, "H must be >= 1 (got %d)", H);
  const void *ptrs[4] = {q, k, v, out};
  for (int i = 0; i < 4; ++i)
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0)
      return fail_fmt(SA_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return fail_fmt(SA_ERR_INVALID_ARG, "lse must be 4-byte aligned");

  Problem p;
  p.B = B;
  p.H = H;
  p.N = N;
  p.D = D;
  p.window = window;
  p.half = window / 2;
  if (dilation)
    p.dilation.assign(dilation, dilation + H);
  else
    p.dilation.assign(H, 1);
  p.scale = scale;
  p.dtype = dtype;
  for (int i = 0; i < n_global; ++i)
    if (global_idx[i] < 0 || global_idx[i] >= N)
      return fail_fmt(SA_ERR_INVALID_ARG, "global_idx[%d] = %d outside [0, %d)", i, global_idx[i], N);
  p.globals = global_set(global_idx, n_global);
  std::string why = validate(p);
  if (!why.empty()) return fail_fmt(SA_ERR_INVALID_ARG, "%s", why.c_str());
  if (D != 64 && D != 128) return fail_fmt(SA_ERR_UNSUPPORTED, "D = %d (supported: 64, 128)", D);
  if ((int)p.globals.size() > SA_MAX_GLOBALS)
    return fail_fmt(SA_ERR_UNSUPPORTED, "%d distinct globals (at most %d)",
                    (int)p.globals.size(), SA_MAX_GLOBALS);

  // Work-list sizes (host arithmetic only) and the global-row chunking; while
  // the split-K partials would not fit, halve the number of key chunks (fewer,
  // longer chunks, same result).
  Plan L;
  L.item_off.assign(H + 1, 0);
  L.slot_off.assign(H + 1, 0);
  for (int h = 0; h < H; ++h) {
    const int d = p.dilation[h];
    int64_t items = 0;
    for (int r = 0; r < d && r < N; ++r) items += ((N - r + d - 1) / d + kTile - 1) / kTile;
    if (L.item_off[h] + items > INT32_MAX / 2 || (int64_t)L.slot_off[h] + std::min(d, N) > INT32_MAX / 2)
      return fail_fmt(SA_ERR_UNSUPPORTED, "problem too large for sa_forward_noalloc (use sa_forward)");
    L.item_off[h + 1] = L.item_off[h] + (int32_t)items;
    L.slot_off[h + 1] = L.slot_off[h] + std::min(d, N);
  }
  const int n_g = (int)p.globals.size();
  const int64_t bh = (int64_t)B * H;
  if (n_g > 0) {
    L.g_pad = ((n_g + kTile - 1) / kTile) * kTile;
    L.g_items = (n_g + kTile - 1) / kTile;
    const int64_t max_tiles = (N + kTile - 1) / kTile;
    int64_t want = (kSimtTiling.target_ctas + bh * L.g_items - 1) / (bh * L.g_items);
    std::tie(L.chunk_len, L.n_chunks) = key_chunks(N, want, kTile, max_tiles);
    layout(p, L);
    while (L.total > kStaticScratchBytes && L.n_chunks > 1) {
      std::tie(L.chunk_len, L.n_chunks) = key_chunks(N, L.n_chunks / 2, kTile, max_tiles);
      layout(p, L);
    }
  } else {
    layout(p, L);
  }
  if (L.total > kStaticScratchBytes)
    return fail_fmt(SA_ERR_UNSUPPORTED,
                    "problem needs %zu bytes of scratch; the static scratch of "
                    "sa_forward_noalloc holds %zu bytes (use sa_forward)",
                    L.total, kStaticScratchBytes);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_fmt(SA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  char *base = nullptr;
  sa_status st = static_scratch_address(dev, &base);
  if (st != SA_OK) return st;

  // the work lists, written on the device from kernel parameters
  {
    static thread_local BuildParams bp;  // ~4.5 KB: off the stack
    for (int h0 = 0; h0 < H; h0 += kBuildHeads) {
      std::memset(&bp, 0, sizeof bp);
      bp.N = N;
      bp.half = std::min(p.half, N);
      bp.H = H;
      bp.B = B;
      bp.h0 = h0;
      bp.nh = std::min(kBuildHeads, H - h0);
      bp.items_per_batch = L.item_off[H];
      for (int i = 0; i < bp.nh; ++i) {
        bp.dil[i] = p.dilation[h0 + i];
        bp.item_off[i] = L.item_off[h0 + i];
        bp.slot_off[i] = L.slot_off[h0 + i];
      }
      bp.n_slots_here = L.slot_off[h0 + bp.nh] - L.slot_off[h0];
      bp.n_items_here = L.item_off[h0 + bp.nh] - L.item_off[h0];
      bp.first = h0 == 0;
      bp.n_g = n_g;
      bp.n_chunks = L.n_chunks;
      bp.g_items = L.g_items;
      bp.bh = (int)bh;
      for (int g = 0; g < n_g; ++g) bp.globals[g] = p.globals[g];
      bp.slots = reinterpret_cast<Slot *>(base + L.slots);
      bp.band = reinterpret_cast<BandItem *>(base + L.band);
      bp.gitems = reinterpret_cast<GlobalItem *>(base + L.global);
      bp.glist = reinterpret_cast<int32_t *>(base + L.globals);
      const int64_t work = std::max<int64_t>(
          std::max<int64_t>((int64_t)B * bp.n_items_here, bp.n_slots_here),
          std::max<int64_t>(bh * L.n_chunks * L.g_items, n_g));
      const int blocks = (int)std::min<int64_t>(1024, std::max<int64_t>(1, (work + 255) / 256));
      build_work_lists_kernel<<<blocks, 256, 0, stream>>>(bp);
      if ((e = cudaGetLastError()) != cudaSuccess)
        return fail_fmt(SA_ERR_CUDA, "work-list launch: %s", cudaGetErrorString(e));
    }
  }

  DevProblem dp{};
  dp.q = q;
  dp.k = k;
  dp.v = v;
  dp.gq_src = q;
  dp.gk_src = k;
  dp.gv_src = v;
  dp.g_first = -1;  // the CUDA-core kernels read gathered rows
  dp.out = out;
  dp.lse = lse;
  dp.N = N;
  dp.D = D;
  dp.H = H;
  dp.half = std::min(p.half, N);
  dp.scale_log2 = scale * 1.4426950408889634f;
  dp.globals = reinterpret_cast<const int32_t *>(base + L.globals);
  dp.n_g = n_g;
  dp.g_pad = L.g_pad;
  dp.slots = reinterpret_cast<const Slot *>(base + L.slots);
  dp.n_slots = L.slot_off[H];
  dp.band = reinterpret_cast<const BandItem *>(base + L.band);
  dp.n_band = B * L.item_off[H];
  dp.BH = B * H;
  dp.gitems = reinterpret_cast<const GlobalItem *>(base + L.global);
  dp.n_gitems = (int)(bh * L.n_chunks * L.g_items);
  dp.n_chunks = L.n_chunks;
  dp.chunk_len = L.chunk_len;
  dp.part_sets = L.n_chunks;
  dp.part_sub = 1;
  dp.g_alt = 0;  // the CUDA-core kernels: one partial set per chunk
  dp.g_packed = 0;
  dp.qg = base + L.qg;
  dp.kg = base + L.kg;
  dp.vg = base + L.vg;
  dp.part_o = reinterpret_cast<float *>(base + L.part_o);
  dp.part_ml = reinterpret_cast<float *>(base + L.part_ml);
  dp.err = nullptr;  // the CUDA-core kernels have no waits that could stall

  const int BH = B * H;
  if (dp.n_g > 0 && (e = launch_gather(dp, BH, dtype, stream)) != cudaSuccess)
    return fail_fmt(SA_ERR_CUDA, "gather launch: %s", cudaGetErrorString(e));
  if ((e = launch_band_simt(dp, dtype, stream)) != cudaSuccess)
    return fail_fmt(SA_ERR_CUDA, "band launch: %s", cudaGetErrorString(e));
  if (dp.n_g > 0) {
    if ((e = launch_global_simt(dp, dtype, stream)) != cudaSuccess)
      return fail_fmt(SA_ERR_CUDA, "global-row launch: %s", cudaGetErrorString(e));
    if ((e = launch_merge(dp, BH, dtype, stream)) != cudaSuccess)
      return fail_fmt(SA_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
  }
  return SA_OK;
}
