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
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
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

// Device address of g_static_scratch on each device, resolved once per device
// with that device current.  In host code the symbol itself is only a host
// stand-in; kernels must be given this address instead.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
char *g_scratch_addr[kMaxDevices] = {};

sa_status static_scratch_address(int dev, char **out) {
  if (dev < 0 || dev >= kMaxDevices)
    return record_error(SA_ERR_UNSUPPORTED, "device ordinal beyond the static-scratch table");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess || !ptr) {
      std::string m = std::string("cudaGetSymbolAddress(static scratch): ") + cudaGetErrorString(e);
      return record_error(SA_ERR_CUDA, m.c_str());
    }
    g_scratch_addr[dev] = static_cast<char *>(ptr);
  }
  *out = g_scratch_addr[dev];
  return SA_OK;
}

struct Layout {
  size_t slots, band, global, globals, qg, kg, vg, part_o, part_ml, total;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

Layout layout_of(const Problem &p, const Schedule &s) {
  Layout L{};
  size_t at = 0;
  auto take = [&at](size_t bytes) {
    size_t here = at;
    at += round256(bytes);
    return here;
  };
  const size_t BH = (size_t)p.B * p.H;
  const size_t es = p.dtype == SA_BF16 ? 2 : 4;
  L.slots = take(sizeof(Slot) * s.slots.size());
  L.band = take(sizeof(BandItem) * s.band.size());
  L.global = take(sizeof(GlobalItem) * s.global.size());
  L.globals = take(sizeof(int32_t) * p.globals.size());
  const size_t g_rows = BH * s.g_pad * p.D;
  L.qg = take(g_rows * es);
  L.kg = take(g_rows * es);
  L.vg = take(g_rows * es);
  const size_t part_rows = BH * (size_t)s.part_sets * s.g_pad;
  L.part_o = take(part_rows * p.D * sizeof(float));
  L.part_ml = take(part_rows * 2 * sizeof(float));
  L.total = at;
  return L;
}

template <typename X>
cudaError_t put(char *base, size_t off, const std::vector<X> &v, cudaStream_t st) {
  if (v.empty()) return cudaSuccess;
  return cudaMemcpyAsync(base + off, v.data(), sizeof(X) * v.size(), cudaMemcpyHostToDevice, st);
}

sa_status fail_fmt(sa_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
sa_status fail_fmt(sa_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
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

  // Schedule; while the split-K partials would not fit, halve the number of
  // key chunks of the global-row pass (fewer, longer chunks, same result).
  Tiling t = kSimtTiling;
  Schedule s = build_schedule(p, t);
  Layout L = layout_of(p, s);
  const int g_items = p.globals.empty() ? 1 : (int)((p.globals.size() + t.g_item_rows - 1) / t.g_item_rows);
  while (L.total > kStaticScratchBytes && s.n_chunks > 1) {
    const int64_t want = (int64_t)(s.n_chunks / 2) * B * H * g_items;
    t.target_ctas = (int)std::min<int64_t>(want, INT32_MAX);
    s = build_schedule(p, t);
    L = layout_of(p, s);
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

  if ((e = put(base, L.slots, s.slots, stream)) != cudaSuccess ||
      (e = put(base, L.band, s.band, stream)) != cudaSuccess ||
      (e = put(base, L.global, s.global, stream)) != cudaSuccess ||
      (e = put(base, L.globals, p.globals, stream)) != cudaSuccess)
    return fail_fmt(SA_ERR_CUDA, "copy of the schedule into static scratch: %s",
                    cudaGetErrorString(e));

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
  dp.half = p.half;
  dp.scale_log2 = scale * 1.4426950408889634f;
  dp.globals = reinterpret_cast<const int32_t *>(base + L.globals);
  dp.n_g = (int)p.globals.size();
  dp.g_pad = s.g_pad;
  dp.slots = reinterpret_cast<const Slot *>(base + L.slots);
  dp.band = reinterpret_cast<const BandItem *>(base + L.band);
  dp.n_band = (int)s.band.size();
  dp.gitems = reinterpret_cast<const GlobalItem *>(base + L.global);
  dp.n_gitems = (int)s.global.size();
  dp.n_chunks = s.n_chunks;
  dp.chunk_len = s.chunk_len;
  dp.part_sets = s.part_sets;
  dp.part_sub = s.part_sub;
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
