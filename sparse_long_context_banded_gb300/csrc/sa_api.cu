// sa_api.cu -- the C ABI: argument checks, schedule cache, scratch, launches.
//
// One sa_forward call enqueues, on the caller's stream:
//   1. gather    -- q/k/v rows of a scattered global set into compact buffers
//                   (contiguous globals are read in place on the tensor cores)
//   2. band      -- per query tile: the key tiles of its band, then the global
//                   key tile(s); writes every row of `out` (global rows too).
//      global    -- the global rows against all N keys, split over key chunks,
//                   each CTA leaving partials (max, sum, unnormalised output).
//                   On the tensor cores both kinds of work run in one launch,
//                   on CTAs of their own (the global rows' CTAs read K and V
//                   while the band CTAs compute); on the CUDA cores, and when
//                   one launch cannot address every residue class, the global
//                   rows are a launch of their own.
//   3. merge     -- combines the partials and overwrites the global rows
// Steps 1 and 3 and the global-row work run only when the global set is not
// empty.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "sa.h"
#include "sa_internal.h"
#include "sa_kernels.h"
#include "sa_tc.h"

#include <nvtx3/nvToolsExt.h>

namespace sa {
namespace {

thread_local std::string t_last_error;

sa_status fail(sa_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

// A failed runtime call also leaves its error as the thread's "last error",
// which a later launch check (cudaGetLastError after a launch) would report as
// its own: once recorded here, the error is consumed (a sticky error, which
// poisons the context, stays whatever is done).
sa_status cuda_fail(cudaError_t e, const char *what) {
  cudaGetLastError();
  return fail(SA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

sa_status no_memory(cudaError_t e, const char *what, size_t bytes) {
  cudaGetLastError();
  return fail(SA_ERR_NO_MEMORY, "%s of %zu bytes: %s", what, bytes, cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------
// per-device state: error word, scratch pool, cached schedules
//
// One mutex guards this state; it is held only while a call looks up or
// builds its schedule and while it hands the schedule back, never across the
// launches.  A schedule evicted from the cache is retired: its device buffers
// are freed once no call is still enqueuing with it and every event recorded
// after a call that used it has completed (no device-wide synchronisation).  A
// schedule used by a call under stream capture is never freed, since the
// captured graph may run it at any later time.

struct DeviceSchedule {
  Schedule host;
  Slot *slots = nullptr;
  BandItem *band = nullptr;
  GlobalItem *global = nullptr;
  int32_t *globals = nullptr;
  int active = 0;                       // calls between lookup and release
  std::vector<cudaEvent_t> inflight;    // recorded after each call that used it
  bool captured = false;                // used under stream capture: keep forever
};

struct DeviceState {
  int *err = nullptr;
  cudaMemPool_t pool = nullptr;
  int sms = 0;
  std::map<std::string, std::unique_ptr<DeviceSchedule>> schedules;
  std::vector<std::unique_ptr<DeviceSchedule>> retired;
  std::vector<cudaEvent_t> spare_events;
};

std::mutex g_mutex;
std::map<int, std::unique_ptr<DeviceState>> g_devices;
constexpr size_t kMaxCachedSchedules = 256;

sa_status device_state(int dev, DeviceState **out) {
  auto it = g_devices.find(dev);
  if (it != g_devices.end()) {
    *out = it->second.get();
    return SA_OK;
  }
  auto ds = std::make_unique<DeviceState>();
  cudaError_t e = cudaMalloc(&ds->err, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
  e = cudaMemset(ds->err, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
  e = cudaDeviceGetAttribute(&ds->sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  cudaMemPoolProps props{};
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = cudaMemLocationTypeDevice;
  props.location.id = dev;
  // SA_POOL_MAX_BYTES (decimal, read once per device) caps the pool, so that
  // the out-of-memory path can be exercised without filling the device
  if (const char *cap = std::getenv("SA_POOL_MAX_BYTES")) {
    const unsigned long long c = std::strtoull(cap, nullptr, 10);
    if (c > 0) props.maxSize = (size_t)c;
  }
  e = cudaMemPoolCreate(&ds->pool, &props);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
  uint64_t keep = ~0ull;  // keep freed scratch in the pool between calls
  cudaMemPoolSetAttribute(ds->pool, cudaMemPoolAttrReleaseThreshold, &keep);
  *out = ds.get();
  g_devices[dev] = std::move(ds);
  return SA_OK;
}

// Schedule buffers come from the device's stream-ordered pool, so that
// freeing a retired one never synchronises the device.
template <typename X>
sa_status upload(const std::vector<X> &v, X **dst, cudaMemPool_t pool, cudaStream_t stream) {
  *dst = nullptr;
  if (v.empty()) return SA_OK;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(dst), sizeof(X) * v.size(), pool,
                                          stream);
  if (e != cudaSuccess) {
    *dst = nullptr;
    return no_memory(e, "schedule buffer", sizeof(X) * v.size());
  }
  e = cudaMemcpyAsync(*dst, v.data(), sizeof(X) * v.size(), cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_fail(e, "copy of the schedule");
  return SA_OK;
}

void free_schedule(DeviceSchedule &s, cudaStream_t stream) {
  void *bufs[4] = {s.slots, s.band, s.global, s.globals};
  for (void *b : bufs)
    if (b) cudaFreeAsync(b, stream);
  s.slots = nullptr;
  s.band = nullptr;
  s.global = nullptr;
  s.globals = nullptr;
}

// Drops the completed events of a schedule (returned to the spare list).
void prune_events(DeviceState &ds, DeviceSchedule &s) {
  size_t keep = 0;
  for (cudaEvent_t ev : s.inflight) {
    if (cudaEventQuery(ev) == cudaSuccess)
      ds.spare_events.push_back(ev);
    else
      s.inflight[keep++] = ev;
  }
  s.inflight.resize(keep);
}

// Frees the retired schedules that nothing can still read (the frees are
// enqueued on `stream`, which is not capturing).
void collect_retired(DeviceState &ds, cudaStream_t stream) {
  size_t keep = 0;
  for (auto &r : ds.retired) {
    prune_events(ds, *r);
    if (r->active == 0 && r->inflight.empty() && !r->captured)
      free_schedule(*r, stream);
    else
      ds.retired[keep++] = std::move(r);
  }
  ds.retired.resize(keep);
}

std::string schedule_key(const Problem &p, int family) {
  std::string k;
  auto put = [&k](const void *x, size_t n) { k.append(static_cast<const char *>(x), n); };
  int head[9] = {family, p.B, p.H, p.N, p.D, p.window, (int)p.globals.size(), p.chunk, p.memory};
  put(head, sizeof head);
  put(p.dilation.data(), sizeof(int32_t) * p.dilation.size());
  put(p.globals.data(), sizeof(int32_t) * p.globals.size());
  return k;
}

// Looks up (or builds and uploads) the schedule and marks it in use; the call
// hands it back with release_schedule once its work is enqueued.  Schedules
// are immutable once uploaded, so calls on any stream may share them.  A new
// schedule is uploaded on `stream` and waited for, so it cannot be built
// while the stream is capturing.  Called with g_mutex held.
sa_status acquire_schedule(DeviceState &ds, const Problem &p, int family, const Tiling &t,
                           cudaStream_t stream, bool capturing, DeviceSchedule **out) {
  if (!capturing) collect_retired(ds, stream);
  const std::string key = schedule_key(p, family);
  auto it = ds.schedules.find(key);
  if (it != ds.schedules.end()) {
    it->second->active += 1;
    *out = it->second.get();
    return SA_OK;
  }
  if (capturing)
    return fail(SA_ERR_INVALID_ARG, "first call for this problem shape made while the stream is "
                "capturing: make one call outside capture first (it builds and uploads the "
                "schedule)");
  if (ds.schedules.size() >= kMaxCachedSchedules) {
    for (auto &kv : ds.schedules) ds.retired.push_back(std::move(kv.second));
    ds.schedules.clear();
    collect_retired(ds, stream);
  }
  auto s = std::make_unique<DeviceSchedule>();
  s->host = build_schedule(p, t);
  s->host.globals_sorted = p.globals;
  sa_status st;
  if ((st = upload(s->host.slots, &s->slots, ds.pool, stream)) != SA_OK ||
      (st = upload(s->host.band, &s->band, ds.pool, stream)) != SA_OK ||
      (st = upload(s->host.global, &s->global, ds.pool, stream)) != SA_OK ||
      (st = upload(s->host.globals_sorted, &s->globals, ds.pool, stream)) != SA_OK) {
    free_schedule(*s, stream);
    return st;
  }
  // later calls may come on other streams: the upload has to be complete
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    free_schedule(*s, stream);
    return cuda_fail(e, "upload of the schedule");
  }
  s->active = 1;
  *out = s.get();
  ds.schedules[key] = std::move(s);
  return SA_OK;
}

// Hands a schedule back after the call's work on `stream` is enqueued: an event
// recorded there marks when the device is done reading it.  Takes g_mutex.
void release_schedule(DeviceState &ds, DeviceSchedule &s, cudaStream_t stream, bool capturing) {
  std::lock_guard<std::mutex> lock(g_mutex);
  s.active -= 1;
  if (capturing) {
    s.captured = true;
    return;
  }
  prune_events(ds, s);
  cudaEvent_t ev = nullptr;
  if (!ds.spare_events.empty()) {
    ev = ds.spare_events.back();
    ds.spare_events.pop_back();
  } else if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
    s.captured = true;  // cannot track its last use: keep it
    return;
  }
  if (cudaEventRecord(ev, stream) != cudaSuccess) {
    ds.spare_events.push_back(ev);
    s.captured = true;
    return;
  }
  s.inflight.push_back(ev);
}

// ---------------------------------------------------------------------------
// profiling events (a lock of their own: launches happen outside g_mutex)

struct ProfileRecord {
  int stage;
  int launches;  // kernel launches between the two events
  cudaEvent_t start, stop;
};
struct Profiler {
  std::mutex mutex;
  bool on = false;
  std::vector<ProfileRecord> records;
  std::vector<cudaEvent_t> spare;
  cudaEvent_t get() {
    if (!spare.empty()) {
      cudaEvent_t e = spare.back();
      spare.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
} g_prof;

struct StageTimer {
  int stage;
  cudaStream_t stream;
  cudaEvent_t start = nullptr;
  // (no events for a call under stream capture: the graph would record them
  // at each replay, after the profile has been read)
  StageTimer(int s, cudaStream_t st, bool capturing) : stage(s), stream(st) {
    std::lock_guard<std::mutex> lock(g_prof.mutex);
    if (g_prof.on && !capturing) {
      start = g_prof.get();
      cudaEventRecord(start, stream);
    }
  }
  void done(int launches = 1) {
    if (start) {
      std::lock_guard<std::mutex> lock(g_prof.mutex);
      cudaEvent_t stop = g_prof.get();
      cudaEventRecord(stop, stream);
      g_prof.records.push_back({stage, launches, start, stop});
      start = nullptr;
    }
  }
};

// ---------------------------------------------------------------------------
// precision of the P V product on the bf16 tensor-core path

std::atomic<int> g_pv_mode{SA_PV_AUTO};

// Automatic choice: split P into two bf16 parts when the softmax of some row
// can concentrate on a few keys, where the rounding of single bf16 weights no
// longer averages out -- rows with fewer than kSplitMinKeys keys, or a score
// scale |scale| sqrt(D) above kSplitMaxScale (unit-variance q and k give
// scores of standard deviation |scale| sqrt(D)).
constexpr int kSplitMinKeys = 128;
constexpr float kSplitMaxScale = 1.25f;

bool split_p(const Problem &p) {
  const int mode = g_pv_mode.load(std::memory_order_relaxed);
  if (mode == SA_PV_SINGLE) return false;
  if (mode == SA_PV_SPLIT) return true;
  if (std::fabs(p.scale) * std::sqrt((float)p.D) > kSplitMaxScale) return true;
  // fewest keys of a non-global row: a band row at the sequence edge sees
  // half + 1 keys (of its residue class); a chunk row its chunk (the last
  // chunk may be short) plus the memory
  int64_t min_keys;
  if (p.chunk > 0) {
    const int64_t main = (int64_t)p.N - p.memory;
    const int64_t last = main > 0 ? (main % p.chunk == 0 ? p.chunk : main % p.chunk) : p.chunk;
    min_keys = std::min<int64_t>(p.chunk, last) + p.memory;
  } else {
    int64_t shortest = p.N;
    for (int d : p.dilation) shortest = std::min<int64_t>(shortest, ((int64_t)p.N + d - 1) / d);
    min_keys = std::min<int64_t>((int64_t)p.half + 1, shortest) + (int64_t)p.globals.size();
  }
  return min_keys < kSplitMinKeys;
}

// ---------------------------------------------------------------------------

// The problem of one call, checked before anything is enqueued: every
// argument but the device pointers.
sa_status build_problem(int B, int H, int N, int D, int window, const int32_t *dilation,
                        const int32_t *global_idx, int n_global, float scale, sa_dtype dtype,
                        int chunk, int memory, Problem *out) {
  if (n_global < 0) return fail(SA_ERR_INVALID_ARG, "n_global must be >= 0");
  if (n_global > 0 && !global_idx)
    return fail(SA_ERR_INVALID_ARG, "global_idx is null but n_global = %d", n_global);
  if (H < 1) return fail(SA_ERR_INVALID_ARG, "H must be >= 1 (got %d)", H);
  Problem &p = *out;
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
  p.chunk = chunk;
  p.memory = memory;
  for (int i = 0; i < n_global; ++i)
    if (global_idx[i] < 0 || global_idx[i] >= N)
      return fail(SA_ERR_INVALID_ARG, "global_idx[%d] = %d outside [0, %d)", i, global_idx[i], N);
  p.globals = global_set(global_idx, n_global);
  std::string why = validate(p);
  if (!why.empty()) return fail(SA_ERR_INVALID_ARG, "%s", why.c_str());
  if (D != 64 && D != 128) return fail(SA_ERR_UNSUPPORTED, "D = %d (supported: 64, 128)", D);
  if ((int)p.globals.size() > SA_MAX_GLOBALS)
    return fail(SA_ERR_UNSUPPORTED, "%d distinct globals (at most %d)", (int)p.globals.size(),
                SA_MAX_GLOBALS);
  if (dtype == SA_TF32 && !tc_supports(dtype, D))
    return fail(SA_ERR_UNSUPPORTED, "SA_TF32 supports D = 64 (got %d)", D);
  return SA_OK;
}

sa_status forward_impl(const void *q, const void *k, const void *v, void *out, float *lse,
                       int B, int H, int N, int D, int window, const int32_t *dilation,
                       const int32_t *global_idx, int n_global, float scale, sa_dtype dtype,
                       cudaStream_t stream, int chunk = 0, int memory = 0,
                       const void *q_glob = nullptr, const void *k_glob = nullptr,
                       const void *v_glob = nullptr) {
  if (!q || !k || !v || !out) return fail(SA_ERR_INVALID_ARG, "q, k, v and out must be non-null");
  if (!q_glob) q_glob = q;
  if (!k_glob) k_glob = k;
  if (!v_glob) v_glob = v;
  const void *ptrs[7] = {q, k, v, out, q_glob, k_glob, v_glob};
  for (int i = 0; i < 7; ++i)
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0)
      return fail(SA_ERR_INVALID_ARG, "q, k, v, out (and the global projections) must be "
                  "16-byte aligned");
  if (reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return fail(SA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  Problem p;
  sa_status vst = build_problem(B, H, N, D, window, dilation, global_idx, n_global, scale, dtype,
                                chunk, memory, &p);
  if (vst != SA_OK) return vst;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  const bool capturing = cs != cudaStreamCaptureStatusNone;

  // bf16 -> tensor cores (kind::f16); tf32 (fp32 in memory, D = 64) -> tensor
  // cores (kind::tf32, no cast of the inputs); fp32 -> CUDA cores, fp32 throughout
  const bool tc = tc_supports(dtype, D);
  const bool precise = tc && dtype == SA_BF16 && split_p(p);

  DeviceState *ds = nullptr;
  DeviceSchedule *sched = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    sa_status st = device_state(dev, &ds);
    if (st != SA_OK) return st;
    const Tiling tiling = tc ? tc_tiling(D, ds->sms) : kSimtTiling;
    st = acquire_schedule(*ds, p, tc ? 1 : 0, tiling, stream, capturing, &sched);
    if (st != SA_OK) return st;
  }
  // the schedule is handed back once everything is enqueued, on every path
  struct Release {
    DeviceState *ds;
    DeviceSchedule *s;
    cudaStream_t stream;
    bool capturing;
    ~Release() { release_schedule(*ds, *s, stream, capturing); }
  } release{ds, sched, stream, capturing};
  const Schedule &hs = sched->host;

  DevProblem dp{};
  dp.q = q;
  dp.k = k;
  dp.v = v;
  dp.gq_src = q_glob;
  dp.gk_src = k_glob;
  dp.gv_src = v_glob;
  dp.out = out;
  dp.lse = lse;
  dp.N = N;
  dp.D = D;
  dp.H = H;
  dp.half = std::min(p.half, p.N);  // a wider band changes nothing
  dp.chunk = p.chunk;
  dp.memory = p.memory;
  dp.scale_log2 = scale * 1.4426950408889634f;
  dp.globals = sched->globals;
  dp.n_g = (int)p.globals.size();
  dp.g_pad = hs.g_pad;
  // contiguous globals (a first token, a memory prefix): the tensor-core kernels
  // read them through views of the inputs, and nothing is gathered
  dp.g_first = -1;
  if (tc && !p.globals.empty() &&
      p.globals.back() - p.globals.front() + 1 == (int32_t)p.globals.size())
    dp.g_first = p.globals.front();
  dp.slots = sched->slots;
  dp.n_slots = (int)hs.slots.size();
  dp.band = sched->band;
  dp.n_band = (int)hs.band.size();
  dp.BH = B * H;
  dp.gitems = sched->global;
  dp.n_gitems = (int)hs.global.size();
  dp.n_chunks = hs.n_chunks;
  dp.chunk_len = hs.chunk_len;
  dp.part_sets = hs.part_sets;
  dp.part_sub = hs.part_sub;
  dp.g_alt = hs.g_alt ? 1 : 0;
  dp.g_packed = hs.g_packed ? 1 : 0;
  dp.err = ds->err;

  const int BH = B * H;
  const size_t esize = dtype == SA_BF16 ? 2 : 4;
  const size_t g_rows = (size_t)BH * hs.g_pad * D;
  const size_t part_rows = (size_t)BH * hs.part_sets * hs.g_pad;
  size_t off_q = 0, off_k = 0, off_v = 0, off_po = 0, off_ml = 0, total = 0;
  auto carve = [&total](size_t bytes) {
    size_t at = total;
    total += (bytes + 255) & ~size_t(255);
    return at;
  };
  if (dp.n_g > 0) {
    if (dp.g_first < 0) {
      off_q = carve(g_rows * esize);
      off_k = carve(g_rows * esize);
      off_v = carve(g_rows * esize);
    }
    off_po = carve(part_rows * D * sizeof(float));
    off_ml = carve(part_rows * 2 * sizeof(float));
  }
  // fp32 on the tensor cores: transposed values (per slot, the global-row
  // pass's, the gathered globals')
  const bool tf32 = dtype == SA_TF32;
  size_t off_vts = 0, off_vtp = 0, off_vtg = 0;
  if (tf32) {
    size_t per_slot = 0;
    for (const Slot &sl : hs.slots) per_slot += (size_t)BH * D * values_len_pad(sl.len) * 4;
    off_vts = carve(per_slot);
    if (dp.n_g > 0) {
      off_vtp = carve((size_t)BH * D * values_len_pad(N) * 4);
      off_vtg = carve((size_t)BH * D * hs.g_pad * 4);
    }
  }
  char *scratch = nullptr;
  if (total > 0) {
    e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&scratch), total, ds->pool, stream);
    if (e != cudaSuccess)
      return no_memory(e, "scratch", total);
    if (dp.g_first < 0) {
      dp.qg = scratch + off_q;
      dp.kg = scratch + off_k;
      dp.vg = scratch + off_v;
    }
    dp.part_o = reinterpret_cast<float *>(scratch + off_po);
    dp.part_ml = reinterpret_cast<float *>(scratch + off_ml);
    if (tf32) {
      dp.vT_slots = reinterpret_cast<float *>(scratch + off_vts);
      if (dp.n_g > 0) {
        dp.vT_plain = reinterpret_cast<float *>(scratch + off_vtp);
        dp.vgT = reinterpret_cast<float *>(scratch + off_vtg);
      }
    }
  }

  sa_status result = SA_OK;
  auto step = [&](int stage, const char *range, auto &&launch, const char *what, int launches = 1) {
    if (result != SA_OK) return;
    nvtxRangePushA(range);
    StageTimer timer(stage, stream, capturing);
    cudaError_t le = launch();
    timer.done(launches);
    nvtxRangePop();
    if (le != cudaSuccess) result = cuda_fail(le, what);
  };
  if (dp.n_g > 0 && dp.g_first < 0)
    step(0, "sa.gather", [&] { return launch_gather(dp, BH, dtype, stream); }, "gather launch");
  if (tf32) {
    step(0, "sa.transpose_values", [&] {
      size_t off = 0;
      for (const Slot &sl : hs.slots) {
        const int lp = values_len_pad(sl.len);
        cudaError_t le = launch_transpose_values(static_cast<const float *>(v), dp.vT_slots + off, N,
                                                 D, sl.r, sl.d, sl.len, lp, BH, stream);
        if (le != cudaSuccess) return le;
        off += (size_t)BH * D * lp;
      }
      if (dp.n_g == 0) return cudaSuccess;
      cudaError_t le = launch_transpose_values(static_cast<const float *>(dp.gv_src), dp.vT_plain, N,
                                               D, 0, 1, N, values_len_pad(N), BH, stream);
      if (le != cudaSuccess) return le;
      if (dp.g_first >= 0)  // straight from the contiguous rows of v
        return launch_transpose_values(static_cast<const float *>(v), dp.vgT, N, D, dp.g_first, 1,
                                       std::min(hs.g_pad, N - dp.g_first), hs.g_pad, BH, stream);
      return launch_transpose_values(static_cast<const float *>(dp.vg), dp.vgT, hs.g_pad, D, 0, 1,
                                     hs.g_pad, hs.g_pad, BH, stream);
    }, "value transposition launch", (int)hs.slots.size() + (dp.n_g > 0 ? 2 : 0));
  }
  // tensor cores: the global-row items run on CTAs of the band launch when
  // the schedule assigns them some (hs.g_ctas), else in a launch of their own
  const bool fused = tc && dp.n_g > 0 && hs.g_ctas > 0;
  if (tc)
    step(1, fused ? "sa.band+global_rows" : "sa.band", [&] {
      return launch_band_tc(dp, dtype, precise, hs.slots.data(), (int)hs.slots.size(), hs.group_begin,
                            BH, ds->sms, fused ? hs.g_ctas : 0, hs.band_ctas, stream);
    }, "band (tensor-core) launch", (int)hs.group_begin.size() - 1);
  else
    step(1, "sa.band", [&] { return launch_band_simt(dp, dtype, stream); }, "band launch");
  if (dp.n_g > 0) {
    if (tc && !fused)
      step(2, "sa.global_rows", [&] { return launch_global_tc(dp, dtype, precise, BH, ds->sms, stream); },
           "global-row (tensor-core) launch");
    else if (!tc)
      step(2, "sa.global_rows", [&] { return launch_global_simt(dp, dtype, stream); }, "global-row launch");
    step(3, "sa.merge", [&] { return launch_merge(dp, BH, dtype, stream); }, "merge launch");
  }
  if (scratch) {
    e = cudaFreeAsync(scratch, stream);
    if (e != cudaSuccess && result == SA_OK) result = cuda_fail(e, "cudaFreeAsync(scratch)");
  }
  return result;
}

}  // namespace

sa_status record_error(sa_status s, const char *message) {
  t_last_error = message;
  return s;
}

}  // namespace sa

using namespace sa;

extern "C" sa_status sa_forward(const void *q, const void *k, const void *v, void *out, int B,
                                int H, int N, int D, int window, const int32_t *dilation,
                                const int32_t *global_idx, int n_global, float scale,
                                sa_dtype dtype, sa_stream_t stream) {
  return forward_impl(q, k, v, out, nullptr, B, H, N, D, window, dilation, global_idx,
                      n_global, scale, dtype, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" sa_status sa_forward_lse(const void *q, const void *k, const void *v, void *out,
                                    float *lse, int B, int H, int N, int D, int window,
                                    const int32_t *dilation, const int32_t *global_idx,
                                    int n_global, float scale, sa_dtype dtype,
                                    sa_stream_t stream) {
  return forward_impl(q, k, v, out, lse, B, H, N, D, window, dilation, global_idx, n_global,
                      scale, dtype, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" sa_status sa_forward_chunked(const void *q, const void *k, const void *v, void *out,
                                        float *lse, int B, int H, int N, int D, int n_memory,
                                        int chunk, float scale, sa_dtype dtype,
                                        sa_stream_t stream) {
  if (chunk < 1) return fail(SA_ERR_INVALID_ARG, "chunk must be >= 1 (got %d)", chunk);
  if (n_memory < 0 || n_memory > N)
    return fail(SA_ERR_INVALID_ARG, "n_memory = %d outside [0, N = %d]", n_memory, N);
  if (n_memory > SA_MAX_GLOBALS)
    return fail(SA_ERR_UNSUPPORTED, "%d memory tokens (at most %d)", n_memory, SA_MAX_GLOBALS);
  std::vector<int32_t> mem(n_memory);
  for (int i = 0; i < n_memory; ++i) mem[i] = i;
  return forward_impl(q, k, v, out, lse, B, H, N, D, 0, nullptr, mem.data(), n_memory, scale,
                      dtype, reinterpret_cast<cudaStream_t>(stream), chunk, n_memory);
}

extern "C" sa_status sa_forward_global_proj(const void *q, const void *k, const void *v,
                                            const void *q_global, const void *k_global,
                                            const void *v_global, void *out, float *lse, int B,
                                            int H, int N, int D, int window,
                                            const int32_t *dilation, const int32_t *global_idx,
                                            int n_global, float scale, sa_dtype dtype,
                                            sa_stream_t stream) {
  if (!q_global || !k_global || !v_global)
    return fail(SA_ERR_INVALID_ARG, "q_global, k_global and v_global must be non-null");
  return forward_impl(q, k, v, out, lse, B, H, N, D, window, dilation, global_idx, n_global,
                      scale, dtype, reinterpret_cast<cudaStream_t>(stream), 0, 0, q_global,
                      k_global, v_global);
}

// ---------------------------------------------------------------------------
// Host buffers.  Each (b, h) slice is a problem of its own (its mask, its
// global rows and its output involve that slice only), so the call cuts the
// slices into groups of consecutive heads and runs a three-stage pipeline
// over two sets of device buffers: group g+1's inputs are copied in while
// group g is computed and group g-1's output is copied out.

namespace sa {
namespace {

constexpr int kHostGroups = 16;                      // groups wanted per call
constexpr int64_t kHostGroupMinBytes = 32ll << 20;   // inputs of one group, at least

// Batches b0 .. b0+nb-1, heads h0 .. h0+nh-1 of each (nb > 1 only with all heads).
struct HostGroup {
  int b0, nb, h0, nh;
};

std::vector<HostGroup> host_groups(int B, int H, int64_t head_input_bytes, int heads_per_group) {
  const int64_t units = (int64_t)B * H;
  int64_t g = heads_per_group;
  if (g <= 0) {
    const int64_t min_heads = (kHostGroupMinBytes + head_input_bytes - 1) / head_input_bytes;
    g = std::max<int64_t>({(units + kHostGroups - 1) / kHostGroups, min_heads, 1});
  }
  std::vector<HostGroup> groups;
  if (g < H) {
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; h += (int)g) groups.push_back({b, 1, h, (int)std::min<int64_t>(g, H - h)});
  } else {
    const int nb = (int)std::min<int64_t>(B, g / H);
    for (int b = 0; b < B; b += nb) groups.push_back({b, std::min(nb, B - b), 0, H});
  }
  return groups;
}

}  // namespace
}  // namespace sa

extern "C" sa_status sa_forward_host(const void *q, const void *k, const void *v, void *out,
                                     float *lse, int B, int H, int N, int D, int window,
                                     const int32_t *dilation, const int32_t *global_idx,
                                     int n_global, float scale, sa_dtype dtype,
                                     int heads_per_group) {
  if (!q || !k || !v || !out) return fail(SA_ERR_INVALID_ARG, "q, k, v and out must be non-null");
  if (heads_per_group < 0)
    return fail(SA_ERR_INVALID_ARG, "heads_per_group must be >= 0 (got %d)", heads_per_group);
  {
    Problem p;  // every argument checked before any copy
    sa_status st = build_problem(B, H, N, D, window, dilation, global_idx, n_global, scale, dtype,
                                 0, 0, &p);
    if (st != SA_OK) return st;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceState *ds = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    sa_status st = device_state(dev, &ds);
    if (st != SA_OK) return st;
  }
  const size_t es = dtype == SA_BF16 ? 2 : 4;
  const size_t head_elems = (size_t)N * D;
  const std::vector<HostGroup> groups =
      host_groups(B, H, (int64_t)(3 * head_elems * es), heads_per_group);
  size_t max_heads = 0;
  for (const HostGroup &g : groups) max_heads = std::max(max_heads, (size_t)g.nb * g.nh);
  auto round256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t r = round256(max_heads * head_elems * es);  // one tensor of one set
  const size_t set_bytes = 4 * r + (lse ? round256(max_heads * N * sizeof(float)) : 0);

  // stages: 0 copies in, 1 computes, 2 copies out; per buffer set, the event
  // each stage records after its work on that set
  cudaStream_t st[3] = {nullptr, nullptr, nullptr};
  cudaEvent_t ev[3][2] = {};
  char *set[2] = {nullptr, nullptr};
  sa_status result = SA_OK;
  auto check = [&result](cudaError_t ce, const char *what) {
    if (ce != cudaSuccess && result == SA_OK) result = cuda_fail(ce, what);
    return result == SA_OK;
  };
  for (int i = 0; i < 3 && result == SA_OK; ++i)
    check(cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking), "cudaStreamCreate");
  for (int i = 0; i < 3 && result == SA_OK; ++i)
    for (int b = 0; b < 2 && result == SA_OK; ++b)
      check(cudaEventCreateWithFlags(&ev[i][b], cudaEventDisableTiming), "cudaEventCreate");
  // both sets are allocated on the copy-in stream; every later use waits for
  // an event recorded there after the allocation
  for (int b = 0; b < 2 && result == SA_OK && b < (int)groups.size(); ++b) {
    e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&set[b]), set_bytes, ds->pool, st[0]);
    if (e != cudaSuccess)
      result = no_memory(e, "host-call buffers", set_bytes);
  }
  for (size_t gi = 0; gi < groups.size() && result == SA_OK; ++gi) {
    const HostGroup &g = groups[gi];
    const int b = (int)(gi & 1);
    const size_t u0 = (size_t)g.b0 * H + g.h0, nu = (size_t)g.nb * g.nh;
    const size_t off = u0 * head_elems * es, bytes = nu * head_elems * es;
    char *dq = set[b], *dk = dq + r, *dv = dk + r, *dout = dv + r;
    float *dlse = lse ? reinterpret_cast<float *>(dout + r) : nullptr;
    // group gi-2 used this set: its inputs must have been read before they are
    // overwritten, its output copied out before it is overwritten
    if (gi >= 2 && !check(cudaStreamWaitEvent(st[0], ev[1][b], 0), "cudaStreamWaitEvent")) break;
    if (!check(cudaMemcpyAsync(dq, static_cast<const char *>(q) + off, bytes,
                               cudaMemcpyHostToDevice, st[0]), "copy of q to the device") ||
        !check(cudaMemcpyAsync(dk, static_cast<const char *>(k) + off, bytes,
                               cudaMemcpyHostToDevice, st[0]), "copy of k to the device") ||
        !check(cudaMemcpyAsync(dv, static_cast<const char *>(v) + off, bytes,
                               cudaMemcpyHostToDevice, st[0]), "copy of v to the device") ||
        !check(cudaEventRecord(ev[0][b], st[0]), "cudaEventRecord") ||
        !check(cudaStreamWaitEvent(st[1], ev[0][b], 0), "cudaStreamWaitEvent") ||
        (gi >= 2 && !check(cudaStreamWaitEvent(st[1], ev[2][b], 0), "cudaStreamWaitEvent")))
      break;
    sa_status fs = forward_impl(dq, dk, dv, dout, dlse, g.nb, g.nh, N, D, window,
                                dilation ? dilation + g.h0 : nullptr, global_idx, n_global, scale,
                                dtype, st[1]);
    if (fs != SA_OK) {
      result = fs;
      break;
    }
    if (!check(cudaEventRecord(ev[1][b], st[1]), "cudaEventRecord") ||
        !check(cudaStreamWaitEvent(st[2], ev[1][b], 0), "cudaStreamWaitEvent") ||
        !check(cudaMemcpyAsync(static_cast<char *>(out) + off, dout, bytes,
                               cudaMemcpyDeviceToHost, st[2]), "copy of out to the host") ||
        (lse && !check(cudaMemcpyAsync(lse + u0 * N, dlse, nu * N * sizeof(float),
                                       cudaMemcpyDeviceToHost, st[2]), "copy of lse to the host")) ||
        !check(cudaEventRecord(ev[2][b], st[2]), "cudaEventRecord"))
      break;
  }
  // whatever was enqueued finishes before the host buffers are handed back
  // (a failure here is reported only when nothing failed before)
  for (int i = 0; i < 3; ++i)
    if (st[i]) check(cudaStreamSynchronize(st[i]), "stream synchronize");
  int word = 0;
  if (st[2]) {
    for (int b = 0; b < 2; ++b)
      if (set[b]) check(cudaFreeAsync(set[b], st[2]), "cudaFreeAsync(host-call buffers)");
    // the device error word, read (and cleared) as sa_sync_status does, but on
    // this call's own stream rather than the legacy default stream
    if (result == SA_OK &&
        check(cudaMemcpyAsync(&word, ds->err, sizeof(int), cudaMemcpyDeviceToHost, st[2]),
              "read error word") &&
        check(cudaStreamSynchronize(st[2]), "stream synchronize") && word != 0)
      check(cudaMemsetAsync(ds->err, 0, sizeof(int), st[2]), "clear error word");
    check(cudaStreamSynchronize(st[2]), "stream synchronize");
  }
  for (int i = 0; i < 3; ++i)
    for (int b = 0; b < 2; ++b)
      if (ev[i][b]) cudaEventDestroy(ev[i][b]);
  for (int i = 0; i < 3; ++i)
    if (st[i]) cudaStreamDestroy(st[i]);
  if (result != SA_OK) return result;
  if (word & kErrWaitTimeout)
    return fail(SA_ERR_TIMEOUT, "a kernel gave up on a stalled wait (error word 0x%x)", word);
  if (word != 0)
    return fail(SA_ERR_CUDA, "a kernel failed a device-side check (error word 0x%x)", word);
  return SA_OK;
}

extern "C" sa_status sa_forward_gather(const void *q, const void *k, const void *v,
                                       const int32_t *idx, void *out, float *lse, int B, int H,
                                       int Nq, int Nk, int D, int K, float scale,
                                       sa_dtype dtype, sa_stream_t stream) {
  if (!q || !k || !v || !out) return fail(SA_ERR_INVALID_ARG, "q, k, v and out must be non-null");
  if (K > 0 && !idx) return fail(SA_ERR_INVALID_ARG, "idx is null but K = %d", K);
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1)
    return fail(SA_ERR_INVALID_ARG, "B, H, Nq and Nk must be >= 1 (got %d, %d, %d, %d)", B, H, Nq, Nk);
  if (K < 0) return fail(SA_ERR_INVALID_ARG, "K must be >= 0 (got %d)", K);
  if (!std::isfinite(scale)) return fail(SA_ERR_INVALID_ARG, "scale must be finite");
  if (dtype != SA_BF16 && dtype != SA_FP32) return fail(SA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  const void *ptrs[4] = {q, k, v, out};
  for (int i = 0; i < 4; ++i)
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16 != 0)
      return fail(SA_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(idx) % 4 != 0 || reinterpret_cast<uintptr_t>(lse) % 4 != 0)
    return fail(SA_ERR_INVALID_ARG, "idx and lse must be 4-byte aligned");
  if (D != 64 && D != 128) return fail(SA_ERR_UNSUPPORTED, "D = %d (supported: 64, 128)", D);
  GatherProblem gp{};
  gp.q = q;
  gp.k = k;
  gp.v = v;
  gp.idx = idx;
  gp.out = out;
  gp.lse = lse;
  gp.rows = (int64_t)B * H * Nq;
  gp.Nq = Nq;
  gp.Nk = Nk;
  gp.K = K;
  gp.D = D;
  gp.scale_log2 = scale * 1.4426950408889634f;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
  StageTimer timer(1, s, cs != cudaStreamCaptureStatusNone);
  cudaError_t e = launch_gather_attention(gp, dtype, s);
  timer.done();
  if (e != cudaSuccess) return cuda_fail(e, "list-gather attention launch");
  return SA_OK;
}

extern "C" sa_status sa_count_pairs_chunked(int N, int n_memory, int chunk, int64_t *per_head) {
  if (N < 1) return fail(SA_ERR_INVALID_ARG, "N must be >= 1 (got %d)", N);
  if (chunk < 1) return fail(SA_ERR_INVALID_ARG, "chunk must be >= 1 (got %d)", chunk);
  if (n_memory < 0 || n_memory > N)
    return fail(SA_ERR_INVALID_ARG, "n_memory = %d outside [0, N = %d]", n_memory, N);
  if (!per_head) return fail(SA_ERR_INVALID_ARG, "per_head must be non-null");
  *per_head = pairs_chunked(N, n_memory, chunk);
  return SA_OK;
}

extern "C" sa_status sa_count_pairs(int N, int window, const int32_t *dilation, int H,
                                    const int32_t *global_idx, int n_global, int64_t *per_head,
                                    int64_t *total) {
  if (n_global < 0) return fail(SA_ERR_INVALID_ARG, "n_global must be >= 0");
  if (n_global > 0 && !global_idx)
    return fail(SA_ERR_INVALID_ARG, "global_idx is null but n_global = %d", n_global);
  if (H < 1) return fail(SA_ERR_INVALID_ARG, "H must be >= 1 (got %d)", H);
  Problem p;
  p.B = 1;
  p.H = H;
  p.N = N;
  p.D = 64;
  p.window = window;
  p.half = window / 2;
  if (dilation)
    p.dilation.assign(dilation, dilation + H);
  else
    p.dilation.assign(H, 1);
  p.scale = 1.f;
  p.dtype = SA_BF16;
  for (int i = 0; i < n_global; ++i)
    if (global_idx[i] < 0 || global_idx[i] >= N)
      return fail(SA_ERR_INVALID_ARG, "global_idx[%d] = %d outside [0, %d)", i, global_idx[i], N);
  p.globals = global_set(global_idx, n_global);
  std::string why = validate(p);
  if (!why.empty()) return fail(SA_ERR_INVALID_ARG, "%s", why.c_str());
  if ((int)p.globals.size() > SA_MAX_GLOBALS)
    return fail(SA_ERR_UNSUPPORTED, "%d distinct globals (at most %d)", (int)p.globals.size(),
                SA_MAX_GLOBALS);
  int64_t sum = 0;
  for (int h = 0; h < H; ++h) {
    const int64_t c = pairs_of_head(N, p.half, p.dilation[h], p.globals);
    if (per_head) per_head[h] = c;
    sum += c;
  }
  if (total) *total = sum;
  return SA_OK;
}

extern "C" const char *sa_last_error(void) { return t_last_error.c_str(); }

extern "C" sa_status sa_check_stalled_wait(uint32_t limit_us, sa_stream_t stream) {
  if (limit_us < 1 || limit_us > 2000000)
    return fail(SA_ERR_INVALID_ARG, "limit_us must be in [1, 2000000] (got %u)", limit_us);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceState *ds = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    sa_status st = device_state(dev, &ds);
    if (st != SA_OK) return st;
  }
  e = launch_stalled_wait_check(ds->err, limit_us, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stalled-wait check launch");
  return SA_OK;
}

extern "C" sa_status sa_sync_status(sa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int *word = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_devices.find(dev);
    if (it == g_devices.end()) return SA_OK;  // nothing ever ran here
    word = it->second->err;
  }
  int h = 0;
  e = cudaMemcpy(&h, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (h != 0) {
    cudaMemset(word, 0, sizeof(int));
    if (h & kErrWaitTimeout)
      return fail(SA_ERR_TIMEOUT, "a kernel gave up on a stalled wait (error word 0x%x)", h);
    return fail(SA_ERR_CUDA, "a kernel failed a device-side check (error word 0x%x)", h);
  }
  return SA_OK;
}

extern "C" sa_status sa_profile_begin(void) {
  std::lock_guard<std::mutex> lock(g_prof.mutex);
  for (auto &r : g_prof.records) {
    g_prof.spare.push_back(r.start);
    g_prof.spare.push_back(r.stop);
  }
  g_prof.records.clear();
  g_prof.on = true;
  return SA_OK;
}

extern "C" sa_status sa_profile_end(sa_profile *out) {
  std::lock_guard<std::mutex> lock(g_prof.mutex);
  g_prof.on = false;
  sa_profile res{};
  sa_status st = SA_OK;
  for (auto &r : g_prof.records) {
    cudaError_t e = cudaEventSynchronize(r.stop);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
    if (e != cudaSuccess && st == SA_OK) st = cuda_fail(e, "profile event");
    res.launches[r.stage] += r.launches;
    res.ms[r.stage] += ms;
    g_prof.spare.push_back(r.start);
    g_prof.spare.push_back(r.stop);
  }
  g_prof.records.clear();
  if (out) *out = res;
  return st;
}

extern "C" sa_status sa_set_pv_mode(sa_pv_mode mode) {
  if (mode != SA_PV_AUTO && mode != SA_PV_SINGLE && mode != SA_PV_SPLIT)
    return fail(SA_ERR_INVALID_ARG, "unknown P V mode %d", (int)mode);
  g_pv_mode.store((int)mode, std::memory_order_relaxed);
  return SA_OK;
}

extern "C" sa_pv_mode sa_get_pv_mode(void) {
  return (sa_pv_mode)g_pv_mode.load(std::memory_order_relaxed);
}

extern "C" int sa_uses_split_p(int N, int D, int window, const int32_t *dilation, int H,
                               const int32_t *global_idx, int n_global, int chunk, int n_memory,
                               float scale) {
  Problem p;
  p.B = 1;
  p.H = H < 1 ? 1 : H;
  p.N = N;
  p.D = D;
  p.window = window;
  p.half = window / 2;
  if (dilation && H >= 1)
    p.dilation.assign(dilation, dilation + H);
  else
    p.dilation.assign(p.H, 1);
  p.scale = scale;
  p.dtype = SA_BF16;
  p.chunk = chunk;
  p.memory = n_memory;
  if (global_idx && n_global > 0) p.globals = global_set(global_idx, n_global);
  return split_p(p) ? 1 : 0;
}

extern "C" const char *sa_version(void) { return "sa-gb300 0.2 (sm_103a)"; }
