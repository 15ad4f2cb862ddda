// sa_internal.h -- structures shared by the host scheduler and the kernels.
#pragma once

#include <cstdint>
#include <string>
#include <utility>
#include <vector>

#include "sa.h"

namespace sa {

// One residue class of one dilation value: positions r, r+d, r+2d, ... (< N).
// A dilated band |i-j| <= half*d, d | (i-j) is an ordinary band of half-width
// `half` on each class, so every kernel works in class coordinates t, with
// position = r + d*t and t in [0, len).
struct Slot {
  int32_t d;
  int32_t r;
  int32_t len;  // ceil((N - r) / d)
  int32_t pad;
};

// One CTA of band work: query tiles q_tile, q_tile+1, ... (nq of them, class
// coordinates, `rows` rows each) of head bh in residue class `slot`.  For query
// tile u the key tiles k_lo[u]..k_hi[u] (inclusive, `key_tile` keys each)
// intersect the band; flags bit u says whether any global key falls inside
// that query tile's band reach (so the global tile must drop duplicates).
struct BandItem {
  int32_t bh;
  int32_t slot;
  int32_t q_tile;
  int32_t flags;
  int32_t k_lo[2];
  int32_t k_hi[2];
};

// One CTA of the global-row pass: head bh, key chunk `chunk` (keys
// [chunk*chunk_len, min(N, (chunk+1)*chunk_len))), global-row tile `g_tile`.
struct GlobalItem {
  int32_t bh;
  int32_t chunk;
  int32_t g_tile;
  int32_t pad;
};

// Host-side description of one call.  Two mask patterns share every kernel:
//   band (chunk == 0): row i scores |i-j| <= half*d, d | (i-j), plus the globals;
//   chunked (chunk > 0): positions [0, memory) are the globals (GMAT memory),
//   and a main position i >= memory scores the main positions of its chunk,
//   (i-memory)/chunk, plus the memory.
struct Problem {
  int B, H, N, D;
  int window, half;
  std::vector<int32_t> dilation;  // per head (all 1 for the chunked pattern)
  std::vector<int32_t> globals;   // sorted, unique
  float scale;
  sa_dtype dtype;
  int chunk = 0;   // chunk length C of the chunked pattern, 0 for the band pattern
  int memory = 0;  // memory tokens M of the chunked pattern
};

// Non-global keys of row t (class coordinate; len positions in the class), as
// the interval [lo, hi]: the band t-half..t+half, or the row's chunk.  Rows
// inside the memory (global rows, recomputed densely) take chunk 0.  Both lo
// and hi never decrease with t, so a tile of rows reads keys lo(first row) ..
// hi(last row).
#if defined(__CUDACC__)
__host__ __device__
#endif
inline void row_keys(int half, int chunk, int memory, int len, int t, int &lo, int &hi) {
  if (chunk > 0) {
    const int c = t >= memory ? (t - memory) / chunk : 0;
    lo = memory + c * chunk;
    hi = (lo + chunk < len ? lo + chunk : len) - 1;
  } else {
    lo = t - half;
    hi = (t + half < len - 1 ? t + half : len - 1);
  }
}

// Tiling of one kernel family.
struct Tiling {
  int rows;         // query rows per tile
  int q_tiles;      // query tiles per CTA (1 or 2)
  int key_tile;     // keys per band tile
  int g_tile;       // the gathered global rows are padded to a multiple of this
  int g_item_rows;  // global query rows per CTA of the global-row pass
  int target_ctas;  // CTAs wanted for the global-row pass (separate launch)
  int max_slots;    // residue classes one launch can address (groups items)
  // Tensor-core family: the global-row work runs on CTAs of its own inside the
  // band launch (one CTA per SM, `sms` SMs), each query tile of such a CTA
  // taking every other key tile of the chunk (two chains of dependent MMAs per
  // SM); at most 64 global rows are packed two key halves to a 128-row tile.
  int sms = 0;
  bool fuse_global = false;
};

// Full launch schedule of one problem for one tiling.
struct Schedule {
  std::vector<Slot> slots;
  std::vector<int32_t> head_slot0;  // first slot index of each head's dilation
  std::vector<BandItem> band;          // grouped by slot group, longest first
  std::vector<int32_t> group_begin;    // band[group_begin[g] .. group_begin[g+1])
  std::vector<GlobalItem> global;
  int n_chunks = 0, chunk_len = 0, g_pad = 0;
  // Global-row partials: sets per head (key chunks, or two per chunk when the
  // two query tiles of a CTA take alternate key tiles), and rows per global
  // within a set (2 when the global rows are packed: one partial per key half).
  int part_sets = 0, part_sub = 1;
  bool g_alt = false, g_packed = false;
  // CTAs of the band launch that run global-row items (0: a separate launch)
  // and the CTAs that run band items.
  int g_ctas = 0, band_ctas = 0;
  int64_t band_tile_pairs = 0;  // executed (query tile, key tile) pairs
  std::vector<int32_t> globals_sorted;  // the global set the schedule was built for
};

// Host scheduler (sa_schedule.cpp).
std::string validate(const Problem &p);
std::vector<int32_t> global_set(const int32_t *idx, int n);
Schedule build_schedule(const Problem &p, const Tiling &t);
int64_t pairs_of_head(int N, int half, int d, const std::vector<int32_t> &globals);
int64_t pairs_chunked(int N, int memory, int chunk);
// About `want` key chunks of the N keys, each a multiple of `align` long (at
// most max_chunks): (chunk length, chunk count).
std::pair<int, int> key_chunks(int N, int64_t want, int64_t align, int64_t max_chunks);

// Sets the thread-local message that sa_last_error() returns; returns s.
sa_status record_error(sa_status s, const char *message);

}  // namespace sa
