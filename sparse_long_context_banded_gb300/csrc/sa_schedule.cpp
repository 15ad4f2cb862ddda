// sa_schedule.cpp -- argument checks, the global index set, the band-tile
// schedule and the exact in-mask pair count.  Host code, integer arithmetic.
//
// Mask (Ultralytics glossary "Longformer", section "How the Longformer
// attention works"): row i scores key j when |i-j| <= floor(w/2)*d and d
// divides i-j (the dilated sliding window; d = 1 is the plain window), and
// every row scores every global key while a global row scores every key.
// Global positions form a set: listing one twice changes nothing, as the
// section's mask-count example assigns True to a global row and column.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <numeric>
#include <tuple>
#include <utility>

#include "sa_internal.h"

namespace sa {

std::string validate(const Problem &p) {
  char buf[256];
  if (p.B < 1 || p.H < 1 || p.N < 1) {
    snprintf(buf, sizeof buf, "B, H, N must be >= 1 (got %d, %d, %d)", p.B, p.H, p.N);
    return buf;
  }
  if (p.window < 0) {
    snprintf(buf, sizeof buf, "window must be >= 0 (got %d)", p.window);
    return buf;
  }
  if ((int)p.dilation.size() != p.H) return "dilation must have H entries";
  for (int h = 0; h < p.H; ++h)
    if (p.dilation[h] < 1) {
      snprintf(buf, sizeof buf, "dilation[%d] = %d must be >= 1", h, p.dilation[h]);
      return buf;
    }
  for (int32_t g : p.globals)
    if (g < 0 || g >= p.N) {
      snprintf(buf, sizeof buf, "global index %d outside [0, %d)", g, p.N);
      return buf;
    }
  if (!std::isfinite(p.scale)) return "scale must be finite";
  if (p.chunk < 0) return "chunk must be >= 0";
  if (p.chunk > 0) {
    if (p.memory < 0 || p.memory > p.N) {
      snprintf(buf, sizeof buf, "memory tokens %d outside [0, %d]", p.memory, p.N);
      return buf;
    }
    for (int h = 0; h < p.H; ++h)
      if (p.dilation[h] != 1) return "the chunked pattern takes no dilation";
  }
  if (p.dtype != SA_BF16 && p.dtype != SA_FP32 && p.dtype != SA_TF32) return "unknown dtype";
  const double elems = (double)p.B * p.H * p.N * std::max(p.D, 1);
  if (elems > 9.0e18) return "tensor too large";
  return "";
}

std::vector<int32_t> global_set(const int32_t *idx, int n) {
  std::vector<int32_t> g(idx, idx + std::max(n, 0));
  std::sort(g.begin(), g.end());
  g.erase(std::unique(g.begin(), g.end()), g.end());
  return g;
}

// Number of t with |t| <= half and 0 <= i + t*d < N.
static inline int64_t band_len(int64_t N, int64_t half, int64_t d, int64_t i) {
  const int64_t lo = std::max(-half, -(i / d));
  const int64_t hi = std::min(half, (N - 1 - i) / d);
  return hi - lo + 1;
}

static inline bool in_band(int64_t half, int64_t d, int64_t i, int64_t j) {
  const int64_t diff = i - j;
  return (diff <= half * d && -diff <= half * d) && (diff % d == 0);
}

// |mask| of one head:
//   sum over non-global rows of (band length + globals outside the band)
//   + N per global row.
// The globals-inside-band term is counted from the globals' side (the band
// relation is symmetric), so the cost is O(N + |G|^2).
int64_t pairs_of_head(int N, int half, int d, const std::vector<int32_t> &G) {
  const int64_t n_g = (int64_t)G.size();
  int64_t band_all = 0;
  for (int64_t i = 0; i < N; ++i) band_all += band_len(N, half, d, i);
  int64_t band_g = 0;            // band lengths of the global rows
  int64_t g_in_band_of_g = 0;    // pairs (g, g') of globals inside each other's band
  for (int32_t g : G) {
    band_g += band_len(N, half, d, g);
    for (int32_t g2 : G) g_in_band_of_g += in_band(half, d, g, g2) ? 1 : 0;
  }
  // non-global rows i: band_len(i) + n_g - |{g in band(i)}|
  // sum_{i not in G} |{g in band(i)}| = sum_g (band_len(g) - |{i in G in band(g)}|)
  const int64_t rows_ng = (int64_t)N - n_g;
  const int64_t g_in_band_rows = band_g - g_in_band_of_g;
  return (band_all - band_g) + rows_ng * n_g - g_in_band_rows + n_g * (int64_t)N;
}

// GMAT chunked pattern: M dense memory rows; a main row scores the M memory
// keys and the main keys of its chunk.
int64_t pairs_chunked(int N, int memory, int chunk) {
  int64_t n = (int64_t)memory * N;
  for (int64_t start = memory; start < N; start += chunk) {
    const int64_t len = std::min<int64_t>(chunk, N - start);
    n += len * (memory + len);
  }
  return n;
}

std::pair<int, int> key_chunks(int N, int64_t want, int64_t align, int64_t max_chunks) {
  want = std::max<int64_t>(1, std::min(want, max_chunks));
  const int64_t per = (N + want - 1) / want;
  const int64_t len = ((per + align - 1) / align) * align;
  return std::pair<int, int>((int)len, (int)((N + len - 1) / len));
}

Schedule build_schedule(const Problem &p, const Tiling &t) {
  Schedule s;
  const int half = std::min(p.half, p.N);  // a wider band changes nothing
  // residue-class slots, one group per distinct dilation value
  std::vector<int32_t> dvals(p.dilation);
  std::sort(dvals.begin(), dvals.end());
  dvals.erase(std::unique(dvals.begin(), dvals.end()), dvals.end());
  std::vector<int32_t> first_slot(dvals.size());
  for (size_t a = 0; a < dvals.size(); ++a) {
    first_slot[a] = (int32_t)s.slots.size();
    const int d = dvals[a];
    for (int r = 0; r < d && r < p.N; ++r)
      s.slots.push_back(Slot{d, r, (int32_t)((p.N - r + d - 1) / d), 0});
  }
  s.head_slot0.resize(p.H);
  for (int h = 0; h < p.H; ++h) {
    const size_t a = std::lower_bound(dvals.begin(), dvals.end(), p.dilation[h]) - dvals.begin();
    s.head_slot0[h] = first_slot[a];
  }

  // band work: every query tile of every residue class of every head, with the
  // key tiles that intersect its band
  const int n_g = (int)p.globals.size();
  std::vector<std::pair<int, BandItem>> items;
  for (int b = 0; b < p.B; ++b)
    for (int h = 0; h < p.H; ++h) {
      const int d = p.dilation[h];
      for (int r = 0; r < d && r < p.N; ++r) {
        const int slot = s.head_slot0[h] + r;
        const int64_t len = s.slots[slot].len;
        const int64_t n_tiles = (len + t.rows - 1) / t.rows;
        for (int64_t t0 = 0; t0 < n_tiles; t0 += t.q_tiles) {
          BandItem it{};
          it.bh = b * p.H + h;
          it.slot = slot;
          it.q_tile = (int32_t)t0;
          int work = 0;
          for (int u = 0; u < 2; ++u) {
            const int64_t tt = t0 + u;
            if (u >= t.q_tiles || tt >= n_tiles) {
              it.k_lo[u] = 0;
              it.k_hi[u] = -1;
              continue;
            }
            const int64_t row_lo = tt * t.rows;
            const int64_t row_hi = std::min(len - 1, row_lo + t.rows - 1);
            int reach_lo, reach_hi, unused;
            row_keys(half, p.chunk, p.memory, (int)len, (int)row_lo, reach_lo, unused);
            row_keys(half, p.chunk, p.memory, (int)len, (int)row_hi, unused, reach_hi);
            const int64_t key_lo = std::max<int64_t>(0, reach_lo);
            const int64_t key_hi = std::min<int64_t>(len - 1, reach_hi);
            if (key_hi < key_lo) {  // no non-global key for these rows (all memory)
              it.k_lo[u] = 0;
              it.k_hi[u] = -1;
              continue;
            }
            it.k_lo[u] = (int32_t)(key_lo / t.key_tile);
            it.k_hi[u] = (int32_t)(key_hi / t.key_tile);
            work += it.k_hi[u] - it.k_lo[u] + 1;
            s.band_tile_pairs += it.k_hi[u] - it.k_lo[u] + 1;
            // does a global key of this class fall inside the band reach?
            for (int32_t g : p.globals) {
              if ((g - r) % d != 0) continue;
              const int64_t tg = (g - r) / d;
              if (tg >= reach_lo && tg <= reach_hi) {
                it.flags |= 1 << u;
                break;
              }
            }
          }
          if (it.k_hi[0] >= it.k_lo[0] || it.k_hi[1] >= it.k_lo[1])  // not all memory rows
            items.push_back({work, it});
        }
      }
    }
  // grouped by slot group (a launch addresses at most max_slots residue
  // classes), then longest work first (stable, so equal-work items keep their
  // sequence order and neighbouring CTAs keep sharing key/value tiles in L2)
  auto group_of = [&t](const BandItem &it) { return it.slot / t.max_slots; };
  std::stable_sort(items.begin(), items.end(),
                   [&](const std::pair<int, BandItem> &a, const std::pair<int, BandItem> &b) {
                     const int ga = group_of(a.second), gb = group_of(b.second);
                     if (ga != gb) return ga < gb;
                     return a.first > b.first;
                   });
  s.band.reserve(items.size());
  for (auto &x : items) s.band.push_back(x.second);
  const int n_groups = ((int)s.slots.size() + t.max_slots - 1) / t.max_slots;
  s.group_begin.assign(n_groups + 1, 0);
  for (size_t i = 0, g = 0; g <= (size_t)n_groups; ++g) {
    while (i < s.band.size() && group_of(s.band[i]) < (int)g) ++i;
    s.group_begin[g] = (int32_t)i;
  }
  s.group_begin[n_groups] = (int32_t)s.band.size();

  // global-row pass: split the N keys into chunks
  if (n_g > 0) {
    s.g_pad = ((n_g + t.g_tile - 1) / t.g_tile) * t.g_tile;
    const int g_items = (n_g + t.g_item_rows - 1) / t.g_item_rows;
    const int64_t bh = (int64_t)p.B * p.H;
    const int64_t max_tiles = (p.N + t.key_tile - 1) / t.key_tile;
    // tensor-core family: up to 128 global rows fill one query tile, so the
    // CTA's two query tiles take alternate key tiles of the chunk instead
    // (each leaves its own partial); up to 64 rows are packed twice into the
    // tile, one copy per key half (each half leaves its own partial)
    s.g_alt = t.q_tiles == 2 && n_g <= t.rows;
    s.g_packed = s.g_alt && 2 * n_g <= t.rows;
    const bool fused = t.fuse_global && t.sms > 1 && n_groups == 1;
    auto chunk_of = [&](int64_t want, int64_t align) { return key_chunks(p.N, want, align, max_tiles); };
    if (!fused) {
      int64_t want = (t.target_ctas + bh * g_items - 1) / (bh * g_items);
      std::tie(s.chunk_len, s.n_chunks) = chunk_of(want, t.key_tile);
    } else {
      // Cost model in units of one key tile of both query tiles of a band CTA
      // (the two chains interleave on the tensor core):
      //   band item: max over its query tiles of the band tiles, plus the
      //   global key tiles (64 keys: ~0.6 of a band tile);
      //   global item: its key tiles, alternate tiles going to the two query
      //   tiles (measured at D = 128: a key tile of global rows costs ~2,000
      //   SM cycles, a band unit ~4,300).
      // The band items are spread over S - X CTAs, the global items over X.
      // The key chunks number X (or 2X), so that, with the items in head-major
      // order, every global CTA takes one chunk of each head in turn and the
      // global CTAs move through the heads together with the band CTAs (whose
      // items are in head order too): the keys and values they read were
      // loaded by the band tiles shortly before and come from L2.
      const double kNarrow = 0.6, kGlobTile = 0.93, kMergePerPart = 0.15;
      double band_total = 0.0, band_max = 0.0;
      for (const BandItem &it : s.band) {
        double c = 0.0;
        for (int u = 0; u < 2; ++u)
          if (it.k_hi[u] >= it.k_lo[u])
            c = std::max(c, (it.k_hi[u] - it.k_lo[u] + 1) + kNarrow * ((n_g + 63) / 64));
        band_total += c;
        band_max = std::max(band_max, c);
      }
      const int S = t.sms;
      const int64_t n_band = (int64_t)s.band.size();
      const int64_t align = (s.g_alt ? 2 : 1) * (int64_t)t.key_tile;
      double best = 1e300;
      int best_x = 1, best_len = 0, best_nc = 0;
      for (int x = 1; x < S; ++x) {
        const int64_t bc = std::min<int64_t>(S - x, std::max<int64_t>(n_band, 1));
        const double t_band =
            n_band == 0 ? 0.0 : std::max(band_max, band_total / (double)bc + 0.5 * band_max);
        for (int m = 1; m <= 2; ++m) {
          int len, nc;
          std::tie(len, nc) = chunk_of((int64_t)x * m, align);
          const int64_t n_gi = bh * nc * g_items;
          if (n_gi < x) continue;  // a global CTA without work
          // CTA k runs items k, k + x, ...: the most key tiles any CTA runs
          auto item_cost = [&](int c) {
            const int64_t keys = std::min<int64_t>(p.N, (int64_t)(c + 1) * len) - (int64_t)c * len;
            const int64_t tiles = (keys + t.key_tile - 1) / t.key_tile;
            return kGlobTile * (double)(s.g_alt ? (tiles + 1) / 2 : tiles);
          };
          double t_glob = 0.0;
          if (n_gi <= 16 * (int64_t)S) {
            std::vector<double> per_cta(x, 0.0);
            for (int64_t i = 0; i < n_gi; ++i) per_cta[i % x] += item_cost((int)((i / g_items) % nc));
            t_glob = *std::max_element(per_cta.begin(), per_cta.end());
          } else {  // many items per CTA: the average plus one item
            double sum = 0.0;
            for (int c = 0; c < nc; ++c) sum += item_cost(c);
            t_glob = sum * (double)(bh * g_items) / x + item_cost(0);
          }
          const double tot = std::max(t_band, t_glob) +
                             kMergePerPart * nc * (s.g_alt ? 2 : 1) * (s.g_packed ? 2 : 1);
          if (tot < best) {
            best = tot;
            best_x = x;
            best_len = len;
            best_nc = nc;
          }
        }
      }
      s.chunk_len = best_len;
      s.n_chunks = best_nc;
      s.g_ctas = best_x;
      s.band_ctas = (int)std::min<int64_t>(S - best_x, n_band);
    }
    s.part_sets = s.n_chunks * (s.g_alt ? 2 : 1);
    s.part_sub = s.g_packed ? 2 : 1;
    for (int64_t x = 0; x < bh; ++x)
      for (int c = 0; c < s.n_chunks; ++c)
        for (int gt = 0; gt < g_items; ++gt)
          s.global.push_back(GlobalItem{(int32_t)x, c, gt, 0});
  }
  return s;
}

}  // namespace sa
