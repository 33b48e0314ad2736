// Host-side check of the kernels' work schedule (schedule.cuh): for a list
// of launch shapes, every work item is taken by exactly one CTA, every index
// stays inside its buffer, and the backward's workspace rows a CTA touches
// lie inside the padded row range. Built with nvcc and run on the CPU by
// tests/test_schedule.py; prints "ok" or the first violation.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "schedule.cuh"

using namespace fa;

static int fails = 0;
#define CHECK(c, ...)                                      \
  do {                                                     \
    if (!(c)) {                                            \
      if (fails++ < 10) {                                  \
        std::printf("FAIL %s:%d: ", __FILE__, __LINE__);   \
        std::printf(__VA_ARGS__);                          \
        std::printf("\n");                                 \
      }                                                    \
    }                                                      \
  } while (0)

// heads per group of the causal launch order (same rule as the library)
static int head_group(int N, int d, bool causal) {
  if (!causal) return 1;
  const long long per_head = static_cast<long long>(N) * d * 2 * 2;
  long long g = (48ll << 20) / per_head;
  return static_cast<int>(g < 1 ? 1 : (g > 16 ? 16 : g));
}

// the two-tile forward's group: a power of two within the rule, at most 8
static int fwd_head_group(int N, int d, bool causal) {
  const int g = head_group(N, d, causal);
  int p = 1;
  while (p * 2 <= g && p * 2 <= 8) p *= 2;
  return p;
}

static void check_grouped(int n_heads, int n_tiles, int hgroup, bool reverse, const char *what) {
  std::vector<int> seen(static_cast<size_t>(n_heads) * n_tiles, 0);
  for (int blk = 0; blk < n_heads * n_tiles; ++blk) {
    const WorkItem w = grouped_item(blk, n_heads, n_tiles, hgroup, reverse);
    CHECK(w.bh >= 0 && w.bh < n_heads && w.tile >= 0 && w.tile < n_tiles,
          "%s: block %d -> (%d, %d) outside %d x %d", what, blk, w.bh, w.tile, n_heads, n_tiles);
    if (w.bh >= 0 && w.bh < n_heads && w.tile >= 0 && w.tile < n_tiles)
      seen[static_cast<size_t>(w.bh) * n_tiles + w.tile]++;
  }
  for (size_t i = 0; i < seen.size(); ++i)
    CHECK(seen[i] == 1, "%s: item %zu taken %d times (heads %d, tiles %d, group %d)", what, i, seen[i],
          n_heads, n_tiles, hgroup);
}

static void check_tiles(int n_heads, int nqt, bool reverse) {
  std::vector<int> seen(static_cast<size_t>(n_heads) * nqt, 0);
  for (int blk = 0; blk < n_heads * nqt; ++blk) {
    const WorkItem w = tile_item(blk, nqt, reverse);
    CHECK(w.bh >= 0 && w.bh < n_heads && w.tile >= 0 && w.tile < nqt, "tile item %d out of range", blk);
    seen[static_cast<size_t>(w.bh) * nqt + w.tile]++;
  }
  for (size_t i = 0; i < seen.size(); ++i) CHECK(seen[i] == 1, "query tile %zu taken %d times", i, seen[i]);
}

static void check_splits(int n_all, int splits) {
  int next = 0;
  for (int s = 0; s < splits; ++s) {
    int lo, n;
    split_share(n_all, s, splits, &lo, &n);
    CHECK(lo == next && n >= 0, "split %d of %d over %d tiles: [%d, %d) after %d", s, splits, n_all, lo,
          lo + n, next);
    next = lo + n;
  }
  CHECK(next == n_all, "splits of %d tiles end at %d", n_all, next);
}

// backward: the CTA of (key/value head bkv, key tile kt) reads and adds to
// the workspace rows of query tiles qi of the query heads of its group
static void check_bwd_rows(int B, int H, int Hkv, int N, bool causal) {
  const int nqt = (N + 127) / 128;
  const long long tile_rows = static_cast<long long>(nqt) * 128;
  const long long rows_pad = static_cast<long long>(B) * H * tile_rows;
  std::vector<int> head_seen(static_cast<size_t>(B) * H, 0);
  for (int bkv = 0; bkv < B * Hkv; ++bkv) {
    CHECK(kv_head_of(q_head_of(bkv, 0, H, Hkv), H, Hkv) == bkv, "q_head/kv_head do not invert");
    for (int g = 0; g < H / Hkv; ++g) {
      const int qh = q_head_of(bkv, g, H, Hkv);
      CHECK(qh >= 0 && qh < B * H, "query head %d out of range", qh);
      CHECK(kv_head_of(qh, H, Hkv) == bkv, "query head %d reads %d, not %d", qh, kv_head_of(qh, H, Hkv), bkv);
      head_seen[qh]++;
      for (int kt = 0; kt < nqt; ++kt)
        for (int qi = causal ? kt : 0; qi < nqt; ++qi) {
          const long long r0 = qh * tile_rows + static_cast<long long>(qi) * 128;
          CHECK(r0 >= 0 && r0 + 127 < rows_pad, "workspace rows [%lld, %lld) outside %lld", r0, r0 + 128,
                rows_pad);
        }
    }
  }
  for (size_t i = 0; i < head_seen.size(); ++i) CHECK(head_seen[i] == 1, "query head %zu in %d groups", i, head_seen[i]);
}

int main() {
  struct S { int B, H, Hkv, N, d; };
  const S shapes[] = {{1, 2, 2, 256, 64},      {16, 16, 16, 512, 64},  {8, 12, 12, 1024, 64},
                      {8, 16, 16, 4096, 128},  {4, 16, 16, 8192, 128}, {2, 16, 16, 16384, 128},
                      {2, 8, 8, 16384, 64},    {4, 32, 8, 4096, 128},  {1, 1, 1, 1, 64},
                      {3, 5, 5, 300, 128},     {2, 6, 3, 4500, 64},    {1, 7, 1, 129, 128},
                      {5, 3, 3, 20000, 128},   {1, 1, 1, 8192, 128}};
  for (const S &s : shapes) {
    const int nqt = (s.N + 127) / 128, nqb = (nqt + 1) / 2;
    for (int causal = 0; causal < 2; ++causal) {
      const int hg = head_group(s.N, s.d, causal);
      // two-tile forward: query-tile pairs of B*H heads
      check_grouped(s.B * s.H, nqb, fwd_head_group(s.N, s.d, causal), causal, "two-tile forward");
      // backward: key tiles of B*Hkv heads (group size divided by the query heads per key/value head)
      int hgb = hg / (s.H / s.Hkv);
      if (hgb < 1) hgb = 1;
      check_grouped(s.B * s.Hkv, nqt, hgb, false, "backward");
      check_tiles(s.B * s.H, nqt, causal);
      check_bwd_rows(s.B, s.H, s.Hkv, s.N, causal);
    }
    for (int sp = 1; sp <= 64; sp = sp * 2 + 1) check_splits(nqt, sp);
  }
  for (int g = 1; g <= 16; ++g) check_grouped(37, 11, g, true, "odd group sizes");
  if (fails) {
    std::printf("%d failures\n", fails);
    return 1;
  }
  std::printf("ok\n");
  return 0;
}
