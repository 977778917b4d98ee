// Host-side check of the item deal (deal_items in common.cuh): for chunk
// lists with and without a degree-binned order, the run table must cover
// every item exactly once, segment by segment, with runs between one lane
// group's share and the plain row run, and a grid that matches the blocks
// the table describes; rows of the buckets an ELL slab handles (hybrid
// schedule) must be dealt to no block. Built and run by
// tests/test_deal_host.py; no kernel is launched.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "common.cuh"

using namespace autosage;

static int failures = 0;
#define CHECK(cond, ...)                 \
  do {                                   \
    if (!(cond)) {                       \
      std::printf("FAIL: " __VA_ARGS__); \
      std::printf("\n");                 \
      ++failures;                        \
    }                                    \
  } while (0)

// Replays the block -> item range mapping of ItemQueue on the host.
static void block_range(const ChunkList &cl, int64_t n_rows, int ipb, int b, int64_t &base, int64_t &end) {
  const RunTable &T = cl.runs;
  if (T.n > 0) {
    int sg = 0;
    while (sg + 1 < T.n && b >= T.block0[sg + 1]) ++sg;
    base = T.item0[sg] + (int64_t)(b - T.block0[sg]) * T.run[sg];
    const int64_t stop = base + T.run[sg];
    end = stop < T.item1[sg] ? stop : T.item1[sg];
  } else {
    base = (int64_t)b * ipb;
    const int64_t n_items = n_rows + cl.n_chunks;
    end = base + ipb < n_items ? base + ipb : n_items;
  }
}

static void check_case(const char *name, int n_chunks, int split, const std::vector<int> &bucket_rows, int GE,
                       int G, int ell_from = 32, int ell_to = 32) {
  ChunkList cl;
  cl.n_chunks = n_chunks;
  cl.split = split;
  cl.ell_from = ell_from;
  cl.ell_to = ell_to;
  int64_t n_rows = 0;
  static int32_t dummy_order = 0;
  if (!bucket_rows.empty()) {
    cl.row_order = &dummy_order;  // only its presence matters to the deal
    for (int k = 0; k < 32; ++k) {
      cl.bucket_start[k] = static_cast<int32_t>(n_rows);
      n_rows += k < (int)bucket_rows.size() ? bucket_rows[k] : 0;
    }
    cl.bucket_start[32] = static_cast<int32_t>(n_rows);
  } else {
    n_rows = 100003;
  }
  const Deal d = deal_items(cl, n_rows, GE, G);
  const int64_t items = n_rows + n_chunks;
  const int groups = (kBlock / 32) * (32 / GE);
  const RunTable &T = d.cl.runs;
  CHECK(T.n >= 1 && T.n <= kMaxRuns, "%s: %d segments", name, T.n);
  CHECK(T.item0[0] == 0 && T.item0[T.n] == items, "%s: segments cover %lld of %lld items", name,
        (long long)T.item0[T.n], (long long)items);
  CHECK(T.block0[T.n] == d.grid, "%s: grid %lld, table %d", name, (long long)d.grid, T.block0[T.n]);
  for (int s = 0; s < T.n; ++s) {
    const int64_t count = T.item1[s] - T.item0[s];
    CHECK(T.item1[s] <= T.item0[s + 1], "%s: segment %d overlaps the next", name, s);
    CHECK(count > 0, "%s: empty segment %d", name, s);
    CHECK(T.run[s] >= groups && T.run[s] <= d.ipb && T.run[s] % groups == 0, "%s: run %d of segment %d", name,
          T.run[s], s);
    CHECK(T.block0[s + 1] - T.block0[s] == (count + T.run[s] - 1) / T.run[s], "%s: blocks of segment %d", name, s);
  }
  // every item belongs to exactly one block, blocks in item order; the rows
  // of the ELL buckets belong to none
  std::vector<int> seen(items, 0);
  int64_t next = 0;
  for (int b = 0; b < d.grid; ++b) {
    int64_t base, end;
    block_range(d.cl, n_rows, d.ipb, b, base, end);
    CHECK(base >= next && end > base && end - base <= d.ipb, "%s: block %d covers [%lld, %lld)", name, b,
          (long long)base, (long long)end);
    for (int64_t i = base; i < end && i < items; ++i) ++seen[i];
    next = end;
  }
  for (int64_t i = 0; i < items; ++i) {
    const int64_t pos = i - n_chunks;  // position in the row order
    const bool ell = !bucket_rows.empty() && pos >= 0 && ell_from < 32 && pos >= cl.bucket_start[ell_from] &&
                     pos < cl.bucket_start[ell_to];
    CHECK(seen[i] == (ell ? 0 : 1), "%s: item %lld dealt %d times", name, (long long)i, seen[i]);
  }
  // heavy buckets get short runs: a bucket of rows below 2^bits edges gives a group at most
  // max(1, 512 >> bits) of them
  if (!bucket_rows.empty()) {
    int s = n_chunks > 0 ? 1 : 0;
    for (int k = 0; k < 32; ++k) {
      if (k >= (int)bucket_rows.size() || bucket_rows[k] == 0) continue;
      if (k >= ell_from && k < ell_to) continue;  // no segment: the ELL slab holds these rows
      const int bits = 31 - k;
      if (k < 31 && bits >= 2) {
        const int cap = bits >= 10 ? 1 : (512 >> bits);
        CHECK(T.run[s] / groups <= (cap < 1 ? 1 : cap), "%s: bucket %d run %d per group", name, k,
              T.run[s] / groups);
      }
      ++s;
    }
  }
}

int main() {
  // degree-binned: rows of bit length 10 (512..1023 edges) down to empty rows
  std::vector<int> buckets(32, 0);
  buckets[21] = 37;      // 2^10 > degree >= 2^9
  buckets[22] = 501;     // 256..511
  buckets[23] = 1999;    // 128..255
  buckets[25] = 40000;   // 32..63
  buckets[28] = 123457;  // 4..7
  buckets[31] = 77777;   // empty rows and rows longer than split
  for (int GE : {1, 2, 4, 8, 16, 32})
    for (int G : {1, 16}) {
      if (G > GE) continue;
      check_case("binned", 9000, 512, buckets, GE, G);
      check_case("binned-no-chunks", 0, 128, buckets, GE, G);
      check_case("plain", 12345, 128, {}, GE, G);
      check_case("plain-no-chunks", 0, 0, {}, GE, G);
      check_case("hybrid", 9000, 512, buckets, GE, G, 28, 31);
      check_case("hybrid-no-chunks", 0, 128, buckets, GE, G, 28, 31);
    }
  std::vector<int> tiny(32, 0);
  tiny[31] = 1;
  check_case("one-row", 0, 16, tiny, 32, 32);
  if (failures) {
    std::printf("%d failures\n", failures);
    return 1;
  }
  std::printf("OK\n");
  return 0;
}
