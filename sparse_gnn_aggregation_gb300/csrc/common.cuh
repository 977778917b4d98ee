// Shared device helpers: vector fragments of fp32 / bf16 feature rows,
// streaming loads of the CSR arrays, lane-group geometry, work items.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace autosage {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kBlock = 256;  // threads per block of the gather kernels

// ---------------------------------------------------------------- lane groups
//
// A warp is cut into 32 / (G*E) groups; each group owns one work item (a row
// or a chunk of a row) at a time. Inside a group, lane l = e*G + g: g in
// [0, G) walks the feature vector in VW-element fragments (NV fragments per
// lane: interleaved, fragment g + k*G, or, where a lane should stay inside
// one attention head, consecutive, fragment g*NV + k), e in [0, E) walks the
// item's edges (p = begin + e, e + E, ...). Feature lanes are adjacent, so
// one gathered row is read by adjacent lanes.
struct Lanes {
  int G, E, GE;
  int lane, g, e, slot;
  unsigned group_mask;  // the GE lanes of this group
  unsigned sub_mask;    // the G lanes of this group that share edge lane e
  __device__ __forceinline__ Lanes(int G_, int E_) : G(G_), E(E_), GE(G_ * E_) {
    lane = threadIdx.x & 31;
    const int l = lane % GE;
    g = l % G;
    e = l / G;
    slot = lane / GE;
    group_mask = (GE == 32) ? FULL : (((1u << GE) - 1u) << (slot * GE));
    sub_mask = (G == 32) ? FULL : (((1u << G) - 1u) << (slot * GE + e * G));
  }
};

// ---------------------------------------------------------------- loads

__device__ __forceinline__ int ld_stream_i32(const int32_t *p) { return __ldcs(p); }
__device__ __forceinline__ float ld_stream_f32(const float *p) { return __ldcs(p); }

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half), .y = b
  return *reinterpret_cast<uint32_t *>(&h);
}

// A fragment of VW consecutive elements of type T kept in its raw (packed)
// form; get(i) widens element i to fp32, get2(i) elements 2i and 2i + 1 as a
// pair for the packed fp32x2 arithmetic of sm_100 and later (VW even).
template <typename T, int VW> struct Frag;

template <> struct Frag<float, 4> {
  float4 r;
  __device__ __forceinline__ void load(const float *p) { r = __ldg(reinterpret_cast<const float4 *>(p)); }
  __device__ __forceinline__ void zero() { r = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ float get(int i) const { return i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w; }
  __device__ __forceinline__ float2 get2(int i) const { return i == 0 ? make_float2(r.x, r.y) : make_float2(r.z, r.w); }
};
template <> struct Frag<float, 2> {
  float2 r;
  __device__ __forceinline__ void load(const float *p) { r = __ldg(reinterpret_cast<const float2 *>(p)); }
  __device__ __forceinline__ void zero() { r = make_float2(0.f, 0.f); }
  __device__ __forceinline__ float get(int i) const { return i == 0 ? r.x : r.y; }
  __device__ __forceinline__ float2 get2(int) const { return r; }
};
template <> struct Frag<float, 1> {
  float r;
  __device__ __forceinline__ void load(const float *p) { r = __ldg(p); }
  __device__ __forceinline__ void zero() { r = 0.f; }
  __device__ __forceinline__ float get(int) const { return r; }
};
template <> struct Frag<__nv_bfloat16, 8> {
  uint4 r;
  __device__ __forceinline__ uint32_t word(int i) const { return i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w; }
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { r = __ldg(reinterpret_cast<const uint4 *>(p)); }
  __device__ __forceinline__ void zero() { r = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ float get(int i) const {
    const uint32_t w = i < 2 ? r.x : i < 4 ? r.y : i < 6 ? r.z : r.w;
    return (i & 1) ? bf16hi(w) : bf16lo(w);
  }
  __device__ __forceinline__ float2 get2(int i) const {
    const uint32_t w = i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w;
    return make_float2(bf16lo(w), bf16hi(w));
  }
};
template <> struct Frag<__nv_bfloat16, 4> {
  uint2 r;
  __device__ __forceinline__ uint32_t word(int i) const { return i == 0 ? r.x : r.y; }
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { r = __ldg(reinterpret_cast<const uint2 *>(p)); }
  __device__ __forceinline__ void zero() { r = make_uint2(0u, 0u); }
  __device__ __forceinline__ float get(int i) const {
    const uint32_t w = i < 2 ? r.x : r.y;
    return (i & 1) ? bf16hi(w) : bf16lo(w);
  }
  __device__ __forceinline__ float2 get2(int i) const {
    const uint32_t w = i == 0 ? r.x : r.y;
    return make_float2(bf16lo(w), bf16hi(w));
  }
};
template <> struct Frag<__nv_bfloat16, 2> {
  uint32_t r;
  __device__ __forceinline__ uint32_t word(int) const { return r; }
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { r = __ldg(reinterpret_cast<const unsigned int *>(p)); }
  __device__ __forceinline__ void zero() { r = 0u; }
  __device__ __forceinline__ float get(int i) const { return (i & 1) ? bf16hi(r) : bf16lo(r); }
  __device__ __forceinline__ float2 get2(int) const { return make_float2(bf16lo(r), bf16hi(r)); }
};
template <> struct Frag<__nv_bfloat16, 1> {
  uint32_t r;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
    r = static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(p)));
  }
  __device__ __forceinline__ void zero() { r = 0u; }
  __device__ __forceinline__ float get(int) const { return __uint_as_float(r << 16); }
};

// A running fp32 sum over one fragment slot: VW values kept as pairs, so
// that the accumulation runs on the packed fp32x2 FMA of sm_100 and later
// (one instruction for two elements; each element is still one fp32 FMA,
// rounded to nearest). VW = 1 keeps its one value in .x.
template <int VW>
struct Acc {
  static constexpr int P = (VW + 1) / 2;
  float2 p[P];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < P; ++i) p[i] = make_float2(0.f, 0.f);
  }
  __device__ __forceinline__ void scale(float c) {
#pragma unroll
    for (int i = 0; i < P; ++i) p[i] = __fmul2_rn(p[i], make_float2(c, c));
  }
  template <typename F>
  __device__ __forceinline__ void fma(float w, const F &f) {
    if constexpr (VW >= 2) {
      const float2 ww = make_float2(w, w);
#pragma unroll
      for (int i = 0; i < P; ++i) p[i] = __ffma2_rn(ww, f.get2(i), p[i]);
    } else {
      p[0].x = fmaf(w, f.get(0), p[0].x);
    }
  }
  __device__ __forceinline__ float get(int v) const { return (v & 1) ? p[v >> 1].y : p[v >> 1].x; }
  __device__ __forceinline__ void set(int v, float x) {
    if (v & 1) p[v >> 1].y = x;
    else p[v >> 1].x = x;
  }
};

// <a, b> over one fragment pair: even and odd elements in two packed
// fp32x2 chains, added at the end.
template <typename T, int VW>
__device__ __forceinline__ float frag_dot(const Frag<T, VW> &a, const Frag<T, VW> &b) {
  if constexpr (VW >= 2) {
    float2 d = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VW / 2; ++i) d = __ffma2_rn(a.get2(i), b.get2(i), d);
    return d.x + d.y;
  } else {
    return a.get(0) * b.get(0);
  }
}

// a * b + c for the low (or high) bf16 halves of two packed words with the
// mixed-precision FMA of sm_100 and later: the bf16 operands are multiplied
// exactly and the sum rounded once in fp32, which is the value of widening
// both halves to fp32 and calling fmaf, without the two widening steps.
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
      "fma.rn.f32.bf16 %0, a0, b0, %3;\n\t}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
      "fma.rn.f32.bf16 %0, a1, b1, %3;\n\t}" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

// <a, b> over one bf16 fragment pair: even and odd elements in two chains
// (the order of the packed-pair form above), added at the end.
template <int VW>
__device__ __forceinline__ float frag_dot(const Frag<__nv_bfloat16, VW> &a, const Frag<__nv_bfloat16, VW> &b) {
  if constexpr (VW >= 2) {
    float e = 0.f, o = 0.f;
#pragma unroll
    for (int i = 0; i < VW / 2; ++i) {
      e = fma_bf16_lo(a.word(i), b.word(i), e);
      o = fma_bf16_hi(a.word(i), b.word(i), o);
    }
    return e + o;
  } else {
    return a.get(0) * b.get(0);
  }
}

// Store VW fp32 values as type T (bf16: round to nearest even), streaming.
template <typename T, int VW> __device__ __forceinline__ void store_frag(T *p, const float (&o)[VW]);

template <> __device__ __forceinline__ void store_frag<float, 4>(float *p, const float (&o)[4]) {
  __stcs(reinterpret_cast<float4 *>(p), make_float4(o[0], o[1], o[2], o[3]));
}
template <> __device__ __forceinline__ void store_frag<float, 2>(float *p, const float (&o)[2]) {
  __stcs(reinterpret_cast<float2 *>(p), make_float2(o[0], o[1]));
}
template <> __device__ __forceinline__ void store_frag<float, 1>(float *p, const float (&o)[1]) { __stcs(p, o[0]); }
template <> __device__ __forceinline__ void store_frag<__nv_bfloat16, 8>(__nv_bfloat16 *p, const float (&o)[8]) {
  __stcs(reinterpret_cast<uint4 *>(p), make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]),
                                                  pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7])));
}
template <> __device__ __forceinline__ void store_frag<__nv_bfloat16, 4>(__nv_bfloat16 *p, const float (&o)[4]) {
  __stcs(reinterpret_cast<uint2 *>(p), make_uint2(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3])));
}
template <> __device__ __forceinline__ void store_frag<__nv_bfloat16, 2>(__nv_bfloat16 *p, const float (&o)[2]) {
  __stcs(reinterpret_cast<unsigned int *>(p), pack_bf16(o[0], o[1]));
}
template <> __device__ __forceinline__ void store_frag<__nv_bfloat16, 1>(__nv_bfloat16 *p, const float (&o)[1]) {
  *p = __float2bfloat16_rn(o[0]);
}

// fp32 workspace partials: kept in L2 (the fix-up reads them right after).
template <int VW> __device__ __forceinline__ void store_partial(float *p, const float (&o)[VW]) {
#pragma unroll
  for (int i = 0; i < VW; ++i) __stcg(p + i, o[i]);
}

// ---------------------------------------------------------------- work items
//
// Rows whose degree is at most `split` are work items of their own. Longer
// rows are cut into chunks of `split` edges; chunk c covers edges
// [chunk_begin[c], min(chunk_begin[c] + split, row end)) of row chunk_row[c]
// and writes its partial result at slot c. Long row j owns the consecutive
// chunks [long_ptr[j], long_ptr[j+1]), so a fix-up combines them in order.
// Runs of a launch: the items are cut into segments (the chunks; then the
// rows, one segment per degree bucket when the rows are in degree-binned
// order), and each segment is dealt to its own blocks in runs of run[s]
// items. Set by deal_items for each launch; n == 0 leaves one uniform run.
constexpr int kMaxRuns = 34;  // chunks, 32 degree buckets, rows longer than split
struct RunTable {
  int n = 0;
  int64_t item0[kMaxRuns + 1];  // first item of segment s; item0[n] = items
  int64_t item1[kMaxRuns];      // one past the last item of segment s
  int block0[kMaxRuns + 1];     // first block of segment s; block0[n] = grid
  int run[kMaxRuns];            // items per block in segment s
};

struct ChunkList {
  const int32_t *chunk_row = nullptr;    // [n_chunks]
  const int32_t *chunk_begin = nullptr;  // [n_chunks]
  const int32_t *long_rows = nullptr;    // [n_long]
  const int32_t *long_ptr = nullptr;     // [n_long + 1]
  const int32_t *row_order = nullptr;  // [n_rows] rows in processing order (null: 0, 1, 2, ...)
  int n_chunks = 0;
  int n_long = 0;
  int split = 0;  // 0: no row is cut
  // degree-binned order: rows of bucket k (k = 0: the longest) start at
  // position bucket_start[k] of row_order; bucket_start[32] = n_rows
  int32_t bucket_start[33] = {};
  // buckets [ell_from, ell_to) are handled by an ELL slab (hybrid schedule):
  // the row launch skips their items
  int ell_from = 32, ell_to = 32;
  RunTable runs;
};

// One work item: (row, edge begin, edge end, chunk slot or -1 for a whole row).
// Inactive items (b == e) still take part in their group's shuffles.
struct Item {
  int64_t row;
  int b, e;
  int chunk;
  bool active;
};

// Work item number idx of a launch: the chunks of cut rows come first (the
// longest items start earliest), then every row, in row_order when the plan
// has one (degree-binned schedules: rows sorted by degree bucket, longest
// first, so the lane groups of a warp get rows of similar length).
__device__ __forceinline__ Item item_at(int64_t idx, int64_t n_rows, const int32_t *row_ptr,
                                        const ChunkList &cl) {
  Item it{0, 0, 0, -1, false};
  if (idx < cl.n_chunks) {
    it.chunk = static_cast<int>(idx);
    it.row = cl.chunk_row[idx];
    it.b = cl.chunk_begin[idx];
    const int re = row_ptr[it.row + 1];
    it.e = (re - it.b > cl.split) ? it.b + cl.split : re;
    it.active = true;
  } else if (idx - cl.n_chunks < n_rows) {
    const int64_t r = cl.row_order ? (int64_t)cl.row_order[idx - cl.n_chunks] : idx - cl.n_chunks;
    it.row = r;
    it.b = row_ptr[r];
    it.e = row_ptr[r + 1];
    it.active = !(cl.split > 0 && it.e - it.b > cl.split);
    if (!it.active) it.e = it.b;
  }
  return it;
}

// Items of a launch (the chunks of cut rows, then the rows) are dealt to
// blocks segment by segment (RunTable): chunks a few per lane group, rows of
// a degree bucket so many per lane group that a group gets about 512 edges
// (at most the plain row run), other rows in plain runs. Inside a block the
// lane groups take the block's items one at a time from a shared counter, so
// a group that drew short rows goes on with the next item instead of idling
// until the block's longest row ends. Groups of one warp may take different
// numbers of items; all their shuffles use group or sub-group masks.
struct ItemQueue {
  int64_t base, end;
  int *counter;
  __device__ __forceinline__ ItemQueue(int64_t n_rows, const ChunkList &cl, int ipb, int *shared_counter) {
    const RunTable &T = cl.runs;
    if (T.n > 0) {
      int sg = 0;
      while (sg + 1 < T.n && (int)blockIdx.x >= T.block0[sg + 1]) ++sg;
      base = T.item0[sg] + (int64_t)((int)blockIdx.x - T.block0[sg]) * T.run[sg];
      const int64_t stop = base + T.run[sg];
      end = stop < T.item1[sg] ? stop : T.item1[sg];
    } else {
      base = (int64_t)blockIdx.x * ipb;
      const int64_t n_items = n_rows + cl.n_chunks;
      end = base + ipb < n_items ? base + ipb : n_items;
    }
    counter = shared_counter;
    if (threadIdx.x == 0) *counter = 0;
    __syncthreads();
  }
  __device__ __forceinline__ bool next(const Lanes &L, int64_t &idx) const {
    int local = 0;
    if (L.g == 0 && L.e == 0) local = atomicAdd(counter, 1);
    local = __shfl_sync(L.group_mask, local, L.slot * L.GE);
    idx = base + local;
    return idx < end;
  }
};

// Items per block: a few per lane group, so blocks stay short enough for the
// block scheduler to balance them across SMs. Whole-warp groups over wide
// rows (G >= 16 of 32 lanes) take 16 each, other groups 8 (measured on the
// R-MAT scale-20 step: fewer, longer blocks pay off where items are heavy).
inline int items_per_block_for(int GE, int G) {
  return (kBlock / 32) * (32 / GE) * ((GE == 32 && G >= 16) ? 16 : 8);
}

// The deal of one launch over n_rows rows with lane groups of GE lanes: the
// chunk list with its run table set, the plain row run, and the grid.
struct Deal {
  ChunkList cl;
  int ipb;
  int64_t grid;
};
inline Deal deal_items(const ChunkList &cl, int64_t n_rows, int GE, int G) {
  Deal d{cl, items_per_block_for(GE, G), 0};
  const int groups = (kBlock / 32) * (32 / GE);
  const int max_per_group = d.ipb / groups;
  RunTable &T = d.cl.runs;
  T.n = 0;
  int64_t item = 0, block = 0;
  auto add = [&](int64_t count, int run) {
    if (count <= 0) return;
    T.item0[T.n] = item;
    T.item1[T.n] = item + count;
    T.block0[T.n] = static_cast<int>(block);
    T.run[T.n] = run;
    item += count;
    block += (count + run - 1) / run;
    ++T.n;
  };
  // chunks: about 512 edges per lane group
  int per_group = cl.split > 0 ? 512 / cl.split : 1;
  per_group = per_group < 1 ? 1 : (per_group > max_per_group ? max_per_group : per_group);
  add(cl.n_chunks, groups * per_group);
  if (cl.row_order && cl.bucket_start[32] == n_rows) {
    // degree buckets, longest first: bucket k holds degrees below 2^(31 - k)
    // (the last bucket: rows longer than split, which are inactive items)
    for (int k = 0; k < 32; ++k) {
      if (k >= cl.ell_from && k < cl.ell_to) {  // rows of the ELL slab: not items of this launch
        item += (int64_t)cl.bucket_start[k + 1] - cl.bucket_start[k];
        continue;
      }
      const int bits = 31 - k;
      int pg = k == 31 || bits >= 10 ? 1 : 512 >> bits;
      if (k == 31) pg = max_per_group;
      pg = pg < 1 ? 1 : (pg > max_per_group ? max_per_group : pg);
      add((int64_t)cl.bucket_start[k + 1] - cl.bucket_start[k], groups * pg);
    }
  } else {
    add(n_rows, d.ipb);
  }
  T.item0[T.n] = item;
  T.block0[T.n] = static_cast<int>(block);
  d.grid = block;
  return d;
}

}  // namespace autosage
