// Batch schedule, computed on the device from seq_lens (and the context-parallel
// lengths or local bounds, when given) by every CTA of the split-KV kernel, in
// scratch shared memory before the tile buffers are used.
//
// These functions run once per kernel (or once per piece of work) and are kept out of
// line: the split-KV kernel's twelve warps run different code, so a compact kernel keeps
// their per-tile loops in the instruction cache, and one copy of each helper that the
// prologue has already fetched serves every later caller.
//
// The deal is described in mla_common.cuh: work rows (packed M tiles of
// (token, head) rows), bands of side-by-side clusters over a request's work rows,
// super-rows laid end to end and dealt in equal contiguous shares of virtual
// tiles.  Each cluster extracts its pieces ("segments") in order; the CTAs share
// the writing of the row table the reduction kernel reads.
#pragma once
#include <climits>

#include "mla_common.cuh"

namespace mla {

// K (this rank's keys) of request b, clamped to the page table; out-of-range values
// are flagged
__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b, uint32_t* err) {
  int K = p.seq_lens[b];
  const int cap = p.pt_stride * p.page_size;
  if (K < 0 || K > cap) {
    if (err) atomicOr(err, kErrBadLength);
    K = K < 0 ? 0 : cap;
  }
  return K;
}

// whole-sequence length the causal and window bounds are taken on
__device__ __forceinline__ int global_len(const DecodeParams& p, int b, int K) {
  if (p.cp_world <= 1) return K;
  const int g = p.global_seq_lens[b];
  return g < 0 ? 0 : g;
}

__device__ __forceinline__ void token_keys(const DecodeParams& p, int b, int t, int K, int Kg, int& lo, int& hi) {
  const bool has_lvl = p.local_visible_lens != nullptr;
  const int lvl = has_lvl ? p.local_visible_lens[(size_t)b * p.Sq + t] : 0;
  token_range(K, Kg, lvl, has_lvl, p.Sq, t, p.causal, p.window_left, p.cp_world, p.cp_rank, p.cp_interleave, lo, hi);
}

// union tile span of tokens [t0, t1] of request b with local bounds (arbitrary per token):
// (first tile, tile count)
static __device__ __noinline__ int2 tokens_span_lvl(const DecodeParams& p, int b, int t0, int t1, int K, int Kg) {
  int lo_min = INT_MAX, hi_max = 0;
  for (int t = t0; t <= t1; ++t) {
    int lo, hi;
    token_keys(p, b, t, K, Kg, lo, hi);
    if (hi > lo) {
      lo_min = lo < lo_min ? lo : lo_min;
      hi_max = hi > hi_max ? hi : hi_max;
    }
  }
  int tlo = 0, n = 0;
  if (hi_max > 0) tile_span(lo_min, hi_max, tlo, n);
  return make_int2(tlo, n);
}

// Union tile span of tokens [t0, t1] of request b.  Without local bounds both ends of a
// token's range are non-decreasing in t and consecutive ranges meet (the window floor of
// t + 1 is below the causal bound of t), also through the monotone context-parallel map,
// and a token with an empty range has its floor at the first key any later token sees; so
// the union is [lo(t0), hi(t1)).
__device__ __forceinline__ void tokens_span(const DecodeParams& p, int b, int t0, int t1, int K, int Kg, int& tlo,
                                            int& n) {
  if (p.local_visible_lens) {
    const int2 r = tokens_span_lvl(p, b, t0, t1, K, Kg);
    tlo = r.x;
    n = r.y;
    return;
  }
  int lo0, hi0, lo1, hi1;
  token_range(K, Kg, 0, false, p.Sq, t0, p.causal, p.window_left, p.cp_world, p.cp_rank, p.cp_interleave, lo0, hi0);
  token_range(K, Kg, 0, false, p.Sq, t1, p.causal, p.window_left, p.cp_world, p.cp_rank, p.cp_interleave, lo1, hi1);
  tile_span(lo0, hi1, tlo, n);
}

struct Sched {
  const int32_t* prefix;  // [S + 1] in shared memory
  DealShape d;
  long long T;
  int Gd;  // groups the tiles are dealt to
};

// span of sub-band k of request b (the union of its work rows), given the request's lengths
__device__ __forceinline__ void sub_span(const DecodeParams& p, const DealShape& d, int b, int k, int K, int Kg, int& ulo,
                                int& U) {
  const int i0 = k * d.wb, i1 = min(d.Qb, i0 + d.wb) - 1;
  int t0, t1;
  work_tokens(i0, i1, p.Sq, p.H, t0, t1);
  tokens_span(p, b, t0, t1, K, Kg, ulo, U);
}

// span of work row i of request b
__device__ __forceinline__ void work_span(const DecodeParams& p, int b, int i, int K, int Kg, int& tlo, int& n) {
  int t0, t1;
  work_tokens(i, i, p.Sq, p.H, t0, t1);
  tokens_span(p, b, t0, t1, K, Kg, tlo, n);
}

// Block-wide: fills prefix[0..S] (prefix[S] = T) in shared memory.  scratch needs
// S + 1 + 32 ints.  All threads of the block must call it.
__device__ __forceinline__ Sched build_schedule(const DecodeParams& p, int32_t* scratch, uint32_t* err_flag) {
  const DealShape d = deal_shape(p.B, p.Sq, p.H, p.num_clusters);
  const int S = d.S;
  const int tid = threadIdx.x, nt = blockDim.x;
  int32_t* prefix = scratch;
  int32_t* part = scratch + S + 1;  // 32 ints
  // per-thread contiguous chunk of super-rows
  const int chunk = (S + nt - 1) / nt;
  const int s0 = min(S, tid * chunk), s1 = min(S, s0 + chunk);
  int local = 0;
  for (int s = s0; s < s1; ++s) {
    const int b = s / d.nsub;
    const int K = clamp_len(p, b, s % d.nsub == 0 ? err_flag : nullptr);  // a bad length flagged once
    int ulo, U;
    sub_span(p, d, b, s % d.nsub, K, global_len(p, b, K), ulo, U);
    const int cost = U > 0 ? p.piece_units + kUnitsPerTile * U : 0;
    prefix[s] = cost;
    local += cost;
  }
  // inclusive scan of per-thread sums: warp scans, then a scan of warp totals
  const int lane = tid & 31, warp = tid >> 5;
  int v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  if (lane == 31) part[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const int nw = (nt + 31) / 32;
    int w = lane < nw ? part[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int x = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += x;
    }
    if (lane < nw) part[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  int run = (v - local) + (warp > 0 ? part[warp - 1] : 0);  // exclusive prefix of this thread's chunk
  for (int s = s0; s < s1; ++s) {
    int n = prefix[s];
    prefix[s] = run;
    run += n;
  }
  if (tid == nt - 1) prefix[S] = run;  // last thread: run == T (also correct when its chunk is empty)
  __syncthreads();
  Sched sc;
  sc.prefix = prefix;
  sc.d = d;
  sc.T = prefix[S];
  sc.Gd = deal_groups(d.Gg, sc.T);
  return sc;
}

// largest super-row s with prefix[s] <= x (x < T): the super-row holding unit x
__device__ __forceinline__ int super_row_of_tile(const Sched& sc, long long x) {
  int lo = 0, hi = sc.d.S - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (sc.prefix[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// pieces of a work row whose own tiles start tlo - ulo into super-row s: n_parts and the
// group of its first piece (the groups owning its first and last tiles, and every one between)
__device__ __forceinline__ int row_parts(const Sched& sc, int pu, int s, int ulo, int tlo, int n, int& g_first) {
  if (n <= 0) {
    g_first = 0;
    return 0;
  }
  const long long xf = tile_unit(sc.prefix[s], pu, tlo - ulo), xl = tile_unit(sc.prefix[s], pu, tlo - ulo + n - 1);
  g_first = group_of_tile(xf, sc.T, sc.Gd);
  return group_of_tile(xl, sc.T, sc.Gd) - g_first + 1;
}

// Extract the pieces of cluster c, in order: one warp, a lane per super-row of the
// cluster's share (the spans of a super-row take one read of the request's lengths, and
// the lanes read theirs together).  The first kSmemSegs go to `segs` in shared memory,
// the rest to `overflow` (workspace).  Returns the number of pieces (in every lane).
__device__ __forceinline__ int build_segments(const DecodeParams& p, const Sched& sc, int c, Segment* segs,
                                     Segment* overflow) {
  const DealShape& d = sc.d;
  const int lane = threadIdx.x & 31;
  const int g = c / d.wb, j = c % d.wb;
  if (sc.T <= 0 || g >= sc.Gd) return 0;
  const long long cb = group_tile_begin(g, sc.T, sc.Gd), ce = group_tile_begin(g + 1, sc.T, sc.Gd);
  if (cb >= ce) return 0;
  const int first = super_row_of_tile(sc, cb), last = super_row_of_tile(sc, ce - 1);
  int n = 0;
  for (int base = first; base <= last; base += 32) {
    const int s = base + lane;
    bool has = false;
    Segment sg{};
    if (s <= last) {
      const int b = s / d.nsub, k = s % d.nsub, i = k * d.wb + j;
      if (i < d.Qb) {
        const int K = clamp_len(p, b, nullptr), Kg = global_len(p, b, K);
        int ulo, U, tlo, nt;
        sub_span(p, d, b, k, K, Kg, ulo, U);
        work_span(p, b, i, K, Kg, tlo, nt);
        // the sub-band's tiles whose first unit lies in [cb, ce): i in [ceil((cb - pb) / 4),
        // ceil((ce - pb) / 4)), pb the unit of its tile 0; then those of this work row
        const long long pb = tile_unit(sc.prefix[s], p.piece_units, 0);
        const long long ib = cb <= pb ? 0 : (cb - pb + kUnitsPerTile - 1) / kUnitsPerTile;
        const long long ie = ce <= pb ? 0 : (ce - pb + kUnitsPerTile - 1) / kUnitsPerTile;
        const int t_begin = max(ulo + (int)min(ib, (long long)U), tlo);
        const int t_end = min(ulo + (int)min(ie, (long long)U), tlo + nt);
        if (U > 0 && t_begin < t_end) {
          int g_first;
          const int np = row_parts(sc, p.piece_units, s, ulo, tlo, nt, g_first);
          const int slot = np == 1 ? -1 : (s + g) * d.wb + j;
          sg.row_slot = (uint32_t)(b * d.Qb + i) | ((uint32_t)(slot + 1) << 14);
          sg.tile_begin = t_begin;
          sg.tile_end = t_end;
          sg.K = K;
          sg.parts = (uint32_t)np | ((uint32_t)(g - g_first) << 16);
          has = true;
        }
      }
    }
    const uint32_t mask = __ballot_sync(0xffffffffu, has);
    if (has) {
      const int at = n + __popc(mask & ((1u << lane) - 1u));
      if (at < kSmemSegs) segs[at] = sg;
      else overflow[at - kSmemSegs] = sg;
    }
    n += __popc(mask);
  }
  return n;
}

// Row table for the reduction and the header: the work rows spread over every CTA of
// the split-KV kernel, the header from block 0.
__device__ __forceinline__ void write_row_table(const DecodeParams& p, const Sched& sc) {
  const DealShape& d = sc.d;
  const WsLayout L = ws_layout(p.B, p.Sq, p.H, p.num_clusters, p.partial_f16);
  RowInfo* info = reinterpret_cast<RowInfo*>(p.ws + L.row_info);
  for (int w = blockIdx.x * blockDim.x + threadIdx.x; w < d.Rw; w += gridDim.x * blockDim.x) {
    const int b = w / d.Qb, i = w % d.Qb;
    const int k = i / d.wb, j = i % d.wb, s = b * d.nsub + k;
    const int K = clamp_len(p, b, nullptr), Kg = global_len(p, b, K);
    int tlo, n;
    work_span(p, b, i, K, Kg, tlo, n);
    RowInfo ri;
    ri.tile_lo = tlo;
    ri.n_tiles = n;
    ri.first_slot = 0;
    ri.n_parts = 0;
    if (n > 0) {
      int ulo, U, g_first;
      sub_span(p, d, b, k, K, Kg, ulo, U);
      ri.n_parts = row_parts(sc, p.piece_units, s, ulo, tlo, n, g_first);
      ri.first_slot = (s + g_first) * d.wb + j;
    }
    info[w] = ri;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    WsHeader* h = reinterpret_cast<WsHeader*>(p.ws);
    h->total_tiles = (int)sc.T;
    h->num_rows = d.Rw;
    h->num_clusters = p.num_clusters;
    h->deal_groups = sc.Gd;
    h->band = d.wb;
    h->super_rows = d.S;
    h->partial_f16 = p.partial_f16;
    h->pad = 0;
  }
}

}  // namespace mla
