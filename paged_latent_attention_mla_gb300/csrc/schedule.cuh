// Batch schedule, computed on the device from seq_lens by every CTA of the
// split-KV kernel (in scratch shared memory, before the tile buffers are used).
//
// Every (request, token) row r = b * Sq + t has visible keys [lo, hi) and the
// KV tiles [tile_lo, tile_lo + n_r) that hold them.  Each row with n_r > 0 costs
// n_r + kPieceCost virtual tiles: kPieceCost for starting a piece, then its real
// tiles.  The rows' virtual tiles are laid end to end (row r starts at the prefix
// sum P_r, its real tiles at P_r + kPieceCost) and dealt out in equal contiguous
// shares to G = min(clusters launched, T) clusters of one persistent wave:
// cluster c owns virtual tiles [floor(c*T/G), floor((c+1)*T/G)) and works on the
// real tiles among them.
// The piece of row r owned by cluster c writes partial slot r + c, and the
// reduction kernel turns each row's slots into its output.
#pragma once
#include "mla_common.cuh"

namespace mla {

struct RowWork {
  int row, b, t;
  int key_lo, key_hi;    // visible keys of the row
  int tile_begin;        // first tile (key index / kTileN) of this piece
  int tile_end;          // one past its last tile
  int slot;              // partial slot (r + c)
  int n_parts;           // pieces the row is cut into
};

struct ScheduleView {
  const int32_t* prefix;  // [R + 1] in shared memory
  int R, T;
  int G;         // clusters the tiles are dealt to: min(launched, T), at least 1
  int G_layout;  // clusters launched (sizes the workspace)
};

__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b, uint32_t* err) {
  int K = p.seq_lens[b];
  const int cap = p.pt_stride * kPageSize;
  if (K < 0 || K > cap) {
    if (err) atomicOr(err, kErrBadLength);
    K = K < 0 ? 0 : cap;
  }
  return K;
}

__device__ __forceinline__ void row_span(const DecodeParams& p, int r, int K, int& lo, int& hi, int& tile_lo,
                                         int& n) {
  const int t = r % p.Sq;
  visible_range(K, p.Sq, t, p.causal, p.window_left, lo, hi);
  tile_span(lo, hi, tile_lo, n);
}

// Block-wide: fills prefix[0..R] (prefix[R] = T) in shared memory.  scratch
// needs R + 1 + 32 ints.  All threads of the block must call it.
__device__ inline ScheduleView build_schedule(const DecodeParams& p, int32_t* scratch, uint32_t* err_flag) {
  const int R = p.B * p.Sq;
  const int tid = threadIdx.x, nt = blockDim.x;
  int32_t* prefix = scratch;
  int32_t* part = scratch + R + 1;  // 32 ints
  // per-thread contiguous chunk of rows
  const int chunk = (R + nt - 1) / nt;
  const int r0 = min(R, tid * chunk), r1 = min(R, r0 + chunk);
  int local = 0;
  for (int r = r0; r < r1; ++r) {
    int lo, hi, tlo, n;
    row_span(p, r, clamp_len(p, r / p.Sq, err_flag), lo, hi, tlo, n);
    const int cost = n > 0 ? n + kPieceCost : 0;
    prefix[r] = cost;
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
  for (int r = r0; r < r1; ++r) {
    int n = prefix[r];
    prefix[r] = run;
    run += n;
  }
  if (tid == nt - 1) prefix[R] = run;  // last thread: run == T (also correct when its chunk is empty)
  __syncthreads();
  ScheduleView s;
  s.prefix = prefix;
  s.R = R;
  s.T = prefix[R];
  s.G_layout = p.num_clusters;
  s.G = deal_clusters(p.num_clusters, s.T);
  return s;
}

// largest row r with prefix[r] <= x (x < T): the row holding virtual tile x
__device__ inline int row_of_tile(const ScheduleView& s, int x) {
  int lo = 0, hi = s.R - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (s.prefix[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// rows [first, last] that hold cluster c's tiles (first > last: none)
__device__ inline void cluster_rows(const ScheduleView& s, int c, int& first, int& last) {
  first = 1;
  last = 0;
  if (s.T <= 0 || c >= s.G) return;
  const long long b = cluster_tile_begin(c, s.T, s.G), e = cluster_tile_begin(c + 1, s.T, s.G);
  if (b >= e) return;
  first = row_of_tile(s, (int)b);
  last = row_of_tile(s, (int)(e - 1));
}

// the piece of row r that cluster c owns (call for r in cluster_rows(c)): the row's
// real tiles inside the cluster's share, if any
__device__ inline bool row_piece(const DecodeParams& p, const ScheduleView& s, int c, int r, RowWork& w) {
  const int n = s.prefix[r + 1] - s.prefix[r] - kPieceCost;
  if (n <= 0) return false;
  const long long cb = cluster_tile_begin(c, s.T, s.G), ce = cluster_tile_begin(c + 1, s.T, s.G);
  const long long pb = s.prefix[r] + kPieceCost, pe = pb + n;
  const long long gb = pb > cb ? pb : cb, ge = pe < ce ? pe : ce;
  if (gb >= ge) return false;
  int lo, hi, tlo, nn;
  const int b = r / p.Sq;
  row_span(p, r, clamp_len(p, b, nullptr), lo, hi, tlo, nn);
  w.row = r;
  w.b = b;
  w.t = r % p.Sq;
  w.key_lo = lo;
  w.key_hi = hi;
  w.tile_begin = tlo + (int)(gb - pb);
  w.tile_end = tlo + (int)(ge - pb);
  w.slot = r + c;
  const int c_first = cluster_of_tile(pb, s.T, s.G), c_last = cluster_of_tile(pe - 1, s.T, s.G);
  w.n_parts = c_last - c_first + 1;
  return true;
}

// Row table for the reduction (written once, by CTA 0 of the split-KV kernel).
__device__ inline void write_row_table(const DecodeParams& p, const ScheduleView& s) {
  const WsLayout L = ws_layout(s.R, s.G_layout);
  RowInfo* info = reinterpret_cast<RowInfo*>(p.ws + L.row_info);
  for (int r = threadIdx.x; r < s.R; r += blockDim.x) {
    int lo, hi, tlo, n;
    row_span(p, r, clamp_len(p, r / p.Sq, nullptr), lo, hi, tlo, n);
    RowInfo ri;
    ri.tile_lo = tlo;
    ri.n_tiles = n;
    ri.prefix = s.prefix[r];
    ri.key_lo = lo;
    ri.key_hi = hi;
    ri.pad = 0;
    if (n > 0) {
      const long long pb = (long long)s.prefix[r] + kPieceCost;
      const int c_first = cluster_of_tile(pb, s.T, s.G);
      const int c_last = cluster_of_tile(pb + n - 1, s.T, s.G);
      ri.first_slot = r + c_first;
      ri.n_parts = c_last - c_first + 1;
    } else {
      ri.first_slot = 0;
      ri.n_parts = 0;
    }
    info[r] = ri;
  }
  if (threadIdx.x == 0) {
    WsHeader* h = reinterpret_cast<WsHeader*>(p.ws);
    h->total_tiles = s.T;
    h->num_rows = s.R;
    h->num_clusters = s.G_layout;
    h->deal_clusters = s.G;
  }
}

}  // namespace mla

namespace mla {

// One piece of work of a cluster: tiles [tile_begin, tile_end) of row `row`.
struct Segment {
  int32_t row;
  int32_t tile_begin;
  int32_t tile_end;
};

// Extract cluster c's pieces, in row order, into segs[0..n) (thread 0 of the
// block; the caller synchronizes).  Returns the number of pieces, capped at
// max_segs (an overflow sets kErrBadLength in *err).
__device__ inline int build_segments(const DecodeParams& p, const ScheduleView& s, int c, Segment* segs, int max_segs,
                                     uint32_t* err) {
  int first, last, n = 0;
  cluster_rows(s, c, first, last);
  for (int r = first; r <= last; ++r) {
    RowWork w;
    if (!row_piece(p, s, c, r, w)) continue;
    if (n == max_segs) {
      atomicOr(err, kErrBadLength);
      break;
    }
    segs[n].row = r;
    segs[n].tile_begin = w.tile_begin;
    segs[n].tile_end = w.tile_end;
    ++n;
  }
  return n;
}

}  // namespace mla
