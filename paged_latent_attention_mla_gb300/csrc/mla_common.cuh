// Shared definitions of the paged MLA decode kernels: sizes, the decode
// parameters, the visibility rule, the batch deal and the workspace layout.
// Host code (the plan, the workspace size) and device code (the schedule every
// CTA builds) use the same functions, so the two always agree.
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/mla.h"

namespace mla {

constexpr int kDLatent = 512;  // d_c, the latent width (also the value width)
constexpr int kDRope = 64;     // d_r, the rope width
constexpr int kDQK = kDLatent + kDRope;
constexpr int kKeyGroup = 64;  // keys per load unit: one [64 rows x 128 B] swizzled block per column block
constexpr int kTileN = 256;    // keys per KV tile: four key groups, two per CTA of a pair
constexpr int kRowsPerCta = 64;
constexpr int kTileM = 2 * kRowsPerCta;  // (token, head) rows of one work row: the M tile of the pair
constexpr int kMaxHeads = kTileM;
constexpr int kMinPageSize = 8;     // one 8-row group of the 128-byte swizzle
constexpr int kMaxPageSize = 1024;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // bounded device waits give up after 2 s
// The batch deal counts work in units of a quarter tile: a tile of 256 keys is 4 units,
// and every (sub-)band with visible keys is charged piece_units ahead of its tiles, what
// starting a piece costs a cluster (its Q, the pipeline refill, the epilogue), so that a
// cluster dealt many short rows gets fewer tiles.  Measured on GB300 (3 to 6 units swept
// over the benchmark batches), a whole tile is best: below it batches of many short rows
// overload the clusters dealt them, above it nothing gains.
constexpr int kUnitsPerTile = 4;
__host__ __device__ constexpr int piece_units(bool) { return kUnitsPerTile; }
// Segments (pieces of work) each CTA keeps in shared memory; a cluster dealt more keeps
// the rest in its workspace region.
constexpr int kSmemSegs = 192;

// status bits each CTA of the split-KV kernel leaves in its own status word
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrBadPage = 2u;
constexpr uint32_t kErrBadLength = 4u;

// -------------------------------------------------------------- decode parameters
struct DecodeParams {
  const void* q_latent;
  const void* q_rope;
  const void* ckv;
  const void* kpe;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* global_seq_lens;     // [B] whole-sequence lengths (context parallelism), or null
  const int32_t* local_visible_lens;  // [B, Sq] exclusive local bounds, or null
  void* out;
  float* lse;
  uint8_t* ws;
  int B, Sq, H, num_pages, pt_stride, page_size, page_shift, causal, window_left;
  int cp_world, cp_rank, cp_interleave;
  int qkv_e4m3, out_f32, partial_f16;
  int piece_units;             // the deal's charge for starting a piece (quarter tiles)
  int fused_combine;           // the last piece of a row combines it (no reduction kernel)
  uint32_t epoch;              // this call's tag in the rows' arrival counters
  int num_clusters;            // clusters launched (G)
  int reduce_d_tiles;          // CTAs per work row across the 512 output dims (1, 2, 4 or 8)
  float scale;                 // softmax scale
  float q_descale, ckv_descale, kpe_descale;
  float score_scale_log2;      // scale * q_descale * k_descale * log2(e) folded for exp2
};

__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }

// -------------------------------------------------------------- visibility
// Local keys of this rank below global position g: positions are dealt to the ranks in
// runs of I, run k to rank k % W, so full cycles of W*I positions hold I keys of each rank
// and the partial cycle holds min(I, max(0, rem - rank*I)).  W <= 1: g itself.
__host__ __device__ inline int dcp_local_bound(int g, int W, int rank, int I) {
  if (W <= 1) return g;
  if (g <= 0) return 0;
  const long long cycle = (long long)W * I;
  const long long full = g / cycle;
  long long tail = g - full * cycle - (long long)rank * I;
  tail = tail < 0 ? 0 : (tail > I ? I : tail);
  return (int)(full * I + tail);
}

// Visible local keys [lo, hi) of query token t of a request with K local keys.
//   hi: local_visible_lens[b, t] when given; else the causal bound Kg - (Sq - 1 - t) on the
//       whole sequence (Kg = K without context parallelism), mapped to this rank's keys;
//       else every key.
//   lo: the sliding-window floor Kg - Sq - window_left + t, mapped likewise (0 without a window).
// Both clamped to [0, K], lo <= hi.
__host__ __device__ inline void token_range(int K, int Kg, int lvl, bool has_lvl, int Sq, int t, int causal,
                                            int window_left, int W, int rank, int I, int& lo, int& hi) {
  int h;
  if (has_lvl) h = lvl;
  else if (causal) h = dcp_local_bound(Kg - (Sq - 1 - t), W, rank, I);
  else h = K;
  int l = window_left >= 0 ? dcp_local_bound(Kg - Sq - window_left + t, W, rank, I) : 0;
  h = h < 0 ? 0 : (h > K ? K : h);
  l = l < 0 ? 0 : (l > K ? K : l);
  if (l > h) l = h;
  lo = l;
  hi = h;
}

// tiles of kTileN keys that hold keys in [lo, hi)
__host__ __device__ inline void tile_span(int lo, int hi, int& tile_lo, int& n_tiles) {
  if (hi <= lo) {
    tile_lo = 0;
    n_tiles = 0;
    return;
  }
  tile_lo = lo / kTileN;
  n_tiles = (hi + kTileN - 1) / kTileN - tile_lo;
}

// -------------------------------------------------------------- the batch deal
// Work rows.  A request's Sq * H (token, head) rows, token-major, are cut into Qb =
// ceil(Sq * H / 128) work rows of 128: M row m of work row i is flat row 128 i + m, token
// (128 i + m) / H, head (128 i + m) % H (consecutive tokens pack into one M tile when
// H < 128).  Work row w = b * Qb + i.
//
// Bands.  The work rows of a request read the same KV, so they are dealt side by side:
// with G clusters launched, a group of wb = min(Qb, G) clusters walks the same tiles of a
// request together, lane j of the group taking work rows j, j + wb, ... (sub-band k holds
// work rows [k wb, k wb + wb)).  Super-row s = b * nsub + k is one sub-band; it costs
// piece_units + 4 U units, U the tiles of the union of its work rows' spans.  The
// super-rows' units are laid end to end (prefix sums) and dealt in equal contiguous shares
// to Gd = min(G / wb, T / 4) groups (every share at least one tile's worth): group g owns
// units [g T / Gd, (g+1) T / Gd), and a tile belongs to the group whose share holds its
// first unit.  Tile i of super-row s (counted from the sub-band's first tile) starts at
// unit prefix[s] + piece_units + 4 i; inside a row's tiles any 4 consecutive units hold
// one tile start, so every group between a row's first and last piece owns tiles of it.
//
// Slots.  The piece of work row k wb + j that group g computes writes partial slot
// (s + g) * wb + j: the groups holding one super-row are consecutive, so these never
// collide, and a work row's pieces sit wb slots apart.
struct DealShape {
  int Qb;     // work rows per request
  int wb;     // band width: clusters of a group
  int nsub;   // sub-bands (super-rows) per request
  int S;      // super-rows
  int Rw;     // work rows
  int Gg;     // groups that fit the clusters launched
  int slots;  // partial slots
};

__host__ __device__ inline DealShape deal_shape(int B, int Sq, int H, int G) {
  DealShape d;
  d.Qb = cdiv(Sq * H, kTileM);
  d.wb = d.Qb < G ? d.Qb : G;
  if (d.wb < 1) d.wb = 1;
  d.nsub = cdiv(d.Qb, d.wb);
  d.S = B * d.nsub;
  d.Rw = B * d.Qb;
  d.Gg = G / d.wb;
  if (d.Gg < 1) d.Gg = 1;
  d.slots = (d.S + d.Gg) * d.wb;
  return d;
}

// tokens [t0, t1] held by work rows [i0, i1] of a request
__host__ __device__ inline void work_tokens(int i0, int i1, int Sq, int H, int& t0, int& t1) {
  t0 = (kTileM * i0) / H;
  const int last = (kTileM * (i1 + 1) < Sq * H ? kTileM * (i1 + 1) : Sq * H) - 1;
  t1 = last / H;
}

// group holding unit x when T units are dealt to Gd groups in equal contiguous shares
// [floor(g*T/Gd), floor((g+1)*T/Gd))
// (32-bit arithmetic when the products fit, as they do for any batch of practical size)
__host__ __device__ inline int group_of_tile(long long x, long long T, long long Gd) {
  if (T < (1 << 20) && Gd <= 2048) return (int)((((uint32_t)x + 1u) * (uint32_t)Gd - 1u) / (uint32_t)T);
  return (int)(((x + 1) * Gd - 1) / T);
}

__host__ __device__ inline long long group_tile_begin(long long g, long long T, long long Gd) {
  if (T < (1 << 20) && Gd <= 2048) return (long long)(((uint32_t)g * (uint32_t)T) / (uint32_t)Gd);
  return g * T / Gd;
}

// groups the T units are dealt to: every share at least one tile's worth of units
__host__ __device__ inline int deal_groups(int Gg, long long T) {
  const long long most = T / kUnitsPerTile;
  return most < 1 ? 1 : (most < Gg ? (int)most : Gg);
}

// first unit of tile i (counted from the sub-band's first tile) of a super-row whose
// units start at `start`
__host__ __device__ inline long long tile_unit(long long start, int pu, int i) {
  return start + pu + (long long)kUnitsPerTile * i;
}

// -------------------------------------------------------------- workspace
// [header 256 B][cta_status 2G][row_info Rw][overflow segments 2G x max(0, S - kSmemSegs)]
// [partial_lse slots x 128 fp32][fp16: partial_scale slots x 2 x 128 fp32]
// [partial_o slots x 128 x 512, fp32 or fp16]
// A slot's O is laid out [dim / V][row][dim % V] with V = 4 (fp32) or 8 (fp16): a warp's
// 16-byte store (V dims of 32 consecutive rows) is 512 contiguous bytes.  fp16 partials
// are scaled by a power of two per (row, half of the dims: 256 c + 128 h + [0, 128)) so the
// half's largest |value| lands in [2^14, 2^15): any finite value fits, with fp16's 11 bits;
// partial_scale holds the base-2 exponent that undoes it.
// Every CTA of the split-KV kernel overwrites its own status word on every call and the
// schedule rewrites the header and row table, so the workspace needs no clearing.
struct WsHeader {
  int32_t total_tiles;
  int32_t num_rows;       // work rows Rw
  int32_t num_clusters;   // clusters launched (the layout's G)
  int32_t deal_groups;    // groups the tiles were dealt to
  int32_t band;           // wb
  int32_t super_rows;     // S
  int32_t partial_f16;
  int32_t pad;
};

struct RowInfo {
  int32_t tile_lo;     // first KV tile holding a visible key of the work row
  int32_t n_tiles;     // tiles from tile_lo on (0: no visible key in any of its rows)
  int32_t first_slot;  // partial slot of the first piece (pieces sit wb slots apart)
  int32_t n_parts;     // pieces (0: empty, 1: written to the output by the split-KV kernel)
};

// One piece of work of a cluster.  The work row (< 2^14) and the partial slot + 1 (0: the
// row's only piece, written to the output) share one word; K is the request's local key
// count, so the roles start a piece without reading seq_lens.
struct Segment {
  uint32_t row_slot;   // row | (slot + 1) << 14
  int32_t tile_begin;  // tiles [tile_begin, tile_end) of the work row
  int32_t tile_end;
  int32_t K;
  uint32_t parts;      // the row's pieces | this piece's index among them << 16
  __host__ __device__ int row() const { return (int)(row_slot & 0x3FFFu); }
  __host__ __device__ int slot() const { return (int)(row_slot >> 14) - 1; }
  __host__ __device__ int n_parts() const { return (int)(parts & 0xFFFFu); }
  __host__ __device__ int piece() const { return (int)(parts >> 16); }
};
constexpr int kMaxWorkRows = 1 << 14;
constexpr int kMaxClusters = 1024;  // the partial slot of a segment has 18 bits

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t cta_status, row_info, counters, segs, partial_lse, partial_scale, partial_o, total;
  size_t slot_bytes;  // bytes of one slot's O
  int seg_cap;        // overflow segments per CTA
};

__host__ __device__ inline WsLayout ws_layout(int B, int Sq, int H, int G, int partial_f16) {
  const DealShape d = deal_shape(B, Sq, H, G);
  WsLayout l{};
  l.seg_cap = d.S > kSmemSegs ? d.S - kSmemSegs : 0;
  l.slot_bytes = (size_t)kTileM * kDLatent * (partial_f16 ? 2 : 4);
  size_t off = align256(sizeof(WsHeader));
  l.cta_status = off;
  off = align256(off + sizeof(uint32_t) * 2 * (size_t)kMaxClusters);
  // [work row][CTA of the pair] arrival counters, epoch << 32 | pieces arrived: at the same
  // offset and size for every shape, so no other region of an earlier call's layout lands
  // on them (a zeroed workspace stays valid across plans of any shape)
  l.counters = off;
  off = align256(off + sizeof(unsigned long long) * 2 * (size_t)kMaxWorkRows);
  l.row_info = off;
  off = align256(off + sizeof(RowInfo) * (size_t)d.Rw);
  l.segs = off;
  off = align256(off + sizeof(Segment) * 2 * (size_t)G * (size_t)l.seg_cap);
  l.partial_lse = off;
  off = align256(off + sizeof(float) * (size_t)d.slots * kTileM);
  l.partial_scale = off;  // fp16: [slot][half][row]
  if (partial_f16) off = align256(off + sizeof(float) * (size_t)d.slots * 2 * kTileM);
  l.partial_o = off;
  off = align256(off + l.slot_bytes * (size_t)d.slots);
  l.total = off;
  return l;
}

// -------------------------------------------------------------- launch entry points (mla_kernels.cu)
cudaError_t launch_reduce(const DecodeParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_merge(const void* o_parts, const float* lse_parts, int world, long long rows, int out_f32,
                         void* out, float* lse, cudaStream_t stream);

}  // namespace mla
