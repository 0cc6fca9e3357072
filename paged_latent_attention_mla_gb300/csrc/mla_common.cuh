// Shared definitions of the paged MLA decode kernels: sizes, the workspace
// layout, the visibility rule and the batch schedule.
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/mla.h"

namespace mla {

constexpr int kDLatent = 512;  // d_c, the latent width (also the value width)
constexpr int kDRope = 64;     // d_r, the rope width
constexpr int kDQK = kDLatent + kDRope;
constexpr int kPageSize = 64;  // keys per cache page
constexpr int kTileN = 256;    // keys per KV tile: four pages, two per CTA of a pair
constexpr int kRowsPerCta = 64;
constexpr int kHeadsPad = 2 * kRowsPerCta;  // one M=128 tile of heads per (request, token) row
constexpr int kMaxHeads = kHeadsPad;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // bounded device waits give up after 2 s
// The batch deal charges every row with visible keys this many virtual tiles ahead of its
// real ones: what starting a piece costs a cluster (its Q, the pipeline refill, the
// epilogue), so that a cluster dealt many short rows gets fewer tiles.
constexpr int kPieceCost = 1;

// status bits each CTA of the split-KV kernel leaves in its own status word
constexpr uint32_t kErrTimeout = 1u;
constexpr uint32_t kErrBadPage = 2u;
constexpr uint32_t kErrBadLength = 4u;

// -------------------------------------------------------------- workspace
// [header 256 B][cta_status 2G][row_info R][partial_lse S x 128][partial_o S x 128 x 512]
// with S = R + G partial slots: the pieces of row r dealt to cluster c use slot r + c.
// Every CTA of the split-KV kernel overwrites its own status word on every call,
// so the workspace needs no clearing between calls.
struct WsHeader {
  int32_t total_tiles;
  int32_t num_rows;
  int32_t num_clusters;   // clusters launched (the layout's G)
  int32_t deal_clusters;  // clusters the tiles were dealt to
};

struct RowInfo {
  int32_t tile_lo;     // first KV tile (key index / kTileN) holding a visible key
  int32_t n_tiles;     // tiles from tile_lo on that hold visible keys (0: empty row)
  int32_t prefix;      // virtual tiles of all earlier rows (the batch deal's row start)
  int32_t first_slot;  // partial slot of the row's first piece
  int32_t n_parts;     // pieces the row is cut into (0: empty, 1: written directly)
  int32_t key_lo;      // visible keys [key_lo, key_hi)
  int32_t key_hi;
  int32_t pad;
};

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t cta_status, row_info, partial_lse, partial_o, total;
  int slots;
};

__host__ __device__ inline WsLayout ws_layout(int num_rows, int num_clusters) {
  WsLayout l{};
  l.slots = num_rows + num_clusters;
  size_t off = align256(sizeof(WsHeader));
  l.cta_status = off;
  off = align256(off + sizeof(uint32_t) * 2 * (size_t)num_clusters);
  l.row_info = off;
  off = align256(off + sizeof(RowInfo) * (size_t)num_rows);
  l.partial_lse = off;
  off = align256(off + sizeof(float) * (size_t)l.slots * kHeadsPad);
  l.partial_o = off;
  off = align256(off + sizeof(float) * (size_t)l.slots * kHeadsPad * kDLatent);
  l.total = off;
  return l;
}

// -------------------------------------------------------------- visibility
// Visible keys [lo, hi) of query token t of a request with K cached keys: the
// causal bound K - (Sq - 1 - t) and the sliding-window floor
// K - Sq - window_left + t, both clamped to [0, K].
__host__ __device__ inline void visible_range(int K, int Sq, int t, int causal, int window_left, int& lo, int& hi) {
  int h = causal ? K - (Sq - 1 - t) : K;
  int l = window_left >= 0 ? K - Sq - window_left + t : 0;
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

// cluster holding virtual tile x when T virtual tiles are dealt to G clusters in equal
// contiguous shares [floor(c*T/G), floor((c+1)*T/G))
__host__ __device__ inline int cluster_of_tile(long long x, long long T, long long G) {
  return (int)(((x + 1) * G - 1) / T);
}

__host__ __device__ inline long long cluster_tile_begin(long long c, long long T, long long G) { return c * T / G; }

// clusters the T tiles are dealt to: never more than T, so none is empty
__host__ __device__ inline int deal_clusters(int launched, long long T) {
  return T < 1 ? 1 : (T < launched ? (int)T : launched);
}

// -------------------------------------------------------------- launch entry points (mla_kernels.cu)
struct DecodeParams {
  const void* q_latent;
  const void* q_rope;
  const void* ckv;
  const void* kpe;
  const int32_t* page_table;
  const int32_t* seq_lens;
  void* out;
  float* lse;
  uint8_t* ws;
  int B, Sq, H, num_pages, pt_stride, causal, window_left;
  int qkv_e4m3, out_f32;
  int num_clusters;
  float scale;                 // softmax scale
  float q_descale, ckv_descale, kpe_descale;
  float score_scale_log2;      // scale * q_descale * k_descale * log2(e) folded for exp2
};

cudaError_t launch_reduce(const DecodeParams& p, cudaStream_t stream);

}  // namespace mla
