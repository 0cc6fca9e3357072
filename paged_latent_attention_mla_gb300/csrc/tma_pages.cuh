// Paged KV tile loads: TMA boxes of one page's rows x 128 bytes of columns.
//
// The caches are described to TMA as 3-D tensors [num_pages][page_size][D]
// (innermost first: D, slot, page) with 128-byte swizzle (64-byte for the e4m3
// rope), so a box {128 B of columns, r rows, 1 page} lands as r swizzled 128-byte
// rows that the tensor core reads directly.  The load unit is a group of 64 keys
// (one [64 rows x 128 B] block per column block): with page_size P >= 64 it is one
// box of 64 rows at a row offset inside its page, with P < 64 it is 64 / P boxes
// of P rows, one per page (P >= 8 keeps every box on whole 8-row swizzle groups).
// A box past a request's length, or whose page id is outside [0, num_pages), is
// pointed at page num_pages, which TMA answers with zeros (out-of-bounds fill).
#pragma once
#include "mla_common.cuh"
#include "ptx.cuh"

namespace mla {

struct KvMaps {
  CUtensorMap ckv;       // [pages][P][512], box {128 B, box_rows, 1}
  CUtensorMap kpe;       // [pages][P][64],  box {128 B (e4m3: 64 B), box_rows, 1}
  CUtensorMap q_latent;  // [B][Sq*H][512], box {128 B, 64 rows, 1}
  CUtensorMap q_rope;    // [B][Sq*H][64]
};

// elements per 128-byte column block
template <bool E4M3>
__host__ __device__ constexpr int blk_elems() {
  return E4M3 ? 128 : 64;
}
template <bool E4M3>
__host__ __device__ constexpr int latent_blocks() {
  return kDLatent / blk_elems<E4M3>();
}
constexpr int kBlockBytes = 64 * 128;  // one [64 rows x 128 B] block

// boxes per 64-key group and rows per box for page size P
__host__ __device__ constexpr int boxes_per_group(int P) { return P >= kKeyGroup ? 1 : kKeyGroup / P; }
__host__ __device__ constexpr int box_rows(int P) { return P >= kKeyGroup ? kKeyGroup : P; }

// Zero rows [row0, 64) of a [64 x 128 B] swizzled block (the slots past the
// last valid key of a request): any bits there (NaN included) must not reach
// the P.V product.  Generic-proxy writes: fence before the tensor core reads.
__device__ __forceinline__ void zero_block_rows(uint8_t* block, int row0, int lane, int nlanes) {
  for (int i = row0 * 8 + lane; i < 64 * 8; i += nlanes)
    *reinterpret_cast<uint4*>(block + i * 16) = make_uint4(0, 0, 0, 0);
}

// Page id and row offset of the box of keys starting at key0 of request b (K keys),
// P = 1 << page_shift: key0 >= K or an invalid page id -> page num_pages (zero fill),
// bad set for the latter.  Branch-free after the load, so a caller that reads ahead
// does not wait for the page table until it uses the page.
__device__ __forceinline__ void box_page(const int32_t* page_table, int pt_stride, int num_pages, int page_shift, int b,
                                         int key0, int K, int& page, int& row, bool& bad) {
  const bool in = key0 < K;
  const int lp = key0 >> page_shift;
  const int v = in ? __ldg(page_table + (size_t)b * pt_stride + lp) : num_pages;
  bad = in && (unsigned)v >= (unsigned)num_pages;
  page = in && !bad ? v : num_pages;
  row = in ? key0 - (lp << page_shift) : 0;
}

}  // namespace mla
