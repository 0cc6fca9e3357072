// Paged KV tile loads: one TMA box per (page, 128-byte column block).
//
// The caches are described to TMA as 3-D tensors [num_pages][64 slots][D]
// (innermost first: D, slot, page) with 128-byte swizzle, so one box
// {128 B of columns, 64 slots, 1 page} lands as a [64 rows x 128 B] swizzled
// block that the tensor core reads directly.  A page id outside [0, num_pages)
// is replaced by num_pages, which TMA answers with zeros (out-of-bounds fill).
#pragma once
#include "mla_common.cuh"
#include "ptx.cuh"

namespace mla {

struct KvMaps {
  CUtensorMap ckv;  // [pages][64][512], box {128 B, 64, 1}
  CUtensorMap kpe;  // [pages][64][64],  box {128 B, 64, 1} (e4m3: 64 B of data + 64 B zero fill)
  CUtensorMap q_latent;  // [B*Sq][H][512], box {128 B, 64 heads, 1}
  CUtensorMap q_rope;    // [B*Sq][H][64]
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

// page id of key page `lp` (logical page index) of request b, or num_pages
// (out of range: zero fill) for an invalid entry
__device__ __forceinline__ int page_of(const int32_t* page_table, int pt_stride, int num_pages, int b, int lp,
                                       bool& bad) {
  const int pg = __ldg(page_table + (size_t)b * pt_stride + lp);
  bad = (unsigned)pg >= (unsigned)num_pages;
  return bad ? num_pages : pg;
}

// Zero rows [row0, 64) of a [64 x 128 B] swizzled block (the slots past the
// last valid key of a request): any bits there (NaN included) must not reach
// the P.V product.  Generic-proxy writes: fence before the tensor core reads.
__device__ __forceinline__ void zero_block_rows(uint8_t* block, int row0, int lane, int nlanes) {
  for (int i = row0 * 8 + lane; i < 64 * 8; i += nlanes)
    *reinterpret_cast<uint4*>(block + i * 16) = make_uint4(0, 0, 0, 0);
}

}  // namespace mla
