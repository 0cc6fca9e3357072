// Launch entry points of the device kernels (host side of the C ABI calls them).
#pragma once
#include <cuda_runtime.h>

#include "mla_common.cuh"
#include "tma_pages.cuh"

namespace mla {

cudaError_t launch_debug_wait_timeout(uint64_t timeout_ns, uint32_t* status_words, cudaStream_t stream);
cudaError_t launch_debug_mask(const DecodeParams& p, int max_k, uint32_t* bits, cudaStream_t stream);
cudaError_t launch_debug_gather(const KvMaps& maps, bool e4m3, const int32_t* page_table, const int32_t* seq_lens,
                                int B, int pt_stride, int num_pages, int page_size, int max_k, void* out,
                                uint32_t* err, cudaStream_t stream);
// split-KV decode kernel: one persistent wave of 2-CTA clusters
cudaError_t launch_split_kv(const DecodeParams& p, const KvMaps& maps, cudaStream_t stream);
// clusters of the split-KV kernel resident at once on `device` (0 on error)
int split_kv_max_clusters(int device, bool e4m3);

}  // namespace mla
