// Split-KV reduction and the debug kernels (gather, mask).
//
// The reduction follows reduction_kernel of the kv_balanced_mla kernel page:
// the global base-2 log-sum-exp of a row's pieces is lse = max + log2(sum
// 2^(lse_i - max)) (max taken as 0 when every piece is empty), and the output
// is sum_i 2^(lse_i - lse) * O_i over the row's normalized partials.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla_common.cuh"
#include "mla_kernels.cuh"
#include "ptx.cuh"
#include "schedule.cuh"
#include "tma_pages.cuh"

namespace mla {

// ------------------------------------------------------------------ reduction
// grid (ceil(H / 4), R), block 128: each warp combines one head of one row,
// each lane 16 consecutive dims (four float4 loads per piece).
__global__ void __launch_bounds__(128) reduce_kernel(const DecodeParams p) {
  const int r = blockIdx.y;
  const int h = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= p.H) return;
  const WsLayout L = ws_layout(p.B * p.Sq, p.num_clusters);
  const RowInfo ri = reinterpret_cast<const RowInfo*>(p.ws + L.row_info)[r];
  if (ri.n_parts == 1) return;  // the split-KV kernel wrote this row directly
  const size_t out_row = (size_t)r * p.H + h;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float lse2 = -INFINITY;
  if (ri.n_parts > 1) {
    const float* plse = reinterpret_cast<const float*>(p.ws + L.partial_lse);
    const float* po = reinterpret_cast<const float*>(p.ws + L.partial_o);
    float mx = -INFINITY;
    for (int i = 0; i < ri.n_parts; ++i) mx = fmaxf(mx, plse[(size_t)(ri.first_slot + i) * kHeadsPad + h]);
    const float m0 = mx == -INFINITY ? 0.f : mx;
    float sum = 0.f;
    for (int i = 0; i < ri.n_parts; ++i) sum += exp2f(plse[(size_t)(ri.first_slot + i) * kHeadsPad + h] - m0);
    lse2 = sum > 0.f ? m0 + log2f(sum) : -INFINITY;
    if (sum > 0.f) {
      for (int i = 0; i < ri.n_parts; ++i) {
        const size_t slot = (size_t)(ri.first_slot + i);
        const float li = plse[slot * kHeadsPad + h];
        if (li == -INFINITY) continue;  // an empty piece adds nothing (and its partial is never read)
        const float w = exp2f(li - lse2);
        const float4* src = reinterpret_cast<const float4*>(po + (slot * kHeadsPad + h) * kDLatent) + lane * 4;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 x = __ldcs(src + v);
          acc[4 * v + 0] += w * x.x;
          acc[4 * v + 1] += w * x.y;
          acc[4 * v + 2] += w * x.z;
          acc[4 * v + 3] += w * x.w;
        }
      }
    }
  }
  // n_parts == 0: no visible key, O = 0 and LSE = -inf
  if (p.out_f32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + out_row * kDLatent) + lane * 4;
#pragma unroll
    for (int v = 0; v < 4; ++v) dst[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
  } else {
    __nv_bfloat162 b2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b2[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + out_row * kDLatent) + lane * 2;
    dst[0] = *reinterpret_cast<uint4*>(&b2[0]);
    dst[1] = *reinterpret_cast<uint4*>(&b2[4]);
  }
  if (p.lse && lane == 0) p.lse[out_row] = lse2 * 0.69314718055994530942f;
}

cudaError_t launch_reduce(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid((p.H + 3) / 4, p.B * p.Sq);
  reduce_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ debug mask
__global__ void debug_mask_kernel(const int32_t* seq_lens, int Sq, int causal, int window_left, int max_k,
                                  uint32_t* bits) {
  const int row = blockIdx.x;  // b * Sq + t
  const int b = row / Sq, t = row % Sq;
  int lo, hi;
  visible_range(seq_lens[b], Sq, t, causal, window_left, lo, hi);
  const int n_words = (max_k + 31) / 32;
  for (int w = threadIdx.x; w < n_words; w += blockDim.x) {
    uint32_t word = 0;
    for (int i = 0; i < 32; ++i) {
      const int k = 32 * w + i;
      if (k < max_k && k >= lo && k < hi) word |= 1u << i;
    }
    bits[(size_t)row * n_words + w] = word;
  }
}

cudaError_t launch_debug_mask(const int32_t* seq_lens, int B, int Sq, int causal, int window_left, int max_k,
                              uint32_t* bits, cudaStream_t stream) {
  debug_mask_kernel<<<B * Sq, 128, 0, stream>>>(seq_lens, Sq, causal, window_left, max_k, bits);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ debug gather
// One CTA per (page of keys, request): the decode kernel's page lookup and TMA
// boxes bring the page's latent and rope blocks into swizzled shared memory,
// the slots past the request's length are zeroed as the decode kernel zeroes
// them, and the block is written back densely.
template <bool E4M3>
__global__ void __launch_bounds__(256) debug_gather_kernel(const __grid_constant__ KvMaps maps,
                                                           const int32_t* page_table, const int32_t* seq_lens,
                                                           int pt_stride, int num_pages, int max_k, uint8_t* out,
                                                           uint32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int es = E4M3 ? 1 : 2;
  constexpr int nlat = latent_blocks<E4M3>();
  const int lp = blockIdx.x, b = blockIdx.y;
  const int K = min(max(seq_lens[b], 0), pt_stride * kPageSize);
  const int key0 = lp * kPageSize;
  if (key0 >= max_k) return;
  const int valid = min(max(K - key0, 0), kPageSize);
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (valid > 0) {
    if (threadIdx.x == 0) {
      bool bad;
      const int pg = page_of(page_table, pt_stride, num_pages, b, lp, bad);
      if (bad && err) atomicOr(err, kErrBadPage);
      constexpr uint32_t rope_bytes = E4M3 ? 64 * 64 : kBlockBytes;
      mbar_arrive_expect_tx(smem_addr(&bar), nlat * kBlockBytes + rope_bytes);
      for (int kb = 0; kb < nlat; ++kb)
        tma_load_3d(smem_addr(smem + kb * kBlockBytes), &maps.ckv, kb * blk_elems<E4M3>(), 0, pg, smem_addr(&bar));
      tma_load_3d(smem_addr(smem + nlat * kBlockBytes), &maps.kpe, 0, 0, pg, smem_addr(&bar));
    }
    if (!mbar_wait_bounded(smem_addr(&bar), 0, kWaitTimeoutNs)) {
      if (threadIdx.x == 0 && err) atomicOr(err, kErrTimeout);
      return;
    }
    // slots past the request's length: zero, as the decode kernel does before P.V
    if (valid < kPageSize)
      for (int kb = 0; kb < nlat; ++kb) zero_block_rows(smem + kb * kBlockBytes, valid, threadIdx.x, blockDim.x);
    __syncthreads();
  }
  // write back: row j of this page -> out[b][key0 + j][0:576]
  const int row_bytes = kDQK * es;
  const int rows = min(kPageSize, max_k - key0);
  for (int i = threadIdx.x; i < rows * (row_bytes / 16); i += blockDim.x) {
    const int j = i / (row_bytes / 16), ch = i % (row_bytes / 16);  // 16-byte chunk of the dense row
    uint4 v = make_uint4(0, 0, 0, 0);
    if (j < valid) {
      const int byte = ch * 16;
      if (byte < kDLatent * es) {
        const int kb = byte / 128, within = byte % 128;
        v = *reinterpret_cast<const uint4*>(smem + kb * kBlockBytes + sw128_offset(j, within / 16));
      } else {
        const int within = byte - kDLatent * es;
        if (E4M3)  // 64-byte swizzled rows: chunk index XOR (row / 2) & 3
          v = *reinterpret_cast<const uint4*>(smem + nlat * kBlockBytes + j * 64 + (((within / 16) ^ ((j >> 1) & 3)) << 4));
        else
          v = *reinterpret_cast<const uint4*>(smem + nlat * kBlockBytes + sw128_offset(j, within / 16));
      }
    }
    *reinterpret_cast<uint4*>(out + ((size_t)b * max_k + key0 + j) * row_bytes + ch * 16) = v;
  }
}

cudaError_t launch_debug_gather(const KvMaps& maps, bool e4m3, const int32_t* page_table, const int32_t* seq_lens,
                                int B, int pt_stride, int num_pages, int max_k, void* out, uint32_t* err,
                                cudaStream_t stream) {
  dim3 grid((max_k + kPageSize - 1) / kPageSize, B);
  const int smem = 9 * kBlockBytes + 1024;
  cudaError_t e;
  if (e4m3) {
    e = cudaFuncSetAttribute(debug_gather_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    debug_gather_kernel<true><<<grid, 256, smem, stream>>>(maps, page_table, seq_lens, pt_stride, num_pages, max_k,
                                                            static_cast<uint8_t*>(out), err);
  } else {
    e = cudaFuncSetAttribute(debug_gather_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    debug_gather_kernel<false><<<grid, 256, smem, stream>>>(maps, page_table, seq_lens, pt_stride, num_pages, max_k,
                                                             static_cast<uint8_t*>(out), err);
  }
  return cudaGetLastError();
}

}  // namespace mla
