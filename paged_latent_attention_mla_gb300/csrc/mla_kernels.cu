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

// One CTA per (row, 64 dims): the row's pieces combined with weights
// exp2(lse_i - lse), lse = log2 of the summed exp2(lse_i) (one piece: weight 1, a
// copy).  Pieces are workspace slots laid out [dim / 4][head][dim % 4], so a
// warp's float4 loads are 512 contiguous bytes; the block transposes through
// shared memory and writes the output head-major with each head's dims contiguous.
constexpr int kReduceDims = 64;

__global__ void __launch_bounds__(256) reduce_kernel(const DecodeParams p) {
  __shared__ float tile[kHeadsPad][kReduceDims + 1];  // [head][dim], padded against bank conflicts
  const int r = blockIdx.y, d0 = blockIdx.x * kReduceDims;
  const int h = threadIdx.x & (kHeadsPad - 1), dg = threadIdx.x >> 7;  // 32 dims per thread
  const WsLayout L = ws_layout(p.B * p.Sq, p.num_clusters);
  const RowInfo ri = reinterpret_cast<const RowInfo*>(p.ws + L.row_info)[r];
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  float lse2 = -INFINITY;
  if (h < p.H && ri.n_parts > 0) {
    const float* plse = reinterpret_cast<const float*>(p.ws + L.partial_lse) + (size_t)ri.first_slot * kHeadsPad + h;
    const float4* po = reinterpret_cast<const float4*>(p.ws + L.partial_o) +
                       ((size_t)ri.first_slot * (kDLatent / 4) + (d0 + 32 * dg) / 4) * kHeadsPad + h;
    const int np = ri.n_parts;
    // two pieces per round; each round's partial loads are issued before its weights are
    // known (the first round's before the LSE arithmetic).  An empty piece (LSE -inf, slot
    // never written) gets weight 0 and is selected away.
    float4 x[2][8];
    auto load_round = [&](int i0) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = i0 + u < np ? i0 + u : i0;
        const float4* src = po + (size_t)i * (kDLatent / 4) * kHeadsPad;
#pragma unroll
        for (int q = 0; q < 8; ++q) x[u][q] = __ldcs(src + (size_t)q * kHeadsPad);
      }
    };
    load_round(0);
    // the pieces' LSEs: loads issued together, then max and sum
    float mx = -INFINITY;
#pragma unroll 4
    for (int i = 0; i < np; ++i) mx = fmaxf(mx, plse[(size_t)i * kHeadsPad]);
    const float m0 = mx == -INFINITY ? 0.f : mx;
    float sum = 0.f;
#pragma unroll 4
    for (int i = 0; i < np; ++i) sum += exp2f(plse[(size_t)i * kHeadsPad] - m0);
    lse2 = sum > 0.f ? m0 + log2f(sum) : -INFINITY;
    for (int i0 = 0; i0 < np; i0 += 2) {
      if (i0 > 0) load_round(i0);
      float w[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float li = plse[(size_t)(i0 + u < np ? i0 + u : i0) * kHeadsPad];
        w[u] = (sum > 0.f && i0 + u < np && li != -INFINITY) ? exp2f(li - lse2) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (w[u] == 0.f) continue;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          acc[4 * q] += w[u] * x[u][q].x;
          acc[4 * q + 1] += w[u] * x[u][q].y;
          acc[4 * q + 2] += w[u] * x[u][q].z;
          acc[4 * q + 3] += w[u] * x[u][q].w;
        }
      }
    }
  }
  // n_parts == 0: no visible key, O = 0 and LSE = -inf
#pragma unroll
  for (int e = 0; e < 32; ++e) tile[h][32 * dg + e] = acc[e];
  __syncthreads();
  const int hh = threadIdx.x >> 1, part = threadIdx.x & 1;  // one head's 32 dims per thread
  if (hh < p.H) {
    const size_t out_row = (size_t)r * p.H + hh;
    const float* t = &tile[hh][32 * part];
    if (p.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + out_row * kDLatent + d0 + 32 * part);
#pragma unroll
      for (int v = 0; v < 8; ++v) dst[v] = make_float4(t[4 * v], t[4 * v + 1], t[4 * v + 2], t[4 * v + 3]);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + out_row * kDLatent + d0 + 32 * part);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(t[8 * v + 2 * e], t[8 * v + 2 * e + 1]);
          w[e] = *reinterpret_cast<uint32_t*>(&b2);
        }
        dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  if (p.lse && blockIdx.x == 0 && dg == 0 && h < p.H) p.lse[(size_t)r * p.H + h] = lse2 * 0.69314718055994530942f;
}

cudaError_t launch_reduce(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid(kDLatent / kReduceDims, p.B * p.Sq);
  reduce_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ debug wait timeout
// One 2-CTA cluster: tensor memory allocated, then a bounded wait on an mbarrier that
// nothing arrives at.  The wait gives up after timeout_ns, the CTAs meet, free the tensor
// memory and report the timeout bit in their status words.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64, 1) debug_wait_timeout_kernel(uint64_t timeout_ns,
                                                                                           uint32_t* status_words) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(smem_addr(&tmem_slot), 32);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  uint32_t err = 0;
  if (tid == 0 && !mbar_wait_bounded(smem_addr(&bar), 0, timeout_ns)) err = kErrTimeout;
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc_pair(tmem_slot, 32);
  if (tid == 0) status_words[cluster_ctarank()] = err;
}

cudaError_t launch_debug_wait_timeout(uint64_t timeout_ns, uint32_t* status_words, cudaStream_t stream) {
  debug_wait_timeout_kernel<<<2, 64, 0, stream>>>(timeout_ns, status_words);
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
