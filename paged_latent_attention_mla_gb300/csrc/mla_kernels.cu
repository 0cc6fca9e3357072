// Split-KV reduction, the context-parallel merge and the debug kernels (gather, mask).
//
// The reduction follows reduction_kernel of the kv_balanced_mla kernel page:
// the global base-2 log-sum-exp of a row's pieces is lse = max + log2(sum
// 2^(lse_i - max)) (max taken as 0 when every piece is empty), and the output
// is output_scale * sum_i 2^(lse_i - lse) * O_i over the row's normalized
// partials (fp32, or fp16 as __init__'s partial_fp16 allows: a normalized partial
// is a convex combination of stored value codes), in 1, 2, 4 or 8 bands of the 512
// output dims (reducer_d_tiles).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mla_common.cuh"
#include "mla_kernels.cuh"
#include "ptx.cuh"
#include "schedule.cuh"
#include "tma_pages.cuh"

namespace mla {

// One CTA per (work row, band of 512 / d_tiles output dims), 256 threads: thread
// (m, dg) with m = tid & 127 the work row's M row and dg = tid >> 7 the half of each
// 64-dim chunk it accumulates.  A row's pieces are combined with weights
// 2^(lse_i - lse) times the value scale (the partials hold O / l in the stored codes'
// units), lse = log2 of the summed 2^(lse_i).  Slots are laid out [dim / V][row][dim % V]
// (V = 4 fp32, 8 fp16), so a warp's 16-byte loads are 512 contiguous bytes; the block
// transposes each 64-dim chunk through shared memory and writes the output row-major.
// Work rows written whole by the split-KV kernel (one piece) are skipped.
template <bool F16>
__global__ void __launch_bounds__(256, 2) reduce_kernel(const DecodeParams p) {
  grid_dependency_wait();  // the split-KV kernel's partials (programmatic dependent launch)
  __shared__ float tile[kTileM][64 + 1];  // [row][dim], padded against bank conflicts
  const int w = blockIdx.y;
  const WsLayout L = ws_layout(p.B, p.Sq, p.H, p.num_clusters, p.partial_f16);
  const DealShape d = deal_shape(p.B, p.Sq, p.H, p.num_clusters);
  const RowInfo ri = reinterpret_cast<const RowInfo*>(p.ws + L.row_info)[w];
  if (ri.n_parts == 1) return;
  const int m = threadIdx.x & (kTileM - 1), dg = threadIdx.x >> 7;
  const int rows_q = p.Sq * p.H;
  const int b = w / d.Qb, flat0 = kTileM * (w % d.Qb);
  const bool live = flat0 + m < rows_q;
  const int np = live ? ri.n_parts : 0;
  const float* plse = reinterpret_cast<const float*>(p.ws + L.partial_lse) + m;
  const uint8_t* po = p.ws + L.partial_o;
  auto slot_of = [&](int i) { return (size_t)ri.first_slot + (size_t)i * d.wb; };
  // fp16 partials carry a power-of-two scale per (row, half of each 256-dim chunk); a
  // thread's 32 dims lie in one half
  const float* pscale = reinterpret_cast<const float*>(p.ws + L.partial_scale) + m;
  // 32 dims of piece i from d0 into x, and their scale exponent (loaded with them)
  auto load = [&](int i, int d0, float (&x)[32], float& sc) {
    const size_t sl = slot_of(i);
    if constexpr (F16) {
      sc = pscale[(sl * 2 + ((d0 >> 7) & 1)) * kTileM];
      const uint4* src = reinterpret_cast<const uint4*>(po + sl * L.slot_bytes) + m;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = __ldcs(src + (size_t)(d0 / 8 + q) * kTileM);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[e]));
          x[8 * q + 2 * e] = f.x;
          x[8 * q + 2 * e + 1] = f.y;
        }
      }
    } else {
      sc = 0.f;
      const float4* src = reinterpret_cast<const float4*>(po + sl * L.slot_bytes) + m;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 v = __ldcs(src + (size_t)(d0 / 4 + q) * kTileM);
        x[4 * q] = v.x;
        x[4 * q + 1] = v.y;
        x[4 * q + 2] = v.z;
        x[4 * q + 3] = v.w;
      }
    }
  };
  const int band = kDLatent / p.reduce_d_tiles;
  // the first round's partials (pieces 0 and 1 of the first chunk) go out with the LSE
  // loads, before the LSE arithmetic: one dependent round trip fewer
  float x[2][32], xs[2] = {0.f, 0.f};
  if (np > 0) {
    load(0, blockIdx.x * band + 32 * dg, x[0], xs[0]);
    load(np > 1 ? 1 : 0, blockIdx.x * band + 32 * dg, x[1], xs[1]);
  }
  // the pieces' LSEs: max, sum, the row's LSE
  float mx = -INFINITY;
  for (int i = 0; i < np; ++i) mx = fmaxf(mx, plse[slot_of(i) * kTileM]);
  const float m0 = mx == -INFINITY ? 0.f : mx;
  float sum = 0.f;
  for (int i = 0; i < np; ++i) sum += exp2f(plse[slot_of(i) * kTileM] - m0);
  const float lse2 = sum > 0.f ? m0 + log2f(sum) : -INFINITY;
  auto weight = [&](int i, float sc) {
    const float li = plse[slot_of(i) * kTileM];
    return (sum > 0.f && li != -INFINITY) ? exp2f(li - lse2 + sc) * p.ckv_descale : 0.f;
  };
  for (int c = 0; c < band / 64; ++c) {
    const int d0 = blockIdx.x * band + 64 * c + 32 * dg;  // this thread's 32 dims
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
    // two pieces per round, both rounds' loads issued before their weights are applied;
    // an empty piece (LSE -inf) gets weight 0 and is selected away
    for (int i0 = 0; i0 < np; i0 += 2) {
      if (c > 0 || i0 > 0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) load(i0 + u < np ? i0 + u : i0, d0, x[u], xs[u]);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float wt = i0 + u < np ? weight(i0 + u, xs[u]) : 0.f;
        if (wt == 0.f) continue;
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] += wt * x[u][e];
      }
    }
    // np == 0: no visible key, O = 0
#pragma unroll
    for (int e = 0; e < 32; ++e) tile[m][32 * dg + e] = acc[e];
    __syncthreads();
    const int hh = threadIdx.x >> 1, part = threadIdx.x & 1;  // one row's 32 dims per thread
    if (flat0 + hh < rows_q) {
      const size_t out_row = (size_t)b * rows_q + flat0 + hh;
      const int od = blockIdx.x * band + 64 * c + 32 * part;
      const float* t = &tile[hh][32 * part];
      if (p.out_f32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + out_row * kDLatent + od);
#pragma unroll
        for (int v = 0; v < 8; ++v) dst[v] = make_float4(t[4 * v], t[4 * v + 1], t[4 * v + 2], t[4 * v + 3]);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + out_row * kDLatent + od);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(t[8 * v + 2 * e], t[8 * v + 2 * e + 1]);
            wv[e] = *reinterpret_cast<uint32_t*>(&b2);
          }
          dst[v] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
    __syncthreads();
  }
  if (p.lse && blockIdx.x == 0 && dg == 0 && live)
    p.lse[(size_t)b * rows_q + flat0 + m] = lse2 * 0.69314718055994530942f;
}

cudaError_t launch_reduce(const DecodeParams& p, cudaStream_t stream, bool pdl) {
  const DealShape d = deal_shape(p.B, p.Sq, p.H, p.num_clusters);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.reduce_d_tiles, d.Rw);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return p.partial_f16 ? cudaLaunchKernelEx(&cfg, reduce_kernel<true>, p)
                       : cudaLaunchKernelEx(&cfg, reduce_kernel<false>, p);
}

// ------------------------------------------------------------------ context-parallel merge
// One warp per row, 16 dims per lane: the ranks' pieces of a row (normalized O and
// natural-log LSE over disjoint key sets) combined with weights e^(lse_r - lse),
// lse = m + ln(sum_r e^(lse_r - m)); empty pieces (-inf) add nothing, and a row whose
// pieces are all empty gets O = 0, LSE = -inf.
template <bool F32>
__global__ void __launch_bounds__(256) merge_kernel(const void* o_parts, const float* lse_parts, int world,
                                                    long long rows, void* out, float* lse) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int r = 0; r < world; ++r) mx = fmaxf(mx, lse_parts[(size_t)r * rows + row]);
  float acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0.f;
  float l = -INFINITY;
  if (mx != -INFINITY) {
    float z = 0.f;
    for (int r = 0; r < world; ++r) z += expf(lse_parts[(size_t)r * rows + row] - mx);
    l = mx + logf(z);
    for (int r = 0; r < world; ++r) {
      const float lr = lse_parts[(size_t)r * rows + row];
      if (lr == -INFINITY) continue;
      const float wt = expf(lr - l);
      const size_t base = ((size_t)r * rows + row) * kDLatent + 16 * lane;
      if constexpr (F32) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(o_parts) + base);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v = src[q];
          acc[4 * q] += wt * v.x;
          acc[4 * q + 1] += wt * v.y;
          acc[4 * q + 2] += wt * v.z;
          acc[4 * q + 3] += wt * v.w;
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(o_parts) + base);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 v = src[q];
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[e]));
            acc[8 * q + 2 * e] += wt * f.x;
            acc[8 * q + 2 * e + 1] += wt * f.y;
          }
        }
      }
    }
  }
  const size_t obase = (size_t)row * kDLatent + 16 * lane;
  if constexpr (F32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + obase);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + obase);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t wv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[8 * q + 2 * e], acc[8 * q + 2 * e + 1]);
        wv[e] = *reinterpret_cast<uint32_t*>(&b2);
      }
      dst[q] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
  }
  if (lse && lane == 0) lse[row] = l;
}

cudaError_t launch_merge(const void* o_parts, const float* lse_parts, int world, long long rows, int out_f32,
                         void* out, float* lse, cudaStream_t stream) {
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  if (out_f32) merge_kernel<true><<<blocks, 256, 0, stream>>>(o_parts, lse_parts, world, rows, out, lse);
  else merge_kernel<false><<<blocks, 256, 0, stream>>>(o_parts, lse_parts, world, rows, out, lse);
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
// One block per (request, token): the decode kernel's visible key range of the row, as bits.
__global__ void debug_mask_kernel(const DecodeParams p, int max_k, uint32_t* bits) {
  const int row = blockIdx.x;  // b * Sq + t
  const int b = row / p.Sq, t = row % p.Sq;
  const int K = clamp_len(p, b, nullptr);
  int lo, hi;
  token_keys(p, b, t, K, global_len(p, b, K), lo, hi);
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

cudaError_t launch_debug_mask(const DecodeParams& p, int max_k, uint32_t* bits, cudaStream_t stream) {
  debug_mask_kernel<<<p.B * p.Sq, 128, 0, stream>>>(p, max_k, bits);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ debug gather
// One CTA per (64-key group, request): the decode kernel's page boxes bring the group's
// latent and rope blocks into swizzled shared memory, the slots past the request's length
// are zeroed as the decode kernel zeroes them, and the block is written back densely.
template <bool E4M3>
__global__ void __launch_bounds__(256) debug_gather_kernel(const __grid_constant__ KvMaps maps,
                                                           const int32_t* page_table, const int32_t* seq_lens,
                                                           int pt_stride, int num_pages, int page_size, int max_k,
                                                           uint8_t* out, uint32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int es = E4M3 ? 1 : 2;
  constexpr int nlat = latent_blocks<E4M3>();
  constexpr int rope_row = E4M3 ? 64 : 128;
  const int grp = blockIdx.x, b = blockIdx.y;
  const int K = min(max(seq_lens[b], 0), pt_stride * page_size);
  const int key0 = grp * kKeyGroup;
  if (key0 >= max_k) return;
  const int valid = min(max(K - key0, 0), kKeyGroup);
  const int nb = boxes_per_group(page_size), br = box_rows(page_size);
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (valid > 0) {
    if (threadIdx.x == 0) mbar_arrive_expect_tx(smem_addr(&bar), nlat * kBlockBytes + 64 * rope_row);
    __syncthreads();
    if (threadIdx.x < nb) {
      const int i = threadIdx.x;
      int pg, rw, shift = 0;
      bool bad;
      while ((1 << shift) < page_size) ++shift;
      box_page(page_table, pt_stride, num_pages, shift, b, key0 + i * br, K, pg, rw, bad);
      if (bad && err) atomicOr(err, kErrBadPage);
      for (int kb = 0; kb < nlat; ++kb)
        tma_load_3d(smem_addr(smem + kb * kBlockBytes + i * br * 128), &maps.ckv, kb * blk_elems<E4M3>(), rw, pg,
                    smem_addr(&bar));
      tma_load_3d(smem_addr(smem + nlat * kBlockBytes + i * br * rope_row), &maps.kpe, 0, rw, pg, smem_addr(&bar));
    }
    if (!mbar_wait_bounded(smem_addr(&bar), 0, kWaitTimeoutNs)) {
      if (threadIdx.x == 0 && err) atomicOr(err, kErrTimeout);
      return;
    }
    // slots past the request's length: zero, as the decode kernel does before P.V
    if (valid < kKeyGroup)
      for (int kb = 0; kb < nlat; ++kb) zero_block_rows(smem + kb * kBlockBytes, valid, threadIdx.x, blockDim.x);
    __syncthreads();
  }
  // write back: row j of this group -> out[b][key0 + j][0:576]
  const int row_bytes = kDQK * es;
  const int rows = min(kKeyGroup, max_k - key0);
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
                                int B, int pt_stride, int num_pages, int page_size, int max_k, void* out,
                                uint32_t* err, cudaStream_t stream) {
  dim3 grid((max_k + kKeyGroup - 1) / kKeyGroup, B);
  const int smem = 9 * kBlockBytes + 1024;
  cudaError_t e;
  if (e4m3) {
    e = cudaFuncSetAttribute(debug_gather_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    debug_gather_kernel<true><<<grid, 256, smem, stream>>>(maps, page_table, seq_lens, pt_stride, num_pages,
                                                            page_size, max_k, static_cast<uint8_t*>(out), err);
  } else {
    e = cudaFuncSetAttribute(debug_gather_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    debug_gather_kernel<false><<<grid, 256, smem, stream>>>(maps, page_table, seq_lens, pt_stride, num_pages,
                                                             page_size, max_k, static_cast<uint8_t*>(out), err);
  }
  return cudaGetLastError();
}

}  // namespace mla
