// Split-KV decode on CUDA cores: a plain correctness baseline for the schedule,
// workspace and reduction, before the tensor-core kernel takes over.
//
// Grid: 2 CTAs per cluster of the schedule; CTA (c, r) walks cluster c's pieces
// for the head groups g = r, r + 2, ... of 16 heads, with an online softmax over
// 32-key chunks.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "mla_common.cuh"
#include "mla_kernels.cuh"
#include "schedule.cuh"

namespace mla {

namespace v0 {
constexpr int kHeads = 16;
constexpr int kChunk = 32;
constexpr int kThreads = 256;
constexpr int kMaxSegs = 512;

template <bool E4M3>
__device__ __forceinline__ float ld(const void* base, size_t i) {
  if constexpr (E4M3) {
    __nv_fp8_e4m3 x;
    *reinterpret_cast<uint8_t*>(&x) = static_cast<const uint8_t*>(base)[i];
    return float(x);
  } else {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
  }
}

struct Smem {
  float q[kHeads][kDQK];
  float kv[kChunk][kDQK];
  float s[kHeads][kChunk];
  float m[kHeads], l[kHeads], corr[kHeads];
  Segment segs[kMaxSegs];
  int nseg;
  uint32_t err;
};

template <bool E4M3>
__global__ void __launch_bounds__(kThreads) split_kv_v0(const DecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int c = blockIdx.x >> 1;
  const int tid = threadIdx.x;
  if (tid == 0) S.err = 0;
  __syncthreads();
  {
    int32_t* scratch = reinterpret_cast<int32_t*>(&S.kv[0][0]);  // R + 33 ints fit (checked on the host)
    ScheduleView sv = build_schedule(p, scratch, &S.err);
    if (blockIdx.x == 0) write_row_table(p, sv);
    if (tid == 0) S.nseg = build_segments(p, sv, c, S.segs, kMaxSegs, &S.err);
    __syncthreads();
  }
  const float ln2 = 0.69314718055994530942f;
  const WsLayout L = ws_layout(p.B * p.Sq, p.num_clusters);
  const int hh = tid / 16;          // head within the group (PV phase)
  const int d0 = (tid % 16) * 32;   // 32 output dims per thread
  for (int hg = blockIdx.x & 1; hg * kHeads < p.H; hg += 2)
  for (int si = 0; si < S.nseg; ++si) {
    const int h_out = hg * kHeads + hh;
    const Segment seg = S.segs[si];
    const int b = seg.row / p.Sq, t = seg.row % p.Sq;
    int lo, hi;
    const int K = clamp_len(p, b, nullptr);
    visible_range(K, p.Sq, t, p.causal, p.window_left, lo, hi);
    const int ka = max(lo, seg.tile_begin * kTileN), kb = min(hi, seg.tile_end * kTileN);
    // Q for this head group, dequantized
    for (int i = tid; i < kHeads * kDQK; i += kThreads) {
      const int h = hg * kHeads + i / kDQK, d = i % kDQK;
      float v = 0.f;
      if (h < p.H) {
        const size_t row = (size_t)seg.row * p.H + h;
        v = d < kDLatent ? ld<E4M3>(p.q_latent, row * kDLatent + d) : ld<E4M3>(p.q_rope, row * kDRope + d - kDLatent);
        v *= p.q_descale;
      }
      S.q[i / kDQK][d] = v;
    }
    if (tid < kHeads) {
      S.m[tid] = -INFINITY;
      S.l[tid] = 0.f;
    }
    float o[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = 0.f;
    __syncthreads();
    for (int k0 = ka; k0 < kb; k0 += kChunk) {
      for (int i = tid; i < kChunk * kDQK; i += kThreads) {
        const int j = i / kDQK, d = i % kDQK, key = k0 + j;
        float v = 0.f;
        if (key < kb) {
          const int pg = p.page_table[(size_t)b * p.pt_stride + key / kPageSize];
          if ((unsigned)pg < (unsigned)p.num_pages) {
            const size_t slot = (size_t)pg * kPageSize + key % kPageSize;
            v = d < kDLatent ? ld<E4M3>(p.ckv, slot * kDLatent + d) * p.ckv_descale
                             : ld<E4M3>(p.kpe, slot * kDRope + d - kDLatent) * p.kpe_descale;
          } else if (d == 0) {
            atomicOr(&S.err, kErrBadPage);
          }
        }
        S.kv[j][d] = v;
      }
      __syncthreads();
      for (int i = tid; i < kHeads * kChunk; i += kThreads) {
        const int h = i / kChunk, j = i % kChunk;
        float acc = 0.f;
        for (int d = 0; d < kDQK; ++d) acc += S.q[h][d] * S.kv[j][d];
        S.s[h][j] = (k0 + j < kb) ? acc * p.scale : -INFINITY;
      }
      __syncthreads();
      if (tid < kHeads) {
        float mx = S.m[tid];
        for (int j = 0; j < kChunk; ++j) mx = fmaxf(mx, S.s[tid][j]);
        const float corr = S.m[tid] == -INFINITY ? 0.f : __expf(S.m[tid] - mx);
        float sum = 0.f;
        for (int j = 0; j < kChunk; ++j) {
          const float e = S.s[tid][j] == -INFINITY ? 0.f : __expf(S.s[tid][j] - mx);
          S.s[tid][j] = e;
          sum += e;
        }
        S.l[tid] = S.l[tid] * corr + sum;
        S.m[tid] = mx;
        S.corr[tid] = corr;
      }
      __syncthreads();
      const float cf = S.corr[hh];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float acc = o[i] * cf;
        for (int j = 0; j < kChunk; ++j) acc += S.s[hh][j] * S.kv[j][d0 + i];
        o[i] = acc;
      }
      __syncthreads();
    }
    // finish the piece
    if (h_out < p.H) {
      const float l = S.l[hh], m = S.m[hh];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse_e = l > 0.f ? m + __logf(l) : -INFINITY;
      if (seg.whole) {
        const size_t orow = (size_t)seg.row * p.H + h_out;
        if (p.out_f32) {
          float* dst = static_cast<float*>(p.out) + orow * kDLatent + d0;
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[i] = o[i] * inv;
        } else {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + orow * kDLatent + d0;
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[i] = __float2bfloat16_rn(o[i] * inv);
        }
        if (p.lse && (tid % 16) == 0) p.lse[orow] = lse_e;
      } else {
        const size_t slot = (size_t)seg.row + c;
        float* dst = reinterpret_cast<float*>(p.ws + L.partial_o) + (slot * kHeadsPad + h_out) * kDLatent + d0;
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[i] = o[i] * inv;
        if ((tid % 16) == 0)
          reinterpret_cast<float*>(p.ws + L.partial_lse)[slot * kHeadsPad + h_out] = lse_e / ln2;
      }
    }
    __syncthreads();
  }
  __syncthreads();
  if (tid == 0) reinterpret_cast<uint32_t*>(p.ws + L.cta_status)[2 * c + (blockIdx.x & 1)] = S.err;
}
}  // namespace v0

cudaError_t launch_split_kv_v0(const DecodeParams& p, cudaStream_t stream) {
  const int smem = (int)sizeof(v0::Smem);
  dim3 grid(2 * p.num_clusters);
  cudaError_t e;
  if (p.qkv_e4m3) {
    e = cudaFuncSetAttribute(v0::split_kv_v0<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    v0::split_kv_v0<true><<<grid, v0::kThreads, smem, stream>>>(p);
  } else {
    e = cudaFuncSetAttribute(v0::split_kv_v0<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    v0::split_kv_v0<false><<<grid, v0::kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace mla
