// Split-KV paged MLA decode on the tensor cores (tcgen05, 2-CTA clusters).
//
// One cluster = two CTAs on two SMs working on the same (request, token) row:
// CTA r holds heads [64r, 64r + 64) of the 128-row M tile and the keys of its
// two pages of every 256-key tile.  The leader CTA issues cta_group::2 MMAs:
//   S[128 heads x 256 keys]  = Q[128 x 576] . [c | kpe]^T      (QK^T, K = 576)
//   O[128 heads x 512 dims] += P[128 x 256] . c[256 x 512]      (V is c itself)
// with S (two stages) and O in tensor memory.  Roles (12 warps per CTA):
//   warps 0-3  softmax: online max / exp2 / row sums, P (bf16 or e4m3) into
//              tensor memory over the S it came from (below)
//   warps 4-7  correction: rescale O when the row max moves, final epilogue
//   warp 8     MMA issue (leader CTA, one thread) and TMEM allocation: QK^T(t + 1)
//              then P.V(t) over all of the cluster's tiles, across pieces too
//   warp 9     TMA loads of Q (once per piece of work)
//   warps 10-11 TMA loads of K blocks and V pages into one ring of 16 KB slots,
//              in exactly the order the MMAs consume them (even fills by warp 10,
//              odd fills by warp 11), page ids read a tile ahead
// P.V takes P as an A operand in tensor memory, where lane half h of a CTA reads
// its rows from its own lanes: S leaves keys [0, 128) of a row in the lower half
// and keys [128, 256) in the upper half, so each softmax thread writes its own
// keys of P over S columns it has already read, the two halves swap theirs
// through a small shared buffer, and both halves end with the whole row.  P thus
// lives in the S stage of its tile: two tiles' P in flight, no shared-memory P
// buffer held until P.V completes, and no shared-memory reads of A in P.V.
// A work row is an M tile of 128 (token, head) rows of one request (consecutive
// tokens pack into it when H < 128); every M row has its own visible key range
// (its token's causal, window or local bound, on this rank's keys under decode
// context parallelism).  The split follows the batch schedule (schedule.cuh): a
// work row cut into several pieces writes each to a workspace slot (fp32, or fp16
// scaled by a power of two per row and half of the dims) that the reduction kernel
// combines, or that the last of its pieces combines here (combine_in_kernel); a work
// row in one piece is written to the output directly.  Every mbarrier wait is bounded: on timeout the
// kernel records kErrTimeout, tells its peer CTA, unwinds its roles, and before
// freeing tensor memory proves with bounded waits that every copy it issued has
// landed and every MMA it issued has completed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "mla_common.cuh"
#include "mla_kernels.cuh"
#include "ptx.cuh"
#include "schedule.cuh"
#include "tma_pages.cuh"

namespace mla {
namespace tc {


constexpr int kThreads = 384;
// Rescale O only when a row's max grows by more than 2^8: P stays <= 256
// (exact enough in bf16, below the e4m3 maximum of 448) and most tiles skip it.
constexpr float kSkipCorrectionLog2 = 8.0f;
// bounded waits of the abort teardown (anything legitimate lands within microseconds)
constexpr uint64_t kDrainTimeoutNs = 50000000ull;
// work rows a CTA combines at its end: a cluster's share cuts at most the work rows at its
// two ends, so two (more are combined at once by the correction warps)
constexpr int kCombList = 4;

template <bool E4M3>
struct Cfg {
  static constexpr int kBlk = E4M3 ? 128 : 64;  // elements per 128-byte column block
  static constexpr int kNLat = kDLatent / kBlk;  // latent column blocks: 8 or 4
  static constexpr int kNKb = kNLat + 1;         // QK^T contraction blocks (latent + rope)
  static constexpr int kRopeSteps = E4M3 ? 2 : 4;
  static constexpr int kRopeRow = E4M3 ? 64 : 128;  // bytes of a key's rope row in shared memory
  static constexpr uint32_t kQBytes = kNLat * 8192 + (E4M3 ? 4096 : 8192);
  // P of one row-half of 128 keys in 32-bit words.  The halves swap P through an
  // exchange buffer of [row][half] regions: e4m3 in one round (128 B a region), bf16 in
  // two rounds of 64 keys (128 B a region), which halves its size.
  static constexpr int kPWords = E4M3 ? 32 : 64;
  static constexpr int kXRegion = 128;
  static constexpr int kXBytes = 64 * 2 * kXRegion;
  static constexpr int kPCols = E4M3 ? 64 : 128;  // TMEM columns of a full P row
  // One ring of 16 KB slots holds, in consumption order, the K blocks of a tile (one
  // slot each: this CTA's 128 keys x 128 B) and its V key groups (this CTA's columns of
  // 64 keys: two slots in bf16, one per output chunk; one slot in e4m3).
  static constexpr int kSlot = 16384;
  static constexpr int kNS = E4M3 ? 10 : 8;  // even: each loader warp owns every other slot
  static_assert(kNS % 2 == 0, "the two loader warps own alternate slots");
  static constexpr int kVItems = E4M3 ? 1 : 2;    // ring slots per V key group
  static constexpr int kPvSteps = E4M3 ? 2 : 4;  // MMAs per key group and output chunk (32 or 16 keys each)
  static constexpr uint32_t kIdescQK = instr_desc(E4M3 ? 0u : 1u, 128, 256, 0, 0);
  static constexpr uint32_t kIdescPV = instr_desc(E4M3 ? 0u : 1u, 128, 256, 0, 1);
  static constexpr int kOffQ = 0;
  static constexpr int kOffX = kOffQ + kNKb * 8192;
  static constexpr int kOffRing = kOffX + kXBytes;
  static constexpr int kOffSeg = kOffRing + kNS * kSlot;
  static constexpr int kOffMisc = kOffSeg + kSmemSegs * (int)sizeof(Segment);
};

struct Misc {
  uint64_t q_full, q_empty;
  uint64_t full[10], empty[10];  // ring slots
  uint64_t s_full[2];
  // the per-tile barriers come in pairs indexed by tile parity: the softmax may run one
  // tile ahead of the correction and of the P.V, never two
  uint64_t pv_ready[2];   // leader: one arrival per CTA, P written and O corrected for the next P.V
  uint64_t pv_local[2];   // this CTA's 4 softmax + 4 correction warps, forwarded to the leader's pv_ready
  // leader: the peer zeroed the tail of a request's last key group (one arrival a slot); two,
  // alternating by tail group, so the peer (at most a ring ahead of the MMA, and tail groups
  // a tile's fills apart) can never complete a phase the MMA has not yet waited for
  uint64_t tail_ready[2];
  uint64_t o_done[2];     // P.V of a tile complete
  uint64_t cor_ready[2];  // softmax -> correction: the tile's rescale factor is posted
  uint64_t tail_bar[2], xchg_bar;  // tail_bar: one per loader warp
  uint64_t drain;                  // abort teardown: the MMA thread's final commit
  uint64_t comb_in, comb_out;      // fused combine: the 4 correction warps' partials written; the verdict posted
  float xchg[2][128];             // per-tile row-max exchange between the two halves of a row
  float xsum[128];                // final row-sum exchange
  float corr[2][128];             // per-tile rescale factor, softmax -> correction
  float fin_l[2][128], fin_m[2][128];  // final row statistics, double-buffered by segment
  // what this CTA issued, for the abort teardown: fills per ring slot, the bytes the
  // slot's latest fill brings to the leader's barrier (0: a tail fill, which lands on the
  // loader's own tail barrier), tail fills issued and waited per loader warp, Q loads
  uint32_t nfill[10], fbytes[10];
  uint32_t ntail[2], ntail_done[2];
  // page sizes below 64: each loader warp's page ids of the boxes of three tiles (the one
  // whose V is loaded, the one whose K is loaded, the next), written by its lanes
  int32_t boxes[2][3][32];
  uint32_t nq;
  // in-kernel combine: the verdict of this CTA's latest arrival (1: combine the row now),
  // and the work rows it arrived last on, combined at the end (row, first slot, pieces)
  uint32_t last_piece;
  uint32_t ncl;
  int4 comb_list[kCombList];
  uint32_t tmem_base;
  uint32_t err;
  uint32_t abort;
  int nseg;
};

template <bool E4M3>
constexpr int smem_bytes() {
  return Cfg<E4M3>::kOffMisc + (int)sizeof(Misc) + 1024;
}
static_assert(smem_bytes<false>() <= 232448, "bf16 kernel exceeds shared memory");
static_assert(smem_bytes<true>() <= 232448, "e4m3 kernel exceeds shared memory");

// record a timeout and tell both CTAs of the pair to unwind
__device__ __noinline__ void abort_pair(Misc& M) {
  atomicOr(&M.err, kErrTimeout);
  *reinterpret_cast<volatile uint32_t*>(&M.abort) = 1u;
  st_shared_cluster(map_to_rank(smem_addr(&M.abort), cluster_ctarank() ^ 1u), 1u);
}

// bounded wait that also gives up when this CTA or its peer already aborted (the spin
// is out of line: one copy for every wait site keeps the kernel compact)
__device__ __noinline__ bool kwait_spin(Misc& M, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*reinterpret_cast<volatile uint32_t*>(&M.abort)) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
        abort_pair(M);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool kwait(Misc& M, uint32_t bar, uint32_t parity) {
  return mbar_try_wait(bar, parity) || kwait_spin(M, bar, parity);
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// 2^x with the hardware approximation (relative error ~2^-22; denormal results flush to 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 probabilities to bf16 pairs (16 words) or e4m3 quadruples (8 words), key order
template <bool E4M3>
__device__ __forceinline__ void pack_p(const float (&p)[32], uint32_t (&w)[E4M3 ? 8 : 16]) {
  if constexpr (!E4M3) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      __nv_bfloat162 h2 = __floats2bfloat162_rn(p[2 * e], p[2 * e + 1]);
      w[e] = *reinterpret_cast<uint32_t*>(&h2);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(p[4 * e], p[4 * e + 1]), __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(p[4 * e + 2], p[4 * e + 3]), __NV_SATFINITE, __NV_E4M3);
      w[e] = lo | (hi << 16);
    }
  }
}

// Order in which a thread turns its four 32-key chunks of S into P.  P chunk c of
// half h lands in columns (kPCols / 2) h + (kPCols / 8) c; each order writes only
// columns of S chunks the thread has already read (S chunk c: columns 32 c .. +32).
template <bool E4M3>
__device__ __forceinline__ int chunk_order(int half, int k) {
  if (half == 0) return k;
  return E4M3 ? (k < 2 ? 1 - k : k) : 3 - k;
}

// 8 consecutive floats times `scale` to 16 bytes of bf16 or fp16
__device__ __forceinline__ uint4 pack8_bf16(const uint32_t* r, float scale) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(u2f(r[2 * e]) * scale, u2f(r[2 * e + 1]) * scale);
    w[e] = *reinterpret_cast<uint32_t*>(&h2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 pack8_f16(const uint32_t* r, float scale) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __half2 h2 = __floats2half2_rn(u2f(r[2 * e]) * scale, u2f(r[2 * e + 1]) * scale);
    w[e] = *reinterpret_cast<uint32_t*>(&h2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}


// Abort teardown (a bounded wait gave up in this CTA or its peer): before the memory goes
// away, prove with bounded waits that every copy the pair issued has landed and every MMA
// has completed.  Of each ring slot only the latest fill can be outstanding (a fill waits
// for the MMA to consume the one before), and its phase completes on the leader's barrier
// once the leader armed it and both CTAs' bytes landed: the leader arms a fill only the
// peer issued, and completes the bytes of a fill only the leader issued.  Tail fills land
// on each loader's own barrier.  All threads of the CTA call it (it ends in a barrier).
template <bool E4M3>
__device__ __noinline__ void drain_after_abort(Misc& M, uint32_t rank, int warp, int lane, int tid) {
  using C = Cfg<E4M3>;
  if (rank == 0 && tid == 0) {
    const uint32_t peer = 1u;
    for (int sl = 0; sl < C::kNS; ++sl) {
      const uint32_t a = M.nfill[sl], bcnt = ld_shared_cluster(map_to_rank(smem_addr(&M.nfill[sl]), peer));
      const uint32_t nf = a > bcnt ? a : bcnt;
      if (nf == 0) continue;
      const uint32_t f = nf - 1;
      const uint32_t bytes = a == nf ? M.fbytes[sl] : ld_shared_cluster(map_to_rank(smem_addr(&M.fbytes[sl]), peer));
      const uint32_t bar = smem_addr(&M.full[sl]);
      if (bytes == 0 || mbar_try_wait(bar, f & 1)) continue;
      if (a < nf) mbar_arrive_expect_tx(bar, bytes);
      if (bcnt < nf) mbar_complete_tx(bar, bytes);
      mbar_wait_bounded(bar, f & 1, kDrainTimeoutNs);
    }
    const uint32_t a = M.nq, bcnt = ld_shared_cluster(map_to_rank(smem_addr(&M.nq), peer));
    const uint32_t nq = a > bcnt ? a : bcnt;
    if (nq > 0) {
      const uint32_t bar = smem_addr(&M.q_full);
      if (!mbar_try_wait(bar, (nq - 1) & 1)) {
        if (a < nq) mbar_arrive_expect_tx(bar, C::kQBytes);
        if (bcnt < nq) mbar_complete_tx(bar, C::kQBytes);
        mbar_wait_bounded(bar, (nq - 1) & 1, kDrainTimeoutNs);
      }
    }
  }
  if (warp >= 10 && lane == 0) {
    const int own = warp - 10;
    if (M.ntail[own] > M.ntail_done[own])
      mbar_wait_bounded(smem_addr(&M.tail_bar[own]), M.ntail_done[own] & 1, kDrainTimeoutNs);
  }
  // the MMA thread's final commit arrives on both CTAs' drain barrier once all its MMAs
  // (and their shared-memory reads) are complete
  if (warp == 8 && lane == 0 && rank == 0) mma_commit_pair(smem_addr(&M.drain), 0x3);
  if (warp == 8 && lane == 0) mbar_wait_bounded(smem_addr(&M.drain), 0, kDrainTimeoutNs);
  __syncthreads();
}

// The request's last key group, when its length is not a multiple of 64 (loader warp
// `own`): each CTA landed the group locally on its tail barrier; wait for it, zero the
// slots' rows past the length (any bits there, NaN included, must not reach P.V), then
// the leader completes its slots' phases and the peer reports on the leader's
// tail_ready[tg & 1], tg the CTA's tail groups so far (the MMA waits for both on this
// group).  Out of line: once per piece.
template <bool E4M3>
__device__ __noinline__ bool tail_group(Misc& M, uint8_t* smem, int own, uint32_t rank, int lane, uint32_t tph,
                                        uint32_t tg, int slot0, int slot1, bool mine0, bool mine1, int tail_rows) {
  using C = Cfg<E4M3>;
  if (!kwait(M, smem_addr(&M.tail_bar[own]), tph & 1)) return false;
  if (lane == 0) M.ntail_done[own] += 1;
#pragma unroll
  for (int it = 0; it < C::kVItems; ++it) {
    const bool mine = it == 0 ? mine0 : mine1;
    const int slot = it == 0 ? slot0 : slot1;
    if (mine)
      for (int u = 0; u < 2; ++u) zero_block_rows(smem + C::kOffRing + slot * C::kSlot + u * 8192, tail_rows, lane, 32);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
#pragma unroll
    for (int it = 0; it < C::kVItems; ++it) {
      const bool mine = it == 0 ? mine0 : mine1;
      const int slot = it == 0 ? slot0 : slot1;
      if (!mine) continue;
      if (rank == 0)
        mbar_arrive(smem_addr(&M.full[slot]));
      else
        mbar_arrive_cluster(map_to_rank(smem_addr(&M.tail_ready[tg & 1]), 0));
    }
  }
  __syncwarp();
  return true;
}

// In-kernel combine, arrival (the correction warps, 128 threads, once the piece's
// partial is written): count this CTA's piece of the work row; the last of the row's
// pieces to arrive combines them.  The counter holds this call's epoch in its high half,
// so a word left by an earlier call counts as zero.  The last arrival queues the row for
// the end of the kernel (every role idle then, so more threads and loads in flight), or
// asks for the combine now when the queue is full.  The two syncs among the correction
// warps are mbarriers waited with the bounded waits (phase parity `ph`).  Returns 1 to
// combine now, 0 otherwise, -1 when a wait gave up.
__device__ __noinline__ int arrive_piece(Misc& M, const DecodeParams& p, unsigned long long* counter, uint32_t ph,
                                         int w, int first_slot, int np, int L) {
  __threadfence();  // this thread's partial stores before the arrival
  __syncwarp();
  if ((L & 31) == 0) mbar_arrive(smem_addr(&M.comb_in));
  if (!kwait(M, smem_addr(&M.comb_in), ph)) return -1;
  if (L == 0) {
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(counter), seen, want;
    do {
      seen = cur;
      want = (seen >> 32) == p.epoch ? seen + 1 : ((unsigned long long)p.epoch << 32) | 1ull;
      cur = atomicCAS(counter, seen, want);
    } while (cur != seen);
    uint32_t now = 0;
    if ((uint32_t)(want & 0xFFFFFFFFull) == (uint32_t)np) {
      const uint32_t k = M.ncl++;
      if (k < (uint32_t)kCombList) M.comb_list[k] = make_int4(w, first_slot, np, 0);
      else now = 1;
    }
    *reinterpret_cast<volatile uint32_t*>(&M.last_piece) = now;
    mbar_arrive(smem_addr(&M.comb_out));
  }
  if (!kwait(M, smem_addr(&M.comb_out), ph)) return -1;
  return (int)*reinterpret_cast<volatile uint32_t*>(&M.last_piece);
}

// In-kernel combine of work row w for this CTA's 64 M rows, as the reduction kernel does:
// lse = log2 of the summed 2^(lse_i), out = output_scale * sum_i 2^(lse_i - lse) O_i over
// its np slots (first_slot, wb apart); an empty piece (lse_i = -inf) adds nothing.  nthr
// threads (a multiple of 64), t this one: M row 64 rank + (t & 63), 32-column blocks
// t / 64 + k nthr / 64; two pieces' loads are issued before either is applied.
__device__ __noinline__ void combine_row(const DecodeParams& p, const uint8_t* part_o, const float* part_lse,
                                         const float* part_scale, size_t slot_bytes, int w, int first_slot, int np,
                                         int wb, int Qb, uint32_t rank, int t, int nthr) {
  __threadfence();  // the other pieces' stores, published before their arrivals
  const int rows_q = p.Sq * p.H;
  const int m = 64 * (int)rank + (t & 63);
  const int flat = kTileM * (w % Qb) + m;
  if (flat >= rows_q) return;
  const float* plse = part_lse + m;
  float mx = -INFINITY;
  for (int i = 0; i < np; ++i) mx = fmaxf(mx, __ldcg(plse + (size_t)(first_slot + i * wb) * kTileM));
  const float m0 = mx == -INFINITY ? 0.f : mx;
  float sum = 0.f;
  for (int i = 0; i < np; ++i) sum += exp2f(__ldcg(plse + (size_t)(first_slot + i * wb) * kTileM) - m0);
  const float lse2 = sum > 0.f ? m0 + log2f(sum) : -INFINITY;
  const size_t orow = (size_t)(w / Qb) * rows_q + flat;
  if (t < 64 && p.lse) p.lse[orow] = lse2 * 0.69314718055994530942f;
#pragma unroll 1
  for (int cb = t >> 6; cb < kDLatent / 32; cb += nthr >> 6) {
    const int d0 = 32 * cb;
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll 1
    for (int i0 = 0; i0 < np; i0 += 2) {
      float x[2][32];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint8_t* so = part_o + (size_t)(first_slot + min(i0 + u, np - 1) * wb) * slot_bytes;
        if (p.partial_f16) {
          const uint4* src = reinterpret_cast<const uint4*>(so) + m;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldcg(src + (size_t)(d0 / 8 + q) * kTileM);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[e]));
              x[u][8 * q + 2 * e] = f.x;
              x[u][8 * q + 2 * e + 1] = f.y;
            }
          }
        } else {
          const float4* src = reinterpret_cast<const float4*>(so) + m;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 v = __ldcg(src + (size_t)(d0 / 4 + q) * kTileM);
            x[u][4 * q] = v.x;
            x[u][4 * q + 1] = v.y;
            x[u][4 * q + 2] = v.z;
            x[u][4 * q + 3] = v.w;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const size_t sl = (size_t)(first_slot + (i0 + u) * wb);
        const float li = i0 + u < np ? __ldcg(plse + sl * kTileM) : -INFINITY;
        if (!(sum > 0.f) || li == -INFINITY) continue;
        // fp16 partials: undo the half's power-of-two scale (d0's half of its 256-dim chunk)
        const float sc = p.partial_f16 ? __ldcg(part_scale + (sl * 2 + ((d0 >> 7) & 1)) * kTileM + m) : 0.f;
        const float wt = exp2f(li - lse2 + sc) * p.ckv_descale;
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] += wt * x[u][e];
      }
    }
    if (p.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kDLatent + d0);
#pragma unroll
      for (int q = 0; q < 8; ++q) dst[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    } else {
      uint32_t r[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(acc[e]);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow * kDLatent + d0);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = pack8_bf16(r + 8 * q, 1.f);
    }
  }
}

// Fused combine: the work rows with no visible key in any of their M rows have no piece;
// this CTA's share of them (every gridDim.x-th) gets O = 0 and LSE = -inf (the correction
// warps, 128 threads, one M row each).  Out of line: once per kernel.
__device__ __noinline__ void write_empty_rows(const DecodeParams& p, const DealShape& DS, int L) {
  const int rows_q = p.Sq * p.H;
  for (int w = blockIdx.x; w < DS.Rw; w += gridDim.x) {
    const int b = w / DS.Qb, i = w % DS.Qb;
    const int K = clamp_len(p, b, nullptr);
    int tlo, n;
    work_span(p, b, i, K, global_len(p, b, K), tlo, n);
    if (n > 0) continue;
    const int flat = kTileM * i + L;
    if (flat >= rows_q) continue;
    const size_t orow = (size_t)b * rows_q + flat;
    if (p.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kDLatent);
      for (int q = 0; q < kDLatent / 4; ++q) dst[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow * kDLatent);
      for (int q = 0; q < kDLatent / 8; ++q) dst[q] = make_uint4(0, 0, 0, 0);
    }
    if (p.lse) p.lse[orow] = -INFINITY;
  }
}

// Epilogue of one piece for this thread's M row (correction warps, once per piece): a
// work row in one piece goes to the output (O / l times the value scale, natural-log
// LSE); a piece of a longer row goes to its slot (O / l in the stored codes' units and
// the base-2 LSE, combined and scaled by the reduction kernel).  A row with no visible
// key in the piece gets O = 0 and LSE = -inf.  TMEM columns [128 c', +128) of this lane
// hold D columns 256 c' + 128 half + [0, 128).  Out of line: it runs once per piece.
__device__ __noinline__ void piece_epilogue(const DecodeParams& p, uint8_t* slot_o, float* slot_lse, float* slot_scale,
                                            uint32_t obase, int half, int m, int b, int flat, bool live, bool direct,
                                            float lrow, float mrow) {
  const bool empty = !(lrow > 0.f);
  const int rows_q = p.Sq * p.H;
  if (direct) {
    // P.V ran on the stored codes of c: the value scale (the key cache's descale) applies here
    const float inv = empty ? 0.f : p.ckv_descale / lrow;
    const size_t orow = (size_t)b * rows_q + flat;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t r[32];
      tmem_ld32(obase + c * 32, r);
      tmem_ld_wait();
      const int d0 = 256 * (c >> 2) + 128 * half + 32 * (c & 3);
      if (!live) continue;
      if (p.out_f32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kDLatent + d0);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(u2f(r[4 * q]) * inv, u2f(r[4 * q + 1]) * inv, u2f(r[4 * q + 2]) * inv,
                               u2f(r[4 * q + 3]) * inv);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow * kDLatent + d0);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = pack8_bf16(r + 8 * q, inv);
      }
    }
    if (live && half == 0 && p.lse) p.lse[orow] = empty ? -INFINITY : (mrow + log2f(lrow)) * 0.69314718055994530942f;
  } else {
    float inv = empty ? 0.f : 1.f / lrow;
    uint8_t* so = slot_o;
    if (p.partial_f16) {
      // this thread's power-of-two scale: the largest |O / l| of its 256 dims to [2^14, 2^15)
      float amax = 0.f;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t r[32];
        tmem_ld32(obase + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(u2f(r[e])));
      }
      amax *= inv;
      int ex = 0;
      if (amax > 0.f && amax <= 3.0e38f) frexpf(amax, &ex);  // amax = f 2^ex, f in [0.5, 1)
      const int sh = amax > 0.f && amax <= 3.0e38f ? ex - 15 : 0;
      inv = ldexpf(inv, -sh);
      if (live) slot_scale[half * kTileM + m] = (float)sh;
    }
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t r[32];
      tmem_ld32(obase + c * 32, r);
      tmem_ld_wait();
      const int d0 = 256 * (c >> 2) + 128 * half + 32 * (c & 3);
      if (!live) continue;
      if (p.partial_f16) {
        // [dim / 8][row][dim % 8] halves: a warp's 16-byte stores are 512 contiguous bytes
        uint4* po = reinterpret_cast<uint4*>(so) + m;
#pragma unroll
        for (int q = 0; q < 4; ++q) __stcg(po + (size_t)(d0 / 8 + q) * kTileM, pack8_f16(r + 8 * q, inv));
      } else {
        float4* po = reinterpret_cast<float4*>(so) + m;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          __stcg(po + (size_t)(d0 / 4 + q) * kTileM, make_float4(u2f(r[4 * q]) * inv, u2f(r[4 * q + 1]) * inv,
                                                                u2f(r[4 * q + 2]) * inv, u2f(r[4 * q + 3]) * inv));
      }
    }
    if (live && half == 0) slot_lse[m] = empty ? -INFINITY : mrow + log2f(lrow);
  }
}

// E4M3: e4m3 inputs (else bf16).  ONE_BOX: page_size >= 64, one page box per 64-key group
// (else 64 / page_size boxes, looked up through the loader's shared table).
template <bool E4M3, bool ONE_BOX>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    split_kv_tc(const __grid_constant__ DecodeParams p, const __grid_constant__ KvMaps maps) {
  using C = Cfg<E4M3>;
  constexpr int KIND = E4M3 ? 1 : 0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& M = *reinterpret_cast<Misc*>(smem + C::kOffMisc);
  Segment* segs = reinterpret_cast<Segment*>(smem + C::kOffSeg);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + C::kOffQ, sRing = sbase + C::kOffRing;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = blockIdx.x >> 1;
  const WsLayout WL = ws_layout(p.B, p.Sq, p.H, p.num_clusters, p.partial_f16);
  const DealShape DS = deal_shape(p.B, p.Sq, p.H, p.num_clusters);
  const int rows_q = p.Sq * p.H;  // (token, head) rows of a request
  Segment* overflow = reinterpret_cast<Segment*>(p.ws + WL.segs) + (size_t)blockIdx.x * WL.seg_cap;

  if (tid == 0) {
    M.err = 0;
    M.abort = 0;
    for (int i = 0; i < 10; ++i) M.nfill[i] = M.fbytes[i] = 0;
    M.ntail[0] = M.ntail[1] = M.ntail_done[0] = M.ntail_done[1] = 0;
    M.nq = 0;
    M.ncl = 0;
    mbar_init(smem_addr(&M.q_full), 1);  // armed by the leader with both CTAs' bytes
    mbar_init(smem_addr(&M.q_empty), 1);
    for (int i = 0; i < C::kNS; ++i) {
      mbar_init(smem_addr(&M.full[i]), 1);   // armed by the leader with both CTAs' bytes
      mbar_init(smem_addr(&M.empty[i]), 1);  // the leader's MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&M.s_full[i]), 1);
      mbar_init(smem_addr(&M.pv_ready[i]), 2);
      mbar_init(smem_addr(&M.pv_local[i]), 8);
      mbar_init(smem_addr(&M.o_done[i]), 1);
      mbar_init(smem_addr(&M.cor_ready[i]), 4);
    }
    mbar_init(smem_addr(&M.tail_ready[0]), C::kVItems);
    mbar_init(smem_addr(&M.tail_ready[1]), C::kVItems);
    mbar_init(smem_addr(&M.tail_bar[0]), 1);
    mbar_init(smem_addr(&M.tail_bar[1]), 1);
    mbar_init(smem_addr(&M.xchg_bar), 4);
    mbar_init(smem_addr(&M.drain), 1);
    mbar_init(smem_addr(&M.comb_in), 4);
    mbar_init(smem_addr(&M.comb_out), 1);
    fence_mbar_init();
  }
  // what needs no schedule goes first: the barriers above, tensor memory, the descriptors
  if (warp == 8) {
    tmem_alloc_pair(smem_addr(&M.tmem_base), 512);
    tmem_relinquish_pair();
  }
  if (warp == 9 && lane == 0) {
    tma_prefetch_desc(&maps.ckv);
    tma_prefetch_desc(&maps.kpe);
    tma_prefetch_desc(&maps.q_latent);
    tma_prefetch_desc(&maps.q_rope);
  }
  __syncthreads();
  {
    // the batch schedule, in the ring memory before any tile lands there
    int32_t* scratch = reinterpret_cast<int32_t*>(smem + C::kOffRing);
    Sched sc = build_schedule(p, scratch, &M.err);
    // this CTA's pieces first (every role waits for them), then the row table's share
    // (measured: the other order held the segments back by 1.6 us)
    if (warp == 0) {
      const int nseg = build_segments(p, sc, cl, segs, overflow);
      if (lane == 0) M.nseg = nseg;
    }
    if (blockIdx.x * blockDim.x < DS.Rw) write_row_table(p, sc);  // the CTAs that own rows of the table
  }
  __syncthreads();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();

  const uint32_t tmem = M.tmem_base;
  const int nseg = M.nseg;
  auto lead = [&](uint64_t& bar) { return map_to_rank(smem_addr(&bar), 0); };
  auto seg_at = [&](int s) -> Segment { return s < kSmemSegs ? segs[s] : overflow[s - kSmemSegs]; };

  if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int L = tid, row = L & 63, half = L >> 6;
    const uint32_t lanebase = static_cast<uint32_t>(warp * 32) << 16;
    const float cl2 = p.score_scale_log2;
    int j = 0;  // global tile counter of this cluster
    uint32_t xph = 0;
    bool ok = true;
    for (int s = 0; s < nseg && ok; ++s) {
      const Segment sg = seg_at(s);
      // this thread's M row: its token's visible keys (none for a padding row)
      const int b = sg.row() / DS.Qb, flat = kTileM * (sg.row() % DS.Qb) + 64 * (int)rank + row;
      int key_lo = 0, key_hi = 0;
      if (flat < rows_q) token_keys(p, b, flat / p.H, sg.K, global_len(p, b, sg.K), key_lo, key_hi);
      const int n = sg.tile_end - sg.tile_begin;
      float m_ref = -INFINITY, l = 0.f;
      for (int i = 0; i < n; ++i, ++j) {
        const int st = j & 1;
        if (!(ok = kwait(M, smem_addr(&M.s_full[st]), (j >> 1) & 1))) break;
        tc_fence_after();
        const int key0 = (sg.tile_begin + i) * kTileN + 128 * half;
        const bool full = key0 >= key_lo && key0 + 128 <= key_hi;
        const uint32_t sbase_t = tmem + lanebase + st * 128;
        // visible keys of this thread's 128: [vlo, vhi) relative to key0 (all of them on most
        // tiles); the mask is one unsigned compare, so the loops stay branch-free
        const int vlo = full ? 0 : min(max(key_lo - key0, 0), 128);
        const int vhi = full ? 128 : min(max(key_hi - key0, 0), 128);
        const uint32_t vspan = static_cast<uint32_t>(max(vhi - vlo, 0));
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t r[32];
          tmem_ld32(sbase_t + ch * 32, r);
          tmem_ld_wait();
          if (full) {
#pragma unroll
            for (int e = 0; e < 32; ++e) mq[e & 3] = fmaxf(mq[e & 3], u2f(r[e]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const bool vis = static_cast<uint32_t>(ch * 32 + e - vlo) < vspan;
              mq[e & 3] = fmaxf(mq[e & 3], vis ? u2f(r[e]) : -INFINITY);
            }
          }
        }
        const float mloc = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        M.xchg[j & 1][L] = mloc;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&M.xchg_bar));
        if (!(ok = kwait(M, smem_addr(&M.xchg_bar), xph & 1))) break;
        ++xph;
        // -inf when no key of this tile is visible to the row (a packed row of an earlier
        // token, a window edge): its P is then all zero and its statistics stay empty
        const float mt = fmaxf(mloc, M.xchg[j & 1][L ^ 64]);
        const float mts = mt * cl2;
        float m_new, fac;
        if (i == 0) {
          m_new = mts;
          fac = 0.f;
        } else if (mts > m_ref + kSkipCorrectionLog2) {
          m_new = mts;
          fac = ex2(m_ref - m_new);
        } else {
          m_new = m_ref;
          fac = 1.f;
        }
        l *= fac;
        // P of this tile overwrites its S stage, which this tile's QK^T (complete at s_full)
        // wrote after the P.V of tile j - 2 had read the stage's previous P
        const uint32_t pcol = tmem + lanebase + st * 128;
        // this thread's and its partner's exchange regions (16-byte units XOR-swizzled by row)
        uint8_t* xmine = smem + C::kOffX + (row * 2 + half) * C::kXRegion;
        const uint8_t* xpart = smem + C::kOffX + (row * 2 + (half ^ 1)) * C::kXRegion;
        const int xsw = row & 7;
        auto xput = [&](int unit, const uint32_t* w4) {
          *reinterpret_cast<uint4*>(xmine + 16 * (unit ^ xsw)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        };
        auto xget = [&](int unit, uint32_t* w4) {
          const uint4 v = *reinterpret_cast<const uint4*>(xpart + 16 * (unit ^ xsw));
          w4[0] = v.x;
          w4[1] = v.y;
          w4[2] = v.z;
          w4[3] = v.w;
        };
        auto xbarrier = [&]() -> bool {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&M.xchg_bar));
          const bool r = kwait(M, smem_addr(&M.xchg_bar), xph & 1);
          ++xph;
          return r;
        };
        float lq[2] = {0.f, 0.f};
        uint32_t hold0[16], hold1[16];  // bf16: this half's second-round chunks
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          const int ch = chunk_order<E4M3>(half, k);
          uint32_t r[32];
          tmem_ld32(sbase_t + ch * 32, r);
          tmem_ld_wait();
          float pv[32];
          if (full) {
#pragma unroll
            for (int e = 0; e < 32; ++e) pv[e] = ex2(fmaf(u2f(r[e]), cl2, -m_new));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const bool vis = static_cast<uint32_t>(ch * 32 + e - vlo) < vspan;
              pv[e] = vis ? ex2(fmaf(u2f(r[e]), cl2, -m_new)) : 0.f;
            }
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) lq[e & 1] += pv[e];
          constexpr int kW = E4M3 ? 8 : 16;
          uint32_t w[kW];
          pack_p<E4M3>(pv, w);
          if constexpr (E4M3) {
            tmem_st8(pcol + (C::kPCols / 2) * half + (C::kPCols / 8) * ch, w);
            // the region holds this half's 128 keys in key order: chunk ch at units 2 ch, 2 ch + 1
#pragma unroll
            for (int q = 0; q < 2; ++q) xput(2 * ch + q, w + 4 * q);
          } else {
            tmem_st16(pcol + (C::kPCols / 2) * half + (C::kPCols / 8) * ch, w);
            // first round: this half's chunks k = 0, 1 at units 4 k .. +4; the others wait
            if (k < 2) {
#pragma unroll
              for (int q = 0; q < 4; ++q) xput(4 * k + q, w + 4 * q);
            } else if (k == 2) {
#pragma unroll
              for (int e = 0; e < 16; ++e) hold0[e] = w[e];
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) hold1[e] = w[e];
            }
          }
        }
        l += lq[0] + lq[1];
        // swap halves: this thread's row gets the other half's 128 keys of P
        if (!(ok = xbarrier())) break;
        if constexpr (E4M3) {
          uint32_t w[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) xget(q, w + 4 * q);
          tmem_st32(pcol + (C::kPCols / 2) * (half ^ 1), w);
        } else {
          const int hp = half ^ 1;
#pragma unroll 1
          for (int rd = 0; rd < 2; ++rd) {
            if (rd == 1) {
              // the partner has read the first round: this half's second round goes out
              if (!(ok = xbarrier())) break;
#pragma unroll
              for (int q = 0; q < 4; ++q) xput(q, hold0 + 4 * q);
#pragma unroll
              for (int q = 0; q < 4; ++q) xput(4 + q, hold1 + 4 * q);
              if (!(ok = xbarrier())) break;
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              uint32_t w[16];
#pragma unroll
              for (int q = 0; q < 4; ++q) xget(4 * c2 + q, w + 4 * q);
              tmem_st16(pcol + (C::kPCols / 2) * hp + (C::kPCols / 8) * chunk_order<E4M3>(hp, 2 * rd + c2), w);
            }
          }
          if (!ok) break;
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&M.pv_local[st]));
        M.corr[st][L] = fac;
        if (i == n - 1) {
          // final row statistics: the two halves of the row add their sums
          M.xsum[L] = l;
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&M.xchg_bar));
          if (!(ok = kwait(M, smem_addr(&M.xchg_bar), xph & 1))) break;
          ++xph;
          M.fin_l[s & 1][L] = l + M.xsum[L ^ 64];
          M.fin_m[s & 1][L] = m_new;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&M.cor_ready[st]));
        m_ref = m_new;
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ correction + epilogue
    const int L = tid - 128, row = L & 63, half = L >> 6;
    const uint32_t lanebase = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const uint32_t obase = tmem + lanebase + 256;
    const int m = 64 * (int)rank + row;  // this thread's M row
    int j = 0;
    uint32_t ncomb = 0;  // fused combines so far (the parity of their syncs)
    bool ok = true;
    for (int s = 0; s < nseg && ok; ++s) {
      const Segment sg = seg_at(s);
      const int n = sg.tile_end - sg.tile_begin;
      float fl = 0.f, fm = 0.f;  // the piece's final row statistics
      for (int i = 0; i < n; ++i, ++j) {
        const int st = j & 1;
        if (!(ok = kwait(M, smem_addr(&M.cor_ready[st]), (j >> 1) & 1))) break;
        const float fac = M.corr[st][L];
        if (i == n - 1) {
          // read before this tile's arrival below: the softmax can then run at most two
          // tiles ahead, and writes these statistics again only for the piece after next
          fl = M.fin_l[s & 1][L];
          fm = M.fin_m[s & 1][L];
        }
        if (i > 0 && __any_sync(0xffffffffu, fac != 1.f)) {
          // O holds tiles < j once the P.V of tile j - 1 completes
          if (!(ok = kwait(M, smem_addr(&M.o_done[st ^ 1]), ((j - 1) >> 1) & 1))) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            tmem_ld32(obase + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(u2f(r[e]) * fac);
            tmem_st32(obase + c * 32, r);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&M.pv_local[st]));
        if (warp == 4) {
          // forward this CTA's readiness to the leader: one cross-CTA arrive per tile.  P and
          // the corrected O are in tensor memory (ordered by the writers' tcgen05 waits and
          // fences), so the arrive need not release generic memory at cluster scope
          if (!(ok = kwait(M, smem_addr(&M.pv_local[st]), (j >> 1) & 1))) break;
          if (lane == 0) mbar_arrive_remote(lead(M.pv_ready[st]));
          __syncwarp();
        }
      }
      if (!ok) break;
      // epilogue: the piece to the output or to its slot
      if (!(ok = kwait(M, smem_addr(&M.o_done[(j - 1) & 1]), ((j - 1) >> 1) & 1))) break;
      tc_fence_after();
      const int b = sg.row() / DS.Qb, flat = kTileM * (sg.row() % DS.Qb) + m;
      const int slot = sg.slot();
      const size_t sl = slot < 0 ? 0 : (size_t)slot;
      piece_epilogue(p, p.ws + WL.partial_o + sl * WL.slot_bytes,
                     reinterpret_cast<float*>(p.ws + WL.partial_lse) + sl * kTileM,
                     reinterpret_cast<float*>(p.ws + WL.partial_scale) + sl * 2 * kTileM, obase, half, m, b, flat,
                     flat < rows_q, slot < 0, fl, fm);
      if (p.fused_combine && slot >= 0) {
        tc_fence_before();
        const int first = slot - sg.piece() * DS.wb;
        const int v = arrive_piece(M, p,
                                   reinterpret_cast<unsigned long long*>(p.ws + WL.counters) + 2 * (size_t)sg.row() + rank,
                                   ncomb & 1, sg.row(), first, sg.n_parts(), L);
        ++ncomb;
        ok = v >= 0;
        if (!ok) break;
        if (v > 0)
          combine_row(p, p.ws + WL.partial_o, reinterpret_cast<const float*>(p.ws + WL.partial_lse),
                      reinterpret_cast<const float*>(p.ws + WL.partial_scale), WL.slot_bytes, sg.row(), first,
                      sg.n_parts(), DS.wb, DS.Qb, rank, L, 128);
      }
      tc_fence_before();
    }
    if (ok && p.fused_combine) write_empty_rows(p, DS, L);
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issue (leader CTA)
    if (rank == 0 && lane == 0) {
      int j = 0, pvc = 0, tcount = 0;
      int rslot = 0;        // next ring slot in consumption order
      uint32_t rphase = 0;  // and the parity of its fill
      bool ok = true;
      // next ring slot: wait until both CTAs' copies landed (one CTA-scope test in the
      // common case, the bounded wait otherwise)
      auto take = [&](uint32_t& addr, int& slot) -> bool {
        slot = rslot;
        const uint32_t bar = smem_addr(&M.full[rslot]);
        if (!mbar_try_wait_cta(bar, rphase) && !kwait_spin(M, bar, rphase)) return false;
        addr = sRing + slot * C::kSlot;
        if (++rslot == C::kNS) {
          rslot = 0;
          rphase ^= 1u;
        }
        return true;
      };
      auto qk = [&](int jt) -> bool {
        // S stage jt & 1 was last read by the softmax of tile jt - 2 and, as its P, by that
        // tile's P.V, issued after its pv_ready and before this QK^T; the tensor pipe runs
        // MMAs in issue order: no separate wait
        const int st = jt & 1;
        const uint32_t d = tmem + st * 128;
        // the descriptors of step t are the block's plus 32 bytes per step
#pragma unroll
        for (int kb = 0; kb < C::kNKb; ++kb) {
          uint32_t ka;
          int slot;
          if (!take(ka, slot)) return false;
          tc_fence_after();
          const uint32_t qa = sQ + kb * 8192;
          if (E4M3 && kb == C::kNLat) {
            const uint64_t ad = smem_desc_sw64(qa, 512), bd = smem_desc_sw64(ka, 512);
#pragma unroll
            for (int t = 0; t < C::kRopeSteps; ++t) mma_ss<KIND>(d, ad + 2 * t, bd + 2 * t, C::kIdescQK, 1u);
          } else {
            const uint64_t ad = smem_desc_sw128(qa, 16, 1024), bd = smem_desc_sw128(ka, 16, 1024);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              mma_ss<KIND>(d, ad + 2 * t, bd + 2 * t, C::kIdescQK, (kb | t) != 0 ? 1u : 0u);
          }
          mma_commit_pair(smem_addr(&M.empty[slot]), 0x3);
        }
        mma_commit_pair(smem_addr(&M.s_full[st]), 0x3);
        return true;
      };
      // P.V of tile `tile` of a request with ngroups key groups, the last tail_rows long
      auto pv = [&](bool first, int tile, int ngroups, int tail_rows) -> bool {
        const int pst = pvc & 1;
        if (!kwait(M, smem_addr(&M.pv_ready[pst]), (pvc >> 1) & 1)) return false;
        tc_fence_after();
#pragma unroll 1
        for (int vp = 0; vp < 4; ++vp) {
          // bf16: slot c holds the columns of output chunk c; e4m3: one slot holds both
          uint32_t va[2];
          int slot[2];
#pragma unroll
          for (int it = 0; it < C::kVItems; ++it)
            if (!take(va[it], slot[it])) return false;
          if (4 * tile + vp == ngroups - 1 && tail_rows != 0) {
            // the request's last key group: the peer zeroed its slots' tail too
            if (!kwait(M, smem_addr(&M.tail_ready[tcount & 1]), (tcount >> 1) & 1)) return false;
            ++tcount;
          }
          tc_fence_after();
          // output chunk c's V columns: e4m3 at 8 KB into the group's slot, bf16 in slot c;
          // step t moves 16 (bf16) or 32 (e4m3) keys of 128 B down
          const uint64_t vd0 = smem_desc_sw128(va[0], 8192, 1024);
          const uint64_t vd1 = E4M3 ? vd0 + (8192 >> 4) : smem_desc_sw128(va[1], 8192, 1024);
#pragma unroll
          for (int t = 0; t < C::kPvSteps; ++t) {
            const uint32_t acc = (first && vp == 0 && t == 0) ? 0u : 1u;
            // keys [64 vp + (32 or 16) t, ...) of P: 8 columns of stage pst per step
            const uint32_t a_tm = tmem + pst * 128 + (C::kPCols / 4) * vp + 8 * t;
            const uint64_t dt = static_cast<uint64_t>(t) * ((E4M3 ? 4096 : 2048) >> 4);
            mma_ts<KIND>(tmem + 256, a_tm, vd0 + dt, C::kIdescPV, acc);
            mma_ts<KIND>(tmem + 384, a_tm, vd1 + dt, C::kIdescPV, acc);
          }
#pragma unroll
          for (int it = 0; it < C::kVItems; ++it) mma_commit_pair(smem_addr(&M.empty[slot[it]]), 0x3);
        }
        mma_commit_pair(smem_addr(&M.o_done[pst]), 0x3);
        ++pvc;
        return true;
      };
      // One software pipeline over the CTA's tiles, across pieces: QK^T(t + 1) then P.V(t),
      // also when t + 1 opens the next piece (the ring holds K(t + 1) ahead of V(t))
      bool pend = false, pend_first = false;  // the tile whose P.V is still to be issued
      int pend_tile = 0, pend_ng = 0, pend_tr = 0;
      for (int s = 0; s < nseg && ok; ++s) {
        const Segment sg = seg_at(s);
        const int n = sg.tile_end - sg.tile_begin;
        const int ng = cdiv(sg.K, kKeyGroup), tr = sg.K % kKeyGroup;
        if (!(ok = kwait(M, smem_addr(&M.q_full), s & 1))) break;
        tc_fence_after();
        for (int i = 0; i < n && ok; ++i) {
          ok = qk(j + i);
          // Q is free once the piece's last QK^T completes: the next piece's Q load need
          // not wait for the P.V issued after it
          if (ok && i == n - 1) mma_commit_pair(smem_addr(&M.q_empty), 0x3);
          if (ok && pend) ok = pv(pend_first, pend_tile, pend_ng, pend_tr);
          pend = true;
          pend_first = i == 0;
          pend_tile = sg.tile_begin + i;
          pend_ng = ng;
          pend_tr = tr;
        }
        j += n;
      }
      if (ok && pend) ok = pv(pend_first, pend_tile, pend_ng, pend_tr);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ Q loads
    // lane kb issues Q block kb (one copy a lane: a thread's copies go out one after another);
    // lane 0 waits and the warp follows its verdict, so the count of issued loads is exact
    for (int s = 0; s < nseg; ++s) {
      bool okq = true;
      if (s > 0 && lane == 0) okq = kwait(M, smem_addr(&M.q_empty), (s - 1) & 1);
      if (!__shfl_sync(0xffffffffu, okq ? 1 : 0, 0)) break;
      const uint32_t bar = lead(M.q_full);
      // the leader arms the barrier with both CTAs' bytes; the peer's copies only complete bytes on it
      if (lane == 0 && rank == 0) mbar_arrive_expect_tx(smem_addr(&M.q_full), 2 * C::kQBytes);
      const int wr = seg_at(s).row(), b = wr / DS.Qb;
      const int r0 = kTileM * (wr % DS.Qb) + 64 * (int)rank;  // this CTA's 64 (token, head) rows
      if (lane < C::kNLat) tma_load_3d_pair(sQ + lane * 8192, &maps.q_latent, lane * C::kBlk, r0, b, bar);
      else if (lane == C::kNLat) tma_load_3d_pair(sQ + C::kNLat * 8192, &maps.q_rope, 0, r0, b, bar);
      if (lane == 0) M.nq = s + 1;
      __syncwarp();
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------------ K blocks and V key groups, one ring
    // Consumption order over the CTA's tiles, across pieces: K(t0), then K(t), V(t - 1) for
    // every following tile, then V(last); a K block is this CTA's two key groups x 128 B of
    // columns, a V key group this CTA's output columns of 64 keys.  Two warps issue the
    // copies: warp 10 the even fills, warp 11 the odd ones.  The slot count is even, so a
    // slot always has the same owner, and an owner only ever waits for the release of its
    // own previous fill of the slot.  Lane q of the owning warp issues box q of a fill
    // (page boxes: tma_pages.cuh).
    const int own = warp - 10;
    const int nb = ONE_BOX ? 1 : boxes_per_group(p.page_size), br = ONE_BOX ? kKeyGroup : box_rows(p.page_size);
    constexpr bool one_box = ONE_BOX;
    int32_t* table = &M.boxes[own][0][0];
    int fill = 0;
    uint32_t tph = 0;
    uint32_t ntg = 0;  // tail groups so far (this warp's or not): their tail_ready barrier
    bool ok = true;
    // the next fill in consumption order: this warp's (wait until its slot is free) or the
    // other warp's (skip); lane-uniform
    auto acquire = [&](int& slot, bool& mine) -> bool {
      slot = fill % C::kNS;
      mine = (fill & 1) == own;
      if (mine && fill >= C::kNS && !kwait(M, smem_addr(&M.empty[slot]), ((fill / C::kNS) - 1) & 1)) return false;
      ++fill;
      return true;
    };
    // Page boxes of a tile, loaded a tile ahead into registers and used a tile later (the
    // validity check is a select, and a bad page id is reported at the end).  page_size >= 64:
    // one box per key group, every lane holds the four; below 64: lane k holds box k and
    // writes its page to the warp's table when the tile comes up, where the issuing lanes
    // read it.
    struct TileBoxes {
      int pg[4], rw[4];
    };
    bool bad_page = false;
    auto fetch = [&](int b, int K, int tile, TileBoxes& tb) {
      bool bad;
      if constexpr (one_box) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          box_page(p.page_table, p.pt_stride, p.num_pages, p.page_shift, b, tile * kTileN + q * kKeyGroup, K, tb.pg[q],
                   tb.rw[q], bad);
          bad_page |= bad;
        }
      } else if (lane < 4 * nb) {
        box_page(p.page_table, p.pt_stride, p.num_pages, p.page_shift, b, tile * kTileN + lane * br, K, tb.pg[0],
                 tb.rw[0], bad);
        bad_page |= bad;
      } else {
        tb.pg[0] = p.num_pages;
      }
    };
    // below 64: this lane's box of the tile into the warp's table, at the loader's tile
    // count ti mod 3 (the tile whose V is loaded, the one whose K is loaded, the next)
    auto publish = [&](int ti, const TileBoxes& tb) {
      if constexpr (one_box) return;
      table[(ti % 3) * 32 + lane] = tb.pg[0];
      __syncwarp();
    };
    // page and row of box k (k < 4 nb) of a tile, in the issuing lane
    auto box = [&](const TileBoxes& tb, int ti, int k, int& pg, int& rw) {
      if constexpr (one_box) {
        // selects, not a runtime index: the boxes stay in registers
        pg = k == 0 ? tb.pg[0] : k == 1 ? tb.pg[1] : k == 2 ? tb.pg[2] : tb.pg[3];
        rw = k == 0 ? tb.rw[0] : k == 1 ? tb.rw[1] : k == 2 ? tb.rw[2] : tb.rw[3];
      } else {
        pg = table[(ti % 3) * 32 + k];
        rw = 0;
      }
    };
    auto load_k = [&](int ti, const TileBoxes& tb) -> bool {
      for (int kb = 0; kb < C::kNKb; ++kb) {
        int slot;
        bool mine;
        if (!acquire(slot, mine)) return false;
        if (mine && lane < 2 * nb) {
          // lane q issues box q of the fill: a thread's copies go out one after another, so
          // the fill's boxes leave from separate lanes
          const bool rope = kb == C::kNLat;
          const int rowb = rope ? C::kRopeRow : 128;  // bytes per key row of the block
          const uint32_t bar = lead(M.full[slot]);
          const uint32_t dst = sRing + slot * C::kSlot;
          // both CTAs' two key groups
          if (lane == 0 && rank == 0) mbar_arrive_expect_tx(smem_addr(&M.full[slot]), 4 * 64 * rowb);
          const int k0 = 2 * (int)rank * nb;  // this CTA's boxes: key groups 2 rank, 2 rank + 1
          int pg, rw;
          box(tb, ti, k0 + lane, pg, rw);
          const uint32_t d = dst + lane * br * rowb;
          if (!rope) tma_load_3d_pair(d, &maps.ckv, kb * C::kBlk, rw, pg, bar);
          else tma_load_3d_pair(d, &maps.kpe, 0, rw, pg, bar);
          if (lane == 0) {
            M.nfill[slot] += 1;
            M.fbytes[slot] = 2 * 64 * rowb;
          }
        }
        __syncwarp();
      }
      return true;
    };
    // V of tile `tile` of a request with ngroups key groups, the last tail_rows long (0: full)
    auto load_v = [&](int tile, int ti, int ngroups, int tail_rows, const TileBoxes& tb) -> bool {
      for (int vp = 0; vp < 4; ++vp) {
        int slot[2];
        bool mine[2];
        int nmine = 0;
#pragma unroll
        for (int it = 0; it < C::kVItems; ++it) {
          if (!acquire(slot[it], mine[it])) return false;
          nmine += mine[it] ? 1 : 0;
        }
        const bool tail_grp = 4 * tile + vp == ngroups - 1 && tail_rows != 0;
        const bool tail = tail_grp && nmine != 0;
        // this CTA's 128-byte column blocks of V: bf16 blocks {0,1,4,5} or {2,3,6,7}
        // (two per slot, one slot per output chunk), e4m3 blocks {rank, 2 + rank}
        const uint32_t tbar = smem_addr(&M.tail_bar[own]);
        if (lane < 2 * nb) {
          // lane 2 q + u issues page box q of column block u (see load_k: one box a lane)
          if (tail && lane == 0) mbar_arrive_expect_tx(tbar, nmine * C::kSlot);
          const int q = lane >> 1, u = lane & 1;
#pragma unroll
          for (int it = 0; it < C::kVItems; ++it) {
            if (!mine[it]) continue;
            const uint32_t dst = sRing + slot[it] * C::kSlot;
            const uint32_t bar = lead(M.full[slot[it]]);
            if (!tail && lane == 0 && rank == 0) mbar_arrive_expect_tx(smem_addr(&M.full[slot[it]]), 2 * C::kSlot);
            int pg, rw;
            box(tb, ti, vp * nb + q, pg, rw);
            const int gb = E4M3 ? 2 * u + (int)rank : 4 * it + 2 * (int)rank + u;
            const uint32_t d = dst + u * 8192 + q * br * 128;
            if (tail) tma_load_3d(d, &maps.ckv, gb * C::kBlk, rw, pg, tbar);
            else tma_load_3d_pair(d, &maps.ckv, gb * C::kBlk, rw, pg, bar);
            if (lane == 0) {
              M.nfill[slot[it]] += 1;
              M.fbytes[slot[it]] = tail ? 0u : (uint32_t)C::kSlot;
            }
          }
          if (tail && lane == 0) M.ntail[own] += 1;
        }
        __syncwarp();
        if (tail) {
          if (!tail_group<E4M3>(M, smem, own, rank, lane, tph, ntg, slot[0], slot[C::kVItems - 1], mine[0],
                                mine[C::kVItems - 1], tail_rows))
            return false;
          ++tph;
        }
        if (tail_grp) ++ntg;
      }
      return true;
    };
    // e4m3, page size >= 64: this CTA's K rows of a tile (its two key groups, latent and
    // rope: each a page's contiguous rows) prefetched into L2 a tile ahead of their copies
    // (measured: shorter e4m3 launches, slightly longer bf16 ones)
    auto prefetch_k = [&](const TileBoxes& tb) {
      if constexpr (one_box && E4M3) {
        if (own == 0 && lane < 4) {
          int pg, rw;
          box(tb, 0, 2 * (int)rank + (lane & 1), pg, rw);
          if (pg < p.num_pages) {
            const bool rope = lane >= 2;
            const size_t rb = (size_t)(rope ? kDRope : kDLatent) * (E4M3 ? 1 : 2);  // bytes per key row
            const uint8_t* base = static_cast<const uint8_t*>(rope ? p.kpe : p.ckv);
            prefetch_l2_bulk(base + ((size_t)pg * p.page_size + rw) * rb, (uint32_t)(kKeyGroup * rb));
          }
        }
      }
    };
    // One software pipeline over the CTA's tiles, across pieces: K(t + 1) goes ahead of V(t)
    // also when t + 1 opens the next piece, so a piece's last P.V never drains the ring
    bool pend = false;  // the tile whose V is still to be loaded
    int pend_tile = 0, pend_ti = 0, pend_ng = 0, pend_tr = 0;
    TileBoxes pend_tb;
    int ti = 0;  // tiles of this CTA so far
    for (int s = 0; s < nseg && ok; ++s) {
      const Segment sg = seg_at(s);
      const int b = sg.row() / DS.Qb;
      const int K = sg.K;
      const int ng = cdiv(K, kKeyGroup), tr = K % kKeyGroup;
      TileBoxes cur, next;
      fetch(b, K, sg.tile_begin, cur);
      for (int tile = sg.tile_begin; tile < sg.tile_end && ok; ++tile, ++ti) {
        // the next tile's page ids: bf16, read once this tile's K copies are out (its first
        // copy then waits only for its own page ids); e4m3, before them, a tile ahead of its
        // L2 prefetch (each order measured faster for its type)
        if (E4M3 && tile + 1 < sg.tile_end) fetch(b, K, tile + 1, next);
        publish(ti, cur);
        ok = load_k(ti, cur);
        if (!E4M3 && tile + 1 < sg.tile_end) fetch(b, K, tile + 1, next);
        if (ok && tile + 1 < sg.tile_end) prefetch_k(next);
        if (ok && pend) ok = load_v(pend_tile, pend_ti, pend_ng, pend_tr, pend_tb);
        pend = true;
        pend_tile = tile;
        pend_ti = ti;
        pend_ng = ng;
        pend_tr = tr;
        pend_tb = cur;
        cur = next;
      }
    }
    if (ok && pend) ok = load_v(pend_tile, pend_ti, pend_ng, pend_tr, pend_tb);
    if (__any_sync(0xffffffffu, bad_page) && own == 0 && lane == 0) atomicOr(&M.err, kErrBadPage);
  }

  // ------------------------------------------------------------ teardown
  __syncwarp();
  grid_launch_dependents();
  __syncthreads();
  tc_fence_before();
  cluster_sync();  // both CTAs have stopped issuing; an abort of either is visible in both
  tc_fence_after();
  if (*reinterpret_cast<volatile uint32_t*>(&M.abort)) drain_after_abort<E4M3>(M, rank, warp, lane, tid);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 8) tmem_dealloc_pair(tmem, 512);
  if (tid == 0) reinterpret_cast<uint32_t*>(p.ws + WL.cta_status)[2 * cl + rank] = M.err;
  // the work rows this CTA arrived last on, by 8 warps (no abort: every piece arrived)
  if (p.fused_combine && !*reinterpret_cast<volatile uint32_t*>(&M.abort) && tid < 256) {
    const int n = min((int)M.ncl, kCombList);
    for (int e = 0; e < n; ++e) {
      const int4 E = M.comb_list[e];
      combine_row(p, p.ws + WL.partial_o, reinterpret_cast<const float*>(p.ws + WL.partial_lse),
                  reinterpret_cast<const float*>(p.ws + WL.partial_scale), WL.slot_bytes, E.x, E.y, E.z, DS.wb, DS.Qb,
                  rank, tid, 256);
    }
  }
}

}  // namespace tc

template <bool E4M3, bool ONE_BOX>
static cudaError_t launch_variant(const DecodeParams& p, const KvMaps& maps, cudaStream_t stream) {
  const dim3 grid(2 * p.num_clusters), block(tc::kThreads);
  const int smem = tc::smem_bytes<E4M3>();
  cudaError_t e = cudaFuncSetAttribute(tc::split_kv_tc<E4M3, ONE_BOX>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  tc::split_kv_tc<E4M3, ONE_BOX><<<grid, block, smem, stream>>>(p, maps);
  return cudaGetLastError();
}

cudaError_t launch_split_kv(const DecodeParams& p, const KvMaps& maps, cudaStream_t stream) {
  const bool one = p.page_size >= kKeyGroup;
  if (p.qkv_e4m3) return one ? launch_variant<true, true>(p, maps, stream) : launch_variant<true, false>(p, maps, stream);
  return one ? launch_variant<false, true>(p, maps, stream) : launch_variant<false, false>(p, maps, stream);
}

int split_kv_max_clusters(int device, bool e4m3) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(tc::kThreads);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e;
  if (e4m3) {
    cfg.dynamicSmemBytes = tc::smem_bytes<true>();
    cudaFuncSetAttribute(tc::split_kv_tc<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes);
    e = cudaOccupancyMaxActiveClusters(&n, tc::split_kv_tc<true, true>, &cfg);
  } else {
    cfg.dynamicSmemBytes = tc::smem_bytes<false>();
    cudaFuncSetAttribute(tc::split_kv_tc<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes);
    e = cudaOccupancyMaxActiveClusters(&n, tc::split_kv_tc<false, true>, &cfg);
  }
  if (e != cudaSuccess || n <= 0) return sms / 2;
  return n;
}

}  // namespace mla
