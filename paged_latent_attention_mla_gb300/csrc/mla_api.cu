// C ABI of the paged MLA decode library (declared in include/mla.h).
//
// Host-side work only: argument validation, the plan (a host mirror of the
// device schedule, used to size the workspace), TMA descriptor encoding and
// kernel launches.  Nothing here allocates device memory or synchronizes the
// stream on the decode path.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/mla.h"
#include "mla_common.cuh"
#include "mla_kernels.cuh"

using namespace mla;

namespace {

constexpr int kMaxRows = 16384;   // B * seq_len_q (schedule scratch in shared memory)
constexpr int kMaxSeqLenQ = 64;
constexpr int kMaxWorld = 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

mla_status_t validate_cfg(const mla_config_t* cfg, int B, int H, int page_size, int window_left) {
  if (!cfg) return MLA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || cfg->seq_len_q < 1 || cfg->num_pages < 1 || cfg->page_table_stride < 1) return MLA_ERR_INVALID_ARG;
  if (window_left < -1 || cfg->num_clusters < 0) return MLA_ERR_INVALID_ARG;
  if (cfg->qkv_dtype != MLA_BF16 && cfg->qkv_dtype != MLA_E4M3) return MLA_ERR_INVALID_ARG;
  if (cfg->out_dtype != MLA_F32 && cfg->out_dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
  if (!(std::isfinite(cfg->q_descale) && std::isfinite(cfg->ckv_descale) && std::isfinite(cfg->kpe_descale)) ||
      cfg->q_descale <= 0.f || cfg->ckv_descale <= 0.f || cfg->kpe_descale <= 0.f)
    return MLA_ERR_INVALID_ARG;
  if (cfg->qkv_dtype == MLA_BF16 && (cfg->q_descale != 1.f || cfg->ckv_descale != 1.f || cfg->kpe_descale != 1.f))
    return MLA_ERR_INVALID_ARG;
  // one scale for the whole key (latent and rope parts are one contraction)
  if (cfg->qkv_dtype == MLA_E4M3 && cfg->ckv_descale != cfg->kpe_descale) return MLA_ERR_UNSUPPORTED;
  if (page_size < 1) return MLA_ERR_INVALID_ARG;
  if (!pow2(page_size) || page_size < kMinPageSize || page_size > kMaxPageSize) return MLA_ERR_UNSUPPORTED;
  if (H > kMaxHeads || cfg->seq_len_q > kMaxSeqLenQ) return MLA_ERR_UNSUPPORTED;
  if ((long long)B * cfg->seq_len_q > kMaxRows) return MLA_ERR_UNSUPPORTED;
  if ((long long)B * ((cfg->seq_len_q * H + kTileM - 1) / kTileM) > kMaxWorkRows) return MLA_ERR_UNSUPPORTED;
  if (cfg->num_clusters > kMaxClusters) return MLA_ERR_UNSUPPORTED;
  if ((long long)cfg->page_table_stride * page_size > (1ll << 30)) return MLA_ERR_UNSUPPORTED;
  if (cfg->cp_world < 0 || cfg->cp_interleave < 0) return MLA_ERR_INVALID_ARG;
  if (cfg->cp_world > 1) {
    if (cfg->cp_world > kMaxWorld || cfg->cp_rank < 0 || cfg->cp_rank >= cfg->cp_world) return MLA_ERR_INVALID_ARG;
  }
  if (cfg->partial_fp16 != 0 && cfg->partial_fp16 != 1) return MLA_ERR_INVALID_ARG;
  if (cfg->combine_in_kernel != 0 && cfg->combine_in_kernel != 1) return MLA_ERR_INVALID_ARG;
  if (cfg->reducer_d_tiles != 0 && cfg->reducer_d_tiles != 1 && cfg->reducer_d_tiles != 2 &&
      cfg->reducer_d_tiles != 4 && cfg->reducer_d_tiles != 8)
    return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

int cp_world_of(const mla_config_t* cfg) { return cfg->cp_world > 1 ? cfg->cp_world : 1; }
int cp_interleave_of(const mla_config_t* cfg) { return cfg->cp_interleave > 0 ? cfg->cp_interleave : 1; }
int d_tiles_of(const mla_config_t* cfg) { return cfg->reducer_d_tiles > 0 ? cfg->reducer_d_tiles : 8; }

// clusters of one persistent wave on the current device (cached per device)
int resolve_clusters(const mla_config_t* cfg, bool e4m3, int* out) {
  if (cfg->num_clusters > 0) {
    *out = cfg->num_clusters;
    return 0;
  }
  static std::mutex mu;
  static int cache[64][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> g(mu);
  int& c = cache[dev][e4m3 ? 1 : 0];
  if (c == 0) c = split_kv_max_clusters(dev, e4m3);
  if (c <= 0) return -1;
  *out = c;
  return 0;
}

// Host mirror of the device deal (same functions, same integer arithmetic) over host
// lengths: the most pieces any work row is cut into.  Under context parallelism or with
// local bounds (whose device values the host does not have) every local key is taken
// as visible, which makes the count an estimate.
int plan_max_parts(const int32_t* seq_lens, int B, int H, int page_size, int window_left, const mla_config_t* cfg,
                   int G) {
  const int Sq = cfg->seq_len_q;
  const DealShape d = deal_shape(B, Sq, H, G);
  const int pu = piece_units(cfg->qkv_dtype == MLA_E4M3);
  const bool exact = cp_world_of(cfg) == 1 && !cfg->local_visible_lens;
  auto span = [&](int b, int t0, int t1, int& tlo, int& n) {
    int K = seq_lens[b];
    K = K < 0 ? 0 : (K > cfg->page_table_stride * page_size ? cfg->page_table_stride * page_size : K);
    int lo_min = INT_MAX, hi_max = 0;
    for (int t = t0; t <= t1; ++t) {
      int lo = 0, hi = K;
      if (exact) token_range(K, K, 0, false, Sq, t, cfg->causal, window_left, 1, 0, 1, lo, hi);
      if (hi > lo) {
        lo_min = std::min(lo_min, lo);
        hi_max = std::max(hi_max, hi);
      }
    }
    if (hi_max > 0) tile_span(lo_min, hi_max, tlo, n);
    else tlo = n = 0;
  };
  std::vector<long long> prefix(d.S + 1, 0);
  std::vector<int> ulo(d.S), U(d.S);
  for (int s = 0; s < d.S; ++s) {
    const int b = s / d.nsub, k = s % d.nsub;
    int t0, t1;
    work_tokens(k * d.wb, std::min(d.Qb, k * d.wb + d.wb) - 1, Sq, H, t0, t1);
    span(b, t0, t1, ulo[s], U[s]);
    prefix[s + 1] = prefix[s] + (U[s] > 0 ? pu + kUnitsPerTile * U[s] : 0);
  }
  const long long T = prefix[d.S];
  const int Gd = deal_groups(d.Gg, T);
  int most = 1;
  for (int w = 0; w < d.Rw; ++w) {
    const int b = w / d.Qb, i = w % d.Qb, s = b * d.nsub + i / d.wb;
    int t0, t1, tlo, n;
    work_tokens(i, i, Sq, H, t0, t1);
    span(b, t0, t1, tlo, n);
    if (n <= 0) continue;
    const long long xf = tile_unit(prefix[s], pu, tlo - ulo[s]), xl = tile_unit(prefix[s], pu, tlo - ulo[s] + n - 1);
    most = std::max(most, group_of_tile(xl, T, Gd) - group_of_tile(xf, T, Gd) + 1);
  }
  return most;
}

// ------------------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over [d2][d1][d0] (d0 innermost, elements of es bytes), box {box0, box1, 1}
bool encode3d(CUtensorMap* m, const void* base, bool e4m3, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
              uint32_t box1, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t es = e4m3 ? 1 : 2;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// KV maps: [pages][P][D] with boxes of one page's box_rows(P) rows; Q maps: [B][Sq * H][D]
// with boxes of 64 (token, head) rows (a work row's rows past Sq * H read as zeros).
bool encode_kv_maps(KvMaps* maps, const void* ckv, const void* kpe, const void* q_latent, const void* q_rope, bool e4m3,
                    int num_pages, int page_size, int B, int rows_q) {
  const uint32_t blk = e4m3 ? 128 : 64;
  const CUtensorMapSwizzle rope_sw = e4m3 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  const uint32_t br = (uint32_t)box_rows(page_size);
  memset(maps, 0, sizeof(*maps));
  bool ok = encode3d(&maps->ckv, ckv, e4m3, kDLatent, (uint64_t)page_size, (uint64_t)num_pages, blk, br,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
            encode3d(&maps->kpe, kpe, e4m3, kDRope, (uint64_t)page_size, (uint64_t)num_pages, kDRope, br, rope_sw);
  if (ok && q_latent)
    ok = encode3d(&maps->q_latent, q_latent, e4m3, kDLatent, (uint64_t)rows_q, (uint64_t)B, blk, kRowsPerCta,
                  CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode3d(&maps->q_rope, q_rope, e4m3, kDRope, (uint64_t)rows_q, (uint64_t)B, kDRope, kRowsPerCta, rope_sw);
  return ok;
}

// A tag for this call's arrival counters (never 0, so a zeroed workspace matches no call).
uint32_t next_epoch() {
  static std::atomic<uint32_t> epoch{0};
  uint32_t e = ++epoch;
  if (e == 0) e = ++epoch;
  return e;
}

// decode parameters from the call's arguments (validated)
DecodeParams make_params(const void* q_latent, const void* q_rope, const void* ckv_cache, const void* kpe_cache,
                         const int32_t* page_table, const int32_t* seq_lens, float scale, int window_left, void* out,
                         float* lse, void* workspace, int B, int H, int page_size, const mla_config_t* cfg, int G) {
  DecodeParams p{};
  p.q_latent = q_latent;
  p.q_rope = q_rope;
  p.ckv = ckv_cache;
  p.kpe = kpe_cache;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.global_seq_lens = cp_world_of(cfg) > 1 ? cfg->global_seq_lens : nullptr;
  p.local_visible_lens = cfg->local_visible_lens;
  p.out = out;
  p.lse = lse;
  p.ws = static_cast<uint8_t*>(workspace);
  p.B = B;
  p.Sq = cfg->seq_len_q;
  p.H = H;
  p.num_pages = cfg->num_pages;
  p.pt_stride = cfg->page_table_stride;
  p.page_size = page_size;
  p.page_shift = 0;
  while ((1 << p.page_shift) < page_size) ++p.page_shift;
  p.causal = cfg->causal ? 1 : 0;
  p.window_left = window_left;
  p.cp_world = cp_world_of(cfg);
  p.cp_rank = p.cp_world > 1 ? cfg->cp_rank : 0;
  p.cp_interleave = cp_interleave_of(cfg);
  p.qkv_e4m3 = cfg->qkv_dtype == MLA_E4M3 ? 1 : 0;
  p.out_f32 = cfg->out_dtype == MLA_F32 ? 1 : 0;
  p.partial_f16 = cfg->partial_fp16 ? 1 : 0;
  p.piece_units = piece_units(p.qkv_e4m3 != 0);
  p.fused_combine = cfg->combine_in_kernel;
  p.epoch = next_epoch();
  p.num_clusters = G;
  p.reduce_d_tiles = d_tiles_of(cfg);
  p.scale = scale;
  p.q_descale = cfg->q_descale;
  p.ckv_descale = cfg->ckv_descale;
  p.kpe_descale = cfg->kpe_descale;
  p.score_scale_log2 = scale * cfg->q_descale * cfg->ckv_descale * 1.4426950408889634f;
  return p;
}

mla_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
  }
  return "MLA_ERR_UNKNOWN";
}

mla_status_t mla_plan(const int32_t* seq_lens, int B, int H, int page_size, int window_left, const mla_config_t* cfg,
                      int* split_kv, size_t* workspace_bytes) {
  if (!seq_lens || !split_kv || !workspace_bytes) return MLA_ERR_INVALID_ARG;
  mla_status_t st = validate_cfg(cfg, B, H, page_size, window_left);
  if (st != MLA_OK) return st;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < 0 || (long long)seq_lens[b] > (long long)cfg->page_table_stride * page_size)
      return MLA_ERR_INVALID_ARG;
  int G;
  if (resolve_clusters(cfg, cfg->qkv_dtype == MLA_E4M3, &G) != 0) return MLA_ERR_CUDA;
  *split_kv = plan_max_parts(seq_lens, B, H, page_size, window_left, cfg, G);
  *workspace_bytes = ws_layout(B, cfg->seq_len_q, H, G, cfg->partial_fp16 ? 1 : 0).total;
  return MLA_OK;
}

mla_status_t mla_decode(const void* q_latent, const void* q_rope, const void* ckv_cache, const void* kpe_cache,
                        const int32_t* page_table, const int32_t* seq_lens, float scale, int window_left, void* out,
                        float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream, int B, int H,
                        int page_size, const mla_config_t* cfg) {
  mla_status_t st = validate_cfg(cfg, B, H, page_size, window_left);
  if (st != MLA_OK) return st;
  if (!q_latent || !q_rope || !ckv_cache || !kpe_cache || !page_table || !seq_lens || !out || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (cp_world_of(cfg) > 1 && !cfg->global_seq_lens) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_latent) || !aligned16(q_rope) || !aligned16(ckv_cache) || !aligned16(kpe_cache) ||
      !aligned16(page_table) || !aligned16(seq_lens) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return MLA_ERR_INVALID_ARG;
  const bool e4m3 = cfg->qkv_dtype == MLA_E4M3;
  int G;
  if (resolve_clusters(cfg, e4m3, &G) != 0) return MLA_ERR_CUDA;
  if (workspace_bytes < ws_layout(B, cfg->seq_len_q, H, G, cfg->partial_fp16 ? 1 : 0).total)
    return MLA_ERR_WORKSPACE_TOO_SMALL;

  const DecodeParams p = make_params(q_latent, q_rope, ckv_cache, kpe_cache, page_table, seq_lens, scale, window_left,
                                     out, lse, workspace, B, H, page_size, cfg, G);
  KvMaps maps;
  if (!encode_kv_maps(&maps, ckv_cache, kpe_cache, q_latent, q_rope, e4m3, cfg->num_pages, page_size, B,
                      cfg->seq_len_q * H))
    return MLA_ERR_CUDA;
  const bool timed = cfg->split_timing[0] && cfg->split_timing[1];
  if (timed && cudaEventRecord(static_cast<cudaEvent_t>(cfg->split_timing[0]), stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  cudaError_t e = launch_split_kv(p, maps, stream);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  if (timed && cudaEventRecord(static_cast<cudaEvent_t>(cfg->split_timing[1]), stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (p.fused_combine) return MLA_OK;  // the split-KV kernel combined every row itself
  // the PDL reduction starts its launch while the split-KV kernel drains; it is not used
  // when the split kernel is timed alone (its end event would then come late)
  return cuda_status(launch_reduce(p, stream, cfg->use_pdl != 0 && !timed));
}

mla_status_t mla_merge(const void* o_parts, const float* lse_parts, int world, long long rows, mla_dtype_t dtype,
                       void* out, float* lse, cudaStream_t stream) {
  if (!o_parts || !lse_parts || !out || world < 1 || world > kMaxWorld || rows < 1) return MLA_ERR_INVALID_ARG;
  if (dtype != MLA_F32 && dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_merge(o_parts, lse_parts, world, rows, dtype == MLA_F32 ? 1 : 0, out, lse, stream));
}

mla_status_t mla_debug_gather(const void* ckv_cache, const void* kpe_cache, const int32_t* page_table,
                              const int32_t* seq_lens, int B, int page_size, int max_k, const mla_config_t* cfg,
                              void* dense_out, cudaStream_t stream) {
  mla_status_t st = validate_cfg(cfg, B, 1, page_size, -1);
  if (st != MLA_OK) return st;
  if (!ckv_cache || !kpe_cache || !page_table || !seq_lens || !dense_out || max_k < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned16(ckv_cache) || !aligned16(kpe_cache) || !aligned16(dense_out)) return MLA_ERR_INVALID_ARG;
  const bool e4m3 = cfg->qkv_dtype == MLA_E4M3;
  KvMaps maps;
  if (!encode_kv_maps(&maps, ckv_cache, kpe_cache, nullptr, nullptr, e4m3, cfg->num_pages, page_size, 1, 1))
    return MLA_ERR_CUDA;
  return cuda_status(launch_debug_gather(maps, e4m3, page_table, seq_lens, B, cfg->page_table_stride, cfg->num_pages,
                                         page_size, max_k, dense_out, nullptr, stream));
}

mla_status_t mla_debug_mask(const int32_t* seq_lens, int B, int window_left, int max_k, const mla_config_t* cfg,
                            uint32_t* bits, cudaStream_t stream) {
  mla_status_t st = validate_cfg(cfg, B, 1, kKeyGroup, window_left);
  if (st != MLA_OK) return st;
  if (!seq_lens || !bits || max_k < 1) return MLA_ERR_INVALID_ARG;
  if (cp_world_of(cfg) > 1 && !cfg->global_seq_lens) return MLA_ERR_INVALID_ARG;
  const DecodeParams p = make_params(nullptr, nullptr, nullptr, nullptr, nullptr, seq_lens, 1.f, window_left, nullptr,
                                     nullptr, nullptr, B, 1, kKeyGroup, cfg, 1);
  return cuda_status(launch_debug_mask(p, max_k, bits, stream));
}

mla_status_t mla_debug_wait_timeout(unsigned timeout_us, uint32_t* status_words, cudaStream_t stream) {
  if (!status_words || timeout_us < 1 || timeout_us > 2000000u || !aligned16(status_words)) return MLA_ERR_INVALID_ARG;
  if (launch_debug_wait_timeout(1000ull * timeout_us, status_words, stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  uint32_t words[2] = {0, 0};
  if (cudaMemcpy(words, status_words, sizeof words, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  return (words[0] & kErrTimeout) && (words[1] & kErrTimeout) ? MLA_ERR_TIMEOUT : MLA_OK;
}

mla_status_t mla_workspace_status(const void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!workspace || workspace_bytes < sizeof(WsHeader)) return MLA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, workspace, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (h.num_clusters <= 0 || h.num_rows <= 0) return MLA_ERR_INVALID_ARG;
  // the status words follow the header (the start of every workspace layout)
  const size_t off = align256(sizeof(WsHeader));
  if (workspace_bytes < off + 8 * (size_t)h.num_clusters) return MLA_ERR_INVALID_ARG;
  std::vector<uint32_t> words(2 * (size_t)h.num_clusters);
  if (cudaMemcpy(words.data(), static_cast<const uint8_t*>(workspace) + off, words.size() * 4,
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;
  uint32_t all = 0;
  for (uint32_t w : words) all |= w;
  if (all & kErrTimeout) return MLA_ERR_TIMEOUT;
  if (all & (kErrBadPage | kErrBadLength)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

}  // extern "C"
