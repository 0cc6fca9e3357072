/*
 * Paged Multi-Head Latent Attention (MLA) decode for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libmla_gb300.so.  The operation is the one the vLLM Kimi-K3
 * kv_balanced_mla kernel page describes (BlackwellMultiHeadLatentAttentionForwardFP8,
 * __call__ docstring and reduction_kernel): for every request b, query token
 * t < seq_len_q and head h < H,
 *
 *   s_j = scale * (q_latent[b,t,h,:] . c_j + q_rope[b,t,h,:] . kpe_j)
 *   out[b,t,h,:] = sum_j softmax(s)_j * c_j        (V is the latent c itself)
 *   lse[b,t,h]   = log(sum_j exp(s_j))              (natural log)
 *
 * over the visible keys j of request b, fetched through the page table:
 * key j lives in page page_table[b][j / page_size], slot j % page_size.
 * Visible keys of token t (K = seq_lens[b], which counts the seq_len_q new
 * tokens): j < K - (seq_len_q - 1 - t) when causal, else j < K (the softmax
 * K bound); and j >= K - seq_len_q - window_left + t when window_left >= 0
 * (the window_left docstring of __init__).  A row with no visible key gets
 * out = 0 and lse = -inf (write_empty_output).
 *
 * Work is split along the KV axis across the GPU.  A row cut into several pieces
 * has each piece write a normalized partial output and its base-2 log-sum-exp
 * into the caller's workspace, and a reduction combines them with weights
 * 2^(lse_i - lse) (reduction_kernel): a second kernel, or the split kernel
 * itself with combine_in_kernel.  A row in one piece is written directly.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless marked host.  The caller owns every
 *    buffer and the stream; the library allocates nothing and never
 *    synchronizes the stream on the decode path.
 *  - Errors are return codes.  Arguments are validated before anything is
 *    launched; on any error nothing is launched and no output is touched.
 *  - Tensors are dense and contiguous in the shapes given, and every pointer
 *    is 16-byte aligned.
 *  - Asynchronous CUDA faults surface as MLA_ERR_CUDA from a later call.
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,         /* a NULL / misaligned pointer, a bad size or shape */
  MLA_ERR_UNSUPPORTED = 2,         /* valid, but outside what the library implements */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < what mla_plan reported */
  MLA_ERR_CUDA = 4,                /* a CUDA runtime call failed (launch or an earlier fault) */
  MLA_ERR_TIMEOUT = 5              /* a bounded device wait gave up (read by mla_workspace_status) */
} mla_status_t;

typedef enum { MLA_BF16 = 0, MLA_E4M3 = 1, MLA_F32 = 2 } mla_dtype_t;

/*
 * Tensor metadata the decode call needs beyond its pointers.  A zero-initialized
 * struct with the first six fields and the descales set is a plain decode.
 *  seq_len_q          query tokens per request (1 = plain decode; >1 = speculative block)
 *  num_pages          pages in the cache pool (first dim of ckv / kpe)
 *  page_table_stride  int32 entries per request row of page_table (its second dim)
 *  qkv_dtype          MLA_BF16, or MLA_E4M3 (float8 e4m3fn) for q, ckv and kpe together
 *  out_dtype          MLA_F32 or MLA_BF16 for out; lse is always fp32
 *  causal             1: token t sees keys before K - (seq_len_q - 1 - t)
 *  q_descale ...      per-tensor fp32 scales of the e4m3 inputs (value = code * descale);
 *                     must be 1 for bf16 inputs.  The latent and rope parts of a key
 *                     feed one contraction, so kpe_descale must equal ckv_descale
 *                     (MLA_ERR_UNSUPPORTED otherwise): one scale for the key cache.
 *  num_clusters       0: one persistent wave sized from the device (default);
 *                     >0: use this many 2-CTA clusters (testing and partitioning)
 *  split_timing       optional pair of cudaEvent_t handles (caller-owned, already
 *                     created): when both are non-NULL, mla_decode records [0] just
 *                     before and [1] just after the split-KV kernel on the call's
 *                     stream, so the kernel can be timed alone; NULL: nothing recorded
 *
 * Decode context parallelism (the kv_balanced_mla kernel page: __init__'s cp_world,
 * cp_rank, cp_interleave_size and __call__'s causal_seqs).  Every sequence's key
 * positions are dealt to cp_world ranks in runs of cp_interleave consecutive
 * positions, run k to rank k % cp_world.  Each rank's cache and page table hold its
 * own keys in position order and its seq_lens count them; the causal and window
 * bounds are taken on the whole sequence, whose lengths global_seq_lens gives.  Each
 * rank's decode then yields its share (O, LSE) of every row, and mla_merge combines
 * the ranks' shares into the whole decode.
 *  cp_world           0 or 1: no context parallelism
 *  cp_rank            this rank, 0 <= cp_rank < cp_world
 *  cp_interleave      positions per run (0 is taken as 1)
 *  global_seq_lens    device [B] int32, the whole sequences' lengths; required when
 *                     cp_world > 1, ignored otherwise
 *
 *  local_visible_lens device [B, seq_len_q] int32 or NULL (__call__'s local_visible_lens):
 *                     query token t of request b sees local keys below this bound (and
 *                     above the window floor, when a window is set); it replaces the causal
 *                     bound.  NULL: the causal flag decides.
 *  partial_fp16       1: store the split pieces' normalized partial outputs as fp16
 *                     (__init__'s partial_fp16) instead of fp32: half the bytes written by
 *                     the split-KV kernel and read by the reduction.  Each (row, half of
 *                     the dims) is scaled by a power of two that puts its largest |value|
 *                     in [2^14, 2^15), so any finite value fits (fp16's 11 significant bits
 *                     each, in a sum rounded to the output type afterwards).
 *  reducer_d_tiles    CTAs per work row across the 512 output dims in the reduction:
 *                     1, 2, 4 or 8 (0: 8)
 *  use_pdl            1: launch the reduction with programmatic dependent launch, so its
 *                     launch overlaps the split-KV kernel's end (not with split_timing)
 *  combine_in_kernel  0 (default): a separate reduction kernel combines the pieces of a row
 *                     cut into several (reducer_d_tiles, use_pdl); 1: the split-KV kernel
 *                     combines them, the last piece of a row to finish counting its arrival
 *                     in the workspace, and mla_decode launches one kernel
 */
typedef struct {
  int seq_len_q;
  int num_pages;
  int page_table_stride;
  mla_dtype_t qkv_dtype;
  mla_dtype_t out_dtype;
  int causal;
  float q_descale;
  float ckv_descale;
  float kpe_descale;
  int num_clusters;
  void* split_timing[2];
  int cp_world;
  int cp_rank;
  int cp_interleave;
  const int32_t* global_seq_lens;
  const int32_t* local_visible_lens;
  int partial_fp16;
  int reducer_d_tiles;
  int use_pdl;
  int combine_in_kernel;
} mla_config_t;

/*
 * Plan a decode batch (host only; reads the host copy of seq_lens).
 *
 * A request's seq_len_q * H (token, head) rows are cut into M tiles of 128 rows
 * ("work rows"; consecutive tokens share a tile when H < 128, the page's pack_q).
 * The KV range of every work row is cut into tiles of 256 keys; the visible
 * tiles of all requests are laid end to end and dealt out in equal contiguous
 * shares to a persistent wave of clusters, so unequal lengths balance (the page's
 * get_split_kv / get_k_tile_count plan the same split per request; this plan splits
 * the whole batch at once), with a request's work rows given to side-by-side
 * clusters that read its KV together.  Tiles wholly outside every row's window are
 * skipped.
 *
 *  seq_lens        host [B] int32, 0 <= seq_lens[b] <= page_table_stride * page_size
 *  B, H            requests and heads, 1 <= H <= 128, B * seq_len_q <= 16384
 *  page_size       keys per page: a power of two from 8 to 1024
 *  window_left     -1 for full history, else >= 0
 *  cfg             tensor metadata as above
 *  split_kv        out: the most pieces any work row is cut into (1 = no reduction
 *                  needed); with context parallelism or local_visible_lens, whose
 *                  device values the host does not see, an estimate that takes every
 *                  local key as visible
 *  workspace_bytes out: device workspace mla_decode needs; it depends on B, H,
 *                  seq_len_q, the cluster count and partial_fp16 only, not on the lengths
 *
 * Returns MLA_ERR_CUDA when cfg->num_clusters == 0 and no device can be queried.
 */
MLA_API mla_status_t mla_plan(const int32_t *seq_lens, int B, int H, int page_size, int window_left, const mla_config_t *cfg,
                      int *split_kv, size_t *workspace_bytes);

/*
 * Decode: out = softmax(q.[c;kpe]^T * scale).c and lse, for all B * seq_len_q * H rows.
 *
 *  q_latent   [B, seq_len_q, H, 512]   qkv_dtype
 *  q_rope     [B, seq_len_q, H, 64]    qkv_dtype
 *  ckv_cache  [num_pages, page_size, 512] qkv_dtype  (latent c, also the value)
 *  kpe_cache  [num_pages, page_size, 64]  qkv_dtype  (rope key)
 *  page_table [B, page_table_stride] int32; entries [0, ceil(seq_lens[b]/page_size))
 *             must be page ids in [0, num_pages); later entries are never read
 *  seq_lens   [B] int32, device copy of the lengths given to mla_plan
 *  scale      softmax scale (e.g. 1/sqrt(576))
 *  window_left -1, or the sliding-window span (same value as given to mla_plan)
 *  out        [B, seq_len_q, H, 512] out_dtype
 *  lse        [B, seq_len_q, H] fp32 natural-log LSE, or NULL to skip it
 *  workspace  device scratch of at least the planned size, 256-byte aligned.  With
 *             combine_in_kernel, zero it once after allocating it (the rows' arrival
 *             counters must start at zero or hold an earlier call's tag); it needs no
 *             clearing otherwise, nor between calls
 *  stream     the CUDA stream all work is enqueued on
 *
 * Cache slots past a request's length and pages no visible key uses may hold
 * any bits (NaN included) without affecting the result.
 *
 * Conditions only the device sees (a visible page id outside the pool, a device
 * seq_lens value outside [0, page_table_stride * page_size], a bounded wait that
 * gave up) do not change this return value: read them with mla_workspace_status.
 */
MLA_API mla_status_t mla_decode(const void *q_latent, const void *q_rope, const void *ckv_cache, const void *kpe_cache,
                        const int32_t *page_table, const int32_t *seq_lens, float scale, int window_left, void *out,
                        float *lse, void *workspace, size_t workspace_bytes, cudaStream_t stream, int B, int H,
                        int page_size, const mla_config_t *cfg);

/*
 * Decode without allocation: mla_decode with its scratch in a fixed array
 * inside this library instead of a caller-provided workspace.  The pages this
 * library follows have no counterpart of this call; it exists for callers that
 * must not allocate device memory at all (code running under a runtime that
 * owns all device memory once it serves, plugins given no allocator, paths that
 * cannot afford an allocation's implicit synchronization).
 *
 * Same arguments and results as mla_decode, minus workspace and its size.
 * The array is 64 MiB on every GPU that loads the library, held until the
 * process exits; a batch needing more (see mla_plan's workspace_bytes) returns
 * MLA_ERR_WORKSPACE_TOO_SMALL and launches nothing.  The first call on a device
 * looks the array's address up, so make it before any stream capture; the
 * address is cached for the life of the device context (after cudaDeviceReset
 * reload the library).  All calls share the one array: calls that overlap on
 * the GPU race (serialize them, e.g. on one stream).  Nothing in it needs
 * clearing between calls.  Device-side errors of a call (see mla_decode) are
 * read with mla_noalloc_status; the output of a call that reports one is
 * incomplete.
 */
MLA_API mla_status_t mla_decode_noalloc(const void *q_latent, const void *q_rope, const void *ckv_cache,
                                        const void *kpe_cache, const int32_t *page_table, const int32_t *seq_lens,
                                        float scale, int window_left, void *out, float *lse, cudaStream_t stream,
                                        int B, int H, int page_size, const mla_config_t *cfg);

/*
 * Device-side status of the last mla_decode_noalloc on the current device: what
 * mla_workspace_status reports for a workspace, read from the library's own
 * array.  Synchronizes the stream.  Not for the decode path.
 */
MLA_API mla_status_t mla_noalloc_status(cudaStream_t stream);

/*
 * Combine the ranks' shares of a context-parallel decode (see mla_config_t):
 *  o_parts   [world, rows, 512] in dtype (MLA_F32 or MLA_BF16), rank r's output
 *  lse_parts [world, rows] fp32 natural-log LSEs (-inf: the rank saw no visible key)
 *  out       [rows, 512] in dtype;  lse [rows] fp32 or NULL
 * lse = m + ln(sum_r e^(lse_r - m)), out = sum_r e^(lse_r - lse) o_r (the same combine
 * as the split-KV reduction, reduction_kernel); rows with no visible key on any rank
 * get out = 0 and lse = -inf.  rows = B * seq_len_q * H for a decode's outputs.  The
 * exchange of the shares between ranks is the caller's (an all-gather).
 */
MLA_API mla_status_t mla_merge(const void *o_parts, const float *lse_parts, int world, long long rows,
                               mla_dtype_t dtype, void *out, float *lse, cudaStream_t stream);

/*
 * Debug gather: the decode kernel's page walk and tile load, written back densely.
 *  dense_out [B, max_k, 576] elements of qkv_dtype: row j of request b is
 *  (c_j | kpe_j) for j < seq_lens[b] and zero bytes for j >= seq_lens[b].
 * Byte-for-byte equal to a host gather through the page table.
 */
MLA_API mla_status_t mla_debug_gather(const void *ckv_cache, const void *kpe_cache, const int32_t *page_table,
                              const int32_t *seq_lens, int B, int page_size, int max_k, const mla_config_t *cfg,
                              void *dense_out, cudaStream_t stream);

/*
 * Debug mask: the decode kernel's visibility rule, one bit per key (with the
 * context-parallel lengths and local bounds of cfg when set).
 *  bits [B, seq_len_q, ceil(max_k/32)] uint32: bit i of word w is set iff key
 *  32*w + i is visible to that (request, token) row.
 */
MLA_API mla_status_t mla_debug_mask(const int32_t *seq_lens, int B, int window_left, int max_k, const mla_config_t *cfg,
                            uint32_t *bits, cudaStream_t stream);

/*
 * Debug check of the bounded device waits: launches one 2-CTA cluster that allocates
 * tensor memory and waits on an mbarrier nothing arrives at, giving up after
 * timeout_us microseconds (1 .. 2000000) the way every wait of the decode kernel
 * gives up after 2 s: it records a timeout bit, meets its peer, frees the tensor
 * memory and writes a status word per CTA to status_words (device, 2 x uint32,
 * caller-owned) instead of hanging or faulting.  Synchronizes the stream and returns
 * MLA_ERR_TIMEOUT when both words report the timeout, MLA_OK if a wait did not time
 * out, MLA_ERR_INVALID_ARG for a bad argument.  Not for the decode path.
 */
MLA_API mla_status_t mla_debug_wait_timeout(unsigned timeout_us, uint32_t *status_words, cudaStream_t stream);

/*
 * Device-side status of the last mla_decode on this workspace: synchronizes the
 * stream and reads the status words the decode kernel left there.
 *   MLA_OK               nothing went wrong on the device
 *   MLA_ERR_TIMEOUT      a bounded device wait gave up (the kernel unwound instead of hanging)
 *   MLA_ERR_INVALID_ARG  a visible page-table entry outside [0, num_pages) (read as zeros),
 *                        or a device seq_lens value outside [0, page_table_stride * page_size)
 *                        (clamped into it)
 * mla_decode cannot see these conditions (it returns once the kernels are
 * enqueued); the output of a call that reports one is incomplete.  Not for the
 * decode path.
 */
MLA_API mla_status_t mla_workspace_status(const void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Static string naming a status code. */
MLA_API const char *mla_status_string(mla_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
