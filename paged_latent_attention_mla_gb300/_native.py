"""ctypes binding of libmla_gb300.so (include/mla.h): argument marshalling only.

Every step of the decode runs in the library's CUDA kernels; this module turns
torch tensors into pointers and status codes into exceptions.  There is no
fallback: if the library is missing the calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE_TOO_SMALL, MLA_ERR_CUDA, MLA_ERR_TIMEOUT = range(6)
MLA_BF16, MLA_E4M3, MLA_F32 = 0, 1, 2

_DTYPES = {torch.bfloat16: MLA_BF16, torch.float8_e4m3fn: MLA_E4M3, torch.float32: MLA_F32}

EXPORTS = ("mla_plan", "mla_decode", "mla_decode_noalloc", "mla_noalloc_status", "mla_merge", "mla_debug_gather",
           "mla_debug_mask", "mla_debug_wait_timeout", "mla_workspace_status", "mla_status_string")


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


class MlaConfig(ctypes.Structure):
    _fields_ = [
        ("seq_len_q", ctypes.c_int),
        ("num_pages", ctypes.c_int),
        ("page_table_stride", ctypes.c_int),
        ("qkv_dtype", ctypes.c_int),
        ("out_dtype", ctypes.c_int),
        ("causal", ctypes.c_int),
        ("q_descale", ctypes.c_float),
        ("ckv_descale", ctypes.c_float),
        ("kpe_descale", ctypes.c_float),
        ("num_clusters", ctypes.c_int),
        ("split_timing", ctypes.c_void_p * 2),
        ("cp_world", ctypes.c_int),
        ("cp_rank", ctypes.c_int),
        ("cp_interleave", ctypes.c_int),
        ("global_seq_lens", ctypes.c_void_p),
        ("local_visible_lens", ctypes.c_void_p),
        ("partial_fp16", ctypes.c_int),
        ("reducer_d_tiles", ctypes.c_int),
        ("use_pdl", ctypes.c_int),
        ("combine_in_kernel", ctypes.c_int),
    ]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load the library (built in-tree by build()); raises if it is not there."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is not built: run paged_latent_attention_mla_gb300.build.build() first")
            lib = ctypes.CDLL(p)
            P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            cfgp = ctypes.POINTER(MlaConfig)
            lib.mla_plan.argtypes = [P, I, I, I, I, cfgp, ctypes.POINTER(I), ctypes.POINTER(S)]
            lib.mla_decode.argtypes = [P, P, P, P, P, P, F, I, P, P, P, S, P, I, I, I, cfgp]
            lib.mla_decode_noalloc.argtypes = [P, P, P, P, P, P, F, I, P, P, P, I, I, I, cfgp]
            lib.mla_debug_gather.argtypes = [P, P, P, P, I, I, I, cfgp, P, P]
            lib.mla_debug_mask.argtypes = [P, I, I, I, cfgp, P, P]
            lib.mla_debug_wait_timeout.argtypes = [ctypes.c_uint, P, P]
            lib.mla_workspace_status.argtypes = [P, S, P]
            lib.mla_noalloc_status.argtypes = [P]
            lib.mla_merge.argtypes = [P, P, I, ctypes.c_longlong, I, P, P, P]
            lib.mla_status_string.argtypes = [I]
            lib.mla_status_string.restype = ctypes.c_char_p
            for fn in ("mla_plan", "mla_decode", "mla_decode_noalloc", "mla_noalloc_status", "mla_merge",
                       "mla_debug_gather", "mla_debug_mask", "mla_debug_wait_timeout", "mla_workspace_status"):
                getattr(lib, fn).restype = I
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().mla_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != MLA_OK:
        raise MlaError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_config(*, seq_len_q: int, num_pages: int, page_table_stride: int, qkv_dtype, out_dtype=torch.bfloat16,
                causal: bool = False, q_descale: float = 1.0, ckv_descale: float = 1.0, kpe_descale: float = 1.0,
                num_clusters: int = 0, cp_world: int = 1, cp_rank: int = 0, cp_interleave: int = 1,
                partial_fp16: bool = False, reducer_d_tiles: int = 0, use_pdl: bool = False,
                combine_in_kernel: bool = False) -> MlaConfig:
    """The C config; the device pointers global_seq_lens / local_visible_lens are set per call
    (set_call_inputs), since their tensors belong to the call."""
    qd = _DTYPES[qkv_dtype] if isinstance(qkv_dtype, torch.dtype) else int(qkv_dtype)
    od = _DTYPES[out_dtype] if isinstance(out_dtype, torch.dtype) else int(out_dtype)
    c = MlaConfig(int(seq_len_q), int(num_pages), int(page_table_stride), qd, od, int(bool(causal)),
                  float(q_descale), float(ckv_descale), float(kpe_descale), int(num_clusters))
    c.cp_world, c.cp_rank, c.cp_interleave = int(cp_world), int(cp_rank), int(cp_interleave)
    c.partial_fp16, c.reducer_d_tiles, c.use_pdl = int(bool(partial_fp16)), int(reducer_d_tiles), int(bool(use_pdl))
    c.combine_in_kernel = int(bool(combine_in_kernel))
    return c


def set_call_inputs(cfg: MlaConfig, global_seq_lens=None, local_visible_lens=None):
    """Point the config at this call's device tensors (or clear them)."""
    cfg.global_seq_lens = None if global_seq_lens is None else global_seq_lens.data_ptr()
    cfg.local_visible_lens = None if local_visible_lens is None else local_visible_lens.data_ptr()


def mla_plan(seq_lens, B: int, H: int, page_size: int, window_left: int, cfg: MlaConfig):
    """Returns (split_kv, workspace_bytes).  seq_lens: host int32 tensor or list."""
    sl = torch.as_tensor(seq_lens, dtype=torch.int32).cpu().contiguous()
    split = ctypes.c_int()
    ws = ctypes.c_size_t()
    _check("mla_plan", load().mla_plan(_ptr(sl), int(B), int(H), int(page_size), int(window_left), ctypes.byref(cfg),
                                       ctypes.byref(split), ctypes.byref(ws)))
    return split.value, ws.value


def mla_decode(q_latent, q_rope, ckv_cache, kpe_cache, page_table, seq_lens, scale: float, window_left: int, out,
               lse, workspace, cfg: MlaConfig, stream=None):
    B, Sq, H = q_latent.shape[0], q_latent.shape[1], q_latent.shape[2]
    page_size = ckv_cache.shape[1]
    _check("mla_decode", load().mla_decode(
        _ptr(q_latent), _ptr(q_rope), _ptr(ckv_cache), _ptr(kpe_cache), _ptr(page_table), _ptr(seq_lens),
        float(scale), int(window_left), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream), int(B), int(H), int(page_size), ctypes.byref(cfg)))


def mla_decode_noalloc(q_latent, q_rope, ckv_cache, kpe_cache, page_table, seq_lens, scale: float, window_left: int,
                       out, lse, cfg: MlaConfig, stream=None):
    """mla_decode with the library's own fixed scratch array: for callers that must not allocate."""
    B, H = q_latent.shape[0], q_latent.shape[2]
    _check("mla_decode_noalloc", load().mla_decode_noalloc(
        _ptr(q_latent), _ptr(q_rope), _ptr(ckv_cache), _ptr(kpe_cache), _ptr(page_table), _ptr(seq_lens),
        float(scale), int(window_left), _ptr(out), _ptr(lse), _stream(stream), int(B), int(H),
        int(ckv_cache.shape[1]), ctypes.byref(cfg)))


def mla_merge(o_parts, lse_parts, out, lse=None, stream=None):
    """Combine per-rank shares: o_parts [world, rows, 512] (fp32 or bf16), lse_parts [world, rows] fp32."""
    world = o_parts.shape[0]
    rows = o_parts.numel() // (world * 512)
    _check("mla_merge", load().mla_merge(_ptr(o_parts), _ptr(lse_parts), int(world), int(rows),
                                         _DTYPES[o_parts.dtype], _ptr(out), _ptr(lse), _stream(stream)))


def mla_noalloc_status(stream=None) -> int:
    """Device-side status of the last mla_decode_noalloc on the current device (synchronizes)."""
    return load().mla_noalloc_status(_stream(stream))


def mla_debug_gather(ckv_cache, kpe_cache, page_table, seq_lens, max_k: int, dense_out, cfg: MlaConfig, stream=None):
    B = page_table.shape[0]
    _check("mla_debug_gather", load().mla_debug_gather(
        _ptr(ckv_cache), _ptr(kpe_cache), _ptr(page_table), _ptr(seq_lens), int(B), int(ckv_cache.shape[1]),
        int(max_k), ctypes.byref(cfg), _ptr(dense_out), _stream(stream)))


def mla_debug_mask(seq_lens, window_left: int, max_k: int, bits, cfg: MlaConfig, stream=None):
    B = seq_lens.shape[0]
    _check("mla_debug_mask", load().mla_debug_mask(_ptr(seq_lens), int(B), int(window_left), int(max_k),
                                                   ctypes.byref(cfg), _ptr(bits), _stream(stream)))


def mla_debug_wait_timeout(timeout_us: int, status_words, stream=None):
    """Raises MlaError(MLA_ERR_TIMEOUT) when the device wait gave up, as it should."""
    _check("mla_debug_wait_timeout", load().mla_debug_wait_timeout(ctypes.c_uint(int(timeout_us)), _ptr(status_words),
                                                                   _stream(stream)))


def mla_workspace_status(workspace, stream=None) -> int:
    return load().mla_workspace_status(_ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))


def mla_status_string(status: int) -> str:
    return status_string(status)
