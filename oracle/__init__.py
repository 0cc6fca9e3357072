"""fp64 CPU oracle for paged MLA decode.

TEST INFRASTRUCTURE ONLY: the correctness reference for the CUDA path.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import it; the product package never does.  It shares no code with the CUDA
path.  The arithmetic lives in ``mla_oracle.c`` (plain C, fp64, OpenMP over
rows); this module compiles it with gcc on first use and marshals arguments.

Every function follows the kv_balanced_mla kernel page of the vLLM Kimi-K3 MLA
docs (BlackwellMultiHeadLatentAttentionForwardFP8): ``decode`` is the
definition (softmax(q.[c;kpe]^T * scale) . c with a natural-log LSE),
``decode_split`` the page's split-KV tiling (get_k_tile_count) plus its base-2
LSE-weighted combine (reduction_kernel), ``gather`` and ``visibility_bits`` the
page-table walk and the causal / sliding-window visible range.  ``decode_ex``
adds decode context parallelism (``__init__``'s cp_world, cp_rank and
cp_interleave_size, ``__call__``'s causal_seqs) and ``__call__``'s
local_visible_lens; ``merge`` combines the ranks' pieces.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, E4M3 = 0, 1
D_LATENT, D_ROPE = 512, 64


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i, d, i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
            lib.oracle_mla_decode.argtypes = [P, P, P, P, i, d, d, d, P, i, P, i, i, i, i, i, d, i, i, P, i64, i, P, P]
            lib.oracle_mla_decode_ex.argtypes = [P, P, P, P, i, d, d, d, P, i, P, i, i, i, i, i, d, i, i,
                                                 i, i, i, P, P, i, P, P]
            lib.oracle_merge.argtypes = [P, P, i, i64, P, P]
            lib.oracle_mla_decode_split.argtypes = [P, P, P, P, i, d, d, d, P, i, P, i, i, i, i, i, d, i, i, i, i, i, P, P]
            lib.oracle_gather.argtypes = [P, P, i, P, i, P, i, i, i, P]
            lib.oracle_visibility_bits.argtypes = [P, i, i, i, i, i, P]
            lib.oracle_visibility_bits_ex.argtypes = [P, i, i, i, i, i, i, i, P, P, i, P]
            lib.oracle_visible_range.argtypes = [i, i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = d
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_f64.restype = d
            lib.oracle_max_threads.restype = i
            _lib = lib
    return _lib


def _bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits of a CPU tensor (bf16 -> uint16, e4m3 -> uint8)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.uint16).numpy()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    raise TypeError(f"oracle takes bf16 or float8_e4m3fn inputs, got {t.dtype}")


def _dtype_code(t: torch.Tensor) -> int:
    return BF16 if t.dtype == torch.bfloat16 else E4M3


def _i32(t) -> np.ndarray:
    return np.ascontiguousarray(torch.as_tensor(t).to("cpu", torch.int32).numpy())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return _load().oracle_max_threads()


def _common(p: dict):
    ql, qr, ckv, kpe = (_bits(p[k]) for k in ("q_latent", "q_rope", "ckv", "kpe"))
    pt, sl = _i32(p["page_table"]), _i32(p["seq_lens"])
    B, Sq, H = p["q_latent"].shape[:3]
    num_pages, page_size = p["ckv"].shape[:2]
    keep = (ql, qr, ckv, kpe, pt, sl)
    args = [_ptr(ql), _ptr(qr), _ptr(ckv), _ptr(kpe), _dtype_code(p["ckv"]),
            float(p.get("q_descale", 1.0)), float(p.get("ckv_descale", 1.0)), float(p.get("kpe_descale", 1.0)),
            _ptr(pt), pt.shape[1], _ptr(sl), B, Sq, H, page_size, num_pages,
            float(p["scale"]), int(bool(p.get("causal", False))), int(p.get("window_left", -1))]
    return keep, args, (B, Sq, H)


def decode(p: dict, rows=None, threads: int = 0):
    """The definition, for all rows or a list of flat row ids (b*Sq + t)*H + h.

    ``p`` holds CPU tensors q_latent [B,Sq,H,512], q_rope [B,Sq,H,64],
    ckv [pages,P,512], kpe [pages,P,64] (bf16 or float8_e4m3fn), page_table
    [B,stride] and seq_lens [B] (int32), plus scale, causal, window_left and
    the per-tensor descales.  Returns (O [n,512], LSE [n]) as float64 arrays,
    LSE in natural log.
    """
    lib = _load()
    keep, args, (B, Sq, H) = _common(p)
    if rows is None:
        n = B * Sq * H
        rows_arr, rows_ptr = None, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows_arr.shape[0]
        rows_ptr = _ptr(rows_arr)
    O = np.empty((n, D_LATENT), dtype=np.float64)
    L = np.empty((n,), dtype=np.float64)
    lib.oracle_mla_decode(*args, rows_ptr, n, int(threads), _ptr(O), _ptr(L))
    del keep, rows_arr
    return O, L


def decode_ex(p: dict, cp_world: int = 1, cp_rank: int = 0, cp_interleave: int = 1, global_seq_lens=None,
              local_visible_lens=None, threads: int = 0):
    """The definition with decode context parallelism and per-token local bounds, all rows.

    Under context parallelism (cp_world > 1) ``p`` holds one rank's share: its keys in
    position order behind its own page table, ``seq_lens`` counting them, and
    ``global_seq_lens`` [B] the whole sequences' lengths, on which the causal and window
    bounds are taken.  ``local_visible_lens`` [B, Sq], when given, bounds each query
    token's keys by local index (replacing the causal bound).  Returns (O, LSE) of
    this share: merge the ranks' shares with ``merge``.
    """
    lib = _load()
    keep, args, (B, Sq, H) = _common(p)
    gsl = None if global_seq_lens is None else _i32(global_seq_lens)
    lvl = None if local_visible_lens is None else _i32(local_visible_lens).reshape(B, Sq).copy()
    n = B * Sq * H
    O = np.empty((n, D_LATENT), dtype=np.float64)
    L = np.empty((n,), dtype=np.float64)
    rc = lib.oracle_mla_decode_ex(*args, int(cp_world), int(cp_rank), int(cp_interleave),
                                  None if gsl is None else _ptr(gsl), None if lvl is None else _ptr(lvl),
                                  int(threads), _ptr(O), _ptr(L))
    if rc != 0:
        raise ValueError("bad context-parallel arguments")
    del keep, gsl, lvl
    return O, L


def merge(O_parts, L_parts):
    """Combine per-rank (O [rows, 512], LSE [rows]) pieces over disjoint key sets."""
    lib = _load()
    Op = np.ascontiguousarray(np.stack([np.asarray(o, dtype=np.float64) for o in O_parts]))
    Lp = np.ascontiguousarray(np.stack([np.asarray(x, dtype=np.float64) for x in L_parts]))
    world, rows = Lp.shape
    O = np.empty((rows, D_LATENT), dtype=np.float64)
    L = np.empty((rows,), dtype=np.float64)
    lib.oracle_merge(_ptr(Op), _ptr(Lp), int(world), int(rows), _ptr(O), _ptr(L))
    return O, L


def decode_split(p: dict, split_kv: int, tile_n: int, threads: int = 0):
    """The split-KV route: partials per split (get_k_tile_count) + base-2 combine."""
    lib = _load()
    keep, args, (B, Sq, H) = _common(p)
    n = B * Sq * H
    O = np.empty((n, D_LATENT), dtype=np.float64)
    L = np.empty((n,), dtype=np.float64)
    rc = lib.oracle_mla_decode_split(*args, int(split_kv), int(tile_n), int(threads), _ptr(O), _ptr(L))
    if rc != 0:
        raise ValueError("bad split_kv / tile_n")
    del keep
    return O, L


def gather(p: dict, max_k: int) -> np.ndarray:
    """Dense [B, max_k, 576] raw element bits through the page table (zeros past K)."""
    lib = _load()
    ckv, kpe = _bits(p["ckv"]), _bits(p["kpe"])
    pt, sl = _i32(p["page_table"]), _i32(p["seq_lens"])
    B = pt.shape[0]
    out = np.zeros((B, max_k, D_LATENT + D_ROPE), dtype=ckv.dtype)
    lib.oracle_gather(_ptr(ckv), _ptr(kpe), _dtype_code(p["ckv"]), _ptr(pt), pt.shape[1], _ptr(sl), B,
                      p["ckv"].shape[1], max_k, _ptr(out))
    return out


def visibility_bits(seq_lens, Sq: int, causal: bool, window_left: int, max_k: int) -> np.ndarray:
    """[B, Sq, ceil(max_k/32)] uint32 words, bit i of word w = key 32w+i visible."""
    lib = _load()
    sl = _i32(seq_lens)
    B = sl.shape[0]
    out = np.zeros((B, Sq, (max_k + 31) // 32), dtype=np.uint32)
    lib.oracle_visibility_bits(_ptr(sl), B, Sq, int(bool(causal)), int(window_left), max_k, _ptr(out))
    return out


def visibility_bits_ex(seq_lens, Sq: int, causal: bool, window_left: int, max_k: int, cp_world: int = 1,
                       cp_rank: int = 0, cp_interleave: int = 1, global_seq_lens=None,
                       local_visible_lens=None) -> np.ndarray:
    """visibility_bits under decode context parallelism and local bounds (decode_ex's rule)."""
    lib = _load()
    sl = _i32(seq_lens)
    B = sl.shape[0]
    gsl = None if global_seq_lens is None else _i32(global_seq_lens)
    lvl = None if local_visible_lens is None else _i32(local_visible_lens).reshape(B, Sq).copy()
    out = np.zeros((B, Sq, (max_k + 31) // 32), dtype=np.uint32)
    rc = lib.oracle_visibility_bits_ex(_ptr(sl), B, Sq, int(bool(causal)), int(window_left), int(cp_world),
                                       int(cp_rank), int(cp_interleave), None if gsl is None else _ptr(gsl),
                                       None if lvl is None else _ptr(lvl), max_k, _ptr(out))
    if rc != 0:
        raise ValueError("bad context-parallel arguments")
    return out


def visible_range(K: int, Sq: int, t: int, causal: bool, window_left: int):
    lib = _load()
    lo, hi = ctypes.c_int(), ctypes.c_int()
    lib.oracle_visible_range(K, Sq, t, int(bool(causal)), window_left, ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


def e4m3_to_f64(bits: int) -> float:
    return _load().oracle_e4m3_to_f64(bits)
