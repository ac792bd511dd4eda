"""ctypes shim over the CPU oracle (``ep_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports, links or runs anything in this folder.

The shim only marshals numpy arrays; every step of the arithmetic is in the C
file.  The shared object is built from source with gcc on first use (or by
``build_oracle()``), with ``-ffp-contract=off`` so no multiply-add is fused
unless the C code asks for it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "ep_oracle.c")
_SRC_MT = os.path.join(_DIR, "ep_oracle_mt.c")
_LIB = os.path.join(_DIR, "libep_oracle.so")

OK, ERR_INVALID_ARG, ERR_EXPERT_RANGE, ERR_DUP_EXPERT, ERR_CAPACITY = range(5)


def build_oracle(force: bool = False) -> str:
    """Compile ``ep_oracle.c`` (and its multi-threaded driver
    ``ep_oracle_mt.c``) into ``libep_oracle.so`` next to them."""
    srcs = [_SRC, _SRC_MT, os.path.join(_DIR, "ep_oracle.h")]
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(f) for f in srcs
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra", "-o", tmp, _SRC, _SRC_MT,
             "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build_oracle())
        _declare(_lib)
    return _lib


_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


def _declare(L):
    L.oracle_bf16_to_f32.restype = ctypes.c_float
    L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_e4m3_to_f32.restype = ctypes.c_float
    L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    for name in ("oracle_f32_to_bf16_n", "oracle_bf16_to_f32_n",
                 "oracle_f32_to_e4m3_n", "oracle_e4m3_to_f32_n"):
        getattr(L, name).restype = None
        getattr(L, name).argtypes = [_i64, _p, _p]
    L.oracle_recv_capacity.restype = _i64
    L.oracle_recv_capacity.argtypes = [_i32, _i32, _i32, _i32]
    L.oracle_layout.restype = ctypes.c_int
    L.oracle_layout.argtypes = [_i32, _i32, _i32, _i32, _i32, _p, _i64] + [_p] * 8
    L.oracle_dispatch_bf16.restype = None
    L.oracle_dispatch_bf16.argtypes = [_i32, _i32, _i32, _i32, _p, _p, _p, _p, _p,
                                       ctypes.c_int, _p, _p]
    L.oracle_dispatch_fp8.restype = None
    L.oracle_dispatch_fp8.argtypes = [_i32, _i32, _i32, _i32, _p, _p, _p, _p, _p,
                                      ctypes.c_int, _p, _p, _p]
    L.oracle_combine.restype = None
    L.oracle_combine.argtypes = [_i32, _i32, _i32, _p, _p, _p, _p]
    L.oracle_dispatch_bf16_mt.restype = ctypes.c_int
    L.oracle_dispatch_bf16_mt.argtypes = [_i32, _i32, _i32, _i32, _p, _p, _p, _p, _p,
                                          ctypes.c_int, _p, _p, _i32]
    L.oracle_dispatch_fp8_mt.restype = ctypes.c_int
    L.oracle_dispatch_fp8_mt.argtypes = [_i32, _i32, _i32, _i32, _p, _p, _p, _p, _p,
                                         ctypes.c_int, _p, _p, _p, _i32]
    L.oracle_combine_mt.restype = ctypes.c_int
    L.oracle_combine_mt.argtypes = [_i32, _i32, _i32, _p, _p, _p, _p, _i32]
    L.oracle_combine_epilogue.restype = None
    L.oracle_combine_epilogue.argtypes = [_i32, _i32, _i32] + [_p] * 8
    L.oracle_dispatch_backward.restype = None
    L.oracle_dispatch_backward.argtypes = [_i32, _i32, _i32] + [_p] * 5
    L.oracle_combine_backward.restype = None
    L.oracle_combine_backward.argtypes = [_i32, _i32, _i32] + [_p] * 6
    L.oracle_rank_layout.restype = None
    L.oracle_rank_layout.argtypes = [_i32, _i32, _p, _p, _p, _p]
    L.oracle_dispatch_ranks.restype = None
    L.oracle_dispatch_ranks.argtypes = [_i32] * 5 + [_p] * 7
    L.oracle_expand.restype = None
    L.oracle_expand.argtypes = [_i32] * 5 + [_p] * 7
    L.oracle_reduce_ranks.restype = None
    L.oracle_reduce_ranks.argtypes = [_i32] * 5 + [_p] * 6
    L.oracle_combine_ranks.restype = None
    L.oracle_combine_ranks.argtypes = [_i32] * 3 + [_p] * 3
    L.oracle_scale_ld.restype = _i64
    L.oracle_scale_ld.argtypes = [_i64]
    L.oracle_scales_to_col_major.restype = None
    L.oracle_scales_to_col_major.argtypes = [_i64, _i32, _p, _i64, _p]
    L.oracle_dispatch_fp8_prequant.restype = None
    L.oracle_dispatch_fp8_prequant.argtypes = [_i32, _i32, _i32, _i32] + [_p] * 6 + \
        [ctypes.c_int, _p, _p, _p]


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar codecs (vectorised by looping in Python: small inputs only) ----

def bf16_to_f32(h) -> float:
    return lib().oracle_bf16_to_f32(int(h))


def f32_to_bf16(f) -> int:
    return lib().oracle_f32_to_bf16(float(np.float32(f)))


def e4m3_to_f32(c) -> float:
    return lib().oracle_e4m3_to_f32(int(c))


def f32_to_e4m3(v) -> int:
    return lib().oracle_f32_to_e4m3(float(np.float32(v)))


def _map(fn, a, in_dtype, out_dtype):
    a = _c(a, in_dtype)
    out = np.empty(a.shape, out_dtype)
    getattr(lib(), fn)(a.size, _ptr(a), _ptr(out))
    return out


def f32_to_bf16_array(a) -> np.ndarray:
    return _map("oracle_f32_to_bf16_n", a, np.float32, np.uint16)


def bf16_to_f32_array(a) -> np.ndarray:
    return _map("oracle_bf16_to_f32_n", a, np.uint16, np.float32)


def f32_to_e4m3_array(a) -> np.ndarray:
    return _map("oracle_f32_to_e4m3_n", a, np.float32, np.uint8)


def e4m3_to_f32_array(a) -> np.ndarray:
    return _map("oracle_e4m3_to_f32_n", a, np.uint8, np.float32)


# ---- method -----------------------------------------------------------------

def recv_capacity(max_tokens, num_topk, num_experts, alignment) -> int:
    return int(lib().oracle_recv_capacity(max_tokens, num_topk, num_experts, alignment))


def layout(topk_idx: np.ndarray, num_experts: int, num_ranks: int,
           alignment: int, cap: Optional[int] = None) -> dict:
    """Layout from the definition.  Returns a dict of numpy arrays + status."""
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    E, R, A = num_experts, num_ranks, alignment
    if cap is None:
        cap = recv_capacity(T, K, E, A)
    out = dict(
        expert_count=np.zeros(E, np.int32),
        expert_start=np.zeros(E + 1, np.int32),
        expert_end=np.zeros(E, np.int32),
        rank_start=np.zeros(R + 1, np.int32),
        tokens_per_rank=np.zeros(R, np.int32),
        is_token_in_rank=np.zeros((T, R), np.uint8),
        slot_of=np.zeros((T, K), np.int32),
        src_info=np.zeros((cap, 2), np.int32),
    )
    st = lib().oracle_layout(
        T, K, E, R, A, _ptr(idx), cap,
        _ptr(out["expert_count"]), _ptr(out["expert_start"]), _ptr(out["expert_end"]),
        _ptr(out["rank_start"]), _ptr(out["tokens_per_rank"]),
        _ptr(out["is_token_in_rank"]), _ptr(out["slot_of"]), _ptr(out["src_info"]))
    out["status"] = int(st)
    out["cap"] = cap
    return out


def dispatch_bf16(x, topk_weights, lay: dict, zero_padding=False, fill=0xFFFF,
                  out=None, nthreads=1):
    """Expanded bf16 dispatch; rows the method does not write keep ``fill``
    (or their previous contents when ``out=(recv_x, recv_w)`` is given).
    nthreads > 1 runs the same function on token slices in that many threads
    (identical result)."""
    x = _c(x, np.uint16)
    T, H = x.shape
    slot_of = _c(lay["slot_of"], np.int32)
    K = slot_of.shape[1]
    E = lay["expert_count"].shape[0]
    cap = lay["cap"]
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    if out is not None:
        recv_x, recv_w = out
        assert recv_x.shape == (cap, H) and recv_x.dtype == np.uint16
        assert recv_w.shape == (cap,) and recv_w.dtype == np.float32
    else:
        recv_x = np.full((cap, H), fill, np.uint16)
        recv_w = np.full(cap, np.nan, np.float32)
    args = (T, H, K, E, _ptr(x), _ptr(w), _ptr(slot_of),
            _ptr(_c(lay["expert_start"], np.int32)), _ptr(_c(lay["expert_end"], np.int32)),
            int(bool(zero_padding)), _ptr(recv_x), _ptr(recv_w))
    if nthreads > 1:
        lib().oracle_dispatch_bf16_mt(*args, int(nthreads))
    else:
        lib().oracle_dispatch_bf16(*args)
    return recv_x, recv_w


def dispatch_fp8(x, topk_weights, lay: dict, zero_padding=False, fill=0xFF, out=None,
                 nthreads=1):
    """Expanded dispatch with fused 1x128 E4M3 quantisation (``out=(recv_q,
    recv_scale, recv_w)`` writes into given arrays; nthreads as in
    dispatch_bf16)."""
    x = _c(x, np.uint16)
    T, H = x.shape
    slot_of = _c(lay["slot_of"], np.int32)
    K = slot_of.shape[1]
    E = lay["expert_count"].shape[0]
    cap = lay["cap"]
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    if out is not None:
        recv_q, recv_scale, recv_w = out
        assert recv_q.shape == (cap, H) and recv_q.dtype == np.uint8
        assert recv_scale.shape == (cap, H // 128) and recv_scale.dtype == np.float32
        assert recv_w.shape == (cap,) and recv_w.dtype == np.float32
    else:
        recv_q = np.full((cap, H), fill, np.uint8)
        recv_scale = np.full((cap, H // 128), np.nan, np.float32)
        recv_w = np.full(cap, np.nan, np.float32)
    args = (T, H, K, E, _ptr(x), _ptr(w), _ptr(slot_of),
            _ptr(_c(lay["expert_start"], np.int32)), _ptr(_c(lay["expert_end"], np.int32)),
            int(bool(zero_padding)), _ptr(recv_q), _ptr(recv_scale), _ptr(recv_w))
    if nthreads > 1:
        lib().oracle_dispatch_fp8_mt(*args, int(nthreads))
    else:
        lib().oracle_dispatch_fp8(*args)
    return recv_q, recv_scale, recv_w


def combine(expert_out, topk_weights, slot_of, out=None, nthreads=1) -> np.ndarray:
    """Combine from the definition: returns y (uint16 bf16 bits [T, H]);
    nthreads as in dispatch_bf16."""
    Y = _c(expert_out, np.uint16)
    H = Y.shape[1]
    slot_of = _c(slot_of, np.int32)
    T, K = slot_of.shape
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    if out is not None:
        y = out
        assert y.shape == (T, H) and y.dtype == np.uint16
    else:
        y = np.zeros((T, H), np.uint16)
    if nthreads > 1:
        lib().oracle_combine_mt(T, H, K, _ptr(Y), _ptr(w), _ptr(slot_of), _ptr(y),
                                int(nthreads))
    else:
        lib().oracle_combine(T, H, K, _ptr(Y), _ptr(w), _ptr(slot_of), _ptr(y))
    return y


def combine_tokens(expert_out, topk_weights, slot_of, tokens) -> np.ndarray:
    """Combine for a sample of tokens only: the oracle's own definition applied
    to the rows those tokens select, so that it can be checked at full size."""
    tokens = np.asarray(tokens, dtype=np.int64)
    so = np.asarray(slot_of)[tokens]
    used = so >= 0
    rows = so[used]
    sub = np.full(so.shape, -1, np.int32)
    sub[used] = np.arange(rows.size, dtype=np.int32)
    Ysub = np.asarray(expert_out)[rows] if rows.size else np.zeros((0, np.asarray(expert_out).shape[1]), np.uint16)
    w = None if topk_weights is None else np.asarray(topk_weights)[tokens]
    if rows.size == 0:
        Ysub = np.zeros((1, np.asarray(expert_out).shape[1]), np.uint16)
    return combine(Ysub, w, sub)


def combine_epilogue(expert_out, topk_weights, slot_of, bias0=None, bias1=None,
                     recv_w=None):
    """Combine with the epilogue: bias terms after the fold, and the gate
    weights gathered back per (t, k).  Returns (y, combined_w or None)."""
    Y = _c(expert_out, np.uint16)
    H = Y.shape[1]
    slot_of = _c(slot_of, np.int32)
    T, K = slot_of.shape
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    b0 = None if bias0 is None else _c(bias0, np.uint16)
    b1 = None if bias1 is None else _c(bias1, np.uint16)
    rw = None if recv_w is None else _c(recv_w, np.float32)
    y = np.zeros((T, H), np.uint16)
    cw = None if rw is None else np.zeros((T, K), np.float32)
    lib().oracle_combine_epilogue(T, H, K, _ptr(Y), _ptr(w), _ptr(slot_of), _ptr(b0),
                                  _ptr(b1), _ptr(rw), _ptr(y), _ptr(cw))
    return y, cw


def scale_ld(cap: int) -> int:
    return int(lib().oracle_scale_ld(cap))


def scales_to_col_major(row_major, fill=np.nan):
    rm = _c(row_major, np.float32)
    cap, nb = rm.shape
    ld = scale_ld(cap)
    col = np.full((nb, ld), fill, np.float32)
    lib().oracle_scales_to_col_major(cap, nb, _ptr(rm), ld, _ptr(col))
    return col


def dispatch_fp8_prequant(x_q, x_scale, topk_weights, lay: dict, zero_padding=False,
                          fill=0xFF):
    """Expanded dispatch of pre-quantised FP8 rows and their scales."""
    xq = _c(x_q, np.uint8)
    xs = _c(x_scale, np.float32)
    T, H = xq.shape
    slot_of = _c(lay["slot_of"], np.int32)
    K = slot_of.shape[1]
    E = lay["expert_count"].shape[0]
    cap = lay["cap"]
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    recv_q = np.full((cap, H), fill, np.uint8)
    recv_scale = np.full((cap, H // 128), np.nan, np.float32)
    recv_w = np.full(cap, np.nan, np.float32)
    lib().oracle_dispatch_fp8_prequant(T, H, K, E, _ptr(xq), _ptr(xs), _ptr(w),
                                       _ptr(slot_of),
                                       _ptr(_c(lay["expert_start"], np.int32)),
                                       _ptr(_c(lay["expert_end"], np.int32)),
                                       int(bool(zero_padding)), _ptr(recv_q),
                                       _ptr(recv_scale), _ptr(recv_w))
    return recv_q, recv_scale, recv_w


def dispatch_backward(grad_recv, slot_of, grad_recv_w=None):
    """Transpose of dispatch: (grad_x [T,H] bf16 bits, grad_w [T,K] or None)."""
    G = _c(grad_recv, np.uint16)
    H = G.shape[1]
    slot_of = _c(slot_of, np.int32)
    T, K = slot_of.shape
    gw_in = None if grad_recv_w is None else _c(grad_recv_w, np.float32)
    gx = np.zeros((T, H), np.uint16)
    gw = None if gw_in is None else np.zeros((T, K), np.float32)
    lib().oracle_dispatch_backward(T, H, K, _ptr(G), _ptr(gw_in), _ptr(slot_of),
                                   _ptr(gx), _ptr(gw))
    return gx, gw


def combine_backward(dy, topk_weights, slot_of, cap, expert_out=None,
                     want_grad_w=True, fill=0xFFFF):
    """Combine backward: (grad_Y [cap,H] bf16 bits -- unwritten rows keep
    `fill` --, grad_w [T,K] fp32 or None)."""
    D = _c(dy, np.uint16)
    T, H = D.shape
    slot_of = _c(slot_of, np.int32)
    K = slot_of.shape[1]
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    Y = None if expert_out is None else _c(expert_out, np.uint16)
    gY = np.full((cap, H), fill, np.uint16)
    gw = np.zeros((T, K), np.float32) if want_grad_w else None
    lib().oracle_combine_backward(T, H, K, _ptr(D), _ptr(w), _ptr(slot_of), _ptr(Y),
                                  _ptr(gY), _ptr(gw))
    return gY, gw


# ---- non-expanded (destination-major) stage -----------------------------------

def rank_layout(lay: dict) -> dict:
    """Rank rows from the layout's per-rank flags."""
    itr = _c(lay["is_token_in_rank"], np.uint8)
    T, R = itr.shape
    out = dict(rank_row_start=np.zeros(R + 1, np.int32),
               rank_slot_of=np.zeros((T, R), np.int32),
               rank_src=np.full(max(T * R, 1), -1, np.int32))
    lib().oracle_rank_layout(T, R, _ptr(itr), _ptr(out["rank_row_start"]),
                             _ptr(out["rank_slot_of"]), _ptr(out["rank_src"]))
    out["rows"] = int(out["rank_row_start"][-1])
    return out


def dispatch_ranks(x, topk_idx, topk_weights, rl: dict, num_experts, fill=0xFFFF):
    x = _c(x, np.uint16)
    T, H = x.shape
    idx = _c(topk_idx, np.int64)
    K = idx.shape[1]
    R = rl["rank_slot_of"].shape[1]
    n = max(rl["rows"], 1)
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    rank_x = np.full((n, H), fill, np.uint16)
    rank_idx = np.full((n, K), -7, np.int32)
    rank_w = np.full((n, K), np.nan, np.float32)
    lib().oracle_dispatch_ranks(T, H, K, num_experts, R, _ptr(x), _ptr(idx), _ptr(w),
                                _ptr(_c(rl["rank_slot_of"], np.int32)), _ptr(rank_x),
                                _ptr(rank_idx), _ptr(rank_w))
    return rank_x, rank_idx, rank_w


def expand(topk_idx, lay: dict, rl: dict, rank_x, rank_topk_w, num_experts, fill=0xFFFF):
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    R = rl["rank_slot_of"].shape[1]
    rx = _c(rank_x, np.uint16)
    H = rx.shape[1]
    rw = None if rank_topk_w is None else _c(rank_topk_w, np.float32)
    recv_x = np.full((lay["cap"], H), fill, np.uint16)
    recv_w = np.full(lay["cap"], np.nan, np.float32)
    lib().oracle_expand(T, H, K, num_experts, R, _ptr(idx),
                        _ptr(_c(lay["slot_of"], np.int32)),
                        _ptr(_c(rl["rank_slot_of"], np.int32)), _ptr(rx), _ptr(rw),
                        _ptr(recv_x), _ptr(recv_w))
    return recv_x, recv_w


def reduce_ranks(topk_idx, lay: dict, rl: dict, expert_out, topk_weights, num_experts,
                 fill=0xFFFF):
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    R = rl["rank_slot_of"].shape[1]
    Y = _c(expert_out, np.uint16)
    H = Y.shape[1]
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    rank_y = np.full((max(rl["rows"], 1), H), fill, np.uint16)
    lib().oracle_reduce_ranks(T, H, K, num_experts, R, _ptr(idx),
                              _ptr(_c(lay["slot_of"], np.int32)),
                              _ptr(_c(rl["rank_slot_of"], np.int32)), _ptr(Y), _ptr(w),
                              _ptr(rank_y))
    return rank_y


def combine_ranks(rl: dict, rank_y):
    so = _c(rl["rank_slot_of"], np.int32)
    T, R = so.shape
    ry = _c(rank_y, np.uint16)
    H = ry.shape[1]
    y = np.zeros((T, H), np.uint16)
    lib().oracle_combine_ranks(T, H, R, _ptr(so), _ptr(ry), _ptr(y))
    return y
