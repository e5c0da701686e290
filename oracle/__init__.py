"""CPU oracle of the local MoE layer (route, dispatch, SwiGLU expert FFN, combine).

TEST INFRASTRUCTURE ONLY: the tests, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg use it; the product library never does.

The arithmetic lives in `oracle.c` (plain C, fp64, OpenMP over tokens), which
cites the passages of "Hosting Qwen on Blackwell" it follows. This module only
marshals numpy arrays through ctypes.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

NONFINITE = 5


def build(force=False):
    """Compile liboracle.so with gcc (OpenMP when available)."""
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", _SO + ".tmp", "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        subprocess.run(base, check=True)
    os.replace(_SO + ".tmp", _SO)
    return _SO


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.oracle_route.argtypes = [i64, i32, i32, vp, vp, vp]
    lib.oracle_route.restype = i32
    lib.oracle_dispatch.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.oracle_dispatch.restype = i64
    lib.oracle_expert_ffn_rows.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, i64, i64, vp]
    lib.oracle_expert_ffn_rows.restype = None
    lib.oracle_expert_ffn_rowlist.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, i64, vp]
    lib.oracle_expert_ffn_rowlist.restype = None
    lib.oracle_combine_tokens.argtypes = [i32, i32, vp, vp, vp, vp, i64, vp]
    lib.oracle_combine_tokens.restype = None
    lib.oracle_moe_layer_tokens.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i64, vp]
    lib.oracle_moe_layer_tokens.restype = i32
    lib.oracle_mxfp8_quantize.argtypes = [i64, i32, vp, vp, vp]
    lib.oracle_mxfp8_quantize.restype = i32
    lib.oracle_mxfp8_dequantize.argtypes = [i64, i32, vp, vp, vp]
    lib.oracle_mxfp8_dequantize.restype = None
    lib.oracle_expert_ffn_mxfp8_rowlist.argtypes = [i32, i32, i32] + [vp] * 9 + [vp, i64] + [vp] * 6
    lib.oracle_expert_ffn_mxfp8_rowlist.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_SO))
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def num_threads():
    return int(_load().oracle_num_threads())


def route(logits, k):
    """-> (status, topk_idx int32 [T,k], topk_w float64 [T,k])"""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    st = _load().oracle_route(T, E, k, _p(lg), _p(idx), _p(w))
    return int(st), idx, w


def dispatch(topk_idx, e0, e1):
    """-> dict(counts, offsets, row_pair [R], pair_row [T*k], R)"""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    n = e1 - e0
    counts = np.zeros(n, np.int32)
    offsets = np.zeros(n + 1, np.int32)
    row_pair = np.full(T * k, -1, np.int32)
    pair_row = np.full(T * k, -1, np.int32)
    R = _load().oracle_dispatch(T, k, e0, e1, _p(idx), _p(counts), _p(offsets), _p(row_pair), _p(pair_row))
    if R < 0:
        raise ValueError("oracle_dispatch: bad arguments")
    return dict(counts=counts, offsets=offsets, row_pair=row_pair[:R].copy(), pair_row=pair_row, R=int(R))


def expert_ffn_rows(x_perm, offsets, w_gate, w_up, w_down, row_lo=0, row_hi=None):
    """FFN of grouped rows [row_lo, row_hi) -> float64 [rows, H]."""
    xp = _c(x_perm, np.uint16)
    H = xp.shape[1]
    n, I, _ = w_gate.shape
    if row_hi is None:
        row_hi = int(offsets[-1])
    off = _c(offsets, np.int32)
    wg, wu, wd = _c(w_gate, np.uint16), _c(w_up, np.uint16), _c(w_down, np.uint16)
    y = np.zeros((row_hi - row_lo, H), np.float64)
    _load().oracle_expert_ffn_rows(H, I, n, _p(xp), _p(off), _p(wg), _p(wu), _p(wd), row_lo, row_hi, _p(y))
    return y


def expert_ffn_rowlist(x_perm, offsets, w_gate, w_up, w_down, rows):
    """FFN of the listed grouped rows -> float64 [len(rows), H]."""
    xp = _c(x_perm, np.uint16)
    H = xp.shape[1]
    n, I, _ = w_gate.shape
    off = _c(offsets, np.int32)
    rr = _c(rows, np.int64)
    wg, wu, wd = _c(w_gate, np.uint16), _c(w_up, np.uint16), _c(w_down, np.uint16)
    y = np.zeros((rr.size, H), np.float64)
    _load().oracle_expert_ffn_rowlist(H, I, n, _p(xp), _p(off), _p(wg), _p(wu), _p(wd), _p(rr), rr.size, _p(y))
    return y


def combine_tokens(y_perm, pair_row, topk_w, tokens=None):
    """Weighted combine of grouped fp32 rows -> float64 [ntok, H]."""
    yp = _c(y_perm, np.float32)
    H = yp.shape[1]
    tw = _c(topk_w, np.float32)
    T, k = tw.shape
    toks = np.arange(T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    pr = _c(pair_row, np.int32)
    out = np.zeros((toks.size, H), np.float64)
    _load().oracle_combine_tokens(H, k, _p(yp), _p(pr), _p(tw), _p(toks), toks.size, _p(out))
    return out


def moe_layer_tokens(logits, x, w_gate, w_up, w_down, k, e0, e1, tokens=None):
    """Token-major full layer for the listed tokens -> (status, float64 [ntok, H])."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    xx = _c(x, np.uint16)
    H = xx.shape[1]
    I = w_gate.shape[1]
    toks = np.arange(T, dtype=np.int64) if tokens is None else _c(tokens, np.int64)
    wg, wu, wd = _c(w_gate, np.uint16), _c(w_up, np.uint16), _c(w_down, np.uint16)
    out = np.zeros((toks.size, H), np.float64)
    st = _load().oracle_moe_layer_tokens(H, I, E, k, e0, e1, _p(lg), _p(xx), _p(wg), _p(wu), _p(wd),
                                         _p(toks), toks.size, _p(out))
    return int(st), out


# ---------------------------------------------------------------- MXFP8
def mxfp8_quantize(a):
    """MXFP8 (E4M3 elements, UE8M0 scales, blocks of 32 along the last axis) of a
    bf16 bit-pattern matrix [rows, K] -> (q uint8 [rows, K], s uint8 [rows, K/32])."""
    src = _c(a, np.uint16)
    rows, K = src.shape
    q = np.empty((rows, K), np.uint8)
    s = np.empty((rows, K // 32), np.uint8)
    if _load().oracle_mxfp8_quantize(rows, K, _p(src), _p(q), _p(s)) != 0:
        raise ValueError("oracle_mxfp8_quantize: K must be a multiple of 32")
    return q, s


def mxfp8_dequantize(q, s):
    """float64 values of an MXFP8 matrix."""
    qq, ss = _c(q, np.uint8), _c(s, np.uint8)
    rows, K = qq.shape
    out = np.empty((rows, K), np.float64)
    _load().oracle_mxfp8_dequantize(rows, K, _p(qq), _p(ss), _p(out))
    return out


def expert_ffn_mxfp8_rowlist(xq, xs, offsets, wg, wu, wd, rows, h_in=None, want_h=False):
    """MXFP8 expert FFN of the listed grouped rows.  wg, wu, wd are (q, s) pairs with
    the shapes of the bf16 weights ([n, I, H], [n, I, H], [n, H, I]) and of their
    scales.  h_in: optional (hq, hs) [len(rows), I] / [len(rows), I/32] used for the
    down GEMM instead of the oracle's own quantised h.  Returns y float64
    [len(rows), H], and with want_h also (h fp64, hq, hs) of the oracle's h."""
    xq_, xs_ = _c(xq, np.uint8), _c(xs, np.uint8)
    H = xq_.shape[1]
    n, I, _ = wg[0].shape
    off, rr = _c(offsets, np.int32), _c(rows, np.int64)
    w = [_c(a, np.uint8) for pair in (wg, wu, wd) for a in pair]
    y = np.zeros((rr.size, H), np.float64)
    h = np.zeros((rr.size, I), np.float64) if want_h else None
    hq = np.zeros((rr.size, I), np.uint8) if want_h else None
    hs = np.zeros((rr.size, I // 32), np.uint8) if want_h else None
    hin = [None, None] if h_in is None else [_c(h_in[0], np.uint8), _c(h_in[1], np.uint8)]
    p = lambda a: None if a is None else _p(a)
    _load().oracle_expert_ffn_mxfp8_rowlist(H, I, n, _p(xq_), _p(xs_), _p(off), *[_p(a) for a in w], _p(rr),
                                            rr.size, p(hin[0]), p(hin[1]), p(h), p(hq), p(hs), _p(y))
    return (y, h, hq, hs) if want_h else y
