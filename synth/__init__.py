"""Seeded synthetic inputs for the MoE layer (shared by the oracle tests and the
CUDA path tests / benchmark). Holds no MoE arithmetic: random numbers only.

`make_inputs(cfg)` returns numpy arrays:
  x        uint16 [T, H]         bf16 bits, N(0, x_std)
  logits   float32 [T, E]        N(0, logit_std) (+ fp32 Zipf bias if asked)
  w_gate   uint16 [n, I, H]      bf16 bits, N(0, w_std), local experts e0..e1-1
  w_up     uint16 [n, I, H]
  w_down   uint16 [n, H, I]
"""
import ctypes
import math
import os
import subprocess

import numpy as np

from .configs import CONFIGS, TID_AUX, TID_LOGITS, TID_W_DOWN, TID_W_GATE, TID_W_UP, TID_X, dims_of  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force=False):
    """Compile libsynth.so with gcc (OpenMP if the compiler has it)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", _SO + ".tmp", "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        subprocess.run(base, check=True)
    os.replace(_SO + ".tmp", _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, f64, f64, vp]
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, i64, f64, vp]
        lib.synth_uniform_int.argtypes = [u64, u64, u64, i64, i64, vp]
        lib.synth_f32_to_bf16.argtypes = [vp, i64, vp]
        for f in (lib.synth_normal_f32, lib.synth_normal_bf16, lib.synth_uniform_int, lib.synth_f32_to_bf16):
            f.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def normal_f32(seed, tid, shape, mean=0.0, std=1.0, start=0):
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(seed, tid, start, out.size, float(mean), float(std), _ptr(out))
    return out


def normal_bf16(seed, tid, shape, std=1.0, start=0):
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(seed, tid, start, out.size, float(std), _ptr(out))
    return out


def uniform_int(seed, tid, n, m, start=0):
    out = np.empty(n, dtype=np.int32)
    _load().synth_uniform_int(seed, tid, start, n, m, _ptr(out))
    return out


def f32_to_bf16(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().synth_f32_to_bf16(_ptr(a), a.size, _ptr(out))
    return out


def bf16_to_f32(a):
    """Exact widening of bf16 bit patterns (storage conversion only)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def zipf_bias(E):
    """bias_e = 3 ln(1/(e+1)), rounded to fp32."""
    return np.array([3.0 * math.log(1.0 / (e + 1)) for e in range(E)], dtype=np.float32)


def make_logits(cfg, seed=0):
    T, E = cfg["T"], cfg["E"]
    lg = normal_f32(seed, TID_LOGITS, (T, E), 0.0, cfg["logit_std"])
    if cfg.get("zipf_bias"):
        lg = (lg + zipf_bias(E)[None, :]).astype(np.float32)  # fp32 add
    if cfg.get("one_token_per_expert"):
        # token t's largest logit is at expert e0 + t (a margin of 64 over N(0,1) noise)
        t = np.arange(T)
        lg[t, cfg["e0"] + t] += np.float32(64.0)
    return lg


def make_x(cfg, seed=0):
    return normal_bf16(seed, TID_X, (cfg["T"], cfg["H"]), cfg["x_std"])


def make_weights(cfg, seed=0, which=("gate", "up", "down")):
    """Local-expert slices [e0, e1) of the global weight tensors."""
    H, I, e0, e1 = cfg["H"], cfg["I"], cfg["e0"], cfg["e1"]
    n = e1 - e0
    out = {}
    if "gate" in which:
        out["w_gate"] = normal_bf16(seed, TID_W_GATE, (n, I, H), cfg["w_std"], start=e0 * I * H)
    if "up" in which:
        out["w_up"] = normal_bf16(seed, TID_W_UP, (n, I, H), cfg["w_std"], start=e0 * I * H)
    if "down" in which:
        out["w_down"] = normal_bf16(seed, TID_W_DOWN, (n, H, I), cfg["w_std"], start=e0 * H * I)
    return out


def make_inputs(cfg, seed=0, weights=True):
    d = {"x": make_x(cfg, seed), "logits": make_logits(cfg, seed)}
    if weights:
        d.update(make_weights(cfg, seed))
    return d


def config(name, **over):
    c = dict(CONFIGS[name])
    c.update(over)
    c["name"] = name
    return c
