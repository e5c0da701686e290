"""Python binding of libmoe, the GB300 (sm_103a) local MoE layer of one
expert-parallel rank: route -> dispatch -> grouped SwiGLU expert FFN -> combine.

Argument marshalling only: every step runs in the CUDA kernels behind the C ABI
declared in include/moe.h.  Functions carry the C names and take either torch
CUDA tensors (their data_ptr is passed) or raw integer device addresses; the
stream defaults to torch's current stream.  A non-zero status raises MoeError.
There is no CPU path: if libmoe.so cannot be loaded, every call raises.
"""
import ctypes
import os

__all__ = [
    "MoeError", "Dims", "lib", "build", "moe_route", "moe_dispatch", "moe_dispatch_noalloc", "moe_expert_ffn", "moe_combine",
    "moe_layer", "moe_layer_gather", "moe_combine_accumulate", "moe_expert_gate_up", "moe_expert_down", "moe_workspace_size", "moe_dispatch_workspace_size", "moe_expert_ffn_workspace_size",
    "moe_status_string", "alloc_workspace", "EXPORTED", "moe_testing_layer_stalled_barrier", "FUSED_MAX_PAIRS",
    "moe_quantize_mxfp8", "moe_expert_ffn_mxfp8_workspace_size", "moe_expert_ffn_mxfp8", "moe_layer_mxfp8_workspace_size",
    "moe_layer_mxfp8", "moe_testing_expert_gate_up_stalled", "moe_testing_expert_ffn_mxfp8_stalled",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe.so")

# every symbol include/moe.h declares
EXPORTED = ("moe_status_string", "moe_dispatch_workspace_size", "moe_expert_ffn_workspace_size",
            "moe_workspace_size", "moe_route", "moe_dispatch", "moe_dispatch_noalloc", "moe_expert_ffn", "moe_expert_gate_up",
            "moe_expert_down", "moe_combine", "moe_combine_accumulate", "moe_layer", "moe_layer_gather",
            "moe_testing_layer_stalled_barrier", "moe_quantize_mxfp8", "moe_expert_ffn_mxfp8_workspace_size",
            "moe_expert_ffn_mxfp8", "moe_layer_mxfp8_workspace_size", "moe_layer_mxfp8",
            "moe_testing_expert_gate_up_stalled", "moe_testing_expert_ffn_mxfp8_stalled")

FUSED_MAX_PAIRS = 8192  # MOE_FUSED_MAX_PAIRS in include/moe.h

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_NONFINITE", 6: "MOE_ERR_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({moe_status_string(status)})")


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "I", "E", "k", "e0", "e1")]

    def __init__(self, T, H, I, E, k, e0, e1):
        super().__init__(T, H, I, E, k, e0, e1)

    @classmethod
    def of(cls, d):
        if isinstance(d, cls):
            return d
        if isinstance(d, dict):
            return cls(*(d[n] for n in ("T", "H", "I", "E", "k", "e0", "e1")))
        return cls(*d)


_lib = None


def build(force=False):
    from . import _build as _b
    return _b.build(force=force)


def lib():
    """Load libmoe.so (raises OSError if it is missing: no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"libmoe.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        pd = ctypes.POINTER(Dims)
        L.moe_status_string.argtypes = [i32]
        L.moe_status_string.restype = ctypes.c_char_p
        for f in (L.moe_workspace_size, L.moe_dispatch_workspace_size, L.moe_expert_ffn_workspace_size,
                  L.moe_expert_ffn_mxfp8_workspace_size, L.moe_layer_mxfp8_workspace_size):
            f.argtypes = [pd]
            f.restype = sz
        L.moe_route.argtypes = [pd, vp, vp, vp, vp, vp]
        L.moe_dispatch.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_dispatch_noalloc.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_expert_ffn.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
        L.moe_expert_gate_up.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp]
        L.moe_testing_expert_gate_up_stalled.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp]
        L.moe_expert_down.argtypes = [pd, vp, vp, vp, vp, vp, vp]
        L.moe_combine.argtypes = [pd, vp, vp, vp, vp, vp]
        L.moe_combine_accumulate.argtypes = [pd, vp, vp, vp, vp, vp]
        L.moe_layer.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
        L.moe_layer_gather.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
        L.moe_testing_layer_stalled_barrier.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
        L.moe_quantize_mxfp8.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, vp, vp, vp]
        L.moe_expert_ffn_mxfp8.argtypes = [pd] + [vp] * 11 + [sz, vp, vp]
        L.moe_testing_expert_ffn_mxfp8_stalled.argtypes = [pd] + [vp] * 11 + [sz, vp, vp]
        L.moe_layer_mxfp8.argtypes = [pd] + [vp] * 12 + [sz, vp, vp]
        for f in (L.moe_route, L.moe_dispatch, L.moe_dispatch_noalloc, L.moe_expert_ffn, L.moe_expert_gate_up, L.moe_expert_down,
                  L.moe_combine, L.moe_combine_accumulate, L.moe_layer, L.moe_layer_gather,
                  L.moe_testing_layer_stalled_barrier,
                  L.moe_quantize_mxfp8, L.moe_expert_ffn_mxfp8, L.moe_layer_mxfp8,
                  L.moe_testing_expert_gate_up_stalled, L.moe_testing_expert_ffn_mxfp8_stalled):
            f.restype = i32
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    if t is None:
        return 0
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st, where):
    if st != 0:
        raise MoeError(st, where)


def moe_status_string(status):
    try:
        return lib().moe_status_string(int(status)).decode()
    except OSError:
        return STATUS.get(status, "unknown")


def moe_workspace_size(dims):
    return int(lib().moe_workspace_size(ctypes.byref(Dims.of(dims))))


def moe_dispatch_workspace_size(dims):
    return int(lib().moe_dispatch_workspace_size(ctypes.byref(Dims.of(dims))))


def moe_expert_ffn_workspace_size(dims):
    return int(lib().moe_expert_ffn_workspace_size(ctypes.byref(Dims.of(dims))))


def alloc_workspace(nbytes, device="cuda"):
    """A uint8 CUDA tensor of at least nbytes (torch's allocator returns >= 512-byte alignment)."""
    import torch
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def moe_route(dims, logits, topk_idx, topk_w, status=None, stream=None):
    d = Dims.of(dims)
    _check(lib().moe_route(ctypes.byref(d), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(status),
                           _stream(stream)), "moe_route")


def moe_dispatch(dims, x, topk_idx, counts, offsets, row_pair, pair_row, x_perm, ws, ws_bytes=None, stream=None):
    d = Dims.of(dims)
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().moe_dispatch(ctypes.byref(d), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(offsets), _ptr(row_pair),
                              _ptr(pair_row), _ptr(x_perm), _ptr(ws), nb, _stream(stream)), "moe_dispatch")


def moe_dispatch_noalloc(dims, x, topk_idx, counts, offsets, row_pair, pair_row, x_perm, stream=None):
    """moe_dispatch without a workspace, for callers that cannot allocate device
    memory: the scratch is a fixed 1 MiB array inside libmoe shared by all calls
    (calls that overlap on the GPU race).  Too-large problems raise
    MOE_ERR_UNSUPPORTED."""
    d = Dims.of(dims)
    _check(lib().moe_dispatch_noalloc(ctypes.byref(d), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(offsets),
                                      _ptr(row_pair), _ptr(pair_row), _ptr(x_perm), _stream(stream)),
           "moe_dispatch_noalloc")


def moe_expert_ffn(dims, x_perm, offsets, w_gate, w_up, w_down, y_perm, ws, ws_bytes=None, status=None, stream=None):
    d = Dims.of(dims)
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().moe_expert_ffn(ctypes.byref(d), _ptr(x_perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                _ptr(y_perm), _ptr(ws), nb, _ptr(status), _stream(stream)), "moe_expert_ffn")


def moe_expert_gate_up(dims, x_perm, offsets, w_gate, w_up, h, status=None, stream=None):
    d = Dims.of(dims)
    _check(lib().moe_expert_gate_up(ctypes.byref(d), _ptr(x_perm), _ptr(offsets), _ptr(w_gate), _ptr(w_up), _ptr(h),
                                    _ptr(status), _stream(stream)), "moe_expert_gate_up")


def moe_testing_expert_gate_up_stalled(dims, x_perm, offsets, w_gate, w_up, h, status=None, stream=None):
    """Fault-injection hook: moe_expert_gate_up whose first ring stage never fills;
    the kernel must report MOE_ERR_TIMEOUT in `status` and return."""
    d = Dims.of(dims)
    _check(lib().moe_testing_expert_gate_up_stalled(ctypes.byref(d), _ptr(x_perm), _ptr(offsets), _ptr(w_gate),
                                                    _ptr(w_up), _ptr(h), _ptr(status), _stream(stream)),
           "moe_testing_expert_gate_up_stalled")


def moe_expert_down(dims, h, offsets, w_down, y_perm, status=None, stream=None):
    d = Dims.of(dims)
    _check(lib().moe_expert_down(ctypes.byref(d), _ptr(h), _ptr(offsets), _ptr(w_down), _ptr(y_perm), _ptr(status),
                                 _stream(stream)), "moe_expert_down")


def moe_combine(dims, y_perm, pair_row, topk_w, out, stream=None):
    d = Dims.of(dims)
    _check(lib().moe_combine(ctypes.byref(d), _ptr(y_perm), _ptr(pair_row), _ptr(topk_w), _ptr(out), _stream(stream)),
           "moe_combine")


def moe_combine_accumulate(dims, y_perm, pair_row, topk_w, out, stream=None):
    d = Dims.of(dims)
    _check(lib().moe_combine_accumulate(ctypes.byref(d), _ptr(y_perm), _ptr(pair_row), _ptr(topk_w), _ptr(out),
                                        _stream(stream)), "moe_combine_accumulate")


def moe_layer(dims, x, logits, w_gate, w_up, w_down, out, ws, ws_bytes=None, topk_idx=None, topk_w=None,
              status=None, stream=None):
    d = Dims.of(dims)
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().moe_layer(ctypes.byref(d), _ptr(x), _ptr(logits), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(out),
                           _ptr(topk_idx), _ptr(topk_w), _ptr(ws), nb, _ptr(status), _stream(stream)), "moe_layer")


def moe_layer_gather(dims, x, logits, w_gate, w_up, w_down, out, ws, ws_bytes=None, topk_idx=None, topk_w=None,
                     status=None, stream=None):
    """moe_layer's fused path with the gate/up token rows gathered from x by TMA (no x_perm)."""
    d = Dims.of(dims)
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().moe_layer_gather(ctypes.byref(d), _ptr(x), _ptr(logits), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                  _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(ws), nb, _ptr(status),
                                  _stream(stream)), "moe_layer_gather")


def moe_testing_layer_stalled_barrier(dims, x, logits, w_gate, w_up, w_down, out, ws, ws_bytes=None, status=None,
                                      stream=None):
    """Fault-injection hook: the fused layer with a grid barrier that cannot
    complete; the kernel must report MOE_ERR_TIMEOUT in `status` and return."""
    d = Dims.of(dims)
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().moe_testing_layer_stalled_barrier(ctypes.byref(d), _ptr(x), _ptr(logits), _ptr(w_gate), _ptr(w_up),
                                                   _ptr(w_down), _ptr(out), _ptr(ws), nb, _ptr(status),
                                                   _stream(stream)), "moe_testing_layer_stalled_barrier")


# ---------------------------------------------------------------- MXFP8
def moe_quantize_mxfp8(src, rows, K, q, s, stream=None):
    """q, s = MXFP8 (E4M3 codes, UE8M0 block-32 scales) of the bf16 matrix src [rows, K]."""
    _check(lib().moe_quantize_mxfp8(_ptr(src), int(rows), int(K), _ptr(q), _ptr(s), _stream(stream)),
           "moe_quantize_mxfp8")


def moe_expert_ffn_mxfp8_workspace_size(dims):
    return int(lib().moe_expert_ffn_mxfp8_workspace_size(ctypes.byref(Dims.of(dims))))


def moe_layer_mxfp8_workspace_size(dims):
    return int(lib().moe_layer_mxfp8_workspace_size(ctypes.byref(Dims.of(dims))))


def moe_expert_ffn_mxfp8(dims, x_perm_q, x_perm_s, offsets, w_gate, w_up, w_down, y_perm, ws, ws_bytes=None,
                         status=None, stream=None):
    """w_gate, w_up, w_down: (codes, scales) pairs."""
    d = Dims.of(dims)
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().moe_expert_ffn_mxfp8(ctypes.byref(d), _ptr(x_perm_q), _ptr(x_perm_s), _ptr(offsets),
                                      _ptr(w_gate[0]), _ptr(w_gate[1]), _ptr(w_up[0]), _ptr(w_up[1]),
                                      _ptr(w_down[0]), _ptr(w_down[1]), _ptr(y_perm), _ptr(ws), nb, _ptr(status),
                                      _stream(stream)), "moe_expert_ffn_mxfp8")


def moe_testing_expert_ffn_mxfp8_stalled(dims, x_perm_q, x_perm_s, offsets, w_gate, w_up, w_down, y_perm, ws,
                                         ws_bytes=None, status=None, stream=None):
    """Fault-injection hook: moe_expert_ffn_mxfp8 whose gate/up ring never fills its
    first stage; the kernel must report MOE_ERR_TIMEOUT in `status` and return."""
    d = Dims.of(dims)
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().moe_testing_expert_ffn_mxfp8_stalled(ctypes.byref(d), _ptr(x_perm_q), _ptr(x_perm_s),
                                                      _ptr(offsets), _ptr(w_gate[0]), _ptr(w_gate[1]),
                                                      _ptr(w_up[0]), _ptr(w_up[1]), _ptr(w_down[0]),
                                                      _ptr(w_down[1]), _ptr(y_perm), _ptr(ws), nb, _ptr(status),
                                                      _stream(stream)), "moe_testing_expert_ffn_mxfp8_stalled")


def moe_layer_mxfp8(dims, x, logits, w_gate, w_up, w_down, out, ws, ws_bytes=None, topk_idx=None, topk_w=None,
                    status=None, stream=None):
    """w_gate, w_up, w_down: (codes, scales) pairs from moe_quantize_mxfp8."""
    d = Dims.of(dims)
    nb = _nbytes(ws) if ws_bytes is None else ws_bytes
    _check(lib().moe_layer_mxfp8(ctypes.byref(d), _ptr(x), _ptr(logits), _ptr(w_gate[0]), _ptr(w_gate[1]),
                                 _ptr(w_up[0]), _ptr(w_up[1]), _ptr(w_down[0]), _ptr(w_down[1]), _ptr(out),
                                 _ptr(topk_idx), _ptr(topk_w), _ptr(ws), nb, _ptr(status), _stream(stream)),
           "moe_layer_mxfp8")
