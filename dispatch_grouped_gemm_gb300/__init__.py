"""GB300 (sm_103a) fused MoE-FFN: Python binding of libhmm.so.

The functions ``hmm_*`` mirror the C entry points of ``include/hmm.h`` one to
one and only marshal arguments (torch tensors -> device pointers and sizes,
the current CUDA stream).  Every step of the computation runs in the CUDA
kernels of the library; there is no Python or CPU fallback: if ``libhmm.so``
is missing, every call raises.

``moe_ffn(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight)`` is
the autograd entry point (forward saves what the backward needs, backward
returns one gradient per public argument and None for topk_ids), following
the HyperMegaMoE API (§3.1) and its DFunction semantics (§3.2).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

__all__ = [
    "HmmError", "HmmShape", "hmm_create", "hmm_destroy", "hmm_set_option",
    "hmm_workspace_size", "hmm_route", "hmm_route_static", "hmm_forward", "hmm_backward",
    "hmm_backward_dx", "hmm_backward_dw", "hmm_forward_shared", "hmm_backward_shared",
    "hmm_status",
    "hmm_error_string", "Context", "moe_ffn", "library_path", "load_library",
    "hmm_profile_read", "hmm_phase_name", "hmm_set_trace",
    "HMM_OPT_VALIDATE", "HMM_OPT_WAIT_BUDGET_NS", "HMM_OPT_INJECT_SKIP_READY", "HMM_OPT_PROFILE",
    "HMM_OPT_PAIR_ROWS", "HMM_OPT_OVERLAP_LAUNCHES", "HMM_OPT_FUSED_COMBINE",
    "HMM_DTYPE_BF16", "HMM_DTYPE_F32", "HMM_STATUS_EXPERT_ID", "HMM_STATUS_TIMEOUT",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_LIB_PATH = os.path.join(_HERE, "libhmm.so")
_HEADER = os.path.join(_ROOT, "include", "hmm.h")


def _header_constants():
    consts = {}
    with open(_HEADER) as f:
        for m in re.finditer(r"#define\s+(HMM_\w+)\s+\(?(-?\w+?)u?\)?\s", f.read()):
            try:
                consts[m.group(1)] = int(m.group(2), 0)
            except ValueError:
                pass
    return consts


_C = _header_constants()
HMM_OK = _C["HMM_OK"]
HMM_ERR_TIMEOUT = _C["HMM_ERR_TIMEOUT"]
HMM_ERR_EXPERT_ID = _C["HMM_ERR_EXPERT_ID"]
HMM_OPT_VALIDATE = _C["HMM_OPT_VALIDATE"]
HMM_OPT_WAIT_BUDGET_NS = _C["HMM_OPT_WAIT_BUDGET_NS"]
HMM_OPT_INJECT_SKIP_READY = _C["HMM_OPT_INJECT_SKIP_READY"]
HMM_OPT_PROFILE = _C["HMM_OPT_PROFILE"]
HMM_OPT_PAIR_ROWS = _C["HMM_OPT_PAIR_ROWS"]
HMM_OPT_OVERLAP_LAUNCHES = _C["HMM_OPT_OVERLAP_LAUNCHES"]
HMM_OPT_FUSED_COMBINE = _C["HMM_OPT_FUSED_COMBINE"]
HMM_DTYPE_BF16 = _C["HMM_DTYPE_BF16"]
HMM_DTYPE_F32 = _C["HMM_DTYPE_F32"]
HMM_STATUS_EXPERT_ID = _C["HMM_STATUS_EXPERT_ID"]
HMM_STATUS_TIMEOUT = _C["HMM_STATUS_TIMEOUT"]


class HmmShape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("I", ctypes.c_int64),
                ("E", ctypes.c_int64), ("K", ctypes.c_int64),
                ("weights_dtype", ctypes.c_int32), ("shared", ctypes.c_int32)]


class HmmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {hmm_error_string(code)} (code {code})")


_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libhmm.so (raises if it was not built: there is no fallback)."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing; build it with "
                "`python -m dispatch_grouped_gemm_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sp = ctypes.POINTER(HmmShape)
        sig = {
            "hmm_create": [ctypes.POINTER(vp), i32],
            "hmm_destroy": [vp],
            "hmm_set_option": [vp, i32, i64],
            "hmm_workspace_size": [sp, i32, ctypes.POINTER(sz), ctypes.POINTER(sz),
                                   ctypes.POINTER(sz)],
            "hmm_route": [vp, sp, vp, vp, vp, vp, vp, vp, sz, vp],
            "hmm_route_static": [sp, vp, vp, vp, vp, vp, vp],
            "hmm_forward": [vp, sp, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp],
            "hmm_backward": [vp, sp, vp, vp, vp, vp, vp, sz, vp, vp, vp, vp, vp, sz, vp],
            "hmm_backward_dx": [vp, sp, vp, vp, vp, vp, vp, sz, vp, vp, vp, sz, vp],
            "hmm_forward_shared": [vp, sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp],
            "hmm_backward_shared": [vp, sp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp, vp, vp,
                                    vp, vp, sz, vp],
            "hmm_backward_dw": [vp, sp, vp, sz, vp, vp, vp, sz, vp],
            "hmm_status": [vp, vp, ctypes.POINTER(i32)],
            "hmm_profile_read": [vp, i32, ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_int64)],
            "hmm_set_trace": [vp, vp, sz, i32],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = i32
        lib.hmm_error_string.argtypes = [i32]
        lib.hmm_error_string.restype = ctypes.c_char_p
        lib.hmm_phase_name.argtypes = [i32]
        lib.hmm_phase_name.restype = ctypes.c_char_p
        _lib = lib
        return lib


# ------------------------------------------------------------ marshalling
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != HMM_OK:
        raise HmmError(rc, where)


def make_shape(T, H, I, E, K, weights_dtype=HMM_DTYPE_BF16, shared=0) -> HmmShape:
    return HmmShape(int(T), int(H), int(I), int(E), int(K), int(weights_dtype), int(shared))


def hmm_error_string(code: int) -> str:
    return load_library().hmm_error_string(int(code)).decode()


def hmm_create(device: int = 0):
    h = ctypes.c_void_p()
    _check(load_library().hmm_create(ctypes.byref(h), int(device)), "hmm_create")
    return h


def hmm_destroy(ctx):
    _check(load_library().hmm_destroy(ctx), "hmm_destroy")


def hmm_set_option(ctx, option: int, value: int):
    _check(load_library().hmm_set_option(ctx, int(option), int(value)), "hmm_set_option")


def hmm_workspace_size(shape: HmmShape, training: bool):
    f, s, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().hmm_workspace_size(ctypes.byref(shape), int(bool(training)),
                                             ctypes.byref(f), ctypes.byref(s), ctypes.byref(b)),
           "hmm_workspace_size")
    return f.value, s.value, b.value


def hmm_route(ctx, shape, topk_ids, counts, offsets, slot2row, row2slot, workspace, stream=None):
    rc = load_library().hmm_route(ctx, ctypes.byref(shape), _ptr(topk_ids), _ptr(counts),
                                  _ptr(offsets), _ptr(slot2row), _ptr(row2slot), _ptr(workspace),
                                  _nbytes(workspace), _stream(stream))
    _check(rc, "hmm_route")


def hmm_route_static(shape, topk_ids, counts, offsets, slot2row, row2slot, stream=None):
    """Routing on the current device with the library's static scratch (no
    allocation, no context); see include/hmm.h."""
    rc = load_library().hmm_route_static(ctypes.byref(shape), _ptr(topk_ids), _ptr(counts),
                                         _ptr(offsets), _ptr(slot2row), _ptr(row2slot),
                                         _stream(stream))
    _check(rc, "hmm_route_static")


def hmm_forward(ctx, shape, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, y,
                saved, workspace, stream=None):
    rc = load_library().hmm_forward(ctx, ctypes.byref(shape), _ptr(x), _ptr(topk_ids),
                                    _ptr(topk_weights), _ptr(up_proj_weight),
                                    _ptr(down_proj_weight), _ptr(y), _ptr(saved), _nbytes(saved),
                                    _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check(rc, "hmm_forward")


def hmm_backward(ctx, shape, dy, topk_weights, up_proj_weight, down_proj_weight, saved, dx,
                 d_up_proj_weight, d_down_proj_weight, d_topk_weights, workspace, stream=None):
    rc = load_library().hmm_backward(ctx, ctypes.byref(shape), _ptr(dy), _ptr(topk_weights),
                                     _ptr(up_proj_weight), _ptr(down_proj_weight), _ptr(saved),
                                     _nbytes(saved), _ptr(dx), _ptr(d_up_proj_weight),
                                     _ptr(d_down_proj_weight), _ptr(d_topk_weights),
                                     _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check(rc, "hmm_backward")


def hmm_forward_shared(ctx, shape, x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                       shared_up_proj_weight, shared_down_proj_weight, y, saved, workspace,
                       stream=None):
    rc = load_library().hmm_forward_shared(
        ctx, ctypes.byref(shape), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
        _ptr(up_proj_weight), _ptr(down_proj_weight), _ptr(shared_up_proj_weight),
        _ptr(shared_down_proj_weight), _ptr(y), _ptr(saved), _nbytes(saved), _ptr(workspace),
        _nbytes(workspace), _stream(stream))
    _check(rc, "hmm_forward_shared")


def hmm_backward_shared(ctx, shape, dy, topk_weights, up_proj_weight, down_proj_weight,
                        shared_up_proj_weight, shared_down_proj_weight, saved, dx,
                        d_up_proj_weight, d_down_proj_weight, d_shared_up_proj_weight,
                        d_shared_down_proj_weight, d_topk_weights, workspace, stream=None):
    rc = load_library().hmm_backward_shared(
        ctx, ctypes.byref(shape), _ptr(dy), _ptr(topk_weights), _ptr(up_proj_weight),
        _ptr(down_proj_weight), _ptr(shared_up_proj_weight), _ptr(shared_down_proj_weight),
        _ptr(saved), _nbytes(saved), _ptr(dx), _ptr(d_up_proj_weight), _ptr(d_down_proj_weight),
        _ptr(d_shared_up_proj_weight), _ptr(d_shared_down_proj_weight), _ptr(d_topk_weights),
        _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check(rc, "hmm_backward_shared")


def hmm_backward_dx(ctx, shape, dy, topk_weights, up_proj_weight, down_proj_weight, saved, dx,
                    d_topk_weights, workspace, stream=None):
    rc = load_library().hmm_backward_dx(ctx, ctypes.byref(shape), _ptr(dy), _ptr(topk_weights),
                                        _ptr(up_proj_weight), _ptr(down_proj_weight),
                                        _ptr(saved), _nbytes(saved), _ptr(dx),
                                        _ptr(d_topk_weights), _ptr(workspace), _nbytes(workspace),
                                        _stream(stream))
    _check(rc, "hmm_backward_dx")


def hmm_backward_dw(ctx, shape, saved, d_up_proj_weight, d_down_proj_weight, workspace,
                    stream=None):
    rc = load_library().hmm_backward_dw(ctx, ctypes.byref(shape), _ptr(saved), _nbytes(saved),
                                        _ptr(d_up_proj_weight), _ptr(d_down_proj_weight),
                                        _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check(rc, "hmm_backward_dw")


def hmm_status(ctx, stream=None):
    """Synchronise the stream, read and clear the device status word.
    Returns (return code, HMM_STATUS_* bits) without raising."""
    bits = ctypes.c_int(0)
    rc = load_library().hmm_status(ctx, _stream(stream), ctypes.byref(bits))
    return rc, bits.value


def hmm_phase_name(phase: int):
    r = load_library().hmm_phase_name(int(phase))
    return None if r is None else r.decode()


def hmm_profile_read(ctx):
    """{phase name: (GPU ms, kernel launches)} since the previous read."""
    n = _C["HMM_NUM_PHASES"]
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(load_library().hmm_profile_read(ctx, n, ms, cnt), "hmm_profile_read")
    return {hmm_phase_name(i): (ms[i], cnt[i]) for i in range(n)}


def hmm_set_trace(ctx, buffer, which: int):
    """Record the per-tile timeline of the next GEMM launch of kind `which`
    (0 forward, 1 backward data, 2 backward weight) into `buffer` (a device
    tensor; None disables)."""
    _check(load_library().hmm_set_trace(ctx, _ptr(buffer), _nbytes(buffer), int(which)),
           "hmm_set_trace")


# ------------------------------------------------------------ torch layer
_WDTYPES = {torch.bfloat16: HMM_DTYPE_BF16, torch.float32: HMM_DTYPE_F32}


def _u8(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


class Context:
    """A library context on one device plus shape checks of torch arguments."""

    _cache: dict = {}
    _cache_lock = threading.Lock()

    def __init__(self, device=None):
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else
                           torch.device(device).index or 0)
        self.device = dev
        self.handle = hmm_create(dev.index)

    def close(self):
        if self.handle is not None:
            hmm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @classmethod
    def for_device(cls, device) -> "Context":
        idx = device.index if device.index is not None else torch.cuda.current_device()
        with cls._cache_lock:
            c = cls._cache.get(idx)
            if c is None:
                c = cls._cache[idx] = cls(torch.device("cuda", idx))
            return c

    def set_option(self, option: int, value: int):
        hmm_set_option(self.handle, option, value)

    @staticmethod
    def shape_of(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                 shared_up_proj_weight=None, shared_down_proj_weight=None) -> HmmShape:
        if x.dim() != 2 or topk_ids.dim() != 2 or up_proj_weight.dim() != 3:
            raise ValueError("x [T,H], topk_ids [T,K], up_proj_weight [E,H,2I] expected")
        T, H = x.shape
        E, H1, I2 = up_proj_weight.shape
        if H1 != H or I2 % 2:
            raise ValueError(f"up_proj_weight {tuple(up_proj_weight.shape)} does not match x {tuple(x.shape)}")
        I = I2 // 2
        if tuple(down_proj_weight.shape) != (E, I, H):
            raise ValueError(f"down_proj_weight must be {(E, I, H)}, got {tuple(down_proj_weight.shape)}")
        if topk_ids.shape[0] != T or tuple(topk_weights.shape) != tuple(topk_ids.shape):
            raise ValueError("topk_ids / topk_weights must both be [T, K]")
        if x.dtype != torch.bfloat16 or up_proj_weight.dtype != torch.bfloat16 or \
                down_proj_weight.dtype != torch.bfloat16:
            raise TypeError("x, up_proj_weight and down_proj_weight must be bfloat16")
        if topk_ids.dtype != torch.int32:
            raise TypeError("topk_ids must be int32")
        if topk_weights.dtype not in _WDTYPES:
            raise TypeError("topk_weights must be bfloat16 or float32")
        shared = shared_up_proj_weight is not None or shared_down_proj_weight is not None
        if shared:
            if shared_up_proj_weight is None or shared_down_proj_weight is None:
                raise ValueError("the shared expert needs both shared weights")
            if tuple(shared_up_proj_weight.shape) != (H, 2 * I) or \
                    tuple(shared_down_proj_weight.shape) != (I, H):
                raise ValueError(f"shared weights must be {(H, 2 * I)} and {(I, H)}")
            if shared_up_proj_weight.dtype != torch.bfloat16 or \
                    shared_down_proj_weight.dtype != torch.bfloat16:
                raise TypeError("shared weights must be bfloat16")
        for t in (x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                  shared_up_proj_weight, shared_down_proj_weight):
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError("all arguments must be contiguous CUDA tensors")
        return make_shape(T, H, I, E, topk_ids.shape[1], _WDTYPES[topk_weights.dtype],
                          1 if shared else 0)

    def forward(self, x, topk_ids, topk_weights, W1, W2, training: bool, stream=None,
                Ws1=None, Ws2=None):
        shape = self.shape_of(x, topk_ids, topk_weights, W1, W2, Ws1, Ws2)
        fwd, sv, _ = hmm_workspace_size(shape, training)
        y = torch.empty_like(x)
        ws = _u8(fwd, x.device)
        saved = _u8(sv, x.device) if training else None
        if shape.shared:
            hmm_forward_shared(self.handle, shape, x, topk_ids, topk_weights, W1, W2, Ws1, Ws2, y,
                               saved, ws, stream)
        else:
            hmm_forward(self.handle, shape, x, topk_ids, topk_weights, W1, W2, y, saved, ws,
                        stream)
        return y, saved

    def backward(self, dy, x, topk_ids, topk_weights, W1, W2, saved, need=(True, True, True, True),
                 stream=None, Ws1=None, Ws2=None, need_shared=(True, True)):
        """(dx, dW1, dW2, d_topk_weights) and, with the shared expert, (dWs1, dWs2)
        appended; `need` / `need_shared` skip outputs."""
        shape = self.shape_of(x, topk_ids, topk_weights, W1, W2, Ws1, Ws2)
        _, _, bwd = hmm_workspace_size(shape, True)
        dy = dy.contiguous()
        if dy.dtype != torch.bfloat16 or tuple(dy.shape) != tuple(x.shape):
            raise ValueError("dy must be bfloat16 with the shape of x")
        dx = torch.empty_like(x) if need[0] else None
        dW1 = torch.empty_like(W1) if need[1] else None
        dW2 = torch.empty_like(W2) if need[2] else None
        dw = torch.empty_like(topk_weights) if need[3] else None
        ws = _u8(bwd, x.device)
        if not shape.shared:
            hmm_backward(self.handle, shape, dy, topk_weights, W1, W2, saved, dx, dW1, dW2, dw,
                         ws, stream)
            return dx, dW1, dW2, dw
        dWs1 = torch.empty_like(Ws1) if need_shared[0] else None
        dWs2 = torch.empty_like(Ws2) if need_shared[1] else None
        hmm_backward_shared(self.handle, shape, dy, topk_weights, W1, W2, Ws1, Ws2, saved, dx,
                            dW1, dW2, dWs1, dWs2, dw, ws, stream)
        return dx, dW1, dW2, dw, dWs1, dWs2


class _MoEFFN(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, topk_ids, topk_weights, W1, W2):
        c = Context.for_device(x.device)
        y, saved = c.forward(x, topk_ids, topk_weights, W1, W2, training=True)
        ctx.save_for_backward(x, topk_ids, topk_weights, W1, W2, saved)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, topk_ids, topk_weights, W1, W2, saved = ctx.saved_tensors
        need = (ctx.needs_input_grad[0], ctx.needs_input_grad[3], ctx.needs_input_grad[4],
                ctx.needs_input_grad[2])
        c = Context.for_device(x.device)
        dx, dW1, dW2, dw = c.backward(dy, x, topk_ids, topk_weights, W1, W2, saved, need)
        return dx, None, dw, dW1, dW2


class _MoEFFNShared(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, topk_ids, topk_weights, W1, W2, Ws1, Ws2):
        c = Context.for_device(x.device)
        y, saved = c.forward(x, topk_ids, topk_weights, W1, W2, training=True, Ws1=Ws1, Ws2=Ws2)
        ctx.save_for_backward(x, topk_ids, topk_weights, W1, W2, Ws1, Ws2, saved)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, topk_ids, topk_weights, W1, W2, Ws1, Ws2, saved = ctx.saved_tensors
        n = ctx.needs_input_grad
        c = Context.for_device(x.device)
        dx, dW1, dW2, dw, dWs1, dWs2 = c.backward(dy, x, topk_ids, topk_weights, W1, W2, saved,
                                                  (n[0], n[3], n[4], n[2]), Ws1=Ws1, Ws2=Ws2,
                                                  need_shared=(n[5], n[6]))
        return dx, None, dw, dW1, dW2, dWs1, dWs2


def moe_ffn(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight, *,
            shared_up_proj_weight=None, shared_down_proj_weight=None):
    """y[T,H] = sum_k topk_weights[t,k] * FFN_{topk_ids[t,k]}(x[t]) with SwiGLU
    experts (gate = first I columns of up_proj's 2I outputs), plus FFN_s(x[t])
    of the optional shared expert (keyword-only weights [H, 2I] and [I, H]).
    Differentiable in x, topk_weights and every weight tensor; topk_ids is
    not."""
    shared = (shared_up_proj_weight, shared_down_proj_weight)
    has_shared = shared[0] is not None or shared[1] is not None
    tensors = (x, topk_weights, up_proj_weight, down_proj_weight) + (shared if has_shared else ())
    if not (torch.is_grad_enabled() and any(t.requires_grad for t in tensors)):
        c = Context.for_device(x.device)
        y, _ = c.forward(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                         training=False, Ws1=shared[0], Ws2=shared[1])
        return y
    if has_shared:
        return _MoEFFNShared.apply(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight,
                                   *shared)
    return _MoEFFN.apply(x, topk_ids, topk_weights, up_proj_weight, down_proj_weight)
