"""fp64 CPU oracle for the fused MoE-FFN forward and backward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the
CUDA library and its Python binding) never imports, links or runs it, and it
shares no code with that path.

The arithmetic lives in ``hmm_oracle.c`` (plain loops, fp64); this module only
compiles it with gcc and marshals numpy arrays through ctypes.  Every function
cites the page section it follows; see the C file's header.

Floating inputs are passed either as raw bf16 bit patterns (``np.uint16``) or
as ``np.float64``; outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hmm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16, F64 = 0, 1


def build(force: bool = False) -> str:
    """Compile hmm_oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _configure(lib):
    """Declare the C entry points' signatures on a loaded library."""
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_route.restype = i64
    lib.oracle_route.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp]
    lib.oracle_forward.restype = i64
    lib.oracle_forward.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int,
                                   vp, vp, vp, vp, vp, vp]
    lib.oracle_backward_tokens.restype = i64
    lib.oracle_backward_tokens.argtypes = [i64, i64, i64, i64, i64,
                                           ctypes.c_int, vp, vp, vp, vp,
                                           vp, vp, vp, vp]
    lib.oracle_weight_grad.restype = i64
    lib.oracle_weight_grad.argtypes = [i64, i64, i64, i64, i64,
                                       ctypes.c_int, i64, vp, vp, vp, vp,
                                       vp, vp, vp, vp]
    lib.oracle_expert_ffn.restype = None
    lib.oracle_expert_ffn.argtypes = [i64, i64, ctypes.c_int, vp, i64, vp,
                                      i64, vp, i64, vp, vp, vp]
    lib.oracle_shared_forward.restype = None
    lib.oracle_shared_forward.argtypes = [i64, i64, i64, ctypes.c_int, vp, vp, vp, vp]
    lib.oracle_shared_backward.restype = None
    lib.oracle_shared_backward.argtypes = [i64, i64, i64, ctypes.c_int, vp, vp, vp, vp,
                                           vp, vp, vp]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _configure(ctypes.CDLL(_LIB_PATH))
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().oracle_num_threads())


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _fp(arrs):
    """Common dtype code of the floating inputs; all must agree."""
    dts = {a.dtype for a in arrs}
    if dts == {np.dtype(np.uint16)}:
        return BF16, [np.ascontiguousarray(a) for a in arrs]
    if dts == {np.dtype(np.float64)}:
        return F64, [np.ascontiguousarray(a) for a in arrs]
    raise TypeError(f"floating inputs must all be uint16 (bf16 bits) or all float64, got {dts}")


class InvalidExpertId(ValueError):
    pass


def route(topk_ids: np.ndarray, E: int):
    """Routing metadata: counts[E], offsets[E+1], slot2row[TK], row2slot[TK]."""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, K = ids.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    s2r = np.zeros(T * K, np.int32)
    r2s = np.zeros(T * K, np.int32)
    bad = _load().oracle_route(T, K, E, _ptr(ids), _ptr(counts), _ptr(offsets),
                               _ptr(s2r), _ptr(r2s))
    if bad:
        raise InvalidExpertId(f"{bad} topk_ids outside [0, {E})")
    return counts, offsets, s2r, r2s


def forward(x, topk_ids, topk_weights, W1, W2):
    """y[T,H] (float64) of the fused MoE-FFN forward."""
    dt, (x, w, W1, W2) = _fp([x, topk_weights, W1, W2])
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, H = x.shape
    E, H1, I2 = W1.shape
    I = I2 // 2
    K = ids.shape[1]
    assert H1 == H and W2.shape == (E, I, H) and w.shape == ids.shape == (T, K)
    y = np.zeros((T, H), np.float64)
    bad = _load().oracle_forward(T, H, I, E, K, dt, _ptr(x), _ptr(ids), _ptr(w),
                                 _ptr(W1), _ptr(W2), _ptr(y))
    if bad:
        raise InvalidExpertId(f"{bad} topk_ids outside [0, {E})")
    return y


def expert_ffn(x_row, W1_e, W2_e):
    """(h[2I], a[I], o[H]) of one expert on one token row."""
    dt, (x_row, W1_e, W2_e) = _fp([x_row, W1_e, W2_e])
    H, I2 = W1_e.shape
    I = I2 // 2
    h = np.zeros(2 * I, np.float64)
    a = np.zeros(I, np.float64)
    o = np.zeros(H, np.float64)
    _load().oracle_expert_ffn(H, I, dt, _ptr(x_row), 0, _ptr(W1_e), 0,
                              _ptr(W2_e), 0, _ptr(h), _ptr(a), _ptr(o))
    return h, a, o


def backward_tokens(x, topk_ids, topk_weights, W1, W2, dy):
    """(dx[T,H], d_topk_weights[T,K]) in float64."""
    dt, (x, w, W1, W2, dy) = _fp([x, topk_weights, W1, W2, dy])
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, H = x.shape
    E, _, I2 = W1.shape
    I = I2 // 2
    K = ids.shape[1]
    dx = np.zeros((T, H), np.float64)
    dw = np.zeros((T, K), np.float64)
    bad = _load().oracle_backward_tokens(T, H, I, E, K, dt, _ptr(x), _ptr(ids),
                                         _ptr(w), _ptr(W1), _ptr(W2), _ptr(dy),
                                         _ptr(dx), _ptr(dw))
    if bad:
        raise InvalidExpertId(f"{bad} topk_ids outside [0, {E})")
    return dx, dw


def weight_grad(e, x, topk_ids, topk_weights, W1, W2, dy):
    """(dW1[e] [H,2I], dW2[e] [I,H]) in float64 for one expert e."""
    dt, (x, w, W1, W2, dy) = _fp([x, topk_weights, W1, W2, dy])
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, H = x.shape
    E, _, I2 = W1.shape
    I = I2 // 2
    K = ids.shape[1]
    dW1 = np.zeros((H, 2 * I), np.float64)
    dW2 = np.zeros((I, H), np.float64)
    bad = _load().oracle_weight_grad(T, H, I, E, K, dt, int(e), _ptr(x),
                                     _ptr(ids), _ptr(w), _ptr(W1), _ptr(W2),
                                     _ptr(dy), _ptr(dW1), _ptr(dW2))
    if bad:
        raise InvalidExpertId(f"{bad} topk_ids outside [0, {E})")
    return dW1, dW2


def backward(x, topk_ids, topk_weights, W1, W2, dy):
    """All four gradients (dx, dW1[E,H,2I], dW2[E,I,H], dw) in float64."""
    E = W1.shape[0]
    dx, dw = backward_tokens(x, topk_ids, topk_weights, W1, W2, dy)
    dW1 = np.zeros(W1.shape, np.float64)
    dW2 = np.zeros(W2.shape, np.float64)
    for e in range(E):
        dW1[e], dW2[e] = weight_grad(e, x, topk_ids, topk_weights, W1, W2, dy)
    return dx, dW1, dW2, dw


def shared_forward(x, Ws1, Ws2):
    """The shared expert's term of y (float64 [T,H]): FFN_s(x[t]) for every
    token, unit weight [HyperMegaMoE §6.1]."""
    dt, (x, Ws1, Ws2) = _fp([x, Ws1, Ws2])
    T, H = x.shape
    H1, I2 = Ws1.shape
    I = I2 // 2
    assert H1 == H and Ws2.shape == (I, H)
    ys = np.zeros((T, H), np.float64)
    _load().oracle_shared_forward(T, H, I, dt, _ptr(x), _ptr(Ws1), _ptr(Ws2), _ptr(ys))
    return ys


def shared_backward(x, Ws1, Ws2, dy):
    """The shared expert's part of dx and its weight gradients:
    (dx_s [T,H], dWs1 [H,2I], dWs2 [I,H]) in float64."""
    dt, (x, Ws1, Ws2, dy) = _fp([x, Ws1, Ws2, dy])
    T, H = x.shape
    I = Ws1.shape[1] // 2
    dxs = np.zeros((T, H), np.float64)
    dWs1 = np.zeros((H, 2 * I), np.float64)
    dWs2 = np.zeros((I, H), np.float64)
    _load().oracle_shared_backward(T, H, I, dt, _ptr(x), _ptr(Ws1), _ptr(Ws2), _ptr(dy),
                                   _ptr(dxs), _ptr(dWs1), _ptr(dWs2))
    return dxs, dWs1, dWs2
