"""CPU oracle for the forward pass of one top-k-routed SwiGLU MoE layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never imports it, and it never imports the product library.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 sums, bf16
round-to-nearest-even at logits, h, a and y).  This module only builds that
file with gcc and passes numpy arrays to it through ctypes.

Every function takes and returns numpy arrays.  bf16 tensors travel as their
raw 16-bit patterns in ``numpy.uint16`` arrays.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmoe_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``oracle/_build/libmoe_oracle.so``.

    OpenMP is used when gcc accepts ``-fopenmp``; otherwise the oracle is built
    single-threaded.  Returns the library path.
    """
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cc = os.environ.get("CC") or shutil.which("gcc") or "cc"
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_bf16_round.argtypes = [ctypes.c_double]
    lib.oracle_bf16_round.restype = ctypes.c_uint16
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_round_array.argtypes = [P, ctypes.c_long, P]
    lib.oracle_bf16_round_array.restype = None
    lib.oracle_set_threads.argtypes = [i]
    lib.oracle_set_threads.restype = None
    lib.oracle_get_threads.argtypes = []
    lib.oracle_get_threads.restype = i
    lib.oracle_router_logits.argtypes = [P, P, P, i, i, i, P]
    lib.oracle_router_logits.restype = None
    lib.oracle_topk_softmax.argtypes = [P, i, i, i, i, P, P]
    lib.oracle_topk_softmax.restype = None
    lib.oracle_align_capacity.argtypes = [i, i, i, i]
    lib.oracle_align_capacity.restype = ctypes.c_long
    lib.oracle_align_block_size.argtypes = [P, i, i, i, i, P, P, P, P]
    lib.oracle_align_block_size.restype = i
    lib.oracle_expert_act.argtypes = [P, P, P, i, i, i, i, i, P]
    lib.oracle_expert_act.restype = None
    lib.oracle_expert_down_combine.argtypes = [P, P, P, P, P, i, i, i, i, i, P]
    lib.oracle_expert_down_combine.restype = None
    lib.oracle_moe_forward.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, i, P, P, P, P]
    lib.oracle_moe_forward.restype = i
    lib.oracle_e4m3_round_array.argtypes = [P, ctypes.c_long, P]
    lib.oracle_e4m3_round_array.restype = None
    lib.oracle_e4m3_to_double_array.argtypes = [P, ctypes.c_long, P]
    lib.oracle_e4m3_to_double_array.restype = None
    lib.oracle_quant_rows.argtypes = [P, i, i, P, P]
    lib.oracle_quant_rows.restype = None
    lib.oracle_expert_act_fp8.argtypes = [P, P, P, P, P, i, i, i, i, i, P]
    lib.oracle_expert_act_fp8.restype = None
    lib.oracle_expert_down_combine_fp8.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, P]
    lib.oracle_expert_down_combine_fp8.restype = None
    lib.oracle_moe_forward_fp8.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, P, P, P]
    lib.oracle_moe_forward_fp8.restype = i
    _lib = lib
    return lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def bf16_round(values) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (uint16), element by element."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_bf16_round_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def router_logits(x, w_r, bias=None):
    """logits [M, E] (bf16 bits) = bf16(x @ w_r^T + bias)."""
    x = _c(x, np.uint16)
    w_r = _c(w_r, np.uint16)
    bias = _c(bias, np.float32)
    M, H = x.shape
    E = w_r.shape[0]
    assert w_r.shape == (E, H)
    out = np.empty((M, E), np.uint16)
    _load().oracle_router_logits(_ptr(x), _ptr(w_r), _ptr(bias), M, E, H, _ptr(out))
    return out


def topk_softmax(logits, top_k: int, renormalize: bool = True):
    """(topk_ids int32 [M, k], topk_weights float32 [M, k]) from bf16 logits."""
    logits = _c(logits, np.uint16)
    M, E = logits.shape
    ids = np.empty((M, top_k), np.int32)
    w = np.empty((M, top_k), np.float32)
    _load().oracle_topk_softmax(_ptr(logits), M, E, top_k, int(bool(renormalize)), _ptr(ids), _ptr(w))
    return ids, w


def align_capacity(M: int, top_k: int, E: int, B: int) -> int:
    return int(_load().oracle_align_capacity(M, top_k, E, B))


def align_block_size(topk_ids, E: int, block_size_m: int):
    """(sorted_token_ids [cap], expert_ids [cap/B], expert_offsets [E+1], n_post)."""
    ids = _c(topk_ids, np.int32)
    M, k = ids.shape
    B = int(block_size_m)
    cap = align_capacity(M, k, E, B)
    s = np.empty(cap, np.int32)
    eid = np.empty(cap // B, np.int32)
    off = np.empty(E + 1, np.int32)
    n = np.zeros(1, np.int32)
    rc = _load().oracle_align_block_size(_ptr(ids), M, k, E, B, _ptr(s), _ptr(eid), _ptr(off), _ptr(n))
    if rc != 0:
        raise ValueError("expert id outside [0, E)")
    return s, eid, off, int(n[0])


def expert_act(x, w13, topk_ids):
    """a [M*k, I] (bf16 bits), pair order."""
    x = _c(x, np.uint16)
    w13 = _c(w13, np.uint16)
    ids = _c(topk_ids, np.int32)
    M, H = x.shape
    E, twoI, H2 = w13.shape
    assert H2 == H and twoI % 2 == 0
    I = twoI // 2
    k = ids.shape[1]
    a = np.empty((M * k, I), np.uint16)
    _load().oracle_expert_act(_ptr(x), _ptr(w13), _ptr(ids), M, k, E, H, I, _ptr(a))
    return a


def expert_down_combine(a, w2, topk_ids, topk_weights, residual=None):
    """y [M, H] (bf16 bits) = bf16(sum_j w_j * (W2_{id_j} a_{p}) + residual)."""
    a = _c(a, np.uint16)
    w2 = _c(w2, np.uint16)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_weights, np.float32)
    residual = _c(residual, np.uint16)
    M, k = ids.shape
    E, H, I = w2.shape
    assert a.shape == (M * k, I)
    y = np.empty((M, H), np.uint16)
    _load().oracle_expert_down_combine(_ptr(a), _ptr(w2), _ptr(ids), _ptr(w), _ptr(residual),
                                       M, k, E, H, I, _ptr(y))
    return y


def moe_forward(x, w13, w2, top_k: int, *, w_router=None, router_logits=None,
                router_bias=None, residual=None, renormalize: bool = True):
    """Whole layer.  Returns dict(y, topk_ids, topk_weights, logits)."""
    x = _c(x, np.uint16)
    w13 = _c(w13, np.uint16)
    w2 = _c(w2, np.uint16)
    w_router = _c(w_router, np.uint16)
    router_logits = _c(router_logits, np.uint16)
    router_bias = _c(router_bias, np.float32)
    residual = _c(residual, np.uint16)
    M, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    y = np.empty((M, H), np.uint16)
    ids = np.empty((M, top_k), np.int32)
    w = np.empty((M, top_k), np.float32)
    lg = np.empty((M, E), np.uint16)
    rc = _load().oracle_moe_forward(_ptr(x), _ptr(w_router), _ptr(router_logits), _ptr(router_bias),
                                    _ptr(w13), _ptr(w2), _ptr(residual), M, E, top_k, H, I,
                                    int(bool(renormalize)), _ptr(y), _ptr(ids), _ptr(w), _ptr(lg))
    if rc != 0:
        raise ValueError("oracle_moe_forward: bad arguments")
    return {"y": y, "topk_ids": ids, "topk_weights": w, "logits": lg}


# ----------------------------------------------------------------------------- FP8 (E4M3)

def e4m3_round(values) -> np.ndarray:
    """float64 values -> E4M3 codes (uint8): nearest, ties to even, saturating at +-448."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_round_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_to_f64(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> float64, exactly."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_to_double_array(_ptr(c), c.size, _ptr(out))
    return out


def quant_rows(src):
    """Per-row dynamic E4M3 quantization of bf16 bits [R, K]: (codes uint8 [R, K], scales f32 [R])."""
    src = _c(src, np.uint16)
    R, K = src.shape
    q = np.empty((R, K), np.uint8)
    s = np.empty(R, np.float32)
    _load().oracle_quant_rows(_ptr(src), R, K, _ptr(q), _ptr(s))
    return q, s


def expert_act_fp8(qx, sx, qw13, sw13, topk_ids):
    """a [M*k, I] (bf16 bits) from E4M3 x codes/scales and E4M3 W13 codes/row scales."""
    qx, sx = _c(qx, np.uint8), _c(sx, np.float32)
    qw13, sw13 = _c(qw13, np.uint8), _c(sw13, np.float32)
    ids = _c(topk_ids, np.int32)
    M, H = qx.shape
    E, twoI, H2 = qw13.shape
    assert H2 == H and sw13.shape == (E, twoI) and sx.shape == (M,)
    I = twoI // 2
    k = ids.shape[1]
    a = np.empty((M * k, I), np.uint16)
    _load().oracle_expert_act_fp8(_ptr(qx), _ptr(sx), _ptr(qw13), _ptr(sw13), _ptr(ids), M, k, E,
                                  H, I, _ptr(a))
    return a


def expert_down_combine_fp8(qa, sa, qw2, sw2, topk_ids, topk_weights, residual=None):
    """y [M, H] (bf16 bits) from E4M3 activation codes/scales and E4M3 W2 codes/row scales."""
    qa, sa = _c(qa, np.uint8), _c(sa, np.float32)
    qw2, sw2 = _c(qw2, np.uint8), _c(sw2, np.float32)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_weights, np.float32)
    residual = _c(residual, np.uint16)
    M, k = ids.shape
    E, H, I = qw2.shape
    assert qa.shape == (M * k, I) and sa.shape == (M * k,) and sw2.shape == (E, H)
    y = np.empty((M, H), np.uint16)
    _load().oracle_expert_down_combine_fp8(_ptr(qa), _ptr(sa), _ptr(qw2), _ptr(sw2), _ptr(ids),
                                           _ptr(w), _ptr(residual), M, k, E, H, I, _ptr(y))
    return y


def moe_forward_fp8(x, qw13, sw13, qw2, sw2, top_k: int, *, w_router=None, router_logits=None,
                    router_bias=None, residual=None, renormalize: bool = True):
    """Whole layer with E4M3 expert weights.  Returns dict(y, topk_ids, topk_weights, logits)."""
    x = _c(x, np.uint16)
    qw13, sw13 = _c(qw13, np.uint8), _c(sw13, np.float32)
    qw2, sw2 = _c(qw2, np.uint8), _c(sw2, np.float32)
    w_router = _c(w_router, np.uint16)
    router_logits = _c(router_logits, np.uint16)
    router_bias = _c(router_bias, np.float32)
    residual = _c(residual, np.uint16)
    M, H = x.shape
    E, twoI, _ = qw13.shape
    I = twoI // 2
    y = np.empty((M, H), np.uint16)
    ids = np.empty((M, top_k), np.int32)
    w = np.empty((M, top_k), np.float32)
    lg = np.empty((M, E), np.uint16)
    rc = _load().oracle_moe_forward_fp8(_ptr(x), _ptr(w_router), _ptr(router_logits),
                                        _ptr(router_bias), _ptr(qw13), _ptr(sw13), _ptr(qw2),
                                        _ptr(sw2), _ptr(residual), M, E, top_k, H, I,
                                        int(bool(renormalize)), _ptr(y), _ptr(ids), _ptr(w),
                                        _ptr(lg))
    if rc != 0:
        raise ValueError("oracle_moe_forward_fp8: bad arguments")
    return {"y": y, "topk_ids": ids, "topk_weights": w, "logits": lg}
