"""Python binding of the GB300 MoE-layer CUDA library (``libmoe_gb300.so``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  The functions keep the
C ABI's names (``include/moe_api.h``); each takes preallocated torch tensors
for its outputs and raises ``MoeError`` on a non-OK status.  There is no CPU
fallback: if the library is missing or cannot be loaded, every call raises.

The layer follows the page "Mixture of Experts in vLLM - From First
Principles to fused_moe": router logits, softmax / top-k / renormalize,
grouping of the (token, expert) pairs by expert into block-padded
sorted_token_ids / expert_ids, grouped GEMM 1 with SiLU(gate) * up, grouped
GEMM 2 with the router-weighted per-token combine.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "MoeError", "load_library", "library_path", "moe_workspace_size", "moe_align_capacity",
    "moe_pick_block_size", "moe_workspace_init", "moe_router_logits", "moe_topk_softmax",
    "moe_align_block_size", "moe_grouped_gemm_w13_act", "moe_grouped_gemm_w2_combine",
    "moe_forward", "moe_get_device_status", "moe_status_string", "Workspace",
    "moe_grouped_gemm_w2_combine_noalloc", "moe_route", "moe_selftest_device_timeout",
    "moe_quantize_rows_fp8", "moe_workspace_size_fp8", "moe_grouped_gemm_w13_act_fp8",
    "moe_grouped_gemm_w2_combine_fp8", "moe_forward_fp8",
]

STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
    3: "MOE_ERR_WORKSPACE_TOO_SMALL", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_BAD_EXPERT_ID",
    6: "MOE_ERR_DEVICE_TIMEOUT",
}

# Every symbol include/moe_api.h declares.
EXPORTED = (
    "moe_workspace_size", "moe_align_capacity", "moe_pick_block_size", "moe_router_logits",
    "moe_topk_softmax", "moe_align_block_size", "moe_grouped_gemm_w13_act",
    "moe_grouped_gemm_w2_combine", "moe_forward", "moe_workspace_init", "moe_get_device_status",
    "moe_status_string", "moe_grouped_gemm_w2_combine_noalloc", "moe_route",
    "moe_selftest_device_timeout", "moe_quantize_rows_fp8", "moe_workspace_size_fp8",
    "moe_grouped_gemm_w13_act_fp8", "moe_grouped_gemm_w2_combine_fp8", "moe_forward_fp8",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.status, self.status)}")


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False):
    """Load the CUDA library (optionally building it first)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"CUDA library not built: {path} is missing "
                               "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        _build.build()
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "moe_workspace_size": ([I, I, I, I, I, I], Z),
        "moe_align_capacity": ([I, I, I, I], ctypes.c_long),
        "moe_pick_block_size": ([I, I, I, I, I], I),
        "moe_router_logits": ([P, P, P, I, I, I, P, P], I),
        "moe_topk_softmax": ([P, I, I, I, I, P, P, P], I),
        "moe_align_block_size": ([P, I, I, I, I, P, P, P, P, P, Z, P], I),
        "moe_grouped_gemm_w13_act": ([P, P, P, P, P, I, I, I, I, I, I, P, P], I),
        "moe_route": ([P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P, P, Z, P], I),
        "moe_grouped_gemm_w2_combine": ([P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, Z, P], I),
        "moe_grouped_gemm_w2_combine_noalloc": ([P, P, P, P, P, P, P, I, I, I, I, I, I, P, P], I),
        "moe_forward": ([P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, P, Z, P], I),
        "moe_workspace_init": ([P, Z, P], I),
        "moe_get_device_status": ([P, P], I),
        "moe_selftest_device_timeout": ([P, Z, I, P], I),
        "moe_status_string": ([I], ctypes.c_char_p),
        "moe_quantize_rows_fp8": ([P, I, I, P, P, P], I),
        "moe_workspace_size_fp8": ([I, I, I, I, I, I], Z),
        "moe_grouped_gemm_w13_act_fp8": ([P, P, P, P, P, P, P, I, I, I, I, I, I, P, P], I),
        "moe_grouped_gemm_w2_combine_fp8": ([P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, Z,
                                             P], I),
        "moe_forward_fp8": ([P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P, P, P, P, Z, P],
                            I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


# ----------------------------------------------------------------------------- helpers

def _p(t):
    """Device pointer of a tensor (None for None)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _check_dtype(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ok(rc: int, where: str):
    if rc != 0:
        raise MoeError(rc, where)


# ----------------------------------------------------------------------------- sizes

def moe_workspace_size(M_max: int, E: int, top_k: int, H: int, I: int, block_size_m: int = 0) -> int:
    n = load_library().moe_workspace_size(M_max, E, top_k, H, I, block_size_m)
    if n == 0:
        raise MoeError(2, "moe_workspace_size")
    return int(n)


def moe_align_capacity(M: int, top_k: int, E: int, block_size_m: int) -> int:
    n = load_library().moe_align_capacity(M, top_k, E, block_size_m)
    if n < 0:
        raise MoeError(2, "moe_align_capacity")
    return int(n)


def moe_pick_block_size(M: int, E: int, top_k: int, H: int, I: int) -> int:
    return int(load_library().moe_pick_block_size(M, E, top_k, H, I))


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(int(status)).decode()


def moe_workspace_size_fp8(M_max: int, E: int, top_k: int, H: int, I: int,
                           block_size_m: int = 0) -> int:
    n = load_library().moe_workspace_size_fp8(M_max, E, top_k, H, I, block_size_m)
    if n == 0:
        raise MoeError(2, "moe_workspace_size_fp8")
    return int(n)


class Workspace:
    """One caller-owned workspace buffer, sized once and reused by every call
    (fp8=True sizes it for moe_forward_fp8)."""

    def __init__(self, M_max: int, E: int, top_k: int, H: int, I: int, block_size_m: int = 0,
                 device=None, stream=None, fp8: bool = False):
        size = moe_workspace_size_fp8 if fp8 else moe_workspace_size
        self.nbytes = size(M_max, E, top_k, H, I, block_size_m)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        moe_workspace_init(self.buf, stream=stream)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())


def _ws(ws):
    if isinstance(ws, Workspace):
        return ws.ptr, ws.nbytes
    return _p(ws), ws.numel() * ws.element_size()


def moe_workspace_init(ws, stream=None) -> None:
    ptr, n = _ws(ws)
    _ok(load_library().moe_workspace_init(ptr, n, _stream(stream)), "moe_workspace_init")


def moe_selftest_device_timeout(ws, limit_ms: int = 100, stream=None) -> None:
    """Runs the device timeout self-test; read the result with moe_get_device_status."""
    ptr, n = _ws(ws)
    _ok(load_library().moe_selftest_device_timeout(ptr, n, int(limit_ms), _stream(stream)),
        "moe_selftest_device_timeout")


def moe_get_device_status(ws, stream=None) -> int:
    """Synchronises the stream; returns and clears the device status word.
    ws=None reads only the library-wide word of the entry points that take no
    workspace."""
    ptr = None if ws is None else _ws(ws)[0]
    return int(load_library().moe_get_device_status(ptr, _stream(stream)))


# ----------------------------------------------------------------------------- the steps

def moe_router_logits(x, w_router, logits, router_bias=None, stream=None) -> None:
    _check_dtype(x, torch.bfloat16, "x")
    _check_dtype(w_router, torch.bfloat16, "w_router")
    _check_dtype(logits, torch.bfloat16, "logits")
    _check_dtype(router_bias, torch.float32, "router_bias")
    M, H = x.shape
    E = w_router.shape[0]
    _ok(load_library().moe_router_logits(_p(x), _p(w_router), _p(router_bias), M, E, H, _p(logits),
                                         _stream(stream)), "moe_router_logits")


def moe_topk_softmax(logits, top_k: int, topk_ids, topk_weights, renormalize: bool = True,
                     stream=None) -> None:
    _check_dtype(logits, torch.bfloat16, "logits")
    _check_dtype(topk_ids, torch.int32, "topk_ids")
    _check_dtype(topk_weights, torch.float32, "topk_weights")
    M, E = logits.shape
    _ok(load_library().moe_topk_softmax(_p(logits), M, E, top_k, int(bool(renormalize)),
                                        _p(topk_ids), _p(topk_weights), _stream(stream)),
        "moe_topk_softmax")


def moe_align_block_size(topk_ids, E: int, block_size_m: int, sorted_token_ids, expert_ids,
                         expert_offsets, num_tokens_post_padded, ws, stream=None) -> None:
    _check_dtype(topk_ids, torch.int32, "topk_ids")
    M, top_k = topk_ids.shape
    ptr, n = _ws(ws)
    _ok(load_library().moe_align_block_size(_p(topk_ids), M, top_k, E, block_size_m,
                                            _p(sorted_token_ids), _p(expert_ids),
                                            _p(expert_offsets), _p(num_tokens_post_padded), ptr, n,
                                            _stream(stream)), "moe_align_block_size")


def moe_route(top_k: int, block_size_m: int, topk_ids, topk_weights, sorted_token_ids,
              expert_ids, expert_offsets, num_tokens_post_padded, ws, *, x=None, w_router=None,
              router_logits=None, router_bias=None, renormalize: bool = True,
              router_logits_out=None, stream=None) -> None:
    """Router logits (or the given logits), top-k and align in as few launches as the shape allows.
    router_logits_out [M, E] bf16 (with w_router) receives the logits the routing used."""
    for t, n in ((x, "x"), (w_router, "w_router"), (router_logits, "router_logits")):
        _check_dtype(t, torch.bfloat16, n)
    _check_dtype(router_bias, torch.float32, "router_bias")
    _check_dtype(topk_ids, torch.int32, "topk_ids")
    _check_dtype(topk_weights, torch.float32, "topk_weights")
    _check_dtype(router_logits_out, torch.bfloat16, "router_logits_out")
    if w_router is not None:
        M, H = x.shape
        E = w_router.shape[0]
    else:
        M, E = router_logits.shape
        H = 16
    ptr, n = _ws(ws)
    _ok(load_library().moe_route(_p(x), _p(w_router), _p(router_logits), _p(router_bias), M, E,
                                 top_k, H, int(bool(renormalize)), block_size_m, _p(topk_ids),
                                 _p(topk_weights), _p(sorted_token_ids), _p(expert_ids),
                                 _p(expert_offsets), _p(num_tokens_post_padded),
                                 _p(router_logits_out), ptr, n, _stream(stream)), "moe_route")


def moe_grouped_gemm_w13_act(x, w13, sorted_token_ids, expert_ids, num_tokens_post_padded,
                             top_k: int, block_size_m: int, a, stream=None) -> None:
    _check_dtype(x, torch.bfloat16, "x")
    _check_dtype(w13, torch.bfloat16, "w13")
    _check_dtype(a, torch.bfloat16, "a")
    M, H = x.shape
    E, twoI, _ = w13.shape
    _ok(load_library().moe_grouped_gemm_w13_act(_p(x), _p(w13), _p(sorted_token_ids),
                                                _p(expert_ids), _p(num_tokens_post_padded), M,
                                                top_k, E, H, twoI // 2, block_size_m, _p(a),
                                                _stream(stream)), "moe_grouped_gemm_w13_act")


def moe_grouped_gemm_w2_combine(a, w2, sorted_token_ids, expert_ids, num_tokens_post_padded,
                                topk_weights, top_k: int, block_size_m: int, y, ws,
                                residual=None, stream=None) -> None:
    _check_dtype(a, torch.bfloat16, "a")
    _check_dtype(w2, torch.bfloat16, "w2")
    _check_dtype(y, torch.bfloat16, "y")
    _check_dtype(topk_weights, torch.float32, "topk_weights")
    _check_dtype(residual, torch.bfloat16, "residual")
    M, H = y.shape
    E, _, I = w2.shape
    ptr, n = _ws(ws)
    _ok(load_library().moe_grouped_gemm_w2_combine(_p(a), _p(w2), _p(sorted_token_ids),
                                                   _p(expert_ids), _p(num_tokens_post_padded),
                                                   _p(topk_weights), _p(residual), M, top_k, E, H,
                                                   I, block_size_m, _p(y), ptr, n, _stream(stream)),
        "moe_grouped_gemm_w2_combine")


def moe_grouped_gemm_w2_combine_noalloc(a, w2, sorted_token_ids, expert_ids,
                                        num_tokens_post_padded, topk_weights, top_k: int,
                                        block_size_m: int, y, residual=None, stream=None) -> None:
    """GEMM 2 + combine with the library's built-in accumulator (no workspace).

    For callers that cannot allocate device memory.  M * H must not exceed
    2,097,152; calls that overlap on the GPU share the accumulator and race."""
    _check_dtype(a, torch.bfloat16, "a")
    _check_dtype(w2, torch.bfloat16, "w2")
    _check_dtype(y, torch.bfloat16, "y")
    _check_dtype(topk_weights, torch.float32, "topk_weights")
    _check_dtype(residual, torch.bfloat16, "residual")
    M, H = y.shape
    E, _, I = w2.shape
    _ok(load_library().moe_grouped_gemm_w2_combine_noalloc(
        _p(a), _p(w2), _p(sorted_token_ids), _p(expert_ids), _p(num_tokens_post_padded),
        _p(topk_weights), _p(residual), M, top_k, E, H, I, block_size_m, _p(y), _stream(stream)),
        "moe_grouped_gemm_w2_combine_noalloc")


def moe_forward(x, w13, w2, top_k: int, y, ws, *, w_router=None, router_logits=None,
                router_bias=None, residual=None, renormalize: bool = True, block_size_m: int = 0,
                topk_ids_out=None, topk_weights_out=None, router_logits_out=None,
                stream=None) -> None:
    for t, n in ((x, "x"), (w13, "w13"), (w2, "w2"), (y, "y"), (w_router, "w_router"),
                 (router_logits, "router_logits"), (residual, "residual"),
                 (router_logits_out, "router_logits_out")):
        _check_dtype(t, torch.bfloat16, n)
    _check_dtype(router_bias, torch.float32, "router_bias")
    _check_dtype(topk_ids_out, torch.int32, "topk_ids_out")
    _check_dtype(topk_weights_out, torch.float32, "topk_weights_out")
    M, H = x.shape
    E, twoI, _ = w13.shape
    ptr, n = _ws(ws)
    _ok(load_library().moe_forward(_p(x), _p(w_router), _p(router_logits), _p(router_bias),
                                   _p(w13), _p(w2), _p(residual), M, E, top_k, H, twoI // 2,
                                   int(bool(renormalize)), block_size_m, _p(y), _p(topk_ids_out),
                                   _p(topk_weights_out), _p(router_logits_out), ptr, n,
                                   _stream(stream)), "moe_forward")


# ----------------------------------------------------------------------------- FP8 (E4M3) weights
# Codes are torch.uint8 tensors (E4M3 bit patterns, e.g. a float8_e4m3fn tensor
# viewed as uint8); scales are fp32, one per row.

def moe_quantize_rows_fp8(src, q, scales, stream=None) -> None:
    """Per-row dynamic E4M3 quantization: scales[r] = amax|src[r]| / 448, q = e4m3(src / s)."""
    _check_dtype(src, torch.bfloat16, "src")
    _check_dtype(q, torch.uint8, "q")
    _check_dtype(scales, torch.float32, "scales")
    R, K = src.shape
    _ok(load_library().moe_quantize_rows_fp8(_p(src), R, K, _p(q), _p(scales), _stream(stream)),
        "moe_quantize_rows_fp8")


def moe_grouped_gemm_w13_act_fp8(qx, x_scales, w13, w13_scales, sorted_token_ids, expert_ids,
                                 num_tokens_post_padded, top_k: int, block_size_m: int, a,
                                 stream=None) -> None:
    for t, n in ((qx, "qx"), (w13, "w13")):
        _check_dtype(t, torch.uint8, n)
    for t, n in ((x_scales, "x_scales"), (w13_scales, "w13_scales")):
        _check_dtype(t, torch.float32, n)
    _check_dtype(a, torch.bfloat16, "a")
    M, H = qx.shape
    E, twoI, _ = w13.shape
    _ok(load_library().moe_grouped_gemm_w13_act_fp8(
        _p(qx), _p(x_scales), _p(w13), _p(w13_scales), _p(sorted_token_ids), _p(expert_ids),
        _p(num_tokens_post_padded), M, top_k, E, H, twoI // 2, block_size_m, _p(a),
        _stream(stream)), "moe_grouped_gemm_w13_act_fp8")


def moe_grouped_gemm_w2_combine_fp8(qa, a_scales, w2, w2_scales, sorted_token_ids, expert_ids,
                                    num_tokens_post_padded, topk_weights, top_k: int,
                                    block_size_m: int, y, ws, residual=None, stream=None) -> None:
    for t, n in ((qa, "qa"), (w2, "w2")):
        _check_dtype(t, torch.uint8, n)
    for t, n in ((a_scales, "a_scales"), (w2_scales, "w2_scales"), (topk_weights, "topk_weights")):
        _check_dtype(t, torch.float32, n)
    _check_dtype(y, torch.bfloat16, "y")
    _check_dtype(residual, torch.bfloat16, "residual")
    M, H = y.shape
    E, _, I = w2.shape
    ptr, n = _ws(ws)
    _ok(load_library().moe_grouped_gemm_w2_combine_fp8(
        _p(qa), _p(a_scales), _p(w2), _p(w2_scales), _p(sorted_token_ids), _p(expert_ids),
        _p(num_tokens_post_padded), _p(topk_weights), _p(residual), M, top_k, E, H, I,
        block_size_m, _p(y), ptr, n, _stream(stream)), "moe_grouped_gemm_w2_combine_fp8")


def moe_forward_fp8(x, w13, w13_scales, w2, w2_scales, top_k: int, y, ws, *, w_router=None,
                    router_logits=None, router_bias=None, residual=None,
                    renormalize: bool = True, block_size_m: int = 0, topk_ids_out=None,
                    topk_weights_out=None, router_logits_out=None, stream=None) -> None:
    for t, n in ((x, "x"), (y, "y"), (w_router, "w_router"), (router_logits, "router_logits"),
                 (residual, "residual"), (router_logits_out, "router_logits_out")):
        _check_dtype(t, torch.bfloat16, n)
    for t, n in ((w13, "w13"), (w2, "w2")):
        _check_dtype(t, torch.uint8, n)
    for t, n in ((w13_scales, "w13_scales"), (w2_scales, "w2_scales"),
                 (router_bias, "router_bias"), (topk_weights_out, "topk_weights_out")):
        _check_dtype(t, torch.float32, n)
    _check_dtype(topk_ids_out, torch.int32, "topk_ids_out")
    M, H = x.shape
    E, twoI, _ = w13.shape
    ptr, n = _ws(ws)
    _ok(load_library().moe_forward_fp8(
        _p(x), _p(w_router), _p(router_logits), _p(router_bias), _p(w13), _p(w13_scales), _p(w2),
        _p(w2_scales), _p(residual), M, E, top_k, H, twoI // 2, int(bool(renormalize)),
        block_size_m, _p(y), _p(topk_ids_out), _p(topk_weights_out), _p(router_logits_out), ptr, n,
        _stream(stream)), "moe_forward_fp8")
