"""The C-ABI library loads, exports every symbol include/moe_api.h declares,
and rejects bad arguments on the host before launching anything.

No compute call is made here.  The argument-check cases run only where no
GPU is visible: there an argument check that wrongly let a call through
would end in a CUDA error code (no device), never in a kernel.
"""
import ctypes
import os
import re

import pytest
import torch

import mixture_experts_layer_renorm_gb300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_api.h")

OK, INVALID, SHAPE, WS_SMALL = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_renorm_gb300 import _build
    _build.build()
    return moe.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_bound_functions():
    assert declared_functions() == sorted(moe.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in moe.STATUS_NAMES.items():
        assert moe.moe_status_string(code) == name
    assert moe.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_sizes_and_capacity(lib):
    assert moe.moe_align_capacity(3, 2, 4, 4) == 20           # 6 pairs + 4 experts * 3 = 18 -> 20
    assert moe.moe_align_capacity(1, 8, 128, 16) == 1936       # 8 + 128*15 = 1928 -> 1936
    assert moe.moe_align_capacity(16384, 8, 128, 128) == 147328
    assert lib.moe_align_capacity(1, 8, 128, 0) == -1          # B must be explicit
    assert lib.moe_align_capacity(1, 9, 8, 16) == -1           # top_k > E
    n = moe.moe_workspace_size(64, 128, 8, 2048, 768, 16)
    assert n >= 64 * 8 * 768 * 2 + 64 * 2048 * 4
    assert moe.moe_workspace_size(64, 128, 8, 2048, 768, 0) >= n
    assert lib.moe_workspace_size(64, 128, 8, 2047, 768, 16) == 0   # H not a multiple of 16
    assert lib.moe_workspace_size(64, 2000, 8, 2048, 768, 16) == 0  # E > 1024
    assert lib.moe_workspace_size(64, 128, 8, 2048, 768, 257) == 0  # block size > 256
    for B in (1, 4, 8, 24, 200):                                    # any block size in [1, 256]
        assert moe.moe_workspace_size(3, 4, 2, 128, 64, B) > 0
    # a batch below M_max may need more (it reserves split-K scratch): the size covers it
    assert moe.moe_workspace_size(300, 128, 8, 2048, 768, 16) >= moe.moe_workspace_size(256, 128, 8, 2048, 768, 16)
    # and the router's split scratch (up to 60 tiles of 128 tokens): sizes never
    # shrink as M_max grows, across both limits (E = 128: 7680 tokens; E = 1024:
    # 15 tiles of four weight tiles, 1920 tokens), for the bf16 and E4M3 layers
    for E, edge in ((128, 7680), (1024, 1920)):
        for size in (moe.moe_workspace_size, moe.moe_workspace_size_fp8):
            Ms = [edge - 128, edge - 1, edge, edge + 1, edge + 128, 2 * edge]
            sizes = [size(M, E, 8, 2048, 768, 0) for M in Ms]
            assert all(b >= a for a, b in zip(sizes, sizes[1:])), (E, size.__name__, sizes)
    for M in (1, 8, 64, 512, 4096, 16384):
        assert moe.moe_pick_block_size(M, 128, 8, 2048, 768) in (16, 32, 64, 128, 256)
    # blocks a few times the mean group: 16 up to 6 pairs per expert, 32 up to
    # 12, 64 up to 24, 128 up to 64
    assert moe.moe_pick_block_size(64, 128, 8, 2048, 768) == 16         # 4 per expert
    assert moe.moe_pick_block_size(128, 128, 8, 2048, 768) == 32        # 8 per expert
    assert moe.moe_pick_block_size(256, 128, 8, 2048, 768) == 64        # 16 per expert
    assert moe.moe_pick_block_size(512, 128, 8, 2048, 768) == 128       # 32 per expert
    assert moe.moe_pick_block_size(1024, 128, 8, 2048, 768) == 128      # 64 per expert
    # then 256-token tiles where both GEMMs run 2-SM tiles (even weight-tile
    # counts: ceil(I/64) and ceil(H/128)), else from 1024 per expert
    assert moe.moe_pick_block_size(2048, 128, 8, 2048, 768) == 256      # 128 per expert, 12 and 16 tiles
    assert moe.moe_pick_block_size(4096, 128, 8, 2048, 768) == 256      # 256 per expert
    assert moe.moe_pick_block_size(8192, 60, 4, 2048, 1408) == 256      # 546 per expert, 22 and 16 tiles
    assert moe.moe_pick_block_size(4096, 128, 8, 2048, 704) == 128      # 11 GEMM-1 weight tiles
    assert moe.moe_pick_block_size(16384, 128, 8, 2048, 704) == 256     # 1024 per expert


needs_no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                                  reason="host-only argument checks use fake device pointers")

FAKE = ctypes.c_void_p(1 << 20)     # 16- and 256-byte aligned, never dereferenced
FAKE_MIS = ctypes.c_void_p((1 << 20) + 8)
NULL = None
S = None  # default stream


@needs_no_gpu
def test_forward_argument_checks(lib):
    f = lib.moe_forward
    big = 1 << 40
    args = dict(x=FAKE, wr=FAKE, lg=NULL, bias=NULL, w13=FAKE, w2=FAKE, res=NULL, M=4, E=8, k=2,
                H=64, I=32, renorm=1, B=16, y=FAKE, ids=NULL, wts=NULL, lgo=NULL, ws=FAKE, wsb=big)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["x"], a["wr"], a["lg"], a["bias"], a["w13"], a["w2"], a["res"], a["M"], a["E"],
                 a["k"], a["H"], a["I"], a["renorm"], a["B"], a["y"], a["ids"], a["wts"], a["lgo"],
                 a["ws"], a["wsb"], S)

    assert call(M=0) == OK                      # M == 0 is a no-op
    assert call(M=-1) == INVALID
    assert call(E=0) == SHAPE
    assert call(E=1025) == SHAPE
    assert call(k=9) == SHAPE                   # top_k > E
    assert call(k=0) == SHAPE
    assert call(E=64, k=33) == SHAPE            # top_k > 32
    assert call(H=60) == SHAPE                  # not a multiple of 16
    assert call(I=8) == SHAPE
    assert call(B=257) == SHAPE
    assert call(B=-3) == SHAPE
    assert call(lg=FAKE) == INVALID             # both router weights and logits
    assert call(wr=NULL) == INVALID             # neither
    assert call(wr=NULL, lg=FAKE, bias=FAKE) == INVALID  # a bias without router weights
    assert call(x=NULL) == INVALID
    assert call(w13=NULL) == INVALID
    assert call(y=NULL) == INVALID
    assert call(ws=NULL) == INVALID
    assert call(x=FAKE_MIS) == INVALID          # misaligned matrix
    assert call(ws=FAKE_MIS) == INVALID         # misaligned workspace
    need = moe.moe_workspace_size(4, 8, 2, 64, 32, 16)
    assert call(wsb=need - 1) == WS_SMALL


@needs_no_gpu
def test_step_argument_checks(lib):
    assert lib.moe_topk_softmax(FAKE, 4, 8, 9, 1, FAKE, FAKE, S) == SHAPE
    assert lib.moe_topk_softmax(FAKE, -1, 8, 2, 1, FAKE, FAKE, S) == INVALID
    assert lib.moe_topk_softmax(NULL, 4, 8, 2, 1, FAKE, FAKE, S) == INVALID
    assert lib.moe_topk_softmax(FAKE, 0, 8, 2, 1, FAKE, FAKE, S) == OK
    assert lib.moe_router_logits(FAKE, FAKE, NULL, 4, 8, 63, FAKE, S) == SHAPE
    assert lib.moe_router_logits(NULL, FAKE, NULL, 4, 8, 64, FAKE, S) == INVALID
    assert lib.moe_align_block_size(FAKE, 4, 2, 8, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, S) == SHAPE
    assert lib.moe_align_block_size(FAKE, 4, 2, 8, 16, FAKE, FAKE, FAKE, FAKE, NULL, 1 << 20, S) == INVALID
    assert lib.moe_align_block_size(FAKE, 4, 2, 8, 16, FAKE, FAKE, FAKE, FAKE, FAKE, 16, S) == WS_SMALL
    assert lib.moe_grouped_gemm_w13_act(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 8, 64, 32, 0, FAKE, S) == SHAPE
    assert lib.moe_grouped_gemm_w13_act(FAKE, NULL, FAKE, FAKE, FAKE, 4, 2, 8, 64, 32, 16, FAKE, S) == INVALID
    assert lib.moe_grouped_gemm_w2_combine(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 4, 2, 8, 64, 32,
                                           16, FAKE, FAKE, 64, S) == WS_SMALL
    assert lib.moe_grouped_gemm_w2_combine(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, NULL, 4, 2, 8, 64, 32,
                                           16, FAKE, FAKE, 1 << 30, S) == INVALID
    assert lib.moe_workspace_init(NULL, 1024, S) == INVALID
    assert lib.moe_workspace_init(FAKE_MIS, 1024, S) == INVALID
    # no workspace: only the library-wide word, which needs a device to read
    assert lib.moe_get_device_status(NULL, S) == 4  # MOE_ERR_CUDA
    assert lib.moe_selftest_device_timeout(NULL, 1 << 20, 10, S) == INVALID
    assert lib.moe_selftest_device_timeout(FAKE_MIS, 1 << 20, 10, S) == INVALID
    assert lib.moe_selftest_device_timeout(FAKE, 16, 10, S) == INVALID   # smaller than the status block


def test_fp8_sizes(lib):
    n = moe.moe_workspace_size(64, 128, 8, 2048, 768, 16)
    n8 = moe.moe_workspace_size_fp8(64, 128, 8, 2048, 768, 16)
    # plus x codes [64, 2048], a codes [512, 768] and their row scales
    assert n8 >= n + 64 * 2048 + 512 * 768 + (64 + 512) * 4
    assert lib.moe_workspace_size_fp8(64, 128, 8, 2048, 768, 24) == 0   # not a tensor-core tile
    assert lib.moe_workspace_size_fp8(64, 128, 8, 2040, 768, 16) == 0
    assert moe.moe_workspace_size_fp8(64, 128, 8, 2048, 768, 0) >= n8


@needs_no_gpu
def test_fp8_argument_checks(lib):
    q = lib.moe_quantize_rows_fp8
    assert q(FAKE, 0, 64, FAKE, FAKE, S) == OK
    assert q(FAKE, -1, 64, FAKE, FAKE, S) == INVALID
    assert q(FAKE, 4, 60, FAKE, FAKE, S) == SHAPE            # K not a multiple of 16
    assert q(NULL, 4, 64, FAKE, FAKE, S) == INVALID
    assert q(FAKE, 4, 64, FAKE_MIS, FAKE, S) == INVALID      # misaligned codes
    assert q(FAKE, 4, 64, FAKE, NULL, S) == INVALID
    g1 = lib.moe_grouped_gemm_w13_act_fp8
    assert g1(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 8, 64, 32, 24, FAKE, S) == SHAPE
    assert g1(FAKE, NULL, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 8, 64, 32, 16, FAKE, S) == INVALID
    assert g1(FAKE, FAKE, FAKE, NULL, FAKE, FAKE, FAKE, 4, 2, 8, 64, 32, 16, FAKE, S) == INVALID
    assert g1(FAKE_MIS, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 8, 64, 32, 16, FAKE, S) == INVALID
    g2 = lib.moe_grouped_gemm_w2_combine_fp8
    assert g2(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 4, 2, 8, 64, 32, 16, FAKE, FAKE,
              64, S) == WS_SMALL
    assert g2(FAKE, FAKE, FAKE, NULL, FAKE, FAKE, FAKE, FAKE, NULL, 4, 2, 8, 64, 32, 16, FAKE, FAKE,
              1 << 30, S) == INVALID
    assert g2(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 4, 2, 8, 64, 32, 1, FAKE, FAKE,
              1 << 30, S) == SHAPE
    f = lib.moe_forward_fp8
    args = dict(x=FAKE, wr=FAKE, lg=NULL, bias=NULL, w13=FAKE, s13=FAKE, w2=FAKE, s2=FAKE, res=NULL,
                M=4, E=8, k=2, H=64, I=32, renorm=1, B=16, y=FAKE, ids=NULL, wts=NULL, lgo=NULL,
                ws=FAKE, wsb=1 << 40)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["x"], a["wr"], a["lg"], a["bias"], a["w13"], a["s13"], a["w2"], a["s2"],
                 a["res"], a["M"], a["E"], a["k"], a["H"], a["I"], a["renorm"], a["B"], a["y"],
                 a["ids"], a["wts"], a["lgo"], a["ws"], a["wsb"], S)

    assert call(M=0) == OK
    assert call(M=-1) == INVALID
    assert call(B=48) == SHAPE                  # the FP8 GEMMs tile 16..256 powers of two only
    assert call(H=56) == SHAPE
    assert call(lg=FAKE) == INVALID
    assert call(s13=NULL) == INVALID
    assert call(s2=NULL) == INVALID
    assert call(w2=FAKE_MIS) == INVALID
    assert call(ws=FAKE_MIS) == INVALID
    need = moe.moe_workspace_size_fp8(4, 8, 2, 64, 32, 16)
    assert call(wsb=need - 1) == WS_SMALL
    assert need > moe.moe_workspace_size(4, 8, 2, 64, 32, 16)


def test_product_path_fails_loudly_without_the_library(monkeypatch, tmp_path):
    from mixture_experts_layer_renorm_gb300 import _build
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        moe.load_library()
