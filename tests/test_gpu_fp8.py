"""FP8 (E4M3) expert weights on the GPU against the oracle.

The reading taken (the vLLM page, "fused_experts_impl", leaves format and
scale granularity open): E4M3 codes with one fp32 scale per output row of
W13 and W2, activations quantized per row at run time (x per token, a per
pair) with s = amax / 448, dequantization after the fp32 sums.

Comparisons:
  - the per-row quantization decides every code in fp32 with correctly
    rounded division on both sides, so codes and scales match bit for bit;
  - each grouped GEMM gets the oracle's quantized inputs and is compared at
    the output tolerance of the bf16 layer (tests/_util.py);
  - the layer quantizes its own a: where the GPU's a differs from the
    oracle's by a bf16 rounding, that row's codes may differ too, which the
    output tolerance covers (one code step is 2^-3 relative, on one pair);
  - routing is checked as in tests/test_gpu_parity.py (the router is bf16).
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_renorm_gb300 as moe
import oracle
import synth
from _util import W_ABS, assert_close_bf16, bits
from test_gpu_parity import align_on_device, assert_routing_explained, check_logits, run_route

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_renorm_gb300 import _build
    _build.build()
    moe.load_library()
    oracle.build()
    oracle.set_threads(max(1, len(__import__("os").sched_getaffinity(0))))


def rand_bf16(shape, std, seed, device=DEV):
    return synth.normal_bf16(shape, std, seed, device)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


# ----------------------------------------------------------------------------- quantization

def special_rows(K, seed):
    """Rows that reach the edges of the quantization: zeros (+0 and -0), one
    nonzero, tiny values (codes in the subnormal range), large values, equal
    magnitudes of both signs, values whose quotient lands on code midpoints."""
    g = torch.Generator().manual_seed(seed)
    rows = [torch.zeros(K), -torch.zeros(K)]
    one = torch.zeros(K)
    one[K // 3] = -3.5
    rows.append(one)
    rows.append(torch.randn(K, generator=g) * 1e-30)
    rows.append(torch.randn(K, generator=g) * 3e4)
    pm = torch.full((K,), 0.75)
    pm[::2] = -0.75
    rows.append(pm)
    # amax 448: quotients are the values themselves, many of them code midpoints
    mid = torch.linspace(-448, 448, K)
    mid[0] = 448.0
    rows.append(mid)
    # a wide spread inside one row: most codes subnormal or zero
    spread = torch.randn(K, generator=g) * torch.logspace(-12, 2, K)
    rows.append(spread)
    return torch.stack(rows).to(torch.bfloat16)


# Below 4096 rows the two-pass kernel; from 4096 rows the register-resident
# one, with rows of 1, 2, 4 and 8 16-byte chunks per lane (ragged ones too)
# and more rows than one resident wave; rows past 2048 take two passes.
@pytest.mark.parametrize("R,K", [(1, 16), (37, 2048), (513, 768), (8, 1408), (300, 208),
                                 (70, 496), (4095, 2048), (4096, 2048), (6000, 768),
                                 (4099, 208), (5000, 496), (4100, 1408), (4096, 2064), (9, 4096)])
def test_quantize_rows_matches_the_oracle_bit_for_bit(R, K):
    src = rand_bf16((R, K), 1.0, 100 + R + K)
    sp = special_rows(K, R).to(DEV)
    n = min(R, sp.shape[0])
    src[:n] = sp[:n]
    q = torch.full((R, K), 0x55, dtype=torch.uint8, device=DEV)
    s = torch.full((R,), float("nan"), dtype=torch.float32, device=DEV)
    moe.moe_quantize_rows_fp8(src, q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_rows(bits(src))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32)), "scales"
    gq = q.cpu().numpy()
    bad = np.argwhere(gq != rq)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[0]}: {gq[tuple(bad[0])]:#x} vs {rq[tuple(bad[0])]:#x}"


def test_quantize_rows_byte_order_and_values():
    """A row whose codes are known from the E4M3 definition alone: amax 448
    gives the scale 1, and 448, -448, 1, 2^-9 (the smallest subnormal),
    2^-10 (a tie to 0) and 1.0625 (the midpoint between 1 and 1.125, which
    rounds to the even code of 1) become 0x7E, 0xFE, 0x38, 0x01, 0x00, 0x38
    in this order."""
    vals = [448.0, -448.0, 1.0, 2.0 ** -9, 2.0 ** -10, 1.0625] + [0.0] * 10
    src = torch.tensor([vals], dtype=torch.float32).to(torch.bfloat16).to(DEV)
    q = torch.empty((1, 16), dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    moe.moe_quantize_rows_fp8(src, q, s)
    torch.cuda.synchronize()
    assert s.item() == 1.0
    assert q.cpu().numpy()[0, :6].tolist() == [0x7E, 0xFE, 0x38, 0x01, 0x00, 0x38]


# ----------------------------------------------------------------------------- the grouped GEMMs

FP8_SHAPES = [(3, 4, 2, 128, 64, 16), (64, 128, 8, 2048, 768, 16), (64, 60, 4, 2048, 1408, 16),
              (200, 32, 4, 512, 96, 32), (128, 256, 8, 2048, 512, 16), (1, 128, 8, 2048, 768, 16),
              (300, 8, 2, 192, 48, 64), (1000, 16, 4, 320, 208, 128), (40, 3, 3, 80, 16, 16),
              # 256-token tiles (2-SM where the weight-tile count is even); ragged
              # 128-element K stages (H = 208, 80) and ragged weight tiles
              (700, 4, 2, 256, 128, 256), (1000, 16, 4, 208, 80, 256), (300, 60, 4, 512, 192, 256),
              (2000, 8, 2, 2048, 768, 256), (512, 128, 8, 2048, 768, 32)]


def fp8_weights(E, H, I, seed):
    return (synth.fp8_codes((E, 2 * I, H), seed, DEV), synth.row_scales((E, 2 * I), seed + 1, DEV),
            synth.fp8_codes((E, H, I), seed + 2, DEV), synth.row_scales((E, H), seed + 3, DEV))


def np_of(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("M,E,k,H,I,B", FP8_SHAPES)
def test_grouped_gemm_w13_act_fp8(M, E, k, H, I, B):
    seed = 5 * M + E + H
    x = rand_bf16((M, H), 1.0, seed)
    lg = rand_bf16((M, E), 1.0, seed + 9, "cpu")
    w13, s13, _, _ = fp8_weights(E, H, I, seed)
    qx, sx = oracle.quant_rows(bits(x))
    ids, _ = oracle.topk_softmax(bits(lg), k)
    s, e, n = align_on_device(ids, E, B)
    a = torch.full((M * k, I), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_grouped_gemm_w13_act_fp8(dev(qx), dev(sx), w13, s13, s, e, n, k, B, a)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(None) == 0
    ref = oracle.expert_act_fp8(qx, sx, np_of(w13), np_of(s13), ids)
    assert_close_bf16(bits(a), ref, "a")


@pytest.mark.parametrize("M,E,k,H,I,B", FP8_SHAPES)
@pytest.mark.parametrize("with_residual", [False, True])
def test_grouped_gemm_w2_combine_fp8(M, E, k, H, I, B, with_residual):
    seed = 7 * M + E + I
    lg = rand_bf16((M, E), 1.0, seed + 9, "cpu")
    _, _, w2, s2 = fp8_weights(E, H, I, seed)
    ids, w = oracle.topk_softmax(bits(lg), k)
    # an activation with the spread of SiLU(h_gate) * h_up, quantized per pair
    a_bits = bits(rand_bf16((M * k, I), 0.05, seed + 4, "cpu"))
    qa, sa = oracle.quant_rows(a_bits)
    res = rand_bf16((M, H), 1.0, 77) if with_residual else None
    s, e, n = align_on_device(ids, E, B)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    ws = moe.Workspace(M, E, k, H, I, B)
    moe.moe_grouped_gemm_w2_combine_fp8(dev(qa), dev(sa), w2, s2, s, e, n, dev(w), k, B, y, ws,
                                        residual=res)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    ref = oracle.expert_down_combine_fp8(qa, sa, np_of(w2), np_of(s2), ids, w,
                                         None if res is None else bits(res))
    assert_close_bf16(bits(y), ref, "y")


def test_two_sm_fp8_gemm1_equals_one_cta_tiles(monkeypatch):
    """256-token 2-SM tiles on E4M3 operands (one kind::f8f6f4 M = 256 MMA
    over both CTAs' shared memory) give the bits of one CTA per tile."""
    w = synth.WORKLOADS[3]
    M, B = 4096, 256
    wt = synth.layer_weights_fp8(w, device=DEV)
    x = synth.layer_input(w, M, device=DEV)["x"]
    out, _ = run_route(M, w.E, w.top_k, B, x=x, wr=wt["w_router"], bias=wt["router_bias"])
    s, e, n = (torch.from_numpy(out[key]).to(DEV) for key in ("s", "e", "n"))
    qx = torch.empty((M, w.H), dtype=torch.uint8, device=DEV)
    sx = torch.empty(M, dtype=torch.float32, device=DEV)
    moe.moe_quantize_rows_fp8(x, qx, sx)
    P = M * w.top_k
    monkeypatch.setenv("MOE_FORCE_PATH", "tc1")
    a_one = torch.empty((P, w.I), dtype=torch.bfloat16, device=DEV)
    moe.moe_grouped_gemm_w13_act_fp8(qx, sx, wt["w13"], wt["w13_scale"], s, e, n, w.top_k, B, a_one)
    torch.cuda.synchronize()
    ref_bits = bits(a_one)
    monkeypatch.setenv("MOE_FORCE_PATH", "tc")
    a_two = torch.empty_like(a_one)
    for run in range(5):
        a_two.fill_(float("nan"))
        moe.moe_grouped_gemm_w13_act_fp8(qx, sx, wt["w13"], wt["w13_scale"], s, e, n, w.top_k, B,
                                         a_two)
        torch.cuda.synchronize()
        assert np.array_equal(bits(a_two), ref_bits), f"run {run}: 2-SM tiles differ"
    assert moe.moe_get_device_status(None) == 0
    g = torch.Generator().manual_seed(4097)
    tok = torch.randperm(M, generator=g)[:24].sort().values.numpy()
    rq, rs = oracle.quant_rows(bits(x)[tok])
    ref = oracle.expert_act_fp8(rq, rs, np_of(wt["w13"]), np_of(wt["w13_scale"]), out["ids"][tok])
    pairs = (tok[:, None] * w.top_k + np.arange(w.top_k)[None, :]).reshape(-1)
    assert_close_bf16(ref_bits[pairs], ref, "a (sampled pairs)")


# ----------------------------------------------------------------------------- the layer

def run_forward_fp8(x, wt, k, *, lg=None, wr=None, bias=None, res=None, B=0, renorm=True):
    M, H = x.shape
    E, twoI, _ = wt["w13"].shape
    y = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((M, k), dtype=torch.float32, device=DEV)
    lgo = torch.empty((M, E), dtype=torch.bfloat16, device=DEV) if wr is not None else None
    ws = moe.Workspace(M, E, k, H, twoI // 2, B, fp8=True)
    moe.moe_forward_fp8(x, wt["w13"], wt["w13_scale"], wt["w2"], wt["w2_scale"], k, y, ws,
                        w_router=wr, router_logits=lg, router_bias=bias, residual=res,
                        renormalize=renorm, block_size_m=B, topk_ids_out=ids, topk_weights_out=wts,
                        router_logits_out=lgo)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return bits(y), ids.cpu().numpy(), wts.cpu().numpy(), None if lgo is None else bits(lgo)


def oracle_fp8(x_bits, wt, k, lg_bits, res_bits=None, renorm=True):
    return oracle.moe_forward_fp8(x_bits, np_of(wt["w13"]), np_of(wt["w13_scale"]),
                                  np_of(wt["w2"]), np_of(wt["w2_scale"]), k,
                                  router_logits=lg_bits, residual=res_bits, renormalize=renorm)


@pytest.mark.parametrize("M,E,k,H,I,B", [(3, 4, 2, 128, 64, 16), (1, 60, 4, 2048, 1408, 0),
                                         (64, 60, 4, 2048, 1408, 0), (21, 9, 9, 64, 48, 0),
                                         (300, 64, 6, 256, 128, 0), (700, 8, 2, 208, 80, 256),
                                         # K splits over few 128-element stages: GEMM 2 splits
                                         # 6 stages four ways, GEMM 1 (H = 384) 3 stages three ways
                                         (6, 128, 8, 2048, 768, 0), (6, 128, 8, 384, 208, 0)])
@pytest.mark.parametrize("renorm", [True, False])
def test_forward_fp8_given_logits(M, E, k, H, I, B, renorm):
    seed = 11 * M + E
    x = rand_bf16((M, H), 1.0, seed)
    lg = rand_bf16((M, E), 1.0, seed + 1, "cpu")
    w13, s13, w2, s2 = fp8_weights(E, H, I, seed + 2)
    wt = {"w13": w13, "w13_scale": s13, "w2": w2, "w2_scale": s2}
    yb, ids, wts, _ = run_forward_fp8(x, wt, k, lg=lg.to(DEV), B=B, renorm=renorm)
    ref = oracle_fp8(bits(x), wt, k, bits(lg), renorm=renorm)
    assert np.array_equal(ids, ref["topk_ids"])
    assert np.abs(wts.astype(np.float64) - ref["topk_weights"]).max() <= W_ABS
    assert_close_bf16(yb, ref["y"], "y")


@pytest.mark.parametrize("cfg,M,sampled", [(1, 3, False), (2, 1, False), (2, 6, False), (2, 8, False),
                                           (2, 64, False), (4, 16, False), (3, 4096, True),
                                           (3, 16384, True), (5, 8192, True)])
def test_forward_fp8_on_workloads(cfg, M, sampled):
    """The workloads with E4M3 expert weights: routing (bf16 router) explained
    against the oracle's, y equal to the oracle's FP8 layer on the GPU's
    logits; the prefill sizes on a sample of tokens (every step of the layer
    is per token or per pair, so a token's output depends on its row alone)."""
    w = synth.WORKLOADS[cfg]
    wt = synth.layer_weights_fp8(w, device=DEV)
    inp = synth.layer_input(w, M, device=DEV)
    x, lg = inp["x"], inp["router_logits"]
    res = x if w.residual else None
    yb, ids, _, g_lg = run_forward_fp8(x, wt, w.top_k, lg=lg, wr=wt["w_router"],
                                       bias=wt["router_bias"], res=res, B=w.block_size_m)
    tok = np.arange(M)
    if sampled:
        g = torch.Generator().manual_seed(M + 1)
        tok = torch.randperm(M, generator=g)[:48].sort().values.numpy()
    xb = bits(x)[tok]
    res_b = None if res is None else xb
    if wt["w_router"] is None:
        ref = oracle_fp8(xb, wt, w.top_k, bits(lg)[tok], res_b)
    else:
        g_lg = g_lg[tok]
        check_logits(g_lg, x[torch.from_numpy(tok).to(DEV)], wt["w_router"], wt["router_bias"])
        bias = None if wt["router_bias"] is None else wt["router_bias"].cpu().numpy()
        o_lg = oracle.router_logits(xb, bits(wt["w_router"]), bias)
        o_ids, _ = oracle.topk_softmax(o_lg, w.top_k)
        nd = assert_routing_explained(g_lg, ids[tok], o_lg, o_ids, w.top_k)
        assert nd <= max(1, 0.02 * len(tok))
        ref = oracle_fp8(xb, wt, w.top_k, g_lg, res_b)
    assert np.array_equal(ids[tok], ref["topk_ids"])
    assert_close_bf16(yb[tok], ref["y"], "y")

