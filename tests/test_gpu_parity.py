"""Parity of every C-ABI entry point against the CPU oracle, on the GPU.

The CUDA path and the oracle get the same seeded inputs (module `synth`);
nothing the CUDA path produces is fed to the oracle except, where a test says
so, the router logits the GPU decided on: those are first checked on their
own (each must be the bf16 rounding of a value within the fp32 summation
error bound of the exact dot product), then the GPU's routing must equal the
oracle's top-k of those very logits bit for bit, and the layer output must
match the oracle run on them -- on every token, at the output tolerance
(tests/_util.py).  Where the oracle's own logits (fp64 sums) round a value to
the other side of a bf16 midpoint and that flips a near-tie at the k-th
logit, the GPU's routing may differ from the oracle's own: every such token
must have logits that differ between the two sides, and every expert chosen
by one side only must sit within a few bf16 steps of the k-th largest logit.
Routing outputs given identical logits match bit for bit; router weights
within 1e-6.
"""
import math

import numpy as np
import pytest
import torch

import mixture_experts_layer_renorm_gb300 as moe
import oracle
import synth
from _util import (W_ABS, Y_MAX_REL, Y_MEAN_REL, assert_close_bf16, bits, f64_of_bits, fp32_dot_error_bound,
                   tensor_of_bits)

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


def tie_heavy_logits(M, E, seed):
    g = torch.Generator().manual_seed(seed)
    levels = torch.tensor([-1.0, -0.0, 0.0, 0.25, 0.5, 0.5078125, 1.0])
    return levels[torch.randint(0, len(levels), (M, E), generator=g)].to(torch.bfloat16)


@pytest.fixture(params=["tc", "gemv"])
def gemm_path(request, monkeypatch):
    """Runs a test once per implementation: the tensor-core kernels, and the
    CUDA-core ones (MOE_FORCE_PATH=gemv) that serve shapes the former do not tile."""
    monkeypatch.setenv("MOE_FORCE_PATH", request.param)
    return request.param


# ----------------------------------------------------------------------------- S0 router

def check_logits(got_bits, x, wr, bias):
    """Every GPU logit must be the bf16 rounding of some value within the fp32
    summation error bound of the exact dot product (rounding is monotone, so
    it lies between the roundings of exact - bound and exact + bound).
    Returns how many logits differ from the oracle's."""
    xb, wb = bits(x), bits(wr)
    want = oracle.router_logits(xb, wb, None if bias is None else bias.cpu().numpy())
    diff = got_bits != want
    if not diff.any():
        return 0
    xf, wf = f64_of_bits(xb), f64_of_bits(wb)
    exact = xf @ wf.T
    bound = fp32_dot_error_bound(xf, wf)
    if bias is not None:
        b = bias.cpu().numpy().astype(np.float64)
        exact = exact + b
        bound = bound + 2.0 ** -23 * (np.abs(exact) + np.abs(b))
    lo = f64_of_bits(oracle.bf16_round(exact - bound))
    hi = f64_of_bits(oracle.bf16_round(exact + bound))
    g = f64_of_bits(got_bits)
    assert ((g >= lo) & (g <= hi))[diff].all(), "a logit lies outside the fp32 error bound"
    return int(diff.sum())


@pytest.mark.parametrize("M,E,H,with_bias", [(3, 4, 128, False), (64, 128, 2048, False),
                                             (37, 256, 2048, False), (200, 33, 160, True),
                                             (1, 128, 2048, True), (515, 128, 2048, True),
                                             (4096, 256, 2048, False), (300, 60, 2048, True),
                                             (1000, 1024, 128, True)])
def test_router_logits(M, E, H, with_bias, gemm_path):
    x = rand_bf16((M, H), 1.0, 11 + M)
    wr = rand_bf16((E, H), 0.02, 12 + E)
    bias = synth.zipf_router_bias(E, 1.1).to(DEV) if with_bias else None
    lg = torch.empty((M, E), dtype=torch.bfloat16, device=DEV)
    moe.moe_router_logits(x, wr, lg, router_bias=bias)
    torch.cuda.synchronize()
    n = check_logits(bits(lg), x, wr, bias)
    assert n <= max(2, 0.01 * M * E)


# ----------------------------------------------------------------------------- S1 top-k

@pytest.mark.parametrize("M,E,k", [(3, 4, 2), (64, 128, 8), (1000, 60, 4), (129, 256, 8),
                                   (50, 1024, 32), (77, 32, 32), (40, 7, 1), (300, 128, 1)])
@pytest.mark.parametrize("kind", ["normal", "ties"])
@pytest.mark.parametrize("renorm", [True, False])
def test_topk_softmax(M, E, k, kind, renorm):
    lg = (rand_bf16((M, E), 1.0, 1000 + M + E, "cpu") if kind == "normal"
          else tie_heavy_logits(M, E, 2000 + M + E))
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    w = torch.empty((M, k), dtype=torch.float32, device=DEV)
    moe.moe_topk_softmax(lg.to(DEV), k, ids, w, renormalize=renorm)
    torch.cuda.synchronize()
    rid, rw = oracle.topk_softmax(bits(lg), k, renormalize=renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.abs(w.cpu().numpy().astype(np.float64) - rw).max() <= W_ABS


# ----------------------------------------------------------------------------- S2 align

def skewed_ids(M, E, k, seed, s=1.1):
    """topk_ids with Zipf-skewed expert loads (some experts empty, some heavy)."""
    g = torch.Generator().manual_seed(seed)
    bias = synth.zipf_router_bias(E, s, seed=seed)
    lg = (torch.randn((M, E), generator=g) + bias).to(torch.bfloat16)
    return oracle.topk_softmax(bits(lg), k)[0]


def run_align(ids_np, E, B):
    M, k = ids_np.shape
    cap = moe.moe_align_capacity(M, k, E, B)
    sorted_ids = torch.full((cap,), -7, dtype=torch.int32, device=DEV)
    eids = torch.full((cap // B,), -7, dtype=torch.int32, device=DEV)
    offs = torch.empty((E + 1,), dtype=torch.int32, device=DEV)
    npost = torch.empty((1,), dtype=torch.int32, device=DEV)
    ws = moe.Workspace(M, E, k, 16, 16, B)
    moe.moe_align_block_size(torch.from_numpy(ids_np).to(DEV), E, B, sorted_ids, eids, offs, npost, ws)
    torch.cuda.synchronize()
    return sorted_ids.cpu().numpy(), eids.cpu().numpy(), offs.cpu().numpy(), int(npost.item()), ws


def assert_align_equal(ids_np, E, B):
    s, e, o, n, ws = run_align(ids_np, E, B)
    rs, re_, ro, rn = oracle.align_block_size(ids_np, E, B)
    assert n == rn
    assert np.array_equal(s[:n], rs[:n])
    assert np.array_equal(e[: n // B], re_[: n // B])
    assert np.array_equal(o, ro)
    assert moe.moe_get_device_status(ws) == 0
    return s, e, o, n


@pytest.mark.parametrize("M,E,k,B", [(3, 4, 2, 4), (3, 4, 2, 16), (1, 128, 8, 16), (64, 128, 8, 16),
                                     (128, 256, 8, 16), (64, 60, 4, 16), (512, 128, 8, 32),
                                     (2047, 128, 8, 64), (4096, 128, 8, 128), (16384, 128, 8, 128),
                                     (8192, 60, 4, 128), (100, 1024, 32, 256), (5000, 7, 3, 1),
                                     (3000, 128, 8, 256), (2049, 1, 1, 64)])
def test_align_block_size(M, E, k, B):
    assert_align_equal(skewed_ids(M, E, k, seed=M * 31 + E), E, B)


def test_align_pages_worked_example():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "toy_align.json")))
    ids = np.array(g["our_choice"]["topk_ids"], np.int32)
    s, e, o, n = assert_align_equal(ids, 4, 4)
    assert list(s[:4]) == g["printed_on_page"]["block0_sorted_token_ids"]
    assert e[0] == g["printed_on_page"]["block0_expert"]


def test_align_is_deterministic_and_all_on_one_expert():
    ids = skewed_ids(16384, 128, 8, seed=5)
    first = run_align(ids, 128, 128)[:4]
    for _ in range(3):
        again = run_align(ids, 128, 128)[:4]
        assert all(np.array_equal(a, b) for a, b in zip(first[:3], again[:3])) and first[3] == again[3]
    same = np.zeros((40000, 1), np.int32) + 3
    assert_align_equal(same, 8, 64)


def test_align_reports_a_bad_expert_id():
    ids = skewed_ids(64, 16, 2, seed=9)
    ids[5, 1] = 16
    ids[7, 0] = -2
    s, e, o, n, ws = run_align(ids, 16, 16)
    assert moe.moe_get_device_status(ws) == 5       # MOE_ERR_DEVICE_BAD_EXPERT_ID
    assert moe.moe_get_device_status(ws) == 0       # read clears it
    body = s[:n]
    real = body[body < ids.size]
    assert sorted(real) == sorted(set(range(ids.size)) - {5 * 2 + 1, 7 * 2 + 0})


# ----------------------------------------------------------------------------- S3 / S4

def layer_case(M, E, k, H, I, seed, dev=DEV):
    x = rand_bf16((M, H), 1.0, seed, dev)
    w13 = rand_bf16((E, 2 * I, H), 0.02, seed + 1, dev)
    w2 = rand_bf16((E, H, I), 0.02, seed + 2, dev)
    lg = rand_bf16((M, E), 1.0, seed + 3, "cpu")
    return x, w13, w2, lg


def align_on_device(ids_np, E, B):
    """The oracle's align lists as device tensors (oracle -> CUDA inputs only)."""
    rs, re_, _, rn = oracle.align_block_size(ids_np, E, B)
    return (torch.from_numpy(rs).to(DEV), torch.from_numpy(re_).to(DEV),
            torch.tensor([rn], dtype=torch.int32, device=DEV))


GEMM_SHAPES = [(3, 4, 2, 128, 64, 16), (64, 128, 8, 2048, 768, 16), (64, 60, 4, 2048, 1408, 16),
               (33, 16, 3, 256, 160, 4), (200, 32, 4, 512, 96, 32), (128, 256, 8, 2048, 512, 16),
               (512, 128, 8, 2048, 768, 32), (1, 128, 8, 2048, 768, 16), (300, 8, 2, 192, 48, 64),
               (1000, 16, 4, 320, 208, 128), (700, 4, 2, 256, 128, 256), (40, 3, 3, 80, 16, 16),
               # 256-token tiles: ragged K stage (H = 208), ragged 64-channel and
               # 128-row weight tiles (I = 80, H = 208), mostly-padding blocks, real sizes
               (1000, 16, 4, 208, 80, 256), (300, 60, 4, 512, 192, 256), (2000, 8, 2, 2048, 768, 256)]


@pytest.mark.parametrize("M,E,k,H,I,B", GEMM_SHAPES)
def test_grouped_gemm_w13_act(M, E, k, H, I, B, gemm_path):
    x, w13, w2, lg = layer_case(M, E, k, H, I, seed=M + E + H)
    ids, _ = oracle.topk_softmax(bits(lg), k)
    s, e, n = align_on_device(ids, E, B)
    a = torch.full((M * k, I), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_grouped_gemm_w13_act(x, w13, s, e, n, k, B, a)
    torch.cuda.synchronize()
    ref = oracle.expert_act(bits(x), bits(w13), ids)
    assert_close_bf16(bits(a), ref, "a")


@pytest.mark.parametrize("M,E,k,H,I,B", GEMM_SHAPES)
@pytest.mark.parametrize("with_residual", [False, True])
def test_grouped_gemm_w2_combine(M, E, k, H, I, B, with_residual, gemm_path):
    x, w13, w2, lg = layer_case(M, E, k, H, I, seed=2 * M + E + I)
    ids, w = oracle.topk_softmax(bits(lg), k)
    a_bits = oracle.expert_act(bits(x), bits(w13), ids)     # oracle activation as the input
    res = rand_bf16((M, H), 1.0, 77) if with_residual else None
    s, e, n = align_on_device(ids, E, B)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    ws = moe.Workspace(M, E, k, H, I, B)
    moe.moe_grouped_gemm_w2_combine(tensor_of_bits(a_bits, DEV), w2, s, e, n,
                                    torch.from_numpy(w).to(DEV), k, B, y, ws, residual=res)
    torch.cuda.synchronize()
    ref = oracle.expert_down_combine(a_bits, bits(w2), ids, w, None if res is None else bits(res))
    assert_close_bf16(bits(y), ref, "y")


# ----------------------------------------------------------------------------- the layer

def run_forward(x, w13, w2, k, *, lg=None, wr=None, bias=None, res=None, B=0, renorm=True,
                want_logits=False):
    M, H = x.shape
    E, twoI, _ = w13.shape
    y = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((M, k), dtype=torch.float32, device=DEV)
    lgo = torch.empty((M, E), dtype=torch.bfloat16, device=DEV) if wr is not None else None
    ws = moe.Workspace(M, E, k, H, twoI // 2, B)
    moe.moe_forward(x, w13, w2, k, y, ws, w_router=wr, router_logits=lg, router_bias=bias,
                    residual=res, renormalize=renorm, block_size_m=B, topk_ids_out=ids,
                    topk_weights_out=wts, router_logits_out=lgo)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    out = (bits(y), ids.cpu().numpy(), wts.cpu().numpy())
    if want_logits:
        out = out + (None if lgo is None else bits(lgo),)
    return out


@pytest.mark.parametrize("M,E,k,H,I,B", [(3, 4, 2, 128, 64, 16), (1, 60, 4, 2048, 1408, 0),
                                         (64, 60, 4, 2048, 1408, 0), (21, 9, 9, 64, 48, 0),
                                         (50, 24, 5, 96, 32, 8), (300, 64, 6, 256, 128, 0),
                                         # both GEMMs split K = 4 stages three ways
                                         (6, 128, 8, 208, 208, 0)])
@pytest.mark.parametrize("renorm", [True, False])
def test_forward_given_logits(M, E, k, H, I, B, renorm):
    x, w13, w2, lg = layer_case(M, E, k, H, I, seed=3 * M + E)
    yb, ids, wts = run_forward(x, w13, w2, k, lg=lg.to(DEV), B=B, renorm=renorm)
    ref = oracle.moe_forward(bits(x), bits(w13), bits(w2), k, router_logits=bits(lg), renormalize=renorm)
    assert np.array_equal(ids, ref["topk_ids"])
    assert np.abs(wts.astype(np.float64) - ref["topk_weights"]).max() <= W_ABS
    assert_close_bf16(yb, ref["y"], "y")


def ordered_bf16(bits_):
    """bf16 bit patterns -> integers in the order of the values (+0 and -0 equal)."""
    b = np.asarray(bits_, dtype=np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def assert_routing_explained(g_lg, g_ids, o_lg, o_ids, k, what="routing", max_steps=8):
    """g_ids must be the oracle's top-k of the GPU logits g_lg (bit for bit); a
    token routed differently by the oracle from its own logits o_lg must have
    logits that differ, and every expert chosen by one side only must lie
    within max_steps bf16 steps of the oracle's k-th largest logit (a near-tie
    that the two roundings decide differently).  Returns the number of such
    tokens."""
    want_ids, _ = oracle.topk_softmax(g_lg, k)
    assert np.array_equal(g_ids, want_ids), f"{what}: GPU ids are not the top-k of its own logits"
    differ = ~(g_ids == o_ids).all(axis=1)
    for t in np.nonzero(differ)[0]:
        assert (g_lg[t] != o_lg[t]).any(), f"{what}: token {t} routed differently on equal logits"
        kth = ordered_bf16(o_lg[t][o_ids[t][-1]])
        odd = np.setxor1d(o_ids[t], g_ids[t])
        assert (np.abs(ordered_bf16(o_lg[t][odd]) - kth) <= max_steps).all(), \
            f"{what}: token {t} routed differently away from a near-tie"
    return int(differ.sum())


def compare_routed_layer(yb, ids, g_lg, x, wr, bias, w13, w2, k, res=None, renorm=True):
    """A layer routed by router weights: the GPU logits within the fp32 bound,
    the GPU's routing the top-k of its logits, any difference from the
    oracle's own routing a near-tie, and y equal to the oracle's layer on the
    GPU logits for every token."""
    check_logits(g_lg, x, wr, bias)
    xb = bits(x)
    o_lg = oracle.router_logits(xb, bits(wr), None if bias is None else bias.cpu().numpy())
    o_ids, _ = oracle.topk_softmax(o_lg, k, renormalize=renorm)
    n = assert_routing_explained(g_lg, ids, o_lg, o_ids, k)
    assert n <= max(1, 0.02 * len(ids)), f"{n} of {len(ids)} tokens routed differently"
    ref = oracle.moe_forward(xb, bits(w13), bits(w2), k, router_logits=g_lg,
                             residual=None if res is None else bits(res), renormalize=renorm)
    assert np.array_equal(ids, ref["topk_ids"])
    assert_close_bf16(yb, ref["y"], "y")


@pytest.mark.parametrize("cfg,M", [(1, 3), (2, 1), (2, 8), (2, 32), (2, 64), (4, 16), (4, 128)])
def test_forward_with_router_on_workloads(cfg, M):
    w = synth.WORKLOADS[cfg]
    wt = synth.layer_weights(w, device=DEV)
    inp = synth.layer_input(w, M, device=DEV)
    x = inp["x"]
    res = x if w.residual else None
    yb, ids, _, g_lg = run_forward(x, wt["w13"], wt["w2"], w.top_k, wr=wt["w_router"], res=res,
                                   B=w.block_size_m, want_logits=True)
    compare_routed_layer(yb, ids, g_lg, x, wt["w_router"], None, wt["w13"], wt["w2"], w.top_k, res)


@pytest.mark.parametrize("cfg,M", [(3, 512), (3, 4096), (3, 16384), (5, 8192), (5, 1)])
def test_forward_full_size_sampled(cfg, M):
    """The full workload on the GPU; the oracle recomputes a sample of tokens."""
    w = synth.WORKLOADS[cfg]
    wt = synth.layer_weights(w, device=DEV)
    inp = synth.layer_input(w, M, device=DEV)
    x = inp["x"]
    lg = inp["router_logits"]
    yb, ids, _, g_lg = run_forward(x, wt["w13"], wt["w2"], w.top_k, wr=wt["w_router"], lg=lg,
                                   bias=wt["router_bias"], want_logits=True)
    g = torch.Generator().manual_seed(M)
    sample = torch.randperm(M, generator=g)[: min(M, 48)].sort().values.numpy()
    if wt["w_router"] is None:
        ref = oracle.moe_forward(bits(x)[sample], bits(wt["w13"]), bits(wt["w2"]), w.top_k,
                                 router_logits=bits(lg)[sample])
        assert np.array_equal(ids[sample], ref["topk_ids"])
        assert_close_bf16(yb[sample], ref["y"], "y")
    else:
        compare_routed_layer(yb[sample], ids[sample], g_lg[sample],
                             x[torch.from_numpy(sample).to(DEV)], wt["w_router"], wt["router_bias"],
                             wt["w13"], wt["w2"], w.top_k)
    # routing is complete: every token has top_k distinct experts
    assert (np.sort(ids, axis=1)[:, 1:] != np.sort(ids, axis=1)[:, :-1]).all()


# ----------------------------------------------------------------------------- the 64-layer stack

def test_stack_chain_against_the_oracle_on_sampled_tokens():
    """The 256-expert, 64-layer decode stack: layer l+1 reads y_l computed with
    residual x_l.  The GPU runs all M=16 tokens through every layer.  Two
    checks per layer on 5 sampled tokens:

    same input (the parity check): the oracle gets the very x_l the GPU layer
    received and the router logits the GPU decided on.  At every depth the
    GPU logits must lie within the fp32 bound, the GPU routing must be the
    top-k of them, any difference from the oracle's own routing of x_l must
    be a near-tie, and y_l must match at the unscaled output tolerance.

    chained drift (an extra): the oracle also chains the sampled tokens
    through the layers on its own.  Each layer's y is rounded to bf16 on both
    sides from differently ordered sums and the residual carries the
    difference forward, so the chains drift apart like a random walk; they
    are compared while their routing agrees, with a tolerance growing as
    sqrt(1 + l/4), and the first routing difference must be a near-tie."""
    w = synth.WORKLOADS[4]
    M, sample = 16, [0, 3, 7, 10, 13]
    x0 = synth.layer_input(w, M, device=DEV)["x"]
    ws = moe.Workspace(M, w.E, w.top_k, w.H, w.I, 0)
    cur = x0.clone()
    ox = bits(x0)[sample]
    live = np.ones(len(sample), bool)
    compared = 0
    first_diff = [w.layers] * len(sample)
    for l in range(w.layers):
        wt = synth.layer_weights(w, layer=l, device=DEV)
        y = torch.empty_like(cur)
        ids = torch.empty((M, w.top_k), dtype=torch.int32, device=DEV)
        lg = torch.empty((M, w.E), dtype=torch.bfloat16, device=DEV)
        moe.moe_forward(cur, wt["w13"], wt["w2"], w.top_k, y, ws, w_router=wt["w_router"],
                        residual=cur, topk_ids_out=ids, router_logits_out=lg)
        torch.cuda.synchronize()
        gx = bits(cur)[sample]
        g_y, g_ids, g_lg = bits(y)[sample], ids.cpu().numpy()[sample], bits(lg)[sample]
        wr_b = bits(wt["w_router"])
        # the oracle's own chain for the sampled tokens
        o_lg = oracle.router_logits(ox, wr_b)
        o_ids, o_w = oracle.topk_softmax(o_lg, w.top_k)
        # copy only the experts either check routes to
        used = np.unique(np.concatenate([o_ids.ravel(), g_ids.ravel()]))
        idx = torch.from_numpy(used.astype(np.int64)).to(DEV)
        w13 = np.zeros((w.E, 2 * w.I, w.H), np.uint16)
        w2 = np.zeros((w.E, w.H, w.I), np.uint16)
        w13[used] = bits(wt["w13"].index_select(0, idx))
        w2[used] = bits(wt["w2"].index_select(0, idx))

        # same input: x_l as the GPU layer received it, the GPU's logits
        sub = torch.from_numpy(np.array(sample)).to(DEV)
        check_logits(g_lg, cur.index_select(0, sub), wt["w_router"], None)
        s_lg = oracle.router_logits(gx, wr_b)
        s_ids, _ = oracle.topk_softmax(s_lg, w.top_k)
        assert_routing_explained(g_lg, g_ids, s_lg, s_ids, w.top_k, f"layer {l}")
        ref = oracle.moe_forward(gx, w13, w2, w.top_k, router_logits=g_lg, residual=gx)
        assert np.array_equal(g_ids, ref["topk_ids"])
        assert_close_bf16(g_y, ref["y"], f"y layer {l} (same input)")

        # chained drift
        a = oracle.expert_act(ox, w13, o_ids)
        oy = oracle.expert_down_combine(a, w2, o_ids, o_w, residual=ox)
        for s_i in range(len(sample)):
            if not live[s_i]:
                continue
            if not np.array_equal(o_ids[s_i], g_ids[s_i]):
                # a near-tie: every expert chosen by one side only sits within a few
                # bf16 steps of the oracle's k-th largest logit
                assert (o_lg[s_i] != g_lg[s_i]).any(), f"layer {l}: routing differs, logits equal"
                kth = ordered_bf16(o_lg[s_i][o_ids[s_i][-1]])
                odd = np.setxor1d(o_ids[s_i], g_ids[s_i])
                assert (np.abs(ordered_bf16(o_lg[s_i][odd]) - kth) <= 8).all(), \
                    f"layer {l} token {sample[s_i]}: routing differs away from a near-tie"
                live[s_i] = False
                first_diff[s_i] = l
                continue
            grow = math.sqrt(1.0 + l / 4.0)
            assert_close_bf16(g_y[s_i:s_i + 1], oy[s_i:s_i + 1], f"y layer {l} token {sample[s_i]}",
                              max_rel=Y_MAX_REL * grow, mean_rel=Y_MEAN_REL * grow)
            compared += 1
        ox, cur = oy, y
        del wt
    assert moe.moe_get_device_status(ws) == 0
    assert min(first_diff) >= 2, f"routing differs too early: first differing layers {first_diff}"
    assert compared >= 0.1 * w.layers * len(sample), f"only {compared} pairs compared ({first_diff})"


# ----------------------------------------------------------------------------- S0 + S1 + S2 together

def run_route(M, E, k, B, *, lg=None, x=None, wr=None, bias=None, ws=None, renorm=True, lg_out=None):
    cap = moe.moe_align_capacity(M, k, E, B)
    out = dict(ids=torch.empty((M, k), dtype=torch.int32, device=DEV),
               w=torch.empty((M, k), dtype=torch.float32, device=DEV),
               s=torch.full((cap,), -7, dtype=torch.int32, device=DEV),
               e=torch.full((cap // B,), -7, dtype=torch.int32, device=DEV),
               o=torch.empty((E + 1,), dtype=torch.int32, device=DEV),
               n=torch.empty((1,), dtype=torch.int32, device=DEV))
    ws = ws or moe.Workspace(M, E, k, 16, 16, B)
    moe.moe_route(k, B, out["ids"], out["w"], out["s"], out["e"], out["o"], out["n"], ws, x=x,
                  w_router=wr, router_logits=lg, router_bias=bias, renormalize=renorm,
                  router_logits_out=lg_out)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    return {kk: v.cpu().numpy() for kk, v in out.items()}, ws


@pytest.mark.parametrize("M,E,k,B", [(1, 128, 8, 16), (64, 128, 8, 16), (64, 60, 4, 16), (3, 4, 2, 4),
                                     (256, 256, 8, 16), (200, 1024, 32, 32), (37, 33, 3, 64),
                                     (300, 128, 8, 16)])
def test_route_given_logits_matches_the_steps(M, E, k, B):
    """One launch (M <= 256) or three kernels (M = 300): the same ids, weights and
    lists as the oracle's top-k and align; a second call on the same workspace
    (its counters reset by the first) gives the same result."""
    lg = rand_bf16((M, E), 1.0, 4000 + M + E, "cpu")
    rid, rw = oracle.topk_softmax(bits(lg), k)
    rs, re_, ro, rn = oracle.align_block_size(rid, E, B)
    ws = None
    for _ in range(2):
        out, ws = run_route(M, E, k, B, lg=lg.to(DEV), ws=ws)
        assert np.array_equal(out["ids"], rid)
        assert np.abs(out["w"].astype(np.float64) - rw).max() <= W_ABS
        n = int(out["n"][0])
        assert n == rn
        assert np.array_equal(out["s"][:n], rs[:n])
        assert np.array_equal(out["e"][: n // B], re_[: n // B])
        assert np.array_equal(out["o"], ro)


@pytest.mark.parametrize("cfg,M", [(2, 1), (2, 64), (4, 128), (3, 512)])
def test_route_with_router_weights(cfg, M):
    """Routing from router weights: the logits the routing used (router_logits_out)
    lie within the fp32 bound of the exact products, the ids and weights are
    the oracle's top-k of those logits, the lists are the oracle's align of
    those ids (all bit for bit), and every token the oracle routes differently
    from its own logits is a near-tie."""
    w = synth.WORKLOADS[cfg]
    wt = synth.layer_weights(w, device=DEV)
    x = synth.layer_input(w, M, device=DEV)["x"]
    B = 16
    g_lg = torch.empty((M, w.E), dtype=torch.bfloat16, device=DEV)
    out, _ = run_route(M, w.E, w.top_k, B, x=x, wr=wt["w_router"], bias=wt["router_bias"],
                       lg_out=g_lg)
    g_lg = bits(g_lg)
    check_logits(g_lg, x, wt["w_router"], wt["router_bias"])
    bias_np = None if wt["router_bias"] is None else wt["router_bias"].cpu().numpy()
    o_lg = oracle.router_logits(bits(x), bits(wt["w_router"]), bias_np)
    o_ids, _ = oracle.topk_softmax(o_lg, w.top_k)
    n = assert_routing_explained(g_lg, out["ids"], o_lg, o_ids, w.top_k)
    assert n <= max(1, 0.02 * M), f"{n} of {M} tokens routed differently"
    rid, rw = oracle.topk_softmax(g_lg, w.top_k)
    assert np.array_equal(out["ids"], rid)
    assert np.abs(out["w"].astype(np.float64) - rw).max() <= W_ABS
    rs, re_, ro, rn = oracle.align_block_size(rid, w.E, B)
    nn = int(out["n"][0])
    assert nn == rn
    assert np.array_equal(out["s"][:nn], rs[:nn])
    assert np.array_equal(out["e"][: nn // B], re_[: nn // B])
    assert np.array_equal(out["o"], ro)


@pytest.mark.parametrize("M,E,k,H", [(300, 128, 8, 2048), (512, 128, 8, 2048), (1000, 60, 4, 2048),
                                     (4096, 128, 8, 2048), (7680, 128, 8, 2048),
                                     (2000, 300, 8, 1024), (513, 256, 8, 192)])
def test_route_splits_the_router_k_range(M, E, k, H):
    """Above 256 tokens with a workspace, the tensor-core router splits each
    tile's K range over up to four CTAs when its tiles leave SMs idle (fp32
    partial sums in per-split slices, added in split order by the tile's last
    part): the logits lie within the fp32 bound of the exact products, the
    routing is the oracle's up to near-ties, ids and lists are the oracle's
    top-k and align of the logits used, and a second call on the same
    workspace (tile counters back at zero) gives the same logits bit for bit.
    Four splits of 32 stages (300 to 4096 tokens), two at the 60-tile limit
    (7680), 60 experts (rows past E), 300 experts (two weight tiles), three
    stages over three splits (H = 192) with one token in the last tile."""
    x = rand_bf16((M, H), 1.0, 8100 + M + E)
    wr = rand_bf16((E, H), 0.02, 8200 + E + H)
    bias = synth.zipf_router_bias(E, 1.1).to(DEV) if E % 2 == 0 else None
    B = 64
    ws = moe.Workspace(M, E, k, 16, 16, B)
    first = None
    for call in range(2):
        g_lg = torch.empty((M, E), dtype=torch.bfloat16, device=DEV)
        out, ws = run_route(M, E, k, B, x=x, wr=wr, bias=bias, ws=ws, lg_out=g_lg)
        g_lg = bits(g_lg)
        if first is None:
            first = g_lg
            check_logits(g_lg, x, wr, bias)
            bias_np = None if bias is None else bias.cpu().numpy()
            o_lg = oracle.router_logits(bits(x), bits(wr), bias_np)
            o_ids, _ = oracle.topk_softmax(o_lg, k)
            n = assert_routing_explained(g_lg, out["ids"], o_lg, o_ids, k)
            assert n <= max(1, 0.02 * M), f"{n} of {M} tokens routed differently"
        else:
            assert np.array_equal(g_lg, first), f"call {call}: logits differ from the first call"
        rid, rw = oracle.topk_softmax(g_lg, k)
        assert np.array_equal(out["ids"], rid)
        assert np.abs(out["w"].astype(np.float64) - rw).max() <= W_ABS
        rs, re_, ro, rn = oracle.align_block_size(rid, E, B)
        nn = int(out["n"][0])
        assert nn == rn
        assert np.array_equal(out["s"][:nn], rs[:nn])
        assert np.array_equal(out["o"], ro)


@pytest.mark.parametrize("M,E,k,H,B", [(1, 128, 8, 2048, 16), (8, 128, 8, 2048, 16),
                                       (5, 60, 4, 2048, 16), (2, 20, 3, 256, 16),
                                       (8, 256, 8, 2048, 16), (3, 200, 6, 2112, 32),
                                       (7, 16, 2, 64, 16), (4, 129, 32, 4160, 16)])
def test_route_small_batches_with_router_weights(M, E, k, H, B):
    """Decode batches (M <= 8) with router weights run one thread-block cluster
    (up to 8 CTAs, E/n experts each, logits handed over in shared memory): the
    logits within the fp32 bound, ids and weights the oracle's top-k of those
    logits and the lists the oracle's align of those ids, bit for bit; cluster
    sizes 1 to 8, two experts per warp (E > 128), K over several staged chunks
    (H > 2048) and a ragged last chunk."""
    x = rand_bf16((M, H), 1.0, 600 + M + E)
    wr = rand_bf16((E, H), 0.02, 700 + E)
    bias = synth.zipf_router_bias(E, 1.1).to(DEV) if E % 2 == 0 else None
    g_lg = torch.empty((M, E), dtype=torch.bfloat16, device=DEV)
    ws = moe.Workspace(M, E, k, H, 16, B)
    for rep in range(2):  # a second call on the same workspace
        out, _ = run_route(M, E, k, B, x=x, wr=wr, bias=bias, lg_out=g_lg, ws=ws)
        lg_b = bits(g_lg)
        check_logits(lg_b, x, wr, bias)
        rid, rw = oracle.topk_softmax(lg_b, k)
        assert np.array_equal(out["ids"], rid)
        assert np.abs(out["w"].astype(np.float64) - rw).max() <= W_ABS
        rs, re_, ro, rn = oracle.align_block_size(rid, E, B)
        nn = int(out["n"][0])
        assert nn == rn
        assert np.array_equal(out["s"][:nn], rs[:nn])
        assert np.array_equal(out["e"][: nn // B], re_[: nn // B])
        assert np.array_equal(out["o"], ro)


# ----------------------------------------------------------------------------- small-batch sort skip

@pytest.mark.parametrize("cfg,M", [(2, 1), (2, 4), (5, 1), (4, 1), (4, 8)])
def test_forward_small_batch_skips_the_sort(cfg, M):
    """M * top_k * 4 <= E: moe_forward puts each pair in its own block (vLLM blog,
    "Small batches skip the sort").  Its y must match the always-sort path
    through the step entry points, and both the oracle, on the same logits."""
    w = synth.WORKLOADS[cfg]
    assert M * w.top_k * 4 <= w.E
    wt = synth.layer_weights(w, device=DEV)
    inp = synth.layer_input(w, M, device=DEV)
    x = inp["x"]
    lg = inp["router_logits"]
    if lg is None:  # route from fixed logits so both paths see the same ids
        lg = torch.empty((M, w.E), dtype=torch.bfloat16, device=DEV)
        moe.moe_router_logits(x, wt["w_router"], lg, router_bias=wt["router_bias"])
    B = 16
    y_skip, ids_skip, _ = run_forward(x, wt["w13"], wt["w2"], w.top_k, lg=lg, B=B, renorm=w.renormalize)
    # the always-sort path
    P = M * w.top_k
    cap = moe.moe_align_capacity(M, w.top_k, w.E, B)
    ids = torch.empty((M, w.top_k), dtype=torch.int32, device=DEV)
    wts = torch.empty((M, w.top_k), dtype=torch.float32, device=DEV)
    s = torch.empty(cap, dtype=torch.int32, device=DEV)
    e = torch.empty(cap // B, dtype=torch.int32, device=DEV)
    o = torch.empty(w.E + 1, dtype=torch.int32, device=DEV)
    n = torch.empty(1, dtype=torch.int32, device=DEV)
    ws = moe.Workspace(M, w.E, w.top_k, w.H, w.I, B)
    moe.moe_topk_softmax(lg, w.top_k, ids, wts, renormalize=w.renormalize)
    moe.moe_align_block_size(ids, w.E, B, s, e, o, n, ws)
    a = torch.empty((P, w.I), dtype=torch.bfloat16, device=DEV)
    y_sort = torch.empty((M, w.H), dtype=torch.bfloat16, device=DEV)
    moe.moe_grouped_gemm_w13_act(x, wt["w13"], s, e, n, w.top_k, B, a)
    moe.moe_grouped_gemm_w2_combine(a, wt["w2"], s, e, n, wts, w.top_k, B, y_sort, ws)
    torch.cuda.synchronize()
    assert np.array_equal(ids_skip, ids.cpu().numpy())
    assert_close_bf16(y_skip, bits(y_sort), "y skip vs sort")
    ref = oracle.moe_forward(bits(x), bits(wt["w13"]), bits(wt["w2"]), w.top_k, router_logits=bits(lg),
                             renormalize=w.renormalize)
    assert np.array_equal(ids_skip, ref["topk_ids"])
    assert_close_bf16(y_skip, ref["y"], "y")


# ----------------------------------------------------------------------------- failure path

def test_device_wait_that_runs_out_reports_a_timeout_and_the_context_stays_usable():
    """A bounded device wait whose mbarrier nothing completes gives up, records
    MOE_ERR_DEVICE_TIMEOUT (6) in the workspace status word and returns; the next
    layer on the same workspace runs normally and matches the oracle."""
    w = synth.WORKLOADS[1]
    ws = moe.Workspace(w.Ms[0], w.E, w.top_k, w.H, w.I, w.block_size_m)
    moe.moe_selftest_device_timeout(ws, limit_ms=100)
    assert moe.moe_get_device_status(ws) == 6
    assert moe.moe_get_device_status(ws) == 0       # read clears it
    M = w.Ms[0]
    x, w13, w2, lg = layer_case(M, w.E, w.top_k, w.H, w.I, seed=5)
    y = torch.empty((M, w.H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((M, w.top_k), dtype=torch.int32, device=DEV)
    moe.moe_forward(x, w13, w2, w.top_k, y, ws, router_logits=lg.to(DEV), block_size_m=w.block_size_m,
                    topk_ids_out=ids)
    assert moe.moe_get_device_status(ws) == 0
    ref = oracle.moe_forward(bits(x), bits(w13), bits(w2), w.top_k, router_logits=bits(lg))
    assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
    assert_close_bf16(bits(y), ref["y"], "y")


def test_forward_back_to_back_on_one_workspace_with_changing_batches():
    """One workspace (sized for the largest batch) serves layers of different
    M in a row on one stream, switching between the fused routing launch
    (M <= 256: completion counters, split-K scratch, small-batch skip) and the
    separate routing kernels (M > 256); every layer matches the oracle."""
    w = synth.WORKLOADS[2]
    wt = synth.layer_weights(w, device=DEV)
    Ms = (64, 1, 300, 8, 257, 3, 64)
    ws = moe.Workspace(max(Ms), w.E, w.top_k, w.H, w.I, 16)
    outs = []
    for i, M in enumerate(Ms):
        x = rand_bf16((M, w.H), 1.0, 900 + i)
        lg = rand_bf16((M, w.E), 1.0, 950 + i)
        y = torch.empty((M, w.H), dtype=torch.bfloat16, device=DEV)
        ids = torch.empty((M, w.top_k), dtype=torch.int32, device=DEV)
        moe.moe_forward(x, wt["w13"], wt["w2"], w.top_k, y, ws, router_logits=lg, block_size_m=16,
                        topk_ids_out=ids)
        outs.append((x, lg, y, ids))
    assert moe.moe_get_device_status(ws) == 0
    for x, lg, y, ids in outs:
        ref = oracle.moe_forward(bits(x), bits(wt["w13"]), bits(wt["w2"]), w.top_k,
                                 router_logits=bits(lg))
        assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
        assert_close_bf16(bits(y), ref["y"], "y")


@pytest.mark.parametrize("cfg,M", [(2, 8), (2, 32), (2, 20), (5, 64), (4, 128), (2, 200)])
def test_forward_decode_batches_twice_per_workspace(cfg, M):
    """Decode batches whose GEMM tiles are split along K (the partial sums
    added up in the split-K scratch, the last part of each tile forming its
    output) match the oracle on every token (given logits, so routing is
    exact), on two calls in a row on one workspace: the tile counters must be
    back at zero after each call."""
    w = synth.WORKLOADS[cfg]
    wt = synth.layer_weights(w, device=DEV)
    x = rand_bf16((M, w.H), 1.0, 1300 + M)
    lg = rand_bf16((M, w.E), 1.0, 1400 + M, "cpu")
    res = x if w.residual else None
    ref = oracle.moe_forward(bits(x), bits(wt["w13"]), bits(wt["w2"]), w.top_k,
                             router_logits=bits(lg), residual=None if res is None else bits(res))
    ws = moe.Workspace(M, w.E, w.top_k, w.H, w.I)
    lgd = lg.to(DEV)
    for rep in range(2):  # the split tiles' counters must be back at zero
        y = torch.empty((M, w.H), dtype=torch.bfloat16, device=DEV)
        ids = torch.empty((M, w.top_k), dtype=torch.int32, device=DEV)
        moe.moe_forward(x, wt["w13"], wt["w2"], w.top_k, y, ws, router_logits=lgd, residual=res,
                        topk_ids_out=ids)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws) == 0
        assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
        assert_close_bf16(bits(y), ref["y"], f"y (call {rep})")


# ----------------------------------------------------------------------------- one-kernel decode layer

@pytest.mark.parametrize("M,E,k,H,I,mode", [
    (1, 128, 8, 2048, 768, "router"),      # decode, one token
    (8, 128, 8, 2048, 768, "router"),
    (16, 256, 8, 2048, 512, "residual"),   # a stack layer
    (1, 60, 4, 2048, 1408, "logits"),      # tail: I = 1408 spans two K slices of GEMM 2
    (3, 4, 2, 128, 64, "router"),          # toy: fewer channels than CTAs
    (2, 1024, 32, 256, 64, "bias"),        # the largest E and top_k
    (5, 33, 3, 80, 48, "residual"),        # ragged everything
    (16, 8, 8, 2304, 96, "logits"),        # every expert chosen by every token; H beyond one K slice
])
def test_decode_layer_kernel_matches_the_oracle(M, E, k, H, I, mode, monkeypatch):
    """moe_forward with the whole layer in one persistent kernel (forced on):
    routing, both GEMMs and the combine against the oracle, twice in a row on
    one workspace (its grid-barrier counters must be back at zero)."""
    monkeypatch.setenv("MOE_DECODE_LAYER", "on")
    ws = moe.Workspace(M, E, k, H, I, 0)
    for rep in range(2):
        x, w13, w2, lg = layer_case(M, E, k, H, I, seed=7 * M + E + H + 100 * rep)
        wr = rand_bf16((E, H), 0.02, 3 + E + rep) if mode != "logits" else None
        bias = synth.zipf_router_bias(E, 1.1).to(DEV) if mode == "bias" else None
        res = rand_bf16((M, H), 1.0, 9 + rep) if mode == "residual" else None
        y = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=DEV)
        ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
        wts = torch.empty((M, k), dtype=torch.float32, device=DEV)
        lgo = torch.empty((M, E), dtype=torch.bfloat16, device=DEV) if wr is not None else None
        moe.moe_forward(x, w13, w2, k, y, ws, w_router=wr,
                        router_logits=lg.to(DEV) if wr is None else None, router_bias=bias,
                        residual=res, topk_ids_out=ids, topk_weights_out=wts, router_logits_out=lgo)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws) == 0
        if wr is None:
            ref = oracle.moe_forward(bits(x), bits(w13), bits(w2), k, router_logits=bits(lg),
                                     residual=None if res is None else bits(res))
            assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"])
            assert np.abs(wts.cpu().numpy().astype(np.float64) - ref["topk_weights"]).max() <= W_ABS
            assert_close_bf16(bits(y), ref["y"], "y")
        else:
            compare_routed_layer(bits(y), ids.cpu().numpy(), bits(lgo), x, wr, bias, w13, w2, k, res)
            _, rw = oracle.topk_softmax(bits(lgo), k)
            assert np.abs(wts.cpu().numpy().astype(np.float64) - rw).max() <= W_ABS


@pytest.mark.parametrize("cfg,M", [(2, 1), (2, 8), (4, 16), (5, 1)])
def test_decode_layer_kernel_agrees_with_the_multi_kernel_layer(cfg, M, monkeypatch):
    """The same layer through the one-kernel path and through the routing +
    grouped-GEMM kernels, on the same logits: identical routing, y within the
    output tolerance of each other."""
    w = synth.WORKLOADS[cfg]
    wt = synth.layer_weights(w, device=DEV)
    inp = synth.layer_input(w, M, device=DEV)
    lg = inp["router_logits"]
    if lg is None:
        lg = torch.empty((M, w.E), dtype=torch.bfloat16, device=DEV)
        moe.moe_router_logits(inp["x"], wt["w_router"], lg, router_bias=wt["router_bias"])
    res = inp["x"] if w.residual else None
    outs = {}
    for path in ("on", "off"):
        monkeypatch.setenv("MOE_DECODE_LAYER", path)
        outs[path] = run_forward(inp["x"], wt["w13"], wt["w2"], w.top_k, lg=lg, res=res)
    assert np.array_equal(outs["on"][1], outs["off"][1])
    assert np.abs(outs["on"][2] - outs["off"][2]).max() <= W_ABS
    assert_close_bf16(outs["on"][0], outs["off"][0], "y one kernel vs several")


# ----------------------------------------------------------------------------- 2-SM tiles

def test_two_sm_gemm1_is_stable_and_equals_one_cta_tiles(monkeypatch):
    """Grouped GEMM 1 with 256-token 2-SM tiles (a pair of CTAs, one M = 256
    MMA over both CTAs' shared memory; the odd CTA hands each stage to the
    even CTA's MMA with a release arrival that the even CTA acquires): 20 runs
    at the Zipf prefill shape M = 4096 (no K split, so a is deterministic) must
    equal, bit for bit, the same GEMM with one CTA per 256-token tile, and
    match the oracle on a sample of pairs."""
    w = synth.WORKLOADS[3]
    M, B = 4096, 256
    wt = synth.layer_weights(w, device=DEV)
    x = synth.layer_input(w, M, device=DEV)["x"]
    out, _ = run_route(M, w.E, w.top_k, B, x=x, wr=wt["w_router"], bias=wt["router_bias"])
    s = torch.from_numpy(out["s"]).to(DEV)
    e = torch.from_numpy(out["e"]).to(DEV)
    n = torch.from_numpy(out["n"]).to(DEV)
    P = M * w.top_k
    monkeypatch.setenv("MOE_FORCE_PATH", "tc1")
    a_one = torch.empty((P, w.I), dtype=torch.bfloat16, device=DEV)
    moe.moe_grouped_gemm_w13_act(x, wt["w13"], s, e, n, w.top_k, B, a_one)
    torch.cuda.synchronize()
    ref_bits = bits(a_one)
    monkeypatch.setenv("MOE_FORCE_PATH", "tc")
    a_two = torch.empty_like(a_one)
    for run in range(20):
        a_two.fill_(float("nan"))
        moe.moe_grouped_gemm_w13_act(x, wt["w13"], s, e, n, w.top_k, B, a_two)
        torch.cuda.synchronize()
        assert np.array_equal(bits(a_two), ref_bits), f"run {run}: 2-SM tiles differ from one-CTA tiles"
    assert moe.moe_get_device_status(None) == 0
    g = torch.Generator().manual_seed(4096)
    tok = torch.randperm(M, generator=g)[:24].sort().values.numpy()
    ids = out["ids"][tok]
    ref = oracle.expert_act(bits(x)[tok], bits(wt["w13"]), ids)
    pairs = (tok[:, None] * w.top_k + np.arange(w.top_k)[None, :]).reshape(-1)
    assert_close_bf16(ref_bits[pairs], ref, "a (sampled pairs)")
