"""moe_forward captured once in a CUDA graph and replayed with new inputs.

The whole layer is asynchronous and allocates nothing, so a caller can
capture it (the MoE execution analysis page, "Per-decode-step kernel
launches", counts the launches a decode step pays for without that).  Replay
is where state kept on the device between calls would show: the routing
kernel's completion counters, the split-K tile counters and the accumulators
cleared inside the layer all live in the workspace and must be back at their
starting values after every layer.  Each case captures one layer, replays it
three times with a fresh x (and fresh logits) copied into the captured input
buffers, and compares every replay with the oracle (tests/test_gpu_parity.py
has the comparison rules).
"""
import numpy as np
import pytest
import torch

import mixture_experts_layer_renorm_gb300 as moe
import oracle
import synth
from _util import assert_close_bf16, bits
from test_gpu_parity import compare_routed_layer

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


# decode M = 1 (small-batch skip of the sort), 8 and 64 (grouped, split K);
# the 256-expert stack layer with its residual; the 60-expert tail from given logits
@pytest.mark.parametrize("cfg,M,one_kernel", [(2, 1, False), (2, 8, False), (2, 64, False),
                                              (4, 16, False), (5, 64, False),
                                              # the whole layer as one persistent kernel: its
                                              # grid-barrier counters must reset for each replay
                                              (2, 1, True), (2, 8, True), (4, 16, True), (5, 1, True)])
def test_forward_replayed_from_a_cuda_graph(cfg, M, one_kernel, monkeypatch):
    monkeypatch.setenv("MOE_DECODE_LAYER", "on" if one_kernel else "off")
    w = synth.WORKLOADS[cfg]
    wt = synth.layer_weights(w, device=DEV)
    x_in = torch.empty((M, w.H), dtype=torch.bfloat16, device=DEV)
    lg_in = torch.empty((M, w.E), dtype=torch.bfloat16, device=DEV) if w.logits_given else None
    y = torch.empty((M, w.H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((M, w.top_k), dtype=torch.int32, device=DEV)
    lg_out = None if w.logits_given else torch.empty((M, w.E), dtype=torch.bfloat16, device=DEV)
    ws = moe.Workspace(M, w.E, w.top_k, w.H, w.I, 0)

    def load(rep):
        inp = synth.layer_input(w, M, rep=rep, device=DEV)
        x_in.copy_(inp["x"])
        if lg_in is not None:
            lg_in.copy_(inp["router_logits"])

    def layer():
        moe.moe_forward(x_in, wt["w13"], wt["w2"], w.top_k, y, ws,
                        w_router=None if w.logits_given else wt["w_router"], router_logits=lg_in,
                        router_bias=wt["router_bias"], residual=x_in if w.residual else None,
                        renormalize=w.renormalize, topk_ids_out=ids, router_logits_out=lg_out)

    load(0)
    layer()  # per-device set-up (tensor maps, shared-memory limits) outside the capture
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer()
    for rep in (1, 2, 3):
        load(rep)
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws) == 0
        g_ids = ids.cpu().numpy()
        if w.logits_given:
            ref = oracle.moe_forward(bits(x_in), bits(wt["w13"]), bits(wt["w2"]), w.top_k,
                                     router_logits=bits(lg_in), renormalize=w.renormalize)
            assert np.array_equal(g_ids, ref["topk_ids"]), f"replay {rep}: routing"
            assert_close_bf16(bits(y), ref["y"], f"y (replay {rep})")
        else:
            compare_routed_layer(bits(y), g_ids, bits(lg_out), x_in, wt["w_router"],
                                 wt["router_bias"], wt["w13"], wt["w2"], w.top_k,
                                 x_in if w.residual else None, w.renormalize)


# E4M3 expert weights: the two row quantizations join the captured chain and
# the GEMMs' K splits run on 128-element stages.  Given logits keep routing
# exact, so every replay is compared with the oracle's E4M3 layer directly;
# with router weights (last case) the replay's logits are checked against
# their fp32 bound and the oracle's layer is run on them.
@pytest.mark.parametrize("cfg,M,given", [(2, 1, True), (2, 8, True), (2, 64, True), (5, 64, True),
                                         (2, 8, False)])
def test_forward_fp8_replayed_from_a_cuda_graph(cfg, M, given):
    from test_gpu_fp8 import oracle_fp8
    from test_gpu_parity import check_logits
    w = synth.WORKLOADS[cfg]
    wt = synth.layer_weights_fp8(w, device=DEV)
    wr = None if given else wt["w_router"]
    x_in = torch.empty((M, w.H), dtype=torch.bfloat16, device=DEV)
    lg_in = torch.empty((M, w.E), dtype=torch.bfloat16, device=DEV) if given else None
    lg_out = None if given else torch.empty((M, w.E), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((M, w.H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((M, w.top_k), dtype=torch.int32, device=DEV)
    ws = moe.Workspace(M, w.E, w.top_k, w.H, w.I, 0, fp8=True)

    def load(rep):
        x_in.copy_(synth.normal_bf16((M, w.H), 1.0, 7100 + 31 * rep + M, DEV))
        if given:
            lg_in.copy_(synth.normal_bf16((M, w.E), 1.0, 7200 + 31 * rep + M, DEV))

    def layer():
        moe.moe_forward_fp8(x_in, wt["w13"], wt["w13_scale"], wt["w2"], wt["w2_scale"], w.top_k,
                            y, ws, w_router=wr, router_logits=lg_in, router_bias=wt["router_bias"],
                            renormalize=w.renormalize, topk_ids_out=ids, router_logits_out=lg_out)

    load(0)
    layer()  # per-device set-up outside the capture
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(ws) == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer()
    for rep in (1, 2, 3):
        load(rep)
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(ws) == 0
        if given:
            lg = bits(lg_in)
        else:
            lg = bits(lg_out)
            check_logits(lg, x_in, wt["w_router"], wt["router_bias"])
        ref = oracle_fp8(bits(x_in), wt, w.top_k, lg, renorm=w.renormalize)
        assert np.array_equal(ids.cpu().numpy(), ref["topk_ids"]), f"replay {rep}: routing"
        assert_close_bf16(bits(y), ref["y"], f"y (replay {rep})")
