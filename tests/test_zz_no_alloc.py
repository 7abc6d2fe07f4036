"""moe_grouped_gemm_w2_combine_noalloc: GEMM 2 + combine for callers that
cannot allocate device memory (plugin code whose host application owns all
device allocations, latency-critical code that may not call cudaMalloc).

It keeps its fp32 accumulator in an array built into the library instead of
a caller workspace.  This test calls it through the C ABI twice in a row, on
different inputs (the second call must not see the first call's sums), and
compares each result with the oracle's GEMM 2 + combine and with the
workspace entry point moe_grouped_gemm_w2_combine, within the output
tolerance.  Without a workspace a caller learns of a device-side problem
through the library-wide status word (moe_get_device_status(NULL)); it must
read MOE_OK after every call.  The file is named to be collected last.
"""
import pytest
import torch

import mixture_experts_layer_renorm_gb300 as moe
import oracle
import synth
from _util import assert_close_bf16, bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT = 1 << 21  # accumulator elements built into the library (M * H)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_layer_renorm_gb300 import _build
    _build.build()
    moe.load_library()
    oracle.build()


def _case(M, E, k, H, I, B, seed, residual):
    x = synth.normal_bf16((M, H), 1.0, seed, DEV)
    w13 = synth.normal_bf16((E, 2 * I, H), 0.02, seed + 1, DEV)
    w2 = synth.normal_bf16((E, H, I), 0.02, seed + 2, DEV)
    lg = synth.normal_bf16((M, E), 1.0, seed + 3, "cpu")
    ids, w = oracle.topk_softmax(bits(lg), k)
    a_bits = oracle.expert_act(bits(x), bits(w13), ids)
    s, e, _, n = oracle.align_block_size(ids, E, B)
    s, e = torch.from_numpy(s).to(DEV), torch.from_numpy(e).to(DEV)
    n = torch.tensor([n], dtype=torch.int32, device=DEV)
    wts = torch.from_numpy(w).to(DEV)
    a = synth.from_bits(a_bits, DEV)    # the oracle's activation as the input
    res = synth.normal_bf16((M, H), 1.0, seed + 4, DEV) if residual else None
    ref = oracle.expert_down_combine(a_bits, bits(w2), ids, w, None if res is None else bits(res))
    return a, w2, s, e, n, wts, res, ref


@pytest.mark.parametrize("shape", [(64, 128, 8, 2048, 768, 16), (3, 4, 2, 128, 64, 16)])
def test_noalloc_matches_the_oracle_and_the_workspace_entry_point_on_two_calls(shape):
    M, E, k, H, I, B = shape
    assert moe.moe_get_device_status(None) == 0
    for call, (seed, residual) in enumerate([(501, False), (907, True)]):
        a, w2, s, e, n, wts, res, ref = _case(M, E, k, H, I, B, seed + M, residual)
        y_ws = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
        ws = moe.Workspace(M, E, k, H, I, B)
        moe.moe_grouped_gemm_w2_combine(a, w2, s, e, n, wts, k, B, y_ws, ws, residual=res)
        y_na = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=DEV)
        moe.moe_grouped_gemm_w2_combine_noalloc(a, w2, s, e, n, wts, k, B, y_na, residual=res)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(None) == 0
        assert moe.moe_get_device_status(ws) == 0
        assert_close_bf16(bits(y_na), ref, f"y against the oracle (call {call + 1})")
        assert_close_bf16(bits(y_na), bits(y_ws), f"y against the workspace path (call {call + 1})")


def test_noalloc_rejects_sizes_beyond_its_accumulator():
    H = 2048
    M = LIMIT // H + 1
    lib = moe.load_library()
    # rejected on the host before anything is launched; the buffer is zeros
    # (num_tokens_post_padded = 0), so even a launch would find no work
    dummy = torch.zeros(1 << 22, dtype=torch.int32, device=DEV)
    p = dummy.data_ptr()
    rc = lib.moe_grouped_gemm_w2_combine_noalloc(p, p, p, p, p, p, None, M, 8, 128, H, 768, 16, p,
                                                 None)
    assert rc == 2  # MOE_ERR_UNSUPPORTED_SHAPE
