"""Pins for the CPU oracle, each against something other than the oracle itself.

Sources: "Mixture of Experts in vLLM - From First Principles to fused_moe"
(the vLLM page): sections "An expert is a small SwiGLU MLP", "One token uses
only 8 experts", "A batch: (token, expert) pairs", "Group by expert",
"The two index lists", "One GEMM 1 program, step by step", "Put the results
back, and combine them per token".

What pins what:
  bf16 rounding      torch fp32->bf16 casts; brute-force nearest search over all bf16 values
  router logits      numpy fp64 matmul (library) + brute-force rounding; one-hot closed form
  top-k              numpy stable lexsort on (-value, id); forced ties; +0/-0
  weights            sum to 1; k=E equals scipy softmax; k=1 gives 1; no-renorm equals softmax
  align              the page's worked example (golden file); invariants; numpy stable argsort
  expert MLP         closed form on one-hot inputs (gate/up order, SiLU); dense expansion with
                     torch fp64 matmuls and torch's silu; k=E dense softmax mixture; E=1 SwiGLU
                     FFN; linearity in W2; residual
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- helpers

def _all_finite_bf16_positive():
    bits = np.arange(0x0000, 0x7F80, dtype=np.uint32)  # +0 .. largest finite
    vals = (bits << 16).view(np.float32).astype(np.float64)
    return bits.astype(np.uint16), vals


_BF_BITS, _BF_VALS = _all_finite_bf16_positive()
_BF_MAX = _BF_VALS[-1]
_BF_HALF_ULP_TOP = 2.0 ** (127 - 8)


def nearest_bf16_bruteforce(v):
    """Nearest bf16 by searching the sorted table of every finite bf16 value.

    Ties go to the pattern whose last bit is 0 (the even significand); beyond
    the largest finite value, the midpoint to 2^128 and above round to inf."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    n = len(_BF_VALS)
    i = np.searchsorted(_BF_VALS, a, side="left")          # _BF_VALS[i-1] < a <= _BF_VALS[i]
    i_hi = np.clip(i, 0, n - 1)
    i_lo = np.clip(i - 1, 0, n - 1)
    lo, hi = _BF_VALS[i_lo], _BF_VALS[i_hi]
    dlo, dhi = a - lo, hi - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((_BF_BITS[i_hi] & 1) == 0))
    bits = np.where(pick_hi, _BF_BITS[i_hi], _BF_BITS[i_lo])
    over = np.where(a >= _BF_MAX + _BF_HALF_ULP_TOP, np.uint16(0x7F80), np.uint16(0x7F7F))
    bits = np.where(a > _BF_MAX, over, bits)
    return (bits | np.where(np.signbit(v), np.uint16(0x8000), np.uint16(0))).astype(np.uint16)


def f64(bits):
    return oracle.bf16_to_f64(bits)


def torch_bf16_bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def rand_bf16(rng, shape, std):
    return torch_bf16_bits(torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)))


def ulp_diff(a_bits, b_bits):
    """Distance in bf16 ulps between two same-sign bf16 arrays (sign-magnitude aware)."""
    def ordered(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(ordered(a_bits) - ordered(b_bits))


# ----------------------------------------------------------------------------- bf16

def test_bf16_round_matches_torch_cast_on_fp32_patterns():
    rng = np.random.default_rng(0)
    pats = rng.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    edge = []
    for e in list(range(0, 4)) + list(range(120, 136)) + list(range(250, 256)):
        for m in (0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x17FFF, 0x18000, 0x7FFFFF):
            edge.append((e << 23) | m)
    pats = np.concatenate([pats, np.array(edge, np.uint32), np.array(edge, np.uint32) | 0x80000000])
    f = pats.view(np.float32)
    f = f[~np.isnan(f)]
    want = torch_bf16_bits(torch.from_numpy(f.copy()))
    got = oracle.bf16_round(f.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_round_is_nearest_on_doubles():
    rng = np.random.default_rng(1)
    mags = np.exp2(rng.uniform(-140, 128, size=200_000))
    v = mags * rng.choice([-1.0, 1.0], size=mags.size)
    # exact midpoints between neighbours, in normal and subnormal range
    lo = _BF_VALS[1000:1200]
    mids = (lo + _BF_VALS[1001:1201]) / 2
    v = np.concatenate([v, mids, -mids, [0.0, -0.0, 3.3961e38, 3.39e38, 1e-45, 2.0**-134]])
    assert np.array_equal(oracle.bf16_round(v), nearest_bf16_bruteforce(v))


# ----------------------------------------------------------------------------- router

def test_router_logits_against_library_matmul():
    rng = np.random.default_rng(2)
    M, E, H = 9, 13, 96
    x = rand_bf16(rng, (M, H), 1.0)
    w = rand_bf16(rng, (E, H), 0.02)
    bias = rng.standard_normal(E).astype(np.float32)
    got = oracle.router_logits(x, w, bias)
    exact = f64(x) @ f64(w).T + bias.astype(np.float64)
    want = nearest_bf16_bruteforce(exact)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.router_logits(x, w), nearest_bf16_bruteforce(f64(x) @ f64(w).T))


def test_router_logits_one_hot_rows_pick_a_weight_column():
    rng = np.random.default_rng(3)
    E, H = 5, 32
    w = rand_bf16(rng, (E, H), 0.5)
    x = torch_bf16_bits(torch.eye(H, dtype=torch.float32))  # token h = unit vector e_h
    got = oracle.router_logits(x, w)
    assert np.array_equal(got, w.T)  # logits[h, e] = W_r[e, h]


# ----------------------------------------------------------------------------- top-k

def _lexsort_topk(lg_bits, k):
    vals = f64(lg_bits)
    M, E = vals.shape
    out = np.empty((M, k), np.int32)
    for t in range(M):
        order = np.lexsort((np.arange(E), -vals[t]))  # primary: value desc, then id asc
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("E,k", [(4, 2), (60, 4), (128, 8), (256, 8), (33, 33), (7, 1)])
def test_topk_matches_stable_lexsort_with_ties(E, k):
    rng = np.random.default_rng(E * 7 + k)
    M = 64
    # few distinct values -> many ties, including at the k / k+1 boundary
    levels = torch_bf16_bits(torch.tensor([-1.0, -0.0, 0.0, 0.25, 0.5, 0.5078125, 1.0]))
    lg = levels[rng.integers(0, len(levels), size=(M, E))]
    ids, _ = oracle.topk_softmax(lg, k)
    assert np.array_equal(ids, _lexsort_topk(lg, k))
    lg2 = rand_bf16(rng, (M, E), 1.0)
    ids2, _ = oracle.topk_softmax(lg2, k)
    assert np.array_equal(ids2, _lexsort_topk(lg2, k))


def test_topk_all_equal_and_signed_zero():
    lg = np.full((3, 10), 0x3F80, np.uint16)  # all 1.0
    ids, w = oracle.topk_softmax(lg, 4)
    assert (ids == np.arange(4)).all()
    np.testing.assert_allclose(w, 0.25, atol=1e-7)
    z = np.zeros((1, 6), np.uint16)
    z[0, ::2] = 0x8000  # -0 at even ids: -0 == +0, ties by id
    ids, _ = oracle.topk_softmax(z, 6)
    assert (ids[0] == np.arange(6)).all()


def test_topk_weights_renormalized_and_softmax_special_cases():
    from scipy.special import softmax
    rng = np.random.default_rng(4)
    M, E = 50, 24
    lg = rand_bf16(rng, (M, E), 2.0)
    ids, w = oracle.topk_softmax(lg, 5, renormalize=True)
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert (np.diff(f64(lg)[np.arange(M)[:, None], ids], axis=1) <= 0).all()
    p = softmax(f64(lg), axis=1)
    # k = E with renormalize: the full softmax, in id order after sorting by slot
    idsE, wE = oracle.topk_softmax(lg, E, renormalize=True)
    np.testing.assert_allclose(wE, p[np.arange(M)[:, None], idsE], rtol=1e-6, atol=1e-7)
    # no renormalize: the softmax probabilities of the kept experts
    ids0, w0 = oracle.topk_softmax(lg, 5, renormalize=False)
    np.testing.assert_allclose(w0, p[np.arange(M)[:, None], ids0], rtol=1e-6, atol=1e-8)
    # k = 1 with renormalize: weight exactly 1
    _, w1 = oracle.topk_softmax(lg, 1, renormalize=True)
    assert (w1 == 1.0).all()


# ----------------------------------------------------------------------------- align

def test_align_reproduces_the_pages_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "toy_align.json")))
    pg = g["printed_on_page"]
    ids = np.array(g["our_choice"]["topk_ids"], np.int32)
    M, k, E, B = pg["M"], pg["top_k"], pg["E"], pg["block_size_m"]
    for p, e in pg["pair_expert"].items():
        assert ids.reshape(-1)[int(p)] == e
    s, eid, off, n_post = oracle.align_block_size(ids, E, B)
    # printed on the page: block 0 = [p1, p2, pad, pad], expert e0, pad id 6
    assert list(s[:B]) == pg["block0_sorted_token_ids"]
    assert eid[0] == pg["block0_expert"]
    assert M * k == pg["pad_id"]
    real = [p for p in s[:B] if p < M * k]
    assert [p // k for p in real] == pg["block0_input_rows"]
    assert real == pg["block0_output_rows"]
    assert 0 // k == pg["pair0_input_row"]
    want = g["our_choice"]["expected_by_definition"]
    assert list(s[:n_post]) == want["sorted_token_ids"]
    assert list(eid[: n_post // B]) == want["expert_ids"]
    assert list(off) == want["expert_offsets"]
    assert n_post == want["num_tokens_post_padded"]


def _check_align_invariants(ids, E, B, s, eid, off, n_post):
    P = ids.size
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    assert counts.sum() == P                                   # sum_e n_e = M * top_k
    padded = (counts + B - 1) // B * B
    assert n_post == padded.sum() and n_post % B == 0
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(padded)]))
    body = s[:n_post]
    real = body[body < P]
    assert np.array_equal(np.sort(real), np.arange(P))        # each pair exactly once
    assert (body[body >= P] == P).all()                        # pads hold M * top_k
    blocks = eid[: n_post // B]
    assert (np.diff(blocks) >= 0).all()                        # experts ascending
    for b, e in enumerate(blocks):
        seg = body[b * B:(b + 1) * B]
        r = seg[seg < P]
        assert (flat[r] == e).all()                            # one expert per block
        assert len(r) > 0                                      # no all-pad block
    assert np.array_equal(real, np.argsort(flat, kind="stable"))  # library cross-check


@pytest.mark.parametrize("seed", range(12))
def test_align_invariants_random(seed):
    rng = np.random.default_rng(100 + seed)
    E = int(rng.integers(1, 70))
    k = int(rng.integers(1, min(E, 8) + 1))
    M = int(rng.integers(1, 300))
    B = int(rng.choice([1, 4, 16, 32, 64, 128, 256]))
    # skewed ids: some experts empty, some heavy
    pz = rng.zipf(1.5, size=E).astype(np.float64)
    pz /= pz.sum()
    ids = np.stack([rng.choice(E, size=k, replace=False, p=pz) for _ in range(M)]).astype(np.int32)
    s, eid, off, n_post = oracle.align_block_size(ids, E, B)
    assert len(s) == oracle.align_capacity(M, k, E, B) >= n_post
    _check_align_invariants(ids, E, B, s, eid, off, n_post)


def test_align_edge_cases():
    # every pair on one expert
    ids = np.zeros((40, 1), np.int32)
    s, eid, off, n = oracle.align_block_size(ids, 5, 16)
    _check_align_invariants(ids, 5, 16, s, eid, off, n)
    assert n == 48 and list(off) == [0, 48, 48, 48, 48, 48]
    # B = 1: no padding at all
    ids = np.array([[3, 1], [1, 0]], np.int32)
    s, eid, off, n = oracle.align_block_size(ids, 4, 1)
    assert n == 4 and list(s[:4]) == [3, 1, 2, 0] and list(eid[:4]) == [0, 1, 1, 3]
    with pytest.raises(ValueError):
        oracle.align_block_size(np.array([[0, 4]], np.int32), 4, 16)


# ----------------------------------------------------------------------------- expert MLP

def _dense_reference(x, w13, w2, ids, w, residual=None):
    """y by brute force: every expert evaluated on every token with torch fp64
    matmuls and torch's silu, bf16 rounding at h, a and y, then the routing mask."""
    M, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    xt = torch.from_numpy(f64(x))
    acc = torch.zeros((M, w2.shape[1]), dtype=torch.float64)
    gate = np.zeros((M, E))
    for t in range(M):
        for j in range(ids.shape[1]):
            gate[t, ids[t, j]] += float(w[t, j])
    for e in range(E):
        h = xt @ torch.from_numpy(f64(w13[e])).T                      # [M, 2I]
        h = torch.from_numpy(f64(nearest_bf16_bruteforce(h.numpy())))
        a = torch.nn.functional.silu(h[:, :I]) * h[:, I:]
        a = torch.from_numpy(f64(nearest_bf16_bruteforce(a.numpy())))
        o = a @ torch.from_numpy(f64(w2[e])).T                        # [M, H]
        acc += torch.from_numpy(gate[:, e:e + 1]) * o
    if residual is not None:
        acc += torch.from_numpy(f64(residual))
    return nearest_bf16_bruteforce(acc.numpy())


def test_expert_closed_form_gate_up_order_and_silu():
    # x = e_0 so h = W13[:, 0]; gate rows hold g, up rows hold u; a = SiLU(g) * u
    H, I = 16, 4
    g_vals = [2.0, -1.5, 0.0, 4.0]
    u_vals = [3.0, 0.5, 7.0, -0.25]
    w13 = np.zeros((1, 2 * I, H), np.float32)
    w13[0, :I, 0] = g_vals
    w13[0, I:, 0] = u_vals
    w13b = torch_bf16_bits(torch.from_numpy(w13))
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    a = oracle.expert_act(torch_bf16_bits(torch.from_numpy(x)), w13b, np.zeros((1, 1), np.int32))
    want = [g / (1.0 + math.exp(-g)) * u for g, u in zip(g_vals, u_vals)]
    assert np.array_equal(a[0], nearest_bf16_bruteforce(np.array(want)))
    swapped = [u / (1.0 + math.exp(-u)) * g for g, u in zip(g_vals, u_vals)]
    assert not np.array_equal(a[0], nearest_bf16_bruteforce(np.array(swapped)))


@pytest.mark.parametrize("M,E,k,H,I", [(3, 4, 2, 128, 64), (7, 6, 3, 48, 32), (5, 1, 1, 64, 16),
                                       (4, 5, 5, 32, 48)])
def test_layer_matches_dense_expansion(M, E, k, H, I):
    rng = np.random.default_rng(M * 1000 + E * 10 + k)
    x = rand_bf16(rng, (M, H), 1.0)
    w13 = rand_bf16(rng, (E, 2 * I, H), 0.3)
    w2 = rand_bf16(rng, (E, H, I), 0.3)
    lg = rand_bf16(rng, (M, E), 1.0)
    res = rand_bf16(rng, (M, H), 1.0)
    out = oracle.moe_forward(x, w13, w2, k, router_logits=lg, residual=res)
    ids, w = out["topk_ids"], out["topk_weights"]
    want = _dense_reference(x, w13, w2, ids, w, res)
    assert ulp_diff(out["y"], want).max() <= 1
    assert (out["y"] == want).mean() > 0.97


def test_k_equals_E_is_the_dense_softmax_mixture():
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    M, E, H, I = 6, 5, 64, 32
    x = rand_bf16(rng, (M, H), 1.0)
    w13 = rand_bf16(rng, (E, 2 * I, H), 0.3)
    w2 = rand_bf16(rng, (E, H, I), 0.3)
    lg = rand_bf16(rng, (M, E), 1.0)
    out = oracle.moe_forward(x, w13, w2, E, router_logits=lg)
    p = softmax(f64(lg), axis=1)
    dense_ids = np.tile(np.arange(E, dtype=np.int32), (M, 1))
    want = _dense_reference(x, w13, w2, dense_ids, p)
    assert ulp_diff(out["y"], want).max() <= 1


def test_single_expert_is_a_swiglu_ffn():
    rng = np.random.default_rng(6)
    M, H, I = 8, 64, 48
    x = rand_bf16(rng, (M, H), 1.0)
    w13 = rand_bf16(rng, (1, 2 * I, H), 0.2)
    w2 = rand_bf16(rng, (1, H, I), 0.2)
    y = oracle.moe_forward(x, w13, w2, 1, router_logits=np.zeros((M, 1), np.uint16))["y"]
    W1, W3, W2 = (torch.from_numpy(f64(w13[0, :I])), torch.from_numpy(f64(w13[0, I:])),
                  torch.from_numpy(f64(w2[0])))
    xt = torch.from_numpy(f64(x))
    g = torch.from_numpy(f64(nearest_bf16_bruteforce((xt @ W1.T).numpy())))
    u = torch.from_numpy(f64(nearest_bf16_bruteforce((xt @ W3.T).numpy())))
    a = torch.from_numpy(f64(nearest_bf16_bruteforce((torch.nn.functional.silu(g) * u).numpy())))
    want = nearest_bf16_bruteforce((a @ W2.T).numpy())
    assert ulp_diff(y, want).max() <= 1


def test_linearity_in_w2_and_residual():
    rng = np.random.default_rng(7)
    M, E, k, H, I = 5, 8, 2, 64, 32
    x = rand_bf16(rng, (M, H), 1.0)
    w13 = rand_bf16(rng, (E, 2 * I, H), 0.1)
    w2 = rand_bf16(rng, (E, H, I), 0.1)
    lg = rand_bf16(rng, (M, E), 1.0)
    y1 = oracle.moe_forward(x, w13, w2, k, router_logits=lg)["y"]
    w2x2 = torch_bf16_bits(torch.from_numpy(f64(w2) * 2.0))
    y2 = oracle.moe_forward(x, w13, w2x2, k, router_logits=lg)["y"]
    assert np.array_equal(f64(y2), 2.0 * f64(y1))
    zero = np.zeros((M, H), np.uint16)
    y3 = oracle.moe_forward(x, w13, w2, k, router_logits=lg, residual=zero)["y"]
    assert np.array_equal(y3, y1)


def test_forward_is_the_composition_of_the_steps():
    rng = np.random.default_rng(8)
    M, E, k, H, I = 11, 9, 3, 64, 32
    x = rand_bf16(rng, (M, H), 1.0)
    wr = rand_bf16(rng, (E, H), 0.1)
    bias = rng.standard_normal(E).astype(np.float32)
    w13 = rand_bf16(rng, (E, 2 * I, H), 0.1)
    w2 = rand_bf16(rng, (E, H, I), 0.1)
    out = oracle.moe_forward(x, w13, w2, k, w_router=wr, router_bias=bias)
    lg = oracle.router_logits(x, wr, bias)
    ids, w = oracle.topk_softmax(lg, k)
    a = oracle.expert_act(x, w13, ids)
    y = oracle.expert_down_combine(a, w2, ids, w)
    assert np.array_equal(out["logits"], lg) and np.array_equal(out["topk_ids"], ids)
    assert np.array_equal(out["y"], y)


def test_forward_rejects_bad_router_arguments():
    x = np.zeros((1, 16), np.uint16)
    w13 = np.zeros((2, 32, 16), np.uint16)
    w2 = np.zeros((2, 16, 16), np.uint16)
    with pytest.raises(ValueError):
        oracle.moe_forward(x, w13, w2, 1)  # neither router weights nor logits


# ----------------------------------------------------------------------------- FP8 (E4M3)
#
# What pins what:
#   E4M3 decode        every code against torch.float8_e4m3fn; closed forms (448, 2^-6, 2^-9)
#   E4M3 rounding      torch fp32 -> float8_e4m3fn casts on 200k values within +-448;
#                      brute-force nearest search (ties to the even code) over every code;
#                      saturation to +-448 beyond the range
#   row quantization   closed forms: the largest element maps to 448, an all-zero row to scale 1
#                      and codes 0, dequantized values within half an E4M3 step of the input
#   FP8 expert MLP     reduces to the pinned bf16 expert MLP when codes dequantize to bf16
#                      values and scales are powers of two (both exact)

def _finite_e4m3():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    keep = np.isfinite(vals)
    return codes[keep], vals[keep]


def test_e4m3_decode_matches_torch_and_closed_forms():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(mine[fin], ref[fin])
    assert mine[0x7E] == 448.0 and mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9
    assert mine[0xFE] == -448.0 and np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])


def test_e4m3_round_matches_torch_cast_on_fp32_values():
    g = np.random.default_rng(7)
    v = g.standard_normal(200000) * np.exp(g.uniform(-14, 6.5, 200000))
    v = v[np.abs(v) <= 448].astype(np.float32)
    mine = oracle.e4m3_round(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_e4m3_round_is_nearest_ties_to_even_and_saturates():
    codes, vals = _finite_e4m3()
    pos = codes < 0x80                       # the sign-clear codes: +0 .. 448, ascending
    pc, pv = codes[pos], vals[pos]
    order = np.argsort(pv, kind="stable")
    pc, pv = pc[order], pv[order]
    g = np.random.default_rng(11)
    mids = (pv[1:] + pv[:-1]) / 2            # every tie between neighbouring codes
    v = np.concatenate([g.uniform(0, 448, 50000), mids, pv])
    i = np.clip(np.searchsorted(pv, v, side="left"), 1, len(pv) - 1)
    lo, hi = pv[i - 1], pv[i]
    pick_hi = (hi - v < v - lo) | ((hi - v == v - lo) & ((pc[i] & 1) == 0))
    want = np.where(pick_hi, pc[i], pc[i - 1])
    want = np.where(v == pv[i - 1], pc[i - 1], want)
    assert np.array_equal(oracle.e4m3_round(v), want)
    assert np.array_equal(oracle.e4m3_round(-v), want | 0x80)
    assert list(oracle.e4m3_round(np.array([448.0, 460.0, 1e6, -1e30]))) == [0x7E, 0x7E, 0x7E, 0xFE]


def test_quant_rows_closed_forms_and_error_bound():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(40, 300, generator=g) * torch.logspace(-3, 3, 40)[:, None]).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    xb[5] = 0                                  # an all-zero row
    q, s = oracle.quant_rows(xb)
    xf = x.float().numpy().astype(np.float64)
    xf[5] = 0
    amax = np.abs(xf).max(axis=1)
    assert s[5] == 1.0 and (q[5] == 0).all()
    rows = amax > 0
    assert np.array_equal(s[rows], (amax[rows].astype(np.float32) / np.float32(448)))
    # the largest element of a row maps to the largest code
    arg = np.abs(xf).argmax(axis=1)
    assert ((q[np.arange(40), arg] & 0x7F)[rows] == 0x7E).all()
    # dequantized values lie within half an E4M3 step (2^-4 relative, or the
    # subnormal half step) of the inputs
    deq = oracle.e4m3_to_f64(q) * s[:, None]
    tol = np.maximum(np.abs(xf) * 2.0 ** -4, (2.0 ** -10) * s[:, None]) * (1 + 1e-6)
    assert (np.abs(deq - xf) <= tol).all()


def _random_codes(shape, seed, spread=64.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * spread).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _bf16_of(vals):
    return torch.from_numpy(np.ascontiguousarray(vals, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def test_fp8_expert_mlp_reduces_to_the_bf16_oracle():
    """E4M3 values are bf16 values, and power-of-two scales are exact: the FP8
    expert MLP on codes and scales must equal, bit for bit, the pinned bf16
    expert MLP on the dequantized tensors."""
    M, E, k, H, I = 5, 6, 3, 64, 48
    qx = _random_codes((M, H), 1, spread=8.0)
    qw13 = _random_codes((E, 2 * I, H), 2, spread=8.0)
    qw2 = _random_codes((E, H, I), 3, spread=8.0)
    g = np.random.default_rng(5)
    sx = (2.0 ** g.integers(-4, 2, M)).astype(np.float32)
    sw13 = (2.0 ** g.integers(-9, -5, (E, 2 * I))).astype(np.float32)
    sw2 = (2.0 ** g.integers(-9, -5, (E, H))).astype(np.float32)
    ids = np.stack([g.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    wts = g.uniform(0.1, 1.0, (M, k)).astype(np.float32)
    x_deq = _bf16_of(oracle.e4m3_to_f64(qx) * sx[:, None])
    w13_deq = _bf16_of(oracle.e4m3_to_f64(qw13) * sw13[:, :, None])
    w2_deq = _bf16_of(oracle.e4m3_to_f64(qw2) * sw2[:, :, None])
    a8 = oracle.expert_act_fp8(qx, sx, qw13, sw13, ids)
    a16 = oracle.expert_act(x_deq, w13_deq, ids)
    assert np.array_equal(a8, a16)
    qa = _random_codes((M * k, I), 4, spread=8.0)
    sa = (2.0 ** g.integers(-3, 3, M * k)).astype(np.float32)
    a_deq = _bf16_of(oracle.e4m3_to_f64(qa) * sa[:, None])
    y8 = oracle.expert_down_combine_fp8(qa, sa, qw2, sw2, ids, wts)
    y16 = oracle.expert_down_combine(a_deq, w2_deq, ids, wts)
    assert np.array_equal(y8, y16)


def test_fp8_forward_quantizes_x_and_a_per_row():
    """The FP8 layer with every quantization step written out by hand from the
    pinned pieces above: x's codes and scales from the row quantizer, GEMM 1,
    a's codes and scales, GEMM 2 and the combine."""
    M, E, k, H, I = 4, 8, 2, 64, 32
    g = torch.Generator().manual_seed(9)
    x = torch.randn(M, H, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    lg = torch.randn(M, E, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qw13, qw2 = _random_codes((E, 2 * I, H), 21), _random_codes((E, H, I), 22)
    sw13 = np.full((E, 2 * I), 0.02 / 64, np.float32)
    sw2 = np.full((E, H), 0.02 / 64, np.float32)
    out = oracle.moe_forward_fp8(x, qw13, sw13, qw2, sw2, k, router_logits=lg)
    ids, wts = oracle.topk_softmax(lg, k)
    qx, sx = oracle.quant_rows(x)
    a = oracle.expert_act_fp8(qx, sx, qw13, sw13, ids)
    qa, sa = oracle.quant_rows(a)
    y = oracle.expert_down_combine_fp8(qa, sa, qw2, sw2, ids, wts)
    assert np.array_equal(out["topk_ids"], ids)
    assert np.array_equal(out["y"], y)
