"""Pins of the CPU oracle against what the mathematics fixes.

Each test checks one building block (or the whole step) against a closed
form, an invariant, a special case that reduces to a library routine
(numpy / scipy / torch), or a brute-force composition of such routines on a
tiny model.  They are chosen so that a plausible slip - eps outside the
square root, NeoX pairing instead of adjacent pairs, a sign or frequency
error in RoPE, a missing 1/sqrt(hd), GQA heads grouped modulo instead of by
block, a window one position too wide or narrow, a softmax over all experts,
a tie broken upwards - fails at least one of them.
"""
import dataclasses
import math
import zlib

import numpy as np
import pytest
import scipy.special as sp
import torch

import oracle
import synth
import synth.workloads as wl
from synth import BF16, F32
from synth.workloads import Shape

RNG = np.random.default_rng(20261202)


@pytest.fixture(autouse=True)
def _rng_per_test(request):
    """Each test draws from its own generator, seeded by its name, so its inputs do
    not depend on which other tests ran before it."""
    global RNG
    RNG = np.random.default_rng(zlib.crc32(request.node.name.encode()))


def f32(a):
    return np.asarray(a, dtype=np.float32)


# --------------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("c", [0.5, -3.0, 1e-3, 7.25])
def test_rmsnorm_constant_vector_closed_form(c):
    n, eps = 64, 1e-5
    x = np.full(n, c, np.float32)
    w = f32(np.linspace(0.5, 2.0, n))
    out = oracle.rmsnorm(x, w, eps)
    expect = w.astype(np.float64) * np.float64(np.float32(c)) / math.sqrt(float(np.float32(c)) ** 2 + eps)
    assert np.allclose(out, expect, rtol=2e-7, atol=0)


def test_rmsnorm_unit_rms_and_scale_invariance():
    x = f32(RNG.standard_normal(4096) * 3)
    ones = np.ones(4096, np.float32)
    out = oracle.rmsnorm(x, ones, 0.0)
    assert abs(math.sqrt(np.mean(out.astype(np.float64) ** 2)) - 1.0) < 1e-6
    # a power-of-two scale is exact in fp32, so with eps = 0 the output is identical
    assert np.array_equal(out, oracle.rmsnorm(x * np.float32(8.0), ones, 0.0))


def test_rmsnorm_eps_inside_square_root():
    x = np.full(16, 1e-6, np.float32)
    out = oracle.rmsnorm(x, np.ones(16, np.float32), 1e-5)
    inside = 1e-6 / math.sqrt(1e-12 + 1e-5)       # eps under the root
    outside = 1e-6 / (1e-6 + 1e-5)                 # eps added to the rms
    assert np.allclose(out, inside, rtol=1e-6)
    assert not np.allclose(out, outside, rtol=1e-2)


# ------------------------------------------------------------------------ RoPE

def _complex_rotation(v, p, theta):
    """Textbook RoPE: pair (2i, 2i+1) as a complex number times exp(i p theta^(-2i/d))."""
    d = v.size
    z = v[0::2].astype(np.float64) + 1j * v[1::2].astype(np.float64)
    z = z * np.exp(1j * p * np.power(theta, -2.0 * np.arange(d // 2) / d))
    out = np.empty(d)
    out[0::2], out[1::2] = z.real, z.imag
    return out


@pytest.mark.parametrize("hd", [32, 128])
@pytest.mark.parametrize("p", [1, 7, 2049, 8191])
@pytest.mark.parametrize("theta", [1e4, 5e5, 1e6])
def test_rope_is_complex_rotation_of_adjacent_pairs(hd, p, theta):
    v = f32(RNG.standard_normal(hd))
    got = oracle.rope(v, p, theta)
    assert np.allclose(got, _complex_rotation(v, p, theta), rtol=0, atol=1e-6 * np.abs(v).max())


def test_rope_position_zero_is_identity():
    v = f32(RNG.standard_normal(128))
    assert np.array_equal(oracle.rope(v, 0, 1e4), v)


def test_rope_preserves_pair_norms():
    v = f32(RNG.standard_normal(128))
    got = oracle.rope(v, 1234, 1e4).astype(np.float64)
    n0 = v[0::2].astype(np.float64) ** 2 + v[1::2].astype(np.float64) ** 2
    n1 = got[0::2] ** 2 + got[1::2] ** 2
    assert np.allclose(n1, n0, rtol=1e-6)


@pytest.mark.parametrize("theta", [1e4, 1e6])
def test_rope_frequency_closed_forms(theta):
    hd, p = 128, 3
    for pair, angle in ((0, p * 1.0), (hd // 4, p / math.sqrt(theta))):
        v = np.zeros(hd, np.float32)
        v[2 * pair] = 1.0
        got = oracle.rope(v, p, theta).astype(np.float64)
        turned = math.atan2(got[2 * pair + 1], got[2 * pair])
        want = math.atan2(math.sin(angle), math.cos(angle))
        assert abs(turned - want) < 1e-6
        others = np.delete(got, [2 * pair, 2 * pair + 1])
        assert np.all(others == 0)


def test_rope_dot_products_depend_on_relative_position_only():
    q, k = f32(RNG.standard_normal(128)), f32(RNG.standard_normal(128))
    for (m, n) in ((5, 2), (100, 97), (4000, 3997)):
        d0 = np.dot(oracle.rope(q, m, 1e4).astype(np.float64), oracle.rope(k, n, 1e4).astype(np.float64))
        d1 = np.dot(oracle.rope(q, m + 777, 1e4).astype(np.float64),
                    oracle.rope(k, n + 777, 1e4).astype(np.float64))
        assert abs(d0 - d1) < 1e-4 * (np.linalg.norm(q) * np.linalg.norm(k))


def _complex_rotation_halves(v, p, theta):
    """Textbook NeoX RoPE: pair (i, i + d/2) as a complex number times exp(i p theta^(-2i/d))."""
    d = v.size
    z = v[: d // 2].astype(np.float64) + 1j * v[d // 2:].astype(np.float64)
    z = z * np.exp(1j * p * np.power(theta, -2.0 * np.arange(d // 2) / d))
    return np.concatenate([z.real, z.imag])


@pytest.mark.parametrize("hd", [32, 128])
@pytest.mark.parametrize("p", [1, 7, 2049])
@pytest.mark.parametrize("theta", [1e4, 1e6])
def test_rope_neox_is_complex_rotation_of_half_pairs(hd, p, theta):
    v = f32(RNG.standard_normal(hd))
    got = oracle.rope_neox(v, p, theta)
    assert np.allclose(got, _complex_rotation_halves(v, p, theta), rtol=0,
                       atol=1e-6 * np.abs(v).max())
    assert np.array_equal(oracle.rope_neox(v, 0, theta), v)


def test_rope_neox_is_adjacent_rope_on_interleaved_halves():
    # the layout the GPU library uses for NeoX models: a head's dimensions in
    # the order 0, d/2, 1, d/2 + 1, ... make the NeoX pairs adjacent, and the
    # adjacent-pair rotation of the reordered vector is the reordered NeoX
    # rotation (same angle per pair)
    hd = 64
    perm = np.empty(hd, dtype=np.int64)
    perm[0::2], perm[1::2] = np.arange(hd // 2), np.arange(hd // 2) + hd // 2
    for p in (1, 5, 300):
        v = f32(RNG.standard_normal(hd))
        assert np.allclose(oracle.rope(v[perm], p, 1e4), oracle.rope_neox(v, p, 1e4)[perm],
                           rtol=0, atol=1e-6)
    # and the two forms differ on the same vector
    v = f32(RNG.standard_normal(hd))
    assert not np.allclose(oracle.rope(v, 3, 1e4), oracle.rope_neox(v, 3, 1e4), atol=1e-3)


# ------------------------------------------------------------------- attention

def _rand_kv(npos, nkv, hd):
    return f32(RNG.standard_normal((npos, nkv, hd))), f32(RNG.standard_normal((npos, nkv, hd)))


def test_attention_first_position_returns_v0_exactly():
    H, Hkv, hd = 8, 2, 32
    K, V = _rand_kv(4, Hkv, hd)
    q = f32(RNG.standard_normal(H * hd) * 10)
    o = oracle.attention(q, K, V, H, Hkv, 0).reshape(H, hd)
    for h in range(H):
        assert np.array_equal(o[h], V[0, h // (H // Hkv)])


def test_attention_equal_keys_average_values():
    H, Hkv, hd, p = 4, 4, 16, 9
    K, V = _rand_kv(p + 1, Hkv, hd)
    K[:] = K[0]
    q = f32(RNG.standard_normal(H * hd))
    o = oracle.attention(q, K, V, H, Hkv, p).reshape(H, hd)
    assert np.allclose(o, V[: p + 1].astype(np.float64).mean(axis=0), rtol=0, atol=1e-6)


def test_attention_two_positions_logistic_weights():
    hd, a = 4, 1.7
    K = np.zeros((2, 1, hd), np.float32)
    K[0, 0, 0], K[1, 0, 0] = 1.0, -1.0
    V = f32(RNG.standard_normal((2, 1, hd)))
    q = np.zeros(hd, np.float32)
    q[0] = a
    o = oracle.attention(q, K, V, 1, 1, 1)
    # scores +-a/sqrt(hd) = +-a/2, so the first value gets weight 1/(1+e^-a)
    w0 = 1.0 / (1.0 + math.exp(-a))
    assert np.allclose(o, w0 * V[0, 0] + (1 - w0) * V[1, 0], rtol=0, atol=1e-6)


def test_attention_matches_scipy_softmax():
    H, Hkv, hd, p = 6, 3, 8, 12
    K, V = _rand_kv(p + 1, Hkv, hd)
    q = f32(RNG.standard_normal(H * hd))
    o = oracle.attention(q, K, V, H, Hkv, p).reshape(H, hd)
    for h in range(H):
        g = h // (H // Hkv)
        s = K[:, g, :].astype(np.float64) @ q[h * hd:(h + 1) * hd].astype(np.float64) / math.sqrt(hd)
        assert np.allclose(o[h], sp.softmax(s) @ V[:, g, :].astype(np.float64), rtol=0, atol=1e-6)


def test_attention_huge_score_selects_its_value():
    hd, p = 8, 5
    K = np.zeros((p + 1, 1, hd), np.float32)
    K[3, 0, 0] = 1000.0
    V = f32(RNG.standard_normal((p + 1, 1, hd)))
    q = np.zeros(hd, np.float32)
    q[0] = 1.0
    assert np.allclose(oracle.attention(q, K, V, 1, 1, p), V[3, 0], atol=1e-6)


def test_gqa_consecutive_query_heads_share_a_kv_head():
    H, Hkv, hd, p = 8, 2, 4, 3
    K, V = _rand_kv(p + 1, Hkv, hd)
    for g in range(Hkv):
        V[:, g, :] = g + 1.0
    o = oracle.attention(f32(RNG.standard_normal(H * hd)), K, V, H, Hkv, p).reshape(H, hd)
    for h in range(H):
        assert np.allclose(o[h], h // (H // Hkv) + 1.0)   # block grouping, not h % Hkv


@pytest.mark.parametrize("W", [1, 4, 7])
def test_window_masks_exactly_the_older_positions(W):
    H, Hkv, hd, p = 4, 2, 8, 10
    K, V = _rand_kv(p + 1, Hkv, hd)
    q = f32(RNG.standard_normal(H * hd))
    base = oracle.attention(q, K, V, H, Hkv, p, W)
    K2, V2 = K.copy(), V.copy()
    K2[: p - W + 1] = 1e4      # everything at j <= p - W
    V2[: p - W + 1] = -1e4
    assert np.array_equal(oracle.attention(q, K2, V2, H, Hkv, p, W), base)
    V3 = V.copy()
    V3[p - W + 1] += 1.0        # the oldest position inside the window
    assert not np.array_equal(oracle.attention(q, K, V3, H, Hkv, p, W), base)


def test_window_wider_than_context_is_no_window():
    H, Hkv, hd, p = 4, 2, 8, 10
    K, V = _rand_kv(p + 1, Hkv, hd)
    q = f32(RNG.standard_normal(H * hd))
    full = oracle.attention(q, K, V, H, Hkv, p, 0)
    assert np.array_equal(oracle.attention(q, K, V, H, Hkv, p, p + 1), full)
    assert np.array_equal(oracle.attention(q, K, V, H, Hkv, p, 1000), full)
    assert not np.array_equal(oracle.attention(q, K, V, H, Hkv, p, p), full)


# ---------------------------------------------------------------- FFN and MoE

def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    for z in np.linspace(-20, 20, 81):
        assert math.isclose(oracle.silu(z), z * sp.expit(z), rel_tol=1e-14, abs_tol=1e-300)
    assert math.isclose(oracle.silu(50.0), 50.0, rel_tol=1e-15)


def test_ffn_is_swiglu_of_library_ops():
    E, F = 24, 40
    wg, wu, wd = (f32(RNG.standard_normal(s) * 0.3) for s in ((F, E), (F, E), (E, F)))
    xn = f32(RNG.standard_normal(E))
    g = wg.astype(np.float64) @ xn.astype(np.float64)
    u = wu.astype(np.float64) @ xn.astype(np.float64)
    want = wd.astype(np.float64) @ (g * sp.expit(g) * u)
    assert np.allclose(oracle.ffn(wg, wu, wd, xn), want, rtol=1e-5, atol=1e-6)


def test_matvec_matches_numpy_fp64():
    W, x = f32(RNG.standard_normal((300, 77))), f32(RNG.standard_normal(77))
    want = (W.astype(np.float64) @ x.astype(np.float64)).astype(np.float32)
    got = oracle.matvec(W, x)
    assert np.max(np.abs(got.view(np.int32) - want.view(np.int32))) <= 1


def test_topk_picks_largest_and_breaks_ties_to_lower_index():
    assert list(oracle.topk_softmax(f32([0.5, 2.0, 2.0, -1.0]), 2)[0]) == [1, 2]
    assert list(oracle.topk_softmax(f32([0.5, 2.0, 2.0, -1.0]), 1)[0]) == [1]
    assert list(oracle.topk_softmax(f32([1.0, 1.0, 1.0]), 2)[0]) == [0, 1]
    assert list(oracle.topk_softmax(f32([-5, 3, 0, 2, 9, -1, 2, 3]), 3)[0]) == [4, 1, 7]


def test_topk_softmax_is_over_the_selected_logits_only():
    idx, g = oracle.topk_softmax(f32([3.0, 1.0, 0.0, 2.0]), 2)
    assert list(idx) == [0, 3]
    assert np.allclose(g, [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))], rtol=1e-14)
    r = f32(RNG.standard_normal(8))
    idx, g = oracle.topk_softmax(r, 8)
    full = np.zeros(8)
    full[idx] = g
    assert np.allclose(full, sp.softmax(r.astype(np.float64)), rtol=1e-13)


def test_argmax_ties_go_to_the_lowest_id():
    assert oracle.argmax(f32([1, 3, 3, 2])) == 1
    assert oracle.argmax(np.zeros(10, np.float32)) == 0
    assert oracle.argmax(f32([-1, -1, -0.5, -0.5])) == 2


def test_bf16_rounding_matches_torch():
    x = f32(RNG.standard_normal(5000))
    ours = np.array([oracle.round_bf16(float(v)) for v in x], np.float32)
    assert np.array_equal(ours, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


# ---------------------------------------------------------------- whole step

TS = Shape(n_vocab=16, n_embd=16, n_head=4, n_kv_head=2, n_layer=2, n_ff=24, n_ctx=12,
           rope_theta=100.0, rms_norm_eps=1e-5, dtype=F32)


def _bf16(a):
    return torch.from_numpy(f32(a)).to(torch.bfloat16).float().numpy()


def _rand_arrays(shape: Shape, scale=0.3):
    """Explicit random weights for every tensor of `shape` (storage values)."""
    arrays = {}
    for spec in wl.weight_specs(shape):
        k = spec.name if spec.name in ("tok_embd", "out_norm", "output") else (spec.name, spec.layer, spec.sub)
        if spec.const is not None:
            a = f32(1.0 + 0.1 * RNG.standard_normal((spec.rows, spec.cols)))
        else:
            a = f32(RNG.standard_normal((spec.rows, spec.cols)) * scale)
        arrays[k] = _bf16(a) if shape.dtype == BF16 else a
    return arrays


def _library_forward(shape: Shape, arrays, tokens, margins=None):
    """Brute force: the decode steps composed of library routines (numpy norm, complex
    exponentials, scipy softmax / expit, matmul), fp64 throughout; the cache stores
    torch-rounded bf16 values when the model is bf16."""
    E, H, Hkv, F = shape.n_embd, shape.n_head, shape.n_kv_head, shape.n_ff
    hd, eps, W = shape.head_dim, shape.rms_norm_eps, shape.sliding_window
    d = lambda a: np.asarray(a, np.float64)
    Kc = [[] for _ in range(shape.n_layer)]
    Vc = [[] for _ in range(shape.n_layer)]

    def norm(x, w):
        return d(w).ravel() * x / math.sqrt(np.linalg.norm(x) ** 2 / x.size + eps)

    def rot(v, p):
        if shape.rope_neox:
            return _complex_rotation_halves(v, p, shape.rope_theta)
        return _complex_rotation(v, p, shape.rope_theta)

    def store(v):
        return _bf16(v).astype(np.float64) if shape.dtype == BF16 else f32(v).astype(np.float64)

    def swiglu(prefix, l, e, xn):
        g = d(arrays[("wgate", l, e)]) @ xn
        u = d(arrays[("wup", l, e)]) @ xn
        return d(arrays[("wdown", l, e)]) @ (g * sp.expit(g) * u)

    out = []
    for p, tok in enumerate(tokens):
        x = d(arrays["tok_embd"])[tok].copy()
        step_margin = math.inf
        for l in range(shape.n_layer):
            xn = norm(x, arrays[("attn_norm", l, 0)])
            q = d(arrays[("wq", l, 0)]) @ xn
            k = d(arrays[("wk", l, 0)]) @ xn
            v = d(arrays[("wv", l, 0)]) @ xn
            if shape.qkv_bias:
                q = q + d(arrays[("bq", l, 0)]).ravel()
                k = k + d(arrays[("bk", l, 0)]).ravel()
                v = v + d(arrays[("bv", l, 0)]).ravel()
            q = np.concatenate([rot(q[h * hd:(h + 1) * hd], p) for h in range(H)])
            k = np.concatenate([rot(k[g * hd:(g + 1) * hd], p) for g in range(Hkv)])
            Kc[l].append(store(k))
            Vc[l].append(store(v))
            lo = max(0, p - W + 1) if W > 0 else 0
            Kl, Vl = np.array(Kc[l][lo:p + 1]), np.array(Vc[l][lo:p + 1])
            o = []
            for h in range(H):
                g = h // (H // Hkv)
                s = Kl[:, g * hd:(g + 1) * hd] @ q[h * hd:(h + 1) * hd] / math.sqrt(hd)
                o.append(sp.softmax(s) @ Vl[:, g * hd:(g + 1) * hd])
            x = x + d(arrays[("wo", l, 0)]) @ np.concatenate(o)
            xn = norm(x, arrays[("ffn_norm", l, 0)])
            if shape.expert_count > 0:
                r = d(arrays[("wrouter", l, 0)]) @ xn
                top = np.argsort(-r, kind="stable")[: shape.expert_used]
                if shape.expert_used < shape.expert_count:
                    rest = np.argsort(-r, kind="stable")[shape.expert_used]
                    step_margin = min(step_margin, (r[top[-1]] - r[rest]) / np.max(np.abs(r)))
                gate = sp.softmax(r[top])
                x = x + sum(gi * swiglu("", l, int(e), xn) for gi, e in zip(gate, top))
            else:
                x = x + swiglu("", l, 0, xn)
        out.append(d(arrays["output"]) @ norm(x, arrays["out_norm"]))
        if margins is not None:
            margins.append(step_margin)
    return out


def _oracle_run(shape, arrays, tokens):
    m = oracle.Model(shape, arrays=arrays)
    s = m.new_state()
    res = [s.forward(t) for t in tokens]
    return [r[0] for r in res], [r[1] for r in res]


@pytest.mark.parametrize("variant", ["mha_f32", "gqa_f32", "gqa_bf16", "window_bf16", "moe_f32",
                                     "moe_bf16", "qkv_bias_bf16", "neox_f32", "bias_neox_f32"])
def test_whole_step_matches_library_composition(variant):
    shape = {
        "mha_f32": dataclasses.replace(TS, n_kv_head=4),
        "gqa_f32": TS,
        "gqa_bf16": dataclasses.replace(TS, dtype=BF16),
        "window_bf16": dataclasses.replace(TS, dtype=BF16, sliding_window=3),
        "moe_f32": dataclasses.replace(TS, expert_count=4, expert_used=2),
        "moe_bf16": dataclasses.replace(TS, expert_count=3, expert_used=2, dtype=BF16),
        "qkv_bias_bf16": dataclasses.replace(TS, dtype=BF16, qkv_bias=True),
        "neox_f32": dataclasses.replace(TS, rope_neox=True),
        "bias_neox_f32": dataclasses.replace(TS, qkv_bias=True, rope_neox=True),
    }[variant]
    arrays = _rand_arrays(shape)
    tokens = [int(t) for t in RNG.integers(0, shape.n_vocab, size=shape.n_ctx)]
    want = _library_forward(shape, arrays, tokens)
    got, am = _oracle_run(shape, arrays, tokens)
    for p in range(len(tokens)):
        scale = np.abs(want[p]).max()
        assert np.allclose(got[p], want[p], rtol=0, atol=1e-5 * scale), (variant, p)
        srt = np.sort(want[p])
        if srt[-1] - srt[-2] > 1e-4 * scale:
            assert am[p] == int(np.argmax(want[p]))



def test_route_margin_is_the_top_k_gap_of_the_router_logits():
    """The oracle's routing near-tie diagnostic: after each forward, the smallest
    gap between the k-th chosen router logit and the best unchosen one, over the
    layers, relative to the layer's largest |logit|, as the brute-force
    composition's fp64 router logits give it; an exact tie gives 0 and a dense
    model infinity."""
    shape = dataclasses.replace(TS, expert_count=4, expert_used=2)
    arrays = _rand_arrays(shape)
    tokens = [int(t) for t in RNG.integers(0, shape.n_vocab, size=shape.n_ctx)]
    want = []
    _library_forward(shape, arrays, tokens, margins=want)
    m = oracle.Model(shape, arrays=arrays)
    st = m.new_state()
    for t, w in zip(tokens, want):
        st.forward(t)
        assert w > 0 and abs(st.route_margin - w) <= 1e-5, (st.route_margin, w)
    # three identical router rows, top-2: the unchosen expert ties the second
    shape3 = dataclasses.replace(TS, expert_count=3, expert_used=2)
    arrays3 = _rand_arrays(shape3)
    for l in range(shape3.n_layer):
        wr = arrays3[("wrouter", l, 0)]
        wr[1] = wr[0]
        wr[2] = wr[0]
    st3 = oracle.Model(shape3, arrays=arrays3).new_state()
    st3.forward(3)
    assert st3.route_margin == 0.0
    st_dense = oracle.Model(TS, arrays=_rand_arrays(TS)).new_state()
    st_dense.forward(3)
    assert st_dense.route_margin == math.inf

def test_residual_only_model_gives_closed_form_logits():
    arrays = _rand_arrays(TS)
    for l in range(TS.n_layer):
        arrays[("wo", l, 0)][:] = 0.0
        arrays[("wdown", l, 0)][:] = 0.0
    tokens = [3, 9, 3, 0, 15]
    got, _ = _oracle_run(TS, arrays, tokens)
    for p, t in enumerate(tokens):
        x = arrays["tok_embd"][t].astype(np.float64)
        xn = arrays["out_norm"][0] * x / np.sqrt(np.mean(x * x) + TS.rms_norm_eps)
        assert np.allclose(got[p], arrays["output"].astype(np.float64) @ xn, rtol=0, atol=1e-6)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    arrays = _rand_arrays(TS)
    mha = dataclasses.replace(TS, n_kv_head=TS.n_head)
    dup = dict(arrays)
    grp, hd = TS.n_head // TS.n_kv_head, TS.head_dim
    for l in range(TS.n_layer):
        for name in ("wk", "wv"):
            a = arrays[(name, l, 0)].reshape(TS.n_kv_head, hd, TS.n_embd)
            dup[(name, l, 0)] = np.repeat(a, grp, axis=0).reshape(TS.n_head * hd, TS.n_embd)
    tokens = [1, 5, 7, 2, 2, 11, 4, 0]
    a, _ = _oracle_run(TS, arrays, tokens)
    b, _ = _oracle_run(mha, dup, tokens)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_single_expert_top1_equals_dense_ffn():
    arrays = _rand_arrays(TS)
    moe = dataclasses.replace(TS, expert_count=1, expert_used=1)
    m_arrays = dict(arrays)
    for l in range(TS.n_layer):
        m_arrays[("wrouter", l, 0)] = f32(RNG.standard_normal((1, TS.n_embd)))
    tokens = [4, 4, 8, 1, 13]
    a, _ = _oracle_run(TS, arrays, tokens)
    b, _ = _oracle_run(moe, m_arrays, tokens)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_window_at_least_context_equals_no_window():
    arrays = _rand_arrays(TS)
    win = dataclasses.replace(TS, sliding_window=TS.n_ctx)
    tokens = [int(t) for t in RNG.integers(0, 16, size=TS.n_ctx)]
    a, _ = _oracle_run(TS, arrays, tokens)
    b, _ = _oracle_run(win, arrays, tokens)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_reset_then_replay_is_identical():
    m = oracle.Model(TS, arrays=_rand_arrays(TS))
    s = m.new_state()
    tokens = [2, 14, 6, 6, 1]
    first = [s.forward(t)[0] for t in tokens]
    s.reset()
    assert s.pos == 0 and np.all(s.kv(0, 0) == 0)
    second = [s.forward(t)[0] for t in tokens]
    for x, y in zip(first, second):
        assert np.array_equal(x, y)


def test_bad_token_and_full_cache_are_errors():
    m = oracle.Model(TS, arrays=_rand_arrays(TS))
    s = m.new_state()
    with pytest.raises(ValueError):
        s.forward(TS.n_vocab)
    s.pos = TS.n_ctx
    with pytest.raises(ValueError):
        s.forward(0)


def test_synth_prefill_writes_generated_cache_contents():
    shape = dataclasses.replace(TS, dtype=BF16)
    m = oracle.Model(shape, seed=9)
    s = m.new_state()
    s.prefill_synth(9, 3, 2, 7)
    assert s.pos == 7
    per = shape.n_kv_head * shape.head_dim
    for l in range(shape.n_layer):
        for kind, kk in ((0, synth.KCACHE), (1, synth.VCACHE)):
            kv = s.kv(l, kind).reshape(shape.n_ctx, per)
            want = synth.values(synth.key(9, kk, l, 3), 2 * per, 5 * per, 1.0, BF16).reshape(5, per)
            assert np.array_equal(kv[2:7], want)
            assert np.all(kv[:2] == 0) and np.all(kv[7:] == 0)


def test_synth_model_uses_generated_weights():
    """A seeded oracle model equals the same model given the generated arrays explicitly."""
    shape = dataclasses.replace(TS, dtype=BF16)
    arrays = {}
    for spec in wl.weight_specs(shape):
        k = spec.name if spec.name in ("tok_embd", "out_norm", "output") else (spec.name, spec.layer, spec.sub)
        if spec.const is None:
            arrays[k] = synth.values(spec.key(11), 0, spec.rows * spec.cols, wl.WEIGHT_SIGMA,
                                     BF16).reshape(spec.rows, spec.cols)
    a, _ = _oracle_run(shape, arrays, [1, 2, 3])
    m = oracle.Model(shape, seed=11)
    s = m.new_state()
    b = [s.forward(t)[0] for t in [1, 2, 3]]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_tiny_workload_matches_stored_oracle_run():
    """Regression guard: the stored run was written by tests/golden/make_tiny_golden.py,
    which calls only the oracle; a change to the oracle's arithmetic shows up here."""
    import importlib.util
    import os
    here = os.path.join(os.path.dirname(__file__), "golden")
    spec = importlib.util.spec_from_file_location("make_tiny_golden",
                                                  os.path.join(here, "make_tiny_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    stored = {}
    with open(os.path.join(here, "tiny_oracle_greedy.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            k, *vals = line.split()
            stored[k] = vals
    prompt, gen, top = mod.run()
    assert prompt == [int(v) for v in stored["prompt"]]
    assert gen == [int(v) for v in stored["generated"]]
    for (i, v), s in zip(top, stored["top5"]):
        si, sv = s.split(":")
        assert i == int(si) and math.isclose(v, float(sv), rel_tol=1e-6)


def test_step_in_parts_equals_forward():
    """embed + every layer + head (pos advanced by hand) reproduces forward bit for bit."""
    shape = dataclasses.replace(TS, dtype=BF16, sliding_window=4)
    arrays = _rand_arrays(shape)
    m = oracle.Model(shape, arrays=arrays)
    a, b = m.new_state(), m.new_state()
    for t in [3, 1, 4, 1, 5, 9, 2]:
        la, ama = a.forward(t)
        x = b.embed(t)
        for l in range(shape.n_layer):
            b.layer(l, x)
        lb, amb = b.head(x)
        b.pos = b.pos + 1
        assert np.array_equal(la, lb) and ama == amb


# ------------------------------------------------------------------ Q8 weights

def test_f16_conversion_matches_numpy():
    """The generator's fp32 -> fp16 rounding (nearest even) is numpy's, normal and subnormal."""
    vals = np.concatenate([RNG.uniform(1e-8, 6.1e-5, 2000), RNG.uniform(6.1e-5, 6.0e4, 4000),
                           np.float32(1.0) + np.float32(2.0 ** -11) * np.arange(8, dtype=np.float32),
                           [0.0, 5.960464477539063e-08, 6.103515625e-05, 65504.0]]).astype(np.float32)
    for v in vals:
        want = int(np.float32(v).astype(np.float16).view(np.uint16))
        got = synth.f32_to_f16_bits(float(v))
        assert got == want, (float(v), hex(got), hex(want))
        assert synth.f16_to_f32(got) == float(np.uint16(want).view(np.float16).astype(np.float32))


@pytest.mark.parametrize("cols,sigma", [(64, 0.02), (256, 1.0), (96, 3e-4)])
def test_q8_blocks_follow_their_definition(cols, sigma):
    """Each block of 32: d = fp16(max|w| / 127), q = clip(rint(w / d), -127, 127), from the
    generator's fp32 values, recomputed here with numpy; an unclamped weight d * q is
    within d / 2 of w (sigma 3e-4 gives subnormal fp16 scales)."""
    k = synth.key(5, synth.WQ, 3, 0)
    rows = 6
    raw, deq = synth.q8_rows(k, 2, rows, cols, sigma)
    for r in range(rows):
        w = synth.values(k, (2 + r) * cols, cols, sigma, F32)
        q = raw[r, :cols].view(np.int8)
        d = raw[r, cols:].view(np.uint16)
        for b in range(cols // 32):
            wb = w[32 * b:32 * b + 32]
            dw = (np.float32(np.max(np.abs(wb))) / np.float32(127)).astype(np.float16)
            assert d[b] == dw.view(np.uint16)
            df = np.float32(dw)
            qw = np.clip(np.rint(wb / df), -127, 127).astype(np.int8)
            assert np.array_equal(q[32 * b:32 * b + 32], qw)
            assert np.array_equal(deq[r, 32 * b:32 * b + 32], df * qw.astype(np.float32))
            inner = np.abs(qw) < 127   # clamped values (a coarse subnormal d) excepted
            assert np.all(np.abs(wb - df * qw)[inner] <= 0.5 * df * (1 + 2.0 ** -9))
            if df >= 2.0 ** -14:   # normal fp16 scale: the largest value uses the range
                assert np.max(np.abs(qw)) >= 126


@pytest.mark.parametrize("experts", [0, 4])
def test_q8_model_is_the_model_of_its_dequantized_weights(experts):
    """A seeded Q8 oracle model (with experts: router and experts in blocks too)
    equals the bf16-cache model given d * q explicitly."""
    shape = dataclasses.replace(TS, dtype=synth.Q8, n_embd=64, n_head=4, n_kv_head=2, n_ff=96,
                                expert_count=experts, expert_used=2 if experts else 0)
    arrays = {}
    for spec in wl.weight_specs(shape):
        k = spec.name if spec.name in ("tok_embd", "out_norm", "output") else (spec.name, spec.layer, spec.sub)
        if spec.const is None:
            arrays[k] = synth.q8_rows(spec.key(11), 0, spec.rows, spec.cols, wl.WEIGHT_SIGMA)[1]
    a, _ = _oracle_run(dataclasses.replace(shape, dtype=BF16), arrays, [1, 2, 3])
    m = oracle.Model(shape, seed=11)
    s = m.new_state()
    b = [s.forward(t)[0] for t in [1, 2, 3]]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ------------------------------------------------------------------ Q4 weights

@pytest.mark.parametrize("cols,sigma", [(64, 0.02), (256, 1.0), (96, 3e-4)])
def test_q4_blocks_follow_their_definition(cols, sigma):
    """Each block of 32: d = fp16(max|w| / 7), code u = clip(rint(w / d), -8, 7) + 8, two
    codes per byte (element 2j in the low nibble of byte j), the scales after the codes;
    the weight is d * (u - 8), recomputed here with numpy; an unclamped weight is within
    d / 2 of w (sigma 3e-4 gives subnormal fp16 scales)."""
    k = synth.key(5, synth.WQ, 3, 0)
    rows = 6
    raw, deq = synth.q4_rows(k, 2, rows, cols, sigma)
    assert raw.shape == (rows, cols // 2 + cols // 16)
    for r in range(rows):
        w = synth.values(k, (2 + r) * cols, cols, sigma, F32)
        packed = raw[r, :cols // 2]
        u = np.empty(cols, dtype=np.int32)
        u[0::2] = packed & 0xF
        u[1::2] = packed >> 4
        d = raw[r, cols // 2:].view(np.uint16)
        for b in range(cols // 32):
            wb = w[32 * b:32 * b + 32]
            dw = (np.float32(np.max(np.abs(wb))) / np.float32(7)).astype(np.float16)
            assert d[b] == dw.view(np.uint16)
            df = np.float32(dw)
            qw = np.clip(np.rint(wb / df), -8, 7).astype(np.int32)
            assert np.array_equal(u[32 * b:32 * b + 32], qw + 8)
            assert np.array_equal(deq[r, 32 * b:32 * b + 32], df * qw.astype(np.float32))
            inner = (qw > -8) & (qw < 7)
            assert np.all(np.abs(wb - df * qw)[inner] <= 0.5 * df * (1 + 2.0 ** -9))
            if df >= 2.0 ** -14:   # normal fp16 scale: the largest value uses the range
                assert np.max(np.abs(qw)) >= 6


@pytest.mark.parametrize("experts", [0, 4])
def test_q4_model_is_the_model_of_its_dequantized_weights(experts):
    """A seeded Q4 oracle model (with experts: router and experts in blocks too)
    equals the bf16-cache model given d * (u - 8) explicitly."""
    shape = dataclasses.replace(TS, dtype=synth.Q4, n_embd=64, n_head=4, n_kv_head=2, n_ff=96,
                                expert_count=experts, expert_used=2 if experts else 0)
    arrays = {}
    for spec in wl.weight_specs(shape):
        k = spec.name if spec.name in ("tok_embd", "out_norm", "output") else (spec.name, spec.layer, spec.sub)
        if spec.const is None:
            arrays[k] = synth.q4_rows(spec.key(11), 0, spec.rows, spec.cols, wl.WEIGHT_SIGMA)[1]
    a, _ = _oracle_run(dataclasses.replace(shape, dtype=BF16), arrays, [1, 2, 3])
    m = oracle.Model(shape, seed=11)
    s = m.new_state()
    b = [s.forward(t)[0] for t in [1, 2, 3]]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ------------------------------------------------------------------ sampling

def test_sample_uniform_is_splitmix64_published_sequence():
    # SplitMix64 seeded with 1234567: the first three outputs of the published
    # generator (Steele, Lea & Flood 2014; the sequence Vigna's reference C
    # code prints), top 24 bits scaled to [0, 1)
    for n, word in enumerate((6457827717110365317, 3203168211198807973, 9817491932198370423)):
        assert oracle.sample_uniform(1234567, n) == (word >> 40) / 2.0**24
    u = np.array([oracle.sample_uniform(99, n) for n in range(20000)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 0.01 and abs(u.var() - 1 / 12) < 0.005


def test_sample_temperature_zero_is_argmax_lowest_id():
    lg = f32([0.5, 3.0, -1.0, 3.0, 2.9])
    for T in (0.0, -1.0):
        for u in (0.0, 0.5, 0.999):
            assert oracle.sample(lg, T, u=u)[0] == 1


def test_sample_top_k_one_is_argmax_at_any_temperature():
    rng = np.random.default_rng(4)
    lg = f32(rng.normal(size=300))
    for T in (0.1, 1.0, 7.0):
        for u in (0.0, 0.37, 0.9999):
            tok, idx, cum = oracle.sample(lg, T, top_k=1, u=u)
            assert tok == int(np.argmax(lg)) and list(idx) == [tok] and cum[-1] == 1.0


def test_sample_three_token_closed_form():
    # logits ln 1, ln 2, ln 4 at T = 1: probabilities 1/7, 2/7, 4/7, drawn in
    # the order token 2, 1, 0 (cumulative 4/7, 6/7, 1)
    lg = f32(np.log([1.0, 2.0, 4.0]))
    tok, idx, cum = oracle.sample(lg, 1.0)
    assert list(idx) == [2, 1, 0]
    assert np.allclose(cum, [4 / 7, 6 / 7, 1.0], rtol=1e-6)
    for u, want in ((0.0, 2), (0.5, 2), (0.58, 1), (0.85, 1), (0.86, 0), (0.9999, 0)):
        assert oracle.sample(lg, 1.0, u=u)[0] == want
    # top-p 0.5: token 2 alone exceeds it; top-p 0.6: tokens 2 and 1 (2/3, 1/3)
    for u in (0.0, 0.5, 0.99):
        assert oracle.sample(lg, 1.0, top_p=0.5, u=u)[0] == 2
    _, idx, cum = oracle.sample(lg, 1.0, top_p=0.6)
    assert list(idx) == [2, 1] and np.allclose(cum, [2 / 3, 1.0])
    assert oracle.sample(lg, 1.0, top_p=0.6, u=0.66)[0] == 2
    assert oracle.sample(lg, 1.0, top_p=0.6, u=0.67)[0] == 1
    # top-k 2 keeps 2 and 1 whatever p
    _, idx, cum = oracle.sample(lg, 1.0, top_k=2)
    assert list(idx) == [2, 1] and np.allclose(cum, [2 / 3, 1.0])


def test_sample_top_p_boundary_is_exceeds_not_reaches():
    # four equal logits: probabilities 1/4 each (exact in binary), cumulative
    # 1/4, 1/2, 3/4, 1 - it reaches p = 1/2 at the second token and exceeds
    # it only at the third
    lg = f32([0.7, 0.7, 0.7, 0.7])
    _, idx, cum = oracle.sample(lg, 1.0, top_p=0.5)
    assert list(idx) == [0, 1, 2] and np.array_equal(cum, [1 / 3, 2 / 3, 1.0])
    _, idx, _ = oracle.sample(lg, 1.0, top_p=0.49)
    assert list(idx) == [0, 1]
    _, idx, _ = oracle.sample(lg, 1.0, top_p=0.0)
    assert list(idx) == [0]
    _, idx, _ = oracle.sample(lg, 1.0, top_p=1.0)
    assert list(idx) == [0, 1, 2, 3]


def test_sample_temperature_scales_the_logits():
    # logits 0, ln 2 at T = 1/2: z = 0, 2 ln 2, probabilities 1/5, 4/5
    lg = f32([0.0, np.log(2.0)])
    _, idx, cum = oracle.sample(lg, 0.5)
    assert list(idx) == [1, 0] and np.allclose(cum, [0.8, 1.0], rtol=1e-6)
    # very high temperature: uniform
    lg = f32(np.arange(10.0))
    _, idx, cum = oracle.sample(lg, 1e6)
    assert list(idx) == list(range(9, -1, -1)) and np.allclose(cum, np.arange(1, 11) / 10, atol=1e-4)


@pytest.mark.parametrize("a", [1.5, -1.5])
def test_sample_repetition_penalty_two_token_logistic(a):
    # token 0 has logit a, token 1 logit 0; token 0 repeated (twice: once
    # counts). Penalised z0 = a / 1.3 when a > 0, a * 1.3 when a < 0, so
    # p0 = 1 / (1 + exp(-z0))
    lg = f32([a, 0.0])
    z0 = a / 1.3 if a > 0 else a * 1.3
    p0 = 1.0 / (1.0 + math.exp(-z0))
    _, idx, cum = oracle.sample(lg, 1.0, repeat_penalty=1.3, recent=[0, 0, 7, -2])
    first = 0 if a > 0 else 1
    assert idx[0] == first
    assert math.isclose(cum[0], p0 if first == 0 else 1 - p0, rel_tol=1e-6)
    # penalty 1 and an empty window change nothing
    for kw in ({"repeat_penalty": 1.0, "recent": [0, 1]}, {"repeat_penalty": 2.0, "recent": []}):
        _, _, c = oracle.sample(lg, 1.0, **kw)
        assert math.isclose(c[0], max(1 / (1 + math.exp(-a)), 1 / (1 + math.exp(a))), rel_tol=1e-6)


def test_sample_penalty_follows_temperature():
    # temperature first, then the penalty: logit 2 at T = 2 is z = 1, divided
    # by 4 gives 0.25 - below token 1's z = 0.3 (logit 0.6)
    lg = f32([2.0, 0.6])
    _, idx, _ = oracle.sample(lg, 2.0, repeat_penalty=4.0, recent=[0])
    assert list(idx[:2]) == [1, 0]


def test_sample_ties_keep_lower_ids_in_top_k():
    lg = f32([1.0, 5.0, 5.0, 5.0, 0.0, 5.0])
    _, idx, cum = oracle.sample(lg, 1.0, top_k=3)
    assert list(idx) == [1, 2, 3] and np.allclose(cum, [1 / 3, 2 / 3, 1.0])


def test_sample_empirical_frequencies_match_kept_probabilities():
    # brute force: draws with uniform u land on each kept token with its
    # probability (the renormalised softmax of the kept z), nothing else is drawn
    rng = np.random.default_rng(8)
    lg = f32(rng.normal(size=40) * 2)
    T, k, p = 0.8, 12, 0.9
    _, idx, cum = oracle.sample(lg, T, top_k=k, top_p=p)
    z = lg.astype(np.float64) / T
    order = np.argsort(-z, kind="stable")[:k]
    assert list(idx) == list(order[:len(idx)])
    pk = sp.softmax(z[order])
    assert np.sum(pk[:len(idx) - 1]) <= p < np.sum(pk[:len(idx)])
    probs = sp.softmax(z[idx])
    n = 20000
    counts = np.zeros(40)
    for i in range(n):
        counts[oracle.sample(lg, T, top_k=k, top_p=p, u=oracle.sample_uniform(5, i))[0]] += 1
    assert counts.sum() == n and np.all(counts[np.setdiff1d(np.arange(40), idx)] == 0)
    sd = np.sqrt(n * probs * (1 - probs))
    assert np.all(np.abs(counts[idx] - n * probs) < 5 * sd + 1)


def test_qkv_bias_on_zero_projections_is_the_bias():
    # with Wq = Wk = Wv = 0 every value vector is the v bias, so whatever the
    # attention weights, each head's output is its KV head's v bias; with the
    # FFN zeroed the logits then have a closed form
    shape = dataclasses.replace(TS, qkv_bias=True, n_layer=1)
    arrays = _rand_arrays(shape)
    H, Hkv, hd = shape.n_head, shape.n_kv_head, shape.head_dim
    for name in ("wq", "wk", "wv"):
        arrays[(name, 0, 0)] = np.zeros_like(arrays[(name, 0, 0)])
    for name in ("wgate", "wup", "wdown"):
        arrays[(name, 0, 0)] = np.zeros_like(arrays[(name, 0, 0)])
    m = oracle.Model(shape, arrays=arrays)
    s = m.new_state()
    bv = arrays[("bv", 0, 0)].ravel().astype(np.float64)
    o = np.concatenate([bv[(h // (H // Hkv)) * hd:(h // (H // Hkv) + 1) * hd] for h in range(H)])
    for p, tok in enumerate((3, 9, 4)):
        lg, _ = s.forward(tok)
        x = arrays["tok_embd"][tok].astype(np.float64) + arrays[("wo", 0, 0)].astype(np.float64) @ o
        xn = arrays["out_norm"].ravel() * x / math.sqrt(np.mean(x * x) + shape.rms_norm_eps)
        want = arrays["output"].astype(np.float64) @ xn
        assert np.allclose(lg, want, rtol=0, atol=1e-5 * np.abs(want).max()), p


def test_bias_and_neox_models_differ_from_the_plain_model():
    # each variant flag changes the result (a dropped bias or rotation form fails here)
    base = dataclasses.replace(TS, qkv_bias=True)
    arrays = _rand_arrays(base)
    tokens = [int(t) for t in RNG.integers(0, TS.n_vocab, size=6)]
    plain = {k: v for k, v in arrays.items() if not (isinstance(k, tuple) and k[0][0] == "b")}
    runs = {}
    for name, shape, arr in (("plain", TS, plain), ("bias", base, arrays),
                             ("neox", dataclasses.replace(TS, rope_neox=True), plain)):
        runs[name] = _oracle_run(shape, arr, tokens)[0]
    for other in ("bias", "neox"):
        assert not np.allclose(runs["plain"][-1], runs[other][-1], atol=1e-3)
