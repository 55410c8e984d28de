"""Pins of the CPU oracle to facts other than itself: library routines (bf16 rounding,
sorting), closed forms, invariants and special cases of the decode step.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign, index or grouping, a transposed operand, a sequential instead of parallel
block) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import synth

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------- bf16

def test_bf16_widen_matches_torch_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_bf16_rounding_matches_torch_nearest_even():
    x = RNG.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # exact ties: bf16 value plus half an ulp, with even and odd low bit
    base = RNG.standard_normal(5000).astype(np.float32)
    b16 = base.view(np.uint32) & np.uint32(0xFFFF0000)
    ties = (b16 | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1.0, -2.5, 1e30, -1e-30])])
    ours = O.f64_to_bf16(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    big = np.abs(x) >= np.float32(2.0 ** -126)
    assert np.array_equal(ours[big], ref[big])


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    d, c, eps = 64, -0.37, 1e-6
    g = RNG.standard_normal(d)
    h = O.rms_norm(np.full(d, c), g, eps)
    assert np.allclose(h, g * c / math.sqrt(c * c + eps), rtol=0, atol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    x = RNG.standard_normal(128)
    h = O.rms_norm(x, np.ones(128), 0.0)
    assert abs(np.sqrt(np.mean(h * h)) - 1.0) < 1e-14
    assert np.allclose(O.rms_norm(7.5 * x, np.ones(128), 0.0), h, atol=1e-14)


# ----------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    v = RNG.standard_normal((3, 16))
    assert np.array_equal(O.rope(v, 0, 1e4), v)


def test_rope_preserves_norm_and_depends_on_relative_position():
    q, k = RNG.standard_normal(64), RNG.standard_normal(64)
    for p in (1, 17, 4095):
        assert abs(np.linalg.norm(O.rope(q, p, 1e6)) - np.linalg.norm(q)) < 1e-12
    a = O.rope(q, 100, 1e4) @ O.rope(k, 37, 1e4)
    b = O.rope(q, 163, 1e4) @ O.rope(k, 100, 1e4)
    assert abs(a - b) < 1e-11


def test_rope_basis_vector_closed_form_rotate_half():
    hd, theta, p = 32, 1e4, 5
    for i in (0, 3, 15):
        e = np.zeros(hd); e[i] = 1.0
        ang = p * theta ** (-2.0 * i / hd)
        want = np.zeros(hd); want[i] = math.cos(ang); want[i + hd // 2] = math.sin(ang)
        assert np.allclose(O.rope(e, p, theta), want, atol=1e-15)
        e2 = np.zeros(hd); e2[i + hd // 2] = 1.0
        want2 = np.zeros(hd); want2[i] = -math.sin(ang); want2[i + hd // 2] = math.cos(ang)
        assert np.allclose(O.rope(e2, p, theta), want2, atol=1e-15)


# ----------------------------------------------------------------- attention

def test_attention_single_key_returns_its_value():
    q = RNG.standard_normal((4, 8)); K = RNG.standard_normal((1, 2, 8))
    V = RNG.standard_normal((1, 2, 8))
    o = O.attention(q, K, V)
    assert np.allclose(o[:2], V[0, 0]) and np.allclose(o[2:], V[0, 1])


def test_attention_equal_keys_average_values():
    q = RNG.standard_normal((2, 8)); k = RNG.standard_normal(8)
    K = np.tile(k, (10, 1, 1)); V = RNG.standard_normal((10, 1, 8))
    assert np.allclose(O.attention(q, K, V), V[:, 0].mean(0), atol=1e-14)


def test_attention_two_keys_closed_form_with_sqrt_hd_scale():
    hd = 16
    q = np.zeros((1, hd)); q[0, 0] = 2.0
    K = np.zeros((2, 1, hd)); K[0, 0, 0] = 3.0; K[1, 0, 0] = -1.0
    V = RNG.standard_normal((2, 1, hd))
    s0, s1 = 6.0 / math.sqrt(hd), -2.0 / math.sqrt(hd)
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert np.allclose(O.attention(q, K, V)[0], p0 * V[0, 0] + (1 - p0) * V[1, 0],
                       atol=1e-14)


def test_attention_gqa_contiguous_groups():
    Hq, Hkv, hd, n = 8, 2, 8, 5
    q = RNG.standard_normal((Hq, hd)); K = RNG.standard_normal((n, Hkv, hd))
    V = RNG.standard_normal((n, Hkv, hd)); V[:, 1] = 0.0
    o = O.attention(q, K, V)
    assert np.all(o[4:] == 0.0)                 # heads 4..7 -> kv head 1
    assert np.all(np.abs(o[:4]).sum(1) > 0)     # heads 0..3 -> kv head 0


def test_split_kv_merge_equals_full_softmax():
    q = RNG.standard_normal((8, 32)); K = RNG.standard_normal((300, 2, 32)) * 2
    V = RNG.standard_normal((300, 2, 32))
    full = O.attention(q, K, V)
    for cuts in ([100], [1, 2, 299], [37, 64, 200, 250]):
        edges = [0] + cuts + [300]
        parts = [O.attention_partial(q, K[a:b], V[a:b]) for a, b in zip(edges, edges[1:])]
        assert np.allclose(O.merge_partials(parts), full, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- router / experts

def test_topk_matches_stable_full_sort_with_ties():
    for _ in range(200):
        r = np.round(RNG.standard_normal(32), 1)      # many exact ties
        k = int(RNG.integers(1, 9))
        idx, w, margin = O.router_topk(r, k)
        ref = np.lexsort((np.arange(32), -r))[:k]   # by -r, then index
        assert np.array_equal(idx, ref)
        assert abs(w.sum() - 1.0) < 1e-12
        srt = np.sort(r)[::-1]
        assert margin == srt[k - 1] - srt[k]


def test_topk_softmax_closed_forms():
    r = np.array([0.3, 2.0, -1.0, 1.5])
    idx, w, _ = O.router_topk(r, 1)
    assert list(idx) == [1] and w[0] == 1.0
    idx, w, _ = O.router_topk(r, 2)
    assert list(idx) == [1, 3]
    assert abs(w[0] - 1 / (1 + math.exp(1.5 - 2.0))) < 1e-15


def test_swiglu_scalar_closed_form():
    h = np.array([0.7]); wg = np.array([[1.3]]); wu = np.array([[-0.4]])
    wd = np.array([[2.0]])
    z = 1.3 * 0.7
    want = 2.0 * (z / (1 + math.exp(-z))) * (-0.4 * 0.7)
    assert abs(O.swiglu_expert(h, wg, wu, wd)[0] - want) < 1e-15


# ----------------------------------------------------------------- whole layer

TINY = dict(n_layers=2, d_model=32, n_q_heads=4, n_kv_heads=2, head_dim=8, n_experts=4,
            top_k=2, d_ff=16, vocab=50, rope_theta=1e4, rms_eps=1e-6, sliding_window=0,
            swa_layers=(), page_size=16)


def _setup(cfg=TINY, lens=(37, 5), seed=0, gain_jitter=0.2, std=0.2):
    W = synth.make_weights(cfg, seed=seed, gain_jitter=gain_jitter, std=std)
    pt, npages = synth.make_page_table(list(lens), seed=seed)
    k, v = synth.make_kv(cfg, npages, seed=seed)
    return W, pt, k, v


def _x(B, d, seed=3):
    return np.random.default_rng(seed).standard_normal((B, d))


def test_parallel_block_is_additive_in_its_two_branches():
    W, pt, k, v = _setup()
    x = _x(2, 32)
    kv = synth.HostKV(k, v)
    full, _ = O.layer_step(TINY, synth.HostWeights(W), kv, 0, x, [37, 5], pt)
    Wa = dict(W); Wa["w_down"] = torch.zeros_like(W["w_down"])
    attn_only, _ = O.layer_step(TINY, synth.HostWeights(Wa), kv, 0, x, [37, 5], pt)
    Wm = dict(W); Wm["wo"] = torch.zeros_like(W["wo"])
    moe_only, _ = O.layer_step(TINY, synth.HostWeights(Wm), kv, 0, x, [37, 5], pt)
    assert np.allclose(full - x, (attn_only - x) + (moe_only - x), atol=1e-13)
    assert np.abs(attn_only - x).max() > 1e-3 and np.abs(moe_only - x).max() > 1e-3


def test_zero_branches_leave_residual_and_logits_reduce_to_head_matvec():
    W, pt, k, v = _setup()
    W["wo"] = torch.zeros_like(W["wo"]); W["w_down"] = torch.zeros_like(W["w_down"])
    tok = [7, 41]
    out = O.decode_step(TINY, synth.HostWeights(W), synth.HostKV(k, v), tok, [37, 5], pt)
    x0 = O.bf16_to_f64(W["embed"][tok].view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(out["hidden"][-1], x0)
    g = O.bf16_to_f64(W["final_norm"].view(torch.int16).numpy().view(np.uint16))
    lm = O.bf16_to_f64(W["lm_head"].view(torch.int16).numpy().view(np.uint16))
    for b in range(2):
        h = x0[b] / math.sqrt(np.mean(x0[b] ** 2) + 1e-6) * g
        assert np.allclose(out["logits"][b], lm @ h, atol=1e-12)
        assert out["greedy"][b] == int(np.argmax(lm @ h))


def test_all_experts_with_identical_weights_equal_dense_swiglu():
    cfg = dict(TINY, top_k=4)
    W, pt, k, v = _setup(cfg)
    for name in ("w_gate", "w_up", "w_down"):
        W[name][:, 1:] = W[name][:, :1]
    W["wo"] = torch.zeros_like(W["wo"])
    x = _x(2, 32)
    HW = synth.HostWeights(W)
    y, info = O.layer_step(cfg, HW, synth.HostKV(k, v), 0, x, [37, 5], pt)
    g = O.bf16_to_f64(HW.attn_norm(0))
    wg, wu, wd = (O.bf16_to_f64(a) for a in HW.expert(0, 0))
    for b in range(2):
        h = x[b] / math.sqrt(np.mean(x[b] ** 2) + 1e-6) * g
        dense = wd @ ((wg @ h) / (1 + np.exp(-(wg @ h))) * (wu @ h))
        assert np.allclose(y[b] - x[b], dense, atol=1e-13)
        assert sorted(info["idx"][b]) == [0, 1, 2, 3]


def test_dense_layer_equals_moe_layer_of_identical_experts():
    """A dense layer of a mixed stack (one SwiGLU FFN for every token) equals an MoE
    layer whose experts are all copies of that FFN, whatever the routing (the weights
    sum to 1); the dense layer does not use the router."""
    cfg = dict(TINY, top_k=2)
    W, pt, k, v = _setup(cfg)
    for name in ("w_gate", "w_up", "w_down"):
        W[name][:, 1:] = W[name][:, :1]
    dcfg = dict(cfg, dense_layers=(0,), dense_ff=cfg["d_ff"])
    Wd = dict(W, ffn_gate=W["w_gate"][:, 0].clone(), ffn_up=W["w_up"][:, 0].clone(),
              ffn_down=W["w_down"][:, 0].clone(), router=torch.zeros_like(W["router"]))
    x = _x(2, 32)
    kv = synth.HostKV(k, v)
    y_moe, _ = O.layer_step(cfg, synth.HostWeights(W), kv, 0, x, [37, 5], pt)
    y_dense, info = O.layer_step(dcfg, synth.HostWeights(Wd), kv, 0, x, [37, 5], pt)
    assert np.allclose(y_dense, y_moe, atol=1e-13)
    assert info["experts"] == {} and info["idx"].shape == (2, 0)
    # layer 1 of the same stack is still routed
    _, info1 = O.layer_step(dcfg, synth.HostWeights(Wd), kv, 1, x, [37, 5], pt)
    assert info1["idx"].shape == (2, 2)


def test_first_token_attends_only_to_itself():
    W, pt, k, v = _setup(lens=(0,))
    W["w_down"] = torch.zeros_like(W["w_down"])
    x = _x(1, 32)
    HW = synth.HostWeights(W)
    y, info = O.layer_step(TINY, HW, synth.HostKV(k, v), 0, x, [0], pt)
    v16 = O.bf16_to_f64(info["kv"][0]["v"])             # [Hkv, hd]
    o = np.concatenate([v16[(i * 2) // 4] for i in range(4)])
    assert np.allclose(y[0] - x[0], O.bf16_to_f64(HW.wo(0)) @ o, atol=1e-13)


# ----------------------------------------------------------------- the query's rotation
# The rope() pins above test the rotation alone.  These two pin that layer_step
# rotates the QUERY at the token's own position: the first by the relative-position
# property of a whole layer, the second by where the attention peaks when query and
# keys share one raw vector.

Q1 = dict(n_layers=1, d_model=32, n_q_heads=4, n_kv_heads=2, head_dim=8, n_experts=4,
          top_k=2, d_ff=16, vocab=50, rope_theta=1e4, rms_eps=1e-6, sliding_window=0,
          swa_layers=(), page_size=16)


def _bf16_tensor(a):
    return torch.from_numpy(O.f64_to_bf16(a).view(np.int16)).view(torch.bfloat16)


def _with_query_rope(mutation, fn):
    """Run fn() with the query's rotation inside layer_step replaced by mutation(v, pos,
    theta, rope) (the query is the rope() argument with n_q_heads rows; keys have
    n_kv_heads); mutation None runs the oracle as it is."""
    if mutation is None:
        return fn()
    orig = O.rope

    def patched(v, pos, theta):
        v = np.asarray(v)
        if v.ndim == 2 and v.shape[0] == 4:
            return mutation(v, pos, theta, orig)
        return orig(v, pos, theta)
    O.rope = patched
    try:
        return fn()
    finally:
        O.rope = orig


_Q_MUTATIONS = {
    "unrotated": lambda v, pos, th, r: np.asarray(v, dtype=np.float64),
    "at position 0": lambda v, pos, th, r: r(v, 0, th),
    "one position late": lambda v, pos, th, r: r(v, pos + 1, th),
    "one position early": lambda v, pos, th, r: r(v, pos - 1, th),
    "negative angle": lambda v, pos, th, r: r(v, -pos, th),
}


def _shift_case(cfg, p, delta, x, raw_k, raw_v):
    """Attention branch of layer 1 (a sliding-window layer) at position p + delta, the
    cache holding at position j >= delta raw key raw_k[j - delta] rotated at j."""
    W = synth.make_weights(cfg, seed=0, std=0.2)
    W["w_down"] = torch.zeros_like(W["w_down"])
    n = p + delta
    pt, npages = synth.make_page_table([n], seed=0)
    k = torch.zeros((2, npages, 2, 16, 8), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    for j in range(delta, n):
        k[1, pt[0][j // 16], :, j % 16] = _bf16_tensor(O.rope(raw_k[j - delta], j, cfg["rope_theta"]))
        v[1, pt[0][j // 16], :, j % 16] = _bf16_tensor(raw_v[j - delta])
    y, _ = O.layer_step(cfg, synth.HostWeights(W), synth.HostKV(k, v), 1, x, [n], pt)
    return y - x


@pytest.mark.parametrize("mutation", [None] + list(_Q_MUTATIONS))
def test_layer_attention_depends_only_on_relative_positions(mutation):
    """RoPE makes a layer's attention invariant to shifting every position by delta
    (the window moves along; cached keys are re-rotated at their new positions).  Only
    bf16 rounding of the re-rotated keys differs, a relative error of ~1e-3 here; an
    unrotated query, one rotated at a fixed position or with the wrong sign breaks the
    invariance by O(1).  (A constant offset of the query's position keeps it: the next
    test pins that.)"""
    cfg = dict(Q1, n_layers=2, sliding_window=12, swa_layers=(1,))
    rng = np.random.default_rng(5)
    x = rng.standard_normal((1, 32))
    p = 20
    raw_k = rng.standard_normal((p, 2, 8)) * 3.0
    raw_v = rng.standard_normal((p, 2, 8))
    errs = []
    for delta in (1, 13, 1000, 70000):
        a, b = _with_query_rope(_Q_MUTATIONS.get(mutation), lambda: (
            _shift_case(cfg, p, 0, x, raw_k, raw_v), _shift_case(cfg, p, delta, x, raw_k, raw_v)))
        errs.append(np.linalg.norm(a - b) / np.linalg.norm(a))
    if mutation is None:
        assert max(errs) < 1e-2, errs
    elif mutation in ("one position late", "one position early"):
        assert max(errs) < 1e-2, errs        # a constant offset is shift-invariant
    else:
        assert max(errs) > 0.2, errs


@pytest.mark.parametrize("p", [37, 300])
@pytest.mark.parametrize("mutation", [None] + list(_Q_MUTATIONS))
def test_query_rotated_at_its_own_position(p, mutation):
    """Query and key share one raw vector u per KV group (the query rows of each head are
    the key rows of its KV group), and the cache holds at every position j the key u
    rotated at j + 2.  A rotation preserves length, so by Cauchy-Schwarz the score
    rot(u, p) . rot(u, j + 2) is largest exactly where the two rotations agree: at the
    cached position j = p - 2 and at the new token's own key (rotated at p), with equal
    bf16 bits.  With |u| large every other key's weight vanishes, so each head's output
    is the mean of those two values.  A query rotated at any other position moves the
    peak."""
    W = synth.make_weights(Q1, seed=0, std=0.2)
    W["w_down"] = torch.zeros_like(W["w_down"])
    W["wk"][0] = (W["wk"][0].float() * 15).to(torch.bfloat16)
    for i in range(4):
        g = (i * 2) // 4
        W["wq"][0, i * 8:(i + 1) * 8] = W["wk"][0, g * 8:(g + 1) * 8]
    W["wo"][0] = torch.eye(32, dtype=torch.bfloat16)
    W["attn_norm"][0] = 1.0
    HW = synth.HostWeights(W)
    x = np.random.default_rng(2).standard_normal((1, 32))
    u = (O.bf16_to_f64(HW.wk(0)) @ O.rms_norm(x, 1.0, 1e-6)[0]).reshape(2, 8)
    pt, npages = synth.make_page_table([p], seed=0)
    k = torch.zeros((1, npages, 2, 16, 8), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    vals = O.bf16_to_f64(O.f64_to_bf16(np.random.default_rng(9).standard_normal((p, 2, 8))))
    for j in range(p):
        k[0, pt[0][j // 16], :, j % 16] = _bf16_tensor(O.rope(u, j + 2, 1e4))
        v[0, pt[0][j // 16], :, j % 16] = _bf16_tensor(vals[j])
    y, info = _with_query_rope(_Q_MUTATIONS.get(mutation), lambda: O.layer_step(
        Q1, HW, synth.HostKV(k, v), 0, x, [p], pt))
    o = (y - x)[0].reshape(4, 8)                      # Wo = I: the heads' outputs
    v_new = O.bf16_to_f64(info["kv"][0]["v"])
    want = np.stack([(vals[p - 2, (i * 2) // 4] + v_new[(i * 2) // 4]) / 2 for i in range(4)])
    err = float(np.abs(o - want).max())
    if mutation is None:
        assert err < 5e-3, err
    else:
        assert err > 0.5, (mutation, err)


# ----------------------------------------------------------------- routing weights x experts

def _pairing_layer(swap_weights=False):
    """One MoE layer reduced to a closed form: constant inputs x_b = +-1 (so h_b = s_b 1,
    s_b = +-1/sqrt(1 + eps)), router row e = a_e / 32 (logit a_e s_b), gate and up rows
    g_e / 32 and u_e / 32 (every f-row gets g_e s_b and u_e s_b), and a down matrix that
    writes 1/16 of each f-row into output rows 8e..8e+7 only.  Expert e then adds
    w_{b,e} silu(g_e s_b) u_e s_b to its own eight outputs."""
    W = synth.make_weights(Q1, seed=0, std=0.2)
    W["wo"] = torch.zeros_like(W["wo"])
    W["attn_norm"][0] = 1.0
    a, g, u = [1.0, 0.5, -0.25, -2.0], [1.5, -0.75, 1.25, 0.5], [0.5, 1.0, -1.5, 0.75]
    for e in range(4):
        W["router"][0, e] = a[e] / 32
        W["w_gate"][0, e] = g[e] / 32
        W["w_up"][0, e] = u[e] / 32
        W["w_down"][0, e] = 0.0
        W["w_down"][0, e, 8 * e:8 * e + 8] = 1.0 / 16
    x = np.stack([np.full(32, 1.0), np.full(32, -1.0)])
    pt, npages = synth.make_page_table([3, 9], seed=0)
    k, v = synth.make_kv(Q1, npages, seed=0)
    orig = O.router_topk
    if swap_weights:                                   # a planted pairing slip
        def swapped(r, kk, forced=None):
            idx, w, m = orig(r, kk, forced)
            return idx, w[::-1].copy(), m
        O.router_topk = swapped
    try:
        y, info = O.layer_step(Q1, synth.HostWeights(W), synth.HostKV(k, v), 0, x, [3, 9], pt)
    finally:
        O.router_topk = orig
    want = np.zeros((2, 32))
    sel_want = []
    for b, sb in enumerate((1 / math.sqrt(1 + 1e-6), -1 / math.sqrt(1 + 1e-6))):
        logit = [a[e] * sb for e in range(4)]
        first, second = sorted(range(4), key=lambda e: -logit[e])[:2]
        sel_want.append([first, second])
        w_first = 1 / (1 + math.exp(logit[second] - logit[first]))   # 2-way softmax
        for e, w in ((first, w_first), (second, 1 - w_first)):
            z = g[e] * sb
            want[b, 8 * e:8 * e + 8] = w * (z / (1 + math.exp(-z))) * (u[e] * sb)
    return y - x, want, info, sel_want


def test_moe_combine_pairs_each_weight_with_its_expert():
    got, want, info, sel = _pairing_layer()
    assert info["idx"].tolist() == sel == [[0, 1], [3, 2]]
    assert np.abs(got - want).max() < 1e-13
    # the planted slip (weights handed to the wrong experts) is seen
    got_bad, _, _, _ = _pairing_layer(swap_weights=True)
    assert np.abs(got_bad - want).max() > 0.1


def test_kv_write_goes_to_page_table_slot_with_rotated_bf16_k():
    W, pt, k, v = _setup()
    x = _x(2, 32)
    HW = synth.HostWeights(W)
    _, info = O.layer_step(TINY, HW, synth.HostKV(k, v), 1, x, [37, 5], pt)
    for b, p in ((0, 37), (1, 5)):
        rec = info["kv"][b]
        assert rec["page"] == pt[b][p // 16] and rec["slot"] == p % 16
        g = O.bf16_to_f64(HW.attn_norm(1))
        h = x[b] / math.sqrt(np.mean(x[b] ** 2) + 1e-6) * g
        kn = O.rope((O.bf16_to_f64(HW.wk(1)) @ h).reshape(2, 8), p, 1e4)
        assert np.array_equal(rec["k"], O.f64_to_bf16(kn))


def test_paged_gather_equals_contiguous_cache_bit_exact():
    W, pt, k, v = _setup(lens=(45,))
    x = _x(1, 32)
    HW = synth.HostWeights(W)
    y1, _ = O.layer_step(TINY, HW, synth.HostKV(k, v), 0, x, [45], pt)
    # same logical cache stored contiguously: logical page i at physical page i
    n = pt.shape[1]
    idx = torch.as_tensor(pt[0].astype(np.int64))
    k2, v2 = k[:, idx].clone(), v[:, idx].clone()
    pt2 = np.arange(n, dtype=np.int32)[None]
    y2, _ = O.layer_step(TINY, HW, synth.HostKV(k2, v2), 0, x, [45], pt2)
    assert np.array_equal(y1, y2)


def test_sliding_window_ignores_keys_outside_and_full_window_matches():
    cfg = dict(TINY, sliding_window=8, swa_layers=(1,))
    W, pt, k, v = _setup(cfg, lens=(40,))
    x = _x(1, 32)
    HW = synth.HostWeights(W)
    base, _ = O.layer_step(cfg, HW, synth.HostKV(k, v), 1, x, [40], pt)
    k2, v2 = k.clone(), v.clone()
    for pos in range(0, 33):             # window of 8 at p=40 keeps 33..40
        k2[1, pt[0][pos // 16], :, pos % 16] = float("nan")
        v2[1, pt[0][pos // 16], :, pos % 16] = float("nan")
    got, _ = O.layer_step(cfg, HW, synth.HostKV(k2, v2), 1, x, [40], pt)
    assert np.array_equal(base, got)
    full_cfg = dict(cfg, sliding_window=41)
    a, _ = O.layer_step(full_cfg, HW, synth.HostKV(k, v), 1, x, [40], pt)
    b, _ = O.layer_step(TINY, HW, synth.HostKV(k, v), 1, x, [40], pt)
    assert np.array_equal(a, b)
    # the window really cuts: a NaN at position 33 must reach the output
    k2[1, pt[0][33 // 16], :, 33 % 16] = float("nan")
    got, _ = O.layer_step(cfg, HW, synth.HostKV(k2, v2), 1, x, [40], pt)
    assert np.isnan(got).any()


def test_argmax_lowest_index_on_ties():
    assert O.argmax_lowest([1.0, 3.0, 3.0, 2.0]) == 1


# ----------------------------------------------------------------- SoL arithmetic

def _golden(name):
    import os
    vals = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                kk, vv = line.split("=")
                vals[kk.strip()] = float(vv)
    return vals


def test_sol_arithmetic_reproduces_the_pages_h100_numbers():
    from persistent_moe_decode_cta_gb300 import sol
    g = _golden("sol_h100.txt")
    nbytes = g["weight_bytes"] + g["kv_bytes_8k"]
    assert abs(nbytes - g["bytes_per_token"]) < 1e-9 * nbytes
    tok = sol.sol_tok_s(nbytes, g["hbm_bytes_per_s"])
    assert abs(tok - g["sol_tok_s"]) / g["sol_tok_s"] < 0.01
    assert round(1e3 * sol.sol_seconds(nbytes, g["hbm_bytes_per_s"]), 1) == g["floor_ms"]
    assert round(100 * g["megakernel_tok_s"] / g["sol_tok_s"]) == g["megakernel_pct_of_sol"]
    assert round(100 * g["vllm_tok_s"] / g["sol_tok_s"]) == g["vllm_pct_of_sol"]
    assert round(1e3 / g["vllm_tok_s"], 1) == g["vllm_ms_per_step"]
    assert round(1e3 / g["megakernel_tok_s"], 1) == g["megakernel_ms_per_step"]
    floor = g["floor_ms"]
    assert round(g["vllm_ms_per_step"] - floor, 1) == g["vllm_ms_above_floor"]
    assert round(g["megakernel_ms_per_step"] - floor, 1) == g["megakernel_ms_above_floor"]
    closed = g["vllm_ms_per_step"] - g["megakernel_ms_per_step"]
    assert round(closed, 1) == g["gap_closed_ms"]
    assert abs(100 * closed / g["vllm_ms_above_floor"] - g["gap_closed_pct"]) < 2
    assert round(g["megakernel_tok_s"] / g["vllm_tok_s"], 2) == g["speedup"]


def test_param_counts_of_the_pages_scale_model():
    from persistent_moe_decode_cta_gb300 import sol
    g = _golden("sol_h100.txt")
    pc = sol.param_counts(synth.MODELS["pages"])
    assert pc["total"] == 30_532_012_032
    # the pages round down: "30B" total, "3.3B" active (the full embedding table counted)
    assert int(pc["total"] / 1e9) == int(g["total_params"] / 1e9)
    assert int(pc["active_with_embedding"] / 1e8) == int(g["active_params"] / 1e8)
    assert pc["active_step"] == 3_041_757_184


def test_step_bytes_pages_b1_8k():
    from persistent_moe_decode_cta_gb300 import sol
    cfg = synth.model_config("pages_b1_8k")
    sb = sol.step_bytes(cfg, [8192], [8] * 48)
    assert sb["kv"] == 48 * 8192 * 2 * 4 * 128 * 2
    assert abs(sb["weights"] - 6.0835e9) < 1e6


# ---------------------------------------------------------------- FP8 (E4M3) weights
def test_e4m3_every_finite_code_decodes_and_encodes_back_to_itself():
    c = np.arange(256, dtype=np.uint8)
    finite = (c & 0x7F) != 0x7F
    v = O.e4m3_to_f64(c[finite])
    assert np.array_equal(O.f32_to_e4m3(v.astype(np.float32)), c[finite])
    assert O.e4m3_to_f64(np.uint8(0x7E)) == 448.0 and O.e4m3_to_f64(np.uint8(0x01)) == 2.0 ** -9
    assert O.e4m3_to_f64(np.uint8(0x08)) == 2.0 ** -6 and O.e4m3_to_f64(np.uint8(0x38)) == 1.0


def test_e4m3_rounding_is_nearest_even_with_saturation_by_brute_force():
    """Against the nearest of all 254 finite values by exhaustive search (ties to the
    even code), for random values across the whole range and for exact midpoints."""
    c = np.arange(256, dtype=np.uint8)
    c = c[(c & 0x7F) != 0x7F]
    vals = O.e4m3_to_f64(c)
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(3000) * 10.0, rng.standard_normal(1000) * 1e-2,
                        rng.uniform(-600, 600, 500)]).astype(np.float32)
    srt = np.unique(vals)
    mids = ((srt[1:] + srt[:-1]) / 2).astype(np.float32)            # exact in float32
    x = np.concatenate([x, mids, -mids])
    got = O.f32_to_e4m3(x)
    for xi, gi in zip(x.astype(np.float64), got):
        t = np.clip(xi, -448.0, 448.0)
        d = np.abs(vals - t)
        best = c[d == d.min()]
        if len(best) > 1:                                           # a tie: the even code
            best = best[(best & 1) == 0]
            if len(best) > 1:                                       # +0 / -0
                best = best[(best & 0x80) == (0x80 if np.signbit(xi) else 0)]
        assert gi == best[0], (xi, gi, best)


def test_e4m3_row_quantisation_scale_and_error_bound():
    rng = np.random.default_rng(3)
    w = O.f64_to_bf16(rng.standard_normal((16, 96)) * 0.02)
    for block in (None, 32):
        codes, scale = O.quantize_e4m3_rows(w, block)
        wq = O.dequantize_e4m3(codes, scale, block)
        wf = O.bf16_to_f64(w)
        nb = 1 if block is None else 96 // block
        amax = np.abs(wf.reshape(16, nb, -1)).max(axis=2)
        # the largest magnitude of each row (block) maps to the code 448
        assert np.allclose(np.abs(O.e4m3_to_f64(codes).reshape(16, nb, -1)).max(axis=2), 448.0)
        assert np.array_equal(np.asarray(scale).reshape(16, nb), (amax / 448.0).astype(np.float32))
        # error at most half a step of the code's binade (relative 2^-4) or of the subnormal grid
        s = np.repeat(np.asarray(scale, dtype=np.float64).reshape(16, nb), 96 // nb, axis=1)
        err = np.abs(wq - wf) / s
        assert np.all(err <= np.maximum(np.abs(wf) / s * 2.0 ** -4, 2.0 ** -10) + 1e-12)


def test_fp8_experts_change_the_layer_only_by_the_quantisation():
    """With expert_dtype fp8 the layer equals the bf16 layer computed on the decoded
    weights, and differs from the bf16 weights' layer by a small amount."""
    cfg = dict(TINY, d_ff=64)
    W, pt, k, v = _setup(cfg)
    x = _x(2, 32)
    HW = synth.HostWeights(W)
    kv = synth.HostKV(k, v)
    y16, info16 = O.layer_step(cfg, HW, kv, 0, x, [37, 5], pt)
    y8, info8 = O.layer_step(dict(cfg, expert_dtype="fp8"), HW, kv, 0, x, [37, 5], pt)
    assert [list(a) for a in info8["idx"]] == [list(a) for a in info16["idx"]]
    rel = np.linalg.norm(y8 - y16) / np.linalg.norm(y16 - x)
    assert 0 < rel < 0.1
    # the same layer computed by hand from the decoded expert matrices
    g = O.bf16_to_f64(HW.attn_norm(0))
    for b in range(2):
        h = x[b] / math.sqrt(np.mean(x[b] ** 2) + 1e-6) * g
        moe = sum(w * O.swiglu_expert(h, *O.fp8_expert(*HW.expert(0, int(e))))
                  for e, w in zip(info8["idx"][b], info8["w"][b]))
        moe16 = sum(w * O.swiglu_expert(h, *(O.bf16_to_f64(a) for a in HW.expert(0, int(e))))
                    for e, w in zip(info16["idx"][b], info16["w"][b]))
        assert np.allclose((y8[b] - y16[b]), moe - moe16, atol=1e-12)


def test_fp8_expert_scales_are_per_output_channel():
    """Every decoded row of gate, up and down is an E4M3 value times one scale, the
    row's max|w| / 448 computed here from the bf16 weights, and the row's largest
    weight decodes to 448 times it (per-block scales would fail the first check on
    rows whose blocks have different maxima)."""
    cfg = dict(TINY, d_ff=64)
    W, _, _, _ = _setup(cfg)
    HW = synth.HostWeights(W)
    grid = np.unique(np.abs(O.e4m3_to_f64(np.arange(256, dtype=np.uint8)[(np.arange(256) & 0x7F) != 0x7F])))
    for e in range(3):
        for w16, wq in zip(HW.expert(0, e), O.fp8_expert(*HW.expert(0, e))):
            wf = O.bf16_to_f64(w16)
            scale = (np.abs(wf).max(axis=1).astype(np.float32) / np.float32(448.0)).astype(np.float64)
            v = np.abs(wq) / scale[:, None]
            assert np.all(np.isin(v, grid)), e
            assert np.array_equal(v.max(axis=1), np.full(wf.shape[0], 448.0))


# ----------------------------------------------------------------- FP8 dense projections

def _e4m3_grid_bf16(shape, k, seed):
    """bf16 matrices whose rows lie exactly on the E4M3 grid of scale 2^-k: random finite
    codes times 2^-k, each row's first element +-448 * 2^-k (so the row's max|w| / 448 is
    2^-k and quantisation is lossless)."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=shape).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10                     # no NaN codes
    v = O.e4m3_to_f64(codes) * 2.0 ** -k
    v[..., 0] = np.where(rng.random(shape[:-1]) < 0.5, -448.0, 448.0) * 2.0 ** -k
    return torch.from_numpy(v).to(torch.bfloat16)            # exact: 4 significant bits


def _fp8w(cfg):
    return dict(cfg, expert_dtype="fp8", dense_dtype="fp8")


def test_fp8_dense_projections_are_lossless_on_the_e4m3_grid():
    """Projections whose weights lie on the E4M3 grid of their row scales quantise
    without loss, so the layer and the LM head with FP8 dense projections (and FP8
    experts on the grid too) equal the bf16 ones exactly: the FP8 reading applies the
    same matrices in the same places."""
    cfg = dict(TINY, d_ff=64)
    W, pt, k, v = _setup(cfg)
    for i, name in enumerate(("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")):
        W[name] = _e4m3_grid_bf16(tuple(W[name].shape), 9, seed=i)
    W["lm_head"] = _e4m3_grid_bf16(tuple(W["lm_head"].shape), 8, seed=9)
    HW, kv = synth.HostWeights(W), synth.HostKV(k, v)
    x = _x(2, 32)
    for l in (0, 1):
        y16, i16 = O.layer_step(cfg, HW, kv, l, x, [37, 5], pt)
        y8, i8 = O.layer_step(_fp8w(cfg), HW, kv, l, x, [37, 5], pt)
        assert np.array_equal(y8, y16) and np.array_equal(i8["idx"], i16["idx"])
        for r16, r8 in zip(i16["kv"], i8["kv"]):
            assert np.array_equal(r8["k"], r16["k"]) and np.array_equal(r8["v"], r16["v"])
    assert np.array_equal(O.lm_head(_fp8w(cfg), HW, x), O.lm_head(cfg, HW, x))


def test_fp8_dense_projections_change_the_layer_only_by_the_quantisation():
    """On random weights the FP8 projections move the layer's output and the logits by
    a small relative amount (E4M3 keeps 3 mantissa bits: per-weight error <= 1/16 of
    the value), the routing weights' source -- the bf16 router -- is untouched, and the
    query, key and value heads differ from the bf16 ones only through Wq, Wk, Wv."""
    cfg = dict(TINY, d_ff=64)
    W, pt, k, v = _setup(cfg)
    HW, kv = synth.HostWeights(W), synth.HostKV(k, v)
    x = _x(2, 32)
    y16, i16 = O.layer_step(dict(cfg, expert_dtype="fp8"), HW, kv, 0, x, [37, 5], pt)
    y8, i8 = O.layer_step(_fp8w(cfg), HW, kv, 0, x, [37, 5], pt)
    assert np.array_equal(i8["router_logits"], i16["router_logits"])   # router stays bf16
    rel = np.linalg.norm(y8 - y16) / np.linalg.norm(y16 - x)
    assert 0 < rel < 0.1, rel
    # the K the layer writes is bf16(RoPE(decoded Wk h))
    g = O.bf16_to_f64(HW.attn_norm(0))
    for b, p in ((0, 37), (1, 5)):
        h = x[b] / math.sqrt(np.mean(x[b] ** 2) + 1e-6) * g
        kn = O.rope((O.fp8_matrix(HW.wk(0)) @ h).reshape(2, 8), p, 1e4)
        assert np.array_equal(i8["kv"][b]["k"], O.f64_to_bf16(kn))
    l8, l16 = O.lm_head(_fp8w(cfg), HW, x), O.lm_head(cfg, HW, x)
    assert 0 < np.abs(l8 - l16).max() < 0.1 * np.abs(l16).max()


def test_fp8_dense_scales_are_per_output_channel():
    """Each decoded row of Wq, Wk, Wv, Wo and the LM head is an E4M3 value times one
    scale, the row's max|w| / 448, and the row's largest weight decodes to 448 times it."""
    W, _, _, _ = _setup(dict(TINY, d_ff=64))
    HW = synth.HostWeights(W)
    grid = np.unique(np.abs(O.e4m3_to_f64(np.arange(256, dtype=np.uint8)[(np.arange(256) & 0x7F) != 0x7F])))
    for w16 in (HW.wq(0), HW.wk(1), HW.wv(0), HW.wo(1), HW.lm_head()):
        wf = O.bf16_to_f64(w16)
        scale = (np.abs(wf).max(axis=1).astype(np.float32) / np.float32(448.0)).astype(np.float64)
        vq = np.abs(O.fp8_matrix(w16)) / scale[:, None]
        assert np.all(np.isin(vq, grid))
        assert np.array_equal(vq.max(axis=1), np.full(wf.shape[0], 448.0))
