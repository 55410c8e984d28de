"""GPU behaviour beyond single-step parity: consecutive steps (device seq_len advance
and the cache each step leaves), sliding-window layers, ragged batches on the small
model, per-op/graph equivalence, and the device error paths (bad page id, bad token,
a dependency that can never complete) -- none of which faults the GPU."""
import numpy as np
import pytest
import torch

import oracle
import synth
from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


def _engine(workload, seq_lens=None, steps=1, seed=0, **kw):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seed=seed, seq_lens=seq_lens,
                                                      steps=steps)
    cfg = dict(cfg, **kw)
    mk = B.Megakernel(cfg, W, max_batch=8)
    pt_dev = torch.as_tensor(pt, device="cuda")
    mk.plan(seq, pt_dev, npages)
    return cfg, W, seq, pt, pt_dev, npages, k, v, tokens, mk


def test_three_consecutive_steps_match_oracle_and_advance_seq_lens():
    cfg, W, seq, pt, pt_dev, npages, k, v, tokens, mk = _engine("tiny_b1_64", [61, 14], steps=3)
    logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
    cur = list(seq)
    for step in range(3):
        kb, vb = k.clone(), v.clone()
        mk.step(tokens, k, v, logits)
        assert mk.status()["code"] == 0
        PU.check_step(cfg, mk, W, cur, pt, (kb, vb), tokens.cpu().numpy(), logits, k, v)
        cur = [c + 1 for c in cur]
        assert list(mk.seq_lens()) == cur
        # feed back the greedy tokens (the crosses page boundaries: 61 -> 64)
        tokens = logits.argmax(-1).to(torch.int32)
    mk.close()


def test_sliding_window_layers_match_oracle():
    cfg = dict(synth.model_config("tiny_b1_64"), sliding_window=20, swa_layers=(1,))
    W = synth.make_weights(cfg, seed=3, device="cuda", gain_jitter=0.1)
    seq = [64, 19, 20, 21, 0]
    pt, npages = synth.make_page_table(seq, seed=3)
    k, v = synth.make_kv(cfg, npages, seed=3, device="cuda")
    tokens = synth.make_tokens(len(seq), cfg["vocab"], seed=3, device="cuda")
    kb, vb = k.clone(), v.clone()
    mk = B.Megakernel(cfg, W)
    mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
    logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
    mk.step(tokens, k, v, logits)
    assert mk.status()["code"] == 0
    PU.check_step(cfg, mk, W, seq, pt, (kb, vb), tokens.cpu().numpy(), logits, k, v)
    mk.close()


def test_small_model_batch8_ragged_matches_oracle():
    cfg, W, seq, pt, pt_dev, npages, k, v, tokens, mk = _engine(
        "small_b1_2k", [2048, 1, 700, 16, 15, 17, 1023, 300])
    kb, vb = k.clone(), v.clone()
    logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
    mk.step(tokens, k, v, logits)
    assert mk.status()["code"] == 0
    PU.check_step(cfg, mk, W, seq, pt, (kb, vb), tokens.cpu().numpy(), logits, k, v)
    mk.close()


def test_perop_graph_and_megakernel_agree():
    """Each mode is checked against the oracle.  The modes are not bit-identical: the
    MoE combine adds fp32 partials atomically, and a last-bit difference in the sum
    can move the next layer's bf16 operand across a rounding boundary (one bf16 ulp,
    which shifts every GEMV output of that layer by ~1e-4), or decide a router near-tie
    the other way.  Rows whose expert selections match in every layer must therefore
    agree within the logit tolerance of the oracle comparison; a row whose selection
    differs has already been accepted as a near-tie by the oracle check."""
    cfg, W, seq, pt, pt_dev, npages, k, v, tokens, mk = _engine("small_b1_2k", [900, 31])
    mk.set_fixed(True)
    outs, routes = [], []
    for mode in ("mega", "perop", "graph", "mega"):
        kb, vb = k.clone(), v.clone()
        lg = torch.empty(len(seq), cfg["vocab"], device="cuda")
        if mode == "mega":
            mk.step(tokens, k, v, lg)
        else:
            mk.step_perop(tokens, k, v, lg, use_graph=(mode == "graph"))
        assert mk.status()["code"] == 0
        PU.check_step(cfg, mk, W, seq, pt, (kb, vb), tokens.cpu().numpy(), lg, k, v)
        outs.append(lg.cpu().numpy())
        routes.append(np.sort(mk.routes()[0], axis=-1))
    same = [b for b in range(len(seq)) if all(np.array_equal(r[:, b], routes[0][:, b])
                                              for r in routes[1:])]
    for o in outs[1:]:
        if same:
            assert np.abs(o[same] - outs[0][same]).max() <= PU.LOGIT_ABS
    assert list(mk.seq_lens()) == seq
    mk.close()


def test_bad_page_id_reports_error_without_writing():
    cfg, W, seq, pt, pt_dev, npages, k, v, tokens, mk = _engine("tiny_b1_64", [40])
    pt_dev[0, 40 // 16] = npages + 5            # the page of the new token is invalid
    kb = k.clone()
    logits = torch.empty(1, cfg["vocab"], device="cuda")
    mk.step(tokens, k, v, logits)
    st = mk.status()
    assert st["code"] == B.MK_ERR_BAD_PAGE and st["observed"] == npages + 5
    assert torch.equal(k.view(torch.int16), kb.view(torch.int16))
    assert mk.status()["code"] == 0           # cleared once read
    mk.close()


def test_bad_token_reports_error():
    cfg, W, seq, pt, pt_dev, npages, k, v, tokens, mk = _engine("tiny_b1_64", [8])
    bad = torch.tensor([cfg["vocab"] + 3], dtype=torch.int32, device="cuda")
    logits = torch.empty(1, cfg["vocab"], device="cuda")
    mk.step(bad, k, v, logits)
    st = mk.status()
    assert st["code"] == B.MK_ERR_BAD_TOKEN and st["observed"] == cfg["vocab"] + 3
    mk.close()


@pytest.mark.parametrize("batch", [1, 3])
def test_exact_router_ties_go_to_the_lower_expert_id(batch):
    """Three experts with identical router rows, scaled to be every token's largest
    logits, give bit-equal logits: top-2 must take the two lowest ids of the three, in
    that order, with equal weights (the oracle's tie rule)."""
    lens = [40, 7, 100][:batch]
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup("tiny_b1_64", seq_lens=lens, gain_jitter=0.0)
    W["attn_norm"][:] = 1.0
    for l in range(cfg["n_layers"]):
        W["router"][l] *= 0.1
        row = W["router"][l, 0].clone() * 0.0 + 0.05      # every logit of these rows: 0.05 * sum(h)
        for e in (6, 1, 4):
            W["router"][l, e] = row
    # sum(h) > 0 for every token makes the tied logits the largest
    mk = B.Megakernel(cfg, W, max_batch=8)
    mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
    logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
    mk.step(tokens, k, v, logits)
    assert mk.status()["code"] == 0
    lg = mk.router_logits()
    idx, w = mk.routes()
    for l in range(cfg["n_layers"]):
        for b in range(len(seq)):
            if lg[l, b, 1] > np.sort(lg[l, b])[-4]:     # the tied three lead this token
                assert lg[l, b, 1] == lg[l, b, 4] == lg[l, b, 6]
                assert [int(e) for e in idx[l, b]] == [1, 4], (l, b, idx[l, b])
                assert w[l, b, 0] == w[l, b, 1]
    mk.close()


def test_nan_router_logit_reports_error_and_routes_to_valid_experts():
    """A router row of NaNs (non-finite weights: invalid input the route step checks)
    makes that expert's logit NaN: the step completes with a full, valid top-k that
    skips it, and reports MK_ERR_NAN with the layer and the logit's index."""
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup("tiny_b1_64", seq_lens=[40, 7])
    W["router"][1, 3] = float("nan")
    mk = B.Megakernel(cfg, W)
    mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
    logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
    mk.step(tokens, k, v, logits)
    st = mk.status()
    assert st["code"] == B.MK_ERR_NAN and st["observed"] == 1 and st["target"] % cfg["n_experts"] == 3
    idx, w = mk.routes()
    for b in range(len(seq)):
        sel = [int(e) for e in idx[1, b]]
        assert len(set(sel)) == cfg["top_k"] and 3 not in sel and all(0 <= e < cfg["n_experts"] for e in sel)
        assert abs(float(w[1, b].sum()) - 1.0) < 1e-5
    assert not mk.counters().any()
    mk.step(tokens, k, v, logits)               # the context and the handle still work
    assert mk.status()["code"] == B.MK_ERR_NAN
    mk.close()


def test_dropped_signal_times_out_and_the_context_survives():
    """A QKV tile whose completion signal is dropped (host-side injection): the
    attention splits waiting for its KV group give up after timeout_ms, the step
    reports MK_ERR_TIMEOUT naming the group's counter, every CTA exits, and after
    re-planning the next step is correct."""
    cfg, W, seq, pt, pt_dev, npages, k, v, tokens, mk0 = _engine("tiny_b1_64", [40])
    mk0.close()
    mk = B.Megakernel(cfg, W, timeout_ms=200)
    mk.plan(seq, pt_dev, npages)
    T, off, lst, info = B.mk_plan_dry(cfg, 1, mk.query(B.MK_Q_NUM_SMS))
    qkv0 = [t for t in range(len(T)) if T[t][0] == 2 and T[t][1] == 0 and T[t][2] == 0][0]
    B.mk_plan_drop_signal(mk.h, qkv0)
    logits = torch.empty(1, cfg["vocab"], device="cuda")
    mk.step(tokens, k, v, logits)
    st = mk.status()
    assert st["code"] == B.MK_ERR_TIMEOUT, st
    assert st["counter"] == info[17] + 0      # QKV group 0 of layer 0
    assert st["target"] == info[10] and st["observed"] == info[10] - 1
    # re-plan: the same context runs a correct step
    kb, vb = k.clone(), v.clone()
    mk.plan(seq, pt_dev, npages)
    mk.step(tokens, k, v, logits)
    assert mk.status()["code"] == 0
    PU.check_step(cfg, mk, W, seq, pt, (kb, vb), tokens.cpu().numpy(), logits, k, v)
    mk.close()
