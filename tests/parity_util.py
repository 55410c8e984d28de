"""Shared helpers for the GPU-vs-oracle parity tests.

Acceptance (from the decode-step contract):
  * bookkeeping bit-exact: written K/V page/slot, untouched cache bytes unchanged,
    active-expert sets and per-expert token lists, counters back at zero;
  * expert selection identical wherever the oracle's top-k margin >= 1e-3, the
    oracle's router being evaluated on the GPU's own layer input (below that margin
    either set is correct); the free-running oracle then takes the GPU's selections;
  * per-layer hidden-state relative L2 error <= 1e-2;
  * logits max |diff| <= 0.05 and the same greedy argmax (unless the oracle's
    top-2 gap is below 2 * max|diff|, a reported tie).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

MARGIN = 1e-3
REL_L2 = 1e-2
LOGIT_ABS = 0.05


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def setup(workload, seed=0, steps=1, gain_jitter=0.1, device="cuda", seq_lens=None, batch=None,
          cfg_update=None):
    cfg = synth.model_config(workload)
    cfg.update(cfg_update or {})
    W = synth.make_weights(cfg, seed=seed, device=device, gain_jitter=gain_jitter)
    seq = list(seq_lens) if seq_lens is not None else synth.seq_lens_for(workload, seed)
    if batch is not None:
        seq = (seq * batch)[:batch]
    pt, npages = synth.make_page_table(seq, steps=steps, seed=seed)
    k, v = synth.make_kv(cfg, npages, seed=seed, device=device)
    tokens = synth.make_tokens(len(seq), cfg["vocab"], seed=seed, device=device)
    return cfg, W, seq, pt, npages, k, v, tokens


def check_routing_teacher_forced(cfg, HW, hid, gidx, gw, B):
    """Routing decisions, layer by layer, against the oracle's router evaluated on the
    GPU's own residual x_l: identical expert sets wherever the oracle's top-k margin
    is >= MARGIN; weights within 1e-3 of the oracle's softmax over the GPU's
    selection.  Returns the number of (layer, token) near-ties seen."""
    ties = 0
    dense = tuple(cfg.get("dense_layers", ()))
    for l in range(cfg["n_layers"]):
        if l in dense:  # a dense layer of a mixed stack routes nothing
            continue
        h = oracle.rms_norm(hid[l].astype(np.float64), oracle.bf16_to_f64(HW.attn_norm(l)),
                            cfg["rms_eps"])
        r = h @ oracle.bf16_to_f64(HW.router(l)).T
        for b in range(B):
            idx, _, margin = oracle.router_topk(r[b], cfg["top_k"])
            g_sel = [int(e) for e in gidx[l, b]]
            if margin >= MARGIN:
                assert sorted(g_sel) == sorted(int(e) for e in idx), (l, b, margin, g_sel, idx)
            else:
                ties += 1
            _, w_forced, _ = oracle.router_topk(r[b], cfg["top_k"], forced=g_sel)
            assert np.abs(w_forced - gw[l, b]).max() < 1e-3, (l, b, w_forced, gw[l, b])
    return ties


def check_step(cfg, mk, W, seq, pt, kv_before, tokens_np, logits_gpu, k_after=None, v_after=None):
    """Compare one GPU step with the oracle.  Returns a dict of measured errors.

    Routing is validated teacher-forced (above); the numerics are then compared with
    the oracle run free on its own residual stream but taking the GPU's (validated)
    expert selections, so that a near-tie decided the other way does not turn into a
    different model."""
    HW = synth.HostWeights(W)
    HK = synth.HostKV(*kv_before)
    B = len(seq)
    hid = mk.hidden()
    gidx, gw = mk.routes()
    out = dict(near_ties=check_routing_teacher_forced(cfg, HW, hid, gidx, gw, B))
    forced = {(l, b): [int(e) for e in gidx[l, b]]
              for l in range(cfg["n_layers"]) for b in range(B)
              if l not in tuple(cfg.get("dense_layers", ()))}
    ref = oracle.decode_step(cfg, HW, HK, tokens_np, seq, pt, forced=forced)
    # active-expert bookkeeping: slot order = ascending expert id, token lists by (b, j)
    act = mk.active()
    for l, info in enumerate(ref["layers"]):
        want = [(e, sorted(info["experts"][e])) for e in sorted(info["experts"])]
        assert act[l] == want, (l, act[l], want)
    # hidden states
    errs = [rel_l2(hid[i], ref["hidden"][i]) for i in range(cfg["n_layers"] + 1)]
    out["hidden_rel_l2_max"] = max(errs)
    assert max(errs) <= REL_L2, errs
    # logits
    lg = logits_gpu.detach().float().cpu().numpy()
    dmax = float(np.abs(lg - ref["logits"]).max())
    out["logits_max_abs"] = dmax
    assert dmax <= LOGIT_ABS, dmax
    for b in range(len(seq)):
        srt = np.sort(ref["logits"][b])[::-1]
        if srt[0] - srt[1] >= 2 * dmax:
            assert int(np.argmax(lg[b])) == int(ref["greedy"][b])
    # K/V writes: bit-exact location, values within bf16 rounding of the oracle's
    if k_after is not None:
        kb, vb = kv_before
        written = set()
        for l, info in enumerate(ref["layers"]):
            for rec in info["kv"]:
                page, slot, b = rec["page"], rec["slot"], rec["b"]
                written.add((l, page, slot))
                gk = k_after[l, page, :, slot].float().cpu().numpy()
                gv = v_after[l, page, :, slot].float().cpu().numpy()
                ok = oracle.bf16_to_f64(rec["k"])
                ov = oracle.bf16_to_f64(rec["v"])
                assert rel_l2(gk, ok) < REL_L2 and rel_l2(gv, ov) < REL_L2, (l, b)
        mask = torch.ones(kb.shape[:2] + (kb.shape[3],), dtype=torch.bool)
        for (l, page, slot) in written:
            mask[l, page, slot] = False
        mask = mask.to(kb.device)
        kb_m = kb.permute(0, 1, 3, 2, 4)[mask]
        ka_m = k_after.permute(0, 1, 3, 2, 4)[mask]
        assert torch.equal(kb_m.view(torch.int16), ka_m.view(torch.int16))
        assert torch.equal(kv_before[1].permute(0, 1, 3, 2, 4)[mask].view(torch.int16),
                           v_after.permute(0, 1, 3, 2, 4)[mask].view(torch.int16))
    return out


def check_layer_teacher_forced(cfg, HW, HK, hid, gidx, gw, act, k, v, seq, pt, l):
    """Layer l checked on the GPU's own input x_l: routing (where the oracle's top-k
    margin >= MARGIN; the oracle then takes the GPU's selection), the layer output
    x_{l+1}, the active-expert bookkeeping and the K/V written at the layer."""
    x = hid[l].astype(np.float64)
    Bn = len(seq)
    # routing on the GPU's own layer input
    h = oracle.rms_norm(x, oracle.bf16_to_f64(HW.attn_norm(l)), cfg["rms_eps"])
    r = h @ oracle.bf16_to_f64(HW.router(l)).T
    forced = {}
    for b in range(Bn):
        idx, _, margin = oracle.router_topk(r[b], cfg["top_k"])
        g_sel = [int(e) for e in gidx[l, b]]
        if margin >= MARGIN:
            assert sorted(g_sel) == sorted(int(e) for e in idx), (l, b, margin)
        _, w_forced, _ = oracle.router_topk(r[b], cfg["top_k"], forced=g_sel)
        assert np.abs(w_forced - gw[l, b]).max() < 1e-3, (l, b)
        forced[b] = g_sel
    x_next, info = oracle.layer_step(cfg, HW, HK, l, x, seq, pt, forced=forced)
    err = rel_l2(hid[l + 1], x_next)
    assert err <= REL_L2, (l, err)
    want = []
    per = {}
    for b in range(Bn):
        for j, e in enumerate(info["idx"][b]):
            per.setdefault(int(e), []).append((b, j))
    want = [(e, sorted(per[e])) for e in sorted(per)]
    assert act[l] == want, (l, act[l], want)
    for rec in info["kv"]:
        gk = k[l, rec["page"], :, rec["slot"]].float().cpu().numpy()
        gv = v[l, rec["page"], :, rec["slot"]].float().cpu().numpy()
        assert rel_l2(gk, oracle.bf16_to_f64(rec["k"])) < REL_L2, (l, rec["b"])
        assert rel_l2(gv, oracle.bf16_to_f64(rec["v"])) < REL_L2, (l, rec["b"])
    return err


def expected_split_count(cfg, l, pos, split_pages):
    """Attention splits of a sequence at layer l: the oracle's attended cached keys
    [window_start, pos) cut into pages of 16 and groups of split_pages pages."""
    window = cfg["sliding_window"] if l in tuple(cfg.get("swa_layers", ())) else 0
    lo = oracle.window_start(pos, window)
    if pos <= lo:
        return 0
    npg = (pos - 1) // oracle.PAGE - lo // oracle.PAGE + 1
    return -(-npg // split_pages)


def check_bookkeeping(mk, cfg, seq, megakernel=True):
    """The schedule's bookkeeping after an inspected step, bit-exact:
      * every counter's final value equals what the step must leave there -- each
        descriptor's wait and signal targets (as planned), the per-(layer, sequence, KV
        group) attention split counts + 1 from the oracle's attended ranges and the
        GPU's split size, one route step per routed layer, the grid;
      * every queue drained: head = items + one failing claim per SM, and the expert
        queue's count = the routed experts' items (from the active lists).  The O-proj
        queue serves the megakernel's MoE drains only (megakernel=False: the per-op
        launches deal the O-proj tiles as a wave of their own)."""
    from persistent_moe_decode_cta_gb300 import binding as Bd
    T = mk.tasks()
    fin = mk.final_counters().astype(np.int64)
    heads, counts = mk.final_queues()
    n_sm = mk.query(Bd.MK_Q_NUM_SMS)
    Bn, L, Hkv = len(seq), cfg["n_layers"], cfg["n_kv_heads"]
    # (on the handle's SM count: the QKV tiling follows the SMs free of router tiles)
    _, _, _, I = Bd.mk_plan_dry(cfg, Bn, n_sm, max_batch=mk.max_batch)
    maxa, t_moe, qkv_tpg, n_router = int(I[3]), int(I[5]), int(I[10]), int(I[11])
    c_lr, c_qkvg, c_rt, c_rr, c_att, c_og, c_md, c_od = (int(x) for x in I[16:24])
    od_target, c_done, c_oa, t_dense, nrb_d = int(I[12]), int(I[13]), int(I[26]), int(I[27]), int(I[24])
    dense = set(cfg.get("dense_layers", ()))
    sp = mk.query(Bd.MK_Q_SPLIT_PAGES)
    # 1. every descriptor's waits and signals end exactly at their planned targets
    for t in T:
        for c, tg in ((t[7], t[8]), (t[17], t[18]), (t[9], t[10])):
            if c >= 0:
                assert fin[c] == tg, (list(t[:3]), int(c), int(fin[c]), int(tg))
    # 2. every counter, including those no descriptor names
    want = np.zeros_like(fin)
    want[c_lr:c_lr + L + 1] = nrb_d
    want[c_qkvg:c_qkvg + L * Hkv] = qkv_tpg
    want[c_og:c_og + L * Hkv] = Bn
    want[c_od:c_od + L] = od_target
    want[c_oa:c_oa + L] = Hkv * Bn
    want[c_done] = n_sm
    splits = np.zeros((L, Bn), dtype=np.int64)
    for l in range(L):
        routed = l not in dense
        want[c_rt + l] = n_router if routed else 0
        want[c_rr + l] = 1 if routed else 0
        want[c_md + l] = maxa * t_moe if routed else t_dense
        for b in range(Bn):
            splits[l, b] = expected_split_count(cfg, l, seq[b], sp)
            for g in range(Hkv):
                want[c_att + (l * Bn + b) * Hkv + g] = splits[l, b] + 1
    bad = np.flatnonzero(fin != want)
    assert bad.size == 0, [(int(i), int(fin[i]), int(want[i])) for i in bad[:10]]
    # 3. queues drained, each item claimed once
    act = mk.active()
    oq = {int(t[1]) for t in T if t[0] == 5 and t[6] > 0} if megakernel else set()
    for l in range(L):
        assert heads[l] == Hkv * int((splits[l] + 1).sum()) + n_sm, (l, heads[l])
        items = t_dense if l in dense else len(act[l]) * t_moe
        assert heads[L + l] == items + n_sm, (l, heads[L + l], items)
        assert counts[L + l] == (0 if l in dense else items), (l, counts[L + l])
        assert heads[2 * L + l] == (od_target + n_sm if l in oq else 0), (l, heads[2 * L + l])
    return dict(splits=splits)
