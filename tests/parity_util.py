"""Shared helpers for the GPU-vs-oracle parity tests.

Acceptance (from the decode-step contract):
  * bookkeeping bit-exact: written K/V page/slot, untouched cache bytes unchanged,
    active-expert sets and per-expert token lists, counters back at zero;
  * expert selection identical wherever the oracle's top-k margin >= 1e-3 (below
    that either set is correct: the oracle is re-run with the GPU's choice forced);
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


def setup(workload, seed=0, steps=1, gain_jitter=0.1, device="cuda", seq_lens=None, batch=None):
    cfg = synth.model_config(workload)
    W = synth.make_weights(cfg, seed=seed, device=device, gain_jitter=gain_jitter)
    seq = list(seq_lens) if seq_lens is not None else synth.seq_lens_for(workload, seed)
    if batch is not None:
        seq = (seq * batch)[:batch]
    pt, npages = synth.make_page_table(seq, steps=steps, seed=seed)
    k, v = synth.make_kv(cfg, npages, seed=seed, device=device)
    tokens = synth.make_tokens(len(seq), cfg["vocab"], seed=seed, device=device)
    return cfg, W, seq, pt, npages, k, v, tokens


def gpu_forced_routes(cfg, ref, gpu_idx):
    """(l, b) -> GPU selection wherever the sets differ; asserts each such place is
    a near-tie of the oracle (margin < MARGIN)."""
    forced = {}
    for l, info in enumerate(ref["layers"]):
        for b in range(gpu_idx.shape[1]):
            o_set = set(int(e) for e in info["idx"][b])
            g_set = set(int(e) for e in gpu_idx[l, b])
            if o_set != g_set:
                assert info["margin"][b] < MARGIN, (
                    f"layer {l} seq {b}: expert sets differ with margin {info['margin'][b]}")
                forced[(l, b)] = [int(e) for e in gpu_idx[l, b]]
    return forced


def check_step(cfg, mk, W, seq, pt, kv_before, tokens_np, logits_gpu, k_after=None, v_after=None):
    """Compare one GPU step with the oracle.  Returns a dict of measured errors."""
    HW = synth.HostWeights(W)
    HK = synth.HostKV(*kv_before)
    ref = oracle.decode_step(cfg, HW, HK, tokens_np, seq, pt)
    gidx, gw = mk.routes()
    forced = gpu_forced_routes(cfg, ref, gidx)
    if forced:
        ref = oracle.decode_step(cfg, HW, HK, tokens_np, seq, pt, forced=forced)
    out = dict(forced=len(forced))
    # routing: identical sets everywhere now (forced where near-tied); weights close
    for l, info in enumerate(ref["layers"]):
        for b in range(len(seq)):
            assert sorted(int(e) for e in info["idx"][b]) == sorted(int(e) for e in gidx[l, b])
            og = dict(zip((int(e) for e in info["idx"][b]), info["w"][b]))
            for e, wv in zip(gidx[l, b], gw[l, b]):
                assert abs(og[int(e)] - wv) < 2e-2, (l, b, e, og[int(e)], wv)
    # active-expert bookkeeping: slot order = ascending expert id, token lists by (b, j)
    act = mk.active()
    for l, info in enumerate(ref["layers"]):
        want = []
        for e in sorted(info["experts"]):
            want.append((e, sorted(info["experts"][e])))
        got = [(e, lst) for e, lst in act[l]]
        # the GPU's slot j for token b is its own selection order; compare (b) and expert
        assert [e for e, _ in got] == [e for e, _ in want], (l, got, want)
        for (e, gl), (_, wl) in zip(got, want):
            assert [b for b, _ in gl] == [b for b, _ in wl]
            for b, j in gl:
                assert int(gidx[l, b, j]) == e
    # hidden states
    hid = mk.hidden()
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
        vb_m = kb_m = None
        assert torch.equal(kv_before[1].permute(0, 1, 3, 2, 4)[mask].view(torch.int16),
                           v_after.permute(0, 1, 3, 2, 4)[mask].view(torch.int16))
    return out
