"""FP8 experts (expert_dtype "fp8"): the routed experts' matrices stored as E4M3 codes
with float32 scales, decoded in the kernel.

* The stored codes and scales, read back through mk_read_expert_fp8, are bit-equal to
  the oracle's quantisation of the same bf16 weights (nearest code, ties to even,
  saturating; one scale per row = max|row| / 448 in float32) -- every expert of the tiny model,
  sampled experts of the small and the pages-scale ones.
* A decode step matches the oracle run on the decoded weights (routing teacher-forced,
  the same tolerances as the bf16 path) through the megakernel, the per-op path and
  its CUDA graph, at batch 1 to 8; and at the pages-scale sizes, on sampled layers in
  the launch configuration the benchmark times.
* Several steps in one launch equal the same steps with the greedy token fed back on
  the host.
* With the projections in FP8 as well (expert_dtype MK_WEIGHTS_FP8: QKV, O-proj and
  LM head as E4M3 codes with one float32 scale per output row, read back through
  mk_read_weight_fp8), the same: stored form bit-equal to the oracle's quantisation,
  steps against the oracle on the decoded weights."""
import numpy as np
import pytest
import torch

import oracle
import synth
from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


def _check_stored(mk, HW, l, e):
    got = mk.expert_fp8(l, e)
    wg, wu, wd = HW.expert(l, e)
    for name, w in (("gate", wg), ("up", wu), ("down", wd)):
        codes, scales = oracle.quantize_e4m3_rows(w)
        assert np.array_equal(got[name + "_codes"], codes), (l, e, name)
        assert np.array_equal(got[name + "_scales"].view(np.uint32), scales.view(np.uint32)), (l, e, name)


# max_batch 8: expert items of 64 rows of d_ff; below 4: of 32 rows
@pytest.mark.parametrize("workload,pairs,max_batch", [
    ("tiny_fp8_b1_64", "all", 8),
    ("tiny_fp8_b1_64", "all", 2),
    ("small_fp8_b1_2k", [(0, 0), (3, 17), (7, 31)], 8),
])
def test_stored_codes_and_scales_equal_the_oracle_quantisation(workload, pairs, max_batch):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload)
    mk = B.Megakernel(cfg, W, max_batch=max_batch)
    try:
        HW = synth.HostWeights(W)
        if pairs == "all":
            pairs = [(l, e) for l in range(cfg["n_layers"]) for e in range(cfg["n_experts"])]
        for l, e in pairs:
            _check_stored(mk, HW, l, e)
    finally:
        mk.close()


@pytest.mark.parametrize("workload,seq_lens,mode,max_batch", [
    ("tiny_fp8_b1_64", [64], "mega", 8),
    ("tiny_fp8_b1_64", [61, 0, 17], "mega", 8),
    ("tiny_fp8_b1_64", [61, 0, 17], "perop", 8),
    ("tiny_fp8_b1_64", [61, 17], "mega", 2),
    ("tiny_fp8_b1_64", [64], "perop", 1),
    ("small_fp8_b1_2k", [2048, 300], "mega", 8),
    ("small_fp8_b1_2k", [2048, 300], "graph", 8),
    ("small_fp8_b1_2k", [2048, 300], "mega", 2),
    ("small_fp8_b1_2k", [2048, 5, 900, 17, 64, 1, 333, 2000], "mega", 8),
    # FP8 experts and projections
    ("tiny_fp8w_b1_64", [64], "mega", 8),
    ("tiny_fp8w_b1_64", [61, 0, 17], "mega", 8),
    ("tiny_fp8w_b1_64", [61, 0, 17], "perop", 8),
    ("tiny_fp8w_b1_64", [64], "graph", 1),
    ("small_fp8w_b1_2k", [2048], "mega", 1),
    ("small_fp8w_b1_2k", [2048, 300], "graph", 8),
    ("small_fp8w_b1_2k", [2048, 5, 900, 17, 64, 1, 333, 2000], "mega", 8),
    ("tiny_dense_fp8w_b1_64", [61, 0, 17], "mega", 8),
    # FP8 experts beside bf16 dense layers (a mixed stack)
    ("tiny_dense_fp8_b1_64", [61, 0, 17], "mega", 8),
    ("tiny_dense_fp8_b1_64", [61, 17], "perop", 2),
    ("small_dense_fp8_b1_2k", [2048, 300], "mega", 8),
    ("small_dense_fp8_b1_2k", [2048], "graph", 1),
])
def test_fp8_step_matches_oracle(workload, seq_lens, mode, max_batch):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seq_lens=seq_lens)
    mk = B.Megakernel(cfg, W, max_batch=max_batch)
    try:
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
        kb, vb = k.clone(), v.clone()
        logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
        if mode == "mega":
            mk.step(tokens, k, v, logits)
        else:
            mk.step_perop(tokens, k, v, logits, use_graph=(mode == "graph"))
        assert mk.status()["code"] == 0
        PU.check_step(cfg, mk, W, seq, pt, (kb, vb), tokens.cpu().numpy(), logits, k, v)
    finally:
        mk.close()


@pytest.mark.parametrize("workload", ["tiny_fp8_b1_64", "tiny_fp8w_b1_64"])
def test_fp8_multi_step_equals_single_steps(workload):
    n = 4
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seq_lens=[62, 9, 30], steps=n)
    pt_dev = torch.as_tensor(pt, device="cuda")
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        k1, v1 = k.clone(), v.clone()
        mk.plan(seq, pt_dev, npages)
        lg1 = torch.empty(len(seq), cfg["vocab"], device="cuda")
        t = tokens.clone()
        host = []
        for _ in range(n):
            mk.step(t, k1, v1, lg1)
            assert mk.status()["code"] == 0
            t = lg1.argmax(-1).to(torch.int32)
            host.append(t.cpu().numpy())
        mk.plan(seq, pt_dev, npages)
        lg2 = torch.empty_like(lg1)
        out = mk.steps(tokens, n, k, v, lg2)
        assert mk.status()["code"] == 0
        assert np.array_equal(out.cpu().numpy(), np.stack(host))
        assert PU.rel_l2(k.float().cpu().numpy(), k1.float().cpu().numpy()) < PU.REL_L2
        assert PU.rel_l2(v.float().cpu().numpy(), v1.float().cpu().numpy()) < PU.REL_L2
        assert float((lg1 - lg2).abs().max()) <= PU.LOGIT_ABS
    finally:
        mk.close()


def _check_stored_projections(mk, HW, cfg, layers, lm=True):
    pairs = [(B.MK_W_Q, HW.wq), (B.MK_W_K, HW.wk), (B.MK_W_V, HW.wv), (B.MK_W_O, HW.wo)]
    for l in layers:
        for m, get in pairs:
            codes, scales = mk.weight_fp8(m, l)
            want_c, want_s = oracle.quantize_e4m3_rows(get(l))
            assert np.array_equal(codes, want_c), (m, l)
            assert np.array_equal(scales.view(np.uint32), want_s.view(np.uint32)), (m, l)
    if lm:
        codes, scales = mk.weight_fp8(B.MK_W_LM)
        want_c, want_s = oracle.quantize_e4m3_rows(HW.lm_head())
        assert np.array_equal(codes, want_c) and np.array_equal(scales.view(np.uint32), want_s.view(np.uint32))


@pytest.mark.parametrize("workload,layers,lm", [
    ("tiny_fp8w_b1_64", (0, 1), True),
    ("small_fp8w_b1_2k", (0, 7), True),
])
def test_stored_projection_codes_and_scales_equal_the_oracle_quantisation(workload, layers, lm):
    cfg, W, *_ = PU.setup(workload)
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        HW = synth.HostWeights(W)
        _check_stored_projections(mk, HW, cfg, layers, lm)
        _check_stored(mk, HW, layers[-1], 3)          # the experts as with FP8 experts alone
        with pytest.raises(B.MkError) as e:             # out of range
            mk.weight_fp8(B.MK_W_Q, cfg["n_layers"])
        assert e.value.code == B.MK_ERR_INVALID
    finally:
        mk.close()
    cfg, W, *_ = PU.setup("tiny_fp8_b1_64")            # FP8 experts only: bf16 projections
    mk = B.Megakernel(cfg, W)
    try:
        with pytest.raises(B.MkError) as e:
            mk.weight_fp8(B.MK_W_Q, 0)
        assert e.value.code == B.MK_ERR_STATE
    finally:
        mk.close()


@pytest.mark.parametrize("workload,layers", [
    ("pages_fp8_b1_8k", (0, 24, 47)),
    ("pages_fp8_b8_ragged_swa", (0, 1, 47)),   # 1 and 47 are sliding-window layers
    ("pages_fp8w_b1_8k", (0, 24, 47)),
    ("pages_fp8w_b8_ragged_swa", (0, 1, 47)),
])
def test_fp8_pages_scale_sampled_layers_and_stored_form(workload, layers):
    cfg = synth.model_config(workload)
    W = synth.make_weights(cfg, seed=0, device="cuda")
    seq = synth.seq_lens_for(workload, 0)
    pt, npages = synth.make_page_table(seq, seed=0)
    k, v = synth.make_kv(cfg, npages, seed=0, device="cuda")
    tokens = synth.make_tokens(len(seq), cfg["vocab"], seed=0, device="cuda")
    mk = B.Megakernel(cfg, W, max_batch=len(seq))  # as the benchmark sizes it
    try:
        HW, HK = synth.HostWeights(W), synth.HostKV(k, v)
        for l, e in ((0, 0), (24, 63), (47, 127)):
            _check_stored(mk, HW, l, e)
        if cfg.get("dense_dtype") == "fp8":
            _check_stored_projections(mk, HW, cfg, (0, 47), lm=False)
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
        logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
        mk.step(tokens, k, v, logits)
        assert mk.status()["code"] == 0
        hid = mk.hidden()
        gidx, gw = mk.routes()
        act = mk.active()
        for l in layers:
            PU.check_layer_teacher_forced(cfg, HW, HK, hid, gidx, gw, act, k, v, seq, pt, l)
            HW.drop_cache()
        ref = oracle.lm_head(cfg, HW, hid[cfg["n_layers"]].astype(np.float64))
        dmax = float(np.abs(logits.float().cpu().numpy() - ref).max())
        assert dmax <= PU.LOGIT_ABS, dmax
    finally:
        mk.close()
        del W, k, v
        torch.cuda.empty_cache()


def test_read_expert_fp8_errors():
    cfg, W, *_ = PU.setup("tiny_b1_64")
    mk = B.Megakernel(cfg, W)
    try:  # a bf16 handle has no FP8 form
        with pytest.raises(B.MkError) as e:
            mk.expert_fp8(0, 0)
        assert e.value.code == B.MK_ERR_STATE
    finally:
        mk.close()
    cfg, W, *_ = PU.setup("tiny_fp8_b1_64")
    mk = B.Megakernel(cfg, W)
    try:
        for l, e_ in ((cfg["n_layers"], 0), (0, cfg["n_experts"]), (-1, 0)):
            with pytest.raises(B.MkError) as e:
                mk.expert_fp8(l, e_)
            assert e.value.code == B.MK_ERR_INVALID
        d, f = cfg["d_model"], cfg["d_ff"]
        buf = np.empty(3 * f * d + 4 * (2 * f + d) - 4, dtype=np.uint8)  # one float short
        rc = B.load_library().mk_read_expert_fp8(mk.h, 0, 0, buf.ctypes.data, buf.nbytes)
        assert rc == B.MK_ERR_INVALID
    finally:
        mk.close()
    cfg, W, *_ = PU.setup("tiny_dense_fp8_b1_64")
    mk = B.Megakernel(cfg, W)
    try:  # layer 0 of this mixed stack is dense: no routed experts to read back
        with pytest.raises(B.MkError) as e:
            mk.expert_fp8(0, 0)
        assert e.value.code == B.MK_ERR_INVALID
        _check_stored(mk, synth.HostWeights(W), 1, 3)
    finally:
        mk.close()
