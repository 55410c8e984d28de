"""The tensor-core build (MK_LM_UMMA=1 at mk_create, and MK_MOE_UMMA=1 beside it): the
LM head's 64-row tiles and, with the second, the bf16 expert / dense-FFN items (32-row
f-slices), their weight chunks in shared memory in the K-major core-matrix layout, the
tokens' operands staged beside them, tcgen05.mma (M = 128) into f32 accumulators in
tensor memory, read back with tcgen05.ld (FP8 expert items stay on mma.sync).  Through
the C ABI against the oracle: whole steps (batch 1 and ragged batch 8, megakernel /
per-op / graph, MoE and dense FFN layers), greedy multi-step launches, and the
pages-scale LM head on the GPU's own final hidden state."""
import numpy as np
import pytest
import torch

import oracle
import synth
from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu

OP_LMHEAD = 8


@pytest.fixture(autouse=True, params=["lm", "lm+ffn"])
def umma(request, monkeypatch):
    monkeypatch.setenv("MK_LM_UMMA", "1")
    monkeypatch.setenv("MK_MOE_UMMA", "1" if request.param == "lm+ffn" else "0")
    return request.param


@pytest.mark.parametrize("workload,lens,mode", [
    ("tiny_b1_64", [64], "mega"),
    ("tiny_b1_64", [64, 1, 0, 17, 33, 200, 15, 16], "mega"),
    ("small_b1_2k", [2048], "mega"),
    ("small_b1_2k", [2048, 5, 700, 1500, 33, 1024, 64, 300], "mega"),
    ("small_b1_2k", [2048, 37], "perop"),
    ("small_b1_2k", [2048, 37], "graph"),
    ("small_fp8_b1_2k", [2048, 9, 300], "mega"),
    ("small_dense_b1_2k", [2048, 9, 300, 1024], "mega"),
    ("tiny_dense_b1_64", [64, 3], "graph"),
])
def test_tensor_core_lm_head_matches_oracle(workload, lens, mode, umma):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seq_lens=lens)
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        # the FFN items move to the tensor cores only where they are bf16
        ffn = umma == "lm+ffn" and cfg.get("expert_dtype", "bf16") == "bf16"
        assert mk.query(B.MK_Q_TENSOR_CORES) == (3 if ffn else 1)
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
        T = mk.tasks()
        lm = T[T[:, 0] == OP_LMHEAD]
        assert len(lm) and (lm[:, 4] == 64).all()
        kv0 = (k.clone(), v.clone())
        logits = torch.full((len(seq), cfg["vocab"]), float("nan"), device="cuda")
        if mode == "mega":
            mk.step(tokens, k, v, logits)
        else:
            mk.step_perop(tokens, k, v, logits, use_graph=(mode == "graph"))
        assert mk.status()["code"] == 0, mk.status()
        PU.check_step(cfg, mk, W, seq, pt, kv0, tokens.cpu().numpy(), logits, k, v)
    finally:
        mk.close()


def test_tensor_core_lm_head_greedy_multistep():
    """Four greedy steps in one launch equal four single steps with the greedy token fed
    back on the host (the argmax keys come out of the tensor-memory epilogue)."""
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup("tiny_b1_64", seq_lens=[40, 7, 0], steps=4)
    pt_dev = torch.as_tensor(pt, device="cuda")
    a = B.Megakernel(cfg, W)
    b = B.Megakernel(cfg, W)
    try:
        a.plan(seq, pt_dev, npages)
        b.plan(seq, pt_dev, npages)
        ka, va, kb, vb = k.clone(), v.clone(), k.clone(), v.clone()
        la = torch.empty(len(seq), cfg["vocab"], device="cuda")
        toks = torch.empty(4, len(seq), dtype=torch.int32, device="cuda")
        a.steps(tokens, 4, ka, va, la, toks)
        assert a.status()["code"] == 0
        t = tokens.clone()
        lb = torch.empty_like(la)
        for s in range(4):
            b.step(t, kb, vb, lb)
            t = lb.argmax(dim=1).to(torch.int32)
            assert torch.equal(t, toks[s]), (s, t, toks[s])
    finally:
        a.close()
        b.close()


def test_tensor_core_lm_head_pages_scale():
    """The pages-scale LM head (151936 x 2048, 2374 tiles) on the GPU's own final hidden
    state, batch 1 at 8K and batch 8 ragged, in the benchmark's launch configuration."""
    for wl in ("pages_l1_b1_8k", "pages_l2_b8_ragged_swa"):
        cfg = synth.model_config(wl)
        W = synth.make_weights(cfg, seed=0, device="cuda")
        seq = synth.seq_lens_for(wl, 0)
        pt, npages = synth.make_page_table(seq, seed=0)
        k, v = synth.make_kv(cfg, npages, seed=0, device="cuda")
        tokens = synth.make_tokens(len(seq), cfg["vocab"], seed=0, device="cuda")
        mk = B.Megakernel(cfg, W, max_batch=8)
        try:
            mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
            logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
            mk.step(tokens, k, v, logits)
            assert mk.status()["code"] == 0
            HW = synth.HostWeights(W)
            hid = mk.hidden()
            ref = oracle.lm_head(cfg, HW, hid[cfg["n_layers"]].astype(np.float64))
            lg = logits.cpu().numpy()
            dmax = float(np.abs(lg - ref).max())
            assert dmax <= PU.LOGIT_ABS, dmax
            for b in range(len(seq)):
                srt = np.sort(ref[b])[::-1]
                if srt[0] - srt[1] >= 2 * dmax:
                    assert int(np.argmax(lg[b])) == int(np.argmax(ref[b]))
        finally:
            mk.close()
            del W, k, v
            torch.cuda.empty_cache()
