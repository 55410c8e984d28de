"""The allocation-free step (mk_decode_step_noalloc) for callers that cannot call
cudaMalloc while decoding: called through the C ABI twice in a row after one
mk_decode_step on the same plan, each of the three steps is checked against the oracle
in the same way (whole steps on the tiny models; sampled layers teacher-forced and the
LM head at the pages scale) -- not against each other: the MoE combine adds fp32
partials atomically, so two runs may differ in the last bits and, at a router near-tie,
in the experts chosen.  A plan whose step scratch does not fit the static buffer is
refused before anything runs.  This file is collected last so that a run that stops at
the first failure has already run every other test; it passes alone in a fresh process
as well as after the others."""
import numpy as np
import pytest
import torch

import oracle
import synth
from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


def _allocating_then_noalloc(mk, cfg, seq, tokens, k, v, check):
    """One allocating step, then two allocation-free steps on the same plan at the same
    position, each checked against the oracle by check(logits, kv_before) through the
    handle's reads (which follow the last step, wherever its buffers were)."""
    mk.set_fixed(True)          # every step then writes the same K/V slot
    kv0 = (k.clone(), v.clone())
    ref = torch.empty(len(seq), cfg["vocab"], device="cuda")
    mk.step(tokens, k, v, ref)
    assert mk.status()["code"] == 0
    check(ref, kv0)
    for _ in range(2):
        out = torch.full((len(seq), cfg["vocab"]), float("nan"), device="cuda")
        B.mk_decode_step_noalloc(mk.h, tokens, k, v, out)
        assert mk.status()["code"] == 0
        check(out, kv0)
    assert list(mk.seq_lens()) == list(seq)


@pytest.mark.parametrize("workload,lens", [("tiny_b1_64", [64, 3]),
                                           ("tiny_b1_64", [64, 1, 0, 17, 33, 40, 15, 16]),
                                           ("tiny_dense_fp8_b1_64", [64, 9, 30])])
def test_noalloc_step_matches_the_allocating_step(workload, lens):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seq_lens=lens)
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)

        def check(logits, kv0):   # the whole step against the oracle
            PU.check_step(cfg, mk, W, seq, pt, kv0, tokens.cpu().numpy(), logits, k, v)
        _allocating_then_noalloc(mk, cfg, seq, tokens, k, v, check)
    finally:
        mk.close()


def test_noalloc_refuses_a_plan_beyond_the_static_buffer():
    """64 layers x 8 KV groups of 8 query heads at batch 8 with up to 1024 pages a
    sequence: the attention partials alone need ~147 MB, more than the 64 MiB buffer.
    The call fails with MK_ERR_UNSUPPORTED and the size needed, before any launch; the
    allocating step runs the same plan."""
    cfg = dict(n_layers=64, d_model=256, n_q_heads=64, n_kv_heads=8, head_dim=32, n_experts=8,
               top_k=2, d_ff=128, vocab=64, rope_theta=1e4, rms_eps=1e-6, sliding_window=0,
               swa_layers=(), page_size=16)
    W = synth.make_weights(cfg, seed=0, device="cuda")
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        pt = torch.full((8, 1024), -1, dtype=torch.int32, device="cuda")
        pt[:, 0] = torch.arange(8, dtype=torch.int32, device="cuda")
        mk.plan([5] * 8, pt, 8)
        k, v = synth.make_kv(cfg, 8, seed=0, device="cuda")
        tokens = synth.make_tokens(8, cfg["vocab"], device="cuda")
        out = torch.empty(8, cfg["vocab"], device="cuda")
        with pytest.raises(B.MkError) as ei:
            B.mk_decode_step_noalloc(mk.h, tokens, k, v, out)
        assert ei.value.code == B.MK_ERR_UNSUPPORTED
        msg = str(ei.value)
        need = int(msg.split("needs ")[1].split(" bytes")[0])
        assert need > 64 << 20 and str(64 << 20) in msg
        mk.step(tokens, k, v, out)
        assert mk.status()["code"] == 0 and torch.isfinite(out).all()
    finally:
        mk.close()


def test_noalloc_pages_scale_b1_8k():
    """The pages-scale batch-1 8K step (~21 MiB of step scratch): the allocating step
    against the oracle on layers 0 and 47 (teacher-forced) and the LM head, then the
    allocation-free step twice against it."""
    wl = "pages_b1_8k"
    cfg = synth.model_config(wl)
    W = synth.make_weights(cfg, seed=0, device="cuda")
    seq = synth.seq_lens_for(wl, 0)
    pt, npages = synth.make_page_table(seq, seed=0)
    k, v = synth.make_kv(cfg, npages, seed=0, device="cuda")
    tokens = synth.make_tokens(len(seq), cfg["vocab"], seed=0, device="cuda")
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
        HW = synth.HostWeights(W)

        def check(logits, kv0):   # sampled layers teacher-forced, and the LM head
            hid = mk.hidden()
            gidx, gw = mk.routes()
            act = mk.active()
            HK = synth.HostKV(*kv0)
            for l in (0, 23, 47):
                PU.check_layer_teacher_forced(cfg, HW, HK, hid, gidx, gw, act, k, v, seq, pt, l)
                HW.drop_cache()
            ref = oracle.lm_head(cfg, HW, hid[cfg["n_layers"]].astype(np.float64))
            lg = logits.cpu().numpy()
            dmax = float(np.abs(lg - ref).max())
            assert dmax <= PU.LOGIT_ABS, dmax
            srt = np.sort(ref[0])[::-1]
            if srt[0] - srt[1] >= 2 * dmax:
                assert int(np.argmax(lg[0])) == int(np.argmax(ref[0]))
            HW.drop_cache()
        _allocating_then_noalloc(mk, cfg, seq, tokens, k, v, check)
    finally:
        mk.close()
        del W, k, v
        torch.cuda.empty_cache()
