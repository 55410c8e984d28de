"""Multi-step decode (mk_decode_steps): N greedy steps in one launch, each step's
token fed to the next on the device.  On the tiny model it must equal N single steps
with the greedy token fed back on the host -- the same tokens and seq_lens, the K/V
cache and the last step's logits within the parity tolerance (the order of the fp32
atomic adds into the layer accumulator is not fixed, so the last bits may differ
between any two runs) -- and the last step of a multi-step launch must match the
oracle (routing teacher-forced, as in the single-step parity tests); the single steps
themselves are pinned to the oracle there."""
import numpy as np
import pytest
import torch

import oracle
import synth
from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


def test_steps_in_one_launch_equal_single_steps_with_host_feedback():
    n = 5  # position 61 -> 65 crosses a page boundary
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup("tiny_b1_64", seq_lens=[61, 14], steps=n)
    pt_dev = torch.as_tensor(pt, device="cuda")
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        k1, v1 = k.clone(), v.clone()
        mk.plan(seq, pt_dev, npages)
        lg1 = torch.empty(len(seq), cfg["vocab"], device="cuda")
        t = tokens.clone()
        host_tokens = []
        for _ in range(n):
            mk.step(t, k1, v1, lg1)
            assert mk.status()["code"] == 0
            t = lg1.argmax(-1).to(torch.int32)
            host_tokens.append(t.cpu().numpy())
        k2, v2 = k.clone(), v.clone()
        mk.plan(seq, pt_dev, npages)
        lg2 = torch.empty_like(lg1)
        out = mk.steps(tokens, n, k2, v2, lg2)
        assert mk.status()["code"] == 0
        assert np.array_equal(out.cpu().numpy(), np.stack(host_tokens))
        assert list(mk.seq_lens()) == [s + n for s in seq]
        assert PU.rel_l2(k2.float().cpu().numpy(), k1.float().cpu().numpy()) < PU.REL_L2
        assert PU.rel_l2(v2.float().cpu().numpy(), v1.float().cpu().numpy()) < PU.REL_L2
        assert float((lg1 - lg2).abs().max()) <= PU.LOGIT_ABS
        # the launch can be repeated: counters, queues and the argmax keys are reset
        out2 = mk.steps(out[-1].clone(), 2, k2, v2, lg2)
        assert mk.status()["code"] == 0
        assert list(mk.seq_lens()) == [s + n + 2 for s in seq]
        assert int(out2[1, 0]) == int(lg2[0].argmax())
    finally:
        mk.close()


@pytest.mark.parametrize("workload,seq_lens", [("tiny_b1_64", [40, 7, 63]), ("small_b1_2k", [700, 31])])
def test_last_step_of_a_launch_matches_oracle(workload, seq_lens):
    n = 3
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seq_lens=seq_lens, steps=n)
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
        logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
        out = mk.steps(tokens, n, k, v, logits)
        assert mk.status()["code"] == 0
        assert list(mk.seq_lens()) == [s + n for s in seq]
        toks = out.cpu().numpy()
        # every step's token is the greedy token of that step; the last one of the
        # logits the launch returns (lowest index on ties)
        lg = logits.float().cpu().numpy()
        assert np.array_equal(toks[-1], np.argmax(lg, axis=-1))
        # the last step against the oracle, on the cache the earlier steps wrote (the
        # oracle computes the new token's K/V itself and reads the earlier positions)
        last_seq = [s + n - 1 for s in seq]
        res = PU.check_step(cfg, mk, W, last_seq, pt, (k, v), toks[-2], logits)
        assert res["logits_max_abs"] <= PU.LOGIT_ABS
        # the K/V the last step wrote, against the oracle's
        HW, HK = synth.HostWeights(W), synth.HostKV(k, v)
        gidx = mk.routes()[0]
        forced = {(l, b): [int(e) for e in gidx[l, b]] for l in range(cfg["n_layers"]) for b in range(len(seq))}
        ref = oracle.decode_step(cfg, HW, HK, toks[-2], last_seq, pt, forced=forced)
        for l, info in enumerate(ref["layers"]):
            for rec in info["kv"]:
                gk = k[l, rec["page"], :, rec["slot"]].float().cpu().numpy()
                gv = v[l, rec["page"], :, rec["slot"]].float().cpu().numpy()
                assert PU.rel_l2(gk, oracle.bf16_to_f64(rec["k"])) < PU.REL_L2
                assert PU.rel_l2(gv, oracle.bf16_to_f64(rec["v"])) < PU.REL_L2
    finally:
        mk.close()


def test_steps_argument_errors():
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup("tiny_b1_64", seq_lens=[8])
    mk = B.Megakernel(cfg, W)
    try:
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
        logits = torch.empty(1, cfg["vocab"], device="cuda")
        out = torch.empty(1, 1, dtype=torch.int32, device="cuda")
        for bad in (0, 4097):
            with pytest.raises(B.MkError):
                B.mk_decode_steps(mk.h, tokens, bad, k, v, logits, out)
    finally:
        mk.close()
