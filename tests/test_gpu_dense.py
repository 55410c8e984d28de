"""Mixed dense/MoE stacks: a dense layer (dense_layer_mask) runs one SwiGLU FFN of
width dense_ff for every token in place of the routed experts, with no router.  The
GPU step must match the oracle (routing checked teacher-forced on the routed layers
only), through the megakernel and the per-op path, at several batch sizes."""
import numpy as np
import pytest
import torch

from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("workload,seq_lens,mode", [
    ("tiny_dense_b1_64", [64], "mega"),
    ("tiny_dense_b1_64", [61, 0, 17], "mega"),
    ("tiny_dense_b1_64", [61, 0, 17], "perop"),
    ("small_dense_b1_2k", [2048, 300], "mega"),
    ("small_dense_b1_2k", [2048, 300], "graph"),
])
def test_mixed_stack_step_matches_oracle(workload, seq_lens, mode):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seq_lens=seq_lens)
    assert cfg["dense_layers"]
    mk = B.Megakernel(cfg, W, max_batch=8)
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
        # the dense layers publish no active experts
        act = mk.active()
        for l in cfg["dense_layers"]:
            assert act[l] == []
    finally:
        mk.close()


def test_mixed_stack_multi_step_equals_single_steps():
    n = 4
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup("tiny_dense_b1_64", seq_lens=[62, 9], steps=n)
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
        # the same greedy tokens; cache and logits agree within the parity tolerance (the
        # order of the fp32 atomic adds into the layer accumulator is not fixed)
        assert np.array_equal(out.cpu().numpy(), np.stack(host))
        assert PU.rel_l2(k.float().cpu().numpy(), k1.float().cpu().numpy()) < PU.REL_L2
        assert PU.rel_l2(v.float().cpu().numpy(), v1.float().cpu().numpy()) < PU.REL_L2
        assert float((lg1 - lg2).abs().max()) <= PU.LOGIT_ABS
    finally:
        mk.close()
