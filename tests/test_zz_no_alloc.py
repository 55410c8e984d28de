"""The allocation-free step (mk_decode_step_noalloc) for callers that cannot call
cudaMalloc while decoding: called through the C ABI twice in a row, it must give the
same logits and the same K/V writes as mk_decode_step, within the logit tolerance of
the parity tests (the MoE combine adds fp32 partials atomically, so the order of the
additions, and with it a router near-tie, may differ between calls).  This file is collected last so that a run that
stops at the first failure has already run every other test; it passes alone in a
fresh process as well as after the others."""
import numpy as np
import pytest
import torch

from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("workload,lens", [("tiny_b1_64", [64, 3]),
                                           ("tiny_b1_64", [64, 1, 0, 17, 33, 40, 15, 16])])
def test_noalloc_step_matches_the_allocating_step(workload, lens):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seq_lens=lens)
    mk = B.Megakernel(cfg, W, max_batch=8)
    mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
    mk.set_fixed(True)          # both entry points then write the same K/V slot
    ref = torch.empty(len(seq), cfg["vocab"], device="cuda")
    mk.step(tokens, k, v, ref)
    assert mk.status()["code"] == 0
    k_ref, v_ref = k.clone(), v.clone()
    for _ in range(2):
        out = torch.full((len(seq), cfg["vocab"]), float("nan"), device="cuda")
        B.mk_decode_step_noalloc(mk.h, tokens, k, v, out)
        assert mk.status()["code"] == 0
        diff = (out - ref).abs().max().item()
        assert diff <= PU.LOGIT_ABS, diff
        top2 = ref.topk(2, dim=-1).values
        clear = (top2[:, 0] - top2[:, 1]) >= 2 * diff      # not a reported tie
        assert torch.equal(out.argmax(-1)[clear], ref.argmax(-1)[clear])
        dk = (k.float() - k_ref.float()).abs().max().item()
        dv = (v.float() - v_ref.float()).abs().max().item()
        assert dk < 0.05 and dv < 0.05
    assert list(mk.seq_lens()) == seq
    mk.close()
