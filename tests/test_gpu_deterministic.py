"""Deterministic steps (mk_set_deterministic): the layer accumulators hold 64-bit
fixed-point sums, so that the order in which expert items and O-proj tiles finish does
not reach the results.  Through the C ABI, each case checks a step against the oracle
and then repeats the step at the same position: hidden states, routing, K/V and logits
must be bit-identical between the runs.  The default (float) mode is not expected to
repeat bit for bit; it is covered by the other parity tests."""
import numpy as np
import pytest
import torch

import synth
from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


def _run_twice(workload, lens, max_batch=8):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seq_lens=lens)
    mk = B.Megakernel(cfg, W, max_batch=max_batch)
    try:
        mk.set_deterministic(True)
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
        mk.set_fixed(True)  # both steps write the same K/V slot
        kv0 = (k.clone(), v.clone())
        runs = []
        for _ in range(2):
            k.copy_(kv0[0])
            v.copy_(kv0[1])
            logits = torch.full((len(seq), cfg["vocab"]), float("nan"), device="cuda")
            mk.step(tokens, k, v, logits)
            assert mk.status()["code"] == 0, mk.status()
            idx, w = mk.routes()
            runs.append(dict(logits=logits.cpu().numpy(), hidden=mk.hidden(), idx=idx, w=w,
                             act=mk.active(), k=k.cpu(), v=v.cpu()))
        # the first run against the oracle
        k.copy_(runs[0]["k"].cuda())
        v.copy_(runs[0]["v"].cuda())
        PU.check_step(cfg, mk, W, seq, pt, kv0, tokens.cpu().numpy(), torch.as_tensor(runs[0]["logits"]).cuda(),
                      k, v)
        a, b = runs
        assert np.array_equal(a["logits"], b["logits"])
        assert np.array_equal(a["hidden"], b["hidden"])
        assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(a["w"], b["w"])
        assert a["act"] == b["act"]
        assert torch.equal(a["k"], b["k"]) and torch.equal(a["v"], b["v"])
    finally:
        mk.close()


@pytest.mark.parametrize("workload,lens", [
    ("small_b1_2k", [2048]),
    ("small_b1_2k", [2048, 5, 700, 1500, 33, 1024, 64, 300]),
    ("tiny_b1_64", [64, 1, 0, 17, 33, 40, 15, 16]),
])
def test_deterministic_steps_repeat_bit_for_bit(workload, lens):
    _run_twice(workload, lens)


def test_deterministic_fp8_mixed_stack_repeats_bit_for_bit():
    _run_twice("small_dense_fp8_b1_2k", [2048, 9, 300], max_batch=3)


def test_deterministic_mode_takes_effect_at_the_next_plan():
    """Switching the mode re-sizes the accumulators at the next plan: both modes then
    step correctly on the same handle."""
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup("tiny_b1_64", seq_lens=[64, 7])
    mk = B.Megakernel(cfg, W)
    try:
        pt_dev = torch.as_tensor(pt, device="cuda")
        for det in (True, False, True):
            mk.set_deterministic(det)
            mk.plan(seq, pt_dev, npages)
            mk.set_fixed(True)
            kv0 = (k.clone(), v.clone())
            logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
            mk.step(tokens, k, v, logits)
            assert mk.status()["code"] == 0
            PU.check_step(cfg, mk, W, seq, pt, kv0, tokens.cpu().numpy(), logits, k, v)
            k.copy_(kv0[0])
            v.copy_(kv0[1])
    finally:
        mk.close()
