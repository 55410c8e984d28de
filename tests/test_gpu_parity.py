"""GPU parity: the megakernel (through the C ABI) against the CPU oracle on the
same seeded inputs."""
import numpy as np
import pytest
import torch

import synth
from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


def _run(workload, seed=0, seq_lens=None, batch=None, mode="mega", steps=1):
    cfg, W, seq, pt, npages, k, v, tokens = PU.setup(workload, seed=seed, seq_lens=seq_lens,
                                                      batch=batch, steps=steps)
    kb, vb = k.clone(), v.clone()
    mk = B.Megakernel(cfg, W, max_batch=max(8, len(seq)))
    pt_dev = torch.as_tensor(pt, device="cuda")
    mk.plan(seq, pt_dev, npages)
    logits = torch.full((len(seq), cfg["vocab"]), float("nan"), device="cuda")
    if mode == "mega":
        mk.step(tokens, k, v, logits)
    else:
        mk.step_perop(tokens, k, v, logits, use_graph=(mode == "graph"))
    st = mk.status()
    assert st["code"] == 0, st
    res = PU.check_step(cfg, mk, W, seq, pt, (kb, vb), tokens.cpu().numpy(), logits, k, v)
    assert np.array_equal(mk.seq_lens(), np.array(seq) + 1)
    assert not mk.counters().any()
    mk.close()
    return res


def test_tiny_megakernel_matches_oracle():
    _run("tiny_b1_64")


def test_tiny_perop_and_graph_match_oracle():
    _run("tiny_b1_64", mode="perop")
    _run("tiny_b1_64", mode="graph")


def test_tiny_batch8_ragged_matches_oracle():
    _run("tiny_b1_64", seq_lens=[64, 1, 0, 17, 33, 200, 15, 16])


def test_small_b1_matches_oracle():
    _run("small_b1_2k")
