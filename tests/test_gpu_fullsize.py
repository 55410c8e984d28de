"""Parity at the pages-scale sizes, in the launch configuration the benchmark times (one
cooperative megakernel launch per step, 48 layers, d 2048, 128 experts top-8, vocab
151936): the batch-1 8K-context workload, the batch-8 ragged workload with a 4096-
token window on odd layers, and batch 1 at the 128K context.

A full float64 oracle step at this size is chained through 48 layers; instead, sampled
layers are checked teacher-forced -- the oracle runs layer l on the GPU's own input x_l
(its routing checked against the GPU's wherever the top-k margin is >= 1e-3, then
forced to the GPU's selection) and its output must match the GPU's x_{l+1}; the K/V the
GPU wrote at those layers, the active-expert bookkeeping, and the LM head applied to
the GPU's final hidden state are checked the same way.  Chained, these cover every
opcode of the step at the benchmark's sizes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from persistent_moe_decode_cta_gb300 import binding as B

import parity_util as PU

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pages_weights():
    # the benchmark's weights: seed 0, unit gains
    W = synth.make_weights(synth.model_config("pages_b1_8k"), seed=0, device="cuda")
    yield W
    del W
    torch.cuda.empty_cache()


@pytest.mark.parametrize("workload,layers", [
    ("pages_b1_8k", [0, 1, 24, 47]),
    ("pages_b8_ragged_swa", [0, 1, 24, 47]),   # 1 and 47 are sliding-window layers
    ("pages_b1_128k", [0, 47]),                 # the longest context (8192 pages a sequence)
])
def test_pages_scale_step_sampled_layers_and_lm_head(pages_weights, workload, layers):
    W = pages_weights
    cfg = synth.model_config(workload)
    seq = synth.seq_lens_for(workload, 0)
    pt, npages = synth.make_page_table(seq, seed=0)
    k, v = synth.make_kv(cfg, npages, seed=0, device="cuda")
    tokens = synth.make_tokens(len(seq), cfg["vocab"], seed=0, device="cuda")
    mk = B.Megakernel(cfg, W, max_batch=8)
    try:
        mk.plan(seq, torch.as_tensor(pt, device="cuda"), npages)
        mk.inspect(True)
        logits = torch.empty(len(seq), cfg["vocab"], device="cuda")
        mk.step(tokens, k, v, logits)
        assert mk.status()["code"] == 0
        assert list(mk.seq_lens()) == [s + 1 for s in seq]
        PU.check_bookkeeping(mk, cfg, seq)   # counters, split counts and queues, bit-exact
        hid = mk.hidden()
        gidx, gw = mk.routes()
        act = mk.active()
        HW, HK = synth.HostWeights(W), synth.HostKV(k, v)
        for l in layers:
            PU.check_layer_teacher_forced(cfg, HW, HK, hid, gidx, gw, act, k, v, seq, pt, l)
            HW.drop_cache()
        # the LM head on the GPU's final hidden state
        ref = oracle.lm_head(cfg, HW, hid[cfg["n_layers"]].astype(np.float64))
        lg = logits.float().cpu().numpy()
        dmax = float(np.abs(lg - ref).max())
        assert dmax <= PU.LOGIT_ABS, dmax
        for b in range(len(seq)):
            srt = np.sort(ref[b])[::-1]
            if srt[0] - srt[1] >= 2 * dmax:
                assert int(np.argmax(lg[b])) == int(np.argmax(ref[b]))
    finally:
        mk.close()
        del k, v
        torch.cuda.empty_cache()
