"""Host-only checks of the megakernel schedule (no GPU): the planner's per-SM lists,
simulated with the kernel's wait/signal semantics under random interleavings, must
run to completion with every counter ending exactly at the target its waiters use
and every work queue drained.

The simulator models what each opcode waits on and signals (descriptor fields, the
claimer queues, the fan-in follow-ups: route step, attention combine), with a random
routing, so that a wrong counter target, a missing arrival or a list order that can
deadlock shows up here."""
import collections

import numpy as np
import pytest

import synth
from persistent_moe_decode_cta_gb300 import binding as B

OP_EMBED, OP_QKV, OP_ROUTER, OP_ATT, OP_MOE, OP_OPROJ, OP_LM, OP_RESID = 1, 2, 3, 4, 5, 7, 8, 9
OP_PREFETCH, OP_PREFETCH_KV = 10, 11
D_OP, D_LAYER, D_AUX, D_ROW0, D_K0, D_KLEN = 0, 1, 2, 3, 5, 6
D_WAIT, D_WAIT_T, D_SIG, D_SIG_T, D_WAIT2, D_WAIT2_T = 7, 8, 9, 10, 17, 18
PAGE = 16


def att_splits(cfg, l, p, split_pages):
    w = cfg["sliding_window"] if l in cfg.get("swa_layers", ()) else 0
    lo = max(0, p - w + 1) if w > 0 else 0
    if p <= lo:
        return 0
    npg = (p - 1) // PAGE - lo // PAGE + 1
    return (npg + split_pages - 1) // split_pages


class Sim:
    def __init__(self, cfg, batch, n_sm, seq_lens, seed):
        self.cfg, self.B = cfg, batch
        self.T, off, lst, self.I = B.mk_plan_dry(cfg, batch, n_sm)
        self.lists = [list(lst[off[s]:off[s + 1]]) for s in range(n_sm)]
        self.rng = np.random.default_rng(seed)
        self.seq = seq_lens
        self.ctr = collections.Counter()
        self.split_pages = 8
        I = self.I
        self.maxa, self.t_moe, self.qkv_tpg, self.n_router = I[3], I[5], I[10], I[11]
        (self.c_lr, self.c_qkvg, self.c_rt, self.c_rr, self.c_att, self.c_og, self.c_md,
         self.c_od) = I[16:24]
        self.nrb_d, self.L, self.Hkv = I[24], cfg["n_layers"], cfg["n_kv_heads"]
        self.c_oa = I[26]
        self.t_dense = I[27]
        mask = (int(I[28]) & 0xffffffff) | ((int(I[29]) & 0xffffffff) << 32)
        self.dense = {l for l in range(self.L) if (mask >> l) & 1}
        self.pending = [None] * n_sm   # a claimed O-proj tile waiting for its group
        self.held = [None] * n_sm      # layer of an O-proj tile claimed before C_OA was full
        # queues
        self.att_items = {}
        self.moe_count = {}
        self.heads = collections.Counter()
        self.targets = {}          # counter -> the value its waiters need (checked at end)
        self.arrivals_att = {}

    def C(self, base, *idx):
        if base == self.c_att:
            l, b, g = idx
            return self.c_att + (l * self.B + b) * self.Hkv + g
        if base in (self.c_qkvg, self.c_og):
            l, g = idx
            return base + l * self.Hkv + g
        return base + idx[0]

    def att_queue(self, l):
        if l not in self.att_items:
            per_g = []
            for b in range(self.B):
                ns = att_splits(self.cfg, l, self.seq[b], self.split_pages)
                per_g += [(b, s, ns) for s in range(ns + 1)]
            # the kernel's queue order: KV groups interleaved
            self.att_items[l] = [(g, b, s, ns) for (b, s, ns) in per_g for g in range(self.Hkv)]
        return self.att_items[l]

    def route(self, l):
        E, k = self.cfg["n_experts"], self.cfg["top_k"]
        active = set()
        for b in range(self.B):
            active |= set(self.rng.choice(E, size=k, replace=False).tolist())
        self.moe_count[l] = len(active) * self.t_moe
        self.ctr[self.c_rr + l] += 1
        self.ctr[self.c_md + l] += (self.maxa - len(active)) * self.t_moe

    def ready(self, ci, t):
        self.targets.setdefault(ci, set()).add(t)
        return self.ctr[ci] >= t

    def step_task(self, sm):
        """Try to advance SM `sm` by one task or one claimed item; True if it did."""
        if self.pending[sm] is not None:
            T = self.T[self.pending[sm]]
            if not self.ready(T[D_WAIT], T[D_WAIT_T]):
                return False
            self.ctr[T[D_SIG]] += 1
            self.pending[sm] = None
            return True
        if not self.lists[sm]:
            return False
        ti = self.lists[sm][0]
        T = self.T[ti]
        op, l = T[D_OP], T[D_LAYER]
        if op in (OP_PREFETCH, OP_PREFETCH_KV):   # producer-only, no dependency
            self.lists[sm].pop(0)
            return True
        if op in (OP_QKV, OP_ROUTER, OP_OPROJ, OP_LM, OP_RESID, OP_EMBED):
            if T[D_WAIT] >= 0 and not self.ready(T[D_WAIT], T[D_WAIT_T]):
                return False
            if T[D_WAIT2] >= 0 and not self.ready(T[D_WAIT2], T[D_WAIT2_T]):
                return False
            # the layer's last router tile (D_AUX = 1) collects every tile's logits
            if op == OP_ROUTER and T[D_AUX] == 1 and self.ctr[T[D_SIG]] < T[D_SIG_T] - 1:
                return False
            self.lists[sm].pop(0)
            if op == OP_EMBED:
                self.ctr[T[D_SIG]] += self.nrb_d
            elif op == OP_ROUTER:
                self.ctr[T[D_SIG]] += 1
                if T[D_AUX] == 1:
                    assert self.ctr[T[D_SIG]] == T[D_SIG_T]
                    self.route(l)
            elif op == OP_RESID:
                self.ctr[self.c_lr + l + 1] += 1
            elif op != OP_LM:
                self.ctr[T[D_SIG]] += 1
            return True
        if op == OP_ATT:
            q = self.att_queue(l)
            h = self.heads[("att", l)]
            if h >= len(q):
                self.lists[sm].pop(0)
                return True
            g, b, s, ns = q[h]
            if not self.ready(self.C(self.c_qkvg, l, g), self.qkv_tpg):
                return False
            self.heads[("att", l)] += 1
            ca = self.C(self.c_att, l, b, g)
            self.ctr[ca] += 1
            self.targets.setdefault(ca, set()).add(ns + 1)
            if self.ctr[ca] == ns + 1:
                self.ctr[self.C(self.c_og, l, g)] += 1
                self.ctr[self.c_oa + l] += 1
            return True
        if op == OP_MOE:
            # the drain also serves the layer's O-proj tiles (D_KLEN from task D_K0): ahead
            # of expert items once every attention output is complete, and the remaining
            # ones once the items are gone
            n_o, o_base = T[D_KLEN], T[D_K0]
            ho = self.heads[("oproj", l)]
            if n_o and ho < n_o and self.ready(self.c_oa + l, self.Hkv * self.B):
                self.heads[("oproj", l)] += 1
                self.pending[sm] = o_base + ho
                return True
            # the route words of the layer (a dense layer has none: its FFN's items take
            # every token), and the ADD_RMSNORM outputs (the items' operand)
            if l in self.dense:
                self.moe_count[l] = self.t_dense
            elif not self.ready(self.c_rr + l, 1):
                return False
            if not self.ready(self.c_lr + l, self.nrb_d):
                return False
            h = self.heads[("moe", l)]
            if h < self.moe_count[l]:
                self.heads[("moe", l)] += 1
                self.ctr[self.c_md + l] += 1
                return True
            if n_o and ho < n_o:
                # while the layer's attention outputs are incomplete a drain holds at
                # most one O-proj tile
                full = self.Hkv * self.B
                if self.held[sm] == l and not self.ready(self.c_oa + l, full):
                    return False
                self.held[sm] = l if self.ctr[self.c_oa + l] < full else None
                self.heads[("oproj", l)] += 1
                self.pending[sm] = o_base + ho
                return True
            self.lists[sm].pop(0)
            return True
        raise AssertionError(f"unknown op {op}")

    def run(self):
        n = len(self.lists)
        while any(self.lists) or any(x is not None for x in self.pending):
            order = self.rng.permutation(n)
            progressed = False
            for sm in order:
                if self.step_task(int(sm)):
                    progressed = True
                    break
            assert progressed, f"deadlock: heads {[self.T[l[0]][:3] for l in self.lists if l]}"
        # every counter ends at exactly the value its waiters wait for
        for ci, ts in self.targets.items():
            assert len(ts) == 1, (ci, ts)
            assert self.ctr[ci] == next(iter(ts)), (ci, self.ctr[ci], ts)
        for l in range(self.L):
            assert self.heads[("moe", l)] == self.moe_count[l]
            assert self.heads[("att", l)] == len(self.att_queue(l))
            assert self.ctr[self.c_md + l] == (self.t_dense if l in self.dense else self.maxa * self.t_moe)
        assert self.ctr[self.c_lr + self.L] == self.nrb_d


@pytest.mark.parametrize("workload,batch,n_sm,lens", [
    ("tiny_b1_64", 1, 152, [64]),
    ("tiny_b1_64", 1, 3, [0]),
    ("tiny_b1_64", 8, 5, [64, 1, 0, 17, 33, 200, 15, 16]),
    ("small_b1_2k", 3, 16, [2048, 5, 700]),
    ("pages_b8_ragged_swa", 8, 152, [1024, 5000, 9000, 4097, 4096, 32768, 17, 0]),
    ("tiny_dense_b1_64", 3, 7, [64, 1, 30]),
    ("small_dense_b1_2k", 2, 152, [2048, 100]),
])
def test_schedule_completes_with_exact_counter_targets(workload, batch, n_sm, lens):
    cfg = synth.model_config(workload)
    for seed in range(3):
        Sim(cfg, batch, n_sm, lens, seed).run()


def valid_orders():
    """Every per-layer wave order the planner accepts: the letters r q a m o x with QKV
    before attention before O-proj, the router before the MoE drain, and the MoE drain
    and O-proj before ADD_RMSNORM."""
    import itertools
    out = []
    for perm in itertools.permutations("rqamox"):
        s = "".join(perm)
        i = s.index
        if i("q") < i("a") < i("o") and i("r") < i("m") < i("x") and i("o") < i("x"):
            out.append(s)
    return out


# the pages' three named orders, as read here: the tuned order they state (QKV,
# router, attention, MoE projections, O-proj and RMSNorm), attention-first (the whole
# attention branch before the router), interleaved (the MoE branch's waves ahead of the
# attention branch's, alternating)
PAGES_ORDERS = {"tuned": "qramox", "attention-first": "qaormx", "interleaved": "rqmaox"}


def test_valid_orders_include_the_pages_orders_and_reject_broken_ones(monkeypatch):
    orders = valid_orders()
    assert len(orders) == 10 and "rqamox" in orders
    assert set(PAGES_ORDERS.values()) <= set(orders)
    cfg = synth.model_config("tiny_b1_64")
    for bad in ("aqrmox", "rqaxmo", "rqamo", "rqamoxx", "rqamoz"):
        monkeypatch.setenv("MK_WAVE_ORDER", bad)
        with pytest.raises(B.MkError):
            B.mk_plan_dry(cfg, 1, 4)


@pytest.mark.parametrize("order", valid_orders())
@pytest.mark.parametrize("workload,batch,n_sm,lens", [
    ("tiny_b1_64", 8, 3, [64, 1, 0, 17, 33, 200, 15, 16]),
    ("small_b1_2k", 2, 5, [2048, 37]),
    ("tiny_dense_b1_64", 2, 2, [64, 9]),
])
def test_every_wave_order_completes_with_exact_counter_targets(monkeypatch, order, workload, batch, n_sm,
                                                                lens):
    """Any order that respects the dependencies, dealt to fewer SMs than a layer has
    O-proj tiles (the case in which a MoE drain ahead of the attention drain could hold
    an O-proj tile on every SM), runs to completion with exact counter targets."""
    monkeypatch.setenv("MK_WAVE_ORDER", order)
    cfg = synth.model_config(workload)
    for seed in range(2):
        Sim(cfg, batch, n_sm, lens, seed).run()


def test_tasks_are_dealt_round_robin_within_waves():
    cfg = synth.model_config("small_b1_2k")
    T, off, lst, info = B.mk_plan_dry(cfg, 1, 7)
    # static tasks appear in exactly one list; the first wave of layer 0 (after the
    # embedding on SM 0) deals task k to SM k mod 7
    owner = {}
    for s in range(7):
        for t in lst[off[s]:off[s + 1]]:
            if T[t][0] not in (OP_ATT, OP_MOE, OP_PREFETCH_KV):
                assert t not in owner
                owner[t] = s
    # the O-proj tiles are served by the MoE drains, not dealt
    assert not any(T[t][0] == OP_OPROJ for t in owner)
    router0 = [t for t in range(len(T)) if T[t][0] == OP_ROUTER and T[t][1] == 0]
    assert [owner[t] for t in router0] == [k % 7 for k in range(len(router0))]
    # claimer tasks: one per SM per layer
    for s in range(7):
        ops = [T[t][0] for t in lst[off[s]:off[s + 1]]]
        assert ops.count(OP_ATT) == cfg["n_layers"] and ops.count(OP_MOE) == cfg["n_layers"]


def test_descriptor_weight_offsets_are_tile_aligned_and_disjoint():
    cfg = synth.model_config("small_b1_2k")
    T, off, lst, info = B.mk_plan_dry(cfg, 2, 9)
    spans = []
    for t in T:
        if t[0] in (OP_QKV, OP_ROUTER, OP_OPROJ, OP_LM):
            o = (int(t[12]) << 32) | (int(t[11]) & 0xFFFFFFFF)
            n = int(t[13])
            assert o % 512 == 0 and n % 512 == 0 and n == t[4] * t[6] * 2
            spans.append((o, o + n))
    spans.sort()
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
