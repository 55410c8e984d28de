"""Seeded synthetic inputs for the MoE decode step: model shapes, weights, paged KV
cache, page tables and tokens.

This module is shared by the tests, the benchmark and the oracle's callers. It holds
no arithmetic of the decode step itself: only shapes, random draws and data movement
(device tensors -> host numpy views for the oracle).

Shapes follow the workloads the megakernel pages measure (a parallel-block MoE decoder
in BF16, paged KV in 16-token pages, batch 1-8); the model itself (North Mini Code)
and its checkpoint are not available, so every tensor is drawn from a seeded normal
distribution: matrices ~N(0, 0.02) in bf16, K/V ~N(0, 1) in bf16, norm gains 1.0.
"""
from __future__ import annotations

import hashlib
import math

import numpy as np
import torch

PAGE = 16

# Model shapes.  The three shapes are the tiny and small parity models and the
# pages-scale model (about 30.5B total / 3.3B active parameters).
MODELS = {
    "tiny": dict(n_layers=2, d_model=256, n_q_heads=8, n_kv_heads=2, head_dim=32,
                 n_experts=8, top_k=2, d_ff=128, vocab=1024, rope_theta=1e4,
                 rms_eps=1e-6, sliding_window=0, swa_layers=()),
    "small": dict(n_layers=8, d_model=1024, n_q_heads=16, n_kv_heads=4, head_dim=64,
                  n_experts=32, top_k=4, d_ff=512, vocab=32000, rope_theta=1e4,
                  rms_eps=1e-6, sliding_window=0, swa_layers=()),
    "pages": dict(n_layers=48, d_model=2048, n_q_heads=32, n_kv_heads=4, head_dim=128,
                  n_experts=128, top_k=8, d_ff=768, vocab=151936, rope_theta=1e6,
                  rms_eps=1e-6, sliding_window=0, swa_layers=()),
}
# Mixed dense/MoE stacks (a dense layer: one SwiGLU FFN of width dense_ff for every
# token, no router): the tiny and small parity models with some layers dense.
MODELS["tiny_dense"] = dict(MODELS["tiny"], dense_layers=(0,), dense_ff=256)
MODELS["small_dense"] = dict(MODELS["small"], dense_layers=(0, 5), dense_ff=1024)
# Two layers of the pages-scale shape: small enough (3.7 GB) for profiler captures
# and for the oracle to run in seconds, with every tile size of the full model.
MODELS["pages_l2"] = dict(MODELS["pages"], n_layers=2)
MODELS["pages_l1"] = dict(MODELS["pages"], n_layers=1)
# The pages-scale shape with its first three layers dense (FFN width 4096), for the
# mixed-stack measurement.
MODELS["pages_dense3"] = dict(MODELS["pages"], dense_layers=(0, 1, 2), dense_ff=4096)
# The same shapes with the routed experts stored as E4M3 codes + float32 scales (the
# weights drawn are the bf16 ones; quantisation happens when the model is loaded).
for _m in ("tiny", "small", "pages", "pages_l2", "tiny_dense", "small_dense"):
    MODELS[_m + "_fp8"] = dict(MODELS[_m], expert_dtype="fp8")
# ... and with the dense projections (QKV, O-proj, LM head) in FP8 as well
for _m in ("tiny", "small", "pages", "pages_l2", "pages_l1", "tiny_dense", "small_dense"):
    MODELS[_m + "_fp8w"] = dict(MODELS[_m], expert_dtype="fp8", dense_dtype="fp8")

# Workloads: a model plus a batch of cached sequence lengths.
WORKLOADS = {
    "tiny_b1_64": dict(model="tiny", batch=1, lens=("fixed", 64)),
    "small_b1_2k": dict(model="small", batch=1, lens=("fixed", 2048)),
    "pages_b1_8k": dict(model="pages", batch=1, lens=("fixed", 8192)),
    "pages_b8_ragged_swa": dict(model="pages", batch=8, lens=("uniform", 1024, 32768),
                                sliding_window=4096, swa="odd"),
    "pages_b1_128k": dict(model="pages", batch=1, lens=("fixed", 131072)),
    "pages_l2_b1_8k": dict(model="pages_l2", batch=1, lens=("fixed", 8192)),
    "pages_l1_b1_8k": dict(model="pages_l1", batch=1, lens=("fixed", 8192)),
    "pages_l2_b8_ragged_swa": dict(model="pages_l2", batch=8, lens=("uniform", 1024, 32768),
                                   sliding_window=4096, swa="odd"),
    "tiny_dense_b1_64": dict(model="tiny_dense", batch=1, lens=("fixed", 64)),
    "pages_dense3_b1_8k": dict(model="pages_dense3", batch=1, lens=("fixed", 8192)),
    "small_dense_b1_2k": dict(model="small_dense", batch=1, lens=("fixed", 2048)),
    "tiny_fp8_b1_64": dict(model="tiny_fp8", batch=1, lens=("fixed", 64)),
    "small_fp8_b1_2k": dict(model="small_fp8", batch=1, lens=("fixed", 2048)),
    "pages_fp8_b1_8k": dict(model="pages_fp8", batch=1, lens=("fixed", 8192)),
    "pages_l2_fp8_b1_8k": dict(model="pages_l2_fp8", batch=1, lens=("fixed", 8192)),
    "tiny_dense_fp8_b1_64": dict(model="tiny_dense_fp8", batch=1, lens=("fixed", 64)),
    "small_dense_fp8_b1_2k": dict(model="small_dense_fp8", batch=1, lens=("fixed", 2048)),
    "pages_fp8_b8_ragged_swa": dict(model="pages_fp8", batch=8, lens=("uniform", 1024, 32768),
                                    sliding_window=4096, swa="odd", lens_of="pages_b8_ragged_swa"),
    "pages_l2_fp8_b8_ragged_swa": dict(model="pages_l2_fp8", batch=8, lens=("uniform", 1024, 32768),
                                       sliding_window=4096, swa="odd", lens_of="pages_b8_ragged_swa"),
    # FP8 experts and dense projections
    "tiny_fp8w_b1_64": dict(model="tiny_fp8w", batch=1, lens=("fixed", 64)),
    "small_fp8w_b1_2k": dict(model="small_fp8w", batch=1, lens=("fixed", 2048)),
    "tiny_dense_fp8w_b1_64": dict(model="tiny_dense_fp8w", batch=1, lens=("fixed", 64)),
    "pages_fp8w_b1_8k": dict(model="pages_fp8w", batch=1, lens=("fixed", 8192)),
    "pages_l1_fp8w_b1_8k": dict(model="pages_l1_fp8w", batch=1, lens=("fixed", 8192)),
    "pages_l2_fp8w_b1_8k": dict(model="pages_l2_fp8w", batch=1, lens=("fixed", 8192)),
    "pages_fp8w_b8_ragged_swa": dict(model="pages_fp8w", batch=8, lens=("uniform", 1024, 32768),
                                     sliding_window=4096, swa="odd", lens_of="pages_b8_ragged_swa"),
}


def model_config(workload: str) -> dict:
    """Model shape dict for a workload, with the workload's sliding-window setting."""
    w = WORKLOADS[workload]
    cfg = dict(MODELS[w["model"]])
    if w.get("sliding_window"):
        cfg["sliding_window"] = w["sliding_window"]
        if w.get("swa") == "odd":
            cfg["swa_layers"] = tuple(l for l in range(cfg["n_layers"]) if l % 2 == 1)
    cfg["page_size"] = PAGE
    return cfg


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def seq_lens_for(workload: str, seed: int = 0) -> list[int]:
    w = WORKLOADS[workload]
    kind = w["lens"][0]
    if kind == "fixed":
        return [w["lens"][1]] * w["batch"]
    lo, hi = w["lens"][1], w["lens"][2]
    # (a variant of a workload -- e.g. its FP8 form -- draws the same lengths)
    rng = np.random.default_rng(_seed("seq_lens", w.get("lens_of", workload), seed))
    return [int(v) for v in rng.integers(lo, hi + 1, size=w["batch"])]


EXPERT_TENSORS = ("w_gate", "w_up", "w_down")


def make_weights(cfg: dict, seed: int = 0, device="cpu", gain_jitter: float = 0.0,
                 std: float = 0.02) -> dict:
    """All model tensors, bf16, row-major [out, in] for every projection.

    embed/lm_head [V, d]; attn_norm [L, d]; final_norm [d]; wq [L, Hq*hd, d];
    wk/wv [L, Hkv*hd, d]; wo [L, d, Hq*hd]; router [L, E, d];
    w_gate/w_up [L, E, f, d]; w_down [L, E, d, f].
    Gains are 1.0, or 1 + gain_jitter * N(0, 1) when gain_jitter > 0 (so that tests
    see the gain multiply).  Each layer slice (and each expert of a layer) has its own
    generator.
    """
    L, d, Hq, Hkv, hd = (cfg[k] for k in ("n_layers", "d_model", "n_q_heads",
                                          "n_kv_heads", "head_dim"))
    E, f, V = cfg["n_experts"], cfg["d_ff"], cfg["vocab"]
    bf = torch.bfloat16
    shapes = {
        "wq": (Hq * hd, d), "wk": (Hkv * hd, d), "wv": (Hkv * hd, d),
        "wo": (d, Hq * hd), "router": (E, d),
        "w_gate": (E, f, d), "w_up": (E, f, d), "w_down": (E, d, f),
    }
    W = {}
    for name, shp in shapes.items():
        t = torch.empty((L,) + shp, dtype=bf, device=device)
        for l in range(L):
            if name in EXPERT_TENSORS:
                for e in range(E):
                    t[l, e].normal_(0.0, std, generator=_gen(device, seed, name, l, e))
            else:
                t[l].normal_(0.0, std, generator=_gen(device, seed, name, l))
        W[name] = t
    for name in ("embed", "lm_head"):
        W[name] = torch.empty((V, d), dtype=bf, device=device).normal_(
            0.0, std, generator=_gen(device, seed, name))
    def gains(name, shape):
        g = torch.ones(shape, dtype=torch.float32, device=device)
        if gain_jitter > 0:
            g += gain_jitter * torch.randn(shape, generator=_gen(device, seed, name),
                                           device=device)
        return g.to(bf)
    W["attn_norm"] = gains("attn_norm", (L, d))
    W["final_norm"] = gains("final_norm", (d,))
    dense = tuple(cfg.get("dense_layers", ()))
    if dense:
        # the dense FFNs of a mixed stack: ffn_gate/ffn_up [L, Fd, d], ffn_down [L, d, Fd]
        # (drawn for the dense layers, zero elsewhere)
        fd = cfg["dense_ff"]
        for name, shp in (("ffn_gate", (fd, d)), ("ffn_up", (fd, d)), ("ffn_down", (d, fd))):
            t = torch.zeros((L,) + shp, dtype=bf, device=device)
            for l in dense:
                t[l].normal_(0.0, std, generator=_gen(device, seed, name, l))
            W[name] = t
    return W


def pages_needed(seq_lens, steps: int = 1) -> list[int]:
    """Pages each sequence needs to hold its cached tokens plus `steps` new ones."""
    return [(n + steps + PAGE - 1) // PAGE for n in seq_lens]


def make_page_table(seq_lens, steps: int = 1, seed: int = 0, spare: int = 0):
    """Shuffled physical page ids.  Returns (page_table int32 [B, max_pages] with -1
    for unused entries, n_pages in the pool)."""
    need = pages_needed(seq_lens, steps)
    total = sum(need) + spare
    rng = np.random.default_rng(_seed("pages", seed, tuple(seq_lens)))
    perm = rng.permutation(total).astype(np.int32)
    maxp = max(need)
    pt = np.full((len(seq_lens), maxp), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[o:o + n]
        o += n
    return pt, total


def make_kv(cfg: dict, n_pages: int, seed: int = 0, device="cpu"):
    """K and V pools, bf16 [L, n_pages, Hkv, 16, hd], ~N(0, 1); cached K counts as
    already rotated."""
    L, Hkv, hd = cfg["n_layers"], cfg["n_kv_heads"], cfg["head_dim"]
    shp = (n_pages, Hkv, PAGE, hd)
    k = torch.empty((L,) + shp, dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    for l in range(L):
        k[l].normal_(0.0, 1.0, generator=_gen(device, seed, "k", l))
        v[l].normal_(0.0, 1.0, generator=_gen(device, seed, "v", l))
    return k, v


def make_tokens(batch: int, vocab: int, seed: int = 0, device="cpu"):
    g = _gen("cpu", seed, "tokens")
    return torch.randint(0, vocab, (batch,), generator=g, dtype=torch.int32).to(device)


# ---------------------------------------------------------------------------
# Host views for the oracle: bf16 tensors handed over as uint16 numpy arrays,
# copied from the device lazily (the pages-scale model does not fit in host RAM
# in fp64, and the oracle only needs the experts that were routed to).

def _u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


class HostWeights:
    """Adapter from the tensor dict of make_weights() to the oracle's weight
    accessors.  cache_experts=True also keeps the host copy of every expert asked for
    (for repeated oracle steps; the dense matrices are always kept)."""

    def __init__(self, W: dict, cache_experts: bool = False):
        self.W = W
        self._cache = {}
        self.cache_experts = cache_experts

    def _get(self, key, fn):
        if key not in self._cache:
            self._cache[key] = fn()
        return self._cache[key]

    def embed_rows(self, tokens):
        idx = torch.as_tensor(np.asarray(tokens, dtype=np.int64),
                              device=self.W["embed"].device)
        return _u16(self.W["embed"].index_select(0, idx))

    def attn_norm(self, l): return self._get(("an", l), lambda: _u16(self.W["attn_norm"][l]))
    def wq(self, l): return self._get(("wq", l), lambda: _u16(self.W["wq"][l]))
    def wk(self, l): return self._get(("wk", l), lambda: _u16(self.W["wk"][l]))
    def wv(self, l): return self._get(("wv", l), lambda: _u16(self.W["wv"][l]))
    def wo(self, l): return self._get(("wo", l), lambda: _u16(self.W["wo"][l]))
    def router(self, l): return self._get(("wr", l), lambda: _u16(self.W["router"][l]))

    def expert(self, l, e):
        fn = lambda: (_u16(self.W["w_gate"][l, e]), _u16(self.W["w_up"][l, e]),
                      _u16(self.W["w_down"][l, e]))
        return self._get(("ex", l, e), fn) if self.cache_experts else fn()

    def dense_ffn(self, l):
        return (_u16(self.W["ffn_gate"][l]), _u16(self.W["ffn_up"][l]), _u16(self.W["ffn_down"][l]))

    def final_norm(self): return self._get(("fn",), lambda: _u16(self.W["final_norm"]))
    def lm_head(self): return self._get(("lm",), lambda: _u16(self.W["lm_head"]))

    def drop_cache(self):
        self._cache.clear()


class HostKV:
    """Adapter from K/V pool tensors [L, n_pages, Hkv, 16, hd] to the oracle's page
    gather accessor.  cache=True keeps each layer's gathered pages (repeated oracle
    steps over the same pages)."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor, cache: bool = False):
        self.k, self.v = k, v
        self._cache = {} if cache else None

    def pages(self, l, page_ids):
        key = (l, tuple(int(p) for p in page_ids)) if self._cache is not None else None
        if key is not None and key in self._cache:
            return self._cache[key]
        idx = torch.as_tensor(np.asarray(page_ids, dtype=np.int64), device=self.k.device)
        out = _u16(self.k[l].index_select(0, idx)), _u16(self.v[l].index_select(0, idx))
        if key is not None:
            self._cache[key] = out
        return out


class LazyHostWeights:
    """Oracle weight accessors that draw each tensor on the host when first asked
    for, from the same per-layer / per-expert seeds as make_weights (host and device
    generators differ, so the values differ from a device draw; shapes and
    distribution are the same).  Used to time the oracle on a slice of the
    pages-scale model without materialising all 61 GB."""

    def __init__(self, cfg: dict, seed: int = 0, std: float = 0.02):
        self.cfg, self.seed, self.std = cfg, seed, std
        self._cache = {}

    def _draw(self, key, shape, *parts):
        if key not in self._cache:
            t = torch.empty(shape, dtype=torch.bfloat16).normal_(
                0.0, self.std, generator=_gen("cpu", self.seed, *parts))
            self._cache[key] = _u16(t)
        return self._cache[key]

    def _dims(self):
        c = self.cfg
        return (c["d_model"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["n_experts"],
                c["d_ff"], c["vocab"])

    def embed_rows(self, tokens):
        d = self.cfg["d_model"]
        out = np.empty((len(tokens), d), dtype=np.uint16)
        for i, t in enumerate(tokens):
            out[i] = self._draw(("emb", int(t)), (d,), self.seed, "embed_row", int(t))
        return out

    def attn_norm(self, l):
        return _u16(torch.ones(self.cfg["d_model"], dtype=torch.bfloat16))

    def final_norm(self):
        return _u16(torch.ones(self.cfg["d_model"], dtype=torch.bfloat16))

    def wq(self, l):
        d, Hq, _, hd, _, _, _ = self._dims()
        return self._draw(("wq", l), (Hq * hd, d), "wq", l)

    def wk(self, l):
        d, _, Hkv, hd, _, _, _ = self._dims()
        return self._draw(("wk", l), (Hkv * hd, d), "wk", l)

    def wv(self, l):
        d, _, Hkv, hd, _, _, _ = self._dims()
        return self._draw(("wv", l), (Hkv * hd, d), "wv", l)

    def wo(self, l):
        d, Hq, _, hd, _, _, _ = self._dims()
        return self._draw(("wo", l), (d, Hq * hd), "wo", l)

    def router(self, l):
        d, _, _, _, E, _, _ = self._dims()
        return self._draw(("wr", l), (E, d), "router", l)

    def expert(self, l, e):
        d, _, _, _, _, f, _ = self._dims()
        return (self._draw(("g", l, e), (f, d), "w_gate", l, e),
                self._draw(("u", l, e), (f, d), "w_up", l, e),
                self._draw(("dn", l, e), (d, f), "w_down", l, e))

    def lm_head(self, rows=None):
        d, V = self.cfg["d_model"], self.cfg["vocab"]
        n = V if rows is None else rows
        return self._draw(("lm", n), (n, d), "lm_head", n)


class LazyHostKV:
    """K/V page accessor that draws pages on the host on demand (same role as
    HostKV, for timing the oracle on a slice of a long context)."""

    def __init__(self, cfg: dict, seed: int = 0):
        self.cfg, self.seed = cfg, seed
        self._cache = {}

    def pages(self, l, page_ids):
        Hkv, hd = self.cfg["n_kv_heads"], self.cfg["head_dim"]
        key = (l, tuple(int(p) for p in page_ids))
        if key not in self._cache:
            n = len(page_ids)
            g = _gen("cpu", self.seed, "kvpages", l)
            k = torch.empty((n, Hkv, PAGE, hd), dtype=torch.bfloat16).normal_(0, 1, generator=g)
            v = torch.empty((n, Hkv, PAGE, hd), dtype=torch.bfloat16).normal_(0, 1, generator=g)
            self._cache = {key: (_u16(k), _u16(v))}
        return self._cache[key]


def max_active_experts(cfg: dict, batch: int) -> int:
    return min(cfg["n_experts"], batch * cfg["top_k"])


def describe(workload: str) -> str:
    w = WORKLOADS[workload]
    c = model_config(workload)
    return (f"{workload}: {c['n_layers']}L d{c['d_model']} {c['n_q_heads']}/{c['n_kv_heads']}x"
            f"{c['head_dim']} E{c['n_experts']} top{c['top_k']} f{c['d_ff']} V{c['vocab']} "
            f"B={w['batch']} lens={w['lens']}")


__all__ = ["MODELS", "WORKLOADS", "PAGE", "model_config", "seq_lens_for", "make_weights",
           "make_page_table", "make_kv", "make_tokens", "HostWeights", "HostKV",
           "LazyHostWeights", "LazyHostKV",
           "pages_needed", "max_active_experts", "describe"]
