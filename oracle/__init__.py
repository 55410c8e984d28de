"""CPU oracle for one batched decode step of a parallel-block MoE transformer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this package:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
use it.  It shares no code with the CUDA path.

What it computes is the plain definition of the decode step the megakernel pages
describe, in float64 over the same bf16 weight bits (widened exactly):

* one pre-norm per layer feeding both branches of a parallel block, with the
  residual ``x <- x + attn(h) + moe(h)``
  [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "One kernel for the
  full decode step": attention and MoE branches of a layer are independent;
  Cohere open-sources fused LLM decode kernel with 1.58x vLLM claim: the 16 task
  types, one of them ADD_RMSNORM];
* QKV projection with RoPE, the new K/V stored in bf16 into a paged cache, grouped-
  query attention over the cached keys plus the new one, O projection
  [same pages: QKV_PROJ, ATTN_DECODE/ATTN_COMBINE, O_PROJ; Cohere Megakernel,
  "Overview": paged KV cache and sliding-window attention];
* router GEMM, top-k, softmax over the selected logits, SwiGLU experts and the
  weighted combine [same pages: ROUTER_GEMM, ROUTER_TOPK, MOE_UPGATE_ACT,
  MOE_DOWN, MOE_COMBINE; the calling-convention section names the SiLU-and-multiply
  epilogue];
* final RMSNorm and LM head, fp logits, greedy argmax [Cohere's Open-Source
  Megakernel ..., "Current limitations": greedy sampling].

Readings taken where the pages are silent:
rotate-half RoPE with inv_freq_i = theta^(-2i/hd) over the full head; cached K is
already rotated; the new token sits at position L_b and attends to itself; the
attention window of a sliding-window layer is {j : p - W < j <= p}; q head i uses
KV head floor(i * Hkv / Hq); top-k ties go to the lower expert index; argmax ties
to the lower token id; norm gains multiply after the normalisation; a dense layer of
a mixed stack (cfg["dense_layers"]) replaces the routed experts by one SwiGLU FFN of
width cfg["dense_ff"] applied to every token with weight 1, sharing the layer's pre-norm.

Parity status: every building block below is pinned by tests/test_oracle_pins.py
(closed forms, invariants, special cases, library routines for bf16 rounding and
sorting), and so are the two steps of layer_step that combine them: the query's
rotation at the token's own position (a whole layer's invariance to shifting every
position, and the attention peak when query and keys share one raw vector) and the
pairing of each routing weight with its expert (a layer reduced to a closed form with
distinct experts on disjoint outputs).  Whole-model values on the larger models have no published example and
are pinned only through those blocks ("parity unpinned" beyond them).
"""
from __future__ import annotations

import numpy as np

PAGE = 16


# ---------------------------------------------------------------------------
# bf16 <-> float64

def bf16_to_f64(u16) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 to the nearest bf16 (ties to even), returning uint16 bits.

    Rounds directly from float64 (one rounding), for finite normal values of bf16
    range; values below the smallest normal are flushed to signed zero."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    u = x.view(np.uint64)
    sign = (u >> np.uint64(63)).astype(np.uint32)
    mag = u & np.uint64(0x7FFFFFFFFFFFFFFF)
    exp = (mag >> np.uint64(52)).astype(np.int64) - 1023 + 127
    mant = mag & np.uint64((1 << 52) - 1)
    out = np.zeros(x.shape, dtype=np.uint32)
    normal = (exp >= 1) & (exp < 255)
    comb = (exp.clip(0, 255).astype(np.uint64) << np.uint64(52)) | mant
    q = comb >> np.uint64(45)
    rem = comb & np.uint64((1 << 45) - 1)
    half = np.uint64(1 << 44)
    up = (rem > half) | ((rem == half) & ((q & np.uint64(1)) == np.uint64(1)))
    q = q + up.astype(np.uint64)
    out = np.where(normal, q.astype(np.uint32), out)
    out = np.where(exp >= 255, np.uint32(0x7F80), out)          # overflow -> inf
    out = np.where(np.isnan(x), np.uint32(0x7FC0), out)
    return (out | (sign << 15)).astype(np.uint16)


# ---------------------------------------------------------------------------
# building blocks

# ---------------------------------------------------------------- FP8 (E4M3) weights
# The FP8 weight path stores expert matrices as E4M3 codes with float32 scales, one
# scale per output channel (row) of each of gate, up and down; a code decodes as
# sign * value(code) * scale.
# E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
# subnormal (m/8 * 2^-6); the largest finite value is 448; 0x7F/0xFF are NaN.
# Quantisation rounds x / scale (a float32 division) to the nearest code, ties to
# even, saturating to +-448; scale = max|row| / 448 (float32), 1 for an all-zero row.
# [Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "Current limitations":
# FP8 weights are on the roadmap; the pages fix no format: E4M3 with per-channel
# float32 scales is the reading taken]
# cfg["expert_dtype"] == "fp8": the routed experts are stored so; cfg["dense_dtype"] ==
# "fp8" as well: QKV, O-proj and LM-head matrices too (router and embedding stay bf16).
E4M3_MAX = 448.0


def e4m3_to_f64(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    return sign * val


def f32_to_e4m3(x) -> np.ndarray:
    """Nearest E4M3 code of each float32 value, ties to even, saturating to +-448."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)      # exact
    neg = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))                      # a = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)                                     # binade (subnormals share -6)
    step = np.exp2((e - 3).astype(np.float64))                     # spacing of 3 mantissa bits
    v = np.minimum(np.round(a / step) * step, E4M3_MAX)           # np.round: ties to even
    _, ev = np.frexp(np.where(v > 0, v, 1.0))
    ev = ev - 1
    sub = v < 2.0 ** -6
    mant_sub = np.round(v / 2.0 ** -9).astype(np.int64)
    mant_nrm = np.round((v / np.exp2(ev.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    code = np.where(sub, mant_sub, ((ev + 7) << 3) | mant_nrm)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def quantize_e4m3_rows(w_u16, block=None):
    """E4M3 codes and float32 scales of a bf16 matrix [rows, cols]: one scale per row,
    or per row and `block` columns.  Returns (codes uint8 [rows, cols], scales float32
    [rows] or [rows, cols // block])."""
    w = bf16_to_f64(w_u16).astype(np.float32)                       # exact
    rows, cols = w.shape
    if block is not None and (cols % block or cols < block):
        raise ValueError(f"{cols} columns are not whole {block}-column blocks")
    nb = 1 if block is None else cols // block
    wb = w.reshape(rows, nb, cols // nb)
    amax = np.max(np.abs(wb), axis=2)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    codes = f32_to_e4m3((wb / scale[:, :, None]).astype(np.float32)).reshape(rows, cols)
    return codes, (scale[:, 0] if block is None else scale)


def dequantize_e4m3(codes, scales, block=None) -> np.ndarray:
    v = e4m3_to_f64(codes)
    if block is None:
        return v * np.asarray(scales, dtype=np.float64)[:, None]
    rows, cols = v.shape
    s = np.repeat(np.asarray(scales, dtype=np.float64), block, axis=1)
    return v * s


def fp8_expert(wg_u16, wu_u16, wd_u16):
    """The expert's matrices as the FP8 path stores them (per-row scales), decoded to
    float64."""
    return tuple(dequantize_e4m3(*quantize_e4m3_rows(w)) for w in (wg_u16, wu_u16, wd_u16))


def fp8_matrix(w_u16):
    """A dense projection (QKV, O-proj, LM head) as the FP8 weight path stores it: E4M3
    codes with one float32 scale per output channel (row), the reading taken for the
    experts, decoded to float64.  The router and the embedding stay bf16."""
    return dequantize_e4m3(*quantize_e4m3_rows(w_u16))


def _dense(cfg, w_u16):
    return fp8_matrix(w_u16) if cfg.get("dense_dtype") == "fp8" else bf16_to_f64(w_u16)


def rms_norm(x, gain, eps):
    """x / sqrt(mean(x^2) + eps) * gain, over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * gain


def rope(v, pos, theta):
    """Rotate-half rotary embedding of v [..., hd] at integer position pos.

    Pairs (i, i + hd/2) rotate by angle pos * theta^(-2i/hd)."""
    v = np.asarray(v, dtype=np.float64)
    hd = v.shape[-1]
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    ang = float(pos) * theta ** (-2.0 * i / hd)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = v[..., :half], v[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(s):
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - s.max())
    return e / e.sum()


def attention(q, K, V):
    """Grouped-query attention of one token.

    q [Hq, hd]; K, V [n_keys, Hkv, hd].  Head i uses KV head floor(i*Hkv/Hq); scores
    are q.k / sqrt(hd) and the softmax runs over all n_keys keys."""
    Hq, hd = q.shape
    Hkv = K.shape[1]
    o = np.empty((Hq, hd))
    for i in range(Hq):
        g = (i * Hkv) // Hq
        s = K[:, g, :] @ q[i] / np.sqrt(hd)
        o[i] = softmax(s) @ V[:, g, :]
    return o


def attention_partial(q, K, V):
    """Unnormalised softmax partial over a subset of keys: per head (m, l, o) with
    m = max score, l = sum exp(s - m), o = sum exp(s - m) v."""
    Hq, hd = q.shape
    Hkv = K.shape[1]
    m = np.empty(Hq); l = np.empty(Hq); o = np.empty((Hq, hd))
    for i in range(Hq):
        g = (i * Hkv) // Hq
        s = K[:, g, :] @ q[i] / np.sqrt(hd)
        m[i] = s.max()
        e = np.exp(s - m[i])
        l[i] = e.sum()
        o[i] = e @ V[:, g, :]
    return m, l, o


def merge_partials(parts):
    """Log-sum-exp merge of attention partials [(m, l, o), ...] -> normalised o."""
    M = np.max(np.stack([p[0] for p in parts]), axis=0)
    L = sum(p[1] * np.exp(p[0] - M) for p in parts)
    O = sum(p[2] * np.exp(p[0] - M)[:, None] for p in parts)
    return O / L[:, None]


def router_topk(r, k, forced=None):
    """Top-k experts of router logits r [E] and softmax weights over the selected
    logits.  Ties go to the lower expert index.  `forced` replaces the selection
    (used when a near-tie lets either set be correct).  Returns (idx, w, margin)
    with margin = r_(k) - r_(k+1) in descending order."""
    r = np.asarray(r, dtype=np.float64)
    E = r.shape[0]
    order = sorted(range(E), key=lambda e: (-r[e], e))
    margin = (r[order[k - 1]] - r[order[k]]) if k < E else np.inf
    idx = list(order[:k]) if forced is None else list(forced)
    w = softmax(r[idx])
    return np.array(idx, dtype=np.int64), w, margin


def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu_expert(h, wg, wu, wd):
    """Down(silu(Gate h) * (Up h)) with float64 matrices [f,d], [f,d], [d,f]."""
    return wd @ (silu(wg @ h) * (wu @ h))


def window_start(p, window):
    """First key position attended by a token at position p (window 0 = full)."""
    return 0 if window <= 0 else max(0, p - window + 1)


def argmax_lowest(v):
    """Index of the maximum, lowest index on ties."""
    v = np.asarray(v)
    return int(np.flatnonzero(v == v.max())[0])


# ---------------------------------------------------------------------------
# one layer, one step

def _mat(u16):
    return bf16_to_f64(u16)


def layer_step(cfg, W, kv, l, x, positions, page_table, forced=None):
    """Layer l of the decode step for every sequence of the batch.

    x [B, d] float64 residual entering the layer; positions[b] = cached length L_b
    (the new token's position); page_table [B, max_pages] physical page ids; W and
    kv are accessor objects (see synth.HostWeights / synth.HostKV).  forced maps
    b -> expert list to use instead of the top-k.

    Returns (x_next [B, d], info) where info records router logits, the selection,
    weights and margins, and the bf16 K/V written with their page and slot.
    """
    B, d = x.shape
    Hq, Hkv, hd = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    k_top, eps, theta = cfg["top_k"], cfg["rms_eps"], cfg["rope_theta"]
    window = cfg["sliding_window"] if l in tuple(cfg.get("swa_layers", ())) else 0

    dense = l in tuple(cfg.get("dense_layers", ()))
    g = bf16_to_f64(W.attn_norm(l))
    Wq, Wk, Wv, Wo = (_dense(cfg, W.wq(l)), _dense(cfg, W.wk(l)), _dense(cfg, W.wv(l)),
                      _dense(cfg, W.wo(l)))
    h = rms_norm(x, g, eps)                                   # [B, d]

    info = dict(router_logits=np.empty((B, cfg["n_experts"])), idx=[], w=[], margin=[],
                kv=[])
    attn_out = np.empty((B, d))
    for b in range(B):
        p = int(positions[b])
        q = rope((Wq @ h[b]).reshape(Hq, hd), p, theta)
        k_new = rope((Wk @ h[b]).reshape(Hkv, hd), p, theta)
        v_new = (Wv @ h[b]).reshape(Hkv, hd)
        k16, v16 = f64_to_bf16(k_new), f64_to_bf16(v_new)    # stored in the bf16 cache
        page, slot = int(page_table[b][p // PAGE]), p % PAGE
        info["kv"].append(dict(b=b, page=page, slot=slot, k=k16, v=v16))

        lo = window_start(p, window)
        keys = np.empty((p - lo + 1, Hkv, hd))
        vals = np.empty_like(keys)
        if p > lo:
            pos = np.arange(lo, p)
            pages = np.asarray(page_table[b])[pos // PAGE]
            uniq, inv = np.unique(pages, return_inverse=True)
            Kp, Vp = kv.pages(l, uniq)                        # [n, Hkv, 16, hd] uint16
            keys[:-1] = bf16_to_f64(Kp[inv, :, pos % PAGE, :])
            vals[:-1] = bf16_to_f64(Vp[inv, :, pos % PAGE, :])
        keys[-1] = bf16_to_f64(k16)
        vals[-1] = bf16_to_f64(v16)
        o = attention(q, keys, vals)
        attn_out[b] = Wo @ o.reshape(-1)

    if dense:
        # a dense layer of a mixed stack: one SwiGLU FFN for every token, no router
        # [Cohere open-sources fused LLM decode kernel with 1.58x vLLM claim: the dense
        # GEMM task types FFN_UPGATE_ACT and FFN_DOWN]
        wg, wu, wd = (_mat(a) for a in W.dense_ffn(l))
        ffn_out = np.stack([swiglu_expert(h[b], wg, wu, wd) for b in range(B)])
        info["router_logits"] = None
        info["experts"] = {}
        info["idx"] = np.zeros((B, 0), dtype=np.int64)
        info["w"] = np.zeros((B, 0))
        info["margin"] = np.full(B, np.inf)
        return x + attn_out + ffn_out, info

    Wr = _mat(W.router(l))
    r = h @ Wr.T                                              # [B, E]
    info["router_logits"][:] = r
    moe_out = np.zeros((B, d))
    per_expert = {}
    for b in range(B):
        fb = None if forced is None else forced.get(b)
        idx, w, margin = router_topk(r[b], k_top, fb)
        info["idx"].append(idx); info["w"].append(w); info["margin"].append(margin)
        for j, e in enumerate(idx):
            per_expert.setdefault(int(e), []).append((b, j))
    fp8 = cfg.get("expert_dtype") == "fp8"
    for e in sorted(per_expert):
        wg, wu, wd = fp8_expert(*W.expert(l, e)) if fp8 else (_mat(a) for a in W.expert(l, e))
        for b, j in per_expert[e]:
            moe_out[b] += info["w"][b][j] * swiglu_expert(h[b], wg, wu, wd)
    info["experts"] = {e: per_expert[e] for e in sorted(per_expert)}
    info["idx"] = np.array(info["idx"]); info["w"] = np.array(info["w"])
    info["margin"] = np.array(info["margin"])
    return x + attn_out + moe_out, info


def lm_head(cfg, W, x, rows_per_chunk=16384):
    """logits [B, V] = (RMSNorm(x) * g_final) @ Wlm^T."""
    h = rms_norm(x, bf16_to_f64(W.final_norm()), cfg["rms_eps"])
    Wlm = W.lm_head()
    V = Wlm.shape[0]
    out = np.empty((x.shape[0], V))
    for r0 in range(0, V, rows_per_chunk):    # (per-row scales: chunks of rows decode alone)
        out[:, r0:r0 + rows_per_chunk] = h @ _dense(cfg, Wlm[r0:r0 + rows_per_chunk]).T
    return out


def embed(W, tokens):
    return bf16_to_f64(W.embed_rows(tokens))


def decode_step(cfg, W, kv, tokens, seq_lens, page_table, forced=None):
    """One full decode step.  forced maps (l, b) -> expert list.

    Returns dict(logits [B,V], greedy [B], hidden [L+1,B,d], layers=[info per layer])."""
    x = embed(W, tokens)
    hidden = [x]
    layers = []
    for l in range(cfg["n_layers"]):
        fl = None
        if forced:
            fl = {b: e for (ll, b), e in forced.items() if ll == l} or None
        x, info = layer_step(cfg, W, kv, l, x, seq_lens, page_table, fl)
        hidden.append(x)
        layers.append(info)
    logits = lm_head(cfg, W, x)
    greedy = np.array([argmax_lowest(row) for row in logits])
    return dict(logits=logits, greedy=greedy, hidden=np.stack(hidden), layers=layers)


__all__ = ["e4m3_to_f64", "f32_to_e4m3", "quantize_e4m3_rows", "dequantize_e4m3", "fp8_expert", "fp8_matrix",
           "bf16_to_f64", "f64_to_bf16", "rms_norm", "rope", "softmax", "attention",
           "attention_partial", "merge_partials", "router_topk", "silu", "swiglu_expert",
           "window_start", "argmax_lowest", "layer_step", "lm_head", "embed",
           "decode_step", "PAGE"]
