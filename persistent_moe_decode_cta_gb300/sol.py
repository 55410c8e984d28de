"""Speed-of-light arithmetic for one decode step.

The pages define speed of light as the bytes a decode step must stream (active
weights plus the KV cache read) divided by the HBM bandwidth
[Cohere's Open-Source Megakernel Beats vLLM by 1.58x on H100, "Why decode leaves the
GPU idle"; Fuse decode into one megakernel for 1.58x higher H100 throughput, "Where
the bandwidth actually goes"].  This module counts those bytes for a model shape and
a batch: every dense weight once, the union of experts the batch routed to at each
layer, the LM head, the embedding rows actually read, the cached K/V each token
attends to, and the step's writes (new K/V slots and fp32 logits).
"""
from __future__ import annotations

BF16 = 2


def param_counts(cfg: dict) -> dict:
    """Total parameters, and the per-token active ones (top-k experts) with and
    without the full embedding table."""
    L, d, Hq, Hkv, hd = (cfg[k] for k in ("n_layers", "d_model", "n_q_heads",
                                          "n_kv_heads", "head_dim"))
    E, k, f, V = cfg["n_experts"], cfg["top_k"], cfg["d_ff"], cfg["vocab"]
    dense_layer = d * (Hq + 2 * Hkv) * hd + Hq * hd * d + d * E + d
    expert = 3 * d * f
    total = L * (dense_layer + E * expert) + 2 * V * d + d
    active_no_embed = L * (dense_layer + k * expert) + V * d + d
    return dict(total=total, active_with_embedding=active_no_embed + V * d,
                active_step=active_no_embed, dense_layer=dense_layer, expert=expert)


def expert_bytes(cfg: dict) -> int:
    """Bytes of one routed expert: bf16 matrices, or (expert_dtype "fp8") E4M3 codes
    plus one float32 scale per row of gate, up and down."""
    d, f = cfg["d_model"], cfg["d_ff"]
    if cfg.get("expert_dtype", "bf16") == "fp8":
        return 3 * d * f + 4 * (2 * f + d)
    return BF16 * 3 * d * f


def attended_cached_keys(p: int, window: int) -> int:
    """Cached keys (positions < p) read by a token at position p."""
    lo = 0 if window <= 0 else max(0, p - window + 1)
    return p - lo


def step_bytes(cfg: dict, seq_lens, union_sizes) -> dict:
    """Algorithmic bytes of one decode step.

    seq_lens: cached length per sequence (= the new token's position).
    union_sizes: distinct experts routed to at each layer (len n_layers)."""
    L, d, Hkv, hd = cfg["n_layers"], cfg["d_model"], cfg["n_kv_heads"], cfg["head_dim"]
    V, f = cfg["vocab"], cfg["d_ff"]
    B = len(seq_lens)
    pc = param_counts(cfg)
    # a dense layer of a mixed stack reads its FFN instead of a router and experts
    dense = set(cfg.get("dense_layers", ()))
    n_dense = sum(1 for l in range(L) if l in dense)
    routed_union = sum(u for l, u in enumerate(union_sizes) if l not in dense)
    dense_ffn = 3 * d * cfg.get("dense_ff", 0)
    weights = BF16 * (L * pc["dense_layer"] - n_dense * d * cfg["n_experts"]
                      + n_dense * dense_ffn + V * d + d + B * d) + routed_union * expert_bytes(cfg)
    if cfg.get("dense_dtype", "bf16") == "fp8":
        # QKV, O-proj and LM head as E4M3 codes plus a float32 scale per row (router,
        # norms and embedding stay bf16)
        Hq = cfg["n_q_heads"]
        qkv_rows, o_rows = (Hq + 2 * Hkv) * hd, d
        fp8_elems = L * (qkv_rows * d + o_rows * Hq * hd) + V * d
        weights += (1 - BF16) * fp8_elems + 4 * (L * (qkv_rows + o_rows) + V)
    swa = set(cfg.get("swa_layers", ()))
    kv_read = 0
    for p in seq_lens:
        for l in range(L):
            w = cfg.get("sliding_window", 0) if l in swa else 0
            kv_read += 2 * Hkv * hd * BF16 * attended_cached_keys(p, w)
    writes = B * L * 2 * Hkv * hd * BF16 + B * V * 4
    return dict(weights=weights, kv=kv_read, writes=writes,
                total=weights + kv_read + writes)


def sol_seconds(nbytes: float, bw_bytes_per_s: float) -> float:
    return nbytes / bw_bytes_per_s


def sol_tok_s(nbytes: float, bw_bytes_per_s: float, batch: int = 1) -> float:
    """Tokens per second at speed of light: batch tokens per step."""
    return batch * bw_bytes_per_s / nbytes
