"""Bytes per decoded token and the bandwidth bound on batch-1 decode speed.

At batch 1 every generated token streams every active weight, plus the KV cache
it attends over, through HBM, so decode speed is bounded by

    tokens/s <= effective bandwidth / (beta * active parameters + KV bytes)

with beta the bytes per parameter ("Real-time LLM inference on standard GPUs:
3,000 tokens/s per request", hakusoku.com summary, section
"GPU推論の速度制限要因：メモリ帯域幅"). The pages' own numbers (a 2B FP16 model
of about 4 GB on 8xH200 at ~30.7 TB/s and 8xMI300X at ~33.6 TB/s giving
7,700-8,400 tokens/s) fix beta as bytes per parameter; for mixed precision the
product is the byte count of every active tensor, which is what
`bytes_per_token` adds up exactly for a workload configuration.

The same pages model the multi-kernel stack's launch cost (4.5 µs x 10 kernels x
25 layers = 1,125 µs per token, a cap of about 890 tokens/s; section
"標準推論スタックのボトルネックとKogの工夫") and the per-token and per-layer
budgets at 3,000 tokens/s (333 µs and 13.3 µs over 25 layers; aether-echoes.com
reading, section "どう出したか").
"""
from __future__ import annotations

_EB = {"f16": 2, "bf16": 2, "e4m3": 1, "f32": 4}


def page_bound(bandwidth_bytes_per_s: float, active_params: float, beta_bytes_per_param: float,
               kv_bytes: float = 0.0) -> float:
    """tokens/s <= BW / (beta * active params + KV bytes)."""
    return bandwidth_bytes_per_s / (beta_bytes_per_param * active_params + kv_bytes)


def launch_overhead_per_token_s(launch_s: float, kernels_per_layer: int, layers: int) -> float:
    return launch_s * kernels_per_layer * layers


def per_token_budget_s(tokens_per_s: float) -> float:
    return 1.0 / tokens_per_s


def generation_time_s(n_tokens: float, tokens_per_s: float) -> float:
    return n_tokens / tokens_per_s


def weight_bytes_per_token(cfg: dict) -> int:
    """Bytes of every weight one decode step reads once: all layer weights (for MoE the
    attention, router, norms and top-k experts with their fp32 scales), the LM head, one
    embedding row and the final norm gain."""
    c = cfg
    fp4 = c["weight_dtype"] == "nvfp4"    # half a byte per element + one e4m3 scale per 16 elements
    q8 = c["weight_dtype"] in ("e4m3", "nvfp4")  # layer matrices with an fp32 scale per row
    ee = _EB[c.get("embed_dtype") or c["weight_dtype"]]  # embedding, LM head, norm gains

    def mb(n_elems: int) -> int:
        """Bytes of n_elems layer-matrix elements."""
        return n_elems * 9 // 16 if fp4 else n_elems * _EB[c["weight_dtype"]]

    d, hq, hkv, hd, V = c["d_model"], c["n_heads"], c["n_kv_heads"], c["head_dim"], c["vocab"]
    attn = mb(hq * hd * d * 2 + 2 * hkv * hd * d) + ((hq * hd + 2 * hkv * hd + d) * 4 if q8 else 0)
    norms = 2 * d * ee
    if c["n_experts"]:
        f, k = c["d_expert"], c["top_k"]
        xeb = _EB[c["expert_dtype"]]
        router = c["n_experts"] * d * _EB[c["router_dtype"]]
        experts = k * (3 * f * d * xeb + (2 * f + d) * 4)
        ffn = router + experts
    else:
        ffn = mb(3 * c["d_ff"] * d) + ((2 * c["d_ff"] + d) * 4 if q8 else 0)
    per_layer = attn + norms + ffn
    head = V * d * ee
    return c["n_layers"] * per_layer + head + d * ee + d * ee


def kv_read_bytes(cfg: dict, context: int) -> int:
    """K and V of positions 0..context-1 for every layer (the new row included)."""
    return 2 * cfg["n_layers"] * cfg["n_kv_heads"] * cfg["head_dim"] * _EB[cfg["kv_dtype"]] * context


def kv_write_bytes(cfg: dict) -> int:
    return 2 * cfg["n_layers"] * cfg["n_kv_heads"] * cfg["head_dim"] * _EB[cfg["kv_dtype"]]


def bytes_per_token(cfg: dict, context: int) -> int:
    """Algorithmic HBM bytes of one decode step that ends with `context` cached positions."""
    return weight_bytes_per_token(cfg) + kv_read_bytes(cfg, context) + kv_write_bytes(cfg)


def mean_bytes_per_token(cfg: dict, first_context: int, n_steps: int) -> float:
    """Average over steps whose contexts are first_context, first_context + 1, ..."""
    w = weight_bytes_per_token(cfg) + kv_write_bytes(cfg)
    per_pos = kv_read_bytes(cfg, 1)
    mean_ctx = first_context + (n_steps - 1) / 2.0
    return w + per_pos * mean_ctx


def batch_step_bytes(cfg: dict, contexts) -> int:
    """Algorithmic HBM bytes of one batched decode step: every weight once for the whole batch,
    plus each request's KV cache up to its own context and its new KV row."""
    return weight_bytes_per_token(cfg) + sum(kv_read_bytes(cfg, c) + kv_write_bytes(cfg) for c in contexts)


def mean_batch_step_bytes(cfg: dict, nb: int, first_context: int, n_steps: int) -> float:
    """Average batched-step bytes over steps in which all nb requests sit at contexts
    first_context, first_context + 1, ..."""
    mean_ctx = first_context + (n_steps - 1) / 2.0
    return weight_bytes_per_token(cfg) + nb * (kv_write_bytes(cfg) + kv_read_bytes(cfg, 1) * mean_ctx)


def roofline_tokens_per_s(cfg: dict, context: float, bandwidth_bytes_per_s: float) -> float:
    w = weight_bytes_per_token(cfg) + kv_write_bytes(cfg)
    return bandwidth_bytes_per_s / (w + kv_read_bytes(cfg, 1) * context)
