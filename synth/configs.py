"""Workload shapes.

The 2.3B-class dense decoder is the model class the pages measure: a 2.3B
parameter FP16 decoder with 25 layers and context 4096, decoded at batch 1
("Real-time LLM inference on standard GPUs: 3,000 tokens/s per request",
aether-echoes.com reading, sections "どう出したか" (25 layers, 333 µs/token) and
"モデルは 2B・HumanEval 50%" (FP16, context 4096); studioglobal.ai, table
"Laneformer 2B: 実証済みの性能" (2.3B, FP16, batch 1)). Its inner widths, and
the tiny, 8B-class and MoE shapes beside it, are the engine's workload set;
the MoE one follows the pages' projection of the method to FP8 mixture-of-experts
models (hakusoku.com, author reply in "Hackerたちの意見").

Every weight is a seeded std-0.02 normal rounded to its storage dtype;
RMSNorm gains are 1.0.
"""
from __future__ import annotations

import copy

_BASE = dict(
    rms_eps=1e-5,
    rope_theta=10000.0,
    tied_embeddings=True,
    weight_dtype="f16",
    embed_dtype=None,  # embedding, LM head and norm gains: None = weight_dtype
    kv_dtype="f16",
    n_experts=0,
    top_k=0,
    d_expert=0,
    router_dtype="f16",
    expert_dtype="e4m3",
    temperature=0.0,
)


def _cfg(**kw):
    c = dict(_BASE)
    c.update(kw)
    return c


CONFIGS = [
    # 0: tiny dense decoder (L2-resident; parity and latency)
    _cfg(index=0, name="tiny", n_layers=2, d_model=256, n_heads=4, n_kv_heads=2, head_dim=64,
         d_ff=688, vocab=4096, max_ctx=256, prompt_len=16, decode_steps=64),
    # 1: 2.3B-class dense fp16 decoder, greedy, context 513..1024
    _cfg(index=1, name="dense-2.3b-fp16", n_layers=25, d_model=2560, n_heads=20, n_kv_heads=4,
         head_dim=128, d_ff=9728, vocab=32000, max_ctx=4096, prompt_len=512, decode_steps=512),
    # 2: same model, long context 3585..4096, temperature 0.7 sampling
    _cfg(index=2, name="dense-2.3b-fp16-long-t0.7", n_layers=25, d_model=2560, n_heads=20,
         n_kv_heads=4, head_dim=128, d_ff=9728, vocab=32000, max_ctx=4096, prompt_len=3584,
         decode_steps=512, temperature=0.7),
    # 3: 8B-class dense bf16 decoder, untied 128256 vocabulary, theta 5e5
    _cfg(index=3, name="dense-8b-bf16", n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8,
         head_dim=128, d_ff=14336, vocab=128256, max_ctx=8192, rope_theta=500000.0,
         tied_embeddings=False, weight_dtype="bf16", kv_dtype="bf16", prompt_len=1024,
         decode_steps=256),
    # 4: MoE decoder: bf16 attention, fp16 router over 32 e4m3 SwiGLU experts, top-4
    _cfg(index=4, name="moe-32x1408-top4-e4m3", n_layers=24, d_model=2048, n_heads=16,
         n_kv_heads=4, head_dim=128, d_ff=0, vocab=32000, max_ctx=4096, weight_dtype="bf16",
         kv_dtype="bf16", n_experts=32, top_k=4, d_expert=1408, router_dtype="f16",
         expert_dtype="e4m3", prompt_len=256, decode_steps=512),
    # 5: the 2.3B model with fp8 layer weights: every layer matrix e4m3 with per-output-channel
    #    fp32 scales (applied after the dot), embedding / tied LM head and norm gains fp16
    _cfg(index=5, name="dense-2.3b-e4m3", n_layers=25, d_model=2560, n_heads=20, n_kv_heads=4,
         head_dim=128, d_ff=9728, vocab=32000, max_ctx=4096, weight_dtype="e4m3", embed_dtype="f16",
         prompt_len=512, decode_steps=512),
    # 6: the 2.3B model with nvfp4 layer weights (e2m1 elements, an e4m3 scale per 16 consecutive
    #    elements of a row, an fp32 scale per row), embedding / tied LM head and norm gains fp16
    _cfg(index=6, name="dense-2.3b-nvfp4", n_layers=25, d_model=2560, n_heads=20, n_kv_heads=4,
         head_dim=128, d_ff=9728, vocab=32000, max_ctx=4096, weight_dtype="nvfp4", embed_dtype="f16",
         prompt_len=512, decode_steps=512),
    # 7, 8: the 8B model with e4m3 / nvfp4 layer matrices (scales as in 5 and 6); embedding, the
    #    untied LM head and norm gains stay bf16, the KV cache bf16
    _cfg(index=7, name="dense-8b-e4m3", n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8,
         head_dim=128, d_ff=14336, vocab=128256, max_ctx=8192, rope_theta=500000.0,
         tied_embeddings=False, weight_dtype="e4m3", embed_dtype="bf16", kv_dtype="bf16", prompt_len=1024,
         decode_steps=256),
    _cfg(index=8, name="dense-8b-nvfp4", n_layers=32, d_model=4096, n_heads=32, n_kv_heads=8,
         head_dim=128, d_ff=14336, vocab=128256, max_ctx=8192, rope_theta=500000.0,
         tied_embeddings=False, weight_dtype="nvfp4", embed_dtype="bf16", kv_dtype="bf16", prompt_len=1024,
         decode_steps=256),
]

BY_NAME = {c["name"]: c for c in CONFIGS}


def get_config(key) -> dict:
    if isinstance(key, int):
        return copy.deepcopy(CONFIGS[key])
    return copy.deepcopy(BY_NAME[key])


def shrink(cfg: dict, **overrides) -> dict:
    """A small variant of a workload that keeps its code path (dtypes, GQA ratio,
    tying, theta, MoE routing) but with few layers and narrow widths, for fast checks."""
    c = copy.deepcopy(cfg)
    c["name"] = cfg["name"] + "-shrunk"
    group = cfg["n_heads"] // cfg["n_kv_heads"]
    c.update(n_layers=2, d_model=256, head_dim=64, n_kv_heads=2, n_heads=2 * group,
             vocab=2048, max_ctx=256, prompt_len=8, decode_steps=8)
    if cfg["n_experts"]:
        c.update(n_experts=8, top_k=cfg["top_k"], d_expert=192)
    else:
        # nvfp4 matrices keep every reduction length a multiple of 128
        c.update(d_ff=640 if cfg["weight_dtype"] == "nvfp4" else 688)
    c.update(overrides)
    return c


def n_params(cfg: dict) -> int:
    d, hq, hkv, hd, V, L = (cfg[k] for k in ("d_model", "n_heads", "n_kv_heads", "head_dim", "vocab", "n_layers"))
    attn = d * hq * hd * 2 + 2 * d * hkv * hd + 2 * d
    if cfg["n_experts"]:
        ffn = cfg["n_experts"] * 3 * d * cfg["d_expert"] + cfg["n_experts"] * d
    else:
        ffn = 3 * d * cfg["d_ff"]
    emb = V * d * (1 if cfg["tied_embeddings"] else 2)
    return L * (attn + ffn) + emb + d
