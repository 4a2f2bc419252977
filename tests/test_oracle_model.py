"""Whole-step pins of the CPU oracle: the float64 brute force (no KV cache, the full prefix
recomputed at every position) against the oracle's plain and exact modes (no GPU)."""
import numpy as np
import pytest

import synth
from oracle import EXACT, PLAIN, OracleModel, brute


def run_oracle(cfg, W, tokens_in, n_decode, mode, force=None):
    """Prefill tokens_in, then n_decode greedy steps. Returns (tokens, logits per position, model)."""
    m = OracleModel(cfg, W)
    toks = [int(t) for t in tokens_in]
    logits, routes = [], []
    out = None
    for i, t in enumerate(toks):
        out = m.step(t, mode)
        logits.append(out["logits"])
        routes.append(out.get("experts"))
    for _ in range(n_decode):
        t = out["next"]
        toks.append(t)
        out = m.step(t, mode)
        logits.append(out["logits"])
        routes.append(out.get("experts"))
    return toks, np.array(logits), routes, m


def check_against_brute(cfg, n_prompt, n_decode, tol=1e-4):
    W = synth.model_weights(cfg)
    prompt = synth.prompt(cfg, n_prompt)
    toks, lp, routes, mp = run_oracle(cfg, W, prompt, n_decode, PLAIN)
    toks_e, le, routes_e, me = run_oracle(cfg, W, prompt, n_decode, EXACT)
    # teacher forcing: both oracle modes and the brute force run on the plain mode's tokens
    bl, broutes = brute.forward(cfg, W, toks[:-1] + [toks[-1]])
    assert np.max(np.abs(lp - bl[: len(lp)])) < tol
    if toks_e == toks:
        assert np.max(np.abs(le - bl[: len(le)])) < tol
        assert np.max(np.abs(le - lp)) < tol
    # greedy decisions agree wherever the float64 top-2 margin is not razor thin
    for i in range(len(lp)):
        top2 = np.sort(bl[i])[-2:]
        if top2[1] - top2[0] > 1e-3:
            assert int(np.argmax(lp[i])) == int(np.argmax(bl[i]))
    if cfg["n_experts"]:
        for pos in range(len(routes)):
            assert np.array_equal(np.sort(routes[pos], axis=1), np.sort(broutes[pos], axis=1))
    return mp, me


def test_tiny_against_brute_force():
    cfg = synth.get_config("tiny")
    mp, me = check_against_brute(cfg, cfg["prompt_len"], cfg["decode_steps"])
    # KV rows: exact and plain differ only in rare last-bit roundings
    n = cfg["prompt_len"] + cfg["decode_steps"]
    diff = np.mean(mp.kc[:, :, :n] != me.kc[:, :, :n])
    assert diff < 0.05


@pytest.mark.parametrize("name", ["dense-2.3b-fp16", "dense-8b-bf16", "moe-32x1408-top4-e4m3", "dense-2.3b-e4m3",
                                  "dense-2.3b-nvfp4", "dense-8b-e4m3", "dense-8b-nvfp4"])
def test_shrunk_workloads_against_brute_force(name):
    over = {}
    if name in ("dense-8b-e4m3", "dense-8b-nvfp4"):
        # fp16 KV storage: a bf16 cache element that fp32 and float64 arithmetic round one ulp apart
        # moves these logits by ~1e-4 by itself; the bf16 cache path is pinned by dense-8b-bf16
        over["kv_dtype"] = "f16"
    cfg = synth.shrink(synth.get_config(name), **over)
    check_against_brute(cfg, 8, 24)


@pytest.mark.parametrize("overrides", [{"embed_dtype": "bf16"}, {"tied_embeddings": False},
                                       {"head_dim": 128, "n_heads": 4, "n_kv_heads": 4, "d_model": 512}])
def test_nvfp4_variants_against_brute_force(overrides):
    """NVFP4 layer matrices with a bf16 embedding / LM head / gains, with an untied LM head, and
    with 128-wide heads (MHA): the paths around the 4-bit matrices the 2.3B case does not take."""
    cfg = synth.shrink(synth.get_config("dense-2.3b-nvfp4"), **overrides)
    check_against_brute(cfg, 8, 12)


def test_multi_head_attention_variant_against_brute_force():
    cfg = synth.shrink(synth.get_config("tiny"), n_kv_heads=4, n_heads=4)
    check_against_brute(cfg, 8, 16)


def test_single_kv_head_long_block_tail_against_brute_force():
    # one KV head for 6 query heads, 77 positions: several 32-position blocks and a ragged tail
    cfg = synth.shrink(synth.get_config("tiny"), n_kv_heads=1, n_heads=6)
    check_against_brute(cfg, 40, 37)


def test_oracle_rejects_position_beyond_context():
    cfg = synth.shrink(synth.get_config("tiny"), max_ctx=8)
    m = OracleModel(cfg, synth.model_weights(cfg))
    for t in range(8):
        m.step(t)
    with pytest.raises(RuntimeError):
        m.step(1)
