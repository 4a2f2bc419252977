"""Shared drivers for the GPU parity tests: run the engine (through the C ABI) and the CPU
oracle on the same seeded inputs, teacher-forced on the oracle's token stream."""
from __future__ import annotations

import numpy as np

import synth
from oracle import EXACT, PLAIN, OracleModel

# Parity tolerances of the engine's logits against the plain fp32 oracle, per step.
LOGIT_MAX_ABS = 2e-2
LOGIT_REL_L2 = 5e-3
ARGMAX_MARGIN = 0.05


def oracle_free_run(cfg, W, prompt, n_decode, mode=EXACT, temperature=0.0, us=None, kv_prefix=None):
    """Oracle run: prompt, then n_decode steps fed with its own choices.
    Returns (input tokens per step, logits per step, next token per step, oracle model)."""
    m = OracleModel(cfg, W)
    if kv_prefix is not None:
        m.load_kv_prefix(*kv_prefix)
    toks, logits, nexts, experts = [], [], [], []
    seq = [int(t) for t in prompt]
    i = 0
    while True:
        t = seq[i]
        u = float(us[i]) if us is not None else 0.0
        out = m.step(t, mode, temperature=temperature, u=u)
        toks.append(t)
        logits.append(out["logits"])
        nexts.append(out["next"])
        experts.append(out.get("experts"))
        if i + 1 >= len(seq):
            if len(seq) - len(prompt) >= n_decode:
                break
            seq.append(out["next"])
        i += 1
    return toks, np.array(logits), nexts, experts, m


def oracle_forced(cfg, W, toks, mode=PLAIN, temperature=0.0, us=None, kv_prefix=None):
    m = OracleModel(cfg, W)
    if kv_prefix is not None:
        m.load_kv_prefix(*kv_prefix)
    logits, nexts = [], []
    for i, t in enumerate(toks):
        out = m.step(t, mode, temperature=temperature, u=float(us[i]) if us is not None else 0.0)
        logits.append(out["logits"])
        nexts.append(out["next"])
    return np.array(logits), nexts, m


def engine_forced(model, toks, temperature=0.0, us=None, kv_prefix=None, read_experts=False):
    """Engine run through adp_decode_step, one step per input token."""
    import torch
    cfg = model.cfg
    kv = model.new_kv()
    if kv_prefix is not None:
        kv.load(*kv_prefix)
    lg = torch.empty(cfg["vocab"], dtype=torch.float32, device=model.device)
    logits, nexts, experts = [], [], []
    for i, t in enumerate(toks):
        nxt = kv.step(int(t), temperature, float(us[i]) if us is not None else 0.0, lg)
        logits.append(lg.cpu().numpy().copy())
        nexts.append(nxt)
        if read_experts:
            from autoregressive_decode_persistent_gb300 import adp
            experts.append(adp.adp_debug_read_experts(model.handle, cfg["n_layers"], cfg["top_k"]))
    k, v = kv.read()
    kv.close()
    return np.array(logits), nexts, k, v, experts


def assert_logits_within_tolerance(got, ref):
    for i in range(len(ref)):
        d = got[i].astype(np.float64) - ref[i]
        assert np.max(np.abs(d)) <= LOGIT_MAX_ABS, (i, np.max(np.abs(d)))
        assert np.linalg.norm(d) / np.linalg.norm(ref[i].astype(np.float64)) <= LOGIT_REL_L2, i
        top2 = np.sort(ref[i])[-2:]
        if top2[1] - top2[0] > ARGMAX_MARGIN:
            assert int(np.argmax(got[i])) == int(np.argmax(ref[i])), i


def kv_used(k, v, n):
    return k[:, :, :n], v[:, :, :n]


def seeded_model(cfg):
    return synth.model_weights(cfg)
