"""Pin of the oracle's forced-expert branch (no GPU).

When the experts of a layer are forced (the teacher-forcing hook of MoE parity), the step uses the
forced experts with the router's softmax probabilities of those experts, renormalised over the
forced set (the routing stage of the step: hakusoku.com, "標準GPUによるリアルタイムLLM推論",
section "Kog Inference Engineの特徴とイノベーション"; the top-k gate renormalisation of the MoE
configuration).  The float64 brute force, which recomputes the whole prefix with NumPy and shares
no code with oracle.c, applies the same forced choices; both oracle modes must agree with it within
1e-4 on every position.

Planted mistakes (mutated copies of oracle.c compiled into a temporary directory, never the
oracle itself): gates taken from the router's own top-k instead of the forced experts, and gates
left unnormalised (the plain probabilities) must both fail the same check."""
import os

import numpy as np
import pytest

import synth
from oracle import EXACT, PLAIN, OracleModel, brute
from oracle import oracle as orc

FORCED_GATES = "for (int i = 0; i < K; ++i) gate[i] = P[sel[i]] / Zs;"


def _forced(cfg, W, n_pos):
    """For each position and layer, top_k distinct experts drawn from a seeded permutation."""
    E, K, L = cfg["n_experts"], cfg["top_k"], cfg["n_layers"]
    assert 2 * K <= E
    rng = np.random.default_rng(7)
    out = np.zeros((n_pos, L, K), dtype=np.int32)
    for t in range(n_pos):
        for l in range(L):
            out[t, l] = rng.permutation(E)[:K]
    return out


def _run(cfg, W, toks, force, mode, library=None):
    m = OracleModel(cfg, W, library=library)
    lg = []
    for t, tok in enumerate(toks):
        r = m.step(int(tok), mode, force=force[t])  # r["experts"]: the router's own (unforced) choice
        lg.append(r["logits"])
    return np.array(lg, dtype=np.float64)


@pytest.fixture(scope="module")
def moe():
    # fp16 KV storage: with the model's bf16 cache, about 0.5% of stored K/V elements round one bf16
    # ulp differently in fp32 and float64 arithmetic, which alone moves the logits by ~1e-4; with
    # fp16 (three more fraction bits) the check below measures the branch, not the storage rounding.
    cfg = synth.shrink(synth.get_config("moe-32x1408-top4-e4m3"), kv_dtype="f16")
    W = synth.model_weights(cfg)
    toks = [int(t) for t in synth.prompt(cfg, 12)]
    force = _forced(cfg, W, len(toks))
    bl, broutes = brute.forward(cfg, W, toks, force=force)
    return cfg, W, toks, force, bl


def test_forced_experts_match_the_brute_force(moe):
    cfg, W, toks, force, bl = moe
    for mode in (PLAIN, EXACT):
        lg = _run(cfg, W, toks, force, mode)
        assert np.max(np.abs(lg - bl)) < 1e-4, mode


def test_forcing_changes_the_result(moe):
    """The forced experts are not the router's own: unforced logits differ far beyond the tolerance,
    so the check above exercises the branch."""
    cfg, W, toks, force, bl = moe
    free, _ = brute.forward(cfg, W, toks)
    assert np.max(np.abs(free - bl)) > 1e-2


@pytest.mark.parametrize("mutation", [
    # gates of the router's own top-k, applied to the forced experts
    "(void)Zs;",
    # probabilities of the forced experts, not renormalised over them
    "for (int i = 0; i < K; ++i) gate[i] = P[sel[i]];",
])
def test_planted_mistakes_in_the_branch_fail(moe, tmp_path, mutation):
    cfg, W, toks, force, bl = moe
    src = open(os.path.join(os.path.dirname(orc.__file__), "oracle.c")).read()
    assert src.count(FORCED_GATES) == 1
    bad = tmp_path / "oracle_mutant.c"
    bad.write_text(src.replace(FORCED_GATES, mutation))
    lib = orc.load(orc.compile_c(str(bad), str(tmp_path / "liboracle_mutant.so")))
    lg = _run(cfg, W, toks, force, PLAIN, library=lib)
    assert np.max(np.abs(lg - bl)) > 1e-2
