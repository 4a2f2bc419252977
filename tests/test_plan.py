"""The decode step's plan, from the engine itself (adp_plan: host only, no GPU), checked against
the rules the kernels rely on: every tile of every CTA fits one 32 KB ring slot and is a bulk copy
(16-byte aligned start and size), K-chunks start at multiples of 256 elements, regions do not
overlap and add up to the weight image, and the phases come in step order.  For NVFP4 layer
matrices the inside of each tile is replayed: the repack's code and scale bytes of every row
block, and the consumer warps' reads, land on the tile's bytes exactly once."""
import math

import numpy as np
import pytest

import synth

SLOT = 32768
WARPS = 15  # consumer warps per CTA: at most one unit per warp and round
ALIGN = 256
KINDS = {"qkv": 0, "attn": 1, "wo": 2, "gu": 3, "down": 4, "router": 5, "egu": 6, "edown": 7, "lm": 8, "sample": 9}
F16, BF16, E4M3, F32, NVFP4 = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def adp():
    from autoregressive_decode_persistent_gb300 import adp, build
    build.build()
    return adp


def _plan(adp, cfg, n_sms=152):
    from autoregressive_decode_persistent_gb300.model import make_config
    return adp.adp_plan(make_config(cfg), n_sms)


def wbytes(dtype, n):
    """Image bytes of n consecutive elements of one row."""
    if dtype == NVFP4:
        assert n % 16 == 0
        return n // 16 * 9
    return n * {F16: 2, BF16: 2, E4M3: 1, F32: 4}[dtype]


def _cases():
    out = []
    for c in synth.CONFIGS:
        out.append(c)
        out.append(synth.shrink(c))
    out.append(synth.shrink(synth.get_config("dense-2.3b-nvfp4"), n_layers=1, d_model=2560, d_ff=9728))
    out.append(synth.shrink(synth.get_config("tiny"), head_dim=128, n_heads=4, n_kv_heads=2, d_model=384,
                            d_ff=1000))
    return out


CASES = _cases()
IDS = [f'{c["name"]}-{i}' for i, c in enumerate(CASES)]


def _shares(n_units, G, replicated=0):
    """(u0, n) of every CTA: units [floor(c n / G), floor((c + 1) n / G)); a replicated phase gives
    every CTA all units (one shared region of the image)."""
    if replicated:
        return [(0, n_units)] * G
    return [(c * n_units // G, (c + 1) * n_units // G - c * n_units // G) for c in range(G)]


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_phases_come_in_step_order(adp, cfg):
    ph, _ = _plan(adp, cfg)
    L = cfg["n_layers"]
    per_layer = ["qkv", "attn", "wo"] + (["router", "egu", "edown"] if cfg["n_experts"] else ["gu", "down"])
    want = [(KINDS[k], l) for l in range(L) for k in per_layer] + [(KINDS["lm"], L), (KINDS["sample"], L)]
    assert [(p["kind"], p["layer"]) for p in ph] == want


@pytest.mark.parametrize("n_sms", [152, 148, 132])
@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_tiles_fit_one_slot_and_are_bulk_copies(adp, cfg, n_sms):
    ph, _ = _plan(adp, cfg, n_sms)
    for p in ph:
        if p["dtype"] < 0:
            assert p["n_units"] == 0
            continue
        K, KC, upr, ur, s, dt = p["K"], p["KC"], p["upr"], p["unit_rows"], p["slots"], p["dtype"]
        assert KC % ALIGN == 0 and KC > 0 and p["n_chunks"] == math.ceil(K / KC)
        assert 1 <= upr <= WARPS
        # a full round at the full chunk width fills at most one slot, and the next wider chunk
        # would not fit (unless the chunk already spans the whole row)
        assert wbytes(dt, upr * ur * s * KC) <= SLOT
        if KC < math.ceil(K / ALIGN) * ALIGN:
            assert wbytes(dt, upr * ur * s * (KC + ALIGN)) > SLOT
        unit_bytes = wbytes(dt, ur * K)
        for u0, n in set(_shares(p["n_units"], n_sms, p["replicated"])):
            assert (p["region"] + u0 * unit_bytes) % 16 == 0
            if n == 0:
                continue
            pos = 0
            for r in range(math.ceil(n / upr)):
                m = min(upr, n - r * upr)
                for ck in range(p["n_chunks"]):
                    kck = min(KC, K - ck * KC)
                    b = wbytes(dt, m * ur * kck)
                    off = r * upr * unit_bytes + wbytes(dt, m * ur * ck * KC)
                    assert off == pos, "tiles follow one another in consumption order"
                    assert b % 16 == 0 and off % 16 == 0 and 0 < b * s <= SLOT
                    pos += b
            assert pos == n * unit_bytes


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_only_the_router_is_replicated(adp, cfg):
    """Every CTA computes all router logits (its experts are chosen without a hop); every other
    phase splits its units over the CTAs."""
    ph, _ = _plan(adp, cfg)
    for p in ph:
        assert p["replicated"] == (1 if p["kind"] == KINDS["router"] else 0), p


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_regions_are_disjoint_and_make_up_the_image(adp, cfg):
    ph, img = _plan(adp, cfg)
    end = 0
    for p in ph:
        if p["dtype"] < 0:
            continue
        experts = cfg["n_experts"] if p["kind"] in (KINDS["egu"], KINDS["edown"]) else 1
        size = wbytes(p["dtype"], p["n_units"] * p["unit_rows"] * p["K"])
        assert p["region"] == end and p["region"] % ALIGN == 0
        assert p["expert_stride"] == math.ceil(size / ALIGN) * ALIGN
        end += p["expert_stride"] * experts
    assert end == img


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_every_weight_row_is_in_the_plan_once(adp, cfg):
    """The units of each phase cover its matrices' rows: QKV pairs the RoPE halves of every q, k
    and v head, gate|up pairs one gate and one up row, the rest are row groups."""
    ph, _ = _plan(adp, cfg)
    d, hq, hkv, hd = cfg["d_model"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    rows = {KINDS["qkv"]: ((hq + 2 * hkv) * hd, d), KINDS["wo"]: (d, hq * hd), KINDS["lm"]: (cfg["vocab"], d)}
    if cfg["n_experts"]:
        rows.update({KINDS["router"]: (cfg["n_experts"], d), KINDS["egu"]: (2 * cfg["d_expert"], d),
                     KINDS["edown"]: (d, cfg["d_expert"])})
    else:
        rows.update({KINDS["gu"]: (2 * cfg["d_ff"], d), KINDS["down"]: (d, cfg["d_ff"])})
    for p in ph:
        if p["kind"] in rows:
            want_rows, want_k = rows[p["kind"]]
            assert p["n_units"] * p["unit_rows"] == want_rows and p["K"] == want_k, p


def _nvfp4_tile_replay(p, G, ctas):
    """Replay the NVFP4 repack and consumer addressing for the given CTAs of phase p; every byte
    of each CTA's share is written exactly once and every consumer read hits a written byte."""
    K, KC, upr, ur = p["K"], p["KC"], p["upr"], p["unit_rows"]
    unit_bytes = wbytes(NVFP4, ur * K)
    for c in ctas:
        u0 = c * p["n_units"] // G
        n = (c + 1) * p["n_units"] // G - u0
        if n == 0:
            continue
        hits = np.zeros(n * unit_bytes, np.int32)
        lu, j, cb = np.meshgrid(np.arange(n), np.arange(ur), np.arange(K // 16), indexing="ij")
        lu, j, cb = lu.ravel(), j.ravel(), cb.ravel()
        col = cb * 16
        ck = col // KC
        kck = np.minimum(KC, K - ck * KC)
        r, i = lu // upr, lu % upr
        m = np.minimum(upr, n - r * upr)
        tile = r * upr * unit_bytes + m * ur * ck * KC // 16 * 9
        row = i * ur + j
        kc0 = col - ck * KC
        code = tile + row * (kck // 2) + kc0 // 2
        scale = tile + m * ur * (kck // 2) + row * (kck // 16) + kc0 // 16
        tile_end = tile + m * ur * kck // 16 * 9
        assert np.all(code % 8 == 0)
        assert np.all(code + 8 <= tile_end) and np.all(scale < tile_end)
        assert np.all(scale >= tile + m * ur * (kck // 2))
        for b in range(8):
            np.add.at(hits, code + b, 1)
        np.add.at(hits, scale, 1)
        assert hits.min() == 1 and hits.max() == 1
        # consumer warp i reads, for vector v of row j, 4 code bytes and the scale byte of v // 2
        for v_off in (0, 1):
            v = kc0 // 8 + v_off
            rc = tile + (i * ur) * (kck // 2) + j * (kck // 2) + v * 4
            rs = tile + m * ur * (kck // 2) + (i * ur) * (kck // 16) + j * (kck // 16) + v // 2
            assert np.array_equal(rc, code + 4 * v_off) and np.array_equal(rs, scale)


def test_nvfp4_tiles_hold_codes_then_scales(adp):
    cfg = synth.shrink(synth.get_config("dense-2.3b-nvfp4"))
    ph, _ = _plan(adp, cfg)
    dense = [p for p in ph if p["dtype"] == NVFP4]
    assert len(dense) == 4 * cfg["n_layers"]
    for p in dense[:4]:
        _nvfp4_tile_replay(p, 152, range(152))


def test_nvfp4_tiles_at_full_size(adp):
    """The 2.3B widths: multi-chunk rows with ragged last chunks (a sample of CTAs: the first, the
    last, and those whose share size changes)."""
    cfg = synth.get_config("dense-2.3b-nvfp4")
    ph, _ = _plan(adp, cfg)
    layer0 = [p for p in ph if p["dtype"] == NVFP4 and p["layer"] == 0]
    assert max(p["n_chunks"] for p in layer0) >= 4
    for p in layer0:
        sizes = [n for _, n in _shares(p["n_units"], 152)]
        ctas = {0, 151} | {c for c in range(1, 152) if sizes[c] != sizes[c - 1]}
        _nvfp4_tile_replay(p, 152, sorted(ctas)[:6])


def test_plan_rejects_what_the_kernels_cannot_run(adp):
    from autoregressive_decode_persistent_gb300.model import make_config
    cfg = synth.shrink(synth.get_config("dense-2.3b-nvfp4"))
    with pytest.raises(adp.AdpError) as e:
        adp.adp_plan(make_config(dict(cfg, d_ff=704)), 152)  # not a multiple of 128
    assert e.value.code == adp.ADP_ERR_UNSUPPORTED_CONFIG
    with pytest.raises(adp.AdpError) as e:
        adp.adp_plan(make_config(dict(cfg, head_dim=96)), 152)
    assert e.value.code == adp.ADP_ERR_UNSUPPORTED_CONFIG
    with pytest.raises(adp.AdpError) as e:
        adp.adp_plan(make_config(cfg), 0)
    assert e.value.code == adp.ADP_ERR_INVALID_ARG


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_streamed_bytes_are_the_roofline_bytes(adp, cfg):
    """The weight bytes the roofline counts per step (bound.py, from the model's definition) are
    the bytes the plan streams (layer matrices and LM head; for MoE the top-k experts' tiles)
    plus what the kernel reads in place: norm gains, one embedding row, and the fp32 scales."""
    from autoregressive_decode_persistent_gb300 import bound
    ph, _ = _plan(adp, cfg)
    d, hq, hkv, hd, L = cfg["d_model"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["n_layers"]
    ee = 2  # 16-bit embedding, LM head and gains in every workload
    streamed = 0
    for p in ph:
        if p["dtype"] < 0:
            continue
        b = wbytes(p["dtype"], p["n_units"] * p["unit_rows"] * p["K"])
        streamed += b * (cfg["top_k"] if p["kind"] in (KINDS["egu"], KINDS["edown"]) else 1)
    in_place = L * 2 * d * ee + 2 * d * ee  # norm gains, final norm, embedding row
    if cfg["weight_dtype"] in ("e4m3", "nvfp4"):
        in_place += L * (hq * hd + 2 * hkv * hd + d + 2 * cfg["d_ff"] + d) * 4  # row scales
    if cfg["n_experts"]:
        in_place += L * cfg["top_k"] * (2 * cfg["d_expert"] + d) * 4  # expert output-channel scales
    assert streamed + in_place == bound.weight_bytes_per_token(cfg)


@pytest.mark.parametrize("cfg", CASES, ids=IDS)
def test_each_phase_waits_on_the_phases_that_produce_its_inputs(adp, cfg):
    """The step's dataflow, from the model's definition: QKV reads the residual x (layer 0: the
    embedding row, which layer 0's QKV phase publishes as x), attention reads QKV, Wo reads the
    attention output and adds to x, gate|up (or the router and the experts' gate|up) reads x,
    down reads the FFN activations and adds to x, the experts take the router's choice, and the
    LM head reads the last x. Every awaited phase comes earlier in the step."""
    ph, _ = _plan(adp, cfg)
    x_writer = -1  # latest writer of the residual
    router = -1
    for i, p in enumerate(ph):
        k = p["kind"]
        want = {KINDS["qkv"]: (x_writer, -1, -1), KINDS["lm"]: (x_writer, -1, -1), KINDS["sample"]: (-1, -1, -1)}
        if k == KINDS["attn"]:
            want[k] = (i - 1, -1, -1)
        elif k == KINDS["wo"]:
            want[k] = (i - 1, x_writer, -1)
        elif k in (KINDS["gu"], KINDS["router"]):
            want[k] = (x_writer, -1, -1)
        elif k == KINDS["egu"]:
            want[k] = (x_writer, -1, router)
        elif k in (KINDS["down"], KINDS["edown"]):
            want[k] = (i - 1, x_writer, router if k == KINDS["edown"] else -1)
        assert (p["src_phase"], p["res_phase"], p["sel_phase"]) == want[k], (i, p)
        assert all(j < i for j in (p["src_phase"], p["res_phase"], p["sel_phase"]))
        if k == KINDS["qkv"] and p["layer"] == 0:
            x_writer = i  # x = the embedding row, published by layer 0's QKV phase
        elif k in (KINDS["wo"], KINDS["down"], KINDS["edown"]):
            x_writer = i
        elif k == KINDS["router"]:
            router = i


GB300_SMEM_OPTIN = 232448  # opt-in shared memory per block on sm_103 (227 KB)


@pytest.mark.parametrize("name", ["tiny", "dense-2.3b-fp16", "dense-2.3b-nvfp4", "dense-8b-bf16", "dense-8b-nvfp4",
                                  "moe-32x1408-top4-e4m3"])
def test_batch_layouts_fit_and_segment_only_when_needed(adp, name):
    """The batched kernel's shared-memory layout per batch size (adp_batch_plan, the same function
    the first batched call runs): every batch that fits has a ring of at least two 32 KB slots and
    a staging area holding every request's input vector (the down projection's whole, or a segment
    of whole K-chunks), all within the opt-in limit; the down input is segmented only when whole
    vectors beside a two-slot ring would not fit; with whole vectors the ring is as deep as the
    limit allows.  MoE models are not batched."""
    import synth
    from autoregressive_decode_persistent_gb300.model import make_config
    cfg = synth.get_config(name)
    lay, max_nb = adp.adp_batch_plan(make_config(cfg), 152, GB300_SMEM_OPTIN)
    if cfg["n_experts"]:
        assert max_nb == 0 and all(o["ring_slots"] == 0 for o in lay)
        return
    assert max_nb >= 1
    phases, _ = _plan(adp, cfg)
    down_kc = next(P["KC"] for P in phases if P["kind"] == 4)
    pad = lambda n: (n + 255) // 256 * 256
    d, hq, hd, ff = cfg["d_model"], cfg["n_heads"], cfg["head_dim"], cfg["d_ff"]
    for nb in range(1, 5):
        o = lay[nb - 1]
        if nb > max_nb:
            assert o["ring_slots"] == 0
            continue
        assert 2 <= o["ring_slots"] <= 6 and o["attention_slots"] >= 1
        assert o["smem_bytes"] == o["ring_slots"] * 32768 + o["xbuf_floats"] * 4 + o["control_bytes"]
        assert o["smem_bytes"] <= GB300_SMEM_OPTIN
        seg = o["down_segment"]
        assert seg == ff or (seg % down_kc == 0 and seg < ff)
        assert o["xbuf_floats"] >= nb * max(pad(d), pad(hq * hd), pad(seg))
        whole = nb * max(pad(d), pad(hq * hd), pad(ff)) * 4 + 2 * 32768 + o["control_bytes"]
        if seg < ff:
            assert whole > GB300_SMEM_OPTIN  # whole vectors would not have fit
        else:
            assert o["ring_slots"] == 6 or o["smem_bytes"] + 32768 > GB300_SMEM_OPTIN
    if name == "dense-2.3b-fp16":
        # three whole inputs (3 x 38.9 KB); four only in two segments of 7 K-chunks of 768
        assert max_nb == 4
        assert [o["down_segment"] for o in lay] == [ff, ff, ff, 7 * 768]
