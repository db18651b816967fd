"""Workload shapes and storage formats against what the pages print, and the
oracle's whole-path composition on the tiny workload."""

import json
import os

import numpy as np
import torch

import synth
from oracle import csa_oracle as O
from oracle import pipeline as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "v4_attention_shapes.json")


def test_pro_shapes_match_printed_table():
    g = json.load(open(GOLDEN))
    pro = g["pro"]
    for name in ("csa_decode_128k", "csa_prefill_32k", "csa_decode_1m_mixed"):
        c = synth.get(name)
        assert (c["m"], c["H_I"], c["c_I"], c["k"], c["n_h"], c["d"], c["n_win"], c["r"]) == (
            pro["m"], pro["n_h_I"], pro["c_I"], pro["top_k"], pro["n_h"], pro["c"], pro["n_win"],
            g["rope_dims"])
    for name in ("hca_decode_1m", "hca_prefill_64k"):
        c = synth.get(name)
        assert (c["m"], c["n_h"], c["d"], c["n_win"], c["r"]) == (
            pro["m_prime"], pro["n_h"], pro["c"], pro["n_win"], g["rope_dims"])
    assert synth.get("csa_decode_1m_mixed")["N"] == g["csa_candidates_1m"]
    assert synth.get("hca_decode_1m")["N"] == g["hca_entries_1m"]
    assert synth.get("csa_decode_1m_mixed")["L"] == g["context_1m"]


def test_flash_shapes_match_printed_table():
    g = json.load(open(GOLDEN))
    fl = g["flash"]
    for name in ("csa_decode_flash_128k", "csa_prefill_flash_32k"):
        c = synth.get(name)
        assert (c["m"], c["H_I"], c["c_I"], c["k"], c["n_h"], c["d"], c["n_win"], c["r"]) == (
            fl["m"], fl["n_h_I"], fl["c_I"], fl["top_k"], fl["n_h"], fl["c"], fl["n_win"],
            g["rope_dims"])
    # the Flash decode differs from the Pro decode only in heads and top-k
    pro, fla = synth.get("csa_decode_128k"), synth.get("csa_decode_flash_128k")
    diff = {k for k in pro if pro[k] != fla.get(k)}
    assert diff == {"n_h", "k", "name"}


def test_mixed_storage_halves_the_entry_bytes():
    g = json.load(open(GOLDEN))
    c = synth.scaled("csa_decode_1m_mixed", L=1024, B=1)
    x = synth.make_inputs(c)
    d, r = c["d"], c["r"]
    mixed = x["ent_nope"].shape[-1] * 1 + x["ent_rope"].shape[-1] * 2
    assert mixed == (d - r) + 2 * r
    # per-entry scale aside, FP8 + BF16-RoPE storage is ~half of pure BF16
    assert abs(mixed / (2 * d) - g["mixed_kv_vs_bf16"]) < 0.07


def test_quantised_inputs_decode_close_to_source():
    # the encoders round to nearest: decoded FP4 blocks stay within half a code
    # step (relative 1/4 of the block scale * 2) of the source values
    gen = torch.Generator().manual_seed(7)
    v = torch.randn(64, 128, generator=gen) / 11.3
    packed, sf = synth.generate.quantise_fp4_blocks(v)
    dec = O.decode_fp4_blocks(packed.numpy(), sf.numpy())
    scale = np.repeat(O.decode_e4m3(sf.numpy()), 16, axis=-1)
    assert np.all(np.abs(dec - v.double().numpy()) <= scale * 1.0 + 1e-12)
    assert np.all(np.abs(v.double().numpy()) <= 6 * scale + 1e-12)
    e = torch.randn(16, 512, generator=gen)
    nope, s, rope = synth.generate.quantise_mixed_entries(e, 64)
    dec = O.decode_mixed_entries(nope.numpy(), s.numpy(), rope.float().numpy())
    np.testing.assert_allclose(dec, e.double().numpy(), rtol=0.07, atol=0.02 * float(e.abs().max()))


def test_oracle_pipeline_tiny_workload():
    cfg = synth.get("tiny_csa_prefill_f32")
    x = {k: v.numpy() for k, v in synth.make_inputs(cfg).items()}
    rows = [0, 3, 4, 15, 16, 17, 100, 255]
    res = P.run_rows(cfg, x, 0, rows)
    assert res["out"].shape == (len(rows), cfg["n_h"], cfg["d"])
    assert np.all(np.isfinite(res["out"]))
    for i, t in enumerate(rows):
        vis = O.visible_count(t, cfg["m"])
        assert len(res["selected"][i]) == min(cfg["k"], vis)
        assert np.all(res["scores"][i, :vis] >= 0)
    # the attention output of a token is a convex combination (times the sink
    # share) of rotated unit-RMS rows: bounded by the largest row norm
    assert np.abs(res["out"]).max() < 10
