"""Pins of the oracle's whole-path composition (``oracle/pipeline.py``).

``run_rows``, ``entries_of``, ``window_of`` and ``indexer_inputs`` map query
rows to positions, pick each sequence's window rows and decode the stored
formats.  Each test below checks them against something that does not come
from the oracle (DeepSeek-V4 report, Chinese translation, blog.uika.cn,
§2.3.1 visibility rule and top-k selector, §2.3.3 window and sink, §2.3.4
storage formats):

* a second, independently written brute-force forward (tests/brute_force.py)
  on tiny CSA / HCA prefill and decode workloads, decode batches at mixed
  context lengths and the FP8 / FP4 storage formats;
* closed forms: identical keys with unit head weights make every visible score
  equal, so the selection is the lowest indices and the finite-score pattern is
  exactly (s+1)m <= t+1; a zero query makes every logit 0, so with one-hot
  window rows the output shows exactly which tokens the window took, and the
  denominator shows how many rows the query attended;
* invariants: moving the query, every entry and every window token by the same
  multiple of m leaves scores, selection (shifted) and output unchanged; a
  b-row of block j reaches compressed entry j+1 only, an a-row entry j only;
* the stored formats decode to within their rounding step of the float
  values they were quantised from.
"""

import numpy as np
import pytest

import synth
from oracle import csa_oracle as O
from oracle import pipeline as OP
from tests import brute_force as BF


def _np(x):
    return {k: v.float().numpy() if v.is_floating_point() else v.numpy() for k, v in x.items()}


TINY = {
    "csa_prefill": ("tiny_csa_prefill_f32", dict(T=64, d=32, r=8, n_h=2, H_I=3, c_I=8, k=5, n_win=6)),
    "hca_prefill": ("hca_prefill_64k", dict(T=300, m=16, d=32, r=8, n_h=2, n_win=6)),
    "csa_decode": ("csa_decode_128k", dict(B=3, lengths=[41, 30, 9], d=32, r=8, n_h=2, H_I=3,
                                            c_I=16, k=4, n_win=5)),
    "csa_decode_mixed": ("csa_decode_1m_mixed", dict(B=2, lengths=[70, 33], d=48, r=16, n_h=2,
                                                     H_I=2, c_I=32, k=5, n_win=6)),
    "hca_decode": ("hca_decode_1m", dict(B=2, lengths=[200, 60], m=16, d=32, r=8, n_h=2, n_win=7)),
}


@pytest.mark.parametrize("case", sorted(TINY))
def test_pipeline_matches_independent_brute_force(case):
    name, over = TINY[case]
    cfg = synth.scaled(name, **over)
    x = _np(synth.make_inputs(cfg, seed=1))
    rows = list(range(cfg["Tq"]))
    for b in range(cfg["B"]):
        res = OP.run_rows(cfg, x, b, rows)
        bf = BF.run(cfg, x, b, rows)
        for i, (sc, sel, out) in enumerate(bf):
            np.testing.assert_allclose(res["out"][i], np.array(out), rtol=1e-10, atol=1e-12,
                                       err_msg=f"{case} b={b} row {i} output")
            if sc is None:
                continue
            got = res["scores"][i]
            fin = np.isfinite(got)
            assert sorted(np.nonzero(fin)[0].tolist()) == sorted(sc), f"{case} visible set"
            np.testing.assert_allclose(got[fin], [sc[s] for s in np.nonzero(fin)[0]],
                                       rtol=1e-11, atol=1e-14)
            assert sorted(res["selected"][i].tolist()) == sel, f"{case} b={b} row {i} top-k"


def _decode_cfg(lengths, **over):
    base = dict(B=len(lengths), lengths=lengths, d=64, r=16, n_h=2, H_I=4, c_I=16, k=6, n_win=6)
    base.update(over)
    return synth.scaled("csa_decode_128k", **base)


def test_pipeline_equal_keys_select_lowest_visible_indices():
    # t = 4v-1 sees v entries, t = 4v-2 sees v-1: an off-by-one in the row ->
    # position map changes the visible count of one of them
    v = 37
    cfg = _decode_cfg([4 * v, 4 * v - 1, 10], k=8)
    x = _np(synth.make_inputs(cfg, seed=2))
    x["K"][:] = x["K"][:, :1]                # every key equals key 0 of its sequence
    x["w"][:] = 1.0
    for b, L in enumerate(cfg["lengths"]):
        t = L - 1
        vis = (t + 1) // cfg["m"]
        res = OP.run_rows(cfg, x, b, [0])
        s = res["scores"][0]
        assert int(res["t"][0]) == t
        assert np.all(np.isfinite(s[:vis])) and np.all(np.isneginf(s[vis:]))
        want = sum(max(0.0, float(np.dot(x["qI"][b, 0, h].astype(np.float64),
                                         x["K"][b, 0].astype(np.float64))))
                   for h in range(cfg["H_I"]))
        np.testing.assert_allclose(s[:vis], want, rtol=1e-12)
        assert sorted(res["selected"][0].tolist()) == list(range(min(cfg["k"], vis)))


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_pipeline_window_is_exactly_the_last_n_win_tokens(kind):
    # zero query: every logit is 0, so out = sum of the attended rows / (J + e^sink).
    # Entries are zero; window token p is one-hot on channel p - base of a buffer
    # that holds 4 more tokens than the window, so the lit channels name the
    # attended tokens and their common value names J, the number of rows.
    n_win, extra = 6, 4
    if kind == "csa":
        cfg = _decode_cfg([90, 23], n_win=n_win)
    else:
        cfg = synth.scaled("hca_decode_1m", B=2, lengths=[90, 23], m=16, d=64, r=16, n_h=2,
                           n_win=n_win)
    x = _np(synth.make_inputs(cfg, seed=3))
    d, r = cfg["d"], cfg["r"]
    T_win = n_win + extra
    x["q"][:] = 0.0
    if "entries" in x:
        x["entries"][:] = 0.0
    x["win"] = np.zeros((cfg["B"], T_win, d), dtype=np.float32)
    for j in range(T_win):
        x["win"][:, j, j] = 1.0               # channel j < d - r: outside the RoPE dims
    assert T_win <= d - r
    for b, L in enumerate(cfg["lengths"]):
        t = L - 1
        x["win_base"][b] = t - T_win + 1      # the buffer ends at the query's token
        res = OP.run_rows(cfg, x, b, [0])
        vis = (t + 1) // cfg["m"]
        J = (min(cfg["k"], vis) if kind == "csa" else vis) + n_win
        lit = np.arange(extra, T_win)         # tokens t-n_win+1 .. t
        for h in range(cfg["n_h"]):
            want = np.zeros(d)
            want[lit] = 1.0 / (J + np.exp(float(x["sink"][h])))
            np.testing.assert_allclose(res["out"][0, h], want, atol=1e-15, rtol=1e-12)


def test_pipeline_shift_by_whole_blocks_is_invisible():
    # prepend delta entries whose keys score exactly 0 (zero vectors), and move
    # the query, the window tokens and every real entry by m*delta positions:
    # scores and selection shift by delta, the output does not change
    # (RoPE depends on position differences only)
    delta = 3
    cfg = _decode_cfg([97], H_I=8, k=5)
    x = _np(synth.make_inputs(cfg, seed=4))
    m = cfg["m"]
    base = OP.run_rows(cfg, x, 0, [0])
    cfg2 = dict(cfg, N=cfg["N"] + delta, lengths=[97 + m * delta], L=97 + m * delta)
    x2 = dict(x)
    rng = np.random.default_rng(0)
    x2["entries"] = np.concatenate([rng.standard_normal((1, delta, cfg["d"])).astype(np.float32),
                                    x["entries"]], axis=1)
    x2["K"] = np.concatenate([np.zeros((1, delta, cfg["c_I"]), np.float32), x["K"]], axis=1)
    x2["q_pos"] = x["q_pos"] + m * delta
    x2["win_base"] = x["win_base"] + m * delta
    moved = OP.run_rows(cfg2, x2, 0, [0])
    assert np.all(moved["scores"][0, :delta] == 0.0)
    np.testing.assert_allclose(moved["scores"][0, delta:], base["scores"][0], rtol=1e-13)
    assert np.min(base["scores"][0][np.isfinite(base["scores"][0])][base["selected"][0]]) > 0
    assert sorted(moved["selected"][0].tolist()) == sorted((base["selected"][0] + delta).tolist())
    np.testing.assert_allclose(moved["out"], base["out"], rtol=1e-9, atol=1e-12)


def test_entries_of_takes_a_rows_of_block_i_and_b_rows_of_block_i_minus_1():
    name, over = TINY["csa_prefill"]
    cfg = synth.scaled(name, **over)
    x = _np(synth.make_inputs(cfg, seed=5))
    m = cfg["m"]
    ref = OP.entries_of(cfg, x, 0)
    for j in (0, 3, cfg["N"] - 1):
        for nm, target in (("Ca", j), ("Za", j), ("Cb", j + 1), ("Zb", j + 1)):
            y = {k: v.copy() for k, v in x.items()}
            y[nm][0, m * j:m * (j + 1)] += np.linspace(0.5, 1.5, m)[:, None]
            moved = np.nonzero(np.abs(OP.entries_of(cfg, y, 0) - ref).max(axis=1) > 1e-12)[0]
            assert moved.tolist() == ([target] if target < cfg["N"] else []), (nm, j, moved)


def test_stored_formats_decode_close_to_their_source():
    # the FP8/BF16-RoPE rows and FP4 indexer tensors of the mixed workload
    # against the float32 values they were quantised from (same workload name,
    # so the same seeded normals): e4m3 keeps 3 mantissa bits (relative step
    # 2^-3, so rounding error <= 2^-4 |x| above the subnormal range, where the
    # step is 2^-9 of the row scale); bf16 keeps 8 bits; e2m1 with a block
    # scale s rounds to within s of the source and |source| <= 6 s
    name, over = TINY["csa_decode_mixed"]
    cfg = synth.scaled(name, **over)
    src_cfg = dict(cfg, dtype="f32")
    xq = _np(synth.make_inputs(cfg, seed=6))
    xs = _np(synth.make_inputs(src_cfg, seed=6))
    d, r = cfg["d"], cfg["r"]
    for b in range(cfg["B"]):
        for got, src, scale in ((OP.entries_of(cfg, xq, b), xs["entries"][b], xq["ent_scale"][b]),
                                (OP.window_of(xq, b), xs["win"][b], xq["win_scale"][b])):
            err = np.abs(got - src)
            bound_nope = 2.0 ** -4 * np.abs(src[:, :d - r]) + 2.0 ** -10 * scale[:, None]
            assert np.all(err[:, :d - r] <= bound_nope + 1e-12)
            assert np.all(err[:, d - r:] <= 2.0 ** -8 * np.abs(src[:, d - r:]) + 1e-30)
        qI, K = OP.indexer_inputs(xq, b, [0])
        for got, src, sf in ((qI, xs["qI"][b][[0]], xq["qI_sf"][b][[0]]),
                             (K, xs["K"][b], xq["K_sf"][b])):
            s = np.repeat(O.decode_e4m3(sf), 16, axis=-1)
            assert np.all(np.abs(got - src) <= s + 1e-12)
            assert np.all(np.abs(src) <= 6 * s + 1e-12)
