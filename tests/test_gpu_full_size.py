"""Parity at the full workload sizes, in the launch configuration the benchmark times.

Each test runs one whole layer forward (``path.forward``: the same C-ABI calls,
shapes and work split that ``bench.py`` times) on the full-size seeded
workload, then checks sampled outputs against the float64 oracle one by one:

* compressed entries (prefill workloads) at sampled entry indices;
* indexer score rows at sampled query rows (relative 1e-3, identical -inf);
* the top-k set of each sampled row, bit-exact against the oracle's rule
  applied to the GPU's own fp32 scores;
* the attention output of each sampled row, against the oracle's attention on
  the GPU-selected entries (2e-2 for bf16 storage, 6e-2 for FP8/FP4 storage).

Sampled rows include the block and window boundaries (t = 0, m-1, m, 127, 128,
4095, 4096, T-1) for prefill, and every sequence's new token for decode.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import csa_oracle as O
from tests.parity import TOL_BF16, TOL_MIXED, assert_close, assert_scores_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    import compressed_sparse_long_05_b300 as k
    k.lib()
    return k


def _np(t):
    return t.cpu().numpy() if t.dtype in (torch.uint8, torch.int32) else f64(t)


def _entries(cfg, x, buf, b):
    """The compressed entries the GPU attention used, float64 and unrotated."""
    if cfg["kind"].endswith("prefill"):
        e = f64(buf.entries[b])
        if cfg.get("entry_rope"):           # stored rotated at m(s+1)-1: turn them back
            e = O.rope_rotate(e, -O.entry_position(np.arange(e.shape[0]), cfg["m"]), cfg["r"],
                              cfg["rope_base"])
        return e
    if "entries" in x:
        return f64(x["entries"][b])
    return O.decode_mixed_entries(_np(x["ent_nope"][b]), _np(x["ent_scale"][b]), f64(x["ent_rope"][b]))


def _window(x, b):
    if "win" in x:
        return f64(x["win"][b])
    return O.decode_mixed_entries(_np(x["win_nope"][b]), _np(x["win_scale"][b]), f64(x["win_rope"][b]))


def _indexer(x, b, i, buf=None):
    """(q [H, c], K [N, c]) float64 for query row i of batch row b (the keys
    the GPU indexed: its own compression when the workload compresses them)."""
    if "CIa" in x:
        return f64(x["qI"][b, i]), f64(buf.K[b])
    if "qI" in x:
        return f64(x["qI"][b, i]), f64(x["K"][b])
    q = O.decode_fp4_blocks(_np(x["qI_fp4"][b, i]), _np(x["qI_sf"][b, i]))
    k = O.decode_fp4_blocks(_np(x["K_fp4"][b]), _np(x["K_sf"][b]))
    return q, k


def _rows(cfg):
    if cfg["kind"].endswith("decode"):
        return [0]
    T = cfg["T"]
    m = cfg["m"]
    fixed = [0, m - 1, m, 127, 128, 4095, 4096, T - 1]
    rng = np.random.default_rng(7)
    return sorted({r for r in fixed + rng.integers(0, T, 2).tolist() if r < T})


def _check_workload(K, name, batch_rows=None):
    from compressed_sparse_long_05_b300 import path as P
    cfg = synth.get(name)
    x = synth.make_inputs(cfg, seed=0, device=DEV)
    buf = P.Buffers()
    out = P.forward(cfg, x, buf)
    torch.cuda.synchronize()
    K.device_error()
    m, r, n_win, base = cfg["m"], cfg["r"], cfg["n_win"], cfg["rope_base"]
    tol = TOL_MIXED if cfg["dtype"] == "mixed" else TOL_BF16
    sink = f64(x["sink"])
    rows = _rows(cfg)
    for b in (batch_rows if batch_rows is not None else range(cfg["B"])):
        ent = _entries(cfg, x, buf, b)
        if cfg["kind"] == "csa_prefill":
            probe = [0, 1, 2, cfg["N"] // 2, cfg["N"] - 1]
            ref = O.compress_csa(f64(x["Ca"][b]), f64(x["Cb"][b]), f64(x["Za"][b]), f64(x["Zb"][b]), m)
            if cfg.get("entry_norm"):
                ref = O.rms_norm(ref, eps=cfg["entry_norm_eps"])
            assert_close(ent[probe], ref[probe], TOL_BF16, TOL_BF16, f"{name} compress")
            if "CIa" in x:
                kref = O.compress_csa(f64(x["CIa"][b]), f64(x["CIb"][b]), f64(x["ZIa"][b]),
                                      f64(x["ZIb"][b]), m)
                assert_close(f64(buf.K[b])[probe], kref[probe], TOL_BF16, TOL_BF16,
                             f"{name} indexer-key compress")
        if cfg["kind"] == "hca_prefill":
            probe = [0, 1, cfg["N"] // 2, cfg["N"] - 1]
            ref = O.compress_hca(f64(x["C"][b]), f64(x["Z"][b]), m)
            assert_close(ent[probe], ref[probe], TOL_BF16, TOL_BF16, f"{name} compress")
        win = _window(x, b)
        win_base = int(x["win_base"][b])
        for i in rows:
            t = int(x["q_pos"][b, i])
            q = f64(x["q"][b, i])
            if cfg["kind"].startswith("csa"):
                qI, Kc = _indexer(x, b, i, buf)
                ref_s = O.index_scores(qI[None], f64(x["w"][b, i])[None], Kc, np.array([t]), m)[0]
                got_s = f64(buf.scores[b, i])
                assert_scores_close(got_s, ref_s, f"{name} scores b={b} i={i}")
                vis = min(cfg["N"], O.visible_count(t, m))
                want = np.sort(O.topk_select(got_s, cfg["k"], vis))
                got_i = buf.idx[b, i].cpu().numpy()
                n = min(cfg["k"], vis)
                assert np.array_equal(got_i[:n], want), f"{name} top-k b={b} i={i}"
                assert np.all(got_i[n:] == -1)
                ref_o = O.csa_attend_token(q, t, ent, got_i, win, win_base, sink, m, n_win, r, base)
            else:
                ref_o = O.hca_attend_token(q, t, ent, win, win_base, sink, m, n_win, r, base)
            assert_close(f64(out[b, i]), ref_o, tol, tol, f"{name} attend b={b} i={i} t={t}")


def test_csa_decode_128k_full(K):
    _check_workload(K, "csa_decode_128k")


def test_csa_prefill_32k_full(K):
    _check_workload(K, "csa_prefill_32k")


def test_hca_decode_1m_full(K):
    _check_workload(K, "hca_decode_1m")


def test_hca_prefill_64k_full(K):
    _check_workload(K, "hca_prefill_64k")


def test_csa_decode_1m_mixed_full(K):
    # all 8 sequences run; two are checked row by row (each oracle row decodes
    # and scores 262,144 FP4 keys in float64)
    _check_workload(K, "csa_decode_1m_mixed", batch_rows=[0, 7])


def test_csa_decode_flash_128k_full(K):
    # V4-Flash attention shape: one 64-head group, top-k 512
    _check_workload(K, "csa_decode_flash_128k")


def test_csa_prefill_flash_32k_full(K):
    _check_workload(K, "csa_prefill_flash_32k")


def test_csa_prefill_32k_producer_full(K):
    # indexer keys compressed from raw index rows, entries RMS-normalised and
    # stored pre-rotated by the compression epilogue
    _check_workload(K, "csa_prefill_32k_producer")
