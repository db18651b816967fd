"""Whole-path composition of the oracle stages for one workload.

TEST INFRASTRUCTURE ONLY (see csa_oracle).  Takes numpy copies of a workload's
inputs (as produced by the seeded generators) and runs the four stages of the
DeepSeek-V4 CSA forward (compress -> index -> top-k -> attend; DeepSeek-V4
Chinese translation, blog.uika.cn, §2.3.1) or the two of HCA (compress ->
dense attend, §2.3.2) for a chosen subset of query rows.
"""

from __future__ import annotations

import numpy as np

from . import csa_oracle as O


def entries_of(cfg: dict, x: dict, b: int) -> np.ndarray:
    """Compressed entries of batch row b, float64 [N, d] (unrotated).

    Prefill workloads compress the raw rows; with cfg["entry_norm"] each
    compressed entry is then RMS-normalised with eps cfg["entry_norm_eps"]
    ([uika] §2.3.3)."""
    kind = cfg["kind"]
    if kind in ("csa_prefill", "hca_prefill"):
        if kind == "csa_prefill":
            ent = O.compress_csa(x["Ca"][b], x["Cb"][b], x["Za"][b], x["Zb"][b], cfg["m"])
        else:
            ent = O.compress_hca(x["C"][b], x["Z"][b], cfg["m"])
        return O.rms_norm(ent, eps=cfg["entry_norm_eps"]) if cfg.get("entry_norm") else ent
    if "entries" in x:
        return np.asarray(x["entries"][b], dtype=np.float64)
    return O.decode_mixed_entries(x["ent_nope"][b], x["ent_scale"][b], x["ent_rope"][b])


def window_of(x: dict, b: int) -> np.ndarray:
    if "win" in x:
        return np.asarray(x["win"][b], dtype=np.float64)
    return O.decode_mixed_entries(x["win_nope"][b], x["win_scale"][b], x["win_rope"][b])


def indexer_inputs(x: dict, b: int, rows, m: int = 4):
    """(qI [len(rows), H, c], K [N, c]) of batch row b, float64.

    With raw per-token indexer keys (CIa, CIb, ZIa, ZIb) the keys are their
    overlapped compression, K^IComp of [uika] §2.3.1 ([notes] 关键设计 1:
    the index keys go through the same weighted overlap compression)."""
    if "CIa" in x:
        qI = np.asarray(x["qI"][b][rows], dtype=np.float64)
        K = O.compress_csa(x["CIa"][b], x["CIb"][b], x["ZIa"][b], x["ZIb"][b], m)
    elif "qI" in x:
        qI = np.asarray(x["qI"][b][rows], dtype=np.float64)
        K = np.asarray(x["K"][b], dtype=np.float64)
    else:
        qI = O.decode_fp4_blocks(x["qI_fp4"][b][rows], x["qI_sf"][b][rows])
        K = O.decode_fp4_blocks(x["K_fp4"][b], x["K_sf"][b])
    return qI, K


def run_rows(cfg: dict, x: dict, b: int, rows, selected=None, entries=None):
    """Oracle outputs for query rows ``rows`` of batch row b.

    Query row i sits at absolute position x["q_pos"][b][i]; row j of the
    window buffer of batch row b holds raw token x["win_base"][b] + j.

    Returns a dict with 't' (the rows' positions), 'scores' [len(rows), N]
    (CSA only), 'selected' (list of index arrays, CSA only) and 'out'
    [len(rows), n_h, d].  ``selected`` may supply the index sets the attention
    uses (e.g. a set already checked against the oracle's own top-k rule);
    ``entries`` may supply precomputed compressed entries.
    """
    rows = np.asarray(rows, dtype=np.int64)
    m, r, base, n_win = cfg["m"], cfg["r"], cfg["rope_base"], cfg["n_win"]
    t_pos = np.asarray(x["q_pos"][b], dtype=np.int64)[rows]
    win_base = int(np.asarray(x["win_base"])[b])
    ent = entries_of(cfg, x, b) if entries is None else entries
    win = window_of(x, b)
    q = x["q"][b]
    res = {"t": t_pos}
    outs = []
    if cfg["kind"].startswith("csa"):
        qI, K = indexer_inputs(x, b, rows, m)
        w = np.asarray(x["w"][b][rows], dtype=np.float64)
        scores = O.index_scores(qI, w, K, t_pos, m)
        res["scores"] = scores
        if selected is None:
            selected = [O.topk_select(scores[i], cfg["k"], min(cfg["N"], O.visible_count(int(t), m)))
                        for i, t in enumerate(t_pos)]
        res["selected"] = selected
        for i, t in enumerate(t_pos):
            outs.append(O.csa_attend_token(np.asarray(q[rows[i]], dtype=np.float64), int(t), ent,
                                           selected[i], win, win_base, x["sink"], m, n_win, r, base))
    else:
        for i, t in enumerate(t_pos):
            outs.append(O.hca_attend_token(np.asarray(q[rows[i]], dtype=np.float64), int(t), ent,
                                           win, win_base, x["sink"], m, n_win, r, base))
    res["out"] = np.stack(outs) if outs else np.zeros((0,))
    return res
