"""One CSA or HCA attention layer forward, composed from the C-ABI stages.

DeepSeek-V4 report (Chinese translation, blog.uika.cn) §2.3.1: compress the
per-token entries (m = 4, overlapped), score every visible compressed entry
with the lightning indexer, keep the top-k, and run shared-KV MQA over them
plus the 128-token window with the per-head sink.  §2.3.2: HCA compresses
with m' = 128 and attends densely.  Decode steps start from a given
compressed cache (a new entry is compressed only when a block closes).

The functions take a dict of device tensors named as in ``synth.generate``
and a size dict as in ``synth.configs``; they only allocate outputs and call
the library.
"""

from __future__ import annotations

from . import _lib as L


class Buffers:
    """Reusable intermediate and output buffers of one layer forward."""

    def __init__(self):
        self.entries = None
        self.scores = None
        self.idx = None
        self.out = None
        self.ws = None
        self.ws_topk = None


def _entries_arg(x):
    if "entries" in x:
        return x["entries"]
    return (x["ent_nope"], x["ent_scale"], x["ent_rope"])


def _win_arg(x):
    if "win" in x:
        return x["win"]
    return (x["win_nope"], x["win_scale"], x["win_rope"])


def _indexer_args(x):
    if "qI" in x:
        return x["qI"], None, x["K"], None
    return x["qI_fp4"], x["qI_sf"], x["K_fp4"], x["K_sf"]


def forward(cfg: dict, x: dict, buf: Buffers | None = None):
    """All stages of one layer forward; returns the attention output [B, Tq, n_h, d]."""
    buf = buf or Buffers()
    kind = cfg["kind"]
    m, r, n_win = cfg["m"], cfg["r"], cfg["n_win"]
    q_pos0, win_base, base = cfg["q_pos0"], cfg["win_base"], cfg["rope_base"]
    if kind == "csa_prefill":
        buf.entries = L.csa_compress(x["Ca"], x["Za"], m, Cb=x["Cb"], Zb=x["Zb"], out=buf.entries)
        entries = buf.entries
    elif kind == "hca_prefill":
        buf.entries = L.csa_compress(x["C"], x["Z"], m, out=buf.entries)
        entries = buf.entries
    else:
        entries = _entries_arg(x)
    win = _win_arg(x)
    if kind.startswith("csa"):
        qI, qI_sf, K, K_sf = _indexer_args(x)
        buf.scores, buf.idx, buf.ws_topk = L.csa_index_topk(
            qI, x["w"], K, cfg["k"], m, q_pos0, qI_sf=qI_sf, K_sf=K_sf, scores=buf.scores,
            idx=buf.idx, ws=buf.ws_topk)
        if buf.ws is None:
            n = L.attend_workspace_size(x["q"], entries, win, cfg["k"], m, n_win, q_pos0, r, False)
            buf.ws = L._workspace(None, n, x["q"].device)
        buf.out = L.csa_attend(x["q"], entries, buf.idx, win, x["sink"], m, n_win, win_base,
                               q_pos0, r, base, out=buf.out, ws=buf.ws)
    else:
        if buf.ws is None:
            n = L.attend_workspace_size(x["q"], entries, win, 0, m, n_win, q_pos0, r, True)
            buf.ws = L._workspace(None, n, x["q"].device)
        buf.out = L.hca_attend(x["q"], entries, win, x["sink"], m, n_win, win_base, q_pos0, r,
                               base, out=buf.out, ws=buf.ws)
    return buf.out
