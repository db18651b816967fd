"""Workload shapes for the CSA / HCA forward path.

Each workload is a plain dict of sizes.  The five main workloads follow the
shapes the DeepSeek-V4 report gives for V4-Pro (Chinese translation,
blog.uika.cn, §4.2.1 model settings table: m=4, n_h^I=64, c^I=128, top-k 1024,
m'=128, n_h=128, c=512, n_win=128; §2.3.3: RoPE on the last 64 dims) and a tiny
fp32 prefill case.  ``scaled`` derives smaller cases of the same structure for
the parity tests.

This module holds no arithmetic of the method: only sizes.
"""

from __future__ import annotations

import copy

# kind: what the workload exercises
#   csa_prefill : compress (overlapped, m) -> index -> top-k -> sparse attend
#   csa_decode  : index -> top-k -> sparse attend against a given compressed cache
#   hca_prefill : compress (non-overlapped, m') -> dense attend
#   hca_decode  : dense attend against a given compressed cache
WORKLOADS = {
    "tiny_csa_prefill_f32": dict(
        kind="csa_prefill", dtype="f32", B=1, T=256, m=4, d=128, r=32, n_h=4,
        H_I=4, c_I=32, k=16, n_win=16, w_scale=0.25, qk_scale=32 ** -0.5),
    "csa_decode_128k": dict(
        kind="csa_decode", dtype="bf16", B=4, L=131072, m=4, d=512, r=64,
        n_h=128, H_I=64, c_I=128, k=1024, n_win=128, w_scale=1.0 / 64,
        qk_scale=128 ** -0.5),
    "csa_prefill_32k": dict(
        kind="csa_prefill", dtype="bf16", B=1, T=32768, m=4, d=512, r=64,
        n_h=128, H_I=64, c_I=128, k=1024, n_win=128, w_scale=1.0 / 64,
        qk_scale=128 ** -0.5),
    "hca_decode_1m": dict(
        kind="hca_decode", dtype="bf16", B=2, L=1048576, m=128, d=512, r=64,
        n_h=128, n_win=128),
    "hca_prefill_64k": dict(
        kind="hca_prefill", dtype="bf16", B=1, T=65536, m=128, d=512, r=64,
        n_h=128, n_win=128),
    "csa_decode_1m_mixed": dict(
        kind="csa_decode", dtype="mixed", B=8, L=1048576, m=4, d=512, r=64,
        n_h=128, H_I=64, c_I=128, k=1024, n_win=128, w_scale=1.0 / 64,
        qk_scale=128 ** -0.5),
    # V4-Flash attention shape (same report, §4.2.1: n_h=64, top-k 512; m, the
    # indexer, c and the window as Pro), decode and prefill at the Pro sizes
    "csa_decode_flash_128k": dict(
        kind="csa_decode", dtype="bf16", B=4, L=131072, m=4, d=512, r=64,
        n_h=64, H_I=64, c_I=128, k=512, n_win=128, w_scale=1.0 / 64,
        qk_scale=128 ** -0.5),
    # the producer side of the CSA prefill (same report, §2.3.1: the indexer
    # keys K^IComp are the overlapped compression of per-token index rows;
    # §2.3.3: compressed entries are RMS-normalised before core attention):
    # keys compressed from raw rows, entries RMS-normalised (eps 1e-6, no
    # weight: the pages give neither) and stored pre-rotated at compression
    "csa_prefill_32k_producer": dict(
        kind="csa_prefill", dtype="bf16", B=1, T=32768, m=4, d=512, r=64,
        n_h=128, H_I=64, c_I=128, k=1024, n_win=128, w_scale=1.0 / 64,
        qk_scale=128 ** -0.5, index_keys="compressed", entry_norm=True,
        entry_norm_eps=1e-6, entry_rope=True),
    "csa_prefill_flash_32k": dict(
        kind="csa_prefill", dtype="bf16", B=1, T=32768, m=4, d=512, r=64,
        n_h=64, H_I=64, c_I=128, k=512, n_win=128, w_scale=1.0 / 64,
        qk_scale=128 ** -0.5),
}

ROPE_BASE = 10000.0


def get(name: str) -> dict:
    cfg = copy.deepcopy(WORKLOADS[name])
    cfg["name"] = name
    return derive(cfg)


def scaled(name: str, **overrides) -> dict:
    """A copy of workload ``name`` with some sizes replaced (for parity cases);
    ``lengths`` (decode) gives each sequence its own context length."""
    cfg = copy.deepcopy(WORKLOADS[name])
    cfg.update(overrides)

    def tag(v):
        return "-".join(map(str, v)) if isinstance(v, (list, tuple)) else str(v)
    cfg["name"] = name + "".join(f"_{k}{tag(v)}" for k, v in sorted(overrides.items()))
    return derive(cfg)


def derive(cfg: dict) -> dict:
    """Fill in the derived sizes: entry count N, query count and the context
    length of each sequence.

    Prefill: every sequence has T tokens, query row i sits at token i and the
    window buffer holds all T tokens.  Decode: sequence b holds lengths[b]
    tokens (default L for every sequence; the new token is the last one, at
    position lengths[b] - 1), the compressed cache is sized for the longest
    sequence and the window buffer holds each sequence's last n_win tokens.
    """
    kind = cfg["kind"]
    if kind.endswith("prefill"):
        cfg["N"] = cfg["T"] // cfg["m"]
        cfg["Tq"] = cfg["T"]
        cfg["T_win"] = cfg["T"]      # window buffer holds every token
        cfg["lengths"] = [cfg["T"]] * cfg["B"]
    else:
        lengths = list(cfg.get("lengths") or [cfg["L"]] * cfg["B"])
        if len(lengths) != cfg["B"] or min(lengths) < 1:
            raise ValueError("one context length >= 1 per sequence")
        cfg["lengths"] = lengths
        cfg["L"] = max(lengths)
        cfg["N"] = cfg["L"] // cfg["m"]
        cfg["Tq"] = 1
        cfg["T_win"] = cfg["n_win"]  # window buffer holds the last n_win tokens
    cfg.setdefault("rope_base", ROPE_BASE)
    return cfg


def query_positions(cfg: dict):
    """Absolute token position of every query row: [B][Tq] nested lists."""
    if cfg["kind"].endswith("prefill"):
        return [list(range(cfg["T"])) for _ in range(cfg["B"])]
    return [[L - 1] for L in cfg["lengths"]]


def window_bases(cfg: dict):
    """Token held by row 0 of each sequence's window buffer."""
    if cfg["kind"].endswith("prefill"):
        return [0] * cfg["B"]
    return [max(0, L - cfg["n_win"]) for L in cfg["lengths"]]
