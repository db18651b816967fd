"""A second, independently written restatement of the CSA / HCA forward for
tiny inputs, used to pin the float64 oracle's whole-path composition.

Test code only.  It shares nothing with ``oracle/``: plain Python loops over
lists with the ``math`` / ``cmath`` modules (no numpy arithmetic), and it is
structured differently wherever the mathematics allows, so that a slip in one
is unlikely to repeat in the other:

* compression (DeepSeek-V4 report, Chinese translation, blog.uika.cn, §2.3.1
  compression equations; §2.3.2 for HCA): the members of entry i are listed
  as (logit, value) pairs per channel and normalised by an explicit sum;
* the lightning indexer (§2.3.1): sum over heads of w * max(0, dot);
* top-k (§2.3.1; ties toward the lower index): a full sort of (-score, s);
* RoPE (§2.3.3): the pair (x[2i], x[2i+1]) is the complex number
  x[2i] + 1j x[2i+1], rotated by multiplication with exp(1j * p * theta_i),
  theta_i = base ** (-2i / r);
* attention (§2.3.1 shared-KV MQA, §2.3.3 window and sink): logits over the
  explicit row list, exp(logit - M) weights, denominator plus exp(sink - M);
  the output is rotated back by multiplying with exp(-1j * t * theta_i);
* stored formats (§2.3.4): e4m3 and e2m1 codes decoded from their bit fields
  by explicit branches, packed FP4 nibbles unpacked low-first.

Positions come from the inputs as the library takes them: query row i of
batch row b sits at q_pos[b][i]; window-buffer row j of batch row b holds
token win_base[b] + j.
"""

from __future__ import annotations

import cmath
import math


def _e4m3(byte: int) -> float:
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    f = byte & 0x7
    if e == 0xF and f == 0x7:
        return float("nan")
    if e == 0:
        return s * (f / 8.0) * 2.0 ** -6
    return s * (1.0 + f / 8.0) * 2.0 ** (e - 7)


_E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1(code: int) -> float:
    v = _E2M1[code & 7]
    return -v if code & 8 else v


def fp4_row(packed, scales):
    """One row of packed e2m1 bytes and its e4m3 block-16 scale bytes -> floats."""
    vals = []
    for byte in packed:
        vals.append(_e2m1(int(byte) & 0xF))
        vals.append(_e2m1(int(byte) >> 4))
    return [v * _e4m3(int(scales[j // 16])) for j, v in enumerate(vals)]


def mixed_row(nope, scale, rope):
    """FP8 non-RoPE dims times the row scale, then the bf16 RoPE dims."""
    return [_e4m3(int(b)) * float(scale) for b in nope] + [float(v) for v in rope]


def compress(A, Bv, ZA, ZB, m, overlap):
    T, d = len(A), len(A[0])
    out = []
    for i in range(T // m):
        members = [(ZA[j], A[j]) for j in range(m * i, m * i + m)]
        if overlap and i > 0:
            members += [(ZB[j], Bv[j]) for j in range(m * (i - 1), m * i)]
        row = []
        for c in range(d):
            top = max(z[c] for z, _ in members)
            den = sum(math.exp(z[c] - top) for z, _ in members)
            row.append(sum(math.exp(z[c] - top) * v[c] for z, v in members) / den)
        out.append(row)
    return out


def _dot(a, b):
    return sum(x * y for x, y in zip(a, b))


def index_score(qh, w, key):
    return sum(w[h] * max(0.0, _dot(qh[h], key)) for h in range(len(qh)))


def _rotate(vec, pos, r, base):
    d = len(vec)
    out = list(vec)
    for i in range(r // 2):
        theta = base ** (-(2.0 * i) / r)
        z = complex(vec[d - r + 2 * i], vec[d - r + 2 * i + 1]) * cmath.exp(1j * pos * theta)
        out[d - r + 2 * i] = z.real
        out[d - r + 2 * i + 1] = z.imag
    return out


def attend(q, t, rows, sink, r, base):
    """q: [n_h][d] for the query at t; rows: list of (vector, position)."""
    d = len(q[0])
    rot = [(_rotate(v, p, r, base)) for v, p in rows]
    out = []
    for h in range(len(q)):
        qh = _rotate(q[h], t, r, base)
        logits = [_dot(qh, v) / math.sqrt(d) for v in rot]
        M = max(logits + [sink[h]])
        wts = [math.exp(l - M) for l in logits]
        den = sum(wts) + math.exp(sink[h] - M)
        o = [sum(wts[j] * rot[j][c] for j in range(len(rot))) / den for c in range(d)]
        out.append(_rotate(o, -t, r, base))
    return out


def run(cfg, x, b, rows):
    """Per query row of batch row b: (scores or None, selected set or None, out)."""
    kind, m, r, base, n_win = cfg["kind"], cfg["m"], cfg["r"], cfg["rope_base"], cfg["n_win"]

    def L(a):
        return a.tolist() if hasattr(a, "tolist") else list(a)

    if kind == "csa_prefill":
        ent = compress(L(x["Ca"][b]), L(x["Cb"][b]), L(x["Za"][b]), L(x["Zb"][b]), m, True)
    elif kind == "hca_prefill":
        ent = compress(L(x["C"][b]), None, L(x["Z"][b]), None, m, False)
    elif "entries" in x:
        ent = L(x["entries"][b])
    else:
        ent = [mixed_row(x["ent_nope"][b][s], x["ent_scale"][b][s], x["ent_rope"][b][s])
               for s in range(len(x["ent_nope"][b]))]
    if "win" in x:
        win = L(x["win"][b])
    else:
        win = [mixed_row(x["win_nope"][b][j], x["win_scale"][b][j], x["win_rope"][b][j])
               for j in range(len(x["win_nope"][b]))]
    wb = int(x["win_base"][b])
    N = len(ent)
    res = []
    for i in rows:
        t = int(x["q_pos"][b][i])
        vis = [s for s in range(N) if (s + 1) * m <= t + 1]
        scores = sel = None
        if kind.startswith("csa"):
            if "qI" in x:
                qh = L(x["qI"][b][i])
                keys = L(x["K"][b])
            else:
                qh = [fp4_row(x["qI_fp4"][b][i][h], x["qI_sf"][b][i][h])
                      for h in range(len(x["qI_fp4"][b][i]))]
                keys = [fp4_row(x["K_fp4"][b][s], x["K_sf"][b][s]) for s in range(N)]
            w = L(x["w"][b][i])
            scores = {s: index_score(qh, w, keys[s]) for s in vis}
            order = sorted(vis, key=lambda s: (-scores[s], s))
            sel = sorted(order[: cfg["k"]])
            chosen = sel
        else:
            chosen = vis
        rows_list = [(ent[s], m * (s + 1) - 1) for s in chosen]
        for p in range(max(0, t - n_win + 1), t + 1):
            rows_list.append((win[p - wb], p))
        out = attend(L(x["q"][b][i]), t, rows_list, L(x["sink"]), r, base)
        res.append((scores, sel, out))
    return res
