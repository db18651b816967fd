"""Float64 CPU oracle for the DeepSeek-V4 CSA / HCA attention forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module.  It shares no
code with the CUDA path and imports nothing from it.

Every function is the plain definition written out in float64 numpy, one query
(or one compressed entry) at a time, with library matmuls as the only building
block.  Stored low-precision inputs (bf16, e4m3, e2m1) are decoded exactly
before any arithmetic.

Sources (the DeepSeek-V4 technical report as restated by the pages):
  [uika]  DeepSeek-V4 Chinese translation, blog.uika.cn — §2.3.1 "Compressed
          Sparse Attention" (compression, lightning indexer, shared-KV MQA),
          §2.3.2 "Heavily Compressed Attention", §2.3.3 "other key details"
          (partial RoPE with inverse rotation of the output, sliding window,
          attention sink), §2.3.4 (FP8/BF16 KV storage, FP4 indexer QK),
          §3.6.1 (tail tokens stay uncompressed until a block closes).
  [notes] DeepSeek-V4 paper notes, awesome.papernotes.org — "关键设计 1" (CSA
          compression and indexer equations, C_t = TopK_k(I_t,:)), "关键设计 2"
          (HCA equations).

Readings taken where the pages leave a step open (each is listed in the design
notes with its reason):
  * entry 0 of CSA has no previous block: its softmax runs over the m a-rows only;
  * the learnable position biases B^a, B^b, B are [m, d] (one per in-block row
    and channel) and default to zero;
  * tail tokens (T mod m) are not compressed: N = floor(T / m);
  * compressed entry s is visible to query t iff (s+1)*m <= t+1, and its RoPE
    position is the last raw token it summarises, m*(s+1)-1;
  * RoPE rotates interleaved pairs (x[2i], x[2i+1]) of the last r dims with
    theta_i = base^(-2i/r); the output is rotated back at position -t;
  * the window of query t is tokens max(0, t-n_win+1) .. t, inclusive;
  * logits are scaled by 1/sqrt(d) with the full head dim d;
  * the sink adds exp(z'_h) to the softmax denominator only;
  * top-k orders visible entries by (score descending, index ascending) and
    keeps the first min(k, vis); the result is a set.
"""

from __future__ import annotations

import math

import numpy as np

# ----------------------------------------------------------------------------
# stored formats -> float64 ([uika] §2.3.4: FP8 non-RoPE dims + BF16 RoPE dims;
# FP4 indexer QK; scales per the OCP/NV 4-bit block format)
# ----------------------------------------------------------------------------


def decode_e4m3(b) -> np.ndarray:
    """e4m3fn byte -> value: 1 sign, 4 exponent (bias 7), 3 mantissa bits.

    Exponent field 0 is subnormal (mant/8 * 2^-6); 0x7f / 0xff are NaN.
    """
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 15
    mant = (b & 7).astype(np.float64)
    val = np.where(e == 0, mant / 8.0 * 2.0 ** -6,
                   (1.0 + mant / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 15) & ((b & 7) == 7), np.nan, val)
    return sign * val


def decode_e2m1(code) -> np.ndarray:
    """e2m1 4-bit code -> value: 1 sign, 2 exponent (bias 1), 1 mantissa bit."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    mb = (c & 1).astype(np.float64)
    val = np.where(e == 0, 0.5 * mb, (1.0 + 0.5 * mb) * np.exp2(e.astype(np.float64) - 1.0))
    return sign * val


def decode_fp4_blocks(packed, scale_bytes, block: int = 16) -> np.ndarray:
    """Packed e2m1 (element 2j in the low nibble of byte j) times its e4m3 block scale."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = decode_e2m1(packed & 15)
    hi = decode_e2m1(packed >> 4)
    vals = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    sf = decode_e4m3(scale_bytes)
    return vals * np.repeat(sf, block, axis=-1)


def decode_mixed_entries(nope_bytes, scale, rope) -> np.ndarray:
    """[..., d-r] e4m3 * per-entry scale, followed by the [..., r] RoPE dims."""
    nope = decode_e4m3(nope_bytes) * np.asarray(scale, dtype=np.float64)[..., None]
    return np.concatenate([nope, np.asarray(rope, dtype=np.float64)], axis=-1)


# ----------------------------------------------------------------------------
# 1. compression  ([uika] §2.3.1 compression equations; §2.3.2; [notes] 关键设计 1/2)
# ----------------------------------------------------------------------------


def _softmax_down_rows(logits: np.ndarray) -> np.ndarray:
    """Softmax of each column over the rows (the per-channel 'Softmax_row')."""
    mx = logits.max(axis=0, keepdims=True)
    e = np.exp(logits - mx)
    return e / e.sum(axis=0, keepdims=True)


def compress_csa(Ca, Cb, Za, Zb, m: int, Ba=None, Bb=None) -> np.ndarray:
    """Overlapped compression of one sequence: [T, d] x4 -> [floor(T/m), d].

    Entry i weighs the a-rows of block i and the b-rows of block i-1 with one
    softmax per channel over those 2m rows; block -1 does not exist, so entry 0
    uses its m a-rows alone.
    """
    Ca, Cb, Za, Zb = (np.asarray(x, dtype=np.float64) for x in (Ca, Cb, Za, Zb))
    T, d = Ca.shape
    N = T // m
    ba = np.zeros((m, d)) if Ba is None else np.asarray(Ba, dtype=np.float64)
    bb = np.zeros((m, d)) if Bb is None else np.asarray(Bb, dtype=np.float64)
    out = np.zeros((N, d))
    for i in range(N):
        a = slice(m * i, m * (i + 1))
        logits = Za[a] + ba
        values = Ca[a]
        if i >= 1:
            b = slice(m * (i - 1), m * i)
            logits = np.concatenate([logits, Zb[b] + bb], axis=0)
            values = np.concatenate([values, Cb[b]], axis=0)
        S = _softmax_down_rows(logits)
        out[i] = (S * values).sum(axis=0)
    return out


def compress_hca(C, Z, m: int, Bias=None) -> np.ndarray:
    """Non-overlapped compression of one sequence: [T, d] x2 -> [floor(T/m), d]."""
    C, Z = np.asarray(C, dtype=np.float64), np.asarray(Z, dtype=np.float64)
    T, d = C.shape
    N = T // m
    bias = np.zeros((m, d)) if Bias is None else np.asarray(Bias, dtype=np.float64)
    out = np.zeros((N, d))
    for i in range(N):
        blk = slice(m * i, m * (i + 1))
        S = _softmax_down_rows(Z[blk] + bias)
        out[i] = (S * C[blk]).sum(axis=0)
    return out


def rms_norm(x, weight=None, eps: float = 0.0) -> np.ndarray:
    """RMSNorm of each vector along the last axis: x / sqrt(mean(x^2) + eps),
    times an optional per-channel weight ([uika] §2.3.3: the compressed KV
    entries, and each query head, are RMS-normalised before core attention)."""
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return y if weight is None else y * np.asarray(weight, dtype=np.float64)


# ----------------------------------------------------------------------------
# 2. lightning indexer  ([uika] §2.3.1 "Lightning Indexer"; [notes] 关键设计 1)
# ----------------------------------------------------------------------------


def visible_count(t: int, m: int) -> int:
    """Number of compressed entries query t may see: entries s with (s+1)m <= t+1
    (none for a query at a negative position)."""
    return max(0, (t + 1) // m)


def index_scores(qI, w, K, t_pos, m: int) -> np.ndarray:
    """I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . K[s,:]) for visible s, -inf otherwise.

    qI [Tq, H, c], w [Tq, H], K [N, c], t_pos [Tq] absolute query positions.
    """
    qI = np.asarray(qI, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    Tq = qI.shape[0]
    N = K.shape[0]
    out = np.full((Tq, N), -np.inf)
    for i in range(Tq):
        vis = min(N, visible_count(int(t_pos[i]), m))
        if vis == 0:
            continue
        dots = qI[i] @ K[:vis].T                 # [H, vis]
        out[i, :vis] = w[i] @ np.maximum(dots, 0.0)
    return out


# ----------------------------------------------------------------------------
# 3. top-k  ([uika] §2.3.1 "top-k selector"; [notes] C_t = TopK_k(I_t,:))
# ----------------------------------------------------------------------------


def topk_select(scores_row, k: int, vis: int) -> np.ndarray:
    """Indices of the min(k, vis) largest scores among s < vis; ties -> lower s.

    Returned in selection order (score descending, index ascending).
    """
    s = np.asarray(scores_row, dtype=np.float64)[:vis]
    order = np.lexsort((np.arange(vis), -s))   # last key is primary
    return order[: min(k, vis)].astype(np.int64)


# ----------------------------------------------------------------------------
# 4. attention  ([uika] §2.3.1 shared-KV MQA, §2.3.3 partial RoPE / window / sink)
# ----------------------------------------------------------------------------


def rope_rotate(x, pos, r: int, base: float) -> np.ndarray:
    """Rotate the last r dims of x by position pos, pairs (x[2i], x[2i+1]).

    x [..., d]; pos broadcasts against x[..., 0].  Dims before the last r are
    returned unchanged.  theta_i = base^(-2i/r), angle = pos * theta_i.
    """
    x = np.array(x, dtype=np.float64, copy=True)
    if r == 0:
        return x
    d = x.shape[-1]
    i = np.arange(r // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / r)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    x0 = x[..., d - r::2].copy()
    x1 = x[..., d - r + 1::2].copy()
    x[..., d - r::2] = x0 * c - x1 * s
    x[..., d - r + 1::2] = x0 * s + x1 * c
    return x


def entry_position(s, m: int):
    """RoPE position of compressed entry s: the last raw token of its block."""
    return m * (np.asarray(s) + 1) - 1


def window_positions(t: int, n_win: int) -> np.ndarray:
    """Raw tokens in the sliding window of query t: max(0, t-n_win+1) .. t."""
    return np.arange(max(0, t - n_win + 1), t + 1)


def attend_rows(q, t: int, rows, pos, sink, r: int, base: float) -> np.ndarray:
    """One query token, all heads, over an explicit set of key=value rows.

    q [n_h, d] un-rotated; rows [J, d] un-rotated with RoPE positions pos [J];
    sink [n_h].  Returns the inverse-rotated output [n_h, d].
    """
    q = np.asarray(q, dtype=np.float64)
    n_h, d = q.shape
    qr = rope_rotate(q, t, r, base)
    er = rope_rotate(rows, pos, r, base)
    logits = qr @ er.T / math.sqrt(d)            # [n_h, J]
    sink = np.asarray(sink, dtype=np.float64)
    mx = np.maximum(logits.max(axis=1) if logits.shape[1] else -np.inf, sink)
    p = np.exp(logits - mx[:, None])
    denom = p.sum(axis=1) + np.exp(sink - mx)
    o = (p @ er) / denom[:, None]
    return rope_rotate(o, -t, r, base)


def _window_rows(win, win_base: int, t: int, n_win: int):
    pos = window_positions(t, n_win)
    win = np.asarray(win, dtype=np.float64)
    return win[pos - win_base], pos


def csa_attend_token(q, t: int, entries, selected, win, win_base: int, sink,
                     m: int, n_win: int, r: int, base: float) -> np.ndarray:
    """CSA core attention for query t: the selected compressed entries plus the window.

    entries [N, d] (row s = compressed entry s), selected: indices into entries
    (entries of -1 are ignored), win [T_win, d] with row j holding raw token
    win_base + j.
    """
    sel = np.asarray([s for s in np.asarray(selected).ravel() if s >= 0], dtype=np.int64)
    ent = np.asarray(entries, dtype=np.float64)
    wrows, wpos = _window_rows(win, win_base, t, n_win)
    rows = np.concatenate([ent[sel], wrows], axis=0)
    pos = np.concatenate([entry_position(sel, m), wpos])
    return attend_rows(q, t, rows, pos, sink, r, base)


def hca_attend_token(q, t: int, entries, win, win_base: int, sink, m: int,
                     n_win: int, r: int, base: float) -> np.ndarray:
    """HCA core attention for query t: every visible compressed entry plus the window."""
    ent = np.asarray(entries, dtype=np.float64)
    vis = min(ent.shape[0], visible_count(t, m))
    s = np.arange(vis)
    wrows, wpos = _window_rows(win, win_base, t, n_win)
    rows = np.concatenate([ent[s], wrows], axis=0)
    pos = np.concatenate([entry_position(s, m), wpos])
    return attend_rows(q, t, rows, pos, sink, r, base)


# ----------------------------------------------------------------------------
# 5. grouped output projection  ([uika] §2.3.1 "分组输出投影"; §4.2.1 g, d_g)
# ----------------------------------------------------------------------------


def grouped_projection(A, W) -> np.ndarray:
    """Group j of the columns of A times its own weight: the n_h head outputs
    split into G groups, each projected to N = d_g dims.

    A [M, >= G*K]; W [G, N, K] (row n of W[j] holds output n's weights).
    Returns [M, G*N] with columns j*N .. (j+1)*N - 1 = A[:, j*K:(j+1)*K] @ W[j]^T.
    The final projection to the model width is the same with G = 1.
    """
    A = np.asarray(A, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    G, N, K = W.shape
    return np.concatenate([A[:, j * K:(j + 1) * K] @ W[j].T for j in range(G)], axis=1)
