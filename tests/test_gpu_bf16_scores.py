"""BF16 index scores (DeepSeek-V4 report, Chinese translation, blog.uika.cn,
§3.4: the index scores are quantised from FP32 to BF16, which makes the top-k
selector faster while keeping 99.7% recall of the selected KV entries).

With score_dtype BF16 the index kernel stores each score rounded to bf16 and
the selector ranks those rounded values (ties toward the lower index).  The
tests check:
* the stored scores against the float64 oracle within the float32 tolerance
  plus one bf16 rounding (relative 2^-9 of the score, bounded here by 2^-8);
* the selected set, bit-exact, against the oracle's rule applied to the GPU's
  own bf16 scores (bf16 rounding makes equal scores common, so the
  lower-index tie rule is exercised; negative scores exercise the keys of
  negative numbers);
* the recall of the float32 selection: the share of the entries selected
  from float32 scores that the bf16 selection keeps.
"""

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O
from tests.parity import TOL_SCORES_REL, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gen(seed):
    return torch.Generator(device=DEV).manual_seed(seed)


def _inputs(fmt, B, N, H=64, c=128, seed=300):
    w = torch.rand((B, 1, H), generator=_gen(seed), device=DEV) / H
    q = (torch.randn((B, 1, H, c), generator=_gen(seed + 1), device=DEV) / c ** 0.5)
    k = (torch.randn((B, N, c), generator=_gen(seed + 2), device=DEV) / c ** 0.5)
    if fmt == "bf16":
        return q.to(torch.bfloat16), None, k.to(torch.bfloat16), None, w
    from synth.generate import quantise_fp4_blocks
    qp, qs = quantise_fp4_blocks(q)
    kp, ks = quantise_fp4_blocks(k)
    return qp, qs, kp, ks, w


def _oracle_scores(fmt, qI, q_sf, Kt, k_sf, w, b, t, m):
    if fmt == "bf16":
        q64, k64 = f64(qI[b]), f64(Kt[b])
    else:
        q64 = O.decode_fp4_blocks(qI[b].cpu().numpy(), q_sf[b].cpu().numpy())
        k64 = O.decode_fp4_blocks(Kt[b].cpu().numpy(), k_sf[b].cpu().numpy())
    return O.index_scores(q64, f64(w[b]), k64, np.array([t]), m)[0]


def _check_selection(scores, idx, k, m, q_pos):
    sc, ix = f64(scores), idx.cpu().numpy()
    B, Tq, N = sc.shape
    for b in range(B):
        for i in range(Tq):
            vis = min(N, O.visible_count(int(q_pos[b][i]), m))
            n = min(k, vis)
            want = np.sort(O.topk_select(sc[b, i], k, vis))
            assert np.array_equal(ix[b, i][:n], want), f"row ({b},{i})"
            assert np.all(ix[b, i][n:] == -1)


@pytest.mark.parametrize("fmt,B,N,k", [
    ("bf16", 4, 32768, 1024),      # V4-Pro decode rows at 128K context
    ("fp4", 2, 262144, 1024),      # 1M-context rows, FP4 indexer, 16-CTA clusters
    ("bf16", 3, 5001, 333),        # odd N
    ("bf16", 2, 700, 1024),        # every visible entry selected
])
def test_index_topk_bf16_scores(fmt, B, N, k):
    import compressed_sparse_long_05_b300 as K
    m = 4
    qI, q_sf, Kt, k_sf, w = _inputs(fmt, B, N)
    q_pos = torch.tensor([[4 * N - 1 - 3 * b] for b in range(B)], dtype=torch.int32, device=DEV)
    s, idx, _ = K.csa_index_topk(qI, w, Kt, k, m, q_pos, qI_sf=q_sf, K_sf=k_sf,
                                 score_dtype=torch.bfloat16)
    s32, idx32, _ = K.csa_index_topk(qI, w, Kt, k, m, q_pos, qI_sf=q_sf, K_sf=k_sf)
    torch.cuda.synchronize()
    K.device_error()
    assert s.dtype == torch.bfloat16
    # scores: within one bf16 rounding of the oracle (plus the float32 tolerance)
    for b in (0, B - 1):
        t = int(q_pos[b, 0])
        ref = _oracle_scores(fmt, qI, q_sf, Kt, k_sf, w, b, t, m)
        got = f64(s[b, 0])
        assert np.array_equal(np.isneginf(got), np.isneginf(ref))
        fin = np.isfinite(ref)
        err = np.abs(got[fin] - ref[fin])
        bound = 2.0 ** -8 * np.abs(ref[fin]) + TOL_SCORES_REL * np.abs(ref[fin]).max()
        assert np.all(err <= bound), f"b={b}: max excess {(err - bound).max():.3g}"
        # and bf16 rounding of the GPU's own float32 score, exactly
        assert torch.equal(s[b, 0], s32[b, 0].to(torch.bfloat16))
    _check_selection(s, idx, k, m, q_pos.cpu().numpy())
    # recall of the float32 selection
    rec = []
    for b in range(B):
        a32 = set(idx32[b, 0].cpu().numpy().tolist()) - {-1}
        a16 = set(idx[b, 0].cpu().numpy().tolist()) - {-1}
        rec.append(len(a32 & a16) / max(1, len(a32)))
    print(f"recall of the float32 selection ({fmt}, N={N}, k={k}): {np.mean(rec):.4f}")
    assert np.mean(rec) >= 0.9


@pytest.mark.parametrize("B,Tq,N,k,q_pos0,levels", [
    (1, 300, 64, 16, 0, 0),          # prefill rows, vis <= k on the first rows
    (1, 40, 9000, 4096, 35990, 0),   # large k
    (2, 3, 20000, 7, 79999, 1),      # every score equal: lowest indices win
    (1, 64, 2048, 100, 8000, 7),     # few distinct values
])
def test_topk_bf16_scores_with_negatives(B, Tq, N, k, q_pos0, levels):
    import compressed_sparse_long_05_b300 as K
    g = _gen(23)
    if levels:
        scores = (torch.randint(0, levels, (B, Tq, N), generator=g, device=DEV).float() - 3.0)
    else:
        scores = torch.randn((B, Tq, N), generator=g, device=DEV)   # half of them negative
    scores = scores.to(torch.bfloat16)
    idx = K.csa_topk(scores, k, 4, q_pos0)
    torch.cuda.synchronize()
    K.device_error()
    q_pos = (q_pos0 + np.arange(Tq))[None].repeat(B, 0)
    _check_selection(scores, idx, k, 4, q_pos)
