"""Decode batches whose sequences sit at different context lengths.

Each sequence b of a decode batch has its own length L_b; its new token is at
position t_b = L_b - 1 (DeepSeek-V4 report, Chinese translation, blog.uika.cn,
§2.3.1: visibility (s+1)m <= t+1 is decided per query t).  The library takes
the positions as a per-row device array q_pos [B, Tq] and each sequence's
window-buffer base as win_base [B].  These tests run one whole decode step
(``path.forward``, the launch configuration the benchmark times) on batches
that mix a full-length sequence, one whose length is not a multiple of m, one
that sees fewer than k entries and one shorter than the window, and compare
every sequence with the float64 oracle: scores (1e-3 relative, identical -inf
pattern), the top-k set (bit-exact, from the GPU's own scores) and the
attention output (2e-2 bf16, 6e-2 FP8/FP4 storage).
"""

import numpy as np
import pytest
import torch

import synth
from oracle import csa_oracle as O
from oracle import pipeline as OP
from tests.parity import TOL_BF16, TOL_MIXED, assert_close, assert_scores_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _host(x):
    return {k: (v.float().cpu().numpy() if v.dtype in (torch.bfloat16, torch.float32)
                else v.cpu().numpy()) for k, v in x.items()}


@pytest.mark.parametrize("name,lengths", [
    # V4-Pro CSA decode: full 128K, L mod 4 = 1, vis = 512 < k = 1024, L < n_win
    ("csa_decode_128k", [131072, 70001, 2050, 77]),
    # FP8 / BF16-RoPE entries and FP4 indexer at up to 64K tokens
    ("csa_decode_1m_mixed", [65536, 40003, 3000, 130]),
    # HCA (m' = 128): vis = 0 on the shortest, L mod 128 != 0 on the second
    ("hca_decode_1m", [262144, 100001, 129, 50]),
])
def test_decode_batch_at_mixed_lengths(name, lengths):
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import path as P
    cfg = synth.scaled(name, B=len(lengths), lengths=lengths)
    x = synth.make_inputs(cfg, seed=3, device=DEV)
    buf = P.Buffers()
    out = P.forward(cfg, x, buf)
    torch.cuda.synchronize()
    K.device_error()
    xn = _host(x)
    tol = TOL_MIXED if cfg["dtype"] == "mixed" else TOL_BF16
    m, k = cfg["m"], cfg.get("k")
    for b, L in enumerate(lengths):
        t = L - 1
        assert int(xn["q_pos"][b, 0]) == t
        if cfg["kind"].startswith("csa"):
            res = OP.run_rows(cfg, xn, b, [0], selected=[buf.idx[b, 0].cpu().numpy()])
            got_s = f64(buf.scores[b, 0])
            assert_scores_close(got_s, res["scores"][0], f"{name} L={L} scores")
            vis = min(cfg["N"], O.visible_count(t, m))
            n = min(k, vis)
            want = np.sort(O.topk_select(got_s, k, vis))
            got_i = buf.idx[b, 0].cpu().numpy()
            assert np.array_equal(got_i[:n], want), f"{name} L={L} top-k"
            assert np.all(got_i[n:] == -1)
        else:
            res = OP.run_rows(cfg, xn, b, [0])
        assert_close(f64(out[b, 0]), res["out"][0], tol, tol, f"{name} L={L} attend")


def test_index_topk_rows_at_their_own_positions():
    # several query rows per sequence at arbitrary (not consecutive) positions:
    # the two-call path (csa_index + csa_topk) reads each row's position
    import compressed_sparse_long_05_b300 as K
    B, Tq, N, H, c, m, k = 2, 5, 3000, 64, 128, 4, 256
    g = torch.Generator(device=DEV).manual_seed(11)
    qI = (torch.randn((B, Tq, H, c), generator=g, device=DEV) / c ** 0.5).to(torch.bfloat16)
    Kt = (torch.randn((B, N, c), generator=g, device=DEV) / c ** 0.5).to(torch.bfloat16)
    w = torch.rand((B, Tq, H), generator=g, device=DEV) / H
    pos = [[11999, 3, 1025, 400, 7000], [0, 11998, 5000, 1027, 64]]
    q_pos = torch.tensor(pos, dtype=torch.int32, device=DEV)
    s = K.csa_index(qI, w, Kt, m, q_pos)
    idx = K.csa_topk(s, k, m, q_pos)
    torch.cuda.synchronize()
    K.device_error()
    for b in range(B):
        ref = O.index_scores(f64(qI[b]), f64(w[b]), f64(Kt[b]), np.array(pos[b]), m)
        for i in range(Tq):
            assert_scores_close(f64(s[b, i]), ref[i], f"b={b} i={i}")
            vis = min(N, O.visible_count(pos[b][i], m))
            n = min(k, vis)
            want = np.sort(O.topk_select(f64(s[b, i]), k, vis))
            assert np.array_equal(idx[b, i].cpu().numpy()[:n], want)
            assert np.all(idx[b, i].cpu().numpy()[n:] == -1)


def test_negative_position_is_flagged_and_sees_nothing():
    # a position below 0 is an input error the host cannot see: the kernels
    # flag it in the device error word and the row selects nothing
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import CsaError
    B, Tq, N, k, m = 1, 2, 500, 16, 4
    scores = torch.rand((B, Tq, N), device=DEV)
    q_pos = torch.tensor([[-5, 1999]], dtype=torch.int32, device=DEV)
    idx = K.csa_topk(scores, k, m, q_pos)
    torch.cuda.synchronize()
    with pytest.raises(CsaError) as e:
        K.device_error()
    assert e.value.status == 6                        # CSA_ERR_DEVICE (bad-index bit)
    assert np.all(idx[0, 0].cpu().numpy() == -1)
    want = np.sort(O.topk_select(f64(scores[0, 1]), k, 500))
    assert np.array_equal(idx[0, 1].cpu().numpy(), want)
    K.device_error()                                  # the word was cleared by the read
