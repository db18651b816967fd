"""GPU parity of each C-ABI stage against the float64 oracle on the same inputs."""

import numpy as np
import pytest
import torch

import synth
from oracle import csa_oracle as O
from tests.parity import (TOL_BF16, TOL_F32, assert_close, assert_scores_close, f64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    import compressed_sparse_long_05_b300 as k
    k.lib()
    return k


def _gen(seed):
    return torch.Generator(device=DEV).manual_seed(seed)


def _randn(shape, dtype, seed, scale=1.0):
    return (torch.randn(shape, generator=_gen(seed), device=DEV) * scale).to(dtype)


# ----------------------------------------------------------------------------
# compress
# ----------------------------------------------------------------------------


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,T,d,m", [(1, 256, 128, 4), (2, 1037, 512, 4), (1, 3, 64, 4),
                                     (2, 999, 512, 128), (1, 77, 64, 1), (1, 1000, 256, 16)])
def test_compress_csa(K, dtype, B, T, d, m):
    Ca, Cb = _randn((B, T, d), dtype, 1), _randn((B, T, d), dtype, 2)
    Za, Zb = _randn((B, T, d), dtype, 3), _randn((B, T, d), dtype, 4)
    out = K.csa_compress(Ca, Za, m, Cb=Cb, Zb=Zb)
    torch.cuda.synchronize()
    N = T // m
    assert out.shape == (B, N, d)
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for b in range(B):
        ref = O.compress_csa(f64(Ca[b]), f64(Cb[b]), f64(Za[b]), f64(Zb[b]), m)
        assert_close(f64(out[b]), ref, tol, tol, f"compress csa b={b}")
    K.device_error()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,T,d,m", [(1, 1000, 512, 128), (2, 300, 128, 128), (1, 50, 64, 7)])
def test_compress_hca(K, dtype, B, T, d, m):
    C, Z = _randn((B, T, d), dtype, 5), _randn((B, T, d), dtype, 6)
    out = K.csa_compress(C, Z, m)
    torch.cuda.synchronize()
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for b in range(B):
        assert_close(f64(out[b]), O.compress_hca(f64(C[b]), f64(Z[b]), m), tol, tol, "hca")


def test_compress_bias(K):
    B, T, d, m = 1, 64, 128, 4
    Ca, Cb, Za, Zb = (_randn((B, T, d), torch.float32, s) for s in (7, 8, 9, 10))
    Ba, Bb = _randn((m, d), torch.float32, 11), _randn((m, d), torch.float32, 12)
    out = K.csa_compress(Ca, Za, m, Cb=Cb, Zb=Zb, Ba=Ba, Bb=Bb)
    torch.cuda.synchronize()
    ref = O.compress_csa(f64(Ca[0]), f64(Cb[0]), f64(Za[0]), f64(Zb[0]), m, Ba=f64(Ba), Bb=f64(Bb))
    assert_close(f64(out[0]), ref, TOL_F32, TOL_F32, "bias")


# ----------------------------------------------------------------------------
# index (float32 path)
# ----------------------------------------------------------------------------


def test_index_f32(K):
    cfg = synth.get("tiny_csa_prefill_f32")
    x = synth.make_inputs(cfg, device=DEV)
    s = K.csa_index(x["qI"], x["w"], x["K"], cfg["m"], cfg["q_pos0"])
    torch.cuda.synchronize()
    ref = O.index_scores(f64(x["qI"][0]), f64(x["w"][0]), f64(x["K"][0]), np.arange(cfg["T"]), cfg["m"])
    for t in range(cfg["T"]):
        assert_scores_close(f64(s[0, t]), ref[t], f"row {t}")


# ----------------------------------------------------------------------------
# top-k
# ----------------------------------------------------------------------------


def _check_topk(scores, idx, k, m, q_pos0):
    sc, ix = f64(scores), idx.cpu().numpy()
    B, Tq, N = sc.shape
    for b in range(B):
        for i in range(Tq):
            vis = min(N, O.visible_count(q_pos0 + i, m))
            ref = np.sort(O.topk_select(sc[b, i], k, vis))
            n = min(k, vis)
            got = ix[b, i]
            assert np.array_equal(got[:n], ref), f"row ({b},{i}) vis={vis}"
            assert np.all(got[n:] == -1)


@pytest.mark.parametrize("B,Tq,N,k,q_pos0,levels", [
    (1, 300, 64, 16, 0, 0),          # prefill rows, vis <= k on the first rows
    (1, 64, 2048, 100, 8000, 7),     # ties from few distinct values
    (4, 1, 32768, 1024, 131071, 0),  # decode rows, cluster of 16 CTAs
    (3, 2, 40000, 1024, 159990, 3),  # several rows, ties, ragged slices
    (1, 40, 9000, 4096, 35990, 0),   # large k
    (2, 3, 20000, 7, 79999, 1),      # every score equal: lowest indices win
])
def test_topk(K, B, Tq, N, k, q_pos0, levels):
    g = _gen(21)
    if levels:
        scores = torch.randint(0, levels, (B, Tq, N), generator=g, device=DEV).float()
    else:
        scores = torch.rand((B, Tq, N), generator=g, device=DEV)
    idx = K.csa_topk(scores, k, 4, q_pos0)
    torch.cuda.synchronize()
    _check_topk(scores, idx, k, 4, q_pos0)


def test_topk_negative_and_inf_scores(K):
    g = _gen(22)
    scores = torch.randn((2, 5, 3000), generator=g, device=DEV)
    scores[:, :, ::7] = -float("inf")
    scores[0, 0, 5] = float("inf")
    idx = K.csa_topk(scores, 50, 4, 11990)
    torch.cuda.synchronize()
    _check_topk(scores, idx, 50, 4, 11990)


# ----------------------------------------------------------------------------
# attention (float32 path)
# ----------------------------------------------------------------------------


def test_attend_f32_tiny(K):
    cfg = synth.get("tiny_csa_prefill_f32")
    x = synth.make_inputs(cfg, device=DEV)
    m = cfg["m"]
    ent = K.csa_compress(x["Ca"], x["Za"], m, Cb=x["Cb"], Zb=x["Zb"])
    s = K.csa_index(x["qI"], x["w"], x["K"], m, 0)
    idx = K.csa_topk(s, cfg["k"], m, 0)
    out = K.csa_attend(x["q"], ent, idx, x["win"], x["sink"], m, cfg["n_win"], 0, 0, cfg["r"])
    torch.cuda.synchronize()
    ent64, win64, q64, sink = f64(ent[0]), f64(x["win"][0]), f64(x["q"][0]), f64(x["sink"])
    ix = idx[0].cpu().numpy()
    for t in range(cfg["T"]):
        ref = O.csa_attend_token(q64[t], t, ent64, ix[t], win64, 0, sink, m, cfg["n_win"],
                                 cfg["r"], cfg["rope_base"])
        assert_close(f64(out[0, t]), ref, TOL_F32, TOL_F32, f"t={t}")
    K.device_error()


def test_hca_attend_f32(K):
    B, T, d, r, n_h, m, n_win = 2, 700, 128, 32, 4, 128, 16
    C, Z = _randn((B, T, d), torch.float32, 31), _randn((B, T, d), torch.float32, 32)
    q = _randn((B, T, n_h, d), torch.float32, 33)
    win = _randn((B, T, d), torch.float32, 34)
    sink = _randn((n_h,), torch.float32, 35)
    ent = K.csa_compress(C, Z, m)
    out = K.hca_attend(q, ent, win, sink, m, n_win, 0, 0, r)
    torch.cuda.synchronize()
    for b in range(B):
        e64, w64, q64 = f64(ent[b]), f64(win[b]), f64(q[b])
        for t in (0, 1, 126, 127, 128, 300, 699):
            ref = O.hca_attend_token(q64[t], t, e64, w64, 0, f64(sink), m, n_win, r, 1e4)
            assert_close(f64(out[b, t]), ref, TOL_F32, TOL_F32, f"b={b} t={t}")


# ----------------------------------------------------------------------------
# index (bf16, tcgen05 path)
# ----------------------------------------------------------------------------


@pytest.mark.parametrize("B,Tq,N,H,c,q_pos0", [
    (2, 1, 5000, 64, 128, 19999),      # decode rows, ragged last tile
    (1, 1030, 257, 64, 128, 0),        # causal prefill, ragged query groups
    (1, 9, 300, 64, 128, 700),         # mid-sequence query block
    (3, 5, 1000, 64, 64, 3990),        # c = 64
    (1, 33, 700, 32, 128, 2700),       # H = 32
    (1, 6, 640, 128, 128, 2540),       # H = 128
])
def test_index_bf16(K, B, Tq, N, H, c, q_pos0):
    m = 4
    qI = _randn((B, Tq, H, c), torch.bfloat16, 41, scale=c ** -0.5)
    Kt = _randn((B, N, c), torch.bfloat16, 42, scale=c ** -0.5)
    w = torch.rand((B, Tq, H), generator=_gen(43), device=DEV) / H
    s = K.csa_index(qI, w, Kt, m, q_pos0)
    torch.cuda.synchronize()
    K.device_error()
    for b in range(B):
        ref = O.index_scores(f64(qI[b]), f64(w[b]), f64(Kt[b]), q_pos0 + np.arange(Tq), m)
        got = f64(s[b])
        for i in range(Tq):
            assert_scores_close(got[i], ref[i], f"b={b} row {i}")
