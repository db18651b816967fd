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
    s = K.csa_index(x["qI"], x["w"], x["K"], cfg["m"], x["q_pos"])
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
    (1, 1, 40000, 4096, 159999, 3),  # the keys equal to the k-th span three ranks' slices
    (1, 40, 9000, 4096, 35990, 0),   # large k
    (2, 3, 20000, 7, 79999, 1),      # every score equal: lowest indices win
    (2, 1, 262144, 1024, 1048575, 0),   # 1M-context decode rows: 16-CTA clusters
    (1, 2, 262144, 1024, 1048574, 2),   # ties across a 16-CTA cluster
    (1, 1, 600000, 1024, 2399999, 0),   # beyond 16 x 32768 keys: 8-bit radix over 16 CTAs
    (1, 3, 70001, 333, 280003, 0),      # odd N: unaligned row starts, ragged slices
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


# ----------------------------------------------------------------------------
# attention (bf16, tcgen05 path)
# ----------------------------------------------------------------------------


def _rms(shape, seed):
    x = torch.randn(shape, generator=_gen(seed), device=DEV)
    return (x * torch.rsqrt(x.square().mean(-1, keepdim=True))).to(torch.bfloat16)


def _attend_case(K, B, Tq, N, k, q_pos0, T_win, win_base, n_h=128, m=4, n_win=128, dense=False,
                 rows=None, seed=50):
    d, r = 512, 64
    q = _rms((B, Tq, n_h, d), seed)
    ent = _rms((B, N, d), seed + 1)
    win = _rms((B, T_win, d), seed + 2)
    sink = torch.randn((n_h,), generator=_gen(seed + 3), device=DEV)
    if dense:
        out = K.hca_attend(q, ent, win, sink, m, n_win, win_base, q_pos0, r)
        idx = None
    else:
        scores = torch.rand((B, Tq, N), generator=_gen(seed + 4), device=DEV)
        idx = K.csa_topk(scores, k, m, q_pos0)
        out = K.csa_attend(q, ent, idx, win, sink, m, n_win, win_base, q_pos0, r)
    torch.cuda.synchronize()
    K.device_error()
    e64, w64, s64 = f64(ent), f64(win), f64(sink)
    rows = range(Tq) if rows is None else rows
    for b in range(B):
        for i in rows:
            t = q_pos0 + i
            q64 = f64(q[b, i])
            if dense:
                ref = O.hca_attend_token(q64, t, e64[b], w64[b], win_base, s64, m, n_win, r, 1e4)
            else:
                ref = O.csa_attend_token(q64, t, e64[b], idx[b, i].cpu().numpy(), w64[b], win_base,
                                         s64, m, n_win, r, 1e4)
            assert_close(f64(out[b, i]), ref, TOL_BF16, TOL_BF16, f"b={b} i={i} t={t}")


def test_attend_bf16_decode_split(K):
    # few query rows: rows split over CTAs, partials merged by the combine kernel
    N = 3000
    L = 4 * N
    _attend_case(K, B=2, Tq=1, N=N, k=1024, q_pos0=L - 1, T_win=128, win_base=L - 128)


def test_attend_bf16_decode_small_k(K):
    N = 800
    _attend_case(K, B=3, Tq=2, N=N, k=200, q_pos0=4 * N - 2, T_win=129, win_base=4 * N - 129, seed=60)


def test_attend_bf16_prefill_prerotated(K):
    # many query rows: one chunk per row, rows rotated once up front, early rows
    # see fewer than k entries and fewer than n_win window tokens
    T = 700
    _attend_case(K, B=1, Tq=T, N=T // 4, k=64, q_pos0=0, T_win=T, win_base=0,
                 rows=[0, 1, 3, 4, 5, 127, 128, 255, 256, 257, 400, 511, 600, 699], seed=70)


def test_attend_bf16_rotate_in_smem_single_chunk(K):
    # many query rows over a long cache: in-kernel RoPE of gathered rows
    N = 20000
    _attend_case(K, B=1, Tq=160, N=N, k=256, q_pos0=4 * N - 160, T_win=300,
                 win_base=4 * N - 300, rows=[0, 1, 77, 159], seed=80)


def test_hca_attend_bf16_decode(K):
    N = 2500
    L = 128 * N
    _attend_case(K, B=2, Tq=1, N=N, k=0, q_pos0=L - 1, T_win=128, win_base=L - 128, m=128,
                 dense=True, seed=90)


def test_hca_attend_bf16_decode_cluster_partials(K):
    # 33 row chunks per head group (8320 rows): more than one co-resident cluster
    # can hold, so clusters of fewer chunks merge into partials that the combine
    # kernel finishes.  The scratch size shows the plan: far fewer 128 KB
    # partials than the 132 work items.
    from compressed_sparse_long_05_b300 import _lib
    N = 8192
    L = 128 * N
    ws = _lib.lib().csa_attend_workspace_size(2, 1, N, 0, 128, 128, 512, 64, 128, 128, 1, 1, 1)
    part = 64 * 512 * 4
    assert 0 < ws < 132 * part
    assert ws // part < 66
    _attend_case(K, B=2, Tq=1, N=N, k=0, q_pos0=L - 1, T_win=128, win_base=L - 128, m=128,
                 dense=True, seed=95)


def test_hca_attend_bf16_prefill(K):
    T = 1100
    _attend_case(K, B=1, Tq=T, N=T // 128, k=0, q_pos0=0, T_win=T, win_base=0, m=128, dense=True,
                 rows=[0, 5, 126, 127, 128, 129, 300, 1023, 1099], seed=100)


def test_attend_bf16_heads_64(K):
    N = 500
    _attend_case(K, B=1, Tq=3, N=N, k=128, q_pos0=4 * N - 3, T_win=140, win_base=4 * N - 140,
                 n_h=64, seed=110)


# ----------------------------------------------------------------------------
# index (FP4 e2m1 + e4m3 block scales, block-scaled tcgen05 path)
# ----------------------------------------------------------------------------


def _fp4(shape, seed, scale):
    from synth.generate import quantise_fp4_blocks
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(shape, generator=g) * scale
    packed, sf = quantise_fp4_blocks(v)
    return packed.to(DEV), sf.to(DEV)


@pytest.mark.parametrize("B,Tq,N,H,q_pos0", [
    (2, 1, 5000, 64, 19999),      # decode rows, ragged last tile
    (3, 3, 1001, 64, 3999),       # odd N: scale rows of batch row 1 start on an odd row
    (1, 300, 257, 64, 0),         # causal prefill, vis < one tile for most rows
    (1, 7, 700, 128, 2790),       # H = 128
    (1, 9, 640, 32, 2550),        # H = 32, four queries per group
])
def test_index_fp4(K, B, Tq, N, H, q_pos0):
    m, c = 4, 128
    q_p, q_sf = _fp4((B, Tq, H, c), 44, c ** -0.5)
    k_p, k_sf = _fp4((B, N, c), 45, c ** -0.5)
    w = torch.rand((B, Tq, H), generator=_gen(46), device=DEV) / H
    s = K.csa_index(q_p, w, k_p, m, q_pos0, qI_sf=q_sf, K_sf=k_sf)
    torch.cuda.synchronize()
    K.device_error()
    for b in range(B):
        qd = O.decode_fp4_blocks(q_p[b].cpu().numpy(), q_sf[b].cpu().numpy())
        kd = O.decode_fp4_blocks(k_p[b].cpu().numpy(), k_sf[b].cpu().numpy())
        ref = O.index_scores(qd, f64(w[b]), kd, q_pos0 + np.arange(Tq), m)
        got = f64(s[b])
        for i in range(Tq):
            assert_scores_close(got[i], ref[i], f"b={b} row {i}")


# ----------------------------------------------------------------------------
# attention over FP8 (e4m3 + per-row scale) / BF16-RoPE rows
# ----------------------------------------------------------------------------


def _mixed(rows_bf16):
    from synth.generate import quantise_mixed_entries
    return quantise_mixed_entries(rows_bf16.float(), 64)


@pytest.mark.parametrize("B,Tq,N,k,split", [(2, 1, 3000, 1024, True), (1, 40, 2000, 256, False)])
def test_attend_mixed_rows(K, B, Tq, N, k, split):
    from tests.parity import TOL_MIXED
    d, r, n_h, m, n_win = 512, 64, 128, 4, 128
    q_pos0 = 4 * N - Tq
    T_win = n_win + Tq
    win_base = 4 * N - T_win
    q = _rms((B, Tq, n_h, d), 120)
    ent = _mixed(_rms((B, N, d), 121))
    win = _mixed(_rms((B, T_win, d), 122))
    sink = torch.randn((n_h,), generator=_gen(123), device=DEV)
    scores = torch.rand((B, Tq, N), generator=_gen(124), device=DEV)
    idx = K.csa_topk(scores, k, m, q_pos0)
    out = K.csa_attend(q, ent, idx, win, sink, m, n_win, win_base, q_pos0, r)
    torch.cuda.synchronize()
    K.device_error()
    for b in range(B):
        e64 = O.decode_mixed_entries(ent[0][b].cpu().numpy(), ent[1][b].cpu().numpy(), f64(ent[2][b]))
        w64 = O.decode_mixed_entries(win[0][b].cpu().numpy(), win[1][b].cpu().numpy(), f64(win[2][b]))
        for i in sorted({0, Tq // 2, Tq - 1}):
            t = q_pos0 + i
            ref = O.csa_attend_token(f64(q[b, i]), t, e64, idx[b, i].cpu().numpy(), w64, win_base,
                                     f64(sink), m, n_win, r, 1e4)
            assert_close(f64(out[b, i]), ref, TOL_MIXED, TOL_MIXED, f"b={b} i={i}")


# ----------------------------------------------------------------------------
# index + top-k in one call (decode rows: histogram built by the index kernel)
# ----------------------------------------------------------------------------


@pytest.mark.parametrize("fmt,B,N,k", [
    ("bf16", 3, 32768, 1024),       # 128K-context decode rows over a 16-CTA cluster
    ("bf16", 2, 700, 1024),         # every visible entry selected (vis < k)
    ("bf16", 1, 5001, 333),         # odd N
    ("fp4", 2, 262144, 1024),       # 1M-context decode rows over an 8-CTA cluster
    ("fp4", 1, 40001, 512),         # past 32768: cluster of 8, ragged slices
    ("fp4", 200, 3000, 512),        # more rows than SMs: CTAs flush two rows' histograms
    ("bf16", 200, 3000, 512),
])
def test_index_topk_fused_matches_separate_calls(K, fmt, B, N, k):
    m, H, c = 4, 64, 128
    q_pos0 = 4 * N - 1
    w = torch.rand((B, 1, H), generator=_gen(47), device=DEV) / H
    if fmt == "bf16":
        qI = _randn((B, 1, H, c), torch.bfloat16, 48, scale=c ** -0.5)
        Kt = _randn((B, N, c), torch.bfloat16, 49, scale=c ** -0.5)
        q_sf = k_sf = None
    else:
        qI, q_sf = _fp4((B, 1, H, c), 48, c ** -0.5)
        Kt, k_sf = _fp4((B, N, c), 49, c ** -0.5)
    s_ref = K.csa_index(qI, w, Kt, m, q_pos0, qI_sf=q_sf, K_sf=k_sf)
    i_ref = K.csa_topk(s_ref, k, m, q_pos0)
    s, i, _ = K.csa_index_topk(qI, w, Kt, k, m, q_pos0, qI_sf=q_sf, K_sf=k_sf)
    torch.cuda.synchronize()
    K.device_error()
    assert torch.equal(s, s_ref)
    assert torch.equal(i, i_ref)
    _check_topk(s, i, k, m, q_pos0)


def test_index_topk_every_score_equal(K):
    # w = 0 makes every visible score 0: the first-digit bin the index kernel
    # counted holds the whole row, every radix pass finds one digit, and the
    # lowest indices win across the cluster's slices
    m, H, c, k, B, N = 4, 64, 128, 1024, 2, 32768
    q_pos0 = 4 * N - 1
    w = torch.zeros((B, 1, H), device=DEV)
    qI = _randn((B, 1, H, c), torch.bfloat16, 68, scale=c ** -0.5)
    Kt = _randn((B, N, c), torch.bfloat16, 69, scale=c ** -0.5)
    s, i, _ = K.csa_index_topk(qI, w, Kt, k, m, q_pos0)
    torch.cuda.synchronize()
    K.device_error()
    assert int(s.count_nonzero()) == 0
    assert torch.equal(i.cpu(), torch.arange(k, dtype=i.dtype).expand(B, 1, k))
    _check_topk(s, i, k, m, q_pos0)


@pytest.mark.parametrize("fmt,B,N", [("bf16", 3, 32768), ("bf16", 2, 700), ("fp4", 2, 40001)])
def test_index_topk_workspace_left_zero(K, fmt, B, N):
    # the histograms in the workspace start zero and every call leaves them zero,
    # so repeated calls on one workspace agree with the first
    m, H, c, k = 4, 64, 128, 1024
    q_pos0 = 4 * N - 1
    w = torch.rand((B, 1, H), generator=_gen(57), device=DEV) / H
    if fmt == "bf16":
        qI = _randn((B, 1, H, c), torch.bfloat16, 58, scale=c ** -0.5)
        Kt = _randn((B, N, c), torch.bfloat16, 59, scale=c ** -0.5)
        q_sf = k_sf = None
    else:
        qI, q_sf = _fp4((B, 1, H, c), 58, c ** -0.5)
        Kt, k_sf = _fp4((B, N, c), 59, c ** -0.5)
    s0, i0, ws = K.csa_index_topk(qI, w, Kt, k, m, q_pos0, qI_sf=q_sf, K_sf=k_sf)
    torch.cuda.synchronize()
    K.device_error()
    assert ws is not None and int(ws.count_nonzero()) == 0
    for _ in range(2):
        s, i, ws = K.csa_index_topk(qI, w, Kt, k, m, q_pos0, qI_sf=q_sf, K_sf=k_sf, ws=ws)
        torch.cuda.synchronize()
        K.device_error()
        assert torch.equal(s, s0) and torch.equal(i, i0)
        assert int(ws.count_nonzero()) == 0


@pytest.mark.parametrize("kind,m,T,ents", [("csa", 4, 4096, [0, 1, 2, 511, 1023]), ("hca", 128, 4096, [0, 1, 31])])
def test_compress_entry_matches_whole_sequence(K, kind, m, T, ents):
    # the entry a closing block adds during decode equals that entry of the
    # whole-sequence compression (oracle)
    from compressed_sparse_long_05_b300 import path as P
    B, d = 2, 512
    Ca = _rms((B, T, d), 140)
    Za = _randn((B, T, d), torch.bfloat16, 141)
    Cb = _rms((B, T, d), 142) if kind == "csa" else None
    Zb = _randn((B, T, d), torch.bfloat16, 143) if kind == "csa" else None
    for b in range(B):
        if kind == "csa":
            ref = O.compress_csa(f64(Ca[b]), f64(Cb[b]), f64(Za[b]), f64(Zb[b]), m)
        else:
            ref = O.compress_hca(f64(Ca[b]), f64(Za[b]), m)
        for i in ents:
            got = P.compress_entry(i, m, Ca, Za, Cb=Cb, Zb=Zb)
            torch.cuda.synchronize()
            assert_close(f64(got[b]), ref[i], TOL_BF16, TOL_BF16, f"{kind} entry {i} b={b}")


# ----------------------------------------------------------------------------
# producer side: RMSNorm and RoPE pre-rotation in the compression epilogue,
# attention on pre-rotated entries, indexer keys compressed at d = c_I
# ----------------------------------------------------------------------------


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,T,d,m,overlap,norm,weight,rope", [
    (2, 1037, 512, 4, True, True, False, 64),     # CSA, V4 entry shape, ragged tail
    (1, 999, 512, 128, False, True, True, 64),    # HCA, weighted RMSNorm
    (1, 515, 128, 4, True, False, False, 0),      # indexer keys: d = c_I, plain
    (1, 300, 64, 4, True, True, False, 0),        # small d: partial last warp
    (1, 260, 128, 1, False, True, False, 32),     # m = 1
])
def test_compress_epilogue(K, dtype, B, T, d, m, overlap, norm, weight, rope):
    Ca, Za = _randn((B, T, d), dtype, 150), _randn((B, T, d), dtype, 151)
    Cb = _randn((B, T, d), dtype, 152) if overlap else None
    Zb = _randn((B, T, d), dtype, 153) if overlap else None
    w = (torch.rand((d,), generator=_gen(154), device=DEV) + 0.5) if weight else None
    eps = 1e-6
    out = K.csa_compress(Ca, Za, m, Cb=Cb, Zb=Zb, rms_norm=norm, norm_eps=eps, norm_weight=w,
                         rope_dims=rope)
    torch.cuda.synchronize()
    K.device_error()
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    for b in range(B):
        if overlap:
            ref = O.compress_csa(f64(Ca[b]), f64(Cb[b]), f64(Za[b]), f64(Zb[b]), m)
        else:
            ref = O.compress_hca(f64(Ca[b]), f64(Za[b]), m)
        if norm:
            ref = O.rms_norm(ref, None if w is None else f64(w), eps)
        if rope:
            ref = O.rope_rotate(ref, O.entry_position(np.arange(ref.shape[0]), m), rope, 1e4)
        assert_close(f64(out[b]), ref, tol, tol, f"compress epilogue b={b}")


def test_compress_epilogue_rejects_bad_options(K):
    Ca, Za = _randn((1, 64, 128), torch.bfloat16, 155), _randn((1, 64, 128), torch.bfloat16, 156)
    from compressed_sparse_long_05_b300 import CsaError
    with pytest.raises(CsaError):
        K.csa_compress(Ca, Za, 4, rope_dims=12)      # not a multiple of the 8-element vector
    with pytest.raises(CsaError):
        K.csa_compress(Ca, Za, 4, rope_dims=7)       # odd


@pytest.mark.parametrize("case", ["decode", "prefill", "hca_decode", "f32"])
def test_attend_pre_rotated_entries(K, case):
    # entries stored rotated at their positions (compression epilogue) give the
    # oracle's attention over the unrotated entries: decode rotates each
    # gathered row by -t only, prefill skips its rotation pre-pass for them
    d, r, m = 512, 64, 4
    n_h, n_win, dt = 128, 128, torch.bfloat16
    if case == "decode":
        B, Tq, T, k = 2, 1, 12000, 1024
    elif case == "prefill":
        B, Tq, T, k = 1, 600, 600, 64
    elif case == "hca_decode":
        B, Tq, T, k, m = 2, 1, 128 * 900, 0, 128
    else:
        B, Tq, T, k, d, r, n_h, n_win, dt = 1, 200, 200, 16, 128, 32, 4, 16, torch.float32
    Ca, Za = _rms((B, T, d), 160).to(dt), _randn((B, T, d), dt, 161)
    if m == 4:
        Cb, Zb = _rms((B, T, d), 162).to(dt), _randn((B, T, d), dt, 163)
    else:
        Cb = Zb = None
    ent_rot = K.csa_compress(Ca, Za, m, Cb=Cb, Zb=Zb, rope_dims=r)
    ent = K.csa_compress(Ca, Za, m, Cb=Cb, Zb=Zb)
    N = T // m
    q_pos0 = T - Tq
    T_win = n_win + Tq if Tq == 1 else T
    win_base = T - T_win
    q = _rms((B, Tq, n_h, d), 164).to(dt)
    win = _rms((B, T_win, d), 165).to(dt)
    sink = torch.randn((n_h,), generator=_gen(166), device=DEV)
    if k:
        scores = torch.rand((B, Tq, N), generator=_gen(167), device=DEV)
        idx = K.csa_topk(scores, k, m, q_pos0)
        out = K.csa_attend(q, ent_rot, idx, win, sink, m, n_win, win_base, q_pos0, r,
                           entries_rotated=True)
    else:
        out = K.hca_attend(q, ent_rot, win, sink, m, n_win, win_base, q_pos0, r, entries_rotated=True)
    torch.cuda.synchronize()
    K.device_error()
    tol = TOL_F32 if dt == torch.float32 else TOL_BF16
    for b in range(B):
        e64, w64 = f64(ent[b]), f64(win[b])
        for i in sorted({0, Tq // 2, Tq - 1}):
            t = q_pos0 + i
            if k:
                ref = O.csa_attend_token(f64(q[b, i]), t, e64, idx[b, i].cpu().numpy(), w64, win_base,
                                         f64(sink), m, n_win, r, 1e4)
            else:
                ref = O.hca_attend_token(f64(q[b, i]), t, e64, w64, win_base, f64(sink), m, n_win, r,
                                         1e4)
            assert_close(f64(out[b, i]), ref, tol, tol, f"{case} b={b} i={i}")
