"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each test states which closed form, library routine, invariant or printed fact
it uses.  The sources are the DeepSeek-V4 report pages: the Chinese translation
(blog.uika.cn, §2.3.1-§2.3.4) and the paper notes (awesome.papernotes.org,
"关键设计 1" / "关键设计 2").
"""

import math

import numpy as np
import pytest
import torch
from scipy.special import expit

from oracle import csa_oracle as O

RNG = np.random.default_rng(1234)


def rnd(*shape):
    return RNG.standard_normal(shape)


# ----------------------------------------------------------------------------
# compression
# ----------------------------------------------------------------------------


def test_compress_equal_logits_is_block_mean():
    # Equal Z makes every softmax weight 1/(rows): entry i is the mean of the
    # 2m rows {a-rows of block i, b-rows of block i-1}; entry 0 the mean of m rows.
    m, T, d = 4, 37, 6
    Ca, Cb = rnd(T, d), rnd(T, d)
    Z = np.full((T, d), 0.3)
    out = O.compress_csa(Ca, Cb, Z, Z, m)
    N = T // m
    assert out.shape == (N, d)
    np.testing.assert_allclose(out[0], Ca[0:m].mean(axis=0), rtol=0, atol=1e-14)
    for i in range(1, N):
        rows = np.concatenate([Ca[m * i:m * (i + 1)], Cb[m * (i - 1):m * i]])
        np.testing.assert_allclose(out[i], rows.mean(axis=0), rtol=0, atol=1e-14)


def test_compress_two_row_closed_form():
    # m = 1: entry i mixes a_i and b_{i-1} with weights sigmoid(za - zb), sigmoid(zb - za).
    T, d = 9, 3
    Ca, Cb, Za, Zb = rnd(T, d), rnd(T, d), rnd(T, d), rnd(T, d)
    out = O.compress_csa(Ca, Cb, Za, Zb, 1)
    np.testing.assert_allclose(out[0], Ca[0], atol=1e-15)
    for i in range(1, T):
        wa = expit(Za[i] - Zb[i - 1])
        np.testing.assert_allclose(out[i], wa * Ca[i] + (1 - wa) * Cb[i - 1], atol=1e-14)


def test_compress_overlap_locality():
    # C^a / Z^a of block j feed entry j only; C^b / Z^b of block j feed entry j+1 only;
    # tail tokens (T mod m) feed nothing.
    m, T, d = 4, 30, 5
    Ca, Cb, Za, Zb = rnd(T, d), rnd(T, d), rnd(T, d), rnd(T, d)
    base = O.compress_csa(Ca, Cb, Za, Zb, m)
    N = T // m
    for j in range(N):
        blk = slice(m * j, m * (j + 1))
        for name in ("Ca", "Za", "Cb", "Zb"):
            args = dict(Ca=Ca.copy(), Cb=Cb.copy(), Za=Za.copy(), Zb=Zb.copy())
            args[name][blk] += rnd(m, d)      # not a per-channel constant (that is a softmax shift)
            out = O.compress_csa(args["Ca"], args["Cb"], args["Za"], args["Zb"], m)
            changed = np.nonzero(np.abs(out - base).max(axis=1) > 1e-12)[0].tolist()
            target = j if name in ("Ca", "Za") else j + 1
            assert changed == ([target] if target < N else []), (name, j, changed)
    args = dict(Ca=Ca.copy(), Cb=Cb.copy(), Za=Za.copy(), Zb=Zb.copy())
    for v in args.values():
        v[N * m:] += 5.0
    np.testing.assert_array_equal(O.compress_csa(**args, m=m), base)


def test_compress_one_hot_selects_row():
    m, T, d = 4, 16, 3
    Ca, Cb = rnd(T, d), rnd(T, d)
    Za, Zb = np.zeros((T, d)), np.zeros((T, d))
    Zb[5, 1] = 800.0           # block 1, in-block row 1, channel 1 -> entry 2
    Za[9, 2] = 800.0           # block 2, row 1, channel 2 -> entry 2
    out = O.compress_csa(Ca, Cb, Za, Zb, m)
    assert out[2, 1] == pytest.approx(Cb[5, 1], abs=1e-12)
    assert out[2, 2] == pytest.approx(Ca[9, 2], abs=1e-12)


def test_compress_shift_invariance_and_bias():
    # Adding one constant per channel to all logits of a group leaves it unchanged;
    # a bias constant over the in-block rows is such a shift.
    m, T, d = 4, 24, 4
    Ca, Cb, Za, Zb = rnd(T, d), rnd(T, d), rnd(T, d), rnd(T, d)
    base = O.compress_csa(Ca, Cb, Za, Zb, m)
    c = rnd(d)
    Za2, Zb2 = Za + c, Zb + c
    np.testing.assert_allclose(O.compress_csa(Ca, Cb, Za2, Zb2, m), base, atol=1e-13)
    Ba = np.tile(c, (m, 1))
    np.testing.assert_allclose(O.compress_csa(Ca, Cb, Za, Zb, m, Ba=Ba, Bb=Ba), base, atol=1e-13)
    # a bias that is large on one in-block row picks that row in every entry
    Ba = np.zeros((m, d)); Ba[3] = 900.0
    Bb = np.zeros((m, d))
    out = O.compress_csa(Ca, Cb, Za, Zb, m, Ba=Ba, Bb=Bb)
    for i in range(T // m):
        np.testing.assert_allclose(out[i], Ca[m * i + 3], atol=1e-12)


def test_compress_hca_block_mean_and_one_hot():
    m, T, d = 128, 300, 4
    C = rnd(T, d)
    out = O.compress_hca(C, np.zeros((T, d)), m)
    assert out.shape == (2, d)
    for i in range(2):
        np.testing.assert_allclose(out[i], C[m * i:m * (i + 1)].mean(axis=0), atol=1e-14)
    Z = np.zeros((T, d)); Z[200, 3] = 900.0
    out = O.compress_hca(C, Z, m)
    assert out[1, 3] == pytest.approx(C[200, 3], abs=1e-12)
    # HCA has no overlap: block 0 never reaches entry 1
    C2 = C.copy(); C2[:m] += 1.0
    np.testing.assert_array_equal(O.compress_hca(C2, np.zeros((T, d)), m)[1], O.compress_hca(C, np.zeros((T, d)), m)[1])


# ----------------------------------------------------------------------------
# indexer
# ----------------------------------------------------------------------------


def test_index_visibility_pattern():
    # entry s is visible to query t iff (s+1) m <= t+1
    m, N, H, c = 4, 10, 3, 5
    qI, K, w = rnd(41, H, c), rnd(N, c), RNG.random((41, H))
    t_pos = np.arange(41)
    I = O.index_scores(qI, w, K, t_pos, m)
    for t in range(41):
        for s in range(N):
            assert np.isneginf(I[t, s]) == ((s + 1) * m > t + 1)
    assert np.all(np.isneginf(I[: m - 1]))      # t < m-1 sees nothing
    assert np.isfinite(I[m - 1, 0]) and np.isneginf(I[m - 1, 1])


def test_index_nonnegative_and_relu():
    # ReLU with non-negative head weights gives non-negative scores; with H=1,
    # w=1, scores(q) + scores(-q) = |q.K| (the ReLU identity relu(x)+relu(-x)=|x|).
    m, N, c = 4, 32, 8
    t_pos = np.array([200])
    qI, K = rnd(1, 5, c), rnd(N, c)
    I = O.index_scores(qI, RNG.random((1, 5)), K, t_pos, m)
    assert np.all(I >= 0)
    q1 = rnd(1, 1, c)
    w1 = np.ones((1, 1))
    both = O.index_scores(q1, w1, K, t_pos, m) + O.index_scores(-q1, w1, K, t_pos, m)
    absdot = np.array([abs(sum(q1[0, 0, j] * K[s, j] for j in range(c))) for s in range(N)])
    np.testing.assert_allclose(both[0], absdot, atol=1e-13)


def test_index_unit_queries_pick_key_columns():
    # q_{t,h} = e_{j_h} makes q.K[s] = K[s, j_h]: score = sum_h w_h relu(K[s, j_h]).
    m, N, c, H = 4, 16, 6, 3
    K = rnd(N, c)
    js = [0, 4, 4]
    qI = np.zeros((1, H, c))
    for h, j in enumerate(js):
        qI[0, h, j] = 1.0
    w = np.array([[0.5, 2.0, -1.0]])
    I = O.index_scores(qI, w, K, np.array([N * m - 1]), m)
    for s in range(N):
        expect = sum(w[0, h] * max(0.0, K[s, j]) for h, j in enumerate(js))
        assert I[0, s] == pytest.approx(expect, abs=1e-14)


def test_index_linear_in_w_and_homogeneous_in_K():
    m, N, c, H = 4, 20, 7, 4
    qI, K = rnd(3, H, c), rnd(N, c)
    t_pos = np.array([79, 50, 3])
    w1, w2 = RNG.random((3, H)), RNG.random((3, H))
    a = O.index_scores(qI, w1 + w2, K, t_pos, m)
    b = O.index_scores(qI, w1, K, t_pos, m) + O.index_scores(qI, w2, K, t_pos, m)
    fin = np.isfinite(a)
    np.testing.assert_allclose(a[fin], b[fin], atol=1e-12)
    c2 = O.index_scores(qI, w1, 2.5 * K, t_pos, m)
    np.testing.assert_allclose(c2[fin], 2.5 * O.index_scores(qI, w1, K, t_pos, m)[fin], atol=1e-12)


# ----------------------------------------------------------------------------
# top-k
# ----------------------------------------------------------------------------


def test_topk_matches_full_sort_with_ties():
    for trial in range(200):
        vis = int(RNG.integers(0, 40))
        k = int(RNG.integers(1, 30))
        s = RNG.integers(0, 6, size=50).astype(np.float64)   # many ties
        got = O.topk_select(s, k, vis)
        ref = sorted(range(vis), key=lambda i: (-s[i], i))[: min(k, vis)]
        assert got.tolist() == ref


def test_topk_k_at_least_vis_returns_all():
    s = rnd(64)
    for vis in (0, 1, 17, 64):
        assert sorted(O.topk_select(s, 64, vis).tolist()) == list(range(vis))


def test_topk_tie_rule_lower_index_wins():
    s = np.array([1.0, 3.0, 3.0, 2.0, 3.0, 3.0])
    assert O.topk_select(s, 3, 6).tolist() == [1, 2, 4]
    assert O.topk_select(s, 2, 6).tolist() == [1, 2]
    assert O.topk_select(np.zeros(9), 4, 9).tolist() == [0, 1, 2, 3]


# ----------------------------------------------------------------------------
# RoPE
# ----------------------------------------------------------------------------


def test_rope_matches_complex_rotation():
    # Pairs as complex numbers: (x0 + i x1) * exp(i p theta_k), theta_k = base^(-2k/r).
    d, r, base = 16, 8, 10000.0
    x = rnd(5, d)
    pos = np.array([0, 1, 7, 4095, 1048575])
    got = O.rope_rotate(x, pos, r, base)
    z = x[:, d - r::2] + 1j * x[:, d - r + 1::2]
    th = np.array([base ** (-2.0 * k / r) for k in range(r // 2)])
    zr = z * np.exp(1j * np.outer(pos, th))
    np.testing.assert_allclose(got[:, d - r::2], zr.real, atol=1e-12)
    np.testing.assert_allclose(got[:, d - r + 1::2], zr.imag, atol=1e-12)
    np.testing.assert_array_equal(got[:, : d - r], x[:, : d - r])


def test_rope_known_value_and_inverse():
    # r = 2: theta_0 = 1, so (1, 0) at p = 1 becomes (cos 1, sin 1).
    v = O.rope_rotate(np.array([[1.0, 0.0]]), np.array([1]), 2, 10000.0)
    np.testing.assert_allclose(v[0], [math.cos(1.0), math.sin(1.0)], atol=1e-15)
    x = rnd(7, 32)
    p = RNG.integers(0, 1 << 20, size=7)
    back = O.rope_rotate(O.rope_rotate(x, p, 16, 10000.0), -p, 16, 10000.0)
    np.testing.assert_allclose(back, x, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(O.rope_rotate(x, p, 16, 10000.0), axis=1),
                               np.linalg.norm(x, axis=1), rtol=1e-13)


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------


def _sdpa(q, k, v):
    """Library attention (torch, float64): softmax(q k^T / sqrt(dk)) v."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None])[0].numpy()


def test_attend_no_rope_no_sink_is_library_attention():
    n_h, d, J = 4, 16, 9
    q, E = rnd(n_h, d), rnd(J, d)
    sink = np.full(n_h, -np.inf)
    got = O.attend_rows(q, 5, E, np.arange(J), sink, 0, 10000.0)
    np.testing.assert_allclose(got, _sdpa(q, E, E), atol=1e-12)


def test_attend_sink_is_an_extra_zero_value_key():
    # The sink adds exp(z'_h) to the denominator only: the same as one extra key
    # with logit z'_h whose value is zero.  Built for the library routine with an
    # extra coordinate: q' = [q, sqrt(d+1) z'], keys [E, 0] and [0, 1], value [E; 0].
    n_h, d, J = 3, 8, 6
    q, E = rnd(n_h, d), rnd(J, d)
    sink = rnd(n_h)
    got = O.attend_rows(q, 0, E, np.arange(J), sink, 0, 10000.0)
    # library logits are scaled by 1/sqrt(d+1); rescale q so they equal q.E/sqrt(d)
    scale = math.sqrt(d + 1) / math.sqrt(d)
    for h in range(n_h):
        qe = np.concatenate([q[h] * scale, [sink[h] * math.sqrt(d + 1)]])[None]
        ke = np.concatenate([np.concatenate([E, np.zeros((J, 1))], 1), [[0] * d + [1.0]]])
        ve = np.concatenate([E, np.zeros((1, d))])
        np.testing.assert_allclose(got[h], _sdpa(qe, ke, ve)[0], atol=1e-12)


def test_attend_sink_at_logsumexp_halves_output_and_single_entry():
    n_h, d, J = 2, 8, 5
    q, E = rnd(n_h, d), rnd(J, d)
    no_sink = O.attend_rows(q, 0, E, np.arange(J), np.full(n_h, -np.inf), 0, 1e4)
    lse = np.log(np.exp(q @ E.T / math.sqrt(d)).sum(axis=1))
    np.testing.assert_allclose(O.attend_rows(q, 0, E, np.arange(J), lse, 0, 1e4), no_sink / 2, atol=1e-13)
    z = rnd(n_h)
    one = O.attend_rows(q, 0, E[:1], np.zeros(1), z, 0, 1e4)
    ell = q @ E[0] / math.sqrt(d)
    np.testing.assert_allclose(one, np.outer(expit(ell - z), E[0]), atol=1e-14)


def test_attend_shift_invariance():
    # Moving the query and every key position by the same offset changes nothing:
    # logits see only p - t and the output is rotated back by -t.
    n_h, d, r, J = 4, 32, 16, 11
    q, E = rnd(n_h, d), rnd(J, d)
    pos = RNG.integers(0, 500, size=J)
    sink = rnd(n_h)
    a = O.attend_rows(q, 600, E, pos, sink, r, 10000.0)
    for delta in (1, 37, 123456):
        b = O.attend_rows(q, 600 + delta, E, pos + delta, sink, r, 10000.0)
        np.testing.assert_allclose(a, b, atol=1e-9)


def test_attend_same_position_keys_reduce_to_plain_attention():
    # All keys at the query's own position: logits are rotation-free and the
    # inverse rotation undoes the value rotation, so the result is plain attention.
    n_h, d, r, J, t = 3, 16, 16, 7, 98765
    q, E = rnd(n_h, d), rnd(J, d)
    got = O.attend_rows(q, t, E, np.full(J, t), np.full(n_h, -np.inf), r, 10000.0)
    np.testing.assert_allclose(got, _sdpa(q, E, E), atol=1e-10)


def test_csa_with_k_at_least_visible_equals_dense():
    # With k >= vis(t), CSA attends every visible compressed entry plus the
    # window: the HCA-style dense computation with the same block size m.
    m, T, d, r, n_h, n_win = 4, 64, 16, 8, 2, 8
    ent = rnd(T // m, d)
    win = rnd(T, d)
    sink = rnd(n_h)
    for t in (0, 3, 4, 17, 63):
        vis = O.visible_count(t, m)
        q = rnd(n_h, d)
        a = O.csa_attend_token(q, t, ent, np.arange(vis), win, 0, sink, m, n_win, r, 1e4)
        b = O.hca_attend_token(q, t, ent, win, 0, sink, m, n_win, r, 1e4)
        np.testing.assert_allclose(a, b, atol=1e-13)
        # -1 padding is ignored
        pad = np.concatenate([np.arange(vis), [-1, -1]])
        c = O.csa_attend_token(q, t, ent, pad, win, 0, sink, m, n_win, r, 1e4)
        np.testing.assert_allclose(a, c, atol=0)


def test_window_membership():
    assert O.window_positions(0, 128).tolist() == [0]
    assert O.window_positions(5, 4).tolist() == [2, 3, 4, 5]
    assert len(O.window_positions(1000, 128)) == 128
    assert O.entry_position(np.array([0, 1, 2]), 4).tolist() == [3, 7, 11]


# ----------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------


def test_decode_e4m3_matches_library_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.decode_e4m3(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_decode_e2m1_table_and_packing():
    # The e2m1 value set of the OCP microscaling formats spec.
    vals = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    np.testing.assert_array_equal(O.decode_e2m1(np.arange(8)), vals)
    np.testing.assert_array_equal(O.decode_e2m1(np.arange(8, 16)), [-v for v in vals])
    # byte j holds element 2j in its low nibble; one scale per 16 elements
    packed = np.array([[0x21, 0xF7] + [0] * 6 + [0x01] + [0] * 7], dtype=np.uint8)   # 32 elements
    sf = np.array([[0x38, 0x40]], dtype=np.uint8)        # e4m3: 1.0, 2.0
    got = O.decode_fp4_blocks(packed, sf)
    assert got.shape == (1, 32)
    assert got[0, :4].tolist() == [0.5, 1.0, 6.0, -6.0]
    assert got[0, 16] == 1.0 and got[0, 17] == 0.0


# ----------------------------------------------------------------------------
# RMSNorm of the compressed entries ([uika] §2.3.3)
# ----------------------------------------------------------------------------


def test_rms_norm_unit_rms_same_direction():
    x = rnd(7, 33) * np.exp(rnd(7, 1))           # rows of very different scales
    y = O.rms_norm(x)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(y / np.linalg.norm(y, axis=-1, keepdims=True),
                               x / np.linalg.norm(x, axis=-1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(O.rms_norm(3.7 * x), y, rtol=1e-13)     # scale invariant


def test_rms_norm_weight_and_eps_closed_forms():
    x = rnd(4, 16)
    w = rnd(16)
    np.testing.assert_allclose(O.rms_norm(x, w), O.rms_norm(x) * w, rtol=1e-14)
    # a constant vector a: mean(x^2) = a^2, so y = a / sqrt(a^2 + eps)
    a, eps = 0.3, 0.05
    np.testing.assert_allclose(O.rms_norm(np.full((1, 8), a), eps=eps), a / math.sqrt(a * a + eps),
                               rtol=1e-14)


# ----------------------------------------------------------------------------
# grouped output projection ([uika] §2.3.1; §4.2.1: g groups of d_g outputs)
# ----------------------------------------------------------------------------


def test_grouped_projection_is_a_block_diagonal_projection():
    # the grouped projection is one projection whose weight is block diagonal
    # (group j's inputs feed only group j's outputs): library block_diag + matmul
    from scipy.linalg import block_diag
    G, N, K, M = 4, 3, 5, 7
    A, W = rnd(M, G * K), rnd(G, N, K)
    full = block_diag(*[W[j].T for j in range(G)])          # [G*K, G*N]
    np.testing.assert_allclose(O.grouped_projection(A, W), A @ full, rtol=1e-13, atol=1e-13)
    # extra columns of A beyond G*K are not read
    A2 = np.concatenate([A, rnd(M, 3)], axis=1)
    np.testing.assert_array_equal(O.grouped_projection(A2, W), O.grouped_projection(A, W))


def test_grouped_projection_one_hot_picks_a_weight_column():
    # A = e_i (one row, one-hot at column j*K + c) selects W[j][:, c] into group j's outputs
    G, N, K = 3, 4, 6
    W = rnd(G, N, K)
    for j, c in ((0, 0), (1, 5), (2, 3)):
        a = np.zeros((1, G * K))
        a[0, j * K + c] = 1.0
        want = np.zeros(G * N)
        want[j * N:(j + 1) * N] = W[j][:, c]
        np.testing.assert_array_equal(O.grouped_projection(a, W)[0], want)
