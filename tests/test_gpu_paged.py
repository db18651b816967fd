"""The paged KV-cache layout (DeepSeek-V4 report, Chinese translation,
blog.uika.cn, §3.6.1): blocks of lcm(m, m') raw tokens, each holding lcm/m
CSA entries and indexer keys and lcm/m' HCA entries in pools shared by every
sequence, one block table per sequence, and the sliding window as a
fixed-size ring per sequence (the state cache).

Paging changes only where rows are read from and written to, not the
arithmetic, so every paged result must be bit-identical to the flat layout on
the same logical rows: the whole decode step (index, top-k, attention) of the
bf16 and FP8/FP4 CSA workloads and of HCA, at mixed lengths, with the blocks
handed out in a scrambled order; the index call at several block sizes
(smaller than, equal to and larger than a 128-entry tile); causal prefill,
whose attention pre-rotates paged rows; compression straight into the pools
(prefill, and the entry a closing block adds in decode).  The decode step
through the cache is also compared with the float64 oracle, and a block-table
entry outside the pool is flagged in the device error word, not followed.
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


def _scrambled_cache(P, cfg, lengths, storage, extra_blocks=7, seed=0):
    """A cache whose blocks are handed out round-robin over the sequences after
    a scrambled set of releases, so no sequence's blocks are contiguous."""
    B = len(lengths)
    L_max = max(lengths)
    per_seq = -(-L_max // 128)
    cache = P.PagedKVCache(B, L_max, B * per_seq + extra_blocks, d=cfg["d"], r=cfg["r"],
                           c_I=cfg.get("c_I", 128), T_win=cfg["T_win"], m=4, m_hca=128,
                           storage=storage, device=DEV)
    rng = np.random.default_rng(seed)
    junk = cache.pool.alloc(extra_blocks)              # occupy some ids, release a few later
    grown = [0] * B
    while any(grown[b] < -(-lengths[b] // 128) for b in range(B)):
        for b in rng.permutation(B):
            if grown[b] < -(-lengths[b] // 128):
                grown[b] += 1
                cache.reserve(int(b), grown[b] * 128)
        if junk and rng.random() < 0.5:
            cache.pool.release([junk.pop()])
    return cache


def _fill(cache, cfg, x, lengths, kind):
    """Copies the workload's flat cache tensors into the cache, sequence by sequence."""
    N = cfg["N"]
    for b, Lb in enumerate(lengths):
        Nb = Lb // cfg["m"]
        if cfg["dtype"] == "mixed":
            cache.load("entries", b, (x["ent_nope"][b, :Nb], x["ent_scale"][b, :Nb],
                                      x["ent_rope"][b, :Nb]))
            cache.load("keys", b, x["K_fp4"][b, :Nb], sf=x["K_sf"][b, :Nb])
            cache.load_window(b, (x["win_nope"][b], x["win_scale"][b], x["win_rope"][b]),
                              int(x["win_base"][b]))
        else:
            cache.load("hca" if kind == "hca" else "entries", b, x["entries"][b, :Nb])
            if kind == "csa":
                cache.load("keys", b, x["K"][b, :Nb])
            cache.load_window(b, x["win"][b], int(x["win_base"][b]))
    return N


@pytest.mark.parametrize("name,lengths", [
    ("csa_decode_128k", [131072, 70001, 2050, 77]),
    ("csa_decode_1m_mixed", [65536, 40003, 3000, 130]),
    ("hca_decode_1m", [262144, 100001, 129, 50]),
])
def test_paged_decode_step_is_bit_identical_to_flat(name, lengths):
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import path as P
    cfg = synth.scaled(name, B=len(lengths), lengths=lengths)
    kind = "csa" if cfg["kind"].startswith("csa") else "hca"
    x = synth.make_inputs(cfg, seed=5, device=DEV)
    flat = P.Buffers()
    out_flat = P.forward(cfg, x, flat).clone()
    torch.cuda.synchronize()
    K.device_error()
    cache = _scrambled_cache(P, cfg, lengths, "mixed" if cfg["dtype"] == "mixed" else "bf16")
    N = _fill(cache, cfg, x, lengths, kind)
    x2 = dict(x)
    x2.update(cache.views(kind, N))
    paged = P.Buffers()
    out = P.forward(cfg, x2, paged)
    torch.cuda.synchronize()
    K.device_error()
    assert torch.equal(out, out_flat)
    if kind == "csa":
        assert torch.equal(paged.idx, flat.idx)
        for b, Lb in enumerate(lengths):
            vis = min(N, O.visible_count(Lb - 1, cfg["m"]))
            assert torch.equal(paged.scores[b, 0, :vis], flat.scores[b, 0, :vis])


def test_paged_decode_step_matches_the_oracle():
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import path as P
    lengths = [131072, 9001, 600, 40]
    cfg = synth.scaled("csa_decode_128k", B=len(lengths), lengths=lengths)
    x = synth.make_inputs(cfg, seed=8, device=DEV)
    cache = _scrambled_cache(P, cfg, lengths, "bf16", seed=3)
    N = _fill(cache, cfg, x, lengths, "csa")
    x2 = dict(x)
    x2.update(cache.views("csa", N))
    buf = P.Buffers()
    out = P.forward(cfg, x2, buf)
    torch.cuda.synchronize()
    K.device_error()
    xn = _host(x)
    for b, Lb in enumerate(lengths):
        res = OP.run_rows(cfg, xn, b, [0], selected=[buf.idx[b, 0].cpu().numpy()])
        got_s = f64(buf.scores[b, 0])
        assert_scores_close(got_s, res["scores"][0], f"L={Lb} scores")
        vis = min(N, O.visible_count(Lb - 1, cfg["m"]))
        n = min(cfg["k"], vis)
        got_i = buf.idx[b, 0].cpu().numpy()
        assert np.array_equal(got_i[:n], np.sort(O.topk_select(got_s, cfg["k"], vis)))
        assert_close(f64(out[b, 0]), res["out"][0], TOL_BF16, TOL_BF16, f"L={Lb} attend")


def _pool_from_flat(flat, block_rows, num_blocks, perm):
    """[B, N, ...] rows -> (pool [num_blocks*block_rows, ...], table [B, max_blocks])."""
    B, N = flat.shape[:2]
    nb = -(-N // block_rows)
    pool = torch.zeros((num_blocks * block_rows,) + tuple(flat.shape[2:]), dtype=flat.dtype,
                       device=flat.device)
    table = torch.tensor(perm[:B * nb], dtype=torch.int32).view(B, nb).to(flat.device)
    for b in range(B):
        for j in range(nb):
            lo, hi = j * block_rows, min(N, (j + 1) * block_rows)
            p0 = int(table[b, j]) * block_rows
            pool[p0:p0 + hi - lo] = flat[b, lo:hi]
    return pool, table


@pytest.mark.parametrize("fmt", ["bf16", "fp4", "f32"])
@pytest.mark.parametrize("block_rows", [8, 32, 128, 512])
def test_paged_index_topk_at_block_sizes(fmt, block_rows):
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300._lib import Paged
    from synth.generate import quantise_fp4_blocks
    B, N, H, c, m, k = 3, 9000, 64, 128, 4, 512
    g = torch.Generator(device=DEV).manual_seed(21)
    qI = torch.randn((B, 1, H, c), generator=g, device=DEV) / c ** 0.5
    Kt = torch.randn((B, N, c), generator=g, device=DEV) / c ** 0.5
    w = torch.rand((B, 1, H), generator=g, device=DEV) / H
    q_pos = torch.tensor([[4 * N - 1], [4 * 5000 + 2], [4 * 70]], dtype=torch.int32, device=DEV)
    q_sf = k_sf = None
    if fmt == "bf16":
        qI, Kt = qI.to(torch.bfloat16), Kt.to(torch.bfloat16)
    elif fmt == "fp4":
        qI, q_sf = quantise_fp4_blocks(qI)
        Kt, k_sf = quantise_fp4_blocks(Kt)
    num_blocks = B * -(-N // block_rows) + 5
    perm = np.random.default_rng(block_rows).permutation(num_blocks).tolist()
    s0, i0, _ = K.csa_index_topk(qI, w, Kt, k, m, q_pos, qI_sf=q_sf, K_sf=k_sf)
    pool, table = _pool_from_flat(Kt, block_rows, num_blocks, perm)
    sf_pool = None if k_sf is None else _pool_from_flat(k_sf, block_rows, num_blocks, perm)[0]
    s1, i1, _ = K.csa_index_topk(qI, w, Paged(pool, table, block_rows, N), k, m, q_pos,
                                 qI_sf=q_sf, K_sf=sf_pool)
    s2 = K.csa_index(qI, w, Paged(pool, table, block_rows, N), m, q_pos, qI_sf=q_sf, K_sf=sf_pool)
    torch.cuda.synchronize()
    K.device_error()
    assert torch.equal(i1, i0)
    for b in range(B):
        vis = O.visible_count(int(q_pos[b, 0]), m)
        assert torch.equal(s1[b, 0, :vis], s0[b, 0, :vis])
        assert torch.equal(s2[b, 0, :vis], s0[b, 0, :vis])
        assert bool(torch.isneginf(s1[b, 0, vis:]).all())


def test_paged_prefill_compress_and_attention():
    # causal prefill with the entries compressed straight into a paged pool:
    # the pool rows equal the flat compression bit for bit, and the attention
    # (absolute-RoPE mode: it rotates every stored row once, here read through
    # the block table) equals the flat attention bit for bit
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import path as P
    cfg = synth.scaled("csa_prefill_32k", T=3000)
    x = synth.make_inputs(cfg, seed=9, device=DEV)
    flat = P.Buffers()
    out_flat = P.forward(cfg, x, flat).clone()
    torch.cuda.synchronize()
    K.device_error()
    N = cfg["N"]
    cache = _scrambled_cache(P, dict(cfg, T_win=128), [cfg["T"]], "bf16", seed=4)
    cache.compress("entries", x["Ca"], x["Za"], Cb=x["Cb"], Zb=x["Zb"])
    cache.compress("keys", x["Ca"][..., :128].contiguous(), x["Za"][..., :128].contiguous(),
                   Cb=x["Cb"][..., :128].contiguous(), Zb=x["Zb"][..., :128].contiguous())
    torch.cuda.synchronize()
    K.device_error()
    rows = cache._rows_of(0, N, cache.csa_rows)
    assert torch.equal(cache.ent[rows], flat.entries[0])
    keys_flat = K.csa_compress(x["Ca"][..., :128].contiguous(), x["Za"][..., :128].contiguous(), 4,
                               Cb=x["Cb"][..., :128].contiguous(), Zb=x["Zb"][..., :128].contiguous())
    assert torch.equal(cache.keys[rows], keys_flat[0])
    # attention over the paged entries (indexer and window as in the flat run)
    out = K.csa_attend(x["q"], cache.entries(N), flat.idx, x["win"], x["sink"], cfg["m"],
                       cfg["n_win"], x["win_base"], x["q_pos"], cfg["r"], cfg["rope_base"])
    torch.cuda.synchronize()
    K.device_error()
    assert torch.equal(out, out_flat)


def test_decode_block_close_writes_its_entry_into_the_cache():
    # in decode, each sequence whose block just closed passes its last 2m raw rows;
    # local entry 1 (a-rows of the closing block, b-rows of the one before) lands
    # at its logical row, rotated at its own position; sequences whose block did
    # not close (entry0 = -1) write nothing; a first block takes -inf b-row logits
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import path as P
    m, d, T = 4, 512, 4096
    cfg = synth.scaled("csa_prefill_32k", T=T)
    x = synth.make_inputs(cfg, seed=12, device=DEV)
    B = 4
    Ca = x["Ca"].expand(B, T, d).contiguous()
    Cb = x["Cb"].expand(B, T, d).contiguous()
    Za = (x["Za"] + torch.arange(B, device=DEV).view(B, 1, 1) * 0.25).to(torch.bfloat16)
    Zb = x["Zb"].expand(B, T, d).contiguous()
    opts = dict(rms_norm=True, norm_eps=1e-6, rope_dims=64, rope_base=10000.0)
    full = K.csa_compress(Ca, Za, m, Cb=Cb, Zb=Zb, **opts)       # every entry, flat
    cache = P.PagedKVCache(B, T, B * T // 128 + 3, storage="bf16", device=DEV)
    for b in range(B):
        cache.reserve(b, T)
    closing = [517, 0, -1, 1000]                      # entry index closing now, or -1
    win_a, win_b, z_a, z_b = (torch.empty((B, 2 * m, d), dtype=torch.bfloat16, device=DEV)
                              for _ in range(4))
    for b, s in enumerate(closing):
        s_ = max(s, 0)
        lo = m * (s_ - 1)
        if s_ == 0:                                   # no previous block: b-row logits -inf
            win_a[b, :m] = 0
            win_b[b, :m] = 0
            z_a[b, :m] = 0
            z_b[b, :m] = float("-inf")
            win_a[b, m:], z_a[b, m:] = Ca[b, :m], Za[b, :m]
            win_b[b, m:], z_b[b, m:] = Cb[b, :m], Zb[b, :m]
        else:
            win_a[b], z_a[b] = Ca[b, lo:lo + 2 * m], Za[b, lo:lo + 2 * m]
            win_b[b], z_b[b] = Cb[b, lo:lo + 2 * m], Zb[b, lo:lo + 2 * m]
    cache.ent.fill_(7.0)
    e0 = torch.tensor(closing, dtype=torch.int32, device=DEV)
    cache.compress("entries", win_a, z_a, Cb=win_b, Zb=z_b, entry0=e0, first=1, **opts)
    torch.cuda.synchronize()
    K.device_error()
    written = 0
    for b, s in enumerate(closing):
        rows = cache._rows_of(b, T // m, cache.csa_rows)
        got = cache.ent[rows]
        if s < 0:
            assert bool((got == 7.0).all())
            continue
        written += 1
        if s > 0:
            assert torch.equal(got[s], full[b, s])
        else:
            ref = O.compress_csa(f64(Ca[b, :m]), f64(Cb[b, :m]), f64(Za[b, :m]), f64(Zb[b, :m]), m)
            ref = O.rope_rotate(O.rms_norm(ref, eps=1e-6), np.array([m - 1]), 64, 10000.0)
            assert_close(f64(got[0]), ref[0], TOL_BF16, TOL_BF16, "first block")
        untouched = torch.ones(T // m, dtype=torch.bool, device=DEV)
        untouched[s] = False
        assert bool((got[untouched] == 7.0).all())
    assert written == 3


def test_block_outside_the_pool_is_flagged_not_followed():
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import CsaError
    from compressed_sparse_long_05_b300 import path as P
    lengths = [20000, 3000]
    cfg = synth.scaled("csa_decode_128k", B=2, lengths=lengths)
    x = synth.make_inputs(cfg, seed=2, device=DEV)
    cache = _scrambled_cache(P, cfg, lengths, "bf16", seed=1)
    N = _fill(cache, cfg, x, lengths, "csa")
    x2 = dict(x)
    x2.update(cache.views("csa", N))
    good = P.forward(cfg, x2, P.Buffers()).clone()
    torch.cuda.synchronize()
    K.device_error()
    saved = cache.table[0, 3].item()
    cache.table[0, 3] = cache.num_blocks               # one past the pool
    P.forward(cfg, x2, P.Buffers())
    torch.cuda.synchronize()
    with pytest.raises(CsaError) as e:
        K.device_error()
    assert e.value.status == 6
    cache.table[0, 3] = saved
    again = P.forward(cfg, x2, P.Buffers())
    torch.cuda.synchronize()
    K.device_error()
    assert torch.equal(again, good)
