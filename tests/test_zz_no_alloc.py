"""csa_attend_noalloc: the attention call for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc: a host application or
serving engine that owns every device allocation and hands the attention layer
only its input and output buffers, or a latency-critical loop that cannot take
cudaMalloc's implicit device synchronisation.  csa_attend_noalloc serves them by
keeping its scratch in one fixed device array inside the library.  These tests
call it through the C ABI and compare it with csa_attend (which takes a
caller-allocated workspace) on the same inputs, twice in a row, because every
call reuses the array the previous call left behind.

The file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes

import pytest
import torch

from tests.parity import TOL_BF16, assert_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCRATCH_BYTES = 16 << 20       # CSA_NOALLOC_SCRATCH_BYTES in include/csa.h


def _rms(shape, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(shape, generator=g, device=DEV)
    return (x * torch.rsqrt(x.square().mean(-1, keepdim=True))).to(torch.bfloat16)


def _decode_case(K, B, N, k, seed):
    """One decode row per sequence at V4-Pro head shapes over a cache of N entries."""
    m, n_win, d, n_h = 4, 128, 512, 128
    L = m * N
    q = _rms((B, 1, n_h, d), seed)
    ent = _rms((B, N, d), seed + 1)
    win = _rms((B, n_win, d), seed + 2)
    sink = torch.randn((n_h,), generator=torch.Generator(device=DEV).manual_seed(seed + 3),
                       device=DEV)
    scores = torch.rand((B, 1, N), generator=torch.Generator(device=DEV).manual_seed(seed + 4),
                        device=DEV)
    idx = K.csa_topk(scores, k, m, L - 1)
    return dict(q=q, ent=ent, win=win, sink=sink, idx=idx, m=m, n_win=n_win, win_base=L - n_win,
                q_pos0=L - 1, r=64)


def test_noalloc_matches_workspace_call_twice():
    # k = 4096 splits each row set over more CTAs than one cluster holds, so the
    # chunks merge through fp32 partials in the scratch array
    import compressed_sparse_long_05_b300 as K
    c = _decode_case(K, B=1, N=20000, k=4096, seed=500)
    need = K.attend_workspace_size(c["q"], c["ent"], c["win"], 4096, c["m"], c["n_win"],
                                   c["q_pos0"], c["r"], False)
    assert 0 < need <= SCRATCH_BYTES      # the case really uses scratch, and it fits
    ref = K.csa_attend(c["q"], c["ent"], c["idx"], c["win"], c["sink"], c["m"], c["n_win"],
                       c["win_base"], c["q_pos0"], c["r"])
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(c["q"], float("nan"))
        K.csa_attend_noalloc(c["q"], c["ent"], c["idx"], c["win"], c["sink"], c["m"], c["n_win"],
                             c["win_base"], c["q_pos0"], c["r"], out=out)
        torch.cuda.synchronize()
        K.device_error()
        assert_close(f64(out), f64(ref), TOL_BF16, TOL_BF16, f"noalloc call {call}")


def test_noalloc_second_call_other_sizes():
    # a smaller call after a larger one: stale scratch from the first must not leak in
    import compressed_sparse_long_05_b300 as K
    big = _decode_case(K, B=1, N=20000, k=4096, seed=510)
    small = _decode_case(K, B=2, N=9000, k=2048, seed=520)
    for c, k in ((big, 4096), (small, 2048)):
        need = K.attend_workspace_size(c["q"], c["ent"], c["win"], k, c["m"], c["n_win"],
                                       c["q_pos0"], c["r"], False)
        assert 0 < need <= SCRATCH_BYTES
        ref = K.csa_attend(c["q"], c["ent"], c["idx"], c["win"], c["sink"], c["m"], c["n_win"],
                           c["win_base"], c["q_pos0"], c["r"])
        out = K.csa_attend_noalloc(c["q"], c["ent"], c["idx"], c["win"], c["sink"], c["m"],
                                   c["n_win"], c["win_base"], c["q_pos0"], c["r"])
        torch.cuda.synchronize()
        K.device_error()
        assert_close(f64(out), f64(ref), TOL_BF16, TOL_BF16, f"noalloc k={k}")


def test_noalloc_rejects_sizes_beyond_the_array():
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import _lib
    c = _decode_case(K, B=4, N=40000, k=4096, seed=530)
    need = K.attend_workspace_size(c["q"], c["ent"], c["win"], 4096, c["m"], c["n_win"],
                                   c["q_pos0"], c["r"], False)
    assert need > SCRATCH_BYTES
    out = torch.zeros_like(c["q"])
    B, Tq, n_h, d = c["q"].shape
    st = _lib.lib().csa_attend_noalloc(
        _lib._p(c["q"]), _lib._kv(c["ent"]), _lib._p(c["idx"]), _lib._kv(c["win"]),
        _lib._p(c["sink"]), _lib._p(out), B, Tq, c["ent"].shape[1], 4096, c["win"].shape[1],
        c["win_base"], n_h, d, c["r"], c["m"], c["n_win"], c["q_pos0"], ctypes.c_float(1e4),
        _lib._stream())
    assert st == 3                      # CSA_ERR_WORKSPACE, before any launch
    assert b"above the fixed" in _lib.lib().csa_last_cuda_error()
    torch.cuda.synchronize()
    assert int(out.abs().sum().item()) == 0
