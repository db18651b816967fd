"""csa_attend_noalloc: the attention call for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc: a host application or
serving engine that owns every device allocation and hands the attention layer
only its input and output buffers, or a latency-critical loop that cannot take
cudaMalloc's implicit device synchronisation.  csa_attend_noalloc serves them by
keeping its scratch in one fixed device array inside the library.  These tests
call it through the C ABI and compare it with csa_attend (which takes a
caller-allocated workspace) on the same inputs, twice in a row, because every
call reuses the array the previous call left behind.  Both calls run the same
plan and the same kernels, so their outputs must agree bit for bit; one case is
also checked against the float64 oracle directly.

The file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O
from tests.parity import TOL_BF16, assert_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"
SCRATCH_BYTES = 16 << 20       # CSA_NOALLOC_SCRATCH_BYTES in include/csa.h


def _rms(shape, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(shape, generator=g, device=DEV)
    return (x * torch.rsqrt(x.square().mean(-1, keepdim=True))).to(torch.bfloat16)


def _decode_case(K, lengths, N, k, seed):
    """One decode row per sequence at V4-Pro head shapes; sequence b holds
    lengths[b] tokens (its new token at lengths[b] - 1) over a cache of N entries."""
    m, n_win, d, n_h = 4, 128, 512, 128
    B = len(lengths)
    q = _rms((B, 1, n_h, d), seed)
    ent = _rms((B, N, d), seed + 1)
    win = _rms((B, n_win, d), seed + 2)
    sink = torch.randn((n_h,), generator=torch.Generator(device=DEV).manual_seed(seed + 3),
                       device=DEV)
    q_pos = torch.tensor([[L - 1] for L in lengths], dtype=torch.int32, device=DEV)
    win_base = torch.tensor([max(0, L - n_win) for L in lengths], dtype=torch.int32, device=DEV)
    scores = torch.rand((B, 1, N), generator=torch.Generator(device=DEV).manual_seed(seed + 4),
                        device=DEV)
    idx = K.csa_topk(scores, k, m, q_pos)
    return dict(q=q, ent=ent, win=win, sink=sink, idx=idx, m=m, n_win=n_win, win_base=win_base,
                q_pos=q_pos, r=64, k=k)


def _ref(K, c):
    return K.csa_attend(c["q"], c["ent"], c["idx"], c["win"], c["sink"], c["m"], c["n_win"],
                        c["win_base"], c["q_pos"], c["r"])


def _noalloc(K, c, out=None):
    return K.csa_attend_noalloc(c["q"], c["ent"], c["idx"], c["win"], c["sink"], c["m"],
                                c["n_win"], c["win_base"], c["q_pos"], c["r"], out=out)


def _need(K, c):
    return K.attend_workspace_size(c["q"], c["ent"], c["win"], c["k"], c["m"], c["n_win"],
                                   c["r"], False)


def test_noalloc_matches_workspace_call_twice():
    # k = 4096 splits each row set over more CTAs than one cluster holds, so the
    # chunks merge through fp32 partials in the scratch array
    import compressed_sparse_long_05_b300 as K
    c = _decode_case(K, lengths=[80000], N=20000, k=4096, seed=500)
    assert 0 < _need(K, c) <= SCRATCH_BYTES      # the case really uses scratch, and it fits
    ref = _ref(K, c)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(c["q"], float("nan"))
        _noalloc(K, c, out=out)
        torch.cuda.synchronize()
        K.device_error()
        assert torch.equal(out, ref), f"noalloc call {call} differs from csa_attend"
    # and the result itself against the float64 oracle on the selected entries
    t = 80000 - 1
    o = O.csa_attend_token(f64(c["q"][0, 0]), t, f64(c["ent"][0]), c["idx"][0, 0].cpu().numpy(),
                           f64(c["win"][0]), t - c["n_win"] + 1, f64(c["sink"]), c["m"],
                           c["n_win"], c["r"], 1e4)
    assert_close(f64(out[0, 0]), o, TOL_BF16, TOL_BF16, "noalloc vs oracle")


def test_noalloc_second_call_other_sizes():
    # a smaller call after a larger one: stale scratch from the first must not
    # leak in; the second has sequences at different context lengths
    import compressed_sparse_long_05_b300 as K
    big = _decode_case(K, lengths=[80000], N=20000, k=4096, seed=510)
    small = _decode_case(K, lengths=[36000, 30001], N=9000, k=2048, seed=520)
    for c in (big, small):
        assert 0 < _need(K, c) <= SCRATCH_BYTES
        ref = _ref(K, c)
        out = _noalloc(K, c)
        torch.cuda.synchronize()
        K.device_error()
        assert torch.equal(out, ref), f"noalloc k={c['k']} differs from csa_attend"


def _raw_call(K, c, k, d=512, out=None):
    from compressed_sparse_long_05_b300 import _lib
    B, Tq, n_h, _ = c["q"].shape
    return _lib.lib().csa_attend_noalloc(
        _lib._p(c["q"]), _lib._kv(c["ent"]), _lib._p(c["idx"]), _lib._kv(c["win"]),
        _lib._p(c["q_pos"]), _lib._p(c["win_base"]), _lib._p(c["sink"]), _lib._p(out), B, Tq,
        c["ent"].shape[1], k, c["win"].shape[1], n_h, d, c["r"], c["m"], c["n_win"],
        ctypes.c_float(1e4), _lib._stream())


def test_noalloc_rejects_sizes_beyond_the_array():
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import _lib
    # 16 sequences at k = 4096: 160 work items, more than one per SM, so every
    # chunk keeps a 128 KB float32 partial (20 MB)
    c = _decode_case(K, lengths=[160000] * 16, N=40000, k=4096, seed=530)
    assert _need(K, c) > SCRATCH_BYTES
    out = torch.zeros_like(c["q"])
    assert _raw_call(K, c, 4096, out=out) == 3          # CSA_ERR_WORKSPACE, before any launch
    assert b"above the fixed" in _lib.lib().csa_last_cuda_error()
    # an invalid argument is reported as such, not as a scratch overflow
    assert _raw_call(K, c, 5000, out=out) == 1          # k above 4096: CSA_ERR_INVALID_ARG
    assert _raw_call(K, c, 4096, d=500, out=out) == 2   # no kernel for d = 500: unsupported
    torch.cuda.synchronize()
    assert int(out.abs().sum().item()) == 0
