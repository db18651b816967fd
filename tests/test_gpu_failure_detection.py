"""Failure detection: a bounded wait that runs out is reported, and the GPU
context stays usable.

Every mbarrier wait in the tensor-core kernels gives up after a time limit,
sets the timeout bit of the library's sticky device error word and raises its
CTA's abort flag so that the CTA's other warp roles leave their loops; copies
already in flight are waited for and tensor memory is freed before the kernel
returns.  ``csa_selftest_wait_timeout`` plants the fault on the host side: the
TMA producer of CTA 0 leaves out one K-tile copy (nothing ever fills that
stage) and the launch's wait limit is 1 ms.  No GPU fault, trap or hang is
involved: the kernel returns by itself.
"""

import time

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O
from tests.parity import assert_scores_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _inputs(B=2, N=5000, H=64, c=128, seed=61):
    g = torch.Generator(device=DEV).manual_seed(seed)
    qI = (torch.randn((B, 1, H, c), generator=g, device=DEV) / c ** 0.5).to(torch.bfloat16)
    Kt = (torch.randn((B, N, c), generator=g, device=DEV) / c ** 0.5).to(torch.bfloat16)
    w = torch.rand((B, 1, H), generator=g, device=DEV) / H
    q_pos = torch.full((B, 1), 4 * N - 1, dtype=torch.int32, device=DEV)
    return qI, Kt, w, q_pos


def test_wait_that_runs_out_is_reported_and_the_next_call_is_correct():
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import CsaError, _lib
    qI, Kt, w, q_pos = _inputs()
    B, _, H, c = qI.shape
    N, m = Kt.shape[1], 4
    scores = torch.empty((B, 1, N), dtype=torch.float32, device=DEV)
    K.device_error()                                  # start from a clear error word
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = _lib.lib().csa_selftest_wait_timeout(_lib._p(qI), _lib._p(w), _lib._p(Kt), _lib._p(q_pos),
                                              _lib._p(scores), B, 1, N, m, 1000, _lib._stream())
    assert st == 0                                    # the launch itself is fine
    torch.cuda.synchronize()                          # the kernel returns by itself
    elapsed = time.perf_counter() - t0
    with pytest.raises(CsaError) as e:
        K.device_error()
    assert e.value.status == 5                        # CSA_ERR_TIMEOUT
    assert elapsed < 1.0, f"the 1 ms limit took {elapsed:.3f} s to end the kernel"
    K.device_error()                                  # the read cleared the word
    # the same context runs the normal kernel correctly afterwards
    s = K.csa_index(qI, w, Kt, m, q_pos)
    torch.cuda.synchronize()
    K.device_error()
    for b in range(B):
        ref = O.index_scores(f64(qI[b]), f64(w[b]), f64(Kt[b]), np.array([4 * N - 1]), m)
        assert_scores_close(f64(s[b, 0]), ref[0], f"b={b} after the timeout")


def test_selftest_rejects_bad_limits():
    from compressed_sparse_long_05_b300 import _lib
    qI, Kt, w, q_pos = _inputs(B=1, N=300)
    scores = torch.empty((1, 1, 300), dtype=torch.float32, device=DEV)
    for lim in (0, 2000001):
        assert _lib.lib().csa_selftest_wait_timeout(
            _lib._p(qI), _lib._p(w), _lib._p(Kt), _lib._p(q_pos), _lib._p(scores), 1, 1, 300, 4,
            lim, _lib._stream()) == 1


@pytest.mark.parametrize("fmt", ["bf16", "fp4"])
def test_stale_histogram_workspace_is_flagged_not_used(fmt):
    # csa_index_topk's workspace must start zero.  A stale one (here: every bin
    # holds 1 extra count) no longer describes the scores: the selector checks
    # that the histogram's total equals the row's visible count, flags the
    # mismatch in the device error word and leaves the row empty instead of
    # selecting from a wrong threshold.  Its writes stay inside the row either
    # way (every output position is bounds-checked).
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import CsaError
    from synth.generate import quantise_fp4_blocks
    B, N, H, c, m, k = 2, 40001, 64, 128, 4, 512
    qI, Kt, w, q_pos = _inputs(B=B, N=N)
    q_sf = k_sf = None
    if fmt == "fp4":
        qI, q_sf = quantise_fp4_blocks(qI.float())
        Kt, k_sf = quantise_fp4_blocks(Kt.float())
    s_ref, i_ref, ws = K.csa_index_topk(qI, w, Kt, k, m, q_pos, qI_sf=q_sf, K_sf=k_sf)
    torch.cuda.synchronize()
    K.device_error()
    ws.view(torch.int32).fill_(1)                     # stale counts in every bin
    s, i, ws = K.csa_index_topk(qI, w, Kt, k, m, q_pos, qI_sf=q_sf, K_sf=k_sf, ws=ws)
    torch.cuda.synchronize()
    with pytest.raises(CsaError) as e:
        K.device_error()
    assert e.value.status == 6                        # CSA_ERR_DEVICE (histogram bit)
    assert torch.equal(s, s_ref)                      # the scores themselves are right
    assert bool((i == -1).all())                      # no selection from a wrong threshold
    assert int(ws.count_nonzero()) == 0               # the selector cleared the histograms
    s, i, ws = K.csa_index_topk(qI, w, Kt, k, m, q_pos, qI_sf=q_sf, K_sf=k_sf, ws=ws)
    torch.cuda.synchronize()
    K.device_error()
    assert torch.equal(i, i_ref)
