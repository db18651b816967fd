"""The grouped output projection on the tensor cores against the float64 oracle.

DeepSeek-V4 report (Chinese translation, blog.uika.cn) §2.3.1 "分组输出投影":
the n_h head outputs are split into g groups, each projected to d_g dims, and
the g * d_g intermediate outputs are projected to the model width d (§4.2.1:
V4-Pro g = 16, d_g = 1024, d = 7168; V4-Flash g = 8, d = 4096).  Inputs are
bf16; the oracle multiplies the same bf16 values in float64.  The GPU
accumulates in float32 and rounds each output once to bf16, so outputs of
unit scale agree within 2e-2.
"""

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O
from tests.parity import TOL_BF16, assert_close, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _randn(shape, seed, scale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, generator=g, device=DEV) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("M,G,N,K", [
    (300, 16, 1024, 4096),     # V4-Pro grouped step, ragged token count
    (77, 3, 200, 72),          # partial N tile, partial K step
    (129, 1, 7168, 16384),     # V4-Pro final step to the model width
    (5, 8, 1024, 4096),        # decode batch: a few tokens, V4-Flash groups
])
def test_grouped_proj_matches_oracle(M, G, N, K):
    import compressed_sparse_long_05_b300 as Kb
    A = _randn((M, G * K), 200)
    W = _randn((G, N, K), 201, scale=K ** -0.5)
    C = Kb.csa_grouped_proj(A, W)
    torch.cuda.synchronize()
    Kb.device_error()
    ref = O.grouped_projection(f64(A), f64(W))
    assert_close(f64(C), ref, TOL_BF16, TOL_BF16, f"grouped proj M={M} G={G} N={N} K={K}")


def test_output_projection_of_an_attention_output():
    # the full two-step projection of a [B, Tq, n_h, d] attention output, with
    # A read at a row stride larger than G*K (a wider buffer)
    import compressed_sparse_long_05_b300 as Kb
    from compressed_sparse_long_05_b300 import path as P
    B, Tq, n_h, d, g, d_g, d_model = 2, 3, 128, 512, 16, 1024, 7168
    out = _randn((B, Tq, n_h, d), 210)
    Wg = _randn((g, d_g, (n_h // g) * d), 211, scale=((n_h // g) * d) ** -0.5)
    Wo = _randn((1, d_model, g * d_g), 212, scale=(g * d_g) ** -0.5)
    z = P.output_projection(out, Wg, Wo)
    torch.cuda.synchronize()
    Kb.device_error()
    y_ref = O.grouped_projection(f64(out).reshape(B * Tq, n_h * d), f64(Wg))
    # the GPU's intermediate y is bf16: project the oracle's y rounded the same way
    y_bf16 = torch.tensor(y_ref, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    z_ref = O.grouped_projection(y_bf16, f64(Wo))
    assert_close(f64(z), z_ref, TOL_BF16, TOL_BF16, "output projection")
    wide = torch.zeros((B * Tq, n_h * d + 64), dtype=torch.bfloat16, device=DEV)
    wide[:, :n_h * d] = out.reshape(B * Tq, n_h * d)
    y2 = Kb.csa_grouped_proj(wide, Wg)
    torch.cuda.synchronize()
    assert_close(f64(y2), y_ref, TOL_BF16, TOL_BF16, "grouped proj, wide A")
