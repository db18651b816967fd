"""path.GraphForward: host copies, every stage and the output read-back as one graph.

The replayed graph must give what eager ``path.forward`` gives on the same
inputs, and must pick up new host inputs written in place between calls.
"""

import pytest
import torch

import synth
from tests.parity import assert_close, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,over", [
    ("csa_decode_128k", dict(B=2, L=16384)),
    ("hca_decode_1m", dict(B=1, L=65536)),
    ("csa_decode_1m_mixed", dict(B=2, L=32768)),
])
def test_graph_forward_matches_eager(name, over):
    from compressed_sparse_long_05_b300 import path as P
    cfg = synth.scaled(name, **over)
    x = synth.make_inputs(cfg, seed=3, device="cuda")
    names = ["q"] + [n for n in ("qI", "qI_fp4", "qI_sf", "w") if n in x]
    fw = P.GraphForward(cfg, x, names)
    for step in range(2):
        if step == 1:                       # new inputs for the second step, written in place
            g = torch.Generator().manual_seed(11)
            fw.host["q"].copy_(torch.randn(fw.host["q"].shape, generator=g).to(fw.host["q"].dtype))
        got = fw().clone()
        xe = dict(x)
        for n in names:
            xe[n] = fw.host[n].to("cuda")
        want = P.forward(cfg, xe).cpu()
        torch.cuda.synchronize()
        # the same kernels on the same bytes: bit-identical
        assert torch.equal(got, want), f"{name} step {step}"
        assert_close(f64(got), f64(want), 0, 0, name)
