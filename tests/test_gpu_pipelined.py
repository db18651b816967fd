"""path.PipelinedForward: a stream of prefill steps whose host transfers overlap
other steps' compute must give, step by step, what eager ``path.forward`` gives."""

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,over", [
    ("csa_prefill_32k", dict(T=2048)),
    ("hca_prefill_64k", dict(T=4096)),
])
def test_pipelined_forward_matches_eager(name, over):
    from compressed_sparse_long_05_b300 import path as P
    cfg = synth.scaled(name, **over)
    x = synth.make_inputs(cfg, seed=5, device="cuda")
    names = ["q"] + [n for n in ("qI", "w", "Ca", "Cb", "Za", "Zb", "C", "Z", "win") if n in x]
    pf = P.PipelinedForward(cfg, x, names)
    # three different steps: the inputs of step s are x scaled by (1 + s/8)
    hosts = []
    for s in range(3):
        h = {}
        for n in names:
            t = x[n].float() * (1.0 + s / 8.0) if x[n].is_floating_point() else x[n]
            h[n] = t.to(x[n].dtype).cpu().pin_memory()
        hosts.append(h)
    outs = []
    for s in range(3):
        if s >= 2:
            pf.wait(s - 2)
            outs.append(pf.out_host[(s - 2) % 2].clone())
        pf.submit(hosts[s])
    for s in (1, 2):
        pf.wait(s)
        outs.append(pf.out_host[s % 2].clone())
    for s in range(3):
        xe = dict(x)
        for n in names:
            xe[n] = hosts[s][n].to("cuda")
        want = P.forward(cfg, xe).cpu()
        torch.cuda.synchronize()
        assert torch.equal(outs[s], want), f"{name} step {s}"
