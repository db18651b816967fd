"""csa_decode_step_host: one CSA decode step through the C ABI from host
buffers (the step's inputs copied from pinned host memory, index, top-k and
attention against the device-resident cache, the output copied back).

It runs the same kernels on the same inputs as the device-side layer forward
(`path.forward`), so its output must agree bit for bit: on decode batches at
mixed context lengths in the bf16 and the FP8/FP4 formats, on two calls in a
row (the top-k histograms it keeps in its workspace must be left zero), as a
captured CUDA graph replayed twice, and through the paged cache.  The
device-side forward is itself checked against the float64 oracle in
test_gpu_mixed_lengths.py and test_gpu_paged.py.
"""

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _host_inputs(x):
    names = ["q", "w"] + (["qI_fp4", "qI_sf"] if "qI_fp4" in x else ["qI"])
    h = {n: x[n].cpu().pin_memory() for n in names}
    h["q_pos"] = x["q_pos"][:, 0].contiguous().cpu().pin_memory()
    h["win_base"] = x["win_base"].cpu().pin_memory()
    return h


def _cache(x):
    mixed = "ent_nope" in x
    c = {"sink": x["sink"]}
    c["entries"] = (x["ent_nope"], x["ent_scale"], x["ent_rope"]) if mixed else x["entries"]
    c["win"] = (x["win_nope"], x["win_scale"], x["win_rope"]) if mixed else x["win"]
    if mixed:
        c["K"], c["K_sf"] = x["K_fp4"], x["K_sf"]
    else:
        c["K"] = x["K"]
    return c


@pytest.mark.parametrize("name,lengths", [
    ("csa_decode_128k", [131072, 70001, 2050, 77]),
    ("csa_decode_1m_mixed", [65536, 40003, 3000, 130]),
])
def test_host_step_equals_the_device_forward(name, lengths):
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import path as P
    cfg = synth.scaled(name, B=len(lengths), lengths=lengths)
    x = synth.make_inputs(cfg, seed=7, device=DEV)
    ref = P.forward(cfg, x, P.Buffers()).cpu()
    torch.cuda.synchronize()
    K.device_error()
    step = K.DecodeStepHost(_cache(x), _host_inputs(x), cfg["k"], cfg["m"], cfg["n_win"], cfg["r"],
                            cfg["rope_base"])
    for _ in range(2):                       # the second call reuses the histograms the first cleared
        out = step()
        K.device_error()
        assert torch.equal(out, ref)
    assert step.h2d_bytes > 0 and step.d2h_bytes == ref.numel() * 2
    # the same call captured once into a CUDA graph and replayed
    gstep = K.DecodeStepHost(_cache(x), _host_inputs(x), cfg["k"], cfg["m"], cfg["n_win"], cfg["r"],
                             cfg["rope_base"], graph=True)
    for _ in range(2):
        out = gstep()
        K.device_error()
        assert torch.equal(out, ref)


def test_host_step_through_the_paged_cache():
    import compressed_sparse_long_05_b300 as K
    from compressed_sparse_long_05_b300 import path as P
    lengths = [40000, 9001, 600]
    cfg = synth.scaled("csa_decode_128k", B=3, lengths=lengths)
    x = synth.make_inputs(cfg, seed=9, device=DEV)
    ref = P.forward(cfg, x, P.Buffers()).cpu()
    cache, views = P.PagedKVCache.from_inputs(cfg, x)
    c = {"sink": x["sink"], "entries": views["entries"], "win": views["win"], "K": views["K"]}
    step = K.DecodeStepHost(c, _host_inputs(x), cfg["k"], cfg["m"], cfg["n_win"], cfg["r"],
                            cfg["rope_base"])
    out = step()
    K.device_error()
    assert torch.equal(out, ref)
