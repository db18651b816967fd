"""Seeded synthetic inputs for the CSA / HCA forward path.

The recipe (one generator per tensor, seeded by a CRC of workload name, tensor
name and seed):

* per-token/per-entry vectors that the attention reads (C^a, C^b, C, the
  compressed entries of a decode cache, the raw window entries, the queries):
  N(0,1) in float32, then each vector divided by its RMS, then stored in the
  workload dtype;
* compression logits Z^a, Z^b, Z: N(0,1);
* indexer queries and keys: N(0,1) * qk_scale (1/sqrt(c_I)); workloads whose
  keys are compressed from raw rows get those rows (CIa, CIb ~ N(0,1) *
  qk_scale) and their compression logits (ZIa, ZIb ~ N(0,1)) instead;
* indexer head weights w: U(0,1) * w_scale;
* per-head sink logits z'_h: N(0,1);
* query positions q_pos [B, Tq] and window-buffer bases win_base [B] (int32)
  from the workload's context lengths (synth.configs.derive).

The mixed-precision workload stores the first d-r dims of every entry as FP8
e4m3 with one float32 scale per entry (amax/448) and the last r (RoPE) dims as
bf16; indexer queries and keys are FP4 e2m1 codes, two per byte (element 2j in
the low nibble), with one e4m3 scale byte per 16 elements (the smallest e4m3
value >= amax/6).  Quantisation happens here, once; every consumer reads the
same bytes.

Values depend on the device the generator runs on (torch's CPU and CUDA
generators differ); a parity check always feeds both sides the same tensors.
This module holds none of the method's arithmetic.
"""

from __future__ import annotations

import zlib

import torch

_CHUNK = 1 << 26  # elements generated per call, bounds float32 temporaries

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def seed_for(workload: str, tensor: str, seed: int = 0) -> int:
    return zlib.crc32(f"{workload}/{tensor}/{seed}".encode()) & 0x7FFFFFFF


def _gen(device, workload, tensor, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(workload, tensor, seed))
    return g


def _rows(shape):
    inner = shape[-1]
    rows = 1
    for s in shape[:-1]:
        rows *= s
    return rows, inner


def normal(shape, dtype, device, g, scale=1.0, rms_normalise=False):
    """N(0,1)*scale, optionally each last-dim vector divided by its RMS."""
    rows, inner = _rows(shape)
    out = torch.empty((rows, inner), dtype=dtype, device=device)
    step = max(1, _CHUNK // inner)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = torch.randn((r1 - r0, inner), generator=g, device=device,
                        dtype=torch.float32)
        if rms_normalise:
            x = x * torch.rsqrt(x.square().mean(dim=1, keepdim=True))
        if scale != 1.0:
            x = x * scale
        out[r0:r1] = x.to(dtype)
    return out.view(shape)


def uniform(shape, dtype, device, g, scale=1.0):
    rows, inner = _rows(shape)
    out = torch.empty((rows, inner), dtype=dtype, device=device)
    step = max(1, _CHUNK // inner)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        x = torch.rand((r1 - r0, inner), generator=g, device=device,
                       dtype=torch.float32) * scale
        out[r0:r1] = x.to(dtype)
    return out.view(shape)


# ----------------------------------------------------------------------------
# storage-format encoders (input preparation only)
# ----------------------------------------------------------------------------

def encode_e4m3(x: torch.Tensor) -> torch.Tensor:
    """float32 -> e4m3fn bytes, round to nearest even, saturating at +-448."""
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def e4m3_ceil(v: torch.Tensor) -> torch.Tensor:
    """Smallest non-negative e4m3 code whose value is >= v (v >= 0), as bytes."""
    v = v.clamp(min=2.0 ** -9, max=E4M3_MAX)
    code = v.to(torch.float8_e4m3fn)
    back = code.to(torch.float32)
    b = code.view(torch.uint8).to(torch.int16)
    b = torch.where(back < v, b + 1, b)
    return b.to(torch.uint8)


_E2M1_TIES_UP = (0.75, 1.75, 3.5)
_E2M1_BOUNDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def encode_e2m1(x: torch.Tensor) -> torch.Tensor:
    """float32 (|x| <= 6) -> e2m1 4-bit codes (uint8, one code per element).

    Round to nearest; a value half-way between two codes goes to the code with
    an even mantissa bit.
    """
    a = x.abs().clamp(max=E2M1_MAX)
    mag = torch.zeros_like(a, dtype=torch.uint8)
    for b in _E2M1_BOUNDS:
        mag += (a > b).to(torch.uint8)
    for b in _E2M1_TIES_UP:
        mag += (a == b).to(torch.uint8)
    sign = ((x < 0) & (mag > 0)).to(torch.uint8) << 3
    return mag | sign


def quantise_fp4_blocks(x: torch.Tensor, block: int = 16):
    """x [..., c] -> (packed e2m1 [..., c/2] uint8, e4m3 scales [..., c/block])."""
    shape = x.shape
    xb = x.float().reshape(*shape[:-1], shape[-1] // block, block)
    amax = xb.abs().amax(dim=-1)
    sf = e4m3_ceil(amax / E2M1_MAX)
    sf_val = sf.view(torch.float8_e4m3fn).to(torch.float32)
    codes = encode_e2m1(xb / sf_val.unsqueeze(-1)).reshape(shape)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed.contiguous(), sf.contiguous()


def quantise_mixed_entries(x: torch.Tensor, r: int):
    """Entries [..., d] -> (e4m3 bytes [..., d-r], fp32 scale [...], bf16 rope [..., r])."""
    d = x.shape[-1]
    nope = x[..., : d - r].float()
    amax = nope.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q8 = encode_e4m3(nope / scale.unsqueeze(-1))
    rope = x[..., d - r:].to(torch.bfloat16)
    return q8.contiguous(), scale.float().contiguous(), rope.contiguous()


# ----------------------------------------------------------------------------

def _storage_dtype(cfg):
    return torch.float32 if cfg["dtype"] == "f32" else torch.bfloat16


def make_inputs(cfg: dict, seed: int = 0, device="cpu") -> dict:
    """All inputs of workload ``cfg`` (see synth.configs) as torch tensors."""
    name = cfg["name"]
    dt = _storage_dtype(cfg)
    B, d, n_h = cfg["B"], cfg["d"], cfg["n_h"]
    Tq, N, T_win = cfg["Tq"], cfg["N"], cfg["T_win"]
    kind = cfg["kind"]
    mixed = cfg["dtype"] == "mixed"
    out = {}

    def g(t):
        return _gen(device, name, t, seed)

    from .configs import query_positions, window_bases
    out["q_pos"] = torch.tensor(query_positions(cfg), dtype=torch.int32, device=device)
    out["win_base"] = torch.tensor(window_bases(cfg), dtype=torch.int32, device=device)
    out["q"] = normal((B, Tq, n_h, d), dt, device, g("q"), rms_normalise=True)
    out["sink"] = normal((n_h,), torch.float32, device, g("sink"))

    win = normal((B, T_win, d), torch.float32 if mixed else dt, device, g("win"),
                 rms_normalise=True)
    if mixed:
        out["win_nope"], out["win_scale"], out["win_rope"] = quantise_mixed_entries(win, cfg["r"])
    else:
        out["win"] = win

    if kind.startswith("csa"):
        H, c = cfg["H_I"], cfg["c_I"]
        qI = normal((B, Tq, H, c), torch.float32 if mixed else dt, device, g("qI"),
                    scale=cfg["qk_scale"])
        if cfg.get("index_keys") == "compressed":
            # raw per-token index rows; the keys are their overlapped compression
            T = cfg["T"]
            for nm in ("CIa", "CIb"):
                out[nm] = normal((B, T, c), dt, device, g(nm), scale=cfg["qk_scale"])
            for nm in ("ZIa", "ZIb"):
                out[nm] = normal((B, T, c), dt, device, g(nm))
            K = None
        else:
            K = normal((B, N, c), torch.float32 if mixed else dt, device, g("K"),
                       scale=cfg["qk_scale"])
        if mixed:
            out["qI_fp4"], out["qI_sf"] = quantise_fp4_blocks(qI)
            out["K_fp4"], out["K_sf"] = quantise_fp4_blocks(K)
        else:
            out["qI"] = qI
            if K is not None:
                out["K"] = K
        out["w"] = uniform((B, Tq, H), torch.float32, device, g("w"), scale=cfg["w_scale"])

    if kind == "csa_prefill":
        T = cfg["T"]
        for nm in ("Ca", "Cb"):
            out[nm] = normal((B, T, d), dt, device, g(nm), rms_normalise=True)
        for nm in ("Za", "Zb"):
            out[nm] = normal((B, T, d), dt, device, g(nm))
    elif kind == "hca_prefill":
        T = cfg["T"]
        out["C"] = normal((B, T, d), dt, device, g("C"), rms_normalise=True)
        out["Z"] = normal((B, T, d), dt, device, g("Z"))
    else:  # decode: the compressed cache is given
        ent = normal((B, N, d), torch.float32 if mixed else dt, device, g("entries"),
                     rms_normalise=True)
        if mixed:
            out["ent_nope"], out["ent_scale"], out["ent_rope"] = quantise_mixed_entries(ent, cfg["r"])
        else:
            out["entries"] = ent
    return out
