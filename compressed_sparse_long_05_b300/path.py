"""One CSA or HCA attention layer forward, composed from the C-ABI stages.

DeepSeek-V4 report (Chinese translation, blog.uika.cn) §2.3.1: compress the
per-token entries (m = 4, overlapped), score every visible compressed entry
with the lightning indexer, keep the top-k, and run shared-KV MQA over them
plus the 128-token window with the per-head sink.  §2.3.2: HCA compresses
with m' = 128 and attends densely.  Decode steps start from a given
compressed cache (a new entry is compressed only when a block closes).

The functions take a dict of device tensors named as in ``synth.generate``
(including the per-row query positions ``q_pos`` [B, Tq] and the window-buffer
bases ``win_base`` [B]) and a size dict as in ``synth.configs``; they only
allocate outputs and call the library.
"""

from __future__ import annotations

from . import _lib as L


class Buffers:
    """Reusable intermediate and output buffers of one layer forward."""

    def __init__(self):
        self.entries = None
        self.K = None
        self.scores = None
        self.idx = None
        self.out = None
        self.ws = None
        self.ws_topk = None


def _entries_arg(x):
    if "entries" in x:
        return x["entries"]
    return (x["ent_nope"], x["ent_scale"], x["ent_rope"])


def _win_arg(x):
    if "win" in x:
        return x["win"]
    return (x["win_nope"], x["win_scale"], x["win_rope"])


def _indexer_args(x, buf=None):
    if "CIa" in x:                      # keys compressed from raw index rows
        return x["qI"], None, buf.K, None
    if "qI" in x:
        return x["qI"], None, x["K"], None
    return x["qI_fp4"], x["qI_sf"], x["K_fp4"], x["K_sf"]


def compress_stage(cfg: dict, x: dict, buf: Buffers):
    """Prefill compression: the entries (CSA m overlapped, HCA m' plain), with
    the workload's optional RMSNorm and RoPE pre-rotation, and, when the
    workload gives raw index rows, the indexer keys K^IComp (same overlapped
    compression at d = c_I; DeepSeek-V4 report, Chinese translation, §2.3.1)."""
    m, r = cfg["m"], cfg["r"]
    opts = dict(rms_norm=bool(cfg.get("entry_norm")), norm_eps=cfg.get("entry_norm_eps", 0.0),
                rope_dims=r if cfg.get("entry_rope") else 0, rope_base=cfg["rope_base"])
    if cfg["kind"] == "csa_prefill":
        buf.entries = L.csa_compress(x["Ca"], x["Za"], m, Cb=x["Cb"], Zb=x["Zb"], out=buf.entries,
                                     **opts)
        if "CIa" in x:
            buf.K = L.csa_compress(x["CIa"], x["ZIa"], m, Cb=x["CIb"], Zb=x["ZIb"], out=buf.K)
    else:
        buf.entries = L.csa_compress(x["C"], x["Z"], m, out=buf.entries, **opts)
    return buf.entries


def forward(cfg: dict, x: dict, buf: Buffers | None = None):
    """All stages of one layer forward; returns the attention output [B, Tq, n_h, d]."""
    buf = buf or Buffers()
    kind = cfg["kind"]
    m, r, n_win = cfg["m"], cfg["r"], cfg["n_win"]
    q_pos, win_base, base = x["q_pos"], x["win_base"], cfg["rope_base"]
    rot = bool(cfg.get("entry_rope"))
    if kind.endswith("prefill"):
        entries = compress_stage(cfg, x, buf)
    else:
        entries = _entries_arg(x)
    win = _win_arg(x)
    if kind.startswith("csa"):
        qI, qI_sf, K, K_sf = _indexer_args(x, buf)
        buf.scores, buf.idx, buf.ws_topk = L.csa_index_topk(
            qI, x["w"], K, cfg["k"], m, q_pos, qI_sf=qI_sf, K_sf=K_sf, scores=buf.scores,
            idx=buf.idx, ws=buf.ws_topk)
        if buf.ws is None:
            n = L.attend_workspace_size(x["q"], entries, win, cfg["k"], m, n_win, r, False)
            buf.ws = L._workspace(None, n, x["q"].device)
        buf.out = L.csa_attend(x["q"], entries, buf.idx, win, x["sink"], m, n_win, win_base,
                               q_pos, r, base, out=buf.out, ws=buf.ws, entries_rotated=rot)
    else:
        if buf.ws is None:
            n = L.attend_workspace_size(x["q"], entries, win, 0, m, n_win, r, True)
            buf.ws = L._workspace(None, n, x["q"].device)
        buf.out = L.hca_attend(x["q"], entries, win, x["sink"], m, n_win, win_base, q_pos, r,
                               base, out=buf.out, ws=buf.ws, entries_rotated=rot)
    return buf.out


def output_projection(out, W_groups, W_out, y=None, z=None):
    """The grouped output projection after the core attention (DeepSeek-V4
    report, Chinese translation, §2.3.1 "分组输出投影"): the [B, Tq, n_h, d]
    attention output, viewed as [B*Tq, n_h*d], is split into g groups of
    (n_h/g)*d columns, group j is projected by W_groups[j] ([d_g, (n_h/g)*d])
    to d_g dims, and the concatenated [B*Tq, g*d_g] result is projected by
    W_out ([1, d_model, g*d_g]) to the model width.  Returns z [B*Tq, d_model];
    y and z may be supplied for reuse."""
    B, Tq, n_h, d = out.shape
    A = out.reshape(B * Tq, n_h * d)
    y = L.csa_grouped_proj(A, W_groups, C=y)
    return L.csa_grouped_proj(y, W_out, C=z)


def compress_entry(i: int, m: int, Ca, Za, Cb=None, Zb=None, Ba=None, Bb=None):
    """Compressed entry i alone, for each batch row: the entry a decode step adds
    to the cache when block i closes (DeepSeek-V4 report, Chinese translation,
    blog.uika.cn, §3.6.1: raw tokens wait in a buffer until their block is full).

    Ca, Za (and Cb, Zb for CSA) are [B, T, d] raw-token buffers holding at least
    tokens [m*(i-1), m*(i+1)) (CSA) or [m*i, m*(i+1)) (HCA).  Entry i of the
    overlapped compression depends only on the a-rows of block i and the b-rows
    of block i-1, so ``csa_compress`` over the two-block window [m*(i-1),
    m*(i+1)) yields it as the window's entry 1 (entry 0 of the window is not
    entry i-1 and is discarded); i = 0 and HCA take the one block.  Returns a
    [B, d] view of the kernel's output.
    """
    import torch
    B, T, d = Ca.shape
    overlap = Cb is not None
    lo = m * (i - 1) if (overlap and i > 0) else m * i
    hi = m * (i + 1)
    if i < 0 or hi > T:
        raise ValueError(f"entry {i} needs tokens [{lo}, {hi}) of a {T}-token buffer")
    row = 1 if (overlap and i > 0) else 0
    res = torch.empty((B, (hi - lo) // m, d), dtype=Ca.dtype, device=Ca.device)
    for b in range(B):   # one call per batch row: the window of each row is contiguous
        L.csa_compress(Ca[b:b + 1, lo:hi], Za[b:b + 1, lo:hi], m,
                       Cb=None if Cb is None else Cb[b:b + 1, lo:hi],
                       Zb=None if Zb is None else Zb[b:b + 1, lo:hi], Ba=Ba, Bb=Bb,
                       out=res[b:b + 1])
    return res[:, row]


class GraphForward:
    """A layer forward replayed as one CUDA graph, host transfers included.

    For a decode loop whose per-step work is tens of microseconds, launching
    each stage from Python costs more than the stages.  This captures, once:
    the copy of every name in ``host_inputs`` from its pinned host buffer into
    the device input, every stage of :func:`forward`, and the copy of the
    output back into a pinned host tensor.  Each call then replays the graph
    and waits for it.  The caller refreshes ``self.host[name]`` in place
    between calls (the graph reads those exact buffers) and reads the returned
    host output before the next call overwrites it.

    ``x`` holds the device inputs the graph reads and writes; they and the
    buffers stay owned by this object for its lifetime.
    """

    def __init__(self, cfg: dict, x: dict, host_inputs, stream=None):
        import torch
        self.cfg = cfg
        self.x = dict(x)
        self.host = {n: self.x[n].cpu().pin_memory() for n in host_inputs}
        self.buf = Buffers()
        self.stream = stream or torch.cuda.Stream()
        with torch.cuda.stream(self.stream):
            forward(cfg, self.x, self.buf)          # sizes every buffer before capture
        self.out_host = torch.empty(self.buf.out.shape, dtype=self.buf.out.dtype).pin_memory()
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream, capture_error_mode="relaxed"):
            for n, t in self.host.items():
                self.x[n].copy_(t, non_blocking=True)
            forward(cfg, self.x, self.buf)
            self.out_host.copy_(self.buf.out, non_blocking=True)
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host.values())
        self.d2h_bytes = self.out_host.numel() * self.out_host.element_size()

    def __call__(self):
        """Runs one forward on the current host inputs; returns the pinned host output."""
        import torch
        with torch.cuda.stream(self.stream):      # replay() launches on the current stream
            self.graph.replay()
        self.stream.synchronize()
        return self.out_host


class PipelinedForward:
    """A stream of independent layer forwards (e.g. prefill requests) with the
    host transfers overlapped with compute.

    Two device copies of every input in ``host_inputs`` and of the output
    alternate between steps: step s copies its inputs host -> device on one
    stream, runs every stage of :func:`forward` on a second once they are in,
    and copies its output device -> host on a third, so that step s's compute
    overlaps step s+1's upload and step s-1's download.  Each step still
    moves its own inputs and output across PCIe.

    ``submit(host)`` queues one step whose inputs are the pinned host tensors
    ``host`` (same names, shapes and dtypes as ``x``); it returns the pinned
    host output buffer that step fills, valid after ``wait(step)``.  Outputs
    alternate between two host buffers, so read a step's output before
    submitting step + 2, and leave a step's host inputs unchanged until
    ``wait(step)`` returns.
    """

    def __init__(self, cfg: dict, x: dict, host_inputs):
        import torch
        self.cfg = cfg
        self.names = list(host_inputs)
        self.sets = []
        for _ in range(2):
            xs = dict(x)
            for n in self.names:
                xs[n] = torch.empty_like(x[n])
            self.sets.append((xs, Buffers()))
        self.s_in = torch.cuda.Stream()
        self.s_run = torch.cuda.Stream()
        self.s_out = torch.cuda.Stream()
        self.ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of the set landed
        self.ev_run = [torch.cuda.Event() for _ in range(2)]     # compute of the set done
        self.ev_out = [torch.cuda.Event() for _ in range(2)]     # output of the set read back
        self.out_host = [None, None]
        self.step = 0
        for xs, buf in self.sets:                                 # size every buffer once
            with torch.cuda.stream(self.s_run):
                forward(cfg, xs, buf)
        torch.cuda.synchronize()
        self.out_host = [torch.empty(buf.out.shape, dtype=buf.out.dtype).pin_memory()
                         for _, buf in self.sets]

    def submit(self, host: dict):
        import torch
        i = self.step % 2
        xs, buf = self.sets[i]
        if self.step >= 2:
            # the set's previous compute must be done before its inputs are overwritten
            self.s_in.wait_event(self.ev_run[i])
        with torch.cuda.stream(self.s_in):
            for n in self.names:
                xs[n].copy_(host[n], non_blocking=True)
            self.ev_in[i].record(self.s_in)
        self.s_run.wait_event(self.ev_in[i])
        if self.step >= 2:
            self.s_run.wait_event(self.ev_out[i])                 # its output was read back
        with torch.cuda.stream(self.s_run):
            forward(self.cfg, xs, buf)
            self.ev_run[i].record(self.s_run)
        self.s_out.wait_event(self.ev_run[i])
        with torch.cuda.stream(self.s_out):
            self.out_host[i].copy_(buf.out, non_blocking=True)
            self.ev_out[i].record(self.s_out)
        self.step += 1
        return self.out_host[i]

    def wait(self, step: int):
        """Blocks until step ``step``'s output is in its host buffer."""
        self.ev_out[step % 2].synchronize()


class PagedKVCache:
    """The heterogeneous KV cache of one CSA and one HCA layer (DeepSeek-V4
    report, Chinese translation, blog.uika.cn, §3.6.1).

    Every block covers lcm(m, m') raw tokens, so it holds lcm/m CSA entries,
    as many indexer keys, and lcm/m' HCA entries (32, 32 and 1 at m = 4,
    m' = 128).  One block table per sequence (int32 [B, max_blocks] on the
    device, mirrored on the host) addresses all three pools; the physical
    blocks come from a native :class:`~._lib.BlockPool`.  The state cache is a
    ring of T_win window rows per sequence (token p at row p mod T_win), which
    takes each new token in place.  The raw tokens of a block that has not
    closed yet stay with the caller; :meth:`compress` writes the entries they
    produce straight into the pools (a whole prefill, or, in decode, the entry
    of each block that just closed).

    ``storage`` "bf16": bf16 entries and keys; "mixed": FP8 entries with bf16
    RoPE dims and FP4 keys with e4m3 block scales (§2.3.4, §3.4).  The
    :meth:`views` dict replaces the cache tensors of an input dict for
    :func:`forward`.
    """

    def __init__(self, B, max_tokens, num_blocks, d=512, r=64, c_I=128, T_win=128, m=4, m_hca=128,
                 storage="bf16", device="cuda"):
        import math
        import torch
        self.B, self.d, self.r, self.c_I, self.T_win = B, d, r, c_I, T_win
        self.m, self.m_hca, self.storage, self.device = m, m_hca, storage, device
        self.block_tokens = math.lcm(m, m_hca)
        self.csa_rows = self.block_tokens // m          # CSA entries (and keys) per block
        self.hca_rows = self.block_tokens // m_hca      # HCA entries per block
        self.max_blocks = -(-max_tokens // self.block_tokens)
        self.num_blocks = num_blocks
        self.pool = L.BlockPool(num_blocks)
        self.blocks = [[] for _ in range(B)]
        self.table = torch.zeros((B, self.max_blocks), dtype=torch.int32, device=device)
        nc, nh = num_blocks * self.csa_rows, num_blocks * self.hca_rows
        u8, bf = torch.uint8, torch.bfloat16
        if storage == "bf16":
            self.ent = torch.zeros((nc, d), dtype=bf, device=device)
            self.hca = torch.zeros((nh, d), dtype=bf, device=device)
            self.keys = torch.zeros((nc, c_I), dtype=bf, device=device)
            self.keys_sf = None
            self.win = torch.zeros((B, T_win, d), dtype=bf, device=device)
        elif storage == "mixed":
            def rows(lead):      # (e4m3 dims, float32 scale, bf16 RoPE dims)
                return (torch.zeros(lead + (d - r,), dtype=u8, device=device),
                        torch.zeros(lead, dtype=torch.float32, device=device),
                        torch.zeros(lead + (r,), dtype=bf, device=device))
            self.ent = rows((nc,))
            self.hca = rows((nh,))
            self.keys = torch.zeros((nc, c_I // 2), dtype=u8, device=device)
            self.keys_sf = torch.zeros((nc, c_I // 16), dtype=u8, device=device)
            self.win = rows((B, T_win))
        else:
            raise ValueError(f"storage {storage!r}: 'bf16' or 'mixed'")

    # ---------------- blocks ----------------
    def reserve(self, b, tokens):
        """Gives sequence b enough blocks for its first ``tokens`` raw tokens."""
        import torch
        need = -(-tokens // self.block_tokens)
        if need > self.max_blocks:
            raise ValueError(f"{tokens} tokens need {need} blocks; the table holds {self.max_blocks}")
        have = len(self.blocks[b])
        if need > have:
            new = self.pool.alloc(need - have)
            self.blocks[b] += new
            self.table[b, have:need] = torch.tensor(new, dtype=torch.int32).to(self.device)

    def release(self, b):
        """Returns sequence b's blocks to the pool."""
        if self.blocks[b]:
            self.pool.release(self.blocks[b])
        self.blocks[b] = []

    # ---------------- views for the kernels ----------------
    def entries(self, N):
        return L.Paged(self.ent, self.table, self.csa_rows, N)

    def hca_entries(self, N):
        return L.Paged(self.hca, self.table, self.hca_rows, N)

    def index_keys(self, N):
        return L.Paged(self.keys, self.table, self.csa_rows, N)

    def window(self):
        return L.Paged(self.win, None, 0, self.T_win, ring=True)

    def views(self, kind, N):
        """Replacements for the cache tensors of an input dict of :func:`forward`
        (``kind`` "csa" or "hca"; N entries per sequence)."""
        v = {"win": self.window()}
        if kind == "hca":
            v["entries"] = self.hca_entries(N)
            return v
        v["entries"] = self.entries(N)
        if self.storage == "mixed":
            v["K_fp4"] = self.index_keys(N)
            v["K_sf"] = self.keys_sf
        else:
            v["K"] = self.index_keys(N)
        return v

    # ---------------- writes ----------------
    def _rows_of(self, b, n, per_block):
        """Physical pool rows of logical rows 0..n-1 of sequence b (host side)."""
        import torch
        j = torch.arange(n)
        blk = torch.tensor(self.blocks[b], dtype=torch.int64)[j // per_block]
        return (blk * per_block + j % per_block).to(self.device)

    def load(self, kind, b, rows, sf=None):
        """Copies sequence b's logical rows 0..n-1 (a [n, ...] tensor, or the
        (e4m3, scale, rope) tuple) into its blocks; ``kind`` "entries", "hca" or
        "keys" (``sf``: the keys' e4m3 scale bytes)."""
        per = self.hca_rows if kind == "hca" else self.csa_rows
        pool = {"entries": self.ent, "hca": self.hca, "keys": self.keys}[kind]
        n = (rows[0] if isinstance(rows, (tuple, list)) else rows).shape[0]
        idx = self._rows_of(b, n, per)
        if isinstance(pool, tuple):
            for p, src in zip(pool, rows):
                p[idx] = src
        else:
            pool[idx] = rows
        if sf is not None:
            self.keys_sf[idx] = sf

    def load_window(self, b, rows, base):
        """Puts sequence b's window tokens base .. base+n-1 (rows [n, ...], or the
        (e4m3, scale, rope) tuple) at their ring rows."""
        import torch
        n = (rows[0] if isinstance(rows, (tuple, list)) else rows).shape[0]
        ring = (torch.arange(n) + base) % self.T_win
        ring = ring.to(self.device)
        if isinstance(self.win, tuple):
            for p, src in zip(self.win, rows):
                p[b][ring] = src
        else:
            self.win[b][ring] = rows

    def compress(self, kind, Ca, Za, Cb=None, Zb=None, entry0=None, first=0, **opts):
        """Compresses raw rows [B, T, d] straight into the bf16 pool of ``kind``
        ("entries", "hca" or "keys"): entry i >= first of sequence b goes to
        logical row entry0[b] + i - first (int32 [B] device tensor, None = 0;
        negative: nothing written).  ``opts``: the csa_compress epilogue."""
        if self.storage != "bf16":
            raise ValueError("compression writes bf16 pools")
        per = self.hca_rows if kind == "hca" else self.csa_rows
        pool = {"entries": self.ent, "hca": self.hca, "keys": self.keys}[kind]
        m = self.m_hca if kind == "hca" else self.m
        out = L.Paged(pool, self.table, per, self.max_blocks * per)
        L.csa_compress(Ca, Za, m, Cb=Cb, Zb=Zb, out=out, out_entry0=entry0, out_first=first, **opts)

    @classmethod
    def from_inputs(cls, cfg: dict, x: dict, extra_blocks=16, seed=0):
        """A cache holding a decode workload's flat cache tensors (the input dict
        of :func:`forward`), its blocks handed out round-robin over the
        sequences in a shuffled order (so no sequence's blocks are contiguous);
        returns (cache, views) with ``views`` as from :meth:`views`."""
        import numpy as np
        B, L, m = cfg["B"], cfg["L"], cfg["m"]
        kind = "csa" if cfg["kind"].startswith("csa") else "hca"
        lengths = cfg.get("lengths") or [L] * B
        mixed = cfg["dtype"] == "mixed"
        cache = cls(B, L, B * -(-L // 128) + extra_blocks, d=cfg["d"], r=cfg["r"],
                    c_I=cfg.get("c_I", 128), T_win=cfg["T_win"], m=4, m_hca=128,
                    storage="mixed" if mixed else "bf16", device=x["q"].device)
        rng = np.random.default_rng(seed)
        for j in range(-(-L // cache.block_tokens)):
            for b in rng.permutation(B):
                if j * cache.block_tokens < lengths[b]:
                    cache.reserve(int(b), min(lengths[b], (j + 1) * cache.block_tokens))
        for b, Lb in enumerate(lengths):
            Nb = Lb // m
            if mixed:
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
        return cache, cache.views(kind, cfg["N"])
