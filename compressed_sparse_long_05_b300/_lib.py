"""ctypes binding of libcsa_b300.so (include/csa.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory and
the current stream); shapes are read from them and passed as plain ints.
Loading fails loudly when the library has not been built.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# CSA_LIB_TRACE=1 loads the phase-trace build of the same sources (build --trace)
TRACE = os.environ.get("CSA_LIB_TRACE") == "1"
LIB_PATH = os.path.join(HERE, "lib", "libcsa_b300_trace.so" if TRACE else "libcsa_b300.so")

DT_F32, DT_BF16, DT_E4M3_BF16ROPE, DT_E2M1_BLOCK16 = 0, 1, 2, 3
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported shape or dtype",
          3: "workspace missing or too small", 4: "CUDA runtime error",
          5: "device wait timed out", 6: "device-side fault"}


class CsaError(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))


class Pages(ctypes.Structure):
    """csa_pages_t: block table (device int32 [B, max_blocks]) of a paged row set."""
    _fields_ = [("block_table", ctypes.c_void_p), ("max_blocks", ctypes.c_int32),
                ("block_rows", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("ring", ctypes.c_int32)]


class KV(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("flags", ctypes.c_int32), ("data", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("rope", ctypes.c_void_p), ("pages", Pages)]


class CompressOpts(ctypes.Structure):
    _fields_ = [("rms_norm", ctypes.c_int32), ("norm_eps", ctypes.c_float),
                ("norm_weight", ctypes.c_void_p), ("rope_dims", ctypes.c_int32),
                ("rope_base", ctypes.c_float), ("out_pages", Pages), ("out_entry0", ctypes.c_void_p),
                ("out_first", ctypes.c_int32)]


class Paged:
    """Rows of a paged cache, or of a per-sequence ring buffer.

    ``pool``: the rows, [num_blocks * block_rows, d] (or the (e4m3, scale,
    rope) tuple of pools for FP8 rows; for FP4 keys the packed bytes, with the
    scale bytes passed separately); ``table``: int32 device tensor
    [B, max_blocks] naming the physical block of each logical block, or None
    for a flat [B, rows, d] ``pool``; ``rows``: logical rows per sequence (N,
    or T_win); ``ring``: window rows, token p at logical row p mod rows.
    """

    def __init__(self, pool, table=None, block_rows=0, rows=None, ring=False):
        self.pool, self.table, self.block_rows, self.ring = pool, table, block_rows, ring
        first = pool[0] if isinstance(pool, (tuple, list)) else pool
        if table is None:
            self.B, self.rows = first.shape[0], first.shape[1]
            self.num_blocks = 0
        else:
            if table.dtype != torch.int32 or table.dim() != 2 or not table.is_contiguous():
                raise ValueError("table must be a contiguous int32 [B, max_blocks] tensor")
            if rows is None:
                raise ValueError("a paged row set needs its logical row count")
            self.B, self.rows = table.shape[0], rows
            self.num_blocks = first.shape[0] // block_rows
        self.d = None if isinstance(pool, (tuple, list)) else first.shape[-1]
        if isinstance(pool, (tuple, list)):
            self.d = pool[0].shape[-1] + pool[2].shape[-1]

    def pages(self):
        if self.table is None:
            return Pages(None, 0, 0, 0, 1 if self.ring else 0)
        return Pages(self.table.data_ptr(), self.table.shape[1], self.block_rows, self.num_blocks,
                     1 if self.ring else 0)


KV_ROTATED = 1


_lib = None

_I, _P, _F, _Z = ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "csa_compress": [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P],
    "csa_compress_ex": [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                        ctypes.POINTER(CompressOpts), _P],
    "csa_index": [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P],
    "csa_topk": [_P, _I, _P, _P, _I, _I, _I, _I, _I, _P],
    "csa_index_topk": [_P, _P, _P, _P, _P, _P, _P, _I, _P] + [_I] * 8 + [_P, _Z, _P],
    "csa_index_topk_workspace_size": [_I] * 4,
    "csa_attend": [_P, KV, _P, KV, _P, _P, _P, _P] + [_I] * 10 + [_F, _P, _Z, _P],
    "hca_attend": [_P, KV, KV, _P, _P, _P, _P] + [_I] * 9 + [_F, _P, _Z, _P],
    "csa_attend_noalloc": [_P, KV, _P, KV, _P, _P, _P, _P] + [_I] * 10 + [_F, _P],
    "csa_attend_workspace_size": [_I] * 13,
    "csa_selftest_wait_timeout": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P],
    "csa_grouped_proj": [_P, ctypes.c_int64, _P, _P, ctypes.c_int64, _I, _I, _I, _I, _P],
    "csa_index_paged": [_P, _P, _P, _P, _P, ctypes.POINTER(Pages), _P, _P, _I] + [_I] * 7 + [_P],
    "csa_index_topk_paged": [_P, _P, _P, _P, _P, ctypes.POINTER(Pages), _P, _P, _I, _P] + [_I] * 8
                            + [_P, _Z, _P],
    "csa_decode_step_host": [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(Pages), KV, KV, _P, _P]
                            + [_I] * 12 + [_F, _P, _Z, _P],
    "csa_decode_step_workspace_size": [_I] * 13,
    "csa_block_pool_create": [ctypes.c_int32],
    "csa_block_pool_destroy": [_P],
    "csa_block_pool_free_count": [_P],
    "csa_block_pool_alloc": [_P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
    "csa_block_pool_release": [_P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
    "csa_device_error": [_P],
    "csa_status_string": [_I],
    "csa_last_cuda_error": [],
    "csa_version": [],
}
_RESTYPES = {"csa_decode_step_workspace_size": _Z, "csa_block_pool_create": _P, "csa_block_pool_destroy": None,
             "csa_block_pool_free_count": ctypes.c_int32, "csa_attend_workspace_size": _Z, "csa_index_topk_workspace_size": _Z, "csa_status_string": ctypes.c_char_p,
             "csa_last_cuda_error": ctypes.c_char_p}


def lib():
    """The loaded library (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m compressed_sparse_long_05_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _RESTYPES.get(name, ctypes.c_int)
        if TRACE:
            L.csa_trace_read.argtypes = [_P, _I]
            L.csa_trace_read.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(fn, status):
    if status != 0:
        detail = lib().csa_last_cuda_error().decode() if status == 4 else ""
        raise CsaError(fn, status, detail)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dt(t):
    if t.dtype == torch.float32:
        return DT_F32
    if t.dtype == torch.bfloat16:
        return DT_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _kv(rows, rotated=False):
    """A row set: a float32/bf16 tensor [B, rows, d], (e4m3 bytes, scale, bf16 rope),
    or a :class:`Paged` of either; ``rotated``: its RoPE dims are already
    rotated at each entry's position."""
    fl = KV_ROTATED if rotated else 0
    pg = Pages()
    if isinstance(rows, Paged):
        pg = rows.pages()
        rows = rows.pool
    if isinstance(rows, (tuple, list)):
        nope, scale, rope = rows
        return KV(DT_E4M3_BF16ROPE, fl, nope.data_ptr(), scale.data_ptr(), rope.data_ptr(), pg)
    return KV(_dt(rows), fl, rows.data_ptr(), None, None, pg)


def positions(q_pos, B, Tq, device):
    """Query positions as the library takes them: None (row i at position i),
    an int p0 (row i of every batch row at p0 + i) made into a [B, Tq] int32
    device tensor, or such a tensor as given."""
    if q_pos is None or (isinstance(q_pos, int) and q_pos == 0):
        return None
    if isinstance(q_pos, int):
        t = torch.arange(q_pos, q_pos + Tq, dtype=torch.int32, device=device)
        return t.unsqueeze(0).expand(B, Tq).contiguous()
    if q_pos.dtype != torch.int32 or tuple(q_pos.shape) != (B, Tq) or not q_pos.is_contiguous():
        raise ValueError(f"q_pos must be a contiguous int32 [{B}, {Tq}] tensor")
    return q_pos


def window_bases(win_base, B, device):
    """Window buffer bases: None (0), an int shared by every batch row, or an
    int32 [B] device tensor."""
    if win_base is None or (isinstance(win_base, int) and win_base == 0):
        return None
    if isinstance(win_base, int):
        return torch.full((B,), win_base, dtype=torch.int32, device=device)
    if win_base.dtype != torch.int32 or tuple(win_base.shape) != (B,) or not win_base.is_contiguous():
        raise ValueError(f"win_base must be a contiguous int32 [{B}] tensor")
    return win_base


def _rows_shape(rows):
    if isinstance(rows, Paged):
        return rows.B, rows.rows, rows.d
    if isinstance(rows, (tuple, list)):
        nope, _, rope = rows
        return nope.shape[0], nope.shape[1], nope.shape[2] + rope.shape[2]
    return rows.shape[0], rows.shape[1], rows.shape[2]


# ----------------------------------------------------------------------------


def csa_compress(Ca, Za, m, Cb=None, Zb=None, Ba=None, Bb=None, out=None, rms_norm=False,
                 norm_eps=0.0, norm_weight=None, rope_dims=0, rope_base=10000.0, out_entry0=None,
                 out_first=0):
    """Compressed entries [B, T//m, d] (Cb = Zb = None: HCA, no overlap).

    ``rms_norm`` / ``rope_dims``: the optional epilogue of csa_compress_ex
    (RMSNorm of every entry, then RoPE of its last rope_dims dims at its
    position).  ``out`` may be a :class:`Paged` pool: entry i >= out_first of
    sequence b then goes to logical row out_entry0[b] + i - out_first
    (``out_entry0``: int32 [B] device tensor, None = 0; negative: nothing
    written for that sequence)."""
    B, T, d = Ca.shape
    if out is None:
        out = torch.empty((B, T // m, d), dtype=Ca.dtype, device=Ca.device)
    if isinstance(out, Paged):
        opts = CompressOpts(1 if rms_norm else 0, norm_eps,
                            None if norm_weight is None else norm_weight.data_ptr(), rope_dims,
                            rope_base, out.pages(), None if out_entry0 is None else out_entry0.data_ptr(),
                            out_first)
        _check("csa_compress_ex", lib().csa_compress_ex(
            _p(Ca), _p(Cb), _p(Za), _p(Zb), _p(Ba), _p(Bb), _p(out.pool), B, T, d, m, _dt(Ca),
            ctypes.byref(opts), _stream()))
        return out
    if not rms_norm and not rope_dims:
        _check("csa_compress", lib().csa_compress(_p(Ca), _p(Cb), _p(Za), _p(Zb), _p(Ba), _p(Bb),
                                                  _p(out), B, T, d, m, _dt(Ca), _stream()))
        return out
    opts = CompressOpts(1 if rms_norm else 0, norm_eps,
                        None if norm_weight is None else norm_weight.data_ptr(), rope_dims,
                        rope_base, Pages(), None, 0)
    _check("csa_compress_ex", lib().csa_compress_ex(
        _p(Ca), _p(Cb), _p(Za), _p(Zb), _p(Ba), _p(Bb), _p(out), B, T, d, m, _dt(Ca),
        ctypes.byref(opts), _stream()))
    return out


def csa_index(qI, w, K, m, q_pos, qI_sf=None, K_sf=None, scores=None, score_dtype=torch.float32):
    """Indexer scores [B, Tq, N] (-inf where not visible), float32 or bf16.

    ``q_pos``: query positions (see :func:`positions`).  ``score_dtype``
    torch.bfloat16 stores every score rounded to bf16."""
    fp4 = qI.dtype == torch.uint8
    B, Tq, H = qI.shape[:3]
    c = qI.shape[3] * (2 if fp4 else 1)
    Kt, kpg, N = _keys(K)
    dt = DT_E2M1_BLOCK16 if fp4 else _dt(qI)
    qp = positions(q_pos, B, Tq, qI.device)
    if scores is None:
        scores = torch.empty((B, Tq, N), dtype=score_dtype, device=qI.device)
    _check("csa_index", lib().csa_index_paged(
        _p(qI), _p(qI_sf), _p(w), _p(Kt), _p(K_sf), kpg, _p(qp), _p(scores), _dt(scores), B, Tq, N,
        H, c, m, dt, _stream()))
    return scores


def _keys(K):
    """(key tensor or pool, csa_pages_t pointer or None, keys per sequence)."""
    if isinstance(K, Paged):
        return K.pool, (ctypes.byref(K.pages()) if K.table is not None else None), K.rows
    return K, None, K.shape[1]


def csa_topk(scores, k, m, q_pos, idx=None):
    """Selected entry indices [B, Tq, k] int32, ascending, -1 padded (float32 or
    bf16 scores)."""
    B, Tq, N = scores.shape
    qp = positions(q_pos, B, Tq, scores.device)
    if idx is None:
        idx = torch.empty((B, Tq, k), dtype=torch.int32, device=scores.device)
    _check("csa_topk", lib().csa_topk(_p(scores), _dt(scores), _p(qp), _p(idx), B, Tq, N, k, m,
                                      _stream()))
    return idx


def csa_index_topk(qI, w, K, k, m, q_pos, qI_sf=None, K_sf=None, scores=None, idx=None, ws=None,
                   score_dtype=torch.float32):
    """Indexer scores and the top-k index sets of one call (same results as
    csa_index then csa_topk); returns (scores, idx, ws).

    ``ws`` (returned for reuse) must be zero-filled before its first call: a new
    one is allocated zeroed, and every successful call leaves it zero.  After a
    failed call pass ``ws=None`` (or zero it) again."""
    fp4 = qI.dtype == torch.uint8
    B, Tq, H = qI.shape[:3]
    c = qI.shape[3] * (2 if fp4 else 1)
    Kt, kpg, N = _keys(K)
    dt = DT_E2M1_BLOCK16 if fp4 else _dt(qI)
    if scores is None:
        scores = torch.empty((B, Tq, N), dtype=score_dtype, device=qI.device)
    if idx is None:
        idx = torch.empty((B, Tq, k), dtype=torch.int32, device=qI.device)
    qp = positions(q_pos, B, Tq, qI.device)
    nbytes = lib().csa_index_topk_workspace_size(B, Tq, N, dt)
    ws = _workspace(ws, nbytes, qI.device, zero=True)   # histograms start zero; calls leave them zero
    _check("csa_index_topk", lib().csa_index_topk_paged(
        _p(qI), _p(qI_sf), _p(w), _p(Kt), _p(K_sf), kpg, _p(qp), _p(scores), _dt(scores), _p(idx), B,
        Tq, N, H, c, m, k, dt, _p(ws) if nbytes else None, nbytes, _stream()))
    return scores, idx, ws


def attend_workspace_size(q, entries, win, k, m, n_win, r, is_hca):
    B, Tq, n_h, d = q.shape
    _, N, _ = _rows_shape(entries)
    _, T_win, _ = _rows_shape(win)
    kv_dt = _kv(entries).dtype
    return lib().csa_attend_workspace_size(B, Tq, N, k, T_win, n_h, d, r, m, n_win,
                                           _dt(q), kv_dt, 1 if is_hca else 0)


def _workspace(ws, nbytes, device, zero=False):
    if nbytes == 0:
        return ws
    if ws is None or ws.numel() < nbytes:
        ws = (torch.zeros if zero else torch.empty)(nbytes, dtype=torch.uint8, device=device)
    return ws


def csa_attend(q, entries, idx, win, sink, m, n_win, win_base, q_pos, r, rope_base=10000.0,
               out=None, ws=None, entries_rotated=False):
    """Sparse shared-KV attention output [B, Tq, n_h, d] (dtype of q).

    ``q_pos``: query positions (see :func:`positions`); ``win_base``: token of
    window row 0 per batch row (see :func:`window_bases`); ``entries_rotated``:
    the entries' RoPE dims are already rotated (csa_compress with rope_dims)."""
    B, Tq, n_h, d = q.shape
    _, N, _ = _rows_shape(entries)
    _, T_win, _ = _rows_shape(win)
    k = idx.shape[2]
    qp, wb = positions(q_pos, B, Tq, q.device), window_bases(win_base, B, q.device)
    if out is None:
        out = torch.empty_like(q)
    nbytes = attend_workspace_size(q, entries, win, k, m, n_win, r, False)
    ws = _workspace(ws, nbytes, q.device)
    _check("csa_attend", lib().csa_attend(
        _p(q), _kv(entries, entries_rotated), _p(idx), _kv(win), _p(qp), _p(wb), _p(sink), _p(out), B, Tq, N, k,
        T_win, n_h, d, r, m, n_win, rope_base, _p(ws) if nbytes else None, nbytes, _stream()))
    return out


def csa_attend_noalloc(q, entries, idx, win, sink, m, n_win, win_base, q_pos, r,
                       rope_base=10000.0, out=None):
    """csa_attend with its scratch in the library's fixed device array (no workspace).

    For callers that must not allocate device memory beyond the output; see
    include/csa.h for the size limit and the sharing rules of that array.
    """
    B, Tq, n_h, d = q.shape
    _, N, _ = _rows_shape(entries)
    _, T_win, _ = _rows_shape(win)
    k = idx.shape[2]
    qp, wb = positions(q_pos, B, Tq, q.device), window_bases(win_base, B, q.device)
    if out is None:
        out = torch.empty_like(q)
    _check("csa_attend_noalloc", lib().csa_attend_noalloc(
        _p(q), _kv(entries), _p(idx), _kv(win), _p(qp), _p(wb), _p(sink), _p(out), B, Tq, N, k,
        T_win, n_h, d, r, m, n_win, rope_base, _stream()))
    return out


def hca_attend(q, entries, win, sink, m, n_win, win_base, q_pos, r, rope_base=10000.0,
               out=None, ws=None, entries_rotated=False):
    """Dense (HCA) shared-KV attention output [B, Tq, n_h, d] (dtype of q)."""
    B, Tq, n_h, d = q.shape
    _, N, _ = _rows_shape(entries)
    _, T_win, _ = _rows_shape(win)
    qp, wb = positions(q_pos, B, Tq, q.device), window_bases(win_base, B, q.device)
    if out is None:
        out = torch.empty_like(q)
    nbytes = attend_workspace_size(q, entries, win, 0, m, n_win, r, True)
    ws = _workspace(ws, nbytes, q.device)
    _check("hca_attend", lib().hca_attend(
        _p(q), _kv(entries, entries_rotated), _kv(win), _p(qp), _p(wb), _p(sink), _p(out), B, Tq, N, T_win, n_h, d,
        r, m, n_win, rope_base, _p(ws) if nbytes else None, nbytes, _stream()))
    return out


def csa_grouped_proj(A, W, C=None, G=None, lda=None, ldc=None):
    """One grouped projection GEMM: for j < G, C[:, jN:(j+1)N] = A[:, jK:(j+1)K] W[j]^T.

    A: [M, >= G*K] bf16 (row stride ``lda``, default its row length); W:
    [G, N, K] bf16; returns C [M, G*N] bf16 (or fills ``C``)."""
    Gw, N, K = W.shape
    G = Gw if G is None else G
    M = A.shape[0]
    lda = A.stride(0) if lda is None else lda
    if C is None:
        C = torch.empty((M, G * N), dtype=torch.bfloat16, device=A.device)
    ldc = C.stride(0) if ldc is None else ldc
    _check("csa_grouped_proj", lib().csa_grouped_proj(_p(A), lda, _p(W), _p(C), ldc, M, N, K, G,
                                                      _stream()))
    return C


def device_error():
    """Reads and clears the library's sticky device error word; raises if it was set."""
    _check("csa_device_error", lib().csa_device_error(_stream()))


class BlockPool:
    """Host-side allocator of the physical blocks of a paged cache
    (csa_block_pool_*): ids 0 .. num_blocks-1, handed out and taken back."""

    def __init__(self, num_blocks):
        self._h = lib().csa_block_pool_create(num_blocks)
        if not self._h:
            raise CsaError("csa_block_pool_create", 1, f"num_blocks={num_blocks}")
        self.num_blocks = num_blocks

    def free_count(self):
        return int(lib().csa_block_pool_free_count(self._h))

    def alloc(self, n):
        ids = (ctypes.c_int32 * max(n, 1))()
        _check("csa_block_pool_alloc", lib().csa_block_pool_alloc(self._h, n, ids))
        return [int(ids[i]) for i in range(n)]

    def release(self, ids):
        arr = (ctypes.c_int32 * max(len(ids), 1))(*ids)
        _check("csa_block_pool_release", lib().csa_block_pool_release(self._h, len(ids), arr))

    def close(self):
        if self._h:
            lib().csa_block_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DecodeStepHost:
    """One CSA decode step through the C ABI from host buffers
    (csa_decode_step_host): the step's inputs are copied from pinned host
    tensors, the index, top-k and attention run against the device-resident
    cache, and the output lands in a pinned host tensor.

    ``cache``: device tensors or :class:`Paged` views as :func:`csa_attend`
    takes them (``entries``, ``win``, ``K`` with ``K_sf`` for FP4 keys) plus
    ``sink``; ``B`` sequences, ``k``, ``m``, ``n_win``, ``r`` as the layer's.
    ``host`` holds pinned tensors ``q`` [B,1,n_h,d] bf16, ``qI`` (or ``qI_fp4``
    and ``qI_sf``), ``w``, ``q_pos`` [B] int32 and ``win_base`` [B] int32; the
    caller refreshes them in place between steps.  ``__call__`` queues one step
    on the current stream, waits for it and returns the pinned output.  With
    ``graph=True`` the call is captured once into a CUDA graph (it only queues
    asynchronous work, so the copies from the same pinned buffers, the kernels
    and the copy back replay as they were queued) and each step replays it.
    """

    def __init__(self, cache, host, k, m, n_win, r, rope_base=10000.0, graph=False):
        self.cache, self.host = cache, host
        self.k, self.m, self.n_win, self.r, self.rope_base = k, m, n_win, r, rope_base
        q = host["q"]
        self.B, _, self.n_h, self.d = q.shape
        qI = host.get("qI", host.get("qI_fp4"))
        self.fp4 = "qI_fp4" in host
        self.H = qI.shape[2]
        self.c = qI.shape[3] * (2 if self.fp4 else 1)
        self.Kt, self.kpg, self.N = _keys(cache["K"])
        self.T_win = _rows_shape(cache["win"])[1]
        self.dt = DT_E2M1_BLOCK16 if self.fp4 else DT_BF16
        self.ent_kv, self.win_kv = _kv(cache["entries"]), _kv(cache["win"])
        nbytes = lib().csa_decode_step_workspace_size(self.B, self.N, self.H, self.c, k, self.T_win,
                                                      self.n_h, self.d, r, m, n_win, self.dt,
                                                      self.ent_kv.dtype)
        if nbytes == 0:
            raise CsaError("csa_decode_step_workspace_size", 1)
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=q.device if q.is_cuda else "cuda")
        self.out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for n, t in host.items()
                             if n in ("q", "qI", "qI_fp4", "qI_sf", "w", "q_pos", "win_base"))
        self.d2h_bytes = self.out.numel() * self.out.element_size()
        self.graph = None
        if graph:
            self._queue()                          # sets kernel attributes, caches the plans
            torch.cuda.current_stream().synchronize()
            self.graph = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            with torch.cuda.graph(self.graph, stream=side, capture_error_mode="relaxed"):
                self._queue()

    def __call__(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self._queue()
        torch.cuda.current_stream().synchronize()
        return self.out

    def _queue(self):
        h = self.host
        st = _stream()
        _check("csa_decode_step_host", lib().csa_decode_step_host(
            _p(h["q"]), _p(h["qI_fp4"] if self.fp4 else h["qI"]), _p(h.get("qI_sf")), _p(h["w"]),
            _p(h["q_pos"]), _p(h.get("win_base")), _p(self.Kt), _p(self.cache.get("K_sf")), self.kpg,
            self.ent_kv, self.win_kv, _p(self.cache["sink"]), _p(self.out), self.B, self.N, self.H,
            self.c, self.k, self.T_win, self.n_h, self.d, self.r, self.m, self.n_win, self.dt,
            self.rope_base, _p(self.ws), self.ws.numel(), st))
