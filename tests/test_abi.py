"""The C-ABI library builds for sm_103a, loads, exports every symbol that
include/csa.h declares, and rejects bad arguments on the host (no GPU needed:
these calls return before touching CUDA)."""

import ctypes
import os
import re

import pytest

from compressed_sparse_long_05_b300 import build as B


@pytest.fixture(scope="module")
def L():
    B.build()
    from compressed_sparse_long_05_b300 import _lib
    return _lib.lib()


def declared(root):
    txt = open(os.path.join(root, "include", "csa.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"^\s*(?:csa_status_t|size_t|int|int32_t|void|const char\*|csa_block_pool_t\*)"
                       r"\s+(\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(L, root):
    names = declared(root)
    assert "csa_attend" in names and "csa_topk" in names and len(names) >= 10
    assert "csa_block_pool_alloc" in names and "csa_index_topk_paged" in names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    assert L.csa_status_string(0) == b"ok"
    assert L.csa_status_string(2) == b"unsupported shape or dtype"
    assert L.csa_version() >= 1


def _p(v):
    return ctypes.c_void_p(v)


def test_host_side_argument_errors(L):
    from compressed_sparse_long_05_b300._lib import KV
    fake = _p(0x10000)      # never dereferenced: every call below fails validation first
    mis = _p(0x10002)
    # null output / input
    assert L.csa_compress(None, None, None, None, None, None, None, 1, 8, 64, 4, 1, None) == 1
    # half an overlap pair
    assert L.csa_compress(fake, fake, fake, None, None, None, fake, 1, 8, 64, 4, 1, None) == 1
    # misaligned pointer
    assert L.csa_compress(mis, None, fake, None, None, None, fake, 1, 8, 64, 4, 1, None) == 1
    # unsupported dtype / width
    assert L.csa_compress(fake, None, fake, None, None, None, fake, 1, 8, 64, 4, 3, None) == 2
    assert L.csa_compress(fake, None, fake, None, None, None, fake, 1, 8, 60, 4, 1, None) == 2
    # top-k: k out of range, negative sizes, misaligned positions, unknown score type
    assert L.csa_topk(fake, 0, None, fake, 1, 1, 100, 0, 4, None) == 1
    assert L.csa_topk(fake, 0, None, fake, 1, 1, 100, 5000, 4, None) == 1
    assert L.csa_topk(fake, 0, None, fake, -1, 1, 100, 5, 4, None) == 1
    assert L.csa_topk(fake, 0, mis, fake, 1, 1, 100, 5, 4, None) == 1
    assert L.csa_topk(fake, 3, None, fake, 1, 1, 100, 5, 4, None) == 2
    # bf16 scores beyond 16 x 32768 keys per row: the 8-bit selector reads float32 only
    assert L.csa_topk(fake, 1, None, fake, 1, 1, 600000, 5, 4, None) == 2
    # index: null scores
    assert L.csa_index(fake, None, fake, fake, None, None, None, 0, 1, 1, 8, 4, 32, 4, 0, None) == 1
    kv = KV(dtype=1, flags=0, data=0x10000)
    # attend: odd rope dims
    assert L.csa_attend(fake, kv, fake, kv, None, None, fake, fake, 1, 1, 8, 4, 128, 128, 512, 63,
                        4, 128, 10000.0, None, 0, None) == 1
    # attend: misaligned window bases
    assert L.csa_attend(fake, kv, fake, kv, None, mis, fake, fake, 1, 1, 8, 4, 128, 128, 512, 64,
                        4, 128, 10000.0, None, 0, None) == 1
    # attend: no index list
    assert L.csa_attend(fake, kv, None, kv, None, None, fake, fake, 1, 1, 8, 4, 128, 128, 512, 64,
                        4, 128, 10000.0, None, 0, None) == 1
    # attend: no kernel for d = 500 with bf16 rows
    assert L.csa_attend(fake, kv, fake, kv, None, None, fake, fake, 1, 1, 8, 4, 128, 128, 500, 64,
                        4, 128, 10000.0, None, 0, None) == 2
    # attend: a workspace the plan needs but the caller did not pass (prefill-shaped:
    # every stored row is rotated once into the workspace)
    assert L.csa_attend(fake, kv, fake, kv, None, None, fake, fake, 1, 4096, 1024, 64, 4096, 128,
                        512, 64, 4, 128, 10000.0, None, 0, None) == 3
    # empty batch is a no-op
    assert L.csa_topk(fake, 0, None, fake, 0, 1, 100, 5, 4, None) == 0


def test_workspace_sizes_follow_the_plan(L):
    # host-side planning only (no device is touched)
    L.csa_index_topk_workspace_size.restype = ctypes.c_size_t
    L.csa_attend_workspace_size.restype = ctypes.c_size_t
    # the histogram workspace of the fused decode call: one 2048-bin row per batch row
    assert L.csa_index_topk_workspace_size(4, 1, 32768, 1) == 4 * 2048 * 4
    assert L.csa_index_topk_workspace_size(8, 1, 262144, 3) == 8 * 2048 * 4
    assert L.csa_index_topk_workspace_size(1, 2, 32768, 1) == 0          # not a decode row
    assert L.csa_index_topk_workspace_size(1, 1, 32768, 0) == 0          # fp32 scores: two calls
    # decode, 128K context, batch 4: 9 chunks of 128 rows per head group; unless the
    # chunks merge inside a cluster, each keeps a [64 heads][512] fp32 partial
    ws = L.csa_attend_workspace_size(4, 1, 32768, 1024, 128, 128, 512, 64, 4, 128, 1, 1, 0)
    assert ws == 0 or ws >= 72 * 64 * 512 * 4
    # causal prefill: every stored row is rotated once into the workspace (1 KB per row)
    ws = L.csa_attend_workspace_size(1, 32768, 8192, 1024, 32768, 128, 512, 64, 4, 128, 1, 1, 0)
    assert ws >= (8192 + 32768) * 1024
    # shapes the tensor-core path does not take need no workspace
    assert L.csa_attend_workspace_size(1, 1, 100, 16, 16, 4, 128, 32, 4, 16, 0, 0, 0) == 0


def test_paged_argument_errors(L):
    # row maps (csa_pages_t) are checked on the host before any launch
    from compressed_sparse_long_05_b300._lib import KV, CompressOpts, Pages
    fake = _p(0x10000)
    mis = 0x10002
    tab = 0x20000
    kv = KV(dtype=1, flags=0, data=0x10000)
    def att(ent_pages, win_pages):
        e = KV(dtype=1, flags=0, data=0x10000, pages=ent_pages)
        w = KV(dtype=1, flags=0, data=0x10000, pages=win_pages)
        return L.csa_attend(fake, e, fake, w, None, None, fake, fake, 1, 1, 1000, 64, 128, 128,
                            512, 64, 4, 128, 10000.0, None, 0, None)
    # too few table columns for N = 1000 entries of 128 rows per block
    assert att(Pages(tab, 7, 128, 64, 0), Pages()) == 1
    # misaligned table, zero block rows, empty pool
    assert att(Pages(mis, 10, 128, 64, 0), Pages()) == 1
    assert att(Pages(tab, 10, 0, 64, 0), Pages()) == 1
    assert att(Pages(tab, 10, 128, 0, 0), Pages()) == 1
    # ring order applies to window rows only
    assert att(Pages(tab, 10, 128, 64, 1), Pages()) == 1
    # index keys: tiled loads need power-of-two block rows >= 8 (bf16)
    for rows, want in ((12, 2), (4, 2)):
        pg = Pages(tab, 1000, rows, 64, 0)
        assert L.csa_index_paged(fake, None, fake, fake, None, ctypes.byref(pg), None, fake, 0, 1, 1,
                                 1000, 64, 128, 4, 1, None) == want
    # compress into pages: negative first entry, misaligned entry offsets
    o = CompressOpts(out_pages=Pages(tab, 10, 32, 64, 0), out_first=-1)
    assert L.csa_compress_ex(fake, fake, fake, fake, None, None, fake, 1, 8, 64, 4, 1,
                             ctypes.byref(o), None) == 1
    o = CompressOpts(out_pages=Pages(tab, 10, 32, 64, 0), out_entry0=mis)
    assert L.csa_compress_ex(fake, fake, fake, fake, None, None, fake, 1, 8, 64, 4, 1,
                             ctypes.byref(o), None) == 1
    o = CompressOpts(out_pages=Pages(tab, 10, 32, 64, 1))
    assert L.csa_compress_ex(fake, fake, fake, fake, None, None, fake, 1, 8, 64, 4, 1,
                             ctypes.byref(o), None) == 1


def test_block_pool():
    # host-only allocator of the paged cache's physical blocks (no GPU involved)
    from compressed_sparse_long_05_b300._lib import BlockPool, CsaError
    p = BlockPool(6)
    assert p.free_count() == 6
    a = p.alloc(4)
    assert a == [0, 1, 2, 3] and p.free_count() == 2
    with pytest.raises(CsaError) as e:
        p.alloc(3)                              # only 2 free: nothing is taken
    assert e.value.status == 3 and p.free_count() == 2
    for bad in ([4], [0, 0], [7], [-1], [1, 5]):  # free, repeated, out of range, mixed
        with pytest.raises(CsaError) as e:
            p.release(bad)
        assert e.value.status == 1
    assert p.free_count() == 2                  # refused releases change nothing
    p.release([2, 0])
    assert p.free_count() == 4
    b = p.alloc(4)
    assert sorted(b) == [0, 2, 4, 5] and p.free_count() == 0
    p.release(a[1:2] + a[3:] + b)
    assert p.free_count() == 6 and sorted(p.alloc(6)) == list(range(6))
    p.close()
    from compressed_sparse_long_05_b300._lib import lib
    lib().csa_block_pool_create.restype = ctypes.c_void_p
    assert lib().csa_block_pool_create(0) is None
    assert lib().csa_block_pool_create((1 << 30) + 1) is None


def test_decode_step_host_arguments(L):
    # host-side checks of the host-buffer decode step (no device is touched)
    from compressed_sparse_long_05_b300._lib import KV
    L.csa_decode_step_workspace_size.restype = ctypes.c_size_t
    args = (4, 32768, 64, 128, 1024, 128, 128, 512, 64, 4, 128)
    n = L.csa_decode_step_workspace_size(*args, 1, 1)
    # at least the staged queries, the float32 scores, the indices and the device output
    assert n >= 4 * 128 * 512 * 2 * 2 + 4 * 32768 * 4 + 4 * 1024 * 4
    assert L.csa_decode_step_workspace_size(*args, 0, 1) == 0        # float32 keys: not a decode format
    assert L.csa_decode_step_workspace_size(0, *args[1:], 1, 1) == 0
    fake = _p(0x10000)
    kv = KV(dtype=1, flags=0, data=0x10000)
    call = lambda q, ws, nbytes: L.csa_decode_step_host(
        q, fake, None, fake, fake, None, fake, None, None, kv, kv, fake, fake, *args[:4], 1024, 128,
        128, 512, 64, 4, 128, 1, ctypes.c_float(1e4), ws, ctypes.c_size_t(nbytes), None)
    assert call(None, None, 0) == 1                    # no host queries
    assert call(fake, None, 0) == 3                    # no workspace
    assert call(fake, _p(0x10100), 16) == 3            # workspace too small
