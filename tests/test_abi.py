"""The C ABI library: it loads, exports every declared symbol, and rejects bad
arguments on the host (no CUDA call is reached, so this runs without a GPU)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_269_gb300 as pa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    return pa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(pa.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.pa_version() >= 10000
    for code in pa.STATUS:
        assert lib.pa_status_string(code)
    assert lib.pa_status_string(12345) == b"unknown status"


def _dims(S=2, H=4, D=128, B=16, N=32):
    return pa.Dims(S, H, D, B, N)


SIZE_ERROR = (1 << 64) - 1


def test_workspace_bytes(lib):
    d = _dims(S=64, H=32, D=128, B=16, N=5000)
    single = lib.pa_decode_workspace_bytes(ctypes.byref(d), 128, 128 * 16)
    split = lib.pa_decode_workspace_bytes(ctypes.byref(d), 128, 256)
    assert single == 0 < split
    # 8 partitions x 64 x 32 pairs x (128 acc + 2) floats
    assert split >= 64 * 32 * 8 * 130 * 4
    assert lib.pa_decode_workspace_bytes(ctypes.byref(d), 128, 17) == SIZE_ERROR  # not k*B
    assert lib.pa_decode_workspace_bytes(ctypes.byref(d), 0, 256) == SIZE_ERROR
    assert lib.pa_decode_workspace_bytes(None, 128, 256) == SIZE_ERROR
    ctr = lib.pa_decode_counters_bytes(ctypes.byref(d))
    assert ctr >= (2 + 64 * 32) * 4 and ctr % 256 == 0
    assert lib.pa_decode_counters_bytes(None) == 0


@pytest.mark.parametrize("D,B,expect", [(96, 16, -3), (128, 12, -3), (0, 16, -2), (128, 0, -2)])
def test_decode_rejects_dims(lib, D, B, expect):
    d = _dims(D=D, B=B)
    rc = lib.pa_decode_ws(None, None, None, None, None, None, 0.1, 8, ctypes.byref(d), 0,
                          None, 0, None, 0, None)
    assert rc == expect


def test_decode_rejects_null_and_alignment(lib):
    d = _dims()
    fake = ctypes.c_void_p(0x100000)           # never dereferenced: checks fail first
    big = 1 << 20

    def call(out=fake, ws=fake, ws_n=big, ctr=fake, ctr_n=big, scale=0.1, mb=8, P=0):
        return lib.pa_decode_ws(out, fake, fake, fake, fake, fake, scale, mb, ctypes.byref(d), P,
                                ws, ws_n, ctr, ctr_n, None)

    assert call(out=None) == -1
    assert call(out=ctypes.c_void_p(0x100002)) == -4
    assert call(ctr=None) == -5
    assert call(ctr_n=16) == -5                  # counter buffer too small
    assert call(ws=None, P=16) == -5             # partials needed but no workspace
    assert call(ws_n=16, P=16) == -5
    assert call(scale=float("nan")) == -2
    assert call(mb=0) == -2
    assert call(P=24) == -2                      # not a multiple of block_size
    assert lib.pa_decode(fake, fake, fake, fake, fake, fake, 0.1, 0, ctypes.byref(d), None) == -2
    assert lib.pa_decode(fake, fake, fake, fake, fake, fake, 0.1, 8, None, None) == -1


def test_decode_static_rejects_before_touching_the_device(lib):
    # Every rejection below happens on the host, before the scratch array's
    # address is looked up or its counters are cleared: no CUDA call is made,
    # which is why this runs without a GPU.
    d = _dims()
    fake = ctypes.c_void_p(0x100000)           # never dereferenced: checks fail first

    def call(out=fake, q=fake, scale=0.1, mb=8, dims=d):
        return lib.pa_decode_static(out, q, fake, fake, fake, fake, scale, mb,
                                    ctypes.byref(dims) if dims is not None else None, None)

    assert call(out=None) == -1
    assert call(q=None) == -1
    assert call(dims=None) == -1
    assert call(out=ctypes.c_void_p(0x100002)) == -4
    assert call(scale=float("nan")) == -2
    assert call(scale=float("inf")) == -2
    assert call(mb=0) == -2
    assert call(dims=_dims(D=96)) == -3
    assert call(dims=_dims(S=0), out=None) == 0   # an empty batch is a no-op
    # 70000 x 64 (sequence, head) tickets need more than the 16 MiB array
    assert call(dims=pa.Dims(70000, 64, 128, 16, 1024)) == -5


def test_empty_batches_are_noops(lib):
    d = _dims(S=0)
    assert lib.pa_decode_ws(None, None, None, None, None, None, 0.1, 8, ctypes.byref(d), 0,
                            None, 0, None, 0, None) == 0
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, ctypes.byref(d), None) == 0


def test_reshape_rejects(lib):
    d = _dims()
    fake = ctypes.c_void_p(0x100000)
    assert lib.pa_reshape_and_cache(fake, fake, fake, fake, fake, -1, ctypes.byref(d), None) == -2
    assert lib.pa_reshape_and_cache(fake, None, fake, fake, fake, 4, ctypes.byref(d), None) == -1
    odd = ctypes.c_void_p(0x100008)
    assert lib.pa_reshape_and_cache(fake, odd, fake, fake, fake, 4, ctypes.byref(d), None) == -4
    bad = _dims(D=80)
    assert lib.pa_reshape_and_cache(fake, fake, fake, fake, fake, 4, ctypes.byref(bad), None) == -3


def test_prefill_rejects(lib):
    fake = ctypes.c_void_p(0x100000)           # never dereferenced: checks fail first
    d = _dims()

    def call(dims=d, out=fake, total=300, maxq=200, scale=0.1, mb=8, ctr=fake, ctr_n=8):
        return lib.pa_prefill_ws(out, fake, fake, fake, fake, fake, fake, total, maxq, scale, mb,
                                 ctypes.byref(dims) if dims is not None else None, ctr, ctr_n, None)

    assert call(dims=None) == -1
    assert call(dims=_dims(D=64)) == -3          # head_dim 128 only
    assert call(dims=_dims(B=32)) == -3          # block_size 16 only
    assert call(dims=_dims(D=0)) == -2
    assert call(total=-1) == -2
    assert call(maxq=-1) == -2
    assert call(mb=0) == -2
    assert call(dims=_dims(S=0)) == 0            # nothing to do
    assert call(total=0) == 0
    assert call(maxq=0) == 0
    assert call(out=None) == -1
    assert call(ctr=None) == -1
    assert call(ctr_n=4) == -5                   # the two work-queue counters need 8 bytes
    assert call(out=ctypes.c_void_p(0x100002)) == -4
    assert call(ctr=ctypes.c_void_p(0x100002)) == -4
    assert call(scale=float("inf")) == -2
    # more work items (pairs of 128-row tiles x sequences x heads) than an int32 counts
    assert call(dims=_dims(S=65535, H=65535, N=1), maxq=256) == -2
    # the allocating entry point validates the same way before any allocation
    assert lib.pa_prefill(fake, fake, fake, fake, fake, fake, fake, 300, 200, 0.1, 8,
                          ctypes.byref(_dims(D=64)), None) == -3
    assert lib.pa_prefill(fake, fake, fake, fake, fake, fake, fake, -1, 200, 0.1, 8,
                          ctypes.byref(d), None) == -2


def test_decode_shared_prefix_rejects(lib):
    fake = ctypes.c_void_p(0x100000)           # never dereferenced: checks fail first
    d = _dims()
    ws_need = lib.pa_decode_shared_prefix_workspace_bytes(ctypes.byref(d), 8, 0)
    ctr_need = lib.pa_decode_shared_prefix_counters_bytes(ctypes.byref(d))
    # one extra partial slot per (sequence, head) for the prefix, always present
    plain = lib.pa_decode_workspace_bytes(ctypes.byref(d), 8, 0)
    assert ws_need > plain and ws_need >= d.num_seqs * d.num_heads * 2 * (d.head_dim + 2) * 4
    assert ctr_need > lib.pa_decode_counters_bytes(ctypes.byref(d))

    def call(dims=d, out=fake, gs=fake, gp=fake, G=1, maxg=4, scale=0.1, mb=8, ws=fake,
             ws_n=ws_need, ctr=fake, ctr_n=ctr_need, pt=0):
        return lib.pa_decode_shared_prefix_ws(
            out, fake, fake, fake, fake, fake, scale, mb,
            ctypes.byref(dims) if dims is not None else None, gs, gp, G, maxg, pt, ws, ws_n,
            ctr, ctr_n, None)

    assert call(dims=None) == -1
    assert call(dims=_dims(D=64)) == -3          # the prefix kernel: head_dim 128 only
    assert call(dims=_dims(B=32)) == -3          # and block_size 16
    assert call(G=-1) == -2
    assert call(maxg=-1) == -2
    assert call(mb=0) == -2
    assert call(pt=24) == -2                     # not a multiple of the block size
    assert call(dims=_dims(S=0)) == 0            # nothing to do
    assert call(out=None) == -1
    assert call(gs=None) == -1
    assert call(gp=None) == -1
    assert call(out=ctypes.c_void_p(0x100002)) == -4
    assert call(scale=float("nan")) == -2
    assert call(ctr=None) == -5
    assert call(ctr_n=ctr_need - 4) == -5
    assert call(ctr=ctypes.c_void_p(0x100002)) == -5
    assert call(ws=None) == -5                   # the prefix partials always need a workspace
    assert call(ws_n=ws_need - 16) == -5
    assert call(ws=ctypes.c_void_p(0x100008)) == -5
    # more prefix work items (tile pairs x groups x heads) than an int32 counts
    assert call(G=1 << 24, maxg=1 << 16) == -2
    assert lib.pa_decode_shared_prefix(fake, fake, fake, fake, fake, fake, 0.1, 8,
                                       ctypes.byref(_dims(D=64)), fake, fake, 1, 4, None) == -3


def test_copy_blocks_rejects(lib):
    fake = ctypes.c_void_p(0x100000)
    d = _dims()

    def call(dims=d, n=2, src_n=32, dst_n=32, pairs=fake, dst_k=fake):
        return lib.pa_copy_blocks(fake, fake, src_n, dst_k, fake, dst_n, pairs, n,
                                  ctypes.byref(dims) if dims is not None else None, None)

    assert call(dims=None) == -1
    assert call(n=-1) == -2
    assert call(src_n=0) == -2
    assert call(dims=_dims(D=80)) == -3
    assert call(n=0) == 0                        # nothing to copy
    assert call(pairs=None) == -1
    assert call(dst_k=ctypes.c_void_p(0x100008)) == -4
    assert call(pairs=ctypes.c_void_p(0x100002)) == -4
