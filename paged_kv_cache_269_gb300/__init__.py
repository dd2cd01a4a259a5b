"""PagedAttention decode on GB300: the Python binding of libpa.

libpa is a C-ABI shared library of hand-written sm_103a CUDA kernels (see
include/pa.h).  This module only marshals arguments: it checks torch tensors,
passes their device pointers and the current CUDA stream through ctypes, and
turns non-zero status codes into exceptions.  Every step of the computation
runs in libpa's kernels; there is no CPU or PyTorch fallback, and a missing or
unbuildable library raises.

Functions (names follow the C ABI):
  reshape_and_cache(k, v, k_cache, v_cache, slot_mapping)
  copy_blocks(src_k, src_v, dst_k, dst_v, block_pairs)
  decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, ...)
  decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                       group_start, group_prefix_blocks, ...)
  decode_workspace_bytes(...), decode_counters_bytes(...), device_errors(), version(),
  selftest_wait_timeout()
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

__all__ = ["PaError", "Dims", "KVManager", "lib", "reshape_and_cache", "copy_blocks", "decode",
           "decode_shared_prefix", "selftest_wait_timeout",
           "prefill", "decode_workspace_bytes", "decode_shared_prefix_workspace_bytes",
           "decode_shared_prefix_counters_bytes",
           "decode_counters_bytes", "device_errors", "reset_workspaces", "version", "DEVERR_TABLE", "DEVERR_CONTEXT",
           "DEVERR_SLOT", "DEVERR_TIMEOUT", "DEVERR_PREFIX"]

DEVERR_TABLE = 0x1
DEVERR_CONTEXT = 0x2
DEVERR_SLOT = 0x4
DEVERR_TIMEOUT = 0x8
DEVERR_PREFIX = 0x10

STATUS = {0: "PA_OK", -1: "PA_ERR_NULL", -2: "PA_ERR_SHAPE", -3: "PA_ERR_UNSUPPORTED",
          -4: "PA_ERR_ALIGN", -5: "PA_ERR_WORKSPACE", -6: "PA_ERR_CUDA",
          -7: "PA_ERR_OUT_OF_BLOCKS"}

# Every symbol include/pa.h declares.
EXPORTS = ("pa_reshape_and_cache", "pa_copy_blocks", "pa_decode", "pa_prefill", "pa_prefill_ws",
           "pa_decode_workspace_bytes",
           "pa_decode_counters_bytes", "pa_decode_ws", "pa_decode_static", "pa_device_errors",
           "pa_status_string", "pa_last_cuda_error", "pa_version",
           "pa_kvm_create", "pa_kvm_destroy", "pa_kvm_num_free_blocks", "pa_kvm_refcount",
           "pa_kvm_add_sequence", "pa_kvm_fork", "pa_kvm_append", "pa_kvm_free",
           "pa_kvm_context_len", "pa_kvm_slot", "pa_kvm_block_tables", "pa_selftest_wait_timeout",
           "pa_decode_shared_prefix", "pa_decode_shared_prefix_ws",
           "pa_decode_shared_prefix_workspace_bytes", "pa_decode_shared_prefix_counters_bytes",
           "pa_kvm_prefix_groups")
_SIZE_ERROR = (1 << 64) - 1


class PaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


DTYPE_F16 = 0
DTYPE_BF16 = 1


class Dims(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def _declare(l):
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    dp = ctypes.POINTER(Dims)
    l.pa_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i32, dp, vp]
    l.pa_copy_blocks.argtypes = [vp, vp, i32, vp, vp, i32, vp, i32, dp, vp]
    l.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, i32, dp, vp]
    l.pa_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, ctypes.c_float, i32, dp, vp]
    l.pa_selftest_wait_timeout.argtypes = [vp, vp]
    l.pa_selftest_wait_timeout.restype = ctypes.c_int
    l.pa_prefill_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, ctypes.c_float, i32, dp, vp,
                                ctypes.c_size_t, vp]
    l.pa_decode_workspace_bytes.argtypes = [dp, i32, i32]
    l.pa_decode_workspace_bytes.restype = sz
    l.pa_decode_counters_bytes.argtypes = [dp]
    l.pa_decode_counters_bytes.restype = sz
    l.pa_decode_ws.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, i32, dp, i32, vp, sz, vp,
                               sz, vp]
    l.pa_decode_static.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, i32, dp, vp]
    l.pa_decode_shared_prefix_workspace_bytes.argtypes = [dp, i32, i32]
    l.pa_decode_shared_prefix_workspace_bytes.restype = sz
    l.pa_decode_shared_prefix_counters_bytes.argtypes = [dp]
    l.pa_decode_shared_prefix_counters_bytes.restype = sz
    l.pa_decode_shared_prefix_ws.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, i32, dp, vp, vp,
                                             i32, i32, i32, vp, sz, vp, sz, vp]
    l.pa_decode_shared_prefix.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, i32, dp, vp, vp,
                                          i32, i32, vp]
    l.pa_decode_static.restype = ctypes.c_int
    l.pa_device_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    l.pa_status_string.argtypes = [ctypes.c_int]
    l.pa_status_string.restype = ctypes.c_char_p
    l.pa_last_cuda_error.argtypes = []
    l.pa_version.argtypes = []
    i32p = ctypes.POINTER(ctypes.c_int32)
    l.pa_kvm_create.argtypes = [i32, i32, i32, ctypes.c_uint64]
    l.pa_kvm_create.restype = vp
    l.pa_kvm_destroy.argtypes = [vp]
    l.pa_kvm_destroy.restype = None
    l.pa_kvm_num_free_blocks.argtypes = [vp]
    l.pa_kvm_refcount.argtypes = [vp, i32]
    l.pa_kvm_add_sequence.argtypes = [vp, i32, i32, i32, i32p]
    l.pa_kvm_fork.argtypes = [vp, i32, i32p]
    l.pa_kvm_append.argtypes = [vp, i32, i32p, i32p, i32p]
    l.pa_kvm_free.argtypes = [vp, i32]
    l.pa_kvm_context_len.argtypes = [vp, i32]
    l.pa_kvm_slot.argtypes = [vp, i32, i32, i32p]
    l.pa_kvm_block_tables.argtypes = [vp, vp, i32, vp, i32, vp]
    l.pa_kvm_prefix_groups.argtypes = [vp, vp, i32, vp, vp, i32, ctypes.POINTER(ctypes.c_int32)]
    for name in ("pa_kvm_num_free_blocks", "pa_kvm_refcount", "pa_kvm_add_sequence",
                 "pa_kvm_fork", "pa_kvm_append", "pa_kvm_free", "pa_kvm_context_len",
                 "pa_kvm_slot", "pa_kvm_block_tables", "pa_kvm_prefix_groups"):
        getattr(l, name).restype = i32
    for name in ("pa_reshape_and_cache", "pa_copy_blocks", "pa_decode", "pa_prefill", "pa_prefill_ws",
                 "pa_decode_ws", "pa_decode_shared_prefix", "pa_decode_shared_prefix_ws",
                 "pa_device_errors",
                 "pa_last_cuda_error", "pa_version"):
        getattr(l, name).restype = ctypes.c_int
    return l


def lib(path: str | None = None):
    """The loaded libpa (built first if missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.build()
            _lib = _declare(ctypes.CDLL(p))
        return _lib


def version() -> int:
    return lib().pa_version()


def _check(rc: int, what: str):
    if rc != 0:
        l = lib()
        msg = l.pa_status_string(rc).decode()
        if rc == -6:
            msg += f" (cudaError {l.pa_last_cuda_error()})"
        raise PaError(rc, f"{what}: {STATUS.get(rc, rc)}: {msg}")


# ----------------------------------------------------------------------------
# torch marshalling
# ----------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_handle(device, stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream), stream


def _need(t, name, dtype, ndim, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _need_out(t, et, ndim, device):
    """The output of a decode: a CUDA tensor on `device`, or pinned host
    memory, which the kernel then writes directly over the host link."""
    torch = _torch()
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError("out must be a CUDA tensor or pinned host memory")
        if t.dtype != et or t.dim() != ndim or not t.is_contiguous():
            raise ValueError(f"out must be a contiguous {ndim}-d tensor of {et}")
        return
    _need(t, "out", et, ndim, device)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _element_dtype(k_cache):
    """The library dtype code of a cache tensor (fp16 or bf16)."""
    torch = _torch()
    if k_cache.dtype == torch.float16:
        return DTYPE_F16
    if k_cache.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"k_cache must be float16 or bfloat16, got {k_cache.dtype}")


def _cache_dims(k_cache, num_seqs=0):
    N, H, B, D = k_cache.shape
    return Dims(num_seqs, H, D, B, N, _element_dtype(k_cache))


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """k_cache[slot // B, :, slot % B, :] = k[i] (same for v) for every i with
    slot = slot_mapping[i] >= 0.  Caches are updated in place."""
    torch = _torch()
    _element_dtype(k_cache)
    et = k_cache.dtype
    _need(k_cache, "k_cache", et, 4)
    dev = k_cache.device
    _need(v_cache, "v_cache", et, 4, dev)
    _need(k, "k", et, 3, dev)
    _need(v, "v", et, 3, dev)
    _need(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    N, H, B, D = k_cache.shape
    T = k.shape[0]
    if v_cache.shape != k_cache.shape or k.shape != (T, H, D) or v.shape != k.shape \
            or slot_mapping.shape[0] != T:
        raise ValueError("reshape_and_cache: inconsistent shapes")
    dims = _cache_dims(k_cache)
    sh, _ = _stream_handle(dev, stream)
    with torch.cuda.device(dev):
        rc = lib().pa_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(slot_mapping), T, ctypes.byref(dims), sh)
    _check(rc, "pa_reshape_and_cache")


def copy_blocks(src_k, src_v, dst_k, dst_v, block_pairs, stream=None):
    """Copy K and V of block src to block dst (all heads) for every row
    (src, dst) of block_pairs [n, 2] int32 (a CUDA tensor).  The pools are
    [N, H, B, D] tensors of one 16-bit dtype, each on the CUDA device or in
    pinned host memory, so one call does copy-on-write (same pool), swap-out
    (device -> pinned host) or swap-in (pinned host -> device)."""
    torch = _torch()
    if not isinstance(block_pairs, torch.Tensor) or not block_pairs.is_cuda:
        raise ValueError("block_pairs must be a CUDA tensor")
    dev = block_pairs.device
    if block_pairs.dtype != torch.int32 or block_pairs.dim() != 2 or block_pairs.shape[1] != 2 \
            or not block_pairs.is_contiguous():
        raise ValueError("block_pairs must be a contiguous int32 [n, 2] tensor")
    _element_dtype(src_k)
    for name, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v)):
        if not isinstance(t, torch.Tensor) or t.dtype != src_k.dtype or t.dim() != 4 \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-d tensor of {src_k.dtype}")
        if t.is_cuda:
            if t.device != dev:
                raise ValueError(f"{name} is on {t.device}, expected {dev}")
        elif not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if src_v.shape != src_k.shape or dst_v.shape != dst_k.shape or src_k.shape[1:] != dst_k.shape[1:]:
        raise ValueError("copy_blocks: inconsistent pool shapes")
    N_src, H, B, D = src_k.shape
    dims = Dims(0, H, D, B, N_src, _element_dtype(src_k))
    sh, _ = _stream_handle(dev, stream)
    with torch.cuda.device(dev):
        rc = lib().pa_copy_blocks(_ptr(src_k), _ptr(src_v), N_src, _ptr(dst_k), _ptr(dst_v),
                                  dst_k.shape[0], _ptr(block_pairs), block_pairs.shape[0],
                                  ctypes.byref(dims), sh)
    _check(rc, "pa_copy_blocks")


PREFILL_COUNTERS_BYTES = 8


def prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
            max_query_len=None, stream=None, counters=None, allocate_in_library=False):
    """Causal attention of the last q_len_s tokens of each sequence over its
    paged K/V (pa_prefill_ws; pa_prefill with allocate_in_library).  q, out
    [total_q, H, D]; query_start [S + 1] int32 on the device; max_query_len
    bounds every q_len_s (computed from query_start, with a device sync, when
    None).  counters: a zeroed int32 CUDA tensor of at least 2 elements for
    the kernel's work queue (left zeroed); by default one cached per (device,
    stream)."""
    torch = _torch()
    _element_dtype(k_cache)
    et = k_cache.dtype
    _need(k_cache, "k_cache", et, 4)
    dev = k_cache.device
    _need(v_cache, "v_cache", et, 4, dev)
    _need(q, "q", et, 3, dev)
    _need(out, "out", et, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(query_start, "query_start", torch.int32, 1, dev)
    N, H, B, D = k_cache.shape
    S = context_lens.shape[0]
    if out.shape != q.shape or q.shape[1:] != (H, D) or query_start.shape[0] != S + 1 \
            or block_tables.shape[0] != S:
        raise ValueError("prefill: inconsistent shapes")
    if max_query_len is None:
        max_query_len = int((query_start[1:] - query_start[:-1]).max()) if S else 0
    dims = _cache_dims(k_cache, S)
    sh, st = _stream_handle(dev, stream)
    with torch.cuda.device(dev):
        if allocate_in_library:
            rc = lib().pa_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(block_tables), _ptr(context_lens), _ptr(query_start),
                                  q.shape[0], int(max_query_len), float(scale),
                                  block_tables.shape[1], ctypes.byref(dims), sh)
        else:
            if counters is None:
                counters = _prefill_counters_for(dev, st)
            _need(counters, "counters", torch.int32, 1, dev)
            rc = lib().pa_prefill_ws(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_tables), _ptr(context_lens), _ptr(query_start),
                                     q.shape[0], int(max_query_len), float(scale),
                                     block_tables.shape[1], ctypes.byref(dims), _ptr(counters),
                                     counters.numel() * 4, sh)
    _check(rc, "pa_prefill")
    return out


_prefill_counters = {}


def _prefill_counters_for(device, stream):
    torch = _torch()
    key = (device.index, stream.cuda_stream)
    with _buf_lock:
        ctr = _prefill_counters.get(key)
        if ctr is None:
            with torch.cuda.stream(stream):
                ctr = torch.zeros(16, dtype=torch.int32, device=device)
            _prefill_counters[key] = ctr
        return ctr


def decode_workspace_bytes(num_seqs, num_heads, head_dim, block_size, num_blocks,
                           max_blocks_per_seq, partition_tokens=0, dtype=DTYPE_F16) -> int:
    """Bytes of partial-result workspace pa_decode_ws needs (0: none)."""
    dims = Dims(num_seqs, num_heads, head_dim, block_size, num_blocks, dtype)
    n = lib().pa_decode_workspace_bytes(ctypes.byref(dims), max_blocks_per_seq, partition_tokens)
    if n == _SIZE_ERROR:
        raise PaError(-2, "pa_decode_workspace_bytes: invalid sizes")
    return n


def decode_counters_bytes(num_seqs, num_heads, head_dim=128, block_size=16, num_blocks=1) -> int:
    """Bytes of the (zeroed, reusable) counter buffer pa_decode_ws needs."""
    dims = Dims(num_seqs, num_heads, head_dim, block_size, num_blocks)
    n = lib().pa_decode_counters_bytes(ctypes.byref(dims))
    if n == 0:
        raise PaError(-2, "pa_decode_counters_bytes: invalid sizes")
    return n


def decode_shared_prefix_workspace_bytes(num_seqs, num_heads, head_dim, block_size, num_blocks,
                                         max_blocks_per_seq, partition_tokens=0,
                                         dtype=DTYPE_F16) -> int:
    """Bytes of workspace pa_decode_shared_prefix_ws needs."""
    dims = Dims(num_seqs, num_heads, head_dim, block_size, num_blocks, dtype)
    n = lib().pa_decode_shared_prefix_workspace_bytes(ctypes.byref(dims), max_blocks_per_seq,
                                                      partition_tokens)
    if n == _SIZE_ERROR:
        raise PaError(-2, "pa_decode_shared_prefix_workspace_bytes: invalid sizes")
    return n


def decode_shared_prefix_counters_bytes(num_seqs, num_heads, head_dim=128, block_size=16,
                                        num_blocks=1) -> int:
    """Bytes of the (zeroed, reusable) counter buffer pa_decode_shared_prefix_ws needs."""
    dims = Dims(num_seqs, num_heads, head_dim, block_size, num_blocks)
    n = lib().pa_decode_shared_prefix_counters_bytes(ctypes.byref(dims))
    if n == 0:
        raise PaError(-2, "pa_decode_shared_prefix_counters_bytes: invalid sizes")
    return n


# Per (device, stream): a zeroed counter buffer, which every successful call
# leaves zeroed, and a scratch workspace for partial results (no initialisation
# needed).  Both grow on demand.
_buffers: dict = {}
_buf_lock = threading.Lock()


def _buffers_for(device, stream, counters_bytes, workspace_bytes):
    torch = _torch()
    key = (device.index, stream.cuda_stream)
    with _buf_lock:
        ctr, ws = _buffers.get(key, (None, None))
        with torch.cuda.stream(stream):
            if ctr is None or ctr.numel() * 4 < counters_bytes:
                ctr = torch.zeros(max(counters_bytes, 1 << 16) // 4, dtype=torch.int32,
                                  device=device)
            if workspace_bytes and (ws is None or ws.numel() < workspace_bytes):
                ws = torch.empty(max(workspace_bytes, 1 << 20), dtype=torch.uint8, device=device)
        _buffers[key] = (ctr, ws)
        return ctr, ws


def reset_workspaces():
    """Zero every cached counter buffer (needed after a device error)."""
    with _buf_lock:
        for ctr, _ in _buffers.values():
            ctr.zero_()
        for ctr in _prefill_counters.values():
            ctr.zero_()


def decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
           max_blocks_per_seq=None, partition_tokens=0, workspace=None, counters=None,
           stream=None, allocate_in_library=False):
    """Paged-attention decode into `out` [S, H, D] (a CUDA tensor, or pinned
    host memory that the kernel writes directly).

    q [S, H, D]; k_cache / v_cache [N, H, B, D], all float16 or all
    bfloat16; block_tables
    [S, MB] int32; context_lens [S] int32.  partition_tokens = 0 picks the
    library default.  counters (a zeroed int32 CUDA tensor of at least
    decode_counters_bytes(...) bytes) and workspace (a uint8 CUDA tensor of at
    least decode_workspace_bytes(...) bytes) are optional; by default cached
    per-stream buffers are used.  allocate_in_library=True calls pa_decode,
    which allocates both itself with cudaMallocAsync on the stream.
    """
    torch = _torch()
    _element_dtype(k_cache)
    et = k_cache.dtype
    _need(k_cache, "k_cache", et, 4)
    dev = k_cache.device
    _need(v_cache, "v_cache", et, 4, dev)
    _need(q, "q", et, 3, dev)
    _need_out(out, et, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    N, H, B, D = k_cache.shape
    S = q.shape[0]
    if v_cache.shape != k_cache.shape or q.shape != (S, H, D) or out.shape != q.shape \
            or block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("decode: inconsistent shapes")
    MB = block_tables.shape[1] if max_blocks_per_seq is None else int(max_blocks_per_seq)
    if MB != block_tables.shape[1]:
        raise ValueError("max_blocks_per_seq must equal block_tables.shape[1]")
    dims = _cache_dims(k_cache, S)
    sh, st = _stream_handle(dev, stream)
    l = lib()
    with torch.cuda.device(dev):
        if allocate_in_library:
            rc = l.pa_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                             _ptr(context_lens), float(scale), MB, ctypes.byref(dims), sh)
            _check(rc, "pa_decode")
            return out
        need_ws = l.pa_decode_workspace_bytes(ctypes.byref(dims), MB, int(partition_tokens))
        need_ctr = l.pa_decode_counters_bytes(ctypes.byref(dims))
        if need_ws == _SIZE_ERROR or need_ctr == 0:
            raise PaError(-2, "decode: invalid sizes")
        if counters is None or (workspace is None and need_ws):
            c2, w2 = _buffers_for(dev, st, need_ctr, need_ws)
            counters = c2 if counters is None else counters
            workspace = w2 if workspace is None else workspace
        _need(counters, "counters", torch.int32, 1, dev)
        if workspace is not None:
            _need(workspace, "workspace", torch.uint8, 1, dev)
        ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
        ws_n = workspace.numel() if workspace is not None else 0
        rc = l.pa_decode_ws(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            _ptr(context_lens), float(scale), MB, ctypes.byref(dims),
                            int(partition_tokens), ws_ptr, ws_n, _ptr(counters),
                            counters.numel() * 4, sh)
    _check(rc, "pa_decode_ws")
    return out


def decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                         group_start, group_prefix_blocks, max_group_size=None,
                         partition_tokens=0, workspace=None, counters=None, stream=None,
                         allocate_in_library=False):
    """decode() for a batch whose sequences form groups sharing the first
    blocks of their tables (pa_decode_shared_prefix_ws; pa_decode_shared_prefix
    with allocate_in_library).  group_start [G + 1] and group_prefix_blocks [G]
    are int32 CUDA tensors: group g is sequences group_start[g] ..
    group_start[g + 1] - 1, sharing their first group_prefix_blocks[g] table
    entries.  max_group_size bounds the group sizes (computed from
    group_start, with a device sync, when None).  The output equals decode()'s;
    a sequence that does not really share its group's prefix is decoded in
    full and flags DEVERR_PREFIX.  counters / workspace: as decode(), sized by
    the shared-prefix byte counts; by default cached per-stream buffers."""
    torch = _torch()
    _element_dtype(k_cache)
    et = k_cache.dtype
    _need(k_cache, "k_cache", et, 4)
    dev = k_cache.device
    _need(v_cache, "v_cache", et, 4, dev)
    _need(q, "q", et, 3, dev)
    _need_out(out, et, 3, dev)
    _need(block_tables, "block_tables", torch.int32, 2, dev)
    _need(context_lens, "context_lens", torch.int32, 1, dev)
    _need(group_start, "group_start", torch.int32, 1, dev)
    _need(group_prefix_blocks, "group_prefix_blocks", torch.int32, 1, dev)
    N, H, B, D = k_cache.shape
    S = q.shape[0]
    G = group_prefix_blocks.shape[0]
    if v_cache.shape != k_cache.shape or q.shape != (S, H, D) or out.shape != q.shape \
            or block_tables.shape[0] != S or context_lens.shape[0] != S \
            or group_start.shape[0] != G + 1:
        raise ValueError("decode_shared_prefix: inconsistent shapes")
    if max_group_size is None:
        max_group_size = int((group_start[1:] - group_start[:-1]).max()) if G else 0
    MB = block_tables.shape[1]
    dims = _cache_dims(k_cache, S)
    sh, st = _stream_handle(dev, stream)
    l = lib()
    with torch.cuda.device(dev):
        if allocate_in_library:
            rc = l.pa_decode_shared_prefix(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(block_tables), _ptr(context_lens), float(scale),
                                           MB, ctypes.byref(dims), _ptr(group_start),
                                           _ptr(group_prefix_blocks), G, int(max_group_size), sh)
            _check(rc, "pa_decode_shared_prefix")
            return out
        need_ws = l.pa_decode_shared_prefix_workspace_bytes(ctypes.byref(dims), MB,
                                                            int(partition_tokens))
        need_ctr = l.pa_decode_shared_prefix_counters_bytes(ctypes.byref(dims))
        if need_ws == _SIZE_ERROR or need_ctr == 0:
            raise PaError(-2, "decode_shared_prefix: invalid sizes")
        if counters is None or workspace is None:
            c2, w2 = _buffers_for(dev, st, need_ctr, need_ws)
            counters = c2 if counters is None else counters
            workspace = w2 if workspace is None else workspace
        _need(counters, "counters", torch.int32, 1, dev)
        _need(workspace, "workspace", torch.uint8, 1, dev)
        rc = l.pa_decode_shared_prefix_ws(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(block_tables), _ptr(context_lens), float(scale),
                                          MB, ctypes.byref(dims), _ptr(group_start),
                                          _ptr(group_prefix_blocks), G, int(max_group_size),
                                          int(partition_tokens), _ptr(workspace),
                                          workspace.numel(), _ptr(counters),
                                          counters.numel() * 4, sh)
    _check(rc, "pa_decode_shared_prefix_ws")
    return out


class KVManager:
    """Host-side KV block manager (pa_kvm_* in the C ABI): a free list of
    blocks, reference-counted sharing and per-sequence block tables.  Pure
    host code -- usable without a GPU."""

    def __init__(self, num_blocks, block_size=16, max_blocks_per_seq=128, shuffle_seed=0):
        self._l = lib()
        self._h = self._l.pa_kvm_create(num_blocks, block_size, max_blocks_per_seq,
                                        ctypes.c_uint64(shuffle_seed))
        if not self._h:
            raise PaError(-2, "pa_kvm_create: invalid sizes")
        self.num_blocks, self.block_size = num_blocks, block_size
        self.max_blocks_per_seq = max_blocks_per_seq

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._l.pa_kvm_destroy(h)

    @staticmethod
    def _out():
        return ctypes.c_int32(-1)

    def add_sequence(self, num_tokens, parent=-1, shared_blocks=0) -> int:
        sid = self._out()
        _check(self._l.pa_kvm_add_sequence(self._h, num_tokens, parent, shared_blocks,
                                           ctypes.byref(sid)), "pa_kvm_add_sequence")
        return sid.value

    def fork(self, parent) -> int:
        sid = self._out()
        _check(self._l.pa_kvm_fork(self._h, parent, ctypes.byref(sid)), "pa_kvm_fork")
        return sid.value

    def append(self, seq):
        """(slot, copy_src, copy_dst); copy_src = copy_dst = -1 unless the
        token lands in a shared block (copy-on-write)."""
        slot, src, dst = self._out(), self._out(), self._out()
        _check(self._l.pa_kvm_append(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                     ctypes.byref(dst)), "pa_kvm_append")
        return slot.value, src.value, dst.value

    def free(self, seq):
        _check(self._l.pa_kvm_free(self._h, seq), "pa_kvm_free")

    def context_len(self, seq) -> int:
        return self._l.pa_kvm_context_len(self._h, seq)

    def slot(self, seq, token) -> int:
        out = self._out()
        _check(self._l.pa_kvm_slot(self._h, seq, token, ctypes.byref(out)), "pa_kvm_slot")
        return out.value

    def num_free_blocks(self) -> int:
        return self._l.pa_kvm_num_free_blocks(self._h)

    def refcount(self, block) -> int:
        return self._l.pa_kvm_refcount(self._h, block)

    def block_tables(self, seqs, row_len=None):
        """(tables [n, row_len] int32, context_lens [n] int32) for the batch
        rows `seqs` (a negative id gives an empty padding row)."""
        import numpy as np
        row_len = row_len or self.max_blocks_per_seq
        ids = np.ascontiguousarray(seqs, dtype=np.int32)
        tables = np.empty((len(ids), row_len), np.int32)
        lens = np.empty(len(ids), np.int32)
        _check(self._l.pa_kvm_block_tables(self._h, ids.ctypes.data, len(ids),
                                           tables.ctypes.data, row_len, lens.ctypes.data),
               "pa_kvm_block_tables")
        return tables, lens

    def prefix_groups(self, seqs, max_groups=None):
        """(group_start [G + 1] int32, group_prefix_blocks [G] int32) for the
        batch rows `seqs`, as decode_shared_prefix takes them: runs of adjacent
        rows whose tables start with the same full blocks (pa_kvm_prefix_groups)."""
        import numpy as np
        ids = np.ascontiguousarray(seqs, dtype=np.int32)
        cap = len(ids) if max_groups is None else int(max_groups)
        starts = np.empty(cap + 1, np.int32)
        pre = np.empty(max(cap, 1), np.int32)
        g = ctypes.c_int32(0)
        _check(self._l.pa_kvm_prefix_groups(self._h, ids.ctypes.data, len(ids), starts.ctypes.data,
                                            pre.ctypes.data, cap, ctypes.byref(g)),
               "pa_kvm_prefix_groups")
        return starts[:g.value + 1].copy(), pre[:g.value].copy()


def selftest_wait_timeout(stream=None, device=None):
    """Run the bounded-wait self-test (pa_selftest_wait_timeout, about 3 s):
    returns, per wait (mbarrier, shared word, drain), 1 if it wrongly
    succeeded and 0 if it gave up.  PA_DEVERR_TIMEOUT is left in the device
    error word."""
    torch = _torch()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    sh, _ = _stream_handle(device, stream)
    res = (ctypes.c_int32 * 3)()
    with torch.cuda.device(device):
        rc = lib().pa_selftest_wait_timeout(res, sh)
    _check(rc, "pa_selftest_wait_timeout")
    return [int(v) for v in res]


def device_errors(stream=None, device=None) -> int:
    """Synchronise the stream and return-and-clear the device error word."""
    torch = _torch()
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    sh, _ = _stream_handle(device, stream)
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(device):
        rc = lib().pa_device_errors(sh, ctypes.byref(flags))
    _check(rc, "pa_device_errors")
    return int(flags.value)
