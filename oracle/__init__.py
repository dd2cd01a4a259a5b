"""CPU fp64 oracle for paged-attention decode and reshape_and_cache.

TEST INFRASTRUCTURE.  Only tests/, the smoke check in __graft_entry__ and the
benchmark's cpu_baseline / reference leg may import this package.  The product
library never loads it and there is no CPU fallback built on it.

The arithmetic lives in pa_oracle.c (plain C, fp64, OpenMP over (sequence,
head) pairs); this module compiles it with the host C compiler and marshals
numpy arrays through ctypes.  See pa_oracle.c for what each function computes
and which passage of the pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {
    -1: "bad argument",
    -2: "context length out of range",
    -3: "block table entry out of range",
    -4: "slot out of range",
    -5: "out of host memory",
}


class OracleError(RuntimeError):
    pass


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle into a shared library (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [os.environ.get("CC", "gcc"), "-O2", "-std=c11", "-fPIC", "-shared",
           "-fopenmp", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str = _LIB_PATH, src: str = _SRC):
    """Load (building first if needed) an oracle library and declare its ABI."""
    build(src=src, out=path)
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    ci = ctypes.c_int
    lib.oracle_decode.argtypes = [dp, u16p, u16p, u16p, i32p, i32p, ctypes.c_double,
                                  ci, ci, ci, ci, ci, ci, ci]
    lib.oracle_decode.restype = ci
    lib.oracle_reshape_and_cache.argtypes = [u16p, u16p, u16p, u16p, i32p,
                                             ci, ci, ci, ci, ci]
    lib.oracle_reshape_and_cache.restype = ci
    lib.oracle_prefill.argtypes = [dp, u16p, u16p, u16p, i32p, i32p, i32p, ctypes.c_double,
                                   ci, ci, ci, ci, ci, ci, ci]
    lib.oracle_prefill.restype = ci
    lib.oracle_copy_blocks.argtypes = [u16p, u16p, ci, u16p, u16p, ci, i32p, ci, ci, ci, ci]
    lib.oracle_copy_blocks.restype = ci
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ci
    return lib


def _get():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load()
        return _lib


def _u16(a: np.ndarray):
    a = np.ascontiguousarray(a)
    assert a.dtype in (np.float16, np.uint16), a.dtype
    return a.view(np.uint16), a.view(np.uint16).ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _i32(a: np.ndarray):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def num_threads(lib=None) -> int:
    return (lib or _get()).oracle_num_threads()


def half_to_double(bits: int, lib=None) -> float:
    return (lib or _get()).oracle_half_to_double(int(bits))


DTYPES = {"f16": 0, "bf16": 1}


def bf16_to_double(bits: int, lib=None) -> float:
    return (lib or _get()).oracle_bf16_to_double(int(bits))


def decode(q, k_cache, v_cache, block_tables, context_lens, scale,
           lib=None, dtype: str = "f16") -> np.ndarray:
    """fp64 attention output [S, H, D] for q [S, H, D] over a paged cache
    [N, H, B, D] reached through block_tables [S, MB] and context_lens [S].
    dtype "f16": arrays are float16; "bf16": uint16 arrays of bfloat16 bits."""
    lib = lib or _get()
    S, H, D = q.shape
    N, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or v_cache.shape != k_cache.shape:
        raise OracleError("shape mismatch")
    MB = block_tables.shape[1] if block_tables.ndim == 2 else 1
    out = np.zeros((S, H, D), dtype=np.float64)
    keep = [_u16(q), _u16(k_cache), _u16(v_cache), _i32(block_tables), _i32(context_lens)]
    rc = lib.oracle_decode(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                           keep[0][1], keep[1][1], keep[2][1], keep[3][1], keep[4][1],
                           float(scale), S, H, D, B, N, max(1, MB), DTYPES[dtype])
    if rc != 0:
        raise OracleError(ERRORS.get(rc, str(rc)))
    return out


def reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, lib=None):
    """Return updated copies of (k_cache, v_cache) with each new token's K/V
    stored at its slot."""
    lib = lib or _get()
    T, H, D = k.shape
    N, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise OracleError("shape mismatch")
    kc = np.array(k_cache, copy=True, order="C")
    vc = np.array(v_cache, copy=True, order="C")
    kk, vv, ss = _u16(k), _u16(v), _i32(slot_mapping)
    kcu, vcu = _u16(kc), _u16(vc)
    rc = lib.oracle_reshape_and_cache(kk[1], vv[1], kcu[1], vcu[1], ss[1], T, H, D, B, N)
    if rc != 0:
        raise OracleError(ERRORS.get(rc, str(rc)))
    return kc, vc


def reshape_and_cache_into(k, v, k_cache, v_cache, slot_mapping, lib=None):
    """Store each new token's K/V at its slot in the given caches, in place
    (C-contiguous arrays of the 16-bit element type).  Same C routine as
    reshape_and_cache, without the copies: for timing the oracle."""
    lib = lib or _get()
    T, H, D = k.shape
    N, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise OracleError("shape mismatch")
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise OracleError("caches must be C-contiguous")
    kk, vv, ss = _u16(k), _u16(v), _i32(slot_mapping)
    kcu, vcu = _u16(k_cache), _u16(v_cache)
    rc = lib.oracle_reshape_and_cache(kk[1], vv[1], kcu[1], vcu[1], ss[1], T, H, D, B, N)
    if rc != 0:
        raise OracleError(ERRORS.get(rc, str(rc)))


def prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
            lib=None, dtype: str = "f16") -> np.ndarray:
    """fp64 causal attention output [total_q, H, D]: sequence s's queries are
    rows query_start[s] .. query_start[s+1]-1 of q, the last tokens of its
    context, each attending to keys 0 .. its own position."""
    lib = lib or _get()
    T, H, D = q.shape
    N, H2, B, D2 = k_cache.shape
    if (H2, D2) != (H, D) or v_cache.shape != k_cache.shape:
        raise OracleError("shape mismatch")
    S = int(np.asarray(context_lens).shape[0])
    MB = block_tables.shape[1]
    out = np.zeros((T, H, D), dtype=np.float64)
    keep = [_u16(q), _u16(k_cache), _u16(v_cache), _i32(block_tables), _i32(context_lens),
            _i32(query_start)]
    rc = lib.oracle_prefill(out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                            keep[0][1], keep[1][1], keep[2][1], keep[3][1], keep[4][1], keep[5][1],
                            float(scale), S, H, D, B, N, max(1, MB), DTYPES[dtype])
    if rc != 0:
        raise OracleError(ERRORS.get(rc, str(rc)))
    return out


def copy_blocks(src_k, src_v, dst_k, dst_v, block_pairs, lib=None):
    """Return updated copies of (dst_k, dst_v) with K/V of block src copied to
    block dst for every row (src, dst) of block_pairs [n, 2]."""
    lib = lib or _get()
    Ns, H, B, D = src_k.shape
    Nd = dst_k.shape[0]
    if src_v.shape != src_k.shape or dst_v.shape != dst_k.shape or dst_k.shape[1:] != (H, B, D):
        raise OracleError("shape mismatch")
    dk = np.array(dst_k, copy=True, order="C")
    dv = np.array(dst_v, copy=True, order="C")
    sk, sv, pp = _u16(src_k), _u16(src_v), _i32(np.asarray(block_pairs).reshape(-1, 2))
    dku, dvu = _u16(dk), _u16(dv)
    rc = lib.oracle_copy_blocks(sk[1], sv[1], Ns, dku[1], dvu[1], Nd, pp[1], pp[0].shape[0], H, D, B)
    if rc != 0:
        raise OracleError(ERRORS.get(rc, str(rc)))
    return dk, dv


def decode_case(case, lib=None) -> np.ndarray:
    """Oracle output for a workloads.DecodeCase (after its new tokens, if any,
    have been stored with reshape_and_cache)."""
    kc, vc = case.k_cache, case.v_cache
    if case.slot_mapping is not None and case.num_new_tokens:
        kc, vc = reshape_and_cache(case.k_new, case.v_new, kc, vc, case.slot_mapping, lib=lib)
    return decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale, lib=lib,
                  dtype=case.dtype)
