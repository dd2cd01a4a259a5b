"""Helpers for the GPU parity tests: upload a case, run it through the C ABI,
compare with the fp64 oracle under the decode tolerance.

Tolerance, fp16 outputs (the stated decode tolerance): max |gpu - oracle|
<= 2e-3 over all elements, and max |gpu - oracle| / |oracle| <= 1e-2 over
elements with |oracle| >= 1e-3 (near-zero outputs are governed by the absolute
bound).

Tolerance, bf16 outputs (derived; the stated one is for fp16): bf16 keeps 8
significant bits, so rounding the fp32 result to nearest even moves it by at
most 2^-8 |o|; fp32 accumulation adds well under 1e-5 at these sizes.  Each
element must satisfy |gpu - oracle| <= 2^-8 |oracle| + 1e-5.
"""
from __future__ import annotations

import numpy as np

ABS_TOL = 2e-3
REL_TOL = 1e-2
REL_FLOOR = 1e-3
BF16_REL = 2.0 ** -8
BF16_ABS = 1e-5


def bf16_bits_to_float64(bits):
    return (np.ascontiguousarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def torch_dtype(case):
    import torch
    return torch.bfloat16 if case.dtype == "bf16" else torch.float16


def to_numpy(t, case):
    """Device tensor -> numpy in the case's storage convention."""
    import torch
    if case.dtype == "bf16":
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


def as_float64(arr, dtype="f16"):
    return bf16_bits_to_float64(arr) if dtype == "bf16" else np.asarray(arr, dtype=np.float64)


def upload(case, dev):
    import torch

    def t(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:  # bf16 bit patterns
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    d = dict(q=t(case.q), k_cache=t(case.k_cache), v_cache=t(case.v_cache),
             block_tables=t(case.block_tables), context_lens=t(case.context_lens))
    if case.slot_mapping is not None:
        d.update(k_new=t(case.k_new), v_new=t(case.v_new), slot_mapping=t(case.slot_mapping))
    return d


def run_gpu(case, dev, partition_tokens=0, tensors=None, reshape=True, stream=None,
            allocate_in_library=False):
    """reshape_and_cache (if the case has new tokens) then decode; returns the
    fp16 output as numpy, the device error flags and the device tensors."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    d = tensors or upload(case, dev)
    if reshape and case.slot_mapping is not None and case.num_new_tokens:
        pa.reshape_and_cache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                             d["slot_mapping"], stream=stream)
    out = torch.full(case.q.shape, float("nan"), dtype=torch_dtype(case), device=dev)
    pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
              case.scale, partition_tokens=partition_tokens, stream=stream,
              allocate_in_library=allocate_in_library)
    flags = pa.device_errors(stream=stream)
    return to_numpy(out, case), flags, d


def errors(got_f16, ref):
    got = np.asarray(got_f16, dtype=np.float64)
    err = np.abs(got - ref)
    big = np.abs(ref) >= REL_FLOOR
    rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return float(np.nanmax(err)) if err.size else 0.0, rel, int((~big).sum())


def assert_parity(got, ref, what="", dtype="f16"):
    """got: the GPU output in storage form (fp16 values, or bf16 bits when
    dtype == "bf16"); ref: the fp64 oracle."""
    g = as_float64(got, dtype)
    assert g.shape == ref.shape
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    if dtype == "bf16":
        err = np.abs(g - ref)
        bound = BF16_REL * np.abs(ref) + BF16_ABS
        worst = float((err / bound).max()) if err.size else 0.0
        assert worst <= 1.0, f"{what}: bf16 error {worst:.3g} x the bound"
        return float(err.max()) if err.size else 0.0, worst
    abs_err, rel_err, _ = errors(g, ref)
    assert abs_err <= ABS_TOL, f"{what}: max abs err {abs_err:.3g} > {ABS_TOL}"
    assert rel_err <= REL_TOL, f"{what}: max rel err {rel_err:.3g} > {REL_TOL}"
    return abs_err, rel_err
