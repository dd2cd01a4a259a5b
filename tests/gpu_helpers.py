"""Helpers for the GPU parity tests: upload a case, run it through the C ABI,
compare with the fp64 oracle under the decode tolerance.

Tolerance (fp16 output vs fp64 oracle): max |gpu - oracle| <= 2e-3 over all
elements, and max |gpu - oracle| / |oracle| <= 1e-2 over elements with
|oracle| >= 1e-3 (near-zero outputs are governed by the absolute bound).
"""
from __future__ import annotations

import numpy as np

ABS_TOL = 2e-3
REL_TOL = 1e-2
REL_FLOOR = 1e-3


def upload(case, dev):
    import torch
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
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
    out = torch.full(case.q.shape, float("nan"), dtype=torch.float16, device=dev)
    pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
              case.scale, partition_tokens=partition_tokens, stream=stream,
              allocate_in_library=allocate_in_library)
    flags = pa.device_errors(stream=stream)
    return out.cpu().numpy(), flags, d


def errors(got_f16, ref):
    got = np.asarray(got_f16, dtype=np.float64)
    err = np.abs(got - ref)
    big = np.abs(ref) >= REL_FLOOR
    rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return float(np.nanmax(err)) if err.size else 0.0, rel, int((~big).sum())


def assert_parity(got_f16, ref, what=""):
    got = np.asarray(got_f16, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    abs_err, rel_err, _ = errors(got_f16, ref)
    assert abs_err <= ABS_TOL, f"{what}: max abs err {abs_err:.3g} > {ABS_TOL}"
    assert rel_err <= REL_TOL, f"{what}: max rel err {rel_err:.3g} > {REL_TOL}"
    return abs_err, rel_err
