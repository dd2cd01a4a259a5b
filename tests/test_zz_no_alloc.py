"""pa_decode_static: decode that allocates no device memory.

Callers that cannot let a library call cudaMalloc (a process that reserved
nearly all device memory for its KV pool, a decode loop that must not stall on
the allocator, a plugin that does not own the allocator) use this entry point;
its counters and partial results live in a fixed array inside the library.

The test calls it through the C ABI twice in a row on each case and compares
with the regular entry point (pa_decode_ws through the binding) within the
decode tolerance.  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh
process, where its first call performs the per-device set-up.
"""
import ctypes

import numpy as np
import pytest

import workloads
from gpu_helpers import assert_parity, upload

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_269_gb300 as pa
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    pa.lib()
    pa.device_errors()
    return d


def _static_call(case, d, out, stream):
    import paged_kv_cache_269_gb300 as pa
    dims = pa.Dims(case.num_seqs, case.num_heads, case.head_dim, case.block_size, case.num_blocks)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return pa.lib().pa_decode_static(p(out), p(d["q"]), p(d["k_cache"]), p(d["v_cache"]),
                                     p(d["block_tables"]), p(d["context_lens"]),
                                     ctypes.c_float(case.scale), case.max_blocks_per_seq,
                                     ctypes.byref(dims), ctypes.c_void_p(stream.cuda_stream))


def _check_against_regular(case, dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    d = upload(case, dev)
    stream = torch.cuda.current_stream(dev)
    ref = torch.empty(case.q.shape, dtype=torch.float16, device=dev)
    pa.decode(ref, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
              case.scale)
    assert pa.device_errors() == 0
    ref_np = ref.cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full(case.q.shape, float("nan"), dtype=torch.float16, device=dev)
        rc = _static_call(case, d, out, stream)
        assert rc == 0, pa.lib().pa_status_string(rc)
        assert pa.device_errors() == 0
        assert_parity(out.cpu().numpy(), ref_np, f"{case.name}: static call {call + 1}")


def test_split_case_matches_regular_entry_point(dev):
    rng = np.random.default_rng(29)
    case = workloads.build_case("static_split", rng.integers(1, 3000, size=16), num_heads=8,
                                head_dim=128, seed=29)
    _check_against_regular(case, dev)


def test_partition_grows_to_fit_the_array(dev):
    # 64 x 32 pairs with 512-block table rows: the default 512-token
    # partition's partial results (16 partitions, about 17 MB) do not fit the
    # 16 MiB array, so a longer partition is used; four long contexts still
    # need several partitions each.
    import paged_kv_cache_269_gb300 as pa
    rng = np.random.default_rng(31)
    lens = np.concatenate([rng.integers(1, 600, size=60), np.full(4, 4096)])
    case = workloads.build_case("static_grow", lens, num_heads=32, head_dim=128, seed=31,
                                max_blocks_per_seq=512)
    default_partials = pa.decode_workspace_bytes(64, 32, 128, 16, case.num_blocks, 512)
    assert default_partials > STATIC_SCRATCH_BYTES
    _check_against_regular(case, dev)


def test_rejects_sizes_beyond_the_array(dev):
    import paged_kv_cache_269_gb300 as pa
    # 70000 x 64 (sequence, head) tickets need more than 16 MiB of counters
    dims = pa.Dims(70000, 64, 128, 16, 1024)
    rc = pa.lib().pa_decode_static(None, None, None, None, None, None, ctypes.c_float(0.1), 8,
                                   ctypes.byref(dims), None)
    assert rc == -5  # PA_ERR_WORKSPACE, nothing launched
