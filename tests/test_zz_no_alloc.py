"""pa_decode_static: decode that allocates no device memory.

Some callers cannot let a library call cudaMalloc: a serving process that
reserved nearly all device memory for its KV-block pool at start-up, a decode
loop that must never stall on the allocator, or a plugin inside a host
program that does not own the allocator.  They use this entry point; its
counters and partial results live in a fixed array inside the library.

Each case calls the entry point through the C ABI three times and checks
every output element by element against the fp64 oracle, within the decode
tolerance, and against the regular entry point (pa_decode through the
binding).  The first case makes its static calls before any regular decode
in this module, so that, run alone in a fresh process, its first call
performs the per-device set-up.  Around the second and third calls, made in
a row, the test checks through the CUDA driver that neither the device's
default stream-ordered memory pool nor the device's free memory moved:
nothing was allocated.

This file sorts last, so a run that stops at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_parity, upload

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 16 << 20
CU_MEMPOOL_ATTR_USED_MEM_CURRENT = 7
CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_269_gb300 as pa
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    torch.zeros(1, device=d)          # the primary context is current on this thread
    pa.lib()
    return d


class DeviceMemory:
    """Allocation evidence from the CUDA driver: the default memory pool's
    used bytes (current and high-water mark, which stream-ordered
    allocations move) and the device's free bytes (which cudaMalloc moves)."""

    def __init__(self, ordinal):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), ordinal) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def _pool_attr(self, attr):
        v = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset_high_water(self):
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH,
                                             ctypes.byref(zero)) == 0

    def snapshot(self):
        free, total = ctypes.c_size_t(), ctypes.c_size_t()
        assert self.cu.cuMemGetInfo_v2(ctypes.byref(free), ctypes.byref(total)) == 0
        return (self._pool_attr(CU_MEMPOOL_ATTR_USED_MEM_CURRENT),
                self._pool_attr(CU_MEMPOOL_ATTR_USED_MEM_HIGH), free.value)


def _static_call(case, d, out, stream):
    import paged_kv_cache_269_gb300 as pa
    dims = pa.Dims(case.num_seqs, case.num_heads, case.head_dim, case.block_size, case.num_blocks)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return pa.lib().pa_decode_static(p(out), p(d["q"]), p(d["k_cache"]), p(d["v_cache"]),
                                     p(d["block_tables"]), p(d["context_lens"]),
                                     ctypes.c_float(case.scale), case.max_blocks_per_seq,
                                     ctypes.byref(dims), ctypes.c_void_p(stream.cuda_stream))


def _check(case, dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    d = upload(case, dev)
    stream = torch.cuda.current_stream(dev)
    want = oracle.decode_case(case)
    outs = [torch.full(case.q.shape, float("nan"), dtype=torch.float16, device=dev)
            for _ in range(3)]
    torch.cuda.synchronize(dev)
    # Call 1 may be the process's first on this device: it looks up the
    # array's address, and the CUDA runtime may load the library's device
    # code and its static array then (module loading, not an allocation the
    # library makes).  Calls 2 and 3, in a row, are watched for allocations.
    rc = _static_call(case, d, outs[0], stream)
    assert rc == 0, pa.lib().pa_status_string(rc)
    torch.cuda.synchronize(dev)
    mem = DeviceMemory(dev.index)
    mem.reset_high_water()
    before = mem.snapshot()
    for out in outs[1:]:
        rc = _static_call(case, d, out, stream)
        assert rc == 0, pa.lib().pa_status_string(rc)
    torch.cuda.synchronize(dev)
    after = mem.snapshot()
    assert after[0] == before[0] and after[1] <= before[0], "the default memory pool was used"
    assert after[2] == before[2], "device free memory changed across the static calls"
    assert pa.device_errors() == 0
    for i, out in enumerate(outs):
        assert_parity(out.cpu().numpy(), want, f"{case.name}: static call {i + 1} vs oracle")

    ref = torch.empty(case.q.shape, dtype=torch.float16, device=dev)
    pa.decode(ref, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
              case.scale)
    assert pa.device_errors() == 0
    ref_np = ref.cpu().numpy().astype(np.float64)
    for i, out in enumerate(outs):
        assert_parity(out.cpu().numpy(), ref_np, f"{case.name}: static call {i + 1} vs pa_decode")


def test_split_case_matches_oracle_and_regular_entry_point(dev):
    rng = np.random.default_rng(29)
    case = workloads.build_case("static_split", rng.integers(1, 3000, size=16), num_heads=8,
                                head_dim=128, seed=29)
    _check(case, dev)


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
    _check(case, dev)


def test_rejects_sizes_beyond_the_array(dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    # 70000 x 64 (sequence, head) tickets need more than 16 MiB of counters;
    # the call returns before it touches any of these buffers
    buf = torch.zeros(64, dtype=torch.float16, device=dev)
    p = ctypes.c_void_p(buf.data_ptr())
    dims = pa.Dims(70000, 64, 128, 16, 1024)
    rc = pa.lib().pa_decode_static(p, p, p, p, p, p, ctypes.c_float(0.1), 8, ctypes.byref(dims),
                                   None)
    assert rc == -5  # PA_ERR_WORKSPACE, nothing launched
