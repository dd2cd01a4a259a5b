"""GPU parity of pa_copy_blocks: copy-on-write inside the cache, swap-out to
pinned host memory and swap-in back to the device, all bit-exact against the
oracle, and decode unchanged (bit for bit) after the blocks move."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import run_gpu, to_numpy, upload

pytestmark = pytest.mark.gpu


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


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint16)


def _pairs(rows, dev):
    import torch
    return torch.tensor(np.asarray(rows, np.int32).reshape(-1, 2), dtype=torch.int32, device=dev)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_copy_on_write_then_decode(dev, dtype):
    import paged_kv_cache_269_gb300 as pa
    case = workloads.build_case("cow", [600, 570, 530, 700], num_heads=4, head_dim=128, seed=5,
                                shared_prefix_blocks=32, spare_frac=2.0, dtype=dtype)
    before, f0, d = run_gpu(case, dev)
    assert f0 == 0
    used = set(case.block_tables[case.block_tables >= 0].tolist())
    free = [b for b in range(case.num_blocks) if b not in used]
    rows, tables = [], case.block_tables.copy()
    for s in (1, 3):                       # two sequences take private prefix copies
        for b in range(32):
            dst = free.pop()
            rows.append((int(case.block_tables[s, b]), dst))
            tables[s, b] = dst
    pa.copy_blocks(d["k_cache"], d["v_cache"], d["k_cache"], d["v_cache"], _pairs(rows, dev))
    assert pa.device_errors() == 0
    ref_k, ref_v = oracle.copy_blocks(case.k_cache, case.v_cache, case.k_cache, case.v_cache,
                                      np.asarray(rows, np.int32))
    assert np.array_equal(_bits(to_numpy(d["k_cache"], case)), _bits(ref_k))
    assert np.array_equal(_bits(to_numpy(d["v_cache"], case)), _bits(ref_v))
    case.block_tables = tables
    import torch
    d["block_tables"] = torch.from_numpy(tables).to(dev)
    after, f1, _ = run_gpu(case, dev, tensors=d)
    assert f1 == 0
    assert np.array_equal(after.view(np.uint16), before.view(np.uint16))


def test_swap_out_and_in(dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    case = workloads.build_case("swap", [700, 300, 1024, 45, 1], num_heads=8, head_dim=128,
                                seed=9, spare_frac=1.0)
    before, f0, d = run_gpu(case, dev)
    ids = np.array(sorted(set(case.block_tables[case.block_tables >= 0].tolist())), np.int32)
    n = len(ids)
    host_k = torch.zeros((n,) + tuple(case.k_cache.shape[1:]), dtype=torch.float16).pin_memory()
    host_v = torch.zeros_like(host_k).pin_memory()
    out_rows = np.stack([ids, np.arange(n, dtype=np.int32)], 1)
    pa.copy_blocks(d["k_cache"], d["v_cache"], host_k, host_v, _pairs(out_rows, dev))
    assert pa.device_errors() == 0          # synchronises the stream
    ref_hk, ref_hv = oracle.copy_blocks(case.k_cache, case.v_cache, np.zeros_like(host_k.numpy()),
                                        np.zeros_like(host_v.numpy()), out_rows)
    assert np.array_equal(_bits(host_k.numpy()), _bits(ref_hk))
    assert np.array_equal(_bits(host_v.numpy()), _bits(ref_hv))
    # swap back in at shuffled places of a fresh device pool
    perm = np.random.default_rng(2).permutation(case.num_blocks)[:n].astype(np.int32)
    in_rows = np.stack([np.arange(n, dtype=np.int32), perm], 1)
    new_k = torch.full_like(d["k_cache"], float("nan"))
    new_v = torch.full_like(d["v_cache"], float("nan"))
    pa.copy_blocks(host_k, host_v, new_k, new_v, _pairs(in_rows, dev))
    assert pa.device_errors() == 0
    remap = dict(zip(ids.tolist(), perm.tolist()))
    tables = np.vectorize(lambda b: remap.get(int(b), -1))(case.block_tables).astype(np.int32)
    d2 = dict(d, k_cache=new_k, v_cache=new_v, block_tables=torch.from_numpy(tables).to(dev))
    after, f1, _ = run_gpu(case, dev, tensors=d2)
    assert f1 == 0
    assert np.array_equal(after.view(np.uint16), before.view(np.uint16))


def test_many_blocks_device_copy(dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    N, H, B, D = 4096, 32, 16, 128
    g = torch.Generator(device=dev).manual_seed(3)
    kc = torch.randn((N, H, B, D), generator=g, device=dev).half()
    vc = torch.randn((N, H, B, D), generator=g, device=dev).half()
    src = torch.randperm(N, device=dev, generator=g)[:2048]
    dst = torch.randperm(N, device=dev, generator=g)[:2048]
    # destinations must not be sources: copy into a second pool
    dk, dv = torch.zeros_like(kc), torch.zeros_like(vc)
    pairs = torch.stack([src, dst], 1).to(torch.int32).contiguous()
    pa.copy_blocks(kc, vc, dk, dv, pairs)
    assert pa.device_errors() == 0
    assert torch.equal(dk[dst], kc[src]) and torch.equal(dv[dst], vc[src])
    untouched = torch.ones(N, dtype=torch.bool, device=dev)
    untouched[dst] = False
    assert int(dk[untouched].abs().sum()) == 0


def test_bad_block_id_is_reported(dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    kc = torch.randn((8, 2, 16, 64), device=dev).half()
    vc = torch.randn_like(kc)
    dk, dv = torch.zeros_like(kc), torch.zeros_like(vc)
    pa.copy_blocks(kc, vc, dk, dv, _pairs([(1, 2), (9, 3), (4, -1)], dev))
    assert pa.device_errors() & pa.DEVERR_TABLE
    assert torch.equal(dk[2], kc[1]) and int(dk[3].abs().sum()) == 0


def test_unpinned_host_memory_is_rejected_or_addressable(dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    kc = torch.randn((4, 2, 16, 64), device=dev).half()
    host = torch.zeros((4, 2, 16, 64), dtype=torch.float16)       # pageable
    with pytest.raises(ValueError):                                # the binding refuses it
        pa.copy_blocks(kc, kc, host, host, _pairs([(0, 1)], dev))
