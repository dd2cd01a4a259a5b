"""GPU parity of pa_prefill (tcgen05 tensor cores) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_parity, to_numpy, torch_dtype, upload

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


def run_prefill(case, dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    d = upload(case, dev)
    qs = torch.from_numpy(case.query_start).to(dev)
    out = torch.full(case.q.shape, float("nan"), dtype=torch_dtype(case), device=dev)
    pa.prefill(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], qs,
               case.scale)
    return to_numpy(out, case), pa.device_errors()


CTX = [1, 15, 16, 17, 64, 65, 127, 128, 129, 300, 513]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("mode", ["whole", "chunk", "single"])
def test_ragged_prefill(dev, dtype, mode):
    ctx = np.array(CTX)
    if mode == "whole":
        ql = ctx                                   # the whole prompt
    elif mode == "chunk":
        ql = np.minimum(ctx, [1, 7, 16, 5, 64, 1, 100, 128, 129, 200, 257])
    else:
        ql = np.ones_like(ctx)                     # one query each (decode-like)
    case = workloads.build_prefill_case(f"pf_{mode}", ctx, ql, num_heads=2, head_dim=128,
                                        seed=40 + len(mode), dtype=dtype)
    got, flags = run_prefill(case, dev)
    assert flags == 0
    ref = oracle.prefill(case.q, case.k_cache, case.v_cache, case.block_tables,
                         case.context_lens, case.query_start, case.scale, dtype=dtype)
    assert_parity(got, ref, f"prefill {mode} {dtype}", dtype=dtype)


def test_many_short_prompts(dev):
    # Hundreds of items of one or two key tiles in a row: the loader then
    # fills a whole item's V tiles while the P V threads are still on the
    # previous item, which must not let the per-item V barrier run ahead of
    # them.  Repeated launches on the same counters.
    rng = np.random.default_rng(44)
    ctx = rng.integers(1, 129, size=96)
    ql = np.minimum(ctx, rng.integers(1, 129, size=96))
    case = workloads.build_prefill_case("pf_short", ctx, ql, num_heads=8, head_dim=128, seed=44)
    ref = oracle.prefill(case.q, case.k_cache, case.v_cache, case.block_tables,
                         case.context_lens, case.query_start, case.scale)
    for rep in range(3):
        got, flags = run_prefill(case, dev)
        assert flags == 0
        assert_parity(got, ref, f"short prompts, launch {rep + 1}")


@pytest.mark.parametrize("kind", workloads.PREFILL_WORKLOADS)
def test_prefill_workloads_full_size(dev, kind):
    case = workloads.make_prefill_workload(kind)
    got, flags = run_prefill(case, dev)
    assert flags == 0
    ref = oracle.prefill(case.q, case.k_cache, case.v_cache, case.block_tables,
                         case.context_lens, case.query_start, case.scale)
    assert_parity(got, ref, kind)


def test_prefill_llama7b_bf16_full_size(dev):
    case = workloads.make_prefill_workload("prefill_llama7b", dtype="bf16")
    got, flags = run_prefill(case, dev)
    assert flags == 0
    ref = oracle.prefill(case.q, case.k_cache, case.v_cache, case.block_tables,
                         case.context_lens, case.query_start, case.scale, dtype="bf16")
    assert_parity(got, ref, "prefill_llama7b bf16", dtype="bf16")


def test_prefill_bad_query_count_is_reported(dev):
    import paged_kv_cache_269_gb300 as pa
    case = workloads.build_prefill_case("pf_bad", [40, 40], [40, 40], num_heads=2, head_dim=128,
                                        seed=3)
    lens = case.context_lens.copy()
    lens[1] = 20                                   # fewer tokens than queries
    case.context_lens = lens
    got, flags = run_prefill(case, dev)
    assert flags & pa.DEVERR_CONTEXT
    ref = oracle.prefill(case.q[:40], case.k_cache, case.v_cache, case.block_tables[:1],
                         case.context_lens[:1], case.query_start[:2], case.scale)
    assert_parity(got[:40], ref, "the valid sequence is still computed")


def _set_rising_scores(case, slope, q0):
    """Scores that grow with the key's position: K[t, 0] = slope * t and
    q[:, 0] = q0, so each row's running maximum rises tile after tile and the
    kernel must rescale its accumulated output several times."""
    bf16 = case.dtype == "bf16"
    enc = (lambda v: workloads.f32_to_bf16_bits(np.asarray(v, np.float32))) if bf16 else \
        (lambda v: np.asarray(v, np.float16))
    B = case.k_cache.shape[2]
    for s, ctx in enumerate(case.context_lens):
        for t in range(int(ctx)):
            case.k_cache[case.block_tables[s, t // B], :, t % B, 0] = enc(slope * t)
    case.q[:, :, 0] = enc(q0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_rising_maximum(dev, dtype):
    ctx = np.array([513, 300, 129, 1000])
    case = workloads.build_prefill_case("pf_rising", ctx, np.minimum(ctx, [513, 300, 129, 600]),
                                        num_heads=2, head_dim=128, seed=47, dtype=dtype)
    _set_rising_scores(case, 0.2, 4.0)
    got, flags = run_prefill(case, dev)
    assert flags == 0
    ref = oracle.prefill(case.q, case.k_cache, case.v_cache, case.block_tables,
                         case.context_lens, case.query_start, case.scale, dtype=dtype)
    assert_parity(got, ref, f"prefill rising {dtype}", dtype=dtype)


def test_prefill_counters_reused_and_left_zero(dev):
    """One work-queue counter buffer across calls of different shapes: each
    result matches the oracle and the kernel leaves the counters at zero."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    ctr = torch.zeros(2, dtype=torch.int32, device=dev)
    shapes = [([700, 33, 256], [700, 20, 256]), ([1, 2, 3], [1, 2, 3]), ([513, 1000], [300, 1000])]
    for i, (ctx, ql) in enumerate(shapes):
        case = workloads.build_prefill_case(f"pf_ctr{i}", np.array(ctx), np.array(ql), num_heads=3,
                                            head_dim=128, seed=60 + i)
        d = upload(case, dev)
        qs = torch.from_numpy(case.query_start).to(dev)
        out = torch.full(case.q.shape, float("nan"), dtype=torch.float16, device=dev)
        pa.prefill(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                   qs, case.scale, counters=ctr)
        torch.cuda.synchronize(dev)
        assert pa.device_errors() == 0
        assert ctr.cpu().tolist() == [0, 0]
        ref = oracle.prefill(case.q, case.k_cache, case.v_cache, case.block_tables,
                             case.context_lens, case.query_start, case.scale)
        assert_parity(to_numpy(out, case), ref, f"prefill counters call {i}")


def test_prefill_library_allocated_counters(dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    case = workloads.build_prefill_case("pf_lib", np.array([300, 129]), np.array([300, 64]),
                                        num_heads=2, head_dim=128, seed=70)
    d = upload(case, dev)
    qs = torch.from_numpy(case.query_start).to(dev)
    out = torch.full(case.q.shape, float("nan"), dtype=torch.float16, device=dev)
    pa.prefill(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], qs,
               case.scale, allocate_in_library=True)
    assert pa.device_errors() == 0
    ref = oracle.prefill(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                         case.query_start, case.scale)
    assert_parity(to_numpy(out, case), ref, "prefill, library-allocated counters")


def test_prefill_bad_table_entry_is_reported(dev):
    """A block-table entry outside the pool is skipped (never read) and
    flagged; a clean call afterwards is exact."""
    import paged_kv_cache_269_gb300 as pa
    case = workloads.build_prefill_case("pf_badtab", [200, 90], [200, 90], num_heads=2,
                                        head_dim=128, seed=80)
    tables = case.block_tables.copy()
    tables[0, 3] = case.num_blocks + 7
    case.block_tables = tables
    _, flags = run_prefill(case, dev)
    assert flags & pa.DEVERR_TABLE
    ok = workloads.build_prefill_case("pf_ok", [200, 90], [200, 90], num_heads=2, head_dim=128,
                                      seed=81)
    got, flags = run_prefill(ok, dev)
    assert flags == 0
    ref = oracle.prefill(ok.q, ok.k_cache, ok.v_cache, ok.block_tables, ok.context_lens,
                         ok.query_start, ok.scale)
    assert_parity(got, ref, "prefill after a reported error")


def test_prefill_understated_max_query_len_is_reported(dev):
    """Rows past max_query_len (rounded up to 256) cannot be computed: the
    call flags it; the rows below are still exact."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    case = workloads.build_prefill_case("pf_maxq", [600, 100], [600, 100], num_heads=2,
                                        head_dim=128, seed=90)
    d = upload(case, dev)
    qs = torch.from_numpy(case.query_start).to(dev)
    out = torch.full(case.q.shape, float("nan"), dtype=torch.float16, device=dev)
    pa.prefill(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"], qs,
               case.scale, max_query_len=200)          # pairs of 256 rows: only one
    assert pa.device_errors() & pa.DEVERR_CONTEXT
    got = to_numpy(out, case)
    ref = oracle.prefill(case.q, case.k_cache, case.v_cache, case.block_tables, case.context_lens,
                         case.query_start, case.scale)
    rows = np.r_[0:256, 600:700]                     # pair 0 of both sequences
    assert_parity(got[rows], ref[rows], "rows inside the stated bound")
