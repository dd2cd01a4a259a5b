"""GPU parity of the shared-prefix decode (pa_decode_shared_prefix_ws).

The call must give pa_decode's output -- the fp64 oracle's, within the decode
tolerance -- for every batch: groups of every size (one row, several 128-row
tiles, several tile pairs), prefixes that end inside a 64-key tile, members
whose suffix is empty or spans several partitions, sequences in no group, and
every kind of misuse (a member whose table does not share the prefix, a
context shorter than the prefix, an understated max_group_size, malformed
group arrays), which must be decoded in full and flagged with DEVERR_PREFIX.
"""
import ctypes

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
    pa.device_errors()  # start from a clear error word
    return d


def _buffers(dev, case, partition_tokens=0):
    import torch
    import paged_kv_cache_269_gb300 as pa
    l = pa.lib()
    dims = pa.Dims(case.num_seqs, case.num_heads, case.head_dim, case.block_size,
                   case.num_blocks, 1 if case.dtype == "bf16" else 0)
    ws = l.pa_decode_shared_prefix_workspace_bytes(ctypes.byref(dims), case.max_blocks_per_seq,
                                                   partition_tokens)
    ctr = l.pa_decode_shared_prefix_counters_bytes(ctypes.byref(dims))
    return (torch.zeros(ctr // 4, dtype=torch.int32, device=dev),
            torch.empty(ws, dtype=torch.uint8, device=dev))


def run_shared(case, gs, gp, dev, partition_tokens=0, max_group_size=None, counters=None,
               workspace=None, tensors=None, allocate_in_library=False):
    import torch
    import paged_kv_cache_269_gb300 as pa
    d = tensors or upload(case, dev)
    g_start = torch.from_numpy(np.ascontiguousarray(gs, dtype=np.int32)).to(dev)
    g_pre = torch.from_numpy(np.ascontiguousarray(gp, dtype=np.int32)).to(dev)
    out = torch.full(case.q.shape, float("nan"), dtype=torch_dtype(case), device=dev)
    pa.decode_shared_prefix(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                            d["context_lens"], case.scale, g_start, g_pre,
                            max_group_size=max_group_size, partition_tokens=partition_tokens,
                            counters=counters, workspace=workspace,
                            allocate_in_library=allocate_in_library)
    flags = pa.device_errors()
    return to_numpy(out, case), flags


# a batch with every shape the two kernels must agree on
def _layout(rng):
    return [
        (5, [80, 81, 700]),                              # prefix ends inside a key tile; empty suffix
        (0, [33, 1000]),                                 # in no group
        (8, [int(c) for c in rng.integers(128, 600, 130)]),   # 130 rows: two 128-row tiles
        (1, [20]),                                       # a group of one
        (40, [int(c) for c in rng.integers(641, 1400, 300)]),  # two tile pairs; long suffixes
        (3, [48, 49, 63, 64, 65]),                       # suffixes of 0, 1, 15, 16, 17 tokens
    ]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("partition_tokens", [0, 256])
def test_ragged_groups(dev, dtype, partition_tokens):
    rng = np.random.default_rng(21)
    case, gs, gp = workloads.build_grouped_case("groups", _layout(rng), num_heads=2,
                                                head_dim=128, seed=21, dtype=dtype)
    ctr, ws = _buffers(dev, case, partition_tokens)
    got, flags = run_shared(case, gs, gp, dev, partition_tokens, counters=ctr, workspace=ws)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), f"groups {dtype} P={partition_tokens}",
                  dtype=dtype)
    assert int(ctr.count_nonzero()) == 0        # the counters are left zeroed


@pytest.mark.parametrize("partition_tokens", [0, 256])
def test_work_order_over_several_chunks(dev, partition_tokens):
    """140 sequences (four full 32-sequence chunks and a ragged one) in the
    per-sequence layout: the longest-first work order is built by several
    warps, one chunk each, and must come out the same in every CTA."""
    rng = np.random.default_rng(23)
    layout = [(4, [int(c) for c in rng.integers(70, 900, 50)]), (0, [30, 700]),
              (6, [int(c) for c in rng.integers(97, 620, 60)]),
              (2, [int(c) for c in rng.integers(33, 1200, 28)])]
    case, gs, gp = workloads.build_grouped_case("order", layout, num_heads=4, head_dim=128,
                                                seed=23)
    ctr, ws = _buffers(dev, case, partition_tokens)
    for _ in range(2):
        got, flags = run_shared(case, gs, gp, dev, partition_tokens, counters=ctr, workspace=ws)
        assert flags == 0
        assert_parity(got, oracle.decode_case(case), f"order P={partition_tokens}")
        assert int(ctr.count_nonzero()) == 0


def test_shared_prefix_workload_full_size(dev):
    """The 128-sequence, 512-token-prompt batch, in the launch configuration the
    benchmark times: one group of 128 sharing 32 blocks."""
    case = workloads.make_workload("shared_prefix")
    gs = np.array([0, case.num_seqs], dtype=np.int32)
    gp = np.array([case.shared_prefix_blocks], dtype=np.int32)
    got, flags = run_shared(case, gs, gp, dev)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), "shared_prefix (shared reads)")


def test_matches_plain_decode_and_library_allocation(dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    rng = np.random.default_rng(5)
    case, gs, gp = workloads.build_grouped_case("alloc", _layout(rng)[:4], num_heads=4,
                                                head_dim=128, seed=5)
    d = upload(case, dev)
    got, flags = run_shared(case, gs, gp, dev, tensors=d, allocate_in_library=True)
    assert flags == 0
    ref = oracle.decode_case(case)
    assert_parity(got, ref, "library-allocated buffers")
    plain = torch.empty(case.q.shape, dtype=torch.float16, device=dev)
    pa.decode(plain, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
              case.scale)
    assert_parity(plain.cpu().numpy(), ref, "plain decode")
    # two correct answers: they differ by rounding only
    diff = np.abs(got.astype(np.float64) - plain.cpu().numpy().astype(np.float64))
    assert float(diff.max()) <= 2e-3


def test_with_new_tokens_after_reshape(dev):
    """reshape_and_cache, then the two shared-prefix launches, back to back on one
    stream: each sequence's new token (in its private suffix) must be seen."""
    import paged_kv_cache_269_gb300 as pa
    rng = np.random.default_rng(9)
    layout = [(4, [int(c) for c in rng.integers(70, 400, 40)]), (0, [17, 300]),
              (12, [int(c) for c in rng.integers(200, 900, 20)])]
    case, gs, gp = workloads.build_grouped_case("step", layout, num_heads=4, head_dim=128,
                                                seed=9, new_tokens=True)
    d = upload(case, dev)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    got, flags = run_shared(case, gs, gp, dev, tensors=d)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), "after reshape_and_cache")


def test_counters_serve_calls_of_any_size(dev):
    """One zeroed counter buffer and workspace, sized for the largest batch,
    serve a sequence of calls of different sizes (each leaves them zeroed)."""
    rng = np.random.default_rng(13)
    big, gs_b, gp_b = workloads.build_grouped_case("big", _layout(rng), num_heads=2,
                                                   head_dim=128, seed=13)
    small, gs_s, gp_s = workloads.build_grouped_case("small", [(2, [40, 50]), (0, [7])],
                                                     num_heads=2, head_dim=128, seed=14,
                                                     max_blocks_per_seq=big.max_blocks_per_seq)
    ctr, ws = _buffers(dev, big, 256)
    for case, gs, gp in ((big, gs_b, gp_b), (small, gs_s, gp_s), (big, gs_b, gp_b)):
        got, flags = run_shared(case, gs, gp, dev, 256, counters=ctr, workspace=ws)
        assert flags == 0
        assert_parity(got, oracle.decode_case(case), case.name)
        assert int(ctr.count_nonzero()) == 0


# ----------------------------------------------------------------------------
# misuse: always pa_decode's output, plus the DEVERR_PREFIX flag
# ----------------------------------------------------------------------------

def _misuse_case():
    rng = np.random.default_rng(17)
    return workloads.build_grouped_case(
        "misuse", [(6, [int(c) for c in rng.integers(100, 500, 12)]), (0, [60]),
                   (3, [int(c) for c in rng.integers(50, 300, 300)])],
        num_heads=2, head_dim=128, seed=17)


def _expect_full_decode(dev, case, gs, gp, what, **kw):
    import paged_kv_cache_269_gb300 as pa
    ctr, ws = _buffers(dev, case)
    got, flags = run_shared(case, gs, gp, dev, counters=ctr, workspace=ws, **kw)
    assert flags & pa.DEVERR_PREFIX, what
    assert (flags & ~pa.DEVERR_PREFIX) == 0, what
    assert_parity(got, oracle.decode_case(case), what)
    assert int(ctr.count_nonzero()) == 0, what


def test_member_with_a_different_prefix_block(dev):
    case, gs, gp = _misuse_case()
    # member 3 of the first group points its block 2 at another block of the pool
    spare = int(case.block_tables[20, 0])
    case.block_tables[3, 2] = spare
    workloads.poison_unused(case)
    _expect_full_decode(dev, case, gs, gp, "foreign prefix block")


def test_member_shorter_than_the_prefix(dev):
    case, gs, gp = _misuse_case()
    case.context_lens[5] = 6 * case.block_size - 3       # inside the group's prefix
    workloads.poison_unused(case)
    _expect_full_decode(dev, case, gs, gp, "context shorter than the prefix")


def test_understated_max_group_size(dev):
    case, gs, gp = _misuse_case()
    # the 300-row group needs two tile pairs; one is planned: rows 256.. decode in full
    _expect_full_decode(dev, case, gs, gp, "max_group_size understated", max_group_size=100)


@pytest.mark.parametrize("bad", ["decreasing", "past_batch", "prefix_too_long"])
def test_malformed_group_arrays(dev, bad):
    case, gs, gp = _misuse_case()
    gs, gp = gs.copy(), gp.copy()
    if bad == "decreasing":
        gs[1], gs[2] = gs[2], gs[1]
    elif bad == "past_batch":
        gs[-1] = case.num_seqs + 5
    else:
        gp[0] = case.max_blocks_per_seq + 1
    _expect_full_decode(dev, case, gs, gp, bad, max_group_size=int(np.abs(np.diff(gs)).max()))


def test_no_groups_is_plain_decode_bit_for_bit(dev):
    """With no group (or max_group_size 0) the call is pa_decode itself."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    rng = np.random.default_rng(3)
    case, gs, gp = workloads.build_grouped_case("nogroups", _layout(rng)[:3], num_heads=2,
                                                head_dim=128, seed=3)
    d = upload(case, dev)
    plain = torch.empty(case.q.shape, dtype=torch.float16, device=dev)
    pa.decode(plain, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
              case.scale, partition_tokens=256)
    for g_start, g_pre, mgs in ((np.zeros(1, np.int32), np.zeros(0, np.int32), 0), (gs, gp, 0)):
        out = torch.full_like(plain, float("nan"))
        pa.decode_shared_prefix(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"], case.scale, torch.from_numpy(g_start).to(dev),
                                torch.from_numpy(g_pre).to(dev), max_group_size=mgs,
                                partition_tokens=256)
        assert pa.device_errors() == 0
        assert torch.equal(out.view(torch.int16), plain.view(torch.int16))


def test_output_in_pinned_host_memory(dev):
    """out may be pinned host memory: the decode kernel writes the rows there
    directly; the result equals the device-memory output bit for bit."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    rng = np.random.default_rng(4)
    case, gs, gp = workloads.build_grouped_case("hostout", _layout(rng)[:4], num_heads=2,
                                                head_dim=128, seed=4)
    d = upload(case, dev)
    g_start, g_pre = torch.from_numpy(gs).to(dev), torch.from_numpy(gp).to(dev)
    on_dev = torch.empty(case.q.shape, dtype=torch.float16, device=dev)
    on_host = torch.full(case.q.shape, float("nan"), dtype=torch.float16).pin_memory()
    for out in (on_dev, on_host):
        pa.decode_shared_prefix(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"], case.scale, g_start, g_pre)
    plain_host = torch.full(case.q.shape, float("nan"), dtype=torch.float16).pin_memory()
    pa.decode(plain_host, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
              d["context_lens"], case.scale)
    torch.cuda.synchronize(dev)
    assert pa.device_errors() == 0
    assert torch.equal(on_host.view(torch.int16), on_dev.cpu().view(torch.int16))
    assert_parity(on_host.numpy(), oracle.decode_case(case), "shared prefix, host output")
    assert_parity(plain_host.numpy(), oracle.decode_case(case), "plain decode, host output")
    with pytest.raises(ValueError):        # pageable host memory is refused
        pa.decode(torch.empty(case.q.shape, dtype=torch.float16), d["q"], d["k_cache"],
                  d["v_cache"], d["block_tables"], d["context_lens"], case.scale)


@pytest.mark.parametrize("n_groups,members,partition_tokens", [(6, 700, 0), (400, 8, 64)])
def test_serving_size_batches(dev, n_groups, members, partition_tokens):
    # Thousands of sequences: each CTA keeps the group arrays and one
    # partition count per chunk of sequences instead of per-sequence state,
    # and derives a sequence's prefix coverage from its group when it needs
    # it.  Some groups share nothing; 64-token partitions split suffixes.
    rng = np.random.default_rng(71 + n_groups)
    layout = []
    for _ in range(n_groups):
        P = int(rng.integers(0, 6))
        layout.append((P, [int(c) for c in P * 16 + rng.integers(0, 300, members)]))
    case, gs, gp = workloads.build_grouped_case(f"sp_big{n_groups}", layout, num_heads=2,
                                                head_dim=128, seed=71 + n_groups)
    got, flags = run_shared(case, gs, gp, dev, partition_tokens=partition_tokens)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), f"{n_groups} groups x {members}")


def test_one_group_of_4096(dev):
    # one 512-token prompt shared by 4096 requests
    rng = np.random.default_rng(73)
    layout = [(32, [int(c) for c in 512 + rng.integers(0, 200, 4096)])]
    case, gs, gp = workloads.build_grouped_case("sp_4096", layout, num_heads=2, head_dim=128,
                                                seed=73)
    got, flags = run_shared(case, gs, gp, dev)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), "one group of 4096")


def test_shared_prefix_4k_full_size(dev):
    # the shared_prefix_4k workload (4096 sequences x 8 heads, one 512-token
    # prompt) through the shared-prefix call, as the bench times it
    case = workloads.make_workload("shared_prefix_4k")
    S = case.num_seqs
    gs = np.array([0, S], dtype=np.int32)
    gp = np.array([case.shared_prefix_blocks], dtype=np.int32)
    got, flags = run_shared(case, gs, gp, dev, max_group_size=S)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), "shared_prefix_4k")
