"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every test here runs libpa's sm_103a kernels on cuda:0 and compares element by
element with the oracle on the same seeded inputs.  reshape_and_cache must be
bit-exact; decode must meet the tolerance in gpu_helpers.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_parity, run_gpu, upload

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


def _ragged(name, lens, H=4, D=128, B=16, seed=7, **kw):
    return workloads.build_case(name, lens, num_heads=H, head_dim=D, block_size=B, seed=seed,
                                **kw)


# ----------------------------------------------------------------------------
# small cases: several tiles, ragged tails, every partition regime
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("partition_tokens", [0, 16, 32, 48, 256, 4096])
def test_tiny_workload(dev, partition_tokens):
    case = workloads.make_workload("tiny", new_tokens=True)
    got, flags, _ = run_gpu(case, dev, partition_tokens)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), f"tiny P={partition_tokens}")


EDGE_LENS = [0, 1, 2, 15, 16, 17, 31, 255, 256, 257, 511, 512, 513, 1000, 4096]


@pytest.mark.parametrize("partition_tokens", [0, 16, 240, 272, 1 << 16])
def test_edge_lengths(dev, partition_tokens):
    case = _ragged("edges", EDGE_LENS, H=3)
    got, flags, _ = run_gpu(case, dev, partition_tokens)
    assert flags == 0
    ref = oracle.decode_case(case)
    assert_parity(got, ref, f"edges P={partition_tokens}")
    assert (got[0] == 0).all(), "an empty context must give a zero row"
    # a one-token context returns that token's V row exactly (weight 1.0)
    phys = case.block_tables[1, 0]
    assert np.array_equal(got[1].view(np.uint16), case.v_cache[phys, :, 0, :].view(np.uint16))


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_head_dim_block_size_variants(dev, D, B):
    case = _ragged(f"v{D}_{B}", [1, 7, B - 1, B, B + 1, 100, 333, 700], H=2, D=D, B=B,
                   seed=D + B)
    ref = oracle.decode_case(case)
    for P in (0, 2 * B, 5 * B):
        got, flags, _ = run_gpu(case, dev, P)
        assert flags == 0
        assert_parity(got, ref, f"D={D} B={B} P={P}")


@pytest.mark.parametrize("D,B", [(64, 8), (64, 16), (128, 8), (64, 32), (256, 8)])
@pytest.mark.parametrize("H", [4, 6, 12])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_head_group_units(dev, D, B, H, dtype):
    # Small tiles are read several heads per unit (4 heads for 1 KiB tiles, 2
    # for 2 KiB and for the 4 KiB tiles of D 64 x B 32 and D 256 x B 8): one
    # bulk copy moves the adjacent tiles of a block's heads, and each consumer
    # warp keeps one head of the group.  6 heads are not a multiple of 4 (one
    # head per unit instead); 4 and 12 divide every group size.
    case = _ragged(f"hg{D}_{B}_{H}", [1, 2, B - 1, B, B + 1, 100, 333, 700, 1500], H=H, D=D,
                   B=B, seed=D + B + H, dtype=dtype)
    ref = oracle.decode_case(case)
    for P in (0, 2 * B, 5 * B):
        got, flags, _ = run_gpu(case, dev, P)
        assert flags == 0
        assert_parity(got, ref, f"{dtype} D={D} B={B} H={H} P={P}", dtype=dtype)


@pytest.mark.parametrize("D,B", [(64, 8), (64, 16)])
def test_head_group_units_full_size(dev, D, B):
    # the variant batch the bench times: 64 sequences, contexts U[128, 2048],
    # H x D = 4096 (64 heads of 64)
    rng = np.random.default_rng(11)
    case = workloads.build_case(f"v{D}_{B}", rng.integers(128, 2049, size=64), num_heads=64,
                                head_dim=D, block_size=B, seed=31)
    got, flags, _ = run_gpu(case, dev)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), f"D={D} B={B} 64 heads")


def _shape_scores(case, profile, rng):
    """Rewrite every context token's K row so that its score against its
    sequence's query follows `profile`: K_t = c_t * q + small noise, whose
    score is about c_t |q|^2 * scale.  The oracle sees the same (rounded)
    rows.  rising: over the last 8 tiles each tile's scores exceed the
    previous maximum by about 12 (log2), past the lazy reference's margin of
    8, so every such tile raises it; spike: one late token dwarfs the rest;
    falling:
    the first tile holds the maximum; saw: tiles alternate high and low."""
    from gpu_helpers import as_float64
    k = as_float64(case.k_cache, case.dtype).astype(np.float32)
    q = as_float64(case.q, case.dtype).astype(np.float32)
    B = case.block_size
    for s, ctx in enumerate(case.context_lens):
        ctx = int(ctx)
        if ctx == 0:
            continue
        t = np.arange(ctx)
        if profile == "rising":
            # over the last 8 tiles, each tile about 12 (log2) above the one
            # before: |q|^2 ~ D, so a score is about c sqrt(D) log2(e)
            r = 12.0 / (B * np.sqrt(case.head_dim) * np.log2(np.e))
            c = np.maximum(0, t - (ctx - 8 * B)) * r
        elif profile == "spike":
            c = np.full(ctx, 0.05)
            c[int(rng.integers(ctx // 2, ctx))] = 3.0
        elif profile == "falling":
            c = 2.0 * (1.0 - t / ctx)
        else:  # saw
            c = np.where((t // B) % 2 == 0, 1.5, -0.5)
        for h in range(case.num_heads):
            rows = c[:, None] * q[s, h][None, :] + 0.05 * rng.standard_normal(
                (ctx, case.head_dim), dtype=np.float32)
            blocks = case.block_tables[s, t // B]
            k[blocks, h, t % B, :] = rows
    if case.dtype == "bf16":
        case.k_cache[...] = workloads.f32_to_bf16_bits(k)
    else:
        case.k_cache[...] = k.astype(np.float16)


@pytest.mark.parametrize("profile", ["rising", "spike", "falling", "saw"])
@pytest.mark.parametrize("D,B", [(64, 8), (64, 16), (128, 16), (256, 32)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_softmax_reference_profiles(dev, profile, D, B, dtype):
    """Score profiles that drive the lazily raised softmax reference through
    every path: a raise on every tile, one late raise, none after the first
    tile, and alternating tiles; whole contexts and split ones (partials with
    different references, combined)."""
    rng = np.random.default_rng(41)
    H = 4 if D == 64 else 2
    case = _ragged(f"prof_{profile}", [1, 9, 40, 300, 700, 1500], H=H, D=D, B=B, seed=43,
                   dtype=dtype)
    _shape_scores(case, profile, rng)
    ref = oracle.decode_case(case)
    for P in (0, 4 * B):
        got, flags, _ = run_gpu(case, dev, P)
        assert flags == 0
        assert_parity(got, ref, f"{profile} D={D} B={B} {dtype} P={P}", dtype=dtype)


def test_split_matches_single_pass(dev):
    rng = np.random.default_rng(17)
    case = _ragged("split", rng.integers(1, 3000, size=24), H=8)
    ref = oracle.decode_case(case)
    single, f1, d = run_gpu(case, dev, 1 << 20)
    split, f2, _ = run_gpu(case, dev, 128, tensors=d)
    assert f1 == 0 and f2 == 0
    assert_parity(single, ref, "single pass")
    assert_parity(split, ref, "split")
    assert_parity(split, single.astype(np.float64), "split vs single pass")


def test_deterministic_and_stream(dev):
    import torch
    case = workloads.make_workload("tiny")
    a, _, d = run_gpu(case, dev, 32)
    b, _, _ = run_gpu(case, dev, 32, tensors=d)
    s = torch.cuda.Stream(dev)
    c, flags, _ = run_gpu(case, dev, 32, tensors=d, stream=s)
    assert flags == 0
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    assert np.array_equal(a.view(np.uint16), c.view(np.uint16))


def test_library_allocated_workspace(dev):
    case = _ragged("alloc", [3, 300, 1500, 77], H=4)
    a, f1, d = run_gpu(case, dev)
    b, f2, _ = run_gpu(case, dev, tensors=d, allocate_in_library=True)
    assert f1 == 0 and f2 == 0
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_counters_return_to_zero_across_shapes(dev):
    """One counter buffer serves calls of different sizes: every call leaves
    it all zero, and partial results never land in it."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    cases = [_ragged("ws1", [1000, 2000, 5, 333], H=4, seed=1),
             _ragged("ws2", [3000, 17, 900, 1, 64, 2500, 700, 1200], H=8, seed=2),
             _ragged("ws3", [100, 2000], H=2, seed=3)]
    ctr = torch.zeros(1 << 14, dtype=torch.int32, device=dev)
    ws = torch.full((1 << 24,), 0x7F, dtype=torch.uint8, device=dev)   # garbage scratch
    for rep in range(2):
        for case in cases:
            d = upload(case, dev)
            out = torch.empty(case.q.shape, dtype=torch.float16, device=dev)
            pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                      d["context_lens"], case.scale, partition_tokens=64, workspace=ws,
                      counters=ctr)
            assert pa.device_errors() == 0
            assert int(ctr.abs().sum()) == 0
            assert_parity(out.cpu().numpy(), oracle.decode_case(case), f"{case.name} rep {rep}")


def test_many_sequences(dev):
    rng = np.random.default_rng(3)
    case = _ragged("many", rng.integers(0, 40, size=3000), H=2, D=64)
    got, flags, _ = run_gpu(case, dev)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), "3000 sequences")


@pytest.mark.parametrize("n,maxlen,partition_tokens", [(60000, 30, 16), (200000, 20, 0)])
def test_very_large_batches(dev, n, maxlen, partition_tokens):
    # Far more sequences than fit one shared-memory entry each: the CTAs keep
    # one partition count per chunk of 64 (60000) or of 256 and more (200000)
    # sequences, so each lane of the producer warp resolves several
    # sequences; 16-token partitions give most sequences several partitions.
    rng = np.random.default_rng(5)
    case = _ragged(f"huge{n}", rng.integers(0, maxlen, size=n), H=1, D=64)
    got, flags, _ = run_gpu(case, dev, partition_tokens)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), f"{n} sequences, P={partition_tokens}")


def test_empty_batch(dev):
    import torch
    import paged_kv_cache_269_gb300 as pa
    z = torch.zeros((0, 2, 64), dtype=torch.float16, device=dev)
    kc = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device=dev)
    pa.decode(z, z, kc, kc, torch.zeros((0, 3), dtype=torch.int32, device=dev),
              torch.zeros((0,), dtype=torch.int32, device=dev), 0.125)
    assert pa.device_errors() == 0


# ----------------------------------------------------------------------------
# reshape_and_cache: bit-exact
# ----------------------------------------------------------------------------

def test_reshape_and_cache_bit_exact(dev):
    import paged_kv_cache_269_gb300 as pa
    case = _ragged("rc", [5, 16, 17, 200, 1], H=4, new_tokens=True)
    slots = case.slot_mapping.copy()
    slots[1] = -1                                      # skipped
    slots[2] = 0                                       # first slot of the pool
    slots[3] = case.num_blocks * case.block_size - 1   # last slot of the pool
    case.slot_mapping = slots
    d = upload(case, dev)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    assert pa.device_errors() == 0
    ref_k, ref_v = oracle.reshape_and_cache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                            slots)
    assert np.array_equal(d["k_cache"].cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(d["v_cache"].cpu().numpy().view(np.uint16), ref_v.view(np.uint16))


# ----------------------------------------------------------------------------
# device-side range checks: reported, never a fault
# ----------------------------------------------------------------------------

def test_bad_table_entry_is_reported(dev):
    import paged_kv_cache_269_gb300 as pa
    case = _ragged("badtab", [40, 40], H=2)
    tables = case.block_tables.copy()
    tables[0, 1] = case.num_blocks + 5
    case.block_tables = tables
    got, flags, _ = run_gpu(case, dev)
    assert flags & pa.DEVERR_TABLE
    pa.reset_workspaces()
    ok = _ragged("ok", [40, 40], H=2)
    got2, flags2, _ = run_gpu(ok, dev)
    assert flags2 == 0
    assert_parity(got2, oracle.decode_case(ok), "after a reported error")


def test_bad_context_len_is_reported(dev):
    import paged_kv_cache_269_gb300 as pa
    case = _ragged("badctx", [40, 20], H=2)
    lens = case.context_lens.copy()
    lens[1] = case.max_blocks_per_seq * case.block_size + 100
    case.context_lens = lens
    _, flags, _ = run_gpu(case, dev)
    assert flags & pa.DEVERR_CONTEXT
    pa.reset_workspaces()


def test_bad_slot_is_reported(dev):
    import paged_kv_cache_269_gb300 as pa
    case = _ragged("badslot", [5, 9], H=2, new_tokens=True)
    d = upload(case, dev)
    before = d["k_cache"].cpu().numpy().copy()
    import torch
    bad = torch.tensor([case.num_blocks * case.block_size, -3], dtype=torch.int32, device=dev)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], bad)
    assert pa.device_errors() & pa.DEVERR_SLOT
    assert np.array_equal(d["k_cache"].cpu().numpy().view(np.uint16), before.view(np.uint16))


# ----------------------------------------------------------------------------
# the five workloads at full size, in the launch configuration the bench uses
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["tiny", "llama7b_b64", "cb_mix", "shared_prefix", "long_ctx",
                                  "cb_mix_1k", "cb_mix_4k"])
def test_workload_full_size(dev, kind):
    case = workloads.make_workload(kind)
    got, flags, d = run_gpu(case, dev)
    assert flags == 0
    if kind == "shared_prefix":
        dup = workloads.duplicate_prefix(case)
        ref = oracle.decode_case(dup)          # the duplicated-prefix oracle
        got_dup, flags2, _ = run_gpu(dup, dev)
        assert flags2 == 0
        # same arithmetic in the same order: bit-identical on the GPU too
        assert np.array_equal(got.view(np.uint16), got_dup.view(np.uint16))
    else:
        ref = oracle.decode_case(case)
    assert_parity(got, ref, kind)
    if case.num_new_tokens:
        # reshape_and_cache at full size: both caches bit-exact
        ref_k, ref_v = oracle.reshape_and_cache(case.k_new, case.v_new, case.k_cache,
                                                case.v_cache, case.slot_mapping)
        assert np.array_equal(d["k_cache"].cpu().numpy().view(np.uint16), ref_k.view(np.uint16))
        assert np.array_equal(d["v_cache"].cpu().numpy().view(np.uint16), ref_v.view(np.uint16))


def test_back_to_back_steps_keep_their_order(dev):
    """Steps issued without any host synchronisation (reshape_and_cache then
    decode, repeated; both kernels use programmatic dependent launch) must
    each see their own step's new tokens: the new K/V alternate between two
    sets and every step's output is checked against the oracle for its set."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    base = _ragged("b2b", [300, 17, 1024, 640, 1, 2000], H=4, new_tokens=True, seed=11)
    alt = _ragged("b2b", [300, 17, 1024, 640, 1, 2000], H=4, new_tokens=True, seed=11)
    workloads.fill_normal_f16(alt.k_new, 99, 4)
    workloads.fill_normal_f16(alt.v_new, 99, 5)
    refs = [oracle.decode_case(base), oracle.decode_case(alt)]
    d = upload(base, dev)
    news = [(d["k_new"], d["v_new"]), (upload(alt, dev)["k_new"], upload(alt, dev)["v_new"])]
    outs = [torch.empty(base.q.shape, dtype=torch.float16, device=dev) for _ in range(12)]
    for i, out in enumerate(outs):
        kn, vn = news[i % 2]
        pa.reshape_and_cache(kn, vn, d["k_cache"], d["v_cache"], d["slot_mapping"])
        pa.decode(out, d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                  base.scale, partition_tokens=256)
    assert pa.device_errors() == 0
    for i, out in enumerate(outs):
        assert_parity(out.cpu().numpy(), refs[i % 2], f"step {i}")


# ----------------------------------------------------------------------------
# bfloat16 caches (bf16 tolerance derived in gpu_helpers)
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("partition_tokens", [0, 16, 272, 1 << 16])
def test_bf16_edge_lengths(dev, partition_tokens):
    case = _ragged("edges_bf16", EDGE_LENS, H=3, dtype="bf16")
    got, flags, _ = run_gpu(case, dev, partition_tokens)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), f"bf16 edges P={partition_tokens}", dtype="bf16")
    assert (got[0] == 0).all(), "an empty context must give a zero row"
    phys = case.block_tables[1, 0]
    assert np.array_equal(got[1], case.v_cache[phys, :, 0, :]), "ctx 1 must return V exactly"


def test_bf16_head_dim_block_size_variants(dev):
    for D in (64, 128, 256):
        for B in (8, 16, 32):
            case = _ragged(f"bf{D}_{B}", [1, B - 1, B + 1, 333, 700], H=2, D=D, B=B,
                           seed=3 * D + B, dtype="bf16")
            ref = oracle.decode_case(case)
            for P in (0, 2 * B):
                got, flags, _ = run_gpu(case, dev, P)
                assert flags == 0
                assert_parity(got, ref, f"bf16 D={D} B={B} P={P}", dtype="bf16")


def test_bf16_reshape_and_cache_bit_exact(dev):
    import paged_kv_cache_269_gb300 as pa
    from gpu_helpers import to_numpy
    case = _ragged("rc_bf16", [5, 16, 17, 200], H=4, new_tokens=True, dtype="bf16")
    d = upload(case, dev)
    pa.reshape_and_cache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slot_mapping"])
    assert pa.device_errors() == 0
    ref_k, ref_v = oracle.reshape_and_cache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                            case.slot_mapping)
    assert np.array_equal(to_numpy(d["k_cache"], case), ref_k)
    assert np.array_equal(to_numpy(d["v_cache"], case), ref_v)


def test_bf16_llama7b_full_size(dev):
    case = workloads.make_workload("llama7b_b64", dtype="bf16")
    got, flags, _ = run_gpu(case, dev)
    assert flags == 0
    assert_parity(got, oracle.decode_case(case), "bf16 llama7b_b64", dtype="bf16")


def test_concurrent_streams_do_not_interfere(dev):
    """Decodes issued on two streams at once (each with its own cached counter
    buffer and workspace, as the binding keeps them per stream) both match the
    oracle; so does a shared-prefix decode running beside a plain one."""
    import torch
    import paged_kv_cache_269_gb300 as pa
    a = _ragged("streamA", [300, 2000, 17, 1024, 640], H=4, seed=21)
    rng = np.random.default_rng(22)
    b, gs, gp = workloads.build_grouped_case(
        "streamB", [(6, [int(c) for c in rng.integers(100, 900, 40)]), (0, [50, 700])],
        num_heads=4, head_dim=128, seed=22)
    da, db = upload(a, dev), upload(b, dev)
    ref_a, ref_b = oracle.decode_case(a), oracle.decode_case(b)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    g_start, g_pre = torch.from_numpy(gs).to(dev), torch.from_numpy(gp).to(dev)
    torch.cuda.synchronize(dev)
    outs = []
    for i in range(6):
        oa = torch.empty(a.q.shape, dtype=torch.float16, device=dev)
        ob = torch.empty(b.q.shape, dtype=torch.float16, device=dev)
        oc = torch.empty(b.q.shape, dtype=torch.float16, device=dev)
        pa.decode(oa, da["q"], da["k_cache"], da["v_cache"], da["block_tables"],
                  da["context_lens"], a.scale, partition_tokens=256, stream=s1)
        pa.decode_shared_prefix(ob, db["q"], db["k_cache"], db["v_cache"], db["block_tables"],
                                db["context_lens"], b.scale, g_start, g_pre, max_group_size=40,
                                stream=s2)
        pa.decode(oc, db["q"], db["k_cache"], db["v_cache"], db["block_tables"],
                  db["context_lens"], b.scale, stream=s1)
        outs.append((oa, ob, oc))
    torch.cuda.synchronize(dev)
    assert pa.device_errors() == 0
    for i, (oa, ob, oc) in enumerate(outs):
        assert_parity(oa.cpu().numpy(), ref_a, f"stream 1, call {i}")
        assert_parity(ob.cpu().numpy(), ref_b, f"stream 2 (shared prefix), call {i}")
        assert_parity(oc.cpu().numpy(), ref_b, f"stream 1 (plain), call {i}")
