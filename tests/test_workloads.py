"""Invariants of the seeded input generator (CPU only)."""
import numpy as np
import pytest

import workloads


@pytest.mark.parametrize("kind", workloads.WORKLOADS)
def test_tables_are_valid(kind):
    case = workloads.make_workload(kind, values=False)
    B = case.block_size
    lens = case.context_lens
    nb = case.blocks_used()
    assert (nb <= case.max_blocks_per_seq).all()
    used = []
    for s in range(case.num_seqs):
        row = case.block_tables[s]
        assert (row[:nb[s]] >= 0).all() and (row[:nb[s]] < case.num_blocks).all()
        assert (row[nb[s]:] == -1).all()
        used.extend(row[case.shared_prefix_blocks:nb[s]].tolist())
    # private blocks are never shared; the prefix is common to every sequence
    assert len(used) == len(set(used))
    if case.shared_prefix_blocks:
        pref = case.block_tables[:, :case.shared_prefix_blocks]
        assert (pref == pref[0]).all()
        assert not set(pref[0].tolist()) & set(used)


def test_workload_recipes():
    t = workloads.make_workload("tiny", values=False)
    assert t.num_blocks == 64 and t.head_dim == 64 and t.num_heads == 4
    assert ((t.context_lens >= 1) & (t.context_lens <= 100)).all()
    l7 = workloads.make_workload("llama7b_b64", values=False)
    assert l7.num_seqs == 64 and l7.num_heads == 32 and l7.head_dim == 128
    assert ((l7.context_lens >= 128) & (l7.context_lens <= 2048)).all()
    assert l7.num_new_tokens == 64
    cb = workloads.make_workload("cb_mix", values=False)
    assert ((cb.context_lens >= 17) & (cb.context_lens <= 512 + 1000)).all()
    sp = workloads.make_workload("shared_prefix", values=False)
    assert sp.shared_prefix_blocks == 32
    assert ((sp.context_lens >= 512 + 16) & (sp.context_lens <= 1024)).all()
    lc = workloads.make_workload("long_ctx", values=False)
    assert (lc.context_lens == 32768).all() and lc.max_blocks_per_seq == 2048
    assert lc.num_blocks >= 16384
    # a 32768-token fp16 K+V sequence of 32 heads x 128 is 2 GiB / 8 seqs ... 4.3 GB total
    assert workloads.decode_algorithmic_bytes(lc) > 4.29e9


def test_new_token_slots_are_last_positions():
    case = workloads.make_workload("tiny", new_tokens=True)
    B = case.block_size
    for s, slot in enumerate(case.slot_mapping):
        pos = int(case.context_lens[s]) - 1
        assert slot == case.block_tables[s, pos // B] * B + pos % B


def test_values_are_seeded_and_poisoned():
    a = workloads.make_workload("tiny")
    b = workloads.make_workload("tiny")
    assert np.array_equal(a.k_cache.view(np.uint16), b.k_cache.view(np.uint16))
    c = workloads.make_workload("tiny", seed=99)
    assert not np.array_equal(np.nan_to_num(a.q), np.nan_to_num(c.q))
    # covered slots are finite, all others NaN
    B = a.block_size
    covered = np.zeros((a.num_blocks, B), bool)
    for s in range(a.num_seqs):
        for t in range(int(a.context_lens[s])):
            covered[a.block_tables[s, t // B], t % B] = True
    assert np.isfinite(a.k_cache[covered[:, None, :].repeat(a.num_heads, 1)]).all()
    assert np.isnan(a.v_cache.transpose(0, 2, 1, 3)[~covered]).all()
    # roughly N(0, 1)
    vals = a.q.astype(np.float64).ravel()
    assert abs(vals.mean()) < 0.1 and abs(vals.std() - 1) < 0.1


def test_fill_is_thread_count_independent(monkeypatch):
    x = np.empty(workloads._CHUNK * 3 + 5, np.float16)
    y = np.empty_like(x)
    workloads.fill_normal_f16(x, 7, 1)
    monkeypatch.setattr(workloads, "_threads", lambda: 1)
    workloads.fill_normal_f16(y, 7, 1)
    assert np.array_equal(x.view(np.uint16), y.view(np.uint16))


def test_out_of_blocks():
    rng = np.random.default_rng(0)
    with pytest.raises(workloads.OutOfBlocks):
        workloads.allocate_tables(np.array([40, 40]), 16, 5, 4, rng)


def test_grouped_case_tables():
    layout = [(5, [80, 81, 700]), (0, [33, 1000]), (2, [20, 40]), (1, [16])]
    case, gs, gp = workloads.build_grouped_case("g", layout, num_heads=2, head_dim=64, seed=3)
    assert gs.tolist() == [0, 3, 5, 7, 8] and gp.tolist() == [5, 0, 2, 1]
    nb = case.blocks_used()
    private, prefixes = [], []
    for g, (P, _) in enumerate(layout):
        rows = case.block_tables[gs[g]:gs[g + 1]]
        if P:
            assert (rows[:, :P] == rows[0, :P]).all()      # every member starts with the prefix
            prefixes.extend(rows[0, :P].tolist())
        for i, s in enumerate(range(gs[g], gs[g + 1])):
            row = case.block_tables[s]
            assert (row[:nb[s]] >= 0).all() and (row[:nb[s]] < case.num_blocks).all()
            assert (row[nb[s]:] == -1).all()
            private.extend(row[P:nb[s]].tolist())
    # every block is either one group's prefix or one sequence's own
    assert len(private + prefixes) == len(set(private + prefixes))
    # blocks no table references hold NaN; referenced ones hold values
    spare = sorted(set(range(case.num_blocks)) - set(private + prefixes))
    assert spare and np.isnan(case.k_cache[spare].astype(np.float32)).all()
    assert np.isfinite(case.k_cache[prefixes].astype(np.float32)).all()
