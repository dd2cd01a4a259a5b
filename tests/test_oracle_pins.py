"""The oracle against its pins (CPU only)."""
import os

import numpy as np
import pytest

import oracle
import workloads
from pins import PINS, GOLDEN


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("name,fn", PINS, ids=[n for n, _ in PINS])
def test_pin(lib, name, fn):
    fn(lib)


def test_rejects_bad_table_entry(lib):
    case = workloads.build_case("bad", [20, 5], num_heads=1, head_dim=8, seed=1)
    tables = case.block_tables.copy()
    tables[0, 1] = case.num_blocks          # one past the pool
    with pytest.raises(oracle.OracleError, match="block table"):
        oracle.decode(case.q, case.k_cache, case.v_cache, tables, case.context_lens,
                      case.scale, lib=lib)


def test_rejects_context_past_table(lib):
    case = workloads.build_case("bad", [20, 5], num_heads=1, head_dim=8, seed=1)
    lens = case.context_lens.copy()
    lens[1] = case.max_blocks_per_seq * case.block_size + 1
    with pytest.raises(oracle.OracleError, match="context"):
        oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables, lens,
                      case.scale, lib=lib)


def test_rejects_slot_past_pool(lib):
    case = workloads.build_case("bad", [3], num_heads=1, head_dim=8, seed=1, new_tokens=True)
    slots = np.array([case.num_blocks * case.block_size], np.int32)
    with pytest.raises(oracle.OracleError, match="slot"):
        oracle.reshape_and_cache(case.k_new, case.v_new, case.k_cache, case.v_cache,
                                 slots, lib=lib)


def test_zero_context_gives_zero(lib):
    case = workloads.build_case("z", [0, 9], num_heads=2, head_dim=8, seed=2)
    out = oracle.decode_case(case, lib=lib)
    assert (out[0] == 0).all() and np.isfinite(out).all()


def test_kv_bytes_golden():
    vals = {}
    for line in open(os.path.join(GOLDEN, "kv_bytes_llama7b.txt")):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    per_tok = workloads.kv_bytes_per_token(vals["num_heads"], vals["head_dim"], vals["dtype_bytes"])
    assert per_tok == vals["bytes_per_token"]
    assert per_tok * vals["seq_len"] == vals["bytes_per_layer"]
    assert per_tok * vals["seq_len"] * vals["layers"] == vals["bytes_all_layers"]


def test_blocks_needed_golden():
    for line in open(os.path.join(GOLDEN, "blocks_needed.txt")):
        if line.strip() and not line.startswith("#"):
            B, n, nb = (int(x) for x in line.split())
            assert workloads.blocks_needed(n, B) == nb
