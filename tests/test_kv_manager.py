"""The host-side KV block manager (pa_kvm_*) against an independent Python
model of the same rules, under random operation sequences (CPU only)."""
from collections import deque

import numpy as np
import pytest

import paged_kv_cache_269_gb300 as pa


@pytest.fixture
def rng():
    return np.random.default_rng(1234)


def check_invariants(m, live, N):
    refs = np.zeros(N, int)
    for sid in live:
        t, l = m.block_tables([sid])
        nb = -(-int(l[0]) // m.block_size)
        for b in t[0, :nb]:
            refs[b] += 1
    for b in range(N):
        assert m.refcount(b) == refs[b]
    assert m.num_free_blocks() == int((refs == 0).sum())


def test_against_model(rng):
    N, B, MB = 64, 4, 12
    m = pa.KVManager(N, B, MB, shuffle_seed=0)
    free = deque(range(N))
    ref = [0] * N
    model = {}        # seq id -> [blocks, len]
    next_id = [0]
    spare_ids = []

    def pop():
        b = free.popleft()
        ref[b] = 1
        return b

    def release(b):
        ref[b] -= 1
        if ref[b] == 0:
            free.append(b)

    def new_id():
        if spare_ids:
            return spare_ids.pop()
        next_id[0] += 1
        return next_id[0] - 1

    for step in range(3000):
        op = rng.choice(["add", "share", "fork", "append", "append", "append", "free"])
        live = sorted(model)
        if op == "add":
            n = int(rng.integers(0, 20))
            need = -(-n // B)
            if need > MB:
                continue
            if need > len(free):
                with pytest.raises(pa.PaError) as e:
                    m.add_sequence(n)
                assert e.value.status == -7
                continue
            sid = m.add_sequence(n)
            assert sid == new_id()
            model[sid] = [[pop() for _ in range(need)], n]
        elif op == "share" and live:
            p = int(rng.choice(live))
            full = model[p][1] // B
            k = int(rng.integers(0, full + 1))
            n = int(rng.integers(k * B, min(MB * B, k * B + 12) + 1))
            need = -(-n // B)
            if need - k > len(free):
                continue
            sid = m.add_sequence(n, p, k)
            assert sid == new_id()
            blocks = model[p][0][:k]
            for b in blocks:
                ref[b] += 1
            model[sid] = [blocks + [pop() for _ in range(need - k)], n]
        elif op == "fork" and live:
            p = int(rng.choice(live))
            sid = m.fork(p)
            assert sid == new_id()
            for b in model[p][0]:
                ref[b] += 1
            model[sid] = [list(model[p][0]), model[p][1]]
        elif op == "append" and live:
            sid = int(rng.choice(live))
            blocks, n = model[sid]
            lb = n // B
            if lb >= MB:
                with pytest.raises(pa.PaError):
                    m.append(sid)
                continue
            need_new = lb >= len(blocks) or ref[blocks[lb]] > 1
            if need_new and not free:
                with pytest.raises(pa.PaError) as e:
                    m.append(sid)
                assert e.value.status == -7
                continue
            slot, src, dst = m.append(sid)
            if lb >= len(blocks):
                blocks.append(pop())
                assert (src, dst) == (-1, -1)
            elif ref[blocks[lb]] > 1:
                old = blocks[lb]
                nb = pop()
                release(old)
                blocks[lb] = nb
                assert (src, dst) == (old, nb)
            else:
                assert (src, dst) == (-1, -1)
            assert slot == blocks[lb] * B + n % B
            model[sid][1] = n + 1
        elif op == "free" and live:
            sid = int(rng.choice(live))
            m.free(sid)
            for b in model[sid][0]:
                release(b)
            del model[sid]
            spare_ids.append(sid)
        # compare the whole state
        for sid, (blocks, n) in model.items():
            t, l = m.block_tables([sid], MB)
            assert int(l[0]) == n and m.context_len(sid) == n
            assert list(t[0, :len(blocks)]) == blocks and (t[0, len(blocks):] == -1).all()
            if n:
                tok = int(rng.integers(0, n))
                assert m.slot(sid, tok) == blocks[tok // B] * B + tok % B
        assert [m.refcount(b) for b in range(N)] == ref
        assert m.num_free_blocks() == len(free)
        if step % 200 == 0:
            check_invariants(m, list(model), N)


def test_shuffled_free_list_is_a_seeded_permutation():
    a = pa.KVManager(100, 16, 100, shuffle_seed=7)
    b = pa.KVManager(100, 16, 100, shuffle_seed=7)
    c = pa.KVManager(100, 16, 100, shuffle_seed=8)
    ta, _ = a.block_tables([a.add_sequence(1600)], 100)
    tb, _ = b.block_tables([b.add_sequence(1600)], 100)
    tc, _ = c.block_tables([c.add_sequence(1600)], 100)
    assert sorted(ta[0]) == list(range(100)) and list(ta[0]) == list(tb[0])
    assert list(ta[0]) != list(tc[0]) and list(ta[0]) != list(range(100))


def test_padding_rows_and_errors():
    m = pa.KVManager(8, 16, 4)
    s = m.add_sequence(17)
    t, l = m.block_tables([s, -1], 4)
    assert list(l) == [17, 0] and (t[1] == -1).all()
    with pytest.raises(pa.PaError):
        m.add_sequence(100)                      # more blocks than a row holds
    with pytest.raises(pa.PaError):
        m.append(99)                             # unknown sequence
    with pytest.raises(pa.PaError):
        m.add_sequence(10, s, 2)                 # parent has one full block only
    m.free(s)
    with pytest.raises(pa.PaError):
        m.free(s)
    assert m.num_free_blocks() == 8
