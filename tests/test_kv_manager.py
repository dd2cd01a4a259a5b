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


def _model_groups(tables, lens, B):
    """The grouping rule, restated: row i's group prefix is what it shares with
    row i + 1 (full blocks only); later rows join while they share at least
    that much with row i; rows sharing nothing with the next row are gathered
    into prefix-0 groups."""
    n = len(lens)
    full = [int(l) // B for l in lens]

    def common(i, j):
        c = 0
        while c < min(full[i], full[j]) and tables[i][c] == tables[j][c]:
            c += 1
        return c

    starts, pre, i, open0 = [], [], 0, False
    while i < n:
        P = common(i, i + 1) if i + 1 < n else 0
        if P > 0:
            j = i + 1
            while j < n and common(i, j) >= P:
                j += 1
            starts.append(i)
            pre.append(P)
            open0, i = False, j
        else:
            if not open0:
                starts.append(i)
                pre.append(0)
            open0, i = True, i + 1
    return starts + [n], pre


def test_prefix_groups_of_shared_prompts_and_forks():
    B = 16
    m = pa.KVManager(256, B, 32)
    p = m.add_sequence(100)                     # 6 full blocks + a partial one
    c1 = m.add_sequence(130, p, 6)              # shares the 6 full blocks
    c2 = m.add_sequence(101, p, 6)
    x = m.add_sequence(50)                      # shares nothing
    y = m.add_sequence(70)
    f = m.fork(c1)                              # shares all of c1, a partial block included
    gs, gp = m.prefix_groups([p, c1, c2, x, y, c1, f, -1])
    assert gs.tolist() == [0, 3, 5, 7, 8] and gp.tolist() == [6, 0, 8, 0]
    # the members of each group do share those blocks, and they are full in each
    t, l = m.block_tables([p, c1, c2, x, y, c1, f, -1], 32)
    for g in range(len(gp)):
        rows = range(gs[g], gs[g + 1])
        for r in rows:
            assert (t[r, :gp[g]] == t[gs[g], :gp[g]]).all() and gp[g] * B <= l[r]
    es, ep = m.prefix_groups([])
    assert es.tolist() == [0] and ep.tolist() == []
    with pytest.raises(pa.PaError):
        m.prefix_groups([p, c1, x, y], max_groups=1)   # needs 2 groups
    with pytest.raises(pa.PaError):
        m.prefix_groups([p, 999])


def test_prefix_groups_match_the_rule(rng):
    B = 8
    m = pa.KVManager(4000, B, 64, shuffle_seed=3)
    live = []
    for _ in range(300):
        op = rng.integers(0, 4)
        if op == 0 or not live:
            live.append(m.add_sequence(int(rng.integers(1, 200))))
        elif op == 1:
            par = live[int(rng.integers(0, len(live)))]
            full = m.context_len(par) // B
            k = int(rng.integers(0, full + 1))
            live.append(m.add_sequence(k * B + int(rng.integers(0, 60)), par, k))
        elif op == 2:
            live.append(m.fork(live[int(rng.integers(0, len(live)))]))
        else:
            s = live[int(rng.integers(0, len(live)))]
            m.append(s)
        if len(live) > 40:
            m.free(live.pop(int(rng.integers(0, len(live)))))
        if rng.random() < 0.3:
            batch = list(live)
            rng.shuffle(batch)
            batch.sort(key=lambda s: m.block_tables([s], 64)[0][0][0])   # sharers adjacent
            batch += [-1] * int(rng.integers(0, 3))
            t, l = m.block_tables(batch, 64)
            gs, gp = m.prefix_groups(batch)
            want_s, want_p = _model_groups(t, l, B)
            assert gs.tolist() == want_s and gp.tolist() == want_p
