"""Pins for the CPU oracle: checks against facts other than the oracle itself.

Each pin takes an oracle library handle (so the mutation test can run the same
battery against deliberately broken copies of the oracle) and raises
AssertionError when the oracle disagrees with what the pages or the
mathematics fix:

* brute force on tiny inputs (pure Python, math.exp without the max trick,
  math.fsum, numpy's own fp16 decoding);
* equality with an unpaged fp64 library attention (torch's
  scaled_dot_product_attention) on K/V gathered with numpy indexing -- paging
  changes addressing only ("vLLM 2026 推理引擎全解", §2.1);
* invariance under any permutation of physical block placement and under a
  shared versus duplicated prefix ("vLLM 2026 推理引擎全解", §2.1, §2.3);
* closed forms: one token -> that token's V row; q = 0 or scale = 0 -> mean
  of the V rows; two tokens whose scores differ by ln 3 -> weights 1/4, 3/4;
* convexity: each output lies within its V column's range;
* the page example of 16-token pages (tests/golden/page_example.txt);
* exact fp16 decoding of all 65536 bit patterns against numpy;
* reshape_and_cache against numpy scatter assignment.
"""
from __future__ import annotations

import math
import os

import numpy as np

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------
# independent helpers (no oracle code)
# ----------------------------------------------------------------------------

def gather_contiguous(case_or_arrays, s, h):
    """numpy gather of sequence s, head h: (K [ctx, D], V [ctx, D]) as float64."""
    kc, vc, tables, lens, B = case_or_arrays
    ctx = int(lens[s])
    t = np.arange(ctx)
    phys = tables[s, t // B]
    off = t % B
    return kc[phys, h, off, :].astype(np.float64), vc[phys, h, off, :].astype(np.float64)


def brute_force(q, kc, vc, tables, lens, scale):
    """Pure-Python attention: no max subtraction, exact-sum via math.fsum."""
    S, H, D = q.shape
    B = kc.shape[2]
    out = np.zeros((S, H, D))
    for s in range(S):
        for h in range(H):
            ctx = int(lens[s])
            if ctx == 0:
                continue
            qs = [float(x) for x in q[s, h]]
            rows_k, rows_v = [], []
            for t in range(ctx):
                phys = int(tables[s][t // B])
                rows_k.append([float(x) for x in kc[phys, h, t % B]])
                rows_v.append([float(x) for x in vc[phys, h, t % B]])
            e = [math.exp(scale * math.fsum(a * b for a, b in zip(qs, kr))) for kr in rows_k]
            z = math.fsum(e)
            for d in range(D):
                out[s, h, d] = math.fsum(e[t] * rows_v[t][d] for t in range(ctx)) / z
    return out


def library_attention(q, kc, vc, tables, lens, scale):
    """fp64 torch scaled_dot_product_attention over numpy-gathered K/V."""
    import torch
    S, H, D = q.shape
    B = kc.shape[2]
    out = np.zeros((S, H, D))
    for s in range(S):
        for h in range(H):
            if int(lens[s]) == 0:
                continue
            K, V = gather_contiguous((kc, vc, tables, lens, B), s, h)
            qt = torch.from_numpy(q[s, h].astype(np.float64)).view(1, 1, 1, D)
            o = torch.nn.functional.scaled_dot_product_attention(
                qt, torch.from_numpy(K).view(1, 1, -1, D),
                torch.from_numpy(V).view(1, 1, -1, D), scale=float(scale))
            out[s, h] = o.view(D).numpy()
    return out


def small_case(seed, S=3, H=2, D=16, lens=(1, 17, 40), spare=0.5, B=16):
    return workloads.build_case(f"small{seed}", list(lens)[:S], num_heads=H, head_dim=D,
                                seed=seed, block_size=B, spare_frac=spare)


def assert_close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.abs(a - b)
    bound = tol * np.maximum(1.0, np.abs(b))
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: max err {np.nanmax(err)} at {np.argwhere(bad)[:3].tolist()}"


def _decode(lib, case, **over):
    args = dict(q=case.q, k_cache=case.k_cache, v_cache=case.v_cache,
                block_tables=case.block_tables, context_lens=case.context_lens,
                scale=case.scale)
    args.update(over)
    return oracle.decode(lib=lib, **args)


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------

def pin_half_decoding(lib):
    bits = np.arange(65536, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    # sample the whole range through the C decoder (all 2^16 values)
    got = np.array([oracle.half_to_double(int(b), lib=lib) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "NaN patterns differ"
    assert np.array_equal(got[~nan], ref[~nan]), "fp16 decoding differs from numpy"
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), "signed zero"


def bf16_bits_to_float64(bits):
    """Independent bf16 decoding through torch's own bfloat16 type."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).astype(np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def pin_bf16_decoding(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_bits_to_float64(bits)
    got = np.array([oracle.bf16_to_double(int(b), lib=lib) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "bf16 NaN patterns differ"
    assert np.array_equal(got[~nan], ref[~nan]), "bf16 decoding differs from torch"
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), "bf16 signed zero"


def pin_brute_force_bf16(lib):
    """bf16 inputs: brute force over values decoded by torch, not the oracle."""
    case = workloads.build_case("bf16", [1, 16, 17, 40], num_heads=2, head_dim=8, seed=14,
                                spare_frac=0.5, dtype="bf16")
    got = _decode(lib, case, dtype="bf16")
    f = lambda a: bf16_bits_to_float64(a)
    ref = brute_force(f(case.q), f(case.k_cache), f(case.v_cache), case.block_tables,
                      case.context_lens, case.scale)
    assert_close(got, ref, 1e-12, "bf16 brute force")


def pin_brute_force_tiny(lib):
    for seed, D, B, lens in ((11, 8, 16, (1, 16, 17, 40)), (12, 4, 4, (3, 9)),
                             (13, 8, 8, (40, 2))):
        case = workloads.build_case("bf", list(lens), num_heads=2, head_dim=D,
                                    seed=seed, block_size=B, spare_frac=0.5)
        got = _decode(lib, case)
        ref = brute_force(case.q, case.k_cache, case.v_cache, case.block_tables,
                          case.context_lens, case.scale)
        assert_close(got, ref, 1e-12, f"brute force seed {seed}")


def pin_library_attention(lib):
    case = small_case(21, S=4, H=3, D=64, lens=(5, 100, 161, 300))
    got = _decode(lib, case)
    ref = library_attention(case.q, case.k_cache, case.v_cache, case.block_tables,
                            case.context_lens, case.scale)
    assert_close(got, ref, 1e-12, "fp64 library attention")
    tiny = workloads.make_workload("tiny")
    got = _decode(lib, tiny)
    ref = library_attention(tiny.q, tiny.k_cache, tiny.v_cache, tiny.block_tables,
                            tiny.context_lens, tiny.scale)
    assert_close(got, ref, 1e-12, "fp64 library attention (tiny workload)")


def pin_placement_invariance(lib):
    case = small_case(31, S=3, H=2, D=32, lens=(33, 64, 90), spare=1.0)
    base = _decode(lib, case)
    rng = np.random.default_rng(5)
    perm = rng.permutation(case.num_blocks)        # old id -> new id
    inv = np.argsort(perm)                         # new id -> old id
    tables = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    moved = _decode(lib, case, k_cache=case.k_cache[inv], v_cache=case.v_cache[inv],
                    block_tables=tables.astype(np.int32))
    assert np.array_equal(base, moved), "output depends on physical placement"


def pin_shared_vs_duplicated(lib):
    case = workloads.build_case("sp", [40, 57, 33, 48], num_heads=2, head_dim=32, seed=41,
                                shared_prefix_blocks=2)
    assert (case.block_tables[:, :2] == case.block_tables[0, :2]).all()
    dup = workloads.duplicate_prefix(case)
    assert len(np.unique(dup.block_tables[dup.block_tables >= 0])) == int(dup.blocks_used().sum())
    assert np.array_equal(_decode(lib, case), _decode(lib, dup)), "shared != duplicated"


def pin_single_token(lib):
    case = small_case(51, S=3, H=2, D=64, lens=(1, 1, 1))
    got = _decode(lib, case)
    for s in range(3):
        phys = case.block_tables[s, 0]
        assert np.array_equal(got[s], case.v_cache[phys, :, 0, :].astype(np.float64)), \
            "one-token context must return that token's V row exactly"


def pin_uniform_weights(lib):
    case = small_case(61, S=2, H=2, D=32, lens=(7, 50))
    for over in (dict(q=np.zeros_like(case.q)), dict(scale=0.0)):
        got = _decode(lib, case, **over)
        for s in range(2):
            for h in range(2):
                K, V = gather_contiguous((case.k_cache, case.v_cache, case.block_tables,
                                          case.context_lens, case.block_size), s, h)
                mean = np.array([math.fsum(V[:, d]) / V.shape[0] for d in range(V.shape[1])])
                assert_close(got[s, h], mean, 1e-13, f"uniform weights {list(over)}")


def pin_two_token_closed_form(lib):
    """Two tokens whose scores differ by ln 3 get weights 1/4 and 3/4.

    Blocks of one token each: q = e_0, k_0 = 0, k_1 = e_0, scale = ln 3, so
    the scores are 0 and ln 3 and o = (v_0 + 3 v_1) / 4.
    """
    D = 8
    q = np.zeros((1, 1, D), np.float16)
    q[0, 0, 0] = 1.0
    kc = np.zeros((2, 1, 1, D), np.float16)
    kc[1, 0, 0, 0] = 1.0
    rng = np.random.default_rng(71)
    vc = rng.standard_normal((2, 1, 1, D)).astype(np.float16)
    tables = np.array([[0, 1]], np.int32)
    got = oracle.decode(q, kc, vc, tables, np.array([2], np.int32), math.log(3.0), lib=lib)
    ref = (vc[0, 0, 0].astype(np.float64) + 3.0 * vc[1, 0, 0].astype(np.float64)) / 4.0
    assert_close(got[0, 0], ref, 1e-14, "scores differing by ln 3")


def pin_convexity(lib):
    case = small_case(81, S=3, H=3, D=32, lens=(2, 77, 130))
    got = _decode(lib, case)
    for s in range(3):
        for h in range(3):
            _, V = gather_contiguous((case.k_cache, case.v_cache, case.block_tables,
                                      case.context_lens, case.block_size), s, h)
            lo, hi = V.min(axis=0), V.max(axis=0)
            assert (got[s, h] >= lo - 1e-12).all() and (got[s, h] <= hi + 1e-12).all(), \
                "output outside the convex hull of V rows"


def pin_logical_order(lib):
    """Reordering the tokens of a context (moving K and V rows together)
    leaves the output unchanged up to summation order."""
    case = small_case(91, S=1, H=2, D=32, lens=(70,), spare=0.0)
    base = _decode(lib, case)
    B = case.block_size
    ctx = int(case.context_lens[0])
    rng = np.random.default_rng(3)
    perm = rng.permutation(ctx)
    kc, vc = case.k_cache.copy(), case.v_cache.copy()
    t = np.arange(ctx)
    phys = case.block_tables[0, t // B]
    kc[phys, :, t % B, :] = case.k_cache[phys[perm], :, (t % B)[perm], :]
    vc[phys, :, t % B, :] = case.v_cache[phys[perm], :, (t % B)[perm], :]
    moved = _decode(lib, case, k_cache=kc, v_cache=vc)
    assert_close(moved, base, 1e-13, "token order")
    # and swapping only K (not V) must change it
    kc2 = case.k_cache.copy()
    kc2[phys, :, t % B, :] = case.k_cache[phys[perm], :, (t % B)[perm], :]
    assert not np.allclose(_decode(lib, case, k_cache=kc2), base, atol=1e-6)


def pin_page_example(lib):
    lines = [l.split() for l in open(os.path.join(GOLDEN, "page_example.txt"))
             if l.strip() and not l.startswith("#")]
    B = int(next(l for l in lines if l[0] == "page_size")[1])
    table = [int(x) for x in next(l for l in lines if l[0] == "table")[1:]]
    D = 8
    ctx = 48
    kc = np.zeros((3, 1, B, D), np.float16)
    vc = np.zeros((3, 1, B, D), np.float16)
    # the V row at (page p, offset o) holds p in dim 0 and o in dim 1
    for p in range(3):
        for o in range(B):
            vc[p, 0, o, 0] = p
            vc[p, 0, o, 1] = o
    tables = np.array([table], np.int32)
    for l in lines:
        if l[0] != "token":
            continue
        tok, page, off = int(l[1]), int(l[3]), int(l[5])
        k = kc.copy()
        q = np.zeros((1, 1, D), np.float16)
        q[0, 0, 0] = 16.0
        # give logical token `tok` a score of 256 and every other token 0
        k[table[tok // B], 0, tok % B, 0] = 16.0
        got = oracle.decode(q, k, vc, tables, np.array([ctx], np.int32), 1.0, lib=lib)
        assert abs(got[0, 0, 0] - page) < 1e-9 and abs(got[0, 0, 1] - off) < 1e-9, \
            f"token {tok}: expected page {page} offset {off}, got {got[0, 0, :2]}"


def pin_masking(lib):
    """Values beyond the context (NaN-poisoned tail slots and spare blocks)
    never reach the output."""
    case = small_case(101, S=3, H=2, D=16, lens=(1, 15, 33))
    got = _decode(lib, case)
    assert np.isfinite(got).all()
    ref = brute_force(case.q, case.k_cache, case.v_cache, case.block_tables,
                      case.context_lens, case.scale)
    assert_close(got, ref, 1e-12, "masked tail")


def pin_reshape_and_cache(lib):
    case = small_case(111, S=3, H=2, D=16, lens=(5, 16, 30))
    workloads.add_new_tokens(case)
    slots = case.slot_mapping.copy()
    slots[1] = -1                                   # skipped token
    kc, vc = oracle.reshape_and_cache(case.k_new, case.v_new, case.k_cache,
                                      case.v_cache, slots, lib=lib)
    ref_k, ref_v = case.k_cache.copy(), case.v_cache.copy()
    B = case.block_size
    for i, sl in enumerate(slots):
        if sl < 0:
            continue
        ref_k[sl // B, :, sl % B, :] = case.k_new[i]
        ref_v[sl // B, :, sl % B, :] = case.v_new[i]
    assert np.array_equal(kc.view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(vc.view(np.uint16), ref_v.view(np.uint16))
    # edge slots: the first and the last slot of the pool, and a skipped one
    edge = np.array([0, case.num_blocks * B - 1, -7], np.int32)
    kn, vn = case.k_new[:3], case.v_new[:3]
    kc, vc = oracle.reshape_and_cache(kn, vn, case.k_cache, case.v_cache, edge, lib=lib)
    ref_k, ref_v = case.k_cache.copy(), case.v_cache.copy()
    for i, sl in enumerate(edge[:2]):
        ref_k[sl // B, :, sl % B, :] = kn[i]
        ref_v[sl // B, :, sl % B, :] = vn[i]
    assert np.array_equal(kc.view(np.uint16), ref_k.view(np.uint16)), "edge slots (K)"
    assert np.array_equal(vc.view(np.uint16), ref_v.view(np.uint16)), "edge slots (V)"
    # a one-token context then attends only to the stored token: out == v_new
    one = small_case(112, S=2, H=2, D=16, lens=(1, 1))
    workloads.add_new_tokens(one)
    got = oracle.decode_case(one, lib=lib)
    assert np.array_equal(got, one.v_new.astype(np.float64))


def pin_copy_blocks(lib):
    """Block copy against numpy indexing; a copy-on-write of the shared prefix
    followed by retargeting the tables leaves the attention unchanged; a swap
    out to a second pool and back in elsewhere leaves it unchanged too."""
    case = workloads.build_case("cow", [40, 57, 33, 48], num_heads=2, head_dim=16, seed=42,
                                shared_prefix_blocks=2, spare_frac=2.0)
    base = _decode(lib, case)
    used = set(case.block_tables[case.block_tables >= 0].tolist())
    free = [b for b in range(case.num_blocks) if b not in used]
    # sequences 1..3 get private copies of the two prefix blocks
    pairs, tables = [], case.block_tables.copy()
    for s in range(1, 4):
        for b in range(2):
            dst = free.pop()
            pairs.append((int(case.block_tables[s, b]), dst))
            tables[s, b] = dst
    pairs = np.array(pairs, np.int32)
    kc, vc = oracle.copy_blocks(case.k_cache, case.v_cache, case.k_cache, case.v_cache, pairs, lib=lib)
    ref_k, ref_v = case.k_cache.copy(), case.v_cache.copy()
    ref_k[pairs[:, 1]] = case.k_cache[pairs[:, 0]]
    ref_v[pairs[:, 1]] = case.v_cache[pairs[:, 0]]
    assert np.array_equal(kc.view(np.uint16), ref_k.view(np.uint16))
    assert np.array_equal(vc.view(np.uint16), ref_v.view(np.uint16))
    assert np.array_equal(_decode(lib, case, k_cache=kc, v_cache=vc, block_tables=tables), base)
    # swap out every used block to a host pool, back in at shuffled places
    ids = np.array(sorted(used), np.int32)
    host_k = np.zeros((len(ids),) + case.k_cache.shape[1:], case.k_cache.dtype)
    host_v = np.zeros_like(host_k)
    out_pairs = np.stack([ids, np.arange(len(ids), dtype=np.int32)], 1)
    host_k, host_v = oracle.copy_blocks(case.k_cache, case.v_cache, host_k, host_v, out_pairs, lib=lib)
    perm = np.random.default_rng(1).permutation(case.num_blocks)[:len(ids)].astype(np.int32)
    blank_k = np.zeros_like(case.k_cache)
    in_pairs = np.stack([np.arange(len(ids), dtype=np.int32), perm], 1)
    k2, v2 = oracle.copy_blocks(host_k, host_v, blank_k, np.zeros_like(blank_k), in_pairs, lib=lib)
    remap = dict(zip(ids.tolist(), perm.tolist()))
    t2 = np.vectorize(lambda b: remap.get(int(b), -1))(case.block_tables).astype(np.int32)
    assert np.array_equal(_decode(lib, case, k_cache=k2, v_cache=v2, block_tables=t2), base)


def brute_force_prefill(q, kc, vc, tables, lens, qs, scale):
    """Pure-Python causal attention: query i of sequence s sits at position
    ctx - q_len + i and sees keys 0 .. that position."""
    T, H, D = q.shape
    B = kc.shape[2]
    out = np.zeros((T, H, D))
    for s in range(len(lens)):
        ctx, q_len = int(lens[s]), int(qs[s + 1] - qs[s])
        for h in range(H):
            rows_k = [[float(x) for x in kc[int(tables[s][t // B]), h, t % B]] for t in range(ctx)]
            rows_v = [[float(x) for x in vc[int(tables[s][t // B]), h, t % B]] for t in range(ctx)]
            for i in range(q_len):
                row = int(qs[s]) + i
                pos = ctx - q_len + i
                qv = [float(x) for x in q[row, h]]
                e = [math.exp(scale * math.fsum(a * b for a, b in zip(qv, rows_k[t])))
                     for t in range(pos + 1)]
                z = math.fsum(e)
                for d in range(D):
                    out[row, h, d] = math.fsum(e[t] * rows_v[t][d] for t in range(pos + 1)) / z
    return out


def _prefill(lib, case, **over):
    args = dict(q=case.q, k_cache=case.k_cache, v_cache=case.v_cache,
                block_tables=case.block_tables, context_lens=case.context_lens,
                query_start=case.query_start, scale=case.scale, dtype=case.dtype)
    args.update(over)
    return oracle.prefill(lib=lib, **args)


def pin_prefill_brute_force(lib):
    case = workloads.build_prefill_case("pbf", [1, 20, 37, 16], [1, 20, 5, 16], num_heads=2,
                                        head_dim=8, seed=31, spare_frac=0.5)
    got = _prefill(lib, case)
    ref = brute_force_prefill(case.q, case.k_cache, case.v_cache, case.block_tables,
                              case.context_lens, case.query_start, case.scale)
    assert_close(got, ref, 1e-12, "prefill brute force")


def pin_prefill_library_attention(lib):
    """fp64 torch attention with an explicit causal mask on numpy-gathered K/V."""
    import torch
    case = workloads.build_prefill_case("plib", [70, 130], [70, 40], num_heads=3, head_dim=32,
                                        seed=32)
    got = _prefill(lib, case)
    for s in range(case.num_seqs):
        ctx, q0 = int(case.context_lens[s]), int(case.query_start[s])
        q_len = int(case.query_start[s + 1]) - q0
        for h in range(case.num_heads):
            K, V = gather_contiguous((case.k_cache, case.v_cache, case.block_tables,
                                      case.context_lens, case.block_size), s, h)
            Q = case.q[q0:q0 + q_len, h].astype(np.float64)
            pos = np.arange(ctx - q_len, ctx)[:, None]
            mask = torch.from_numpy(np.arange(ctx)[None, :] <= pos)
            o = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(Q)[None, None], torch.from_numpy(K)[None, None],
                torch.from_numpy(V)[None, None], attn_mask=mask[None, None], scale=case.scale)
            assert_close(got[q0:q0 + q_len, h], o[0, 0].numpy(), 1e-12, "prefill vs library")


def pin_prefill_special_cases(lib):
    # one query per sequence, at the last position, is decode
    case = workloads.build_prefill_case("p1", [33, 90, 5], [1, 1, 1], num_heads=2, head_dim=16,
                                        seed=33)
    got = _prefill(lib, case)
    dec = _decode(lib, case)
    assert np.array_equal(got, dec), "a single query must match decode"
    # the first query of a whole-prompt prefill sees only token 0: its V row
    case = workloads.build_prefill_case("p2", [40], [40], num_heads=2, head_dim=16, seed=34)
    got = _prefill(lib, case)
    phys = case.block_tables[0, 0]
    assert np.array_equal(got[0], case.v_cache[phys, :, 0, :].astype(np.float64))


PINS = [
    ("half_decoding", pin_half_decoding),
    ("bf16_decoding", pin_bf16_decoding),
    ("brute_force_tiny", pin_brute_force_tiny),
    ("brute_force_bf16", pin_brute_force_bf16),
    ("library_attention", pin_library_attention),
    ("placement_invariance", pin_placement_invariance),
    ("shared_vs_duplicated", pin_shared_vs_duplicated),
    ("single_token", pin_single_token),
    ("uniform_weights", pin_uniform_weights),
    ("two_token_closed_form", pin_two_token_closed_form),
    ("convexity", pin_convexity),
    ("logical_order", pin_logical_order),
    ("page_example", pin_page_example),
    ("masking", pin_masking),
    ("reshape_and_cache", pin_reshape_and_cache),
    ("copy_blocks", pin_copy_blocks),
    ("prefill_brute_force", pin_prefill_brute_force),
    ("prefill_library_attention", pin_prefill_library_attention),
    ("prefill_special_cases", pin_prefill_special_cases),
]
