"""A continuously batched decode loop over the host-side KV block manager.

Sequences join (some sharing a system prompt's blocks, some forked from a
parent as parallel samples), grow by one token per step, and finish; the
manager hands out slots and copy-on-write copies, the step writes the new K/V
and decodes.  After every step the output is compared with the oracle run on a
host mirror of the cache that receives the same copies and writes.  The loop
runs eagerly and replayed from a CUDA graph, with plain decode and with the
shared-prefix decode (the batch ordered so that sharers are adjacent, the
groups taken from the manager's sharing records every step), in fp16 and
bf16, and pipelined:
two staging slots in turn, each step's upload on a copy stream overlapping the
previous step, and each step's output read after the next one is submitted."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import assert_parity

pytestmark = pytest.mark.gpu

H, D, B, N, MB, SMAX = 4, 128, 16, 1024, 64, 16


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


def _normal(rng, shape, dtype="f16"):
    x = rng.standard_normal(shape, dtype=np.float32)
    return workloads.f32_to_bf16_bits(x) if dtype == "bf16" else x.astype(np.float16)


def _to_dev(a, dev):
    """Host fp16 values or bf16 bit patterns -> a device tensor of that type."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _to_host(t):
    """A device fp16 tensor -> float16 values; bf16 -> uint16 bit patterns."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("use_graph,host_out,shared,pipelined,dtype",
                         [(False, False, False, False, "f16"), (True, False, False, False, "f16"),
                          (True, True, False, False, "f16"), (False, False, True, False, "f16"),
                          (True, False, True, False, "f16"), (True, True, False, True, "f16"),
                          (False, False, True, True, "f16"), (True, True, False, True, "bf16"),
                          (False, False, True, False, "bf16")])
def test_continuous_batching_loop(dev, use_graph, host_out, shared, pipelined, dtype):
    import torch
    import paged_kv_cache_269_gb300 as pa
    from paged_kv_cache_269_gb300.step import DecodeStep, PipelinedDecodeStep
    rng = np.random.default_rng(77 + use_graph)
    mgr = pa.KVManager(N, B, MB, shuffle_seed=5)
    if dtype == "bf16":   # NaN bit patterns in every slot not yet written
        mirror_k = np.full((N, H, B, D), 0x7FC0, np.uint16)
    else:
        mirror_k = np.full((N, H, B, D), np.nan, np.float16)
    mirror_v = mirror_k.copy()
    kc = _to_dev(mirror_k, dev)
    vc = _to_dev(mirror_v, dev)
    scale = float(np.float32(1 / np.sqrt(D)))
    # pipelined: two staging slots, step k + 1's upload overlapping step k,
    # each output checked after the next step has been submitted
    kind = PipelinedDecodeStep if pipelined else DecodeStep
    step = kind(kc, vc, SMAX, MB, scale, use_graph=use_graph, partition_tokens=64,
                host_out=host_out, max_groups=SMAX if shared else 0)
    pending = []   # (ticket, n, reference, label) of submitted steps not yet checked

    def check(ticket, n, ref, label):
        out = step.result(ticket) if pipelined else step.launched_out
        if not pipelined:
            step.stream.synchronize()
        assert out.is_cuda != host_out              # the pinned host copy with host_out
        assert_parity(_to_host(out[:n]), ref, label, dtype=dtype)
        assert (_to_host(out[n:]) == 0).all()              # padding rows
    grouped_steps = 0

    def write(slots, k, v):
        """Store token K/V at slots on the device and in the mirror."""
        nonlocal mirror_k, mirror_v
        slots = np.asarray(slots, np.int32)
        with torch.cuda.stream(step.stream):     # ordered with the steps
            ts = torch.from_numpy(slots).to(dev)
            pa.reshape_and_cache(_to_dev(k, dev), _to_dev(v, dev), kc, vc, ts)
        mirror_k, mirror_v = oracle.reshape_and_cache(k, v, mirror_k, mirror_v, slots)

    def prefill(seq, first):
        n = mgr.context_len(seq)
        if n > first:
            slots = [mgr.slot(seq, t) for t in range(first, n)]
            write(slots, _normal(rng, (n - first, H, D), dtype),
                  _normal(rng, (n - first, H, D), dtype))

    running = []
    system = mgr.add_sequence(80)                 # a 5-block system prompt
    prefill(system, 0)
    running.append(system)
    for _ in range(3):                            # requests sharing its full blocks
        s = mgr.add_sequence(80 + int(rng.integers(1, 40)), system, 5)
        prefill(s, 80)
        running.append(s)
    running.append(mgr.fork(running[1]))          # parallel samples of request 1
    running.append(mgr.fork(running[1]))
    s = mgr.add_sequence(int(rng.integers(1, 300)))
    prefill(s, 0)
    running.append(s)

    for it in range(40):
        # continuous batching: some sequences finish, new ones join
        if it % 7 == 6 and len(running) > 3:
            mgr.free(running.pop(int(rng.integers(0, len(running)))))
        if it % 5 == 4 and len(running) < SMAX:
            parent = running[int(rng.integers(0, len(running)))]
            if rng.random() < 0.5:
                running.append(mgr.fork(parent))
            else:
                s = mgr.add_sequence(int(rng.integers(1, 200)))
                prefill(s, 0)
                running.append(s)
        batch = list(running)
        if shared:   # sharers adjacent: by first block, stably
            batch.sort(key=lambda s: int(mgr.block_tables([s], MB)[0][0][0]))
        slots, cow = [], []
        for s in batch:
            slot, src, dst = mgr.append(s)
            slots.append(slot)
            if src >= 0:
                cow.append((src, dst))
        if cow:
            step.copy_on_write(cow)
            mirror_k, mirror_v = oracle.copy_blocks(mirror_k, mirror_v, mirror_k, mirror_v,
                                                    np.asarray(cow, np.int32))
        n = len(batch)
        q, kn, vn = (_normal(rng, (n, H, D), dtype) for _ in range(3))
        tables, lens = mgr.block_tables(batch, MB)
        groups = mgr.prefix_groups(batch, SMAX) if shared else None
        if shared and (groups[1] > 0).any():
            grouped_steps += 1
        step.prepare(q, kn, vn, np.asarray(slots, np.int32), tables, lens, groups=groups)
        if pipelined:
            ticket = step.launch()
        else:
            step.launched_out = step.launch()
            ticket = it
        mirror_k, mirror_v = oracle.reshape_and_cache(kn, vn, mirror_k, mirror_v,
                                                      np.asarray(slots, np.int32))
        ref = oracle.decode(q, mirror_k, mirror_v, tables, lens, scale, dtype=dtype)
        pending.append((ticket, n, ref, f"step {it} (graph={use_graph}, shared={shared}, "
                                        f"pipelined={pipelined}, {dtype})"))
        # a pipelined step's output is read once the next step is in flight
        while len(pending) > (1 if pipelined else 0):
            check(*pending.pop(0))
    while pending:
        check(*pending.pop(0))
    assert pa.device_errors(stream=step.stream) == 0
    if shared:
        assert grouped_steps >= 20                         # the prefix path was exercised
    assert np.array_equal(_to_host(kc).view(np.uint16), mirror_k.view(np.uint16))
