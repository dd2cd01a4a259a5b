"""The bounded waits that every kernel relies on give up, report a timeout
and leave the context usable (no GPU fault: each wait is limited by the wall
clock)."""
import pytest

import oracle
import workloads
from gpu_helpers import assert_parity, run_gpu

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


def test_bounded_waits_give_up_and_report(dev):
    import paged_kv_cache_269_gb300 as pa
    assert pa.selftest_wait_timeout() == [0, 0, 0]
    assert pa.device_errors() & pa.DEVERR_TIMEOUT
    assert pa.device_errors() == 0          # reading cleared the word
    # the context still works: a small decode matches the oracle
    case = workloads.make_workload("tiny")
    got, flags, _ = run_gpu(case, dev)
    assert flags == 0
    ref = oracle.decode_case(case)
    assert_parity(got, ref, "decode after the wait self-test")
