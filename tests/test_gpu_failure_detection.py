"""Failure detection on the GPU without a fault: a bounded on-chip wait that
runs out (an mbarrier that nothing arrives at) is reported as
FA_ERR_DEVICE_TIMEOUT through the status word, once, and the context keeps
running the attention kernels correctly afterwards."""
import time

import pytest

from attention_forward_fa_gb300 import workloads as W
from oracle import attention as A

from tests.parity import compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_fa_gb300 import build
    build.build()


def test_wait_probe_reports_the_timeout_once():
    import attention_forward_fa_gb300 as fa
    assert fa.fa_check_status() == 0
    fa.fa_set_wait_timeout_ns(1_000_000)   # 1 ms
    try:
        t0 = time.perf_counter()
        assert fa.fa_wait_probe() == 0
        assert fa.fa_check_status() == -7      # FA_ERR_DEVICE_TIMEOUT
        assert time.perf_counter() - t0 < 5.0  # the wait gave up; nothing hung
        assert fa.fa_check_status() == 0       # reported once, then cleared
    finally:
        fa.fa_set_wait_timeout_ns(0)
    # the context is intact: a small causal problem still matches the oracle
    p = W.dense(name="after_probe", B=1, Hq=2, Sq=300, D=128, mask=W.MASK_CAUSAL, seed=31)
    O, L = run_gpu(p, 0.0)
    Or, Lr = A.attention_problem(p)
    compare(O, L, Or, Lr, where=p.name)
