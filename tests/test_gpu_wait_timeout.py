"""GPU: a bounded on-chip wait that runs out is reported, and the context stays usable.

Every pipeline wait of the decode kernel is bounded.  With the consumer's wait
limit cut far below one DRAM round trip (pa_debug_set_wait_limit_ns), its
first waits for query rows and KV tiles run out: the call must come back with
PA_DEV_WAIT_TIMEOUT in its status word, with no fault and no hang (the CTAs
stop issuing, wait for the copies already in flight with the full limit, and
exit).  With the limit restored, the next decode on the same context and the
same buffers is oracle-green.  No GPU fault is provoked: the wait simply has a
short limit.
"""
import pytest

import synth.workloads as W
from gpu_cases import DecodeCase, check_close, status_word, to_numpy

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hkv,dtype", [(32, 8, "bf16"), (8, 8, "bf16"), (4, 4, "f32")])
def test_short_wait_limit_reports_timeout_then_recovers(hq, hkv, dtype):
    import torch
    import paged_kv_cache_280_gb300 as pa

    w = W.random_case(41, 24, hq, hkv, 128 if dtype == "bf16" else 64, 16, dtype, max_len=3000, min_len=500)
    c = DecodeCase(w).device()
    ref = c.oracle(threads=8)
    try:
        pa.pa_debug_set_wait_limit_ns(1)
        ws = c.run()
        torch.cuda.synchronize()
        st = status_word(ws)
    finally:
        pa.pa_debug_set_wait_limit_ns(0)
    assert st & pa.PA_DEV_WAIT_TIMEOUT, f"status {st:#x}: no wait ran out"
    assert not st & ~pa.PA_DEV_WAIT_TIMEOUT, f"status {st:#x}: an unexpected bit"
    # same context, same pools and output buffer, fresh workspace: a normal decode
    c.dout.fill_(float("nan"))
    ws = c.run()
    torch.cuda.synchronize()
    assert status_word(ws) == 0
    check_close(to_numpy(c.dout), ref, dtype)

