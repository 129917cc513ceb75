"""Failure reporting on the GPU without a fault: a bounded device-side wait
that nothing completes gives up, raises the device error word, and the
context stays usable for the next call."""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth
from tests._util import assert_close, cuda_or_skip, ensure_built, to_dev, to_np

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    torch = cuda_or_skip()
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda
    kda.kda_sync_status()  # start clean
    kda.kda_selftest_bounded_wait(2_000_000)  # about 1 ms at the GB300 clock
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_sync_status()
    assert ei.value.status == kda.KDA_ERR_TIMEOUT
    kda.kda_sync_status()  # reported once, then cleared
    # the context is still usable: a decode step right after matches the oracle
    d = synth.decode_inputs(400, 2, 3, 128, True, s0_std=0.5)
    bf = torch.bfloat16
    tq, tk, tv = (to_dev(d[n], bf, torch) for n in ("q", "k", "v"))
    ts = to_dev(d["s0"], torch.float32, torch)
    out = torch.empty_like(tq)
    kda.kda_decode_step(tq, tk, tv, to_dev(d["g"], torch.float32, torch), to_dev(d["beta"], torch.float32, torch),
                        ts, out)
    kda.kda_sync_status()
    ro, rs = oracle.decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"])
    assert_close(to_np(out), ro, True, (0, 1), "out")
    assert_close(to_np(ts), rs, True, (0, 1), "state")
