"""The allocation-free prefill entry point (kda_chunk_prefill_noalloc).

It exists for callers that cannot allocate device memory when they run the
prefill, for example code inside another framework's allocator callback or a
serving path that forbids allocation per request. It must give the same
results as kda_chunk_prefill with a caller-provided workspace. Its scratch is
a fixed array shared by every call, so two calls in a row must both be right
whatever the first one left behind.

This file is collected last on purpose: if it fails, every other test has
already run.
"""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth
from tests._util import BF16_REL, F32_ATOL, cuda_or_skip, ensure_built, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = cuda_or_skip()
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda
    return torch, kda


def _draw(seed, lengths, bf16, D=128):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return synth.prefill_inputs(seed, int(cu[-1]), 3, D, bf16, cu_seqlens=cu, s0_std=0.1, g_scale=0.2)


def _inputs(torch, seed, lengths, bf16, D=128):
    d = _draw(seed, lengths, bf16, D)
    cu = d["cu_seqlens"]
    dt = torch.bfloat16 if bf16 else torch.float32
    t = {n: to_dev(d[n], dt, torch) for n in ("q", "k", "v")}
    t["g"] = to_dev(d["g"], torch.float32, torch)
    t["beta"] = to_dev(d["beta"], torch.float32, torch)
    t["s0"] = to_dev(d["s0"], torch.float32, torch)
    t["cu"] = torch.from_numpy(cu).cuda()
    return t, len(lengths)


def _run(torch, kda, t, N, noalloc):
    out = torch.full_like(t["q"], float("nan"))
    sf = torch.full((N,) + tuple(t["s0"].shape[1:]), float("nan"), dtype=torch.float32, device="cuda")
    fn = kda.kda_chunk_prefill_noalloc if noalloc else kda.kda_chunk_prefill
    fn(t["q"], t["k"], t["v"], t["g"], t["beta"], out, initial_state=t["s0"], final_state=sf,
       cu_seqlens=t["cu"], chunk_size=64)
    kda.kda_sync_status()
    return to_np(out), to_np(sf)


def _close(a, b, bf16):
    assert np.all(np.isfinite(a))
    err = np.max(np.abs(a - b))
    if bf16:
        assert err / max(np.max(np.abs(b)), 1e-6) <= BF16_REL
    else:
        assert err <= F32_ATOL


@pytest.mark.parametrize("bf16", [True, False])
def test_noalloc_prefill_matches_workspace_prefill_twice(env, bf16):
    torch, kda = env
    # two different mixed-length batches, back to back, so that the second
    # call runs on scratch the first one filled
    t1, n1 = _inputs(torch, 901, [70, 5, 0, 300, 33, 129, 64, 1], bf16)
    t2, n2 = _inputs(torch, 902, [10, 200, 3], bf16)
    for t, n in ((t1, n1), (t2, n2)):
        o_ref, s_ref = _run(torch, kda, t, n, noalloc=False)
        o_na, s_na = _run(torch, kda, t, n, noalloc=True)
        _close(o_na, o_ref, bf16)
        _close(s_na, s_ref, bf16)


@pytest.mark.parametrize("bf16", [True, False])
def test_noalloc_single_sequence_and_oracle(env, bf16):
    # N = 1 needs no launch order, so the call passes no scratch at all; then a
    # small mixed batch against the fp64 oracle directly, per (sequence, head)
    torch, kda = env
    for seed, lengths in ((903, [150]), (904, [64, 0, 97, 2])):
        d = _draw(seed, lengths, bf16)
        t, n = _inputs(torch, seed, lengths, bf16)
        o_na, s_na = _run(torch, kda, t, n, noalloc=True)
        ro, rs = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"],
                                   cu_seqlens=d["cu_seqlens"], eps=1e-6)
        cu = d["cu_seqlens"]
        for i in range(n):
            a, b = cu[i], cu[i + 1]
            if b > a:
                _close(o_na[a:b], ro[a:b], bf16)
            _close(s_na[i], rs[i], bf16)


def test_noalloc_rejects_batches_above_its_limit(env):
    torch, kda = env
    L = kda.lib()
    st = L.kda_chunk_prefill_noalloc(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, None, None, 0x60000, 0x70000,
                                     4097, 5000, 2, 128, 64, 1, 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG
    assert "4096" in L.kda_last_error_detail().decode()
