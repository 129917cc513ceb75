"""Host-side checks of the C ABI (no GPU, no compute calls).

The library must load, export every function include/kda.h declares, give
the memory figures of the WARP write-up ("KV缓存从11.25GB缩到0.21GB: WARP中Kimi
Delta Attention线性注意力原理剖析", section "414MB 的 KDA 状态从哪来"), and reject
bad arguments synchronously, before any CUDA call.
"""
import ctypes
import os
import re

import pytest

from tests._util import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda as mod
    mod.lib()
    return mod


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(kda):
    declared = _declared_functions()
    assert "kda_decode_step" in declared and "kda_chunk_prefill" in declared
    handle = ctypes.CDLL(kda.library_path())
    for name in declared:
        assert hasattr(handle, name), f"{name} declared in kda.h but not exported"
    assert set(declared) == set(kda.exported_symbols())


def test_status_strings(kda):
    L = kda.lib()
    for s in range(6):
        assert L.kda_status_string(s)
    assert b"unknown" in L.kda_status_string(99)
    assert L.kda_abi_version() == 1


def test_state_bytes_pins_414_mib(kda):
    # 69 layers x 96 heads x 128 x 128 x 4 B
    assert kda.state_bytes(69, 96, 128, 128) == 434_110_464
    assert kda.state_bytes(69, 96, 128, 128) / 2**20 == 414.0
    assert kda.state_bytes(-1, 96, 128, 128) == 0


def test_ring_bytes_pins_about_30_mib(kda):
    # 69 layers x 96 heads x 3 projections x 3 tokens x 128 x 4 B = 29.1 MiB,
    # the "~30 MiB" of the 4K memory ledger
    b = kda.shortconv_ring_bytes(69, 1, 96, 128, 4)
    assert b == 69 * 96 * 3 * 3 * 128 * 4
    assert 29.0 < b / 2**20 < 29.2


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


@pytest.mark.parametrize("case,detail", [
    (dict(D=24), "D must be"),
    (dict(H=0), "H must be"),
    (dict(B=-1), "B must be"),
    (dict(dtype=7), "dtype"),
    (dict(eps=-1.0), "l2_eps"),
    (dict(q=None), "q is NULL"),
    (dict(state=0x10004), "state is not 16-byte aligned"),
    (dict(out=0x10000), "out must not alias"),
])
def test_decode_rejects_bad_arguments(kda, case, detail):
    a = dict(q=0x10000, k=0x20000, v=0x30000, g=0x40000, beta=0x50000, state=0x60000, out=0x70000,
             B=2, H=3, D=128, dtype=1, eps=1e-6)
    a.update(case)
    L = kda.lib()
    st = L.kda_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["state"], a["out"], a["B"], a["H"],
                           a["D"], a["dtype"], a["eps"], None)
    assert st == kda.KDA_ERR_INVALID_ARG
    assert detail in L.kda_last_error_detail().decode()


@pytest.mark.parametrize("case,detail", [
    (dict(D=8), "D must be"),
    (dict(ring=None), "ring is NULL"),
    (dict(y=0x20000), "y must not alias"),
    (dict(w=0x30008), "w is not 16-byte aligned"),
])
def test_shortconv_rejects_bad_arguments(kda, case, detail):
    a = dict(x=0x10000, ring=0x20000, w=0x30000, y=0x40000, B=2, H=3, D=128, dtype=1)
    a.update(case)
    L = kda.lib()
    st = L.kda_shortconv_step(a["x"], a["ring"], a["w"], a["y"], a["B"], a["H"], a["D"], a["dtype"], None)
    assert st == kda.KDA_ERR_INVALID_ARG
    assert detail in L.kda_last_error_detail().decode()


def test_zero_batch_is_a_noop_without_cuda(kda):
    L = kda.lib()
    assert L.kda_decode_step(None, None, None, None, None, None, None, 0, 3, 128, 1, 1e-6, None) == kda.KDA_OK
    assert L.kda_shortconv_step(None, None, None, None, 0, 3, 128, 1, None) == kda.KDA_OK


@pytest.mark.parametrize("case,detail", [
    (dict(D=48), "D must be"),
    (dict(x=None), "x is NULL"),
    (dict(out=0x20000), "out must not alias"),
    (dict(eps=-0.5), "l2_eps"),
])
def test_fused_decode_rejects_bad_arguments(kda, case, detail):
    a = dict(x=0x10000, ring=0x20000, w=0x30000, g=0x40000, beta=0x50000, state=0x60000, out=0x70000,
             B=2, H=3, D=128, dtype=1, eps=1e-6)
    a.update(case)
    L = kda.lib()
    st = L.kda_shortconv_decode_step(a["x"], a["ring"], a["w"], a["g"], a["beta"], a["state"], a["out"], a["B"],
                                     a["H"], a["D"], a["dtype"], a["eps"], None)
    assert st == kda.KDA_ERR_INVALID_ARG
    assert detail in L.kda_last_error_detail().decode()


def test_prefill_workspace_is_the_launch_order(kda):
    """Mixed-length batches of 2..4096 sequences take one int32 per sequence
    (rounded to 256 bytes) for the longest-first launch order; one sequence
    or very large batches take none."""
    assert kda.kda_chunk_prefill_workspace_bytes(1000, 1, 96, 128, 64) == 0
    assert kda.kda_chunk_prefill_workspace_bytes(1000, 8, 96, 128, 64) == 256
    assert kda.kda_chunk_prefill_workspace_bytes(1000, 100, 96, 128, 64) == 512
    assert kda.kda_chunk_prefill_workspace_bytes(1000, 5000, 96, 128, 64) == 0


def test_prefill_rejects_short_workspace(kda):
    L = kda.lib()
    st = L.kda_chunk_prefill(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, None, None, 0x60000, 0x70000, 8, 100,
                             4, 128, 64, 1, 1e-6, 0x80000, 16, None)
    assert st == kda.KDA_ERR_INVALID_ARG
    assert "workspace too small" in L.kda_last_error_detail().decode()


@pytest.mark.parametrize("case,detail", [
    (dict(C=65), "C must be in 1..64"),
    (dict(C=0), "C must be in 1..64"),
    (dict(N=2, cu=None), "cu_seqlens is NULL but N != 1"),
    (dict(D=100), "D must be"),
    (dict(q=None), "q is NULL"),
])
def test_prefill_rejects_bad_arguments(kda, case, detail):
    a = dict(q=0x10000, cu=0x70000, N=1, T=100, H=4, D=128, C=64)
    a.update(case)
    L = kda.lib()
    st = L.kda_chunk_prefill(a["q"], 0x20000, 0x30000, 0x40000, 0x50000, None, None, 0x60000, a["cu"], a["N"],
                             a["T"], a["H"], a["D"], a["C"], 1, 1e-6, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG
    assert detail in L.kda_last_error_detail().decode()


@pytest.mark.parametrize("case,detail", [
    (dict(N=0), "N must be"),
    (dict(T=-1), "T must be"),
    (dict(D=40), "D must be"),
    (dict(N=3, cu=None), "cu_seqlens may be NULL only"),
    (dict(x=None), "x is NULL"),
    (dict(ring_out=0x50000, ring_in=0x50000), "ring_out must not alias"),
    (dict(y=0x10000), "y must not alias"),
    (dict(cu=0x70004), "cu_seqlens must be 8-byte aligned"),
])
def test_conv_prefill_rejects_bad_arguments(kda, case, detail):
    a = dict(x=0x10000, ring_in=0x20000, w=0x30000, y=0x40000, ring_out=0x60000, cu=0x70000, N=1, T=100,
             H=4, D=128)
    a.update(case)
    L = kda.lib()
    st = L.kda_shortconv_prefill(a["x"], a["ring_in"], a["w"], a["y"], a["ring_out"], a["cu"], a["N"], a["T"],
                                 a["H"], a["D"], 1, None)
    assert st == kda.KDA_ERR_INVALID_ARG
    assert detail in L.kda_last_error_detail().decode()


def test_conv_prefill_empty_without_ring_is_a_noop(kda):
    L = kda.lib()
    assert L.kda_shortconv_prefill(None, None, 0x30000, None, None, None, 1, 0, 4, 128, 1, None) == kda.KDA_OK


def test_gated_calls_reject_unknown_gate(kda):
    L = kda.lib()
    st = L.kda_decode_step_gated(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000, 2, 3, 128, 1, 7,
                                 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "gate must be" in L.kda_last_error_detail().decode()
    st = L.kda_shortconv_decode_step_gated(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000, 2, 3,
                                           128, 1, -1, 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "gate must be" in L.kda_last_error_detail().decode()
    st = L.kda_chunk_prefill_gated(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, None, None, 0x60000, None, 1, 100,
                                   4, 128, 64, 1, 3, 1e-6, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "gate must be" in L.kda_last_error_detail().decode()


def test_gate_none_needs_no_g_but_others_do(kda):
    """With no gate, g may be NULL (the argument checks pass on to the next
    pointer); with a per-head gate a NULL g is rejected."""
    L = kda.lib()
    st = L.kda_decode_step_gated(0x10000, 0x20000, 0x30000, None, None, 0x60000, 0x70000, 2, 3, 128, 1,
                                 kda.KDA_GATE_NONE, 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "beta is NULL" in L.kda_last_error_detail().decode()
    st = L.kda_decode_step_gated(0x10000, 0x20000, 0x30000, None, 0x50000, 0x60000, 0x70000, 2, 3, 128, 1,
                                 kda.KDA_GATE_HEAD, 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "g is NULL" in L.kda_last_error_detail().decode()
    st = L.kda_chunk_prefill_gated(0x10000, 0x20000, 0x30000, None, None, None, None, 0x60000, None, 1, 100,
                                   4, 128, 64, 1, kda.KDA_GATE_NONE, 1e-6, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "beta is NULL" in L.kda_last_error_detail().decode()


def test_selftest_rejects_bad_limit(kda):
    L = kda.lib()
    for bad in (0, -5, 3_000_000_000):
        assert L.kda_selftest_bounded_wait(bad, None) == kda.KDA_ERR_INVALID_ARG
        assert "limit_cycles" in L.kda_last_error_detail().decode()


def test_decode_ex_flags(kda):
    """kda_shortconv_decode_step_ex: unknown flag bits are rejected before
    anything else; KDA_DECODE_OVERLAP_PREV passes on to the usual argument
    checks (here a NULL beta)."""
    L = kda.lib()
    st = L.kda_shortconv_decode_step_ex(0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x70000, 2, 3,
                                        128, 1, kda.KDA_GATE_CHANNEL, 1e-6, 4, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "flags" in L.kda_last_error_detail().decode()
    st = L.kda_shortconv_decode_step_ex(0x10000, 0x20000, 0x30000, 0x40000, None, 0x60000, 0x70000, 2, 3,
                                        128, 1, kda.KDA_GATE_CHANNEL, 1e-6, kda.KDA_DECODE_OVERLAP_PREV, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "beta is NULL" in L.kda_last_error_detail().decode()


def test_gated_rmsnorm_argument_checks(kda):
    """kda_gated_rmsnorm: T = 0 is a no-op before any pointer check; bad
    activation, eps, head dim and NULL pointers are rejected without a launch."""
    L = kda.lib()
    assert L.kda_gated_rmsnorm(None, None, None, None, 0, 4, 128, 1, kda.KDA_ACT_SIGMOID, 1e-6, None) == kda.KDA_OK
    st = L.kda_gated_rmsnorm(0x10000, 0x20000, 0x30000, 0x40000, 8, 4, 128, 1, 7, 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "act must be" in L.kda_last_error_detail().decode()
    st = L.kda_gated_rmsnorm(0x10000, 0x20000, 0x30000, 0x40000, 8, 4, 128, 1, kda.KDA_ACT_SILU, -1.0, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "eps" in L.kda_last_error_detail().decode()
    st = L.kda_gated_rmsnorm(0x10000, 0x20000, 0x30000, 0x40000, 8, 4, 48, 1, kda.KDA_ACT_SILU, 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "D must be" in L.kda_last_error_detail().decode()
    st = L.kda_gated_rmsnorm(0x10000, None, 0x30000, 0x40000, 8, 4, 128, 1, kda.KDA_ACT_SIGMOID, 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "gate is NULL" in L.kda_last_error_detail().decode()
    st = L.kda_gated_rmsnorm(0x10000, 0x20000, 0x30008, 0x40000, 8, 4, 128, 1, kda.KDA_ACT_SIGMOID, 1e-6, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "weight is not 16-byte aligned" in L.kda_last_error_detail().decode()


def test_prefill_scan_argument_checks(kda):
    """kda_chunk_prefill_scan: segments out of range and a short workspace are
    rejected (segments = 0 is the automatic count); one segment falls through
    to the ordinary prefill's checks."""
    L = kda.lib()
    args = (0x10000, 0x20000, 0x30000, 0x40000, 0x50000, None, None, 0x60000, 1000, 2, 128, 64, 1,
            kda.KDA_GATE_CHANNEL, 1e-6)
    for bad in (-1, 4097):
        st = L.kda_chunk_prefill_scan(*args, bad, None, 0, None)
        assert st == kda.KDA_ERR_INVALID_ARG and "segments" in L.kda_last_error_detail().decode()
    for segs in (0, 4):
        st = L.kda_chunk_prefill_scan(*args, segs, None, 0, None)
        assert st == kda.KDA_ERR_INVALID_ARG and "workspace too small" in L.kda_last_error_detail().decode()
    need = L.kda_chunk_prefill_scan_workspace_bytes(1000, 2, 128, 64, 4)
    # four fp32 states per segment and head, and a [T, H, D] fp32 output buffer
    assert need >= 4 * 4 * 2 * 128 * 128 * 4 + 1000 * 2 * 128 * 4
    assert L.kda_chunk_prefill_scan_workspace_bytes(1000, 2, 128, 64, 0) > 0
    st = L.kda_chunk_prefill_scan(None, *args[1:], 1, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "q is NULL" in L.kda_last_error_detail().decode()


def test_prefill_epi_argument_checks(kda):
    """kda_chunk_prefill_epi: bad activation, NULL weight and an out_gate that
    aliases out are rejected before any launch."""
    L = kda.lib()
    base = (0x10000, 0x20000, 0x30000, 0x40000, 0x50000, None, None, 0x60000, None, 1, 100, 2, 128, 64, 1,
            kda.KDA_GATE_CHANNEL, 1e-6)
    st = L.kda_chunk_prefill_epi(*base, 0x70000, 0x80000, 5, 1e-6, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "act must be" in L.kda_last_error_detail().decode()
    st = L.kda_chunk_prefill_epi(*base, 0x70000, None, kda.KDA_ACT_SIGMOID, 1e-6, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "norm_weight is NULL" in L.kda_last_error_detail().decode()
    st = L.kda_chunk_prefill_epi(*base, 0x60000, 0x80000, kda.KDA_ACT_SIGMOID, 1e-6, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG and "out_gate must not alias" in L.kda_last_error_detail().decode()


def test_prefill_route_table(kda):
    """Which kernel each prefill shape runs on (no GPU needed): bf16 d in {64, 128} with C in {16, 32, 64}
    on the tcgen05 kernel, fp32 d = 128 with C >= 16 on the tf32 tensor-core kernel, other d = 128 shapes
    on the register-tiled CUDA-core kernel, everything else on the general one; invalid shapes give None."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    route = kda.kda_chunk_prefill_route
    for D in (64, 128):
        for C in (16, 32, 64):
            assert route(D, C, bf) == "prefill_tc_pipe_kernel", (D, C)
    for C in (16, 48, 64):
        assert route(128, C, f32) == "prefill_tf32_kernel", C
    assert route(128, 7, f32) == "prefill_f32_kernel"
    assert route(128, 48, bf) == "prefill_f32_kernel"
    assert route(64, 64, f32) == "prefill_simt_kernel"
    assert route(32, 64, bf) == "prefill_simt_kernel"
    assert route(64, 7, bf) == "prefill_simt_kernel"
    assert route(48, 64, bf) is None and route(128, 0, bf) is None and route(128, 65, f32) is None
    assert route(128, 64, 7) is None


def test_split_plan(kda):
    """The long-sequence split of kda_chunk_prefill_split, planned on the host for a given SM count: only a
    sequence whose chain outlasts the evenly spread work is split (here the 65,536-token one at 8 heads,
    into 1024 // 57 = 17 segments, capped at (152 - 3 x 8) / 8 = 16 so that the three whole sequences'
    CTAs have SMs of their own), never at H not a multiple of 4, never the bench's varlen batch at 96
    heads (its longest chain is shorter than its work per SM); invalid lengths give -1 (an error)."""
    import numpy as np
    cu = np.array([0, 65536, 66036, 69036, 69156], dtype=np.int64)
    seg, n = kda.kda_chunk_prefill_split_plan(cu, 8, 64, sms=152)
    assert n == 1 and list(seg) == [16, 1, 1, 1]
    # the cap is skipped where it would leave fewer than 4 segments (36 whole sequences x 4 heads)
    many = np.concatenate([[0, 65536], 65536 + 64 * np.arange(1, 37)]).astype(np.int64)
    seg, n = kda.kda_chunk_prefill_split_plan(many, 4, 64, sms=152)
    assert n == 1 and seg[0] == 1024 // -(-(1024 + 36) * 4 // 152) and list(seg[1:]) == [1] * 36
    seg, n = kda.kda_chunk_prefill_split_plan(cu, 6, 64, sms=152)
    assert n == 0 and list(seg) == [1, 1, 1, 1]
    varlen = np.cumsum([0, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536]).astype(np.int64)
    assert kda.kda_chunk_prefill_split_plan(varlen, 96, 64, sms=152)[1] == 0
    # one sequence: floor(chunks / max(ceil(chunks * H / SMs), 8)) segments
    seg, n = kda.kda_chunk_prefill_split_plan(np.array([0, 65536], dtype=np.int64), 8, 64, sms=152)
    assert n == 1 and seg[0] == 1024 // -(-1024 * 8 // 152)
    # a sequence of fewer than 4 x 8 chunks stays whole whatever the SM count
    assert kda.kda_chunk_prefill_split_plan(np.array([0, 1984], dtype=np.int64), 4, 64, sms=1024)[1] == 0
    with pytest.raises(kda.KdaError):
        kda.kda_chunk_prefill_split_plan(np.array([0, 10, 5], dtype=np.int64), 8, 64, sms=152)
    with pytest.raises(kda.KdaError):
        kda.kda_chunk_prefill_split_plan(np.array([3, 10], dtype=np.int64), 8, 64, sms=152)


def test_split_rejects_bad_lengths_without_a_gpu(kda):
    import numpy as np
    lib = kda.lib()
    cu = np.array([0, 10, 20], dtype=np.int64)
    st = lib.kda_chunk_prefill_split(None, None, None, None, None, None, None, None, 8, cu.ctypes.data, 2, 21,
                                     8, 128, 64, kda.KDA_BF16, 0, 1e-6, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG
    assert "host_cu_seqlens[N]" in lib.kda_last_error_detail().decode()
    st = lib.kda_chunk_prefill_split(None, None, None, None, None, None, None, None, None, cu.ctypes.data, 2, 20,
                                     8, 128, 64, kda.KDA_BF16, 0, 1e-6, None, 0, None)
    assert st == kda.KDA_ERR_INVALID_ARG
