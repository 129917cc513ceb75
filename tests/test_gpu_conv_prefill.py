"""GPU parity of kda_shortconv_prefill (the width-4 short conv + SiLU over a
packed prompt batch, with the 3-token ring handed to decode) against the
fp64 oracle, through the C ABI ("KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta
Attention线性注意力原理剖析", section "KDA 递推公式先衰减再差分")."""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth
from tests._util import BF16_REL, F32_ATOL, assert_close, cuda_or_skip, ensure_built, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = cuda_or_skip()
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda
    return torch, kda


def _run(torch, kda, x, w, bf16, ring_in=None, cu=None, want_ring=True):
    dt = torch.bfloat16 if bf16 else torch.float32
    T, _, H, D = x.shape
    N = 1 if cu is None else len(cu) - 1
    tx = to_dev(x, dt, torch)
    tw = to_dev(w, torch.float32, torch)
    tr = None if ring_in is None else to_dev(ring_in, dt, torch)
    ty = torch.full((3, T, H, D), float("nan"), dtype=dt, device="cuda")
    tro = torch.full((N, 3, H, 3, D), float("nan"), dtype=dt, device="cuda") if want_ring else None
    tcu = None if cu is None else torch.tensor(np.asarray(cu, np.int64), device="cuda")
    kda.kda_shortconv_prefill(tx, tw, ty, ring_in=tr, ring_out=tro, cu_seqlens=tcu)
    torch.cuda.synchronize()
    kda.kda_sync_status()
    return to_np(ty), (to_np(tro) if want_ring else None)


def _check_y(y, ref, bf16, what="y"):
    """fp32: max abs error; bf16: each element within the bf16 rounding of
    the reference (half an ulp, 2^-9 relative) plus a small absolute slack."""
    assert np.all(np.isfinite(y)), f"{what}: non-finite"
    if bf16:
        bound = 2.0 ** -8 * np.abs(ref) + 1e-6
        bad = np.abs(y - ref) > bound
        assert not bad.any(), f"{what}: {bad.sum()} elements beyond bf16 rounding"
    else:
        assert np.max(np.abs(y - ref)) <= F32_ATOL


LENS = [0, 1, 2, 3, 64, 65, 130, 5, 0, 61]  # empty, shorter than the window, tile-crossing, ragged


@pytest.mark.parametrize("D", [16, 128])
@pytest.mark.parametrize("bf16", [False, True])
def test_conv_prefill_varlen_matches_oracle(env, D, bf16):
    torch, kda = env
    cu = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int64)
    T, H, N = int(cu[-1]), 3, len(LENS)
    d = synth.conv_prefill_inputs(40 + D, T, H, D, N, bf16)
    y, ro = _run(torch, kda, d["x"], d["w"], bf16, ring_in=d["ring"], cu=cu)
    ry, rro = oracle.shortconv_seq(d["x"], d["w"], ring_in=d["ring"], cu_seqlens=cu)
    _check_y(y, ry, bf16)
    np.testing.assert_array_equal(ro, rro)  # pure data movement: bit-exact


@pytest.mark.parametrize("bf16", [False, True])
def test_conv_prefill_one_sequence_zero_history(env, bf16):
    torch, kda = env
    T, H, D = 200, 2, 64
    d = synth.conv_prefill_inputs(7, T, H, D, 1, bf16)
    y, _ = _run(torch, kda, d["x"], d["w"], bf16, want_ring=False)
    ry, _ = oracle.shortconv_seq(d["x"], d["w"])
    _check_y(y, ry, bf16)


def test_conv_prefill_no_tokens_passes_ring_through(env):
    torch, kda = env
    d = synth.conv_prefill_inputs(8, 0, 2, 32, 3, True)
    _, ro = _run(torch, kda, d["x"], d["w"], True, ring_in=d["ring"], cu=[0, 0, 0, 0])
    np.testing.assert_array_equal(ro, d["ring"].astype(np.float64))
    _, ro = _run(torch, kda, d["x"], d["w"], True, ring_in=None, cu=[0, 0, 0, 0])
    assert np.all(ro == 0.0)


def test_conv_prefill_hands_ring_to_decode_step(env):
    """Prefill conv over T tokens, then one kda_shortconv_step on its ring,
    equals the oracle's conv over T + 1 tokens (last output and ring)."""
    torch, kda = env
    T, H, D, bf16 = 77, 2, 128, True
    d = synth.conv_prefill_inputs(9, T + 1, H, D, 1, bf16)
    dt = torch.bfloat16
    tx = to_dev(d["x"][:T], dt, torch)
    tw = to_dev(d["w"], torch.float32, torch)
    ty = torch.empty((3, T, H, D), dtype=dt, device="cuda")
    ring = torch.empty((1, 3, H, 3, D), dtype=dt, device="cuda")
    kda.kda_shortconv_prefill(tx, tw, ty, ring_in=to_dev(d["ring"], dt, torch), ring_out=ring)
    ys = torch.empty((3, 1, H, D), dtype=dt, device="cuda")
    kda.kda_shortconv_step(to_dev(d["x"][T:T + 1], dt, torch), ring, tw, ys)
    torch.cuda.synchronize()
    ry, rro = oracle.shortconv_seq(d["x"], d["w"], ring_in=d["ring"])
    _check_y(to_np(ys)[:, 0], ry[:, T], bf16, "decode step after prefill")
    np.testing.assert_array_equal(to_np(ring), rro)


def test_conv_prefill_feeds_chunk_prefill(env):
    """The projection-major output is directly the q, k, v of
    kda_chunk_prefill: conv then chunked prefill equals the oracle's conv
    then token recurrence."""
    torch, kda = env
    lens = [70, 3, 130]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, H, D, N = int(cu[-1]), 2, 128, len(lens)
    d = synth.conv_prefill_inputs(10, T, H, D, N, True)
    p = synth.prefill_inputs(10, T, H, D, True, cu_seqlens=cu)
    dt = torch.bfloat16
    ty = torch.empty((3, T, H, D), dtype=dt, device="cuda")
    tcu = torch.tensor(cu, device="cuda")
    kda.kda_shortconv_prefill(to_dev(d["x"], dt, torch), to_dev(d["w"], torch.float32, torch), ty,
                              ring_in=to_dev(d["ring"], dt, torch), cu_seqlens=tcu)
    out = torch.empty((T, H, D), dtype=dt, device="cuda")
    sf = torch.empty((N, H, D, D), dtype=torch.float32, device="cuda")
    kda.kda_chunk_prefill(ty[0], ty[1], ty[2], to_dev(p["g"], torch.float32, torch),
                          to_dev(p["beta"], torch.float32, torch), out, final_state=sf, cu_seqlens=tcu)
    torch.cuda.synchronize()
    ry, _ = oracle.shortconv_seq(d["x"], d["w"], ring_in=d["ring"], cu_seqlens=cu)
    # the API hands the prefill bf16 q, k, v: round the oracle's conv output the same way
    yq = synth.bf16_round(ry.astype(np.float32)).astype(np.float64)
    ro, rs = oracle.recurrence(yq[0], yq[1], yq[2], p["g"], p["beta"], cu_seqlens=cu)
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        assert_close(to_np(out)[a:b], ro[a:b], True, (1,), f"out seq {n}")
    assert_close(to_np(sf), rs, True, (0, 1), "final state")


def test_conv_prefill_full_size_sampled_heads(env):
    """4096 tokens x 96 heads x 128 channels (bf16) in the launch the
    benchmark times; three heads checked in full against the oracle."""
    torch, kda = env
    T, H, D = synth.PREFILL["T"], synth.PREFILL["H"], synth.PREFILL["D"]
    full = synth.conv_prefill_inputs(11, T, H, D, 1, True)
    y, ro = _run(torch, kda, full["x"], full["w"], True, ring_in=full["ring"])
    for h in (0, 47, 95):
        ry, rro = oracle.shortconv_seq(full["x"][:, :, h:h + 1], full["w"][:, h:h + 1],
                                       ring_in=full["ring"][:, :, h:h + 1])
        _check_y(y[:, :, h:h + 1], ry, True, f"head {h}")
        np.testing.assert_array_equal(ro[:, :, h:h + 1], rro)


def test_conv_prefill_invalid_seqlens_reported(env):
    torch, kda = env
    d = synth.conv_prefill_inputs(12, 100, 1, 16, 2, False)
    dt = torch.float32
    ty = torch.zeros((3, 100, 1, 16), dtype=dt, device="cuda")
    bad = torch.tensor([0, 120, 100], dtype=torch.int64, device="cuda")  # decreasing
    kda.kda_shortconv_prefill(to_dev(d["x"], dt, torch), to_dev(d["w"], dt, torch), ty, cu_seqlens=bad)
    torch.cuda.synchronize()
    with pytest.raises(kda.KdaError):
        kda.kda_sync_status()
    kda.kda_sync_status()  # the word is cleared once reported
