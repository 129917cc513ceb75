"""GPU parity of the output epilogue, kda_gated_rmsnorm (gated RMSNorm of the
attention output: "KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力
原理剖析", section "相关源码与文档导航"; "为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透
GPT-2 到 K3 的架构进化", section 6), against the fp64 oracle, one row per
(token, head)."""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth
from tests._util import assert_close, cuda_or_skip, ensure_built, report_rows, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = cuda_or_skip()
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda
    return torch, kda


@pytest.mark.parametrize("act", ["sigmoid", "silu"])
@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("bf16", [False, True])
def test_gated_rmsnorm_matches_oracle(env, act, D, bf16):
    """37 tokens x 3 heads (not a multiple of the rows a warp takes), rows of
    magnitudes spread over e^+-3, one row all zero."""
    torch, kda = env
    T, H = 37, 3
    d = synth.epilogue_inputs(10 + D, T, H, D, bf16)
    d["o"][5, 1] = 0.0
    dt = torch.bfloat16 if bf16 else torch.float32
    o, gate = to_dev(d["o"], dt, torch), to_dev(d["gate"], dt, torch)
    y = torch.empty_like(o)
    kda.kda_gated_rmsnorm(o, gate, to_dev(d["weight"], torch.float32, torch), y, act=act, eps=1e-6)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(d["o"], d["gate"], d["weight"], eps=1e-6, act=act)
    assert_close(to_np(y), ref, bf16, (0, 1), "y")
    assert np.all(to_np(y)[5, 1] == 0.0)


def test_gated_rmsnorm_in_place_and_zero_eps(env):
    """y may be o; with eps = 0 a zero row still gives zeros."""
    torch, kda = env
    T, H, D = 9, 5, 128
    d = synth.epilogue_inputs(77, T, H, D, False)
    d["o"][3] = 0.0
    o = to_dev(d["o"], torch.float32, torch)
    kda.kda_gated_rmsnorm(o, to_dev(d["gate"], torch.float32, torch), to_dev(d["weight"], torch.float32, torch), o,
                          act="silu", eps=0.0)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(d["o"], d["gate"], d["weight"], eps=0.0, act="silu")
    assert_close(to_np(o), ref, False, (0, 1), "y in place")
    assert np.all(to_np(o)[3] == 0.0)


def test_gated_rmsnorm_full_size_sampled_rows(env):
    """The prefill output size, T=4096, H=96, D=128, bf16: 64 sampled rows
    against the oracle (each row is independent, so a sample is exact)."""
    torch, kda = env
    T, H, D = 4096, 96, 128
    d = synth.epilogue_inputs(5, T, H, D, True)
    o, gate = to_dev(d["o"], torch.bfloat16, torch), to_dev(d["gate"], torch.bfloat16, torch)
    y = torch.empty_like(o)
    kda.kda_gated_rmsnorm(o, gate, to_dev(d["weight"], torch.float32, torch), y)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    ts, hs = rng.integers(0, T, 64), rng.integers(0, H, 64)
    got = to_np(y)[ts, hs]
    ref = oracle.gated_rmsnorm(d["o"][ts, hs], d["gate"][ts, hs], d["weight"])
    assert_close(got[:, None], ref[:, None], True, (0, 1), "sampled rows")


def _epi_ref(p, d, act, s0=None):
    ro, rs = oracle.recurrence(p["q"], p["k"], p["v"], p["g"], p["beta"], s_init=s0, cu_seqlens=p["cu_seqlens"])
    return oracle.gated_rmsnorm(ro, d["gate"], d["weight"], eps=1e-6, act=act), rs


@pytest.mark.parametrize("act", ["sigmoid", "silu"])
def test_prefill_epi_tensor_core(env, act):
    """kda_chunk_prefill_epi on the tensor-core path (bf16, d=128, C=64). Two
    sequences of 130 and 77 tokens (short last chunks), carry-in states."""
    torch, kda = env
    H, D = 2, 128
    cu = np.array([0, 130, 207], dtype=np.int64)
    T = int(cu[-1])
    p = synth.prefill_inputs(41, T, H, D, True, cu_seqlens=cu, s0_std=0.05)
    d = synth.epilogue_inputs(42, T, H, D, True)
    bf = torch.bfloat16
    q, k, v = (to_dev(p[n], bf, torch) for n in "qkv")
    out = torch.empty_like(q)
    sf = torch.empty((2, H, D, D), device="cuda")
    kda.kda_chunk_prefill_epi(q, k, v, to_dev(p["g"], torch.float32, torch), to_dev(p["beta"], torch.float32, torch),
                              out, to_dev(d["gate"], bf, torch), to_dev(d["weight"], torch.float32, torch), act=act,
                              initial_state=to_dev(p["s0"], torch.float32, torch), final_state=sf,
                              cu_seqlens=torch.from_numpy(cu).cuda())
    torch.cuda.synchronize()
    kda.kda_sync_status()
    ref, rs = _epi_ref(p, d, act, p["s0"])
    assert_close(to_np(out), ref, True, (1,), "out")
    assert_close(to_np(sf), rs, True, (0, 1), "final state")


def test_prefill_epi_cuda_core(env):
    """fp32, d=16, C=16: the CUDA-core prefill, then the epilogue pass."""
    torch, kda = env
    T, H, D = 90, 3, 16
    p = synth.prefill_inputs(43, T, H, D, False)
    d = synth.epilogue_inputs(44, T, H, D, False)
    q, k, v = (to_dev(p[n], torch.float32, torch) for n in "qkv")
    out = torch.empty_like(q)
    kda.kda_chunk_prefill_epi(q, k, v, to_dev(p["g"], torch.float32, torch), to_dev(p["beta"], torch.float32, torch),
                              out, to_dev(d["gate"], torch.float32, torch), to_dev(d["weight"], torch.float32, torch),
                              act="silu", chunk_size=16)
    torch.cuda.synchronize()
    ref, _ = _epi_ref(p, d, "silu")
    assert_close(to_np(out), ref, False, (1,), "out")


def test_prefill_epi_full_size_matches_separate_pass(env):
    """The 4K workload (T=4096, H=96): the one-call prefill with epilogue
    against the prefill followed by kda_gated_rmsnorm, every row."""
    torch, kda = env
    T, H, D = 4096, 96, 128
    p = synth.prefill_inputs(2, T, H, D, True)
    d = synth.epilogue_inputs(45, T, H, D, True)
    bf = torch.bfloat16
    q, k, v = (to_dev(p[n], bf, torch) for n in "qkv")
    g, b = to_dev(p["g"], torch.float32, torch), to_dev(p["beta"], torch.float32, torch)
    gate, w = to_dev(d["gate"], bf, torch), to_dev(d["weight"], torch.float32, torch)
    fused, plain = torch.empty_like(q), torch.empty_like(q)
    kda.kda_chunk_prefill_epi(q, k, v, g, b, fused, gate, w)
    kda.kda_chunk_prefill(q, k, v, g, b, plain)
    sep = torch.empty_like(q)
    kda.kda_gated_rmsnorm(plain, gate, w, sep)
    torch.cuda.synchronize()
    assert_close(to_np(fused), to_np(sep), True, (1,), "fused vs separate")


# ------------------------------------------------------------------------------------------------------------
# The epilogue fused into the fused conv + decode step (kda_shortconv_decode_step_epi): the oracle's conv
# (fp64) feeds its recurrence, whose output goes through the oracle's gated RMSNorm.
NCPU = max(1, len(__import__("os").sched_getaffinity(0)))


def _gate_arg(d, gate):
    """The decode inputs' g in the layout of `gate` (per-head gate: channel 0 of the drawn per-channel gate)."""
    if gate == "head":
        gh = np.ascontiguousarray(d["g"][..., 0])
        return gh, np.repeat(gh[..., None], d["g"].shape[-1], axis=-1)
    if gate == "none":
        return None, np.zeros_like(d["g"])
    return d["g"], d["g"]


def _oracle_decode_epi(d, e, act, gate="channel"):
    ry, rring = oracle.shortconv_step(d["x"], d["ring"], d["w"])
    _, g_or = _gate_arg(d, gate)
    ro, rs = oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], g_or, d["beta"], d["s0"], nthreads=NCPU)
    B, H, D = ro.shape
    ryo = oracle.gated_rmsnorm(ro.reshape(B, H, D), e["gate"], e["weight"], eps=1e-6, act=act)
    return ryo, rs, rring


def _gpu_decode_epi(torch, kda, d, e, bf16, act, gate="channel", overlap=False):
    dt = torch.bfloat16 if bf16 else torch.float32
    B, _, H, D = d["x"].shape
    tx, tr = to_dev(d["x"], dt, torch), to_dev(d["ring"], dt, torch)
    tw, tb = to_dev(d["w"], torch.float32, torch), to_dev(d["beta"], torch.float32, torch)
    g_in, _ = _gate_arg(d, gate)
    tg = to_dev(g_in, torch.float32, torch) if g_in is not None else None
    ts = to_dev(d["s0"], torch.float32, torch)
    og, nw = to_dev(e["gate"], dt, torch), to_dev(e["weight"], torch.float32, torch)
    y = torch.full((B, H, D), float("nan"), dtype=dt, device="cuda")
    kda.kda_shortconv_decode_step_epi(tx, tr, tw, tg, tb, ts, og, nw, y, gate=gate, act=act, overlap_prev=overlap)
    torch.cuda.synchronize()
    return to_np(y), to_np(ts), to_np(tr)


@pytest.mark.parametrize("act", ["sigmoid", "silu"])
@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("bf16", [False, True])
def test_fused_decode_epilogue_matches_oracle(env, act, D, bf16):
    """3 sequences x 5 heads (D = 128 takes the shared-memory-staged kernel at this size): y, state and ring."""
    torch, kda = env
    d = synth.decode_inputs(500 + D, 3, 5, D, bf16, s0_std=0.5)
    e = synth.epilogue_inputs(600 + D, 3, 5, D, bf16)
    y, st, ring = _gpu_decode_epi(torch, kda, d, e, bf16, act)
    ry, rs, rring = _oracle_decode_epi(d, e, act)
    assert_close(y, ry, bf16, (0, 1), "y")
    assert_close(st, rs, bf16, (0, 1), "state")
    assert np.max(np.abs(st - rs)) <= 1e-4
    assert np.array_equal(ring, rring)


@pytest.mark.parametrize("gate", ["head", "none"])
@pytest.mark.parametrize("overlap", [False, True])
def test_fused_decode_epilogue_gate_forms(env, gate, overlap):
    """Per-head and no gate, plain and programmatic-dependent launches (the staged kernel: B=8, H=12)."""
    torch, kda = env
    d = synth.decode_inputs(700, 8, 12, 128, True, s0_std=0.3)
    e = synth.epilogue_inputs(701, 8, 12, 128, True)
    y, st, ring = _gpu_decode_epi(torch, kda, d, e, True, "sigmoid", gate=gate, overlap=overlap)
    ry, rs, rring = _oracle_decode_epi(d, e, "sigmoid", gate=gate)
    assert_close(y, ry, True, (0, 1), "y")
    assert_close(st, rs, True, (0, 1), "state")
    assert np.array_equal(ring, rring)


@pytest.mark.parametrize("act", ["sigmoid", "silu"])
@pytest.mark.parametrize("gate,overlap", [("channel", False), ("head", True), ("none", False)])
def test_fused_decode_epilogue_acts_gates(env, act, gate, overlap):
    """The staged d = 128 kernel with the epilogue, both activations, on 16 sequences x 5 heads (bf16) in
    three gate and launch forms."""
    torch, kda = env
    d = synth.decode_inputs(720, 16, 5, 128, True, s0_std=0.3)
    e = synth.epilogue_inputs(721, 16, 5, 128, True)
    y, st, ring = _gpu_decode_epi(torch, kda, d, e, True, act, gate=gate, overlap=overlap)
    ry, rs, rring = _oracle_decode_epi(d, e, act, gate=gate)
    assert_close(y, ry, True, (0, 1), "y")
    assert_close(st, rs, True, (0, 1), "state")
    assert np.array_equal(ring, rring)


@pytest.mark.parametrize("act", ["sigmoid", "silu"])
def test_fused_decode_epilogue_1248_heads(env, act):
    """The staged d = 128 kernel with the epilogue on 13 sequences x 96 heads (bf16), against the oracle."""
    torch, kda = env
    d = synth.decode_inputs(730, 13, 96, 128, True, s0_std=0.3)
    e = synth.epilogue_inputs(731, 13, 96, 128, True)
    y, st, ring = _gpu_decode_epi(torch, kda, d, e, True, act)
    ry, rs, rring = _oracle_decode_epi(d, e, act)
    assert_close(y, ry, True, (0, 1), "y")
    assert_close(st, rs, True, (0, 1), "state")
    assert np.array_equal(ring, rring)


def test_fused_decode_epilogue_zero_output_row(env):
    """A head whose output is exactly zero (zero state, zero v: o = 0) maps to zeros with norm eps = 0, as the
    oracle's reading fixes; the other heads are unaffected."""
    torch, kda = env
    d = synth.decode_inputs(710, 2, 3, 64, False, s0_std=None)
    d["x"][0, 2, 1] = 0.0  # v projection of (sequence 0, head 1): conv of zeros plus a zero ring
    d["ring"][0, 2, 1] = 0.0
    e = synth.epilogue_inputs(711, 2, 3, 64, False)
    dt = torch.float32
    tx, tr = to_dev(d["x"], dt, torch), to_dev(d["ring"], dt, torch)
    ts = to_dev(d["s0"], dt, torch)
    y = torch.full((2, 3, 64), float("nan"), dtype=dt, device="cuda")
    kda.kda_shortconv_decode_step_epi(tx, tr, to_dev(d["w"], dt, torch), to_dev(d["g"], dt, torch),
                                      to_dev(d["beta"], dt, torch), ts, to_dev(e["gate"], dt, torch),
                                      to_dev(e["weight"], dt, torch), y, norm_eps=0.0)
    torch.cuda.synchronize()
    ry, _ = oracle.shortconv_step(d["x"], d["ring"], d["w"])
    ro, _ = oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], d["g"], d["beta"], d["s0"])
    ref = oracle.gated_rmsnorm(ro, e["gate"], e["weight"], eps=0.0)
    got = to_np(y)
    assert np.all(got[0, 1] == 0.0) and np.all(ref[0, 1] == 0.0)
    assert_close(got, ref, False, (0, 1), "y")


def test_fused_decode_epilogue_full_size(env):
    """The decode workload at full size (B=64, H=96, d=128, bf16: the staged kernel), every unit against
    the oracle."""
    torch, kda = env
    c = synth.DECODE
    d = synth.decode_inputs(c["seed"], c["B"], c["H"], c["D"], True)
    e = synth.epilogue_inputs(c["seed"] + 50, c["B"], c["H"], c["D"], True)
    y, st, ring = _gpu_decode_epi(torch, kda, d, e, True, "sigmoid")
    ry, rs, rring = _oracle_decode_epi(d, e, "sigmoid")
    r = assert_close(y, ry, True, (0, 1), "y")
    assert_close(st, rs, True, (0, 1), "state")
    assert np.array_equal(ring, rring)
    print(f"fused decode + epilogue, full size: worst per-head relative error {r:.3e}")
    report_rows(y, ry, "fused decode + epilogue, full size")
