"""GPU parity of kda_decode_step and kda_shortconv_step against the fp64
oracle, through the C ABI (ctypes binding)."""
import os

import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth
from tests._util import assert_close, cuda_or_skip, ensure_built, report_rows, to_dev, to_np

pytestmark = pytest.mark.gpu
NCPU = max(1, len(os.sched_getaffinity(0)))


@pytest.fixture(scope="module")
def env():
    torch = cuda_or_skip()
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda
    return torch, kda


def _gpu_decode(torch, kda, q, k, v, g, beta, s0, bf16, eps=1e-6):
    dt = torch.bfloat16 if bf16 else torch.float32
    tq, tk, tv = (to_dev(a, dt, torch) for a in (q, k, v))
    tg, tb = to_dev(g, torch.float32, torch), to_dev(beta, torch.float32, torch)
    ts = to_dev(s0, torch.float32, torch)
    out = torch.empty_like(tq)
    kda.kda_decode_step(tq, tk, tv, tg, tb, ts, out, l2_eps=eps)
    torch.cuda.synchronize()
    return to_np(out), to_np(ts)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("B,H", [(1, 1), (3, 5)])
def test_decode_matches_oracle(env, D, bf16, B, H):
    torch, kda = env
    d = synth.decode_inputs(100 + D + B, B, H, D, bf16, s0_std=0.5)
    out, st = _gpu_decode(torch, kda, d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"], bf16)
    ro, rs = oracle.decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"])
    assert_close(out, ro, bf16, (0, 1), "out")
    assert_close(st, rs, bf16, (0, 1), "state")
    # the state stays fp32 in both paths: hold it to the fp32 bar as well
    assert np.max(np.abs(st - rs)) <= 1e-4


def test_decode_tiny_recurrence_as_single_steps(env):
    """The tiny fp32 workload (H=2, d=16, T=64, zero state, seed 0) run as
    64 consecutive decode steps equals the oracle's token recurrence."""
    torch, kda = env
    p = synth.prefill_inputs(synth.TINY["seed"], 64, 2, 16, bf16=False)
    st = np.zeros((1, 2, 16, 16), np.float32)
    ts = to_dev(st, torch.float32, torch)
    outs = []
    for t in range(64):
        q, k, v, g = (to_dev(p[n][t:t + 1], torch.float32, torch) for n in ("q", "k", "v", "g"))
        b = to_dev(p["beta"][t:t + 1], torch.float32, torch)
        o = torch.empty_like(q)
        kda.kda_decode_step(q, k, v, g, b, ts, o)
        outs.append(o)
    torch.cuda.synchronize()
    out = np.concatenate([to_np(o) for o in outs])
    ro, rs = oracle.recurrence(p["q"], p["k"], p["v"], p["g"], p["beta"])
    assert_close(out, ro, False, (), "out")
    assert_close(to_np(ts), rs, False, (), "state")


def test_decode_worked_example(env):
    """Delta-rule worked example (k=[1,3], v=[2,4] then [0,1], beta=1, g=0),
    padded to D=16: the GPU reads back the newest value."""
    torch, kda = env
    D = 16
    q = np.zeros((1, 1, D), np.float32); q[0, 0, :2] = [1, 3]
    v1 = np.zeros_like(q); v1[0, 0, :2] = [2, 4]
    v2 = np.zeros_like(q); v2[0, 0, :2] = [0, 1]
    g = np.zeros_like(q); b = np.ones((1, 1), np.float32)
    s = np.zeros((1, 1, D, D), np.float32)
    o1, s1 = _gpu_decode(torch, kda, q, q, v1, g, b, s, False, eps=0.0)
    o2, _ = _gpu_decode(torch, kda, q, q, v2, g, b, s1, False, eps=0.0)
    np.testing.assert_allclose(o1[0, 0, :2], [2, 4], atol=1e-6)
    np.testing.assert_allclose(o2[0, 0, :2], [0, 1], atol=1e-6)


def test_decode_beta_zero_no_gate_keeps_state_bitwise(env):
    torch, kda = env
    d = synth.decode_inputs(7, 2, 3, 128, False, s0_std=1.0)
    beta = np.zeros_like(d["beta"]); g = np.zeros_like(d["g"])
    _, st = _gpu_decode(torch, kda, d["q"], d["k"], d["v"], g, beta, d["s0"], False)
    assert np.array_equal(st, d["s0"].astype(np.float64))


def test_decode_very_negative_gate_clears(env):
    torch, kda = env
    d = synth.decode_inputs(8, 2, 3, 64, True, s0_std=1.0)
    g = np.full_like(d["g"], -1.0e4)
    out, st = _gpu_decode(torch, kda, d["q"], d["k"], d["v"], g, d["beta"], d["s0"], True)
    ro, rs = oracle.decode_step(d["q"], d["k"], d["v"], g, d["beta"], d["s0"])
    assert_close(out, ro, True, (0, 1), "out")
    assert np.max(np.abs(st - rs)) <= 1e-5


def test_decode_zero_vectors_and_eps(env):
    """A zero q and k with eps=0 normalise to zero (no NaN); eps enters the norm."""
    torch, kda = env
    d = synth.decode_inputs(9, 2, 2, 32, False, s0_std=0.5)
    q = d["q"].copy(); k = d["k"].copy()
    q[0, 0] = 0; k[0, 0] = 0
    for eps in (0.0, 1.0):
        out, st = _gpu_decode(torch, kda, q, k, d["v"], d["g"], d["beta"], d["s0"], False, eps=eps)
        ro, rs = oracle.decode_step(q, k, d["v"], d["g"], d["beta"], d["s0"], eps=eps)
        assert_close(out, ro, False, (), f"out eps={eps}")
        assert_close(st, rs, False, (), f"state eps={eps}")


def test_decode_full_size_workload(env):
    """Decode workload at full size: B=64 sequences, H=96, d=128, bf16
    q/k/v, state ~ N(0, 0.02^2); every output and state checked."""
    torch, kda = env
    c = synth.DECODE
    d = synth.decode_inputs(c["seed"], c["B"], c["H"], c["D"], True)
    out, st = _gpu_decode(torch, kda, d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"], True)
    ro, rs = oracle.decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["s0"], nthreads=NCPU)
    assert_close(out, ro, True, (0, 1), "out")
    assert_close(st, rs, True, (0, 1), "state")


# ---------------------------------------------------------------- short conv
def _gpu_conv(torch, kda, x, ring, w, bf16):
    dt = torch.bfloat16 if bf16 else torch.float32
    tx, tr = to_dev(x, dt, torch), to_dev(ring, dt, torch)
    tw = to_dev(w, torch.float32, torch)
    B, _, H, D = x.shape
    y = torch.empty((3, B, H, D), dtype=dt, device="cuda")
    kda.kda_shortconv_step(tx, tr, tw, y)
    torch.cuda.synchronize()
    return to_np(y), to_np(tr)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("bf16", [False, True])
def test_shortconv_matches_oracle(env, D, bf16):
    torch, kda = env
    d = synth.decode_inputs(200 + D, 3, 5, D, bf16)
    y, ring = _gpu_conv(torch, kda, d["x"], d["ring"], d["w"], bf16)
    ry, rring = oracle.shortconv_step(d["x"], d["ring"], d["w"])
    ry = ry.transpose(1, 0, 2, 3)  # oracle is [B,3,H,D]; the library writes [3,B,H,D]
    if bf16:
        # one rounding of the fp32 result to bf16
        assert np.all(np.abs(y - ry) <= 4e-3 * np.abs(ry) + 1e-5)
    else:
        assert np.max(np.abs(y - ry)) <= 1e-5
    assert np.array_equal(ring, rring)  # the ring only moves stored values


@pytest.mark.parametrize("B,H,D,bf16", [(70, 2, 128, True), (33, 3, 128, False), (37, 2, 64, False),
                                        (300, 2, 16, True), (130, 1, 16, False), (1, 1, 128, True)])
def test_shortconv_tiles(env, B, H, D, bf16):
    """Batches spanning several sequence tiles of the conv step's CTAs (32 KB of x and ring per
    tile: 32 bf16 or 16 fp32 sequences at d=128, up to 256 at d=16), each with a ragged last
    tile, and a single sequence."""
    torch, kda = env
    d = synth.decode_inputs(300 + B, B, H, D, bf16, s0_std=None)
    y, ring = _gpu_conv(torch, kda, d["x"], d["ring"], d["w"], bf16)
    ry, rring = oracle.shortconv_step(d["x"], d["ring"], d["w"])
    ry = ry.transpose(1, 0, 2, 3)
    if bf16:
        assert np.all(np.abs(y - ry) <= 4e-3 * np.abs(ry) + 1e-5)
    else:
        assert np.max(np.abs(y - ry)) <= 1e-5
    assert np.array_equal(ring, rring)


@pytest.mark.parametrize("graph", [False, True])
def test_shortconv_steps_back_to_back(env, graph):
    """Six conv steps on one ring, launched back to back with no host synchronisation between
    them (and, in the second case, captured into a CUDA graph and replayed). Each launch may
    start while the one before it drains, so each must still read the ring that one wrote:
    the outputs of every step and the final ring match the oracle run step by step."""
    torch, kda = env
    steps, B, H, D = 6, 64, 8, 128
    d = synth.decode_inputs(400, B, H, D, True, s0_std=None)
    xs = [synth.decode_inputs(410 + i, B, H, D, True, s0_std=None)["x"] for i in range(steps)]
    tr = to_dev(d["ring"], torch.bfloat16, torch)
    tw = to_dev(d["w"], torch.float32, torch)
    txs = [to_dev(x, torch.bfloat16, torch) for x in xs]
    ys = [torch.zeros((3, B, H, D), dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    torch.cuda.synchronize()
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps):
                kda.kda_shortconv_step(txs[i], tr, tw, ys[i], stream=torch.cuda.current_stream())
        tr.copy_(to_dev(d["ring"], torch.bfloat16, torch))  # capture ran nothing; start from the ring
        torch.cuda.synchronize()
        g.replay()
    else:
        for i in range(steps):
            kda.kda_shortconv_step(txs[i], tr, tw, ys[i])
    torch.cuda.synchronize()
    kda.kda_sync_status()
    ring = d["ring"]
    for i in range(steps):
        ry, ring = oracle.shortconv_step(xs[i], ring, d["w"])
        ry = ry.transpose(1, 0, 2, 3)
        assert np.all(np.abs(to_np(ys[i]) - ry) <= 4e-3 * np.abs(ry) + 1e-5), i
    assert np.array_equal(to_np(tr), ring)


def test_shortconv_then_decode_full_size(env):
    """The decode workload end to end: short conv (bf16 ring of 3 tokens x
    3 projections x 128 per head, SiLU) feeding the decode step, against the
    oracle's conv (fp64, then stored as bf16 like the library's y) feeding
    the oracle's recurrence."""
    torch, kda = env
    c = synth.DECODE
    d = synth.decode_inputs(c["seed"], c["B"], c["H"], c["D"], True)
    tx, tr = to_dev(d["x"], torch.bfloat16, torch), to_dev(d["ring"], torch.bfloat16, torch)
    tw = to_dev(d["w"], torch.float32, torch)
    tg, tb = to_dev(d["g"], torch.float32, torch), to_dev(d["beta"], torch.float32, torch)
    ts = to_dev(d["s0"], torch.float32, torch)
    y = torch.empty((3,) + tuple(d["q"].shape), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(y[0])
    kda.kda_shortconv_step(tx, tr, tw, y)
    kda.kda_decode_step(y[0], y[1], y[2], tg, tb, ts, out)
    torch.cuda.synchronize()
    ry, rring = oracle.shortconv_step(d["x"], d["ring"], d["w"])
    # y is stored in the call's dtype (bf16) by definition of the API; the
    # oracle's decode takes its own conv output rounded to that storage type
    ry = synth.bf16_round(ry.astype(np.float32))
    ro, rs = oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], d["g"], d["beta"], d["s0"], nthreads=NCPU)
    assert_close(to_np(out), ro, True, (0, 1), "out")
    assert_close(to_np(ts), rs, True, (0, 1), "state")
    assert np.array_equal(to_np(tr), rring)


# ---------------------------------------------------------------- fused short conv + decode
def _oracle_conv_decode(d, s0=None, ring=None, x=None):
    ring = d["ring"] if ring is None else ring
    x = d["x"] if x is None else x
    ry, rring = oracle.shortconv_step(x, ring, d["w"])
    ro, rs = oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], d["g"], d["beta"], d["s0"] if s0 is None else s0,
                                nthreads=NCPU)
    return ro, rs, rring


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("bf16", [False, True])
def test_fused_conv_decode_matches_oracle(env, D, bf16):
    """kda_shortconv_decode_step keeps the post-conv q, k, v in fp32, so it is
    compared with the oracle's conv (fp64, unrounded) feeding its recurrence."""
    torch, kda = env
    d = synth.decode_inputs(300 + D, 3, 5, D, bf16, s0_std=0.5)
    dt = torch.bfloat16 if bf16 else torch.float32
    tx, tr = to_dev(d["x"], dt, torch), to_dev(d["ring"], dt, torch)
    tw, tg, tb = (to_dev(d[n], torch.float32, torch) for n in ("w", "g", "beta"))
    ts = to_dev(d["s0"], torch.float32, torch)
    out = torch.empty((3, 5, D), dtype=dt, device="cuda")
    kda.kda_shortconv_decode_step(tx, tr, tw, tg, tb, ts, out)
    torch.cuda.synchronize()
    ro, rs, rring = _oracle_conv_decode(d)
    assert_close(to_np(out), ro, bf16, (0, 1), "out")
    assert_close(to_np(ts), rs, bf16, (0, 1), "state")
    assert np.max(np.abs(to_np(ts) - rs)) <= 1e-4
    assert np.array_equal(to_np(tr), rring)


@pytest.mark.parametrize("gate", ["channel", "head", "none"])
@pytest.mark.parametrize("bf16,overlap", [(True, False), (False, False), (True, True)])
def test_fused_conv_decode_gate_forms(env, gate, bf16, overlap):
    """The staged d = 128 kernel on an odd batch (17 sequences x 3 heads) in every gate form, plain and
    programmatic-dependent launches, against the oracle's conv feeding its recurrence."""
    torch, kda = env
    B, H, D = 17, 3, 128
    d = synth.decode_inputs(820, B, H, D, bf16, s0_std=0.5)
    if gate == "head":
        g_in = np.ascontiguousarray(d["g"][..., 0])
        g_or = np.repeat(g_in[..., None], D, axis=-1)
    elif gate == "none":
        g_in, g_or = None, np.zeros_like(d["g"])
    else:
        g_in = g_or = d["g"]
    dt = torch.bfloat16 if bf16 else torch.float32
    tx, tr = to_dev(d["x"], dt, torch), to_dev(d["ring"], dt, torch)
    tw, tb = to_dev(d["w"], torch.float32, torch), to_dev(d["beta"], torch.float32, torch)
    tg = to_dev(g_in, torch.float32, torch) if g_in is not None else None
    ts = to_dev(d["s0"], torch.float32, torch)
    out = torch.full((B, H, D), float("nan"), dtype=dt, device="cuda")
    kda.kda_shortconv_decode_step_ex(tx, tr, tw, tg, tb, ts, out, gate=gate, overlap_prev=overlap)
    torch.cuda.synchronize()
    kda.kda_sync_status()
    ry, rring = oracle.shortconv_step(d["x"], d["ring"], d["w"])
    ro, rs = oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], g_or, d["beta"], d["s0"], nthreads=NCPU)
    assert_close(to_np(out), ro, bf16, (0, 1), "out")
    assert_close(to_np(ts), rs, bf16, (0, 1), "state")
    assert np.max(np.abs(to_np(ts) - rs)) <= 1e-4
    assert np.array_equal(to_np(tr), rring)


@pytest.mark.parametrize("gate", ["channel", "head", "none"])
def test_fused_conv_decode_1248_heads(env, gate):
    """The staged d = 128 kernel on 13 sequences x 96 heads (1248 CTAs: 2.7 waves at three per SM on 152
    SMs) in every gate form, two steps in a row (ring and state carried), against the oracle."""
    torch, kda = env
    B, H, D = 13, 96, 128
    d = synth.decode_inputs(840, B, H, D, True, s0_std=0.3)
    if gate == "head":
        g_in = np.ascontiguousarray(d["g"][..., 0])
        g_or = np.repeat(g_in[..., None], D, axis=-1)
    elif gate == "none":
        g_in, g_or = None, np.zeros_like(d["g"])
    else:
        g_in = g_or = d["g"]
    bf = torch.bfloat16
    tr = to_dev(d["ring"], bf, torch)
    tw, tb = to_dev(d["w"], torch.float32, torch), to_dev(d["beta"], torch.float32, torch)
    tg = to_dev(g_in, torch.float32, torch) if g_in is not None else None
    ts = to_dev(d["s0"], torch.float32, torch)
    xs = [d["x"], synth.bf16_round(np.random.default_rng(841).standard_normal(d["x"].shape).astype(np.float32))]
    ring, st = d["ring"], d["s0"]
    for i, xi in enumerate(xs):
        out = torch.full((B, H, D), float("nan"), dtype=bf, device="cuda")
        kda.kda_shortconv_decode_step_gated(to_dev(xi, bf, torch), tr, tw, tg, tb, ts, out, gate=gate)
        torch.cuda.synchronize()
        kda.kda_sync_status()
        ry, ring = oracle.shortconv_step(xi, ring, d["w"])
        ro, st = oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], g_or, d["beta"], st, nthreads=NCPU)
        assert_close(to_np(out), ro, True, (0, 1), f"out step {i}")
        assert_close(to_np(ts), st, True, (0, 1), f"state step {i}")
        assert np.array_equal(to_np(tr), ring)


def test_fused_decode_after_a_kernel_that_writes_the_state(env):
    """Every d = 128 fused step is a programmatic dependent launch that may start while the kernel
    before it drains, touching only L2 prefetches until that kernel completes. Here a torch kernel
    halves the state (and shifts the ring's newest slot) between two fused steps on the same state;
    the second step must see those writes: both steps against the oracle doing the same."""
    torch, kda = env
    B, H, D = 16, 96, 128
    d = synth.decode_inputs(860, B, H, D, True, s0_std=0.3)
    bf = torch.bfloat16
    tx, tr = to_dev(d["x"], bf, torch), to_dev(d["ring"], bf, torch)
    tw, tg, tb = (to_dev(d[n], torch.float32, torch) for n in ("w", "g", "beta"))
    ts = to_dev(d["s0"], torch.float32, torch)
    outs = [torch.empty((B, H, D), dtype=bf, device="cuda") for _ in range(2)]
    kda.kda_shortconv_decode_step(tx, tr, tw, tg, tb, ts, outs[0])
    ts.mul_(0.5)                         # a plain torch kernel writing the state
    tr[:, :, :, 2].mul_(-1.0)            # and the ring's newest slot
    kda.kda_shortconv_decode_step(tx, tr, tw, tg, tb, ts, outs[1])
    torch.cuda.synchronize()
    kda.kda_sync_status()
    ry, ring = oracle.shortconv_step(d["x"], d["ring"], d["w"])
    ro0, st = oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], d["g"], d["beta"], d["s0"], nthreads=NCPU)
    st = st * 0.5
    ring = ring.copy()
    ring[:, :, :, 2] = -ring[:, :, :, 2]
    ry, ring = oracle.shortconv_step(d["x"], ring, d["w"])
    ro1, st = oracle.decode_step(ry[:, 0], ry[:, 1], ry[:, 2], d["g"], d["beta"], st, nthreads=NCPU)
    assert_close(to_np(outs[0]), ro0, True, (0, 1), "out step 0")
    assert_close(to_np(outs[1]), ro1, True, (0, 1), "out step 1")
    assert_close(to_np(ts), st, True, (0, 1), "state")
    assert np.array_equal(to_np(tr), ring)


def test_fused_conv_decode_consecutive_steps(env):
    """Four fused steps in a row (ring and state carried) against the oracle
    run step by step on the same inputs."""
    torch, kda = env
    B, H, D = 2, 3, 64
    d = synth.decode_inputs(77, B, H, D, True, s0_std=0.3, g_scale=0.1)
    xs = [synth.bf16_round(np.random.default_rng(100 + i).standard_normal(d["x"].shape).astype(np.float32))
          for i in range(4)]
    bf = torch.bfloat16
    tr = to_dev(d["ring"], bf, torch)
    tw, tg, tb = (to_dev(d[n], torch.float32, torch) for n in ("w", "g", "beta"))
    ts = to_dev(d["s0"], torch.float32, torch)
    ring, st = d["ring"], d["s0"]
    for i in range(4):
        out = torch.empty((B, H, D), dtype=bf, device="cuda")
        kda.kda_shortconv_decode_step(to_dev(xs[i], bf, torch), tr, tw, tg, tb, ts, out)
        ro, st, ring = _oracle_conv_decode(d, s0=st, ring=ring, x=xs[i])
        torch.cuda.synchronize()
        assert_close(to_np(out), ro, True, (0, 1), f"out step {i}")
        assert_close(to_np(ts), st, True, (0, 1), f"state step {i}")
        assert np.array_equal(to_np(tr), ring)


def test_fused_conv_decode_full_size(env):
    """Decode workload at full size through the fused call: B=64, H=96, d=128."""
    torch, kda = env
    c = synth.DECODE
    d = synth.decode_inputs(c["seed"], c["B"], c["H"], c["D"], True)
    bf = torch.bfloat16
    tx, tr = to_dev(d["x"], bf, torch), to_dev(d["ring"], bf, torch)
    tw, tg, tb = (to_dev(d[n], torch.float32, torch) for n in ("w", "g", "beta"))
    ts = to_dev(d["s0"], torch.float32, torch)
    out = torch.empty((c["B"], c["H"], c["D"]), dtype=bf, device="cuda")
    kda.kda_shortconv_decode_step(tx, tr, tw, tg, tb, ts, out)
    torch.cuda.synchronize()
    ro, rs, rring = _oracle_conv_decode(d)
    assert_close(to_np(out), ro, True, (0, 1), "out")
    assert_close(to_np(ts), rs, True, (0, 1), "state")
    assert np.array_equal(to_np(tr), rring)
    report_rows(to_np(out), ro, "fused decode outputs, full size")
