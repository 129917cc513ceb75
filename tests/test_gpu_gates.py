"""GPU parity of the gate-form specialisations ("为什么 Kimi K3 敢把 KV Cache 扔掉？
一篇讲透 GPT-2 到 K3 的架构进化", section 7: Gated DeltaNet decays the state by one
factor per head, the delta rule of section 4 not at all) against the fp64
oracle, which takes the per-head gate broadcast over the key channels and no
gate as g = 0 (its pins tie both to those published forms)."""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth
from tests._util import assert_close, cuda_or_skip, ensure_built, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = cuda_or_skip()
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda
    return torch, kda


def _gate_inputs(g_full, gate):
    """(g passed to the kernel, g the oracle sees) for a gate form; the
    per-head gate is channel 0 of the drawn per-channel gate."""
    if gate == "head":
        gh = np.ascontiguousarray(g_full[..., 0])
        return gh, np.repeat(gh[..., None], g_full.shape[-1], axis=-1)
    if gate == "none":
        return None, np.zeros_like(g_full)
    return g_full, g_full


@pytest.mark.parametrize("gate", ["head", "none", "channel"])
@pytest.mark.parametrize("D,bf16", [(16, False), (128, True), (64, True)])
def test_decode_gated_matches_oracle(env, gate, D, bf16):
    torch, kda = env
    B, H = 3, 4
    d = synth.decode_inputs(300 + D, B, H, D, bf16, s0_std=0.5)
    gk, go = _gate_inputs(d["g"], gate)
    dt = torch.bfloat16 if bf16 else torch.float32
    tq, tk, tv = (to_dev(d[n], dt, torch) for n in ("q", "k", "v"))
    ts = to_dev(d["s0"], torch.float32, torch)
    out = torch.empty_like(tq)
    kda.kda_decode_step_gated(tq, tk, tv, None if gk is None else to_dev(gk, torch.float32, torch),
                              to_dev(d["beta"], torch.float32, torch), ts, out, gate=gate)
    torch.cuda.synchronize()
    ro, rs = oracle.decode_step(d["q"], d["k"], d["v"], go, d["beta"], d["s0"])
    assert_close(to_np(out), ro, bf16, (0, 1), "out")
    assert_close(to_np(ts), rs, bf16, (0, 1), "state")


@pytest.mark.parametrize("gate", ["head", "none"])
def test_fused_decode_gated_matches_oracle(env, gate):
    torch, kda = env
    B, H, D = 2, 3, 128
    d = synth.decode_inputs(320, B, H, D, True, s0_std=0.5)
    gk, go = _gate_inputs(d["g"], gate)
    bf = torch.bfloat16
    ring = to_dev(d["ring"], bf, torch)
    ts = to_dev(d["s0"], torch.float32, torch)
    out = torch.empty((B, H, D), dtype=bf, device="cuda")
    kda.kda_shortconv_decode_step_gated(to_dev(d["x"], bf, torch), ring, to_dev(d["w"], torch.float32, torch),
                                        None if gk is None else to_dev(gk, torch.float32, torch),
                                        to_dev(d["beta"], torch.float32, torch), ts, out, gate=gate)
    torch.cuda.synchronize()
    y, rring = oracle.shortconv_step(d["x"], d["ring"], d["w"])
    ro, rs = oracle.decode_step(y[:, 0], y[:, 1], y[:, 2], go, d["beta"], d["s0"])
    assert_close(to_np(out), ro, True, (0, 1), "out")
    assert_close(to_np(ts), rs, True, (0, 1), "state")
    np.testing.assert_array_equal(to_np(ring), rring)


LENS = [130, 64, 1, 0, 77]


@pytest.mark.parametrize("gate", ["head", "none"])
@pytest.mark.parametrize("D,C,bf16", [(128, 64, True), (32, 16, False), (128, 32, True)])
def test_prefill_gated_matches_oracle(env, gate, D, C, bf16):
    """bf16 with D = 128 and C = 64 runs the tensor-core kernel; the others the
    CUDA-core kernel."""
    torch, kda = env
    cu = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int64)
    T, H, N = int(cu[-1]), 2, len(LENS)
    p = synth.prefill_inputs(330 + D + C, T, H, D, bf16, cu_seqlens=cu, s0_std=0.02)
    gk, go = _gate_inputs(p["g"], gate)
    dt = torch.bfloat16 if bf16 else torch.float32
    q, k, v = (to_dev(p[n], dt, torch) for n in ("q", "k", "v"))
    out = torch.empty_like(q)
    sf = torch.empty((N, H, D, D), dtype=torch.float32, device="cuda")
    kda.kda_chunk_prefill_gated(q, k, v, None if gk is None else to_dev(gk, torch.float32, torch),
                                to_dev(p["beta"], torch.float32, torch), out, gate=gate,
                                initial_state=to_dev(p["s0"], torch.float32, torch), final_state=sf,
                                cu_seqlens=torch.tensor(cu, device="cuda"), chunk_size=C)
    torch.cuda.synchronize()
    kda.kda_sync_status()
    ro, rs = oracle.recurrence(p["q"], p["k"], p["v"], go, p["beta"], s_init=p["s0"], cu_seqlens=cu)
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        if b > a:
            assert_close(to_np(out)[a:b], ro[a:b], bf16, (1,), f"out seq {n}")
    assert_close(to_np(sf), rs, bf16, (0, 1), "final state")


def test_prefill_head_gate_strong_decay_exact_chunks(env):
    """Per-head gates of -3 per token give a decay span of about 190 over a
    chunk, beyond the anchored factorisation: those chunks take the exact
    pairwise path (tensor-core kernel)."""
    torch, kda = env
    T, H, D = 200, 2, 128
    p = synth.prefill_inputs(340, T, H, D, True, s0_std=0.5)
    gh = np.full((T, H), -3.0, np.float32)
    gh[::7] = -0.01  # mixed
    bf = torch.bfloat16
    q, k, v = (to_dev(p[n], bf, torch) for n in ("q", "k", "v"))
    out = torch.empty_like(q)
    sf = torch.empty((1, H, D, D), dtype=torch.float32, device="cuda")
    kda.kda_chunk_prefill_gated(q, k, v, to_dev(gh, torch.float32, torch), to_dev(p["beta"], torch.float32, torch),
                                out, gate="head", initial_state=to_dev(p["s0"], torch.float32, torch),
                                final_state=sf)
    torch.cuda.synchronize()
    go = np.repeat(gh[..., None], D, axis=-1)
    ro, rs = oracle.recurrence(p["q"], p["k"], p["v"], go, p["beta"], s_init=p["s0"])
    assert_close(to_np(out), ro, True, (1,), "out")
    assert_close(to_np(sf), rs, True, (0, 1), "final state")


@pytest.mark.parametrize("gate", ["head", "none"])
def test_prefill_gated_full_size_sampled_heads(env, gate):
    """4096 tokens x 96 heads (bf16, d = 128, C = 64) in the launch the
    benchmark times; three heads checked against the oracle."""
    torch, kda = env
    T, H, D = synth.PREFILL["T"], synth.PREFILL["H"], synth.PREFILL["D"]
    p = synth.prefill_inputs(synth.PREFILL["seed"], T, H, D, True)
    gk, _ = _gate_inputs(p["g"], gate)
    bf = torch.bfloat16
    q, k, v = (to_dev(p[n], bf, torch) for n in ("q", "k", "v"))
    out = torch.empty_like(q)
    sf = torch.empty((1, H, D, D), dtype=torch.float32, device="cuda")
    kda.kda_chunk_prefill_gated(q, k, v, None if gk is None else to_dev(gk, torch.float32, torch),
                                to_dev(p["beta"], torch.float32, torch), out, gate=gate, final_state=sf)
    torch.cuda.synchronize()
    heads = [0, 50, 95]
    sub = {n: p[n][:, heads] for n in ("q", "k", "v", "g", "beta")}
    _, go = _gate_inputs(sub["g"], gate)
    ro, rs = oracle.recurrence(sub["q"], sub["k"], sub["v"], go, sub["beta"], nthreads=8)
    assert_close(to_np(out)[:, heads], ro, True, (1,), "out")
    assert_close(to_np(sf)[:, heads], rs, True, (0, 1), "final state")


@pytest.mark.parametrize("gate", ["channel", "head", "none"])
@pytest.mark.parametrize("bf16", [True, False])
def test_fused_decode_many_heads_sampled(env, gate, bf16):
    """A launch of many waves (12 sequences x 128 heads, d = 128) takes the
    register-resident fused kernel (small launches take the shared-memory
    staged one); eight sampled (sequence, head) units are checked against the
    oracle, including the rings they shift."""
    torch, kda = env
    B, H, D = 12, 128, 128
    d = synth.decode_inputs(360 + bf16, B, H, D, bf16, s0_std=0.5)
    gk, go = _gate_inputs(d["g"], gate)
    dt = torch.bfloat16 if bf16 else torch.float32
    ring = to_dev(d["ring"], dt, torch)
    ts = to_dev(d["s0"], torch.float32, torch)
    out = torch.empty((B, H, D), dtype=dt, device="cuda")
    kda.kda_shortconv_decode_step_gated(to_dev(d["x"], dt, torch), ring, to_dev(d["w"], torch.float32, torch),
                                        None if gk is None else to_dev(gk, torch.float32, torch),
                                        to_dev(d["beta"], torch.float32, torch), ts, out, gate=gate)
    torch.cuda.synchronize()
    got_o, got_s, got_r = to_np(out), to_np(ts), to_np(ring)
    for (bb, hh) in [(0, 0), (0, 127), (5, 64), (11, 1), (11, 126), (3, 33), (7, 99), (9, 77)]:
        x1 = d["x"][bb:bb + 1, :, hh:hh + 1]
        r1 = d["ring"][bb:bb + 1, :, hh:hh + 1]
        w1 = d["w"][:, hh:hh + 1]
        y, rr = oracle.shortconv_step(x1, r1, w1)
        ro, rs = oracle.decode_step(y[:, 0], y[:, 1], y[:, 2], go[bb:bb + 1, hh:hh + 1],
                                    d["beta"][bb:bb + 1, hh:hh + 1], d["s0"][bb:bb + 1, hh:hh + 1])
        assert_close(got_o[bb:bb + 1, hh:hh + 1], ro, bf16, (0, 1), f"out {(bb, hh)}")
        assert_close(got_s[bb:bb + 1, hh:hh + 1], rs, bf16, (0, 1), f"state {(bb, hh)}")
        np.testing.assert_array_equal(got_r[bb, :, hh], rr[0, :, 0])


@pytest.mark.parametrize("D,bf16", [(16, False), (128, True)])
def test_fused_decode_overlap_flag(env, D, bf16):
    """kda_shortconv_decode_step_ex with KDA_DECODE_OVERLAP_PREV, two layers
    launched alternately for three steps (each launch follows the other
    layer's, so the promise holds): D=16 takes the register kernel, D=128 the
    shared-memory-staged one with a programmatic dependent launch. Every
    result equals the plain launch bit for bit, and layer 0 matches the fp64
    oracle over the three steps."""
    torch, kda = env
    B, H, steps = 2, 3, 3
    dt = torch.bfloat16 if bf16 else torch.float32
    layers = [synth.decode_inputs(700 + 10 * l + D, B, H, D, bf16, s0_std=0.5) for l in range(2)]
    xs = [[synth.decode_inputs(800 + 10 * l + t, B, H, D, bf16)["x"] for t in range(steps)] for l in range(2)]

    def run(overlap):
        st = [to_dev(d["s0"], torch.float32, torch) for d in layers]
        rg = [to_dev(d["ring"], dt, torch) for d in layers]
        outs = []
        for t in range(steps):
            for l, d in enumerate(layers):
                out = torch.empty((B, H, D), dtype=dt, device="cuda")
                kda.kda_shortconv_decode_step_ex(to_dev(xs[l][t], dt, torch), rg[l], to_dev(d["w"], torch.float32, torch),
                                                 to_dev(d["g"], torch.float32, torch),
                                                 to_dev(d["beta"], torch.float32, torch), st[l], out,
                                                 overlap_prev=overlap)
                outs.append(out)
        torch.cuda.synchronize()
        return [to_np(o) for o in outs], [to_np(s) for s in st], [to_np(r) for r in rg]

    o1, s1, r1 = run(True)
    o0, s0, r0 = run(False)
    for a, b in zip(o1 + s1 + r1, o0 + s0 + r0):
        np.testing.assert_array_equal(a, b)
    d = layers[0]
    S, ring = d["s0"], d["ring"]
    for t in range(steps):
        y, ring = oracle.shortconv_step(xs[0][t], ring, d["w"])
        ro, S = oracle.decode_step(y[:, 0], y[:, 1], y[:, 2], d["g"], d["beta"], S)
        assert_close(o1[2 * t], ro, bf16, (0, 1), f"out step {t}")
    assert_close(s1[0], S, bf16, (0, 1), "state")
