"""GPU parity of kda_chunk_prefill against the fp64 oracle, through the C ABI."""
import os

import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth
from tests._util import BF16_REL, F32_ATOL, cuda_or_skip, ensure_built, report_rows, to_dev, to_np

pytestmark = pytest.mark.gpu
NCPU = max(1, len(os.sched_getaffinity(0)))


@pytest.fixture(scope="module")
def env():
    torch = cuda_or_skip()
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda
    return torch, kda


def run_prefill(torch, kda, d, bf16, C, init=True, final=True, alias=False, eps=1e-6, use_cu=True):
    dt = torch.bfloat16 if bf16 else torch.float32
    q, k, v = (to_dev(d[n], dt, torch) for n in ("q", "k", "v"))
    g, beta = to_dev(d["g"], torch.float32, torch), to_dev(d["beta"], torch.float32, torch)
    cu = d["cu_seqlens"]
    N, H, D = len(cu) - 1, q.shape[1], q.shape[2]
    tcu = torch.from_numpy(cu).cuda() if use_cu else None
    s0 = to_dev(d["s0"], torch.float32, torch) if (init and d["s0"] is not None) else None
    if alias:
        sf = s0
    elif final:
        sf = torch.full((N, H, D, D), float("nan"), dtype=torch.float32, device="cuda")
    else:
        sf = None
    out = torch.full_like(q, float("nan"))
    kda.kda_chunk_prefill(q, k, v, g, beta, out, initial_state=s0, final_state=sf, cu_seqlens=tcu,
                          chunk_size=C, l2_eps=eps)
    kda.kda_sync_status()
    return to_np(out), (to_np(sf) if sf is not None else None)


def oracle_prefill(d, init=True, eps=1e-6, nthreads=NCPU):
    return oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"],
                             s_init=d["s0"] if init else None, cu_seqlens=d["cu_seqlens"], eps=eps,
                             nthreads=nthreads)


def check(got_o, got_s, ref_o, ref_s, cu, bf16, what=""):
    """fp32: max abs <= 1e-4. bf16: per (sequence, head) relative <= 2e-2."""
    assert np.all(np.isfinite(got_o)), f"{what}: non-finite outputs"
    if got_s is not None:
        assert np.all(np.isfinite(got_s)), f"{what}: non-finite state"
    if not bf16:
        if got_o.size:
            assert np.max(np.abs(got_o - ref_o)) <= F32_ATOL, f"{what}: out abs err {np.max(np.abs(got_o - ref_o))}"
        if got_s is not None:
            assert np.max(np.abs(got_s - ref_s)) <= F32_ATOL, f"{what}: state abs err {np.max(np.abs(got_s - ref_s))}"
        return
    worst = 0.0
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        for h in range(ref_o.shape[1]):
            if b > a:
                den = max(np.max(np.abs(ref_o[a:b, h])), 1e-6)
                worst = max(worst, np.max(np.abs(got_o[a:b, h] - ref_o[a:b, h])) / den)
            if got_s is not None:
                den = max(np.max(np.abs(ref_s[n, h])), 1e-6)
                worst = max(worst, np.max(np.abs(got_s[n, h] - ref_s[n, h])) / den)
    assert worst <= BF16_REL, f"{what}: per-(sequence, head) relative error {worst:.3e}"


VARLEN_SMALL = np.array([0, 5, 5, 70, 133, 200], dtype=np.int64)  # empty and short sequences


@pytest.mark.parametrize("C", [1, 2, 5, 16, 64])
def test_prefill_tiny_workload(env, C):
    """Tiny fp32 recurrence (1 layer, H=2, d=16, T=64, zero state, seed 0)."""
    torch, kda = env
    c = synth.TINY
    d = synth.prefill_inputs(c["seed"], c["T"], c["H"], c["D"], bf16=False)
    o, s = run_prefill(torch, kda, d, False, C)
    ro, rs = oracle_prefill(d)
    check(o, s, ro, rs, d["cu_seqlens"], False, f"C={C}")


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("C", [7, 16, 64])
def test_prefill_varlen_carry_in(env, D, bf16, C):
    torch, kda = env
    d = synth.prefill_inputs(300 + D + C, int(VARLEN_SMALL[-1]), 3, D, bf16, cu_seqlens=VARLEN_SMALL,
                             s0_std=0.5, g_scale=0.1)
    o, s = run_prefill(torch, kda, d, bf16, C)
    ro, rs = oracle_prefill(d)
    check(o, s, ro, rs, d["cu_seqlens"], bf16, f"D={D} bf16={bf16} C={C}")


@pytest.mark.parametrize("bf16", [False, True])
def test_prefill_default_gates_full_head_dim(env, bf16):
    """Workload gate distribution (g = -softplus(N(0,1))), d=128, several chunks."""
    torch, kda = env
    cu = np.array([0, 64, 200, 457], dtype=np.int64)
    d = synth.prefill_inputs(41, 457, 4, 128, bf16, cu_seqlens=cu, s0_std=0.02)
    o, s = run_prefill(torch, kda, d, bf16, 64)
    ro, rs = oracle_prefill(d)
    check(o, s, ro, rs, cu, bf16, "default gates")


@pytest.mark.parametrize("bf16", [False, True])
def test_prefill_unsorted_lengths_launch_order(env, bf16):
    """Sequences in no particular length order (including an empty one and a
    long one in the middle): the longest-first launch order must not change
    which outputs and states belong to which sequence."""
    torch, kda = env
    lengths = [70, 5, 0, 300, 33, 129, 64, 1]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    d = synth.prefill_inputs(58, int(cu[-1]), 2, 128, bf16, cu_seqlens=cu, s0_std=0.3, g_scale=0.1)
    o, s = run_prefill(torch, kda, d, bf16, 64)
    ro, rs = oracle_prefill(d)
    check(o, s, ro, rs, cu, bf16, "unsorted lengths")


def test_prefill_final_state_may_alias_initial(env):
    torch, kda = env
    d = synth.prefill_inputs(51, 200, 2, 64, False, cu_seqlens=VARLEN_SMALL, s0_std=0.3, g_scale=0.1)
    o, s = run_prefill(torch, kda, d, False, 16, alias=True)
    ro, rs = oracle_prefill(d)
    check(o, s, ro, rs, d["cu_seqlens"], False, "alias")


def test_prefill_null_states(env):
    torch, kda = env
    d = synth.prefill_inputs(52, 200, 2, 32, False, cu_seqlens=VARLEN_SMALL, s0_std=0.3)
    o, s = run_prefill(torch, kda, d, False, 16, init=False, final=False)
    ro, _ = oracle_prefill(d, init=False)
    check(o, None, ro, None, d["cu_seqlens"], False, "null states")


@pytest.mark.parametrize("bf16", [False, True])
def test_prefill_extreme_gates(env, bf16):
    """g = -1e4 (memory cleared every token) and beta = 0 (state only decays)."""
    torch, kda = env
    cu = np.array([0, 100, 230], dtype=np.int64)
    d = synth.prefill_inputs(53, 230, 2, 128, bf16, cu_seqlens=cu, s0_std=0.5)
    d1 = dict(d, g=np.full_like(d["g"], -1.0e4))
    o, s = run_prefill(torch, kda, d1, bf16, 64)
    ro, rs = oracle_prefill(d1)
    check(o, s, ro, rs, cu, bf16, "g=-1e4")
    d2 = dict(d, beta=np.zeros_like(d["beta"]), g=d["g"] * 0.01)
    o, s = run_prefill(torch, kda, d2, bf16, 64)
    ro, rs = oracle_prefill(d2)
    check(o, s, ro, rs, cu, bf16, "beta=0")


def test_prefill_all_empty_passes_state_through(env):
    torch, kda = env
    cu = np.zeros(4, dtype=np.int64)
    d = synth.prefill_inputs(54, 0, 2, 16, False, cu_seqlens=cu, s0_std=0.5)
    _, s = run_prefill(torch, kda, d, False, 16)
    assert np.array_equal(s, d["s0"].astype(np.float64))


def test_prefill_then_decode_hand_off(env):
    """Prefill of 70 tokens, then 5 decode steps from its final state, equals
    the recurrence over all 75 tokens."""
    torch, kda = env
    d = synth.prefill_inputs(55, 75, 3, 128, True, s0_std=0.02)
    head = {n: (d[n][:70] if n in ("q", "k", "v", "g", "beta") else d[n]) for n in d}
    head["cu_seqlens"] = np.array([0, 70], dtype=np.int64)
    o1, s1 = run_prefill(torch, kda, head, True, 64)
    st = to_dev(s1, torch.float32, torch)
    outs = []
    for t in range(70, 75):
        q, k, v = (to_dev(d[n][t:t + 1], torch.bfloat16, torch) for n in ("q", "k", "v"))
        g, b = to_dev(d["g"][t:t + 1], torch.float32, torch), to_dev(d["beta"][t:t + 1], torch.float32, torch)
        o = torch.empty_like(q)
        kda.kda_decode_step(q, k, v, g, b, st, o)
        outs.append(to_np(o))
    ro, rs = oracle_prefill(d)
    got = np.concatenate([o1] + outs)
    check(got, to_np(st), ro, rs, d["cu_seqlens"], True, "hand-off")


def test_prefill_split_equals_unsplit(env):
    """prefill(T1) then prefill(T2, carry-in) equals prefill(T1+T2), with
    mild gates so the carried state matters."""
    torch, kda = env
    d = synth.prefill_inputs(56, 300, 2, 128, True, s0_std=0.3, g_scale=0.01)
    a = {n: (d[n][:128] if n in ("q", "k", "v", "g", "beta") else d[n]) for n in d}
    a["cu_seqlens"] = np.array([0, 128], dtype=np.int64)
    o1, s1 = run_prefill(torch, kda, a, True, 64)
    b = {n: (d[n][128:] if n in ("q", "k", "v", "g", "beta") else d[n]) for n in d}
    b["cu_seqlens"] = np.array([0, 172], dtype=np.int64)
    b["s0"] = s1.astype(np.float32)
    o2, s2 = run_prefill(torch, kda, b, True, 64)
    ro, rs = oracle_prefill(d)
    check(np.concatenate([o1, o2]), s2, ro, rs, d["cu_seqlens"], True, "split")


def test_prefill_invalid_cu_seqlens_reported(env):
    torch, kda = env
    d = synth.prefill_inputs(57, 64, 2, 16, False, s0_std=0.5)
    q, k, v = (to_dev(d[n], torch.float32, torch) for n in ("q", "k", "v"))
    g, beta = to_dev(d["g"], torch.float32, torch), to_dev(d["beta"], torch.float32, torch)
    out = torch.zeros_like(q)
    sf = torch.zeros((2, 2, 16, 16), dtype=torch.float32, device="cuda")
    bad = torch.tensor([0, 40, 30], dtype=torch.int64, device="cuda")  # decreasing
    kda.kda_chunk_prefill(q, k, v, g, beta, out, final_state=sf, cu_seqlens=bad, chunk_size=16)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_sync_status()
    assert ei.value.status == kda.KDA_ERR_DEVICE_CHECK
    kda.kda_sync_status()  # cleared


def test_prefill_full_size_4k_workload(env):
    """Chunked prefill at full size: T=4096, H=96, d=128, bf16, C=64, zero
    initial state, fp32 final state; every output and state checked."""
    torch, kda = env
    c = synth.PREFILL
    d = synth.prefill_inputs(c["seed"], c["T"], c["H"], c["D"], bf16=True)
    o, s = run_prefill(torch, kda, d, True, c["C"])
    ro, rs = oracle_prefill(d, init=False)
    check(o, s, ro, rs, d["cu_seqlens"], True, "4K prefill")
    report_rows(o, ro, "4K prefill outputs")


def test_prefill_full_size_varlen_sampled_heads(env):
    """Variable-length prefill at full size (8 sequences of 512..65536
    tokens, 130,560 in all, H=96, d=128, bf16, C=64, non-zero initial
    states): the launch covers all 96 heads; four sampled heads are checked
    against the oracle. Heads not sampled are filled on the device with a
    seeded torch generator (same distributions)."""
    torch, kda = env
    c = synth.VARLEN
    cu = synth.varlen_cu_seqlens()
    T, H, D = int(cu[-1]), c["H"], c["D"]
    heads = [0, 33, 66, 95]
    d = synth.prefill_inputs(c["seed"], T, H, D, bf16=True, cu_seqlens=cu, s0_std=0.02, heads=heads)
    gen = torch.Generator(device="cuda").manual_seed(c["seed"])
    bf = torch.bfloat16

    def fill(shape, dt):
        return torch.randn(shape, generator=gen, device="cuda", dtype=torch.float32).to(dt)
    q, k, v = fill((T, H, D), bf), fill((T, H, D), bf), fill((T, H, D), bf)
    g = -torch.nn.functional.softplus(fill((T, H, D), torch.float32))
    beta = torch.sigmoid(fill((T, H), torch.float32))
    s0 = fill((len(cu) - 1, H, D, D), torch.float32) * 0.02
    hs = torch.tensor(heads, device="cuda")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g)):
        t[:, hs] = to_dev(d[name], t.dtype, torch)
    beta[:, hs] = to_dev(d["beta"], torch.float32, torch)
    s0[:, hs] = to_dev(d["s0"], torch.float32, torch)
    out = torch.empty_like(q)
    sf = torch.empty_like(s0)
    kda.kda_chunk_prefill(q, k, v, g, beta, out, initial_state=s0, final_state=sf,
                          cu_seqlens=torch.from_numpy(cu).cuda(), chunk_size=c["C"])
    kda.kda_sync_status()
    got_o = to_np(out[:, hs])
    got_s = to_np(sf[:, hs])
    ro, rs = oracle_prefill(d)
    check(got_o, got_s, ro, rs, cu, True, "varlen full size")
    report_rows(got_o, ro, "varlen prefill outputs (sampled heads)")


def test_prefill_full_size_4k_fp32(env):
    """The 4K workload's shape in fp32 (T=4096, H=96, d=128, C=64, zero initial state): the register-tiled
    fp32 kernel, every output and final state within the fp32 bar (max abs 1e-4)."""
    torch, kda = env
    c = synth.PREFILL
    d = synth.prefill_inputs(c["seed"], c["T"], c["H"], c["D"], bf16=False)
    o, s = run_prefill(torch, kda, d, False, c["C"])
    ro, rs = oracle_prefill(d, init=False)
    check(o, s, ro, rs, d["cu_seqlens"], False, "4K prefill fp32")
    print(f"4K fp32 prefill: max abs error out {np.max(np.abs(o - ro)):.2e}, state {np.max(np.abs(s - rs)):.2e}")


@pytest.mark.parametrize("gate", ["head", "none"])
@pytest.mark.parametrize("C", [64, 48])
def test_prefill_fp32_gate_forms_d128(env, gate, C):
    """fp32, d=128 (the register-tiled kernel) with a per-head gate or none, carry-in states, ragged chunks."""
    torch, kda = env
    cu = np.array([0, 150, 150, 333], dtype=np.int64)
    d = synth.prefill_inputs(60, 333, 3, 128, False, cu_seqlens=cu, s0_std=0.3, g_scale=0.1)
    if gate == "head":
        gk, go = np.ascontiguousarray(d["g"][..., 0]), np.repeat(d["g"][..., :1], 128, axis=-1)
    else:
        gk, go = None, np.zeros_like(d["g"])
    f32 = torch.float32
    q, k, v = (to_dev(d[n], f32, torch) for n in ("q", "k", "v"))
    out = torch.full_like(q, float("nan"))
    sf = torch.full((3, 3, 128, 128), float("nan"), device="cuda")
    kda.kda_chunk_prefill_gated(q, k, v, None if gk is None else to_dev(gk, f32, torch),
                                to_dev(d["beta"], f32, torch), out, gate=gate,
                                initial_state=to_dev(d["s0"], f32, torch), final_state=sf,
                                cu_seqlens=torch.from_numpy(cu).cuda(), chunk_size=C)
    kda.kda_sync_status()
    ro, rs = oracle.recurrence(d["q"], d["k"], d["v"], go, d["beta"], s_init=d["s0"], cu_seqlens=cu)
    check(to_np(out), to_np(sf), ro, rs, cu, False, f"gate={gate} C={C}")


def test_prefill_fp32_some_chunks_exact(env):
    """fp32, d=128: a gate spike of -200 in one token makes that chunk's decay span exceed the range the
    factored form covers, so that chunk (and only it) takes the exact pairwise path; the others stay on the
    factored one. With mild gates elsewhere the carried state matters across the spike's neighbours."""
    torch, kda = env
    d = synth.prefill_inputs(61, 256, 2, 128, False, s0_std=0.3, g_scale=0.02)
    g = d["g"].copy()
    g[100, 0, :64] = -200.0  # head 0, half the channels, in the second chunk
    d1 = dict(d, g=g)
    o, s = run_prefill(torch, kda, d1, False, 64)
    ro, rs = oracle_prefill(d1)
    check(o, s, ro, rs, d1["cu_seqlens"], False, "spike")


@pytest.mark.parametrize("gate", ["channel", "head", "none"])
@pytest.mark.parametrize("D,C", [(64, 64), (64, 32), (64, 16), (128, 32), (128, 16)])
def test_prefill_bf16_tensor_core_shapes(env, D, C, gate):
    """bf16 shapes the tcgen05 kernel takes besides d=128/C=64: d=64 (its channels 64..127 read as zeros)
    and C=16/32 (64-token chunks inside). Ragged varlen batch with an empty sequence, carry-in states,
    several 64-token chunks per sequence and short last chunks; every gate form; against the oracle."""
    torch, kda = env
    assert kda.kda_chunk_prefill_route(D, C, torch.bfloat16) == "prefill_tc_pipe_kernel"
    cu = np.array([0, 150, 150, 333, 397], dtype=np.int64)
    d = synth.prefill_inputs(700 + D + C, int(cu[-1]), 3, D, True, cu_seqlens=cu, s0_std=0.3, g_scale=0.1)
    bf = torch.bfloat16
    q, k, v = (to_dev(d[n], bf, torch) for n in ("q", "k", "v"))
    if gate == "channel":
        gk, go = to_dev(d["g"], torch.float32, torch), d["g"]
    elif gate == "head":
        gk, go = to_dev(np.ascontiguousarray(d["g"][..., 0]), torch.float32, torch), np.repeat(d["g"][..., :1], D, axis=-1)
    else:
        gk, go = None, np.zeros_like(d["g"])
    out = torch.full_like(q, float("nan"))
    N = len(cu) - 1
    sf = torch.full((N, 3, D, D), float("nan"), device="cuda")
    kda.kda_chunk_prefill_gated(q, k, v, gk, to_dev(d["beta"], torch.float32, torch), out, gate=gate,
                                initial_state=to_dev(d["s0"], torch.float32, torch), final_state=sf,
                                cu_seqlens=torch.from_numpy(cu).cuda(), chunk_size=C)
    kda.kda_sync_status()
    ro, rs = oracle.recurrence(d["q"], d["k"], d["v"], go, d["beta"], s_init=d["s0"], cu_seqlens=cu)
    check(to_np(out), to_np(sf), ro, rs, cu, True, f"D={D} C={C} gate={gate}")


@pytest.mark.parametrize("D,C", [(64, 64), (64, 16), (128, 32)])
def test_prefill_bf16_tensor_core_exact_chunks(env, D, C):
    """The tcgen05 kernel's exact-decay path at the shapes it takes besides d=128/C=64: g = -1e4 on every
    token (each chunk's decay span far past the anchored range; memory cleared every token), and a single
    spike of -200 in one chunk of otherwise mild gates (that chunk alone exact, the carried state mattering
    across it). d=64 runs with the kernel's channels 64..127 zero."""
    torch, kda = env
    assert kda.kda_chunk_prefill_route(D, C, torch.bfloat16) == "prefill_tc_pipe_kernel"
    cu = np.array([0, 100, 230], dtype=np.int64)
    d = synth.prefill_inputs(57 + D + C, 230, 2, D, True, cu_seqlens=cu, s0_std=0.5, g_scale=0.02)
    d1 = dict(d, g=np.full_like(d["g"], -1.0e4))
    o, s = run_prefill(torch, kda, d1, True, C)
    ro, rs = oracle_prefill(d1)
    check(o, s, ro, rs, cu, True, f"D={D} C={C} g=-1e4")
    g2 = d["g"].copy()
    g2[170, 1, : D // 2] = -200.0
    d2 = dict(d, g=g2)
    o, s = run_prefill(torch, kda, d2, True, C)
    ro, rs = oracle_prefill(d2)
    check(o, s, ro, rs, cu, True, f"D={D} C={C} spike")


def test_prefill_full_size_varlen_fp32_sampled_heads(env):
    """The variable-length workload at full size in fp32 (8 sequences of 512..65536 tokens, 130,560 in
    all, H=96, d=128, C=64, non-zero initial states): the tf32 tensor-core kernel walks the 65,536-token
    sequence's 1024 chunks per head. Three sampled heads against the oracle at the fp32 bar (max abs
    1e-4); the other heads are filled on the device with a seeded torch generator (same distributions)."""
    torch, kda = env
    c = synth.VARLEN
    cu = synth.varlen_cu_seqlens()
    T, H, D = int(cu[-1]), c["H"], c["D"]
    assert kda.kda_chunk_prefill_route(D, c["C"], torch.float32) == "prefill_tf32_kernel"
    heads = [1, 48, 94]
    d = synth.prefill_inputs(c["seed"] + 100, T, H, D, bf16=False, cu_seqlens=cu, s0_std=0.02, heads=heads)
    gen = torch.Generator(device="cuda").manual_seed(c["seed"] + 100)
    f32 = torch.float32

    def fill(shape):
        return torch.randn(shape, generator=gen, device="cuda", dtype=f32)
    q, k, v = fill((T, H, D)), fill((T, H, D)), fill((T, H, D))
    g = -torch.nn.functional.softplus(fill((T, H, D)))
    beta = torch.sigmoid(fill((T, H)))
    s0 = fill((len(cu) - 1, H, D, D)) * 0.02
    hs = torch.tensor(heads, device="cuda")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g)):
        t[:, hs] = to_dev(d[name], f32, torch)
    beta[:, hs] = to_dev(d["beta"], f32, torch)
    s0[:, hs] = to_dev(d["s0"], f32, torch)
    out = torch.empty_like(q)
    sf = torch.empty_like(s0)
    kda.kda_chunk_prefill(q, k, v, g, beta, out, initial_state=s0, final_state=sf,
                          cu_seqlens=torch.from_numpy(cu).cuda(), chunk_size=c["C"])
    kda.kda_sync_status()
    got_o, got_s = to_np(out[:, hs]), to_np(sf[:, hs])
    ro, rs = oracle_prefill(d)
    check(got_o, got_s, ro, rs, cu, False, "varlen full size fp32")
    print(f"varlen fp32 (sampled heads): max abs error out {np.max(np.abs(got_o - ro)):.2e}, "
          f"state {np.max(np.abs(got_s - rs)):.2e}")
