"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something fixed outside itself: the
pages' worked example, closed forms, published alternative forms of the same
update, invariants, a library convolution, or brute-force equivalences. A
plausible slip in the oracle (dropped term, wrong sign, transposed operand,
decay after instead of before the delta step, missing normalisation) fails
at least one of them.

Sources: "KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析"
("KDA 递推公式先衰减再差分" section) and "为什么 Kimi K3 敢把 KV Cache 扔掉？
一篇讲透 GPT-2 到 K3 的架构进化" (sections 4-7).
"""
import os

import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    return vals


def _unit(x):
    return x / np.linalg.norm(x)


def _rand(seed, T, H, D, g_scale=1.0, s0_std=None, cu=None):
    d = synth.prefill_inputs(seed, T, H, D, bf16=False, cu_seqlens=cu,
                             s0_std=s0_std, g_scale=g_scale)
    # float64 copies so that the numpy-side closed forms run in fp64
    return {key: (val.astype(np.float64) if isinstance(val, np.ndarray) and val.dtype == np.float32
                  else val) for key, val in d.items()}


# ---------------------------------------------------------------- worked example
def _worked_example_inputs(D):
    gold = _golden("worked_example_delta_rule.txt")
    k = np.zeros((2, 1, D))
    k[:, 0, :2] = gold["k"]
    v = np.zeros((2, 1, D))
    v[0, 0, :2] = gold["v1"]
    v[1, 0, :2] = gold["v2"]
    g = np.zeros((2, 1, D))
    beta = np.ones((2, 1))
    return gold, k.copy(), k, v, g, beta


@pytest.mark.parametrize("D", [2, 16])
def test_worked_example_delta_reads_back_new_value(D):
    """Page 2 section 4: the delta rule replaces the value under a repeated
    key; D=16 pads with zero channels, which must not change anything."""
    gold, q, k, v, g, beta = _worked_example_inputs(D)
    out, sf = oracle.recurrence(q, k, v, g, beta, eps=0.0)
    np.testing.assert_allclose(out[0, 0, :2], gold["delta_readout_1"], atol=1e-14, rtol=0)
    np.testing.assert_allclose(out[1, 0, :2], gold["delta_readout_2"], atol=1e-14, rtol=0)
    assert np.all(out[:, 0, 2:] == 0)
    kh = _unit(gold["k"])
    np.testing.assert_allclose(sf[0, 0, :2, :2], np.outer(kh, gold["v2"]), atol=1e-14, rtol=0)


def test_worked_example_additive_memory_is_contaminated():
    """The contrast the page draws: plain additive memory (no delta
    correction) reads back v1+v2 under the same key, unlike the oracle."""
    gold, q, k, v, g, beta = _worked_example_inputs(2)
    kh = _unit(gold["k"])
    s_add = np.outer(kh, gold["v1"]) + np.outer(kh, gold["v2"])
    np.testing.assert_allclose(s_add.T @ kh, gold["additive_readout_2"], atol=1e-14, rtol=0)
    out, _ = oracle.recurrence(q, k, v, g, beta, eps=0.0)
    assert not np.allclose(out[1, 0], gold["additive_readout_2"])


# ---------------------------------------------------------------- closed forms
def test_beta_zero_and_no_gate_leave_state_bitwise():
    d = _rand(11, 20, 3, 8, s0_std=0.5)
    beta = np.zeros_like(d["beta"])
    g = np.zeros_like(d["g"])
    out, sf = oracle.recurrence(d["q"], d["k"], d["v"], g, beta, s_init=d["s0"], eps=0.0)
    s0 = d["s0"].astype(np.float64)
    assert np.array_equal(sf, s0)
    for t in range(20):
        for h in range(3):
            qh = _unit(d["q"][t, h].astype(np.float64))
            np.testing.assert_allclose(out[t, h], s0[0, h].T @ qh, atol=1e-13, rtol=0)


def test_beta_zero_pure_decay_closed_form():
    """beta=0: S_t = Diag(exp(G_t)) S_0 with G_t the running sum of g."""
    d = _rand(12, 16, 2, 8, s0_std=0.5)
    beta = np.zeros_like(d["beta"])
    out, sf = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], beta, s_init=d["s0"], eps=0.0)
    G = np.cumsum(d["g"].astype(np.float64), axis=0)
    s0 = d["s0"].astype(np.float64)
    for h in range(2):
        np.testing.assert_allclose(sf[0, h], np.exp(G[-1, h])[:, None] * s0[0, h], rtol=1e-12)
        for t in range(16):
            qh = _unit(d["q"][t, h].astype(np.float64))
            np.testing.assert_allclose(out[t, h], (np.exp(G[t, h])[:, None] * s0[0, h]).T @ qh,
                                       atol=1e-13, rtol=0)


def test_very_negative_gate_clears_memory():
    """Page 2 section 6: alpha=0 empties the memory. g=-1e4 makes exp(g)=0,
    so S_t = beta_t k_t v_t^T and o_t = beta_t (k_t.q_t) v_t."""
    d = _rand(13, 12, 2, 8, s0_std=1.0)
    g = np.full_like(d["g"], -1.0e4)
    out, sf = oracle.recurrence(d["q"], d["k"], d["v"], g, d["beta"], s_init=d["s0"], eps=0.0)
    for t in range(12):
        for h in range(2):
            qh = _unit(d["q"][t, h].astype(np.float64))
            kh = _unit(d["k"][t, h].astype(np.float64))
            b = float(d["beta"][t, h])
            np.testing.assert_allclose(out[t, h], b * (kh @ qh) * d["v"][t, h], atol=1e-13, rtol=0)
    kh = _unit(d["k"][-1, 1].astype(np.float64))
    np.testing.assert_allclose(sf[0, 1], d["beta"][-1, 1] * np.outer(kh, d["v"][-1, 1]), atol=1e-14, rtol=0)


def test_orthonormal_keys_store_exact_associations():
    """With no decay, beta=1 and orthonormal keys the delta rule stores
    S = sum_i k_i v_i^T, and querying with k_i returns v_i exactly
    (page 2 section 4: finite memory edited without interference)."""
    D = 8
    rng = np.random.default_rng(5)
    Q, _ = np.linalg.qr(rng.standard_normal((D, D)))
    keys = Q.T  # rows orthonormal
    vals = rng.standard_normal((D, D))
    T = 2 * D
    q = np.zeros((T, 1, D)); k = np.zeros((T, 1, D)); v = np.zeros((T, 1, D))
    beta = np.ones((T, 1))
    k[:D, 0] = keys; v[:D, 0] = vals; q[:D, 0] = keys
    # read phase: beta=0 leaves the state unchanged; query each key
    k[D:, 0] = keys; q[D:, 0] = keys; beta[D:] = 0.0
    out, sf = oracle.recurrence(q, k, v, np.zeros((T, 1, D)), beta, eps=0.0)
    np.testing.assert_allclose(sf[0, 0], keys.T @ vals, atol=1e-12, rtol=0)
    np.testing.assert_allclose(out[D:, 0], vals, atol=1e-12, rtol=0)


# ---------------------------------------------------------------- other published forms
def test_no_gate_matches_deltanet_read_diff_write():
    """g=0 is the ungated delta rule of page 2 section 4 (read the stored
    value, take the difference, write it back), written here in that page's
    transposed d_v x d_k form S_t = S_{t-1} - v_old k^T + v_new k^T with
    v_new = beta v + (1-beta) v_old."""
    d = _rand(21, 24, 2, 8, s0_std=0.3)
    g = np.zeros_like(d["g"])
    out, sf = oracle.recurrence(d["q"], d["k"], d["v"], g, d["beta"], s_init=d["s0"], eps=0.0)
    for h in range(2):
        M = d["s0"][0, h].astype(np.float64).T  # d_v x d_k
        for t in range(24):
            kh = _unit(d["k"][t, h].astype(np.float64))
            qh = _unit(d["q"][t, h].astype(np.float64))
            b = float(d["beta"][t, h])
            v_old = M @ kh
            v_new = b * d["v"][t, h] + (1 - b) * v_old
            M = M - np.outer(v_old, kh) + np.outer(v_new, kh)
            np.testing.assert_allclose(out[t, h], M @ qh, atol=1e-12, rtol=0)
        np.testing.assert_allclose(sf[0, h], M.T, atol=1e-12, rtol=0)


def test_scalar_gate_matches_gated_deltanet():
    """A gate equal across key channels is Gated DeltaNet, page 2 section 7:
    S_t = S_{t-1} alpha_t (I - beta_t k k^T) + beta_t v k^T (d_v x d_k)."""
    d = _rand(22, 24, 2, 8, s0_std=0.3)
    g = np.repeat(d["g"][:, :, :1], 8, axis=2)
    out, sf = oracle.recurrence(d["q"], d["k"], d["v"], g, d["beta"], s_init=d["s0"], eps=0.0)
    I = np.eye(8)
    for h in range(2):
        M = d["s0"][0, h].astype(np.float64).T
        for t in range(24):
            kh = _unit(d["k"][t, h].astype(np.float64))
            qh = _unit(d["q"][t, h].astype(np.float64))
            b = float(d["beta"][t, h]); alpha = np.exp(float(g[t, h, 0]))
            M = M * alpha @ (I - b * np.outer(kh, kh)) + b * np.outer(d["v"][t, h], kh)
            np.testing.assert_allclose(out[t, h], M @ qh, atol=1e-12, rtol=0)
        np.testing.assert_allclose(sf[0, h], M.T, atol=1e-12, rtol=0)


def test_per_channel_gate_matches_kimi_product_form():
    """Page 2 section 7, Kimi Linear in product form:
    S_t = (I - beta_t k k^T) Diag(alpha_t) S_{t-1} + beta_t k v^T; o_t = S_t^T q."""
    d = _rand(23, 24, 2, 8, s0_std=0.3)
    out, sf = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"], eps=0.0)
    I = np.eye(8)
    for h in range(2):
        S = d["s0"][0, h].astype(np.float64)
        for t in range(24):
            kh = _unit(d["k"][t, h].astype(np.float64))
            qh = _unit(d["q"][t, h].astype(np.float64))
            b = float(d["beta"][t, h])
            S = (I - b * np.outer(kh, kh)) @ np.diag(np.exp(d["g"][t, h].astype(np.float64))) @ S \
                + b * np.outer(kh, d["v"][t, h])
            np.testing.assert_allclose(out[t, h], S.T @ qh, atol=1e-12, rtol=0)
        np.testing.assert_allclose(sf[0, h], S, atol=1e-12, rtol=0)


def test_decay_applies_before_delta():
    """The page on WARP stresses that the decay comes before the delta step.
    Decay-after would give S_t = Diag(a)(S + beta k (v - S^T k)^T); this
    test checks the oracle differs from that variant and matches the
    decay-first closed form for one step from a random state."""
    D = 6
    rng = np.random.default_rng(3)
    S0 = rng.standard_normal((1, 1, D, D))
    q = rng.standard_normal((1, 1, D)); k = rng.standard_normal((1, 1, D))
    v = rng.standard_normal((1, 1, D)); g = -rng.random((1, 1, D)) * 2
    beta = np.array([[0.7]])
    out, sf = oracle.recurrence(q, k, v, g, beta, s_init=S0, eps=0.0)
    a = np.exp(g[0, 0]); kh = _unit(k[0, 0])
    Sd = a[:, None] * S0[0, 0]
    first = Sd + 0.7 * np.outer(kh, v[0, 0] - Sd.T @ kh)
    after = a[:, None] * (S0[0, 0] + 0.7 * np.outer(kh, v[0, 0] - S0[0, 0].T @ kh))
    np.testing.assert_allclose(sf[0, 0], first, atol=1e-13, rtol=0)
    assert not np.allclose(sf[0, 0], after, atol=1e-6)


# ---------------------------------------------------------------- invariants
def test_l2_normalisation_scale_invariance():
    """q and k are normalised inside the kernel, so positive rescaling of q
    and k (with eps=0) leaves every output unchanged."""
    d = _rand(31, 20, 2, 8, s0_std=0.2)
    out1, s1 = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"], eps=0.0)
    sc = np.random.default_rng(1).uniform(0.1, 10.0, size=(20, 2, 1))
    out2, s2 = oracle.recurrence(d["q"] * sc, d["k"] * sc[::-1], d["v"], d["g"], d["beta"],
                                 s_init=d["s0"], eps=0.0)
    np.testing.assert_allclose(out1, out2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(s1, s2, atol=1e-12, rtol=0)


def test_eps_enters_the_norm():
    """A tiny key with a large eps is barely written: k_hat = k/sqrt(|k|^2+eps)."""
    q = np.ones((1, 1, 4)); k = np.full((1, 1, 4), 1e-3); v = np.ones((1, 1, 4))
    out, sf = oracle.recurrence(q, k, v, np.zeros((1, 1, 4)), np.ones((1, 1)), eps=1.0)
    kh = 1e-3 / np.sqrt(4e-6 + 1.0)
    np.testing.assert_allclose(sf[0, 0], np.full((4, 4), kh), rtol=1e-12)


def test_state_norm_growth_bound():
    """For beta in [0,1], |k|=1, g<=0 the transition (I - beta k k^T)Diag(e^g)
    is a contraction, so |S_t|_2 <= |S_{t-1}|_2 + beta_t |v_t|_2 each step."""
    d = _rand(41, 40, 2, 8, s0_std=1.0, g_scale=0.05)
    S = d["s0"].astype(np.float64)
    for t in range(40):
        _, S_new = oracle.recurrence(d["q"][t:t + 1], d["k"][t:t + 1], d["v"][t:t + 1],
                                     d["g"][t:t + 1], d["beta"][t:t + 1], s_init=S, eps=0.0)
        for h in range(2):
            lhs = np.linalg.norm(S_new[0, h], 2)
            rhs = np.linalg.norm(S[0, h], 2) + d["beta"][t, h] * np.linalg.norm(d["v"][t, h])
            assert lhs <= rhs * (1 + 1e-12)
        S = S_new


# ---------------------------------------------------------------- chunk form / hand-off
@pytest.mark.parametrize("T", [64, 61])
@pytest.mark.parametrize("C", [1, 2, 3, 5, 8, 16, 64, "T"])
def test_chunked_equals_recurrence(T, C):
    """Page 2 section 5: chunked evaluation at any C computes the recurrence
    (C=1 is the recurrence itself, C=T the quadratic form)."""
    C = T if C == "T" else C
    d = _rand(51, T, 2, 16, s0_std=0.3, g_scale=0.2)
    r_out, r_s = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"])
    c_out, c_s = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"], chunk=C)
    np.testing.assert_allclose(c_out, r_out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(c_s, r_s, atol=1e-12, rtol=0)


def test_chunked_equals_recurrence_varlen_default_gates():
    cu = np.array([0, 5, 5, 70, 133, 200], dtype=np.int64)  # includes an empty sequence
    d = _rand(52, 200, 2, 16, s0_std=0.02, cu=cu)
    r_out, r_s = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"],
                                   cu_seqlens=cu, nthreads=4)
    c_out, c_s = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"],
                                   cu_seqlens=cu, chunk=64, nthreads=4)
    np.testing.assert_allclose(c_out, r_out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(c_s, r_s, atol=1e-12, rtol=0)
    np.testing.assert_array_equal(r_s[1], d["s0"][1])  # empty sequence hands S0 through


@pytest.mark.parametrize("g_scale", [1.0, 0.01])
def test_split_prefill_carry_in_equals_unsplit(g_scale):
    d = _rand(61, 150, 2, 16, s0_std=0.3, g_scale=g_scale)
    full_out, full_s = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"])
    a = slice(0, 70); b = slice(70, 150)
    o1, s1 = oracle.recurrence(d["q"][a], d["k"][a], d["v"][a], d["g"][a], d["beta"][a], s_init=d["s0"])
    o2, s2 = oracle.recurrence(d["q"][b], d["k"][b], d["v"][b], d["g"][b], d["beta"][b], s_init=s1)
    np.testing.assert_array_equal(np.concatenate([o1, o2]), full_out)
    np.testing.assert_array_equal(s2, full_s)


def test_decode_steps_equal_one_long_recurrence():
    d = _rand(62, 12, 3, 8, s0_std=0.3, g_scale=0.1)
    full_out, full_s = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"])
    S = d["s0"]
    for t in range(12):
        o, S = oracle.decode_step(d["q"][t:t + 1], d["k"][t:t + 1], d["v"][t:t + 1],
                                  d["g"][t:t + 1], d["beta"][t:t + 1], S)
        np.testing.assert_array_equal(o[0], full_out[t])
    np.testing.assert_array_equal(S, full_s)


def test_threads_do_not_change_results():
    cu = np.array([0, 30, 31, 90], dtype=np.int64)
    d = _rand(63, 90, 5, 8, s0_std=0.1, cu=cu)
    a = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"], cu_seqlens=cu, nthreads=1)
    b = oracle.recurrence(d["q"], d["k"], d["v"], d["g"], d["beta"], s_init=d["s0"], cu_seqlens=cu, nthreads=4)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------- short conv
def _silu(z):
    return z / (1.0 + np.exp(-z))


def test_shortconv_impulse_response_tap_order():
    """An impulse at step 0 comes out through tap 3 (current token), then
    taps 2, 1, 0 on the next steps, then leaves the window."""
    B, H, D = 1, 2, 4
    w = np.random.default_rng(7).standard_normal((3, H, D, 4))
    ring = np.zeros((B, 3, H, 3, D))
    for m in range(5):
        x = np.zeros((B, 3, H, D))
        if m == 0:
            x[:] = 1.0
        y, ring = oracle.shortconv_step(x, ring, w)
        expect = _silu(w[..., 3 - m]) if m < 4 else np.zeros((3, H, D))
        np.testing.assert_allclose(y[0], expect, atol=1e-15, rtol=0)


def test_shortconv_matches_library_convolution():
    """Stepping T tokens through the ring equals SiLU of a causal depthwise
    convolution computed by numpy.convolve, and the ring ends holding the
    last three inputs in order."""
    rng = np.random.default_rng(8)
    B, H, D, T = 2, 3, 5, 17
    w = rng.standard_normal((3, H, D, 4))
    xs = rng.standard_normal((T, B, 3, H, D))
    ring = np.zeros((B, 3, H, 3, D))
    ys = []
    for t in range(T):
        y, ring = oracle.shortconv_step(xs[t], ring, w)
        ys.append(y)
    ys = np.stack(ys)
    for b in range(B):
        for p in range(3):
            for h in range(H):
                for c in range(D):
                    ref = np.convolve(xs[:, b, p, h, c], w[p, h, c, ::-1])[:T]
                    np.testing.assert_allclose(ys[:, b, p, h, c], _silu(ref), atol=1e-13, rtol=0)
    np.testing.assert_array_equal(ring[:, :, :, 0], xs[T - 3])
    np.testing.assert_array_equal(ring[:, :, :, 2], xs[T - 1])


def test_shortconv_silu_special_values():
    w = np.zeros((3, 1, 2, 4)); w[..., 3] = 1.0
    x = np.zeros((1, 3, 1, 2)); x[..., 0] = 40.0
    y, _ = oracle.shortconv_step(x, np.zeros((1, 3, 1, 3, 2)), w)
    assert np.all(y[..., 1] == 0.0)           # SiLU(0) = 0
    np.testing.assert_allclose(y[..., 0], 40.0, rtol=1e-15)  # SiLU(z) -> z for large z


# ------------------------------------------------ short conv over sequences
def _conv_ref(hist, w):
    """SiLU of the causal width-4 convolution of one channel whose first
    three entries are the history: out[t] = silu(sum_m w[m] hist[t + m])."""
    T = len(hist) - 3
    return _silu(np.array([np.dot(w, hist[t:t + 4]) for t in range(T)]))


def test_shortconv_seq_matches_library_convolution():
    """One sequence from zero history equals numpy.convolve per channel,
    with y written projection-major."""
    rng = np.random.default_rng(21)
    T, H, D = 23, 2, 3
    x = rng.standard_normal((T, 3, H, D))
    w = rng.standard_normal((3, H, D, 4))
    y, ring = oracle.shortconv_seq(x, w)
    assert y.shape == (3, T, H, D) and ring.shape == (1, 3, H, 3, D)
    for p in range(3):
        for h in range(H):
            for c in range(D):
                ref = _silu(np.convolve(x[:, p, h, c], w[p, h, c, ::-1])[:T])
                np.testing.assert_allclose(y[p, :, h, c], ref, atol=1e-13, rtol=0)
    np.testing.assert_array_equal(ring[0], np.moveaxis(x[T - 3:], 0, 2))


def test_shortconv_seq_varlen_history_and_ring_out():
    """Sequences of 0, 1, 2, 3 and 9 tokens with a given history: each output
    is the convolution of [history, tokens]; the ring after the sequence is
    its last three entries, so an empty sequence passes its ring through."""
    rng = np.random.default_rng(22)
    lens = [2, 0, 9, 1, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, D, N = int(cu[-1]), 2, 3, len(lens)
    x = rng.standard_normal((T, 3, H, D))
    w = rng.standard_normal((3, H, D, 4))
    rin = rng.standard_normal((N, 3, H, 3, D))
    y, rout = oracle.shortconv_seq(x, w, ring_in=rin, cu_seqlens=cu)
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        for p in range(3):
            for h in range(H):
                for c in range(D):
                    hist = np.concatenate([rin[n, p, h, :, c], x[a:b, p, h, c]])
                    if b > a:
                        np.testing.assert_allclose(y[p, a:b, h, c], _conv_ref(hist, w[p, h, c]),
                                                   atol=1e-13, rtol=0)
                    np.testing.assert_array_equal(rout[n, p, h, :, c], hist[-3:])


def test_shortconv_seq_split_hand_off():
    """Two calls with the ring handed on equal one call over the whole
    sequence, outputs and final ring."""
    rng = np.random.default_rng(23)
    T1, T2, H, D = 7, 2, 1, 4
    x = rng.standard_normal((T1 + T2, 3, H, D))
    w = rng.standard_normal((3, H, D, 4))
    rin = rng.standard_normal((1, 3, H, 3, D))
    y, r = oracle.shortconv_seq(x, w, ring_in=rin)
    y1, r1 = oracle.shortconv_seq(x[:T1], w, ring_in=rin)
    y2, r2 = oracle.shortconv_seq(x[T1:], w, ring_in=r1)
    np.testing.assert_array_equal(np.concatenate([y1, y2], axis=1), y)
    np.testing.assert_array_equal(r2, r)


def test_shortconv_seq_then_decode_step():
    """A prefill conv over T tokens followed by one decode step on its ring
    equals a prefill conv over T + 1 tokens."""
    rng = np.random.default_rng(24)
    T, H, D = 6, 2, 2
    x = rng.standard_normal((T + 1, 3, H, D))
    w = rng.standard_normal((3, H, D, 4))
    y_all, r_all = oracle.shortconv_seq(x, w)
    _, r = oracle.shortconv_seq(x[:T], w)
    y_step, r_step = oracle.shortconv_step(x[T][None], r, w)
    np.testing.assert_array_equal(y_step[0], y_all[:, T])
    np.testing.assert_array_equal(r_step, r_all)


# ---- output epilogue: gated RMSNorm ("WARP中Kimi Delta Attention" section
# "相关源码与文档导航" names it; "为什么 Kimi K3 ..." section 6: an output gate
# that scales the features). The pins below hold for RMS normalisation and
# for the logistic / SiLU gates whatever the implementation.

def _epi_inputs(seed, R=5, D=16):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((R, D)), rng.standard_normal((R, D)), rng.uniform(0.5, 2.0, D)


def test_epilogue_open_gate_gives_unit_mean_square():
    """With the gate fully open (sigmoid(40) = 1 to 1e-17), unit weight and
    eps = 0, every output row has mean square exactly 1 and points the same
    way as its input row."""
    o, _, _ = _epi_inputs(1)
    y = oracle.gated_rmsnorm(o, np.full_like(o, 40.0), np.ones(o.shape[1]), eps=0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-12)
    cos = np.sum(y * o, axis=1) / np.linalg.norm(y, axis=1) / np.linalg.norm(o, axis=1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-12)
    # a closed gate (sigmoid(-40) ~ 4e-18) passes nothing
    z = oracle.gated_rmsnorm(o, np.full_like(o, -40.0), np.ones(o.shape[1]), eps=0.0)
    assert np.max(np.abs(z)) < 1e-16


def test_epilogue_scale_invariance_and_eps():
    """RMS normalisation ignores a positive scale of the row when eps = 0;
    with eps > 0 a zero row maps to zero and a tiny row stays tiny."""
    o, gate, w = _epi_inputs(2)
    y1 = oracle.gated_rmsnorm(o, gate, w, eps=0.0)
    y2 = oracle.gated_rmsnorm(37.5 * o, gate, w, eps=0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-12)
    z = oracle.gated_rmsnorm(np.zeros_like(o), gate, w, eps=1e-6)
    assert np.all(z == 0.0)
    z0 = oracle.gated_rmsnorm(np.zeros_like(o), gate, w, eps=0.0)  # 0 / 0 read as 0
    assert np.all(z0 == 0.0)
    t = oracle.gated_rmsnorm(1e-6 * o, gate, w, eps=1.0)
    assert np.max(np.abs(t)) < 1e-5


def test_epilogue_sigmoid_symmetry_and_weight():
    """sigmoid(z) + sigmoid(-z) = 1, so the outputs for gate and -gate add up
    to the ungated normalised row times the weight; the weight multiplies
    channel by channel (a transposed or shifted weight fails)."""
    o, gate, w = _epi_inputs(3)
    ya = oracle.gated_rmsnorm(o, gate, w, eps=1e-3)
    yb = oracle.gated_rmsnorm(o, -gate, w, eps=1e-3)
    full = oracle.gated_rmsnorm(o, np.full_like(o, 40.0), w, eps=1e-3)
    np.testing.assert_allclose(ya + yb, full, rtol=1e-12, atol=1e-14)
    y1 = oracle.gated_rmsnorm(o, gate, np.ones_like(w), eps=1e-3)
    np.testing.assert_allclose(ya, y1 * w[None, :], rtol=1e-12)
    # gate = 0: sigmoid(0) = 1/2 exactly
    h = oracle.gated_rmsnorm(o, np.zeros_like(o), w, eps=1e-3)
    np.testing.assert_allclose(2.0 * h, full, rtol=1e-12, atol=1e-14)


def test_epilogue_silu_identity():
    """SiLU(z) - SiLU(-z) = z: the SiLU-gated outputs for gate and -gate
    differ by the normalised row times weight times gate; SiLU(0) = 0."""
    o, gate, w = _epi_inputs(4)
    ya = oracle.gated_rmsnorm(o, gate, w, eps=1e-3, act="silu")
    yb = oracle.gated_rmsnorm(o, -gate, w, eps=1e-3, act="silu")
    full = oracle.gated_rmsnorm(o, np.full_like(o, 40.0), w, eps=1e-3)
    np.testing.assert_allclose(ya - yb, full * gate, rtol=1e-11, atol=1e-13)
    z = oracle.gated_rmsnorm(o, np.zeros_like(o), w, eps=1e-3, act="silu")
    assert np.all(z == 0.0)
    # far from zero SiLU(z) -> z (a gate written as z * sigmoid(-z) keeps the
    # odd-part identity above but fails here)
    big = oracle.gated_rmsnorm(o, np.full_like(o, 40.0), w, eps=1e-3, act="silu")
    np.testing.assert_allclose(big, 40.0 * full, rtol=1e-12, atol=1e-14)
