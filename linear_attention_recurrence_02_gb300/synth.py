"""Seeded synthetic inputs for the KDA recurrence.

This module holds no arithmetic of the recurrence itself: it only draws
random numbers with the distributions of the workloads the pages describe
(96 heads, d_k = d_v = 128, 69 KDA layers, 4K context) and rounds them to
bf16 where a workload stores bf16. Both the CUDA path and the CPU oracle are
fed from here; neither imports the other.

Distributions (per workload description):
  q, k, v (or the pre-conv projections x)  ~ N(0, 1)
  g     = -softplus(N(0, 1))   per key channel, log space
  beta  = sigmoid(N(0, 1))     per token and head
  S0    ~ N(0, 0.02^2)         fp32 state, when a workload has a non-zero one
  ring  ~ N(0, 1)              previous pre-conv projections (decode)
  w     ~ N(0, 0.5^2)          short-conv taps (the pages give no weights)

Streams: every independent unit draws from its own PCG64 stream keyed by
(seed, stream id, unit index...), in a fixed order within the stream, so any
unit (a head of a prefill, a (layer, sequence, head) of a decode stack) can be
regenerated alone for sampled checks.
"""
from __future__ import annotations

import numpy as np

# stream ids
_TOK, _STATE, _RING, _CONVW, _DECODE = 0, 1, 2, 3, 4


def bf16_round(a) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 out."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).reshape(a.shape)


def _softplus(x):
    return np.logaddexp(0.0, x)


def _sigmoid(x):
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def _rng(*key):
    return np.random.default_rng([int(x) for x in key])


def _normal(rng, shape, std=1.0):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def gate_from_normal(z, g_scale=1.0):
    """g = -softplus(z) * g_scale (log-space decay, always <= 0)."""
    return (-_softplus(z.astype(np.float64)) * g_scale).astype(np.float32)


def beta_from_normal(z):
    return _sigmoid(z.astype(np.float64)).astype(np.float32)


def head_tokens(seed: int, h: int, T: int, D: int, bf16: bool, g_scale=1.0):
    """Token inputs of one head: q,k,v,g [T,D] and beta [T] (float32)."""
    rng = _rng(seed, _TOK, h)
    q = _normal(rng, (T, D))
    k = _normal(rng, (T, D))
    v = _normal(rng, (T, D))
    g = gate_from_normal(rng.standard_normal((T, D), dtype=np.float32), g_scale)
    beta = beta_from_normal(rng.standard_normal((T,), dtype=np.float32))
    if bf16:
        q, k, v = bf16_round(q), bf16_round(k), bf16_round(v)
    return q, k, v, g, beta


def initial_state(seed: int, n: int, h: int, D: int, std: float = 0.02):
    """fp32 D x D initial state of (sequence n, head h)."""
    return _normal(_rng(seed, _STATE, n, h), (D, D), std)


def prefill_inputs(seed: int, T: int, H: int, D: int, bf16: bool,
                   cu_seqlens=None, s0_std=None, g_scale=1.0, heads=None):
    """Packed prefill inputs.

    Returns a dict with q,k,v,g [T,H',D], beta [T,H'], cu_seqlens [N+1] int64
    and s0 [N,H',D,D] (or None), where H' = len(heads) (default all H heads).
    Head h of a head subset is bit-identical to head h of the full set.
    """
    if cu_seqlens is None:
        cu_seqlens = np.array([0, T], dtype=np.int64)
    cu_seqlens = np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu_seqlens) - 1
    heads = list(range(H)) if heads is None else list(heads)
    Hs = len(heads)
    q = np.empty((T, Hs, D), np.float32)
    k = np.empty_like(q)
    v = np.empty_like(q)
    g = np.empty_like(q)
    beta = np.empty((T, Hs), np.float32)
    for a, h in enumerate(heads):
        q[:, a], k[:, a], v[:, a], g[:, a], beta[:, a] = head_tokens(seed, h, T, D, bf16, g_scale)
    s0 = None
    if s0_std is not None:
        s0 = np.empty((N, Hs, D, D), np.float32)
        for n in range(N):
            for a, h in enumerate(heads):
                s0[n, a] = initial_state(seed, n, h, D, s0_std)
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=cu_seqlens, s0=s0)


def decode_inputs(seed: int, B: int, H: int, D: int, bf16: bool,
                  s0_std=0.02, g_scale=1.0):
    """One decode step for B sequences with its short-conv ring.

    Returns x [B,3,H,D] (pre-conv q,k,v projections), ring [B,3,H,3,D]
    (3 previous tokens, oldest first), w [3,H,D,4], g [B,H,D], beta [B,H],
    s0 [B,H,D,D] (zeros when s0_std is None), and q,k,v [B,H,D] drawn for
    the decode kernel alone (post-conv inputs, same distribution as x).
    """
    rng = _rng(seed, _DECODE)
    x = _normal(rng, (B, 3, H, D))
    g = gate_from_normal(rng.standard_normal((B, H, D), dtype=np.float32), g_scale)
    beta = beta_from_normal(rng.standard_normal((B, H), dtype=np.float32))
    ring = _normal(_rng(seed, _RING), (B, 3, H, 3, D))
    w = _normal(_rng(seed, _CONVW), (3, H, D, 4), 0.5)
    qkv = _normal(_rng(seed, _TOK), (3, B, H, D))
    if s0_std is None:
        s0 = np.zeros((B, H, D, D), np.float32)
    else:
        s0 = _normal(_rng(seed, _STATE), (B, H, D, D), s0_std)
    if bf16:
        x, ring = bf16_round(x), bf16_round(ring)
        qkv = bf16_round(qkv)
    return dict(x=x, ring=ring, w=w, g=g, beta=beta, s0=s0,
                q=qkv[0], k=qkv[1], v=qkv[2])


def conv_prefill_inputs(seed: int, T: int, H: int, D: int, N: int, bf16: bool, heads=None):
    """Pre-conv projections of a packed prompt batch: x [T,3,H,D] ~ N(0,1),
    ring_in [N,3,H,3,D] ~ N(0,1) (history before each sequence), w [3,H,D,4]
    ~ N(0, 0.5^2). With `heads`, only those heads are drawn (each head from
    its own stream, so a subset equals the same heads of the full draw)."""
    heads = list(range(H)) if heads is None else list(heads)
    x = np.empty((T, 3, len(heads), D), np.float32)
    ring = np.empty((N, 3, len(heads), 3, D), np.float32)
    w = np.empty((3, len(heads), D, 4), np.float32)
    for a, h in enumerate(heads):
        x[:, :, a] = _normal(_rng(seed, _TOK, 3, h), (T, 3, D))
        ring[:, :, a] = _normal(_rng(seed, _RING, 3, h), (N, 3, 3, D))
        w[:, a] = _normal(_rng(seed, _CONVW, 3, h), (3, D, 4), 0.5)
    if bf16:
        x, ring = bf16_round(x), bf16_round(ring)
    return dict(x=x, ring=ring, w=w)


def stack_unit(seed: int, layer: int, b: int, h: int, steps: int, D: int,
               bf16: bool = True, s0_std=0.02):
    """Inputs of one (layer, sequence, head) unit of a multi-layer decode
    stack over `steps` steps: S0 [D,D], ring [3,3,D], x [steps,3,D],
    g [steps,D], beta [steps]."""
    rng = _rng(seed, layer, b, h)
    s0 = _normal(rng, (D, D), s0_std)
    ring = _normal(rng, (3, 3, D))
    x = _normal(rng, (steps, 3, D))
    g = gate_from_normal(rng.standard_normal((steps, D), dtype=np.float32))
    beta = beta_from_normal(rng.standard_normal((steps,), dtype=np.float32))
    if bf16:
        ring, x = bf16_round(ring), bf16_round(x)
    return dict(s0=s0, ring=ring, x=x, g=g, beta=beta)


def stack_conv_weights(seed: int, layer: int, H: int, D: int):
    """Short-conv taps of one layer of a decode stack, [3,H,D,4]."""
    return _normal(_rng(seed, layer, _CONVW, 0), (3, H, D, 4), 0.5)


# Workload sizes (named by what they are).
TINY = dict(T=64, H=2, D=16, seed=0)
DECODE = dict(B=64, H=96, D=128, seed=1)
PREFILL = dict(T=4096, H=96, D=128, C=64, seed=2)
STACK = dict(layers=69, B=8, H=96, D=128, steps=256, seed=3)
VARLEN_LENGTHS = [512, 1024, 2048, 4096, 8192, 16384, 32768, 65536]
VARLEN = dict(H=96, D=128, C=64, seed=4)


def epilogue_inputs(seed: int, T: int, H: int, D: int, bf16: bool):
    """Inputs of the output epilogue: o [T,H,D] ~ N(0,1) with a per-row scale
    exp(N(0,1)) (rows of different magnitude), gate [T,H,D] ~ N(0, 2^2),
    weight [D] ~ U(0.5, 1.5). o and gate rounded to bf16 when bf16."""
    rng = _rng(seed, 0xE1)
    o = _normal(rng, (T, H, D)) * np.exp(rng.standard_normal((T, H, 1))).astype(np.float32)
    gate = _normal(rng, (T, H, D), 2.0)
    weight = rng.uniform(0.5, 1.5, D).astype(np.float32)
    if bf16:
        o, gate = bf16_round(o), bf16_round(gate)
    return dict(o=o.astype(np.float32), gate=gate, weight=weight)


def varlen_cu_seqlens(lengths=VARLEN_LENGTHS):
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, np.int64))]).astype(np.int64)
