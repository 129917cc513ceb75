"""Full-stack decode workload on the GPU: 69 independent KDA layers x 8
sequences x 96 heads x 128x128 fp32 states (414 MiB per sequence), 256
consecutive decode steps per sequence with per-layer seeded bf16 inputs and
short-conv rings carried across steps ("KV缓存从11.25GB缩到0.21GB: WARP中Kimi
Delta Attention线性注意力原理剖析", sections "KDA 递推公式先衰减再差分" and
"414MB 的 KDA 状态从哪来").

Every launch of the stack runs (69 fused conv+decode launches per step, in
model order). Twelve sampled (layer, sequence, head) units carry inputs from
the seeded numpy generator and are checked against the fp64 oracle over all
256 steps; the other units are filled on the device by a seeded torch
generator with the same distributions.
"""
import numpy as np
import pytest

import oracle
from linear_attention_recurrence_02_gb300 import synth
from tests._util import BF16_REL, cuda_or_skip, ensure_built, to_dev

pytestmark = pytest.mark.gpu

LAYERS, B, H, D, STEPS = (synth.STACK[k] for k in ("layers", "B", "H", "D", "steps"))
SEED = synth.STACK["seed"]
SAMPLES = [(l, b, h) for l in (0, 34, 68) for b in (0, 7) for h in (0, 95)]


@pytest.mark.parametrize("overlap", [False, True])
def test_full_stack_decode_256_steps(overlap):
    """overlap=True launches every step with KDA_DECODE_OVERLAP_PREV (each
    launch follows another layer's), so each layer's state streams in while
    the previous layer's launch drains; the results must not change."""
    torch = cuda_or_skip()
    ensure_built()
    from linear_attention_recurrence_02_gb300 import kda
    bf = torch.bfloat16
    dev = "cuda"
    gen = torch.Generator(device=dev).manual_seed(SEED)

    def rnd(shape):
        return torch.randn(shape, generator=gen, device=dev)

    # device buffers for the whole stack
    x = [rnd((STEPS, B, 3, H, D)).to(bf) for _ in range(LAYERS)]
    g = [-torch.nn.functional.softplus(rnd((STEPS, B, H, D))) for _ in range(LAYERS)]
    beta = [torch.sigmoid(rnd((STEPS, B, H))) for _ in range(LAYERS)]
    state = [rnd((B, H, D, D)) * 0.02 for _ in range(LAYERS)]
    ring = [rnd((B, 3, H, 3, D)).to(bf) for _ in range(LAYERS)]
    w = [to_dev(synth.stack_conv_weights(SEED, l, H, D), torch.float32, torch) for l in range(LAYERS)]
    out = [torch.empty((STEPS, B, H, D), dtype=bf, device=dev) for _ in range(LAYERS)]
    assert kda.state_bytes(LAYERS, H, D, D) == 434_110_464  # 414 MiB per sequence

    units = {}
    for (l, b, h) in SAMPLES:
        u = synth.stack_unit(SEED, l, b, h, STEPS, D)
        units[(l, b, h)] = u
        x[l][:, b, :, h, :] = to_dev(u["x"], bf, torch)
        g[l][:, b, h, :] = to_dev(u["g"], torch.float32, torch)
        beta[l][:, b, h] = to_dev(u["beta"], torch.float32, torch)
        state[l][b, h] = to_dev(u["s0"], torch.float32, torch)
        ring[l][b, :, h] = to_dev(u["ring"], bf, torch)

    for t in range(STEPS):
        for l in range(LAYERS):
            if overlap:
                kda.kda_shortconv_decode_step_ex(x[l][t], ring[l], w[l], g[l][t], beta[l][t], state[l], out[l][t],
                                                 overlap_prev=True)
            else:
                kda.kda_shortconv_decode_step(x[l][t], ring[l], w[l], g[l][t], beta[l][t], state[l], out[l][t])
    torch.cuda.synchronize()
    kda.kda_sync_status()

    worst = 0.0
    for (l, b, h), u in units.items():
        wl = synth.stack_conv_weights(SEED, l, H, D)[:, h:h + 1]
        S = u["s0"][None, None].astype(np.float64)
        rg = u["ring"][None, :, None].astype(np.float64)  # [1,3,1,3,D]
        ref = np.empty((STEPS, D))
        for t in range(STEPS):
            y, rg = oracle.shortconv_step(u["x"][t][None, :, None], rg, wl)
            o, S = oracle.decode_step(y[:, 0], y[:, 1], y[:, 2], u["g"][t][None, None], u["beta"][t][None, None], S)
            ref[t] = o[0, 0]
        got = out[l][:, b, h].float().cpu().numpy()
        got_s = state[l][b, h].cpu().numpy()
        got_r = ring[l][b, :, h].float().cpu().numpy()
        assert np.all(np.isfinite(got)) and np.all(np.isfinite(got_s))
        e_out = np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-6)
        e_st = np.max(np.abs(got_s - S[0, 0])) / max(np.max(np.abs(S[0, 0])), 1e-6)
        worst = max(worst, e_out, e_st)
        assert np.array_equal(got_r, rg[0, :, 0]), f"ring of unit {(l, b, h)}"
    assert worst <= BF16_REL, f"worst per-unit relative error {worst:.3e}"
