"""GPU parity of kda_chunk_prefill_scan, the prefill of one long sequence cut
into segments that run side by side ("为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透
GPT-2 到 K3 的架构进化", section 5: the chunk steps are affine in the state, so a
run of them is one affine map), against the fp64 token recurrence. The gates
are scaled down (slow decay) so that each segment's state still matters to the
next one: with the workloads' decay a segment forgets its initial state within
a chunk or two and a wrong scan would go unnoticed."""
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


def _run(torch, kda, p, D, bf16, segments, C, gate="channel", with_s0=True):
    dt = torch.bfloat16 if bf16 else torch.float32
    q, k, v = (to_dev(p[n], dt, torch) for n in "qkv")
    g_all = p["g"]
    if gate == "head":
        gk, go = np.ascontiguousarray(g_all[..., 0]), np.repeat(g_all[..., :1], D, axis=-1)
    elif gate == "none":
        gk, go = None, np.zeros_like(g_all)
    else:
        gk, go = g_all, g_all
    s0 = p["s0"][0] if with_s0 else None
    out = torch.empty_like(q)
    sf = torch.empty((q.shape[1], D, D), device="cuda")
    kda.kda_chunk_prefill_scan(q, k, v, None if gk is None else to_dev(gk, torch.float32, torch),
                               to_dev(p["beta"], torch.float32, torch), out, segments,
                               initial_state=None if s0 is None else to_dev(s0, torch.float32, torch),
                               final_state=sf, gate=gate, chunk_size=C)
    torch.cuda.synchronize()
    kda.kda_sync_status()
    ro, rs = oracle.recurrence(p["q"], p["k"], p["v"], go, p["beta"],
                               s_init=None if s0 is None else s0[None])
    return to_np(out), to_np(sf), ro, rs[0]


@pytest.mark.parametrize("segments", [2, 3, 8])
def test_scan_tensor_core_path(env, segments):
    """bf16, d=128, C=64 (the tensor-core kernel for all three passes),
    1061 tokens (a ragged last chunk), carry-in state."""
    torch, kda = env
    T, H, D = 1061, 2, 128
    p = synth.prefill_inputs(31, T, H, D, True, s0_std=0.05, g_scale=0.02)
    o, s, ro, rs = _run(torch, kda, p, D, True, segments, 64)
    assert_close(o, ro, True, (1,), "out")
    assert_close(s, rs, True, (0,), "final state")


@pytest.mark.parametrize("gate", ["head", "none"])
def test_scan_gate_forms(env, gate):
    """Per-head gate and no gate (the state never decays: every segment's map
    A is far from zero)."""
    torch, kda = env
    T, H, D = 640, 2, 128
    p = synth.prefill_inputs(32, T, H, D, True, s0_std=0.05, g_scale=0.02)
    o, s, ro, rs = _run(torch, kda, p, D, True, 4, 64, gate=gate)
    assert_close(o, ro, True, (1,), "out")
    assert_close(s, rs, True, (0,), "final state")


@pytest.mark.parametrize("with_s0", [False, True])
def test_scan_fp32_cuda_core_path(env, with_s0):
    """fp32, d=16, C=16 (the CUDA-core kernel): the fp32 tolerance."""
    torch, kda = env
    T, H, D = 300, 3, 16
    p = synth.prefill_inputs(33, T, H, D, False, s0_std=0.05, g_scale=0.02)
    o, s, ro, rs = _run(torch, kda, p, D, False, 5, 16, with_s0=with_s0)
    assert_close(o, ro, False, (1,), "out")
    assert_close(s, rs, False, (0,), "final state")


def test_scan_matches_the_serial_prefill(env):
    """The workloads' own decay (g_scale 1): the segmented and the serial
    prefill agree to bf16 tolerance."""
    torch, kda = env
    T, H, D = 2048, 4, 128
    p = synth.prefill_inputs(34, T, H, D, True)
    bf = torch.bfloat16
    q, k, v = (to_dev(p[n], bf, torch) for n in "qkv")
    g, b = to_dev(p["g"], torch.float32, torch), to_dev(p["beta"], torch.float32, torch)
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    s1, s2 = torch.empty((H, D, D), device="cuda"), torch.empty((H, D, D), device="cuda")
    kda.kda_chunk_prefill(q, k, v, g, b, o1, final_state=s1[None], chunk_size=64)
    kda.kda_chunk_prefill_scan(q, k, v, g, b, o2, 8, final_state=s2)
    torch.cuda.synchronize()
    assert_close(to_np(o2), to_np(o1), True, (1,), "out")
    assert_close(to_np(s2), to_np(s1), True, (0,), "final state")


def test_scan_tensor_core_path_no_carry_in(env):
    """bf16, d=128, no initial state: the outputs of the first segment need no correction; 1500 tokens in 5
    segments of 320 tokens (not a multiple of the 128-token correction blocks)."""
    torch, kda = env
    T, H, D = 1500, 2, 128
    p = synth.prefill_inputs(35, T, H, D, True, s0_std=0.05, g_scale=0.02)
    o, s, ro, rs = _run(torch, kda, p, D, True, 5, 64, with_s0=False)
    assert_close(o, ro, True, (1,), "out")
    assert_close(s, rs, True, (0,), "final state")


@pytest.mark.parametrize("segments", [0, 19])
def test_scan_longer_sequence_mild_gates(env, segments):
    """8192 tokens, 2 heads, gates scaled by 0.02 so that the carried state matters across every segment;
    19 segments of 448 tokens (and the automatic count, which fills the GPU's SMs once)."""
    torch, kda = env
    T, H, D = 8192, 2, 128
    p = synth.prefill_inputs(36, T, H, D, True, s0_std=0.05, g_scale=0.02)
    o, s, ro, rs = _run(torch, kda, p, D, True, segments, 64)
    assert_close(o, ro, True, (1,), "out")
    assert_close(s, rs, True, (0,), "final state")


def test_prefill_splits_one_long_sequence_automatically(env):
    """kda_chunk_prefill on one 12,288-token sequence with 8 heads: with the workspace that
    kda_chunk_prefill_workspace_bytes asks for, the call takes the segmented path (floor(SMs / 8) segments);
    without one, the serial path. Both against the fp64 oracle with mild gates and a carry-in state, and
    against each other (an empty workspace keeps the serial path)."""
    torch, kda = env
    T, H, D = 12288, 8, 128
    need = kda.kda_chunk_prefill_workspace_bytes(T, 1, H, D, 64)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms // H < 4:
        pytest.skip("too few SMs for the automatic split at 8 heads")
    assert need > 0
    p = synth.prefill_inputs(37, T, H, D, True, s0_std=0.05, g_scale=0.02)
    bf = torch.bfloat16
    q, k, v = (to_dev(p[n], bf, torch) for n in "qkv")
    g, b = to_dev(p["g"], torch.float32, torch), to_dev(p["beta"], torch.float32, torch)
    s0 = to_dev(p["s0"], torch.float32, torch)
    outs = []
    # the binding allocates the asked-for workspace when given none: an empty one keeps the serial path
    for ws in (torch.empty(need, dtype=torch.uint8, device="cuda"), torch.empty(0, dtype=torch.uint8, device="cuda")):
        o = torch.full_like(q, float("nan"))
        sf = torch.full((1, H, D, D), float("nan"), device="cuda")
        kda.kda_chunk_prefill(q, k, v, g, b, o, initial_state=s0, final_state=sf, chunk_size=64, workspace=ws)
        kda.kda_sync_status()
        outs.append((to_np(o), to_np(sf)))
    ro, rs = oracle.recurrence(p["q"], p["k"], p["v"], p["g"], p["beta"], s_init=p["s0"])
    for o, sf in outs:
        assert_close(o, ro, True, (1,), "out")
        assert_close(sf, rs, True, (0, 1), "final state")
    assert_close(outs[0][0], outs[1][0], True, (1,), "split vs serial")


@pytest.mark.parametrize("bf16", [True, False])
def test_split_batch_with_a_long_sequence(env, bf16):
    """kda_chunk_prefill_split on a packed batch with an empty sequence, short ones and one long one, with
    carry-in states and mild gates (g_scale 0.02: the carried state matters across the long sequence's
    segments). The plan for this GPU splits the long sequence (and only it); every output and final state
    against the fp64 recurrence, and against kda_chunk_prefill_gated of the same batch."""
    torch, kda = env
    H, D = 8, 128
    lens = [300, 0, 9000, 50, 1500]
    cu = np.cumsum([0] + lens).astype(np.int64)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    seg, nsplit = kda.kda_chunk_prefill_split_plan(cu, H, 64)
    expect, _ = kda.kda_chunk_prefill_split_plan(cu, H, 64, sms=sms)
    assert list(seg) == list(expect)
    assert nsplit == 1 and seg[2] >= 4 and all(seg[i] == 1 for i in (0, 1, 3, 4)), seg
    p = synth.prefill_inputs(41, int(cu[-1]), H, D, bf16, cu_seqlens=cu, s0_std=0.05, g_scale=0.02)
    dt = torch.bfloat16 if bf16 else torch.float32
    q, k, v = (to_dev(p[n], dt, torch) for n in "qkv")
    g, b = to_dev(p["g"], torch.float32, torch), to_dev(p["beta"], torch.float32, torch)
    s0 = to_dev(p["s0"], torch.float32, torch)
    N = len(lens)
    res = []
    for split in (True, False):
        o = torch.full_like(q, float("nan"))
        sf = torch.full((N, H, D, D), float("nan"), device="cuda")
        if split:
            kda.kda_chunk_prefill_split(q, k, v, g, b, o, torch.from_numpy(cu), initial_state=s0, final_state=sf,
                                        chunk_size=64)
        else:
            kda.kda_chunk_prefill_gated(q, k, v, g, b, o, initial_state=s0, final_state=sf,
                                        cu_seqlens=torch.from_numpy(cu).cuda(), chunk_size=64)
        kda.kda_sync_status()
        res.append((to_np(o), to_np(sf)))
    ro, rs = oracle.recurrence(p["q"], p["k"], p["v"], p["g"], p["beta"], s_init=p["s0"], cu_seqlens=cu)
    for o, sf in res:
        assert_close(o, ro, bf16, (1,), "out")
        assert_close(sf, rs, bf16, (0, 1), "final state")
    assert_close(res[0][0], res[1][0], bf16, (1,), "split vs whole")


def test_split_captured_in_a_cuda_graph(env):
    """kda_chunk_prefill_split captured into a CUDA graph through the C ABI (its side stream forks from and
    joins the capturing stream; the host lengths and every device buffer prepared before the capture) and
    replayed: bit-identical outputs and final states to the direct call."""
    torch, kda = env
    H, D = 4, 128
    lens = [4096, 100, 200]
    cu = np.cumsum([0] + lens).astype(np.int64)
    seg, nsplit = kda.kda_chunk_prefill_split_plan(cu, H, 64)
    assert nsplit == 1 and seg[0] >= 4 and seg[1] == 1 and seg[2] == 1, seg
    p = synth.prefill_inputs(47, int(cu[-1]), H, D, True, cu_seqlens=cu, s0_std=0.05, g_scale=0.02)
    bf = torch.bfloat16
    q, k, v = (to_dev(p[n], bf, torch) for n in "qkv")
    g, b = to_dev(p["g"], torch.float32, torch), to_dev(p["beta"], torch.float32, torch)
    s0 = to_dev(p["s0"], torch.float32, torch)
    dev_cu = torch.from_numpy(cu).cuda()
    lib = kda.lib()
    N, T = len(lens), int(cu[-1])
    need = int(lib.kda_chunk_prefill_split_workspace_bytes(cu.ctypes.data, N, H, D, 64))
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    outs = [(torch.full_like(q, float("nan")), torch.full((N, H, D, D), float("nan"), device="cuda"))
            for _ in range(2)]

    def call(o, sf, stream):
        return lib.kda_chunk_prefill_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), b.data_ptr(),
                                           s0.data_ptr(), sf.data_ptr(), o.data_ptr(), dev_cu.data_ptr(),
                                           cu.ctypes.data, N, T, H, D, 64, kda.KDA_BF16, 0, 1e-6, ws.data_ptr(),
                                           ws.numel(), stream)
    assert call(*outs[0], torch.cuda.current_stream().cuda_stream) == kda.KDA_OK
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        st = call(*outs[1], torch.cuda.current_stream().cuda_stream)
    assert st == kda.KDA_OK, lib.kda_last_error_detail().decode()
    graph.replay()
    torch.cuda.synchronize()
    kda.kda_sync_status()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("gate", ["channel", "head"])
def test_split_batch_with_two_long_sequences(env, gate):
    """kda_chunk_prefill_split with two sequences long enough to split (the scan workspace reused for
    both, the per-head gate's rows offset per sequence) around short ones, bf16, carry-in states and mild
    gates, against the fp64 recurrence."""
    torch, kda = env
    H, D = 8, 128
    lens = [9000, 40, 8500, 300]
    cu = np.cumsum([0] + lens).astype(np.int64)
    seg, nsplit = kda.kda_chunk_prefill_split_plan(cu, H, 64)
    assert nsplit == 2 and seg[0] >= 4 and seg[2] >= 4 and seg[1] == 1 and seg[3] == 1, seg
    p = synth.prefill_inputs(43, int(cu[-1]), H, D, True, cu_seqlens=cu, s0_std=0.05, g_scale=0.02)
    bf = torch.bfloat16
    q, k, v = (to_dev(p[n], bf, torch) for n in "qkv")
    if gate == "head":
        gk, go = np.ascontiguousarray(p["g"][..., 0]), np.repeat(p["g"][..., :1], D, axis=-1)
    else:
        gk, go = p["g"], p["g"]
    o = torch.full_like(q, float("nan"))
    sf = torch.full((len(lens), H, D, D), float("nan"), device="cuda")
    kda.kda_chunk_prefill_split(q, k, v, to_dev(gk, torch.float32, torch), to_dev(p["beta"], torch.float32, torch),
                                o, torch.from_numpy(cu), gate=gate, initial_state=to_dev(p["s0"], torch.float32, torch),
                                final_state=sf, chunk_size=64)
    kda.kda_sync_status()
    ro, rs = oracle.recurrence(p["q"], p["k"], p["v"], go, p["beta"], s_init=p["s0"], cu_seqlens=cu)
    assert_close(to_np(o), ro, True, (1,), "out")
    assert_close(to_np(sf), rs, True, (0, 1), "final state")
