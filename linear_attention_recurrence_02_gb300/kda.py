"""Thin ctypes binding of libkda.so (declared in include/kda.h).

Argument marshalling only: shapes and dtypes are read from the torch tensors
passed in, their device pointers and the current CUDA stream are handed to
the C ABI, and a non-OK status raises ``KdaError``. Every step of the
computation runs in the library's CUDA kernels; there is no fallback. If the
library has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_DEVICE_CHECK = range(6)
# gate forms: one log-gate per key channel (KDA), per head (Gated DeltaNet), none (DeltaNet)
KDA_GATE_CHANNEL, KDA_GATE_HEAD, KDA_GATE_NONE = range(3)
KDA_DECODE_OVERLAP_PREV = 1  # launch flag of kda_shortconv_decode_step_ex
KDA_ACT_SIGMOID, KDA_ACT_SILU = 0, 1  # output-gate activations of kda_gated_rmsnorm
_ACTS = {"sigmoid": KDA_ACT_SIGMOID, "silu": KDA_ACT_SILU}
_GATES = {"channel": KDA_GATE_CHANNEL, "head": KDA_GATE_HEAD, "none": KDA_GATE_NONE}


def _gate_code(gate):
    if isinstance(gate, str):
        return _GATES[gate]
    return int(gate)


def _check_gate(g, gate, lead, H, D):
    """Shape of g for a gate form: [..., H, D], [..., H], or absent."""
    code = _gate_code(gate)
    if code == KDA_GATE_CHANNEL:
        ok = g is not None and tuple(g.shape) == (*lead, H, D)
    elif code == KDA_GATE_HEAD:
        ok = g is not None and tuple(g.shape) == (*lead, H)
    else:
        ok = True
    if not ok:
        raise ValueError("g shape does not match the gate form")
    return code
KDA_F32, KDA_BF16 = 0, 1

_lib = None
_lock = threading.Lock()

_vp = ctypes.c_void_p
_ci = ctypes.c_int
_cf = ctypes.c_float
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t

_SIGNATURES = {
    "kda_status_string": ([_ci], ctypes.c_char_p),
    "kda_last_error_detail": ([], ctypes.c_char_p),
    "kda_abi_version": ([], _ci),
    "kda_state_bytes": ([_ci, _ci, _ci, _ci], _sz),
    "kda_shortconv_ring_bytes": ([_ci, _ci, _ci, _ci, _ci], _sz),
    "kda_shortconv_step": ([_vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _vp], _ci),
    "kda_shortconv_prefill": ([_vp, _vp, _vp, _vp, _vp, _vp, _ci, _i64, _ci, _ci, _ci, _vp], _ci),
    "kda_decode_step": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _cf, _vp], _ci),
    "kda_decode_step_gated": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _cf, _vp], _ci),
    "kda_shortconv_decode_step_gated": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _cf, _vp],
                                        _ci),
    "kda_chunk_prefill_gated": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _i64, _ci, _ci, _ci, _ci, _ci,
                                 _cf, _vp, _sz, _vp], _ci),
    "kda_shortconv_decode_step": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _cf, _vp], _ci),
    "kda_shortconv_decode_step_ex": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _cf,
                                      ctypes.c_uint, _vp], _ci),
    "kda_shortconv_decode_step_epi": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _ci,
                                       _cf, _cf, ctypes.c_uint, _vp], _ci),
    "kda_chunk_prefill_workspace_bytes": ([_i64, _ci, _ci, _ci, _ci], _sz),
    "kda_chunk_prefill_route": ([_ci, _ci, _ci], ctypes.c_char_p),
    "kda_chunk_prefill": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _i64, _ci, _ci, _ci, _ci,
                           _cf, _vp, _sz, _vp], _ci),
    "kda_chunk_prefill_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _i64, _ci, _ci, _ci,
                                   _ci, _cf, _vp], _ci),
    "kda_gated_rmsnorm": ([_vp, _vp, _vp, _vp, _i64, _ci, _ci, _ci, _ci, _cf, _vp], _ci),
    "kda_chunk_prefill_scan_workspace_bytes": ([_i64, _ci, _ci, _ci, _ci], _sz),
    "kda_chunk_prefill_split": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _i64, _ci, _ci, _ci, _ci,
                                 _ci, _cf, _vp, _sz, _vp], _ci),
    "kda_chunk_prefill_split_workspace_bytes": ([_vp, _ci, _ci, _ci, _ci], _sz),
    "kda_chunk_prefill_split_plan": ([_vp, _ci, _ci, _ci, _ci, _vp], _ci),
    "kda_chunk_prefill_epi": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _i64, _ci, _ci, _ci, _ci, _ci,
                               _cf, _vp, _vp, _ci, _cf, _vp, _sz, _vp], _ci),
    "kda_chunk_prefill_scan": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _ci, _ci, _ci, _ci, _ci, _cf, _ci,
                                _vp, _sz, _vp], _ci),
    "kda_sync_status": ([_vp], _ci),
    "kda_selftest_bounded_wait": ([ctypes.c_longlong, _vp], _ci),
}


class KdaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{_status_string(status)} ({detail})")


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded CDLL with argument types set (raises if not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            handle = ctypes.CDLL(path)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
    return _lib


def exported_symbols():
    return list(_SIGNATURES)


def _status_string(status: int) -> str:
    try:
        return lib().kda_status_string(status).decode()
    except Exception:  # library unavailable while formatting an error
        return f"status {status}"


def _check(status: int):
    if status != KDA_OK:
        raise KdaError(status, lib().kda_last_error_detail().decode())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def state_bytes(layers, heads, dk, dv) -> int:
    return int(lib().kda_state_bytes(layers, heads, dk, dv))


def shortconv_ring_bytes(layers, batch, heads, d, elem_bytes) -> int:
    return int(lib().kda_shortconv_ring_bytes(layers, batch, heads, d, elem_bytes))


def kda_shortconv_step(x, ring, w, y, stream=None):
    """x [B,3,H,D], ring [B,3,H,3,D] (in/out), w [3,H,D,4] fp32, y [3,B,H,D]."""
    B, P, H, D = x.shape
    if P != 3 or tuple(ring.shape) != (B, 3, H, 3, D) or tuple(w.shape) != (3, H, D, 4) \
            or tuple(y.shape) != (3, B, H, D):
        raise ValueError("shape mismatch")
    _check(lib().kda_shortconv_step(_ptr(x), _ptr(ring), _ptr(w), _ptr(y), B, H, D, _dtype_code(x),
                                    _stream(stream, x.device)))


def kda_shortconv_prefill(x, w, y, ring_in=None, ring_out=None, cu_seqlens=None, stream=None):
    """x [T,3,H,D]; w [3,H,D,4] fp32; y [3,T,H,D]; rings [N,3,H,3,D] or None;
    cu_seqlens int64 [N+1] on the device (or None for one sequence)."""
    T, P, H, D = x.shape
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    if P != 3 or tuple(w.shape) != (3, H, D, 4) or tuple(y.shape) != (3, T, H, D):
        raise ValueError("shape mismatch")
    for r in (ring_in, ring_out):
        if r is not None and tuple(r.shape) != (N, 3, H, 3, D):
            raise ValueError("ring shape mismatch")
    _check(lib().kda_shortconv_prefill(_ptr(x), _ptr(ring_in), _ptr(w), _ptr(y), _ptr(ring_out),
                                       _ptr(cu_seqlens), N, T, H, D, _dtype_code(x), _stream(stream, x.device)))


def kda_decode_step(q, k, v, g, beta, state, out, l2_eps=1e-6, stream=None):
    """q,k,v,out [B,H,D]; g [B,H,D] fp32; beta [B,H] fp32; state [B,H,D,D] fp32 (in/out)."""
    B, H, D = q.shape
    if tuple(g.shape) != (B, H, D) or tuple(beta.shape) != (B, H) or tuple(state.shape) != (B, H, D, D) \
            or tuple(out.shape) != (B, H, D):
        raise ValueError("shape mismatch")
    _check(lib().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out),
                                 B, H, D, _dtype_code(q), float(l2_eps), _stream(stream, q.device)))


def kda_decode_step_gated(q, k, v, g, beta, state, out, gate="channel", l2_eps=1e-6, stream=None):
    """kda_decode_step with gate "channel" (g [B,H,D]), "head" (g [B,H]) or "none" (g unused)."""
    B, H, D = q.shape
    code = _check_gate(g, gate, (B,), H, D)
    if tuple(beta.shape) != (B, H) or tuple(state.shape) != (B, H, D, D) or tuple(out.shape) != (B, H, D):
        raise ValueError("shape mismatch")
    _check(lib().kda_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(out),
                                       B, H, D, _dtype_code(q), code, float(l2_eps), _stream(stream, q.device)))


def kda_shortconv_decode_step_gated(x, ring, w, g, beta, state, out, gate="channel", l2_eps=1e-6, stream=None):
    """kda_shortconv_decode_step with a gate form as in kda_decode_step_gated."""
    B, P, H, D = x.shape
    code = _check_gate(g, gate, (B,), H, D)
    if P != 3 or tuple(ring.shape) != (B, 3, H, 3, D) or tuple(w.shape) != (3, H, D, 4) \
            or tuple(beta.shape) != (B, H) or tuple(state.shape) != (B, H, D, D) or tuple(out.shape) != (B, H, D):
        raise ValueError("shape mismatch")
    _check(lib().kda_shortconv_decode_step_gated(_ptr(x), _ptr(ring), _ptr(w), _ptr(g), _ptr(beta), _ptr(state),
                                                 _ptr(out), B, H, D, _dtype_code(x), code, float(l2_eps),
                                                 _stream(stream, x.device)))


def kda_shortconv_decode_step_ex(x, ring, w, g, beta, state, out, gate="channel", l2_eps=1e-6,
                                 overlap_prev=False, stream=None):
    """kda_shortconv_decode_step_gated with launch flags. overlap_prev=True is
    the caller's promise that the kernel enqueued just before on the stream
    does not write `state` (e.g. the step of another layer); the launch may
    then overlap that kernel's tail (KDA_DECODE_OVERLAP_PREV)."""
    B, P, H, D = x.shape
    code = _check_gate(g, gate, (B,), H, D)
    if P != 3 or tuple(ring.shape) != (B, 3, H, 3, D) or tuple(w.shape) != (3, H, D, 4) \
            or tuple(beta.shape) != (B, H) or tuple(state.shape) != (B, H, D, D) or tuple(out.shape) != (B, H, D):
        raise ValueError("shape mismatch")
    flags = KDA_DECODE_OVERLAP_PREV if overlap_prev else 0
    _check(lib().kda_shortconv_decode_step_ex(_ptr(x), _ptr(ring), _ptr(w), _ptr(g), _ptr(beta), _ptr(state),
                                              _ptr(out), B, H, D, _dtype_code(x), code, float(l2_eps), flags,
                                              _stream(stream, x.device)))


def kda_shortconv_decode_step_epi(x, ring, w, g, beta, state, out_gate, norm_weight, y, gate="channel",
                                  act="sigmoid", l2_eps=1e-6, norm_eps=1e-6, overlap_prev=False, stream=None):
    """Fused short conv + decode step whose output goes through the gated
    RMSNorm epilogue before it is stored: y = RMSNorm(o) * norm_weight *
    act(out_gate), o the step's output (fp32 inside the kernel). out_gate and
    y [B,H,D] like x; norm_weight [D] fp32; other arguments as
    kda_shortconv_decode_step_ex."""
    B, P, H, D = x.shape
    code = _check_gate(g, gate, (B,), H, D)
    if P != 3 or tuple(ring.shape) != (B, 3, H, 3, D) or tuple(w.shape) != (3, H, D, 4) \
            or tuple(beta.shape) != (B, H) or tuple(state.shape) != (B, H, D, D) or tuple(y.shape) != (B, H, D) \
            or tuple(out_gate.shape) != (B, H, D) or tuple(norm_weight.shape) != (D,):
        raise ValueError("shape mismatch")
    if act not in _ACTS:
        raise ValueError(f"act must be one of {sorted(_ACTS)}")
    flags = KDA_DECODE_OVERLAP_PREV if overlap_prev else 0
    _check(lib().kda_shortconv_decode_step_epi(_ptr(x), _ptr(ring), _ptr(w), _ptr(g), _ptr(beta), _ptr(state),
                                               _ptr(out_gate), _ptr(norm_weight), _ptr(y), B, H, D, _dtype_code(x),
                                               code, _ACTS[act], float(l2_eps), float(norm_eps), flags,
                                               _stream(stream, x.device)))


def kda_shortconv_decode_step(x, ring, w, g, beta, state, out, l2_eps=1e-6, stream=None):
    """Fused short conv + decode step. x [B,3,H,D], ring [B,3,H,3,D] (in/out),
    w [3,H,D,4] fp32, g [B,H,D] fp32, beta [B,H] fp32, state [B,H,D,D] fp32
    (in/out), out [B,H,D]."""
    B, P, H, D = x.shape
    if P != 3 or tuple(ring.shape) != (B, 3, H, 3, D) or tuple(w.shape) != (3, H, D, 4) \
            or tuple(g.shape) != (B, H, D) or tuple(beta.shape) != (B, H) \
            or tuple(state.shape) != (B, H, D, D) or tuple(out.shape) != (B, H, D):
        raise ValueError("shape mismatch")
    _check(lib().kda_shortconv_decode_step(_ptr(x), _ptr(ring), _ptr(w), _ptr(g), _ptr(beta), _ptr(state),
                                           _ptr(out), B, H, D, _dtype_code(x), float(l2_eps),
                                           _stream(stream, x.device)))


def kda_gated_rmsnorm(o, gate, weight, y, act="sigmoid", eps=1e-6, stream=None):
    """Output epilogue: y = RMSNorm(o) * weight * act(gate) per (token, head)
    row. o, gate, y [T,H,D] (y may be o); weight [D] fp32; act "sigmoid" or
    "silu"."""
    T, H, D = o.shape
    if tuple(gate.shape) != (T, H, D) or tuple(y.shape) != (T, H, D) or tuple(weight.shape) != (D,):
        raise ValueError("shape mismatch")
    if act not in _ACTS:
        raise ValueError(f"act must be one of {sorted(_ACTS)}")
    _check(lib().kda_gated_rmsnorm(_ptr(o), _ptr(gate), _ptr(weight), _ptr(y), T, H, D, _dtype_code(o),
                                   _ACTS[act], float(eps), _stream(stream, o.device)))


def kda_chunk_prefill_epi(q, k, v, g, beta, out, out_gate, norm_weight, gate="channel", act="sigmoid",
                          norm_eps=1e-6, initial_state=None, final_state=None, cu_seqlens=None, chunk_size=64,
                          l2_eps=1e-6, workspace=None, stream=None):
    """kda_chunk_prefill_gated whose output goes through the gated RMSNorm
    epilogue in the same call: out = RMSNorm(o) * norm_weight * act(out_gate).
    out_gate [T,H,D] like q; norm_weight [D] fp32."""
    T, H, D = q.shape
    code = _check_gate(g, gate, (T,), H, D)
    if tuple(out_gate.shape) != (T, H, D) or tuple(norm_weight.shape) != (D,):
        raise ValueError("shape mismatch")
    if act not in _ACTS:
        raise ValueError(f"act must be one of {sorted(_ACTS)}")
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    ws_bytes = kda_chunk_prefill_workspace_bytes(T, N, H, D, chunk_size)
    if workspace is None and ws_bytes > 0:
        import torch
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kda_chunk_prefill_epi(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                       _ptr(final_state), _ptr(out), _ptr(cu_seqlens), N, T, H, D, chunk_size,
                                       _dtype_code(q), code, float(l2_eps), _ptr(out_gate), _ptr(norm_weight),
                                       _ACTS[act], float(norm_eps), _ptr(workspace), wsz, _stream(stream, q.device)))


def kda_chunk_prefill_scan_workspace_bytes(T, H, D, C, segments) -> int:
    return int(lib().kda_chunk_prefill_scan_workspace_bytes(T, H, D, C, segments))


def kda_chunk_prefill_scan(q, k, v, g, beta, out, segments, initial_state=None, final_state=None, gate="channel",
                           chunk_size=64, l2_eps=1e-6, workspace=None, stream=None):
    """Prefill of one long sequence split into `segments` runs processed side
    by side. q,k,v,out [T,H,D]; g per `gate`; beta [T,H]; states [H,D,D] fp32.
    workspace: a device uint8 tensor of kda_chunk_prefill_scan_workspace_bytes
    (allocated here when None)."""
    T, H, D = q.shape
    code = _check_gate(g, gate, (T,), H, D)
    need = kda_chunk_prefill_scan_workspace_bytes(T, H, D, chunk_size, segments)
    if workspace is None and need > 0:
        import torch
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib().kda_chunk_prefill_scan(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                        _ptr(final_state), _ptr(out), T, H, D, chunk_size, _dtype_code(q), code,
                                        float(l2_eps), int(segments), _ptr(workspace),
                                        0 if workspace is None else workspace.numel() * workspace.element_size(),
                                        _stream(stream, q.device)))


def kda_chunk_prefill_route(D, C, dtype) -> str | None:
    """Name of the kernel the chunked prefill runs for this head dimension, chunk size and dtype
    (torch.bfloat16 / torch.float32 or the KDA_* dtype code); None for an unsupported shape."""
    if isinstance(dtype, int):
        code = dtype
    else:
        import torch
        code = {torch.bfloat16: KDA_BF16, torch.float32: KDA_F32}[dtype]
    r = lib().kda_chunk_prefill_route(int(D), int(C), int(code))
    return None if r is None else r.decode()


def kda_chunk_prefill_workspace_bytes(total_tokens, num_seqs, H, D, C) -> int:
    return int(lib().kda_chunk_prefill_workspace_bytes(total_tokens, num_seqs, H, D, C))


def kda_chunk_prefill(q, k, v, g, beta, out, initial_state=None, final_state=None, cu_seqlens=None,
                      chunk_size=64, l2_eps=1e-6, workspace=None, stream=None):
    """q,k,v,out [T,H,D]; g [T,H,D] fp32; beta [T,H] fp32; states [N,H,D,D] fp32;
    cu_seqlens int64 [N+1] on the device (or None for one sequence)."""
    T, H, D = q.shape
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    ws_bytes = kda_chunk_prefill_workspace_bytes(T, N, H, D, chunk_size)
    if workspace is None and ws_bytes > 0:
        import torch
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kda_chunk_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                   _ptr(final_state), _ptr(out), _ptr(cu_seqlens), N, T, H, D, chunk_size,
                                   _dtype_code(q), float(l2_eps), _ptr(workspace), wsz,
                                   _stream(stream, q.device)))


def kda_chunk_prefill_gated(q, k, v, g, beta, out, gate="channel", initial_state=None, final_state=None,
                            cu_seqlens=None, chunk_size=64, l2_eps=1e-6, workspace=None, stream=None):
    """kda_chunk_prefill with gate "channel" (g [T,H,D]), "head" (g [T,H]) or "none" (g unused)."""
    T, H, D = q.shape
    code = _check_gate(g, gate, (T,), H, D)
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    ws_bytes = kda_chunk_prefill_workspace_bytes(T, N, H, D, chunk_size)
    if workspace is None and ws_bytes > 0:
        import torch
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kda_chunk_prefill_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                         _ptr(final_state), _ptr(out), _ptr(cu_seqlens), N, T, H, D, chunk_size,
                                         _dtype_code(q), code, float(l2_eps), _ptr(workspace), wsz,
                                         _stream(stream, q.device)))


def _host_cu(cu_seqlens):
    import numpy as np
    a = cu_seqlens.detach().cpu().numpy() if hasattr(cu_seqlens, "detach") else cu_seqlens
    return np.ascontiguousarray(a, dtype=np.int64)


def kda_chunk_prefill_split_plan(cu_seqlens, H, chunk_size=64, sms=0):
    """Segment count per sequence that kda_chunk_prefill_split uses (1: kept whole) and the number of
    split sequences; `sms` <= 0 plans for the current device."""
    import numpy as np
    cu = _host_cu(cu_seqlens)
    N = cu.shape[0] - 1
    seg = np.zeros(max(N, 1), dtype=np.int32)
    n = lib().kda_chunk_prefill_split_plan(cu.ctypes.data, N, H, chunk_size, sms, seg.ctypes.data)
    if n < 0:
        raise KdaError(KDA_ERR_INVALID_ARG, "invalid cu_seqlens")
    return seg[:N], n


def kda_chunk_prefill_split(q, k, v, g, beta, out, cu_seqlens, gate="channel", initial_state=None,
                            final_state=None, chunk_size=64, l2_eps=1e-6, workspace=None, stream=None):
    """Chunked prefill of a packed batch that splits its long sequences through the chunk-state scan.
    cu_seqlens: the [N+1] offsets, on the host or the device (a host copy is taken here, a device
    copy made when it lives on the host); other arguments as kda_chunk_prefill_gated."""
    import torch
    T, H, D = q.shape
    code = _check_gate(g, gate, (T,), H, D)
    host = _host_cu(cu_seqlens)
    dev_cu = cu_seqlens if (hasattr(cu_seqlens, "is_cuda") and cu_seqlens.is_cuda) else \
        torch.from_numpy(host).to(q.device)
    N = host.shape[0] - 1
    need = int(lib().kda_chunk_prefill_split_workspace_bytes(host.ctypes.data, N, H, D, chunk_size))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wsz = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kda_chunk_prefill_split(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                         _ptr(final_state), _ptr(out), _ptr(dev_cu), host.ctypes.data, N, T, H, D,
                                         chunk_size, _dtype_code(q), code, float(l2_eps), _ptr(workspace), wsz,
                                         _stream(stream, q.device)))


def kda_chunk_prefill_noalloc(q, k, v, g, beta, out, initial_state=None, final_state=None, cu_seqlens=None,
                              chunk_size=64, l2_eps=1e-6, stream=None):
    """kda_chunk_prefill without a workspace, for callers that cannot allocate
    device memory: the launch-order scratch lives in a fixed array owned by
    the library (at most 4096 sequences). Overlapping calls race on it."""
    T, H, D = q.shape
    N = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    _check(lib().kda_chunk_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                           _ptr(final_state), _ptr(out), _ptr(cu_seqlens), N, T, H, D, chunk_size,
                                           _dtype_code(q), float(l2_eps), _stream(stream, q.device)))


def kda_selftest_bounded_wait(limit_cycles=2_000_000, stream=None, device=None):
    """Launch the bounded-wait diagnostic (a wait nothing completes); the next
    kda_sync_status on the stream then raises with KDA_ERR_TIMEOUT."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(lib().kda_selftest_bounded_wait(int(limit_cycles), _stream(stream, dev)))


def kda_sync_status(stream=None, device=None):
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(lib().kda_sync_status(_stream(stream, dev)))
