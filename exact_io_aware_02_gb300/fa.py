"""Python binding of the C-ABI library ``libfa_gb300.so`` (argument marshalling only).

Every function here has the name of the C entry point it calls (declared in
``include/fa_gb300.h``).  Tensors are PyTorch CUDA tensors; PyTorch provides
device memory and the stream, the library does all the work.  Importing this
module loads the library and raises ImportError when it has not been built:
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libfa_gb300.so")

FA_OK = 0
FA_ERR_ARG = -1
FA_ERR_ARCH = -2
FA_ERR_LAUNCH = -3
FA_ERR_TIMEOUT = -4
FA_ERR_CUDA = -5
FA_ERR_WORKSPACE_TOO_LARGE = -6
FA_STATIC_WORKSPACE_BYTES = 16 << 20
FA_STATUS_TIMEOUT = 0x1
FA_STATUS_V_RANGE = 0x2

EXPORTED = ("fa_fwd", "fa_fwd_gqa", "fa_fwd_gqa_workspace_bytes", "fa_fwd_gqa_static_workspace",
            "fa_fwd_host", "fa_bwd", "fa_bwd_host", "fa_fwd_fp8", "fa_fwd_fp8_host", "fa_fwd_fp8_workspace_bytes", "fa_status", "fa_fwd_withheld_tile",
            "fa_fwd_withheld_ring_tile",
            "fa_bwd_withheld_tile", "fa_fwd_fp8_withheld_tile", "fa_strerror", "fa_version")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")

lib = ctypes.CDLL(LIB_PATH)
_vp, _i, _f, _d = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double
lib.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]
lib.fa_fwd.restype = _i
lib.fa_fwd_gqa.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp,
                           ctypes.c_size_t, _vp]
lib.fa_fwd_gqa.restype = _i
lib.fa_fwd_gqa_workspace_bytes.argtypes = [_i, _i, _i, _i, _i]
lib.fa_fwd_gqa_workspace_bytes.restype = ctypes.c_size_t
lib.fa_fwd_gqa_static_workspace.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp]
lib.fa_fwd_gqa_static_workspace.restype = _i
lib.fa_fwd_host.argtypes = [_vp] * 10 + [_i, _i, _i, _i, _i, _i, _f, _i, _i, _vp]
lib.fa_fwd_host.restype = _i
lib.fa_fwd_withheld_tile.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _d, _vp]
lib.fa_fwd_withheld_tile.restype = _i
lib.fa_fwd_withheld_ring_tile.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _d, _vp]
lib.fa_fwd_withheld_ring_tile.restype = _i
lib.fa_bwd.argtypes = [_vp] * 10 + [_i, _i, _i, _i, _i, _f, _i, _vp]
lib.fa_bwd.restype = _i
lib.fa_bwd_host.argtypes = [_vp] * 19 + [_i, _i, _i, _i, _i, _f, _i, _i, _vp]
lib.fa_bwd_host.restype = _i
lib.fa_fwd_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, ctypes.c_size_t, _vp]
lib.fa_fwd_fp8.restype = _i
lib.fa_fwd_fp8_host.argtypes = [_vp] * 11 + [_i, _i, _i, _i, _f, _i, _vp, ctypes.c_size_t, _i, _vp]
lib.fa_fwd_fp8_host.restype = _i
lib.fa_fwd_fp8_workspace_bytes.argtypes = [_i, _i, _i, _i]
lib.fa_fwd_fp8_workspace_bytes.restype = ctypes.c_size_t
lib.fa_bwd_withheld_tile.argtypes = [_vp] * 10 + [_i, _i, _i, _i, _i, _f, _i, _d, _vp]
lib.fa_bwd_withheld_tile.restype = _i
lib.fa_fwd_fp8_withheld_tile.argtypes = [_vp] * 6 + [_i, _i, _i, _i, _f, _i, _vp, ctypes.c_size_t, _d, _vp]
lib.fa_fwd_fp8_withheld_tile.restype = _i
lib.fa_status.argtypes = [_i, _vp]
lib.fa_status.restype = _i
lib.fa_strerror.argtypes = [_i]
lib.fa_strerror.restype = ctypes.c_char_p
lib.fa_version.argtypes = []
lib.fa_version.restype = _i


class FAError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(f"fa error {code}: {lib.fa_strerror(code).decode()}")


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _prepare(q, k, v, o, lse):
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    return B, H, N, d, o, lse


def fa_fwd(q, k, v, o=None, lse=None, scale=None, causal=False, stream=None):
    """Exact attention forward.  q, k, v: CUDA bf16 [B, H, N, d] contiguous.

    Returns (o, lse): o bf16 [B, H, N, d], lse fp32 [B, H, N] (natural log).
    Preallocated ``o`` / ``lse`` are written in place.  Raises FAError on a
    nonzero return code.  Shape, dtype and placement checks are the library's.
    """
    B, H, N, d, o, lse = _prepare(q, k, v, o, lse)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    B, H, N, d, float(scale), int(bool(causal)), _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc)
    return o, lse


def fa_fwd_gqa_workspace_bytes(B, Hq, Nq, d, n_splits) -> int:
    return int(lib.fa_fwd_gqa_workspace_bytes(B, Hq, Nq, d, n_splits))


def fa_fwd_gqa(q, k, v, o=None, lse=None, scale=None, causal=False, n_splits=1,
               workspace=None, stream=None):
    """Grouped-K/V, split-K/V forward.  q: [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d]
    (CUDA bf16, contiguous).  Returns (o, lse).  ``workspace`` (a CUDA tensor of at
    least fa_fwd_gqa_workspace_bytes bytes, 256-byte aligned) is allocated here when
    omitted and n_splits > 1."""
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q must be [B, Hq, Nq, d] and k, v [B, Hkv, Nk, d]")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    ws_bytes = fa_fwd_gqa_workspace_bytes(B, Hq, Nq, d, n_splits)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, Hq, Hkv, Nq, Nk, d, float(scale), int(bool(causal)), int(n_splits),
                        ws_ptr, ws_len, _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc)
    return o, lse


def fa_fwd_host(q_host, k_host, v_host, o_host, lse_host, q, k, v, o, lse, scale=None, causal=False,
                groups_per_chunk=0, stream=None):
    """Host-to-host forward with the copies overlapped with the attention, chunk by chunk.

    q_host, k_host, v_host, o_host, lse_host: pinned CPU tensors (``pin_memory()``) in the
    layouts of fa_fwd_gqa; q, k, v, o, lse: CUDA tensors of the same shapes (q, k, v receive
    the copies).  Enqueues on ``stream`` and returns; synchronise it before reading o_host.
    """
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q must be [B, Hq, Nq, d] and k, v [B, Hkv, Nk, d]")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = lib.fa_fwd_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), o_host.data_ptr(),
                         lse_host.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                         lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                         int(groups_per_chunk), _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc)
    return o_host, lse_host


def fa_fwd_gqa_static_workspace(q, k, v, o=None, lse=None, scale=None, causal=False, n_splits=1,
                                stream=None):
    """fa_fwd_gqa without a workspace argument, for callers that cannot allocate device
    memory: the split partials go to the library's fixed 16 MiB device array (shared by
    every call on the device -- do not overlap calls on the GPU).  The outputs ``o`` and
    ``lse`` are still the caller's; pass them preallocated to allocate nothing here."""
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q must be [B, Hq, Nq, d] and k, v [B, Hkv, Nk, d]")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = lib.fa_fwd_gqa_static_workspace(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, float(scale),
                                         int(bool(causal)), int(n_splits), _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc)
    return o, lse


def fa_bwd(q, k, v, o, lse, dout, dq=None, dk=None, dv=None, delta=None, scale=None,
           causal=False, stream=None):
    """Attention backward with recomputation from the forward's (o, lse).
    q, o, dout: CUDA bf16 [B, Hq, N, d]; k, v: [B, Hkv, N, d]; lse: fp32 [B, Hq, N].
    Returns (dq, dk, dv, delta); delta = rowsum(dout * o) in fp32.  Preallocated
    outputs are written in place.  Raises FAError on a nonzero return code."""
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("q, o, dout must be [B, Hq, N, d] and k, v [B, Hkv, N, d]")
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if delta is None:
        delta = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                    dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), delta.data_ptr(),
                    B, Hq, Hkv, N, d, float(scale), int(bool(causal)), _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc)
    return dq, dk, dv, delta


def fa_fwd_fp8_host(q_host, k_host, v_host, o_host, lse_host, q, k, v, signs, o, lse, workspace, scale=None,
                    causal=False, groups_per_chunk=0, stream=None):
    """Host-to-host FP8 forward with the copies overlapped with the kernels, chunk by chunk.
    Host tensors pinned; q, k, v, o, lse, signs, workspace on the device as for fa_fwd_fp8."""
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    rc = lib.fa_fwd_fp8_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), o_host.data_ptr(),
                             lse_host.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), signs.data_ptr(),
                             o.data_ptr(), lse.data_ptr(), B, H, N, d, float(scale), int(bool(causal)),
                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                             int(groups_per_chunk), _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc)
    return o_host, lse_host


def fa_bwd_host(host_inputs, host_outputs, dev_inputs, dev_outputs, delta, scale=None, causal=False,
                groups_per_chunk=0, stream=None):
    """Host-to-host backward with the copies overlapped with the kernels, chunk by chunk.

    host_inputs: pinned CPU (q, k, v, o, lse, dout); host_outputs: pinned CPU (dq, dk, dv);
    dev_inputs / dev_outputs: CUDA tensors of the same shapes (the inputs receive the copies);
    delta: CUDA fp32 [B, Hq, N].  Enqueues on ``stream``; synchronise it before reading the
    host outputs."""
    q, k = dev_inputs[0], dev_inputs[1]
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    ptrs = [t.data_ptr() for t in (*host_inputs, *host_outputs, *dev_inputs, *dev_outputs, delta)]
    rc = lib.fa_bwd_host(*ptrs, B, Hq, Hkv, N, d, float(scale), int(bool(causal)), int(groups_per_chunk),
                         _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc)
    return host_outputs


def fa_fwd_fp8_workspace_bytes(B, H, N, d) -> int:
    return int(lib.fa_fwd_fp8_workspace_bytes(B, H, N, d))


def fa_fwd_fp8(q, k, v, signs, o=None, lse=None, scale=None, causal=False, workspace=None, stream=None):
    """FP8 attention forward (block-wise E4M3 with incoherent processing).  q, k, v: CUDA
    bf16 [B, H, N, 128]; signs: CUDA int8 [128] (the rotation's random signs).  Returns
    (o, lse).  ``workspace`` (a CUDA uint8 tensor of fa_fwd_fp8_workspace_bytes bytes,
    256-byte aligned) is allocated here when omitted; afterwards it holds the quantised
    tensors and their scales (layout in include/fa_gb300.h)."""
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    o = torch.empty_like(q) if o is None else o
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    ws_bytes = fa_fwd_fp8_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    rc = lib.fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), signs.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), B, H, N, d, float(scale), int(bool(causal)), workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    if rc != FA_OK:
        raise FAError(rc)
    return o, lse


def fa_fwd_withheld_tile(q, k, v, o=None, lse=None, scale=None, causal=False,
                         wait_timeout_ms=50.0, stream=None) -> int:
    """Test hook: run the kernel with V tile 0 never loaded; returns the C return code."""
    B, H, N, d, o, lse = _prepare(q, k, v, o, lse)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    return lib.fa_fwd_withheld_tile(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), B, H, N, d, float(scale), int(bool(causal)),
                                    float(wait_timeout_ms), _stream_handle(stream, q.device))


def fa_fwd_withheld_ring_tile(q, k, v, ring_tile, o=None, lse=None, scale=None, causal=False,
                              wait_timeout_ms=50.0, stream=None) -> int:
    """Test hook: run the kernel with K/V ring tile `ring_tile` (K_0 = 0, V_0 = 1, K_1 = 2, ...)
    never loaded; returns the C return code."""
    B, H, N, d, o, lse = _prepare(q, k, v, o, lse)
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    return lib.fa_fwd_withheld_ring_tile(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, H, N, d, float(scale), int(bool(causal)),
                                         int(ring_tile), float(wait_timeout_ms),
                                         _stream_handle(stream, q.device))


def fa_bwd_withheld_tile(q, k, v, o, lse, dout, wait_timeout_ms=50.0, causal=False, stream=None) -> int:
    """Test hook: fa_bwd with the first dK/dV stage and V tile 0 of the dQ kernel never
    loaded; returns the C return code (outputs are allocated here and discarded)."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    return lib.fa_bwd_withheld_tile(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), delta.data_ptr(),
                                    B, Hq, Hkv, N, d, 1.0 / d ** 0.5, int(bool(causal)), float(wait_timeout_ms),
                                    _stream_handle(stream, q.device))


def fa_fwd_fp8_withheld_tile(q, k, v, signs, wait_timeout_ms=50.0, causal=False, stream=None) -> int:
    """Test hook: fa_fwd_fp8 with V tile 0 never loaded; returns the C return code."""
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    ws_bytes = fa_fwd_fp8_workspace_bytes(B, H, N, d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    return lib.fa_fwd_fp8_withheld_tile(q.data_ptr(), k.data_ptr(), v.data_ptr(), signs.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), B, H, N, d, 1.0 / d ** 0.5, int(bool(causal)),
                                        ws.data_ptr(), ws_bytes, float(wait_timeout_ms),
                                        _stream_handle(stream, q.device))


def fa_status(clear=False, stream=None) -> int:
    """Synchronise the stream and return the device status word (optionally clearing it)."""
    dev = torch.cuda.current_device()
    rc = lib.fa_status(int(bool(clear)), _stream_handle(stream, dev))
    if rc < 0:
        raise FAError(rc)
    return rc


def fa_strerror(code: int) -> str:
    return lib.fa_strerror(int(code)).decode()


def fa_version() -> int:
    return lib.fa_version()
