"""gated_delta_rule_21_gb300 -- Python binding of libkda, the GB300 (sm_103a)
chunked Kimi Delta Attention forward.

The binding only marshals arguments: it checks dtypes/shapes/devices of torch
tensors, allocates outputs and the workspace with torch (device memory and
streams are all torch is used for), and calls the C ABI declared in
``include/kda.h`` through ctypes.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU or eager fallback, and importing this
package fails loudly when ``libkda.so`` has not been built.

Entry points (same names as the C ABI, minus the ``kda_`` prefix):

* :func:`chunk_fwd` -- the chunked KDA forward (``kda_chunk_fwd[_ex]``).
* :func:`chunk_bwd` -- its gradient (``kda_chunk_bwd``).
* :func:`short_conv_silu` -- the causal conv + SiLU (+ L2) prologue.
* :func:`workspace_size`, :func:`read_device_status`,
  :func:`clear_device_status`, :func:`status_string`, :func:`version`.
* :func:`lib` -- the raw ctypes library with typed signatures.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK = 0
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED",
                3: "KDA_ERR_ALIGNMENT", 4: "KDA_ERR_WORKSPACE", 5: "KDA_ERR_CUDA",
                6: "KDA_ERR_TIMEOUT", 7: "KDA_ERR_DEVICE"}
IMPLS = {"auto": 0, "simt": 1, "tc": 2, "split": 3}
DTYPES = {torch.float32: 0, torch.bfloat16: 1}
CHUNK = 64


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({status_string(status)})")


class kda_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int),
                ("qkv_dtype", ctypes.c_int)]


_lib = None
_lock = threading.Lock()


def lib():
    """Load libkda.so (raising if it is missing) and return the typed CDLL."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"libkda.so is not built ({LIB_PATH}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` or "
                "`python -m gated_delta_rule_21_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, u64, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        sp = ctypes.POINTER(kda_shape)
        L.kda_chunk_fwd_workspace_size.argtypes = [sp, i]
        L.kda_chunk_fwd_workspace_size.restype = u64
        L.kda_chunk_fwd_workspace_size_for.argtypes = [sp, i, i]
        L.kda_chunk_fwd_workspace_size_for.restype = u64
        L.kda_chunk_fwd_workspace_size_packed.argtypes = [sp, i]
        L.kda_chunk_fwd_workspace_size_packed.restype = u64
        L.kda_chunk_fwd.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp, vp,
                                    vp, vp, u64, vp]
        L.kda_chunk_fwd.restype = i
        L.kda_chunk_fwd_ex.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp,
                                       vp, vp, vp, u64, i, i, vp]
        L.kda_chunk_fwd_ex.restype = i
        L.kda_short_conv_silu.argtypes = [sp, vp, vp, vp, vp, vp, i, vp, vp,
                                          vp, vp]
        L.kda_short_conv_silu.restype = i
        L.kda_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        L.kda_read_device_status.restype = i
        L.kda_clear_device_status.argtypes = [vp, vp]
        L.kda_clear_device_status.restype = i
        L.kda_status_string.argtypes = [i]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_impl_available.argtypes = [i, sp, i]
        L.kda_impl_available.restype = i
        L.kda_version.argtypes = []
        L.kda_version.restype = i
        L.kda_chunk_fwd_host_buffer_size.argtypes = [sp, i]
        L.kda_chunk_fwd_host_buffer_size.restype = u64
        L.kda_chunk_fwd_host.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp, vp,
                                         vp, vp, u64, vp]
        L.kda_chunk_fwd_host.restype = i
        L.kda_chunk_bwd_workspace_size.argtypes = [sp, i]
        L.kda_chunk_bwd_workspace_size.restype = u64
        L.kda_chunk_bwd.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp, vp, vp, vp, vp, vp,
                                    vp, vp, vp, vp, u64, vp]
        L.kda_chunk_bwd.restype = i
        L.kda_chunk_bwd_workspace_size_for.argtypes = [sp, i, i]
        L.kda_chunk_bwd_workspace_size_for.restype = u64
        L.kda_chunk_bwd_workspace_size_packed.argtypes = [sp, i]
        L.kda_chunk_bwd_workspace_size_packed.restype = u64
        L.kda_chunk_fwd_save_workspace_size.argtypes = [sp, i]
        L.kda_chunk_fwd_save_workspace_size.restype = u64
        L.kda_chunk_fwd_save.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp, vp, vp, vp, u64, vp]
        L.kda_chunk_fwd_save.restype = i
        L.kda_chunk_bwd_from_saved.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp, vp, vp, vp,
                                               vp, vp, vp, vp, vp, vp, u64, vp]
        L.kda_chunk_bwd_from_saved.restype = i
        L.kda_chunk_bwd_ex.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp, vp, vp, vp, vp, vp,
                                       vp, vp, vp, vp, u64, i, vp]
        L.kda_chunk_bwd_ex.restype = i
        L.kda_chunk_fwd_scan_workspace_size.argtypes = [sp, i]
        L.kda_chunk_fwd_scan_workspace_size.restype = u64
        L.kda_chunk_fwd_scan_segments.argtypes = [sp, i]
        L.kda_chunk_fwd_scan_segments.restype = i
        L.kda_chunk_fwd_scan.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp, vp, i, vp, u64, vp]
        L.kda_chunk_fwd_scan.restype = i
        L.kda_chunk_fwd_noalloc.argtypes = [sp, vp, vp, vp, vp, vp, f, i, vp, vp, vp, vp, vp]
        L.kda_chunk_fwd_noalloc.restype = i
        L.kda_chunk_fwd_noalloc_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.kda_chunk_fwd_noalloc_status.restype = i
        L.kda_selftest_wait_timeout.argtypes = [vp, ctypes.c_longlong, vp]
        L.kda_selftest_wait_timeout.restype = i
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def version() -> int:
    return lib().kda_version()


def impl_available(impl, B, T, H, K, V, dtype=torch.bfloat16, v_tile=0) -> bool:
    """Whether implementation ``impl`` ("auto"/"simt"/"tc") runs this shape."""
    s = make_shape(B, T, H, K, V, dtype)
    return bool(lib().kda_impl_available(IMPLS[impl], ctypes.byref(s), int(v_tile)))


def make_shape(B, T, H, K, V, dtype) -> kda_shape:
    if dtype not in DTYPES:
        raise TypeError(f"q/k/v dtype must be float32 or bfloat16, got {dtype}")
    return kda_shape(int(B), int(T), int(H), int(K), int(V), DTYPES[dtype])


def workspace_size(B, T, H, K, V, dtype=torch.bfloat16, has_segment_ids=False,
                   impl=None) -> int:
    """Workspace bytes: what the fastest kernel needs (impl None, the C
    default query) or what ``impl`` needs ("simt" gives the smallest size
    any path accepts)."""
    s = make_shape(B, T, H, K, V, dtype)
    if impl is None:
        return int(lib().kda_chunk_fwd_workspace_size(ctypes.byref(s), int(bool(has_segment_ids))))
    return int(lib().kda_chunk_fwd_workspace_size_for(ctypes.byref(s), int(bool(has_segment_ids)),
                                                      IMPLS[impl]))


def workspace_size_packed(B, T, H, K, V, max_runs_per_row, dtype=torch.bfloat16) -> int:
    """Split-path workspace for packed inputs with at most ``max_runs_per_row``
    runs per row."""
    s = make_shape(B, T, H, K, V, dtype)
    return int(lib().kda_chunk_fwd_workspace_size_packed(ctypes.byref(s), int(max_runs_per_row)))


def alloc_workspace(B, T, H, K, V, dtype=torch.bfloat16, has_segment_ids=False,
                    device=None, impl=None, max_runs_per_row=None) -> torch.Tensor:
    """Zero-filled workspace of the size ``impl`` needs (uint8 device tensor);
    with ``max_runs_per_row`` the split path's packed bound is used."""
    n = 0
    if max_runs_per_row is not None and has_segment_ids and impl in ("auto", "split"):
        n = workspace_size_packed(B, T, H, K, V, max_runs_per_row, dtype)
    if n == 0:
        n = workspace_size(B, T, H, K, V, dtype, has_segment_ids, impl)
    if n == 0:
        raise KdaError(1, "workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def chunk_fwd(q, k, v, g, beta, scale=None, chunk_size=CHUNK, initial_state=None,
              segment_ids=None, output_final_state=False, out=None,
              final_state_out=None, workspace=None, impl="auto", v_tile=0,
              stream=None, max_runs_per_row=None):
    """Chunked KDA forward on the GPU.

    q, k: [B,T,H,K]; v: [B,T,H,V] (bf16 or fp32, same dtype); g: [B,T,H,K]
    fp32 log-decay in [-5, 0]; beta: [B,T,H] fp32; initial_state: [B,H,K,V]
    fp32 or None; segment_ids: [B,T] int32 (1-based, 0 = padding) or None.
    ``scale`` None means K**-0.5.  ``max_runs_per_row`` bounds the runs
    per row when the workspace is allocated here for packed inputs.
    Returns ``(o, final_state or None)``.
    """
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("chunk_fwd needs CUDA tensors")
    dt = q.dtype
    _check(q, "q", (B, T, H, K), dt, dev)
    _check(k, "k", (B, T, H, K), dt, dev)
    _check(v, "v", (B, T, H, V), dt, dev)
    _check(g, "g", (B, T, H, K), torch.float32, dev)
    _check(beta, "beta", (B, T, H), torch.float32, dev)
    _check(initial_state, "initial_state", (B, H, K, V), torch.float32, dev)
    _check(segment_ids, "segment_ids", (B, T), torch.int32, dev)
    if scale is None:
        scale = K ** -0.5
    o = out if out is not None else torch.empty(B, T, H, V, dtype=dt, device=dev)
    _check(o, "out", (B, T, H, V), dt, dev)
    fs = None
    if output_final_state:
        fs = final_state_out if final_state_out is not None else torch.empty(
            B, H, K, V, dtype=torch.float32, device=dev)
        _check(fs, "final_state_out", (B, H, K, V), torch.float32, dev)
    if workspace is None:
        workspace = alloc_workspace(B, T, H, K, V, dt, segment_ids is not None, dev, impl=impl,
                                    max_runs_per_row=max_runs_per_row)
    s = make_shape(B, T, H, K, V, dt)
    st = lib().kda_chunk_fwd_ex(
        ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        float(scale), int(chunk_size), _ptr(initial_state), _ptr(segment_ids),
        _ptr(o), _ptr(fs), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        IMPLS[impl], int(v_tile), _stream_ptr(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd")
    return o, fs


def scan_workspace_size(B, T, H, K, V, dtype=torch.bfloat16, n_segments=0) -> int:
    """Workspace bytes of chunk_fwd_scan (0 when the shape is not served)."""
    s = make_shape(B, T, H, K, V, dtype)
    return int(lib().kda_chunk_fwd_scan_workspace_size(ctypes.byref(s), int(n_segments)))


def scan_segments(B, T, H, K, V, dtype=torch.bfloat16, n_segments=0) -> int:
    """Segments per row chunk_fwd_scan uses for this request (0: not served)."""
    s = make_shape(B, T, H, K, V, dtype)
    return int(lib().kda_chunk_fwd_scan_segments(ctypes.byref(s), int(n_segments)))


def chunk_fwd_scan(q, k, v, g, beta, scale=None, chunk_size=CHUNK, initial_state=None,
                   output_final_state=False, n_segments=0, out=None, final_state_out=None,
                   workspace=None, stream=None):
    """The chunked forward as a chunk-parallel state scan over ``n_segments``
    segments per row (0: chosen to fill the GPU); rows without segment ids,
    bf16 with K = V = 128.  Same results as chunk_fwd up to rounding.
    Returns ``(o, final_state or None)``."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev, dt = q.device, q.dtype
    if dev.type != "cuda":
        raise ValueError("chunk_fwd_scan needs CUDA tensors")
    _check(q, "q", (B, T, H, K), dt, dev)
    _check(k, "k", (B, T, H, K), dt, dev)
    _check(v, "v", (B, T, H, V), dt, dev)
    _check(g, "g", (B, T, H, K), torch.float32, dev)
    _check(beta, "beta", (B, T, H), torch.float32, dev)
    _check(initial_state, "initial_state", (B, H, K, V), torch.float32, dev)
    if scale is None:
        scale = K ** -0.5
    o = out if out is not None else torch.empty(B, T, H, V, dtype=dt, device=dev)
    _check(o, "out", (B, T, H, V), dt, dev)
    fs = None
    if output_final_state:
        fs = final_state_out if final_state_out is not None else torch.empty(
            B, H, K, V, dtype=torch.float32, device=dev)
        _check(fs, "final_state_out", (B, H, K, V), torch.float32, dev)
    if workspace is None:
        n = scan_workspace_size(B, T, H, K, V, dt, n_segments)
        if n == 0:
            raise KdaError(2, "kda_chunk_fwd_scan_workspace_size")
        workspace = torch.zeros(n, dtype=torch.uint8, device=dev)
    s = make_shape(B, T, H, K, V, dt)
    st = lib().kda_chunk_fwd_scan(
        ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        int(chunk_size), _ptr(initial_state), _ptr(o), _ptr(fs), int(n_segments),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        _stream_ptr(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd_scan")
    return o, fs


def bwd_workspace_size(B, T, H, K, V, dtype=torch.bfloat16, has_segment_ids=False,
                       impl=None) -> int:
    """Workspace bytes of chunk_bwd for this shape (0 when unsupported):
    the AUTO choice (impl None) or what ``impl`` ("auto", "simt", "tc")
    needs."""
    s = make_shape(B, T, H, K, V, dtype)
    if impl is None:
        return int(lib().kda_chunk_bwd_workspace_size(ctypes.byref(s), int(bool(has_segment_ids))))
    return int(lib().kda_chunk_bwd_workspace_size_for(ctypes.byref(s), int(bool(has_segment_ids)),
                                                      IMPLS[impl]))


def bwd_workspace_size_packed(B, T, H, K, V, max_runs_per_row, dtype=torch.bfloat16) -> int:
    """Tensor-core backward workspace for inputs with segment ids and at most
    ``max_runs_per_row`` runs per row (0 when that path does not apply)."""
    s = make_shape(B, T, H, K, V, dtype)
    return int(lib().kda_chunk_bwd_workspace_size_packed(ctypes.byref(s), int(max_runs_per_row)))


def chunk_bwd(q, k, v, g, beta, d_o, scale=None, chunk_size=CHUNK, initial_state=None,
              segment_ids=None, d_final=None, want_d_initial=True, workspace=None,
              stream=None, impl="auto"):
    """Gradient of chunk_fwd on the GPU: given ``d_o`` [B,T,H,V] (dtype of q)
    and ``d_final`` [B,H,K,V] fp32 or None, returns fp32 ``(dq, dk, dv, dg,
    dbeta, d_initial or None)`` of ``sum(d_o * o) + sum(d_final *
    final_state)``.  Inputs as chunk_fwd; ``impl``: "auto" (the tensor cores
    where they apply), "tc" or "simt"."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("chunk_bwd needs CUDA tensors")
    dt = q.dtype
    _check(q, "q", (B, T, H, K), dt, dev)
    _check(k, "k", (B, T, H, K), dt, dev)
    _check(v, "v", (B, T, H, V), dt, dev)
    _check(d_o, "d_o", (B, T, H, V), dt, dev)
    _check(g, "g", (B, T, H, K), torch.float32, dev)
    _check(beta, "beta", (B, T, H), torch.float32, dev)
    _check(initial_state, "initial_state", (B, H, K, V), torch.float32, dev)
    _check(d_final, "d_final", (B, H, K, V), torch.float32, dev)
    _check(segment_ids, "segment_ids", (B, T), torch.int32, dev)
    if scale is None:
        scale = K ** -0.5
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dg = (torch.empty(B, T, H, K, **f32) for _ in range(3))
    dv = torch.empty(B, T, H, V, **f32)
    dbeta = torch.empty(B, T, H, **f32)
    d_init = torch.empty(B, H, K, V, **f32) if want_d_initial else None
    if workspace is None:
        n = bwd_workspace_size(B, T, H, K, V, dt, segment_ids is not None, impl)
        if n == 0:
            raise KdaError(2, "kda_chunk_bwd_workspace_size")
        workspace = torch.zeros(n, dtype=torch.uint8, device=dev)
    s = make_shape(B, T, H, K, V, dt)
    st = lib().kda_chunk_bwd_ex(
        ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        int(chunk_size), _ptr(initial_state), _ptr(segment_ids), _ptr(d_o), _ptr(d_final),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(d_init), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), IMPLS[impl],
        _stream_ptr(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_bwd_ex")
    return dq, dk, dv, dg, dbeta, d_init


def fwd_save_workspace_size(B, T, H, K, V, dtype=torch.bfloat16, has_segment_ids=False) -> int:
    """Workspace bytes of chunk_fwd_save (0 when that path does not apply)."""
    s = make_shape(B, T, H, K, V, dtype)
    return int(lib().kda_chunk_fwd_save_workspace_size(ctypes.byref(s), int(bool(has_segment_ids))))


def chunk_fwd_save(q, k, v, g, beta, scale=None, chunk_size=CHUNK, initial_state=None,
                   segment_ids=None, output_final_state=True, workspace=None, stream=None):
    """The forward of a training step (``kda_chunk_fwd_save``): returns
    ``(o, final_state or None, workspace)``, o and the final state as
    chunk_fwd's split path computes them, the workspace holding what
    chunk_bwd_from_saved reads.  bf16, K = V = 128."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("chunk_fwd_save needs CUDA tensors")
    dt = q.dtype
    _check(q, "q", (B, T, H, K), dt, dev)
    _check(k, "k", (B, T, H, K), dt, dev)
    _check(v, "v", (B, T, H, V), dt, dev)
    _check(g, "g", (B, T, H, K), torch.float32, dev)
    _check(beta, "beta", (B, T, H), torch.float32, dev)
    _check(initial_state, "initial_state", (B, H, K, V), torch.float32, dev)
    _check(segment_ids, "segment_ids", (B, T), torch.int32, dev)
    if scale is None:
        scale = K ** -0.5
    o = torch.empty(B, T, H, V, dtype=dt, device=dev)
    fs = torch.empty(B, H, K, V, dtype=torch.float32, device=dev) if output_final_state else None
    if workspace is None:
        n = fwd_save_workspace_size(B, T, H, K, V, dt, segment_ids is not None)
        if n == 0:
            raise KdaError(2, "kda_chunk_fwd_save_workspace_size")
        workspace = torch.zeros(n, dtype=torch.uint8, device=dev)
    s = make_shape(B, T, H, K, V, dt)
    st = lib().kda_chunk_fwd_save(
        ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        int(chunk_size), _ptr(initial_state), _ptr(segment_ids), _ptr(o), _ptr(fs),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        _stream_ptr(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd_save")
    return o, fs, workspace


def chunk_bwd_from_saved(q, k, v, g, beta, d_o, workspace, scale=None, chunk_size=CHUNK,
                         initial_state=None, segment_ids=None, d_final=None,
                         want_d_initial=True, stream=None):
    """The backward of a training step (``kda_chunk_bwd_from_saved``) on the
    workspace a chunk_fwd_save of the same inputs left: returns the
    gradients as chunk_bwd."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    dt = q.dtype
    _check(d_o, "d_o", (B, T, H, V), dt, dev)
    _check(d_final, "d_final", (B, H, K, V), torch.float32, dev)
    if scale is None:
        scale = K ** -0.5
    f32 = dict(dtype=torch.float32, device=dev)
    dq, dk, dg = (torch.empty(B, T, H, K, **f32) for _ in range(3))
    dv = torch.empty(B, T, H, V, **f32)
    dbeta = torch.empty(B, T, H, **f32)
    d_init = torch.empty(B, H, K, V, **f32) if want_d_initial else None
    s = make_shape(B, T, H, K, V, dt)
    st = lib().kda_chunk_bwd_from_saved(
        ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        int(chunk_size), _ptr(initial_state), _ptr(segment_ids), _ptr(d_o), _ptr(d_final),
        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(d_init), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _stream_ptr(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_bwd_from_saved")
    return dq, dk, dv, dg, dbeta, d_init


def short_conv_silu(x_q, x_k, x_v, w, segment_ids=None, l2norm_qk=True,
                    stream=None):
    """Segment-aware causal depthwise conv (width 4) + SiLU on q, k, v, then
    optional L2 norm of q and k.  x_q, x_k: [B,T,H,K]; x_v: [B,T,H,V];
    w: fp32 [3, H*K, 4] (q, k, v weight blocks; needs K == V) or a flat
    tensor of 4*(2*H*K + H*V) floats.  Returns (q, k, v)."""
    B, T, H, K = x_q.shape
    V = x_v.shape[-1]
    dev, dt = x_q.device, x_q.dtype
    _check(x_q, "x_q", (B, T, H, K), dt, dev)
    _check(x_k, "x_k", (B, T, H, K), dt, dev)
    _check(x_v, "x_v", (B, T, H, V), dt, dev)
    _check(segment_ids, "segment_ids", (B, T), torch.int32, dev)
    if w.dtype != torch.float32 or w.device != dev or not w.is_contiguous() \
            or w.numel() != 4 * (2 * H * K + H * V):
        raise ValueError("w must be contiguous fp32 with 4*(2*H*K + H*V) elements")
    q = torch.empty_like(x_q)
    k = torch.empty_like(x_k)
    v = torch.empty_like(x_v)
    s = make_shape(B, T, H, K, V, dt)
    st = lib().kda_short_conv_silu(
        ctypes.byref(s), _ptr(x_q), _ptr(x_k), _ptr(x_v), _ptr(w),
        _ptr(segment_ids), int(bool(l2norm_qk)), _ptr(q), _ptr(k), _ptr(v),
        _stream_ptr(stream, dev))
    if st != KDA_OK:
        raise KdaError(st, "kda_short_conv_silu")
    return q, k, v


def host_buffer_size(B, T, H, K, V, dtype=torch.bfloat16, has_segment_ids=False) -> int:
    """Bytes of device memory chunk_fwd_host needs for this shape."""
    s = make_shape(B, T, H, K, V, dtype)
    return int(lib().kda_chunk_fwd_host_buffer_size(ctypes.byref(s), 1 if has_segment_ids else 0))


def chunk_fwd_host(q, k, v, g, beta, scale=None, chunk_size=CHUNK, initial_state=None,
                   segment_ids=None, output_final_state=False, out=None,
                   final_state_out=None, device_buffer=None, stream=None):
    """End-to-end forward on HOST tensors (pin them for asynchronous copies):
    the library copies the inputs in, runs the forward and copies o (and the
    final state) back, pipelined over token ranges (over head groups with
    segment ids).  ``device_buffer`` is a
    zero-filled CUDA uint8 tensor of host_buffer_size() bytes (allocated here
    when None).  The host outputs are valid once ``stream`` synchronises.
    Returns ``(o, final_state or None)`` (CPU tensors)."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    cpu = torch.device("cpu")
    dt = q.dtype
    for t, name, shape, tdt in ((q, "q", (B, T, H, K), dt), (k, "k", (B, T, H, K), dt),
                                (v, "v", (B, T, H, V), dt),
                                (g, "g", (B, T, H, K), torch.float32),
                                (beta, "beta", (B, T, H), torch.float32),
                                (initial_state, "initial_state", (B, H, K, V), torch.float32),
                                (segment_ids, "segment_ids", (B, T), torch.int32)):
        _check(t, name, shape, tdt, cpu)
    if scale is None:
        scale = K ** -0.5
    o = out if out is not None else torch.empty(B, T, H, V, dtype=dt).pin_memory()
    _check(o, "out", (B, T, H, V), dt, cpu)
    fs = None
    if output_final_state:
        fs = final_state_out if final_state_out is not None else torch.empty(
            B, H, K, V, dtype=torch.float32).pin_memory()
        _check(fs, "final_state_out", (B, H, K, V), torch.float32, cpu)
    n = host_buffer_size(B, T, H, K, V, dt, segment_ids is not None)
    if n == 0:
        raise KdaError(2, "kda_chunk_fwd_host_buffer_size")
    dev = torch.device("cuda", torch.cuda.current_device())
    if device_buffer is None:
        device_buffer = torch.zeros(n, dtype=torch.uint8, device=dev)
    s = make_shape(B, T, H, K, V, dt)
    st = lib().kda_chunk_fwd_host(
        ctypes.byref(s), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
        int(chunk_size), _ptr(initial_state), _ptr(segment_ids), _ptr(o), _ptr(fs),
        _ptr(device_buffer), int(device_buffer.numel() * device_buffer.element_size()),
        _stream_ptr(stream, device_buffer.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_chunk_fwd_host")
    return o, fs


def read_device_status(workspace, stream=None) -> int:
    """Synchronise the stream and return the device status bits (0 = clean)."""
    bits = ctypes.c_uint32(0)
    st = lib().kda_read_device_status(_ptr(workspace), _stream_ptr(stream, workspace.device),
                                      ctypes.byref(bits))
    if st not in (KDA_OK, 4, 6, 7):
        raise KdaError(st, "kda_read_device_status")
    return int(bits.value)


def selftest_wait_timeout(workspace, limit_cycles=1 << 20, stream=None) -> None:
    """Enqueue the bounded-wait self-test: one device wait that nothing ends,
    given up after ``limit_cycles`` SM clocks, reported as KDA_DEVICE_TIMEOUT
    in ``workspace``'s status word (read it with read_device_status)."""
    st = lib().kda_selftest_wait_timeout(_ptr(workspace), int(limit_cycles),
                                         _stream_ptr(stream, workspace.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_selftest_wait_timeout")


def clear_device_status(workspace, stream=None) -> None:
    st = lib().kda_clear_device_status(_ptr(workspace), _stream_ptr(stream, workspace.device))
    if st != KDA_OK:
        raise KdaError(st, "kda_clear_device_status")
