"""fp64 CPU oracle for the chunked KDA forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The GPU
library (``gated_delta_rule_21_gb300``) never imports it and shares no code with
it; the only thing both sides use is the seeded input generator
(``kda_inputs``), which holds none of the method's arithmetic.

Every function here is the plain definition of what the path computes, in
float64, following page "feat(kda): integrate KDA attention with tokamax backend
and CP support":

* :func:`kda_forward` -- section "Delta Rule formulation", one token at a time
  (C, ``kda_ref.c``), with the packed-sequence semantics of section
  "Public API" (segment ids [B,T], 1-based, 0 = padding).
* :func:`short_conv_silu` -- section "Layer architecture", step 1 (causal
  depthwise conv + SiLU), segment-aware.
* :func:`l2norm` -- section "Layer architecture", step 5 / "Public API"
  ``use_qk_l2norm_in_kernel``.
* :func:`kda_backward` -- the gradient of :func:`kda_forward` (its
  vector-Jacobian product), reverse-mode differentiation of the same token
  recurrence written out step by step (C, ``kda_ref_bwd.c``).

Pins (tests/test_oracle.py) check these against closed forms, invariants and an
independent brute-force transcription; see the test file for which property
pins which step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "kda_ref.c"), os.path.join(_HERE, "kda_ref_bwd.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_ref.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``kda_ref.c`` and ``kda_ref_bwd.c`` into
    ``oracle/_build/libkda_ref.so`` with gcc.

    Plain -O2, no fast-math (IEEE fp64 exp and arithmetic), no
    machine-specific flags, so it builds the same on x86_64 and aarch64.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-o", tmp] + _SRCS + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    lib.kda_ref_forward.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, dp, dp, dp, dp, dp, ctypes.c_double, dp, ip,
        dp, dp, ctypes.c_int]
    lib.kda_ref_forward.restype = ctypes.c_int
    lib.kda_ref_backward.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, dp, dp, dp, dp, dp, ctypes.c_double, dp, ip,
        dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
    lib.kda_ref_backward.restype = ctypes.c_int
    lib.kda_ref_short_conv_silu.argtypes = [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp,
        dp, ip, dp]
    lib.kda_ref_short_conv_silu.restype = ctypes.c_int
    lib.kda_ref_l2norm_rows.argtypes = [
        ctypes.c_long, ctypes.c_int, ctypes.c_double, dp]
    lib.kda_ref_l2norm_rows.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


class use_library:
    """Context manager that points this module at another build of the
    oracle's C source (the mutation tests use it to plant mistakes)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _f64(x):
    """Exact upcast to a C-contiguous float64 numpy array (bf16/fp32 -> fp64
    is exact)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def kda_forward(q, k, v, g, beta, scale=None, initial_state=None,
                segment_ids=None, output_final_state=True, threads=None):
    """Token-by-token fp64 KDA forward.

    q, k, g: [B,T,H,K]; v: [B,T,H,V]; beta: [B,T,H]; initial_state:
    [B,H,K,V] or None (zeros); segment_ids: [B,T] int32 or None (all ones).
    ``scale`` None means K**-0.5.  Returns ``(o [B,T,H,V], final_state
    [B,H,K,V] or None)`` as float64 numpy arrays.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    S0 = _f64(initial_state)
    seg = _i32(segment_ids)
    B, T, H, K = q.shape
    V = v.shape[-1]
    assert k.shape == (B, T, H, K) and g.shape == (B, T, H, K)
    assert v.shape == (B, T, H, V) and beta.shape == (B, T, H)
    if S0 is not None:
        assert S0.shape == (B, H, K, V)
    if seg is not None:
        assert seg.shape == (B, T)
    if scale is None:
        scale = K ** -0.5
    o = np.zeros((B, T, H, V), dtype=np.float64)
    fs = np.zeros((B, H, K, V), dtype=np.float64) if output_final_state else None
    n = threads if threads is not None else default_threads()
    dp, ip = ctypes.c_double, ctypes.c_int32
    rc = _load().kda_ref_forward(
        B, T, H, K, V, _ptr(q, dp), _ptr(k, dp), _ptr(v, dp), _ptr(g, dp),
        _ptr(beta, dp), float(scale), _ptr(S0, dp), _ptr(seg, ip),
        _ptr(o, dp), _ptr(fs, dp), int(n))
    if rc != 0:
        raise RuntimeError(f"kda_ref_forward failed with status {rc}")
    return o, fs


def kda_backward(q, k, v, g, beta, scale=None, initial_state=None, segment_ids=None,
                 d_o=None, d_final=None, threads=None):
    """fp64 gradient of :func:`kda_forward`: reverse-mode differentiation of
    the token recurrence, given the upstream gradients ``d_o`` [B,T,H,V] of o
    and ``d_final`` [B,H,K,V] of the final state (None = zeros).  Returns
    ``(dq, dk, dv, dg, dbeta, d_initial)`` as float64 numpy arrays (layouts
    of q, k, v, g, beta and the state); ``d_initial`` is the gradient with
    respect to the initial state (a zero one when none is given).
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    S0 = _f64(initial_state)
    seg = _i32(segment_ids)
    B, T, H, K = q.shape
    V = v.shape[-1]
    dO = _f64(d_o) if d_o is not None else np.zeros((B, T, H, V))
    dF = _f64(d_final)
    assert dO.shape == (B, T, H, V)
    if dF is not None:
        assert dF.shape == (B, H, K, V)
    if scale is None:
        scale = K ** -0.5
    dq = np.zeros((B, T, H, K)); dk = np.zeros((B, T, H, K)); dg = np.zeros((B, T, H, K))
    dv = np.zeros((B, T, H, V)); dbeta = np.zeros((B, T, H)); dS0 = np.zeros((B, H, K, V))
    n = threads if threads is not None else default_threads()
    dp, ip = ctypes.c_double, ctypes.c_int32
    rc = _load().kda_ref_backward(
        B, T, H, K, V, _ptr(q, dp), _ptr(k, dp), _ptr(v, dp), _ptr(g, dp),
        _ptr(beta, dp), float(scale), _ptr(S0, dp), _ptr(seg, ip), _ptr(dO, dp),
        _ptr(dF, dp), _ptr(dq, dp), _ptr(dk, dp), _ptr(dv, dp), _ptr(dg, dp),
        _ptr(dbeta, dp), _ptr(dS0, dp), int(n))
    if rc != 0:
        raise RuntimeError(f"kda_ref_backward failed with status {rc}")
    return dq, dk, dv, dg, dbeta, dS0


def short_conv_silu(x, w, segment_ids=None):
    """Segment-aware causal depthwise conv + SiLU, fp64.

    x: [B,T,C]; w: [C,W] (w[:, W-1] multiplies the current token);
    segment_ids: [B,T] or None.  Returns y [B,T,C] float64.
    """
    x = _f64(x)
    w = _f64(w)
    seg = _i32(segment_ids)
    B, T, C = x.shape
    assert w.shape[0] == C
    W = w.shape[1]
    y = np.zeros_like(x)
    dp, ip = ctypes.c_double, ctypes.c_int32
    rc = _load().kda_ref_short_conv_silu(B, T, C, W, _ptr(x, dp), _ptr(w, dp),
                                         _ptr(seg, ip), _ptr(y, dp))
    if rc != 0:
        raise RuntimeError(f"kda_ref_short_conv_silu failed with status {rc}")
    return y


def l2norm(x, head_dim, eps=1e-6):
    """x / sqrt(sum x^2 + eps) over groups of ``head_dim`` trailing channels."""
    x = _f64(x).copy()
    N = x.size // head_dim
    rc = _load().kda_ref_l2norm_rows(N, head_dim, float(eps),
                                     _ptr(x.reshape(-1), ctypes.c_double))
    if rc != 0:
        raise RuntimeError("kda_ref_l2norm_rows failed")
    return x


def round_bf16(x):
    """Round a float64 array to the nearest bfloat16 (ties to even) and return
    it as float64 -- the storage rounding of a bf16 intermediate."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return t.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
