"""fp64 CPU oracle for the chunked gated delta rule, forward and backward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference legs may import this package.  It shares no
code with the CUDA path (``chunked_gated_delta_gdr_gb300``) and never imports
it.

Two independent forms live here:

* ``recurrent`` -- the plain definition: the gated delta rule recurrence run
  token by token in fp64 (C, OpenMP over (segment, head) units;
  ``gdr_oracle.c``).  This is the oracle the GPU path is compared with.
* ``recurrent_bwd`` -- the gradients of ``recurrent``'s outputs with respect to
  all its inputs, by reverse-mode differentiation of the same token recurrence
  (C, ``gdr_oracle.c``).  Pinned by finite differences of ``recurrent``.
* ``chunked_wy`` -- the chunkwise (WY) form in fp64 numpy, used only on tiny
  inputs to cross-check ``recurrent`` and to expose the per-chunk
  intermediates (G, A, Tm, W, U, v_new, h).

Parity pins: ``recurrent`` is pinned by tests against closed forms, a
hand-worked example, invariants and the chunked form (see tests/).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .chunked_wy import chunked_wy  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdr_oracle.so")
_lock = threading.Lock()
_lib = None

_DT = {"float64": 0, "float32": 1, "bfloat16": 2}


def build(force: bool = False) -> str:
    """Compile gdr_oracle.c into a shared library (gcc, OpenMP, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O3", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def open_library(path: str):
    """ctypes handle to a compiled oracle library (the default one, or a
    variant compiled by a test from a modified copy of gdr_oracle.c)."""
    lib = ctypes.CDLL(path)
    vp, ci, cd = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.gdr_oracle_recurrent.argtypes = [
        vp, ci, vp, ci, vp, ci, vp, ci, vp, ci, cd, vp, ci, vp,
        ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, vp, vp, ci]
    lib.gdr_oracle_recurrent.restype = ci
    lib.gdr_oracle_recurrent_ckpt.argtypes = [
        vp, ci, vp, ci, vp, ci, vp, ci, vp, ci, cd, vp, ci, vp,
        ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, vp, vp, ctypes.c_int32, vp, vp, ci]
    lib.gdr_oracle_recurrent_ckpt.restype = ci
    lib.gdr_oracle_recurrent_bwd.argtypes = [
        vp, ci, vp, ci, vp, ci, vp, ci, vp, ci, cd, vp, ci, vp,
        ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, vp, ci, vp, ci, vp, vp, vp, vp, vp, vp, ci]
    lib.gdr_oracle_recurrent_bwd.restype = ci
    lib.gdr_oracle_max_threads.restype = ci
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def max_threads() -> int:
    return int(_load().gdr_oracle_max_threads())


def _as_np(x):
    """Return (contiguous numpy array, dtype code); bf16 stays as raw bits."""
    if x is None:
        return None, 0
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), _DT["bfloat16"]
            x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, _DT["float64"]
    if x.dtype == np.float32:
        return x, _DT["float32"]
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


def recurrent(q, k, v, g, beta, scale, h0, cu_seqlens, want_ht=True,
              o_init=np.nan, n_threads=0, lib=None):
    """Token-by-token fp64 recurrence.

    Arguments are torch tensors or numpy arrays in the layouts
    q, k [T, Hk, dk]; v [T, H, dv]; g, beta [T, H]; h0 [N, H, dk, dv] or None;
    cu_seqlens [N + 1] int32.  Returns (o [T, H, dv] float64, ht [N, H, dk, dv]
    float64 or None).  Tokens outside every segment keep ``o_init``.
    ``lib`` selects another compiled copy of the oracle (tests only).
    """
    lib = _load() if lib is None else lib
    qa, qd = _as_np(q)
    ka, kd = _as_np(k)
    va, vd = _as_np(v)
    ga, gd = _as_np(g)
    ba, bd = _as_np(beta)
    ha, hd = _as_np(h0)
    try:
        import torch
        if isinstance(cu_seqlens, torch.Tensor):
            cu_seqlens = cu_seqlens.cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, Hk, dk = qa.shape
    H, dv = va.shape[1], va.shape[2]
    n_seq = cu.shape[0] - 1
    o = np.full((T, H, dv), o_init, dtype=np.float64)
    ht = np.zeros((n_seq, H, dk, dv), dtype=np.float64) if want_ht else None
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = lib.gdr_oracle_recurrent(
        ptr(qa), qd, ptr(ka), kd, ptr(va), vd, ptr(ga), gd, ptr(ba), bd,
        float(scale), ptr(ha), hd, ptr(cu), n_seq, T, Hk, H, dk, dv,
        ptr(o), ptr(ht), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_recurrent failed with code {rc}")
    return o, ht


def recurrent_checkpoints(q, k, v, g, beta, scale, h0, cu_seqlens, ckpt_every, want_ht=True,
                          o_init=np.nan, n_threads=0, lib=None):
    """``recurrent`` plus state checkpoints every ``ckpt_every`` tokens of each segment.

    Returns (o, ht, ckpt [rows, H, dk, dv] float64, ckpt_off [N + 1] int32): checkpoint m
    (1-based) of segment n is row ckpt_off[n] + m - 1, the state after the segment's first
    m * ckpt_every tokens.
    """
    lib = _load() if lib is None else lib
    qa, qd = _as_np(q)
    ka, kd = _as_np(k)
    va, vd = _as_np(v)
    ga, gd = _as_np(g)
    ba, bd = _as_np(beta)
    ha, hd = _as_np(h0)
    try:
        import torch
        if isinstance(cu_seqlens, torch.Tensor):
            cu_seqlens = cu_seqlens.cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, Hk, dk = qa.shape
    H, dv = va.shape[1], va.shape[2]
    n_seq = cu.shape[0] - 1
    o = np.full((T, H, dv), o_init, dtype=np.float64)
    ht = np.zeros((n_seq, H, dk, dv), dtype=np.float64) if want_ht else None
    rows = max(T // int(ckpt_every), 1)
    ckpt = np.zeros((rows, H, dk, dv), dtype=np.float64)
    off = np.zeros(n_seq + 1, dtype=np.int32)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = lib.gdr_oracle_recurrent_ckpt(
        ptr(qa), qd, ptr(ka), kd, ptr(va), vd, ptr(ga), gd, ptr(ba), bd,
        float(scale), ptr(ha), hd, ptr(cu), n_seq, T, Hk, H, dk, dv,
        ptr(o), ptr(ht), int(ckpt_every), ptr(ckpt), ptr(off), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_recurrent_ckpt failed with code {rc}")
    return o, ht, ckpt[:off[-1]], off


def recurrent_bwd(q, k, v, g, beta, scale, h0, cu_seqlens, dout, dht=None, n_threads=0,
                  lib=None):
    """Gradients of the token recurrence (fp64) for upstream gradients ``dout``
    (dL/do, [T, H, dv]) and ``dht`` (dL/dht, [N, H, dk, dv] or None for zero).

    Returns (dq [T, Hk, dk], dk [T, Hk, dk], dv [T, H, dv], dg [T, H], dbeta [T, H],
    dh0 [N, H, dk, dv]), all float64.  dq and dk sum the value heads that share a
    query/key head (in head order); tokens outside every segment get zeros; dh0 is
    returned whether or not ``h0`` is given (the gradient for a zero initial state).
    """
    lib = _load() if lib is None else lib
    qa, qd = _as_np(q)
    ka, kd = _as_np(k)
    va, vd = _as_np(v)
    ga, gd = _as_np(g)
    ba, bd = _as_np(beta)
    ha, hd = _as_np(h0)
    da, dd = _as_np(dout)
    ta, td = _as_np(dht)
    try:
        import torch
        if isinstance(cu_seqlens, torch.Tensor):
            cu_seqlens = cu_seqlens.cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    T, Hk, dk = qa.shape
    H, dv = va.shape[1], va.shape[2]
    n_seq = cu.shape[0] - 1
    dq_h = np.zeros((T, H, dk), dtype=np.float64)
    dk_h = np.zeros((T, H, dk), dtype=np.float64)
    dvo = np.zeros((T, H, dv), dtype=np.float64)
    dg = np.zeros((T, H), dtype=np.float64)
    db = np.zeros((T, H), dtype=np.float64)
    dh0 = np.zeros((n_seq, H, dk, dv), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    rc = lib.gdr_oracle_recurrent_bwd(
        ptr(qa), qd, ptr(ka), kd, ptr(va), vd, ptr(ga), gd, ptr(ba), bd,
        float(scale), ptr(ha), hd, ptr(cu), n_seq, T, Hk, H, dk, dv,
        ptr(da), dd, ptr(ta), td, ptr(dq_h), ptr(dk_h), ptr(dvo), ptr(dg), ptr(db),
        ptr(dh0), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"gdr_oracle_recurrent_bwd failed with code {rc}")
    group = H // Hk
    dq = dq_h.reshape(T, Hk, group, dk).sum(axis=2)
    dkk = dk_h.reshape(T, Hk, group, dk).sum(axis=2)
    return dq, dkk, dvo, dg, db, dh0
