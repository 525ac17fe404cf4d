"""Python binding of libgdr: argument marshalling only.

Every step of the forward runs in libgdr's CUDA kernels; this module builds
the C descriptors from torch tensors, allocates outputs and scratch through
PyTorch's allocator, and passes torch's current CUDA stream.  There is no CPU
fallback: without libgdr.so or a GB300 the calls raise.

Host (CPU) tensors are accepted by ``chunk_fwd``: they are copied to the
current CUDA device on the current stream (asynchronously when pinned), the
forward runs there, and o / ht are copied back into host tensors.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _native as nat

_DT = {torch.bfloat16: nat.GDR_BF16, torch.float32: nat.GDR_F32, torch.int32: nat.GDR_I32}


class _Desc:
    """A gdr_tensor_t for a torch tensor (keeps the strides array alive)."""

    def __init__(self, t: torch.Tensor):
        if t.dtype not in _DT:
            raise TypeError(f"unsupported dtype {t.dtype}")
        if t.dim() < 1 or t.dim() > 4:
            raise ValueError("tensors must have 1..4 dims")
        self.strides = (ctypes.c_int64 * t.dim())(*t.stride())
        shape = (ctypes.c_int64 * 4)(*(list(t.shape) + [0] * (4 - t.dim())))
        self.c = nat.GdrTensor(ctypes.c_void_p(t.data_ptr() if t.numel() else 0), _DT[t.dtype],
                               t.dim(), shape,
                               ctypes.cast(self.strides, ctypes.POINTER(ctypes.c_int64)))

    @property
    def ref(self):
        return ctypes.byref(self.c)


def _d(t: Optional[torch.Tensor]):
    return None if t is None else _Desc(t)


def _ref(d):
    return None if d is None else d.ref


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def chunk_count_bound(T: int, n_seq: int) -> int:
    return int(nat.lib().gdr_chunk_count_bound(T, n_seq))


def workspace_bytes(T: int, n_seq: int, H: int, dk: int, dv: int, path: str = "auto") -> int:
    return int(nat.lib().gdr_chunk_fwd_workspace_bytes(T, n_seq, H, dk, dv, nat.PATHS[path]))


def stage_workspace_bytes(T: int, n_seq: int) -> int:
    return int(nat.lib().gdr_stage_workspace_bytes(T, n_seq))


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
              beta: torch.Tensor, scale: Optional[float] = None,
              initial_state: Optional[torch.Tensor] = None,
              cu_seqlens: Optional[torch.Tensor] = None, output_final_state: bool = False,
              path: str = "auto", workspace: Optional[torch.Tensor] = None,
              out: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
              stream: Optional[torch.cuda.Stream] = None
              ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked gated delta rule forward (libgdr ``gdr_chunk_fwd_ws``).

    q, k [T, Hk, dk] bf16; v [T, H, dv] bf16; g [T, H] f32; beta [T, H] bf16;
    initial_state [N, H, dk, dv] f32 or None; cu_seqlens [N + 1] int32 (None:
    one segment of T tokens).  Returns (o [T, H, dv] bf16, ht or None).
    """
    host = q.device.type == "cpu"
    if host:
        piped = _chunk_fwd_host_pipelined(q, k, v, g, beta, scale, initial_state, cu_seqlens,
                                          output_final_state, path, out, final_state)
        if piped is not None:
            return piped
        dev = torch.device("cuda", torch.cuda.current_device())
        mv = lambda t: None if t is None else t.to(dev, non_blocking=True)
        q, k, v, g, beta, initial_state = map(mv, (q, k, v, g, beta, initial_state))
        cu_seqlens = mv(cu_seqlens)
    dev = q.device
    T, H, dv = q.shape[0], v.shape[1], v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    n_seq = cu_seqlens.numel() - 1
    if scale is None:
        scale = q.shape[-1] ** -0.5
    o = torch.empty(T, H, dv, dtype=torch.bfloat16, device=dev) if (out is None or host) else out
    ht = None
    if output_final_state:
        ht = (torch.empty(n_seq, H, q.shape[-1], dv, dtype=torch.float32, device=dev)
              if (final_state is None or host) else final_state)
    if workspace is None:
        workspace = _workspace(workspace_bytes(T, n_seq, H, q.shape[-1], dv, path), dev)
    ds = [_Desc(t) for t in (q, k, v, g, beta)]
    dh0, do, dht = _d(initial_state), _Desc(o), _d(ht)
    rc = nat.lib().gdr_chunk_fwd_ws(
        ds[0].ref, ds[1].ref, ds[2].ref, ds[3].ref, ds[4].ref, ctypes.c_float(scale),
        _ref(dh0), _ptr(cu_seqlens), n_seq, do.ref, _ref(dht), nat.PATHS[path],
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream(stream))
    nat.check(rc, "gdr_chunk_fwd_ws")
    if host:
        o_h = out if out is not None else torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        o_h.copy_(o, non_blocking=True)
        ht_h = None
        if ht is not None:
            ht_h = final_state if final_state is not None else torch.empty(
                ht.shape, dtype=ht.dtype, pin_memory=True)
            ht_h.copy_(ht, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return o_h, ht_h
    return o, ht


def _segment_bounds(cu, T: int):
    """Segment bounds after the library's reading of cu_seqlens (clamped to [0, T],
    made non-decreasing by a running maximum)."""
    b, prev = [], 0
    for i, c in enumerate(int(x) for x in cu):
        c = min(max(c, 0), T)
        if i > 0 and c < prev:
            c = prev
        b.append(c)
        prev = c
    return b


def _segment_groups(bounds, parts: int):
    """Cut the segments into at most `parts` runs of consecutive segments with about
    equal token counts: [(first segment, end segment), ...], none without tokens."""
    n, total = len(bounds) - 1, bounds[-1] - bounds[0]
    groups, n0 = [], 0
    for gi in range(parts):
        target = bounds[0] + total * (gi + 1) // parts
        n1 = n0
        while n1 < n and (bounds[n1] < target or n1 == n0):
            n1 += 1
        if gi == parts - 1:
            n1 = n
        if bounds[n1] > bounds[n0]:
            groups.append((n0, n1))
        elif groups and n1 > n0:
            groups[-1] = (groups[-1][0], n1)  # trailing empty segments join the last run
        n0 = n1
        if n0 >= n:
            break
    if groups and groups[-1][1] < n:
        groups[-1] = (groups[-1][0], n)
    return groups


_PIPE_MIN_TOKENS = 16384  # below this one copy-compute-copy sequence is as fast
_PIPE_PARTS = 4


def _chunk_fwd_host_pipelined(q, k, v, g, beta, scale, initial_state, cu_seqlens,
                              output_final_state, path, out, final_state, parts=_PIPE_PARTS,
                              min_tokens=_PIPE_MIN_TOKENS):
    """Host tensors: cut the packed tokens at segment boundaries into a few runs and give
    each run its own stream (copy in, forward, copy out), so that uploads use parallel
    copy engines and downloads overlap later uploads.  Segments are independent and each
    run computes its segments exactly as one call would (whole, never split into
    pieces), so the results are bit-identical to a single call.  Returns None when the
    call is too small, has a single run, or would use the sequence split."""
    T, Hk, dk = q.shape
    H, dv = v.shape[1], v.shape[2]
    if cu_seqlens is None or path not in ("auto", "fused", "fused_whole") or parts < 2:
        return None
    if T < min_tokens:
        return None
    n_seq = cu_seqlens.numel() - 1
    if path != "fused_whole" and split_pieces(T, n_seq, H) > 1:
        return None
    if not all(t.is_pinned() for t in (q, k, v, g, beta)):
        return None
    bounds = _segment_bounds(cu_seqlens.tolist(), T)
    groups = _segment_groups(bounds, parts)
    if len(groups) < 2:
        return None
    dev = torch.device("cuda", torch.cuda.current_device())
    main = torch.cuda.current_stream(dev)
    if scale is None:
        scale = dk ** -0.5
    o_h = out if out is not None else torch.empty(T, H, dv, dtype=torch.bfloat16,
                                                  pin_memory=True)
    ht_h = None
    if output_final_state:
        ht_h = final_state if final_state is not None else torch.empty(
            n_seq, H, dk, dv, dtype=torch.float32, pin_memory=True)
    bufs = {name: torch.empty(t.shape, dtype=t.dtype, device=dev)
            for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta))}
    o_d = torch.empty(T, H, dv, dtype=torch.bfloat16, device=dev)
    h0_d = (torch.empty(initial_state.shape, dtype=initial_state.dtype, device=dev)
            if initial_state is not None else None)
    ht_d = torch.empty(n_seq, H, dk, dv, dtype=torch.float32, device=dev) if ht_h is not None else None
    # fused path (the device copies are aligned) with every (segment, head) whole
    gpath = "fused_whole" if path in ("auto", "fused", "fused_whole") else path
    work = [(_workspace(workspace_bytes(bounds[n1] - bounds[n0], n1 - n0, H, dk, dv, gpath), dev))
            for n0, n1 in groups]
    cus = [torch.tensor([b - bounds[n0] for b in bounds[n0:n1 + 1]], dtype=torch.int32)
           .pin_memory() for n0, n1 in groups]
    ready = torch.cuda.Event()
    ready.record(main)
    streams = [torch.cuda.Stream(dev) for _ in groups]
    for (n0, n1), st, ws, cu_h in zip(groups, streams, work, cus):
        st.wait_event(ready)
        t0, t1 = bounds[n0], bounds[n1]
        with torch.cuda.stream(st):
            for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
                bufs[name][t0:t1].copy_(t[t0:t1], non_blocking=True)
            cu_d = cu_h.to(dev, non_blocking=True)
            h0g = None
            if h0_d is not None:
                h0_d[n0:n1].copy_(initial_state[n0:n1], non_blocking=True)
                h0g = h0_d[n0:n1]
            chunk_fwd(bufs["q"][t0:t1], bufs["k"][t0:t1], bufs["v"][t0:t1], bufs["g"][t0:t1],
                      bufs["beta"][t0:t1], scale=scale, initial_state=h0g, cu_seqlens=cu_d,
                      output_final_state=ht_d is not None, path=gpath, workspace=ws,
                      out=o_d[t0:t1], final_state=None if ht_d is None else ht_d[n0:n1],
                      stream=st)
            o_h[t0:t1].copy_(o_d[t0:t1], non_blocking=True)
            if ht_d is not None:
                ht_h[n0:n1].copy_(ht_d[n0:n1], non_blocking=True)
    for st in streams:
        st.synchronize()
    return o_h, ht_h


def bwd_workspace_bytes(T: int, n_seq: int, Hk: int, H: int, dk: int, dv: int) -> int:
    return int(nat.lib().gdr_chunk_bwd_workspace_bytes(T, n_seq, Hk, H, dk, dv))


def chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
              beta: torch.Tensor, dout: torch.Tensor, scale: Optional[float] = None,
              initial_state: Optional[torch.Tensor] = None,
              cu_seqlens: Optional[torch.Tensor] = None, dht: Optional[torch.Tensor] = None,
              want_dh0: bool = True, workspace: Optional[torch.Tensor] = None,
              stream: Optional[torch.cuda.Stream] = None, out: Optional[tuple] = None):
    """Backward of ``chunk_fwd`` (libgdr ``gdr_chunk_bwd``): gradients of the loss with
    respect to q, k, v, g, beta and the initial state, given dout = dL/do [T, H, dv] bf16
    and dht = dL/dht [N, H, dk, dv] f32 (None: zero).

    Returns (dq [T, Hk, dk], dk [T, Hk, dk], dv [T, H, dv], dg [T, H], dbeta [T, H],
    dh0 [N, H, dk, dv] or None), all fp32 on the inputs' device; ``out`` may give these six
    tensors (compact, fp32, on that device; dh0 may be None) to be written instead.  Host
    (CPU) inputs are copied to the current CUDA device, and the gradients back into pinned
    host tensors (``out`` then names host tensors).
    """
    if q.device.type == "cpu":
        piped = _chunk_bwd_host_pipelined(q, k, v, g, beta, dout, scale, initial_state,
                                          cu_seqlens, dht, want_dh0, out)
        if piped is not None:
            return piped
        dev = torch.device("cuda", torch.cuda.current_device())
        mv = lambda t: None if t is None else t.to(dev, non_blocking=True)
        res = chunk_bwd(*map(mv, (q, k, v, g, beta, dout)), scale=scale,
                        initial_state=mv(initial_state), cu_seqlens=mv(cu_seqlens), dht=mv(dht),
                        want_dh0=want_dh0, workspace=workspace, stream=stream)
        outs = []
        for i, t in enumerate(res):
            if t is None:
                outs.append(None)
                continue
            h = out[i] if out is not None else torch.empty(t.shape, dtype=t.dtype,
                                                           pin_memory=True)
            h.copy_(t, non_blocking=True)
            outs.append(h)
        torch.cuda.current_stream().synchronize()
        return tuple(outs)
    dev = q.device
    T, Hk, dk_ = q.shape
    H, dv_ = v.shape[1], v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    n_seq = cu_seqlens.numel() - 1
    if scale is None:
        scale = dk_ ** -0.5
    f32 = dict(dtype=torch.float32, device=dev)
    if out is not None:
        dq, dkk, dvv, dg, db, dh0 = out
        if not want_dh0:
            dh0 = None
    else:
        dq, dkk = torch.empty(T, Hk, dk_, **f32), torch.empty(T, Hk, dk_, **f32)
        dvv, dg = torch.empty(T, H, dv_, **f32), torch.empty(T, H, **f32)
        db = torch.empty(T, H, **f32)
        dh0 = torch.empty(n_seq, H, dk_, dv_, **f32) if want_dh0 else None
    if workspace is None:
        workspace = _workspace(bwd_workspace_bytes(T, n_seq, Hk, H, dk_, dv_), dev)
    ins = [_Desc(t) for t in (q, k, v, g, beta)]
    outs = [_Desc(t) for t in (dq, dkk, dvv, dg, db)]
    d_h0, d_do, d_dht, d_dh0 = _d(initial_state), _Desc(dout), _d(dht), _d(dh0)
    rc = nat.lib().gdr_chunk_bwd(
        ins[0].ref, ins[1].ref, ins[2].ref, ins[3].ref, ins[4].ref, ctypes.c_float(scale),
        _ref(d_h0), _ptr(cu_seqlens), n_seq, d_do.ref, _ref(d_dht), outs[0].ref, outs[1].ref,
        outs[2].ref, outs[3].ref, outs[4].ref, _ref(d_dh0), ctypes.c_void_p(workspace.data_ptr()),
        workspace.numel(), _stream(stream))
    nat.check(rc, "gdr_chunk_bwd")
    return dq, dkk, dvv, dg, db, dh0


def _chunk_bwd_host_pipelined(q, k, v, g, beta, dout, scale, initial_state, cu_seqlens, dht,
                              want_dh0, out, parts=_PIPE_PARTS, min_tokens=_PIPE_MIN_TOKENS):
    """Host tensors: the backward of runs of whole segments on separate streams (copy in,
    backward, copy out), as the forward's host path does; segments are independent, so
    the gradients equal a single call's.  Gradients of tokens outside every segment are
    zero.  Returns None when the call is too small or has a single run."""
    T, Hk, dk = q.shape
    H, dv = v.shape[1], v.shape[2]
    if cu_seqlens is None or parts < 2 or T < min_tokens:
        return None
    if not all(t.is_pinned() for t in (q, k, v, g, beta, dout)):
        return None
    n_seq = cu_seqlens.numel() - 1
    bounds = _segment_bounds(cu_seqlens.tolist(), T)
    groups = _segment_groups(bounds, parts)
    if len(groups) < 2:
        return None
    dev = torch.device("cuda", torch.cuda.current_device())
    main = torch.cuda.current_stream(dev)
    if scale is None:
        scale = dk ** -0.5
    shapes = [(T, Hk, dk), (T, Hk, dk), (T, H, dv), (T, H), (T, H), (n_seq, H, dk, dv)]
    outs_h = list(out) if out is not None else [
        torch.empty(sh, dtype=torch.float32, pin_memory=True) for sh in shapes]
    if not want_dh0:
        outs_h[5] = None
    for t in outs_h[:5]:  # tokens outside every segment
        t[:bounds[0]].zero_()
        t[bounds[-1]:].zero_()
    ins = {name: torch.empty(t.shape, dtype=t.dtype, device=dev)
           for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("do", dout))}
    outs_d = [torch.empty(sh, dtype=torch.float32, device=dev) for sh in shapes[:5]]
    outs_d.append(torch.empty(shapes[5], dtype=torch.float32, device=dev) if want_dh0 else None)
    h0_d = (torch.empty(initial_state.shape, dtype=initial_state.dtype, device=dev)
            if initial_state is not None else None)
    dht_d = torch.empty(dht.shape, dtype=dht.dtype, device=dev) if dht is not None else None
    work = [_workspace(bwd_workspace_bytes(bounds[n1] - bounds[n0], n1 - n0, Hk, H, dk, dv), dev)
            for n0, n1 in groups]
    cus = [torch.tensor([b - bounds[n0] for b in bounds[n0:n1 + 1]], dtype=torch.int32)
           .pin_memory() for n0, n1 in groups]
    ready = torch.cuda.Event()
    ready.record(main)
    streams = [torch.cuda.Stream(dev) for _ in groups]
    for (n0, n1), st, ws, cu_h in zip(groups, streams, work, cus):
        st.wait_event(ready)
        t0, t1 = bounds[n0], bounds[n1]
        with torch.cuda.stream(st):
            for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta),
                            ("do", dout)):
                ins[name][t0:t1].copy_(t[t0:t1], non_blocking=True)
            cu_d = cu_h.to(dev, non_blocking=True)
            h0g = dhtg = None
            if h0_d is not None:
                h0_d[n0:n1].copy_(initial_state[n0:n1], non_blocking=True)
                h0g = h0_d[n0:n1]
            if dht_d is not None:
                dht_d[n0:n1].copy_(dht[n0:n1], non_blocking=True)
                dhtg = dht_d[n0:n1]
            og = tuple(o[t0:t1] for o in outs_d[:5]) + (
                outs_d[5][n0:n1] if outs_d[5] is not None else None,)
            chunk_bwd(ins["q"][t0:t1], ins["k"][t0:t1], ins["v"][t0:t1], ins["g"][t0:t1],
                      ins["beta"][t0:t1], ins["do"][t0:t1], scale=scale, initial_state=h0g,
                      cu_seqlens=cu_d, dht=dhtg, want_dh0=want_dh0, workspace=ws, stream=st,
                      out=og)
            for oh, od in zip(outs_h[:5], outs_d[:5]):
                oh[t0:t1].copy_(od[t0:t1], non_blocking=True)
            if want_dh0:
                outs_h[5][n0:n1].copy_(outs_d[5][n0:n1], non_blocking=True)
    for st in streams:
        st.synchronize()
    return tuple(outs_h)


class _ChunkGatedDeltaRule(torch.autograd.Function):
    """Autograd wrapper: the forward and backward each run in libgdr."""

    @staticmethod
    def forward(ctx, q, k, v, g, beta, scale, initial_state, cu_seqlens, output_final_state):
        o, ht = chunk_fwd(q, k, v, g, beta, scale=scale, initial_state=initial_state,
                          cu_seqlens=cu_seqlens, output_final_state=output_final_state)
        ctx.save_for_backward(q, k, v, g, beta, initial_state, cu_seqlens)
        ctx.scale = scale
        return o, ht

    @staticmethod
    def backward(ctx, do, dht):
        q, k, v, g, beta, h0, cu = ctx.saved_tensors
        dq, dk, dv, dg, db, dh0 = chunk_bwd(
            q, k, v, g, beta, do.to(torch.bfloat16).contiguous(), scale=ctx.scale,
            initial_state=h0, cu_seqlens=cu,
            dht=None if dht is None else dht.float().contiguous(),
            want_dh0=h0 is not None and ctx.needs_input_grad[6])
        return (dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype), dg.to(g.dtype),
                db.to(beta.dtype), None, dh0, None, None)


def chunk_gated_delta_rule(q, k, v, g, beta, scale: Optional[float] = None,
                           initial_state: Optional[torch.Tensor] = None,
                           output_final_state: bool = False,
                           cu_seqlens: Optional[torch.Tensor] = None):
    """Differentiable chunked gated delta rule: (o, ht) = forward, gradients through
    ``chunk_bwd``.  Layouts as ``chunk_fwd``; device tensors only."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, q.shape[0]], dtype=torch.int32, device=q.device)
    return _ChunkGatedDeltaRule.apply(q, k, v, g, beta, scale, initial_state, cu_seqlens,
                                      output_final_state)


def split_pieces(T: int, n_seq: int, H: int) -> int:
    """Pieces per long segment of the fused path's sequence split on the current device
    (1: the fused path runs every (segment, head) whole)."""
    return int(nat.lib().gdr_fused_split_pieces(T, n_seq, H))


def split_plan(units: int, sms: int) -> tuple:
    """The split planner for ``units`` (segment, value head) pairs on ``sms`` SMs:
    (pieces per long segment, first piece's weight); (1, 1) means no split."""
    lead = ctypes.c_int32(1)
    pieces = int(nat.lib().gdr_split_plan(units, sms, ctypes.byref(lead)))
    return pieces, int(lead.value)


def checkpoint_count_bound(T: int, checkpoint_every_n_tokens: int) -> int:
    """Rows ``chunk_fwd_checkpoints`` may write: floor(T / checkpoint_every_n_tokens)."""
    return int(nat.lib().gdr_ckpt_count_bound(T, checkpoint_every_n_tokens))


def chunk_fwd_checkpoints(q, k, v, g, beta, checkpoint_every_n_tokens: int, scale=None,
                          initial_state=None, cu_seqlens=None, output_final_state=False,
                          path: str = "auto", stream=None):
    """``chunk_fwd`` on device tensors that also returns state checkpoints
    (libgdr ``gdr_chunk_fwd_ckpt``).

    Returns (o, ht or None, state_checkpoints [bound, H, dk, dv] f32,
    checkpoint_cu_starts [N + 1] int32): checkpoint m (1-based) of segment n is the
    state after the segment's first m * checkpoint_every_n_tokens tokens, in row
    checkpoint_cu_starts[n] + m - 1; rows past checkpoint_cu_starts[N] are not written.
    """
    dev = q.device
    T, H, dk, dv = q.shape[0], v.shape[1], q.shape[-1], v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    n_seq = cu_seqlens.numel() - 1
    scale = dk ** -0.5 if scale is None else scale
    o = torch.empty(T, H, dv, dtype=torch.bfloat16, device=dev)
    ht = (torch.empty(n_seq, H, dk, dv, dtype=torch.float32, device=dev)
          if output_final_state else None)
    rows = checkpoint_count_bound(T, checkpoint_every_n_tokens)
    ck = torch.empty(max(rows, 1), H, dk, dv, dtype=torch.float32, device=dev)
    starts = torch.empty(n_seq + 1, dtype=torch.int32, device=dev)
    ws = _workspace(workspace_bytes(T, n_seq, H, dk, dv, path), dev)
    ds = [_Desc(t) for t in (q, k, v, g, beta)]
    dh0, do, dht = _d(initial_state), _Desc(o), _d(ht)
    dck = _Desc(ck[:rows] if rows > 0 else ck[:0])
    rc = nat.lib().gdr_chunk_fwd_ckpt(
        ds[0].ref, ds[1].ref, ds[2].ref, ds[3].ref, ds[4].ref, ctypes.c_float(scale),
        _ref(dh0), _ptr(cu_seqlens), n_seq, do.ref, _ref(dht), dck.ref, _ptr(starts),
        int(checkpoint_every_n_tokens), nat.PATHS[path], ctypes.c_void_p(ws.data_ptr()),
        ws.numel(), _stream(stream))
    nat.check(rc, "gdr_chunk_fwd_ckpt")
    return o, ht, ck[:rows], starts


def chunk_fwd_alloc(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                    output_final_state=False, stream=None):
    """Same as ``chunk_fwd`` on device tensors, but through ``gdr_chunk_fwd``,
    which takes its scratch with cudaMallocAsync on the stream."""
    dev = q.device
    T, H, dv = q.shape[0], v.shape[1], v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    n_seq = cu_seqlens.numel() - 1
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o = torch.empty(T, H, dv, dtype=torch.bfloat16, device=dev)
    ht = (torch.empty(n_seq, H, q.shape[-1], dv, dtype=torch.float32, device=dev)
          if output_final_state else None)
    ds = [_Desc(t) for t in (q, k, v, g, beta)]
    dh0, do, dht = _d(initial_state), _Desc(o), _d(ht)
    rc = nat.lib().gdr_chunk_fwd(ds[0].ref, ds[1].ref, ds[2].ref, ds[3].ref, ds[4].ref,
                                 ctypes.c_float(scale), _ref(dh0), _ptr(cu_seqlens), n_seq,
                                 do.ref, _ref(dht), _stream(stream))
    nat.check(rc, "gdr_chunk_fwd")
    return o, ht


# ---------------------------------------------------------------- stages

def chunk_index(cu_seqlens: torch.Tensor, T: int, stream=None):
    """Device chunk enumeration: (seg_table [N, 4], chunk_table [bound, 4], n_chunks [1])."""
    dev = cu_seqlens.device
    n_seq = cu_seqlens.numel() - 1
    seg = torch.empty(max(n_seq, 1), 4, dtype=torch.int32, device=dev)
    chunks = torch.empty(max(chunk_count_bound(T, n_seq), 1), 4, dtype=torch.int32, device=dev)
    n = torch.empty(1, dtype=torch.int32, device=dev)
    rc = nat.lib().gdr_chunk_index(_ptr(cu_seqlens), n_seq, T, _ptr(seg), _ptr(chunks),
                                   _ptr(n), _stream(stream))
    nat.check(rc, "gdr_chunk_index")
    return seg[:n_seq], chunks[:chunk_count_bound(T, n_seq)], n


def chunk_prep(k, v, g, beta, cu_seqlens, stream=None):
    """Stage 1: returns (w [T, H, dk] bf16, u [T, H, dv] bf16, gcum [T, H] f32)."""
    dev = k.device
    T, H, dk, dv = k.shape[0], v.shape[1], k.shape[2], v.shape[2]
    n_seq = cu_seqlens.numel() - 1
    w = torch.zeros(T, H, dk, dtype=torch.bfloat16, device=dev)
    u = torch.zeros(T, H, dv, dtype=torch.bfloat16, device=dev)
    gc = torch.zeros(T, H, dtype=torch.float32, device=dev)
    ws = _workspace(stage_workspace_bytes(T, n_seq), dev)
    d = [_Desc(t) for t in (k, v, g, beta, w, u, gc)]
    rc = nat.lib().gdr_chunk_prep(d[0].ref, d[1].ref, d[2].ref, d[3].ref, _ptr(cu_seqlens),
                                  n_seq, d[4].ref, d[5].ref, d[6].ref,
                                  ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    nat.check(rc, "gdr_chunk_prep")
    return w, u, gc


def state_scan(k, w, u, gcum, initial_state, cu_seqlens, output_final_state=True, stream=None):
    """Stage 2: returns (h [bound, H, dk, dv] bf16, v_new [T, H, dv] bf16, ht or None)."""
    dev = k.device
    T, H, dk, dv = k.shape[0], w.shape[1], k.shape[2], u.shape[2]
    n_seq = cu_seqlens.numel() - 1
    h = torch.zeros(max(chunk_count_bound(T, n_seq), 0), H, dk, dv, dtype=torch.bfloat16,
                    device=dev)
    vn = torch.zeros(T, H, dv, dtype=torch.bfloat16, device=dev)
    ht = (torch.zeros(n_seq, H, dk, dv, dtype=torch.float32, device=dev)
          if output_final_state else None)
    ws = _workspace(stage_workspace_bytes(T, n_seq), dev)
    d = [_Desc(t) for t in (k, w, u, gcum, h, vn)]
    dh0, dht = _d(initial_state), _d(ht)
    rc = nat.lib().gdr_state_scan(d[0].ref, d[1].ref, d[2].ref, d[3].ref, _ref(dh0),
                                  _ptr(cu_seqlens), n_seq, d[4].ref, d[5].ref, _ref(dht),
                                  ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    nat.check(rc, "gdr_state_scan")
    return h, vn, ht


def chunk_out(q, k, v_new, h, gcum, scale, cu_seqlens, stream=None):
    """Stage 3: returns o [T, H, dv] bf16 (uncovered tokens zero)."""
    dev = q.device
    T, H, dv = q.shape[0], v_new.shape[1], v_new.shape[2]
    n_seq = cu_seqlens.numel() - 1
    o = torch.zeros(T, H, dv, dtype=torch.bfloat16, device=dev)
    ws = _workspace(stage_workspace_bytes(T, n_seq), dev)
    d = [_Desc(t) for t in (q, k, v_new, h, gcum, o)]
    rc = nat.lib().gdr_chunk_out(d[0].ref, d[1].ref, d[2].ref, d[3].ref, d[4].ref,
                                 ctypes.c_float(scale), _ptr(cu_seqlens), n_seq, d[5].ref,
                                 ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    nat.check(rc, "gdr_chunk_out")
    return o


def chunk_out_noalloc(q, k, v_new, h, gcum, scale, cu_seqlens, out=None, stream=None):
    """Stage 3 through ``gdr_chunk_out_noalloc``: no device allocation inside the
    library (its chunk tables live in a static 4 MiB device array).  ``out`` may be
    a preallocated o [T, H, dv] bf16; otherwise one is allocated here by torch."""
    dev = q.device
    T, H, dv = q.shape[0], v_new.shape[1], v_new.shape[2]
    n_seq = cu_seqlens.numel() - 1
    o = torch.zeros(T, H, dv, dtype=torch.bfloat16, device=dev) if out is None else out
    d = [_Desc(t) for t in (q, k, v_new, h, gcum, o)]
    rc = nat.lib().gdr_chunk_out_noalloc(d[0].ref, d[1].ref, d[2].ref, d[3].ref, d[4].ref,
                                         ctypes.c_float(scale), _ptr(cu_seqlens), n_seq,
                                         d[5].ref, _stream(stream))
    nat.check(rc, "gdr_chunk_out_noalloc")
    return o


def check_cu_seqlens(cu_seqlens: torch.Tensor, T: int, stream=None) -> Tuple[int, int]:
    """(number of malformed offsets, index of the first one or -1); synchronises."""
    n_bad = ctypes.c_int32(0)
    first = ctypes.c_int32(0)
    rc = nat.lib().gdr_debug_check_cu_seqlens(_ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                                              ctypes.byref(n_bad), ctypes.byref(first),
                                              _stream(stream))
    nat.check(rc, "gdr_debug_check_cu_seqlens")
    return n_bad.value, first.value


def device_status() -> int:
    s = ctypes.c_int32(0)
    nat.check(nat.lib().gdr_device_status(ctypes.byref(s)), "gdr_device_status")
    return s.value


def wait_selftest(limit_us: int = 2000, stream=None) -> None:
    """Run the bounded-wait self-test kernel (see gdr_debug_wait_selftest)."""
    nat.check(nat.lib().gdr_debug_wait_selftest(limit_us, _stream(stream)), "gdr_debug_wait_selftest")


def clear_device_status() -> None:
    nat.check(nat.lib().gdr_clear_device_status(), "gdr_clear_device_status")
