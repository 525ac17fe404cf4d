"""Shared helpers of the GPU parity tests: run the oracle on a subset of value
heads and compare with the stated tolerances.

Tolerances (floating point, bf16 output against the fp64 oracle):
  o:  max |delta| <= 4e-3 and cosine >= 0.9999 over covered tokens;
  ht: max |delta| / max |ref| <= 1e-2.
They sit about 2x above the o error FlashQLA's maintainer printed for H200
(max_diff 0.0015-0.0020 at max_ref 0.25-0.31) and above the 0.58% relative
final-state error printed there ("FlashQLA GDN backend produces different
tokens from FLA Triton on correctness-test prompts", maintainer's reply).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

O_ATOL = 4e-3
O_COS = 0.9999
HT_REL = 1e-2


def covered_tokens(cu, T):
    """Token mask of the segments after the running-max / clamp reading."""
    cu = [int(c) for c in (cu.tolist() if hasattr(cu, "tolist") else cu)]
    mask = np.zeros(T, dtype=bool)
    prev = 0
    bounds = []
    for i, c in enumerate(cu):
        c = min(max(c, 0), T)
        if i > 0 and c < prev:
            c = prev
        bounds.append(c)
        prev = c
    for s, e in zip(bounds[:-1], bounds[1:]):
        mask[s:e] = True
    return mask


def oracle_heads(w, heads, want_ht=None, n_threads=0):
    """fp64 oracle on the value heads ``heads`` of workload ``w`` (CPU tensors)."""
    heads = list(heads)
    group = w.H // w.Hk
    hk = [h // group for h in heads]
    sel = lambda t, idx: t[:, idx].contiguous()
    h0 = None if w.h0 is None else w.h0[:, heads].contiguous()
    want = w.want_ht if want_ht is None else want_ht
    return oracle.recurrent(sel(w.q, hk), sel(w.k, hk), sel(w.v, heads), sel(w.g, heads),
                            sel(w.beta, heads), w.scale, h0, w.cu_seqlens, want_ht=want,
                            n_threads=n_threads)


def o_errors(o_gpu, o_ref, mask):
    a = o_gpu.float().cpu().numpy().astype(np.float64)[mask]
    b = o_ref[mask]
    if a.size == 0:
        return 0.0, 1.0
    err = float(np.abs(a - b).max())
    cos = float((a * b).sum() / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))
    return err, cos


def assert_o_close(o_gpu, o_ref, mask, atol=O_ATOL, cos_min=O_COS):
    err, cos = o_errors(o_gpu, o_ref, mask)
    assert err <= atol, f"o max|delta| {err:.3e} > {atol}"
    assert cos >= cos_min, f"o cosine {cos:.6f} < {cos_min}"
    return err, cos


def assert_ht_close(ht_gpu, ht_ref, rel=HT_REL):
    a = ht_gpu.float().cpu().numpy().astype(np.float64)
    scale = max(float(np.abs(ht_ref).max()), 1e-30)
    r = float(np.abs(a - ht_ref).max()) / scale
    assert r <= rel, f"ht max|delta|/max|ref| {r:.3e} > {rel}"
    return r


def chunk_enumeration(cu, T, C=64):
    """Python enumeration of (segment, start, length) chunks, ids in segment order."""
    cu = [int(c) for c in (cu.tolist() if hasattr(cu, "tolist") else cu)]
    b = []
    prev = 0
    for i, c in enumerate(cu):
        c = min(max(c, 0), T)
        if i > 0 and c < prev:
            c = prev
        b.append(c)
        prev = c
    segs, chunks = [], []
    for n in range(len(cu) - 1):
        s, e = b[n], b[n + 1]
        nc = (e - s + C - 1) // C
        segs.append((s, e, len(chunks), nc))
        for c in range(nc):
            chunks.append((n, s + c * C, min(C, e - s - c * C), 0))
    return segs, chunks


def run_gpu(w, path="auto", dev="cuda"):
    from chunked_gated_delta_gdr_gb300 import chunk_fwd
    wd = w.to(dev)
    return chunk_fwd(wd.q, wd.k, wd.v, wd.g, wd.beta, scale=w.scale, initial_state=wd.h0,
                     cu_seqlens=wd.cu_seqlens, output_final_state=w.want_ht, path=path)
