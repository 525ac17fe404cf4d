"""C-ABI contract tests that need no GPU: the library loads, exports every
function include/gdr.h declares with the argument count the binding uses,
sizes its workspaces as documented, and rejects malformed descriptors before
touching the device (cf. the undersized-tensor review findings on the KDA
PR, "feat(cake_kda): add paired recurrent training for SM100a and SM103a":
reject invalid calls instead of accessing out of bounds)."""
import ctypes
import os
import re

import pytest
import torch

from chunked_gated_delta_gdr_gb300 import _native as nat
from chunked_gated_delta_gdr_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdr.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(?:int|size_t|int64_t|int32_t|const char \*)\s*\**\s*(gdr_\w+)\s*\(([^;]*?)\)\s*;",
                         src, flags=re.S):
        args = m.group(2).strip()
        n = 0 if args in ("", "void") else args.count(",") + 1
        out[m.group(1)] = n
    return out


@pytest.fixture(scope="module")
def lib():
    from chunked_gated_delta_gdr_gb300 import build
    build.build()
    return nat.lib()


def test_header_declares_entry_points():
    d = _declared()
    for name in ("gdr_chunk_fwd", "gdr_chunk_fwd_ws", "gdr_chunk_fwd_workspace_bytes",
                 "gdr_chunk_prep", "gdr_state_scan", "gdr_chunk_out", "gdr_chunk_index",
                 "gdr_status_string"):
        assert name in d


def test_every_declared_symbol_exported(lib):
    declared = _declared()
    for name, nargs in declared.items():
        assert hasattr(lib, name), f"{name} not exported"
        assert name in nat.SIGNATURES, f"{name} has no binding signature"
        assert len(nat.SIGNATURES[name][1]) == nargs, f"{name}: binding arg count mismatch"
    assert set(nat.SIGNATURES) == set(declared)


def test_version_and_status_strings(lib):
    assert lib.gdr_version() >= 100
    for code in nat.STATUS:
        s = lib.gdr_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.gdr_status_string(12345).decode() == "unknown status"


def test_chunk_bound_and_workspace_sizes(lib):
    assert lib.gdr_chunk_count_bound(0, 0) == 0
    assert lib.gdr_chunk_count_bound(64, 1) == 2
    assert lib.gdr_chunk_count_bound(65536, 17) == 1024 + 17
    assert lib.gdr_chunk_count_bound(-1, 1) == 0
    assert lib.gdr_chunk_fwd_workspace_bytes(-1, 1, 1, 64, 64, 0) == 0
    T, N, H, D = 65536, 17, 32, 128
    st = lib.gdr_chunk_fwd_workspace_bytes(T, N, H, D, D, 2)
    # staged keeps W, U, V' (bf16 [T,H,D]), gcum (f32 [T,H]) and h (bf16 per chunk)
    assert st >= 3 * T * H * D * 2 + T * H * 4 + (1024 + N) * H * D * D * 2
    auto = lib.gdr_chunk_fwd_workspace_bytes(T, N, H, D, D, 0)
    assert auto >= st
    assert lib.gdr_stage_workspace_bytes(T, N) >= 16 * (N + 1024 + N)


class _Fake:
    """Descriptors with plausible fake device addresses; every call below must
    fail validation before any device access."""

    def __init__(self, T=128, Hk=2, H=4, D=64, N=2):
        self.T, self.Hk, self.H, self.D, self.N = T, Hk, H, D, N
        self.keep = []

    def t(self, shape, dtype, strides=None, addr=0x10000):
        shp = (ctypes.c_int64 * 4)(*(list(shape) + [0] * (4 - len(shape))))
        st = None
        if strides is not None:
            st = (ctypes.c_int64 * len(strides))(*strides)
            self.keep.append(st)
        d = nat.GdrTensor(ctypes.c_void_p(addr), dtype, len(shape), shp,
                          ctypes.cast(st, ctypes.POINTER(ctypes.c_int64)) if st else None)
        self.keep.append(d)
        return d

    def args(self, **over):
        T, Hk, H, D, N = self.T, self.Hk, self.H, self.D, self.N
        a = dict(q=self.t([T, Hk, D], nat.GDR_BF16), k=self.t([T, Hk, D], nat.GDR_BF16),
                 v=self.t([T, H, D], nat.GDR_BF16), g=self.t([T, H], nat.GDR_F32),
                 beta=self.t([T, H], nat.GDR_BF16), h0=None, o=self.t([T, H, D], nat.GDR_BF16),
                 ht=None, cu=ctypes.c_void_p(0x20000), n_seq=N)
        a.update(over)
        return a


def _call(lib, a, path=0, ws=0x40000, ws_bytes=1 << 40):
    r = lambda d: None if d is None else ctypes.byref(d)
    return lib.gdr_chunk_fwd_ws(r(a["q"]), r(a["k"]), r(a["v"]), r(a["g"]), r(a["beta"]),
                                ctypes.c_float(0.125), r(a["h0"]), a["cu"], a["n_seq"], r(a["o"]),
                                r(a["ht"]), path, ctypes.c_void_p(ws), ws_bytes, None)


@pytest.mark.parametrize("case,code", [
    ("q_null", -1), ("q_dtype", -2), ("v_rank", -3), ("o_rows", -3), ("inner_stride", -4),
    ("dim_96", -5), ("dk_ne_dv", -5), ("heads", -6), ("nseq_neg", -7), ("h0_nseq", -7),
    ("h0_noncompact", -4), ("cu_null", -1), ("negative_stride", -4), ("bad_path", -9),
])
def test_validation_errors(lib, case, code):
    f = _Fake()
    T, Hk, H, D, N = f.T, f.Hk, f.H, f.D, f.N
    over = {
        "q_null": dict(q=None),
        "q_dtype": dict(q=f.t([T, Hk, D], nat.GDR_F32)),
        "v_rank": dict(v=f.t([T, H * D], nat.GDR_BF16)),
        "o_rows": dict(o=f.t([T - 1, H, D], nat.GDR_BF16)),
        "inner_stride": dict(q=f.t([T, Hk, D], nat.GDR_BF16, strides=[Hk * D * 2, D * 2, 2])),
        "dim_96": dict(q=f.t([T, Hk, 96], nat.GDR_BF16), k=f.t([T, Hk, 96], nat.GDR_BF16),
                       v=f.t([T, H, 96], nat.GDR_BF16), o=f.t([T, H, 96], nat.GDR_BF16)),
        "dk_ne_dv": dict(v=f.t([T, H, 128], nat.GDR_BF16), o=f.t([T, H, 128], nat.GDR_BF16)),
        "heads": dict(v=f.t([T, 3, D], nat.GDR_BF16), o=f.t([T, 3, D], nat.GDR_BF16),
                      g=f.t([T, 3], nat.GDR_F32), beta=f.t([T, 3], nat.GDR_BF16)),
        "nseq_neg": dict(n_seq=-1),
        "h0_nseq": dict(h0=f.t([N + 1, H, D, D], nat.GDR_F32)),
        "h0_noncompact": dict(h0=f.t([N, H, D, D], nat.GDR_F32,
                                     strides=[2 * H * D * D, D * D, D, 1])),
        "cu_null": dict(cu=None),
        "negative_stride": dict(k=f.t([T, Hk, D], nat.GDR_BF16, strides=[-Hk * D, D, 1])),
    }.get(case, {})
    a = f.args(**over)
    path = 7 if case == "bad_path" else 0
    rc = _call(lib, a, path=path)
    if case == "bad_path":
        # path validation happens after the device check; without a GPU the
        # device check fails first with a CUDA error
        assert rc in (code, -10, -12)
    else:
        assert rc == code, (case, rc)


def test_stage_validation_errors(lib):
    f = _Fake()
    T, Hk, H, D, N = f.T, f.Hk, f.H, f.D, f.N
    k = f.t([T, Hk, D], nat.GDR_BF16)
    v = f.t([T, H, D], nat.GDR_BF16)
    g = f.t([T, H], nat.GDR_F32)
    b = f.t([T, H], nat.GDR_BF16)
    w = f.t([T, H, D], nat.GDR_BF16)
    u = f.t([T, H, D + 1], nat.GDR_BF16)
    gc = f.t([T, H], nat.GDR_F32)
    r = ctypes.byref
    rc = lib.gdr_chunk_prep(r(k), r(v), r(g), r(b), ctypes.c_void_p(0x20000), N, r(w), r(u), r(gc),
                            ctypes.c_void_p(0x40000), 1 << 30, None)
    assert rc == -3
    h = f.t([1, H, D, D], nat.GDR_BF16)  # smaller than the chunk bound
    vn = f.t([T, H, D], nat.GDR_BF16)
    u2 = f.t([T, H, D], nat.GDR_BF16)
    rc = lib.gdr_state_scan(r(k), r(w), r(u2), r(gc), None, ctypes.c_void_p(0x20000), N, r(h),
                            r(vn), None, ctypes.c_void_p(0x40000), 1 << 30, None)
    assert rc == -3
    rc = lib.gdr_chunk_index(None, 3, 100, None, None, None, None)
    assert rc == -1
    rc = lib.gdr_chunk_index(None, -1, 100, None, None, ctypes.c_void_p(0x1000), None)
    assert rc == -7


def test_binding_raises_without_gpu(lib):
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    q = torch.zeros(64, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(Exception):
        api.chunk_fwd(q, q, q, torch.zeros(64, 1), torch.zeros(64, 1, dtype=torch.bfloat16))


def _call_ckpt(lib, a, ck, starts, every, path=0, ws=0x40000, ws_bytes=1 << 40):
    r = lambda d: None if d is None else ctypes.byref(d)
    return lib.gdr_chunk_fwd_ckpt(r(a["q"]), r(a["k"]), r(a["v"]), r(a["g"]), r(a["beta"]),
                                  ctypes.c_float(0.125), r(a["h0"]), a["cu"], a["n_seq"],
                                  r(a["o"]), r(a["ht"]), r(ck), starts, every, path,
                                  ctypes.c_void_p(ws), ws_bytes, None)


@pytest.mark.parametrize("case,code", [
    ("every_zero", -14), ("every_not_64", -14), ("rows_short", -14), ("ckpt_dtype", -2),
    ("ckpt_heads", -14), ("starts_null", -1), ("ckpt_null", -1), ("ckpt_noncompact", -4),
])
def test_checkpoint_validation_errors(lib, case, code):
    f = _Fake()
    T, H, D = f.T, f.H, f.D
    every = {"every_zero": 0, "every_not_64": 96}.get(case, 64)
    rows = T // 64
    ck = {
        "rows_short": f.t([rows - 1, H, D, D], nat.GDR_F32),
        "ckpt_dtype": f.t([rows, H, D, D], nat.GDR_BF16),
        "ckpt_heads": f.t([rows, H + 1, D, D], nat.GDR_F32),
        "ckpt_null": None,
        "ckpt_noncompact": f.t([rows, H, D, D], nat.GDR_F32, strides=[2 * H * D * D, D * D, D, 1]),
    }.get(case, f.t([rows, H, D, D], nat.GDR_F32))
    starts = None if case == "starts_null" else ctypes.c_void_p(0x30000)
    rc = _call_ckpt(lib, f.args(), ck, starts, every)
    assert rc == code, (case, rc)


def test_checkpoint_count_bound(lib):
    assert lib.gdr_ckpt_count_bound(1000, 64) == 15
    assert lib.gdr_ckpt_count_bound(1000, 0) == 0
    assert lib.gdr_ckpt_count_bound(-1, 64) == 0


def _call_bwd(lib, a, outs, ws=0x40000, ws_bytes=1 << 40):
    r = lambda d: None if d is None else ctypes.byref(d)
    return lib.gdr_chunk_bwd(r(a["q"]), r(a["k"]), r(a["v"]), r(a["g"]), r(a["beta"]),
                             ctypes.c_float(0.125), r(a["h0"]), a["cu"], a["n_seq"], r(a["o"]),
                             r(a["ht"]), r(outs["dq"]), r(outs["dk"]), r(outs["dv"]),
                             r(outs["dg"]), r(outs["dbeta"]), r(outs["dh0"]), ctypes.c_void_p(ws),
                             ws_bytes, None)


@pytest.mark.parametrize("case,code", [
    ("dout_dtype", -2), ("dq_dtype", -2), ("dq_heads", -3), ("dv_rows", -3), ("dg_rank", -3),
    ("dbeta_noncompact", -4), ("dh0_nseq", -7), ("dh0_dim", -3), ("dk_null", -1),
    ("dht_noncompact", -4),
])
def test_backward_validation_errors(lib, case, code):
    # the backward checks dout like the forward's o and dht like its ht, and its fp32
    # outputs for shape, type and compactness, before touching the device
    f = _Fake()
    T, Hk, H, D, N = f.T, f.Hk, f.H, f.D, f.N
    F = nat.GDR_F32
    outs = dict(dq=f.t([T, Hk, D], F), dk=f.t([T, Hk, D], F), dv=f.t([T, H, D], F),
                dg=f.t([T, H], F), dbeta=f.t([T, H], F), dh0=f.t([N, H, D, D], F))
    over = {}
    if case == "dout_dtype":
        over = dict(o=f.t([T, H, D], F))
    elif case == "dht_noncompact":
        over = dict(ht=f.t([N, H, D, D], F, strides=[2 * H * D * D, D * D, D, 1]))
    outs.update({
        "dq_dtype": dict(dq=f.t([T, Hk, D], nat.GDR_BF16)),
        "dq_heads": dict(dq=f.t([T, H, D], F)),
        "dv_rows": dict(dv=f.t([T - 1, H, D], F)),
        "dg_rank": dict(dg=f.t([T, H, 1], F)),
        "dbeta_noncompact": dict(dbeta=f.t([T, H], F, strides=[2 * H, 1])),
        "dh0_nseq": dict(dh0=f.t([N + 1, H, D, D], F)),
        "dh0_dim": dict(dh0=f.t([N, H, D, D + 1], F)),
        "dk_null": dict(dk=None),
    }.get(case, {}))
    rc = _call_bwd(lib, f.args(**over), outs)
    assert rc == code, (case, rc)


def test_backward_workspace_bytes(lib):
    T, N, Hk, H, D = 1000, 3, 2, 4, 64
    b = lib.gdr_chunk_bwd_workspace_bytes(T, N, Hk, H, D, D)
    # at least the fp32 per-token gradient scratch (dV', dW and the per-value-head dq, dk)
    assert b >= 4 * T * H * D * 4
    assert lib.gdr_chunk_bwd_workspace_bytes(T, N, 3, 4, D, D) == 0  # H not a multiple of Hk
    assert lib.gdr_chunk_bwd_workspace_bytes(-1, N, Hk, H, D, D) == 0
    # one value head per key head needs no per-value-head scratch
    assert lib.gdr_chunk_bwd_workspace_bytes(T, N, H, H, D, D) < b


def test_split_plan_entry_point(lib):
    lead = ctypes.c_int32(0)
    assert lib.gdr_split_plan(32, 152, ctypes.byref(lead)) == 5 and lead.value == 2
    assert lib.gdr_split_plan(32, 152, None) == 5  # lead may be NULL
    lead.value = 7
    assert lib.gdr_split_plan(0, 152, ctypes.byref(lead)) == 1 and lead.value == 1
    assert lib.gdr_split_plan(10, -1, None) == 1
