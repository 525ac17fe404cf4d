"""Pins of the fp64 oracle against things other than itself (CPU only).

Each ``pin_*`` takes the oracle's token recurrence as a callable so the same
pins also run against deliberately broken copies of the oracle (mutation
tests at the bottom): every planted mistake must fail at least one pin.

Sources of truth used here:
  * a hand-worked three-token example (tests/golden/hand_worked_d2.txt);
  * the chunkwise (WY) form, a separately derived algorithm;
  * the unrolled matrix-product solution of the linear recurrence;
  * closed forms: beta = 0 (pure decay), g = 0 / beta = 1 with orthonormal
    keys (exact overwrite), a single token;
  * invariants: length-0 segments change nothing ("Findings from integrating
    FlashQLA's Blackwell GDN kernels into a JAX trainer", section 2), splitting
    a segment and chaining ht -> h0 equals the unsplit run, grouped heads
    equal explicitly repeated heads, linearity in (h0, v), exact bf16 decoding;
  * the magnitude envelope printed in "FlashQLA GDN backend produces different
    tokens from FLA Triton ..." (maintainer's reply), loosely.
"""
import functools
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gdr_gb300.inputs import make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _parse_golden(path):
    vals = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        key, rest = line.split(None, 1)
        rows = [[float(x) for x in r.split()] for r in rest.split(";")]
        vals[key] = np.array(rows if len(rows) > 1 else rows[0], dtype=np.float64)
    return vals


def _random_f64(seed, lengths, Hk, H, dk, dv, h0=True, normalize=True):
    r = _rng(seed)
    T = int(sum(lengths))
    q = r.standard_normal((T, Hk, dk))
    k = r.standard_normal((T, Hk, dk))
    if normalize:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, H, dv))
    g = -np.log1p(np.exp(-(r.standard_normal((T, H)) + 2.0)))  # logsigmoid
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, H))))
    hh = 0.3 * r.standard_normal((len(lengths), H, dk, dv)) if h0 else None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=hh, cu=cu, scale=dk ** -0.5)


def _run(rec, d, **kw):
    return rec(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["h0"], d["cu"], **kw)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_hand_worked(rec):
    gv = _parse_golden(os.path.join(GOLDEN, "hand_worked_d2.txt"))
    T = 3
    q = gv["q"].reshape(T, 1, 2)
    k = gv["k"].reshape(T, 1, 2)
    v = gv["v"].reshape(T, 1, 2)
    g = np.log(gv["alpha"]).reshape(T, 1)
    beta = gv["beta"].reshape(T, 1)
    h0 = gv["h0"].reshape(1, 1, 2, 2)
    cu = np.array([0, T], dtype=np.int32)
    o, ht = rec(q, k, v, g, beta, float(gv["scale"].ravel()[0]), h0, cu)
    np.testing.assert_allclose(o[:, 0], gv["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ht[0, 0], gv["ht"], rtol=0, atol=1e-13)


def pin_chunked_form(rec):
    for seed, lengths, C, dk, dv, Hk, H in [
        (1, [1], 64, 4, 4, 1, 1), (2, [63], 64, 8, 8, 1, 1), (3, [64], 64, 16, 8, 1, 2),
        (4, [65], 64, 8, 16, 2, 2), (5, [150], 64, 16, 8, 1, 2),
        (6, [10, 0, 7, 13], 4, 5, 3, 1, 3), (7, [29, 3, 16], 8, 4, 6, 2, 4)]:
        d = _random_f64(seed, lengths, Hk, H, dk, dv)
        o1, h1 = _run(rec, d)
        o2, h2 = oracle.chunked_wy(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"],
                                   d["h0"], d["cu"], C=C)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(h1, h2, rtol=0, atol=1e-12)


def pin_unrolled_products(rec):
    """S_t = (M_t..M_1) h0 + sum_j (M_t..M_{j+1}) beta_j k_j v_j^T,
    M_t = exp(g_t)(I - beta_t k_t k_t^T): the closed-form solution of the
    linear recurrence, built from explicit matrices."""
    d = _random_f64(11, [7], 1, 1, 3, 4)
    q, k, v, g, b = d["q"][:, 0], d["k"][:, 0], d["v"][:, 0], d["g"][:, 0], d["beta"][:, 0]
    h0 = d["h0"][0, 0]
    o, ht = _run(rec, d)
    M = [math.exp(g[t]) * (np.eye(3) - b[t] * np.outer(k[t], k[t])) for t in range(7)]

    def prod(a, c):  # M_{c-1} ... M_a  (empty -> I)
        P = np.eye(3)
        for t in range(a, c):
            P = M[t] @ P
        return P

    for t in range(7):
        S = prod(0, t + 1) @ h0 + sum(prod(j + 1, t + 1) @ (b[j] * np.outer(k[j], v[j]))
                                      for j in range(t + 1))
        np.testing.assert_allclose(o[t, 0], d["scale"] * S.T @ q[t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ht[0, 0], S, rtol=0, atol=1e-12)


def pin_beta_zero(rec):
    d = _random_f64(21, [40, 25], 2, 2, 6, 5)
    d["beta"] = np.zeros_like(d["beta"])
    o, ht = _run(rec, d)
    for n, (s, e) in enumerate([(0, 40), (40, 65)]):
        for h in range(2):
            G = np.cumsum(d["g"][s:e, h])
            want = d["scale"] * np.exp(G)[:, None] * (d["q"][s:e, h] @ d["h0"][n, h])
            np.testing.assert_allclose(o[s:e, h], want, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(ht[n, h], math.exp(G[-1]) * d["h0"][n, h],
                                       rtol=1e-12, atol=1e-14)


def pin_overwrite(rec):
    """g = 0, beta = 1, orthonormal keys: each token writes v_j into direction
    k_j exactly, so S_t^T k_j = v_j for every j <= t."""
    dk, dv, m = 8, 5, 6
    r = _rng(31)
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    keys = Qm[:m]
    h0 = r.standard_normal((1, 1, dk, dv))
    v = r.standard_normal((m, 1, dv))
    # query at step t is key j(t) = t // 2 (a key already written)
    qsel = [t // 2 for t in range(m)]
    q = keys[qsel].reshape(m, 1, dk)
    d = dict(q=q, k=keys.reshape(m, 1, dk), v=v, g=np.zeros((m, 1)), beta=np.ones((m, 1)),
             h0=h0, cu=np.array([0, m], dtype=np.int32), scale=0.5)
    o, ht = _run(rec, d)
    for t in range(m):
        np.testing.assert_allclose(o[t, 0], 0.5 * v[qsel[t], 0], rtol=0, atol=1e-12)
    P = np.eye(dk) - keys.T @ keys
    want = P @ h0[0, 0] + keys.T @ v[:, 0]
    np.testing.assert_allclose(ht[0, 0], want, rtol=0, atol=1e-12)


def pin_single_token(rec):
    d = _random_f64(41, [1, 1, 1], 1, 3, 7, 4)
    o, ht = _run(rec, d)
    for n in range(3):
        for h in range(3):
            a = math.exp(d["g"][n, h])
            b = d["beta"][n, h]
            kk = d["k"][n, 0]
            S = a * (np.eye(7) - b * np.outer(kk, kk)) @ d["h0"][n, h] + b * np.outer(kk, d["v"][n, h])
            np.testing.assert_allclose(o[n, h], d["scale"] * S.T @ d["q"][n, 0], rtol=0, atol=1e-13)
            np.testing.assert_allclose(ht[n, h], S, rtol=0, atol=1e-13)


def pin_ghosts(rec):
    base = [37, 70, 5]
    d = _random_f64(51, base, 1, 2, 6, 6)
    o, ht = _run(rec, d)
    lens = [0, 37, 0, 0, 70, 0, 5, 0, 0]
    real = [1, 4, 6]
    h0 = np.zeros((len(lens), 2, 6, 6))
    for i, n in enumerate(real):
        h0[n] = d["h0"][i]
    h0[2] = 7.0  # a ghost with an initial state keeps it
    d2 = dict(d, cu=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), h0=h0)
    o2, ht2 = _run(rec, d2)
    assert np.array_equal(o, o2)
    for i, n in enumerate(real):
        assert np.array_equal(ht[i], ht2[n])
    for n in range(len(lens)):
        if n not in real:
            assert np.array_equal(ht2[n], h0[n])


def pin_chaining(rec):
    d = _random_f64(61, [90], 2, 2, 5, 4)
    o, ht = _run(rec, d)
    for cut in (1, 33, 64, 89):
        d1 = dict(d, cu=np.array([0, cut], dtype=np.int32))
        o1, h1 = _run(rec, d1)
        d2 = dict(d, cu=np.array([0, cut, 90], dtype=np.int32),
                  h0=np.stack([d["h0"][0], h1[0]]))
        o2, h2 = _run(rec, d2)
        np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(h2[1], ht[0], rtol=0, atol=1e-12)


def pin_grouped_heads(rec):
    d = _random_f64(71, [30, 12], 2, 6, 4, 3)
    o, ht = _run(rec, d)
    d2 = dict(d, q=np.repeat(d["q"], 3, axis=1), k=np.repeat(d["k"], 3, axis=1))
    o2, ht2 = _run(rec, d2)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(ht, ht2, rtol=0, atol=1e-14)


def pin_linearity(rec):
    d = _random_f64(81, [45], 1, 2, 6, 4)
    o, ht = _run(rec, d)
    oa, ha = _run(rec, dict(d, v=np.zeros_like(d["v"])))
    ob, hb = _run(rec, dict(d, h0=np.zeros_like(d["h0"])))
    np.testing.assert_allclose(o, oa + ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ht, ha + hb, rtol=0, atol=1e-12)
    o2, _ = _run(rec, dict(d, scale=3 * d["scale"]))
    np.testing.assert_allclose(o2, 3 * o, rtol=1e-13, atol=1e-15)


def pin_segment_reading(rec):
    d = _random_f64(91, [40], 1, 1, 4, 4, h0=False)
    T = 40
    # uncovered tail tokens are not written
    o, _ = _run(rec, dict(d, cu=np.array([0, 10, 10, 30], dtype=np.int32)))
    assert np.isnan(o[30:]).all() and not np.isnan(o[:30]).any()
    # a decreasing offset is raised to the running maximum; ends clamp to T
    o1, h1 = _run(rec, dict(d, cu=np.array([0, 20, 10, 30, 99], dtype=np.int32)))
    o2, h2 = _run(rec, dict(d, cu=np.array([0, 20, 20, 30, T], dtype=np.int32)))
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


def pin_bf16_decoding(rec):
    w = make_workload("dec", 3, [33, 31], 2, 2, 16, with_h0=True)
    o1, h1 = rec(w.q, w.k, w.v, w.g, w.beta, w.scale, w.h0, w.cu_seqlens)
    f = lambda t: t.to(torch.float64).numpy()
    o2, h2 = rec(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), w.scale, f(w.h0), w.cu_seqlens)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


def _ckpt(rec, d, every):
    """State checkpoints from the oracle library ``rec`` runs on (mutants included)."""
    lib = getattr(rec, "keywords", {}).get("lib")
    return oracle.recurrent_checkpoints(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"],
                                        d["h0"], d["cu"], every, lib=lib)


def pin_checkpoint_prefixes(rec):
    # checkpoint m of a segment is the final state of the segment cut after m * every
    # tokens (the checkpoint feature of "feat(cake_kda): add paired recurrent training for
    # SM100a and SM103a", kept inference surface); the offsets are the running sum of
    # floor(len / every)
    lens, every = [150, 0, 128, 200, 3], 64
    d = _random_f64(101, lens, 1, 2, 5, 4)
    o, ht, ck, off = _ckpt(rec, d, every)
    assert off.tolist() == [0, 2, 2, 4, 7, 7]
    o2, ht2 = _run(rec, d)
    assert np.array_equal(o, o2) and np.array_equal(ht, ht2)
    starts = d["cu"][:-1]
    for n, L in enumerate(lens):
        for m in range(1, L // every + 1):
            dn = dict(d, cu=np.array([starts[n], starts[n] + m * every], dtype=np.int32),
                      h0=d["h0"][n:n + 1])
            _, hp = _run(rec, dn)
            assert np.array_equal(ck[off[n] + m - 1], hp[0]), (n, m)


def pin_checkpoint_resume(rec):
    # resuming from a checkpoint reproduces the rest of the segment
    d = _random_f64(111, [300], 2, 2, 4, 4)
    o, ht, ck, off = _ckpt(rec, d, 128)
    assert off.tolist() == [0, 2]
    for m in (1, 2):
        cut = 128 * m
        d2 = dict(d, cu=np.array([cut, 300], dtype=np.int32), h0=ck[m - 1:m])
        o2, h2 = _run(rec, d2)
        np.testing.assert_allclose(o2[cut:], o[cut:], rtol=0, atol=1e-12)
        np.testing.assert_allclose(h2[0], ht[0], rtol=0, atol=1e-12)


def pin_affine_state_carry(rec):
    # the state after a span of tokens is affine in the state before it:
    # S_out = M S_in + R with M the span's transition (run from S_in = I with v = 0) and R
    # its zero-start state (run from S_in = 0); the intra-sequence split chains pieces
    # this way (the CP final_correction of "feat(cake_kda): add paired recurrent training
    # for SM100a and SM103a" carries the state across ranks the same way)
    d = _random_f64(121, [77], 1, 2, 5, 5)
    _, ht = _run(rec, d)
    eye = np.broadcast_to(np.eye(5), (1, 2, 5, 5)).copy()
    _, M = _run(rec, dict(d, v=np.zeros_like(d["v"]), h0=eye))
    _, R = _run(rec, dict(d, h0=np.zeros_like(d["h0"])))
    np.testing.assert_allclose(ht[0], np.einsum("hij,hjk->hik", M[0], d["h0"][0]) + R[0],
                               rtol=0, atol=1e-12)


PINS = [pin_hand_worked, pin_chunked_form, pin_unrolled_products, pin_beta_zero,
        pin_overwrite, pin_single_token, pin_ghosts, pin_chaining, pin_grouped_heads,
        pin_linearity, pin_segment_reading, pin_bf16_decoding, pin_checkpoint_prefixes,
        pin_checkpoint_resume, pin_affine_state_carry]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.recurrent)


def test_chunked_form_matches_hand_worked():
    gv = _parse_golden(os.path.join(GOLDEN, "hand_worked_d2.txt"))
    o, ht = oracle.chunked_wy(gv["q"].reshape(3, 1, 2), gv["k"].reshape(3, 1, 2),
                              gv["v"].reshape(3, 1, 2), np.log(gv["alpha"]).reshape(3, 1),
                              gv["beta"].reshape(3, 1), 1.0, gv["h0"].reshape(1, 1, 2, 2),
                              [0, 3], C=2)
    np.testing.assert_allclose(o[:, 0], gv["o"], atol=1e-13)
    np.testing.assert_allclose(ht[0, 0], gv["ht"], atol=1e-13)


def test_oracle_rejects_bad_heads():
    d = _random_f64(1, [4], 2, 3, 4, 4)
    with pytest.raises(RuntimeError):
        _run(oracle.recurrent, d)


def test_magnitude_envelope_plausible():
    """max|o| and max|ht| within a factor 4 of the H200 envelope's max_ref
    (0.25-0.31 and 2.7-3.0); the page does not state H, g, beta or scale."""
    env = [line.split() for line in open(os.path.join(GOLDEN, "flashqla_h200_accuracy.txt"))
           if line.strip() and not line.startswith("#")]
    o_ref = [float(r[3]) for r in env if r[0] == "o"]
    s_ref = [float(r[3]) for r in env if r[0] == "final_state"]
    w = make_workload("env", 7, [512], 8, 8, 128)
    o, ht = oracle.recurrent(w.q, w.k, w.v, w.g, w.beta, w.scale, w.h0, w.cu_seqlens)
    mo, ms = np.abs(o).max(), np.abs(ht).max()
    assert min(o_ref) / 4 <= mo <= max(o_ref) * 4, mo
    assert min(s_ref) / 4 <= ms <= max(s_ref) * 4, ms


# ---------------------------------------------------------------------------
# mutation tests: plant plausible mistakes in a copy of the oracle's C source
# and check that at least one pin catches each.
# ---------------------------------------------------------------------------

MUTATIONS = {
    "decay_dropped_from_delta": ("- alpha * x[j]);", "- x[j]);"),
    "decay_sign": ("exp(orc_load(g, g_dt, t * H + h))", "exp(-orc_load(g, g_dt, t * H + h))"),
    "decay_dropped_from_state": ("row[j] = alpha * row[j] + ki * u[j];", "row[j] = row[j] + ki * u[j];"),
    "beta_dropped": ("u[j] = b * (", "u[j] = ("),
    "query_as_key_in_delta": ("x[j] += row[j] * ki;", "x[j] += row[j] * qv[i];"),
    "key_as_query_in_output": ("const double qi = qv[i];", "const double qi = kv[i];"),
    "scale_dropped": ("ot[j] *= scale;", "ot[j] *= 1.0;"),
    "grouped_head_map": ("const int32_t hk = h / group;", "const int32_t hk = h % Hk;"),
    "last_token_dropped": ("for (int64_t t = s; t < e; ++t)", "for (int64_t t = s; t + 1 < e; ++t)"),
    "h0_head_index": ("((int64_t)n * H + h) * dk * dv + i", "((int64_t)h * n_seq + n) * dk * dv + i"),
    "bf16_decode_shift": ("<< 16;", "<< 15;"),
    "segment_running_max": ("if (i > 0 && c < prev) c = prev;", ""),
    "checkpoint_segment_offset": ("const int64_t row = ckpt_off[n] +",
                                  "const int64_t row = ckpt_off[0] +"),
    "checkpoint_at_segment_end": ("(t - s + 1) % ckpt_every == 0",
                                  "(t - s + 1) % ckpt_every == 0 && t + 1 < e"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    d = tempfile.mkdtemp(prefix="gdr_oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path_c = os.path.join(mutant_dir, f"{name}.c")
    path_so = os.path.join(mutant_dir, f"{name}.so")
    open(path_c, "w").write(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", path_so, path_c, "-lm"],
                   check=True)
    rec = functools.partial(oracle.recurrent, lib=oracle.open_library(path_so))
    caught = []
    for pin in PINS:
        try:
            pin(rec)
        except (AssertionError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"
