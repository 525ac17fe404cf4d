"""Pins of the fp64 oracle's backward (``oracle.recurrent_bwd``) against things other than
itself (CPU only).

The backward is the gradient of the token recurrence; the pages describe a training
backend whose backward is bit-reproducible and tolerates length-0 segments ("Findings
from integrating FlashQLA's Blackwell GDN kernels into a JAX trainer", intro and
section 2) but print no backward formula.  Sources of truth used here:

  * central finite differences of the forward oracle (itself pinned in
    test_oracle_pins.py), along random directions and element by element;
  * splitting a segment and chaining its gradients through dht -> dh0 (the backward
    of the ht -> h0 chaining invariant);
  * length-0 segments: they change no gradient, and their dh0 is their dht;
  * the beta = 0 closed form (pure decay: S_t = e^{G_t} h0);
  * the strong-decay limit (g = -60: every token starts from a wiped state).

Every pin takes the forward and backward as callables, so the same pins also run
against deliberately broken copies of the backward (mutation tests at the bottom).
"""
import functools
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import oracle


def _problem(seed, lengths, Hk, H, dk, dv, h0=True):
    r = np.random.default_rng(seed)
    T = int(sum(lengths))
    q = r.standard_normal((T, Hk, dk))
    k = r.standard_normal((T, Hk, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, H, dv))
    g = -np.log1p(np.exp(-(r.standard_normal((T, H)) + 2.0)))  # logsigmoid
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((T, H))))
    n = len(lengths)
    d = dict(q=q, k=k, v=v, g=g, beta=beta,
             h0=0.3 * r.standard_normal((n, H, dk, dv)) if h0 else None,
             cu=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32), scale=dk ** -0.5,
             dout=r.standard_normal((T, H, dv)), dht=r.standard_normal((n, H, dk, dv)))
    return d


NAMES = ("q", "k", "v", "g", "beta", "h0")


def _loss(fwd, d, **over):
    x = dict(d, **over)
    o, ht = fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["cu"],
                o_init=0.0)
    return float((o * x["dout"]).sum() + (ht * x["dht"]).sum())


def _grads(bwd, d):
    dq, dk, dv, dg, db, dh0 = bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["h0"],
                                  d["cu"], d["dout"], d["dht"])
    return dict(q=dq, k=dk, v=dv, g=dg, beta=db, h0=dh0)


def pin_bwd_directional_fd(fwd, bwd):
    # L = <o, dout> + <ht, dht>; (L(x + e u) - L(x - e u)) / 2e against <grad, u> for a
    # random direction u of each input in turn.  Segments: empty, 70 tokens (across a
    # 64-token recompute block), 5 and 1 tokens; two key heads, each shared by two
    # value heads.
    d = _problem(11, [0, 70, 5, 1], 2, 4, 4, 3)
    gr = _grads(bwd, d)
    r = np.random.default_rng(12)
    eps = 1e-6
    for name in NAMES:
        u = r.standard_normal(d[name].shape)
        fd = (_loss(fwd, d, **{name: d[name] + eps * u}) -
              _loss(fwd, d, **{name: d[name] - eps * u})) / (2 * eps)
        an = float((gr[name] * u).sum())
        assert abs(fd - an) <= 1e-6 * max(abs(fd), 1.0), (name, fd, an)


def pin_bwd_elementwise_fd(fwd, bwd):
    # every element of every input of a small problem (segments of 2 and 4 tokens and
    # an empty one, two value heads on one key head, dk = dv = 2)
    d = _problem(21, [2, 0, 4], 1, 2, 2, 2)
    gr = _grads(bwd, d)
    eps = 1e-6
    for name in NAMES:
        x = d[name]
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            fd = (_loss(fwd, d, **{name: xp}) - _loss(fwd, d, **{name: xm})) / (2 * eps)
            assert abs(fd - gr[name][idx]) <= 1e-7 * max(abs(fd), 1.0), (name, idx, fd,
                                                                        gr[name][idx])


def pin_bwd_chaining(fwd, bwd):
    # a 90-token segment against its pieces of 40 and 50 tokens: piece B starts from the
    # state A ends in, piece A's dht is the dh0 piece B hands back
    d = _problem(31, [90], 1, 1, 4, 4)
    whole = _grads(bwd, dict(d, dht=d["dht"]))
    A = {n: d[n][:40] for n in ("q", "k", "v", "g", "beta", "dout")}
    B = {n: d[n][40:] for n in ("q", "k", "v", "g", "beta", "dout")}
    _, htA = fwd(A["q"], A["k"], A["v"], A["g"], A["beta"], d["scale"], d["h0"], [0, 40])
    gB = _grads(bwd, dict(B, scale=d["scale"], h0=htA, cu=np.array([0, 50], np.int32),
                          dht=d["dht"]))
    gA = _grads(bwd, dict(A, scale=d["scale"], h0=d["h0"], cu=np.array([0, 40], np.int32),
                          dht=gB["h0"]))
    for name in ("q", "k", "v", "g", "beta"):
        np.testing.assert_allclose(whole[name], np.concatenate([gA[name], gB[name]]),
                                   rtol=0, atol=1e-10, err_msg=name)
    np.testing.assert_allclose(whole["h0"], gA["h0"], rtol=0, atol=1e-10)


def pin_bwd_ghosts(fwd, bwd):
    # length-0 segments, leading, in the middle and trailing, change no gradient of the
    # real tokens, and each one hands its dht back as its dh0
    d = _problem(41, [6, 9], 1, 2, 3, 3)
    g1 = _grads(bwd, d)
    r = np.random.default_rng(42)
    cu = np.array([0, 0, 6, 6, 15, 15, 15], np.int32)
    h0 = np.concatenate([r.standard_normal((1, 2, 3, 3)), d["h0"][:1],
                         r.standard_normal((1, 2, 3, 3)), d["h0"][1:],
                         r.standard_normal((2, 2, 3, 3))])
    dht = np.concatenate([r.standard_normal((1, 2, 3, 3)), d["dht"][:1],
                          r.standard_normal((1, 2, 3, 3)), d["dht"][1:],
                          r.standard_normal((2, 2, 3, 3))])
    g2 = _grads(bwd, dict(d, cu=cu, h0=h0, dht=dht))
    for name in ("q", "k", "v", "g", "beta"):
        assert np.array_equal(g1[name], g2[name]), name
    assert np.array_equal(g2["h0"][[1, 3]], g1["h0"])
    assert np.array_equal(g2["h0"][[0, 2, 4, 5]], dht[[0, 2, 4, 5]])


def pin_bwd_beta_zero(fwd, bwd):
    # beta = 0: S_t = e^{G_t} h0 with G_t the segment's running sum of g, so
    # dq_t = scale e^{G_t} h0 do_t, dk = dv = 0, and
    # dh0 = sum_t scale e^{G_t} q_t do_t^T + e^{G_last} dht
    d = _problem(51, [7], 1, 1, 3, 2)
    d["beta"] = np.zeros_like(d["beta"])
    gr = _grads(bwd, d)
    G = np.cumsum(d["g"][:, 0])
    h0, do, q, s = d["h0"][0, 0], d["dout"][:, 0], d["q"][:, 0], d["scale"]
    dq = s * np.exp(G)[:, None] * (do @ h0.T)
    np.testing.assert_allclose(gr["q"][:, 0], dq, rtol=0, atol=1e-12)
    assert not gr["k"].any() and not gr["v"].any()
    dh0 = s * np.einsum("t,ti,tj->ij", np.exp(G), q, do) + np.exp(G[-1]) * d["dht"][0, 0]
    np.testing.assert_allclose(gr["h0"][0, 0], dh0, rtol=0, atol=1e-12)


def pin_bwd_strong_decay(fwd, bwd):
    # g = -60: alpha = e^-60 ~ 1e-26 wipes the previous state at every token, so
    # S_t = beta_t k_t v_t^T up to terms ~1e-26, o_t = scale beta_t (q_t . k_t) v_t, and
    # with L = sum_t <o_t, do_t> + <ht, dht> (ht = S_last):
    #   dq_t = scale beta_t (v_t . do_t) k_t
    #   dk_t = scale beta_t (v_t . do_t) q_t      (+ beta dht v at the last token)
    #   dv_t = scale beta_t (q_t . k_t) do_t      (+ beta dht^T k at the last token)
    #   dbeta_t = scale (q_t . k_t)(v_t . do_t)   (+ k^T dht v at the last token)
    #   dg, dh0 ~ 0
    d = _problem(61, [9], 1, 1, 3, 2)
    d["g"] = np.full_like(d["g"], -60.0)
    o, ht = fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["h0"], d["cu"])
    gr = _grads(bwd, d)
    q, k, v, b, do, s = (d["q"][:, 0], d["k"][:, 0], d["v"][:, 0], d["beta"][:, 0],
                         d["dout"][:, 0], d["scale"])
    qk, vdo = (q * k).sum(1), (v * do).sum(1)
    dht = d["dht"][0, 0]
    np.testing.assert_allclose(o[:, 0], s * (b * qk)[:, None] * v, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ht[0, 0], b[-1] * np.outer(k[-1], v[-1]), rtol=0, atol=1e-12)
    dk = s * (b * vdo)[:, None] * q
    dk[-1] += b[-1] * dht @ v[-1]
    dv = s * (b * qk)[:, None] * do
    dv[-1] += b[-1] * dht.T @ k[-1]
    db = s * qk * vdo
    db[-1] += k[-1] @ dht @ v[-1]
    np.testing.assert_allclose(gr["q"][:, 0], s * (b * vdo)[:, None] * k, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gr["k"][:, 0], dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gr["v"][:, 0], dv, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gr["beta"][:, 0], db, rtol=0, atol=1e-12)
    assert np.abs(gr["g"]).max() < 1e-12 and np.abs(gr["h0"]).max() < 1e-12


PINS = [pin_bwd_directional_fd, pin_bwd_elementwise_fd, pin_bwd_chaining, pin_bwd_ghosts,
        pin_bwd_beta_zero, pin_bwd_strong_decay]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.recurrent, oracle.recurrent_bwd)


def test_bwd_rejects_bad_heads():
    d = _problem(1, [4], 2, 3, 4, 4)
    with pytest.raises(RuntimeError):
        _grads(oracle.recurrent_bwd, d)


# ---------------------------------------------------------------------------
# mutation tests: plant plausible mistakes in a copy of the backward's C source and
# check that at least one pin catches each.
# ---------------------------------------------------------------------------

MUTATIONS = {
    "dq_from_previous_state": ("acc += St[(int64_t)i * dv + j] * dov[j];",
                               "acc += Sp[(int64_t)i * dv + j] * dov[j];"),
    "dq_scale_dropped": ("dqt[i] = scale * acc;", "dqt[i] = acc;"),
    "output_injection_scale_dropped": ("+= scale * qv[i] * dov[j];", "+= qv[i] * dov[j];"),
    "dk_cross_term_dropped": ("dkt[i] = b * dw - a * b * sy;", "dkt[i] = b * dw;"),
    "dv_beta_dropped": ("dvt[j] = b * y[j];", "dvt[j] = y[j];"),
    "dbeta_decay_dropped": ("w[j] = vv[j] - a * x[j];", "w[j] = vv[j] - x[j];"),
    "dg_cross_term_dropped": ("dg[t * H + h] = a * (dsp - b * yx);", "dg[t * H + h] = a * dsp;"),
    "state_grad_decay_dropped": ("= a * (D[(int64_t)i * dv + j] - b * kv[i] * y[j]);",
                                 "= (D[(int64_t)i * dv + j] - b * kv[i] * y[j]);"),
    "state_grad_delta_sign": ("- b * kv[i] * y[j]);", "+ b * kv[i] * y[j]);"),
    "block_restart_state": ("memcpy(blk, starts + bi * SS,",
                            "memcpy(blk, starts + (bi > 0 ? bi - 1 : 0) * SS,"),
    "dht_ignored": ("D[i] = dht ? orc_load(dht, dht_dt,", "D[i] = dht ? 0.0 * orc_load(dht, dht_dt,"),
    "backward_grouped_head_map": ("const int32_t hq = h / group;", "const int32_t hq = h % Hk;"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    d = tempfile.mkdtemp(prefix="gdr_oracle_bwd_mut_")
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
    lib = oracle.open_library(path_so)
    fwd = functools.partial(oracle.recurrent, lib=lib)
    bwd = functools.partial(oracle.recurrent_bwd, lib=lib)
    caught = []
    for pin in PINS:
        try:
            pin(fwd, bwd)
        except (AssertionError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {name}"
