"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

The pages print no worked example for the gated delta rule, so nothing here
is a printed value. Every check is a consequence of the definition
(S <- alpha S (I - beta kh kh^T) + beta v kh^T, o = S qh, the gated delta rule
that "Optimiser l'inference sur appareil pour Apple Silicon", section "Qwen
cree trois formes de charges de travail", describes in words) that is
computed here by a different route:

* beta = 0: pure exponential decay, closed form;
* beta = 1 with a unit key: the state recalls the written value exactly;
* alpha = 1, beta = 1, orthonormal keys: an exact associative memory;
* dk = dv = 1: a first-order linear recurrence with a closed form;
* tiny sizes: explicit products of the per-token transition matrices;
* the block (chunk) evaluation against the scan, for many chunk sizes;
* state carry across calls, packed sequences, shared key heads.

``test_planted_mistakes_are_caught`` rebuilds the oracle with known mistakes
and shows that at least one pin fails for each.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng


def _nrm(x):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + 1e-6)


def _rand(seed, T, Hk, Hv, dk, dv, B=1):
    r = RNG(seed)
    q = r.standard_normal((B * T, Hk, dk))
    k = r.standard_normal((B * T, Hk, dk))
    v = r.standard_normal((B * T, Hv, dv))
    g = -np.log1p(np.exp(r.standard_normal((B * T, Hv))))
    b = r.standard_normal((B * T, Hv))
    s0 = 0.3 * r.standard_normal((B, Hv, dv, dk))
    return q, k, v, g, b, s0


def _both(mutation=0, chunk=3):
    """The two evaluations the oracle offers, as callables with one signature."""
    def seq(q, k, v, g, b, s0=None, cu=None, B=None):
        return oracle.gdn_sequential(q, k, v, g, b, s0, cu, B=B, mutation=mutation)

    def chk(q, k, v, g, b, s0=None, cu=None, B=None):
        return oracle.gdn_chunked(q, k, v, g, b, s0, cu, B=B, chunk=chunk, mutation=mutation)
    return {"sequential": seq, "chunked": chk}


# ----------------------------------------------------------------------------
# Individual pins. Each returns None on success and raises AssertionError.
# ----------------------------------------------------------------------------
def pin_beta_zero(fn):
    q, k, v, g, b, s0 = _rand(1, T=7, Hk=1, Hv=2, dk=4, dv=3)
    b[:] = -np.inf  # beta = sigmoid(-inf) = 0 exactly
    out, st = fn(q, k, v, g, b, s0)
    G = np.cumsum(g, axis=0)  # [T, Hv]
    for h in range(2):
        np.testing.assert_allclose(st[0, h], np.exp(G[-1, h]) * s0[0, h], rtol=1e-12, atol=1e-14)
        for t in range(7):
            expect = np.exp(G[t, h]) * s0[0, h] @ _nrm(q[t, 0])
            np.testing.assert_allclose(out[t, h], expect, rtol=1e-12, atol=1e-14)


def pin_delta_write(fn):
    """beta = 1 and |kh| = 1: after each token, S kh_t = v_t for any gate and any prior state."""
    q, k, v, g, b, s0 = _rand(2, T=6, Hk=1, Hv=1, dk=5, dv=4)
    k *= 1e3  # |k|^2 >> 1e-6, so |kh| = 1 to ~1e-13
    b[:] = np.inf  # beta = 1
    state = s0
    for t in range(6):
        _, state = fn(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], b[t:t + 1], state)
        kh = _nrm(k[t, 0])
        np.testing.assert_allclose(state[0, 0] @ kh, v[t, 0], rtol=1e-9, atol=1e-9)


def pin_retrieval(fn):
    """alpha = 1, beta = 1, orthonormal keys, zero state: S = sum v_s kh_s^T, S kh_j = v_j."""
    r = RNG(3)
    dk, dv, T = 8, 5, 6
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    keys = Qm[:T] * 1e3
    k = keys[:, None, :]
    v = r.standard_normal((T, 1, dv))
    g = np.zeros((T, 1))
    b = np.full((T, 1), np.inf)
    # query token t with the key of token j(t) <= t: the read-out must be v_j(t)
    jt = [0, 0, 1, 3, 2, 5]
    q = keys[jt][:, None, :]
    out, st = fn(q, k, v, g, b, None)
    for t in range(T):
        np.testing.assert_allclose(out[t, 0], v[jt[t], 0], rtol=1e-9, atol=1e-9)
    expect = sum(np.outer(v[s, 0], _nrm(keys[s])) for s in range(T))
    np.testing.assert_allclose(st[0, 0], expect, rtol=1e-9, atol=1e-9)


def pin_scalar_closed_form(fn):
    """dk = dv = 1: s_t = a_t s_{t-1} + c_t, a_t = alpha_t(1 - beta_t kh_t^2), c_t = beta_t v_t kh_t."""
    r = RNG(4)
    T = 11
    q = r.standard_normal((T, 1, 1))
    k = r.standard_normal((T, 1, 1))
    v = r.standard_normal((T, 1, 1))
    g = -np.log1p(np.exp(r.standard_normal((T, 1))))
    b = r.standard_normal((T, 1))
    s0 = np.array([[[[0.7]]]])
    out, st = fn(q, k, v, g, b, s0)
    kh = k[:, 0, 0] / np.sqrt(k[:, 0, 0] ** 2 + 1e-6)
    qh = q[:, 0, 0] / np.sqrt(q[:, 0, 0] ** 2 + 1e-6)
    alpha, beta = np.exp(g[:, 0]), 1 / (1 + np.exp(-b[:, 0]))
    a = alpha * (1 - beta * kh * kh)
    c = beta * v[:, 0, 0] * kh
    for t in range(T):
        # s_t = (prod_{r<=t} a_r) s_0 + sum_{u<=t} (prod_{u<r<=t} a_r) c_u
        s = np.prod(a[:t + 1]) * 0.7 + sum(np.prod(a[u + 1:t + 1]) * c[u] for u in range(t + 1))
        np.testing.assert_allclose(out[t, 0, 0], s * qh[t], rtol=1e-12, atol=1e-14)
        if t == T - 1:
            np.testing.assert_allclose(st[0, 0, 0, 0], s, rtol=1e-12)


def _bruteforce(q, k, v, g, b, s0):
    """Explicit transition matrices M_t = alpha_t (I - beta_t kh kh^T):
    S_t = S_0 M_1...M_t + sum_{u<=t} beta_u v_u kh_u^T M_{u+1}...M_t, o_t = S_t qh_t."""
    T, _, dk = q.shape
    alpha, beta = np.exp(g[:, 0]), 1 / (1 + np.exp(-b[:, 0]))
    kh, qh = _nrm(k[:, 0]), _nrm(q[:, 0])
    M = [alpha[t] * (np.eye(dk) - beta[t] * np.outer(kh[t], kh[t])) for t in range(T)]

    def prod(lo, hi):  # M_lo ... M_hi (inclusive), identity if empty
        P = np.eye(dk)
        for r in range(lo, hi + 1):
            P = P @ M[r]
        return P

    outs, S = [], None
    for t in range(T):
        S = s0 @ prod(0, t) + sum(beta[u] * np.outer(v[u, 0], kh[u]) @ prod(u + 1, t) for u in range(t + 1))
        outs.append(S @ qh[t])
    return np.array(outs), S


def pin_bruteforce(fn):
    for seed, (T, dk, dv) in enumerate([(8, 4, 3), (5, 3, 4), (1, 2, 2), (8, 1, 2)]):
        q, k, v, g, b, s0 = _rand(10 + seed, T=T, Hk=1, Hv=1, dk=dk, dv=dv)
        out, st = fn(q, k, v, g, b, s0)
        eo, es = _bruteforce(q, k, v, g, b, s0[0, 0])
        np.testing.assert_allclose(out[:, 0], eo, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(st[0, 0], es, rtol=1e-11, atol=1e-12)


def pin_gqa_duplication(fn):
    """Hk=2 shared by Hv=6 (groups of 3) equals Hk=6 with the key heads duplicated."""
    q, k, v, g, b, s0 = _rand(5, T=9, Hk=2, Hv=6, dk=4, dv=3)
    out, st = fn(q, k, v, g, b, s0)
    rep = [0, 0, 0, 1, 1, 1]
    out2, st2 = fn(q[:, rep], k[:, rep], v, g, b, s0)
    np.testing.assert_allclose(out, out2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(st, st2, rtol=1e-13, atol=1e-14)


PINS = [pin_beta_zero, pin_delta_write, pin_retrieval, pin_scalar_closed_form, pin_bruteforce,
        pin_gqa_duplication]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
@pytest.mark.parametrize("which", ["sequential", "chunked"])
def test_pin(pin, which):
    pin(_both()[which])


# ----------------------------------------------------------------------------
# Cross-checks of the two evaluations and of the call contract.
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [1, 2, 3, 16, 64])
def test_chunked_equals_sequential(chunk):
    q, k, v, g, b, s0 = _rand(6, T=100, Hk=2, Hv=4, dk=8, dv=6, B=2)
    o1, s1 = oracle.gdn_sequential(q, k, v, g, b, s0, B=2)
    o2, s2 = oracle.gdn_chunked(q, k, v, g, b, s0, B=2, chunk=chunk)
    assert np.max(np.abs(o1 - o2)) <= 1e-10 * np.max(np.abs(o1))
    assert np.linalg.norm(s1 - s2) <= 1e-10 * np.linalg.norm(s1)


@pytest.mark.parametrize("scale", [1.6, 4.0])
def test_chunked_equals_sequential_fast_gates(scale):
    """Decays fast enough that a 64-token block's cumulative log-decay spans ~80 to ~200: the
    block evaluation still matches the token scan (products of e^{G_t - G_s} down to e^-200)."""
    q, k, v, g, b, s0 = _rand(9, T=200, Hk=2, Hv=4, dk=8, dv=6, B=2)
    g = g * scale
    o1, s1 = oracle.gdn_sequential(q, k, v, g, b, s0, B=2)
    o2, s2 = oracle.gdn_chunked(q, k, v, g, b, s0, B=2, chunk=64)
    assert np.max(np.abs(o1 - o2)) <= 1e-10 * np.max(np.abs(o1))
    assert np.linalg.norm(s1 - s2) <= 1e-10 * np.linalg.norm(s1)


def test_chunked_equals_sequential_varlen_with_empty_and_single():
    lens = [5, 0, 1, 37, 16, 64, 3]
    T = sum(lens)
    q, k, v, g, b, _ = _rand(7, T=T, Hk=1, Hv=2, dk=6, dv=5)
    s0 = RNG(8).standard_normal((len(lens), 2, 5, 6))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o1, s1 = oracle.gdn_sequential(q, k, v, g, b, s0, cu)
    o2, s2 = oracle.gdn_chunked(q, k, v, g, b, s0, cu, chunk=16)
    np.testing.assert_allclose(o2, o1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(s2, s1, rtol=1e-10, atol=1e-12)
    # the zero-length sequence passes its state through unchanged
    np.testing.assert_array_equal(s1[1], s0[1])


@pytest.mark.parametrize("which", ["sequential", "chunked"])
def test_state_carry_split_equals_whole(which):
    fn = _both(chunk=4)[which]
    q, k, v, g, b, s0 = _rand(9, T=30, Hk=1, Hv=2, dk=5, dv=4)
    o, s = fn(q, k, v, g, b, s0)
    cut = 13
    oa, sa = fn(q[:cut], k[:cut], v[:cut], g[:cut], b[:cut], s0)
    ob, sb = fn(q[cut:], k[cut:], v[cut:], g[cut:], b[cut:], sa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(sb, s, rtol=1e-11, atol=1e-13)


def test_prefill_equals_decode_steps():
    q, k, v, g, b, s0 = _rand(11, T=12, Hk=2, Hv=4, dk=4, dv=3)
    o, s = oracle.gdn_chunked(q, k, v, g, b, s0, chunk=5)
    st = s0
    for t in range(12):
        ot, st = oracle.gdn_decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], b[t:t + 1], st)
        np.testing.assert_allclose(ot[0], o[t], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(st, s, rtol=1e-11, atol=1e-13)


def test_packed_equals_separate():
    lens = [7, 3, 12]
    T = sum(lens)
    q, k, v, g, b, _ = _rand(12, T=T, Hk=1, Hv=2, dk=4, dv=4)
    s0 = RNG(13).standard_normal((3, 2, 4, 4))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, s = oracle.gdn_sequential(q, k, v, g, b, s0, cu)
    for n in range(3):
        a, e = cu[n], cu[n + 1]
        on, sn = oracle.gdn_sequential(q[a:e], k[a:e], v[a:e], g[a:e], b[a:e], s0[n:n + 1])
        np.testing.assert_allclose(o[a:e], on, rtol=1e-14, atol=0)
        np.testing.assert_allclose(s[n], sn[0], rtol=1e-14, atol=0)


def test_threads_do_not_change_results():
    q, k, v, g, b, s0 = _rand(14, T=40, Hk=2, Hv=4, dk=6, dv=5, B=3)
    o1, s1 = oracle.gdn_sequential(q, k, v, g, b, s0, B=3, threads=1)
    o2, s2 = oracle.gdn_sequential(q, k, v, g, b, s0, B=3, threads=4)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)


def test_prepass_properties():
    lens = [5, 0, 70, 1, 33]
    T = sum(lens)
    q, k, v, g, b, _ = _rand(15, T=T, Hk=2, Hv=4, dk=8, dv=2)
    q[3] *= 1e-4  # a tiny row: the epsilon must keep the inverse norm finite
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    chunk = 16
    rq, rk, beta, gc = oracle.gdn_prepass(q, k, g, b, cu, chunk=chunk)
    # normalised rows have unit length up to the epsilon
    nq = np.linalg.norm(q * rq[..., None], axis=-1)
    big = np.sum(q * q, axis=-1) > 1.0
    np.testing.assert_allclose(nq[big], 1.0, rtol=1e-6)
    assert np.all(np.isfinite(rq)) and np.all(nq <= 1.0)
    np.testing.assert_allclose(np.linalg.norm(k * rk[..., None], axis=-1), 1.0, rtol=1e-5)
    # beta is the logistic function of the logit: log(beta/(1-beta)) = b
    np.testing.assert_allclose(np.log(beta / (1 - beta)), b, rtol=1e-9, atol=1e-9)
    # gcum restarts at every chunk start and every sequence start, and grows by g
    for n in range(len(lens)):
        for t in range(cu[n], cu[n + 1]):
            pos = t - cu[n]
            if pos % chunk == 0:
                np.testing.assert_allclose(gc[t], g[t], rtol=0, atol=0)
            else:
                np.testing.assert_allclose(gc[t] - gc[t - 1], g[t], rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------
# Planted mistakes: each mutation of the oracle must break at least one pin.
# ----------------------------------------------------------------------------
MUTATIONS = {
    1: "gate dropped",
    2: "delta sign flipped",
    3: "read-out before the update",
    4: "interleaved key-head sharing",
    5: "normalisation dropped",
    6: "block form: P loses its diagonal",
    7: "block form: decay sign flipped in the state update",
}


def _pins_pass(mutation) -> bool:
    fns = _both(mutation=mutation, chunk=3)
    checks = [lambda pin=pin, w=w: pin(fns[w]) for pin in PINS for w in fns]

    def block_vs_scan():
        q, k, v, g, b, s0 = _rand(6, T=20, Hk=1, Hv=2, dk=4, dv=3)
        o1, s1 = fns["sequential"](q, k, v, g, b, s0)
        o2, s2 = fns["chunked"](q, k, v, g, b, s0)
        np.testing.assert_allclose(o2, o1, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s2, s1, rtol=1e-10, atol=1e-12)
    checks.append(block_vs_scan)
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


def test_unmutated_oracle_passes_all_pins():
    assert _pins_pass(0)


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=lambda m: MUTATIONS[m])
def test_planted_mistakes_are_caught(mutation):
    assert not _pins_pass(mutation), f"mutation {mutation} ({MUTATIONS[mutation]}) slipped through"
