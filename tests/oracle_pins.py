"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics.

Each pin takes an ``oracle.Oracle`` instance and raises AssertionError when
the oracle disagrees with the fact.  tests/test_oracle_pins.py runs them on
the oracle as built; tests/test_oracle_mutations.py runs them on copies of the
oracle's C source with one plausible mistake planted each, and requires every
planted mistake to fail at least one pin.

Sources (page title, section):
  P4 = "3.6 어텐션 I — 메모리 문제·FlashAttention 원리"
    3.6.4  stable softmax, online recurrence, alpha <= 1, block-order independence
    3.6.5  worked example (tests/golden/p4_worked_example.json)
    3.6.6  causal: keys j > i are skipped
    3.6.7  saved statistic L = m + log l; the backward pass recomputes S, P
    3.6.9  decoding (one query) needs another parallelisation: Nq << Nk
    3.6.10 pitfalls: rescale both l and O; never drop the max shift
    3.6.11 exercise 2 (tests/golden/p4_exercise2.json)
"""
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert np.all(np.isfinite(a)), "%s: non-finite value %r" % (what, a)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, "%s: |%r - %r| = %g > %g" % (what, a, b, err, tol)


def _rel_close(a, b, rtol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert np.all(np.isfinite(a)), "%s: non-finite value" % what
    scale = max(1.0, float(np.max(np.abs(b))))
    err = float(np.max(np.abs(a - b)))
    assert err <= rtol * scale, "%s: err %g > %g" % (what, err, rtol * scale)


def _worked_problem(scores, values):
    """Embed one score row as an attention problem: d = 1, q_0 = [1],
    k_j = [score_j], scale = 1, so s_j = score_j for query row 0."""
    n = len(scores)
    q = np.zeros((1, 1, n, 1))
    q[0, 0, 0, 0] = 1.0
    k = np.asarray(scores, dtype=np.float64).reshape(1, 1, n, 1)
    v = np.asarray(values, dtype=np.float64).reshape(1, 1, n, 1)
    return q, k, v


# ---------------------------------------------------------------------------
# Pins from the pages' printed values


def pin_worked_example_full(orc):
    """P4 3.6.5: full softmax of x=[1,3,2,5] with v=[10,20,30,40]."""
    g = _load("p4_worked_example.json")
    q, k, v = _worked_problem(g["scores"], g["values"])
    s = orc.scores_row(q[0, 0], k[0, 0], 0, 1.0)
    _close(s, g["scores"], 0.0, "scores")
    o, lse = orc.attention_rows(q, k, v, [(0, 0)], 1.0, causal=False, threads=1)
    tol = g["abs_tol"]
    _close(o[0, 0], g["full"]["o"], tol["o"], "O")
    m = g["full"]["m"]
    l = math.exp(lse[0] - m)  # lse = m + ln l with the page's m
    _close(l, g["full"]["l"], tol["l"], "l")
    _close(o[0, 0] * l, g["full"]["o_unnormalised"], tol["o_unnormalised"], "sum p v")


def pin_worked_example_online(orc):
    """P4 3.6.5: the hand-worked online states, and the reversed order."""
    g = _load("p4_worked_example.json")
    tol = g["abs_tol"]
    r = orc.online_row(g["scores"], g["values"], [tuple(b) for b in g["blocks"]])
    st1, st2 = g["block_states"]
    t1, t2 = r["trace"]
    _close(t1["m_tilde"], st1["m_tilde"], 0.0, "block1 m_tilde")
    _close(t1["m_new"], st1["m_new"], 0.0, "block1 m_new")
    _close(t1["alpha"], st1["alpha"], 0.0, "block1 alpha")
    _close(t1["l"], st1["l"], tol["l"], "block1 l")
    _close(t1["O"][0], st1["O"], tol["O_block1"], "block1 O")
    _close(t2["m_tilde"], st2["m_tilde"], 0.0, "block2 m_tilde")
    _close(t2["m_new"], st2["m_new"], 0.0, "block2 m_new")
    _close(t2["alpha"], st2["alpha"], tol["alpha"], "block2 alpha")
    _close(t2["alpha"] * t1["l"], st2["alpha_l"], tol["alpha_l"], "block2 alpha*l")
    _close(t2["l"], st2["l"], tol["l"], "block2 l")
    _close(t2["alpha"] * t1["O"][0], st2["alpha_O"], tol["alpha_O"], "block2 alpha*O")
    _close(t2["O"][0], st2["O"], tol["O_block2"], "block2 O")
    _close(r["o"][0], g["o_final"], tol["o"], "O final")
    # the page: the same result when the second block comes first
    rr = orc.online_row(g["scores"], g["values"], [tuple(b) for b in reversed(g["blocks"])])
    _close(rr["o"][0], r["o"][0], 1e-12, "reversed order O")
    _close(rr["l"], r["l"], 1e-12, "reversed order l")
    # max does not grow on the second step of the reversed order => alpha = 1
    _close(rr["trace"][0]["alpha"], 0.0, 0.0, "reversed first alpha")
    _close(rr["trace"][1]["alpha"], 1.0, 0.0, "reversed second alpha")


def pin_exercise2(orc):
    """P4 3.6.11 exercise 2: all values 1 => O_final = 1."""
    g = _load("p4_exercise2.json")
    r = orc.online_row(g["scores"], g["values"], [tuple(b) for b in g["blocks"]])
    _close(r["o"][0], g["o_final"], g["abs_tol"], "online O_final")
    q, k, v = _worked_problem(g["scores"], g["values"])
    o, _ = orc.attention_rows(q, k, v, [(0, 0)], 1.0, threads=1)
    _close(o[0, 0], g["o_final"], g["abs_tol"], "two-pass O_final")


# ---------------------------------------------------------------------------
# Closed forms


def pin_uniform_when_scale_zero(orc):
    """scale = 0 makes every allowed score 0: O_i is the mean of the allowed
    value rows and lse_i = ln(#allowed).  Causal allows keys 0..i (P4 3.6.6)."""
    rng = np.random.default_rng(101)
    B, H, N, d = 1, 2, 7, 3
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    for causal in (False, True):
        o, lse = orc.attention_fwd(q, k, v, 0.0, causal=causal, threads=2)
        for h in range(H):
            for i in range(N):
                n_allowed = i + 1 if causal else N
                _close(o[0, h, i], v[0, h, :n_allowed].mean(axis=0), 1e-13,
                       "mean of allowed values (causal=%s)" % causal)
                _close(lse[0, h, i], math.log(n_allowed), 1e-13, "ln(#allowed)")


def pin_two_keys_sigmoid(orc):
    """N = 2, non-causal: softmax of two scores is a logistic split,
    O_i = sig(s0-s1) v0 + sig(s1-s0) v1 and lse_i = logaddexp(s0, s1)."""
    rng = np.random.default_rng(202)
    d = 5
    scale = 0.37
    q = rng.standard_normal((1, 1, 2, d))
    k = rng.standard_normal((1, 1, 2, d))
    v = rng.standard_normal((1, 1, 2, d))
    o, lse = orc.attention_fwd(q, k, v, scale, causal=False, threads=1)
    for i in range(2):
        s0 = scale * float(np.dot(q[0, 0, i], k[0, 0, 0]))
        s1 = scale * float(np.dot(q[0, 0, i], k[0, 0, 1]))
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        _close(o[0, 0, i], w0 * v[0, 0, 0] + w1 * v[0, 0, 1], 1e-13, "two-key O")
        _close(lse[0, 0, i], np.logaddexp(s0, s1), 1e-13, "two-key lse")


def pin_causal_first_row_and_prefix(orc):
    """Causal row 0 sees only key 0: O_0 = v_0, lse_0 = s_00.  Causal row i
    equals the non-causal answer on the first i+1 keys (P4 3.6.6)."""
    rng = np.random.default_rng(303)
    B, H, N, d = 2, 1, 9, 4
    scale = 0.5
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    o, lse = orc.attention_fwd(q, k, v, scale, causal=True, threads=3)
    for b in range(B):
        _close(o[b, 0, 0], v[b, 0, 0], 0.0, "causal row 0 O")
        _close(lse[b, 0, 0], scale * float(np.dot(q[b, 0, 0], k[b, 0, 0])), 1e-14,
               "causal row 0 lse")
        for i in (1, 4, N - 1):
            sub = slice(0, i + 1)
            o2, lse2 = orc.attention_fwd(q[b:b + 1, :, sub], k[b:b + 1, :, sub],
                                         v[b:b + 1, :, sub], scale, causal=False, threads=1)
            _close(o[b, 0, i], o2[0, 0, i], 1e-13, "causal prefix O")
            _close(lse[b, 0, i], lse2[0, 0, i], 1e-13, "causal prefix lse")


def pin_large_logits_stay_finite(orc):
    """Scores near 800 overflow exp() without the max shift (P4 3.6.4 and
    3.6.10); with it the two-key closed form still holds."""
    q = np.array([40.0]).reshape(1, 1, 1, 1)
    q = np.concatenate([q, np.zeros((1, 1, 1, 1))], axis=2)  # second query row unused
    k = np.array([20.0, 19.0]).reshape(1, 1, 2, 1)
    v = np.array([3.0, -7.0]).reshape(1, 1, 2, 1)
    o, lse = orc.attention_rows(q, k, v, [(0, 0)], 1.0, threads=1)
    w0 = 1.0 / (1.0 + math.exp(760.0 - 800.0))
    _close(o[0, 0], w0 * 3.0 + (1.0 - w0) * -7.0, 1e-12, "large-logit O")
    _close(lse[0], 800.0 + math.log1p(math.exp(-40.0)), 1e-12, "large-logit lse")
    r = orc.online_row([800.0, 760.0, 790.0], [1.0, 2.0, 4.0], [(2, 1), (0, 2)])
    e10, e40 = math.exp(-10.0), math.exp(-40.0)
    _close(r["o"][0], (1.0 + 2.0 * e40 + 4.0 * e10) / (1.0 + e40 + e10), 1e-12, "online large")
    _close(r["m"], 800.0, 0.0, "online large m")


# ---------------------------------------------------------------------------
# Invariants


def pin_shift_adds_to_lse_only(orc):
    """Adding c to every score of a row leaves O unchanged and adds c to lse
    (softmax shift invariance; L = m + log l, P4 3.6.7).  The shift is built
    by an extra feature: q' = [q, 1], k'_j = [k_j, c / scale]."""
    rng = np.random.default_rng(404)
    B, H, N, d = 1, 2, 11, 4
    scale = 0.25
    c = 3.5
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    q2 = np.concatenate([q, np.ones((B, H, N, 1))], axis=-1)
    k2 = np.concatenate([k, np.full((B, H, N, 1), c / scale)], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, N, 1))], axis=-1)
    for causal in (False, True):
        o, lse = orc.attention_fwd(q, k, v, scale, causal=causal, threads=2)
        o2, lse2 = orc.attention_fwd(q2, k2, v2, scale, causal=causal, threads=2)
        _close(o2[..., :d], o, 1e-12, "shifted O")
        _close(lse2, lse + c, 1e-12, "shifted lse")


def pin_permutation_equivariance(orc):
    """Non-causal attention is a function of the key/value SET: permuting the
    rows of K and V together leaves every output row unchanged."""
    rng = np.random.default_rng(505)
    B, H, N, d = 1, 1, 13, 6
    scale = 0.4
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    perm = rng.permutation(N)
    o, lse = orc.attention_fwd(q, k, v, scale, threads=2)
    o2, lse2 = orc.attention_fwd(q, k[:, :, perm], v[:, :, perm], scale, threads=2)
    _close(o2, o, 1e-12, "permuted O")
    _close(lse2, lse, 1e-12, "permuted lse")


def pin_one_hot_dominance(orc):
    """A score far above all others puts (numerically) all weight on its key:
    O_i equals that key's value row."""
    rng = np.random.default_rng(606)
    N, d = 10, 4
    v = rng.standard_normal((1, 1, N, d))
    q = np.zeros((1, 1, N, d))
    k = np.zeros((1, 1, N, d))
    target = {0: 7, 3: 2, 9: 5}  # query row -> winning key
    # each winner gets its own feature, so the three rows do not interfere
    for n, (i, j) in enumerate(target.items()):
        q[0, 0, i, n] = 50.0
        k[0, 0, j, n] = 2.0
    o, _ = orc.attention_fwd(q, k, v, 1.0, threads=1)
    for i, j in target.items():
        _close(o[0, 0, i], v[0, 0, j], 1e-12, "one-hot row %d" % i)


def pin_constant_values(orc):
    """Rows of softmax weights sum to 1, so constant V gives O = that constant
    (generalises P4 3.6.11 exercise 2)."""
    rng = np.random.default_rng(707)
    B, H, N, d = 2, 2, 17, 3
    q = rng.standard_normal((B, H, N, d)) * 3.0
    k = rng.standard_normal((B, H, N, d))
    v = np.broadcast_to(np.array([1.5, -2.0, 0.25]), (B, H, N, d)).copy()
    for causal in (False, True):
        o, _ = orc.attention_fwd(q, k, v, 0.7, causal=causal, threads=4)
        _close(o, v, 1e-13, "constant V (causal=%s)" % causal)


def pin_online_matches_two_pass(orc):
    """P4 3.6.4: the online recurrence is exact and independent of the block
    split and order; alpha lies in [0, 1] and is 1 when the max does not grow."""
    rng = np.random.default_rng(808)
    for trial in range(12):
        n = int(rng.integers(1, 300))
        d = int(rng.integers(1, 9))
        scale = float(rng.uniform(0.05, 1.5))
        q = rng.standard_normal((1, 1, n, d)) * (8.0 if trial % 3 == 0 else 1.0)
        k = rng.standard_normal((1, 1, n, d))
        v = rng.standard_normal((1, 1, n, d))
        i = int(rng.integers(0, n))
        causal = bool(trial % 2)
        s = orc.scores_row(q[0, 0], k[0, 0], i, scale, causal=causal)
        nk = s.shape[0]
        cuts = sorted(set(rng.integers(1, nk, size=min(nk - 1, int(rng.integers(0, 8))))
                          .tolist())) if nk > 1 else []
        edges = [0] + cuts + [nk]
        blocks = [(edges[t], edges[t + 1] - edges[t]) for t in range(len(edges) - 1)]
        order = rng.permutation(len(blocks))
        blocks = [blocks[t] for t in order]
        r = orc.online_row(s, v[0, 0, :nk], blocks)
        o, lse = orc.attention_rows(q, k, v, [(0, i)], scale, causal=causal, threads=1)
        _rel_close(r["o"], o[0], 1e-12, "online vs two-pass O")
        _close(r["m"] + math.log(r["l"]), lse[0], 1e-12 * max(1.0, abs(lse[0])),
               "online m + ln l vs lse")
        m_prev = -math.inf
        for t in r["trace"]:
            assert 0.0 <= t["alpha"] <= 1.0, "alpha outside [0, 1]: %r" % t["alpha"]
            if t["m_tilde"] <= m_prev:
                assert t["alpha"] == 1.0, "alpha != 1 with no new max"
            assert t["m_new"] == max(m_prev, t["m_tilde"]), "running max"
            m_prev = t["m_new"]


def pin_rows_agree_with_full(orc):
    """The row-list entry point and the full entry point give the same rows,
    whatever the thread count and the row order."""
    rng = np.random.default_rng(909)
    B, H, N, d = 2, 3, 21, 5
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d))
    v = rng.standard_normal((B, H, N, d))
    for causal in (False, True):
        o, lse = orc.attention_fwd(q, k, v, 0.3, causal=causal, threads=1)
        rows = np.array([(bh, i) for bh in range(B * H) for i in range(N)])
        rows = rows[rng.permutation(len(rows))][:50]
        o2, lse2 = orc.attention_rows(q, k, v, rows, 0.3, causal=causal, threads=5)
        ref = o.reshape(B * H, N, d)[rows[:, 0], rows[:, 1]]
        _close(o2, ref, 0.0, "rows vs full O")
        _close(lse2, lse.reshape(B * H, N)[rows[:, 0], rows[:, 1]], 0.0, "rows vs full lse")


# ---------------------------------------------------------------------------
# Backward pass (section 3.6.7: gradients of the same definition).

def _loss(orc, q, k, v, g, scale, causal):
    o, _ = orc.attention_fwd(q, k, v, scale, causal=causal, threads=1)
    return float(np.sum(o * g))


def pin_bwd_finite_differences(orc):
    """Every gradient entry matches a central difference of sum(o * g)
    computed with the (separately pinned) forward oracle."""
    rng = np.random.default_rng(4040)
    B, H, N, d = 1, 2, 5, 3
    q, k, v, g = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    h = 1e-5
    for causal in (False, True):
        grads = orc.attention_bwd(q, k, v, g, 0.7, causal=causal, threads=2)
        for name, x, gx in zip("qkv", (q, k, v), grads):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                up = _loss(orc, q, k, v, g, 0.7, causal)
                x[idx] = old - h
                dn = _loss(orc, q, k, v, g, 0.7, causal)
                x[idx] = old
                fd[idx] = (up - dn) / (2 * h)
            _close(gx, fd, 1e-7, "d%s vs central difference (causal=%d)" % (name, causal))


def pin_bwd_single_key(orc):
    """N = 1: p = 1 whatever the score, so dv = g and dq = dk = 0."""
    rng = np.random.default_rng(4141)
    q, k, v, g = (rng.standard_normal((2, 1, 1, 4)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.attention_bwd(q, k, v, g, 1.3, causal=causal)
        _close(dv, g, 1e-15, "dv with one key")
        _close(dq, np.zeros_like(q), 0.0, "dq with one key")
        _close(dk, np.zeros_like(k), 0.0, "dk with one key")


def pin_bwd_two_keys_closed_form(orc):
    """N = 2, d = 1, non-causal: o_i = sig(a_i) v_0 + (1 - sig(a_i)) v_1 with
    a_i = scale q_i (k_0 - k_1), so
    do_i/dq_i = sig'(a_i) scale (k_0 - k_1)(v_0 - v_1)."""
    q = np.array([0.8, -1.1]).reshape(1, 1, 2, 1)
    k = np.array([0.4, -0.9]).reshape(1, 1, 2, 1)
    v = np.array([2.0, -0.5]).reshape(1, 1, 2, 1)
    g = np.array([1.5, 0.25]).reshape(1, 1, 2, 1)
    scale = 0.6
    dq, dk, dv = orc.attention_bwd(q, k, v, g, scale)
    want_dq = np.zeros(2)
    want_dv = np.zeros(2)
    want_dk = np.zeros(2)
    for i in range(2):
        a = scale * q[0, 0, i, 0] * (k[0, 0, 0, 0] - k[0, 0, 1, 0])
        sig = 1.0 / (1.0 + math.exp(-a))
        ds = g[0, 0, i, 0] * sig * (1 - sig) * (v[0, 0, 0, 0] - v[0, 0, 1, 0])
        want_dq[i] = ds * scale * (k[0, 0, 0, 0] - k[0, 0, 1, 0])
        want_dk[0] += ds * scale * q[0, 0, i, 0]
        want_dk[1] -= ds * scale * q[0, 0, i, 0]
        want_dv[0] += sig * g[0, 0, i, 0]
        want_dv[1] += (1 - sig) * g[0, 0, i, 0]
    _close(dq.ravel(), want_dq, 1e-14, "two-key dq")
    _close(dk.ravel(), want_dk, 1e-14, "two-key dk")
    _close(dv.ravel(), want_dv, 1e-14, "two-key dv")


def pin_bwd_sum_rules(orc):
    """Rows of P sum to 1 and rows of dS sum to 0, so per head
    sum_j dv_j = sum_i g_i and sum_j dk_j = 0; and since q and k enter only
    through s_ij = scale <q_i, k_j>, sum <dq_i, q_i> = sum <dk_j, k_j>."""
    rng = np.random.default_rng(4242)
    B, H, N, d = 2, 2, 17, 6
    q, k, v, g = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.attention_bwd(q, k, v, g, 0.45, causal=causal, threads=3)
        _close(dv.sum(axis=2), g.sum(axis=2), 1e-12, "sum of dv")
        _close(dk.sum(axis=2), np.zeros((B, H, d)), 1e-12, "sum of dk")
        _close(np.einsum("bhnd,bhnd->bh", dq, q), np.einsum("bhnd,bhnd->bh", dk, k), 1e-12,
               "<dq,q> vs <dk,k>")


def pin_bwd_value_shift(orc):
    """Adding one vector c to every value row shifts every o_i by c, which
    does not depend on q or k: dq and dk are unchanged, and so is dv."""
    rng = np.random.default_rng(4343)
    q, k, v, g = (rng.standard_normal((1, 2, 9, 4)) for _ in range(4))
    c = rng.standard_normal(4) * 3.0
    for causal in (False, True):
        a = orc.attention_bwd(q, k, v, g, 0.5, causal=causal)
        b = orc.attention_bwd(q, k, v + c, g, 0.5, causal=causal)
        for name, x, y in zip(("dq", "dk", "dv"), a, b):
            _close(x, y, 1e-12, "%s under a value shift" % name)


def pin_bwd_causal_first_row(orc):
    """Causal: row 0 sees only key 0, so dq_0 = 0, and the last key is seen
    only by the last row, which makes dv_{N-1} = p_{N-1,N-1} g_{N-1}."""
    rng = np.random.default_rng(4444)
    q, k, v, g = (rng.standard_normal((1, 1, 6, 3)) for _ in range(4))
    dq, _, dv = orc.attention_bwd(q, k, v, g, 0.9, causal=True)
    _close(dq[0, 0, 0], np.zeros(3), 0.0, "causal dq_0")
    s = 0.9 * q[0, 0, 5] @ k[0, 0].T
    p_last = math.exp(s[5] - s.max()) / np.exp(s - s.max()).sum()
    _close(dv[0, 0, 5], p_last * g[0, 0, 5], 1e-14, "causal dv of the last key")


def pin_bwd_row_split_matches_whole_heads(orc):
    """Splitting a head's query rows over threads (private dk, dv summed in
    order) gives the gradients of the one-job-per-head run, up to rounding
    order; the dq-rows entry point gives the same dq rows exactly."""
    rng = np.random.default_rng(4545)
    q, k, v, g = (rng.standard_normal((1, 2, 45, 6)) for _ in range(4))
    for causal in (False, True):
        whole = orc.attention_bwd(q, k, v, g, 0.35, causal=causal, threads=1)
        split = orc.attention_bwd(q, k, v, g, 0.35, causal=causal, threads=7)
        for name, a, b in zip(("dq", "dk", "dv"), whole, split):
            _close(b, a, 1e-12, "%s split vs whole (causal=%d)" % (name, causal))
        rows = np.array([[0, 0], [1, 44], [1, 3], [0, 22], [1, 21]])
        dq_rows = orc.attention_bwd_rows(q, k, v, g, rows, 0.35, causal=causal, threads=3)
        _close(dq_rows, whole[0].reshape(2, 45, 6)[rows[:, 0], rows[:, 1]], 0.0,
               "dq rows vs whole (causal=%d)" % causal)


# ---------------------------------------------------------------------------
# Decoding (section 3.6.9: a few queries against a long key sequence).

def pin_decode_square_is_the_forward(orc):
    """Nq = Nk: the decode definition is the square one (causal included:
    with Nq = Nk the end-aligned and start-aligned masks coincide)."""
    rng = np.random.default_rng(4646)
    q, k, v = (rng.standard_normal((2, 1, 13, 5)) for _ in range(3))
    for causal in (False, True):
        o1, l1 = orc.attention_decode(q, k, v, 0.6, causal=causal, threads=2)
        o2, l2 = orc.attention_fwd(q, k, v, 0.6, causal=causal, threads=1)
        _close(o1, o2, 0.0, "decode square O (causal=%d)" % causal)
        _close(l1, l2, 0.0, "decode square LSE (causal=%d)" % causal)


def pin_decode_end_alignment(orc):
    """Causal decode: the last query sees every key (= non-causal); query i
    sees exactly the first Nk - Nq + i + 1 keys (= non-causal on that prefix)."""
    rng = np.random.default_rng(4747)
    Nq, Nk = 4, 23
    q = rng.standard_normal((1, 2, Nq, 6))
    k, v = (rng.standard_normal((1, 2, Nk, 6)) for _ in range(2))
    oc, lc = orc.attention_decode(q, k, v, 0.5, causal=True)
    on, ln = orc.attention_decode(q, k, v, 0.5, causal=False)
    _close(oc[:, :, -1], on[:, :, -1], 0.0, "last query sees all keys")
    for i in range(Nq):
        n = Nk - Nq + i + 1
        oi, li = orc.attention_decode(q[:, :, i:i + 1], k[:, :, :n], v[:, :, :n], 0.5)
        _close(oc[:, :, i], oi[:, :, 0], 1e-15, "query %d on its key prefix" % i)
        _close(lc[:, :, i], li[:, :, 0], 1e-15, "query %d LSE on its key prefix" % i)


def pin_decode_uniform_and_permutation(orc):
    """One query, scale 0: O = mean of V and LSE = ln Nk; permuting the keys
    (with their values) changes nothing (non-causal)."""
    rng = np.random.default_rng(4848)
    q = rng.standard_normal((1, 3, 1, 4))
    k, v = (rng.standard_normal((1, 3, 31, 4)) for _ in range(2))
    o, l = orc.attention_decode(q, k, v, 0.0)
    _close(o[:, :, 0], v.mean(axis=2), 1e-14, "scale 0 mean")
    _close(l, np.full((1, 3, 1), math.log(31)), 1e-14, "scale 0 LSE")
    perm = rng.permutation(31)
    o1, l1 = orc.attention_decode(q, k, v, 0.7)
    o2, l2 = orc.attention_decode(q, k[:, :, perm], v[:, :, perm], 0.7)
    _close(o2, o1, 1e-14, "key permutation O")
    _close(l2, l1, 1e-14, "key permutation LSE")


PINS = [
    pin_worked_example_full,
    pin_worked_example_online,
    pin_exercise2,
    pin_uniform_when_scale_zero,
    pin_two_keys_sigmoid,
    pin_causal_first_row_and_prefix,
    pin_large_logits_stay_finite,
    pin_shift_adds_to_lse_only,
    pin_permutation_equivariance,
    pin_one_hot_dominance,
    pin_constant_values,
    pin_online_matches_two_pass,
    pin_rows_agree_with_full,
    pin_bwd_finite_differences,
    pin_bwd_single_key,
    pin_bwd_two_keys_closed_form,
    pin_bwd_sum_rules,
    pin_bwd_value_shift,
    pin_bwd_causal_first_row,
    pin_bwd_row_split_matches_whole_heads,
    pin_decode_square_is_the_forward,
    pin_decode_end_alignment,
    pin_decode_uniform_and_permutation,
]
