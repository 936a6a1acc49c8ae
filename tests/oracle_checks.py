"""Pins for the CPU oracle: each check_* raises AssertionError on failure.

Every check ties the oracle to something other than itself: a value printed
on the pages (tests/golden), a closed form stated there, a library routine
(scipy softmax, numpy lexsort), an exact rational enumeration of the output
distribution, or a chi-square test against the target distribution.  The same
functions are run against oracle builds with a planted mistake, which must
fail them (test_oracle_mutations.py).
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction as Fr

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# helpers

def logits_for(P, T: float = 1.0) -> np.ndarray:
    """fp32 logits whose softmax at temperature T is P (up to fp32 rounding)."""
    return np.array([[T * math.log(float(p)) if p > 0 else -np.inf for p in row]
                     for row in P], dtype=np.float32)


def rational_rows(rng, n: int, V: int, lo: int = 1, hi: int = 20):
    a = rng.integers(lo, hi + 1, size=(n, V))
    return [[Fr(int(x), int(row.sum())) for x in row] for row in a]


def run_verify(lib, P, Q, tokens, uniforms, T: float = 1.0):
    """Oracle on B rows sharing the logits of P (K+1 rows) and Q (K rows)."""
    tokens = np.asarray(tokens, np.int32)
    B, K = tokens.shape
    zt = logits_for(P, T)
    zd = logits_for(Q, T)
    target = np.broadcast_to(zt[None], (B,) + zt.shape)
    draft = np.broadcast_to(zd[None], (B,) + zd.shape)
    temp = np.full(B, T, np.float32)
    return oracle.verify(target, draft, tokens, temp,
                         np.asarray(uniforms, np.float32), nthreads=0, lib=lib)


def enumerate_pieces(P, Q):
    """Leaves of the verification procedure on which its output is constant.

    Follows the pages' statement of the rule: x_i ~ q_i; accepted on
    U_i in [0, min(1, p_i(x_i)/q_i(x_i))); after the first rejection at n the
    bonus is drawn from max(p_n - q_n, 0)/R by inverse CDF, and from p_K when
    all K are accepted.  Each leaf is (weight, tokens, uniforms) with U at the
    midpoint of its piece; weights are exact rationals.
    """
    K = len(Q)
    V = len(P[0])
    leaves = []

    def bonus(xs, us, w, r):
        R = sum(r)
        assert R > 0
        cum = Fr(0)
        for v in range(V):
            if r[v] > 0:
                mid = (cum + r[v] / 2) / R
                # positions after the first rejection must not matter; they get
                # a uniform that would reject almost any token, so an oracle
                # that kept scanning would show it
                toks = xs + [0] * (K - len(xs))
                uu = us + [Fr(999, 1000)] * (K - len(us)) + [mid]
                leaves.append((w * r[v] / R, toks, uu))
                cum += r[v]

    def rec(i, xs, us, w):
        if i == K:
            bonus(xs, us, w, list(P[K]))
            return
        for x in range(V):
            if Q[i][x] == 0:
                continue
            wx = w * Q[i][x]
            a = min(Fr(1), P[i][x] / Q[i][x])
            if a > 0:
                rec(i + 1, xs + [x], us + [a / 2], wx * a)
            if a < 1:
                r = [max(P[i][v] - Q[i][v], Fr(0)) for v in range(V)]
                bonus(xs + [x], us + [(a + 1) / 2], wx * (1 - a), r)

    rec(0, [], [], Fr(1))
    return leaves


def exact_output_law(lib, P, Q, T: float = 1.0):
    """Exact law of (accept length, emitted tokens) of the oracle on (P, Q)."""
    leaves = enumerate_pieces(P, Q)
    tokens = np.array([lf[1] for lf in leaves], np.int32)
    uniforms = np.array([[float(u) for u in lf[2]] for lf in leaves], np.float32)
    out = run_verify(lib, P, Q, tokens, uniforms, T)
    return leaves, out


# ---------------------------------------------------------------------------
# a1 distribution

def check_softmax_library(lib):
    """Oracle p = scipy.special.softmax(z / T) on random rows; greedy one-hot."""
    from scipy.special import softmax
    rng = np.random.default_rng(7)
    for V in (1, 2, 3, 17, 1000):
        for T in (0.25, 0.7, 1.0, 2.5):
            z = (rng.standard_normal(V) * 3).astype(np.float32)
            p = oracle.row_probs(z, T, lib=lib)
            ref = softmax(z.astype(np.float64) / T)
            assert np.max(np.abs(p - ref)) < 1e-14, (V, T)
            assert abs(p.sum() - 1.0) < 1e-12
    z = np.array([1.0, 3.0, -2.0, 3.0, 0.5], np.float32)
    p = oracle.row_probs(z, 0.0, lib=lib)
    assert p.tolist() == [0.0, 1.0, 0.0, 0.0, 0.0], p  # first maximum wins
    # bf16 bit patterns decode exactly: 1.0, 0.0, -2.0, -inf
    bits = np.array([0x3F80, 0x0000, 0xC000, 0xFF80], np.uint16).view(np.int16)
    try:
        p = oracle.row_probs(bits, 1.0, lib=lib)
    except ValueError as e:  # a valid row refused
        raise AssertionError(f"bf16 row refused: {e}")
    ref = softmax(np.array([1.0, 0.0, -2.0, -np.inf]))
    assert np.max(np.abs(p - ref)) < 1e-15


def check_verify_library(lib):
    """The whole verification of random rows against library routines: p and q
    from scipy softmax (fp64), the accept test u <= p(x)/q(x) up to the first
    rejection, and the bonus as numpy searchsorted (side="right") of U[K] * R
    on the cumulative residual max(p_n - q_n, 0), or on p_K after K
    acceptances.  Rows the oracle flags as boundary cases are skipped."""
    from scipy.special import softmax
    rng = np.random.default_rng(41)
    B, K, V = 300, 3, 40
    zt = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    zd = (zt[:, :K] + rng.standard_normal((B, K, V)) * rng.uniform(0.2, 2.0, (B, 1, 1))).astype(np.float32)
    temps = rng.choice(np.array([0.6, 1.0, 1.7], np.float32), B)
    tok = np.empty((B, K), np.int32)
    for b in range(B):
        for i in range(K):
            q = softmax(zd[b, i].astype(np.float64) / temps[b])
            tok[b, i] = rng.choice(V, p=q)
    u = rng.random((B, K + 1), dtype=np.float32)
    out = oracle.verify(zt, zd, tok, temps, u, nthreads=0, lib=lib)
    checked = 0
    for b in range(B):
        T = float(temps[b])
        p = [softmax(zt[b, i].astype(np.float64) / T) for i in range(K + 1)]
        q = [softmax(zd[b, i].astype(np.float64) / T) for i in range(K)]
        n = K
        for i in range(K):
            x = tok[b, i]
            if not (q[i][x] > 0 and p[i][x] / q[i][x] >= u[b, i]):
                n = i
                break
        r = np.maximum(p[n] - q[n], 0.0) if n < K else p[K]
        t = int(np.searchsorted(np.cumsum(r), float(u[b, K]) * r.sum(), side="right"))
        np.testing.assert_allclose(out["p"][b], [p[i][tok[b, i]] for i in range(K)], rtol=1e-6)
        np.testing.assert_allclose(out["q"][b], [q[i][tok[b, i]] for i in range(K)], rtol=1e-6)
        if out["boundary"][b]:
            continue
        checked += 1
        assert out["accept_len"][b] == n, (b, out["accept_len"][b], n)
        assert out["out_tokens"][b, n] == t, (b, out["out_tokens"][b, n], t)
        assert (out["out_tokens"][b, :n] == tok[b, :n]).all() and (out["out_tokens"][b, n + 1:] == -1).all()
    assert checked > 0.9 * B
    assert 0 < (out["accept_len"] < K).sum() < B  # both a residual and a p_K draw occur
    assert (out["accept_len"] == K).any()


def check_boundary_flags(lib):
    """The boundary flag (spec: a uniform within 1e-6 of a ratio or a CDF
    step) is set exactly where the definition puts it.  Constructed rows at
    T = 1: p_0 = (.5, .3, .2), q_0 = (.25, .5, .25), p_1 = (.2, .3, .5); the
    draft x = 1 has p/q = 0.6.  On random rows the flag is rare."""
    P = [[0.5, 0.3, 0.2], [0.2, 0.3, 0.5]]
    Q = [[0.25, 0.5, 0.25]]
    cases = [  # (x, U_0, U_1, accept length, boundary)
        (1, 0.6 + 5e-7, 0.5, 0, 1),    # U_0 just past the ratio: rejected, on the boundary
        (1, 0.6 - 5e-7, 0.7, 1, 1),    # just below it: accepted, on the boundary
        (1, 0.59, 0.2 + 5e-7, 1, 1),   # accepted; U_1 just past the step 0.2 of p_1
        (1, 0.59, 0.5 - 4e-7, 1, 1),   # accepted; U_1 just below the step 0.5 of p_1
        (1, 0.59, 0.35, 1, 0),         # clear of every ratio and step
        (1, 0.9, 0.5, 0, 0),           # rejected; residual (.25, 0, 0): U_1 * R clear of 0 and R
        (0, 0.999, 0.2 + 5e-7, 1, 1),  # p/q = 2: always accepted; the bonus on a step
    ]
    tok = np.array([[c[0]] for c in cases], np.int32)
    u = np.array([[c[1], c[2]] for c in cases], np.float32)
    Pf = [[Fr(x).limit_denominator(1000) for x in row] for row in P]
    Qf = [[Fr(x).limit_denominator(1000) for x in row] for row in Q]
    out = run_verify(lib, Pf, Qf, tok, u)
    for k, c in enumerate(cases):
        assert out["accept_len"][k] == c[3], (k, out["accept_len"][k])
        assert out["boundary"][k] == c[4], (k, out["boundary"][k])
    rng = np.random.default_rng(43)
    B, K, V = 400, 3, 50
    zt = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    zd = (zt[:, :K] + rng.standard_normal((B, K, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    o = oracle.verify(zt, zd, tok, np.ones(B, np.float32), rng.random((B, K + 1), dtype=np.float32),
                      nthreads=0, lib=lib)
    assert o["boundary"].sum() <= 2, o["boundary"].sum()


def check_thm1_overlap(lib):
    """[SSD] Theorem 1: alpha = sum min(p, q) = 1 - 0.5 * ||p - q||_1."""
    rng = np.random.default_rng(11)
    for V in (2, 5, 64, 3000):
        for T in (0.5, 1.0):
            zt = (rng.standard_normal((2, V)) * 2).astype(np.float32)
            zd = (zt[:1] + rng.standard_normal((1, V))).astype(np.float32)
            p = oracle.row_probs(zt[0], T, lib=lib)
            q = oracle.row_probs(zd[0], T, lib=lib)
            out = oracle.verify(zt[None], zd[None], np.zeros((1, 1), np.int32),
                                np.array([T], np.float32),
                                np.array([[0.5, 0.5]], np.float32), lib=lib)
            a = out["alpha"][0, 0]
            assert abs(a - (1.0 - 0.5 * np.abs(p - q).sum())) < 1e-12, (V, T, a)


# ---------------------------------------------------------------------------
# a2 + a3, worked examples from the pages

def check_exercise_1(lib):
    """Lecture 5 §11 Exercise 1: beta 0.6, residual [1,0,0], accept probs."""
    ex = golden("cs349d_worked_examples.json")["exercise_1"]
    P = [ex["p"], ex["p"]]
    Q = [ex["q"]]
    acc = ex["accept_prob_per_token"]
    rows_t, rows_u = [], []
    for x in range(3):
        for du in (-2e-3, 2e-3):
            u = min(acc[x] + du, 0.999)
            rows_t.append([x])
            rows_u.append([u, 0.5])
    out = run_verify(lib, P, Q, rows_t, rows_u)
    j = 0
    for x in range(3):
        for du in (-2e-3, 2e-3):
            expect_accept = (acc[x] + du) <= acc[x] or acc[x] >= 1.0
            assert out["accept_len"][j] == (1 if expect_accept else 0), (x, du)
            if not expect_accept:
                # residual is one-hot on token 0 whatever the bonus uniform
                assert out["out_tokens"][j, 0] == 0
            j += 1
    assert abs(out["alpha"][0, 0] - ex["acceptance_rate"]) < 1e-6
    # exact law of the first emitted token equals p
    leaves, out = exact_output_law(lib, [[Fr(str(v)) for v in ex["p"]]] * 2,
                                   [[Fr(str(v)) for v in ex["q"]]])
    law = [Fr(0)] * 3
    for (w, _, _), t in zip(leaves, out["out_tokens"][:, 0]):
        law[t] += w
    assert law == [Fr(str(v)) for v in ex["p"]], law


def check_section_2_3(lib):
    """Lecture 5 §2.3: beta 0.75; B accepted w.p. 0.6; residual A:C = 0.2:0.05."""
    ex = golden("cs349d_worked_examples.json")["section_2_3_partial"]
    s = ex["surviving"]
    P = [ex["p"], ex["p"]]
    Q = [ex["q"]]
    out = run_verify(lib, P, Q, [[1], [1], [1], [1]],
                     [[0.599, 0.5], [0.601, 0.79], [0.601, 0.81], [0.601, 0.0]])
    assert out["accept_len"].tolist() == [1, 0, 0, 0]
    a, c = s["residual_ratio_A_to_C"]
    cut = a / (a + c)  # bonus is A below this uniform, C above
    assert abs(cut - 0.8) < 1e-12
    assert out["out_tokens"][1:, 0].tolist() == [0, 2, 0]
    assert abs(out["alpha"][0, 0] - s["acceptance_rate"]) < 1e-6
    assert abs(out["p"][0, 0] - s["p_B"]) < 1e-6
    assert abs(out["p"][0, 0] / out["q"][0, 0] - s["accept_prob_B"]) < 1e-6


# ---------------------------------------------------------------------------
# a2 + a3, exactness by enumeration ([DLN] §3, [CS349D] §2.4, [SSD] §2.1)

def check_exact_enumeration(lib, seed: int = 3, V: int = 5, K: int = 2,
                            T: float = 1.0, pairs: int = 6):
    """The emitted token at position i+1, given the first i drafts accepted,
    has law exactly p_{i+1}; P(accept at i) = sum min(p_i, q_i)."""
    rng = np.random.default_rng(seed)
    for _ in range(pairs):
        P = rational_rows(rng, K + 1, V)
        Q = rational_rows(rng, K, V)
        leaves, out = exact_output_law(lib, P, Q, T)
        n = out["accept_len"]
        toks = out["out_tokens"]
        assert out["status"].max() & oracle.ROW_ERRORS == 0
        for i in range(K + 1):
            mass = Fr(0)
            law = [Fr(0)] * V
            for (w, _, _), ni, tk in zip(leaves, n, toks):
                if ni >= i:
                    mass += w
                    law[tk[i]] += w
            # P(first i accepted) = prod_j alpha_j
            alpha = Fr(1)
            for j in range(i):
                alpha *= sum(min(P[j][v], Q[j][v]) for v in range(V))
            assert mass == alpha, (i, float(mass), float(alpha))
            cond = [l / mass for l in law]
            assert cond == P[i], (i, [float(c) for c in cond], [float(p) for p in P[i]])


def check_chisq(lib, alpha_target: float, draws: int = 1_000_000, V: int = 8,
                K: int = 3, seed: int = 5):
    """Monte-Carlo: first emitted token ~ p_1 and (given n >= i) the (i+1)-th
    ~ p_{i+1}; chi-square p-value above 1e-3 for each position."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(seed)
    P = [rng.dirichlet(np.ones(V)) for _ in range(K + 1)]
    Q = []
    for i in range(K):
        d = np.zeros(V)
        d[np.argsort(P[i])[:2]] = 0.5  # mass where p is small
        lo, hi = 0.0, 1.0
        for _ in range(60):  # bisection on lambda for sum min(p, q) = target
            lam = 0.5 * (lo + hi)
            q = lam * P[i] + (1 - lam) * d
            a = np.minimum(P[i], q).sum()
            lo, hi = (lam, hi) if a < alpha_target else (lo, lam)
        Q.append(q)
    x = np.stack([rng.choice(V, size=draws, p=Q[i] / Q[i].sum()) for i in range(K)], 1)
    u = rng.random((draws, K + 1), dtype=np.float32)
    out = run_verify(lib, [list(p) for p in P], [list(q) for q in Q], x, u)
    n = out["accept_len"]
    toks = out["out_tokens"]
    for i in range(K + 1):
        sel = n >= i
        obs = np.bincount(toks[sel, i], minlength=V)
        exp = P[i] / P[i].sum() * sel.sum()
        pval = chisquare(obs, exp).pvalue
        assert pval > 1e-3, (alpha_target, i, pval)


def check_expected_tokens(lib):
    """E[n+1] = (1 - a^(g+1))/(1 - a) with i.i.d. rows (Lecture 5 §4.1,
    survey blog §4.3); the printed speedups S = E/(g c + 1) of Lecture 5 §4.3
    and Exercises 2-4 follow from the oracle's exact law of n."""
    fx = golden("cs349d_worked_examples.json")["expected_tokens_and_speedup"]
    rows = {  # V=2 pairs with an exact overlap alpha
        0.7: ([Fr(8, 10), Fr(2, 10)], [Fr(5, 10), Fr(5, 10)]),
        0.8: ([Fr(9, 10), Fr(1, 10)], [Fr(7, 10), Fr(3, 10)]),
        0.75: ([Fr(7, 8), Fr(1, 8)], [Fr(5, 8), Fr(3, 8)]),
        0.6: ([Fr(9, 10), Fr(1, 10)], [Fr(5, 10), Fr(5, 10)]),
        0.1: ([Fr(19, 20), Fr(1, 20)], [Fr(1, 20), Fr(19, 20)]),
    }
    cache = {}
    for case in fx["cases"]:
        a, g, c = case["alpha"], case["gamma"], case["c"]
        key = (a, g)
        if key not in cache:
            p, q = rows[a]
            assert sum(min(x, y) for x, y in zip(p, q)) == Fr(str(a))
            leaves, out = exact_output_law(lib, [p] * (g + 1), [q] * g)
            E = sum(w * (int(ni) + 1) for (w, _, _), ni in zip(leaves, out["accept_len"]))
            for k in range(g + 1):
                pk = sum(w for (w, _, _), ni in zip(leaves, out["accept_len"]) if ni == k)
                A = Fr(str(a))
                assert pk == (A ** k * (1 - A) if k < g else A ** g), (a, g, k)
            cache[key] = E
        E = cache[key]
        closed = (1 - Fr(str(a)) ** (g + 1)) / (1 - Fr(str(a)))
        assert E == closed
        if "E" in case:
            assert round(float(E), 3) == case["E"], (case, float(E))
        S = float(E) / (g * c + 1)
        # printed to two decimals; Exercise 3 prints 2.41 at gamma=8 where the
        # closed form gives 2.40495, so allow half a unit in the last digit
        # plus that 0.005 slip
        assert abs(S - case["S"]) <= 0.0051, (case, S)
    bad = fx["contradiction"]
    E = cache.get((bad["alpha"], bad["gamma"]))
    assert E is not None and round(float(E), 2) != bad["printed"]


def check_wrong_method_a_is_biased(lib):
    """Lecture 5 §2.6: resampling from p after a rejection is biased.  The
    oracle's exact law differs from the wrong method's law by a visible TV."""
    rng = np.random.default_rng(21)
    tvs = []
    for _ in range(20):
        P = rational_rows(rng, 2, 5)
        Q = rational_rows(rng, 1, 5)
        alpha = sum(min(P[0][v], Q[0][v]) for v in range(5))
        wrong = [min(P[0][v], Q[0][v]) + (1 - alpha) * P[0][v] for v in range(5)]
        leaves, out = exact_output_law(lib, P, Q)
        law = [Fr(0)] * 5
        for (w, _, _), t in zip(leaves, out["out_tokens"][:, 0]):
            law[t] += w
        assert law == P[0]
        tvs.append(0.5 * sum(abs(float(a - b)) for a, b in zip(law, wrong)))
    assert max(tvs) > 0.05


# ---------------------------------------------------------------------------
# greedy and invariants

def check_greedy(lib):
    """Lecture 5 §2.7: greedy = accept iff the draft's argmax is the target's
    argmax; the bonus is the target argmax.  Ties go to the first index."""
    zt = np.array([[1, 3, 3, 2], [5, 0, 0, 5], [0, 1, 2, 2], [4, 4, 0, 0]], np.float32)
    zd = np.array([[0, 2, 2, 1], [1, 1, 0, 0], [9, 0, 0, 0]], np.float32)
    # draft argmaxes (first max): 1, 0, 0; target argmaxes: 1, 0, 2, 0
    tokens = np.array([[1, 0, 0], [1, 0, 0], [1, 3, 0], [2, 0, 0]], np.int32)
    B = tokens.shape[0]
    out = oracle.verify(np.broadcast_to(zt[None], (B, 4, 4)),
                        np.broadcast_to(zd[None], (B, 3, 4)), tokens,
                        np.zeros(B, np.float32), np.full((B, 4), 0.999, np.float32),
                        lib=lib)
    # row 0: x1=1 ok, x2=0 ok, x3=0 (target argmax 2) rejected -> bonus 2
    assert out["accept_len"][0] == 2 and out["out_tokens"][0].tolist() == [1, 0, 2, -1]
    # row 2: x2=3 is not the draft argmax (q(x2)=0) -> rejected, bonus argmax p_2 = 0
    assert out["accept_len"][2] == 1 and out["out_tokens"][2].tolist() == [1, 0, -1, -1]
    # row 3: x1=2 rejected at once, bonus = target argmax of row 0 = 1
    assert out["accept_len"][3] == 0 and out["out_tokens"][3].tolist() == [1, -1, -1, -1]
    # all-accept path: the bonus is the argmax of p_{K+1}
    tok = np.array([[1, 0, 2]], np.int32)
    zd2 = zt[:3].copy()
    out = oracle.verify(zt[None], zd2[None], tok, np.zeros(1, np.float32),
                        np.zeros((1, 4), np.float32), lib=lib)
    assert out["accept_len"][0] == 3 and out["out_tokens"][0].tolist() == [1, 0, 2, 0]


def check_invariants(lib):
    """Identical target and draft logits accept every draft; after a rejection
    with q(x_j) > 0 the bonus differs from x_j; outputs are well formed."""
    rng = np.random.default_rng(31)
    B, K, V = 400, 4, 50
    zt = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    zd = zt[:, :K].copy()
    temps = rng.choice(np.array([0.0, 0.5, 1.0], np.float32), B)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    tok[temps == 0] = np.argmax(zd[temps == 0], axis=2)
    u = rng.random((B, K + 1), dtype=np.float32)
    out = oracle.verify(zt, zd, tok, temps, u, lib=lib)
    assert (out["accept_len"] == K).all()
    assert (out["out_tokens"][:, :K] == tok).all()
    zd = (zt[:, :K] + rng.standard_normal((B, K, V)) * 1.5).astype(np.float32)
    out = oracle.verify(zt, zd, tok, temps, u, lib=lib)
    n = out["accept_len"]
    for b in range(B):
        nb = n[b]
        assert 0 <= nb <= K
        assert (out["out_tokens"][b, :nb] == tok[b, :nb]).all()
        assert 0 <= out["out_tokens"][b, nb] < V
        assert (out["out_tokens"][b, nb + 1:] == -1).all()
        if nb < K and out["q"][b, nb] > 0 and temps[b] > 0:
            assert out["out_tokens"][b, nb] != tok[b, nb]
    assert out["status"].max() & oracle.ROW_ERRORS == 0


def check_bad_inputs(lib):
    """Bad tokens, non-finite logits and bad temperatures flag the row and
    leave accept length 0 with no tokens."""
    K, V = 2, 6
    zt = np.zeros((5, K + 1, V), np.float32)
    zd = np.zeros((5, K, V), np.float32)
    tok = np.zeros((5, K), np.int32)
    temps = np.ones(5, np.float32)
    tok[0, 1] = V
    zt[1, 2, 3] = np.nan
    zd[2, 0, 0] = np.inf
    temps[3] = -1.0
    zt[4, 1, :] = -np.inf
    out = oracle.verify(zt, zd, tok, temps, np.full((5, K + 1), 0.5, np.float32), lib=lib)
    assert out["status"].tolist() == [oracle.ROW_BAD_TOKEN, oracle.ROW_NONFINITE,
                                      oracle.ROW_NONFINITE, oracle.ROW_BAD_TEMP,
                                      oracle.ROW_NONFINITE]
    assert (out["accept_len"] == 0).all() and (out["out_tokens"] == -1).all()


def check_fallback_zero_residual(lib):
    """A draft token with q = p = 0 is rejected and leaves a zero residual;
    the bonus then falls back to p_n and the row is flagged."""
    zt = np.array([[[0.0, 1.0, -np.inf, 0.5], [0, 0, 0, 0]]], np.float32)
    zd = zt[:, :1].copy()
    out = oracle.verify(zt, zd, np.array([[2]], np.int32), np.ones(1, np.float32),
                        np.array([[0.3, 0.0]], np.float32), lib=lib)
    assert out["accept_len"][0] == 0 and out["out_tokens"][0, 0] == 0
    assert out["status"][0] & oracle.ROW_FALLBACK


# ---------------------------------------------------------------------------
# a4 outcome prediction, a5 hit

def _bf16(x):
    from speculative_decoding_verification_50_gb300.workloads import f32_to_bf16_bits
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def check_predict_library_sort(lib):
    """Keys = numpy lexsort by (logit desc, index asc) minus the sent token,
    first F; bf16 rows with many ties exercise the index tie-break."""
    rng = np.random.default_rng(41)
    for dtype in ("fp32", "bf16"):
        for (B, K, V, F) in ((3, 2, 7, 3), (4, 3, 300, 6), (2, 4, 1000, 32), (2, 1, 4, 6)):
            z = rng.integers(-3, 4, (B, K + 1, V)).astype(np.float32) * 0.5
            zz = _bf16(z) if dtype == "bf16" else z
            tok = rng.integers(0, V, (B, K)).astype(np.int32)
            out = oracle.predict(zz, tok, F, lib=lib)
            for b in range(B):
                for k in range(K + 1):
                    idx = np.arange(V)
                    if k < K:
                        idx = idx[idx != tok[b, k]]
                    order = idx[np.lexsort((idx, -z[b, k, idx]))][:F]
                    want = np.full(F, -1, np.int32)
                    want[:len(order)] = order
                    assert out["keys"][b, k].tolist() == want.tolist(), (dtype, b, k)
                    got_l = out["key_logits"][b, k][:len(order)]
                    assert np.array_equal(got_l, z[b, k, order])


def check_predict_exclusion(lib):
    """[SSD] §4.1.1: the token sent for verification at lookahead k (< K) is
    never a key there; at k = K nothing is excluded."""
    V, K, F = 20, 3, 4
    z = np.tile(np.arange(V, dtype=np.float32)[::-1], (1, K + 1, 1))  # token 0 best
    tok = np.zeros((1, K), np.int32)
    out = oracle.predict(z, tok, F, lib=lib)
    for k in range(K):
        assert out["keys"][0, k].tolist() == [1, 2, 3, 4]
    assert out["keys"][0, K].tolist() == [0, 1, 2, 3]


def check_hit_constructed(lib):
    """[SSD] §3.1: hit iff t* is among the keys of the realised accept length."""
    K, F = 3, 2
    keys = np.array([[[10, 11], [20, 21], [30, 31], [40, 41]]] * 4, np.int32)
    accept_len = np.array([0, 2, 3, 1], np.int32)
    out_tokens = np.array([[11, -1, -1, -1], [5, 6, 30, -1], [1, 2, 3, 41], [7, 30, -1, -1]], np.int32)
    hit = oracle.check_hit(keys, accept_len, out_tokens, lib=lib)
    assert hit.tolist() == [1, 1, 1, 0]


def _hit_objective(F, a: float, r: float):
    """[SSD] Appendix A.2: the hit rate the fan-out maximises under an r-th
    power-law miss model, a^K (1 - F_K^-r) + sum_{k<K} a^k (1-a) (1 - F_k^-r)."""
    K = len(F) - 1
    w = np.array([a ** k * (1 - a) for k in range(K)] + [a ** K])
    return float(np.sum(w * (1.0 - np.asarray(F, float) ** (-r))))


def check_fanout_optimal(lib):
    """[SSD] Theorem 12: the closed-form F_k sum to the budget, satisfy the
    Lagrange condition of Appendix A.2 (equal marginal hit rate at every k)
    and match a library constrained optimiser (scipy SLSQP) on the objective."""
    from scipy.optimize import minimize
    for (K, a, r, budget) in [(4, 0.7, 1.0, 24), (8, 0.5, 0.7, 64), (3, 0.9, 2.0, 10),
                              (6, 0.3, 1.5, 40)]:
        _, x = oracle.geometric_fanout(K, a, r, budget, lib=lib)
        assert abs(x.sum() - budget) < 1e-9 * budget
        marg = [a ** k * (1 - a) * r * x[k] ** (-r - 1) for k in range(K)] + \
               [a ** K * r * x[K] ** (-r - 1)]
        assert np.ptp(marg) < 1e-9 * max(marg), (K, a, r, marg)
        res = minimize(lambda F: -_hit_objective(F, a, r), np.full(K + 1, budget / (K + 1)),
                       method="SLSQP", bounds=[(1e-3, budget)] * (K + 1),
                       constraints=[{"type": "eq", "fun": lambda F: F.sum() - budget}],
                       options={"ftol": 1e-14, "maxiter": 500})
        assert res.success
        np.testing.assert_allclose(x, res.x, rtol=2e-3, atol=2e-3)
        assert _hit_objective(x, a, r) >= _hit_objective(res.x, a, r) - 1e-10
    # the values of the formula at a = 0.7, r = 1, K = 4, budget = 24 (worked
    # out from Theorem 12, not printed on the pages): 5.97 5.00 4.18 3.50 5.35
    _, x = oracle.geometric_fanout(4, 0.7, 1.0, 24, lib=lib)
    np.testing.assert_allclose(x, [5.97, 5.00, 4.18, 3.50, 5.35], atol=0.006)


def check_fanout_rounding(lib):
    """Integer fan-out (our reading of Theorem 12, which leaves rounding open):
    floor, then the leftover budget to the largest fractional parts (lower k on
    ties), then the cap; every F_k within 1 of the real value; sum = budget."""
    rng = np.random.default_rng(12)
    for _ in range(200):
        K = int(rng.integers(1, 10))
        a = float(rng.uniform(0.05, 0.95))
        r = float(rng.uniform(0.2, 3.0))
        budget = int(rng.integers(0, 200))
        fk, x = oracle.geometric_fanout(K, a, r, budget, max_f=10 ** 6, lib=lib)
        fl = np.floor(x).astype(int)
        assert fk.sum() == budget and np.all(fk >= fl) and np.all(fk <= fl + 1)
        frac = x - fl
        up, down = frac[fk > fl], frac[fk == fl]
        if len(up) and len(down):
            assert up.min() >= down.max()
        capped, _ = oracle.geometric_fanout(K, a, r, budget, max_f=3, lib=lib)
        np.testing.assert_array_equal(capped, np.minimum(fk, 3))


def check_predict_fanout(lib):
    """Per-lookahead fan-out keeps the first F_k keys of each lookahead (the
    rest -1): a prefix of the uniform top-F list."""
    rng = np.random.default_rng(13)
    B, K, V, F = 3, 4, 50, 6
    z = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    full = oracle.predict(z, tok, F, lib=lib)
    fan = np.array([6, 0, 3, 1, 5], np.int32)
    part = oracle.predict(z, tok, F, lib=lib, fanout=fan)
    for k in range(K + 1):
        np.testing.assert_array_equal(part["keys"][:, k, :fan[k]], full["keys"][:, k, :fan[k]])
        assert np.all(part["keys"][:, k, fan[k]:] == -1)


def check_no_draft_is_one_hot_draft(lib):
    """[DLN] Appendix, NO_DRAFT_PROBS: the draft probability of the sent token
    is 1, so verification without draft logits equals verification whose draft
    rows are one-hot at the sent tokens (logit 0 there, -inf elsewhere) --
    whose exact output law is pinned by the enumeration checks."""
    rng = np.random.default_rng(31)
    B, K, V = 24, 3, 9
    zt = rng.normal(0, 1.5, (B, K + 1, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    tok[::3] = np.argmax(zt[::3, :K], axis=-1)  # some drafts the target likes
    temp = rng.choice([0.0, 0.7, 1.0], B).astype(np.float32)
    U = rng.uniform(0, 1, (B, K + 1)).astype(np.float32)
    onehot = np.full((B, K, V), -np.inf, np.float32)
    for b in range(B):
        for i in range(K):
            onehot[b, i, tok[b, i]] = 0.0
    a = oracle.verify(zt, None, tok, temp, U, lib=lib, no_draft=True)
    b_ = oracle.verify(zt, onehot, tok, temp, U, lib=lib)
    for k in ("accept_len", "out_tokens", "status"):
        np.testing.assert_array_equal(a[k], b_[k])
    np.testing.assert_allclose(a["p"], b_["p"], rtol=1e-12)
    np.testing.assert_array_equal(a["q"], 1.0)
    np.testing.assert_allclose(a["alpha"], a["p"], rtol=1e-12)  # sum min(p, one-hot) = p(x)


def check_no_draft_exact_law(lib):
    """Deterministic drafts ([DLN] Appendix, NO_DRAFT_PROBS: q one-hot at the
    sent token), run without draft logits: the emitted token at position i+1,
    given the first i accepted, has law exactly p_{i+1}, and the first i are
    accepted with probability prod_j p_j(x_j)."""
    rng = np.random.default_rng(33)
    V, K = 5, 2
    for _ in range(4):
        P = rational_rows(rng, K + 1, V)
        xs = rng.integers(0, V, K)
        Q = [[Fr(1) if v == xs[i] else Fr(0) for v in range(V)] for i in range(K)]
        leaves = enumerate_pieces(P, Q)
        tokens = np.array([lf[1] for lf in leaves], np.int32)
        uniforms = np.array([[float(u) for u in lf[2]] for lf in leaves], np.float32)
        B = len(leaves)
        zt = logits_for(P)
        target = np.broadcast_to(zt[None], (B,) + zt.shape)
        out = oracle.verify(target, None, tokens, np.ones(B, np.float32), uniforms,
                            nthreads=0, lib=lib, no_draft=True)
        assert out["status"].max() & oracle.ROW_ERRORS == 0
        for i in range(K + 1):
            mass = Fr(0)
            law = [Fr(0)] * V
            for (w, _, _), ni, tk in zip(leaves, out["accept_len"], out["out_tokens"]):
                if ni >= i:
                    mass += w
                    law[tk[i]] += w
            alpha = Fr(1)
            for j in range(i):
                alpha *= P[j][int(xs[j])]
            assert mass == alpha, (i, float(mass), float(alpha))
            assert [l / mass for l in law] == P[i], i


def check_ragged_matches_rows(lib):
    """Per-row draft counts ([DLN] Appendix, cu_num_draft_tokens): each packed
    row verifies exactly as that row alone with K = K_b; a row with no drafts
    draws its bonus from p_0 by the inverse CDF (numpy searchsorted); a count
    outside [0, Kmax] flags the row."""
    rng = np.random.default_rng(32)
    B, Kmax, V = 10, 4, 11
    kb = rng.integers(0, Kmax + 1, B)
    kb[1] = 0
    cu = np.cumsum(kb).astype(np.int32)
    T_ = int(cu[-1])
    zt = rng.normal(0, 1.5, (T_ + B, V)).astype(np.float32)
    zd = (np.repeat(zt[:1], T_, 0) * 0 + rng.normal(0, 1.5, (T_, V))).astype(np.float32)
    tok = rng.integers(0, V, T_).astype(np.int32)
    temp = rng.choice([0.0, 0.8, 1.0], B).astype(np.float32)
    U = rng.uniform(0, 1, T_ + B).astype(np.float32)
    out = oracle.verify_ragged(zt, zd, cu, tok, temp, U, Kmax, lib=lib)
    for b in range(B):
        c0 = 0 if b == 0 else int(cu[b - 1])
        k = int(kb[b])
        rows_t = zt[c0 + b: c0 + b + k + 1][None]
        ot = out["out_tokens"][b]
        assert np.all(ot[k + 1:] == -1)
        if k == 0:
            p0 = oracle.row_probs(rows_t[0, 0], float(temp[b]), lib=lib)
            t = int(np.argmax(p0)) if temp[b] == 0 else \
                int(np.searchsorted(np.cumsum(p0), float(U[c0 + b]) * p0.sum(), side="right"))
            assert out["accept_len"][b] == 0 and ot[0] == t, (b, ot, t)
            continue
        one = oracle.verify(rows_t, zd[c0:c0 + k][None], tok[c0:c0 + k][None], temp[b:b + 1],
                            U[c0 + b: c0 + b + k + 1][None], lib=lib)
        assert out["accept_len"][b] == one["accept_len"][0]
        np.testing.assert_array_equal(ot[:k + 1], one["out_tokens"][0])
        np.testing.assert_array_equal(out["p"][c0:c0 + k], one["p"][0])
        assert out["status"][b] == one["status"][0]
    bad = cu.copy()
    bad[3] = bad[2] + Kmax + 1  # K_3 too large (later rows shift, still read in bounds
    bad[4:] = np.maximum(bad[4:], bad[3])  # of the arrays below)
    big_t = np.concatenate([zt, zt, zt])
    big_d = np.concatenate([zd, zd, zd])
    o2 = oracle.verify_ragged(big_t, big_d, bad, np.concatenate([tok, tok, tok]), temp,
                              np.concatenate([U, U, U]), Kmax, lib=lib)
    assert o2["status"][3] == oracle.ROW_BAD_COUNT and o2["accept_len"][3] == 0
    assert np.all(o2["out_tokens"][3] == -1)


def _top_mask(z, F):
    """numpy lexsort: the F largest logits, ties to the lower index."""
    order = np.lexsort((np.arange(len(z)), -z.astype(np.float64)))
    m = np.zeros(len(z), bool)
    m[order[:F]] = True
    return m


def check_saguaro_library(lib):
    """[SSD] §4.2.1: sigma_{F,C}(z/T) = scipy softmax(z/T + log(C) on top_F(z))."""
    from scipy.special import softmax
    rng = np.random.default_rng(41)
    for _ in range(40):
        V = int(rng.integers(2, 40))
        z = (rng.integers(-3, 4, V) * 0.5 if rng.random() < 0.3 else rng.normal(0, 2, V)).astype(np.float32)
        T = float(rng.choice([0.5, 1.0, 2.0]))
        F = int(rng.integers(1, V))
        C = float(rng.choice([0.1, 47 / 147, 0.5, 1.0]))
        want = softmax(z.astype(np.float64) / T + np.where(_top_mask(z, F), np.log(C), 0.0))
        np.testing.assert_allclose(oracle.saguaro_probs(z, T, F, C, lib=lib), want, rtol=1e-12,
                                   atol=1e-15)


def check_saguaro_thm19(lib):
    """[SSD] Theorem 19 (Appendix A.3): p_d = (.49,.49,.01,.01) with F = 2 and
    C = 47/147 becomes (.47,.47,.03,.03); the acceptance rate against
    p_t = (.48,.48,.02,.02) is 0.98 with either; after a rejection the bonus
    lands in the cache (top-2 of the draft) always with Saguaro, never without."""
    g = golden("ssd_theorem19.json")
    F, C = g["F"], g["C_num"] / g["C_den"]
    zd = np.log(np.array(g["p_draft"])).astype(np.float32)
    zt = np.log(np.array(g["p_target"])).astype(np.float32)
    q = oracle.saguaro_probs(zd, 1.0, F, C, lib=lib)
    np.testing.assert_allclose(q, g["p_draft_saguaro"], atol=2e-7)
    # sampling from it: inverse CDF at U
    s = oracle.saguaro_sample(np.stack([zd] * 4), np.ones(4, np.float32), F, C,
                              np.array([0.2, 0.6, 0.95, 0.99], np.float32), lib=lib)
    assert list(s["tokens"]) == [0, 1, 2, 3]
    np.testing.assert_allclose(s["q"], g["p_draft_saguaro"], atol=2e-7)
    B = 64
    rng = np.random.default_rng(19)
    U = rng.uniform(0, 1, (B, 2)).astype(np.float32)
    U[:, 0] = 0.999  # reject whenever p/q < 1
    tgt = np.broadcast_to(np.stack([zt, zt])[None], (B, 2, 4))
    dft = np.broadcast_to(zd[None, None], (B, 1, 4))
    for sg, tok, in_cache in (((F, C), 2, True), (None, 0, False)):
        toks = np.full((B, 1), tok, np.int32)
        o = oracle.verify(tgt, dft, toks, np.ones(B, np.float32), U, lib=lib, saguaro=sg)
        np.testing.assert_allclose(o["alpha"][:, 0], g["acceptance_rate_both"], atol=2e-7)
        assert (o["accept_len"] == 0).all()  # p/q = 2/3 (Saguaro) or 0.98 (plain) < 0.999
        bonus = o["out_tokens"][:, 0]
        assert (np.isin(bonus, [0, 1]) == in_cache).all(), (sg, bonus)


def check_saguaro_thm15_monotone(lib):
    """[SSD] Theorem 15: with the cache S = top_F(z_d), the share of residual
    mass max(p_t - sigma_{F,C}, 0) inside S is non-increasing in C."""
    from scipy.special import softmax
    rng = np.random.default_rng(15)
    Cs = np.linspace(0.0, 1.0, 21)
    for _ in range(30):
        V = int(rng.integers(4, 30))
        zd = rng.normal(0, 1.5, V).astype(np.float32)
        zt = (zd + rng.normal(0, 1.0, V)).astype(np.float32)
        F = int(rng.integers(1, V - 1))
        pt = softmax(zt.astype(np.float64))
        S = _top_mask(zd, F)
        hit = []
        for C in Cs:
            if C == 0.0 and S.all():
                continue
            u = np.maximum(pt - oracle.saguaro_probs(zd, 1.0, F, float(C), lib=lib), 0.0)
            hit.append(u[S].sum() / u.sum() if u.sum() > 0 else 1.0)
        assert all(a >= b - 1e-12 for a, b in zip(hit, hit[1:])), hit


def check_saguaro_exact_law(lib):
    """Verification of drafts sampled from sigma_{F,C}: the output law is
    exactly the target's (the enumeration weights drafts by sigma)."""
    rng = np.random.default_rng(42)
    V, K, F, C = 5, 2, 2, Fr(1, 3)
    for _ in range(3):
        P = rational_rows(rng, K + 1, V)
        Pd = rational_rows(rng, K, V)
        Q = []
        for row in Pd:
            zr = np.array([math.log(float(x)) for x in row])
            m = _top_mask(zr, F)
            w = [x * (C if m[v] else 1) for v, x in enumerate(row)]
            tot = sum(w)
            Q.append([x / tot for x in w])
        leaves = enumerate_pieces(P, Q)
        tokens = np.array([lf[1] for lf in leaves], np.int32)
        uniforms = np.array([[float(u) for u in lf[2]] for lf in leaves], np.float32)
        B = len(leaves)
        zt, zd = logits_for(P), logits_for(Pd)
        out = oracle.verify(np.broadcast_to(zt[None], (B,) + zt.shape),
                            np.broadcast_to(zd[None], (B,) + zd.shape), tokens,
                            np.ones(B, np.float32), uniforms, nthreads=0, lib=lib,
                            saguaro=(F, float(C)))
        for i in range(K + 1):
            mass = Fr(0)
            law = [Fr(0)] * V
            for (w, _, _), ni, tk in zip(leaves, out["accept_len"], out["out_tokens"]):
                if ni >= i:
                    mass += w
                    law[tk[i]] += w
            assert [l / mass for l in law] == P[i], i


def check_saguaro_sampler_inverse_cdf(lib):
    """Draft-side sampling = numpy searchsorted on the cumulative sigma."""
    rng = np.random.default_rng(43)
    B, V = 50, 23
    z = rng.normal(0, 2, (B, V)).astype(np.float32)
    T = rng.choice([0.0, 0.7, 1.0], B).astype(np.float32)
    U = rng.uniform(0, 1, B).astype(np.float32)
    out = oracle.saguaro_sample(z, T, 3, 0.25, U, lib=lib)
    for b in range(B):
        if T[b] == 0:
            assert out["tokens"][b] == int(np.argmax(z[b]))
            continue
        q = oracle.saguaro_probs(z[b], float(T[b]), 3, 0.25, lib=lib)
        t = int(np.searchsorted(np.cumsum(q), float(U[b]), side="right"))
        assert out["tokens"][b] == min(t, V - 1) and abs(out["q"][b] - q[out["tokens"][b]]) < 1e-15


# ---------------------------------------------------------------------------
# Multi-step speculative sampling at a token-tree node ([CS349D] §6.4)

def mss_pieces(P, Q, m: int):
    """Leaves of MSS with m candidates drawn i.i.d. from Q, in exact rationals.

    Each leaf is (probability, candidates, uniforms, token): the candidates
    occur with probability prod Q(x_j); u_j in [0, a_j) accepts x_j, with
    a_j = min(1, P_j(x_j)/Q(x_j)) and P_{j+1} = norm(max(0, P_j - Q)); when
    all m are rejected, u_m picks the token of P_{m+1} by its CDF.  The
    uniforms are interval midpoints, so a correct MSS takes the leaf's token.
    """
    import itertools
    V = len(P)
    half = Fr(1, 2)
    leaves = []
    for x in itertools.product(range(V), repeat=m):
        w = Fr(1)
        for xi in x:
            w *= Q[xi]
        if w == 0:
            continue
        pj = list(P)
        reach = Fr(1)
        pre = []
        for j in range(m):
            a = min(Fr(1), pj[x[j]] / Q[x[j]])
            if a > 0:
                leaves.append((w * reach * a, x, pre + [a / 2] + [half] * (m - j), x[j]))
            if a == 1:
                reach = Fr(0)
                break
            pre.append((a + 1) / 2)
            reach *= 1 - a
            r = [max(Fr(0), pj[v] - Q[v]) for v in range(V)]
            Z = sum(r)
            pj = [rv / Z for rv in r]
        if reach > 0:
            cum = Fr(0)
            for y in range(V):
                if pj[y] > 0:
                    leaves.append((w * reach * pj[y], x, pre + [cum + pj[y] / 2], y))
                cum += pj[y]
    return leaves


def check_mss_exact_enumeration(lib, seed: int = 11, V: int = 5, pairs: int = 3):
    """Theorem 4.2: over candidates drawn i.i.d. from q, the MSS output law is
    exactly p.  The oracle, run on every leaf of the exact enumeration, takes
    each leaf's token, and the leaves' law is P in exact rationals (m = 1..3)."""
    rng = np.random.default_rng(seed)
    for _ in range(pairs):
        P = rational_rows(rng, 1, V)[0]
        Q = rational_rows(rng, 1, V)[0]
        for m in (1, 2, 3):
            leaves = mss_pieces(P, Q, m)
            law = [Fr(0)] * V
            for w, _, _, y in leaves:
                law[y] += w
            assert law == P, m
            B = len(leaves)
            zt, zq = logits_for([P])[0], logits_for([Q])[0]
            out = oracle.mss(np.broadcast_to(zt, (B, V)), np.broadcast_to(zq, (B, V)),
                             np.array([lf[1] for lf in leaves], np.int32),
                             np.ones(B, np.float32),
                             np.array([[float(u) for u in lf[2]] for lf in leaves], np.float32),
                             nthreads=0, lib=lib)
            assert not (out["status"] & oracle.ROW_ERRORS).any()
            got = out["token"]
            want = np.array([lf[3] for lf in leaves])
            assert np.array_equal(got, want), (m, np.nonzero(got != want)[0][:5])
            acc = out["accepted"]
            for i, (w, x, us, y) in enumerate(leaves):
                assert acc[i] == -1 or x[acc[i]] == y


def _dirichlet_pairs(seed: int, n: int, V: int = 5):
    rng = np.random.default_rng(seed)
    return [(rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))) for _ in range(n)]


def check_mss_law_thm42_thm43(lib):
    """The exact-law routine: sum over candidate tuples weighted by prod q is p
    (Theorem 4.2), and MSS accepts at least as often as naive sampling
    (Theorem 4.3), on 200 random pairs over V = 5 with m = 1..3."""
    import itertools
    V = 5
    for p, q in _dirichlet_pairs(5, 200, V):
        for m in (1, 2, 3):
            tot = np.zeros(V)
            pm = pn = 0.0
            for x in itertools.product(range(V), repeat=m):
                w = float(np.prod(q[list(x)]))
                law, pa = oracle.mss_law(p, q, np.array(x), lib=lib)
                _, pan = oracle.mss_law(p, q, np.array(x), naive=True, lib=lib)
                tot += w * law
                pm += w * pa
                pn += w * pan
            assert np.abs(tot - p).max() < 1e-12, m
            assert pm >= pn - 1e-12, (m, pm, pn)


def check_mss_topk_misuse(lib):
    """[CS349D] §6.4: candidates taken deterministically as the top-k of q with
    the same ratio rule do not give p (mean TV 0.24-0.34 on the pages' pairs,
    whose family is not stated; Dirichlet(1) pairs over V = 5 give about 0.30,
    0.36, 0.40 for k = 1, 2, 3), while naive sampling with the same candidates
    gives p exactly."""
    for k in (1, 2, 3):
        tv = []
        for p, q in _dirichlet_pairs(6, 300):
            x = np.argsort(-q, kind="stable")[:k]
            law, _ = oracle.mss_law(p, q, x, lib=lib)
            tv.append(0.5 * np.abs(law - p).sum())
            lawn, pan = oracle.mss_law(p, q, x, naive=True, lib=lib)
            assert np.abs(lawn - p).max() < 1e-15 and abs(pan - p[x].sum()) < 1e-15
        assert 0.2 < float(np.mean(tv)) < 0.5, (k, np.mean(tv))


def check_mss_single_candidate_is_sd(lib):
    """One candidate is plain speculative sampling: the same accept decision
    and token as verification with K = 1 after a rejection."""
    rng = np.random.default_rng(12)
    B, V = 400, 37
    zt = rng.normal(0, 2, (B, V)).astype(np.float32)
    zq = (zt + rng.normal(0, 1, (B, V))).astype(np.float32)
    T = rng.choice([0.7, 1.0, 1.3], B).astype(np.float32)
    x = rng.integers(0, V, (B, 1)).astype(np.int32)
    U = rng.uniform(0, 1, (B, 2)).astype(np.float32)
    o = oracle.mss(zt, zq, x, T, U, lib=lib)
    tgt = np.stack([zt, zt], axis=1)  # K + 1 = 2 target rows (row 1 unused on rejection)
    v = oracle.verify(tgt, zq[:, None, :], x, T, U, lib=lib)
    assert np.array_equal(o["accepted"] == 0, v["accept_len"] == 1)
    rej = v["accept_len"] == 0
    assert np.array_equal(o["token"][rej], v["out_tokens"][rej, 0])
    assert np.array_equal(o["token"][~rej], x[~rej, 0])
    assert np.allclose(o["accept_prob"][:, 0], np.minimum(1.0, v["p"][:, 0] / v["q"][:, 0]))


def check_mss_naive_and_greedy(lib):
    """Naive sampling: the token is the inverse-CDF draw from p (numpy
    searchsorted on the library softmax) and a candidate is accepted iff it is
    that token.  T = 0: the first candidate equal to argmax p, else argmax p."""
    from scipy.special import softmax
    rng = np.random.default_rng(13)
    B, V, M = 300, 29, 3
    zt = rng.normal(0, 2, (B, V)).astype(np.float32)
    zq = (zt + rng.normal(0, 1, (B, V))).astype(np.float32)
    T = rng.choice([0.0, 0.8, 1.0], B).astype(np.float32)
    x = rng.integers(0, V, (B, M)).astype(np.int32)
    x[::4, 1] = np.argmax(zt[::4], axis=1)  # some nodes hold the argmax
    U = rng.uniform(0, 1, (B, M + 1)).astype(np.float32)
    for naive in (False, True):
        o = oracle.mss(zt, zq, x, T, U, naive=naive, lib=lib)
        for b in range(B):
            if T[b] == 0:
                am = int(np.argmax(zt[b]))
                hits = np.nonzero(x[b] == am)[0]
                assert o["token"][b] == am and o["accepted"][b] == (hits[0] if len(hits) else -1)
            elif naive:
                p = softmax(zt[b].astype(np.float64) / T[b])
                y = min(int(np.searchsorted(np.cumsum(p), float(U[b, M]), side="right")), V - 1)
                assert o["token"][b] == y
                hits = np.nonzero(x[b] == y)[0]
                assert o["accepted"][b] == (hits[0] if len(hits) else -1)
                assert (o["accept_prob"][b] == 0).all()


def check_mss_boundary_flags(lib):
    """MSS and naive sampling flag a node as a boundary case where the
    definition puts it: a candidate's uniform within 1e-6 of its acceptance
    ratio, or the draw's U * R within 1e-6 * R of a CDF step.  One node with
    p = (.5, .3, .2), q = (.25, .5, .25) at T = 1; candidate 1 has p/q = 0.6."""
    lp = np.log(np.array([0.5, 0.3, 0.2]))
    lq = np.log(np.array([0.25, 0.5, 0.25]))
    zt = np.tile(lp, (6, 1)).astype(np.float32)
    zq = np.tile(lq, (6, 1)).astype(np.float32)
    x = np.array([[1], [1], [1], [1], [1], [1]], np.int32)
    T = np.ones(6, np.float32)
    U = np.array([[0.6 + 5e-7, 0.5],     # rejected on the boundary of the ratio
                  [0.6 - 5e-7, 0.5],     # accepted on it
                  [0.59, 0.5],           # accepted, clear
                  [0.9, 0.5],            # rejected; residual (.25, 0, 0): draw clear of its steps
                  [0.9, 0.0 + 3e-7],     # rejected; U * R within 1e-6 * R of the step at 0
                  [0.9, 0.5]], np.float32)
    o = oracle.mss(zt, zq, x, T, U, lib=lib)
    assert o["accepted"].tolist() == [-1, 0, 0, -1, -1, -1], o["accepted"]
    assert o["boundary"].tolist() == [1, 1, 0, 0, 1, 0], o["boundary"]
    # naive sampling: the draw from p itself, steps at 0.5 and 0.8
    Un = np.array([[0.0, 0.5 + 5e-7], [0.0, 0.8 - 5e-7], [0.0, 0.65],
                   [0.0, 0.3], [0.0, 0.9], [0.0, 0.1]], np.float32)
    o = oracle.mss(zt, zq, x, T, Un, naive=True, lib=lib)
    assert o["token"].tolist() == [1, 1, 1, 0, 2, 0], o["token"]
    assert o["boundary"].tolist() == [1, 1, 0, 0, 0, 0], o["boundary"]


def check_mss_bad_inputs(lib):
    """Out-of-range candidates (ROW_BAD_TOKEN), counts outside [0, M]
    (ROW_BAD_COUNT) and bad temperatures flag the node and produce no token."""
    V, M = 7, 2
    z = np.zeros((4, V), np.float32)
    x = np.array([[1, 2], [1, 9], [1, 2], [1, 2]], np.int32)
    T = np.array([1.0, 1.0, -1.0, 1.0], np.float32)
    nc = np.array([2, 2, 2, 3], np.int32)
    o = oracle.mss(z, z, x, T, np.full((4, M + 1), 0.5, np.float32), num_cands=nc, lib=lib)
    assert o["status"][0] == 0 and o["token"][0] >= 0
    assert o["status"][1] & oracle.ROW_BAD_TOKEN and o["token"][1] == -1
    assert o["status"][2] & oracle.ROW_BAD_TEMP and o["token"][2] == -1
    assert o["status"][3] & oracle.ROW_BAD_COUNT and o["token"][3] == -1
    # a node with no candidates draws from p (naive and MSS alike)
    o0 = oracle.mss(z[:1], z[:1], x[:1], T[:1], np.full((1, M + 1), 0.5, np.float32),
                    num_cands=np.array([0], np.int32), lib=lib)
    assert o0["accepted"][0] == -1 and o0["token"][0] == 3  # uniform p on 7: U = .5 -> v = 3


ALL_CHECKS = {
    "softmax_library": check_softmax_library,
    "verify_library": check_verify_library,
    "boundary_flags": check_boundary_flags,
    "thm1_overlap": check_thm1_overlap,
    "exercise_1": check_exercise_1,
    "section_2_3": check_section_2_3,
    "exact_enumeration": check_exact_enumeration,
    "exact_enumeration_T07": lambda lib: check_exact_enumeration(lib, seed=4, T=0.7, K=2),
    "exact_enumeration_K3": lambda lib: check_exact_enumeration(lib, seed=9, V=4, K=3, pairs=2),
    "expected_tokens": check_expected_tokens,
    "wrong_method_a_is_biased": check_wrong_method_a_is_biased,
    "greedy": check_greedy,
    "invariants": check_invariants,
    "bad_inputs": check_bad_inputs,
    "fallback_zero_residual": check_fallback_zero_residual,
    "predict_library_sort": check_predict_library_sort,
    "predict_exclusion": check_predict_exclusion,
    "hit_constructed": check_hit_constructed,
    "fanout_optimal": check_fanout_optimal,
    "fanout_rounding": check_fanout_rounding,
    "predict_fanout": check_predict_fanout,
    "no_draft_one_hot": check_no_draft_is_one_hot_draft,
    "no_draft_exact_law": check_no_draft_exact_law,
    "ragged_rows": check_ragged_matches_rows,
    "saguaro_library": check_saguaro_library,
    "saguaro_thm19": check_saguaro_thm19,
    "saguaro_thm15": check_saguaro_thm15_monotone,
    "saguaro_exact_law": check_saguaro_exact_law,
    "saguaro_sampler": check_saguaro_sampler_inverse_cdf,
    "mss_exact_enumeration": check_mss_exact_enumeration,
    "mss_law_thm42_thm43": check_mss_law_thm42_thm43,
    "mss_topk_misuse": check_mss_topk_misuse,
    "mss_single_candidate": check_mss_single_candidate_is_sd,
    "mss_naive_and_greedy": check_mss_naive_and_greedy,
    "mss_boundary_flags": check_mss_boundary_flags,
    "mss_bad_inputs": check_mss_bad_inputs,
}
