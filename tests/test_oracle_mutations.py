"""Negative controls: oracle builds with one planted mistake must fail the pins.

Each mutation rewrites one line of a private copy of the oracle source (the
committed oracle is never changed), builds it with gcc, and asserts that the
listed pins reject it.  This shows the pins would catch a dropped term, a
wrong sign, a wrong index or a transposed operand in the oracle.
"""
import os

import pytest

import oracle
from tests import oracle_checks as oc

MUTATIONS = {
    # resample from p after a rejection (Lecture 5 §2.6, "wrong method A")
    "wrong_method_a": (
        "for (int v = 0; v < V; ++v) { r[v] = p[v] > q[v] ? p[v] - q[v] : 0.0; R += r[v]; }",
        "for (int v = 0; v < V; ++v) { r[v] = p[v]; R += r[v]; (void)q; }",
        ["exact_enumeration", "wrong_method_a_is_biased", "chisq_0.3", "verify_library"]),
    # residual max(q - p, 0), the garbled form on the survey blog
    "swapped_residual": (
        "r[v] = p[v] > q[v] ? p[v] - q[v] : 0.0;",
        "r[v] = q[v] > p[v] ? q[v] - p[v] : 0.0;",
        ["exact_enumeration", "verify_library"]),
    "ratio_inverted": (
        "accept = ratio >= (double)U[i];",
        "accept = 1.0 / ratio >= (double)U[i];",
        ["exercise_1", "exact_enumeration", "verify_library"]),
    "accept_uses_bonus_uniform": (
        "accept = ratio >= (double)U[i];",
        "accept = ratio >= (double)U[K];",
        ["exact_enumeration", "verify_library"]),
    "cdf_off_by_one": (
        "if (cum > tau) { tstar = v; break; }",
        "if (cum > tau) { tstar = v > 0 ? v - 1 : v; break; }",
        ["exact_enumeration", "section_2_3", "verify_library"]),
    "temperature_ignored": (
        "p[v] = exp((load_logit(base, dtype, off + v) - m) / T);",
        "p[v] = exp(load_logit(base, dtype, off + v) - m);",
        ["softmax_library", "exact_enumeration_T07", "verify_library"]),
    "greedy_last_max": (
        "if (z > m) { m = z; am = v; }",
        "if (z >= m) { m = z; am = v; }",
        ["greedy", "softmax_library"]),
    "no_stop_at_first_rejection": (
        "if (!accept) { n = i; break; }",
        "if (!accept) { n = i; }",
        ["exact_enumeration", "verify_library"]),
    "bonus_from_wrong_row": (
        "const double* p = pt + (int64_t)n * V;",
        "const double* p = pt + (int64_t)(n > 0 ? n - 1 : 0) * V;",
        ["exact_enumeration", "verify_library"]),
    "overlap_uses_max": (
        "a += (p[v] < q[v]) ? p[v] : q[v];",
        "a += (p[v] > q[v]) ? p[v] : q[v];",
        ["thm1_overlap", "exercise_1"]),
    "predict_no_exclusion": (
        "if (v == excl) continue;",
        "(void)excl;",
        ["predict_exclusion", "predict_library_sort"]),
    "predict_tie_order": (
        "return (x->v < y->v) ? -1 : (x->v > y->v);",
        "return (x->v > y->v) ? -1 : (x->v < y->v);",
        ["predict_library_sort"]),
    # Theorem 12 with the (1 - a) factor of F_K dropped
    "fanout_no_tail_factor": (
        "x[k] = (k < K) ? F0 * pow(a, k * g) : F0 * aK * pow(1.0 - a, -g);",
        "x[k] = (k < K) ? F0 * pow(a, k * g) : F0 * aK;",
        ["fanout_optimal"]),
    # exponent k/r instead of k/(1+r)
    "fanout_wrong_exponent": (
        "const double g = 1.0 / (1.0 + r);",
        "const double g = 1.0 / r;",
        ["fanout_optimal"]),
    # leftover budget to the smallest fractional parts
    "fanout_rounds_wrong_way": (
        "if (fk[k] == (int32_t)floor(x[k]) && frac > best_frac) { best = k; best_frac = frac; }",
        "if (fk[k] == (int32_t)floor(x[k]) && (best < 0 || frac < best_frac)) { best = k; best_frac = frac; }",
        ["fanout_rounding"]),
    "predict_fanout_ignored": (
        "const int Fk = fanout ? fanout[k] : F;",
        "const int Fk = F; (void)fanout;",
        ["predict_fanout"]),
    # NO_DRAFT_PROBS with a uniform instead of a one-hot draft distribution
    "no_draft_not_one_hot": (
        "for (int v = 0; v < V; ++v) qd[(int64_t)i * V + v] = (v == x[i]) ? 1.0 : 0.0;",
        "for (int v = 0; v < V; ++v) qd[(int64_t)i * V + v] = 1.0 / V;",
        ["no_draft_one_hot", "no_draft_exact_law"]),
    # ragged rows: target rows placed without the per-row bonus-row shift
    "ragged_target_offset": (
        "verify_row(kb, V, dtype, target, (c0 + b) * t_rs, t_rs, draft, c0 * d_rs, d_rs,",
        "verify_row(kb, V, dtype, target, c0 * t_rs, t_rs, draft, c0 * d_rs, d_rs,",
        ["ragged_rows"]),
    # Saguaro sampling down-weighting the F smallest logits
    "saguaro_bottom_f": (
        "for (int f = 0; f < F && f < V; ++f) p[c[f].v] *= C;",
        "for (int f = 0; f < F && f < V; ++f) p[c[V - 1 - f].v] *= C;",
        ["saguaro_library", "saguaro_thm19"]),
    "saguaro_not_renormalised": (
        "if (!(S > 0.0)) return ROW_NONFINITE;\n  for (int v = 0; v < V; ++v) p[v] /= S;",
        "if (!(S > 0.0)) return ROW_NONFINITE;",
        ["saguaro_library"]),
    # accept test with the plain draft probability after Saguaro sampling
    "saguaro_plain_q_in_accept": (
        ": sg_F > 0 ? log(qd[(int64_t)i * V + x[i]])",
        ": sg_F > 0 ? log_prob(draft, dtype, dof, x[i], T, md[i], lsd[i])",
        ["saguaro_exact_law"]),
    # MSS: the target left at p after a rejection (no residual step)
    "mss_no_residual_update": (
        "    for (int v = 0; v < V; ++v) pj[v] = r[v] / Z;\n  }\n  *tok_out = icdf_draw(pj",
        "    (void)Z;\n  }\n  *tok_out = icdf_draw(pj",
        ["mss_exact_enumeration"]),
    # MSS: every candidate tested against p instead of the current residual
    "mss_ratio_from_p": (
        "const double ratio = qx > 0.0 ? pj[x[j]] / qx : 0.0;",
        "const double ratio = qx > 0.0 ? p[x[j]] / qx : 0.0;",
        ["mss_exact_enumeration"]),
    # MSS: all candidates rejected, but the token drawn from p
    "mss_final_draw_from_p": (
        "*tok_out = icdf_draw(pj, V, (double)U[M], &fb, boundary);",
        "*tok_out = icdf_draw(p, V, (double)U[M], &fb, boundary);",
        ["mss_exact_enumeration"]),
    # MSS: candidate j tested with the draw's uniform
    "mss_accept_uses_draw_uniform": (
        "if (qx > 0.0 && ratio >= (double)U[j]) {",
        "if (qx > 0.0 && ratio >= (double)U[M]) {",
        ["mss_exact_enumeration"]),
    # the exact-law routine without the residual step
    "mss_law_no_residual": (
        "    for (int v = 0; v < V; ++v) pj[v] = r[v] / Z;\n  }\n  for (int v = 0; v < V; ++v) law[v] += reach * pj[v];",
        "    (void)Z;\n  }\n  for (int v = 0; v < V; ++v) law[v] += reach * pj[v];",
        ["mss_law_thm42_thm43"]),
    # naive sampling drawing from q
    "mss_naive_draws_from_q": (
        "*tok_out = icdf_draw(p, V, (double)U[M], &fb, boundary);\n    for (int j = 0; j < m; ++j)",
        "*tok_out = icdf_draw(q, V, (double)U[M], &fb, boundary);\n    for (int j = 0; j < m; ++j)",
        ["mss_naive_and_greedy"]),
    # the boundary band dropped, widened, or checked on one side of the step only
    "boundary_never": (
        "#define BOUNDARY_EPS 1e-6",
        "#define BOUNDARY_EPS 0.0",
        ["boundary_flags"]),
    "boundary_too_wide": (
        "#define BOUNDARY_EPS 1e-6",
        "#define BOUNDARY_EPS 1e-2",
        ["boundary_flags"]),
    "boundary_one_side": (
        "} else if (fabs(tau - prev) < BOUNDARY_EPS * R || fabs(cum - tau) < BOUNDARY_EPS * R) {",
        "} else if (fabs(cum - tau) < BOUNDARY_EPS * R) {",
        ["boundary_flags"]),
    "mss_draw_boundary_one_side": (
        "      if (fabs(tau - prev) < BOUNDARY_EPS * R || fabs(cum - tau) < BOUNDARY_EPS * R) *bd = 1;",
        "      if (fabs(cum - tau) < BOUNDARY_EPS * R) *bd = 1;",
        ["mss_boundary_flags"]),
    "mss_ratio_boundary_dropped": (
        "    if (qx > 0.0 && fabs((double)U[j] - ratio) < BOUNDARY_EPS) *boundary = 1;",
        "",
        ["mss_boundary_flags"]),
    # bf16 bits widened to the wrong place
    "bf16_decode_shift": (
        "uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;",
        "uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 15;",
        ["softmax_library"]),
    # NaN logits not flagged
    "nan_not_flagged": (
        "    if (isnan(z) || z == INFINITY) return ROW_NONFINITE;\n    if (z > m) { m = z; am = v; }",
        "    if (z == INFINITY) return ROW_NONFINITE;\n    if (z > m) { m = z; am = v; }",
        ["bad_inputs"]),
    # packed rows: uniforms without the per-row bonus slot
    "ragged_uniform_offset": (
        "tokens + c0, (double)temperature[b], uniforms + c0 + b, no_draft, 0, 1.0,",
        "tokens + c0, (double)temperature[b], uniforms + c0, no_draft, 0, 1.0,",
        ["ragged_rows"]),
    "hit_wrong_length": (
        "const int32_t* kk = keys + ((int64_t)b * (K + 1) + n) * F;",
        "const int32_t* kk = keys + ((int64_t)b * (K + 1) + 0) * F;",
        ["hit_constructed"]),
}


def _check(name):
    if name.startswith("chisq_"):
        a = float(name.split("_")[1])
        return lambda lib: oc.check_chisq(lib, a, draws=200_000)
    return oc.ALL_CHECKS[name]


@pytest.mark.parametrize("mut", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, mut):
    old, new, checks = MUTATIONS[mut]
    with open(oracle.SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor for {mut} not unique"
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = oracle.build(src=path, out=os.path.join(tmp_path, "libmutant.so"),
                      openmp=False, force=True)
    lib = oracle.load(so)
    for name in checks:
        with pytest.raises(AssertionError):
            _check(name)(lib)
