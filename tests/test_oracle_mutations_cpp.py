"""Mutation check of the oracle's pins, on the C++ oracle.

Each case plants one plausible mistake in the source of the C++ oracle
(oracle/sls_oracle.cpp): one or a few exact text substitutions, each of
which must match the source exactly once.  The planted source is compiled
into a temporary library, and the pins of test_oracle_pins run against it in
a child process (so that a planted mistake that breaks memory safety cannot
take the test run down with it).  Some pin must fail for every case.  The
mistakes are the ones the numpy mutation check plants, written for the C++
source.  CPU only; the variants compile in parallel.
"""
import concurrent.futures
import json
import os
import subprocess
import sys

import pytest

from oracle import build_oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SOFTMAX_EMPTY = """    if (m == kNegInf) {
      lse[g] = kNegInf;
      continue;
    }
    double z = 0.0;"""

MARGIN_MAX = """  double best = kNegInf;
  for (int g = 0; g < G; ++g)
    for (int t = 0; t < block; ++t)
      best = std::max(best, scale * dot(q + (i64)g * D, kh.data() + (i64)t * D, D) - mt[g]);
  return best;"""

MARGIN_MIN_OVER_HEADS = """  double best = kPosInf;
  for (int g = 0; g < G; ++g) {
    double bg = kNegInf;
    for (int t = 0; t < block; ++t)
      bg = std::max(bg, scale * dot(q + (i64)g * D, kh.data() + (i64)t * D, D) - mt[g]);
    best = std::min(best, bg);
  }
  return best;"""

SPARSE_TOKENS = """  std::vector<i64> toks((size_t)(npages * P + 1));
  i64 nt = orc_pages_to_tokens(pages, npages, n, P, toks.data());
  std::vector<double> Kt((size_t)(nt * D + 1)), Vt((size_t)(nt * D + 1));
  for (i64 i = 0; i < nt; ++i)
    for (int c = 0; c < D; ++c) {"""

SPARSE_ALL_TOKENS = """  std::vector<i64> toks((size_t)n + 1);
  i64 nt = n;
  for (i64 t = 0; t < n; ++t) toks[t] = t;
  (void)pages;
  std::vector<double> Kt((size_t)(nt * D + 1)), Vt((size_t)(nt * D + 1));
  for (i64 i = 0; i < nt; ++i)
    for (int c = 0; c < D; ++c) {"""

# name: ([(source text, replacement), ...] applied in order, pins expected to catch it)
MUTANTS = {
    "sink multiplied by the softmax scale": (
        [("    if (sink) m = std::max(m, sink[g]);", "    if (sink) m = std::max(m, scale * sink[g]);"),
         ("    if (sink) z += std::exp(sink[g] - m);", "    if (sink) z += std::exp(scale * sink[g] - m);")],
        ["test_attention_golden"]),
    "sink dropped": (
        [("    if (sink) m = std::max(m, sink[g]);", "    if (false) m = std::max(m, sink[g]);"),
         ("    if (sink) z += std::exp(sink[g] - m);", "    if (false) z += std::exp(sink[g] - m);")],
        ["test_attention_golden"]),
    "keys used as values": (
        [("      for (int c = 0; c < Dv; ++c) og[c] += w * V[t * Dv + c];",
          "      for (int c = 0; c < Dv; ++c) og[c] += w * K[t * Dv + c];")],
        ["test_softmax_attention_brute_force"]),
    "softmax scale dropped": (
        [("      x[t] = scale * dot(q + (i64)g * Dq, K + t * Dq, Dq);", "      x[t] = dot(q + (i64)g * Dq, K + t * Dq, Dq);")],
        ["test_softmax_attention_brute_force"]),
    "split slices overlap by one key": (
        [("    i64 a = bounds[2 * s], b = bounds[2 * s + 1];",
          "    i64 a = bounds[2 * s] > 0 ? bounds[2 * s] - 1 : 0, b = bounds[2 * s + 1];")],
        ["test_split_combine_equals_dense"]),
    "split partial not shifted by its max": (
        [("        double w = std::exp(scale * dot(q + (i64)g * Dq, K + t * Dq, Dq) - *ms);",
          "        double w = std::exp(scale * dot(q + (i64)g * Dq, K + t * Dq, Dq));")],
        ["test_split_combine_equals_dense"]),
    "combine does not rescale the accumulators": (
        [("      for (int c = 0; c < D; ++c) og[c] += as[c] * f;", "      for (int c = 0; c < D; ++c) og[c] += as[c];")],
        ["test_split_combine_equals_dense"]),
    "sink added once per split": (
        [("    if (sink) L += std::exp(sink[g] - M);\n", ""),
         ("      double ms = m[(i64)s * G + g];\n",
          "      if (sink) L += std::exp(sink[g] - M);\n      double ms = m[(i64)s * G + g];\n")],
        ["test_split_combine_equals_dense"]),
    "page summaries read past the context": (
        [("    i64 t0 = p * P, t1 = std::min(t0 + P, n);", "    i64 t0 = p * P, t1 = t0 + P;")],
        ["test_partial_pages_equal_minus_inf_padding"]),
    "page min and max swapped": (
        [("      kmin[p * D + c] = lo;\n      kmax[p * D + c] = hi;", "      kmin[p * D + c] = hi;\n      kmax[p * D + c] = lo;")],
        ["test_quest_golden"]),
    "page count rounded down": (
        [("return (n + page_size - 1) / page_size;", "return n / page_size;")],
        ["test_page_minmax_brute_force"]),
    "bound from kmax alone": (
        [("        u += std::max(a, b);", "        u += b + 0.0 * a;")],
        ["test_quest_bound_admissible_and_identity"]),
    "bound takes the smaller product": (
        [("        u += std::max(a, b);", "        u += std::min(a, b);")],
        ["test_quest_bound_admissible_and_identity"]),
    "group score sums its heads": (
        [("    double s = kNegInf;\n    for (int g = 0; g < G; ++g) s = std::max(s, U[(i64)g * NP + p]);",
          "    double s = 0.0;\n    for (int g = 0; g < G; ++g) s += U[(i64)g * NP + p];")],
        ["test_quest_bound_admissible_and_identity"]),
    "group score averages its heads": (
        [("    double s = kNegInf;\n    for (int g = 0; g < G; ++g) s = std::max(s, U[(i64)g * NP + p]);",
          "    double s = 0.0;\n    for (int g = 0; g < G; ++g) s += U[(i64)g * NP + p] / G;")],
        ["test_quest_bound_admissible_and_identity"]),
    "local pages start one page late": (
        [("(i64)0) / P; p < NP; ++p) f[p] = 1;", "(i64)0) / P + 1; p < NP; ++p) f[p] = 1;")],
        ["test_forced_pages"]),
    "sink pages ignored": (
        [("  for (i64 p = 0; p < std::min((i64)n_sink_pages, NP); ++p) f[p] = 1;\n", "")],
        ["test_forced_pages"]),
    "ties go to the higher page index": (
        [("    return a < b;\n  });", "    return a > b;\n  });")],
        ["test_topk_ties_at_the_budget_boundary"]),
    "budget excludes the forced pages": (
        [("  for (i64 i = 0; i < k - nf && i < (i64)cand.size(); ++i)", "  for (i64 i = 0; i < k && i < (i64)cand.size(); ++i)")],
        ["test_topk_brute_force"]),
    "page list left unsorted": (
        [("  std::sort(out, out + cnt);\n", "")],
        ["test_topk_brute_force"]),
    "k-th score off by one": (
        [("  return score[cand[kk - 1]];", "  return score[cand[std::min(kk, (i64)cand.size() - 1)]];")],
        ["test_kth_score_is_the_last_admitted_score"]),
    "page tokens run one past the context": (
        [("t < std::min((p + 1) * P, n); ++t) out[cnt++] = t;", "t < std::min((p + 1) * P, n + 1); ++t) out[cnt++] = t;")],
        ["test_partial_pages_equal_minus_inf_padding"]),
    "bf16 read from the low half-word": (
        [("    uint32_t u = (uint32_t)bits[i] << 16;", "    uint32_t u = (uint32_t)bits[i];")],
        ["test_to_f64_decodes_bf16_bit_patterns"]),
    "values on a threshold take the lower level": (
        [("k >= h ? 3 : (k >= 0.0 ? 2 : (k >= -h ? 1 : 0));", "k > h ? 3 : (k > 0.0 ? 2 : (k > -h ? 1 : 0));")],
        ["test_thumbnail_golden", "test_thumbnail_error_bound_and_packing"]),
    "thumbnail scale from the signed max": (
        [("    double m = 0.0;\n    for (int t = 0; t < T; ++t) m = std::max(m, std::fabs(Kb[(i64)t * D + c]));",
          "    double m = kNegInf;\n    for (int t = 0; t < T; ++t) m = std::max(m, Kb[(i64)t * D + c]);")],
        ["test_thumbnail_error_bound_and_packing"]),
    "thumbnail levels not halved": (
        [("      out[(i64)t * D + c] = ((double)codes[(i64)t * D + c] - 1.5) * (sc / 2.0);",
          "      out[(i64)t * D + c] = ((double)codes[(i64)t * D + c] - 1.5) * sc;")],
        ["test_thumbnail_golden"]),
    "codes packed high bits first": (
        [("& 3) << (2 * j);", "& 3) << (2 * (3 - j));")],
        ["test_pack_format_bits"]),
    "newest block taken as n // block": (
        [("  i64 last = (n - 1) / block;", "  i64 last = n / block;")],
        ["test_delta_invariants"]),
    "pseudo-max from the sink block only": (
        [("  i64 nb = orc_delta_forced_blocks(n, block, fb);\n  std::vector<i64> toks((size_t)(2 * block));",
          "  i64 nb = std::min<i64>(orc_delta_forced_blocks(n, block, fb), 1);\n"
          "  std::vector<i64> toks((size_t)(2 * block));")],
        ["test_pseudo_max_covers_sink_and_local_blocks"]),
    "block margin takes the min over heads": (
        [(MARGIN_MAX, MARGIN_MIN_OVER_HEADS)],
        ["test_delta_invariants"]),
    "strict keep test": (
        [("    if (margins[i] >= -delta) sel[cnt++] = blocks[i];", "    if (margins[i] > -delta) sel[cnt++] = blocks[i];")],
        ["test_delta_keep_rule_at_the_boundary"]),
    "residual on a 512 denominator": (
        [("      double x = (Kb[i] - kh) * kResDenom / s[c];", "      double x = (Kb[i] - kh) * 512.0 / s[c];")],
        ["test_residual_error_bound"]),
    "residual truncated instead of rounded": (
        [("      double j = std::nearbyint(x);", "      double j = std::trunc(x);")],
        ["test_residual_is_the_nearest_level_brute_force"]),
    "residual subtracted from the level": (
        [("      out[(i64)t * D + c] += (double)r[(i64)t * D + c] * (sc / kResDenom);",
          "      out[(i64)t * D + c] -= (double)r[(i64)t * D + c] * (sc / kResDenom);")],
        ["test_residual_golden"]),
    "refinement skipped": (
        [("    if (j < nfull) {", "    if (false) {")],
        ["test_refined_attention_brute_force"]),
    "recall normalised by the selected mass": (
        [("    out[g] = sel / all;", "    out[g] = sel / std::max(sel, 1e-300) + 0.0 * all;")],
        ["test_recall_equals_mass_ratio_of_the_lse"]),
    "empty context recalls nothing": (
        [("    for (int g = 0; g < G; ++g) out[g] = 1.0;", "    for (int g = 0; g < G; ++g) out[g] = 0.0;")],
        ["test_recall_bounds_additivity_and_monotonicity"]),
    "empty split counted as a unit weight": (
        [("      if (b <= a) continue;", "      if (b <= a) {\n        *ms = 0.0;\n        *ls = 1.0;\n        continue;\n      }")],
        ["test_split_combine_equals_dense"]),
    "thumbnails of the partial block too": (
        [("  i64 nfull = n / block;\n  std::vector<double> Kt((size_t)(nt * D + 1))",
          "  i64 nfull = (n + block - 1) / block;\n  std::vector<double> Kt((size_t)(nt * D + 1))")],
        ["test_refined_attention_brute_force"]),
    "codes unpacked high bits first": (
        [(">> (2 * j)) & 3);", ">> (2 * (3 - j))) & 3);")],
        ["test_thumbnail_error_bound_and_packing"]),
    "empty attention gives the mean of nothing": (
        [(SOFTMAX_EMPTY, SOFTMAX_EMPTY.replace("    double z = 0.0;",
                                               "    if (T == 0) {\n      for (int c = 0; c < Dv; ++c) og[c] = std::nan(\"\");\n"
                                               "      lse[g] = 0.0;\n      continue;\n    }\n    double z = 0.0;"))],
        ["test_empty_attention"]),
    "sparse attention ignores the page list": (
        [(SPARSE_TOKENS, SPARSE_ALL_TOKENS)],
        ["test_recall_equals_mass_ratio_of_the_lse"]),
}


def planted_source(subs):
    """The oracle source with the substitutions applied in order; each must
    match exactly once where it is applied."""
    with open(build_oracle.SOURCE) as f:
        text = f.read()
    for old, new in subs:
        count = text.count(old)
        if count != 1:
            raise AssertionError(f"substitution matches {count} times: {old[:60]!r}")
        text = text.replace(old, new)
    return text


_CHILD = """
import json, sys
sys.path.insert(0, {root!r})
from oracle.sls_oracle import Oracle
from tests.pin_runner import first_failing_pin
print(json.dumps(first_failing_pin(Oracle({path!r}), {hints!r})))
"""


def _run_mutant(args):
    name, tmp = args
    subs, hints = MUTANTS[name]
    path = os.path.join(tmp, f"mutant_{list(MUTANTS).index(name)}.so")
    build_oracle.build(out=path, text=planted_source(subs), opt="-O1")
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, path=path, hints=hints)],
                       capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return {"caught": None, "error": f"child exited {r.returncode}: {r.stderr[-400:]}"}
    return {"caught": json.loads(r.stdout.strip().splitlines()[-1]), "error": None}


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    names = list(MUTANTS)
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        res = list(ex.map(_run_mutant, [(n, tmp) for n in names]))
    return dict(zip(names, res))


def test_substitutions_match_the_source_once():
    for name, (subs, _) in MUTANTS.items():
        planted_source(subs)


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_fails_a_pin(name, mutant_results):
    r = mutant_results[name]
    assert r["error"] is None, r["error"]
    assert r["caught"] is not None, f"no pin catches: {name}"
