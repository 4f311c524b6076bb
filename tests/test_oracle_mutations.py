"""Mutation check of the oracle's pins, on the numpy oracle.

Each case plants one plausible mistake in the numpy fp64 oracle (on the CPU,
by replacing one of its functions for the duration of the case): a dropped
or doubled term, a wrong sign, index or comparison, a transposed operand, an
off-by-one bound, another reading of a convention.  The pins in
test_oracle_pins, run against that oracle, must then fail somewhere; a
mistake that every pin lets through would mean the pins do not fix that part
of the oracle.  test_oracle_mutations_cpp plants the same mistakes in the
source of the C++ oracle.  CPU only.
"""
import math

import numpy as np
import pytest

from oracle import numpy_oracle as O
from tests.pin_runner import PIN_CASES, first_failing_pin


def _first_failing_pin(hints):
    return first_failing_pin(O, hints)


# ---------------------------------------------------------------- mistakes

def _split_unshifted(q, K, V, scale, bounds):
    out = []
    G, D = q.shape[0], V.shape[1]
    for a, b in bounds:
        if b <= a:
            out.append((np.full(G, O.NEG_INF), np.zeros(G), np.zeros((G, D))))
            continue
        x = scale * (q @ K[a:b].T)
        w = np.exp(x)                                    # max not subtracted
        out.append((x.max(axis=1), w.sum(axis=1), w @ V[a:b]))
    return out


def _combine(unscaled_acc=False, sink_per_split=False):
    def combine(parts, sink=None):
        G, D = parts[0][2].shape
        M = np.full(G, O.NEG_INF)
        for m, _, _ in parts:
            M = np.maximum(M, m)
        if sink is not None:
            M = np.maximum(M, np.asarray(sink, np.float64))
        o, lse = np.zeros((G, D)), np.full(G, O.NEG_INF)
        for g in range(G):
            if M[g] == O.NEG_INF:
                continue
            L, acc = 0.0, np.zeros(D)
            for m, l, a in parts:
                if sink is not None and sink_per_split:
                    L += math.exp(float(sink[g]) - M[g])
                if m[g] == O.NEG_INF:
                    continue
                f = math.exp(m[g] - M[g])
                L += l[g] * f
                acc += a[g] * (1.0 if unscaled_acc else f)
            if sink is not None and not sink_per_split:
                L += math.exp(float(sink[g]) - M[g])
            o[g] = acc / L
            lse[g] = M[g] + math.log(L)
        return o, lse
    return combine


def _minmax_past_context(K, n, page_size):
    NP = O.num_pages(n, page_size)
    blks = [K[p * page_size:(p + 1) * page_size] for p in range(NP)]   # n ignored
    return np.array([b.min(axis=0) for b in blks]), np.array([b.max(axis=0) for b in blks])


def _bound(kind):
    def bound(q, kmin, kmax, chunk=4096):
        lo, hi = q[:, None, :] * kmin[None], q[:, None, :] * kmax[None]
        if kind == "kmax":
            return hi.sum(axis=2)
        return np.minimum(lo, hi).sum(axis=2)
    return bound


def _forced_late(n, page_size, n_sink_pages, n_local_tokens):
    NP = O.num_pages(n, page_size)
    f = set(range(min(n_sink_pages, NP)))
    if n_local_tokens > 0 and n > 0:
        f.update(range(max(n - n_local_tokens, 0) // page_size + 1, NP))   # one page late
    return np.array(sorted(f), dtype=np.int64)


def _topk(variant):
    def select(score, k, forced):
        NP = score.shape[0]
        if NP <= k:
            return np.arange(NP, dtype=np.int64)
        forced = np.asarray(forced, dtype=np.int64)
        cand = np.setdiff1d(np.arange(NP), forced)
        kk = k if variant == "budget" else k - forced.size
        key = -cand if variant == "ties" else cand
        chosen = cand[np.lexsort((key, -score[cand]))[:kk]]
        out = np.concatenate([forced, chosen])
        return out if variant == "unsorted" else np.sort(out)
    return select


def _kth_off_by_one(score, k, forced):
    NP = score.shape[0]
    if NP <= k:
        return O.NEG_INF
    cand = np.setdiff1d(np.arange(NP), np.asarray(forced, dtype=np.int64))
    kk = k - len(forced)
    if kk <= 0:
        return math.inf
    order = np.lexsort((cand, -score[cand]))
    return float(score[cand[order[min(kk, len(order) - 1)]]])


def _tokens_one_past(pages, n, page_size):
    toks = [np.arange(p * page_size, min((p + 1) * page_size, n + 1)) for p in pages if p >= 0]
    return np.concatenate(toks) if toks else np.zeros(0, dtype=np.int64)


def _thumb(kind):
    def quantize(Kb):
        s = Kb.max(axis=0) if kind == "signed_max" else np.abs(Kb).max(axis=0)
        h = s / 2.0
        if kind == "strict":
            codes = np.where(Kb > h, 3, np.where(Kb > 0, 2, np.where(Kb > -h, 1, 0)))
        else:
            codes = np.where(Kb >= h, 3, np.where(Kb >= 0, 2, np.where(Kb >= -h, 1, 0)))
        return codes.astype(np.uint8), s
    return quantize


def _pack_high_first(codes):
    T, D = codes.shape
    c = codes.reshape(T, D // 4, 4).astype(np.uint32)
    return (c[:, :, 3] | (c[:, :, 2] << 2) | (c[:, :, 1] << 4) | (c[:, :, 0] << 6)).astype(np.uint8)


def _pseudo_max_sink_only(q, K, n, block, scale):
    toks = O.pages_to_tokens(np.array([0]), n, block)
    return (scale * (q @ K[toks].T)).max(axis=1)


def _margin_min_over_heads(q, K, n, block, scale):
    forced = set(O.delta_forced_blocks(n, block).tolist())
    mt = O.pseudo_max(q, K, n, block, scale)
    blocks, margins = [], []
    for j in range(n // block):
        if j in forced:
            continue
        c, s = O.thumb_quantize(K[j * block:(j + 1) * block])
        st = scale * (q @ O.thumb_dequant(c, s).T)
        blocks.append(j)
        margins.append(float((st - mt[:, None]).max(axis=1).min()))   # min over heads
    return np.array(blocks, dtype=np.int64), np.array(margins)


def _delta_strict(q, K, n, block, delta, scale):
    blocks, margins = O.delta_block_margin(q, K, n, block, scale)
    kept = blocks[margins > -delta]
    return np.union1d(O.delta_forced_blocks(n, block), kept).astype(np.int64), (blocks, margins)


def _residual(denom=508.0, rounding=np.rint):
    def quantize(Kb, codes, s):
        Kb = np.asarray(Kb, np.float64)
        s = np.broadcast_to(np.asarray(s, np.float64), Kb.shape)
        e = Kb - O.thumb_dequant(codes, s)
        x = np.where(s > 0, e * denom / np.where(s > 0, s, 1.0), 0.0)
        return np.clip(rounding(x), -127, 127).astype(np.int8)
    return quantize


def _refined_minus(codes, s, r):
    return O.thumb_dequant(codes, s) - np.asarray(r, np.float64) * (np.asarray(s, np.float64) / O.RES_DENOM)


def _refined_unrefined(q, K, V, blocks, n, block, scale, sink=None):
    return O.sparse_attention_row(q, K, V, blocks, n, block, scale, sink)


def _recall_over_selected(q, K, pages, n, page_size, scale):
    if n == 0:
        return np.ones(q.shape[0])
    x = scale * (q @ K[:n].T)
    toks = O.pages_to_tokens(np.asarray(pages), n, page_size)
    w = np.exp(x - x.max(axis=1, keepdims=True))
    return w[:, toks].sum(axis=1) / np.maximum(w[:, toks].sum(axis=1), 1e-300)


def _to_f64_low_half(x, dtype):
    if dtype == "bf16":
        return np.asarray(x, dtype=np.uint16).astype(np.uint32).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def _split_empty_as_one(q, K, V, scale, bounds):
    G, D = q.shape[0], V.shape[1]
    out = []
    for a, b in bounds:
        if b <= a:
            out.append((np.zeros(G), np.ones(G), np.zeros((G, D))))   # an empty slice as a unit weight at 0
            continue
        out.extend(O.split_partials(q, K, V, scale, [(a, b)]))
    return out


def _thumbnails_with_partial(K, n, block):
    nb = -(-n // block)                                  # the partial block quantised too
    D = K.shape[1]
    codes = np.zeros((nb * block, D), dtype=np.uint8)
    scales = np.zeros((nb, D))
    for j in range(nb):
        c, sc = O.thumb_quantize(K[j * block:min((j + 1) * block, n)])
        codes[j * block:j * block + c.shape[0]] = c
        scales[j] = sc
    return codes, scales


def _unpack_reversed(packed):
    T, W = packed.shape
    p = packed.astype(np.uint32)
    return np.stack([(p >> (2 * (3 - j))) & 3 for j in range(4)], axis=2).reshape(T, W * 4).astype(np.uint8)


MUTATIONS = {
    # name: (oracle attribute, replacement built from the original, pins expected to catch it)
    "sink multiplied by the softmax scale": (
        "softmax_attention",
        lambda f: lambda q, K, V, scale, sink=None: f(q, K, V, scale, None if sink is None else np.asarray(sink) * scale),
        ["test_attention_golden"]),
    "sink dropped": (
        "softmax_attention", lambda f: lambda q, K, V, scale, sink=None: f(q, K, V, scale, None),
        ["test_attention_golden"]),
    "keys used as values": (
        "softmax_attention", lambda f: lambda q, K, V, scale, sink=None: f(q, K, K, scale, sink),
        ["test_softmax_attention_brute_force"]),
    "softmax scale dropped": (
        "softmax_attention", lambda f: lambda q, K, V, scale, sink=None: f(q, K, V, 1.0, sink),
        ["test_softmax_attention_brute_force"]),
    "split slices overlap by one key": (
        "split_partials",
        lambda f: lambda q, K, V, scale, bounds: f(q, K, V, scale,
                                                  [(a, min(b + 1, K.shape[0])) if b > a else (a, b) for a, b in bounds]),
        ["test_split_combine_equals_dense"]),
    "split partial not shifted by its max": ("split_partials", lambda f: _split_unshifted,
                                             ["test_split_combine_equals_dense"]),
    "combine does not rescale the accumulators": ("combine_partials", lambda f: _combine(unscaled_acc=True),
                                                  ["test_split_combine_equals_dense"]),
    "sink added once per split": ("combine_partials", lambda f: _combine(sink_per_split=True),
                                  ["test_split_combine_equals_dense"]),
    "page summaries read past the context": ("page_minmax", lambda f: _minmax_past_context,
                                             ["test_page_minmax_brute_force"]),
    "page min and max swapped": ("page_minmax", lambda f: lambda K, n, P: f(K, n, P)[::-1],
                                 ["test_quest_golden"]),
    "page count rounded down": ("num_pages", lambda f: lambda n, P: int(n) // int(P),
                                ["test_page_minmax_brute_force"]),
    "bound from kmax alone": ("quest_bound", lambda f: _bound("kmax"), ["test_quest_bound_admissible_and_identity"]),
    "bound takes the smaller product": ("quest_bound", lambda f: _bound("min"),
                                        ["test_quest_bound_admissible_and_identity"]),
    "group score sums its heads": ("group_score", lambda f: lambda U: U.sum(axis=0), ["test_quest_golden"]),
    "group score averages its heads": ("group_score", lambda f: lambda U: U.mean(axis=0),
                                       ["test_quest_bound_admissible_and_identity"]),
    "local pages start one page late": ("forced_pages", lambda f: _forced_late, ["test_forced_pages"]),
    "sink pages ignored": ("forced_pages", lambda f: lambda n, P, ns, nl: f(n, P, 0, nl), ["test_forced_pages"]),
    "ties go to the higher page index": ("select_topk", lambda f: _topk("ties"),
                                         ["test_topk_ties_at_the_budget_boundary"]),
    "budget excludes the forced pages": ("select_topk", lambda f: _topk("budget"), ["test_topk_brute_force"]),
    "page list left unsorted": ("select_topk", lambda f: _topk("unsorted"), ["test_topk_brute_force"]),
    "k-th score off by one": ("kth_score", lambda f: _kth_off_by_one, ["test_kth_score_is_the_last_admitted_score"]),
    "page tokens run one past the context": ("pages_to_tokens", lambda f: _tokens_one_past,
                                             ["test_partial_pages_equal_minus_inf_padding"]),
    "bf16 read from the low half-word": ("to_f64", lambda f: _to_f64_low_half,
                                         ["test_to_f64_decodes_bf16_bit_patterns"]),
    "values on a threshold take the lower level": ("thumb_quantize", lambda f: _thumb("strict"),
                                                   ["test_thumbnail_golden", "test_thumbnail_error_bound_and_packing"]),
    "thumbnail scale from the signed max": ("thumb_quantize", lambda f: _thumb("signed_max"),
                                            ["test_thumbnail_error_bound_and_packing"]),
    "thumbnail levels not halved": ("thumb_dequant", lambda f: lambda c, s: (c.astype(np.float64) - 1.5) * s,
                                    ["test_thumbnail_golden"]),
    "codes packed high bits first": ("pack_codes", lambda f: _pack_high_first, ["test_pack_format_bits"]),
    "newest block taken as n // block": (
        "delta_forced_blocks",
        lambda f: lambda n, block: np.zeros(0, np.int64) if n <= 0 else np.array(sorted({0, n // block}), np.int64),
        ["test_delta_invariants"]),
    "pseudo-max from the sink block only": ("pseudo_max", lambda f: _pseudo_max_sink_only,
                                            ["test_pseudo_max_covers_sink_and_local_blocks"]),
    "block margin takes the min over heads": ("delta_block_margin", lambda f: _margin_min_over_heads,
                                              ["test_delta_invariants"]),
    "strict keep test": ("delta_select_row", lambda f: _delta_strict, ["test_delta_keep_rule_at_the_boundary"]),
    "residual on a 512 denominator": ("residual_quantize", lambda f: _residual(denom=512.0),
                                      ["test_residual_golden"]),
    "residual truncated instead of rounded": ("residual_quantize", lambda f: _residual(rounding=np.trunc),
                                              ["test_residual_is_the_nearest_level_brute_force"]),
    "residual subtracted from the level": ("refined_keys", lambda f: _refined_minus, ["test_residual_golden"]),
    "refinement skipped": ("refined_attention_row", lambda f: _refined_unrefined,
                           ["test_refined_attention_brute_force"]),
    "recall normalised by the selected mass": ("attention_mass_recall", lambda f: _recall_over_selected,
                                               ["test_recall_equals_mass_ratio_of_the_lse"]),
    "empty context recalls nothing": (
        "attention_mass_recall",
        lambda f: lambda q, K, pages, n, P, scale: np.zeros(q.shape[0]) if n == 0 else f(q, K, pages, n, P, scale),
        ["test_recall_bounds_additivity_and_monotonicity"]),
    "empty split counted as a unit weight": ("split_partials", lambda f: _split_empty_as_one,
                                             ["test_split_combine_equals_dense"]),
    "thumbnails of the partial block too": ("thumbnails_row", lambda f: _thumbnails_with_partial,
                                            ["test_refined_attention_brute_force"]),
    "codes unpacked high bits first": ("unpack_codes", lambda f: _unpack_reversed,
                                       ["test_thumbnail_error_bound_and_packing"]),
    "empty attention gives the mean of nothing": (
        "softmax_attention",
        lambda f: lambda q, K, V, scale, sink=None: (np.full((q.shape[0], q.shape[1]), np.nan), np.zeros(q.shape[0]))
        if K.shape[0] == 0 else f(q, K, V, scale, sink),
        ["test_empty_attention"]),
    "sparse attention ignores the page list": (
        "sparse_attention_row",
        lambda f: lambda q, K, V, pages, n, P, scale, sink=None: O.softmax_attention(q, K[:n], V[:n], scale, sink),
        ["test_recall_equals_mass_ratio_of_the_lse"]),
}


def test_every_pin_runs_clean():
    """Unmutated, every pin case passes (the check below means something)."""
    assert _first_failing_pin([]) is None
    assert len(PIN_CASES) > 50


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_fails_a_pin(name, monkeypatch):
    attr, make, hints = MUTATIONS[name]
    monkeypatch.setattr(O, attr, make(getattr(O, attr)))
    caught = _first_failing_pin(hints)
    assert caught is not None, f"no pin catches: {name}"
