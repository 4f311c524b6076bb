"""Runs the oracle pins of test_oracle_pins in-process against a given
oracle (any object with the oracle's functions), for the mutation checks.

Each test function of test_oracle_pins is called with every combination of
its parametrize marks; the pins named in `hints` run first.  CPU only.
"""
import itertools

from tests import test_oracle_pins as PINS


def _pin_cases():
    cases = []
    for name, fn in vars(PINS).items():
        if not (name.startswith("test_") and callable(fn)):
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names, values = mark.args[0], mark.args[1]
            names = [s.strip() for s in names.split(",")] if isinstance(names, str) else list(names)
            grids.append([dict(zip(names, v if len(names) > 1 else (v,))) for v in values])
        for combo in itertools.product(*grids):
            kw = {}
            for d in combo:
                kw.update(d)
            cases.append((name, fn, kw))
    return cases


PIN_CASES = _pin_cases()


def first_failing_pin(oracle, hints):
    """Name (and arguments) of the first pin case that fails against
    `oracle`, hinted pins first; None when every pin passes."""
    ordered = [c for c in PIN_CASES if c[0] in hints] + [c for c in PIN_CASES if c[0] not in hints]
    saved = PINS.O
    PINS.O = oracle
    try:
        for name, fn, kw in ordered:
            try:
                fn(**kw)
            except Exception:  # an assertion or any error: the planted mistake shows
                return f"{name}{kw or ''}"
        return None
    finally:
        PINS.O = saved
