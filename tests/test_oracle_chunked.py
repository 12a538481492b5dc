"""The oracle's multi-query (chunked) attention against its pins, and planted
mistakes that the pins must catch."""
import pytest

import oracle.paged_ops as ops
from tests import chunked_checks as cc


@pytest.mark.parametrize("check", cc.ALL, ids=lambda f: f.__name__)
def test_chunked_check(check):
    check()


_orig_positions = ops.query_positions
_orig_attend_one = ops.attend_one


def _positions_shifted(L, n):
    return [p + 1 if p + 1 < L else p for p in _orig_positions(L, n)]


def _positions_early(L, n):
    return [max(0, p - 1) for p in _orig_positions(L, n)]


def _positions_relative(L, n):
    _orig_positions(L, n)
    return list(range(n))


def _positions_not_causal(L, n):
    _orig_positions(L, n)
    return [L - 1] * n


def _attend_one_no_scale(q, k, v, scale):
    return _orig_attend_one(q, k, v, 1.0)


MUTANTS = {
    "mask one past the diagonal": ("query_positions", _positions_shifted),
    "mask one before the diagonal": ("query_positions", _positions_early),
    "positions relative to the chunk": ("query_positions", _positions_relative),
    "no causal mask": ("query_positions", _positions_not_causal),
    "scale dropped": ("attend_one", _attend_one_no_scale),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(ops, attr, fn)
    caught = []
    for check in cc.ALL:
        try:
            check()
        except (AssertionError, ValueError, IndexError, RuntimeError):
            caught.append(check.__name__)
    assert caught, f"no pin caught: {name}"
