"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Every mutant replaces one oracle function for the duration of one test; the
pin tests of ``test_oracle_pins.py`` are then run against it and must fail.
"""

import math

import numpy as np
import pytest

import oracle.diffattn_oracle as om
import tests.test_oracle_pins as pins


def _transposed_scores(q, k, scale, causal, rows=None):
    q, k = om._f64(q), om._f64(k)
    rows = om._rows(rows, q.shape[0])
    s = (k @ q.T)[rows] * scale  # operands swapped
    if causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j <= rows[:, None], s, -np.inf)
    return om.softmax_rows(s)


def _off_by_one_mask(q, k, scale, causal, rows=None):
    q, k = om._f64(q), om._f64(k)
    rows = om._rows(rows, q.shape[0])
    s = (q[rows] @ k.T) * scale
    if causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j <= rows[:, None] + 1, s, -np.inf)  # sees one future key
    return om.softmax_rows(s)


def _plus_lambda(q1, k1, q2, k2, lam, causal, rows=None, scale=None):
    scale = 1 / math.sqrt(om._f64(q1).shape[-1]) if scale is None else scale
    return om.attention_map(q1, k1, scale, causal, rows) + lam * om.attention_map(q2, k2, scale, causal, rows)


def _norm_with_lambda_not_init(o, gamma, eps, lam_init):
    o = om._f64(o)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return gamma_or_one(gamma, o) * o / np.sqrt(ms + eps)  # drops the (1 - lambda_init) factor


def gamma_or_one(gamma, o):
    return np.ones(o.shape[-1]) if gamma is None else om._f64(gamma)


def _norm_over_tokens(o, gamma, eps, lam_init):
    o = om._f64(o)
    ms = np.mean(o * o, axis=0, keepdims=True)  # wrong axis
    return (1 - lam_init) * gamma_or_one(gamma, o) * o / np.sqrt(ms + eps)


MUTANTS = [
    ("attention_map", _transposed_scores, lambda: pins.test_lambda_zero_is_sdpa(False)),
    ("attention_map", _off_by_one_mask, lambda: pins.test_lambda_zero_is_sdpa(True)),
    ("difference_map", _plus_lambda, lambda: pins.test_rows_sum_to_one_minus_lambda(False, 0.8)),
    ("head_rmsnorm", _norm_with_lambda_not_init, pins.test_causal_row_zero_closed_form),
    ("head_rmsnorm", _norm_over_tokens, pins.test_head_rmsnorm_matches_torch_rms_norm),
]


@pytest.mark.parametrize("name,mutant,pin", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_pin_catches_mutant(monkeypatch, name, mutant, pin):
    pin()  # passes on the real oracle
    monkeypatch.setattr(om, name, mutant)
    monkeypatch.setattr(pins.oracle, name, mutant)
    with pytest.raises(AssertionError):
        pin()


def test_v2_pin_catches_halves_pairing(monkeypatch):
    real = om.diff_attn_v2

    def halves(*a, **k):
        k["pairing"] = "halves"
        return real(*a, **k)

    monkeypatch.setattr(pins.oracle, "diff_attn_v2", halves)
    with pytest.raises(AssertionError):
        pins.test_v2_against_sdpa(True)


def test_decode_pins_catch_an_ignored_length(monkeypatch):
    real = om.diff_attn_v1_decode

    def all_keys(q1, q2, k1, k2, v, lam, lam_init, gamma=None, eps=om.DEFAULT_EPS, lens=None):
        return real(q1, q2, k1, k2, v, lam, lam_init, gamma, eps, None)  # attends past the sequence's length

    monkeypatch.setattr(pins.oracle, "diff_attn_v1_decode", all_keys)
    with pytest.raises(AssertionError):
        pins.test_decode_matches_brute_force_with_lengths()


def test_decode_pins_catch_a_swapped_map(monkeypatch):
    real = om.diff_attn_v1_decode

    def swapped(q1, q2, k1, k2, v, lam, lam_init, gamma=None, eps=om.DEFAULT_EPS, lens=None):
        return real(q2, q1, k1, k2, v, lam, lam_init, gamma, eps, lens)  # q1 against K2 and q2 against K1

    monkeypatch.setattr(pins.oracle, "diff_attn_v1_decode", swapped)
    with pytest.raises(AssertionError):
        pins.test_decode_is_the_last_row_of_causal_attention()


def test_v2_decode_pin_catches_swapped_pair(monkeypatch):
    real = om.diff_attn_v2_decode

    def swapped(q, k, v, lam_logits, lens=None, scale=None):
        q = om._f64(q).copy()
        q[:, 0::2], q[:, 1::2] = q[:, 1::2].copy(), q[:, 0::2].copy()  # odd head first
        return real(q, k, v, lam_logits, lens, scale)

    monkeypatch.setattr(pins.oracle, "diff_attn_v2_decode", swapped)
    with pytest.raises(AssertionError):
        pins.test_v2_decode_is_the_last_row_of_causal_v2()


def _e4m3_bias8(codes):
    c = np.asarray(codes).astype(np.int64)
    e, m = (c >> 3) & 0xF, (c & 7) / 8.0
    mag = np.where(e == 0, m * 2.0 ** -7, (1 + m) * np.exp2(e - 8.0))  # exponent bias 8 instead of 7
    return np.where(c & 0x80, -mag, mag)


def _e4m3_no_subnormals(codes):
    c = np.asarray(codes).astype(np.int64)
    e, m = (c >> 3) & 0xF, (c & 7) / 8.0
    mag = (1 + m) * np.exp2(e - 7.0)  # treats exponent 0 as normal
    mag = np.where(c & 0x7F, mag, 0.0)
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where(c & 0x80, -mag, mag)


@pytest.mark.parametrize("mutant", [_e4m3_bias8, _e4m3_no_subnormals])
def test_e4m3_pins_catch_mutants(monkeypatch, mutant):
    monkeypatch.setattr(pins.oracle, "e4m3_decode", mutant)
    with pytest.raises(AssertionError):
        pins.test_e4m3_decode_closed_forms()
    with pytest.raises(AssertionError):
        pins.test_e4m3_decode_matches_torch_float8()


def _lambda_init_rate(rate):
    def f(layer_index):
        return 0.8 - 0.6 * math.exp(-rate * (layer_index - 1))  # the rate 0.3 replaced
    return f


def _lambda_init_no_offset(layer_index):
    return 0.8 - 0.6 * math.exp(-0.3 * layer_index)  # l in place of (l - 1)


@pytest.mark.parametrize("mutant", [_lambda_init_rate(0.2), _lambda_init_rate(0.5), _lambda_init_no_offset],
                         ids=["rate0.2", "rate0.5", "no_offset"])
def test_lambda_init_pin_catches_mutants(monkeypatch, mutant):
    pins.test_lambda_init_closed_forms()  # passes on the real oracle
    monkeypatch.setattr(pins.oracle, "lambda_init", mutant)
    with pytest.raises(AssertionError):
        pins.test_lambda_init_closed_forms()
