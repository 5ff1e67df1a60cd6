"""Planted mistakes in the oracle are caught by its pins (CPU only).

Each case edits one expression of the oracle's source text: a dropped term,
a flipped sign, a transposed or wrong operand, a misplaced scale, a wrong
mask, a missing normalisation, a wrong rounding rule.  The edited copy is
loaded as a module of its own, the ``oracle`` package is pointed at it, and
every pin in test_oracle_pins.py runs against it with all of its
parameters.  Each edit must make at least one pin fail on a value check (an
AssertionError, not only a crash); the unedited copy must pass every pin, so
the harness itself is sound.  The edits live only in memory: the oracle's
files are never touched.
"""
import importlib.util
import inspect
import itertools
import os
import types
import warnings

import numpy as np
import pytest

import oracle
import oracle.attention as oracle_attention

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = open(os.path.join(os.path.dirname(HERE), "oracle", "attention.py")).read()


def _load_pins():
    spec = importlib.util.spec_from_file_location("pins_under_mutation", os.path.join(HERE, "test_oracle_pins.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


PINS = _load_pins()


def _pin_cases():
    """(name, function, kwargs) for every parameter combination pytest runs."""
    out = []
    for name, fn in inspect.getmembers(PINS, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            argnames, values = mark.args[0], mark.args[1]
            argnames = [a.strip() for a in argnames.split(",")]
            if len(argnames) == 1:
                values = [(v,) for v in values]
            grids.append([dict(zip(argnames, v)) for v in values])
        params = set(inspect.signature(fn).parameters)
        for combo in itertools.product(*grids):
            kw = {}
            for c in combo:
                kw.update(c)
            assert set(kw) == params, f"{name}: unsupported fixture or parameter"
            out.append((name, fn, kw))
    return out


CASES = _pin_cases()


def _run_pins(source, monkeypatch):
    """Point the oracle package at `source` and run every pin case.
    Returns (value-check failures, other errors)."""
    mod = types.ModuleType("oracle_mutant")
    exec(compile(source, "oracle_mutant", "exec"), mod.__dict__)
    for name in oracle_attention.__all__:
        monkeypatch.setattr(oracle, name, getattr(mod, name))
    value_fail, errors = [], []
    for name, fn, kw in CASES:
        try:
            with np.errstate(all="ignore"), warnings.catch_warnings():
                warnings.simplefilter("ignore")
                fn(**kw)
        except AssertionError:
            value_fail.append(f"{name}{kw}")
        except Exception as e:              # e.g. shapes that no longer fit
            errors.append(f"{name}{kw}: {type(e).__name__}")
    return value_fail, errors


# (label, original text, occurrence to edit, replacement)
MUTANTS = [
    ("standard dS: dropped -P*(P.dP) term",
     "dS = P * dP - P * np.sum(P * dP, axis=1, keepdims=True)", 0, "dS = P * dP"),
    ("standard dS: sign of the row term",
     "dS = P * dP - P * np.sum(P * dP, axis=1, keepdims=True)", 0,
     "dS = P * dP + P * np.sum(P * dP, axis=1, keepdims=True)"),
    ("standard dK: dS not transposed", "dk[b, h] = (dS.T @ q[b, h]) * scale", 0,
     "dk[b, h] = (dS @ q[b, h]) * scale"),
    ("standard dV: P not transposed", "dv[b, h] = P.T @ do[b, h]", 0, "dv[b, h] = P @ do[b, h]"),
    ("standard dQ: scale dropped", "dq[b, h] = (dS @ k[b, h]) * scale", 0, "dq[b, h] = dS @ k[b, h]"),
    ("standard dP: K in place of V", "dP = do[b, h] @ v[b, h].T", 0, "dP = do[b, h] @ k[b, h].T"),
    ("mask direction reversed", "return j <= i", 0, "return j >= i"),
    ("mask drops the diagonal", "return j <= i", 0, "return j < i"),
    ("scores: scale dropped", "return (_f64(q_bh) @ _f64(k_bh).T) * float(scale)", 0,
     "return _f64(q_bh) @ _f64(k_bh).T"),
    ("softmax: not normalised", "P = e / l", 0, "P = e"),
    ("logsumexp: row maximum dropped", "L = m[:, 0] + np.log(l[:, 0])", 0, "L = np.log(l[:, 0])"),
    ("forward: P transposed", "O[b, h] = P @ v[b, h]", 0, "O[b, h] = P.T @ v[b, h]"),
    ("sampled rows: mask drops the diagonal",
     "keep = (np.arange(k_bh.shape[0])[None, :] <= rows[:, None]) if causal else None", 0,
     "keep = (np.arange(k_bh.shape[0])[None, :] < rows[:, None]) if causal else None"),
    ("recompute dS: sign of D", "dS = P * (dP - D[b, h][:, None])", 0, "dS = P * (dP + D[b, h][:, None])"),
    ("recompute P: L broadcast along keys", "P = np.exp(Sm - L[b, h][:, None])", 0,
     "P = np.exp(Sm - L[b, h][None, :])"),
    ("recompute P: mask not applied", "P = np.where(keep, P, 0.0)", 0, "P = P"),
    ("recompute dK: scale dropped", "dk[b, h] = (dS.T @ q[b, h]) * scale", 1, "dk[b, h] = dS.T @ q[b, h]"),
    ("D: dO * dO in place of O * dO", "return np.sum(_f64(o) * _f64(do), axis=-1)", 0,
     "return np.sum(_f64(do) * _f64(do), axis=-1)"),
    ("partial: output not normalised", "o[ok] = (A @ v_bh[key_idx]) / Bsum[ok][:, None]", 0,
     "o[ok] = A @ v_bh[key_idx]"),
    ("merge: left weight on the right output", "o = (wl[:, None] * o_l + wr[:, None] * o_r) / Bm[:, None]", 0,
     "o = (wl[:, None] * o_l + wl[:, None] * o_r) / Bm[:, None]"),
    ("merge: logsumexp without the maximum", "return o, m, Bm, m + np.log(Bm)", 0, "return o, m, Bm, np.log(Bm)"),
    ("query rows: sign of D", "dS_rows = P_rows * (dP_rows - D_rows[:, None])", 0,
     "dS_rows = P_rows * (dP_rows + D_rows[:, None])"),
    ("query rows: scale dropped from dQ", "return (dS_rows @ k_bh) * scale", 0, "return dS_rows @ k_bh"),
    ("query rows: mask drops the diagonal",
     "P_rows = np.where(np.arange(k_bh.shape[0])[None, :] <= rows[:, None], P_rows, 0.0)", 0,
     "P_rows = np.where(np.arange(k_bh.shape[0])[None, :] < rows[:, None], P_rows, 0.0)"),
    ("query rows: D from dO alone", "D_rows = np.sum(o_rows * do_rows, axis=1)", 0,
     "D_rows = np.sum(do_rows * do_rows, axis=1)"),
    ("key rows: mask reversed", "P_cols = np.where(keys[None, :] <= np.arange(n_q)[:, None], P_cols, 0.0)", 0,
     "P_cols = np.where(keys[None, :] >= np.arange(n_q)[:, None], P_cols, 0.0)"),
    ("key rows: L of the key index", "P_cols = np.exp(S_cols - L_bh[:, None])", 0,
     "P_cols = np.exp(S_cols - L_bh[keys][None, :])"),
    ("key rows: dV from dS", "return (dS_cols.T @ q_bh) * scale, P_cols.T @ do_bh", 0,
     "return (dS_cols.T @ q_bh) * scale, dS_cols.T @ do_bh"),
    ("key rows: dK from dO in place of Q", "return (dS_cols.T @ q_bh) * scale, P_cols.T @ do_bh", 0,
     "return (dS_cols.T @ do_bh) * scale, P_cols.T @ do_bh"),
    ("key rows: dP with K", "dP_cols = do_bh @ v_bh[keys].T", 0, "dP_cols = do_bh @ k_bh[keys].T"),
    ("bf16 rounding: ties not to even", "lsb = (u >> 16) & 1", 0, "lsb = 0 * u"),
    ("bf16 rounding: truncation", "r = ((u + 0x7FFF + lsb) >> 16) << 16", 0, "r = (u >> 16) << 16"),
]


def _edit(label, old, occurrence, new):
    parts = SOURCE.split(old)
    assert len(parts) > occurrence + 1, f"{label}: text not found in the oracle"
    return old.join(parts[: occurrence + 1]) + new + old.join(parts[occurrence + 1:])


def test_unedited_oracle_passes_every_pin(monkeypatch):
    value_fail, errors = _run_pins(SOURCE, monkeypatch)
    assert not value_fail and not errors, (value_fail, errors)
    assert len(CASES) >= 40


@pytest.mark.parametrize("label,old,occurrence,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(label, old, occurrence, new, monkeypatch):
    value_fail, errors = _run_pins(_edit(label, old, occurrence, new), monkeypatch)
    assert value_fail, f"no pin caught '{label}' (errors only: {errors})"
