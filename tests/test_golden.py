"""Worked examples in tests/golden/worked_examples.json, checked against the oracle."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests import refmath as R

HERE = os.path.dirname(os.path.abspath(__file__))
DATA = json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))


def _closed_form(expr):
    env = {"e": math.e, "sin": math.sin, "cos": math.cos, "exp": math.exp,
           "sig": lambda x: 1.0 / (1.0 + math.exp(-x))}
    return np.array(eval(expr, {"__builtins__": {}}, env), dtype=np.float64)


@pytest.mark.parametrize("case", DATA["cases"], ids=lambda c: c["name"])
def test_worked_example(case):
    d, hq, hk, P = case["head_dim"], case["n_qh"], case["n_kvh"], case["page_size"]
    L = len(case["cached_k"])
    bits = lambda a: R.f32_to_bf16_bits(np.asarray(a, np.float32))
    q = bits(case["q"]).reshape(1, hq, d)
    k_new = bits(case["k_new"]).reshape(1, hk, d)
    v_new = bits(case["v_new"]).reshape(1, hk, d)
    # one physical page (index 1 of 2, to exercise the table), cached rows first
    kp = np.zeros((2, hk, P, d), np.uint16)
    vp = np.zeros((2, hk, P, d), np.uint16)
    for t in range(L):
        kp[1, :, t] = bits(case["cached_k"][t])
        vp[1, :, t] = bits(case["cached_v"][t])
    bt = np.array([[1]], np.int32)
    lens = np.array([L], np.int32)
    pos = np.array([case["position"]], np.int32)
    out, st = oracle.decode(q, k_new, v_new, kp, vp, bt, lens, pos,
                            case["rope_theta"], case["scale"])
    assert st == 0
    want = _closed_form(case["expected"])
    assert np.max(np.abs(out[0] - want)) < 1e-12


def test_int8_worked_rows():
    for row in DATA["int8_rows"]:
        codes, sc = oracle.quant_int8(np.asarray(row["x"], np.float32))
        assert list(codes) == row["codes"]
        assert sc == np.float32(np.float32(1.0) / np.float32(127.0))
