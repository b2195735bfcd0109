"""Loads tests/golden/hand_cases.json into call-ready numpy inputs (shared by
the oracle pins and the CUDA parity tests; it computes nothing of the method)."""
import json
import os

import numpy as np

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_cases.json")


def load():
    with open(PATH) as f:
        return json.load(f)


def sample_case(c):
    p = np.asarray(c["p"], np.float64)
    target = np.log(p).astype(np.float32)[None]            # softmax(log p) = p at T = 1
    draft = np.asarray(c["q"], np.float32)[None]
    tokens = np.asarray(c["tokens"], np.int32)[None]
    uni = np.asarray(c["u"], np.float32)[None]
    return target, draft, tokens, uni


def greedy_case(c):
    return (np.asarray(c["logits"], np.float32)[None], np.asarray(c["tokens"], np.int32)[None])


def tree_case(c, V=5):
    am = c["argmax"]
    rows = np.zeros((len(am), V), np.float32)
    for i, a in enumerate(am):
        rows[i, a] = 1.0
    return (rows[None], np.asarray(c["parents"], np.int32),
            np.asarray(c["tokens"], np.int32)[None], int(c["max_depth"]))
