"""The oracle and the workloads against the facts the pages print
(tests/golden/pages_examples.json, each entry cites its page and section)."""
import json
import os

import numpy as np

import oracle as O
import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")))


def test_pair_layouts_match_pages():
    o = O.load()
    g = GOLDEN["pair_layouts"]
    D = g["D"]
    h = D // 2
    # a quarter turn on every pair: y[a] = -x[b], y[b] = x[a] for pair (a, b)
    cos = np.zeros((1, h))
    sin = np.ones((1, h))
    for layout, key in ((O.INTERLEAVED, "interleaved"), (O.SPLIT_HALF, "split_half")):
        pairs = []
        for a in range(D):
            x = np.zeros((1, 1, 1, D))
            x[..., a] = 1.0
            _, _, y = o.apply(x, O.F64, 1, 1, 1, D, D, layout, False, False, None, cos, sin,
                              want_bits=False)
            b = int(np.flatnonzero(y[0, 0, 0])[0])
            if y[0, 0, 0, b] == 1.0:          # x[a] moved to b with + sign: a is first of pair (a, b)
                pairs.append([a, b])
        assert sorted(pairs) == g[key]


def test_pair_rotation_quarter_and_half_turn():
    o = O.load()
    for key in ("quarter_turn", "half_turn"):
        t = GOLDEN["pair_rotation"][key]
        x = np.array(t["x"]).reshape(1, 1, 1, 2)
        _, _, y = o.apply(x, O.F64, 1, 1, 1, 2, 2, O.SPLIT_HALF, False, False, None,
                          np.array([[t["cos"]]]), np.array([[t["sin"]]]), want_bits=False)
        assert y.reshape(-1).tolist() == t["y"]


def test_prefix_shift_ids():
    g = GOLDEN["prefix_shift_example"]
    assert (np.arange(g["seq_len"]) + g["prefix_len"]).tolist() == g["rope_ids"]


def test_tiny_workload_is_the_pages_usage_example():
    g = GOLDEN["rotate_queries_or_keys_example"]
    w = W.BY_NAME["tiny_f32_split_half"]
    assert list(w.q_shape) == g["q_shape"] and list(w.k_shape) == g["k_shape"]
    assert w.rotary_dim == g["dim"] and w.theta == GOLDEN["defaults"]["theta"]


def test_masked_workload_encodes_the_pages_pos_mask_example():
    # tokens start..start+count-1 take frequency rows 0..count-1; the leading
    # tokens are not rotated (position -1)
    g = GOLDEN["flash_attn_with_rotary_example"]
    w = W.BY_NAME["partial_rd32_masked_bf16"]
    assert w.S == g["q_shape"][2] and w.D == g["q_shape"][3] and w.rotary_dim == g["rotary_dim"]
    want = np.full(w.S, -1, dtype=np.int32)
    idx = g["rotated_token_indices"]
    tokens = np.arange(idx["start"], idx["start"] + idx["count"] * idx["step"], idx["step"])
    want[tokens] = np.arange(g["freq_positions"])
    assert np.array_equal(W.positions(w), want)
    assert w.interpolate_factor == GOLDEN["defaults"]["interpolate_factor"]


def test_table_is_half_width():
    o = O.load()
    c, s = o.tables(GOLDEN["defaults"]["theta"], 64, 16, 1.0)
    assert c.shape == (16, 32) and s.shape == (16, 32)     # [seq_len, D/2]
