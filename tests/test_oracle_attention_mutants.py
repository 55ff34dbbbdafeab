"""Plant plausible mistakes in copies of the rotary-attention oracle and check
that the pins catch each one.

Every mutant is a textual edit of ``oracle/attention.py``, executed as a
module of its own (the real oracle is never modified), and every pin of
attention_pins.py runs against it: at least one must fail (an exception of
any kind counts as caught).
"""
import importlib.util
import os

import pytest

import oracle  # noqa: F401  (the mutants import from this package)

import attention_pins as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "oracle", "attention.py")

# (name, [(old, new), ...]) -- each a mistake a hand-written attention could contain
MUTANTS = [
    ("scale_over_d", [("1.0 / np.sqrt(D) if scale is None", "1.0 / D if scale is None")]),
    ("causal_strict", [("np.arange(Sk)[None, :] <= (", "np.arange(Sk)[None, :] < (")]),
    ("causal_top_left", [("(np.arange(Sq)[:, None] + (Sk - Sq))", "(np.arange(Sq)[:, None] + 0)")]),
    ("gqa_modulo", [("kh = h // group", "kh = h % Hk")]),
    ("keys_not_rotated", [("k = rotate_rounded(k_bits, dtype, pos_k,",
                           "k = rotate_rounded(k_bits, dtype, np.full(Sk, -1, dtype=np.int32),")]),
    ("queries_not_rotated", [("q = rotate_rounded(q_bits, dtype, pos_q,",
                              "q = rotate_rounded(q_bits, dtype, np.full(Sq, -1, dtype=np.int32),")]),
    ("query_positions_for_keys", [("k = rotate_rounded(k_bits, dtype, pos_k,",
                                   "k = rotate_rounded(k_bits, dtype, pos_q,")]),
    ("not_normalised", [("(p @ v[b, kh]) / np.where(l > 0, l, 1.0)", "(p @ v[b, kh])")]),
    ("values_of_first_head", [("(p @ v[b, kh])", "(p @ v[b, 0])")]),
    ("mask_not_applied", [("            s = np.where(visible, s, -np.inf)\n", ""),
                          ("p = np.where(visible, np.exp(s - np.where(np.isfinite(m), m, 0.0)), 0.0)",
                           "p = np.exp(s - np.where(np.isfinite(m), m, 0.0))")]),
    ("empty_rows_not_zeroed", [("o = np.where(has[:, None], (p @ v[b, kh]) / np.where(l > 0, l, 1.0), 0.0)",
                                "o = (p @ v[b, kh]) / l")]),
    ("rotated_rows_not_rounded", [("return y64 if dtype == F64 else decode16(yb, dtype)",
                                   "return y64 if dtype == F64 else load().apply(x_bits, dtype, B, H, S, D, "
                                   "rotary_dim, layout, False, False, pos, cos32, sin32)[2]")]),
    ("scores_missing_scale", [("s = (q[b, h] @ k[b, kh].T) * scale", "s = q[b, h] @ k[b, kh].T")]),
    ("softmax_over_queries", [("m = s.max(axis=1, keepdims=True)", "m = s.max(axis=0, keepdims=True)"),
                              ("l = p.sum(axis=1, keepdims=True)", "l = p.sum(axis=0, keepdims=True)")]),
    ("bound_w_signed", [("w_abs[b, h] = (p @ av) * inv_l", "w_abs[b, h] = (p @ v[b, kh]) * inv_l")]),
    ("bound_w_unnormalised", [("w_abs[b, h] = (p @ av) * inv_l", "w_abs[b, h] = p @ av")]),
    ("bound_a_all_keys", [("a_abs[b, h] = (visible.astype(np.float64) @ av) * inv_l",
                           "a_abs[b, h] = av.sum(axis=0)[None, :] * inv_l")]),
    ("mask_ignored", [("visible = visible & (mb[None, :] if mb.ndim == 1 else mb)", "pass")]),
    ("mask_inverted", [("visible = visible & (mb[None, :] if mb.ndim == 1 else mb)",
                        "visible = visible & ~(mb[None, :] if mb.ndim == 1 else mb)")]),
    ("mask_replaces_causal", [("visible = visible & (mb[None, :] if mb.ndim == 1 else mb)",
                               "visible = (mb[None, :] if mb.ndim == 1 else mb) | (visible & False)")]),
    ("mask_of_first_batch", [("mb = attn_mask[b]", "mb = attn_mask[0]")]),
]


def _load_mutant(name, edits):
    src = open(SOURCE).read()
    for old, new in edits:
        assert src.count(old) == 1, "mutant %s: anchor not found once: %r" % (name, old)
        src = src.replace(old, new)
    spec = importlib.util.spec_from_loader("oracle._attention_mutant_" + name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    mod.__package__ = "oracle"
    exec(compile(src, "<attention mutant %s>" % name, "exec"), mod.__dict__)
    return mod


def _caught_by(mod):
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(mod)
        except Exception:  # noqa: BLE001 - any failure of a pin catches the mutant
            caught.append(pin.__name__)
    return caught


@pytest.mark.filterwarnings("ignore::RuntimeWarning")   # a mutant may divide by zero
@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_attention_mutant_is_caught(name):
    edits = dict(MUTANTS)[name]
    caught = _caught_by(_load_mutant(name, edits))
    assert caught, "no pin catches the planted mistake %r" % name
