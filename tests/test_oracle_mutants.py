"""Planted mistakes in the oracle must be caught by its pins.

Each mutant is the oracle's own source with one plausible mistake typed into it
(a dropped term, a wrong index or sign, a transposed operand, one key too far, a
merge that drops a part).  The mutant is built on the CPU as a separate module;
the test asserts that at least one pin from test_oracle_pins fails on it.
"""
import importlib.util
import os
import types

import pytest

from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "attention.py")

MUTANTS = {
    "one key too far (prefill)": ("return kv_offset + i + 1", "return kv_offset + i + 2"),
    "one key too far (verify)": ("return kv_len - rows + i + 1", "return kv_len - rows + i + 2"),
    "one key short (row limit)": ("        lim = lims[i]\n", "        lim = lims[i] - 1\n"),
    "wrong scale": ("SCALE = 1.0 / 16.0", "SCALE = 1.0 / 8.0"),
    "interleaved kv heads": ("return h // (Hq // Hkv)", "return h % Hkv"),
    "transposed operand (V for K)": ("s = (Kb[:lim] @ q_rows[i]) * SCALE", "s = (Vb[:lim] @ q_rows[i]) * SCALE"),
    "dropped normalisation": ("o = (p @ Vb[:lim]) / l", "o = (p @ Vb[:lim])"),
    "dropped max shift": ("m = np.max(s)", "m = 0.0 * np.max(s)"),
    "gate sign": ("return 1.0 / (1.0 + np.exp(-x))", "return 1.0 / (1.0 + np.exp(x))"),
    "lse without ln l": ("lse[i] = m + math.log(l)", "lse[i] = m"),
    "merge drops last part": ("live = [s for s in range(S) if lse_parts[s, n] != -np.inf]",
                              "live = [s for s in range(S) if lse_parts[s, n] != -np.inf][:-1]"),
    "merge skips NaN parts": ("live = [s for s in range(S) if lse_parts[s, n] != -np.inf]",
                              "live = [s for s in range(S) if np.isfinite(lse_parts[s, n])]"),
    "sigmoid clamps the gate": ("return 1.0 / (1.0 + np.exp(-x))",
                                "return 1.0 / (1.0 + np.exp(-np.nan_to_num(x)))"),
    "mask: bool inverted": ("                    keep = base & m\n", "                    keep = base & ~m\n"),
    "mask: bias scaled like a score": ("            s = s + bias[i, idx]", "            s = s + bias[i, idx] * SCALE"),
    "mask: chunk slices the full mask": ("                    M = _broadcast_mask(mask, (B, c, Lq, Lkv))\n",
                                         "                    M = _broadcast_mask(mask, (B, Hq, Lq, Lkv))[:, h0:h0 + c]\n"),
    "mask: chunk-local heads reversed": ("                        head_mask[h0 + k] = M[:, k]",
                                         "                        head_mask[h0 + k] = M[:, c - 1 - k]"),
    "mask: causal one key too far": ("np.arange(Lkv)[None, :] <= kv_offset + np.arange(Lq)[:, None]",
                                     "np.arange(Lkv)[None, :] <= kv_offset + 1 + np.arange(Lq)[:, None]"),
    "mask: -inf bias kept": ("                    keep = base & (a != -np.inf)", "                    keep = base"),
    "scores without NaN": ("        m = np.max(s)\n",
                           "        s = np.where(np.isnan(s), -np.inf, s)\n        m = np.max(s)\n"),
    # keys a row does not see weighted by probability 0 instead of excluded: a NaN or
    # Inf in their V rows then reaches the row (0 x Inf = NaN)
    "masked V multiplied by 0": ("o = (p @ Vb[:lim]) / l",
                                 "o = (np.concatenate([p, np.zeros(kmax - lim)]) @ Vb) / l"),
    "merge ignores weights": ("acc += ws * O_parts[s, n]", "acc += O_parts[s, n]"),
    "plan drops remainder": ("    if gqa % c:\n        plan.append(gqa % c)\n", ""),
    "tree: new rows start one key late": ("    base = kv_len - rows\n    return list(range(base))",
                                          "    base = kv_len - rows + 1\n    return list(range(base))"),
    "tree: mask bits shifted": ("if (int(mask) >> k) & 1]", "if (int(mask) >> (k + 1)) & 1]"),
    "tree: self bit ignored": ("for k in range(rows) if (int(mask) >> k) & 1]",
                               "for k in range(rows) if (int(mask) >> k) & 1 and k != i]"),
    "append one row late": ("        L = int(kv_lens[b])\n        r = cu[b + 1] - cu[b]\n        Kc[b, :, L:L + r]",
                            "        L = int(kv_lens[b]) + 1\n        r = cu[b + 1] - cu[b]\n        Kc[b, :, L:L + r]"),
    "keep from the wrong base": ("        base = int(kv_lens[b]) - r\n        src", "        base = int(kv_lens[b]) - r + 1\n        src"),
    "plan chunk one head too wide": ("c = min(gqa, limit // rows)", "c = min(gqa, limit // rows + 1)"),
    "plan ignores the row bound": ("rows > limit or ", ""),
}


def _build(src, name):
    mod = types.ModuleType(name)
    mod.__file__ = SRC
    exec(compile(src, f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def test_unmutated_source_passes():
    with open(SRC) as f:
        mod = _build(f.read(), "oracle_copy")
    bad = [c.__name__ for c in pins.CHECKS if c(mod)]
    assert not bad, bad


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    with open(SRC) as f:
        src = f.read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    mod = _build(src.replace(old, new), name)
    failed = []
    for c in pins.CHECKS:
        try:
            if c(mod):
                failed.append(c.__name__)
        except Exception as e:  # a crash also counts as caught
            failed.append(f"{c.__name__} raised {type(e).__name__}")
    assert failed, f"no pin caught mutant {name!r}"
