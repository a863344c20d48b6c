"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that at least one pin fails for each: the pins are strong enough to notice a
dropped term, a wrong sign or index, or a transposed operand."""
import os
import sys
import types

import pytest

sys.path.insert(0, os.path.dirname(__file__))
from oracle_pins import ALL_PINS  # noqa: E402

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "attention.py")

MUTATIONS = {
    "gqa_index": ("j = h // G                                              # GQA", "j = h % Hkv                                              # GQA"),
    "causal_strict": ("m &= k_pos <= q_pos", "m &= k_pos < q_pos"),
    "dropped_scale": ("S = sc * (_f64(q[rb, h, :]) @ Kj.T)", "S = (_f64(q[rb, h, :]) @ Kj.T)"),
    "scale_1_over_d": ("1.0 / math.sqrt(d) if scale is None", "1.0 / d if scale is None"),
    "transposed_pv": ("O[b0:b0 + len(rb), hi, :] = P @ Vj", "O[b0:b0 + len(rb), hi, :] = P @ Kj"),
    "merge_weight_index": ("cb = np.where(empty, 0.0, np.exp(lse_b - ls))", "cb = np.where(empty, 0.0, np.exp(lse_a - ls))"),
    "merge_dropped_log": ("lse = np.where(empty, NEG_INF, ms + np.log(wa + wb))", "lse = np.where(empty, NEG_INF, ms + (wa + wb))"),
    "zigzag_chunk": ("(2 * R - 1 - r) * c + np.arange(c)", "(2 * R - 2 - r) * c + np.arange(c)"),
    "reshard_transposed": ("y[u, s * n:(s + 1) * n] = x[s, :, u * Hl:(u + 1) * Hl]", "y[u, s * n:(s + 1) * n] = x[u, :, s * Hl:(s + 1) * Hl]"),
    "doc_boundary": ('idx = np.searchsorted(offsets, pos, side="right") - 1', 'idx = np.searchsorted(offsets, pos, side="left") - 1'),
    "bwd_sign": ("dS = P * (dP - D[:, None])\n        dq[:, h, :] = sc * (dS @ k[:, j, :])",
                 "dS = P * (dP + D[:, None])\n        dq[:, h, :] = sc * (dS @ k[:, j, :])"),
    "bwd_rows_sign": ("dS = P * (dP - D[:, None])\n        return", "dS = P * (dP + D[:, None])\n        return"),
    "bwd_rows_dv_operand": ("dv[:, ji, :] += P.T @ dOr", "dv[:, ji, :] += P.T @ Qr"),
    "bwd_gqa_overwrite": ("dk[:, j, :] += sc * (dS.T @ q[:, h, :])", "dk[:, j, :] = sc * (dS.T @ q[:, h, :])"),
    "bwd_dropped_scale": ("dq[:, h, :] = sc * (dS @ k[:, j, :])", "dq[:, h, :] = (dS @ k[:, j, :])"),
    "balanced_ascending": ("key=lambda j: (-int(work[j]), j)", "key=lambda j: (int(work[j]), j)"),
    "balanced_most_loaded": ("load[r] < load[best]", "load[r] > load[best]"),
    "balanced_ignores_docs": ("per_query = pos - doc_start_of(pos, offsets) + 1", "per_query = pos + 1"),
    "bwd_partial_sign": ("dS = P * (dP - D[:, None])\n        dq[:, h, :] = sc * (dS @ kj)",
                         "dS = P * (dP + D[:, None])\n        dq[:, h, :] = sc * (dS @ kj)"),
    "bwd_partial_lse_unused": ("np.exp(sc * (qh @ kj.T) - lse[h][:, None])", "np.exp(sc * (qh @ kj.T))"),
    "bwd_partial_dk_operand": ("dk[:, j, :] += sc * (dS.T @ qh)", "dk[:, j, :] += sc * (dS.T @ doh)"),
    "lse_reshard_back": ("out[s, u * Hl:(u + 1) * Hl, :] = lse[u, :, s * n:(s + 1) * n]", "out[s, u * Hl:(u + 1) * Hl, :] = lse[s, :, u * n:(u + 1) * n]"),
}


def _mutant(old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name):
    mod = _mutant(*MUTATIONS[name])
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception:  # an AssertionError, or a crash the mistake causes
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutation {name}"
