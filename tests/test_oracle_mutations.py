"""Plant plausible mistakes in a copy of the oracle and show that the pins
catch every one of them (CPU only).

Each mutation is a textual edit of oracle/attention.py applied to a fresh,
private copy of the module; the real oracle is never touched.
"""

import inspect
import types

import pytest

import oracle.attention as attention
from oracle_pins import ALL_CHECKS

MUTATIONS = {
    "scores_operands_swapped": ("s = scale * (qh[rows] @ kh.T)", "s = scale * (kh[rows] @ qh.T)"),
    "causal_mask_off_by_one": ("return cols[None, :] <= rows[:, None]", "return cols[None, :] < rows[:, None]"),
    "lse_in_log2": ("lse = np.where(l > 0, m_safe + np.log(l), NEG_INF)",
                    "lse = np.where(l > 0, m_safe + np.log2(l), NEG_INF)"),
    "no_max_subtraction": ("e = np.exp(s - m_safe[:, None])", "e = np.exp(s)"),
    "causal_prefix_drops_diagonal": ("n_k = min(n_k, int(rows.max()) + 1)", "n_k = min(n_k, int(rows.max()))"),
    "dq_missing_scale": ("dq[h] = float(scale) * (ds @ kh[h])", "dq[h] = ds @ kh[h]"),
    "dk_not_transposed": ("dk[h] = float(scale) * (ds.T @ qh[h])", "dk[h] = float(scale) * (ds @ qh[h])"),
    "ds_sign_flipped": ("ds = p * (dp - d_row[:, None])", "ds = p * (dp + d_row[:, None])"),
    "dv_not_transposed": ("dv[h] = p.T @ doh[h]", "dv[h] = p @ doh[h]"),
    "d_rowsum_wrong_axis": ("d_row = (dp * p).sum(axis=1)", "d_row = (dp * p).sum(axis=0)"),
    "dp_uses_v_untransposed": ("dp = doh[rows] @ vh.T", "dp = doh[rows] @ vh[::-1].T"),
    "online_drops_correction": ("l = l * alpha + float(np.exp(b - m_new).sum())",
                                "l = l + float(np.exp(b - m_new).sum())"),
    "online_correction_inverted": ("alpha = math.exp(m - m_new) if m != -math.inf else 0.0",
                                   "alpha = math.exp(m_new - m) if m != -math.inf else 0.0"),
    "three_pass_missing_divide": ("y = np.array([math.exp(float(xi) - m) / l for xi in x])",
                                  "y = np.array([math.exp(float(xi) - m) for xi in x])"),
    "q_outer_drops_o_correction": ("o = alpha[:, None] * o + p @ vh[h][cols]", "o = o + p @ vh[h][cols]"),
    "kv_outer_drops_alpha": ("c_old = np.where(live, alpha * l_i / l_new, 0.0)",
                             "c_old = np.where(live, l_i / l_new, 0.0)"),
    "q_outer_moved_rows_not_rescaled": ("alpha[moved_live] = np.exp(m[moved_live] - m_new[moved_live])",
                                        "alpha[moved_live] = 1.0"),
}


def _mutant(old, new):
    src = inspect.getsource(attention)
    assert src.count(old) == 1, f"mutation anchor not found exactly once: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "<oracle_mutant>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    mod = _mutant(*MUTATIONS[name])
    failed = []
    for check in ALL_CHECKS:
        try:
            with __import__("numpy").errstate(all="ignore"):
                check(mod)
        except Exception:  # an assertion or a crash both count as caught
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
