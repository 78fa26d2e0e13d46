"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one (CPU only; the real oracle is never modified)."""

import os
import types

import pytest

from oracle_pins import ALL_PINS

SRC = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "oracle", "attention.py")).read()

MUTANTS = {
    "transposed_scores": ("s = (q @ k.T) * scale",
                          "s = ((q @ k.T).T if q.shape[0] == k.shape[0] else q @ k.T) * scale"),
    "scale_divides": ("s = (q @ k.T) * scale", "s = (q @ k.T) / scale if scale else (q @ k.T)"),
    "mask_includes_diagonal": ("cols > np.asarray(rows)[:, None]", "cols >= np.asarray(rows)[:, None]"),
    "mask_hides_past": ("cols > np.asarray(rows)[:, None]", "cols < np.asarray(rows)[:, None]"),
    "no_max_subtraction": ("e = np.exp(s - m[:, None])", "e = np.exp(s) * np.exp(0 * m[:, None])"),
    "lse_drops_max": ("lse = m + np.log(l)", "lse = np.log(l)"),
    "unnormalised_p": ("p = e / l[:, None]", "p = e"),
    "dv_untransposed": ("dv[idx] = p.T @ g", "dv[idx] = p @ g"),
    "ds_sign": ("ds = p * (dp - d_row[:, None])", "ds = p * (dp + d_row[:, None])"),
    "ds_drops_d": ("ds = p * (dp - d_row[:, None])", "ds = p * dp"),
    "dq_no_scale": ("dq[idx] = scale * (ds @ k[idx])", "dq[idx] = ds @ k[idx]"),
    "dk_wrong_operand": ("dk[idx] = scale * (ds.T @ q[idx])", "dk[idx] = scale * (ds.T @ k[idx])"),
    "dp_uses_k": ("dp = g @ v[idx].T", "dp = g @ k[idx].T"),
    "decode_no_norm": ("o[idx] = (e @ vc[idx]) / l", "o[idx] = e @ vc[idx]"),
    "decode_lse_no_max": ("lse[idx] = m + math.log(l)", "lse[idx] = math.log(l)"),
    "online_no_rescale": ("l = l * math.exp(m - m_new) + float(np.exp(c - m_new).sum())",
                          "l = l + float(np.exp(c - m_new).sum())"),
    "gqa_head_modulo": ("return h // (hq // hkv)", "return h % hkv"),
    "gqa_dk_overwritten": ("dk[b, g] += scale * (dsg.T @ q[b, h])",
                           "dk[b, g] = scale * (dsg.T @ q[b, h])"),
    "gqa_dv_overwritten": ("dv[b, g] += p.T @ gr", "dv[b, g] = p.T @ gr"),
    "gqa_dk_wrong_operand": ("dk[b, g] += scale * (dsg.T @ q[b, h])",
                             "dk[b, g] += scale * (dsg.T @ k[b, g])"),
    "gqa_decode_head": ("s = (kc[b, g] @ q[b, h]) * scale", "s = (kc[b, h % hkv] @ q[b, h]) * scale"),
    "window_one_too_wide": ("np.asarray(rows)[:, None] - window + 1", "np.asarray(rows)[:, None] - window"),
    "window_one_too_narrow": ("np.asarray(rows)[:, None] - window + 1",
                              "np.asarray(rows)[:, None] - window + 2"),
    "alibi_sign": ("s = s - slope * dist", "s = s + slope * dist"),
    "alibi_scaled_twice": ("s = s - slope * dist", "s = s - slope * scale * dist"),
    "alibi_signed_distance": ("dist = np.abs(np.asarray(rows)[:, None] - np.arange(k.shape[0])[None, :])",
                              "dist = np.asarray(rows)[:, None] - np.arange(k.shape[0])[None, :]"),
    "alibi_next_head": ("return None if alibi_slopes is None else float(alibi_slopes[h])",
                        "return None if alibi_slopes is None else float(alibi_slopes[(h + 1) % len(alibi_slopes)])"),
    "alibi_decode_position": ("(s.shape[0] - 1 - np.arange(s.shape[0]))", "(s.shape[0] - np.arange(s.shape[0]))"),
    "tile_merge_weight_unnormalised": ("w = math.exp(lse_t - total)", "w = math.exp(lse_t - top)"),
    "tile_partial_unnormalised": ("partials.append(((e_t @ vt) / l_t, m_t + math.log(l_t)))",
                                  "partials.append((e_t @ vt, m_t + math.log(l_t)))"),
}


def _load(src):
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


# A mutant whose mask hides a whole row computes -inf - -inf; the NaN it
# leaves is one of the ways a pin catches it.
@pytest.mark.filterwarnings("ignore:invalid value encountered:RuntimeWarning")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = _load(SRC.replace(old, new))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
