"""Mutation tests: plant one plausible mistake in a copy of the oracle (on the
CPU) and show that the pins of test_oracle_pins.py catch it.

Each mutant is the oracle's own source with one textual edit, executed into a
fresh module namespace; the real oracle is untouched.
"""

import os
import types

import pytest

import test_oracle_pins as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _mutant(relpath, old, new):
    path = os.path.join(ROOT, relpath)
    with open(path) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("mutant_" + os.path.basename(relpath)[:-3])
    mod.__dict__["__name__"] = mod.__name__
    exec(compile(src.replace(old, new), path + "<mutant>", "exec"), mod.__dict__)
    return mod


ATT = "oracle/attention.py"
ONL = "oracle/online.py"

MUTANTS = [
    # (id, file, old, new, checks that must fail)
    ("ds_sign", ATT, "ds = p * (dp - dvec)", "ds = p * (dp + dvec)",
     ["check_worked_example_forward", "check_finite_differences", "check_brute_force_scalar"]),
    ("dk_no_scale", ATT, "dk += scale * (ds.T @ q[rr])", "dk += (ds.T @ q[rr])",
     ["check_finite_differences", "check_brute_force_scalar"]),
    ("dq_transposed_operand", ATT, "dq[rr] = scale * (ds @ k)", "dq[rr] = scale * (ds.T[: len(rr), : k.shape[0]] @ k)",
     ["check_finite_differences"]),
    ("dv_uses_ds", ATT, "dv += p.T @ do[rr]", "dv += (p + ds).T @ do[rr]",
     ["check_finite_differences", "check_brute_force_scalar"]),
    ("mask_transposed", ATT, "keys[None, :] <= np.asarray(rows)[:, None]",
     "keys[None, :] >= np.asarray(rows)[:, None]",
     ["check_brute_force_scalar", "check_invariants", "check_closed_forms"]),
    ("lse_drops_max", ATT, "m_safe[:, 0] + np.log(", "0.0 * m_safe[:, 0] + np.log(",
     ["check_worked_example_forward", "check_invariants"]),
    ("gqa_modulo_map", ATT, "_head_views(k, b, seg, h // group)", "_head_views(k, b, seg, h % h_kv)",
     ["check_gqa_is_repeated_heads"]),
    ("gqa_strided_groups", ATT, "for h in range(g * group, (g + 1) * group):", "for h in range(g, h_q, h_kv):",
     ["check_gqa_is_repeated_heads"]),
    ("packed_sequences_overlap", ATT, "return [(s, (int(cu[s]), int(cu[s + 1]))) for s in range(len(cu) - 1)]",
     "return [(s, (int(cu[s]), int(cu[s + 1]) + (1 if s < len(cu) - 2 else 0))) for s in range(len(cu) - 1)]",
     ["check_packed_is_per_sequence"]),
    ("o_from_keys", ATT, "o[r0:r0 + len(rr)] = p @ v", "o[r0:r0 + len(rr)] = p @ k[:, : v.shape[1]]",
     ["check_asymmetric_head_dims", "check_brute_force_scalar"]),
    ("merge_rescales_denominator_only", ONL, "u = c * u + e @ vb", "u = u + e @ vb",
     ["check_online_merge", "check_merges_match_definition"]),
    ("merge_rescales_numerator_only", ONL, "l = c * l + float(np.sum(e))", "l = l + float(np.sum(e))",
     ["check_online_merge", "check_merges_match_definition"]),
    ("lazy_forgets_u", ONL, "u = u * c\n", "u = u\n",
     ["check_merges_match_definition"]),
]


def _run_check(name, mod_att=None, mod_onl=None):
    fn = getattr(P, name)
    if name in ("check_online_merge",):
        return fn(mod_onl)
    if name == "check_merges_match_definition":
        return fn(mod_att or P.A, mod_onl or P.OL)
    return fn(mod_att)


@pytest.mark.parametrize("mid,path,old,new,checks", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(mid, path, old, new, checks):
    mod = _mutant(path, old, new)
    for name in checks:
        with pytest.raises(AssertionError):
            if path == ATT:
                _run_check(name, mod_att=mod)
            else:
                _run_check(name, mod_onl=mod)


def test_unmutated_oracle_passes_every_check():
    for name in ("check_worked_example_forward", "check_finite_differences", "check_brute_force_scalar",
                 "check_invariants", "check_closed_forms", "check_gqa_is_repeated_heads",
                 "check_packed_is_per_sequence", "check_asymmetric_head_dims"):
        getattr(P, name)(P.A)
    P.check_online_merge(P.OL)
    P.check_merges_match_definition(P.A, P.OL)
