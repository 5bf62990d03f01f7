"""Planted mistakes: a mutated copy of the oracle must fail the pins.

Each mutation is a plausible slip (a wrong sign, a dropped term, a wrong
index or stride, a transposed gate, the wrong read point).  The test compiles
a copy of ``oracle/kda_oracle.c`` with the slip into a temporary directory, on
the CPU, and checks that the pin battery below rejects it.  This shows that
the pins in ``test_oracle_pins.py`` are strong enough to catch such mistakes.
"""
import os

import numpy as np
import pytest

import oracle
import chunked_model

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

DECAY = "S[i * W + j] *= alpha[i];"
MUTATIONS = {
    "gate_channel_reversed": [("alpha[i] = exp(gt[i]);", "alpha[i] = exp(gt[dk - 1 - i]);")],
    "gate_dropped": [("alpha[i] = exp(gt[i]);", "alpha[i] = 1.0;")],
    "gate_on_value_axis": [(DECAY, "S[i * W + j] *= alpha[j % dk];")],
    "delta_sign": [("u[j] = bt * (vt[j] - w[j]);", "u[j] = bt * (vt[j] + w[j]);")],
    "beta_dropped": [("u[j] = bt * (vt[j] - w[j]);", "u[j] = (vt[j] - w[j]);")],
    "read_with_query": [("acc += S[i * W + j] * kt[i];\n            w[j] = acc;",
                         "acc += S[i * W + j] * qt[i];\n            w[j] = acc;")],
    "write_along_query": [("S[i * W + j] += kt[i] * u[j];", "S[i * W + j] += qt[i] * u[j];")],
    "write_dropped": [("S[i * W + j] += kt[i] * u[j];", "S[i * W + j] += 0.0 * u[j];")],
    "output_with_key": [("acc += S[i * W + j] * qt[i];\n            ot[j] = acc;",
                         "acc += S[i * W + j] * kt[i];\n            ot[j] = acc;")],
    "beta_head_index": [("const double bt = a->beta[th];", "const double bt = a->beta[t];")],
    "key_stride": [("const double *kt = a->k + th * dk;", "const double *kt = a->k + t * dk;")],
    "last_token_skipped": [("for (int64_t t = bos; t < eos; ++t)",
                            "for (int64_t t = bos; t + 1 < eos; ++t)")],
    # decay applied after the write and read-out instead of before the read
    "decay_after_write": [
        (DECAY, "(void)0;"),
        ("            ot[j] = acc;\n        }\n",
         "            ot[j] = acc;\n        }\n"
         "        for (int i2 = 0; i2 < dk; ++i2)\n"
         "            for (int j2 = 0; j2 < W; ++j2)\n"
         "                S[i2 * W + j2] *= alpha[i2];\n")],
    # read-out taken before the write
    "output_before_write": [
        ("        double *ot = a->o + th * dv + c0;\n", ""),
        ("        for (int i = 0; i < dk; ++i)               /* S = S + k u^T */",
         "        double *ot = a->o + th * dv + c0;\n"
         "        for (int j = 0; j < W; ++j) {\n"
         "            double acc = 0.0;\n"
         "            for (int i = 0; i < dk; ++i)\n"
         "                acc += S[i * W + j] * qt[i];\n"
         "            ot[j] = acc;\n"
         "        }\n"
         "        for (int i = 0; i < dk; ++i)               /* S = S + k u^T */"),
        ("            ot[j] = acc;\n        }\n    }\n    for (int i = 0; i < dk; ++i)\n"
         "        for (int j = 0; j < W; ++j)\n            a->S_T",
         "            (void)acc;\n        }\n    }\n    for (int i = 0; i < dk; ++i)\n"
         "        for (int j = 0; j < W; ++j)\n            a->S_T"),
    ],
}


def _battery(lib) -> list[str]:
    """Run the cheap pins against one library; return the names that fail."""
    fails = []
    rng = np.random.default_rng(0)
    # hand-worked example
    from test_oracle_pins import _read_golden, _brute_force
    toks, final = _read_golden()
    T = len(toks)
    q = np.array([t[4] for t in toks])[:, None, :]
    k = np.array([t[0] for t in toks])[:, None, :]
    v = np.array([t[1] for t in toks])[:, None, :]
    beta = np.array([t[2][0] for t in toks])[:, None]
    g = np.log(np.array([t[3] for t in toks]))[:, None, :]
    o, S_T, _ = lib.prefill(q, k, v, g, beta, None, [0, T])
    if not (np.allclose(o[:, 0], [t[5] for t in toks], atol=1e-9)
            and np.allclose(S_T.reshape(-1), final, atol=1e-9)):
        fails.append("hand_worked")
    # brute force, one head
    T, dk, dv = 6, 4, 3
    q1 = rng.standard_normal((T, dk)); k1 = rng.standard_normal((T, dk))
    v1 = rng.standard_normal((T, dv)); g1 = -np.abs(rng.standard_normal((T, dk)))
    b1 = rng.uniform(0.1, 0.9, T); S01 = rng.standard_normal((dk, dv))
    o_bf, S_bf = _brute_force(q1, k1, v1, g1, b1, S01)
    o, S_T, _ = lib.prefill(q1[:, None], k1[:, None], v1[:, None], g1[:, None],
                            b1[:, None], S01[None, None], [0, T])
    if not (np.allclose(o[:, 0], o_bf, atol=1e-9) and np.allclose(S_T[0, 0], S_bf, atol=1e-9)):
        fails.append("brute_force")
    # chunked algebra model, several heads and sequences
    lengths = [3, 9, 5]
    T, H = sum(lengths), 3
    q2 = rng.standard_normal((T, H, dk)); k2 = rng.standard_normal((T, H, dk))
    v2 = rng.standard_normal((T, H, dv)); g2 = -np.abs(rng.standard_normal((T, H, dk)))
    b2 = rng.uniform(0.1, 0.9, (T, H)); S02 = rng.standard_normal((3, H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, S_T, _ = lib.prefill(q2, k2, v2, g2, b2, S02, cu)
    o_c, S_c = chunked_model.prefill(q2, k2, v2, g2, b2, S02, cu, 4)
    if not (np.allclose(o, o_c, atol=1e-9) and np.allclose(S_T, S_c, atol=1e-9)):
        fails.append("chunked_model")
    return fails


def test_unmutated_oracle_passes_battery():
    assert _battery(oracle._load()) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert old in src, "mutation anchor not found: %r" % old
        src = src.replace(old, new, 1)
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src)
    lib = oracle.OracleLib(oracle.build(force=True, src=str(mpath),
                                        out=str(tmp_path / "libmutant.so")))
    assert _battery(lib), "mutation %s was not caught by any pin" % name
