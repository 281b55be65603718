"""The CPU oracle against facts outside itself (no GPU needed)."""
import os
import shutil

import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin, oracle_lib):
    fails = pin(oracle_lib)
    assert not fails, "\n".join(fails)


# Plausible mistakes, planted in a copy of the oracle's C source: each must be
# caught by at least one pin.  (original text, planted text, what it models)
MUTANTS = [
    ("return (i + 1 < Nk) ? (i + 1) : Nk;", "return (i + 2 < Nk) ? (i + 2) : Nk;",
     "causal rule admits one future key"),
    ("        s[j] = scale * dot;\n", "        s[j] = dot;\n", "scale dropped"),
    ("    *lse = m + log(l);", "    *lse = log(l);", "max term dropped from LSE"),
    ("orow[x] += p * (double)vh[j * d + x];", "orow[x] += p * (double)kh[j * d + x];",
     "keys used in place of values"),
    ("double p = exp(s[j] - m);", "double p = exp(m - s[j]);", "sign of the exponent"),
    ("    for (long x = 0; x < d; ++x) orow[x] /= l;\n    *lse",
     "    for (long x = 0; x < d; ++x) orow[x] /= 1.0;\n    *lse", "normalisation dropped"),
    ("kh[j * d + x];\n        s[j] = scale", "kh[j * d + (d - 1 - x)];\n        s[j] = scale",
     "key reversed along d"),
    ("const float *kh = J->k + bh * J->Nk * J->d;",
     "const float *kh = J->k + (bh % J->H) * J->Nk * J->d;", "wrong head's keys"),
    ("dvh[j * d + x] += p[j] * (double)doi[x];",
     "dvh[j * d + x] += p[j] * (double)doh[(j % Nq) * d + x];",
     "dV takes the key's row of dO (the page's backward indexing slip)"),
    ("            D += p[j] * dot;", "            D += dot;", "D without the probabilities"),
    ("dqh[i * d + x] += J->scale * ds * (double)kh[j * d + x];",
     "dqh[i * d + x] += ds * (double)kh[j * d + x];", "dQ without the scale"),
]


@pytest.mark.parametrize("orig,planted,what", MUTANTS, ids=[m[2] for m in MUTANTS])
def test_planted_mistake_is_caught(orig, planted, what, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.oracle.__file__), "attn_oracle.c")).read()
    assert src.count(orig) == 1, f"mutation anchor not unique: {orig!r}"
    mpath = tmp_path / "attn_oracle_mutant.c"
    mpath.write_text(src.replace(orig, planted))
    path = oracle.oracle.build(src=str(mpath), build_dir=str(tmp_path), force=True)
    lib = oracle.oracle.load(path)
    caught = []
    for pin in P.ALL_PINS:
        try:
            if pin(lib):
                caught.append(pin.__name__)
        except Exception as e:  # a crash or NaN blow-up also counts as caught
            caught.append(f"{pin.__name__} ({type(e).__name__})")
    assert caught, f"no pin caught the planted mistake: {what}"


def test_oracle_rejects_bad_arguments(oracle_lib):
    import numpy as np
    q = np.zeros((1, 1, 2, 2), np.float32)
    with pytest.raises(RuntimeError):
        oracle.attn_rows(q, q, q, [5], 1.0, False, lib=oracle_lib)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd_online(q, q, q, 1.0, False, bc=0, lib=oracle_lib)
