"""Each planted mistake in a copy of the oracle must fail at least one pin.

The mistakes are the plausible ones: a dropped term, a wrong sign, a shifted
index, a transposed operand, a wrong log base.  Every mutant is compiled from
a textual edit of ``oracle/fa_oracle.c`` into a temporary directory; the real
oracle is untouched.
"""
import os

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "fa_oracle.c")

MUTANTS = {
    "dK drops the scale": ("dkj[c] += scale * dsij * qi[c];", "dkj[c] += dsij * qi[c];"),
    "dQ drops the scale": ("dqi[c] += scale * dsij * kj[c];", "dqi[c] += dsij * kj[c];"),
    "dS sign flipped (dQ pass)": ("double dsij = s[j] * (dpij - Di);",
                                  "double dsij = s[j] * (dpij + Di);"),
    "dS drops D (dK/dV pass)": ("double dsij = pij * (dpij - Dout[bh * N + i]);",
                                "double dsij = pij * dpij;"),
    "dV transposed operand": ("dvj[c] += pij * doi[c];",
                              "dvj[c] += pij * dout[(long)j * d + c];"),
    "dK/dV pass: causal start shifted": ("for (int i = causal ? j : 0; i < N; ++i)",
                                        "for (int i = causal ? j + 1 : 0; i < N; ++i)"),
    "dK/dV pass: P from a log2 L": ("double pij = exp(scale * dot(qi, kj, d) - Lrow[bh * N + i]);",
                                   "double pij = exp2(scale * dot(qi, kj, d) - Lrow[bh * N + i]);"),
    "causal mask shifted": ("causal ? (i + 1 < N ? i + 1 : N) : N",
                            "causal ? (i + 2 < N ? i + 2 : N) : N"),
    "L in log2": ("lse[i] = m + log(l);", "lse[i] = m + log2(l);"),
    "sum without max subtraction": ("for (int j = 0; j < nk; ++j) l += exp(s[j] - m);",
                                    "for (int j = 0; j < nk; ++j) l += exp(s[j]);"),
    "online: alpha not applied to l": ("l = l * alpha + psum;", "l = l + psum;"),
    "online: alpha not applied to acc": ("for (int t = 0; t < d; ++t) acc[t] *= alpha;",
                                         "for (int t = 0; t < d; ++t) acc[t] *= 1.0;"),
    "window starts one key early": (
        "return (window > 0 && i - window + 1 > 0) ? i - window + 1 : 0;",
        "return (window > 0 && i - window > 0) ? i - window : 0;"),
    "window: key pass keeps one query too many": (
        "if (window > 0 && i - j >= window) break;", "if (window > 0 && i - j > window) break;"),
    "merge: wrong weight": ("*l_out = a1 * l1 + a2 * l2;", "*l_out = a1 * l1 + a1 * l2;"),
    "scores transposed (k_i . q_j)": (
        "double m = row_scores(q + (long)i * d, k + (long)j0 * d, nk, d, scale, s, &l);\n"
        "                double* oi = o",
        "double m = row_scores(k + (long)i * d, q + (long)j0 * d, nk, d, scale, s, &l);\n"
        "                double* oi = o"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(before) == 1, f"mutation anchor not unique: {before!r}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(before, after))
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(so)
    failures = []
    for pin in pins.ORACLE_PINS:
        if pin is pins.pin_torch_sdpa:
            try:
                pin(orc, shapes=((1, 2, 37, 8, False), (1, 2, 37, 8, True)))
            except AssertionError as e:
                failures.append(pin.__name__)
            continue
        if pin is pins.pin_gqa:
            try:
                pin(orc, shapes=((1, 4, 2, 21, 8, True),))
            except AssertionError:
                failures.append(pin.__name__)
            continue
        try:
            pin(orc)
        except AssertionError:
            failures.append(pin.__name__)
    assert failures, f"no pin caught the planted mistake '{name}'"


# Planted mistakes in the oracle's grouped-query layer (Python, oracle/__init__.py):
# each mutant module is the oracle package's source with one textual edit, run on the
# real compiled core.
PY_SRC = os.path.join(os.path.dirname(oracle.__file__), "__init__.py")
GQA_MUTANTS = {
    "fp8: exponent bias 8": (
        "np.exp2(e - 7.0)", "np.exp2(e - 8.0)"),
    "fp8: subnormals read as normals": (
        "(m / 8.0) * 2.0 ** -6", "(1.0 + m / 8.0) * 2.0 ** -7"),
    "fp8: v descale dropped": (
        "v = self.e4m3_values(v8) * v_scale", "v = self.e4m3_values(v8)"),
    "decode: last cached key dropped": (
        "m, l, acc = self.row_partial(q[b, h], kc[b, h // g, :n], vc[b, h // g, :n], 0, 0,\n"
        "                                             n, False, scale, n)",
        "m, l, acc = self.row_partial(q[b, h], kc[b, h // g, :n], vc[b, h // g, :n], 0, 0,\n"
        "                                             n - 1, False, scale, n)"),
    "varlen: a sequence sees the next one's first key": (
        "qs, ks, vs = (x[a:e].transpose(1, 0, 2)[None] for x in (q, k, v))",
        "qs, ks, vs = (x[a:min(e + 1, total)].transpose(1, 0, 2)[None] for x in (q, k, v))"),
    "GQA: dK averaged over the group": (
        "return (dq, dk.reshape(B, Hkv, g, N, d).sum(axis=2),",
        "return (dq, dk.reshape(B, Hkv, g, N, d).mean(axis=2),"),
    "GQA: dV from the first query head only": (
        "dv.reshape(B, Hkv, g, N, d).sum(axis=2),",
        "dv.reshape(B, Hkv, g, N, d)[:, :, 0],"),
    "GQA: interleaved head mapping": (
        "return self.fwd(q, np.repeat(_f64(k), g, axis=1), np.repeat(_f64(v), g, axis=1), causal,",
        "return self.fwd(q, np.tile(_f64(k), (1, g, 1, 1)), np.tile(_f64(v), (1, g, 1, 1)), causal,"),
}


@pytest.mark.parametrize("name", sorted(GQA_MUTANTS))
def test_gqa_mutant_is_caught(name):
    before, after = GQA_MUTANTS[name]
    text = open(PY_SRC).read()
    assert text.count(before) == 1, f"mutation anchor not unique: {before!r}"
    ns = {"__name__": "oracle_mutant", "__file__": PY_SRC}
    exec(compile(text.replace(before, after), "oracle_mutant", "exec"), ns)
    orc = ns["Oracle"](oracle.build())
    with pytest.raises((AssertionError, ValueError)):
        if name.startswith("varlen"):
            pins.pin_varlen(orc)
        elif name.startswith("decode"):
            pins.pin_decode(orc)
        elif name.startswith("fp8"):
            pins.pin_fp8(orc)
        else:
            pins.pin_gqa(orc, shapes=((1, 4, 2, 21, 8, True),))
