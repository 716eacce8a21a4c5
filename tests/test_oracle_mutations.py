"""Plant one mistake at a time in a copy of the oracle's C source and check
that the pins catch it.  The mistakes are the plausible ones: a dropped term,
a wrong sign, a wrong denominator, a wrong index or row stride, a missing
max subtraction.  Nothing here touches the real oracle or a GPU."""

import os

import pytest

import oracle
from oracle_pins import check_all

# (name, original text, planted text, which occurrence (0-based))
MUTATIONS = [
    ("resln-unbiased-variance", "double variance = sq / (double)width;",
     "double variance = sq / (double)(width - 1);", 0),
    ("ln-unbiased-variance", "double variance = sq / (double)width;",
     "double variance = sq / (double)(width - 1);", 1),
    ("resln-no-eps", "sqrt(variance + eps)", "sqrt(variance)", 0),
    ("ln-no-eps", "sqrt(variance + eps)", "sqrt(variance)", 1),
    ("rms-no-eps", "sqrt(mean_square + eps)", "sqrt(mean_square)", 0),
    ("resln-sign", "(((double)xi[j] + (double)ri[j]) - mean) / denom",
     "(((double)xi[j] + (double)ri[j]) + mean) / denom", 0),
    ("resln-residual-dropped-from-mean", "sum += (double)xi[j] + (double)ri[j];",
     "sum += (double)xi[j];", 0),
    ("resln-row-stride", "const float *ri = r + i * width;", "const float *ri = r + i;", 0),
    ("ln-row-stride", "const float *xi = x + i * width;", "const float *xi = x + i;", 1),
    ("ln-mean-denominator", "double mean = sum / (double)width;",
     "double mean = sum / (double)(width + 1);", 1),
    ("rms-square-dropped", "sq += (double)xi[j] * (double)xi[j];", "sq += (double)xi[j];", 0),
    ("softmax-min-not-max", "if ((double)xi[j] > m)", "if ((double)xi[j] < m)", 0),
    ("softmax-no-max-subtraction", "total += exp((double)xi[j] - m);",
     "total += exp((double)xi[j]);", 0),
    ("softmax-wrong-index", "yi[j] = exp((double)xi[j] - m) / total;",
     "yi[j] = exp((double)xi[0] - m) / total;", 0),
    ("affine-beta-dropped", "yi[j] = normed * (double)gamma[j] + (beta ? (double)beta[j] : 0.0);",
     "yi[j] = normed * (double)gamma[j];", 0),
    ("affine-gamma-beta-swapped",
     "yi[j] = normed * (double)gamma[j] + (beta ? (double)beta[j] : 0.0);",
     "yi[j] = normed * (beta ? (double)beta[j] : 1.0) + (double)gamma[j];", 0),
    ("affine-residual-dropped-from-variance",
     "double centered = ((double)xi[j] + (ri ? (double)ri[j] : 0.0)) - mean;",
     "double centered = (double)xi[j] - mean;", 0),
    ("weighted-rms-gamma-index", "yi[j] = (double)xi[j] / denom * (double)gamma[j];",
     "yi[j] = (double)xi[j] / denom * (double)gamma[0];", 0),
    ("row-sum-float-accumulator", "        double sum = 0.0;\n        for (long j = 0; j < width; ++j)\n            sum += (double)xi[j];\n        s[i] = sum;",
     "        float sum = 0.0f;\n        for (long j = 0; j < width; ++j)\n            sum += xi[j];\n        s[i] = sum;", 0),
    ("row-sum-skips-last", "        for (long j = 0; j < width; ++j)\n            sum += (double)xi[j];\n        s[i] = sum;",
     "        for (long j = 0; j + 1 < width; ++j)\n            sum += (double)xi[j];\n        s[i] = sum;", 0),
    ("minmax-swapped", "        mn[i] = lo;\n        mx[i] = hi;", "        mn[i] = hi;\n        mx[i] = lo;", 0),
    ("sigmoid-derivative-sign", "dy[k] = s * (1.0 - s);", "dy[k] = s * (1.0 + s);", 0),
    ("gelu-cubic-coefficient", "const double a = 0.044715;", "const double a = 0.04715;", 0),
    ("gelu-derivative-missing-3", "(1.0 + 3.0 * a * v * v)", "(1.0 + a * v * v)", 0),
    ("gelu-derivative-tanh-square", "(1.0 - t * t)", "(1.0 - t)", 0),
    ("ln-backward-mean-g-dropped", "out[j] = rstd * (g - mean_g - xhat * mean_gx);",
     "out[j] = rstd * (g - xhat * mean_gx);", 0),
    ("ln-backward-sign", "out[j] = rstd * (g - mean_g - xhat * mean_gx);",
     "out[j] = rstd * (g - mean_g + xhat * mean_gx);", 0),
    ("ln-backward-gamma-ignored", "double g = (double)di[j] * (gamma ? (double)gamma[j] : 1.0);\n            double xhat = ((double)xi[j] - mean) * rstd;\n            out[j]",
     "double g = (double)di[j];\n            double xhat = ((double)xi[j] - mean) * rstd;\n            out[j]", 0),
    ("rms-backward-rstd-dropped", "out[j] = rstd * (g - (double)xi[j] * rstd * mean_gx);",
     "out[j] = rstd * (g - (double)xi[j] * mean_gx);", 0),
    ("softmax-backward-sign", "out[j] = (double)yi[j] * ((double)di[j] - dot);",
     "out[j] = (double)yi[j] * ((double)di[j] + dot);", 0),
    ("param-grad-dbeta", "dbeta[j] += (double)di[j];", "dbeta[j] += (double)di[j] * (double)xi[j];", 0),
    ("param-grad-rms-centred", "        if (!rms) {", "        if (1) {", 0),
]


def _mutate(text, old, new, occurrence):
    pos = -1
    for _ in range(occurrence + 1):
        pos = text.index(old, pos + 1)
    return text[:pos] + new + text[pos + len(old):]


@pytest.mark.parametrize("name,old,new,occ", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, occ):
    src = open(oracle.SOURCE).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    path = tmp_path / "oracle_mut.c"
    path.write_text(mutated)
    lib = oracle.build(str(path), str(tmp_path / f"liboracle_{name}.so"), force=True)
    fails = check_all(oracle.Oracle(lib))
    assert fails, f"planted mistake {name} was not caught by any pin"
