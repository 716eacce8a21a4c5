"""Pins of the FP64 oracle against things other than itself.

``check_all(orc)`` runs every pin against one loaded oracle and returns the
list of failures (empty when the oracle is right).  The same checks run on
the real oracle (all must pass) and on copies of it with a planted mistake
(at least one must fail), see ``test_oracle_mutations.py``.

Pins used:
  * hand-worked golden cases in ``tests/golden`` (exact rationals derived by
    hand from the definitions on the pages);
  * closed forms: constant rows, +-a rows, softmax of logarithms;
  * invariants that follow from the definitions: LayerNorm output has mean 0
    and variance var/(var+eps); RMSNorm output has mean square
    ms/(ms+eps); softmax rows sum to 1 and y_i/y_j = exp(x_i - x_j); shift
    and scale invariance; permutation equivariance; residual symmetry;
    row independence;
  * a library special case: torch's CPU FP64 layer_norm / rms_norm / softmax.
"""

from __future__ import annotations

import glob
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
getcontext().prec = 50


# ---------------------------------------------------------------------------
# golden fixtures
# ---------------------------------------------------------------------------

def load_golden(path):
    case = {"x": [], "r": [], "numer": [], "den": [], "expect": [], "atol": 0.0,
            "min": [], "max": [], "y": [], "dy": []}
    with open(path) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = [s.strip() for s in line.split(":", 1)]
            if key == "op":
                case["op"] = val
            elif key == "eps":
                case["eps"] = val
            elif key == "atol":
                case["atol"] = float(val)
            elif key in ("x", "r", "upstream", "fwd"):
                case.setdefault(key, []).append([float(v) for v in val.split()])
            elif key in ("numer", "expect", "min", "max", "y", "dy"):
                case[key].append([Fraction(v) for v in val.split()])
            elif key in ("gamma", "beta"):
                case[key] = [float(v) for v in val.split()]
            elif key == "den":
                case[key].append(Fraction(val))
            else:
                raise ValueError(f"{path}: unknown key {key}")
    return case


def _dec(f):
    return Decimal(f.numerator) / Decimal(f.denominator)


def _exact(rows):
    return np.array([[float(_dec(f)) for f in row] for row in rows])


def golden_expected(case):
    """Expected outputs of a golden case, evaluated to 50 digits."""
    op = case["op"]
    if op in ("softmax", "row_sum", "softmax_backward"):
        return _exact(case["expect"])
    if op == "row_minmax":
        return _exact(case["min"]), _exact(case["max"])
    if op in ("sigmoid_pair", "gelu_tanh_pair"):
        return _exact(case["y"]), _exact(case["dy"])
    eps = Decimal(case["eps"])
    gamma = case.get("gamma")
    beta = case.get("beta")
    out = []
    for numer, den in zip(case["numer"], case["den"]):
        root = (_dec(den) + eps).sqrt()
        row = []
        for j, f in enumerate(numer):
            v = _dec(f) / root
            if gamma is not None:
                v = v * Decimal(repr(gamma[j])) + (Decimal(repr(beta[j])) if beta else 0)
            row.append(float(v))
        out.append(row)
    return np.array(out)


def golden_cases():
    return sorted(p for p in glob.glob(os.path.join(GOLDEN, "*.txt"))
                  if os.path.basename(p) != "README.txt")


def _run_golden(orc, path):
    case = load_golden(path)
    if "op" not in case:
        return None
    x = np.array(case["x"], dtype=np.float32) if case["x"] else None
    eps = float(case.get("eps", "1e-5"))
    op = case["op"]
    if op == "layernorm_backward":
        got = orc.layernorm_backward(x, np.array(case["upstream"], np.float32), eps=eps)
    elif op == "rmsnorm_backward":
        got = orc.rmsnorm_backward(x, np.array(case["upstream"], np.float32), eps=eps)
    elif op == "softmax_backward":
        got = orc.softmax_backward(np.array(case["fwd"], np.float32),
                                   np.array(case["upstream"], np.float32))
    elif op == "residual_layernorm":
        got = orc.residual_layernorm(x, np.array(case["r"], dtype=np.float32), eps)
    elif op == "layernorm_affine":
        got = orc.layernorm_affine(x, case["gamma"], case.get("beta"), eps=eps)
    elif op == "rmsnorm_weighted":
        got = orc.rmsnorm_weighted(x, case["gamma"], eps=eps)
    elif op == "row_sum":
        got = orc.row_sum(x)[None, :]
    elif op == "row_minmax":
        mn, mx = orc.row_minmax(x)
        got = (mn[None, :], mx[None, :])
    elif op == "sigmoid_pair":
        got = tuple(a.reshape(1, -1) for a in orc.sigmoid_pair(x.reshape(-1)))
    elif op == "gelu_tanh_pair":
        got = tuple(a.reshape(1, -1) for a in orc.gelu_tanh_pair(x.reshape(-1)))
    else:
        got = orc.run(op, x, eps=eps)
    want = golden_expected(case)
    pairs = zip(got, want) if isinstance(want, tuple) else [(got, want)]
    for g, w in pairs:
        tol = 1e-12 + case["atol"] + 1e-12 * np.abs(w)
        if g.shape != w.shape or not np.all(np.abs(g - w) <= tol):
            return f"golden {os.path.basename(path)}: got {np.asarray(got).tolist()} want {w.tolist()}"
    return None


# ---------------------------------------------------------------------------
# closed forms and invariants on seeded inputs
# ---------------------------------------------------------------------------

def _seeded(rows, width, seed, sigma=None):
    n = rows * width
    v = synth.uniform_pm1(seed, n) if sigma is None else synth.normal(seed, n, sigma)
    return v.reshape(rows, width)


def _close(a, b, tol):
    return a.shape == b.shape and bool(np.all(np.abs(a - b) <= tol))


def _pins_layernorm(orc):
    fails = []
    eps = 1e-5
    x = _seeded(9, 257, 11)
    y = orc.layernorm(x, eps)
    var_x = x.astype(np.float64).var(axis=1)
    if not np.all(np.abs(y.mean(axis=1)) <= 1e-12):
        fails.append("layernorm: row mean of output is not 0")
    if not _close(y.var(axis=1), var_x / (var_x + eps), 1e-12):
        fails.append("layernorm: output variance != var/(var+eps)")
    # shift by an exactly representable constant, scale by 2 (eps = 0)
    if not _close(orc.layernorm(x + np.float32(0.5), eps), y, 1e-12):
        fails.append("layernorm: not shift invariant")
    if not _close(orc.layernorm(2 * x, 0.0), orc.layernorm(x, 0.0), 1e-12):
        fails.append("layernorm: not scale invariant at eps=0")
    # permutation equivariance and row independence
    if not _close(orc.layernorm(x[:, ::-1], eps), y[:, ::-1], 1e-13):
        fails.append("layernorm: not permutation equivariant")
    single = np.vstack([orc.layernorm(x[i:i + 1], eps) for i in range(x.shape[0])])
    if not np.array_equal(single, y):
        fails.append("layernorm: rows not independent")
    # constant rows of non-dyadic values give exactly 0
    c = np.full((3, 1000), np.float32(0.1), dtype=np.float32)
    if not np.all(np.abs(orc.layernorm(c, eps)) <= 1e-9):
        fails.append("layernorm: constant row is not 0")
    return fails


def _pins_residual(orc):
    fails = []
    eps = 1e-5
    x = _seeded(7, 1537, 21)
    r = _seeded(7, 1537, 22)
    y = orc.residual_layernorm(x, r, eps)
    if not _close(orc.residual_layernorm(r, x, eps), y, 1e-13):
        fails.append("residual_layernorm: not symmetric in (x, residual)")
    zero = np.zeros_like(x)
    if not _close(orc.residual_layernorm(x, zero, eps), orc.layernorm(x, eps), 1e-13):
        fails.append("residual_layernorm(x, 0) != layernorm(x)")
    c = (x.astype(np.float64) + r.astype(np.float64))
    var_c = c.var(axis=1)
    if not np.all(np.abs(y.mean(axis=1)) <= 1e-12):
        fails.append("residual_layernorm: row mean of output is not 0")
    if not _close(y.var(axis=1), var_c / (var_c + eps), 1e-12):
        fails.append("residual_layernorm: output variance != var/(var+eps)")
    single = np.vstack([orc.residual_layernorm(x[i:i + 1], r[i:i + 1], eps) for i in range(7)])
    if not np.array_equal(single, y):
        fails.append("residual_layernorm: rows not independent")
    return fails


def _pins_rmsnorm(orc):
    fails = []
    eps = 1e-5
    x = _seeded(5, 4096, 31, sigma=3.0)
    y = orc.rmsnorm(x, eps)
    ms = (x.astype(np.float64) ** 2).mean(axis=1)
    if not _close((y ** 2).mean(axis=1), ms / (ms + eps), 1e-12):
        fails.append("rmsnorm: output mean square != ms/(ms+eps)")
    if not _close(orc.rmsnorm(x[:, ::-1], eps), y[:, ::-1], 1e-13):
        fails.append("rmsnorm: not permutation equivariant")
    # +-a rows: y = +-a / sqrt(a^2 + eps)
    a = np.float32(0.3)
    pm = np.where(np.arange(64) % 3 == 0, a, -a).astype(np.float32)[None, :]
    want = np.sign(pm.astype(np.float64)) * float(a) / math.sqrt(float(a) ** 2 + eps)
    if not _close(orc.rmsnorm(pm, eps), want, 1e-14):
        fails.append("rmsnorm: +-a row is not +-a/sqrt(a^2+eps)")
    single = np.vstack([orc.rmsnorm(x[i:i + 1], eps) for i in range(x.shape[0])])
    if not np.array_equal(single, y):
        fails.append("rmsnorm: rows not independent")
    return fails


def _pins_softmax(orc):
    fails = []
    x = _seeded(6, 8192, 41, sigma=3.0)
    x[1, 100] = np.float32(40.0)
    y = orc.softmax(x)
    if not _close(y.sum(axis=1), np.ones(6), 1e-12):
        fails.append("softmax: rows do not sum to 1")
    if not np.all(y > 0):
        fails.append("softmax: non-positive output")
    i, j = 17, 4000
    ratio = y[:, i] / y[:, j]
    want = np.exp(x[:, i].astype(np.float64) - x[:, j].astype(np.float64))
    if not _close(ratio / want, np.ones(6), 1e-12):
        fails.append("softmax: y_i/y_j != exp(x_i - x_j)")
    u = _seeded(3, 1000, 42)       # values k/2^23 in [-1, 1): +0.5 is exact
    if not _close(orc.softmax(u + np.float32(0.5)), orc.softmax(u), 1e-15):
        fails.append("softmax: not shift invariant")
    if not _close(orc.softmax(x[:, ::-1]), y[:, ::-1], 1e-12):
        fails.append("softmax: not permutation equivariant")
    c = np.full((2, 300), np.float32(-1.7), dtype=np.float32)
    if not _close(orc.softmax(c), np.full((2, 300), 1.0 / 300), 1e-15):
        fails.append("softmax: constant row is not 1/width")
    single = np.vstack([orc.softmax(x[k:k + 1]) for k in range(x.shape[0])])
    if not np.array_equal(single, y):
        fails.append("softmax: rows not independent")
    return fails


def _pins_torch(orc):
    """Library special case: torch's CPU FP64 functional ops."""
    import torch
    import torch.nn.functional as F
    fails = []
    eps = 1e-5
    x = _seeded(8, 1537, 51)
    r = _seeded(8, 1537, 52)
    tx = torch.from_numpy(x).double()
    tr = torch.from_numpy(r).double()
    checks = [
        ("layernorm", orc.layernorm(x, eps), F.layer_norm(tx, (1537,), eps=eps)),
        ("residual_layernorm", orc.residual_layernorm(x, r, eps),
         F.layer_norm(tx + tr, (1537,), eps=eps)),
        ("rmsnorm", orc.rmsnorm(x, eps), F.rms_norm(tx, (1537,), eps=eps)),
        ("softmax", orc.softmax(x), torch.softmax(tx, dim=1)),
    ]
    for name, got, want in checks:
        if not _close(got, want.numpy(), 1e-12):
            fails.append(f"{name}: differs from torch FP64")
    return fails


def _pins_affine(orc):
    import torch
    import torch.nn.functional as F
    fails = []
    eps = 1e-5
    x = _seeded(6, 1537, 61)
    r = _seeded(6, 1537, 62)
    g = synth.uniform_pm1(63, 1537) * np.float32(2.0)
    b = synth.uniform_pm1(64, 1537)
    ones = np.ones(1537, np.float32)
    if not np.array_equal(orc.layernorm_affine(x, ones, None, eps=eps), orc.layernorm(x, eps)):
        fails.append("layernorm_affine(gamma=1, no beta) != layernorm")
    if not np.array_equal(orc.layernorm_affine(x, ones, np.zeros_like(ones), r=r, eps=eps),
                          orc.residual_layernorm(x, r, eps)):
        fails.append("layernorm_affine(gamma=1, beta=0, r) != residual_layernorm")
    two = np.full(1537, 2.0, np.float32)
    if not _close(orc.layernorm_affine(x, two, ones * np.float32(0.25), eps=eps),
                  2 * orc.layernorm(x, eps) + 0.25, 1e-14):
        fails.append("layernorm_affine(gamma=2, beta=1/4) != 2 LN + 1/4")
    c = torch.from_numpy(x).double() + torch.from_numpy(r).double()
    want = F.layer_norm(c, (1537,), weight=torch.from_numpy(g).double(),
                        bias=torch.from_numpy(b).double(), eps=eps).numpy()
    if not _close(orc.layernorm_affine(x, g, b, r=r, eps=eps), want, 1e-12):
        fails.append("layernorm_affine differs from torch FP64 layer_norm(weight, bias)")
    want = F.rms_norm(torch.from_numpy(x).double(), (1537,), weight=torch.from_numpy(g).double(),
                      eps=eps).numpy()
    if not _close(orc.rmsnorm_weighted(x, g, eps), want, 1e-12):
        fails.append("rmsnorm_weighted differs from torch FP64 rms_norm(weight)")
    if not np.array_equal(orc.rmsnorm_weighted(x, ones, eps), orc.rmsnorm(x, eps)):
        fails.append("rmsnorm_weighted(gamma=1) != rmsnorm")
    return fails


def _pins_reductions(orc):
    import math
    fails = []
    # integer-valued rows: the FP64 sum is exact, compare with Python integers
    ints = (np.arange(5 * 999, dtype=np.int64) % 97 - 48).reshape(5, 999)
    if not np.array_equal(orc.row_sum(ints.astype(np.float32)), ints.sum(axis=1).astype(np.float64)):
        fails.append("row_sum: integer rows not exact")
    x = _seeded(7, 4096, 71)
    fs = np.array([math.fsum(row.astype(np.float64)) for row in x])
    if not _close(orc.row_sum(x), fs, 1e-10):
        fails.append("row_sum: differs from math.fsum")
    if not _close(orc.row_sum(x[:, ::-1]), orc.row_sum(x), 1e-10):
        fails.append("row_sum: not permutation invariant")
    mn, mx = orc.row_minmax(x)
    if not (np.array_equal(mn, x.min(axis=1).astype(np.float64))
            and np.array_equal(mx, x.max(axis=1).astype(np.float64))):
        fails.append("row_minmax: differs from numpy min/max")
    mn2, mx2 = orc.row_minmax(-x)
    if not (np.array_equal(mn2, -mx) and np.array_equal(mx2, -mn)):
        fails.append("row_minmax: min(-x) != -max(x)")
    return fails


def _pins_pairs(orc):
    import torch
    import torch.nn.functional as F
    fails = []
    x = synth.normal(81, 20000, 4.0)
    y, dy = orc.sigmoid_pair(x)
    yn, _ = orc.sigmoid_pair(-x)
    if not _close(y + yn, np.ones_like(y), 1e-15):
        fails.append("sigmoid: s(x) + s(-x) != 1")
    tx = torch.from_numpy(x).double().requires_grad_(True)
    ts = torch.sigmoid(tx)
    ts.sum().backward()
    if not (_close(y, ts.detach().numpy(), 1e-15) and _close(dy, tx.grad.numpy(), 1e-15)):
        fails.append("sigmoid pair differs from torch FP64 sigmoid / autograd")
    g, dg = orc.gelu_tanh_pair(x)
    gn, _ = orc.gelu_tanh_pair(-x)
    if not _close(g - gn, x.astype(np.float64), 1e-12):
        fails.append("gelu: g(x) - g(-x) != x")
    tx = torch.from_numpy(x).double().requires_grad_(True)
    tg = F.gelu(tx, approximate="tanh")
    tg.sum().backward()
    if not (_close(g, tg.detach().numpy(), 1e-12) and _close(dg, tx.grad.numpy(), 1e-12)):
        fails.append("gelu pair differs from torch FP64 gelu(tanh) / autograd")
    # derivatives against central differences of the value (h = 2^-12)
    xs = np.linspace(-6, 6, 241).astype(np.float32)
    h = 2.0 ** -12
    for name, fn in (("sigmoid", orc.sigmoid_pair), ("gelu", orc.gelu_tanh_pair)):
        _, d = fn(xs)
        up, _ = fn((xs.astype(np.float64) + h).astype(np.float32))
        dn, _ = fn((xs.astype(np.float64) - h).astype(np.float32))
        fd = (up - dn) / (2 * h)
        if not _close(d, fd, 1e-6):
            fails.append(f"{name}: derivative differs from central differences")
    return fails


def _pins_backward(orc):
    """Backward passes against torch autograd in FP64 (library special case),
    directional finite differences of the forward oracle, and invariants."""
    import torch
    import torch.nn.functional as F
    fails = []
    eps = 1e-5
    rows, width = 6, 257
    x = _seeded(rows, width, 91)
    dy = _seeded(rows, width, 92)
    g = synth.uniform_pm1(93, width) + np.float32(1.5)
    for name, fwd, bwd in (
            ("layernorm", lambda t, w: F.layer_norm(t, (width,), weight=w, eps=eps),
             orc.layernorm_backward),
            ("rmsnorm", lambda t, w: F.rms_norm(t, (width,), weight=w, eps=eps),
             orc.rmsnorm_backward)):
        for gamma in (None, g):
            tx = torch.from_numpy(x).double().requires_grad_(True)
            tw = torch.from_numpy(gamma).double() if gamma is not None else None
            fwd(tx, tw).backward(torch.from_numpy(dy).double())
            if not _close(bwd(x, dy, gamma, eps), tx.grad.numpy(), 1e-12):
                fails.append(f"{name} backward differs from torch autograd (gamma={gamma is not None})")
    ty = torch.from_numpy(x).double().requires_grad_(True)
    sm = torch.softmax(ty, dim=1)
    sm.backward(torch.from_numpy(dy).double())
    y32 = sm.detach().numpy().astype(np.float32)
    # the oracle takes the FP32 output; compare with autograd at that y
    tyy = torch.from_numpy(y32).double()
    want = (tyy * (torch.from_numpy(dy).double() - (torch.from_numpy(dy).double() * tyy)
                   .sum(dim=1, keepdim=True))).numpy()
    if not _close(orc.softmax_backward(y32, dy), want, 1e-14):
        fails.append("softmax backward differs from y*(dy - sum(dy*y))")
    if not _close(orc.softmax_backward(sm.detach().numpy().astype(np.float32), dy),
                  ty.grad.numpy(), 1e-6):
        fails.append("softmax backward differs from torch autograd")
    # directional finite differences of the forward oracle: <dy, dF/dx v> = <dx, v>
    v = _seeded(rows, width, 94)
    h = 2.0 ** -10
    for name, f, bwd in (("layernorm", orc.layernorm, orc.layernorm_backward),
                         ("rmsnorm", orc.rmsnorm, orc.rmsnorm_backward)):
        xp = (x.astype(np.float64) + h * v).astype(np.float32)
        xm = (x.astype(np.float64) - h * v).astype(np.float32)
        dirv = (xp.astype(np.float64) - xm.astype(np.float64)) / 2.0   # exact step taken
        lhs = np.sum(dy * (f(xp, eps) - f(xm, eps)), axis=1)
        rhs = np.sum(bwd(x, dy, None, eps) * 2.0 * dirv, axis=1)
        if not _close(lhs, rhs, 1e-5 * np.abs(rhs).max() + 1e-9):
            fails.append(f"{name} backward differs from central differences")
    # invariants: LayerNorm is shift invariant, so rows of dx sum to 0;
    # softmax rows of dx sum to 0 as well
    if not np.all(np.abs(orc.layernorm_backward(x, dy, g, eps).sum(axis=1)) <= 1e-10):
        fails.append("layernorm backward rows do not sum to 0")
    if not np.all(np.abs(orc.softmax_backward(y32, dy).sum(axis=1)) <= 1e-6):
        fails.append("softmax backward rows do not sum to 0")
    # parameter gradients against autograd
    tx = torch.from_numpy(x).double()
    tw = torch.from_numpy(g).double().requires_grad_(True)
    tb = torch.zeros(width, dtype=torch.float64, requires_grad=True)
    F.layer_norm(tx, (width,), weight=tw, bias=tb, eps=eps).backward(torch.from_numpy(dy).double())
    dg, db = orc.norm_param_grad(x, dy, eps)
    if not (_close(dg, tw.grad.numpy(), 1e-12) and _close(db, tb.grad.numpy(), 1e-12)):
        fails.append("layernorm parameter gradients differ from torch autograd")
    tw = torch.from_numpy(g).double().requires_grad_(True)
    F.rms_norm(tx, (width,), weight=tw, eps=eps).backward(torch.from_numpy(dy).double())
    dg, db = orc.norm_param_grad(x, dy, eps, rms=True)
    if db is not None or not _close(dg, tw.grad.numpy(), 1e-12):
        fails.append("rmsnorm parameter gradient differs from torch autograd")
    return fails


def check_all(orc):
    fails = []
    for path in golden_cases():
        f = _run_golden(orc, path)
        if f:
            fails.append(f)
    for group in (_pins_layernorm, _pins_residual, _pins_rmsnorm, _pins_softmax, _pins_torch,
                  _pins_affine, _pins_reductions, _pins_pairs, _pins_backward):
        try:
            fails.extend(group(orc))
        except Exception as exc:  # a mutant may produce NaN shapes etc.
            fails.append(f"{group.__name__}: raised {exc!r}")
    return fails
