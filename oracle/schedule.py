"""Oracle: offset tables and per-layer alpha schedules, in exact rational arithmetic.

TEST INFRASTRUCTURE ONLY. This package is the slow, obviously correct CPU
statement of what the sparse-attention path computes. Only the tests, the
smoke check and the benchmark's CPU-baseline leg may import it; the product
library never calls it and shares no code with it.

Sources (all from "Depth-Staggered Fibonacci Spacing for Sparse Attention: Static
Schedules Beat Learned Dilation and Extrapolate Where Dense Attention Fails",
as explained on gist.science, Portuguese and French pages, and the aimsg.uk
Chinese summary):
  * Metodologia / Arquitetura e Mecanismo de Atencao, "Conjunto Atendido":
    each query at position i attends a dense local window of size W plus a set
    of sparse offsets from fib = [1, 2, 3, 5, ..., 987].
  * same section, "Escalonamento": each offset f_k is scaled by a per-layer
    scalar alpha, target distance d_k = alpha * f_k.
  * Metodologia / Variaveis Experimentais: Fixo (alpha = 1 in every layer),
    Escalonado Linear (alpha rises linearly from the first to the last layer),
    Escalonado Coprimo/HDC (the same multiset of alphas, reassigned with the
    coprime jump l -> (c*l mod L)).
  * Metodologia / Controles: a reach-matched power-of-two (log-sparse) base.
  * Principais Contribuicoes 3, "Sensibilidade de Base": at 4x the training
    length the power-of-two base gains new large offsets (1024, 2048), i.e. the
    power-of-two list is not capped at the training length.

Readings where the pages are silent (each is listed in the design notes):
  * Fibonacci base = exactly the printed 15 values 1,2,3,...,987, independent
    of the sequence length; `base_max` > 0 replaces the cap 987.
  * power-of-two base = 2^k, k >= 0, every one whose scaled offset still fits
    (o <= T-1); `base_max` > 0 caps the base value.
  * integer offset = alpha*F rounded half up, computed exactly: o = floor(alpha*F + 1/2).
  * linear stagger alpha_l = a_min + (a_max - a_min) * l / (L - 1); L = 1 gives a_min.
  * coprime layer l uses the linear-stagger alpha of layer (c*l mod L).
  * keep only W <= o <= T-1 (smaller offsets lie inside the window, larger
    ones never name a key); the table is a set, ascending.
"""
from __future__ import annotations

from fractions import Fraction
from math import gcd

FIB = "fib"
POW2 = "pow2"
FIXED = "fixed"
LINEAR = "linear"
COPRIME = "coprime"

FIB_CAP = 987  # last value of the printed list fib = [1, 2, 3, 5, ..., 987]


def fibonacci_base(base_max: int = 0):
    """The Fibonacci offsets 1, 2, 3, 5, 8, ... (the leading duplicate 1 is not
    repeated), up to 987 or to `base_max` when that is > 0."""
    cap = FIB_CAP if base_max <= 0 else base_max
    out = []
    a, b = 1, 2
    while a <= cap:
        out.append(a)
        a, b = b, a + b
    return out


def alpha_for_layer(kind: str, layer: int, n_layers: int, alpha=Fraction(1),
                    alpha_min=Fraction(1, 2), alpha_max=Fraction(3, 2), coprime_c: int = 7):
    """Exact alpha of `layer` under the schedule `kind`."""
    if not (0 <= layer < n_layers):
        raise ValueError("layer out of range")
    if kind == FIXED:
        return Fraction(alpha)
    if kind == LINEAR:
        return _linear(layer, n_layers, Fraction(alpha_min), Fraction(alpha_max))
    if kind == COPRIME:
        if coprime_c < 1 or gcd(coprime_c, n_layers) != 1:
            raise ValueError("coprime step must satisfy gcd(c, L) = 1")
        return _linear((coprime_c * layer) % n_layers, n_layers,
                       Fraction(alpha_min), Fraction(alpha_max))
    raise ValueError(kind)


def _linear(layer, n_layers, a_min, a_max):
    if n_layers == 1:
        return a_min
    return a_min + (a_max - a_min) * Fraction(layer, n_layers - 1)


def round_half_up(x: Fraction) -> int:
    """floor(x + 1/2) for an exact rational x."""
    y = x + Fraction(1, 2)
    return y.numerator // y.denominator


def offset_table(base: str, alpha: Fraction, W: int, T: int, base_max: int = 0):
    """Sorted, duplicate-free integer offsets round(alpha*F) with W <= o <= T-1."""
    alpha = Fraction(alpha)
    if alpha <= 0:
        raise ValueError("alpha must be > 0")
    keep = set()
    if base == FIB:
        for f in fibonacci_base(base_max):
            o = round_half_up(alpha * f)
            if W <= o <= T - 1:
                keep.add(o)
    elif base == POW2:
        f = 1
        while True:
            if base_max > 0 and f > base_max:
                break
            o = round_half_up(alpha * f)
            if o > T - 1:
                break
            if o >= W:
                keep.add(o)
            f *= 2
    else:
        raise ValueError(base)
    return sorted(keep)


def layer_table(base, kind, layer, n_layers, W, T, base_max=0, **alpha_kw):
    """Offset table of one layer under a schedule (convenience wrapper)."""
    return offset_table(base, alpha_for_layer(kind, layer, n_layers, **alpha_kw), W, T, base_max)


def key_set(i: int, W: int, table) -> list:
    """Keys attended by query i: the window {j : 0 <= i-j < W, j >= 0} united
    with {i-o : o in table, i-o >= 0}; returned sorted, without duplicates."""
    ks = set(range(max(0, i - W + 1), i + 1))
    for o in table:
        if i - o >= 0:
            ks.add(i - o)
    return sorted(ks)


def frac_bases(alpha: float, base: str, W: int, T: int, base_max: int = 0):
    """The base values F behind frac_distances, in the same order."""
    if not alpha > 0:
        raise ValueError("alpha must be > 0")
    if base == FIB:
        fs = fibonacci_base(base_max)
    elif base == POW2:
        fs, f = [], 1
        while float(alpha) * f <= T - 1 and (base_max <= 0 or f <= base_max):
            fs.append(f)
            f *= 2
    else:
        raise ValueError(f"unknown base {base!r}")
    return [f for f in fs if W <= float(alpha) * f <= T - 1]


def frac_distances(alpha: float, base: str, W: int, T: int, base_max: int = 0):
    """Real offset distances d_k = alpha * F of a fractional ("learned") alpha: the pages'
    learned variant interpolates keys between rows instead of rounding (Metodologia /
    Arquitetura, "Implementacao"). alpha is taken as the given float, the products in
    double precision; kept when W <= d <= T - 1 (the integer rule's interval), ascending."""
    if not alpha > 0:
        raise ValueError("alpha must be > 0")
    if base == FIB:
        fs = fibonacci_base(base_max)
    elif base == POW2:
        fs, f = [], 1
        while float(alpha) * f <= T - 1 and (base_max <= 0 or f <= base_max):
            fs.append(f)
            f *= 2
    else:
        raise ValueError(f"unknown base {base!r}")
    return [float(alpha) * f for f in fs if W <= float(alpha) * f <= T - 1]
