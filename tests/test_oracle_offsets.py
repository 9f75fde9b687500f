"""Pins of the oracle's offset tables and schedules (CPU only).

Each check ties the oracle to something other than itself: values printed on the
pages (tests/golden/pages_values.json), Binet's closed form, decimal-module
arithmetic, or brute force.
"""
import math
from decimal import Decimal, ROUND_HALF_UP, localcontext
from fractions import Fraction

import pytest

import oracle
from oracle import schedule as S


def binet(n):
    phi = (1 + 5 ** 0.5) / 2
    return round(phi ** n / 5 ** 0.5)


def test_fibonacci_base_matches_printed_list(golden):
    fib = S.fibonacci_base()
    head = golden["fib_printed_head"]["value"]
    ends = golden["fib_printed_list_ends"]["value"]
    assert fib[: len(head)] == head
    assert fib[:4] == ends["first"]
    assert fib[-1] == ends["last"]
    assert len(fib) == 15


def test_fibonacci_base_matches_binet():
    # Fib(n) = round(phi^n / sqrt 5); the printed list is Fib(2) .. Fib(16).
    assert S.fibonacci_base() == [binet(n) for n in range(2, 17)]
    # base_max extends the list by the same closed form
    ext = S.fibonacci_base(base_max=10 ** 6)
    assert ext == [binet(n) for n in range(2, 2 + len(ext))]
    assert ext[-1] <= 10 ** 6 < binet(2 + len(ext))


def test_linear_stagger_endpoints_pages(golden):
    g = golden["linear_stagger_endpoints"]["value"]
    L = g["n_layers"]
    a0, a1 = Fraction(*g["layer0"]), Fraction(*g["layer15"])
    al = [S.alpha_for_layer(S.LINEAR, l, L, alpha_min=a0, alpha_max=a1) for l in range(L)]
    assert al[0] == a0 and al[L - 1] == a1
    # linear: constant step (a1 - a0) / (L - 1)
    steps = {al[i + 1] - al[i] for i in range(L - 1)}
    assert steps == {(a1 - a0) / (L - 1)}
    rng = golden["alpha_range"]["value"]
    assert min(al) == Fraction(*rng["min"]) and max(al) == Fraction(*rng["max"])


def test_coprime_is_permutation_of_linear_multiset(golden):
    g = golden["coprime_step"]["value"]
    c, L = g["c"], g["n_layers"]
    for (amin, amax) in [(Fraction(1, 2), Fraction(3, 2)), (Fraction(1, 2), Fraction(2))]:
        lin = [S.alpha_for_layer(S.LINEAR, l, L, alpha_min=amin, alpha_max=amax) for l in range(L)]
        for cc in (c, 5, 3, 1):
            cop = [S.alpha_for_layer(S.COPRIME, l, L, alpha_min=amin, alpha_max=amax, coprime_c=cc)
                   for l in range(L)]
            assert sorted(cop) == sorted(lin)
        # layer l takes the ramp value of layer (7 l mod 16): layer 1 -> ramp 7, layer 2 -> ramp 14
        cop = [S.alpha_for_layer(S.COPRIME, l, L, alpha_min=amin, alpha_max=amax, coprime_c=c)
               for l in range(L)]
        assert cop[0] == lin[0] and cop[1] == lin[7] and cop[2] == lin[14] and cop[3] == lin[5]


def test_coprime_spreads_adjacent_layers(golden):
    # The pages' stated purpose of the coprime jump: larger spacing differences between
    # adjacent layers than the plain ramp has.
    g = golden["coprime_step"]["value"]
    L = g["n_layers"]
    lin = [S.alpha_for_layer(S.LINEAR, l, L) for l in range(L)]
    cop = [S.alpha_for_layer(S.COPRIME, l, L, coprime_c=g["c"]) for l in range(L)]
    d_lin = min(abs(lin[i + 1] - lin[i]) for i in range(L - 1))
    d_cop = min(abs(cop[i + 1] - cop[i]) for i in range(L - 1))
    assert d_cop > d_lin


def test_coprime_rejects_non_coprime_step():
    with pytest.raises(ValueError):
        S.alpha_for_layer(S.COPRIME, 1, 16, coprime_c=4)
    with pytest.raises(ValueError):
        S.alpha_for_layer(S.COPRIME, 1, 16, coprime_c=0)


def test_fixed_alpha_one_table_from_printed_list(golden):
    # alpha = 1: the table is just the printed list cut to [W, T-1].
    ends = golden["fib_printed_list_ends"]["value"]
    fib = S.fibonacci_base()
    for (W, T) in [(16, 256), (64, 1024), (64, 4096), (12, 1024), (6, 8)]:
        tab = S.offset_table(S.FIB, Fraction(1), W, T)
        assert tab == [f for f in fib if W <= f <= T - 1]
    assert S.offset_table(S.FIB, Fraction(1), 16, 256) == [21, 34, 55, 89, 144, 233]
    assert S.offset_table(S.FIB, Fraction(1), 64, 1024) == [89, 144, 233, 377, 610, ends["last"]]
    # the Fibonacci list is not extended past 987 at 4x length
    assert max(S.offset_table(S.FIB, Fraction(1), 64, 4096)) == ends["last"]


def _decimal_table(base_vals, alpha_dec, W, T):
    out = set()
    for f in base_vals:
        o = int((alpha_dec * f).quantize(Decimal(1), rounding=ROUND_HALF_UP))
        if W <= o <= T - 1:
            out.add(o)
    return sorted(out)


@pytest.mark.parametrize("T", [1024, 4096])
@pytest.mark.parametrize("amax", ["1.5", "2.0"])
def test_linear_tables_match_decimal_half_up(T, amax):
    # Independent arithmetic: alpha_l = 0.5 + (amax - 0.5) * l / 15 in 60-digit decimal,
    # rounded half up by `decimal`. A rational with denominator dividing 30 is never
    # within 1e-50 of a half-integer unless it is one, so the decimal rounding is exact.
    with localcontext() as ctx:
        ctx.prec = 60
        for l in range(16):
            a = Decimal("0.5") + (Decimal(amax) - Decimal("0.5")) * l / 15
            want = _decimal_table(S.fibonacci_base(), a, 64, T)
            got = S.layer_table(S.FIB, S.LINEAR, l, 16, 64, T, alpha_min=Fraction(1, 2),
                                alpha_max=Fraction(amax))
            assert got == want, (l, a)


def test_half_up_ties_at_the_ramp_ends():
    # Worked by hand: alpha = 1/2: 233/2 = 116.5 -> 117, 377/2 = 188.5 -> 189,
    # 987/2 = 493.5 -> 494 (half up, not half even); alpha = 3/2: 89*1.5 = 133.5 -> 134.
    t0 = S.offset_table(S.FIB, Fraction(1, 2), 64, 4096)
    assert t0 == [72, 117, 189, 305, 494]
    t15 = S.offset_table(S.FIB, Fraction(3, 2), 64, 4096)
    assert 134 in t15 and 350 in t15 and 1481 in t15  # 233*1.5 = 349.5, 987*1.5 = 1480.5


def test_pow2_new_offsets_only_at_4x(golden):
    g = golden["pow2_new_offsets_at_4x"]["value"]
    tr = S.offset_table(S.POW2, Fraction(1), 64, g["train_T"])
    ev = S.offset_table(S.POW2, Fraction(1), 64, g["eval_T"])
    assert tr == [64, 128, 256, 512]
    assert sorted(set(ev) - set(tr)) == g["new_offsets"]
    # every entry is a power of two, within [W, T-1]
    assert all(o & (o - 1) == 0 and 64 <= o <= g["eval_T"] - 1 for o in ev)


def test_pow2_scaled_and_capped():
    # alpha = 1/2: 2^k / 2 = 2^(k-1); ties 1/2 -> 1 (not in range anyway)
    assert S.offset_table(S.POW2, Fraction(1, 2), 16, 1024) == [16, 32, 64, 128, 256, 512]
    assert S.offset_table(S.POW2, Fraction(1), 16, 1024, base_max=100) == [16, 32, 64]
    # alpha = 3/2 on powers of two: 1.5 * 2^k
    assert S.offset_table(S.POW2, Fraction(3, 2), 8, 200) == [12, 24, 48, 96, 192]


def test_table_invariants_brute_force():
    for base in (S.FIB, S.POW2):
        for alpha in (Fraction(1, 3), Fraction(1, 2), Fraction(7, 10), Fraction(1), Fraction(3, 2),
                      Fraction(2), Fraction(13, 7)):
            for (W, T) in [(1, 2), (6, 64), (12, 1024), (64, 1024), (64, 4096), (100, 50)]:
                tab = S.offset_table(base, alpha, W, T)
                assert tab == sorted(set(tab))
                assert all(W <= o <= T - 1 for o in tab)
                # brute force: every base value whose rounded offset lands in range is kept
                vals = S.fibonacci_base() if base == S.FIB else [2 ** k for k in range(40)]
                bf = sorted({math.floor(alpha * f + Fraction(1, 2)) for f in vals} &
                            set(range(W, T)))
                assert tab == bf


def test_invalid_alpha_rejected():
    with pytest.raises(ValueError):
        S.offset_table(S.FIB, Fraction(0), 4, 100)
    with pytest.raises(ValueError):
        S.alpha_for_layer(S.FIXED, 3, 2)


def test_key_set_closed_form_count():
    # |S_i| = min(W, i + 1) + #{o in table : o <= i}; keys unique, sorted, causal.
    for (W, T, tab) in [(16, 256, [21, 34, 55, 89, 144, 233]), (6, 100, [8, 13, 21, 34, 55, 89]),
                        (64, 300, []), (1, 40, [1, 2, 3, 5])]:
        for i in range(T):
            ks = S.key_set(i, W, tab)
            assert len(ks) == min(W, i + 1) + sum(1 for o in tab if W <= o <= i)
            assert ks == sorted(set(ks)) and all(0 <= j <= i for j in ks)
            assert oracle.key_set_c(i, W, tab) == ks


def test_key_set_brute_force_predicate():
    W, T, tab = 10, 200, [13, 21, 34, 55, 89, 144]
    for i in range(T):
        bf = [j for j in range(T) if (0 <= i - j < W) or (i - j in tab)]
        assert S.key_set(i, W, tab) == bf


def test_mean_key_set_size_c1():
    # B1 H2 T256 W16 alpha=1: mean |S_i| over queries (regression value 19.28...)
    tab = S.offset_table(S.FIB, Fraction(1), 16, 256)
    m = sum(len(S.key_set(i, 16, tab)) for i in range(256)) / 256
    assert abs(m - (sum(min(16, i + 1) for i in range(256)) +
                    sum(max(0, 256 - o) for o in tab)) / 256) < 1e-12
