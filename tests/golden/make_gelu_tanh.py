"""Writes gelu_tanh.json: the tanh form of GELU,
0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), evaluated in 50-digit
decimal arithmetic (tanh from its exponential definition, pi by Machin's
formula, square root by Newton's method), independent of any floating-point
library.  The oracle's tanh variant is checked against these values."""

import json
import os
from decimal import Decimal, getcontext

getcontext().prec = 50


def arctan_inv(n: int) -> Decimal:
    # arctan(1/n) by its Taylor series
    x = Decimal(1) / n
    x2 = x * x
    term, total, k = x, x, 1
    while True:
        term *= -x2
        k += 2
        t = term / k
        if abs(t) < Decimal(10) ** -55:
            return total
        total += t


def pi() -> Decimal:
    return 16 * arctan_inv(5) - 4 * arctan_inv(239)   # Machin


def sqrt(v: Decimal) -> Decimal:
    r = Decimal(1)
    for _ in range(200):
        r = (r + v / r) / 2
    return r


def exp(v: Decimal) -> Decimal:
    # exp by range reduction (v / 2^m) and the Taylor series, then squaring
    m = 0
    while abs(v) > 1:
        v /= 2
        m += 1
    term, total, k = Decimal(1), Decimal(1), 0
    while True:
        k += 1
        term = term * v / k
        if abs(term) < Decimal(10) ** -55:
            break
        total += term
    for _ in range(m):
        total *= total
    return total


def tanh(v: Decimal) -> Decimal:
    e2 = exp(2 * v)
    return (e2 - 1) / (e2 + 1)


def gelu_tanh(x: Decimal) -> Decimal:
    c = sqrt(2 / pi())
    return x * (1 + tanh(c * (x + Decimal("0.044715") * x ** 3))) / 2


def main():
    xs = ["-6", "-3.5", "-2", "-1.25", "-0.5", "-0.1", "0", "0.03125", "0.5", "1", "1.75", "2.5", "4", "8"]
    out = {"source": "GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))); 50-digit decimal "
                     "evaluation by tests/golden/make_gelu_tanh.py (Machin's pi, Newton's square root, "
                     "tanh from exp's Taylor series)",
           "values": [[x, str(gelu_tanh(Decimal(x)))] for x in xs]}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "gelu_tanh.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")


if __name__ == "__main__":
    main()
