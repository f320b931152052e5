"""Write closed_form.json: attention cases whose exact answers are rationals.

Construction (exact, no floating point in the expected values): the query is
q_i = (t_i, 0, ...) and the key is k_j = (ln w_j, c_j, ...) with integer
weights w_j, so with scale 1 the score is s_ij = t_i ln w_j and
exp(s_ij) = w_j ** t_i is an integer.  The softmax of the standard-attention
definition (FlashAttention blog, "From Online Softmax to FlashAttention" and
"(Safe) Softmax") then gives P_ij = w_j**t_i / sum_{visible j'} w_j'**t_i,
O_i = sum_j P_ij v_j and LSE_i = ln(sum_{visible j} w_j**t_i), computed here in
Python fractions.  The only rounding on the oracle side is that of ln w_j to
fp64 and of its own arithmetic, so the oracle must match to ~1e-13.

This script calls neither the oracle nor the CUDA library.
Run:  python tests/golden/make_closed_form.py
"""
import json
import math
import os
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))


def case(name, H, Hkv, t, w, c, v, causal):
    """t: [H][N] query exponents; w: [Hkv][N] integer weights; c: [Hkv][N]
    second key channel (ignored by the score since q's second channel is 0);
    v: [Hkv][N][d] integer values.  d = len(v[0][0]) >= 2."""
    N = len(w[0])
    d = len(v[0][0])
    G = H // Hkv
    q = [[[float(t[h][i])] + [0.0] * (d - 1) for i in range(N)] for h in range(H)]
    k = [[[math.log(w[g][j]), float(c[g][j])] + [0.0] * (d - 2) for j in range(N)]
         for g in range(Hkv)]
    o, lse = [], []
    for h in range(H):
        g = h // G
        oh, lh = [], []
        for i in range(N):
            vis = [j for j in range(N) if (not causal or j <= i)]
            ew = {j: Fraction(w[g][j]) ** t[h][i] for j in vis}
            den = sum(ew.values())
            oi = [sum(ew[j] * v[g][j][cc] for j in vis) / den for cc in range(d)]
            oh.append([f"{x.numerator}/{x.denominator}" for x in oi])
            lh.append(f"{den.numerator}/{den.denominator}")  # LSE = ln(this)
        o.append(oh)
        lse.append(lh)
    return {
        "name": name, "B": 1, "H": H, "Hkv": Hkv, "N": N, "d": d,
        "causal": causal, "scale": 1.0,
        "q": [q], "k": [k], "v": [[[[float(x) for x in row] for row in vg] for vg in v]],
        "o_exact": [o], "lse_exp_exact": [lse],
    }


def main():
    cases = [
        case("four_keys_full", 1, 1, [[1, 1, 1, 1]], [[1, 2, 3, 4]], [[5, -1, 2, 0]],
             [[[1, 0], [0, 1], [2, 2], [-1, 3]]], causal=False),
        case("four_keys_causal", 1, 1, [[1, 1, 1, 1]], [[1, 2, 3, 4]], [[5, -1, 2, 0]],
             [[[1, 0], [0, 1], [2, 2], [-1, 3]]], causal=True),
        case("exponents_0_1_2", 1, 1, [[0, 1, 2]], [[2, 3, 5]], [[0, 0, 0]],
             [[[4, 1, 0], [-2, 7, 1], [3, 3, -5]]], causal=False),
        case("gqa_two_heads_causal", 2, 1, [[1, 2, 0, 1], [2, 0, 1, 3]], [[3, 1, 2, 7]],
             [[1, 2, 3, 4]], [[[1, -1], [2, 0], [0, 5], [-3, 2]]], causal=True),
    ]
    src = ("tests/golden/make_closed_form.py: exact rationals from the standard-attention "
           "definition (FlashAttention blog, 'From Online Softmax to FlashAttention', "
           "'(Safe) Softmax'); LSE per FlashAttention-2 review 2 (logsumexp saved)")
    with open(os.path.join(HERE, "closed_form.json"), "w") as f:
        json.dump({"source": src, "cases": cases}, f, indent=1)


if __name__ == "__main__":
    main()
