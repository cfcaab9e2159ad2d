"""Writes exact_elu1_causal.json: causal kernelized attention with the elu+1
feature map on small positive integer-valued inputs, computed in exact
rational arithmetic (Python fractions).

For x > 0 the elu+1 map is phi(x) = x + 1 exactly (review page "Transformers
are RNNs", main results b2: the elu-based map), so every output
    out_i = sum_{j<=i} (phi(q_i).phi(k_j)) v_j / sum_{j<=i} phi(q_i).phi(k_j)
(proposed method b1-b3: kernel similarity, causal cumulative sums, the sums
include j = i) is a rational number.  The file stores the inputs and the
outputs as exact fractions "p/q".  This script uses neither the oracle nor
the CUDA library; the test compares the oracle against the stored values.

    python tests/golden/make_exact_elu1.py
"""
import json
import os
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))

# two heads, N = 5, D = 3, Dv = 2; positive integers (seeded by hand)
Q = [[[1, 2, 1], [3, 1, 2], [2, 2, 2], [1, 4, 1], [5, 1, 3]],
     [[2, 1, 1], [1, 1, 4], [3, 3, 1], [2, 5, 2], [1, 2, 3]]]
K = [[[2, 1, 3], [1, 1, 1], [4, 2, 1], [1, 3, 2], [2, 2, 5]],
     [[1, 3, 2], [2, 2, 2], [5, 1, 1], [1, 1, 3], [3, 2, 4]]]
V = [[[1, 0], [0, 1], [2, 3], [4, 1], [1, 5]],
     [[3, 1], [1, 2], [0, 4], [2, 2], [5, 1]]]


def phi(x):
    return [Fraction(t) + 1 for t in x]   # elu(x) + 1 for x > 0


def causal(q, k, v):
    out = []
    for i in range(len(q)):
        fq = phi(q[i])
        num = [Fraction(0)] * len(v[0])
        den = Fraction(0)
        for j in range(i + 1):
            w = sum(a * b for a, b in zip(fq, phi(k[j])))
            den += w
            num = [n + w * vj for n, vj in zip(num, v[j])]
        out.append([n / den for n in num])
    return out


def main():
    outs = [causal(Q[h], K[h], V[h]) for h in range(len(Q))]
    doc = {"citation": "Transformers are RNNs (review page), proposed method b1-b3, main results b2",
           "map": "elu1", "causal": True, "B": 1, "H": 2, "N": 5, "D": 3, "Dv": 2,
           "q": Q, "k": K, "v": V,
           "out": [[[f"{x.numerator}/{x.denominator}" for x in row] for row in o] for o in outs]}
    with open(os.path.join(HERE, "exact_elu1_causal.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
