"""Write the golden fixtures in this folder from closed forms.

Each fixture is a small, hand-built problem whose output follows from the
definition of the op by a few lines of algebra, written out below case by case
(the valid slots of every token are listed by hand, not computed).  The closed
forms are evaluated with mpmath at 50 digits and stored as decimal strings;
nothing here calls the oracle or the CUDA library.

Definition used ("Sparse MLA training backward", aiter PR #4766, section
"Contract" and the review notes on the sink-inclusive lse and the all-invalid
row; "Tuned sparse MLA prefill for DSv4.1-Flash TP4; fix attn_sink in Triton
fallback", aiter PR #6002, description items "attn_sink", "int64 indices" and
"Invalid KV rows"): over the slots j whose index r_j lies in [0, num_kv),

    O   = sum_j e^{s_j} kv[r_j] / (sum_j e^{s_j} + e^{sink})
    lse = ln(sum_j e^{s_j} + e^{sink}),      s_j = scale <q, kv[r_j]>,

without the e^{sink} terms when there is no sink; a token with no valid slot
has O = 0 and lse = sink (-inf without a sink).

Run ``python tests/golden/make_golden.py`` to rewrite the JSON files.
"""
from __future__ import annotations

import json
import os

import mpmath as mp
import numpy as np

mp.mp.dps = 50
HERE = os.path.dirname(os.path.abspath(__file__))
D = 512
# 1/sqrt(512) rounded to fp32: the value both the kernels and the oracle are given
SCALE = float(np.float32(1.0 / np.sqrt(512.0)))
CITE = ("'Sparse MLA training backward' (aiter PR #4766): section 'Contract'; review notes on "
        "the sink-inclusive lse and on the all-invalid row. 'Tuned sparse MLA prefill for "
        "DSv4.1-Flash TP4; fix attn_sink in Triton fallback' (aiter PR #6002): description "
        "items 'attn_sink', 'int64 indices', 'Invalid KV rows'.")


def _s(x) -> str:
    return mp.nstr(x, 20, min_fixed=-30, max_fixed=30) if x != 0 else "0"


def _write(name, fx):
    with open(os.path.join(HERE, name + ".json"), "w") as f:
        json.dump(fx, f, indent=None, separators=(",", ":"))
        f.write("\n")


def uniform_scores():
    """Every score is exactly 0: q lives in dims 0..255, every kv row in 256..511.

    With n valid slots (counted with multiplicity) over the multiset R of rows,
    den = n + e^{sink}, O = sum_{r in R} kv[r] / den, lse = ln(den); with no
    valid slot O = 0 and lse = sink.  Pins: the validity rule (-1, num_kv, the
    int32 maximum, other negatives), duplicates counted per slot, the sink in
    the denominator only.
    """
    T, H, N, K = 4, 16, 8, 6
    q = [[t, h, (t * 16 + h) % 256, 1.0] for t in range(T) for h in range(H)]
    kv = []
    for r in range(N):
        kv.append([r, 256 + r, float(r + 1)])
        kv.append([r, 511, 0.5 * r - 1.0])
    idx = [[0, 1, 2, 3, -1, 8],
           [5, 5, 5, -1, -1, -1],
           [-1, -1, -1, -1, -1, -1],
           [7, 2147483647, 6, 0, 1, -5]]
    # valid rows of each token, read off by hand (with multiplicity)
    rows = [{0: 1, 1: 1, 2: 1, 3: 1}, {5: 3}, {}, {7: 1, 6: 1, 0: 1, 1: 1}]
    sink = [(h - 8) / 4.0 for h in range(H)]
    kvd = {}
    for r, d, v in kv:
        kvd[(r, d)] = mp.mpf(v)
    lse, O = [], []
    for t in range(T):
        n = sum(rows[t].values())
        lt = []
        for h in range(H):
            es = mp.e ** mp.mpf(sink[h])
            if n == 0:
                lt.append(_s(mp.mpf(sink[h])))
                continue
            den = n + es
            lt.append(_s(mp.log(den)))
            acc = {}
            for r, c in rows[t].items():
                for (rr, d), v in kvd.items():
                    if rr == r:
                        acc[d] = acc.get(d, 0) + c * v
            for d in sorted(acc):
                if acc[d] != 0:
                    O.append([t, h, d, _s(acc[d] / den)])
        lse.append(lt)
    return dict(name="uniform_scores", cite=CITE, derivation=uniform_scores.__doc__.strip(),
                T=T, H=H, num_kv=N, topk=K, index_dtype="int32", scale=SCALE,
                q=q, kv=kv, idx=idx, sink=sink, expected=dict(lse=lse, O=O))


def two_level_scores():
    """Five kv rows with one or two non-zero dims; 128 heads; int64 slots; no sink.

    kv[0] = 2 e_0, kv[1] = -2 e_1, kv[2] = e_2, kv[3] = -1.5 e_3,
    kv[4] = e_300 + 0.5 e_511; q[t, h] = a e_0 + b e_1 + c e_300, so
    s_0 = 2 scale a, s_1 = -2 scale b, s_2 = s_3 = 0, s_4 = scale c.  With slot
    counts c_r, den = sum_r c_r e^{s_r}, lse = ln(den) and
    O = (2 c_0 e^{s_0} e_0 - 2 c_1 e^{s_1} e_1 + c_2 e_2 - 1.5 c_3 e_3
         + c_4 e^{s_4} (e_300 + 0.5 e_511)) / den.
    Token 1 holds 2^32 + 1 (row 1 if cut to 32 bits) and token 2 holds 2^40 + 2
    (row 2 if cut): both are invalid at full width.
    """
    T, H, N, K = 3, 128, 5, 7
    kvl = [[0, 0, 2.0], [1, 1, -2.0], [2, 2, 1.0], [3, 3, -1.5], [4, 300, 1.0], [4, 511, 0.5]]
    idx = [[0, 1, 2, 3, 4, -1, 5],
           [4, 0, 0, 4294967297, -1, 2147483647, 3],
           [-1, -1, 1099511627778, 2, -1, -7, -1]]
    counts = [[1, 1, 1, 1, 1], [2, 0, 0, 1, 1], [0, 0, 1, 0, 0]]   # read off by hand

    def abc(t, h):
        sgn = 1 if t % 2 == 0 else -1
        return 4 * ((h % 16) - 8) * sgn, 4 * ((h // 16) - 4), 8 * ((h % 5) - 2)

    q = []
    for t in range(T):
        for h in range(H):
            for d, v in zip((0, 1, 300), abc(t, h)):
                if v:
                    q.append([t, h, d, float(v)])
    sc = mp.mpf(SCALE)
    lse, O = [], []
    for t in range(T):
        c = counts[t]
        lt = []
        for h in range(H):
            a, b, g = abc(t, h)
            e0, e1, e4 = mp.e ** (2 * sc * a), mp.e ** (-2 * sc * b), mp.e ** (sc * g)
            den = c[0] * e0 + c[1] * e1 + c[2] + c[3] + c[4] * e4
            lt.append(_s(mp.log(den)))
            for d, v in ((0, 2 * c[0] * e0), (1, -2 * c[1] * e1), (2, mp.mpf(c[2])),
                         (3, mp.mpf(-1.5) * c[3]), (300, c[4] * e4), (511, mp.mpf(0.5) * c[4] * e4)):
                if v != 0:
                    O.append([t, h, d, _s(v / den)])
        lse.append(lt)
    return dict(name="two_level_scores", cite=CITE, derivation=two_level_scores.__doc__.strip(),
                T=T, H=H, num_kv=N, topk=K, index_dtype="int64", scale=SCALE,
                q=q, kv=kvl, idx=idx, sink=None, expected=dict(lse=lse, O=O))


def large_scores():
    """Scores of about +-181 and sinks from -1e4 to 300 (far outside fp32's exp range).

    kv[0] = 2 e_0, kv[1] = 1.875 e_0 + e_1, kv[2] = e_0 + e_256.  Head h uses
    pattern p = h % 8 with q[h] = a_p e_0 + b_p e_256, so s_0 = 2 scale a,
    s_1 = 1.875 scale a, s_2 = scale (a + b); with counts c_r and sink z,
    den = sum_r c_r e^{s_r} + e^z, lse = ln(den),
    O = ((2 c_0 e^{s_0} + 1.875 c_1 e^{s_1} + c_2 e^{s_2}) e_0 + c_1 e^{s_1} e_1
         + c_2 e^{s_2} e_256) / den.
    Token 2 has no valid slot: O = 0, lse = z.  In every pattern the top score's
    row also holds the largest part of the score in each half of the head dim.
    """
    T, H, N, K = 3, 128, 3, 4
    kvl = [[0, 0, 2.0], [1, 0, 1.875], [1, 1, 1.0], [2, 0, 1.0], [2, 256, 1.0]]
    pat = [(2048, 0, -1e4), (2048, 0, 0.0), (2048, 0, 181.0), (2048, 0, 300.0),
           (-2048, 0, -1e4), (-2048, 2048, -1e4), (0, 2048, 0.0), (-1024, 0, 0.0)]
    idx = [[0, 1, 2, -1], [2, 2, 0, 5], [-1, 3, 2147483647, -2147483648]]
    counts = [[1, 1, 1], [1, 0, 2], [0, 0, 0]]   # read off by hand
    q = []
    for t in range(T):
        for h in range(H):
            a, b, _ = pat[h % 8]
            if a:
                q.append([t, h, 0, float(a)])
            if b:
                q.append([t, h, 256, float(b)])
    sink = [pat[h % 8][2] for h in range(H)]
    sc = mp.mpf(SCALE)
    lse, O = [], []
    for t in range(T):
        c = counts[t]
        lt = []
        for h in range(H):
            a, b, z = pat[h % 8]
            if sum(c) == 0:
                lt.append(_s(mp.mpf(z)))
                continue
            e0, e1, e2 = mp.e ** (2 * sc * a), mp.e ** (mp.mpf(1.875) * sc * a), mp.e ** (sc * (a + b))
            den = c[0] * e0 + c[1] * e1 + c[2] * e2 + mp.e ** mp.mpf(z)
            lt.append(_s(mp.log(den)))
            for d, v in ((0, 2 * c[0] * e0 + mp.mpf(1.875) * c[1] * e1 + c[2] * e2),
                         (1, c[1] * e1), (256, c[2] * e2)):
                if v != 0:
                    O.append([t, h, d, _s(v / den)])
        lse.append(lt)
    return dict(name="large_scores", cite=CITE, derivation=large_scores.__doc__.strip(),
                T=T, H=H, num_kv=N, topk=K, index_dtype="int32", scale=SCALE,
                q=q, kv=kvl, idx=idx, sink=sink, expected=dict(lse=lse, O=O))


if __name__ == "__main__":
    for fx in (uniform_scores(), two_level_scores(), large_scores()):
        _write(fx["name"], fx)
        print("wrote", fx["name"])
