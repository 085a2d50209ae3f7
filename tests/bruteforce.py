"""Pure-Python brute force for tiny paged attention cases (an oracle pin).

Written independently of the C oracle: nested Python loops, math.exp, no
numpy arithmetic. Positions are read through the block table one token at a
time; nothing is gathered. Only for contexts of a few dozen tokens.
"""

import math


def _f(x):
    return float(x)


def attend(k_cache, v_cache, q, block_tables, context_lens, scale, widen):
    """q: [B][nq][Hq][D] (nested sequences or arrays); caches [Hkv][NB][bs][D].

    ``widen`` maps one stored element to a Python float exactly.
    Returns nested lists [B][nq][Hq][D] of floats.
    """
    hkv = len(k_cache)
    bs = len(k_cache[0][0])
    batch = len(q)
    out = []
    for b in range(batch):
        nq = len(q[b])
        hq_n = len(q[b][0])
        group = hq_n // hkv
        L = int(context_lens[b])
        rows_b = []
        for i in range(nq):
            last = L - nq + i  # query i sits here and sees positions <= last
            rows_i = []
            for hq in range(hq_n):
                h = hq // group
                qv = [widen(x) for x in q[b][i][hq]]
                D = len(qv)
                if last < 0:
                    rows_i.append([0.0] * D)
                    continue
                scores = []
                for t in range(last + 1):
                    blk = int(block_tables[b][t // bs])
                    kr = k_cache[h][blk][t % bs]
                    scores.append(scale * math.fsum(qv[d] * widen(kr[d]) for d in range(D)))
                m = max(scores)
                w = [math.exp(s - m) for s in scores]
                z = math.fsum(w)
                o = []
                for d in range(D):
                    acc = []
                    for t in range(last + 1):
                        blk = int(block_tables[b][t // bs])
                        acc.append(w[t] * widen(v_cache[h][blk][t % bs][d]))
                    o.append(math.fsum(acc) / z)
                rows_i.append(o)
            rows_b.append(rows_i)
        out.append(rows_b)
    return out
