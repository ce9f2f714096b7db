"""Pure-Python brute force of softmax attention for tiny inputs.

Independent of the numpy oracle: nested loops and ``math.exp`` over python
floats, each score exponentiated after subtracting the row maximum.  Used only
to pin the oracle on shapes of a few rows."""
import math


def attention_rows(q, k, v, scale, causal):
    """q: list of Nq rows, k/v: lists of Nk rows (python floats).
    Returns (o rows, lse list).  Causal: query i sees keys 0..i (Nq == Nk)."""
    out, lses = [], []
    for i, qi in enumerate(q):
        scores = []
        for j, kj in enumerate(k):
            if causal and j > i:
                continue
            dot = 0.0
            for a, b in zip(qi, kj):
                dot += a * b
            scores.append((j, scale * dot))
        mx = max(s for _, s in scores)
        weights = [(j, math.exp(s - mx)) for j, s in scores]
        total = sum(w for _, w in weights)
        row = [0.0] * len(v[0])
        for j, w in weights:
            for c in range(len(row)):
                row[c] += w / total * v[j][c]
        out.append(row)
        lses.append(mx + math.log(total))
    return out, lses


def attention_rows_pred(q, k, v, scale, sees):
    """Like attention_rows, with visibility given by a predicate sees(i, j).
    A query that sees no key gets a zero row and lse = -inf."""
    out, lses = [], []
    for i, qi in enumerate(q):
        scores = []
        for j, kj in enumerate(k):
            if not sees(i, j):
                continue
            dot = 0.0
            for a, b in zip(qi, kj):
                dot += a * b
            scores.append((j, scale * dot))
        row = [0.0] * len(v[0])
        if not scores:
            out.append(row)
            lses.append(float("-inf"))
            continue
        mx = max(s for _, s in scores)
        weights = [(j, math.exp(s - mx)) for j, s in scores]
        total = sum(w for _, w in weights)
        for j, w in weights:
            for c in range(len(row)):
                row[c] += w / total * v[j][c]
        out.append(row)
        lses.append(mx + math.log(total))
    return out, lses
