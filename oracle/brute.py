"""Pure-Python scalar twin of the oracle, for tiny inputs only.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every key set is
decided here by testing each key against a membership predicate, an
independent route to the index lists that ``headcast_ref`` builds, so the
two agreeing pins both.  Sources as in ``headcast_ref``: the Pith review of
"HeadCast: Casting Attention Heads for Efficient Autoregressive Video
Generation" ("What carries the argument", major comment 2, the free-parameter
ledger and the Figure 3 caption).
"""
import math


def attend_one(qv, keys, values, scale):
    """softmax(q . k_j * scale) weighted sum of v_j, with plain loops."""
    scores = [scale * sum(a * b for a, b in zip(qv, kv)) for kv in keys]
    m = max(scores)
    e = [math.exp(s - m) for s in scores]
    z = sum(e)
    d = len(values[0])
    return [sum(e[j] * values[j][c] for j in range(len(keys))) / z for c in range(d)]


def position(t, frame_h, frame_w):
    f, rem = divmod(t, frame_h * frame_w)
    return f, rem // frame_w, rem % frame_w


def in_proxy(qh, qw, kh, kw, r):
    """Chebyshev neighbourhood of radius r (clipping is implicit: only keys
    that exist are tested)."""
    return abs(kh - qh) <= r and abs(kw - qw) <= r


def axis_cell(x, n, cell):
    """Index of x's cell along an axis of length n: cells of ``cell``, the
    last absorbing the remainder, n_cells = max(1, round-half-up(n/cell))."""
    n_cells = max(1, int(n / cell + 0.5))
    return min(x // cell, n_cells - 1)


def in_cell(qh, qw, kh, kw, frame_h, frame_w, cell_h, cell_w):
    return (axis_cell(qh, frame_h, cell_h) == axis_cell(kh, frame_h, cell_h) and
            axis_cell(qw, frame_w, cell_w) == axis_cell(kw, frame_w, cell_w))


def in_sliding(qh, qw, kh, kw, cell_h, cell_w):
    """Window of cell_h x cell_w keys with the query at offset (cell_h//2,
    cell_w//2) from its top-left corner."""
    return 0 <= kh - qh + cell_h // 2 < cell_h and 0 <= kw - qw + cell_w // 2 < cell_w


def keyset_outputs(q, k, v, head, frame_h, frame_w, block_tokens, kind, scale,
                   radius=2, cell_h=10, cell_w=10):
    """Outputs of one head for every query, over the key set ``kind``:
    'full', 'sink' (window's first block), 'dummy' (last block), 'proxy',
    'cell', 'sliding'.  q, k, v are nested lists or arrays [tokens][H][d]."""
    nk = len(k)
    out = []
    for i in range(len(q)):
        _, qh, qw = position(i, frame_h, frame_w)
        sel = []
        for j in range(nk):
            _, kh, kw = position(j, frame_h, frame_w)
            if kind == "full":
                ok = True
            elif kind == "sink":
                ok = j < block_tokens
            elif kind == "dummy":
                ok = j >= nk - block_tokens
            elif kind == "proxy":
                ok = in_proxy(qh, qw, kh, kw, radius)
            elif kind == "cell":
                ok = in_cell(qh, qw, kh, kw, frame_h, frame_w, cell_h, cell_w)
            elif kind == "sliding":
                ok = in_sliding(qh, qw, kh, kw, cell_h, cell_w)
            else:
                raise ValueError(kind)
            if ok:
                sel.append(j)
        out.append(attend_one([float(x) for x in q[i][head]],
                              [[float(x) for x in k[j][head]] for j in sel],
                              [[float(x) for x in v[j][head]] for j in sel], scale))
    return out


def cosine(a, b):
    na = math.sqrt(sum(x * x for x in a))
    nb = math.sqrt(sum(x * x for x in b))
    if na == 0.0 and nb == 0.0:
        return 1.0
    if na == 0.0 or nb == 0.0:
        return 0.0
    return sum(x * y for x, y in zip(a, b)) / (na * nb)
