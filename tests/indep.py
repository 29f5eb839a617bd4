"""Independent restatements used to pin the oracle (tests only).

Nothing here is called by the oracle or by the CUDA path.  Each routine states
the same quantity in a different form than the oracle does, so that a slip in
either one shows up as a disagreement:

* ``brute_force_tree`` -- enumerate every lattice path and sort the lot by the
  recursive total order; the best-first tree is the first N paths.
* ``gdn_expand`` -- the gated delta rule unrolled along a root path:
  h_x = A_x h0 + sum_{a on path(x)} decay(a -> x) k_a c_a^T with
  c_a = beta_a v_a - alpha_a beta_a h_{parent(a)}^T k_a, A_x the product of
  alpha over path(x), and decay(a -> x) the product of alpha over the nodes of
  path(x) after a.  No dk x dv state is ever updated in place.
* ``plain_chain_verify`` -- classic speculative verification of a chain of
  drafts (accept while draft_i equals the argmax of the previous row).
* ``rejection_outcomes`` -- the exact law of a stochastic tree verification
  under the literal rejection rule of the speculative-decoding tutorial
  (section 2.3): keep a draft x with probability min(1, p(x) / q(x)), else go
  on with max(0, p - q) renormalised, each draft being a fixed token (q a
  point mass).  Outcomes are enumerated exactly, in float64.
"""
from __future__ import annotations

import functools

import numpy as np


def canonical_order(sc_row):
    return sorted(range(len(sc_row)), key=lambda i: (-float(sc_row[i]), i))


def brute_force_tree(tok, sc, root, N):
    """tok int [m][K], sc f32 [m][K] (all <= 0) -> dict of tree arrays."""
    m, K = tok.shape
    order = [canonical_order(sc[s]) for s in range(m)]
    paths = {}

    def walk(prefix, score):
        d = len(prefix)
        if d == m:
            return
        for r in range(K):
            s = np.float32(score + np.float32(sc[d][order[d][r]]))
            p = prefix + (r,)
            paths[p] = s
            walk(p, s)

    walk((), np.float32(0.0))

    def cmp(a, b):
        if a == b:
            return 0
        sa, sb = paths[a], paths[b]
        if sa != sb:
            return -1 if sa > sb else 1
        if len(a) != len(b):
            return -1 if len(a) < len(b) else 1
        if a[:-1] != b[:-1]:
            return cmp(a[:-1], b[:-1])
        return -1 if a[-1] < b[-1] else 1

    ordered = sorted(paths, key=functools.cmp_to_key(cmp))[:N]
    index = {(): 0}
    for i, p in enumerate(ordered):
        index[p] = i + 1
    T = N + 1
    out = dict(node_tok=np.full(T, -1, np.int32), node_parent=np.full(T, -1, np.int32),
               node_depth=np.full(T, -1, np.int32), node_rank=np.full(T, -1, np.int32),
               node_score=np.zeros(T, np.float32), node_anc=np.zeros((T, 2), np.uint64))
    out["node_tok"][0] = root
    out["node_depth"][0] = 0
    out["node_anc"][0, 0] = 1
    for p in ordered:
        n = index[p]
        assert p[:-1] in index and index[p[:-1]] < n, "prefix must precede the path"
        par = index[p[:-1]]
        d = len(p)
        out["node_tok"][n] = tok[d - 1][order[d - 1][p[-1]]]
        out["node_parent"][n] = par
        out["node_depth"][n] = d
        out["node_rank"][n] = p[-1]
        out["node_score"][n] = paths[p]
        out["node_anc"][n] = out["node_anc"][par]
        out["node_anc"][n, n // 64] |= np.uint64(1) << np.uint64(n % 64)
    out["n_nodes"] = len(ordered) + 1
    return out


def brute_force_ragged(tok, sc, root, N, m_req, budget):
    """A batch sharing a node budget, by brute force: every root path of every
    request (depth <= m_req[b]) sorted by (score desc, request asc, then the
    recursive tree order); paths are taken in that order while their request
    holds fewer than N drafts and fewer than `budget` drafts are taken in all.
    tok int [B][m][K], sc f32 [B][m][K] -> dict of batched tree arrays."""
    B = tok.shape[0]
    per = []
    for b in range(B):
        t = brute_force_tree(tok[b][: m_req[b]], sc[b][: m_req[b]], root[b],
                             sum(tok.shape[2] ** d for d in range(1, m_req[b] + 1)))
        per.append(t)
    # all draft nodes of all full trees, in the global order
    allp = []
    for b in range(B):
        t = per[b]
        for i in range(1, int(t["n_nodes"])):
            allp.append((-float(t["node_score"][i]), b, i))
    allp.sort()
    take = [0] * B
    used = 0
    for _, b, i in allp:
        if budget >= 0 and used >= budget:
            break
        if take[b] >= N:
            continue
        assert i == take[b] + 1, "a request's drafts are taken in its own order"
        take[b] += 1
        used += 1
    T = N + 1
    out = dict(node_tok=np.full((B, T), -1, np.int32), node_parent=np.full((B, T), -1, np.int32),
               node_depth=np.full((B, T), -1, np.int32), node_rank=np.full((B, T), -1, np.int32),
               node_score=np.zeros((B, T), np.float32), node_anc=np.zeros((B, T, 2), np.uint64),
               n_nodes=np.zeros(B, np.int32))
    for b in range(B):
        n = take[b] + 1
        for k in ("node_tok", "node_parent", "node_depth", "node_rank", "node_score", "node_anc"):
            out[k][b, :n] = per[b][k][:n]
        out["n_nodes"][b] = n
    return out


def brute_force_markov(tok, base, W1, W2, root, N, edges):
    """Best-first tree with parent-dependent edges, by brute force: every root
    path (a sequence of ranks, each rank taken among the children of the path's
    last node under that node's token), sorted by the recursive total order.
    edges(x, d) -> fp32 edge scores of position d's candidates under token x.
    tok int [m][K], base f32 [m][K]."""
    m, K = tok.shape
    paths = {}

    def children(x, d):
        e = edges(x, d)
        order = sorted(range(K), key=lambda i: (-float(e[i]), i))
        return [(int(tok[d][i]), np.float32(e[i])) for i in order]

    def walk(prefix, x, score):
        d = len(prefix)
        if d == m:
            return
        for r, (t, e) in enumerate(children(x, d)):
            s = np.float32(score + e)
            p = prefix + (r,)
            paths[p] = (s, t)
            walk(p, t, s)

    walk((), int(root), np.float32(0.0))

    def cmp(a, b):
        if a == b:
            return 0
        sa, sb = paths[a][0], paths[b][0]
        if sa != sb:
            return -1 if sa > sb else 1
        if len(a) != len(b):
            return -1 if len(a) < len(b) else 1
        if a[:-1] != b[:-1]:
            return cmp(a[:-1], b[:-1])
        return -1 if a[-1] < b[-1] else 1

    ordered = sorted(paths, key=functools.cmp_to_key(cmp))[:N]
    index = {(): 0}
    for i, p in enumerate(ordered):
        index[p] = i + 1
    T = N + 1
    out = dict(node_tok=np.full(T, -1, np.int32), node_parent=np.full(T, -1, np.int32),
               node_depth=np.full(T, -1, np.int32), node_rank=np.full(T, -1, np.int32),
               node_score=np.zeros(T, np.float32), node_anc=np.zeros((T, 2), np.uint64))
    out["node_tok"][0] = root
    out["node_depth"][0] = 0
    out["node_anc"][0, 0] = 1
    for p in ordered:
        n = index[p]
        par = index[p[:-1]]
        out["node_tok"][n] = paths[p][1]
        out["node_parent"][n] = par
        out["node_depth"][n] = len(p)
        out["node_rank"][n] = p[-1]
        out["node_score"][n] = paths[p][0]
        out["node_anc"][n] = out["node_anc"][par]
        out["node_anc"][n, n // 64] |= np.uint64(1) << np.uint64(n % 64)
    out["n_nodes"] = len(ordered) + 1
    return out


def root_path(parent, n):
    p = []
    while n >= 0:
        p.append(int(n))
        n = parent[n]
    return p[::-1]


def gdn_expand(parent, n_nodes, h0, q, k, v, alpha, beta):
    """One request.  h0 [Hv][dk][dv], q/k [T][Hk][dk], v [T][Hv][dv],
    alpha/beta [T][Hv] (any float type, computed in float64).
    Returns (o [T][Hv][dv], states dict node -> [Hv][dk][dv])."""
    h0 = np.asarray(h0, np.float64)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    alpha = np.asarray(alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    T = q.shape[0]
    Hv, dk, dv = h0.shape
    Hk = q.shape[1]
    grp = Hv // Hk
    o = np.zeros((T, Hv, dv))
    states = {}
    for j in range(Hv):
        i = j // grp
        Pk = h0[j].T @ k[:, i, :].T          # [dv][T]
        Pq = h0[j].T @ q[:, i, :].T
        c = np.zeros((T, dv))
        for x in range(n_nodes):
            path = root_path(parent, x)
            anc = path[:-1]

            def decay(a, upto):
                # product of alpha over the nodes of `upto` strictly after a
                sl = upto[upto.index(a) + 1:]
                return float(np.prod([alpha[z, j] for z in sl])) if sl else 1.0

            A_par = float(np.prod([alpha[z, j] for z in anc])) if anc else 1.0
            u = A_par * Pk[:, x]
            for a in anc:
                u = u + decay(a, anc) * float(k[a, i] @ k[x, i]) * c[a]
            c[x] = beta[x, j] * v[x, j] - alpha[x, j] * beta[x, j] * u
            A_x = A_par * alpha[x, j]
            ox = A_x * Pq[:, x]
            for a in path:
                ox = ox + decay(a, path) * float(k[a, i] @ q[x, i]) * c[a]
            o[x, j] = ox
            st = A_x * h0[j]
            for a in path:
                st = st + decay(a, path) * np.outer(k[a, i], c[a])
            states.setdefault(x, np.zeros((Hv, dk, dv)))[j] = st
    return o, states


def plain_chain_verify(root_tok, drafts, argmax_rows):
    """Chain speculative verification: row 0 is the root, row i the i-th draft.
    Accept draft i+1 while it equals argmax of row i; return (tau, out_tok)."""
    out = []
    row = 0
    for i, d in enumerate(drafts):
        if d != argmax_rows[row]:
            break
        out.append(int(d))
        row = i + 1
    out.append(int(argmax_rows[row]))
    return len(out), out


def rejection_outcomes(node_tok, node_parent, n_nodes, p_rows, m):
    """Exact law of (accepted draft tokens..., bonus) under the rejection rule.

    At the current node the target distribution is p = p_rows[node]; its
    children are tried in node order.  Child x (a fixed draft, so q = one-hot
    at x) is kept with probability min(1, p(x) / q(x)) = p(x); if it is not,
    p becomes max(0, p - q) renormalised, i.e. x removed.  When no child is
    kept, the bonus is drawn from the final p.  Returns {tuple: probability}.
    """
    children = {}
    for c in range(1, int(n_nodes)):
        children.setdefault(int(node_parent[c]), []).append(c)
    out = {}

    def visit(node, depth, prefix, weight):
        p = np.array(p_rows[node], dtype=np.float64)
        p = p / p.sum()
        for c in (children.get(node, []) if depth < m else []):
            x = int(node_tok[c])
            keep = min(1.0, p[x] / 1.0)
            if keep > 0:
                visit(c, depth + 1, prefix + (x,), weight * keep)
            q = np.zeros_like(p)
            q[x] = 1.0
            r = np.maximum(0.0, p - q)
            if r.sum() == 0:
                return
            p = r / r.sum()
            weight = weight * (1.0 - keep)
        for y in range(len(p)):
            if p[y] > 0:
                key = prefix + (y,)
                out[key] = out.get(key, 0.0) + weight * p[y]

    visit(0, 0, (), 1.0)
    return out
