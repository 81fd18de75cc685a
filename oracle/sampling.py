"""Oracle for the rejection-sampling half of the verify step (fp64).

Follows quant67 "speculative decoding" section 3.1 (accept x_i with
probability min(1, p_i(x_i)/q_i(x_i)); at the first rejection n resample from
max(0, p_n - q_n) / sum(max(0, p_n - q_n)); if all K are accepted draw a bonus
token from p_{K+1}) and "KV Cache + Speculative Decoding" sections 7.1-7.3
and 7.6 (p = target, q = draft, per-position softmax with temperature, the
bonus row is the last target row).

Readings adopted where the pages leave a step open:
  * p = softmax(target_logits / T) and q = softmax(draft_logits / T), or q as
    given when the draft is passed as probabilities.
  * Accept test in multiplicative form: accept x_i iff u_i * q_i(x_i) <
    p_i(x_i). For q_i(x_i) > 0 this is u_i < min(1, p/q) (strict, as in the
    demo's `rand < r`); for q_i(x_i) = 0 it accepts iff p_i(x_i) > 0. The
    1e-9 guards of the demo code are numerical guards, not the definition.
  * Each position carries two uniforms [u_i, v_i]; v_n drives the residual
    draw at the first rejection n, v_{K+1} the bonus draw. u_{K+1} is unused.
  * Inverse CDF in ascending token id with a strict test: y = min{y : C(y) >
    v * C(V-1)}, C the running sum of the weights. Zero-weight tokens can never
    be drawn. If rounding leaves no such y, the largest y with nonzero weight
    is taken. If the residual mass is exactly 0 (impossible in exact
    arithmetic, since a rejection has probability Z), the draw falls back to p_n.
  * Output tokens: x_1 .. x_{n-1}, y, then -1 padding; num_accepted = n - 1
    (0-based: n_rej accepted drafts precede the drawn token).
"""
import numpy as np


def _np64(x):
    import torch
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def softmax(logits, temperature=1.0):
    """softmax(logits / T) over the last axis, fp64, max-subtracted."""
    x = _np64(logits) / float(temperature)
    x = x - x.max(axis=-1, keepdims=True)
    e = np.exp(x)
    return e / e.sum(axis=-1, keepdims=True)


def inverse_cdf(weights, v):
    """Row-wise y = min{y : C(y) > v*Z} with C = running sum in ascending id.

    weights: [N, V] nonnegative fp64; v: [N]. Returns (y, margin, Z) where
    margin is the distance of v from the nearest edge of y's CDF interval,
    as a fraction of Z (the ``CDF boundary'' distance).
    """
    C = np.cumsum(weights, axis=1)
    Z = C[:, -1]
    thr = np.asarray(v, dtype=np.float64) * Z
    above = C > thr[:, None]
    y = np.argmax(above, axis=1)
    none = ~above.any(axis=1)
    if none.any():   # rounding pushed v*Z to the top: largest y with weight
        rev = np.argmax(weights[:, ::-1] > 0, axis=1)
        y = np.where(none, weights.shape[1] - 1 - rev, y)
    rows = np.arange(weights.shape[0])
    c_hi = C[rows, y]
    c_lo = np.where(y > 0, C[rows, np.maximum(y - 1, 0)], 0.0)
    with np.errstate(divide="ignore", invalid="ignore"):
        margin = np.minimum(thr - c_lo, c_hi - thr) / Z
    return y, np.abs(margin), Z


def top_p_nucleus(logits, top_p, temperature=1.0):
    """The top-p set of softmax(logits / T) of every row, and its margin.

    "KV Cache + Speculative Decoding" section 7.5 and Q21: under top-p the
    target distribution becomes p truncated to its own top-p set and
    renormalised. Reading of the set: order the tokens by logit, largest
    first, equal logits by ascending token id; the set is the shortest
    prefix of that order whose probability reaches top_p (mass >= top_p).
    top_p >= 1 keeps every token.

    Returns (mask [..., V] bool, margin [...]) where margin is the distance
    of top_p * Z from the cumulative masses on either side of the cut, as a
    fraction of the row mass Z (inf when nothing is cut).
    """
    x = _np64(logits)
    V = x.shape[-1]
    rows = x.reshape(-1, V)
    mask = np.zeros(rows.shape, dtype=bool)
    margin = np.full(rows.shape[0], np.inf)
    ids = np.arange(V)
    for r in range(rows.shape[0]):
        if top_p >= 1.0:
            mask[r] = True
            continue
        p = softmax(rows[r], temperature)
        order = np.lexsort((ids, -rows[r]))
        c = np.cumsum(p[order])
        Z = c[-1]
        thr = top_p * Z
        k = int(np.argmax(c >= thr))
        mask[r, order[: k + 1]] = True
        below = c[k - 1] if k > 0 else 0.0
        margin[r] = min(c[k] - thr, thr - below) / Z
    return mask.reshape(x.shape), margin.reshape(x.shape[:-1])


def top_p_filter(logits, top_p, temperature=1.0):
    """logits (fp64) with -inf outside the top-p set: softmax of the result
    (at the same T) is p truncated to the set and renormalised."""
    x = _np64(logits)
    mask, _ = top_p_nucleus(x, top_p, temperature)
    return np.where(mask, x, -np.inf)


def rejection_sample(target_logits, draft, draft_tokens, uniforms,
                     draft_is_probs=False, temperature=1.0, top_p=None, draft_top_p=False):
    """Verify one round for every sequence of the batch.

    target_logits [B, K+1, V]; draft [B, K, V] (logits, or probabilities when
    draft_is_probs); draft_tokens [B, K]; uniforms [B, K+1, 2].
    With top_p < 1 the target rows are cut to their top-p sets first (and the
    draft logit rows too when draft_top_p), see top_p_nucleus.
    Returns a dict with out_tokens [B, K+1] (-1 padded), num_accepted [B] and
    diagnostics (p/q at the draft tokens, accept margins |u - p/q|, CDF margin,
    per-row alpha, the sampled row index and its mass).
    """
    if top_p is not None and top_p < 1.0:
        target_logits = top_p_filter(target_logits, top_p, temperature)
        if draft_top_p and not draft_is_probs and draft is not None:
            draft = top_p_filter(draft, top_p, temperature)
    p = softmax(target_logits, temperature)                      # [B, K+1, V]
    q = _np64(draft) if draft_is_probs else softmax(draft, temperature)
    return verify_from_probs(p, q, draft_tokens, uniforms)


def verify_from_probs(p, q, draft_tokens, uniforms):
    """The accept / resample / bonus logic on given distributions.

    p [B, K+1, V] target distributions, q [B, K, V] draft distributions.
    """
    p = _np64(p)
    q = _np64(q)
    x = _np64(draft_tokens).astype(np.int64)
    uv = _np64(uniforms)
    B, K1, V = p.shape
    K = K1 - 1
    bi = np.arange(B)

    p_x = np.empty((B, K))
    q_x = np.empty((B, K))
    acc_margin = np.empty((B, K))
    alive = np.ones(B, dtype=bool)
    n_rej = np.full(B, K, dtype=np.int64)        # K means "all accepted"
    for i in range(K):
        p_x[:, i] = p[bi, i, x[:, i]]
        q_x[:, i] = q[bi, i, x[:, i]]
        u = uv[:, i, 0]
        accept = u * q_x[:, i] < p_x[:, i]
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(q_x[:, i] > 0, p_x[:, i] / q_x[:, i], np.inf)
        acc_margin[:, i] = np.abs(u - ratio)
        newly = alive & ~accept
        n_rej[newly] = i
        alive &= accept

    # weights of the row that is sampled: the residual max(0, p_n - q_n) at
    # the first rejection n, the target row K+1 (index K) when all accepted
    p_n = p[bi, n_rej]                                          # [B, V]
    if K > 0:
        q_n = q[bi, np.minimum(n_rej, K - 1)]
        residual = np.maximum(0.0, p_n - q_n)
        use_residual = (n_rej < K) & (residual.sum(axis=1) > 0.0)
        w = np.where(use_residual[:, None], residual, p_n)
    else:
        w = p_n
    v = uv[bi, n_rej, 1]
    y, cdf_margin, Z = inverse_cdf(w, v)

    col = np.arange(K + 1)[None, :]
    x_pad = np.concatenate([x, np.zeros((B, 1), dtype=np.int64)], axis=1)
    out = np.where(col < n_rej[:, None], x_pad, -1)
    out = np.where(col == n_rej[:, None], y[:, None], out)
    alpha = np.minimum(p[:, :K, :], q).sum(axis=2)
    return {"out_tokens": out, "num_accepted": n_rej, "p_at_draft": p_x,
            "q_at_draft": q_x, "accept_margin": acc_margin,
            "cdf_margin": cdf_margin, "sampled_row": n_rej, "sampled_mass": Z,
            "alpha": alpha}


def rejection_sample_chunked(target_logits, draft, draft_tokens, uniforms,
                             draft_is_probs=False, temperature=1.0, chunk=8,
                             batch_indices=None):
    """rejection_sample over groups of sequences (bounded host memory)."""
    B = target_logits.shape[0]
    idx = list(range(B)) if batch_indices is None else list(batch_indices)
    parts = []
    for s in range(0, len(idx), chunk):
        sel = idx[s:s + chunk]
        parts.append(rejection_sample(target_logits[sel], draft[sel],
                                      draft_tokens[sel], uniforms[sel],
                                      draft_is_probs, temperature))
    return {k: np.concatenate([r[k] for r in parts]) for k in parts[0]}


def entropy(p):
    """H(p) = -sum p ln p in nats over the last axis (0 ln 0 = 0)."""
    p = _np64(p)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(p > 0, p * np.log(np.where(p > 0, p, 1.0)), 0.0)
    return -t.sum(axis=-1)


def tree_rejection_sample(target_logits, draft, tree_parent, tree_tokens, uniforms,
                          draft_is_probs=False, temperature=1.0, typical=None):
    """Verify a draft tree per sequence by recursive rejection sampling.

    The pages give exact rejection sampling for a chain (quant67 section 3.1;
    "KV Cache + Speculative Decoding" sections 7.1-7.3) and the BFS tree with
    its ancestor mask (Q14, section 8.2), leaving the sampling rule over a
    tree open ("standard rejection sampling" when exactness is wanted). The
    reading taken here (the plainest exact one): walk from the root; at node
    u the residual starts as r = p_u; its children, drafted from q_u, are
    tried in BFS order, child c with token x accepted iff
    uniforms[c][0] * q_u(x) < r(x); a rejection replaces r by
    norm(max(0, r - q_u)); an accepted child becomes u; when every child of
    u is rejected (or u is a leaf) the token is drawn from r by the inverse
    CDF with v = uniforms[u][1]. For a chain this is rejection_sample.

    target_logits [B, n, V]: row j is the target distribution after node j;
    draft [B, n, V] logits (or probabilities): row u is what u's children
    were drawn from; tree_parent [B, n] (node 0 the root, parent -1);
    tree_tokens [B, n] (entry 0 unused); uniforms [B, n, 2].
    typical = (epsilon, delta) switches to typical acceptance ("speculative
    decoding" survey section 9.1 and "KV Cache + Speculative Decoding"
    section 8.2 / Q18: the Medusa rule, not exact): child c of u is accepted
    iff p_u(x) > min(epsilon, delta * exp(-H(p_u))), H in nats; the walk is
    otherwise the same, except that no residual is formed: when no child is
    accepted the token is drawn from p_u itself.

    Returns dict: out_tokens [B, n] (accepted tokens, the drawn one, then -1),
    num_accepted [B], path_nodes [B, n] (accepted nodes, then -1),
    margin [B] (the smallest distance of a decision taken from its
    boundary: |u - r/q| of every accept test, or |p(x) - tau| / tau of every
    typical test, and the CDF margin of the draw) and decisions [B]: the
    walk's decisions in the order taken, each a tuple (node u, child c,
    margin, outcome): an accept (or typical) test of child c at u with
    outcome True / False, and last the draw at u with c = -1 and the drawn
    token as its outcome.
    """
    p_all = softmax(target_logits, temperature)
    q_all = _np64(draft) if draft_is_probs else softmax(draft, temperature)
    par = _np64(tree_parent).astype(np.int64)
    tok = _np64(tree_tokens).astype(np.int64)
    uv = _np64(uniforms)
    B, n, V = p_all.shape
    out = np.full((B, n), -1, dtype=np.int64)
    path = np.full((B, n), -1, dtype=np.int64)
    nacc = np.zeros(B, dtype=np.int64)
    margin = np.full(B, np.inf)
    decisions = [[] for _ in range(B)]
    for b in range(B):
        u, depth = 0, 0
        while True:
            r = p_all[b, u].copy()
            q = q_all[b, u]
            accepted = -1
            if typical is not None:
                tau = min(typical[0], typical[1] * np.exp(-entropy(r)))
                for c in [c for c in range(1, n) if par[b, c] == u]:
                    x = tok[b, c]
                    mt = abs(r[x] - tau) / tau
                    margin[b] = min(margin[b], mt)
                    decisions[b].append((u, c, mt, bool(r[x] > tau)))
                    if r[x] > tau:
                        accepted = c
                        break
                if accepted >= 0:
                    out[b, depth] = tok[b, accepted]
                    path[b, depth] = accepted
                    depth += 1
                    u = accepted
                    continue
                y, m, _ = inverse_cdf(r[None, :], np.array([uv[b, u, 1]]))
                out[b, depth] = y[0]
                margin[b] = min(margin[b], m[0])
                decisions[b].append((u, -1, float(m[0]), int(y[0])))
                nacc[b] = depth
                break
            for c in [c for c in range(1, n) if par[b, c] == u]:
                x = tok[b, c]
                accept = uv[b, c, 0] * q[x] < r[x]
                ratio = r[x] / q[x] if q[x] > 0 else np.inf
                margin[b] = min(margin[b], abs(uv[b, c, 0] - ratio))
                decisions[b].append((u, c, float(abs(uv[b, c, 0] - ratio)), bool(accept)))
                if accept:
                    accepted = c
                    break
                res = np.maximum(0.0, r - q)
                z = res.sum()
                r = res / z if z > 0 else p_all[b, u].copy()   # z = 0 cannot happen in exact arithmetic
            if accepted >= 0:
                out[b, depth] = tok[b, accepted]
                path[b, depth] = accepted
                depth += 1
                u = accepted
                continue
            y, m, _ = inverse_cdf(r[None, :], np.array([uv[b, u, 1]]))
            out[b, depth] = y[0]
            margin[b] = min(margin[b], m[0])
            decisions[b].append((u, -1, float(m[0]), int(y[0])))
            nacc[b] = depth
            break
    return {"out_tokens": out, "num_accepted": nacc, "path_nodes": path, "margin": margin,
            "decisions": decisions}
