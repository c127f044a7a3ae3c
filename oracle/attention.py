"""fp64 CPU oracle: zigzag split, causal attention, LSE merge, ring partition.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.  Inputs may be torch tensors or numpy arrays of any float dtype;
they are upcast to float64 (bf16 inputs are therefore exact).  Layouts:

* q, k, v, dout, out, dq, dk, dv: ``[T, H, d]`` in natural token order (THD);
* lse: ``[H, T]``, natural log of the row's softmax normaliser *after* the
  softmax scale (lse_i = log sum_j exp(scale * q_i . k_j) over visible j);
* ``cu_seqlens``: ``n + 1`` ascending ints; sample ``i`` is
  ``[cu[i], cu[i+1])`` and is laid out ``[prefix (N tokens), text]``
  (CP-VLM page §2).

Readings where the pages leave a step open (the same list is kept with the
design notes):

* the mask is causal over the whole ``[prefix, text]`` sample, prefix
  included: a text query sees every prefix token, a prefix query sees the
  prefix causally (CP-VLM page §4.1 step 4 builds ``[image, text chunk]``);
* packed samples are zigzag-split one by one, and a rank's text is the
  concatenation of its two chunks of every sample in sample order
  (CP-VLM page §5.3 only says the split must follow ``cu_seqlens``);
* ring step ``s`` hands rank ``r`` the KV of rank ``(r - s) mod P``; the
  replicated prefix is part of step 0's local KV;
* prefix query rows are computed once, not once per rank; per-rank prefix
  gradients therefore come from text queries only, and the prefix queries'
  own contribution is a separate term of the sum.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# ----------------------------------------------------------------------------
# helpers (shape plumbing only)
# ----------------------------------------------------------------------------
def _f64(x):
    """Upcast a torch tensor or array-like to a float64 numpy array."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _take(x, rows, heads):
    """x[rows][:, heads] as float64 (rows: int array; heads: list)."""
    if hasattr(x, "detach"):
        import torch
        x = x[torch.as_tensor(np.asarray(rows), dtype=torch.long)]
        return _f64(x)[:, heads]
    return np.asarray(x, dtype=np.float64)[np.asarray(rows)][:, heads]


def kv_group(H, H_kv):
    """Grouped-query attention: query head ``h`` reads KV head ``h // G`` with
    ``G = H / H_kv`` (consecutive grouping; ``H_kv = H`` is plain multi-head
    attention, ``H_kv = 1`` is multi-query attention)."""
    if H_kv < 1 or H % H_kv != 0:
        raise ValueError("H=%d is not a multiple of H_kv=%d" % (H, H_kv))
    return H // H_kv


def _expand_kv(x, H):
    """[T, H_kv, d] -> [T, H, d]: KV head j copied to query heads jG .. jG+G-1."""
    return np.repeat(x, kv_group(H, x.shape[1]), axis=1)


def _fold_kv(g, H_kv):
    """Adjoint of :func:`_expand_kv`: the gradients of the G copies of a KV
    head are summed.  [..., H, d] -> [..., H_kv, d]."""
    G = kv_group(g.shape[-2], H_kv)
    return g.reshape(g.shape[:-2] + (H_kv, G, g.shape[-1])).sum(axis=-2)


def _samples(cu_seqlens):
    cu = [int(c) for c in cu_seqlens]
    if any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must be non-decreasing")
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def _positions(cu_seqlens):
    """Sample id and in-sample position of every natural token."""
    samples = _samples(cu_seqlens)
    T = samples[-1][1] if samples else 0
    sid = np.empty(T, dtype=np.int64)
    pos = np.empty(T, dtype=np.int64)
    for i, (a, b) in enumerate(samples):
        sid[a:b] = i
        pos[a:b] = np.arange(b - a)
    return sid, pos


# ----------------------------------------------------------------------------
# zigzag split (CP-VLM page §1.1)
# ----------------------------------------------------------------------------
def zigzag_chunk_ids(P):
    """CP-VLM page §1.1: the sequence is cut into 2P chunks and rank r keeps the
    head-tail pair (r, 2P - r - 1); with CP=2 rank 0 keeps chunks 0 and 3 and
    rank 1 keeps chunks 1 and 2."""
    if P < 1:
        raise ValueError("P must be >= 1")
    return [(r, 2 * P - 1 - r) for r in range(P)]


def _text_layout(cu_seqlens, prefix_len, P):
    """Per sample: natural index of its first text token and its chunk length c
    (text length / 2P).  CP-VLM page §4.1 step 3: only the text is split."""
    out = []
    for a, b in _samples(cu_seqlens):
        L = b - a - prefix_len
        if L < 0:
            raise ValueError("sample shorter than the prefix")
        if L % (2 * P) != 0:
            raise ValueError("text length %d not divisible by 2P=%d" % (L, 2 * P))
        out.append((a + prefix_len, L // (2 * P)))
    return out


def zigzag_index(cu_seqlens, prefix_len, P):
    """Zigzag gather table and its inverse (CP-VLM page §1.1, ``index_select``
    with ``[cp_rank, 2*cp_size - cp_rank - 1]`` on the sequence dimension;
    §5.3 applied per sample).

    Returns ``(fwd_idx, inv_idx)``:

    * ``fwd_idx[k]``: natural token index of permuted text row ``k``.  Rows are
      rank-major; within a rank, sample-major; within a sample, chunk ``r``
      then chunk ``2P - r - 1``.
    * ``inv_idx[m]``: permuted row of the ``m``-th text token in natural order.
    """
    layout = _text_layout(cu_seqlens, prefix_len, P)
    chunks = zigzag_chunk_ids(P)
    fwd = []
    for r in range(P):
        for t0, c in layout:
            for ch in chunks[r]:
                fwd.extend(range(t0 + ch * c, t0 + (ch + 1) * c))
    fwd = np.asarray(fwd, dtype=np.int64)
    text_nat = [t for t0, c in layout for t in range(t0, t0 + 2 * P * c)]
    where = {int(t): k for k, t in enumerate(fwd)}
    inv = np.asarray([where[t] for t in text_nat], dtype=np.int64)
    return fwd, inv


def rank_local_rows(cu_seqlens, prefix_len, P):
    """Natural token indices held by each simulated rank (its text shard)."""
    fwd, _ = zigzag_index(cu_seqlens, prefix_len, P)
    R = len(fwd) // P
    return [fwd[r * R:(r + 1) * R] for r in range(P)]


def _prefix_rows(cu_seqlens, prefix_len):
    return np.asarray([t for a, _ in _samples(cu_seqlens) for t in range(a, a + prefix_len)],
                      dtype=np.int64)


# ----------------------------------------------------------------------------
# the plain result: unpartitioned causal attention per sample
# ----------------------------------------------------------------------------
def _causal_rows(qb, kb, vb, q_pos0, scale):
    """Rows ``q_pos0 ..`` of causal softmax attention of one head over keys
    ``0 .. q_pos0 + len(qb) - 1`` of the same sample: S = scale q k^T with
    keys after the query masked, lse = log sum exp S, o = softmax(S) v."""
    n = qb.shape[0]
    S = scale * (qb @ kb.T)
    qpos = q_pos0 + np.arange(n)[:, None]
    kpos = np.arange(kb.shape[0])[None, :]
    S = np.where(kpos <= qpos, S, NEG_INF)
    m = S.max(axis=1, keepdims=True)          # finite: a query always sees itself
    e = np.exp(S - m)
    l = e.sum(axis=1, keepdims=True)
    return (e / l) @ vb, (m + np.log(l))[:, 0], e / l


def causal_attention_fwd(q, k, v, cu_seqlens, scale, row_block=1024):
    """Unpartitioned causal attention of every sample (the method reaches this
    exactly, only partitioned).  Returns ``out [T,H,d]`` and ``lse [H,T]``.
    Query rows are evaluated ``row_block`` at a time; every row is computed
    from its full set of visible keys.  ``k``/``v`` may hold fewer heads than
    ``q`` (grouped-query attention, :func:`kv_group`)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, d = q.shape
    k, v = _expand_kv(k, H), _expand_kv(v, H)
    out = np.zeros((T, H, d))
    lse = np.full((H, T), NEG_INF)
    for a, b in _samples(cu_seqlens):
        for h in range(H):
            for r0 in range(a, b, row_block):
                r1 = min(b, r0 + row_block)
                o, l, _ = _causal_rows(q[r0:r1, h], k[a:r1, h], v[a:r1, h], r0 - a, scale)
                out[r0:r1, h] = o
                lse[h, r0:r1] = l
    return out, lse


def causal_attention_bwd(q, k, v, dout, cu_seqlens, scale, row_block=1024):
    """Gradient of unpartitioned causal attention (standard softmax-attention
    backward, which the CP-VLM page's §3.2/§4.2 gradient path needs):
    P = softmax(S), dV = P^T dO, dP = dO V^T, D_i = dO_i . o_i,
    dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.
    o is this oracle's own forward result.  Returns ``dq, dk, dv`` (THD).
    With grouped KV heads, dk/dv of a KV head sum its query heads' terms."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, H, d = q.shape
    H_kv = k.shape[1]
    k, v = _expand_kv(k, H), _expand_kv(v, H)
    dq = np.zeros((T, H, d))
    dk = np.zeros((T, H, d))
    dv = np.zeros((T, H, d))
    for a, b in _samples(cu_seqlens):
        for h in range(H):
            for r0 in range(a, b, row_block):
                r1 = min(b, r0 + row_block)
                K, V, Q, dO = k[a:r1, h], v[a:r1, h], q[r0:r1, h], do[r0:r1, h]
                o, _, Pm = _causal_rows(Q, K, V, r0 - a, scale)
                dv[a:r1, h] += Pm.T @ dO
                dP = dO @ V.T
                D = (dO * o).sum(axis=1, keepdims=True)
                dS = Pm * (dP - D)
                dq[r0:r1, h] = scale * (dS @ K)
                dk[a:r1, h] += scale * (dS.T @ Q)
    return dq, _fold_kv(dk, H_kv), _fold_kv(dv, H_kv)


def _sample_of(cu_seqlens, t):
    for a, b in _samples(cu_seqlens):
        if a <= t < b:
            return a, b
    raise IndexError(t)


def causal_attention_fwd_rows(q, k, v, cu_seqlens, scale, rows, heads=None, dout=None,
                              row_block=256):
    """The unpartitioned result at selected natural query rows only (for
    workloads too large for the full oracle).  Returns ``out [n,Hs,d]``,
    ``lse [Hs,n]`` and, when ``dout`` is given, ``dq [n,Hs,d]`` (the row's
    own dP and D make dQ_i computable row by row)."""
    if k.shape[1] != q.shape[1]:
        raise ValueError("the row-sampled oracle takes as many KV heads as query heads")
    rows = np.asarray(rows, dtype=np.int64)
    heads = list(range(q.shape[1])) if heads is None else list(heads)
    qf = _take(q, rows, heads)
    n, d = len(rows), q.shape[2]
    out = np.zeros((n, len(heads), d))
    lse = np.full((len(heads), n), NEG_INF)
    dq = np.zeros((n, len(heads), d)) if dout is not None else None
    groups = {}
    for idx, t in enumerate(rows):
        groups.setdefault(_sample_of(cu_seqlens, int(t)), []).append(idx)
    for (a, b), idxs in groups.items():
        idxs = np.asarray(idxs)
        last = int(rows[idxs].max()) + 1
        Ks = _take(k, np.arange(a, last), heads)
        Vs = _take(v, np.arange(a, last), heads)
        dOs = _take(dout, rows[idxs], heads) if dout is not None else None
        for hi in range(len(heads)):
            for c0 in range(0, len(idxs), row_block):
                sel = idxs[c0:c0 + row_block]
                Q = qf[sel, hi]
                S = scale * (Q @ Ks[:, hi].T)
                qpos = (rows[sel] - a)[:, None]
                kpos = np.arange(Ks.shape[0])[None, :]
                S = np.where(kpos <= qpos, S, NEG_INF)
                m = S.max(axis=1, keepdims=True)
                e = np.exp(S - m)
                l = e.sum(axis=1, keepdims=True)
                Pm = e / l
                o = Pm @ Vs[:, hi]
                out[sel, hi] = o
                lse[hi, sel] = (m + np.log(l))[:, 0]
                if dout is not None:
                    dO = dOs[c0:c0 + row_block, hi]
                    dS = Pm * (dO @ Vs[:, hi].T - (dO * o).sum(axis=1, keepdims=True))
                    dq[sel, hi] = scale * (dS @ Ks[:, hi])
    return out, lse, dq


def causal_attention_bwd_keys(q, k, v, dout, cu_seqlens, scale, keys, heads=None,
                              row_block=256):
    """dK and dV of the unpartitioned result at selected natural key rows.
    Key j receives from queries i >= j of its sample: dV_j = sum_i P_ij dO_i,
    dK_j = scale sum_i P_ij (dO_i . v_j - D_i) q_i, with each query row's
    softmax and D_i = dO_i . o_i taken over its full set of visible keys.
    Cost grows with (sample end - smallest key) x sample length, so pick keys
    near the end of long samples.  Returns ``dk, dv [n,Hs,d]``."""
    if k.shape[1] != q.shape[1]:
        raise ValueError("the key-sampled oracle takes as many KV heads as query heads")
    keys = np.asarray(keys, dtype=np.int64)
    heads = list(range(q.shape[1])) if heads is None else list(heads)
    n, d = len(keys), q.shape[2]
    dk = np.zeros((n, len(heads), d))
    dv = np.zeros((n, len(heads), d))
    groups = {}
    for idx, t in enumerate(keys):
        groups.setdefault(_sample_of(cu_seqlens, int(t)), []).append(idx)
    for (a, b), idxs in groups.items():
        idxs = np.asarray(idxs)
        first = int(keys[idxs].min())
        Ks = _take(k, np.arange(a, b), heads)
        Vs = _take(v, np.arange(a, b), heads)
        Qs = _take(q, np.arange(first, b), heads)
        dOs = _take(dout, np.arange(first, b), heads)
        kcol = keys[idxs] - a
        for hi in range(len(heads)):
            for r0 in range(first, b, row_block):
                r1 = min(b, r0 + row_block)
                Q, dO = Qs[r0 - first:r1 - first, hi], dOs[r0 - first:r1 - first, hi]
                o, _, Pm = _causal_rows(Q, Ks[:r1 - a, hi], Vs[:r1 - a, hi], r0 - a, scale)
                D = (dO * o).sum(axis=1, keepdims=True)
                Pj = Pm[:, kcol] if kcol.max() < Pm.shape[1] else \
                    np.pad(Pm, ((0, 0), (0, b - a - Pm.shape[1])))[:, kcol]
                dPj = dO @ Vs[kcol, hi].T
                dSj = Pj * (dPj - D)
                dv[idxs, hi] += Pj.T @ dO
                dk[idxs, hi] += scale * (dSj.T @ Q)
    return dk, dv


# ----------------------------------------------------------------------------
# LSE merge of partial results (Ring Attention's online-softmax combination)
# ----------------------------------------------------------------------------
def _merge2(o_a, lse_a, o_b, lse_b):
    """(o_a, lse_a) + (o_b, lse_b) for two partial softmax results over
    disjoint key sets: lse = log(e^lse_a + e^lse_b),
    o = e^(lse_a - lse) o_a + e^(lse_b - lse) o_b.  A side with lse = -inf
    (no visible key) contributes nothing; both -inf gives lse = -inf, o = 0.
    o: [rows, H, d]; lse: [H, rows]."""
    m = np.maximum(lse_a, lse_b)
    fin = np.isfinite(m)
    ms = np.where(fin, m, 0.0)
    wa = np.exp(lse_a - ms)
    wb = np.exp(lse_b - ms)
    tot = wa + wb
    lse = np.where(fin, ms + np.log(np.where(fin, tot, 1.0)), NEG_INF)
    safe = np.where(fin, tot, 1.0)
    ca = np.where(fin, wa / safe, 0.0).T[:, :, None]
    cb = np.where(fin, wb / safe, 0.0).T[:, :, None]
    return ca * o_a + cb * o_b, lse


def lse_merge(outs, lses):
    """Fold the partials left to right in the given (ring) order."""
    o, l = _f64(outs[0]), _f64(lses[0])
    for ob, lb in zip(outs[1:], lses[1:]):
        o, l = _merge2(o, l, _f64(ob), _f64(lb))
    return o, l


# ----------------------------------------------------------------------------
# the partitioned method, step by step
# ----------------------------------------------------------------------------
def _masked_partial(qb, kb, vb, mask, scale):
    """Softmax attention of query rows over the keys ``mask`` allows:
    returns o [n,H,d] and lse [H,n]; rows that see no key give o=0, lse=-inf."""
    n, H, d = qb.shape
    o = np.zeros((n, H, d))
    lse = np.full((H, n), NEG_INF)
    if kb.shape[0] == 0 or n == 0:
        return o, lse
    any_key = mask.any(axis=1)
    for h in range(H):
        S = scale * (qb[:, h] @ kb[:, h].T)
        S = np.where(mask, S, NEG_INF)
        m = np.where(any_key, S.max(axis=1), 0.0)[:, None]
        e = np.exp(S - m)
        l = e.sum(axis=1, keepdims=True)
        ls = np.where(l > 0, l, 1.0)
        o[:, h] = (e / ls) @ vb[:, h]
        lse[h] = np.where(any_key, (m + np.log(ls))[:, 0], NEG_INF)
    return o, lse


def _visible(sid, pos, q_rows, k_rows):
    return (sid[k_rows][None, :] == sid[q_rows][:, None]) & \
           (pos[k_rows][None, :] <= pos[q_rows][:, None])


def cp_ring_fwd(q, k, v, cu_seqlens, prefix_len, P, scale, return_partials=False):
    """The partitioned forward, literally (CP-VLM page §1.1 and §4.1):

    1. the image prefix of every sample is replicated to all ranks (§4.1 step 2);
    2. only the text is zigzag-split: rank r keeps chunks r and 2P-r-1 of every
       sample (§1.1, §4.1 step 3, §5.3);
    3. rank r's local KV at step 0 is ``[image prefix, own text]`` (§4.1 step 4);
       at ring step s it holds the text KV of rank (r - s) mod P (§1 Ring
       Attention; Parallelism page §6);
    4. each step gives a partial (o_s, lse_s) under the global causal mask, and
       the partials are merged by log-sum-exp in step order;
    5. results are written back to natural order (the inverse of the gather).

    Prefix query rows attend to their own prefix once.  Returns ``out, lse``
    (and, with ``return_partials``, the per (rank, step) partials).  Grouped
    KV heads are read through :func:`kv_group`."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, d = q.shape
    k, v = _expand_kv(k, H), _expand_kv(v, H)
    sid, pos = _positions(cu_seqlens)
    local = rank_local_rows(cu_seqlens, prefix_len, P)
    pre = _prefix_rows(cu_seqlens, prefix_len)
    out = np.zeros((T, H, d))
    lse = np.full((H, T), NEG_INF)
    partials = {}
    if len(pre):
        o, l = _masked_partial(q[pre], k[pre], v[pre], _visible(sid, pos, pre, pre), scale)
        out[pre], lse[:, pre] = o, l
    for r in range(P):
        qr = local[r]
        o_run = l_run = None
        for s in range(P):
            j = (r - s) % P
            kv = local[j] if s > 0 else np.concatenate([pre, local[r]])
            o_s, l_s = _masked_partial(q[qr], k[kv], v[kv], _visible(sid, pos, qr, kv), scale)
            partials[(r, s)] = (o_s, l_s)
            if o_run is None:
                o_run, l_run = o_s, l_s
            else:
                o_run, l_run = _merge2(o_run, l_run, o_s, l_s)
        out[qr] = o_run
        lse[:, qr] = l_run
    if return_partials:
        return out, lse, partials
    return out, lse


def _masked_grads(qb, kb, vb, dob, lse_q, D_q, mask, scale):
    """Block backward with the final lse: P = exp(S - lse) on visible pairs,
    dV = P^T dO, dS = P * (dO V^T - D), dQ = scale dS K, dK = scale dS^T Q."""
    n, H, d = qb.shape
    m_ = kb.shape[0]
    dq = np.zeros((n, H, d))
    dk = np.zeros((m_, H, d))
    dv = np.zeros((m_, H, d))
    if n == 0 or m_ == 0:
        return dq, dk, dv
    for h in range(H):
        S = scale * (qb[:, h] @ kb[:, h].T)
        Pm = np.where(mask, np.exp(np.where(mask, S, 0.0) - lse_q[h][:, None]), 0.0)
        dv[:, h] = Pm.T @ dob[:, h]
        dS = Pm * (dob[:, h] @ vb[:, h].T - D_q[:, h][:, None])
        dq[:, h] = scale * (dS @ kb[:, h])
        dk[:, h] = scale * (dS.T @ qb[:, h])
    return dq, dk, dv


def cp_ring_bwd(q, k, v, dout, cu_seqlens, prefix_len, P, scale):
    """The partitioned backward (CP-VLM page §4.2): every rank differentiates
    its own text queries against the KV it met at each ring step, using the
    merged (final) lse; text dK/dV travel back to the rank that owns the KV;
    each rank ends with its own gradient of the replicated image prefix, and
    those per-rank prefix gradients are summed (§4.2 step 3, the AllReduce),
    together with the prefix queries' own term.

    Returns ``dq, dk, dv`` (THD) and the per-rank prefix partials
    ``pdk, pdv`` of shape ``[P + 1, n_prefix_rows, H, d]`` (slot P holds the
    prefix queries' own term).  With grouped KV heads (:func:`kv_group`) the
    KV-side gradients, per-rank prefix partials included, are summed over
    each KV head's query heads."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    T, H, d = q.shape
    H_kv = k.shape[1]
    k, v = _expand_kv(k, H), _expand_kv(v, H)
    out, lse = cp_ring_fwd(q, k, v, cu_seqlens, prefix_len, P, scale)
    D = (do * out).sum(axis=2)                     # [T, H]
    sid, pos = _positions(cu_seqlens)
    local = rank_local_rows(cu_seqlens, prefix_len, P)
    pre = _prefix_rows(cu_seqlens, prefix_len)
    npre = len(pre)
    dq = np.zeros((T, H, d))
    dk = np.zeros((T, H, d))
    dv = np.zeros((T, H, d))
    pdk = np.zeros((P + 1, npre, H, d))
    pdv = np.zeros((P + 1, npre, H, d))
    if npre:
        g = _masked_grads(q[pre], k[pre], v[pre], do[pre], lse[:, pre], D[pre],
                          _visible(sid, pos, pre, pre), scale)
        dq[pre] += g[0]
        pdk[P] += g[1]
        pdv[P] += g[2]
    for r in range(P):
        qr = local[r]
        for s in range(P):
            j = (r - s) % P
            kv = local[j] if s > 0 else np.concatenate([pre, local[r]])
            g = _masked_grads(q[qr], k[kv], v[kv], do[qr], lse[:, qr], D[qr],
                              _visible(sid, pos, qr, kv), scale)
            dq[qr] += g[0]
            if s == 0:
                pdk[r] += g[1][:npre]
                pdv[r] += g[2][:npre]
                dk[kv[npre:]] += g[1][npre:]
                dv[kv[npre:]] += g[2][npre:]
            else:
                dk[kv] += g[1]
                dv[kv] += g[2]
    if npre:
        sk = np.zeros((npre, H, d))
        sv = np.zeros((npre, H, d))
        for r in range(P + 1):                     # fixed order: ranks, then self
            sk += pdk[r]
            sv += pdv[r]
        dk[pre] += sk
        dv[pre] += sv
    return (dq, _fold_kv(dk, H_kv), _fold_kv(dv, H_kv), _fold_kv(pdk, H_kv),
            _fold_kv(pdv, H_kv))


def cp_pair_counts(cu_seqlens, prefix_len, P):
    """Unmasked (query, key) pairs met by each rank at each ring step, counted
    by brute force from the masks (text queries only), plus the prefix
    queries' own pairs.  Returns ``(counts [P, P], prefix_self)``."""
    sid, pos = _positions(cu_seqlens)
    local = rank_local_rows(cu_seqlens, prefix_len, P)
    pre = _prefix_rows(cu_seqlens, prefix_len)
    counts = np.zeros((P, P), dtype=np.int64)
    for r in range(P):
        for s in range(P):
            j = (r - s) % P
            kv = local[j] if s > 0 else np.concatenate([pre, local[r]])
            counts[r, s] = int(_visible(sid, pos, local[r], kv).sum())
    self_pairs = int(_visible(sid, pos, pre, pre).sum()) if len(pre) else 0
    return counts, self_pairs
