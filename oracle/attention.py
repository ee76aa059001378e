"""fp64 oracle of document-masked (intra-document causal) attention.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the
benchmark's CPU baseline, never by the library.

Sources (FlashCP paper, "FlashCP: Load-Balanced Communication-Efficient
Context Parallelism for LLM Training"; "LLM Context Parallel in Production"
guide):
  * Document mask: FlashCP §2.1 and Fig. 1(a) -- query i may attend key j only
    when both lie in the same packed document and j <= i.
  * Online-softmax merge of partial results from separate KV blocks: the
    production guide, "Core Principle: Split Q, Circulate KV" and "Ring
    Attention" -- the row maximum and exponential sum of each block are
    combined without forming the full score matrix.

Definitions computed here (scale = 1/sqrt(d), query head h reads KV head
g = h // (Hq // Hkv), i.e. contiguous GQA groups):
  s_ij   = scale * <q_i,h , k_j,g>            for j in K(i)
  K(i)   = {j : doc(j) = doc(i), j <= i} intersected with the allowed key set
  LSE_ih = ln sum_{j in K(i)} exp(s_ij)       (natural log; -inf if K(i) empty)
  O_ih   = sum_{j in K(i)} exp(s_ij - LSE_ih) v_j,g   (0 if K(i) empty)
Backward, the exact gradient of the above for an upstream dO:
  P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D_i = <dO_i, O_i>,
  dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q,
  with dK and dV summed over the query heads of each GQA group.
Merge of B partials over disjoint key sets:
  LSE = ln sum_b exp(LSE_b),  O = sum_b exp(LSE_b - LSE) O_b.

Two forward forms share nothing but the definition: `attention_bruteforce`
builds the full T x T mask and does a dense softmax (tiny T only), and
`attention_per_doc` does one dense causal softmax per document. Rows are
independent, so per-document work may be split into row chunks purely to
bound memory; no other blocking or reordering is done.
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def to_f64(x) -> np.ndarray:
    """Upcast a tensor/array (bf16 torch tensors included) to float64 numpy."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def doc_ids(cu: np.ndarray) -> np.ndarray:
    """doc(t) for every token t of a packed sequence with offsets `cu`."""
    cu = np.asarray(cu, dtype=np.int64)
    T = int(cu[-1])
    out = np.empty(T, dtype=np.int64)
    for i in range(len(cu) - 1):
        out[cu[i]:cu[i + 1]] = i
    return out


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


def _group(Hq: int, Hkv: int) -> int:
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return Hq // Hkv


def _softmax_rows(s: np.ndarray, allowed: np.ndarray):
    """Masked softmax of each row of s; returns (P, lse). Rows with no allowed
    entry get P = 0 and lse = -inf."""
    s = np.where(allowed, s, NEG_INF)
    m = s.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.where(allowed, np.exp(s - m_safe), 0.0)
    l = e.sum(axis=-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[..., 0] > 0, m_safe[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)), NEG_INF)
    return p, lse


def attention_bruteforce(q, k, v, cu, scale=None, key_allowed=None):
    """Full T x T document-masked attention. q [T,Hq,d], k/v [T,Hkv,d].

    key_allowed: optional bool [T] restricting the key set (a partial KV block).
    Returns O [T,Hq,d] and LSE [Hq,T], float64.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = _group(Hq, Hkv)
    scale = default_scale(d) if scale is None else scale
    doc = doc_ids(cu)
    idx = np.arange(T)
    allowed = (doc[:, None] == doc[None, :]) & (idx[None, :] <= idx[:, None])
    if key_allowed is not None:
        allowed &= np.asarray(key_allowed, dtype=bool)[None, :]
    o = np.zeros((T, Hq, d))
    lse = np.zeros((Hq, T))
    for h in range(Hq):
        g = h // G
        s = scale * (q[:, h, :] @ k[:, g, :].T)
        p, lse[h] = _softmax_rows(s, allowed)
        o[:, h, :] = p @ v[:, g, :]
    return o, lse


def _doc_rows_fwd(qd, kd, vd, scale, key_lo, key_hi, row_chunk, key_ok=None):
    """Forward for one document and one head pair.

    qd [L,d], kd/vd [L,d] (document-local). Keys restricted to the local index
    window [key_lo, key_hi) and, if given, to the local keys with key_ok True.
    Returns o [L,d], lse [L].
    """
    L = qd.shape[0]
    o = np.zeros_like(qd)
    lse = np.full(L, NEG_INF)
    jj = np.arange(L)
    for r0 in range(0, L, row_chunk):
        r1 = min(L, r0 + row_chunk)
        ii = np.arange(r0, r1)
        allowed = (jj[None, :] <= ii[:, None]) & (jj[None, :] >= key_lo) & (jj[None, :] < key_hi)
        if key_ok is not None:
            allowed &= key_ok[None, :]
        s = scale * (qd[r0:r1] @ kd.T)
        p, lse[r0:r1] = _softmax_rows(s, allowed)
        o[r0:r1] = p @ vd
    return o, lse


def attention_per_doc(q, k, v, cu, scale=None, docs=None, heads=None,
                      key_range=None, row_chunk=2048, key_allowed=None):
    """Per-document dense causal attention (the same definition, one document
    at a time).

    docs: iterable of document indices to compute (default all); heads: query
    heads to compute (default all); key_range: (a, b) global key window for a
    partial KV block; key_allowed: optional bool [T] restricting the key set
    further (e.g. to the keys one CP owner holds: the block a ring step
    delivers, "LLM Context Parallel in Production", "Ring Attention").
    Rows/heads not computed are left as NaN so that a caller
    cannot mistake them for results.
    Returns O [T,Hq,d], LSE [Hq,T] float64.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = _group(Hq, Hkv)
    scale = default_scale(d) if scale is None else scale
    cu = np.asarray(cu, dtype=np.int64)
    n = len(cu) - 1
    docs = range(n) if docs is None else docs
    heads = range(Hq) if heads is None else heads
    o = np.full((T, Hq, d), np.nan)
    lse = np.full((Hq, T), np.nan)
    for i in docs:
        s0, s1 = int(cu[i]), int(cu[i + 1])
        if s1 == s0:
            continue
        lo, hi = 0, s1 - s0
        if key_range is not None:
            lo = min(max(key_range[0] - s0, 0), s1 - s0)
            hi = min(max(key_range[1] - s0, 0), s1 - s0)
        ok = None if key_allowed is None else np.asarray(key_allowed, dtype=bool)[s0:s1]
        for h in heads:
            g = h // G
            oo, ll = _doc_rows_fwd(q[s0:s1, h], k[s0:s1, g], v[s0:s1, g], scale, lo, hi, row_chunk, ok)
            o[s0:s1, h] = oo
            lse[h, s0:s1] = ll
    return o, lse


def attention_rows(q, k, v, cu, rows, heads, scale=None, q_holds_rows=False):
    """Forward for a sample of (query row, head) pairs: the full definition per
    row, for spot checks at sizes where whole documents are too costly.
    With q_holds_rows, q[a] is the query of row rows[a] (only the sampled rows
    are passed). Returns o [len(rows), len(heads), d] and lse
    [len(heads), len(rows)]."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    _, Hq, d = q.shape
    G = _group(Hq, k.shape[1])
    scale = default_scale(d) if scale is None else scale
    cu = np.asarray(cu, dtype=np.int64)
    doc = doc_ids(cu)
    rows = np.asarray(rows, dtype=np.int64)
    o = np.zeros((len(rows), len(heads), d))
    lse = np.zeros((len(heads), len(rows)))
    for a, i in enumerate(rows):
        s0 = int(cu[doc[i]])
        qi = q[a] if q_holds_rows else q[i]
        for b, h in enumerate(heads):
            g = h // G
            s = scale * (k[s0:i + 1, g] @ qi[h])
            m = s.max()
            e = np.exp(s - m)
            lse[b, a] = m + math.log(e.sum())
            o[a, b] = (e / e.sum()) @ v[s0:i + 1, g]
    return o, lse


def attention_bwd_per_doc(q, k, v, o, lse, do, cu, scale=None, docs=None,
                          row_chunk=2048):
    """Exact gradient of document-masked attention, one document at a time.

    o and lse are the forward results the gradient is taken at (normally the
    oracle's own fp64 forward). Returns dQ [T,Hq,d], dK and dV [T,Hkv,d] as
    float64; rows of documents not in `docs` are NaN.
    """
    q, k, v, o, do = to_f64(q), to_f64(k), to_f64(v), to_f64(o), to_f64(do)
    lse = to_f64(lse)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = _group(Hq, Hkv)
    scale = default_scale(d) if scale is None else scale
    cu = np.asarray(cu, dtype=np.int64)
    n = len(cu) - 1
    docs = range(n) if docs is None else docs
    dq = np.full((T, Hq, d), np.nan)
    dk = np.full((T, Hkv, d), np.nan)
    dv = np.full((T, Hkv, d), np.nan)
    for i in docs:
        s0, s1 = int(cu[i]), int(cu[i + 1])
        L = s1 - s0
        if L == 0:
            continue
        dk[s0:s1] = 0.0
        dv[s0:s1] = 0.0
        jj = np.arange(L)
        for h in range(Hq):
            g = h // G
            qh, kg, vg = q[s0:s1, h], k[s0:s1, g], v[s0:s1, g]
            doh, oh, lh = do[s0:s1, h], o[s0:s1, h], lse[h, s0:s1]
            Dv = np.sum(doh * oh, axis=-1)
            dqh = np.zeros((L, d))
            for r0 in range(0, L, row_chunk):
                r1 = min(L, r0 + row_chunk)
                ii = np.arange(r0, r1)
                allowed = jj[None, :] <= ii[:, None]
                s = scale * (qh[r0:r1] @ kg.T)
                p = np.where(allowed, np.exp(np.where(allowed, s, 0.0) - lh[r0:r1, None]), 0.0)
                dv[s0:s1, g] += p.T @ doh[r0:r1]
                dp = doh[r0:r1] @ vg.T
                ds = p * (dp - Dv[r0:r1, None])
                dqh[r0:r1] = scale * (ds @ kg)
                dk[s0:s1, g] += scale * (ds.T @ qh[r0:r1])
            dq[s0:s1, h] = dqh
    return dq, dk, dv


def _row_softmax(qi, kd, scale):
    """Probabilities and log-sum-exp of one query row over the keys kd."""
    s = scale * (kd @ qi)
    m = s.max()
    e = np.exp(s - m)
    total = e.sum()
    return e / total, m + math.log(total)


def attention_bwd_query_rows(q, k, v, do, cu, rows, heads, scale=None, q_offset=0):
    """dQ at sampled query rows, from the definition of the gradient row by
    row (for spot checks at sizes where whole documents are too costly):
    with the row's keys j in its document up to i,
      P_ij = exp(s_ij - LSE_i), O_i = sum_j P_ij v_j, D_i = <dO_i, O_i>,
      dS_ij = P_ij (<dO_i, v_j> - D_i),  dQ_i = scale sum_j dS_ij k_j.
    q and do hold rows q_offset, q_offset + 1, ... of the sequence (all rows
    when q_offset = 0); k, v and cu describe the whole sequence.
    Returns dq [len(rows), len(heads), d] (fp64)."""
    k, v = to_f64(k), to_f64(v)
    _, Hq, d = q.shape
    G = _group(Hq, k.shape[1])
    scale = default_scale(d) if scale is None else scale
    cu = np.asarray(cu, dtype=np.int64)
    doc = doc_ids(cu)
    dq = np.zeros((len(rows), len(heads), d))
    for a, i in enumerate(np.asarray(rows, dtype=np.int64)):
        s0 = int(cu[doc[i]])
        qi, doi = to_f64(q[i - q_offset]), to_f64(do[i - q_offset])
        for b, h in enumerate(heads):
            g = h // G
            kd, vd = k[s0:i + 1, g], v[s0:i + 1, g]
            p, _ = _row_softmax(qi[h], kd, scale)
            Di = float(doi[h] @ (p @ vd))
            ds = p * (vd @ doi[h] - Di)
            dq[a, b] = scale * (ds @ kd)
    return dq


def attention_bwd_key_rows(q, k, v, do, cu, key_rows, scale=None, q_offset=0):
    """dK and dV at sampled key rows j (every KV head), from the definition:
    every query i >= j of j's document and every query head h of the KV
    head's group contribute
      dV_j += P_ij dO_i,  dK_j += scale dS_ij q_i,
    with P_ij, D_i and dS_ij as in attention_bwd_query_rows (each query row's
    softmax over its own keys recomputed here). Costs O((doc end - j) * i * d)
    per head: meant for key rows near the end of their document. q and do
    hold rows q_offset, q_offset + 1, ... of the sequence, which must include
    every query row from the first key row to its document's end.
    Returns dk, dv [len(key_rows), Hkv, d] (fp64)."""
    q, k, v, do = to_f64(q), to_f64(k), to_f64(v), to_f64(do)
    _, Hq, d = q.shape
    Hkv = k.shape[1]
    G = _group(Hq, Hkv)
    scale = default_scale(d) if scale is None else scale
    cu = np.asarray(cu, dtype=np.int64)
    doc = doc_ids(cu)
    dk = np.zeros((len(key_rows), Hkv, d))
    dv = np.zeros((len(key_rows), Hkv, d))
    for a, j in enumerate(np.asarray(key_rows, dtype=np.int64)):
        s0, s1 = int(cu[doc[j]]), int(cu[doc[j] + 1])
        for h in range(Hq):
            g = h // G
            for i in range(j, s1):
                kd, vd = k[s0:i + 1, g], v[s0:i + 1, g]
                qi, doi = q[i - q_offset, h], do[i - q_offset, h]
                p, _ = _row_softmax(qi, kd, scale)
                Di = float(doi @ (p @ vd))
                pj = p[j - s0]
                dsj = pj * (float(v[j, g] @ doi) - Di)
                dv[a, g] += pj * doi
                dk[a, g] += scale * dsj * qi
    return dk, dv


def merge(o_parts, lse_parts):
    """Merge B partial results over disjoint key sets.

    o_parts [B,rows,Hq,d], lse_parts [B,Hq,rows] (natural log, -inf for a row
    with no keys in that block). Returns O [rows,Hq,d], LSE [Hq,rows]; a row
    empty in every block gets O = 0 and LSE = -inf.
    """
    o_parts = to_f64(o_parts)
    lse_parts = to_f64(lse_parts)
    m = lse_parts.max(axis=0)                       # [Hq, rows]
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.exp(lse_parts - m_safe[None])            # exp(-inf) = 0
    total = w.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, NEG_INF, m_safe + np.log(np.where(empty, 1.0, total)))
    coef = np.where(empty[None], 0.0, w / np.where(empty, 1.0, total)[None])  # [B,Hq,rows]
    o = np.einsum("bhr,brhd->rhd", coef, o_parts)
    return o, lse


def useful_pairs(lengths) -> int:
    """Number of (query, key) pairs a document mask keeps: sum of L(L+1)/2."""
    return int(sum(int(L) * (int(L) + 1) // 2 for L in lengths))
