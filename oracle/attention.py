"""Plain fp64 CPU attention: the definition the CUDA path must reproduce.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product never
imports this module.

Arrays are numpy, laid out ``[..., N, d]`` (any leading batch/head dims).
Inputs are upcast to float64 exactly; nothing is rounded on the way.
Scores are ``S = scale * Q K^T``; ``causal`` masks key ``j`` from query ``i``
when ``j > i`` (top-left alignment, queries and keys both indexed from 0).

Where the full N x N score matrix of one head would not fit in host memory
the functions below walk the query rows in chunks of ``row_chunk`` rows.
Softmax is a per-row operation and dK, dV are sums over query rows, so the
chunked result is the same definition evaluated row by row; every chunk still
materialises whole rows of S and P (no tiling over keys, no online update).
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _masked_scores(q_rows: np.ndarray, k: np.ndarray, scale: float, causal: bool,
                   row0: int) -> np.ndarray:
    """S = scale * Q K^T for query rows ``row0 .. row0+len(q_rows)-1`` of one head.

    [Interrogating-5] "Why is the textbook algorithm memory-bound?", first
    equation (S = Q K^T); the 1/sqrt(d) factor of [aicassindra] "End-to-end
    flow" is carried by ``scale``.  Causal masking ([aicassindra] "End-to-end
    flow": blocks in the future are skipped) sets S_ij = -inf for j > i.
    """
    s = scale * (q_rows @ k.T)
    if causal:
        i = np.arange(row0, row0 + q_rows.shape[0])[:, None]
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j > i, -np.inf, s)
    return s


def _row_softmax(s: np.ndarray):
    """Row softmax with the max subtracted first, returning (P, m, l).

    [Interrogating-5] "How can you softmax a row you never see whole?": each
    e^{s_ij} is divided by the row's sum after subtracting the row maximum.
    A row whose every score is -inf (unreachable for square causal inputs)
    gets P = 0, m = -inf, l = 0.
    """
    m = s.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    e = np.where(np.isfinite(s), np.exp(s - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    p = np.where(finite[:, None], e / np.where(finite, l, 1.0)[:, None], 0.0)
    return p, m, l


def _heads(*arrays):
    lead = arrays[0].shape[:-2]
    for idx in np.ndindex(*lead):
        yield idx


def attention_probs_ref(q, k, scale: float, causal: bool = False) -> np.ndarray:
    """P = softmax(scale * Q K^T) as a full ``[..., Nq, Nk]`` array (small inputs).

    [Interrogating-5] "Why is the textbook algorithm memory-bound?", first
    equation: P = softmax(S).
    """
    q, k = _f64(q), _f64(k)
    out = np.zeros(q.shape[:-1] + (k.shape[-2],))
    for idx in _heads(q):
        s = _masked_scores(q[idx], k[idx], scale, causal, 0)
        out[idx] = _row_softmax(s)[0]
    return out


def attention_fwd_ref(q, k, v, scale: float, causal: bool = False, row_chunk: int = 256):
    """Forward: O = softmax(scale Q K^T) V and LSE_i = m_i + log l_i.

    O follows [Interrogating-5] "Why is the textbook algorithm memory-bound?"
    (O = P V).  LSE is the per-row log-sum-exp of the scaled scores in natural
    log units, [Interrogating-5] "What does the backward pass do without P?",
    equation L_i = m_i + log l_i.  Returns ``(O, LSE)`` with shapes
    ``[..., Nq, dv]`` and ``[..., Nq]``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq = q.shape[-2]
    o = np.zeros(q.shape[:-1] + (v.shape[-1],))
    lse = np.zeros(q.shape[:-1])
    for idx in _heads(q):
        for r0 in range(0, nq, row_chunk):
            r1 = min(nq, r0 + row_chunk)
            s = _masked_scores(q[idx][r0:r1], k[idx], scale, causal, r0)
            p, m, l = _row_softmax(s)
            o[idx][r0:r1] = p @ v[idx]
            with np.errstate(divide="ignore"):
                lse[idx][r0:r1] = np.where(np.isfinite(m), m + np.log(l), -np.inf)
    return o, lse


def recompute_probs_from_lse_ref(q, k, lse, scale: float, causal: bool = False) -> np.ndarray:
    """P_ij = exp(S_ij - L_i) from Q, K and the saved LSE (small inputs).

    [Interrogating-5] "What does the backward pass do without P?": the
    backward pass recovers each probability from the scores and the one
    log-sum-exp per row that the forward pass stored.
    """
    q, k, lse = _f64(q), _f64(k), _f64(lse)
    out = np.zeros(q.shape[:-1] + (k.shape[-2],))
    for idx in _heads(q):
        s = _masked_scores(q[idx], k[idx], scale, causal, 0)
        out[idx] = np.where(np.isfinite(s), np.exp(s - lse[idx][:, None]), 0.0)
    return out


def attention_bwd_preprocess_ref(o, dout) -> np.ndarray:
    """delta_i = sum_k dO_ik * O_ik, one value per query row.

    delta appears in dS = P o (dP - delta) ([Interrogating-5] "What does the
    backward pass do without P?") without a definition on the pages.  The
    reading taken: delta_i = sum_j P_ij dP_ij, the softmax-Jacobian term,
    which equals sum_k dO_ik O_ik because dP = dO V^T and O = P V.
    """
    return (_f64(o) * _f64(dout)).sum(axis=-1)


def attention_bwd_ref(q, k, v, dout, scale: float, causal: bool = False,
                      row_chunk: int = 256):
    """Backward of O = softmax(scale Q K^T) V by the chain rule.

    [Interrogating-5] "What does the backward pass do without P?":
    dV = P^T dO and dS = P o (dP - delta), with dP = dO V^T and
    delta_i = sum_j P_ij dP_ij.  Through S = scale Q K^T:
    dQ = scale dS K and dK = scale dS^T Q.  P is formed from the plain
    softmax here (the oracle may keep it; only the GPU path recomputes).
    Returns ``(dQ, dK, dV)``.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    nq = q.shape[-2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for idx in _heads(q):
        for r0 in range(0, nq, row_chunk):
            r1 = min(nq, r0 + row_chunk)
            qc = q[idx][r0:r1]
            doc = dout[idx][r0:r1]
            s = _masked_scores(qc, k[idx], scale, causal, r0)
            p = _row_softmax(s)[0]
            dv[idx] += p.T @ doc
            dp = doc @ v[idx].T
            delta = (p * dp).sum(axis=1)
            ds = p * (dp - delta[:, None])
            dq[idx][r0:r1] = scale * (ds @ k[idx])
            dk[idx] += scale * (ds.T @ qc)
    return dq, dk, dv


def online_softmax_ref(q, k, v, scale: float, tile: int, causal: bool = False,
                       rescale_threshold: float | None = None):
    """Tile-by-tile streaming softmax attention, as the pages state it.

    Keys and values are visited in tiles of ``tile`` rows.  Each query row
    carries the running maximum m, the running sum l = sum e^{s-m} and the
    unnormalised output o = sum e^{s-m} v.  When a tile raises the maximum to
    m', l and o are multiplied by the correction factor e^{m-m'} before the
    tile's own terms, computed relative to m', are added ([Interrogating-5]
    "How can you softmax a row you never see whole?", online-softmax update
    equation; the same step in [FA-versions] "FlashAttention (2022)" and
    [datarekha] "The online softmax - why it's exact").  At the end
    O = o / l and LSE = m + log l.

    ``rescale_threshold`` (natural-log units) is the conditional rescale of
    [Interrogating-5] "Why did Blackwell need FlashAttention-4?": when the new
    maximum exceeds the one in use by no more than the threshold, the
    correction is skipped and the stale maximum stays the reference for the
    exponentials, l, o and the final LSE.  ``None`` always rescales.

    Returns ``(O, LSE)``.  Reference-only: it pins the algorithm, and is never
    the comparison target for the GPU.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, nk = q.shape[-2], k.shape[-2]
    o_out = np.zeros(q.shape[:-1] + (v.shape[-1],))
    lse_out = np.zeros(q.shape[:-1])
    for idx in _heads(q):
        qh, kh, vh = q[idx], k[idx], v[idx]
        m = np.full(nq, -np.inf)
        l = np.zeros(nq)
        acc = np.zeros((nq, vh.shape[-1]))
        for t0 in range(0, nk, tile):
            t1 = min(nk, t0 + tile)
            s = _masked_scores(qh, kh[t0:t1], scale, False, 0)
            if causal:
                i = np.arange(nq)[:, None]
                j = np.arange(t0, t1)[None, :]
                s = np.where(j > i, -np.inf, s)
            m_new = np.maximum(m, s.max(axis=1))
            if rescale_threshold is not None:
                keep = np.isfinite(m) & (m_new - m <= rescale_threshold)
                m_new = np.where(keep, m, m_new)
            # correction factor e^{m - m'}; a row that has seen only -inf so far
            # has l = 0 and o = 0, so its factor is immaterial (kept at 1)
            with np.errstate(invalid="ignore"):
                alpha = np.exp(m - m_new)
            alpha = np.where(np.isnan(alpha), 1.0, alpha)
            m_ref = np.where(np.isfinite(m_new), m_new, 0.0)
            p = np.where(np.isfinite(s), np.exp(s - m_ref[:, None]), 0.0)
            l = alpha * l + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ vh[t0:t1]
            m = m_new
        o_out[idx] = acc / l[:, None]
        lse_out[idx] = m + np.log(l)
    return o_out, lse_out
