"""Oracle: scaled-dot-product attention, forward and backward, in float64.

Test infrastructure only (see the package docstring): nothing on the product
path may import this module.

What it computes is the plain definition of the quantities the FlashAttention-2
kernels produce, written out with explicit score matrices.  The online-softmax
recurrence of the kernels reaches the same numbers up to rounding order, so the
oracle does not follow the recurrence; it follows the definitions.

Sources (page titles and items):

* "vision-rs 0.1.1 flash_attn2.rs", ``flash_attention2_forward``: the layout
  ``[BATCH*N_HEADS, N_CTX, HEAD_DIM]`` row-major, the score
  ``sum(q*k) * softmax_scale``, the output ``acc / l`` and the saved
  log-sum-exp ``m + log(l)`` (natural log, of the scaled scores).
* same page, ``flash_attention2_backward_dq`` and
  ``flash_attention2_backward_dkv``: ``D = rowsum(O * dO)``,
  ``p = exp(q.k*scale - L)``, ``dS = p * (dO.v - D)``, ``dQ = sum dS*k*scale``,
  ``dK = sum dS*q*scale``, ``dV = sum p*dO``.
* "vyre-libs 0.7.2 flash_attention_2.rs", ``flash_attention_2_reference``:
  the scalar online softmax used there as a parity oracle; its result is the
  softmax-weighted average of V rows that :func:`forward` writes directly.

Inputs are float64 arrays (storage values already widened exactly).  All
contractions are ``numpy.matmul`` in float64.
"""
from __future__ import annotations

import numpy as np


def scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S[b, i, j] = scale * sum_d q[b, i, d] * k[b, j, d]  (flash_attn2.rs forward, score line)."""
    return scale * np.matmul(q, np.swapaxes(k, -1, -2))


def forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """Attention forward.  q [BH, Nq, d], k/v [BH, Nk, d] -> (O [BH, Nq, d], LSE [BH, Nq]).

    m_i = max_j s_ij;  p_ij = exp(s_ij - m_i);  l_i = sum_j p_ij;
    O_i = sum_j (p_ij / l_i) v_j;  LSE_i = m_i + ln l_i.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if q.shape[-2] == 0 or k.shape[-2] == 0:
        raise ValueError("attention needs at least one query and one key row")
    s = scores(q, k, scale)
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=-1, keepdims=True)
    probs = p / l
    o = np.matmul(probs, v)
    lse = m[..., 0] + np.log(l[..., 0])
    return o, lse


def forward_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, bh: int, rows):
    """Forward for selected query rows of one (batch, head) slice.

    Returns (O [len(rows), d], LSE [len(rows)]); the same definition as
    :func:`forward`, restricted to the rows asked for, so that full-size cases
    can be checked one row at a time.
    """
    rows = np.asarray(rows, dtype=np.int64)
    qs = np.asarray(q[bh, rows], dtype=np.float64)[None]
    o, lse = forward(qs, np.asarray(k[bh], dtype=np.float64)[None], np.asarray(v[bh], dtype=np.float64)[None], scale)
    return o[0], lse[0]


def probabilities(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """Row-normalised attention weights P = softmax(S) (the matrix the kernels never store)."""
    s = scores(np.asarray(q, dtype=np.float64), np.asarray(k, dtype=np.float64), scale)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    return p / p.sum(axis=-1, keepdims=True)


def backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, d_o: np.ndarray, scale: float):
    """Attention backward for loss gradient dO.  Returns (dQ, dK, dV), shapes of q, k, v.

    Follows flash_attn2.rs ``flash_attention2_backward_dq`` / ``_dkv``:
    D_i = sum_d O_id dO_id (with the oracle's own O);  P_ij = exp(s_ij - LSE_i);
    dV_j = sum_i P_ij dO_i;  dP_ij = dO_i . v_j;  dS_ij = P_ij (dP_ij - D_i);
    dQ_i = scale sum_j dS_ij k_j;  dK_j = scale sum_i dS_ij q_i.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    d_o = np.asarray(d_o, dtype=np.float64)
    o, lse = forward(q, k, v, scale)
    d_row = np.sum(o * d_o, axis=-1)
    p = np.exp(scores(q, k, scale) - lse[..., None])
    dv = np.matmul(np.swapaxes(p, -1, -2), d_o)
    dp = np.matmul(d_o, np.swapaxes(v, -1, -2))
    ds = p * (dp - d_row[..., None])
    dq = scale * np.matmul(ds, k)
    dk = scale * np.matmul(np.swapaxes(ds, -1, -2), q)
    return dq, dk, dv


def backward_slice(q, k, v, d_o, scale: float, bh: int, row_chunk: int = 1024, o=None, lse=None,
                   rounding_scales: bool = False):
    """Backward of one (batch, head) slice, with the score matrix built in row chunks.

    Same arithmetic as :func:`backward` for ``q[bh]`` etc.; chunking only bounds
    memory for long sequences (each chunk holds ``row_chunk x Nk`` scores).
    Returns (dQ [Nq, d], dK [Nk, d], dV [Nk, d]).

    ``o`` and ``lse`` ([BH, Nq, d] and [BH, Nq]) are the stored forward outputs that
    the backward kernels of flash_attn2.rs read from memory (``D_q = rowsum(O_q *
    dO_q)`` from the stored O, ``p = exp(q.k*scale - L)`` from the stored L); when
    given, D and P are formed from them instead of from this function's own exact O
    and LSE.  With ``rounding_scales``, three more arrays are returned, one per
    gradient element: the root-sum-square of the terms of its last product,
    sqrt(sum_j (dS_ij k_jc)^2) * scale for dQ, sqrt(sum_i (dS_ij q_ic)^2) * scale for
    dK and sqrt(sum_i (P_ij dO_ic)^2) for dV - the scale on which rounding each term's
    16-bit operand (dS, P) moves the sum.
    """
    qb = np.asarray(q[bh], dtype=np.float64)
    kb = np.asarray(k[bh], dtype=np.float64)
    vb = np.asarray(v[bh], dtype=np.float64)
    dob = np.asarray(d_o[bh], dtype=np.float64)
    nq = qb.shape[0]
    dq = np.zeros_like(qb)
    dk = np.zeros_like(kb)
    dv = np.zeros_like(vb)
    if rounding_scales:
        sq_q, sq_k, sq_v = np.zeros_like(qb), np.zeros_like(kb), np.zeros_like(vb)
    for r0 in range(0, nq, row_chunk):
        r1 = min(nq, r0 + row_chunk)
        s = scale * (qb[r0:r1] @ kb.T)
        if o is None or lse is None:
            m = s.max(axis=-1, keepdims=True)
            e = np.exp(s - m)
            l = e.sum(axis=-1, keepdims=True)
            o_rows = (e / l) @ vb
            lse_rows = m + np.log(l)
        if o is not None:
            o_rows = np.asarray(o[bh, r0:r1], dtype=np.float64)
        if lse is not None:
            lse_rows = np.asarray(lse[bh, r0:r1], dtype=np.float64)[:, None]
        p = np.exp(s - lse_rows)
        d_row = np.sum(o_rows * dob[r0:r1], axis=-1, keepdims=True)
        dv += p.T @ dob[r0:r1]
        ds = p * (dob[r0:r1] @ vb.T - d_row)
        dq[r0:r1] = scale * (ds @ kb)
        dk += scale * (ds.T @ qb[r0:r1])
        if rounding_scales:
            sq_q[r0:r1] = (ds * ds) @ (kb * kb)
            sq_k += (ds * ds).T @ (qb[r0:r1] * qb[r0:r1])
            sq_v += (p * p).T @ (dob[r0:r1] * dob[r0:r1])
    if rounding_scales:
        return dq, dk, dv, scale * np.sqrt(sq_q), scale * np.sqrt(sq_k), np.sqrt(sq_v)
    return dq, dk, dv


def psa_backward(packed: np.ndarray, d_o_lo: np.ndarray, d_o_hi: np.ndarray, scale: float) -> np.ndarray:
    """Gradient of the PSA packed buffer [4, BH, N, KD] through both attention calls.

    psa.rs ``psa_fa2_backward`` as ``FlashAttn2PsaRuntimeOp`` wires it for the V_lo
    (section 2) and V_hi (section 3) calls: sections 0 and 1 receive the sums of the
    two calls' dQ and dK, sections 2 and 3 each call's dV.
    """
    q, k, v_lo, v_hi = (np.asarray(packed[s], dtype=np.float64) for s in range(4))
    dq_lo, dk_lo, dv_lo = backward(q, k, v_lo, d_o_lo, scale)
    dq_hi, dk_hi, dv_hi = backward(q, k, v_hi, d_o_hi, scale)
    return np.stack([dq_lo + dq_hi, dk_lo + dk_hi, dv_lo, dv_hi])


def bwd_preprocess(o: np.ndarray, d_o: np.ndarray) -> np.ndarray:
    """D_i = sum_d O_id dO_id  (flash_attn2.rs backward, ``D_q = rowsum(O_q * dO_q)``)."""
    return np.sum(np.asarray(o, dtype=np.float64) * np.asarray(d_o, dtype=np.float64), axis=-1)
