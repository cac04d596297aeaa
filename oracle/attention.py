"""Plain, slow fp64 oracle for exact attention, written from the source pages.

TEST INFRASTRUCTURE ONLY.  ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py`` are the only callers.  Nothing here is
shared with the CUDA path: no kernels, helpers, constants or pre/post
processing.  Every array is converted to float64 on entry.

Pages cited (by title and section):

* "Flash Attention" (sgdbs.github.io, AI_Infra / GPUKernel / FlashAttention):
  "1.FlashAttention 整体结构", "2.Online Softmax", "3.Recomputation(重计算)详解",
  "4. 附录A" with 结论一 (matmul gradient), 结论二 (softmax Jacobian) and
  "反向传播的公式推导" (backward derivation).
* "FlashAttention 反向传播：删掉 O(N²) 的中间结果，怎么还能算对梯度？" (coreui.cn):
  the 1/sqrt(d_k) factor in dQ and dK.
* "当Attention遇见矩阵乘法：一个被忽视的真相" (cnnetsun.cn): §1.1 the
  scaled dot product, §2 the max-subtracted softmax.

Readings taken where the pages are silent or disagree (each is also listed in
the repository's design notes):

* scores are ``scale * Q Kᵀ`` with ``scale = 1/sqrt(d)`` by default;
* dS is the gradient with respect to the *scaled* scores, so
  ``dQ = scale * dS K`` and ``dK = scale * dSᵀ Q`` (the coreui.cn page divides
  both by sqrt(d_k); the tutorial drops the factor "for brevity");
* LSE is the natural-log log-sum-exp of the scaled scores of each row;
* causal means key j is visible to query i iff j <= i (square, top-left);
  with n_q queries over n_k >= n_q keys the queries are the last n_q positions
  of the sequence (tokens after a cached prefix, "2.Online Softmax" §七 item 3),
  so query i sees keys j <= i + (n_k - n_q);
* normalised partial results (O_k, LSE_k) over disjoint key sets merge with
  the §3.1/§4.1 merge taking m = LSE_k, ℓ = 1, Õ = O_k for each part.

Every function below has a pin in ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# Softmax building blocks ("2.Online Softmax")
# --------------------------------------------------------------------------


def naive_softmax(x):
    """y_i = e^{x_i} / sum_j e^{x_j} with no max subtraction.

    "2.Online Softmax" §1.1 (naive definition).  §1.2 explains why it overflows;
    the tests use it only as a negative control.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(x)
        return e / e.sum(axis=-1, keepdims=True)


def softmax_3pass(x):
    """Safe softmax, the three passes of "2.Online Softmax" §1.3.

    Pass 1 finds m = max_j x_j, pass 2 sums ℓ = Σ_j exp(x_j - m), pass 3
    writes y_j = exp(x_j - m) / ℓ.  Works along the last axis.  Returns
    (y, m, ℓ).  A row that is entirely -inf is not defined by the page and is
    rejected.
    """
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=-1, keepdims=True)                      # pass 1
    if not np.all(np.isfinite(m)):
        raise ValueError("softmax of a row with no finite entry is undefined")
    ell = np.exp(x - m).sum(axis=-1, keepdims=True)         # pass 2
    y = np.exp(x - m) / ell                                 # pass 3
    return y, m[..., 0], ell[..., 0]


def online_softmax_steps(x):
    """Element-at-a-time online normaliser, "2.Online Softmax" §2.1-2.2.

    Starts from m = -inf, ℓ = 0 (the table of §六 uses e^{-inf-1} = 0 for the
    first step) and for each new element applies
    m_new = max(m, x_i);  ℓ = ℓ·e^{m - m_new} + e^{x_i - m_new}.
    Returns the list of (m, rescale factor, ℓ) after every step so the worked
    example of §六 can be checked step by step.
    """
    m = -math.inf
    ell = 0.0
    steps = []
    for xi in np.asarray(x, dtype=np.float64).tolist():
        m_new = max(m, xi)
        factor = 0.0 if m == -math.inf else math.exp(m - m_new)
        ell = ell * factor + math.exp(xi - m_new)
        m = m_new
        steps.append((m, factor, ell))
    return steps


def merge_stats(m_a, l_a, m_b, l_b):
    """Two-block merge of (m, ℓ), "2.Online Softmax" §3.1 (boxed formula).

    m = max(m_A, m_B);  ℓ = ℓ_A·e^{m_A - m} + ℓ_B·e^{m_B - m}.
    A block that has seen nothing is (m, ℓ) = (-inf, 0) and contributes 0.
    """
    m = max(m_a, m_b)
    term_a = 0.0 if l_a == 0.0 else l_a * math.exp(m_a - m)
    term_b = 0.0 if l_b == 0.0 else l_b * math.exp(m_b - m)
    return m, term_a + term_b


def merge_outputs(m_a, l_a, o_a, m_b, l_b, o_b):
    """Merge of unnormalised outputs, "2.Online Softmax" §4.1 (boxed Õ formula).

    Õ = Õ_A·e^{m_A - m} + Õ_B·e^{m_B - m}, merged together with (m, ℓ).
    Returns (m, ℓ, Õ); the caller divides Õ by ℓ at the very end.
    """
    m, ell = merge_stats(m_a, l_a, m_b, l_b)
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    fa = 0.0 if l_a == 0.0 else math.exp(m_a - m)
    fb = 0.0 if l_b == 0.0 else math.exp(m_b - m)
    return m, ell, o_a * fa + o_b * fb


# --------------------------------------------------------------------------
# Attention forward, one head ("1.FlashAttention 整体结构" 一, standard form)
# --------------------------------------------------------------------------


def causal_mask(n_q, n_k):
    """Boolean [n_q, n_k] matrix, True where key j is visible to query i.

    Square: j <= i.  With fewer queries than keys the queries are the last n_q
    positions of the sequence ("2.Online Softmax" §七 item 3: the softmax state
    of a prefix is kept and later tokens extend it), so query i is at position
    i + n_k - n_q and sees j <= i + n_k - n_q.  More queries than keys would
    leave the first rows with no key at all and is rejected.
    """
    if n_q > n_k:
        raise ValueError("a causal mask with more queries than keys leaves rows with no key")
    return np.arange(n_k)[None, :] <= np.arange(n_q)[:, None] + (n_k - n_q)


def _scores(q, k, scale, causal):
    """S = scale·Q Kᵀ with masked entries set to -inf (materialised N×N)."""
    s = scale * (q @ k.T)
    if causal:
        s = np.where(causal_mask(q.shape[0], k.shape[0]), s, -np.inf)
    return s


def attention_forward_head(q, k, v, scale, causal=False):
    """O = softmax(scale·Q Kᵀ) V and LSE for one head, every matrix materialised.

    The three steps of "1.FlashAttention 整体结构" 一 (S, then P = softmax(S)
    row by row with the safe softmax of "2.Online Softmax" §1.3, then O = P V).
    LSE_i = m_i + ln ℓ_i, the statistic of "3.Recomputation" 三.
    Returns (O [N, d], LSE [N]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = _scores(q, k, scale, causal)
    p, m, ell = softmax_3pass(s)
    o = p @ v
    lse = m + np.log(ell)
    return o, lse


def attention_forward_rows(q, k, v, rows, scale, causal=False):
    """Forward for a chosen subset of query rows of one head (same definition).

    Row i of O depends only on q_i and all of K, V, so a sample of rows can be
    checked at sizes where the full N×N matrix is too large.
    """
    q_all = q
    q = np.asarray(q, dtype=np.float64)[np.asarray(rows)]
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = scale * (q @ k.T)
    if causal:
        n_q = np.shape(q_all)[0]
        s = np.where(causal_mask(n_q, k.shape[0])[np.asarray(rows)], s, -np.inf)
    p, m, ell = softmax_3pass(s)
    return p @ v, m + np.log(ell)


def tiled_forward_head(q, k, v, scale, block=64, causal=False):
    """The page's tiled forward, "2.Online Softmax" §4.2 pseudocode.

    One pass over K/V blocks of ``block`` keys (the last block may be short):
    per block j, S_j, m_j = rowmax(S_j), P_j = exp(S_j - m_j), ℓ_j = rowsum(P_j);
    m_new = max(m, m_j), α = e^{m - m_new}, β = e^{m_j - m_new};
    ℓ = αℓ + βℓ_j; O = αO + β P_j V_j; and O/ℓ once at the end (the deferred
    normalisation noted under the pseudocode).  Used only by the self-checks,
    which compare it with ``attention_forward_head``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    visible_all = causal_mask(n, k.shape[0]) if causal else None
    m = np.full(n, -np.inf)
    ell = np.zeros(n)
    o = np.zeros((n, v.shape[1]))
    for j0 in range(0, k.shape[0], block):
        kj = k[j0:j0 + block]
        vj = v[j0:j0 + block]
        s = scale * (q @ kj.T)
        if causal:
            s = np.where(visible_all[:, j0:j0 + kj.shape[0]], s, -np.inf)
        m_j = s.max(axis=1)
        # A row whose whole block is masked has m_j = -inf and adds nothing.
        live = np.isfinite(m_j)
        p = np.zeros_like(s)
        p[live] = np.exp(s[live] - m_j[live, None])
        l_j = p.sum(axis=1)
        m_new = np.maximum(m, m_j)
        alpha = np.where(np.isfinite(m), np.exp(m - np.where(np.isfinite(m_new), m_new, 0.0)), 0.0)
        beta = np.where(live, np.exp(m_j - np.where(np.isfinite(m_new), m_new, 0.0)), 0.0)
        ell = alpha * ell + beta * l_j
        o = alpha[:, None] * o + beta[:, None] * (p @ vj)
        m = m_new
    return o / ell[:, None], m + np.log(ell)


# --------------------------------------------------------------------------
# Backward, one head ("4. 附录A")
# --------------------------------------------------------------------------


def matmul_backward(a, b, dy):
    """附录A 结论一: for Y = A B, dA = dY Bᵀ and dB = Aᵀ dY."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    return dy @ b.T, a.T @ dy


def softmax_backward(p, dp):
    """附录A 结论二, row-wise: ds = p ⊙ (dp - ρ) with ρ = Σ_k p_k dp_k.

    ρ is computed directly from P and dP (not through the rowsum(dO⊙O)
    identity), so the identity itself can be checked against this function.
    """
    p = np.asarray(p, dtype=np.float64)
    dp = np.asarray(dp, dtype=np.float64)
    rho = (p * dp).sum(axis=-1, keepdims=True)
    return p * (dp - rho)


def attention_backward_head(q, k, v, do, scale, causal=False, return_intermediates=False):
    """dQ, dK, dV for one head with L = Σ dO ⊙ O, every matrix materialised.

    Follows "反向传播的公式推导" 三-四 in order: step 1 applies 结论一 to
    O = P V (dV = Pᵀ dO, dP = dO Vᵀ); step 2 applies 结论二 row by row
    (dS = P ⊙ (dP - rowsum(dP ⊙ P))); step 3 applies 结论一 to the unscaled
    product Q Kᵀ (dQ = dS K, dK = dSᵀ Q).  Because the scores are
    scale·Q Kᵀ, both of the last two carry the factor ``scale`` (the coreui.cn
    page's dQ = dS K / sqrt(d_k), dK = dSᵀ Q / sqrt(d_k)).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    s = _scores(q, k, scale, causal)
    p, _, _ = softmax_3pass(s)
    dp, dv = matmul_backward(p, v, do)          # step 1: O = P V
    ds = softmax_backward(p, dp)                # step 2: P = softmax(S)
    dq_u, dkt_u = matmul_backward(q, k.T, ds)   # step 3: Q Kᵀ = Q · (Kᵀ)
    dq = scale * dq_u
    dk = scale * dkt_u.T
    if return_intermediates:
        return dq, dk, dv, {"P": p, "dP": dp, "dS": ds}
    return dq, dk, dv


def attention_backward_rows(q, k, v, do, rows, scale, causal=False):
    """The backward restricted to a block of query rows of one head.

    The loss Σ dO ⊙ O is a sum over query rows, so each row's contribution to
    the gradients can be formed on its own with the same three steps as
    ``attention_backward_head``: for the rows R, dV_R = P_Rᵀ dO_R and
    dK_R = scale · dS_Rᵀ Q_R are those rows' (additive) shares of dV and dK,
    and dQ_R = scale · dS_R K is exact.  Returns (dQ_R, dK_R, dV_R).  Used to
    time a bounded sample of a large workload.
    """
    rows = np.asarray(rows)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    qr, dor = q[rows], do[rows]
    s = scale * (qr @ k.T)
    if causal:
        s = np.where(causal_mask(q.shape[0], k.shape[0])[rows], s, -np.inf)
    p, _, _ = softmax_3pass(s)
    dp, dv = matmul_backward(p, v, dor)
    ds = softmax_backward(p, dp)
    dq_u, dkt_u = matmul_backward(qr, k.T, ds)
    return scale * dq_u, scale * dkt_u.T, dv


def merge_partials(o_parts, lse_parts):
    """Merge normalised partial results over disjoint key sets of the same rows.

    "2.Online Softmax" §3.1 and §4.1 (boxed merges), applied part by part: a
    part with output O_k and statistic LSE_k is the state m = LSE_k, ℓ = 1,
    Õ = O_k (since Σ e^{s} over its keys is e^{LSE_k}).  A row a part never
    saw has LSE_k = -inf and contributes nothing.  Returns (O, LSE) with
    O = Õ/ℓ and LSE = m + ln ℓ, per row; rows no part saw get O = 0 and
    LSE = -inf.  Arrays: o_parts [P, rows, d], lse_parts [P, rows].
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    n_rows = lse_parts.shape[1]
    o = np.zeros(o_parts.shape[1:])
    lse = np.full(n_rows, -np.inf)
    for r in range(n_rows):
        m, ell, acc = -math.inf, 0.0, np.zeros(o_parts.shape[2])
        for k in range(o_parts.shape[0]):
            l_k = 0.0 if lse_parts[k, r] == -math.inf else 1.0
            m, ell, acc = merge_outputs(m, ell, acc, float(lse_parts[k, r]), l_k, o_parts[k, r])
        if ell > 0.0:
            o[r] = acc / ell
            lse[r] = m + math.log(ell)
    return o, lse


# --------------------------------------------------------------------------
# Batched wrappers over [B, H, N, d]
# --------------------------------------------------------------------------


def attention_forward(q, k, v, scale, causal=False):
    """Forward over [B, H, N, d] arrays; returns O [B,H,N,d] and LSE [B,H,N] in fp64."""
    q = np.asarray(q, dtype=np.float64)
    b_, h_, n, _ = q.shape
    o = np.empty(q.shape[:3] + (v.shape[-1],))
    lse = np.empty((b_, h_, n))
    for b in range(b_):
        for h in range(h_):
            o[b, h], lse[b, h] = attention_forward_head(q[b, h], k[b, h], v[b, h], scale, causal)
    return o, lse


def attention_backward(q, k, v, do, scale, causal=False):
    """Backward over [B, H, N, d] arrays; returns dQ, dK, dV in fp64."""
    q = np.asarray(q, dtype=np.float64)
    dq = np.empty(q.shape)
    dk = np.empty(np.shape(k))
    dv = np.empty(np.shape(v))
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            dq[b, h], dk[b, h], dv[b, h] = attention_backward_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
    return dq, dk, dv
