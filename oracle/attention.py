"""Plain float64 CPU attention: the oracle that the CUDA path is checked against.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the library never does, and this module
imports nothing from the library.

What it computes is the plain definition of exact softmax attention, written
out step by step with the full score matrix materialised:

  S   = scale * Q K^T                       (one (batch, head) at a time)
  S  += mask   (-inf where a key is not visible to a query)
  m_i = max_j S_ij
  E   = exp(S - m)
  l_i = sum_j E_ij
  P   = E / l
  O   = P V
  LSE_i = m_i + ln l_i

Sources for the definition (page title, then section):
  * "FlashAttention" learn page (aiunderstanding.org), "Deep dive": standard
    attention scores every pair of tokens into an N-by-N matrix; "Technical
    insight" and the FAQ "How does FlashAttention's output compare to standard
    attention?": FlashAttention returns exactly the values of standard attention,
    only the order of the computation changes.  So the oracle is standard
    attention itself.
  * Arabic thread on extending context length (web3.ouzhyi.biz), point 1:
    local attention, where tokens attend only to their neighbours -> the window
    mask.
  * "Tree Attention: Topology-aware Decoding for Long-Context Attention on GPU
    Clusters" (express24.ir), abstract: the reduction along the sequence axis
    can be computed in parallel as a tree -> ``split_partials``, ``lse_merge``
    and ``tree_combine`` below.

Readings taken where the pages are silent (each is also listed in the design
notes): the scale is an explicit argument (1/sqrt(d) in every workload); causal
is square and top-left aligned (row i sees keys 0..i); a window w keeps keys
with |i - j| <= w, intersected with the causal mask when both are set; query
head h reads kv head h // (Hq / Hkv); a row with no visible key gives O = 0 and
LSE = -inf; LSE is the natural logarithm.

Every function here is pinned by the CPU tests (tests/test_oracle.py) against
facts that do not come from this file: a brute-force loop, a library softmax,
closed forms and invariants, and hand-derived golden fixtures.
"""

from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Any array-like (numpy, or a CPU torch tensor of any float dtype) to float64."""
    if hasattr(x, "detach"):  # torch tensor; bf16 has no numpy dtype
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def visible(nq: int, nk: int, causal: bool, window: int) -> np.ndarray:
    """Boolean [nq, nk] matrix: True where key j is visible to query i."""
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    vis = np.ones((nq, nk), dtype=bool)
    if causal:
        vis &= j <= i
    if window >= 0:
        if causal:
            vis &= (i - j) <= window
        else:
            vis &= np.abs(i - j) <= window
    return vis


def attention_head(q, k, v, scale: float, vis=None, return_p: bool = False):
    """One (batch, head): q [Nq, d], k [Nk, d], v [Nk, dv] -> O [Nq, dv], LSE [Nq].

    ``vis`` is the boolean visibility matrix (None: every key visible).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    S = scale * (q @ k.T)
    if vis is not None:
        S = np.where(vis, S, NEG_INF)
    m = S.max(axis=1, initial=NEG_INF)
    empty = ~np.isfinite(m)  # rows with no visible key (or no key at all)
    m_safe = np.where(empty, 0.0, m)
    E = np.exp(S - m_safe[:, None])
    l = E.sum(axis=1)
    l_safe = np.where(empty, 1.0, l)
    P = E / l_safe[:, None]
    O = P @ v
    with np.errstate(divide="ignore"):
        lse = np.where(empty, NEG_INF, m_safe + np.log(l_safe))
    if return_p:
        return O, lse, P
    return O, lse


def attention(q, k, v, causal: bool = False, window: int = -1, scale: float | None = None):
    """Prefill attention.

    q [B, N, Hq, d], k/v [B, N, Hkv, d] -> O [B, N, Hq, d] (float64), LSE [B, Hq, N].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    vis = visible(Nq, Nk, causal, window)
    O = np.zeros((B, Nq, Hq, v.shape[3]))
    LSE = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            O[b, :, h], LSE[b, h] = attention_head(q[b, :, h], k[b, :, hk], v[b, :, hk],
                                                   scale, vis)
    return O, LSE


def attention_varlen(q, k, v, cu_seqlens, causal: bool = False, window: int = -1,
                     scale: float | None = None):
    """Sequences packed back to back: sequence s owns rows [cu[s], cu[s+1]) of
    q [T, Hq, d] and k/v [T, Hkv, d] and attends only within itself (masks
    counted from its first row).  Returns O [T, Hq, d] and LSE [Hq, T]; rows
    outside every sequence stay NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, d = q.shape
    cu = [int(x) for x in cu_seqlens]
    O = np.full((T, Hq, v.shape[2]), np.nan)
    LSE = np.full((Hq, T), np.nan)
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        if e <= a:
            continue
        o_s, l_s = attention(q[None, a:e], k[None, a:e], v[None, a:e], causal=causal,
                             window=window, scale=scale)
        O[a:e] = o_s[0]
        LSE[:, a:e] = l_s[0]
    return O, LSE


def attention_backward(q, k, v, dO, causal: bool = False, window: int = -1,
                       scale: float | None = None):
    """Gradients of O = softmax(scale Q K^T + mask) V with respect to Q, K, V,
    given dO = dLoss/dO, in float64.  For each (batch, head), with P the
    attention weights of the forward definition:

      dV   = P^T dO
      dP   = dO V^T
      dS   = P * (dP - rowsum(P * dP))        (the softmax Jacobian, row by row)
      dQ   = scale dS K
      dK   = scale dS^T Q

    and rowsum(P * dP) = rowsum(dO * O).  Query heads of a group add their
    dK, dV into the shared kv head.  q [B, N, Hq, d], k/v [B, N, Hkv, d],
    dO [B, N, Hq, dv] -> dQ [B, N, Hq, d], dK [B, N, Hkv, d], dV [B, N, Hkv, dv].
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Nq, Hq, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    vis = visible(Nq, Nk, causal, window)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            _, _, P = attention_head(q[b, :, h], k[b, :, hk], v[b, :, hk], scale, vis,
                                     return_p=True)
            do = dO[b, :, h]
            dV[b, :, hk] += P.T @ do
            dP = do @ v[b, :, hk].T
            dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            dQ[b, :, h] = scale * (dS @ k[b, :, hk])
            dK[b, :, hk] += scale * (dS.T @ q[b, :, h])
    return dQ, dK, dV


def attention_rows(q, k, v, b: int, h: int, rows, causal: bool = False, window: int = -1,
                   scale: float | None = None):
    """O and LSE for selected query rows of one (b, h): the same definition,
    restricted to the requested rows (for spot checks of large launches)."""
    rows = np.asarray(rows)
    Hq, Hkv = q.shape[2], k.shape[2]
    hk = h // (Hq // Hkv)
    N = k.shape[1]
    d = q.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    vis = visible(N, N, causal, window)[rows]
    return attention_head(_f64(q[b, rows, h]), _f64(k[b, :, hk]), _f64(v[b, :, hk]),
                          scale, vis)


def attention_band(q, k, v, window: int, scale: float | None = None, block: int = 512,
                   heads=None):
    """Non-causal sliding-window attention computed only over the band of keys
    a block of rows can see.  Keys outside the band carry exactly zero weight
    (exp(-inf) = 0), so this equals ``attention(..., window=window)``; the CPU
    tests check that on small inputs.  ``heads`` optionally restricts the
    (b, h) pairs computed (the others are left at zero).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.zeros((B, N, Hq, v.shape[3]))
    LSE = np.zeros((B, Hq, N))
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        hk = h // G
        for r0 in range(0, N, block):
            r1 = min(N, r0 + block)
            c0 = max(0, r0 - window)
            c1 = min(N, r1 + window)
            i = np.arange(r0, r1)[:, None]
            j = np.arange(c0, c1)[None, :]
            vis = np.abs(i - j) <= window
            O[b, r0:r1, h], LSE[b, h, r0:r1] = attention_head(
                q[b, r0:r1, h], k[b, c0:c1, hk], v[b, c0:c1, hk], scale, vis)
    return O, LSE


def decode(q, k_cache, v_cache, kv_len, scale: float | None = None, heads=None):
    """Single-query decode: the newest token attends to every cached key.

    q [B, Hq, d], caches [B, Lmax, Hkv, d], kv_len [B] -> O [B, Hq, d], LSE [B, Hq].
    Only rows < kv_len[b] are read.  ``heads`` optionally restricts the (b, h)
    pairs computed (the others are left at zero).
    """
    B, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.zeros((B, Hq, v_cache.shape[3]))
    LSE = np.zeros((B, Hq))
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    cached = {}
    for b, h in todo:
        n = int(kv_len[b])
        hk = h // G
        if (b, hk) not in cached:
            cached.clear()
            cached[(b, hk)] = (_f64(k_cache[b, :n, hk]), _f64(v_cache[b, :n, hk]))
        kk, vv = cached[(b, hk)]
        o, lse = attention_head(_f64(q[b, h])[None, :], kk, vv, scale)
        O[b, h], LSE[b, h] = o[0], lse[0]
    return O, LSE


# ---------------------------------------------------------------------------
# Sequence-axis split and its logsumexp merge (Tree Attention abstract: the
# reduction across the sequence axis is associative and can be done as a tree).
# A partial over a set of keys J is the triple
#     m = max_{j in J} s_j,   l = sum_{j in J} exp(s_j - m),   o = sum_{j in J} exp(s_j - m) v_j
# and the empty set has the identity (-inf, 0, 0).
# ---------------------------------------------------------------------------

def partial(s, vv):
    """(m, l, o) of scores s [n] and values vv [n, dv] (n may be 0)."""
    s, vv = _f64(s), _f64(vv)
    if s.size == 0 or not np.isfinite(s.max()):
        return NEG_INF, 0.0, np.zeros(vv.shape[1])
    m = s.max()
    e = np.exp(s - m)
    return m, e.sum(), e @ vv


def lse_merge(a, b):
    """(m, l, o) + (m', l', o'): rescale both to the larger maximum and add."""
    m1, l1, o1 = a
    m2, l2, o2 = b
    M = max(m1, m2)
    if M == NEG_INF:
        return NEG_INF, 0.0, np.zeros_like(o1)
    w1 = 0.0 if m1 == NEG_INF else np.exp(m1 - M)
    w2 = 0.0 if m2 == NEG_INF else np.exp(m2 - M)
    return M, l1 * w1 + l2 * w2, o1 * w1 + o2 * w2


def tree_combine(parts):
    """Merge a list of partials pairwise, level by level (a balanced binary tree
    of depth ceil(log2 n)), then normalise: O = o / l, LSE = m + ln l."""
    level = list(parts)
    while len(level) > 1:
        nxt = [lse_merge(level[i], level[i + 1]) for i in range(0, len(level) - 1, 2)]
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    m, l, o = level[0]
    if l == 0.0:
        return np.zeros_like(o), NEG_INF
    return o / l, m + np.log(l)


def split_partials(q, k_cache, v_cache, kv_len, chunk: int, num_splits: int,
                   scale: float | None = None, heads=None):
    """Per (b, h, split c): the partial over keys [c*chunk, min((c+1)*chunk, kv_len[b])).

    Returns m, l [B, Hq, S] and o [B, Hq, S, dv] (natural-log units).
    """
    B, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dv = v_cache.shape[3]
    M = np.full((B, Hq, num_splits), NEG_INF)
    L = np.zeros((B, Hq, num_splits))
    Ov = np.zeros((B, Hq, num_splits, dv))
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in todo:
        n = int(kv_len[b])
        hk = h // G
        kk = _f64(k_cache[b, :n, hk])
        vv = _f64(v_cache[b, :n, hk])
        s = scale * (kk @ _f64(q[b, h]))
        for c in range(num_splits):
            lo, hi = c * chunk, min((c + 1) * chunk, n)
            M[b, h, c], L[b, h, c], Ov[b, h, c] = partial(s[lo:hi], vv[lo:hi])
    return M, L, Ov


def combine_rows(m, l, o):
    """``tree_combine`` for every row: m, l [R, S], o [R, S, dv] -> O [R, dv], LSE [R]."""
    m, l, o = _f64(m), _f64(l), _f64(o)
    R, S = m.shape
    O = np.zeros((R, o.shape[2]))
    LSE = np.zeros(R)
    for r in range(R):
        O[r], LSE[r] = tree_combine([(m[r, c], l[r, c], o[r, c]) for c in range(S)])
    return O, LSE
