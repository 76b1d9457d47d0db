"""Checks that pin the float64 oracle to facts that do not come from its own code.

Each ``pin_*`` function takes the oracle module as an argument (so the mutation
test can run the same checks against a deliberately broken copy) and raises
AssertionError when the oracle disagrees with:
  * a brute-force scalar loop (pure Python, ``math.exp``) on tiny inputs,
  * PyTorch's library attention/softmax in float64,
  * closed forms and invariants (rows of P sum to 1, constant V, single key,
    causal first row, window limits, scale 0, hard-max limit, key permutation),
  * the hand-derived golden fixtures under tests/golden/,
  * the split/merge identity of the sequence-axis reduction.
"""

from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    diff = np.where(both_inf, 0.0, np.abs(a - b))
    assert np.all(np.isfinite(diff)), f"{what}: non-finite difference"
    err = float(diff.max()) if diff.size else 0.0
    assert err <= tol * max(1.0, float(np.nanmax(np.abs(np.where(np.isinf(b), 0, b))))
                            if b.size else 1.0), f"{what}: max err {err}"


def _rand(shape, rng):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- brute force
def brute_attention(q, k, v, causal, window, scale):
    """Scalar loops over (b, i, h, j) with math.exp: no arrays, no masking
    matrix, no max-subtraction shortcut shared with the oracle."""
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    dv = v.shape[3]
    G = Hq // Hkv
    O = np.zeros((B, N, Hq, dv))
    LSE = np.zeros((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for i in range(N):
                scores = []
                for j in range(k.shape[1]):
                    if causal and j > i:
                        continue
                    if window >= 0:
                        if i - j > window:
                            continue
                        if not causal and j - i > window:
                            continue
                    s = 0.0
                    for t in range(d):
                        s += float(q[b, i, h, t]) * float(k[b, j, hk, t])
                    scores.append((j, scale * s))
                if not scores:
                    LSE[b, h, i] = -math.inf
                    continue
                top = max(s for _, s in scores)
                ws = [(j, math.exp(s - top)) for j, s in scores]
                Z = sum(w for _, w in ws)
                for t in range(dv):
                    O[b, i, h, t] = sum(w * float(v[b, j, hk, t]) for j, w in ws) / Z
                LSE[b, h, i] = top + math.log(Z)
    return O, LSE


def pin_bruteforce(orc, seed=0):
    rng = np.random.default_rng(seed)
    cases = [
        (1, 5, 2, 2, 3, False, -1, 0.7),
        (2, 7, 4, 2, 4, True, -1, 0.5),
        (1, 8, 2, 1, 3, False, 2, 1.3),
        (1, 9, 3, 3, 2, True, 3, 0.9),
        (1, 6, 2, 2, 5, False, 0, 0.4),
    ]
    for B, N, Hq, Hkv, d, causal, window, scale in cases:
        q = _rand((B, N, Hq, d), rng)
        k = _rand((B, N, Hkv, d), rng)
        v = _rand((B, N, Hkv, d + 1), rng)
        O, L = orc.attention(q, k, v, causal=causal, window=window, scale=scale)
        Ob, Lb = brute_attention(q, k, v, causal, window, scale)
        _close(O, Ob, 1e-12, f"brute O {causal} {window}")
        _close(L, Lb, 1e-12, f"brute LSE {causal} {window}")


# --------------------------------------------------------------- library check
def pin_torch_sdpa(orc, seed=1):
    """PyTorch's float64 CPU attention (a library routine) on the tiny
    non-causal shape, plus causal, windowed and grouped-head variants."""
    g = torch.Generator().manual_seed(seed)
    # the first case is the tiny non-causal workload's shape (B=1, H=2, N=256, d=64)
    for idx, (causal, window, Hq, Hkv) in enumerate([(False, -1, 2, 2), (True, -1, 2, 2),
                                                     (False, 17, 4, 2), (True, 9, 4, 1)]):
        B, N, d = 1, (256 if idx == 0 else 64), 64
        q = torch.randn(B, N, Hq, d, generator=g, dtype=torch.float64)
        k = torch.randn(B, N, Hkv, d, generator=g, dtype=torch.float64)
        v = torch.randn(B, N, Hkv, d, generator=g, dtype=torch.float64)
        scale = 1.0 / math.sqrt(d)
        qt, kt, vt = (x.transpose(1, 2) for x in (q, k, v))
        G = Hq // Hkv
        kt = kt.repeat_interleave(G, dim=1)
        vt = vt.repeat_interleave(G, dim=1)
        i = torch.arange(N)[:, None]
        j = torch.arange(N)[None, :]
        mask = torch.ones(N, N, dtype=torch.bool)
        if causal:
            mask &= j <= i
        if window >= 0:
            mask &= ((i - j) <= window) if causal else ((i - j).abs() <= window)
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                               scale=scale)
        scores = torch.matmul(qt, kt.transpose(-1, -2)) * scale
        lse_ref = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
        O, L = orc.attention(q.numpy(), k.numpy(), v.numpy(), causal=causal, window=window,
                             scale=scale)
        _close(O, ref.transpose(1, 2).numpy(), 1e-10, f"sdpa O {causal} {window}")
        _close(L, lse_ref.numpy(), 1e-10, f"sdpa LSE {causal} {window}")


# ------------------------------------------------------- closed forms, invariants
def pin_rows_sum_to_one(orc, seed=2):
    rng = np.random.default_rng(seed)
    for causal, window in [(False, -1), (True, -1), (False, 3), (True, 2)]:
        q, k, v = _rand((12, 6), rng), _rand((12, 6), rng), _rand((12, 5), rng)
        vis = orc.visible(12, 12, causal, window)
        _, _, P = orc.attention_head(q, k, v, 0.8, vis, return_p=True)
        _close(P.sum(axis=1), np.ones(12), 1e-12, "row sums")
        assert np.all(P[~vis] == 0.0), "masked keys must carry exactly zero weight"
        assert np.all(P[vis] > 0.0), "visible keys must carry positive weight"


def pin_constant_v(orc, seed=3):
    rng = np.random.default_rng(seed)
    q = _rand((1, 10, 2, 4), rng)
    k = _rand((1, 10, 2, 4), rng)
    v = np.broadcast_to(np.array([1.5, -2.0, 0.25]), (1, 10, 2, 3)).copy()
    for causal, window in [(False, -1), (True, -1), (False, 2)]:
        O, _ = orc.attention(q, k, v, causal=causal, window=window, scale=0.6)
        _close(O, np.broadcast_to(v[:, :, :1, :], O.shape), 1e-12, "constant V")


def pin_single_key(orc, seed=4):
    rng = np.random.default_rng(seed)
    q = _rand((1, 1, 3, 5), rng)
    k = _rand((1, 1, 3, 5), rng)
    v = _rand((1, 1, 3, 4), rng)
    O, L = orc.attention(q, k, v, scale=0.7)
    _close(O, v, 1e-12, "single key O")
    s = 0.7 * np.einsum("bnhd,bnhd->bhn", q, k)
    _close(L, s, 1e-12, "single key LSE")


def pin_causal_first_row(orc, seed=5):
    rng = np.random.default_rng(seed)
    q, k, v = _rand((2, 9, 2, 4), rng), _rand((2, 9, 2, 4), rng), _rand((2, 9, 2, 3), rng)
    O, L = orc.attention(q, k, v, causal=True, scale=1.1)
    _close(O[:, 0], v[:, 0], 1e-12, "causal row 0 O")
    _close(L[:, :, 0], 1.1 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]), 1e-12,
           "causal row 0 LSE")


def pin_window_limits(orc, seed=6):
    rng = np.random.default_rng(seed)
    N = 11
    q, k, v = _rand((1, N, 2, 4), rng), _rand((1, N, 2, 4), rng), _rand((1, N, 2, 3), rng)
    full = orc.attention(q, k, v, scale=0.5)
    wide = orc.attention(q, k, v, window=N - 1, scale=0.5)
    _close(wide[0], full[0], 1e-12, "window >= N-1 is non-causal")
    _close(wide[1], full[1], 1e-12, "window >= N-1 LSE")
    zero = orc.attention(q, k, v, window=0, scale=0.5)
    _close(zero[0], v, 1e-12, "window 0 returns v_i")
    # causal + window w: row i sees keys max(0, i-w)..i; with scale 0 the output
    # is the plain mean of those values and LSE = ln(count).
    O, L = orc.attention(q, k, v, causal=True, window=3, scale=0.0)
    for i in range(N):
        lo = max(0, i - 3)
        _close(O[0, i], v[0, lo:i + 1].mean(axis=0), 1e-12, "causal window mean")
        _close(L[0, :, i], np.full(2, math.log(i + 1 - lo)), 1e-12, "causal window count")


def pin_scale_zero(orc, seed=7):
    rng = np.random.default_rng(seed)
    N = 13
    q, k, v = _rand((1, N, 1, 4), rng), _rand((1, N, 1, 4), rng), _rand((1, N, 1, 2), rng)
    for causal, window in [(False, -1), (True, -1), (False, 4)]:
        O, L = orc.attention(q, k, v, causal=causal, window=window, scale=0.0)
        for i in range(N):
            lo = 0 if window < 0 else max(0, i - window)
            hi = i if causal else (N - 1 if window < 0 else min(N - 1, i + window))
            _close(O[0, i, 0], v[0, lo:hi + 1, 0].mean(axis=0), 1e-12, "scale 0 mean")
            _close(L[0, 0, i], math.log(hi - lo + 1), 1e-12, "scale 0 LSE")


def pin_hardmax_limit(orc, seed=8):
    """Very large scale: the softmax tends to the arg-max; LSE tends to the max
    score.  Catches a missing max-subtraction (exp overflow) as well."""
    rng = np.random.default_rng(seed)
    q, k, v = _rand((1, 6, 1, 3), rng), _rand((1, 6, 1, 3), rng), _rand((1, 6, 1, 2), rng)
    scale = 1e4
    O, L = orc.attention(q, k, v, scale=scale)
    s = scale * (q[0, :, 0] @ k[0, :, 0].T)
    for i in range(6):
        srt = np.sort(s[i])
        assert srt[-1] - srt[-2] > 50, "test input needs a clear maximum"
        _close(O[0, i, 0], v[0, int(np.argmax(s[i])), 0], 1e-12, "hard max O")
        _close(L[0, 0, i], srt[-1], 1e-12, "hard max LSE")


def pin_key_permutation(orc, seed=9):
    rng = np.random.default_rng(seed)
    q, k, v = _rand((1, 10, 2, 4), rng), _rand((1, 10, 2, 4), rng), _rand((1, 10, 2, 3), rng)
    perm = rng.permutation(10)
    a = orc.attention(q, k, v, scale=0.9)
    b = orc.attention(q, k[:, perm], v[:, perm], scale=0.9)
    _close(a[0], b[0], 1e-12, "key permutation O")
    _close(a[1], b[1], 1e-12, "key permutation LSE")


def pin_gqa_mapping(orc, seed=10):
    """Query head h reads kv head h // (Hq/Hkv): give each kv head a constant,
    distinct V and read it back."""
    rng = np.random.default_rng(seed)
    Hq, Hkv = 6, 3
    q, k = _rand((1, 5, Hq, 4), rng), _rand((1, 5, Hkv, 4), rng)
    v = np.zeros((1, 5, Hkv, 2))
    for hk in range(Hkv):
        v[:, :, hk, :] = 10.0 * (hk + 1)
    O, _ = orc.attention(q, k, v, scale=0.5)
    for h in range(Hq):
        _close(O[0, :, h], np.full((5, 2), 10.0 * (h // 2 + 1)), 1e-12, "GQA mapping")


def pin_band_equals_dense(orc, seed=11):
    rng = np.random.default_rng(seed)
    N, w = 40, 5
    q, k, v = _rand((2, N, 2, 4), rng), _rand((2, N, 2, 4), rng), _rand((2, N, 2, 3), rng)
    a = orc.attention(q, k, v, window=w, scale=0.7)
    b = orc.attention_band(q, k, v, window=w, scale=0.7, block=8)
    _close(a[0], b[0], 1e-12, "band O")
    _close(a[1], b[1], 1e-12, "band LSE")


def pin_golden(orc):
    for name in sorted(os.listdir(GOLDEN)):
        if not name.endswith(".json"):
            continue
        with open(os.path.join(GOLDEN, name)) as f:
            fx = json.load(f)
        if fx["kind"] == "prefill":
            O, L = orc.attention(np.array(fx["q"]), np.array(fx["k"]), np.array(fx["v"]),
                                 causal=fx["causal"], window=fx["window"], scale=fx["scale"])
            _close(O, np.array(fx["O"]), 1e-12, name + " O")
            _close(L, np.array(fx["LSE"]), 1e-12, name + " LSE")
        elif fx["kind"] == "merge":
            parts = [(m, l, np.array(o)) for m, l, o in fx["partials"]]
            M, Lm, Om = orc.lse_merge(parts[0], parts[1])
            _close([M, Lm], fx["merged"][:2], 1e-12, name + " merged m,l")
            _close(Om, np.array(fx["merged"][2]), 1e-12, name + " merged o")
            O, L = orc.tree_combine(parts)
            _close(O, np.array(fx["O"]), 1e-12, name + " O")
            _close(L, fx["LSE"], 1e-12, name + " LSE")


def pin_split_merge(orc, seed=12):
    """Any partition of the key axis, merged in any bracketing, equals the
    unsplit decode (the sequence-axis reduction is associative)."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, L, d = 2, 4, 2, 37, 5
    q = _rand((B, Hq, d), rng)
    kc, vc = _rand((B, L, Hkv, d), rng), _rand((B, L, Hkv, d), rng)
    kv_len = np.array([37, 23])
    O, LSE = orc.decode(q, kc, vc, kv_len, scale=0.6)
    for chunk, S in [(37, 1), (8, 5), (5, 8), (1, 37), (16, 3), (4, 16)]:
        m, l, o = orc.split_partials(q, kc, vc, kv_len, chunk, S, scale=0.6)
        Oc, Lc = orc.combine_rows(m.reshape(B * Hq, S), l.reshape(B * Hq, S),
                                  o.reshape(B * Hq, S, d))
        _close(Oc.reshape(B, Hq, d), O, 1e-12, f"split {chunk}x{S} O")
        _close(Lc.reshape(B, Hq), LSE, 1e-12, f"split {chunk}x{S} LSE")
    # random bracketings of the merge of random partitions
    s = 0.6 * (kc[0, :, 0] @ q[0, 0])
    full = orc.partial(s, vc[0, :, 0])
    for _ in range(20):
        cuts = np.sort(rng.choice(np.arange(1, L), size=rng.integers(1, 8), replace=False))
        pieces = [orc.partial(s[a:b], vc[0, a:b, 0])
                  for a, b in zip(itertools.chain([0], cuts), itertools.chain(cuts, [L]))]
        while len(pieces) > 1:
            i = int(rng.integers(0, len(pieces) - 1))
            pieces[i:i + 2] = [orc.lse_merge(pieces[i], pieces[i + 1])]
        _close([pieces[0][0], pieces[0][1]], [full[0], full[1]], 1e-12, "bracketing m,l")
        _close(pieces[0][2], full[2], 1e-12, "bracketing o")
    # decode equals prefill's last row under a causal mask (same definition)
    qq = np.zeros((1, L, Hq, d))
    qq[0, L - 1] = q[0]
    Op, Lp = orc.attention(qq, kc[:1], vc[:1], causal=True, scale=0.6)
    _close(Op[0, L - 1], O[0], 1e-12, "decode vs causal last row")
    _close(Lp[0, :, L - 1], LSE[0], 1e-12, "decode vs causal last row LSE")


def pin_empty_rows(orc):
    """A row with no visible key: O = 0, LSE = -inf; empty partials are the identity."""
    O, L = orc.decode(np.ones((1, 2, 3)), np.ones((1, 4, 1, 3)), np.ones((1, 4, 1, 3)),
                      np.array([0]), scale=1.0)
    assert np.all(O == 0.0) and np.all(np.isneginf(L))
    ident = orc.partial(np.zeros(0), np.zeros((0, 3)))
    a = orc.partial(np.array([0.3, -1.0]), np.arange(6.0).reshape(2, 3))
    m = orc.lse_merge(ident, a)
    _close([m[0], m[1]], [a[0], a[1]], 1e-15, "identity merge")
    _close(m[2], a[2], 1e-15, "identity merge o")


def pin_varlen_bruteforce(orc, seed=13):
    """Packed sequences: each sequence equals the brute-force loop on that
    sequence alone (positions counted from its first row), and no row of one
    sequence sees another's keys."""
    rng = np.random.default_rng(seed)
    cu = [0, 3, 3, 8, 9, 15]  # lengths 3, 0 (empty), 5, 1, 6
    T, Hq, Hkv, d = cu[-1], 4, 2, 3
    q = _rand((T, Hq, d), rng)
    k = _rand((T, Hkv, d), rng)
    v = _rand((T, Hkv, d + 1), rng)
    for causal, window in [(False, -1), (True, -1), (False, 1), (True, 2)]:
        O, L = orc.attention_varlen(q, k, v, cu, causal=causal, window=window, scale=0.6)
        for s in range(len(cu) - 1):
            a, e = cu[s], cu[s + 1]
            if e == a:
                continue
            Ob, Lb = brute_attention(q[None, a:e], k[None, a:e], v[None, a:e], causal, window, 0.6)
            _close(O[a:e], Ob[0], 1e-12, f"varlen O seq {s} {causal} {window}")
            _close(L[:, a:e], Lb[0], 1e-12, f"varlen LSE seq {s} {causal} {window}")


def pin_backward_finite_differences(orc, seed=14):
    """Gradients against central differences of the brute-force forward's
    loss sum(dO * O): independent of the analytical backward formulas."""
    rng = np.random.default_rng(seed)
    for B, N, Hq, Hkv, d, causal, window, scale in [(1, 4, 2, 1, 3, True, -1, 0.8),
                                                   (1, 5, 2, 2, 2, False, 1, 1.1)]:
        q = _rand((B, N, Hq, d), rng)
        k = _rand((B, N, Hkv, d), rng)
        v = _rand((B, N, Hkv, d), rng)
        dO = _rand((B, N, Hq, d), rng)
        dQ, dK, dV = orc.attention_backward(q, k, v, dO, causal=causal, window=window,
                                            scale=scale)

        def loss(q_, k_, v_):
            O, _ = brute_attention(q_, k_, v_, causal, window, scale)
            return float((O * dO).sum())

        eps = 1e-6
        for arr, grad, which in ((q, dQ, 0), (k, dK, 1), (v, dV, 2)):
            num = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                plus, minus = arr.copy(), arr.copy()
                plus[idx] += eps
                minus[idx] -= eps
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which], args_m[which] = plus, minus
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            _close(grad, num, 1e-7, f"finite differences {which} {causal} {window}")


def pin_backward_torch_autograd(orc, seed=15):
    """Library cross-check: torch float64 autograd through a plain masked
    softmax attention, grouped heads included."""
    rng = np.random.default_rng(seed)
    B, N, Hq, Hkv, d = 2, 9, 4, 2, 5
    for causal, window in [(False, -1), (True, -1), (True, 3), (False, 2)]:
        q = _rand((B, N, Hq, d), rng)
        k = _rand((B, N, Hkv, d), rng)
        v = _rand((B, N, Hkv, d), rng)
        dO = _rand((B, N, Hq, d), rng)
        tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
        G = Hq // Hkv
        kk = tk.repeat_interleave(G, dim=2)
        vv = tv.repeat_interleave(G, dim=2)
        S = torch.einsum("bihd,bjhd->bhij", tq, kk) * 0.7
        i = torch.arange(N)[:, None]
        j = torch.arange(N)[None, :]
        vis = torch.ones(N, N, dtype=torch.bool)
        if causal:
            vis &= j <= i
        if window >= 0:
            vis &= ((i - j) <= window) if causal else ((i - j).abs() <= window)
        S = S.masked_fill(~vis, float("-inf"))
        O = torch.einsum("bhij,bjhd->bihd", torch.softmax(S, dim=-1), vv)
        (O * torch.tensor(dO)).sum().backward()
        dQ, dK, dV = orc.attention_backward(q, k, v, dO, causal=causal, window=window, scale=0.7)
        _close(dQ, tq.grad.numpy(), 1e-12, f"autograd dQ {causal} {window}")
        _close(dK, tk.grad.numpy(), 1e-12, f"autograd dK {causal} {window}")
        _close(dV, tv.grad.numpy(), 1e-12, f"autograd dV {causal} {window}")


def brute_decode(q, kc, vc, kv_len, scale):
    """Scalar loops for single-query decode: query head h of sequence b scores
    keys 0 .. kv_len[b]-1 of kv head h // (Hq / Hkv) with math.exp."""
    B, Hq, d = q.shape
    Hkv = kc.shape[2]
    dv = vc.shape[3]
    G = Hq // Hkv
    O = np.zeros((B, Hq, dv))
    LSE = np.full((B, Hq), -math.inf)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            scores = []
            for j in range(int(kv_len[b])):
                s = 0.0
                for t in range(d):
                    s += float(q[b, h, t]) * float(kc[b, j, hk, t])
                scores.append(scale * s)
            if not scores:
                continue
            top = max(scores)
            ws = [math.exp(s - top) for s in scores]
            Z = sum(ws)
            for t in range(dv):
                O[b, h, t] = sum(w * float(vc[b, j, hk, t]) for j, w in enumerate(ws)) / Z
            LSE[b, h] = top + math.log(Z)
    return O, LSE


def pin_attention_rows_bruteforce(orc, seed=16):
    """``attention_rows`` (the spot-check form used on full-size launches)
    against the brute-force loop on the same rows: unsorted row lists that
    include the first and the last row, every mask kind, grouped heads with
    Hq / Hkv = 3, several batches, numpy and torch bf16 inputs."""
    rng = np.random.default_rng(seed)
    cases = [
        (2, 11, 6, 2, 3, False, -1, 0.7),
        (2, 12, 6, 2, 4, True, -1, 0.5),
        (2, 10, 3, 1, 3, False, 2, 1.2),
        (2, 13, 6, 2, 3, True, 3, 0.9),
    ]
    for B, N, Hq, Hkv, d, causal, window, scale in cases:
        q = _rand((B, N, Hq, d), rng)
        k = _rand((B, N, Hkv, d), rng)
        v = _rand((B, N, Hkv, d + 2), rng)
        Ob, Lb = brute_attention(q, k, v, causal, window, scale)
        rows = [N - 1, 0, N // 2, 3, 1]
        for b in range(B):
            for h in range(Hq):
                O, L = orc.attention_rows(q, k, v, b, h, rows, causal=causal, window=window,
                                          scale=scale)
                _close(O, Ob[b, rows, h], 1e-12, f"rows O b{b} h{h} {causal} {window}")
                _close(L, Lb[b, h, rows], 1e-12, f"rows LSE b{b} h{h} {causal} {window}")
    # torch bf16 inputs (what the GPU tests pass) go through the same path
    qt = torch.randn(1, 9, 3, 4, generator=torch.Generator().manual_seed(seed)).bfloat16()
    kt = torch.randn(1, 9, 1, 4, generator=torch.Generator().manual_seed(seed + 1)).bfloat16()
    vt = torch.randn(1, 9, 1, 4, generator=torch.Generator().manual_seed(seed + 2)).bfloat16()
    Ob, Lb = brute_attention(qt.double().numpy(), kt.double().numpy(), vt.double().numpy(),
                             True, -1, 0.5)
    O, L = orc.attention_rows(qt, kt, vt, 0, 2, [8, 0, 4], causal=True, scale=0.5)
    _close(O, Ob[0, [8, 0, 4], 2], 1e-12, "rows bf16 O")
    _close(L, Lb[0, 2, [8, 0, 4]], 1e-12, "rows bf16 LSE")


def pin_decode_heads_subset(orc, seed=17):
    """``decode`` against the brute-force decode loop, for all heads and for a
    scrambled subset of (sequence, head) pairs that hops between sequences and
    kv heads (so any cache of the per-(sequence, kv head) keys must be rebuilt
    between them); pairs outside the subset stay zero.  Ragged lengths include
    a one-key sequence."""
    rng = np.random.default_rng(seed)
    for B, Hq, Hkv, L, d, kv_len in [(3, 6, 2, 14, 3, [9, 1, 14]),
                                     (2, 8, 2, 11, 4, [11, 6])]:
        q = _rand((B, Hq, d), rng)
        kc, vc = _rand((B, L, Hkv, d), rng), _rand((B, L, Hkv, d + 1), rng)
        kv = np.array(kv_len)
        Ob, Lb = brute_decode(q, kc, vc, kv, 0.8)
        O, LSE = orc.decode(q, kc, vc, kv, scale=0.8)
        _close(O, Ob, 1e-12, "decode O all heads")
        _close(LSE, Lb, 1e-12, "decode LSE all heads")
        pairs = [(B - 1, Hq - 1), (0, 0), (B - 1, 1), (1, Hq // 2), (0, Hq - 2), (B - 1, Hq // 2),
                 (0, 1)]
        O, LSE = orc.decode(q, kc, vc, kv, scale=0.8, heads=pairs)
        for b in range(B):
            for h in range(Hq):
                if (b, h) in pairs:
                    _close(O[b, h], Ob[b, h], 1e-12, f"decode subset O b{b} h{h}")
                    _close(LSE[b, h], Lb[b, h], 1e-12, f"decode subset LSE b{b} h{h}")
                else:
                    assert np.all(O[b, h] == 0.0) and LSE[b, h] == 0.0, "untouched pair"


ALL_PINS = [
    pin_bruteforce, pin_torch_sdpa, pin_rows_sum_to_one, pin_constant_v, pin_single_key,
    pin_causal_first_row, pin_window_limits, pin_scale_zero, pin_hardmax_limit,
    pin_key_permutation, pin_gqa_mapping, pin_band_equals_dense, pin_golden,
    pin_split_merge, pin_empty_rows, pin_varlen_bruteforce, pin_backward_finite_differences,
    pin_backward_torch_autograd, pin_attention_rows_bruteforce, pin_decode_heads_subset,
]
