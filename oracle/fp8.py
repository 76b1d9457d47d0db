"""Float64 oracle for FP8 (e4m3) attention with per-tile power-of-two scales.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with the
CUDA path.

Sources.  The "FlashAttention" learn page (aiunderstanding.org), section on the
future of FlashAttention, and the FlashAttention-3 article (ybx.com),
"FlashAttention-3 innovations" item 3, say that FlashAttention-3 computes
attention in low-precision FP8 and that the order of operations is chosen so
that the low-bit form stays fast and accurate.  The pages fix neither the
format nor the scaling, so this module states one plain reading:

* Format: OCP FP8 e4m3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
  3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; no
  infinities; the largest finite magnitude is 448.  Conversion rounds to
  nearest, ties to even, and saturates to +-448.
* Scaling: a tile of values x shares one integer exponent e, the largest with
  amax * 2^e <= 448 (amax = max |x| over the tile; e = 0 for an all-zero
  tile; e is clamped to [-126, 126] so that 2^e is a normal float32).  The
  stored code is e4m3(x * 2^e); the value it stands for is code * 2^-e.
  A power of two makes the scaling itself exact.
* Tiles: Q and K in blocks of 128 rows (tokens) of one (batch, head), all of
  d; V per (batch, head) over the whole sequence (the PV product accumulates
  over every key block, so one V scale per head keeps the accumulator in one
  unit).
* The attention itself is then exact attention (the float64 oracle) on the
  dequantised Q, K, V.  The GPU path additionally rounds the softmax
  numerators P to e4m3 before the PV product; that rounding is not a plain
  definition (it depends on the running maximum), so it is not modelled here:
  ``p_rounding_bound`` gives the error bound the parity tests use for it.
"""

import math

import numpy as np

from .attention import _f64, attention_head, visible

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6   # exponent field 1, mantissa 0
E4M3_SUBNORMAL_STEP = 2.0 ** -9  # exponent field 0: value = mantissa * 2^-9
TILE = 128
EXP_CLAMP = 126


def e4m3_round(x) -> np.ndarray:
    """Round float64 values to the e4m3 grid: nearest, ties to even, saturating
    at +-448.  Returns float64 values (the grid points themselves)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # spacing of the grid around |x|: 2^(E-3) in binade [2^E, 2^(E+1)),
    # E >= -6; 2^-9 below the smallest normal
    with np.errstate(divide="ignore"):
        E = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    E = np.clip(E, -6, 8)
    step = np.where(a >= E4M3_MIN_NORMAL, 2.0 ** (E - 3), E4M3_SUBNORMAL_STEP)
    r = np.rint(a / step) * step  # np.rint: half to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_encode(g) -> np.ndarray:
    """Codes (uint8) of values already on the e4m3 grid (``e4m3_round`` output)."""
    g = np.asarray(g, dtype=np.float64)
    a = np.abs(g)
    sign = np.signbit(g).astype(np.uint8) << 7
    with np.errstate(divide="ignore"):
        E = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    normal = a >= E4M3_MIN_NORMAL
    exp_field = np.where(normal, E + 7, 0)
    mant = np.where(normal, a / 2.0 ** E * 8 - 8, a / E4M3_SUBNORMAL_STEP)
    assert np.all(mant == np.floor(mant)) and np.all((mant >= 0) & (mant <= 7)), "not on the grid"
    return (sign | (exp_field.astype(np.uint8) << 3) | mant.astype(np.uint8)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of e4m3 codes; 0x7F and 0xFF are NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    ef = (c >> 3) & 0xF
    m = c & 0x7
    v = np.where(ef == 0, m * E4M3_SUBNORMAL_STEP, (1.0 + m / 8.0) * 2.0 ** (ef - 7))
    v = np.where((c & 0x7F) == 0x7F, np.nan, v)
    return s * v


def scale_exponent(amax) -> np.ndarray:
    """Largest integer e with amax * 2^e <= 448 (0 where amax == 0), clamped to
    [-126, 126].  amax = f * 2^x with f in [0.5, 1) (frexp); 448 = 0.875 * 2^9,
    so e = 9 - x when f <= 0.875 and 8 - x otherwise."""
    amax = np.asarray(amax, dtype=np.float64)
    f, x = np.frexp(amax)
    e = np.where(f <= 0.875, 9 - x, 8 - x)
    e = np.clip(e, -EXP_CLAMP, EXP_CLAMP)
    return np.where(amax == 0, 0, e).astype(np.int64)


def quantize_row_tiles(x, tile: int = TILE):
    """x [B, N, H, d] -> codes uint8 [B, N, H, d], exponents int64 [B, H, ceil(N/tile)],
    dequantised float64 [B, N, H, d].  Tile t of (b, h) is rows
    [t*tile, min((t+1)*tile, N)), all of d."""
    x = _f64(x)
    B, N, H, d = x.shape
    nt = (N + tile - 1) // tile
    exps = np.zeros((B, H, nt), dtype=np.int64)
    codes = np.zeros(x.shape, dtype=np.uint8)
    deq = np.zeros(x.shape)
    for b in range(B):
        for h in range(H):
            for t in range(nt):
                blk = x[b, t * tile:(t + 1) * tile, h]
                e = int(scale_exponent(np.abs(blk).max()))
                g = e4m3_round(blk * 2.0 ** e)
                exps[b, h, t] = e
                codes[b, t * tile:(t + 1) * tile, h] = e4m3_encode(g)
                deq[b, t * tile:(t + 1) * tile, h] = g * 2.0 ** -e
    return codes, exps, deq


def quantize_per_head_transposed(v, pad_to: int = 16):
    """V [B, N, H, d] -> codes uint8 [B, H, d, Np] (V transposed per head, the
    key axis zero-padded to Np = N rounded up to pad_to), exponents int64
    [B, H] (one tile = the whole sequence of the head), dequantised float64
    [B, N, H, d]."""
    v = _f64(v)
    B, N, H, d = v.shape
    Np = (N + pad_to - 1) // pad_to * pad_to
    codes = np.zeros((B, H, d, Np), dtype=np.uint8)
    exps = np.zeros((B, H), dtype=np.int64)
    deq = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            blk = v[b, :, h]
            e = int(scale_exponent(np.abs(blk).max())) if N else 0
            g = e4m3_round(blk * 2.0 ** e)
            exps[b, h] = e
            codes[b, h, :, :N] = e4m3_encode(g).T
            deq[b, :, h] = g * 2.0 ** -e
    return codes, exps, deq


def quantize_inputs(q, k, v):
    """The three quantisations of an FP8 attention call (Q, K per 128-row
    tile; V per head, transposed): a dict of codes, exponents and the
    dequantised float64 tensors."""
    q8, qe, qd = quantize_row_tiles(q)
    k8, ke, kd = quantize_row_tiles(k)
    v8t, ve, vd = quantize_per_head_transposed(v)
    return dict(q8=q8, q_exp=qe, q=qd, k8=k8, k_exp=ke, k=kd, v8t=v8t, v_exp=ve, v=vd)


def attention_fp8(q, k, v, causal: bool = False, window: int = -1, scale: float | None = None):
    """O, LSE of exact attention on the dequantised FP8 inputs, and the
    quantisation dict (``quantize_inputs``)."""
    from .attention import attention
    qz = quantize_inputs(q, k, v)
    d = qz["q"].shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O, L = attention(qz["q"], qz["k"], qz["v"], causal=causal, window=window, scale=scale)
    return O, L, qz


def p_rounding_bound(qd, kd, vd, causal: bool = False, window: int = -1,
                     scale: float | None = None, rows=None):
    """Error scale of rounding the softmax numerators to e4m3 before P V.

    With p_j = exp(s_j - m) (m the row maximum, so p_j <= 1) and l = sum p_j,
    the kernel forms sum_j round(p_j 2^c) v_j 2^-c / l for some c >= 0 (its
    running maximum may lag the true one by c < 8 in base-2 units).  Rounding
    to e4m3 moves each numerator by at most eps_j = max(2^-4 p_j, 2^-10) in
    units where the row maximum is 1 (half a step: 2^-4 relative in the normal
    range, 2^-10 absolute below it, less when c > 0).  The returned array
    [B, N, Hq, dv] is sqrt(sum_j eps_j^2 v_jd^2) / l, the standard deviation
    scale of that error when the per-key rounding errors are independent.
    ``rows`` restricts the computation to the given query rows."""
    qd, kd, vd = _f64(qd), _f64(kd), _f64(vd)
    B, N, Hq, d = qd.shape
    Nk, Hkv, dv = kd.shape[1], kd.shape[2], vd.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    G = Hq // Hkv
    rows = np.arange(N) if rows is None else np.asarray(rows)
    out = np.zeros((B, len(rows), Hq, dv))
    vis = visible(N, Nk, causal, window)[rows]
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            _, _, P = attention_head(qd[b, rows, h], kd[b, :, hk], vd[b, :, hk], scale, vis,
                                     return_p=True)
            # P is normalised: P = p / l with p_max = 1, so p = P / max_j P
            pmax = P.max(axis=1, keepdims=True)
            pmax = np.where(pmax > 0, pmax, 1.0)
            p = P / pmax
            eps = np.maximum(2.0 ** -4 * p, 2.0 ** -10) * (P > 0)
            l = 1.0 / pmax  # sum_j p_j = 1 / max_j P_j
            out[b, :, h] = np.sqrt((eps ** 2) @ (vd[b, :, hk] ** 2)) / l
    return out
