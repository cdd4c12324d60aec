"""Pure-Python scalar re-derivation of the latent-MoE tail for tiny shapes.

It pins the numpy oracle by a different route: format values come from a table built
with ``math.ldexp`` on the bit fields, e4m3 rounding is a nearest-value search over the
whole code table, float32 steps are emulated by ``struct`` round trips (exact for one
+,-,*,/ of float32 operands: double rounding through float64 is innocuous for those),
top-k is ``sorted`` and every product is an explicit loop.
"""
from __future__ import annotations

import math
import struct


def f32(v: float) -> float:
    return struct.unpack("f", struct.pack("f", v))[0]


def _e4m3_table():
    vals = {}
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 0xF and m == 7:
            continue
        vals[c] = s * (math.ldexp(m, -9) if e == 0 else math.ldexp(8 + m, e - 10))
    return vals


E4M3 = _e4m3_table()
E4M3_POS = sorted((v, c) for c, v in E4M3.items() if c < 0x80)


def e4m3_value(c: int) -> float:
    return E4M3[c]


def e4m3_round(v: float) -> int:
    """Nearest finite e4m3 code, ties to the code with an even mantissa; saturating."""
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    best = None
    for val, c in E4M3_POS:
        d = abs(val - a)
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1] | sign


def e2m1_value(c: int) -> float:
    s = -1.0 if c & 8 else 1.0
    e, m = (c >> 1) & 3, c & 1
    return s * (0.5 * m if e == 0 else math.ldexp(2 + m, e - 2))


def quant_group(vals):
    """One 128-wide group of float32 values -> (codes, scale)."""
    amax = max(abs(v) for v in vals)
    s = 1.0 if amax == 0 else f32(amax / 448.0)
    return [e4m3_round(f32(v / s)) for v in vals], s


def quant_group_mx(vals):
    """One 32-wide group -> (codes, scale): scale 2**(e - 8) with 2**e <= amax < 2**(e+1),
    found by exact doubling/halving; 1 for an all-zero group."""
    amax = max(abs(v) for v in vals)
    if amax == 0:
        return [e4m3_round(0.0) for _ in vals], 1.0
    e, p = 0, 1.0
    while p > amax:
        p, e = p / 2.0, e - 1
    while p * 2.0 <= amax:
        p, e = p * 2.0, e + 1
    e = max(-127, min(127, e - 8))
    s = math.ldexp(1.0, e)
    return [e4m3_round(f32(v / s)) for v in vals], s


E2M1_POS = sorted((e2m1_value(c), c) for c in range(8))


def e2m1_round(v: float) -> int:
    """Nearest e2m1 code, ties to the code with an even mantissa bit, saturating at 6;
    the sign bit only for a non-zero magnitude."""
    a = abs(v)
    best = None
    for val, c in E2M1_POS:
        key = (abs(val - a), c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    c = best[1]
    return c | 8 if (v < 0 and c > 0) else c


def quant_group_nvfp4(vals):
    """One 16-wide group -> (codes, scale): scale = the e4m3 value nearest fp32(amax/6),
    codes = e2m1 of fp32(v/scale); all codes 0 when the scale is 0."""
    amax = max(abs(v) for v in vals)
    s = e4m3_value(e4m3_round(f32(amax / 6.0)))
    if s == 0.0:
        return [0 for _ in vals], 0.0
    return [e2m1_round(f32(v / s)) for v in vals], s


def silu(v: float) -> float:
    return v / (1.0 + math.exp(-v))


def matvec(w, x):
    return [sum(wr[i] * x[i] for i in range(len(x))) for wr in w]


def tail_token(logits, z, x, k, experts, gamma, eps, ws13, ws2, w_up, mx=False, a4=False):
    """Output vector of one token.  ``experts[e] = (w13 rows, w2 rows)`` dequantised.
    ``mx``: activations quantised per 32 with power-of-two scales instead of per 128;
    ``a4``: activations quantised to NVFP4 (e2m1, e4m3 scale per 16)."""
    G, qg = (32, quant_group_mx) if mx else (16, quant_group_nvfp4) if a4 else \
        (128, quant_group)
    val = e2m1_value if a4 else e4m3_value
    order = sorted(range(len(logits)), key=lambda e: (-logits[e], e))[:k]
    mx = logits[order[0]]
    ex = [math.exp(logits[e] - mx) for e in order]
    tot = sum(ex)
    wts = [v / tot for v in ex]
    zd = []
    for g0 in range(0, len(z), G):
        q, s = qg([f32(v) for v in z[g0:g0 + G]])
        zd += [val(c) * s for c in q]
    L = len(z)
    r = [0.0] * L
    for e, wj in zip(order, wts):
        w13, w2 = experts[e]
        inter = len(w13) // 2
        h = matvec(w13, zd)
        a = [silu(h[i]) * h[inter + i] for i in range(inter)]
        ad = []
        for g0 in range(0, inter, G):
            q, s = qg([f32(v) for v in a[g0:g0 + G]])
            ad += [val(c) * s for c in q]
        y = matvec(w2, ad)
        for c in range(L):
            r[c] += wj * y[c]
    ms = sum(v * v for v in r) / L
    inv = 1.0 / math.sqrt(ms + eps)
    n = [r[c] * inv * gamma[c] for c in range(L)]
    up = matvec(w_up, n)
    hs = matvec(ws13, x)
    inter_s = len(ws13) // 2
    a_s = [silu(hs[i]) * hs[inter_s + i] for i in range(inter_s)]
    s_out = matvec(ws2, a_s)
    return [up[i] + s_out[i] for i in range(len(up))], order, wts


def bf16_value(v: float) -> float:
    """Nearest bfloat16 value (8 significant bits), ties to an even significand, derived
    from the significand/exponent split of the float64 value."""
    if v == 0.0 or math.isinf(v) or math.isnan(v):
        return v
    m, e = math.frexp(v)            # v = m * 2**e, 0.5 <= |m| < 1
    q = m * 256.0                   # significand with 8 bits before the point
    r = math.floor(q)
    frac = q - r
    if frac > 0.5 or (frac == 0.5 and r % 2 == 1):
        r += 1
    return math.ldexp(r, e - 8)


def latent_inputs_token(x, w_lat, w_gate):
    """Latent input z (bf16 values) and router logits of one token by explicit loops."""
    z = [bf16_value(sum(wr[i] * x[i] for i in range(len(x)))) for wr in w_lat]
    logits = [sum(wr[i] * x[i] for i in range(len(x))) for wr in w_gate]
    return z, logits
