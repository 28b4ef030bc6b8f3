"""Plain, slow CPU oracle for the routed MoE expert FFN (MXFP4 weights, online FP8 activations).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and its
Python binding) imports, links or calls this module.  Only the tests, the package
smoke check and the benchmark's CPU-baseline leg may use it.

What it computes, stage by stage, follows the routed-MoE expert path described in
"Pushing the Limits of Serving DeepSeek-V4-Pro" (LMSYS, H20 deployment):
  * §2.2 (capacity): experts stored as MXFP4 weights, activations quantised online
    to FP8 ("Humming MXFP4AFP8");
  * §3.2 (prefill fusion): FP8 quantisation of the activations, top-k reduction
    merged with the shared-expert add;
  * §3.3 (real routing shapes): W13 and W2 are separate grouped GEMMs whose
    per-expert M comes from the routing histogram;
  * §4.3 (decode hot path): SwiGLU fused with the FP8 quantisation that directly
    produces W2's data and scales;
and from the GB10 "Optimization progress report", Optimization 14 (route preplan:
tokens packed by expert before the MoE launch) and Optimization 05 (native NVFP4
MoE: the expert weights kept in NVFP4 and read as such by the expert GEMMs).

The pages do not define bit formats, block sizes, routing or tie rules.  The
readings taken here (each one a plain, checkable definition):
  * E2M1 / E8M0 follow the OCP Microscaling (MX) v1.0 specification; E4M3 is the
    OCP 8-bit floating point "FN" variant (bias 7, max 448, no infinities).
  * MXFP4 weight block = 32 consecutive K elements sharing one E8M0 scale; two
    E2M1 codes per byte with the even K index in the low nibble.
  * NVFP4 weights (the second format): the same E2M1 codes and packing, one FP8
    E4M3 scale per 16 consecutive K elements, and one fp32 scale per weight tensor
    (W13's gate rows and up rows are two tensors, W2 is one).
  * FP8 activations: one power-of-two scale per row per 128 columns; the scale
    exponent is the smallest integer e with amax <= 448 * 2**e, stored as e + 127;
    codes are round-to-nearest-even of x * 2**-e (saturating, never needed).
  * Routing: softmax over E, the k largest logits (ties -> lower expert index),
    weights renormalised over the selected k.
  * W13 rows [0, I) are the gate projection, rows [I, 2I) the up projection;
    h = silu(gate) * up.
  * Rounding points: y13 -> bf16, h -> fp32 then FP8 codes, y2 -> bf16,
    out -> bf16.  All sums are carried in fp64.

Every floating-point accumulation here is float64; integer stages are exact.
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Element formats
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e2m1_decode(codes):
    """Value of 4-bit E2M1 codes (OCP MX v1.0, §5.3.3 FP4 E2M1).

    Bit 3 is the sign, bits 2..1 the exponent (bias 1), bit 0 the mantissa.
    Exponent field 0 is subnormal: 0.5 * mantissa.  No inf/NaN encodings.
    """
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    exp = (c >> 1) & 0x3
    man = c & 0x1
    mag = np.where(exp == 0, 0.5 * man, np.ldexp(1.0 + 0.5 * man, exp - 1))
    return sign * mag


def e8m0_decode(b):
    """Value of an E8M0 (unsigned, exponent-only) scale byte: 2**(b-127); 0xFF is NaN
    (OCP MX v1.0, §5.4 E8M0)."""
    b = np.asarray(b).astype(np.int64)
    v = np.ldexp(1.0, b - 127)
    return np.where(b == 255, np.nan, v)


def e4m3_decode(codes):
    """Value of FP8 E4M3 ("FN") codes (OCP 8-bit FP spec): bias 7, 3 mantissa bits,
    exponent field 0 subnormal (2**-6 * m/8), S.1111.111 is NaN, no infinities."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    mag = np.where(exp == 0, np.ldexp(man / 8.0, -6), np.ldexp(1.0 + man / 8.0, exp - 7))
    mag = np.where((exp == 15) & (man == 7), np.nan, mag)
    return sign * mag


# Non-negative finite E4M3 values in code order 0x00..0x7E (monotonic increasing).
_E4M3_POS = e4m3_decode(np.arange(0x7F))


def e4m3_encode(v):
    """Round float64 values to FP8 E4M3 codes: round to nearest, ties to the even
    code (even mantissa), magnitudes above 448 saturate to 448 (the "satfinite"
    reading; the scale rule below never produces them).  The sign bit is copied from
    the input, so -0.0 and negative values that round to zero give 0x80.
    NaN inputs are outside the contract."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, a, side="left")  # first value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(_E4M3_POS[hi] == a, hi, np.where(pick_hi, hi, lo))
    code = code | np.where(np.signbit(v), 0x80, 0x00)
    return code.astype(np.uint8)


def bf16_round(v):
    """Round float64 values to the nearest bfloat16 value (ties to even), returned as
    float64.  bfloat16 = 8 significant bits, fp32 exponent range (subnormal ulp
    2**-133).  Rounding is done once, from the float64 value."""
    v = np.asarray(v, dtype=np.float64)
    _, p = np.frexp(v)  # v = f * 2**p, f in [0.5, 1)
    ulp = np.ldexp(1.0, np.maximum(p - 8, -133))
    return np.rint(v / ulp) * ulp


def f32_round(v):
    """Round float64 to the nearest float32 value (IEEE round-to-nearest-even)."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16_bits_to_f64(u16):
    """bfloat16 bit patterns (uint16) to float64 values (exact)."""
    u = np.asarray(u16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v):
    """float64 values that are exactly representable in bfloat16 -> uint16 bits."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Online FP8 activation quantisation (per row, per 128-column block)
# ---------------------------------------------------------------------------

QBLOCK = 128


def scale_exponent(amax):
    """Smallest integer e with amax <= 448 * 2**e ("amax/448 rounded up to a power
    of two"), clamped to [-127, 127]; amax == 0 gives e = 0.

    With amax = f * 2**p, f in [0.5, 1) and 448 = 0.875 * 2**9:
    e = p - 9 when f <= 0.875, else p - 8.  No division is involved, so the
    boundary case amax == 448 * 2**e is decided exactly."""
    amax = np.asarray(amax, dtype=np.float64)
    f, p = np.frexp(amax)
    e = np.where(f <= 0.875, p - 9, p - 8)
    e = np.where(amax == 0, 0, e)
    return np.clip(e, -127, 127).astype(np.int64)


def quant_rows(x):
    """FP8 E4M3 quantisation of a [rows, cols] float64 matrix, one power-of-two scale
    per row per 128 columns.  Returns (codes u8 [rows, cols], scale bytes u8
    [rows, cols/128]) with scale byte = e + 127 and codes = RNE_E4M3(x * 2**-e).
    The product x * 2**-e is exact in float64."""
    x = np.asarray(x, dtype=np.float64)
    rows, cols = x.shape
    assert cols % QBLOCK == 0
    xb = x.reshape(rows, cols // QBLOCK, QBLOCK)
    e = scale_exponent(np.abs(xb).max(axis=2))
    codes = e4m3_encode(np.ldexp(xb, -e[:, :, None]))
    return codes.reshape(rows, cols), (e + 127).astype(np.uint8)


def dequant_rows(codes, scales):
    """codes u8 [rows, cols] + scale bytes u8 [rows, cols/128] -> float64 values."""
    rows, cols = codes.shape
    v = e4m3_decode(codes).reshape(rows, cols // QBLOCK, QBLOCK)
    return (v * e8m0_decode(scales)[:, :, None]).reshape(rows, cols)


def quant_act(x_bf16_bits):
    """Stage a3: online FP8 quantisation of the bf16 activations x [T, H]
    (given as uint16 bit patterns).  Pages: LMSYS-H20 §2.2 (online FP8
    activations) and §3.2 (fused FP8 quantisation on the prefill path)."""
    return quant_rows(bf16_bits_to_f64(x_bf16_bits))


# ---------------------------------------------------------------------------
# MXFP4 weights
# ---------------------------------------------------------------------------

MXBLOCK = 32


def mxfp4_dequant(codes, scales):
    """MXFP4 weight matrix -> float64.  codes u8 [N, K/2] (even K index in the low
    nibble), scales u8 [N, K/32] (E8M0).  Returns [N, K]."""
    codes = np.asarray(codes)
    n, kh = codes.shape
    k = kh * 2
    vals = np.empty((n, k), dtype=np.float64)
    vals[:, 0::2] = e2m1_decode(codes & 0xF)
    vals[:, 1::2] = e2m1_decode(codes >> 4)
    s = e8m0_decode(scales)
    return (vals.reshape(n, k // MXBLOCK, MXBLOCK) * s[:, :, None]).reshape(n, k)


# ---------------------------------------------------------------------------
# f3: NVFP4 weights
# ---------------------------------------------------------------------------

NVBLOCK = 16


def nvfp4_dequant(codes, scales, global_scale=None):
    """NVFP4 weight matrix -> float64 (GB10 "Optimization progress report",
    Optimization 05: the MoE expert weights stay in their native NVFP4 form and the
    expert kernel reads them as such).  The page names the format without defining
    it; the reading is NVIDIA's NVFP4: E2M1 values in blocks of 16 consecutive K
    elements, each block with one FP8 E4M3 scale, and one fp32 scale per tensor.

    codes u8 [N, K/2] (two E2M1 codes per byte, even K index in the low nibble, as
    for MXFP4), scales u8 [N, K/16] (E4M3 codes), global_scale: None (1.0), a
    scalar, or an array [S] of fp32 scales for S equal segments of the N rows (W13
    keeps the gate rows and the up rows as two tensors, each with its own scale).
    Returns [N, K]: e2m1(code) * e4m3(scale of its 16-block) * segment scale."""
    codes = np.asarray(codes)
    n, kh = codes.shape
    k = kh * 2
    vals = np.empty((n, k), dtype=np.float64)
    vals[:, 0::2] = e2m1_decode(codes & 0xF)
    vals[:, 1::2] = e2m1_decode(codes >> 4)
    s = e4m3_decode(scales)
    w = (vals.reshape(n, k // NVBLOCK, NVBLOCK) * s[:, :, None]).reshape(n, k)
    if global_scale is not None:
        gs = np.atleast_1d(np.asarray(global_scale, dtype=np.float32).astype(np.float64))
        w = w * np.repeat(gs, n // len(gs))[:, None]
    return w


def weight_dequant(fmt, codes, scales, global_scale=None):
    """Expert weight matrix of either format -> float64 [N, K]."""
    if fmt == "mxfp4":
        return mxfp4_dequant(codes, scales)
    if fmt == "nvfp4":
        return nvfp4_dequant(codes, scales, global_scale)
    raise ValueError(fmt)


# ---------------------------------------------------------------------------
# f4: router gate projection (the scores the TopK step ranks)
# ---------------------------------------------------------------------------

def router_logits(x_bf16_bits, wg):
    """logits[t, e] = sum_h x[t, h] * W_g[e, h], summed in float64 and rounded once
    to float32.  x is the bf16 hidden state [T, H], W_g the fp32 gate weight [E, H].

    The TopK step of the LMSYS H20 post (§3.2) ranks per-expert router scores; the
    pages do not print the gate, so it is read as the plain linear projection of the
    token's hidden state, kept in fp32 (the precision its output is handed on in)."""
    x = bf16_bits_to_f64(x_bf16_bits)
    w = np.asarray(wg, dtype=np.float32).astype(np.float64)
    return f32_round(x @ w.T)


# ---------------------------------------------------------------------------
# a1: top-k routing
# ---------------------------------------------------------------------------

def route(logits, k):
    """Stage a1.  Per token: softmax over the E experts, keep the k largest, and
    renormalise their weights to sum to 1 (LMSYS-H20 §3.2 names the TopK step; the
    softmax -> top-k -> renormalise rule is the stated routing contract).

    Selection compares the fp32 logits themselves (softmax is monotonic), largest
    first, equal logits -> lower expert index first.  Returns idx int32 [T, k] in
    selection order and w float64 [T, k]; the renormalised weight of expert j is
    exp(l_j - l_max) / sum over the selected of exp(l_i - l_max), the full-softmax
    denominator cancelling."""
    logits = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = logits.shape
    order = np.lexsort((np.broadcast_to(np.arange(E), (T, E)), -logits), axis=-1)
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    ex = np.exp(sel - sel[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    return idx, w


# ---------------------------------------------------------------------------
# a2: histogram + exclusive scan + permute
# ---------------------------------------------------------------------------

def permute(idx, E, has_shared):
    """Stage a2 (GB10 report, Optimization 14: tokens packed by expert before the MoE
    launch; LMSYS-H20 §3.3: per-expert M from the routing histogram).

    Routed row r = t*k + j.  Groups are the E experts, plus group E = the shared
    expert (one row per token) when has_shared.  Inside a group rows are ordered by
    ascending token.  Returns
      counts  int32 [E]       tokens routed to each expert,
      offsets int32 [G + 1]   exclusive scan over groups (G = E + has_shared),
      perm_src int32 [R]      packed row -> routed row t*k + j   (R = T*k),
      inv     int32 [R]       routed row t*k + j -> packed row.
    Shared rows occupy packed rows R .. R + T - 1 in token order."""
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    R = T * k
    counts = np.bincount(idx.reshape(-1), minlength=E).astype(np.int64)
    group_sizes = np.concatenate([counts, [T]]) if has_shared else counts
    offsets = np.zeros(len(group_sizes) + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(group_sizes)
    flat = idx.reshape(-1)
    perm_src = np.argsort(flat, kind="stable")  # stable: routed-row order = token order
    inv = np.empty(R, dtype=np.int64)
    inv[perm_src] = np.arange(R)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            perm_src.astype(np.int32), inv.astype(np.int32))


def packed_row_token(perm_src, T, k, has_shared):
    """Token index of every packed row (routed rows first, then the shared rows)."""
    tok = np.asarray(perm_src, dtype=np.int64) // k
    if has_shared:
        tok = np.concatenate([tok, np.arange(T)])
    return tok


# ---------------------------------------------------------------------------
# a4 / a6: grouped GEMMs
# ---------------------------------------------------------------------------

def grouped_gemm(act_codes, act_scales, offsets, w_codes, w_scales, groups=None,
                 fmt="mxfp4", w_global=None):
    """Stages a4 / a6 (LMSYS-H20 §3.3: W13 and W2 grouped GEMMs over the experts).

    For every group g and packed row r in [offsets[g], offsets[g+1]):
        y[r, n] = sum_k deq(act)[r, k] * deq(W[g])[n, k]
    with act = FP8 E4M3 codes [Rows, K] + per-128 scales, W[g] = MXFP4 [N, K] (or
    NVFP4 with fmt="nvfp4" and per-group tensor scales w_global [G] or [G, S]);
    summed in float64 and rounded once to bf16.  Returns float64 [Rows, N] holding
    bf16 values.  `groups` restricts the work to a subset of groups (the other rows
    are left as NaN)."""
    rows = act_codes.shape[0]
    G = len(offsets) - 1
    N = w_codes.shape[1]
    y = np.full((rows, N), np.nan)
    for g in (range(G) if groups is None else groups):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 == r0:
            continue
        a = dequant_rows(act_codes[r0:r1], act_scales[r0:r1])
        gs = None if w_global is None else np.asarray(w_global)[g]
        w = weight_dequant(fmt, w_codes[g], w_scales[g], gs)
        y[r0:r1] = bf16_round(a @ w.T)
    return y


# ---------------------------------------------------------------------------
# a5: SwiGLU + FP8 requantisation
# ---------------------------------------------------------------------------

def swiglu(y13):
    """h = silu(gate) * up with gate = y13[:, :I], up = y13[:, I:], silu(g) = g / (1 +
    exp(-g)), evaluated in float64 (LMSYS-H20 §4.3)."""
    y13 = np.asarray(y13, dtype=np.float64)
    I = y13.shape[1] // 2
    g, u = y13[:, :I], y13[:, I:]
    return g / (1.0 + np.exp(-g)) * u


def swiglu_quant(y13):
    """Stage a5 (LMSYS-H20 §4.3: SwiGLU fused with the quantisation that directly emits
    W2's data and scales).  h is computed in float64, rounded to fp32 (the precision
    in which the kernel takes the quantisation decisions), then quantised per row per
    128 columns with the same rule as the activations.  Returns (hq u8 [Rows, I],
    hs u8 [Rows, I/128])."""
    return quant_rows(f32_round(swiglu(y13)))


# ---------------------------------------------------------------------------
# a7: weighted top-k combine + shared-expert add
# ---------------------------------------------------------------------------

def combine(y2, inv, w, T, k, has_shared):
    """Stage a7 (LMSYS-H20 §3.2: TopK reduction merged with the shared-expert add).

        out[t] = bf16( sum_j w[t, j] * y2[inv[t*k + j]]  +  y2[R + t] (if shared) )

    summed in float64, rounded once to bf16.  Returns float64 [T, H]."""
    y2 = np.asarray(y2, dtype=np.float64)
    inv = np.asarray(inv, dtype=np.int64).reshape(T, k)
    w = np.asarray(w, dtype=np.float64).reshape(T, k)
    acc = np.zeros((T, y2.shape[1]))
    for j in range(k):
        acc += w[:, j:j + 1] * y2[inv[:, j]]
    if has_shared:
        acc += y2[T * k + np.arange(T)]
    return bf16_round(acc)


# ---------------------------------------------------------------------------
# Whole layer
# ---------------------------------------------------------------------------

def moe_forward(x_bf16_bits, logits, k, w13, w13_s, w2, w2_s, has_shared, fmt="mxfp4",
                w13_gs=None, w2_gs=None):
    """The whole routed-expert FFN, stages a1..a7 in order.

    x_bf16_bits uint16 [T, H]; logits fp32 [T, E]; w13 u8 [G, 2I, H/2],
    w13_s u8 [G, 2I, H/32], w2 u8 [G, H, I/2], w2_s u8 [G, H, I/32] with
    G = E + has_shared (the shared expert is group E).  With fmt="nvfp4" the scales
    are E4M3 per 16 K ([G, 2I, H/16], [G, H, I/16]) and w13_gs [G, 2] (gate, up) /
    w2_gs [G] hold the fp32 tensor scales (None: 1).
    Returns a dict with every intermediate (same names as the C interface)."""
    T, H = x_bf16_bits.shape
    E = logits.shape[1]
    idx, w = route(logits, k)
    counts, offsets, perm_src, inv = permute(idx, E, has_shared)
    xq, xs = quant_act(x_bf16_bits)
    tok = packed_row_token(perm_src, T, k, has_shared)
    y13 = grouped_gemm(xq[tok], xs[tok], offsets, w13, w13_s, fmt=fmt, w_global=w13_gs)
    hq, hs = swiglu_quant(y13)
    y2 = grouped_gemm(hq, hs, offsets, w2, w2_s, fmt=fmt, w_global=w2_gs)
    out = combine(y2, inv, w, T, k, has_shared)
    return dict(idx=idx, w=w, counts=counts, offsets=offsets, perm_src=perm_src,
                inv=inv, xq=xq, xs=xs, y13=y13, hq=hq, hs=hs, y2=y2, out=out)


def moe_forward_tokens(x_bf16_bits, logits, k, w13, w13_s, w2, w2_s, has_shared, tokens,
                       fmt="mxfp4", w13_gs=None, w2_gs=None):
    """The layer output for a subset of tokens only (each token's output depends only
    on its own row of x and logits).  Used to check full-size runs on a sample."""
    tokens = np.asarray(tokens, dtype=np.int64)
    res = moe_forward(x_bf16_bits[tokens], np.asarray(logits)[tokens], k,
                      w13, w13_s, w2, w2_s, has_shared, fmt, w13_gs, w2_gs)
    return res


def dense_unrouted_forward(x_bf16_bits, logits, k, w13, w13_s, w2, w2_s, has_shared,
                           fmt="mxfp4", w13_gs=None, w2_gs=None):
    """Independent recomputation for pinning the routed path on tiny shapes: every
    token goes through every expert (no histogram, no permutation, no gather), and
    the top-k mask selects afterwards.  The per-(token, expert) arithmetic is the same
    as the routed path's, so the two agree bit for bit."""
    T, H = x_bf16_bits.shape
    E = logits.shape[1]
    G = w13.shape[0]
    xq, xs = quant_act(x_bf16_bits)
    xa = dequant_rows(xq, xs)
    y2_all = np.zeros((G, T, w2.shape[1]))
    g13 = (lambda g: None) if w13_gs is None else (lambda g: np.asarray(w13_gs)[g])
    g2 = (lambda g: None) if w2_gs is None else (lambda g: np.asarray(w2_gs)[g])
    for g in range(G):
        y13 = bf16_round(xa @ weight_dequant(fmt, w13[g], w13_s[g], g13(g)).T)
        hq, hs = swiglu_quant(y13)
        y2_all[g] = bf16_round(dequant_rows(hq, hs) @ weight_dequant(fmt, w2[g], w2_s[g],
                                                                     g2(g)).T)
    # brute-force selection: k rounds of "largest remaining logit, lowest index on ties"
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    out = np.zeros((T, w2.shape[1]))
    for t in range(T):
        taken = []
        for _ in range(k):
            best = None
            for e in range(E):
                if e in taken:
                    continue
                if best is None or lg[t, e] > lg[t, best]:
                    best = e
            taken.append(best)
        ex = np.exp(lg[t, taken] - lg[t, taken[0]])
        wt = ex / ex.sum()
        acc = np.zeros(w2.shape[1])
        for j, e in enumerate(taken):
            acc += wt[j] * y2_all[e, t]
        if has_shared:
            acc += y2_all[E, t]
        out[t] = bf16_round(acc)
    return out
