"""Float64 CPU oracle for the forward pass of a block-quantized FP8 MoE layer.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  The product path (the CUDA
library and its Python binding) never calls it and shares no code with it.

What it computes, step by step (float64 unless a step says otherwise):

1. e4m3 decoding by a 256-entry table built from the format's definition:
   sign s = b>>7, exponent e = (b>>3)&15, mantissa m = b&7; a zero e gives
   the subnormal m * 2^-9; e == 15 with m == 7 is NaN; otherwise
   (1 + m/8) * 2^(e-7).  (FreeToken PR #662, PR body: normal codes take a
   rebased exponent, a zero exponent field marks a subnormal m * 2^-9, and
   the finite magnitudes run from 2^-9 to 448.)
2. Block dequantisation: weight banks are e4m3 row-major [rows, K], K
   contiguous, with a bf16 scale for each 128 x 128 block (FreeToken PR #662, PR
   body).  The scale of element (n, kk) is scale[n // 128, kk // 128], read
   through the row stride of the scale bank, which may be padded ("honor
   padded fp8 scale strides" commit of the same PR).  When K or the row count
   is not a multiple of 128 the last block is partial (same PR, Tests: the
   ragged-K case); the stacked [gate; up] bank is blocked over its 2I rows
   from row 0, so with I not a multiple of 128 one block holds gate and up
   rows.
3. Activations: W8A16 mode uses the bf16 activations as they are (the CPU
   and GPU decode kernels of FreeToken PR #662, "Call path" / "Kernels").
   W8A8 mode quantises them per token per 128-column group with a dynamic
   scale (fp8-moe-gather page, "Affects" / "Who is affected": dynamic
   activation scales): amax = max |x|, scale = fl32(amax / 448),
   q = e4m3_rne_satfinite(fl32(x / scale)), a = dec(q) * scale.  These
   quantisation steps run in IEEE fp32, the precision the kernel uses, so
   codes and scales are comparable bit for bit.
4. Expert function: the up/gate projection over the stacked [gate | up]
   bank (gate rows [0, I), up rows [I, 2I); tpu-inference PR #3040, review
   of the bias DMA: gate half at n_id*tile_n1, up half at out_n1 +
   n_id*tile_n1), h = silu(gate) * up with silu(z) = z / (1 + exp(-z))
   (fp8-moe-gather page, "Affects": silu experts), then the down projection
   y = W2 h (fp8-moe-gather page, "The fix": down projection in fp32; here
   float64).  In W8A8 mode h is itself quantised per 128-group by the rule
   of step 3 (float64 h rounded to fp32 first) before the down projection.
   The W8A8 decode mode (the Gaudi path of the fp8-moe-gather page, "The
   fix": dynamic activation scales and an FP8 GEMM for the up/gate
   projection, the down projection in fp32) quantises the activations by
   step 3 and keeps h unquantised.
   Optional MLP biases (tpu-inference PR #3040, review of the bias DMA: the
   up/gate bias row is laid out [gate | up] like the weight rows, the up
   half at offset I, and the down projection has a bias of its own with no
   split): gate += b13[0:I], up += b13[I:2I] before silu, y += b2 after the
   down projection.  The biases are fp32 and enter float64 exactly.
5. Combine: out_t = sum_j w[t,j] * y_{ids[t,j]}(x_t).  The all-expert
   evaluation (the stock mixture_of_experts op of the fp8-moe-gather page,
   "Problem", reads every expert) computes y_e for every expert and masks
   it with c[t,e] = sum_{j: ids[t,j]=e} w[t,j]; the gathered evaluation
   (section The fix: it reads at most g = min(E_local, T*k) experts, those
   that are routed) visits routed experts only.  Both are the same number up to
   float64 rounding.
6. Routing lists: a counting sort of the slots s = t*k + j by expert id,
   stable in s; ids outside [0, E) are skipped.

Readings of points the pages leave open (negative ids skip a slot, ids >= E
skip and are flagged, NaN codes are out of contract, amax == 0 gives codes 0
and scale 0, ...) are listed with the design notes of the repository.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128


# ---------------------------------------------------------------- step 1 --
def e4m3_value(b: int) -> float:
    """Value of e4m3 (fn variant) byte b by the format's definition."""
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        v = m * 2.0 ** -9
    else:
        v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -v if s else v


def e4m3_table() -> np.ndarray:
    """256-entry float64 decode table (NaN at 0x7F and 0xFF)."""
    return np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


_TABLE = e4m3_table()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_rne_satfinite(x) -> np.ndarray:
    """fp32 values -> e4m3 codes: round to nearest, ties to even, magnitudes
    beyond the largest finite value (448) clamp to +-448; NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    nan = np.isnan(x)
    sign = np.signbit(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)
    sub = a < 2.0 ** -6
    # subnormal range: spacing 2^-9; m == 8 lands on the smallest normal, code 0x08
    q_sub = np.rint(a / 2.0 ** -9)
    # normal range: a = f * 2^ex with f in [0.5, 1); exponent e = ex - 1, spacing 2^(e-3)
    _, ex = np.frexp(np.where(sub, 1.0, a))
    e = ex - 1
    q_norm = np.rint(np.where(sub, 8.0, a) / np.ldexp(1.0, e - 3))  # in [8, 16]
    code_norm = ((e + 7) << 3) + (q_norm.astype(np.int64) - 8)      # q == 16 carries into the exponent
    code = np.where(sub, q_sub.astype(np.int64), code_norm)
    out[...] = code.astype(np.uint8)
    out |= np.where(sign, 0x80, 0).astype(np.uint8)
    out[nan] = 0x7F
    return out


# ---------------------------------------------------------------- step 2 --
def bf16_bits_to_f64(u16) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def dequant_bank(codes: np.ndarray, scales_bf16: np.ndarray) -> np.ndarray:
    """Dequantise one expert's bank.

    codes: uint8 [R, K] e4m3; scales_bf16: uint16 [ceil(R/128), >= ceil(K/128)]
    (a possibly padded row stride; only the first ceil(K/128) columns are
    read).  Element (n, kk) is dec(codes[n, kk]) * scale[n // 128, kk // 128].
    """
    R, K = codes.shape
    w = e4m3_decode(codes)
    s = bf16_bits_to_f64(scales_bf16)
    rb = np.arange(R) // BLOCK
    kb = np.arange(K) // BLOCK
    return w * s[rb[:, None], kb[None, :]]


# ---------------------------------------------------------------- step 3 --
def quantize_per_128(x32: np.ndarray):
    """Per-row, per-128-column-group dynamic e4m3 quantisation in fp32.

    x32: float32 [n, K].  Returns (codes uint8 [n, K], scales float32
    [n, ceil(K/128)]) with scale = fl32(amax / 448) and
    code = e4m3_rne_satfinite(fl32(x / scale)); a group with amax == 0 has
    scale 0 and all codes 0x00.
    """
    x32 = np.asarray(x32, dtype=np.float32)
    n, K = x32.shape
    G = -(-K // BLOCK)
    codes = np.zeros((n, K), dtype=np.uint8)
    scales = np.zeros((n, G), dtype=np.float32)
    for gi in range(G):
        blk = x32[:, gi * BLOCK:(gi + 1) * BLOCK]
        amax = np.max(np.abs(blk), axis=1)
        sc = (amax / np.float32(E4M3_MAX)).astype(np.float32)
        scales[:, gi] = sc
        with np.errstate(divide="ignore", invalid="ignore"):
            q = (blk / sc[:, None]).astype(np.float32)
        q = np.where((sc == 0)[:, None], np.float32(0), q)
        codes[:, gi * BLOCK:(gi + 1) * BLOCK] = e4m3_encode_rne_satfinite(q)
    return codes, scales


def dequantize_per_128(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    n, K = codes.shape
    kb = np.arange(K) // BLOCK
    return e4m3_decode(codes) * scales.astype(np.float64)[:, kb]


# ---------------------------------------------------------------- step 4 --
def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_forward(a: np.ndarray, w13_codes, w13_scale, w2_codes, w2_scale, act: str,
                   b13=None, b2=None) -> np.ndarray:
    """y = W2 h(a) (+ b2) for one expert and a batch of activation rows
    a [n, H] (float64, already dequantised in the W8A8 modes).  h is
    quantised only in act == "e4m3" (prefill W8A8).  b13: optional fp32 [2I]
    bias row, gate biases in [0, I) and up biases in [I, 2I); b2: optional
    fp32 [H] down-projection bias."""
    I = w13_codes.shape[0] // 2
    W13 = dequant_bank(w13_codes, w13_scale)       # [2I, H]
    gate = a @ W13[:I].T                            # [n, I]
    up = a @ W13[I:].T
    if b13 is not None:
        b13 = np.asarray(b13, dtype=np.float32).astype(np.float64)
        gate = gate + b13[:I]
        up = up + b13[I:2 * I]
    h = silu(gate) * up
    if act == "e4m3":
        hc, hs = quantize_per_128(h.astype(np.float32))
        h = dequantize_per_128(hc, hs)
    W2 = dequant_bank(w2_codes, w2_scale)           # [H, I]
    y = h @ W2.T                                    # [n, H]
    if b2 is not None:
        y = y + np.asarray(b2, dtype=np.float32).astype(np.float64)
    return y


def activations(hidden_bf16: np.ndarray, act: str) -> np.ndarray:
    """bf16 bits [T, H] -> float64 activation rows for the given mode."""
    x = bf16_bits_to_f64(hidden_bf16)
    if act == "bf16":
        return x
    if act in ("e4m3", "e4m3_x"):
        codes, scales = quantize_per_128(x.astype(np.float32))
        return dequantize_per_128(codes, scales)
    raise ValueError(act)


# ---------------------------------------------------------------- step 5 --
def forward(hidden_bf16, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale,
            mode: str = "gathered", act: str = "bf16", tokens=None, w13_bias=None,
            w2_bias=None) -> np.ndarray:
    """Layer output, float64 [len(tokens), H].

    hidden_bf16: uint16 [T, H]; topk_ids: int32 [T, k]; topk_weights: float32
    [T, k]; w13: uint8 [E, 2I, H]; w13_scale: uint16 [E, 2I/128, >= H/128];
    w2: uint8 [E, H, I]; w2_scale: uint16 [E, H/128, >= I/128].
    mode: "gathered" (routed experts only) or "all" (every expert, masked).
    act: "bf16" (W8A16), "e4m3" (W8A8, dynamic per-token-per-128 scales,
    h quantised the same way) or "e4m3_x" (W8A8 decode: activations
    quantised, h kept in float64 for the down projection).
    tokens: optional subset of token indices (all by default).
    w13_bias: optional fp32 [E, 2I] ([gate | up] per expert); w2_bias:
    optional fp32 [E, H].
    """
    E = w13.shape[0]
    T, H = hidden_bf16.shape
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    ids = np.asarray(topk_ids)[tok]
    wts = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)[tok]
    a = activations(np.asarray(hidden_bf16)[tok], act)
    out = np.zeros((len(tok), H), dtype=np.float64)
    if mode == "all":
        for e in range(E):
            c = np.where(ids == e, wts, 0.0).sum(axis=1)        # c[t, e]
            y = expert_forward(a, w13[e], w13_scale[e], w2[e], w2_scale[e], act,
                               None if w13_bias is None else w13_bias[e],
                               None if w2_bias is None else w2_bias[e])
            out += c[:, None] * y
        return out
    if mode == "gathered":
        valid = (ids >= 0) & (ids < E)
        for e in np.unique(ids[valid]):
            rows, js = np.nonzero(ids == e)
            y = expert_forward(a[rows], w13[e], w13_scale[e], w2[e], w2_scale[e], act,
                               None if w13_bias is None else w13_bias[e],
                               None if w2_bias is None else w2_bias[e])
            np.add.at(out, rows, wts[rows, js][:, None] * y)
        return out
    raise ValueError(mode)


# ---------------------------------------------------------------- step 6 --
def route_lists(topk_ids: np.ndarray, E: int):
    """Routing lists of the gathered path.

    Returns dict with counts [E], offsets [E+1] (exclusive scan), perm [S]
    (valid slots s = t*k + j ordered by expert ascending, stable in s; the
    first offsets[E] entries are meaningful, the rest -1), inv [S] (position
    of slot s in perm, -1 if skipped), glist [g] (distinct routed experts
    ascending, padded with -1 to g = min(E, S)), D (number of distinct
    experts), bad_id (an id >= E was seen).
    """
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    S = ids.size
    valid = (ids >= 0) & (ids < E)
    counts = np.bincount(ids[valid], minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.full(S, -1, dtype=np.int32)
    inv = np.full(S, -1, dtype=np.int32)
    fill = offsets[:-1].copy()
    for s in range(S):                    # slots in index order -> stable
        if valid[s]:
            e = ids[s]
            perm[fill[e]] = s
            inv[s] = fill[e]
            fill[e] += 1
    distinct = np.nonzero(counts)[0].astype(np.int32)
    g = min(E, S)
    glist = np.full(g, -1, dtype=np.int32)
    glist[:len(distinct)] = distinct
    return dict(counts=counts, offsets=offsets, perm=perm, inv=inv, glist=glist,
                D=int(len(distinct)), bad_id=bool(np.any(ids >= E)))


def gate_takes_gathered_path(T: int, k: int, E: int, ratio: float = 0.4) -> bool:
    """The path gate: gathered when T*k <= E*ratio (slots against local experts
    times the ratio; fp8-moe-gather page, environment-variable table,
    default ratio 0.4)."""
    return T * k <= E * ratio
