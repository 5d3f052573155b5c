"""Plain CPU oracle of the GPTQ per-layer path. TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import or run this module. The product path (the CUDA library and
its Python binding) never touches it, and this module imports nothing from the
product: the two share no code, table or constant.

What it computes, step by step, in the order and notation of the pages:

* ``hessian``      H = alpha * X^T X summed over token batches (alpha = 2).
* ``damp``         H_d = H + lambda I, lambda = percdamp * mean(diag H).
* ``act_order_perm``  columns in order of decreasing H_qq.
* ``hinv1``        the three-step Cholesky chain: L = chol(H_d), H^-1 from L by a
                   Cholesky solve against the identity, Hinv1 = upper Cholesky factor
                   of H^-1.
* ``quant_params`` / ``quantize`` / ``dequantize``  asymmetric min/max quantizer.
* ``gptq_columns`` blocked column loop: quantize, error Err1 = (w - w_hat)/Hinv1[j,j],
                   rank-one update inside the block, lazy Err1 @ Hinv1[block, rest]
                   after it; per-element losses Losses1 = Err1^2 / 2.
* ``sequential_pass``  layers one after another: each layer's Hessian from the
                   inputs that the already quantized layers before it produce.
* ``pack_codes`` / ``unpack_codes``  b-bit codes as a little-endian bitstream of
                   uint32 words per row.
* ``dequantize_packed`` / ``dequant_matmul``  the stored layer used again: W_hat
                   from packed codes and group scales, and Y = X W_hat^T.
* ``relative_output_error``  ||(W - W_hat) X^T||_F / ||W X^T||_F through H.

Arithmetic is float64 unless ``dtype=np.float32`` is passed; the float32 mode keeps
the same steps in float32 (the working precision of the listing in "GPTQ-style
round-to-nearest with Hessian weighting") and serves to measure how far float32
rounding alone moves the result. NumPy/LAPACK routines (matmul, Cholesky, triangular
solve, stable argsort) serve as single steps; nothing is blocked, fused or reordered
beyond what the pages state.

Readings taken where the pages are silent or disagree (each is also listed in the
design notes of the repository):

* Hessian constant: H = 2 X^T X with no 1/n. Codes do not depend on a positive
  scale of H; only the losses scale.
* Losses1 is named but not defined on the pages; it is taken as the increase of the
  quadratic objective when column j is fixed, Err1^2/2 = (w - w_hat)^2 / (2 Hinv1_jj^2).
* Group statistics are read from the current (already compensated) weights at the
  group's first column; this needs group_size % blocksize == 0 or the reverse.
* Rounding is round-half-to-even (``np.rint``) and w/scale is a true division.
* act-order ties keep the lower column index first (stable sort).
* act-order with groups: groups are formed in processing order; original column j
  uses group (position of j in the order) // group_size.
* Layers one after another: the synthetic model is a chain of linear layers with
  nothing between them; layer l+1 is calibrated on X_l W_hat_l^T (the quantized
  outputs), rounded to bfloat16.
* Code storage: code (r, j) occupies bits [j*b, j*b + b) of row r's stream.
"""
from __future__ import annotations

import numpy as np
import scipy.linalg

__all__ = [
    "hessian", "hessian_accumulate", "hessian_entries", "damp", "act_order_perm",
    "hinv1", "quant_params", "quantize", "dequantize", "gptq_columns", "gptq_layer",
    "rtn", "round_to_bf16", "sequential_pass", "pack_codes", "unpack_codes", "packed_words_per_row",
    "dequantize_packed", "dequant_matmul",
    "relative_output_error", "loss_quadratic_form",
]


# ----------------------------------------------------------------------------------
# Stage 1: Hessian
# ----------------------------------------------------------------------------------
def hessian_accumulate(H: np.ndarray | None, X: np.ndarray, alpha: float = 2.0) -> np.ndarray:
    """H + alpha * X^T X for one token batch X (tokens x channels).

    Follows "The GPTQ Algorithm" (procedure step 2, H = 2XX^T with X channels x
    tokens), "GPTQ: fixing errors as you go" (Objective: H = 2XX^T, the same for every
    row) and the hook of "GPTQ-style round-to-nearest with Hessian weighting" (section
    "Computing the Hessian": x reshaped to tokens x features, H += x^T x per batch).
    X here is token-major, so X^T X is the pages' X X^T.
    """
    X = np.asarray(X, dtype=np.float64)
    G = X.T @ X
    G *= alpha
    return G if H is None else H + G


def hessian(batches, alpha: float = 2.0) -> np.ndarray:
    """H = alpha * sum over batches of X_b^T X_b (float64)."""
    H = None
    for X in batches:
        H = hessian_accumulate(H, X, alpha)
    return H


def hessian_entries(X: np.ndarray, rows: np.ndarray, cols: np.ndarray, alpha: float = 2.0) -> np.ndarray:
    """alpha * sum_t X[t, i] X[t, j] for the given (i, j) pairs, one dot product each."""
    out = np.empty(len(rows), dtype=np.float64)
    for k, (i, j) in enumerate(zip(rows, cols)):
        out[k] = alpha * np.dot(X[:, i].astype(np.float64), X[:, j].astype(np.float64))
    return out


# ----------------------------------------------------------------------------------
# Stage 2: damping, act-order and the Cholesky chain
# ----------------------------------------------------------------------------------
def damp(H: np.ndarray, percdamp: float = 0.01, dtype=np.float64):
    """(H_d, lambda) with lambda = percdamp * mean(diag H) added to every diagonal entry.

    "GPTQ, Line by Line", question "What does percdamp (dampening) do in GPTQ?"; the
    same two steps open the listing of "GPTQ-style round-to-nearest with Hessian
    weighting". The mean runs over all d diagonal entries, dead channels included.
    """
    H = np.array(H, dtype=dtype, copy=True)
    lam = dtype(percdamp) * np.mean(np.diag(H))
    if not np.isfinite(lam) or lam <= 0:
        raise ValueError("damping term must be positive and finite")
    H[np.diag_indices_from(H)] += lam
    return H, lam


def act_order_perm(H: np.ndarray) -> np.ndarray:
    """Column order of decreasing H_qq, ties by lower index first.

    "The GPTQ Algorithm" (ActOrder: decreasing order of the Hessian diagonal) and
    "GPTQ: fixing errors as you go" (act-order / desc_act processes columns in order
    of decreasing H_qq).
    """
    return np.argsort(-np.diag(H), kind="stable").astype(np.int64)


def hinv1(Hd: np.ndarray, dtype=np.float64) -> np.ndarray:
    """Upper Cholesky factor of H_d^-1 by the pages' three-step chain.

    "GPTQ, Line by Line", question "Why does GPTQ use Cholesky factorizations instead
    of inverting the Hessian directly?": factor H into lower L, turn it into H^-1 by a
    Cholesky solve against the identity, take the upper Cholesky factor of H^-1. The
    listing of "GPTQ-style round-to-nearest with Hessian weighting" runs the same
    chain (cholesky, cholesky_inverse, upper cholesky).
    """
    Hd = np.asarray(Hd, dtype=dtype)
    L = np.linalg.cholesky(Hd)
    Hinv = scipy.linalg.cho_solve((L, True), np.eye(Hd.shape[0], dtype=dtype))
    Hinv = (Hinv + Hinv.T) * dtype(0.5)   # cho_solve returns it up to rounding symmetry
    return np.ascontiguousarray(np.linalg.cholesky(Hinv).T, dtype=dtype)


# ----------------------------------------------------------------------------------
# Quantizer
# ----------------------------------------------------------------------------------
def quant_params(w_group: np.ndarray, bits: int):
    """Per-row (scale, zero) of an asymmetric min/max grid over a group of columns.

    Listing of "GPTQ-style round-to-nearest with Hessian weighting": scale =
    (max - min) / (2^b - 1) clamped below at 1e-8, zero = round(-min / scale) clamped
    to [0, 2^b - 1]. Raw min and max are used (0 is not forced into the range).
    """
    qmax = 2 ** bits - 1
    dt = w_group.dtype.type
    wmin = w_group.min(axis=1)
    wmax = w_group.max(axis=1)
    scale = (wmax - wmin) / dt(qmax)
    scale = np.maximum(scale, dt(1e-8))
    zero = np.clip(np.rint(-wmin / scale), dt(0), dt(qmax))
    return scale, zero


def quantize(w: np.ndarray, scale: np.ndarray, zero: np.ndarray, bits: int) -> np.ndarray:
    """q = clamp(round(w / scale + zero), 0, 2^b - 1), returned in w's float type."""
    dt = w.dtype.type
    return np.clip(np.rint(w / scale + zero), dt(0), dt(2 ** bits - 1))


def dequantize(q: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """w_hat = (q - zero) * scale."""
    return (q - zero) * scale


# ----------------------------------------------------------------------------------
# Stage 3: the blocked column loop
# ----------------------------------------------------------------------------------
def _check_groups(d: int, group_size: int, blocksize: int) -> int:
    g = d if group_size in (-1, 0, None) else int(group_size)
    if g <= 0 or d % g:
        raise ValueError("d must be a multiple of group_size")
    if group_size not in (-1, 0, None) and g % blocksize and blocksize % g:
        raise ValueError("group_size and blocksize must divide one another")
    return g


def gptq_columns(W: np.ndarray, U: np.ndarray, bits: int, group_size: int = 128,
                 blocksize: int = 128, dtype=np.float64, return_err: bool = False) -> dict:
    """Quantize W (m x d, columns already in processing order) against Hinv1 = U.

    Blocked loop of "GPTQ, Line by Line", question "Why does GPTQ process the weight
    matrix in blocks of 128 columns?": inside a block each quantized column updates
    the block's remaining columns by a rank-one product; after the block the
    accumulated errors Err1 are applied to the columns right of it by one matrix
    product Err1 @ Hinv1[block, rest]. The per-column steps (group statistics at the
    group's first column, quantize, dequantize, error divided by Hinv1[j, j], update
    along Hinv1[j, j+1:]) follow the listing of "GPTQ-style round-to-nearest with
    Hessian weighting"; with blocksize 1 this is exactly that listing's loop.

    group_size -1 means one (scale, zero) per row, taken from W before any update.
    Returns codes (m x d, int64), scales and zeros (m x G), losses (m x d, the
    increase Err1^2 / 2 of the quadratic objective per element) and W_hat.
    """
    W = np.array(W, dtype=dtype, copy=True)
    U = np.asarray(U, dtype=dtype)
    m, d = W.shape
    g = _check_groups(d, group_size, blocksize)
    G = d // g
    codes = np.zeros((m, d), dtype=np.int64)
    scales = np.zeros((m, G), dtype=dtype)
    zeros = np.zeros((m, G), dtype=dtype)
    losses = np.zeros((m, d), dtype=dtype)
    What = np.zeros((m, d), dtype=dtype)
    errs = np.zeros((m, d), dtype=dtype) if return_err else None
    half = dtype(0.5)
    for i1 in range(0, d, blocksize):
        i2 = min(i1 + blocksize, d)
        Err1 = np.zeros((m, i2 - i1), dtype=dtype)
        for j in range(i1, i2):
            if j % g == 0:
                s, z = quant_params(W[:, j:j + g], bits)
                scales[:, j // g], zeros[:, j // g] = s, z
            s, z = scales[:, j // g], zeros[:, j // g]
            w = W[:, j]
            q = quantize(w, s, z, bits)
            wq = dequantize(q, s, z)
            err = (w - wq) / U[j, j]
            codes[:, j] = q.astype(np.int64)
            What[:, j] = wq
            Err1[:, j - i1] = err
            losses[:, j] = err * err * half
            W[:, j + 1:i2] -= np.outer(err, U[j, j + 1:i2])
        W[:, i2:] -= Err1 @ U[i1:i2, i2:]
        if return_err:
            errs[:, i1:i2] = Err1
    out = {"codes": codes, "scales": scales, "zeros": zeros, "losses": losses, "W_hat": What}
    if return_err:
        out["err"] = errs
    return out


def gptq_layer(W: np.ndarray, H: np.ndarray, bits: int = 4, group_size: int = 128,
               blocksize: int = 128, percdamp: float = 0.01, act_order: bool = False,
               dtype=np.float64) -> dict:
    """Damp H, optionally permute by act-order, build Hinv1, run the column loop and
    return codes, losses and W_hat in the original column order.

    Adds ``perm`` (identity without act-order), ``U`` (Hinv1 of the permuted damped
    H), ``lambda``, ``col_losses`` (losses summed over rows), ``H_d`` and ``g_idx``.

    With act-order and groups, groups are formed in processing order (the pages name
    act-order, "The GPTQ Algorithm", ActOrder, and groups of 128 columns, but not how
    the two combine; this is the plainest reading): the scale and zero of group k come
    from processed columns k*g ... (k+1)*g - 1, and original column j uses group
    g_idx[j] = (position of j in perm) // g. ``scales`` and ``zeros`` stay indexed by
    group.
    """
    W = np.asarray(W, dtype=dtype)
    m, d = W.shape
    Hd, lam = damp(H, percdamp, dtype=dtype)
    perm = act_order_perm(H) if act_order else np.arange(d)
    Hp = Hd[np.ix_(perm, perm)]
    U = hinv1(Hp, dtype=dtype)
    res = gptq_columns(W[:, perm], U, bits, group_size, blocksize, dtype=dtype)
    out = dict(res)
    for key in ("codes", "losses", "W_hat"):
        a = np.empty_like(res[key])
        a[:, perm] = res[key]
        out[key] = a
    g = d if group_size in (-1, 0, None) else group_size
    g_idx = np.empty(d, dtype=np.int64)
    g_idx[perm] = np.arange(d) // g
    out.update(perm=perm, U=U, H_d=Hd, col_losses=out["losses"].sum(axis=0), g_idx=g_idx)
    out["lambda"] = lam
    return out


def rtn(W: np.ndarray, bits: int, group_size: int = 128, dtype=np.float64) -> dict:
    """Round-to-nearest baseline: the same quantizer, each weight on its own.

    "GPTQ: fixing errors as you go" (section "What actually matters": RTN makes each
    weight as close as possible to its original value).
    """
    W = np.asarray(W, dtype=dtype)
    m, d = W.shape
    g = d if group_size in (-1, 0, None) else group_size
    codes = np.zeros((m, d), dtype=np.int64)
    What = np.zeros((m, d), dtype=dtype)
    scales = np.zeros((m, d // g), dtype=dtype)
    zeros = np.zeros((m, d // g), dtype=dtype)
    for k in range(d // g):
        sl = slice(k * g, (k + 1) * g)
        s, z = quant_params(W[:, sl], bits)
        q = quantize(W[:, sl], s[:, None], z[:, None], bits)
        codes[:, sl] = q.astype(np.int64)
        What[:, sl] = dequantize(q, s[:, None], z[:, None])
        scales[:, k], zeros[:, k] = s, z
    return {"codes": codes, "W_hat": What, "scales": scales, "zeros": zeros}


# ----------------------------------------------------------------------------------
# Layers one after another
# ----------------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Each value rounded to the nearest bfloat16 (8 significant bits, ties to even),
    returned as float64. Written from the format's definition: x = f * 2^e with
    0.5 <= |f| < 1, keep rint(f * 2^8) / 2^8. Values are assumed inside bfloat16's
    normal range (|x| between 2^-126 and 2^128) or zero."""
    x = np.asarray(x, dtype=np.float64)
    f, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(f, 8)), e - 8)


def sequential_pass(X0: np.ndarray, weights, bits: int = 4, group_size: int = 128,
                    blocksize: int = 128, percdamp: float = 0.01, act_order: bool = False,
                    propagate: str | None = "bf16") -> dict:
    """Quantize a chain of linear layers one after another, each on the inputs that the
    layers already quantized hand it.

    "The GPTQ Algorithm" (procedure, steps 1-4) and "GPTQ: fixing errors as you go" (the
    algorithm in words: record the layer's inputs, build H = 2 X X^T, go through the
    columns, then move to the next layer). The pages' models are not at hand; the
    plainest synthetic stand-in is a chain of linear layers W_1 (m_1 x d), W_2 (m_2 x
    m_1), ... with nothing between them. Layer l's calibration inputs are the outputs
    of the layers before it with their quantized weights, X_{l+1} = X_l W_hat_l^T,
    rounded to bfloat16 (the activations' storage type) unless ``propagate`` is None
    (kept in float64).

    Returns ``layers`` (one ``gptq_layer`` result per layer), ``inputs`` (X_l of every
    layer, float64), ``H`` (the undamped Hessian of every layer) and ``output`` (the
    last layer's quantized output X_{L+1} before rounding).
    """
    X = np.asarray(X0, dtype=np.float64)
    layers, inputs, hessians = [], [], []
    out = None
    for li, W in enumerate(weights):
        W = np.asarray(W, dtype=np.float64)
        if W.shape[1] != X.shape[1]:
            raise ValueError(f"layer {li}: W has {W.shape[1]} input channels, the inputs {X.shape[1]}")
        H = hessian([X])
        res = gptq_layer(W, H, bits, group_size, blocksize, percdamp, act_order)
        inputs.append(X)
        hessians.append(H)
        layers.append(res)
        out = X @ res["W_hat"].T
        X = round_to_bf16(out) if propagate == "bf16" else out
    return {"layers": layers, "inputs": inputs, "H": hessians, "output": out}


# ----------------------------------------------------------------------------------
# Storage
# ----------------------------------------------------------------------------------
def packed_words_per_row(d: int, bits: int) -> int:
    return (d * bits + 31) // 32


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Codes (m x d, values < 2^b) -> uint32 words (m x ceil(d*b/32)).

    The pages store "4-bit integers and one scale per 128 weights" ("GPTQ: fixing
    errors as you go", example "a 4-bit Llama layer") without fixing a bit order; the
    reading here is a little-endian bitstream per row: bit k of code (r, j) is bit
    j*b + k of row r's stream, and bit t of the stream is bit t % 32 of word t // 32.
    """
    codes = np.asarray(codes, dtype=np.int64)
    m, d = codes.shape
    if codes.min(initial=0) < 0 or codes.max(initial=0) >= 2 ** bits:
        raise ValueError("code out of range")
    nw = packed_words_per_row(d, bits)
    bitstream = ((codes[:, :, None] >> np.arange(bits)) & 1).astype(np.uint8).reshape(m, d * bits)
    padded = np.zeros((m, nw * 32), dtype=np.uint8)
    padded[:, :d * bits] = bitstream
    return np.packbits(padded, axis=1, bitorder="little").view("<u4").reshape(m, nw)


def unpack_codes(words: np.ndarray, bits: int, d: int) -> np.ndarray:
    """Inverse of ``pack_codes``."""
    words = np.ascontiguousarray(words, dtype="<u4")
    m = words.shape[0]
    bitstream = np.unpackbits(words.view(np.uint8).reshape(m, -1), axis=1, bitorder="little")
    b = bitstream[:, :d * bits].reshape(m, d, bits).astype(np.int64)
    return (b << np.arange(bits)).sum(axis=2)


# ----------------------------------------------------------------------------------
# Using the stored layer: dequantize and multiply
# ----------------------------------------------------------------------------------
def dequantize_packed(words: np.ndarray, scales: np.ndarray, zeros: np.ndarray, bits: int, d: int,
                      group_size: int = 128, g_idx=None) -> np.ndarray:
    """W_hat (m x d, float64) from packed codes and per-group scale and zero.

    After quantization the layer is used as before ("GPTQ: fixing errors as you go",
    section on what changes at inference time: the stored low-bit weights and one scale
    per group stand in for the full-precision ones): w_hat = (code - zero) * scale with
    the (scale, zero) of the column's group, g_idx[j] (default j // group_size).
    """
    codes = unpack_codes(words, bits, d).astype(np.float64)
    g = d if group_size in (-1, 0, None) else group_size
    gi = np.arange(d) // g if g_idx is None else np.asarray(g_idx, dtype=np.int64)
    return dequantize(codes, np.asarray(scales, dtype=np.float64)[:, gi], np.asarray(zeros, dtype=np.float64)[:, gi])


def dequant_matmul(X: np.ndarray, words: np.ndarray, scales: np.ndarray, zeros: np.ndarray, bits: int,
                   group_size: int = 128, g_idx=None) -> np.ndarray:
    """Y = X W_hat^T in float64 for tokens X (T x d): the layer's output computed from
    its stored form."""
    X = np.asarray(X, dtype=np.float64)
    return X @ dequantize_packed(words, scales, zeros, bits, X.shape[1], group_size, g_idx).T


# ----------------------------------------------------------------------------------
# Metrics
# ----------------------------------------------------------------------------------
def loss_quadratic_form(dW: np.ndarray, H: np.ndarray) -> float:
    """1/2 * trace(dW H dW^T)."""
    dW = np.asarray(dW, dtype=np.float64)
    return 0.5 * float(np.sum((dW @ np.asarray(H, dtype=np.float64)) * dW))


def relative_output_error(W: np.ndarray, W_hat: np.ndarray, H0: np.ndarray) -> float:
    """||(W - W_hat) X^T||_F / ||W X^T||_F computed as sqrt(tr(dW H0 dW^T) / tr(W H0 W^T))
    with H0 proportional to X^T X (undamped): the objective of "GPTQ: fixing errors as you
    go" (section Objective) relative to the layer's output energy.
    """
    W = np.asarray(W, dtype=np.float64)
    dW = W - np.asarray(W_hat, dtype=np.float64)
    H0 = np.asarray(H0, dtype=np.float64)
    num = np.sum((dW @ H0) * dW)
    den = np.sum((W @ H0) * W)
    return float(np.sqrt(num / den))
