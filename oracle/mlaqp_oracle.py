"""Plain CPU oracle for the fused MLA decode query projection and assembly.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` use it.  It shares no code with
the CUDA path; both sides see the same input *bits*, produced by the seeded
generators in ``mla_decode_query_gb300.inputs``.

What it computes (SparkInfer PR #75 "Add BF16 MLA query projection and
assembly", sections *What* and *Contract*; vLLM PR #174 "Fuse MXFP8 and BF16
MLA query assembly", section *What*):

  for every token m and head h
      acc[m,h,n]  = sum_k q_nope[m,h,k] * W_UK_T[h,k,n]        n < 512
      p[m,h,n]    = bf16_rne(acc[m,h,n])      (the staged operation boundary)
      out[m,h,:512] = p                              (BF16 output)
                    = e4m3_satfinite_rne(p / q_scale)  (E4M3 output)
      out[m,h,512:576] = q_pe[m,h,:]                 (BF16 output, bit copy)
                       = e4m3_satfinite_rne(q_pe / q_scale)  (E4M3 output)

Everything is evaluated in float64.  Products of two BF16 values, or of a
BF16 value and a dequantised MXFP8 weight, are exact in float64, so ``acc``
differs from the exact sum only by float64 summation rounding (about 1e-16
relative), which is negligible against every tolerance used with it.

Readings of the pages taken here (the pages are silent or garbled):

* nope dim K = 128, latent N = 512, rope R = 64 (the pages' GLM example uses
  K = 192; K is a parameter of every function below).
* ``q_nope`` is token-major ``[M,H,K]``; ``q_pe`` is ``[M,H,64]``.
* MXFP8 weights: OCP E4M3FN codes ``[H,K,N]`` with one E8M0 scale per 32
  consecutive latent (N) elements of each (h,k) row, stored ``[H,K,N/32]``
  (the pages say only ``sf_axis="n"``, ``b_major="n"``).
* The E4M3 output cast is ``satfinite``: NaN -> NaN, |x| > 448 -> +-448,
  otherwise round-to-nearest-even including subnormals; the division by
  ``q_scale`` is an IEEE float32 division of the BF16-rounded value.

The V up-projection after attention (``mla_v_up``): the pages name it only
as the downstream step that a separate change handles (vLLM PR #174, section
Safety scope).  Reading taken: per head, the attention output over the latent
cache ``x[M,H,512]`` (BF16) times ``W_UV[H,512,128]``, FP32 accumulation,
BF16 output ``[M,H,128]``; ``W_UV`` is stored with its output (v) axis
fastest, BF16 or MXFP8 with one E8M0 scale per 32 consecutive output
elements of each (h,c) row (``[H,512,4]``), the convention of ``W_UK_T``.

Functions whose behaviour is pinned only by the format specifications and
closed forms (no worked example is printed on the pages): all of them.  The
pins live in ``tests/test_oracle_*.py``.
"""

from __future__ import annotations

import numpy as np

NOPE_DIM = 128
LATENT_DIM = 512
V_HEAD_DIM = 128
ROPE_DIM = 64
OUT_DIM = LATENT_DIM + ROPE_DIM
MX_BLOCK = 32

E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# BF16 (IEEE-754 binary32 with the low 16 significand bits dropped)
# ---------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Decode BF16 bit patterns (uint16) exactly to float64.

    A BF16 value is the binary32 value whose upper 16 bits are the BF16 bits
    and whose lower 16 bits are zero.
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_rne(x) -> np.ndarray:
    """Round float64 values to BF16 with one IEEE round-to-nearest-even step.

    BF16 keeps 8 significant bits and binary32's exponent range: normals from
    2**-126, subnormals in steps of 2**-133, largest finite (2 - 2**-7)*2**127.
    Values that round to 2**128 or beyond become +-inf; NaN stays NaN.
    The rounding is done once from the float64 value (no intermediate
    binary32 rounding, which could round twice).
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    sign = np.signbit(x)
    ax = np.abs(x)
    finite = np.isfinite(ax)
    safe = np.where(finite & (ax > 0), ax, 1.0)
    _, e = np.frexp(safe)  # safe = f * 2**e, f in [0.5, 1)
    # leading bit has weight 2**(e-1); 7 fraction bits -> quantum 2**(e-8),
    # never finer than the subnormal step 2**-133.
    qexp = np.maximum(e - 8, -133)
    q = np.ldexp(1.0, qexp)
    r = np.round(safe / q) * q  # np.round: halves go to the even integer
    r = np.where(ax > 0, r, 0.0)
    overflow = finite & (r >= 2.0 ** 128)
    r32 = np.where(overflow | ~finite, 0.0, r).astype(np.float32)  # exact
    mag = (r32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    mag = np.where(overflow | np.isinf(ax), np.uint16(0x7F80), mag)
    mag = np.where(np.isnan(ax), np.uint16(0x7FC0), mag)
    out[...] = mag | np.where(sign, np.uint16(0x8000), np.uint16(0))
    return out


def bf16_to_f32(bits) -> np.ndarray:
    """Decode BF16 bits to float32 (exact: BF16 is a subset of binary32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# OCP 8-bit floating point, E4M3 "fn" variant (no infinities, NaN = S.1111.111)
# ---------------------------------------------------------------------------

def e4m3_to_f64(codes) -> np.ndarray:
    """Decode E4M3 codes exactly to float64.

    Code bits ``s eeee mmm`` with exponent bias 7:
      e == 15 and m == 7  -> NaN (there is no infinity)
      e == 0              -> (-1)**s * (m/8) * 2**-6        (subnormal)
      otherwise           -> (-1)**s * (1 + m/8) * 2**(e-7)
    The largest finite magnitude is 448 = 1.75 * 2**8.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = c >> 7
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = (m / 8.0) * 2.0 ** -6
    nor = (1.0 + m / 8.0) * np.ldexp(1.0, e - 7)
    v = np.where(e == 0, sub, nor)
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return np.where(s == 1, -v, v)


_E4M3_MAGNITUDES = e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))  # codes 0..126, increasing


def f32_to_e4m3_satfinite(x) -> np.ndarray:
    """Encode float32 values to E4M3 codes, round-to-nearest-even, saturating.

    NaN -> 0x7F with the input's sign bit; |x| > 448 (infinities included)
    -> +-448 (code 0x7E); otherwise the nearest E4M3 value, ties to the code
    with an even mantissa, subnormals (step 2**-9) included; results that
    round to zero keep the input's sign.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x)
    ax = np.abs(x)
    nan = np.isnan(ax)
    sat = ~nan & (ax > E4M3_MAX)
    safe = np.where(nan | sat | (ax == 0), 1.0, ax)
    _, e = np.frexp(safe)  # leading bit weight 2**(e-1), 3 fraction bits
    qexp = np.maximum(e - 4, -9)
    q = np.ldexp(1.0, qexp)
    r = np.round(safe / q) * q
    r = np.where(ax == 0, 0.0, r)
    r = np.where(nan | sat, E4M3_MAX, r)
    code = np.searchsorted(_E4M3_MAGNITUDES, r).astype(np.int64)
    assert np.all(_E4M3_MAGNITUDES[np.minimum(code, 126)] == r), "grid miss"
    code = np.where(nan, 0x7F, code)
    return (code | np.where(sign, 0x80, 0)).astype(np.uint8)


# ---------------------------------------------------------------------------
# OCP Microscaling shared scale, E8M0 (unsigned power of two, 0xFF = NaN)
# ---------------------------------------------------------------------------

def e8m0_to_f64(codes) -> np.ndarray:
    """Decode E8M0 scale bytes: x -> 2**(x - 127), 255 -> NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 255, np.nan, v)


# ---------------------------------------------------------------------------
# The operation
# ---------------------------------------------------------------------------

def decode_weight(weight, weight_scale, weight_format: str) -> np.ndarray:
    """Return a per-head weight (W_UK_T ``[H,K,N]``, or W_UV ``[H,512,128]``
    with K the contraction and N the output axis) as float64.

    ``weight_format == "bf16"``: ``weight`` holds BF16 bits ``[H,K,N]``.
    ``weight_format == "mxfp8"``: ``weight`` holds E4M3 codes ``[H,K,N]`` and
    ``weight_scale`` E8M0 bytes ``[H,K,N/32]``; element (h,k,n) is
    ``e4m3(code[h,k,n]) * 2**(scale[h,k,n//32] - 127)`` (exact in float64).
    """
    if weight_format == "bf16":
        if weight_scale is not None:
            raise ValueError("BF16 weights take no scale tensor")
        return bf16_to_f64(weight)
    if weight_format == "mxfp8":
        w = e4m3_to_f64(weight)
        s = e8m0_to_f64(weight_scale)
        if s.shape[:-1] != w.shape[:-1] or s.shape[-1] * MX_BLOCK != w.shape[-1]:
            raise ValueError("scale shape must be [H,K,N/32]")
        return w * np.repeat(s, MX_BLOCK, axis=-1)
    raise ValueError(f"unknown weight format {weight_format!r}")


def project(q_nope, w64) -> np.ndarray:
    """Per-head contraction in float64: acc[m,h,n] = sum_k q[m,h,k] * w[h,k,n].

    ``q_nope``: BF16 bits ``[M,H,K]``; ``w64``: float64 ``[H,K,N]``.
    One float64 matmul per head (a library primitive); no blocking.
    """
    q = bf16_to_f64(q_nope)  # [M,H,K]
    M, H, K = q.shape
    if w64.shape[0] != H or w64.shape[1] != K:
        raise ValueError("weight must be [H,K,N] matching q_nope [M,H,K]")
    acc = np.empty((M, H, w64.shape[2]), dtype=np.float64)
    for h in range(H):
        acc[:, h, :] = q[:, h, :] @ w64[h]
    return acc


def assemble(acc, q_pe, out_dtype: str, q_scale=None) -> np.ndarray:
    """Build the ``[M,H,N+R]`` query from the projection and ``q_pe``.

    BF16 output (``out_dtype == "bf16"``): uint16 bits; the first N columns
    are ``bf16_rne(acc)``, the last R the ``q_pe`` bits unchanged.
    E4M3 output (``out_dtype == "e4m3"``): uint8 codes; the first N columns
    are ``e4m3_satfinite(f32(bf16_rne(acc)) / f32(q_scale))`` and the last R
    ``e4m3_satfinite(f32(q_pe) / f32(q_scale))``, the division being one
    IEEE binary32 division.  The BF16 rounding precedes the E4M3 conversion
    (page "Add BF16 MLA query projection and assembly", section Contract).
    """
    p = f64_to_bf16_rne(acc)
    pe = np.asarray(q_pe, dtype=np.uint16)
    if pe.shape[:2] != acc.shape[:2]:
        raise ValueError("q_pe must be [M,H,R] matching acc [M,H,N]")
    if out_dtype == "bf16":
        if q_scale is not None:
            raise ValueError("BF16 output takes no q_scale")
        return np.concatenate([p, pe], axis=-1)
    if out_dtype == "e4m3":
        if q_scale is None:
            raise ValueError("E4M3 output requires q_scale")
        qs = np.float32(q_scale)
        with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
            xp = bf16_to_f32(p) / qs
            xr = bf16_to_f32(pe) / qs
        return np.concatenate([f32_to_e4m3_satfinite(xp), f32_to_e4m3_satfinite(xr)], axis=-1)
    raise ValueError(f"unknown output dtype {out_dtype!r}")


def mla_query(q_nope, q_pe, weight, weight_scale, weight_format: str, out_dtype: str,
              q_scale=None):
    """The whole operation for one layer call.

    Returns ``(out, acc)``: ``out`` the assembled ``[M,H,N+R]`` query bits
    (uint16 for BF16, uint8 for E4M3) and ``acc`` the float64 projection
    ``[M,H,N]`` before any rounding, for tolerance checks.
    """
    w64 = decode_weight(weight, weight_scale, weight_format)
    acc = project(q_nope, w64)
    return assemble(acc, q_pe, out_dtype, q_scale), acc


def write_workspace(workspace, out, row_stride: int):
    """Write ``out`` ``[M,H,D]`` into a flat workspace with a row pitch.

    Element (m,h,j) lands at ``workspace[m*row_stride + h*D + j]``; every
    other element (rows >= M, the pitch padding) keeps its previous value.
    Returns the updated copy.
    """
    ws = np.array(workspace, copy=True)
    M, H, D = out.shape
    for m in range(M):
        ws[m * row_stride: m * row_stride + H * D] = out[m].reshape(-1)
    return ws


def e4m3_ordinal(codes) -> np.ndarray:
    """Map E4M3 codes to a monotone integer scale (+0 and -0 both map to 0).

    Adjacent representable values differ by exactly 1, so ``|ord(a)-ord(b)|``
    counts E4M3 ulps between two finite codes.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def algorithmic_bytes(M: int, H: int, weight_format: str, out_dtype: str,
                      nope: int = NOPE_DIM, latent: int = LATENT_DIM, rope: int = ROPE_DIM) -> int:
    """Bytes one layer call must move at least once: weights (+ scales),
    q_nope, q_pe and the written output."""
    wb = 2 if weight_format == "bf16" else 1
    ob = 2 if out_dtype == "bf16" else 1
    w = H * nope * latent * wb
    s = H * nope * (latent // MX_BLOCK) if weight_format == "mxfp8" else 0
    return w + s + 2 * M * H * nope + 2 * M * H * rope + M * H * (latent + rope) * ob


# ---------------------------------------------------------------------------
# The V up-projection (the step after attention over the latent cache)
# ---------------------------------------------------------------------------

def mla_v_up(x, weight, weight_scale, weight_format: str):
    """V up-projection of one layer call.

    ``x``: BF16 bits ``[M,H,512]`` (attention output in the latent space);
    ``weight``: W_UV, BF16 bits or E4M3 codes ``[H,512,128]``;
    ``weight_scale``: E8M0 ``[H,512,4]`` (MXFP8) or None.
    out[m,h,d] = bf16_rne(sum_c x[m,h,c] * W_UV[h,c,d]).
    Returns ``(out, acc)``: uint16 bits ``[M,H,128]`` and the float64 sums.
    """
    w64 = decode_weight(weight, weight_scale, weight_format)
    if w64.shape[1:] != (LATENT_DIM, V_HEAD_DIM):
        raise ValueError("W_UV must be [H,512,128]")
    acc = project(x, w64)
    return f64_to_bf16_rne(acc), acc


def v_up_algorithmic_bytes(M: int, H: int, weight_format: str, latent: int = LATENT_DIM,
                           v_dim: int = V_HEAD_DIM) -> int:
    """Bytes one V up-projection call must move at least once: W_UV (+ scales),
    the attention output x and the BF16 result."""
    wb = 2 if weight_format == "bf16" else 1
    s = H * latent * (v_dim // MX_BLOCK) if weight_format == "mxfp8" else 0
    return H * latent * v_dim * wb + s + 2 * M * H * latent + 2 * M * H * v_dim
