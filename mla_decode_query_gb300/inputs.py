"""Seeded synthetic inputs for the fused MLA decode query projection.

Shared by the tests, the benchmark and the CPU oracle's callers; it holds none
of the operation's arithmetic.  Every tensor is returned as raw bits in numpy
arrays (uint16 for BF16, uint8 for E4M3 / E8M0) so that the CUDA path and the
oracle consume identical bytes.  Float-to-BF16 and float-to-E4M3 conversion
of the *drawn* values uses PyTorch's CPU dtype casts (round-to-nearest-even),
a library routine.

Recipe (one layer, seed ``s``; ``numpy.random.Generator(PCG64(s))``), drawn
in this order so that the weights do not depend on how many tokens are used:

1. weights ``W_UK_T[h,k,n]`` ~ N(0, sigma = 1/sqrt(K)), float32, shape
   ``[H,K,512]`` (nope dim K = 128 unless asked otherwise); BF16 format: cast
   to BF16.  MXFP8 format: cast to E4M3 (the values stay far below the E4M3
   maximum 448);
2. MXFP8 only: scale exponents ``e`` uniform on the integers -4..2, one per
   32 consecutive latent elements of each (h,k) row, stored as the E8M0 byte
   ``127 + e`` in ``[H,K,16]``;
3. ``q_nope`` ~ N(0,1), ``[M_MAX,H,K]``, cast to BF16;
4. ``q_pe``  ~ N(0,1), ``[M_MAX,H,64]``, cast to BF16;
   callers using M < M_MAX tokens take the first M rows.

``q_scale`` (E4M3 output) is drawn once per run, uniform on [0.01, 0.1], as a
float32 from its own seed.
"""

from __future__ import annotations

import numpy as np
import torch

NOPE = 128
LATENT = 512
ROPE = 64
M_MAX = 32
SIGMA_W = 1.0 / np.sqrt(128.0)


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def layer_seed(config_index: int, layer: int) -> int:
    """Seed of layer ``layer`` in workload ``config_index`` (1000*i + l)."""
    return 1000 * int(config_index) + int(layer)


def make_layer(seed: int, H: int, weight_format: str, m_max: int = M_MAX, nope: int = NOPE) -> dict:
    """Draw one layer's inputs.  Returns a dict of numpy bit arrays:

    ``q_nope`` uint16 [m_max,H,nope], ``q_pe`` uint16 [m_max,H,64],
    ``weight`` uint16 (bf16) or uint8 (mxfp8) [H,nope,512],
    ``weight_scale`` uint8 [H,nope,16] or None.  The weight std is
    1/sqrt(nope) (1/sqrt(128) for the default nope dim 128).
    """
    if weight_format not in ("bf16", "mxfp8"):
        raise ValueError(f"unknown weight format {weight_format!r}")
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_normal((H, nope, LATENT), dtype=np.float32) * np.float32(1.0 / np.sqrt(nope))
    if weight_format == "bf16":
        weight = _to_bf16_bits(w)
        scale = None
    else:
        weight = _to_e4m3_bits(w)
        exps = rng.integers(-4, 3, size=(H, nope, LATENT // 32))
        scale = (127 + exps).astype(np.uint8)
    q_nope = _to_bf16_bits(rng.standard_normal((m_max, H, nope), dtype=np.float32))
    q_pe = _to_bf16_bits(rng.standard_normal((m_max, H, ROPE), dtype=np.float32))
    return {"q_nope": q_nope, "q_pe": q_pe, "weight": weight, "weight_scale": scale}


def make_q_scale(seed: int) -> np.float32:
    """Per-run E4M3 output scale, uniform on [0.01, 0.1]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.float32(rng.uniform(0.01, 0.1))


def small_integer_layer(seed: int, H: int, M: int, weight_format: str, nope: int = NOPE) -> dict:
    """Inputs whose products and partial sums are exact in binary32.

    ``q_nope`` in {-2..2}, weights in {-1, 0, 1} (MXFP8: E4M3 codes of
    -1, 0, 1 with scale byte 127).  Every partial sum is an integer of
    magnitude <= 2*nope, so any summation order gives the same binary32
    value, and its BF16 rounding is the same on every path: the projection
    must then match bit for bit.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.integers(-2, 3, size=(M, H, nope)).astype(np.float32)
    w = rng.integers(-1, 2, size=(H, nope, LATENT)).astype(np.float32)
    pe = rng.integers(-8, 9, size=(M, H, ROPE)).astype(np.float32) * np.float32(0.25)
    if weight_format == "bf16":
        weight, scale = _to_bf16_bits(w), None
    else:
        weight = _to_e4m3_bits(w)
        scale = np.full((H, nope, LATENT // 32), 127, dtype=np.uint8)
    return {"q_nope": _to_bf16_bits(q), "q_pe": _to_bf16_bits(pe), "weight": weight,
            "weight_scale": scale}


V_HEAD = 128


def make_v_layer(seed: int, H: int, weight_format: str, m_max: int = M_MAX) -> dict:
    """Draw one layer's V up-projection inputs (same recipe style):

    1. ``W_UV[h,c,d]`` ~ N(0, 1/sqrt(512)), ``[H,512,128]``, cast to BF16 or E4M3;
    2. MXFP8 only: E8M0 bytes ``127 + U{-4..2}``, ``[H,512,4]`` (one per 32
       consecutive output elements of each (h,c) row);
    3. ``x`` (attention output in the latent space) ~ N(0,1), ``[m_max,H,512]``,
       cast to BF16.
    Returns ``x`` uint16, ``weight`` uint16 / uint8, ``weight_scale`` uint8 or None.
    """
    if weight_format not in ("bf16", "mxfp8"):
        raise ValueError(f"unknown weight format {weight_format!r}")
    rng = np.random.Generator(np.random.PCG64(seed))
    w = rng.standard_normal((H, LATENT, V_HEAD), dtype=np.float32) * np.float32(1.0 / np.sqrt(LATENT))
    if weight_format == "bf16":
        weight, scale = _to_bf16_bits(w), None
    else:
        weight = _to_e4m3_bits(w)
        scale = (127 + rng.integers(-4, 3, size=(H, LATENT, V_HEAD // 32))).astype(np.uint8)
    x = _to_bf16_bits(rng.standard_normal((m_max, H, LATENT), dtype=np.float32))
    return {"x": x, "weight": weight, "weight_scale": scale}


def small_integer_v_layer(seed: int, H: int, M: int, weight_format: str) -> dict:
    """V up-projection inputs whose sums are exact in binary32: ``x`` in
    {-2..2}, weights in {-1, 0, 1} (scale byte 127), every partial sum an
    integer of magnitude <= 1024, so any summation order gives the same FP32
    value and the same BF16 rounding."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.integers(-2, 3, size=(M, H, LATENT)).astype(np.float32)
    w = rng.integers(-1, 2, size=(H, LATENT, V_HEAD)).astype(np.float32)
    if weight_format == "bf16":
        weight, scale = _to_bf16_bits(w), None
    else:
        weight = _to_e4m3_bits(w)
        scale = np.full((H, LATENT, V_HEAD // 32), 127, dtype=np.uint8)
    return {"x": _to_bf16_bits(x), "weight": weight, "weight_scale": scale}
