"""Pins of the oracle's E4M3 output branch (``assemble``), CPU only.

The contract (SparkInfer PR #75 "Add BF16 MLA query projection and assembly",
section Contract): the FP32-accumulated projection is rounded to BF16 first,
and only then optionally converted to E4M3 scaled by ``q_scale``.  The
benchmark configuration spells the conversion ``saturate(rne_e4m3(val /
q_scale))``; the reading taken is one IEEE binary32 division of the
BF16-rounded value, then a saturating round-to-nearest-even E4M3 cast.

Each expectation here is built from library calls only -- PyTorch's float64
matmul, its float32 -> bfloat16 cast, its float32 division and its
float32 -> float8_e4m3fn cast (after clamping to +-448, because the library
cast does not saturate) -- never from the oracle's own codecs.  The inputs
are chosen so that a plausible mistake in the branch changes some codes:

* projections that are not BF16 values, so an oracle that skipped the BF16
  rounding before the division fails;
* scales that are not powers of two, and (value, scale) pairs found by search
  whose reciprocal product RN(p * RN(1/q)) converts to a different code than
  the quotient RN(p / q), so an oracle that multiplied by a reciprocal fails;
* pairs whose binary32 quotient is exactly an E4M3 midpoint while the exact
  quotient is not, so an oracle that rounded the float64 quotient straight to
  E4M3 (skipping the binary32 rounding) fails.

Every test also checks, with the same library calls, that the wrong variant
really differs on its inputs, so the pin cannot pass vacuously.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

K, N, R = 128, 512, 64


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _lib_bf16_f32(bits):
    """BF16 bits -> float32 through PyTorch's dtype view and cast."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(torch.float32)


def _lib_e4m3(x_f32):
    """float32 tensor -> E4M3 codes: PyTorch's RNE cast after clamping to +-448."""
    return torch.clamp(x_f32, -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _lib_chain(acc_f32, q_scale):
    """The contract written with library casts: BF16 round, binary32 division, E4M3."""
    p = acc_f32.to(torch.bfloat16).to(torch.float32)
    return _lib_e4m3(p / torch.tensor(q_scale, dtype=torch.float32))


# --------------------------------------------------------------------------- BF16 rounding first

def _few_hot_layer(seed, H, M):
    """q_nope with 8 significant bits in [0.25, 4) and weights with three
    nonzeros per latent column, each with at most 4 significant bits in
    [0.25, 2): every projection is a sum of three products whose exact value
    fits binary32 (so the library's float32 -> bfloat16 cast is the single
    rounding the contract asks for), yet most are not BF16 values."""
    rng = np.random.default_rng(seed)
    sig = 1.0 + rng.integers(0, 128, size=(M, H, K)) / 128.0
    q = sig * np.exp2(rng.integers(-2, 2, size=(M, H, K))) * rng.choice([-1.0, 1.0], size=(M, H, K))
    w = np.zeros((H, K, N))
    wvals = np.array([1.5, 0.375, -0.8125, 1.25, -0.625, 0.875, -1.75, 0.3125])
    for h in range(H):
        for n in range(N):
            ks = rng.choice(K, size=3, replace=False)
            w[h, ks, n] = rng.choice(wvals, size=3)
    qp = rng.standard_normal((M, H, R))
    return _bf16_bits(q), _bf16_bits(qp), _bf16_bits(w)


@pytest.mark.parametrize("q_scale", [0.0371, 0.01, 0.1, 0.0913, 0.037])
def test_e4m3_branch_rounds_to_bf16_before_dividing(q_scale):
    H, M = 2, 8
    qn, qp, w = _few_hot_layer(int(q_scale * 1e4), H, M)
    qs = np.float32(q_scale)
    out, _ = oracle.mla_query(qn, qp, w, None, "bf16", "e4m3", qs)

    # Independent projection: PyTorch float64 matmul of the library-decoded operands.
    q64 = _lib_bf16_f32(qn).to(torch.float64)
    w64 = _lib_bf16_f32(w).to(torch.float64)
    acc = torch.einsum("mhk,hkn->mhn", q64, w64)
    acc32 = acc.to(torch.float32)
    assert torch.equal(acc32.to(torch.float64), acc), "projections must be exact in binary32"
    assert (acc32 != acc32.to(torch.bfloat16).to(torch.float32)).float().mean() > 0.5

    want = _lib_chain(acc32, qs)
    np.testing.assert_array_equal(out[..., :N], want)
    want_pe = _lib_e4m3(_lib_bf16_f32(qp) / torch.tensor(qs))
    np.testing.assert_array_equal(out[..., N:], want_pe)

    # The pin discriminates: without the BF16 rounding, codes change.
    skipped = _lib_e4m3(acc32 / torch.tensor(qs))
    assert (skipped != want).sum() > 0
    # and most codes are not saturated
    assert ((want & 0x7F) < 0x7E).mean() > 0.5


# --------------------------------------------------------------------------- division, not reciprocal

def _e4m3_midpoint_f32(x):
    """True where float32 x is exactly halfway between two adjacent E4M3
    normal values (x in the E4M3 normal range, below 448)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    return ((b & 0xFFFFF) == 0x80000) & (np.abs(x) >= 2.0 ** -6) & (np.abs(x) < 448)


def _search_pairs():
    """(value, scale) pairs for the division pins, found by scanning scales
    that are not powers of two against every BF16 significand.

    Values are (128 + f) * 2^-10 (BF16 values in [0.125, 0.25)), scales lie
    in [0.01, 0.1], so quotients lie in the E4M3 normal range.  Returns
    (recip, tie): pairs where the reciprocal product converts to another code
    than the quotient, and pairs whose binary32 quotient is an E4M3 midpoint
    while the exact quotient is not."""
    p = ((128 + np.arange(128)) * 2.0 ** -10).astype(np.float32)
    qs = np.linspace(0.01, 0.1, 240001, dtype=np.float64).astype(np.float32)
    recip, tie = [], []
    for lo in range(0, qs.size, 20000):
        q = qs[lo:lo + 20000, None]
        div = p[None, :] / q
        mul = p[None, :] * (np.float32(1.0) / q)
        d_code = _lib_e4m3(torch.from_numpy(np.ascontiguousarray(div)))
        m_code = _lib_e4m3(torch.from_numpy(np.ascontiguousarray(mul)))
        for i, j in zip(*np.nonzero(d_code != m_code)):
            recip.append((p[j], q[i, 0]))
        for i, j in zip(*np.nonzero(_e4m3_midpoint_f32(div))):
            if Fraction(float(p[j])) / Fraction(float(q[i, 0])) != Fraction(float(div[i, j])):
                tie.append((p[j], q[i, 0]))
    return recip, tie


_PAIRS = None


def _pairs():
    global _PAIRS
    if _PAIRS is None:
        _PAIRS = _search_pairs()
    return _PAIRS


def _e4m3_of_exact(p, q):
    """E4M3 code of the exact rational p / q, RNE, found by exact comparison
    with the library-decoded E4M3 grid (positive, normal range, below 448)."""
    grid = torch.arange(0x08, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    x = Fraction(float(p)) / Fraction(float(q))
    for i in range(grid.size - 1):
        a, b = Fraction(float(grid[i])), Fraction(float(grid[i + 1]))
        if a <= x <= b:
            mid = (a + b) / 2
            if x < mid:
                return 0x08 + i
            if x > mid:
                return 0x09 + i
            return 0x08 + i if (0x08 + i) % 2 == 0 else 0x09 + i
    raise AssertionError("quotient outside the E4M3 normal range")


def _identity_call(values, q_scale):
    """Oracle E4M3 output of identity weights on one token whose q_nope
    holds `values` (BF16 values): the projection's first columns are exactly
    those values."""
    H, M = 1, 1
    v = np.zeros(K, dtype=np.float32)
    v[:len(values)] = values
    qn = _bf16_bits(v.reshape(M, H, K))
    assert np.array_equal(_lib_bf16_f32(qn).numpy().reshape(-1), v), "values must be BF16 values"
    eye = np.zeros((H, K, N), dtype=np.float32)
    for k in range(K):
        eye[:, k, k] = 1.0
    qp = _bf16_bits(np.zeros((M, H, R)))
    out, _ = oracle.mla_query(qn, qp, _bf16_bits(eye), None, "bf16", "e4m3", np.float32(q_scale))
    return out[0, 0, :len(values)]


def test_e4m3_branch_divides_instead_of_multiplying_by_a_reciprocal():
    recip, _ = _pairs()
    assert len(recip) >= 8, "the scan should find pairs where the reciprocal product decides another code"
    for p, q in recip[:: max(1, len(recip) // 24)]:
        got = _identity_call([p], q)
        want = _lib_e4m3(torch.tensor([p]) / torch.tensor([q]))
        wrong = _lib_e4m3(torch.tensor([p]) * (1.0 / torch.tensor([q])))
        assert want[0] != wrong[0]
        assert got[0] == want[0], (float(p), float(q), int(got[0]), int(want[0]))


def test_e4m3_branch_rounds_the_quotient_to_binary32_first():
    _, tie = _pairs()
    assert len(tie) >= 2, "the scan should find quotients that round onto an E4M3 midpoint"
    differing = 0
    for p, q in tie:
        got = _identity_call([p], q)
        want = _lib_e4m3(torch.tensor([p]) / torch.tensor([q]))
        assert got[0] == want[0], (float(p), float(q), int(got[0]), int(want[0]))
        # RN32 lands on the midpoint, so the tie goes to the even code; the
        # exact quotient lies to one side of it and may round the other way.
        assert want[0] % 2 == 0
        differing += int(_e4m3_of_exact(p, q) != want[0])
    assert differing >= 1, "some tie case must separate binary32 rounding from exact rounding"


def test_e4m3_branch_q_pe_columns_use_the_same_division():
    recip, _ = _pairs()
    for p, q in recip[:8]:
        H, M = 1, 1
        qn = _bf16_bits(np.zeros((M, H, K)))
        pe = np.zeros((M, H, R), dtype=np.float32)
        pe[0, 0, 5] = p
        pe[0, 0, 6] = -p
        out, _ = oracle.mla_query(qn, _bf16_bits(pe), _bf16_bits(np.zeros((H, K, N))), None, "bf16", "e4m3",
                                  np.float32(q))
        want = _lib_e4m3(torch.from_numpy(pe[0, 0]) / torch.tensor(np.float32(q)))
        np.testing.assert_array_equal(out[0, 0, N:], want)
