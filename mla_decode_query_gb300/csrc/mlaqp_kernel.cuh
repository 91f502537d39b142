// Fused MLA decode query projection + assembly for GB300 (sm_103a).
//
// For one layer call (SparkInfer PR #75 "Add BF16 MLA query projection and
// assembly", sections What and Contract; vLLM PR #174 "Fuse MXFP8 and BF16
// MLA query assembly", section What):
//   out[m,h,0:512]   = bf16(sum_k q_nope[m,h,k] * W_UK_T[h,k,:])  (FP32 sum)
//                      or e4m3_satfinite(that / q_scale)
//   out[m,h,512:576] = q_pe[m,h,:]  (bit copy, or the same E4M3 cast)
//
// Work split: CTA (tile, h) owns head h and latent columns
// [64*tile, 64*tile+64): 8 CTAs per head, 128 threads, one 16-column MMA
// tile per warp over the full K = 128.  Every weight byte is read once.
//
// Data path of one CTA:
//  1. thread 0 issues one 2-D TMA copy of the CTA's 128 x 64 weight tile
//     (BF16: straight into a 128B-swizzled BF16 tile; MXFP8: the E4M3 bytes
//     plus a 1-D bulk copy of the head's 2 KB of E8M0 scales);
//  2. warp 0 warms L2 with the head's q_nope / q_pe rows (prefetch only);
//     q_scale is read (a per-tensor constant, like the weights);
//  3. MXFP8: all threads wait for the copy and dequantise into the same
//     swizzled BF16 tile (e4m3 * 2^(e8m0-127), exact); BF16: all threads
//     wait for the copy and load their weight fragments (ldmatrix.trans);
//     E4M3 output: each of 128 threads adds one entry to the exact
//     division table and checks one significand for the exact one-multiply
//     conversion (see e4m3_mul_exact_for);
//  4. griddepcontrol.wait -- everything above is independent of the
//     previous kernel, so under programmatic dependent launch it overlaps
//     that kernel; everything below reads inputs it may have produced;
//  5. q_nope rows into a swizzled smem tile (16-byte loads), q_pe pairs into
//     registers, the MXFP8 weight fragments with ldmatrix.trans;
//  8. q_pe appended (bit copy or E4M3 cast), one value pair per thread,
//     ahead of the contraction so that it overlaps the MMA latency;
//  6. mma.sync m16n8k16 BF16 -> FP32 with the latent axis on the MMA's M
//     side and tokens on its N side (swap-AB: M <= 32 tokens costs at most
//     four 8-wide column tiles);
//  7. epilogue: round to BF16 (optionally divide by q_scale and convert to
//     E4M3 with saturation), transpose the 8x8 blocks with movmatrix so
//     each lane holds consecutive latent columns of one token, and store
//     straight into the caller's strided workspace.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the CTA
// records MLAQP_DEVSTATUS_WAIT_TIMEOUT in a device status word and returns
// without writing its outputs.

#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mlaqp {

constexpr int kNope = 128;     // nope dim of the benchmark configurations; 192 is also built
constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kOutDim = kLatent + kRope;
constexpr int kMxBlock = 32;
constexpr int kMaxM = 32;

constexpr int kNTile = 64;                       // latent columns per CTA
constexpr int kWarps = kNTile / 16;              // one 16-column MMA tile per warp
constexpr int kThreads = kWarps * 32;            // 128 threads per token group

// Token groups per CTA: for M > 8 (two or more 8-token MMA column tiles) a
// second group of four warps takes every other token tile, halving each
// warp's MMA and epilogue work; M <= 8 uses one group.
constexpr int token_groups(int mt) { return mt >= 2 ? 2 : 1; }
constexpr int kTilesPerHead = kLatent / kNTile;  // 8

// Dynamic shared memory layout for nope dim K (offsets from a 1024-byte
// aligned base; every region starts on at least a 16-byte boundary).
template <int K>
struct Smem {
  static constexpr int A = 0;                                 // BF16 [K][64], 128B swizzle
  static constexpr int Raw = A + K * kNTile * 2;              // E4M3 [K][64]
  static constexpr int Scale = Raw + K * kNTile;              // E8M0 [K][16]
  static constexpr int Q = Scale + K * (kLatent / kMxBlock);  // BF16 [32][K], 16B chunks XOR-swizzled
  static constexpr int Div = Q + kMaxM * K * 2;               // FP32 [128]: RN((128+f)/q_scale)
  static constexpr int Bar = Div + 128 * 4;
  static constexpr int Bytes = Bar + 64 + 1024;               // + slack for the 1024-byte alignment
};
constexpr int kSmemBytes = Smem<kNope>::Bytes;

enum WeightFormat : int { kWeightBF16 = 0, kWeightMXFP8 = 1 };
enum OutDtype : int { kOutBF16 = 0, kOutE4M3 = 1 };

constexpr unsigned kDevStatusWaitTimeout = 1u;

struct RunParams {
  CUtensorMap wmap;             // 2-D map of W_UK_T viewed as [H*128 rows][512 cols], box 64 x 128
  const uint16_t* q_nope;       // BF16, element (m,h,k) at m*q_nope_ts + h*q_nope_hs + k
  const uint16_t* q_pe;         // BF16, element (m,h,j) at m*q_pe_ts + h*q_pe_hs + j
  int64_t q_nope_ts, q_nope_hs; // token / head strides (elements)
  int64_t q_pe_ts, q_pe_hs;
  const uint8_t* weight_scale;  // E8M0 [H,128,16] or null
  uint8_t* out;                 // element (m,h,j) at m*out_row_stride + h*576 + j
  int64_t out_row_stride;       // elements
  const float* q_scale;         // device scalar or null
  unsigned long long wait_limit_ns;  // bound on every mbarrier wait
  unsigned int extra_tx;        // test hook: bytes the barrier expects beyond the copies
  int M;
  int H;
};

// One status word per translation unit; read by the host through the
// symbol.  Bits are only ever set by a CTA that gave up waiting.
static __device__ unsigned int g_device_status;

// ---------------------------------------------------------------------------
// PTX helpers (documented PTX instructions only)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of the barrier.  Returns false if the
// limit expired first.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t ld_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_u128(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two FP32 -> packed BF16x2, round to nearest even; `hi` lands in bits 31..16.
__device__ __forceinline__ uint32_t pack_bf16x2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two FP32 -> packed E4M3x2, round to nearest even, saturating to +-448;
// `hi` lands in bits 15..8.
__device__ __forceinline__ uint32_t pack_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// E4M3 codes in bytes 0 and 1 of `two` -> BF16x2 bit patterns of
// code * 2^-120 (byte 0 in the low half).  The E4M3 exponent and mantissa
// land in the low bits of the BF16 exponent and the high bits of its
// mantissa, so every code -- subnormals included -- maps to exactly its
// value times 2^(7-127).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_scaled(uint32_t two) {
  const uint32_t spread = __byte_perm(two, 0u, 0x4140);  // [b0, 0, b1, 0] -> lanes b0, b1
  return ((spread & 0x007F007Fu) << 4) | ((spread & 0x00800080u) << 8);
}

// 2^(x-7) as a BF16 bit pattern, for an E8M0 byte x <= 134 (exponent field
// x + 120 stays below 255).
__device__ __forceinline__ uint32_t pow2_bf16(uint32_t x) { return (x + 120u) << 7; }

// a / q_scale for a BF16 value `a` (bits), as far as the E4M3 conversion
// that follows can tell: the result converts to the same E4M3 code as the
// exact IEEE binary32 quotient RN(a / q_scale).  Uses the CTA's table
// tab[f] = RN((128+f) / q_scale).  A normal BF16 value is (128+f) * 2^(E-134)
// with f its 7 mantissa bits and E its exponent field, and rounding commutes
// with scaling by a power of two while the result stays a normal float, so
// RN(a / q_scale) = tab[f] * 2^(E-134): one multiply by a power of two.
// Requires 2^-100 <= q_scale <= 2^100, which makes every other case one of
//   |a| < 2^-119 (zero and subnormals included), or a result below 2^-126
//                                                    -> +-0   (E4M3 +-0),
//   infinite a, or a result of 2^128 or more         -> +-inf (E4M3 +-448),
//   NaN a                                            -> NaN.
__device__ __forceinline__ float div_by_table(uint32_t a16, const uint32_t* tab) {
  const uint32_t e = (a16 >> 7) & 0xFFu;
  const float t = __uint_as_float(tab[a16 & 0x7Fu]);
  // 2^(E-134) as a float; only used for E >= 8, where it is a normal float.
  const float scale = __uint_as_float((e - 7u) << 23);
  // The product is exact or overflows to inf (E4M3 448) or underflows below
  // 2^-126 (E4M3 0), matching the exact quotient's code.
  float x = __fmul_rn(t, scale);
  x = e < 8u ? 0.f : x;                             // |a| < 2^-119: quotient < 2^-19
  x = e == 0xFFu ? __uint_as_float(a16 << 16) : x;  // inf / NaN pass through
  return __uint_as_float(__float_as_uint(x) | ((a16 & 0x8000u) << 16));
}

// Plain IEEE division for q_scale outside the table's range (kept out of
// line: it is not on the common path).
static __device__ __noinline__ uint32_t e4m3_pair_divide(uint32_t two_bf16, float qs) {
  return pack_e4m3x2(__fdiv_rn(bf16_hi(two_bf16), qs), __fdiv_rn(bf16_lo(two_bf16), qs));
}

// True when one multiply by rcp = RN(1/q_scale) gives, for every BF16 value
// p, the E4M3 code of the IEEE quotient RN(p / q_scale); one thread checks
// one significand 128 + f, and a CTA takes the AND over f = 0..127.
//
// Why it suffices.  A normal BF16 value is p = (128 + f) * 2^j.  While the
// results stay normal binary32 values, RN(p * rcp) = RN((128+f) * rcp) * 2^j
// = m * 2^j and RN(p / q) = t * 2^j with t = RN((128+f) / q), because
// rounding commutes with scaling by a power of two.  The E4M3 code of x * 2^j
// depends on j only through the regime x * 2^j falls in: at or above 2^-6
// (E4M3 normals and saturation) the code is the same 3-bit rounding of the
// significand for every j, in [2^-10, 2^-6) the rounding step is 2^-9, and
// below 2^-10 everything rounds to zero.  m and t are at most a few binary32
// ulps apart, so comparing the codes of m * 2^k and t * 2^k with k chosen to
// put t into each binade 2^-11 .. 2^-7 and into [1, 2) covers every j.
// Values outside the normal range decide the same code either way (zero,
// BF16 subnormals, infinities: +-0 or +-448) given 2^-100 <= q <= 2^100,
// which the caller checks.  A refusal only costs speed: the CTA then uses
// the division table.
__device__ __forceinline__ bool e4m3_mul_exact_for(int f, float qs, float rcp) {
  const float num = static_cast<float>(128 + f);
  const float t = __fdiv_rn(num, qs);
  const float m = __fmul_rn(num, rcp);
  const int et = static_cast<int>((__float_as_uint(t) >> 23) & 0xFFu) - 127;
  bool ok = true;
#pragma unroll
  for (int i = 0; i < 6; ++i) {
    const int target = i < 5 ? -11 + i : 0;
    const float s = __uint_as_float(static_cast<uint32_t>(target - et + 127) << 23);  // 2^(target - et)
    const uint32_t codes = pack_e4m3x2(__fmul_rn(t, s), __fmul_rn(m, s));
    ok = ok && ((codes & 0xFFu) == (codes >> 8));
  }
  return ok;
}

// How a kernel converts value / q_scale to E4M3 (all three give the code of
// the IEEE binary32 quotient, saturating RNE), chosen once per CTA:
//   kE4m3Divide:   plain IEEE division (q_scale outside [2^-100, 2^100]);
//   kE4m3Table:    the division table (div_by_table), when the check below
//                  refuses the multiply;
//   kE4m3MulExact: one multiply by rcp = RN(1/q_scale), when
//                  e4m3_mul_exact_for held for every significand (almost
//                  every scale: 800 of 800 random ones in [2^-99, 2^99] and
//                  [0.01, 0.1] in a CPU check).
enum E4m3Mode : int { kE4m3Divide = 0, kE4m3Table = 1, kE4m3MulExact = 3 };

// Two BF16 values (packed) -> two E4M3 codes (packed, low value in byte 0).
template <int MODE>
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t two_bf16, const uint32_t* tab, float qs, float rcp) {
  if constexpr (MODE == kE4m3MulExact) {
    return pack_e4m3x2(__fmul_rn(bf16_hi(two_bf16), rcp), __fmul_rn(bf16_lo(two_bf16), rcp));
  } else if constexpr (MODE == kE4m3Table) {
    return pack_e4m3x2(div_by_table(two_bf16 >> 16, tab), div_by_table(two_bf16 & 0xFFFFu, tab));
  } else {
    return e4m3_pair_divide(two_bf16, qs);
  }
}

// Byte offset of 16-byte chunk `chunk` (0..K/8-1) of token row `m` in the
// q_nope tile of 2K-byte rows (a multiple of 128 bytes); XOR of the low
// three chunk bits with m mod 8 makes the eight rows an ldmatrix reads hit
// eight different bank groups.
template <int K>
__device__ __forceinline__ uint32_t q_off(int m, int chunk) {
  return static_cast<uint32_t>(m * (2 * K) + ((chunk ^ (m & 7)) << 4));
}

// Byte offset of 16-byte chunk `chunk` (0 or 1) of row k in a BF16 tile of
// 16 columns (32-byte rows) as the TMA 32-byte swizzle stores it (chunk
// index XOR bit 2 of the row): the eight rows one ldmatrix matrix reads then
// fall into eight different bank groups.  Tile bases are multiples of 256
// bytes (the swizzle repeats every 256).
__device__ __forceinline__ uint32_t sw32(int k, int chunk) {
  return static_cast<uint32_t>(32 * k + 16 * (chunk ^ ((k >> 2) & 1)));
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile of 128-byte
// rows stored with the TMA 128B swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Step 7 of the kernel: D rows g / g+8 of warp w's MMA tile are latent
// columns n_cta+16w+g / +8, its columns 2t, 2t+1 are tokens.  After
// movmatrix.trans a lane holds token 8jt+g and columns 16w+2t, +1 (first
// block) and 16w+8+2t, +1 (second block); stores go straight to
// out[m*row_stride + h*576 + n].  BF16: two 4-byte stores per tile.  E4M3:
// the pairs are 2 bytes each, and 2-byte stores measured far slower than
// 4-byte ones, so neighbouring lanes (t, t^1) trade one pair: the even lane
// then holds columns 2t..2t+3, the odd lane 8+2t-2..8+2t+1, and each makes
// one 4-byte store.
template <int OD, int MTW, int TS, int MODE, int CH>
__device__ __forceinline__ void write_projection(const RunParams& p, const float (&acc)[MTW][4], int wcol, int wtok,
                                                 int lane, int h, int n_cta, int m0, int M, const uint32_t* divtab,
                                                 float qs, float rcp) {
  constexpr int MT = MTW;  // this warp's token tiles: jt = wtok + TS*i, i < MTW
  const int g = lane >> 2;
  const int t = lane & 3;
  // Phase 1: every value this thread writes, into registers; phase 2: the
  // stores.  All table reads precede all stores.
  uint32_t r[MT][2];
#pragma unroll
  for (int jt = 0; jt < MT; ++jt) {
    r[jt][0] = movmatrix_trans(pack_bf16x2(acc[jt][1], acc[jt][0]));
    r[jt][1] = movmatrix_trans(pack_bf16x2(acc[jt][3], acc[jt][2]));
  }
  if constexpr (OD == kOutE4M3) {
#pragma unroll
    for (int jt = 0; jt < MT; ++jt) {
      r[jt][0] = e4m3_pair<MODE>(r[jt][0], divtab, qs, rcp);
      r[jt][1] = e4m3_pair<MODE>(r[jt][1], divtab, qs, rcp);
    }
  }
  uint32_t w4[MT];  // E4M3: this lane's 4 contiguous output bytes of tile jt
  if constexpr (OD == kOutE4M3) {
#pragma unroll
    for (int jt = 0; jt < MT; ++jt) {
      const uint32_t lo = r[jt][0] & 0xFFFFu, hi = r[jt][1] & 0xFFFFu;  // first / second block pair
      const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, (t & 1) ? lo : hi, 1);
      w4[jt] = (t & 1) ? (got | (hi << 16)) : (lo | (got << 16));
    }
  }
#pragma unroll
  for (int jt = 0; jt < MT; ++jt) {
    const int m = 8 * (wtok + TS * jt) + g;  // token of the chunk; beyond the last tile m >= M: no store
    if (m < (CH ? M : p.M)) {
      const size_t off = static_cast<size_t>(CH ? m0 + m : m) * p.out_row_stride + static_cast<size_t>(h) * kOutDim +
                         n_cta + 16 * wcol + 2 * t;
      if constexpr (OD == kOutBF16) {
        uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + off;
        *reinterpret_cast<uint32_t*>(o) = r[jt][0];
        *reinterpret_cast<uint32_t*>(o + 8) = r[jt][1];
      } else {
        uint8_t* o = p.out + off - 2 * (t & 1) + 8 * (t & 1);  // odd t: columns 8+2(t-1)..
        *reinterpret_cast<uint32_t*>(o) = w4[jt];
      }
    }
  }
}

// Step 8: the q_pe append for one pair of values (2 BF16 in, 2 BF16 or
// 2 E4M3 out) at element offset `off` of the output.
template <int OD, int MODE>
__device__ __forceinline__ void write_pe_pair(const RunParams& p, size_t off, uint32_t pe2, const uint32_t* divtab,
                                              float qs, float rcp) {
  if constexpr (OD == kOutBF16) {
    *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + off) = pe2;
  } else {
    *reinterpret_cast<uint16_t*>(p.out + off) = static_cast<uint16_t>(e4m3_pair<MODE>(pe2, divtab, qs, rcp));
  }
}

// ---------------------------------------------------------------------------
// The kernel.  MT = number of 8-token column tiles, ceil(M/8) in 1..4.
// TRIG selects where the CTA lets the next kernel on the stream launch:
//   0 = at entry (deepest overlap; the next kernels' CTAs fill free SM slots),
//   1 = right after the dependency wait (at most two kernels in flight),
//   2 = once its weight tile is in shared memory (MXFP8: dequantised).
// ---------------------------------------------------------------------------

template <int WF, int OD, int MT, int TRIG, int K, int TS = token_groups(MT), int CH = 0>
__global__ void __launch_bounds__(kThreads * TS) mlaqp_fused_query_kernel(const __grid_constant__ RunParams p) {
  static_assert(K % 32 == 0 && K <= 256, "nope dim: multiple of 32, at most one TMA box (256 rows)");
  using L = Smem<K>;
  constexpr int kCta = kThreads * TS;       // threads in the CTA
  constexpr int MTW = (MT + TS - 1) / TS;   // token tiles per warp
  constexpr int KS = K / 16;                // MMA k-steps
  constexpr int KC = K / 8;                 // 16-byte chunks per q_nope row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_a = smem_u32(smem + L::A);
  const uint32_t s_bar = smem_u32(smem + L::Bar);

  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int wcol = warp & (kWarps - 1);  // 16-column MMA tile of this warp
  const int wtok = warp / kWarps;        // token group of this warp
  // CH = 1: this CTA's tokens are [m0, m0 + M) of an (8*MT)-token chunk
  // (the grid has ceil(M / (8*MT)) of them); CH = 0: all tokens, with no
  // offset arithmetic on the path (measured 0.02-0.13 us per layer call
  // slower when unchunked launches carried it).
  const int m0 = CH ? static_cast<int>(blockIdx.z) * 8 * MT : 0;
  const int M = CH ? min(8 * MT, p.M - m0) : p.M;
  const int n_cta = tile * kNTile;
  // (Each use below reads the parameter itself when CH = 0, as before.)
  const uint16_t* const q_nope_c = p.q_nope + m0 * p.q_nope_ts;
  const uint16_t* const q_pe_c = p.q_pe + m0 * p.q_pe_ts;

  // The next kernel on the stream may start its independent prologue.
  if constexpr (TRIG == 0) pdl_launch_dependents();

  // q_scale is, like the weights, a per-tensor constant of the layer: it is
  // read (and its division table built) ahead of the dependency wait.
  float qs = 1.f;
  if constexpr (OD == kOutE4M3) qs = *p.q_scale;

  // 1. Weight (and scale) stream: one elected thread, one barrier phase.
  if (tid == 0) {
    prefetch_tensormap(&p.wmap);
    mbar_init(s_bar, 1);
    fence_barrier_init();
    if constexpr (WF == kWeightBF16) {
      mbar_arrive_expect_tx(s_bar, K * kNTile * 2 + p.extra_tx);
      tma_load_2d(s_a, &p.wmap, n_cta, h * K, s_bar);
    } else {
      mbar_arrive_expect_tx(s_bar, K * kNTile + K * (kLatent / kMxBlock) + p.extra_tx);
      tma_load_2d(smem_u32(smem + L::Raw), &p.wmap, n_cta, h * K, s_bar);
      bulk_load_1d(smem_u32(smem + L::Scale), p.weight_scale + static_cast<size_t>(h) * K * (kLatent / kMxBlock),
                   K * (kLatent / kMxBlock), s_bar);
    }
  }

  // 2. Warm L2 with the head's q rows (L2 is the coherence point, so a line
  //    fetched before the producer writes it is updated by that write; the
  //    values themselves are read only after the dependency wait), one
  //    prefetch per 128-byte line (a bulk prefetch per row measured no
  //    faster up to M = 32 and 0.06-0.35 us slower per layer call in the
  //    chunked forms above).
  if (warp == 0 && lane < M) {
    const uint16_t* qrow = (CH ? q_nope_c : p.q_nope) + lane * p.q_nope_ts + h * p.q_nope_hs;
#pragma unroll
    for (int o = 0; o < K; o += 64) prefetch_l2(qrow + o);
    prefetch_l2((CH ? q_pe_c : p.q_pe) + lane * p.q_pe_ts + h * p.q_pe_hs);
  }
  __syncthreads();  // barrier initialised before anyone waits on it

  // E4M3 output: table of RN((128+f)/q_scale) and the per-significand check
  // of the one-multiply form, one significand per thread (both uniform
  // across the grid: q_scale is one value), published and combined by a CTA
  // barrier.  The 32-token chunked form builds it here, while the weight
  // copy is in flight, and lets the barrier after the MXFP8 dequantisation
  // combine it (MXFP8->E4M3, H = 16, M = 40 / 64 / 96: 2.37 / 2.43 / 2.74
  // against 2.47 / 2.54 / 2.87 us per layer call); the other forms build it
  // after the dequantisation (there the early table measured 0.01-0.04 us
  // slower).
  constexpr bool kEarlyTable = CH && MT == 4;
  uint32_t* divtab = reinterpret_cast<uint32_t*>(smem + L::Div);
  bool table_ok = false, mul_ok = false, mine = false;
  float rcp = 1.f;
  auto build_table = [&]() {
    table_ok = qs >= 0x1p-100f && qs <= 0x1p100f;
    rcp = __frcp_rn(qs);
    mine = table_ok;
    if (table_ok && tid < 128) {
      divtab[tid] = __float_as_uint(__fdiv_rn(static_cast<float>(128 + tid), qs));
      mine = e4m3_mul_exact_for(tid, qs, rcp);
    }
  };
  if constexpr (OD == kOutE4M3 && kEarlyTable) build_table();

  // 3. MXFP8: dequantise into the swizzled BF16 tile before the dependency
  //    wait.  Job (row k, chunk c of 8 columns); 8K jobs, 8K/(128 TS) per thread.
  if constexpr (WF == kWeightMXFP8) {
    const bool ok = mbar_wait_bounded(s_bar, 0, p.wait_limit_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
      pdl_wait();  // exit only after the previous kernel: later waits rely on it
      return;
    }
    const uint8_t* raw = smem + L::Raw;
    const uint8_t* sc = smem + L::Scale;
    const int c = tid & 7;
    const int blk = (n_cta + 8 * c) / kMxBlock;
    // Loads of all jobs first, then the arithmetic, then the stores: the
    // phases keep every job's chain independent of the others' stores.
    constexpr int kJobs = 8 * K / kCta;
    uint2 v[kJobs];
    uint32_t xs[kJobs];
#pragma unroll
    for (int i = 0; i < kJobs; ++i) {
      const int k = (tid >> 3) + (kCta / 8) * i;
      v[i] = *reinterpret_cast<const uint2*>(raw + k * kNTile + 8 * c);
      xs[i] = sc[k * (kLatent / kMxBlock) + blk];
    }
    uint32_t o[kJobs][4];
#pragma unroll
    for (int i = 0; i < kJobs; ++i) {
      // value = code * 2^(x-127) = (code * 2^-120) * 2^(x-7), as two exact
      // power-of-two factors so that each stays inside BF16's range.
      const uint32_t x = xs[i];
      const uint32_t s1 = pow2_bf16(min(x, 134u));
      const uint32_t f1 = s1 | (s1 << 16);
      // 2^(x-134) for x > 134 (1.0 otherwise); NaN for the NaN byte 255.
      const uint32_t s2 = x == 255u ? 0x7FC0u : pow2_bf16(max(x, 134u) - 127u);
      const uint32_t f2 = s2 | (s2 << 16);
      const uint32_t w[2] = {v[i].x, v[i].y};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o[i][q] = mul_bf16x2(mul_bf16x2(e4m3x2_to_bf16x2_scaled(w[q >> 1] >> (16 * (q & 1))), f1), f2);
    }
#pragma unroll
    for (int i = 0; i < kJobs; ++i) {
      const int k = (tid >> 3) + (kCta / 8) * i;
      *reinterpret_cast<uint4*>(smem + L::A + sw128(k, c)) = make_uint4(o[i][0], o[i][1], o[i][2], o[i][3]);
    }
    if constexpr (OD == kOutE4M3 && kEarlyTable) {
      mul_ok = __syncthreads_and(mine);  // also publishes the table
    } else {
      __syncthreads();
    }
    if constexpr (TRIG == 2) pdl_launch_dependents();
  } else if constexpr (TRIG == 2) {
    const bool ok = mbar_wait_bounded(s_bar, 0, p.wait_limit_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
      pdl_wait();  // exit only after the previous kernel: later waits rely on it
      return;
    }
    pdl_launch_dependents();
  }
  if constexpr (OD == kOutE4M3 && !(kEarlyTable && WF == kWeightMXFP8)) {
    if constexpr (!kEarlyTable) build_table();
    mul_ok = __syncthreads_and(mine);  // also publishes the table
  }

  // A fragments (weights, transposed by ldmatrix.trans) for all k-steps:
  // lane L addresses row L&7 of matrix L>>3 -- matrices 0/1 = k 16s..+7,
  // 2/3 = k 16s+8..+15; 0/2 = columns 16w..+7, 1/3 = 16w+8..+15.  BF16
  // weights: loaded here, before the dependency wait (measured 0.01-0.03 us
  // faster per layer call); MXFP8: after it (the dequantised tile is ready
  // either way, and there the later load measured faster).
  const int mi = lane >> 3;
  const int chunk = 2 * wcol + (mi & 1);
  uint32_t a[KS][4];
  if constexpr (WF == kWeightBF16 && TRIG != 2) {
    const bool ok = mbar_wait_bounded(s_bar, 0, p.wait_limit_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
      pdl_wait();  // exit only after the previous kernel: later waits rely on it
      return;
    }
  }
  if constexpr (WF == kWeightBF16) {
#pragma unroll
    for (int s = 0; s < KS; ++s) ldmatrix_x4_trans(a[s], s_a + sw128(16 * s + 8 * (mi >> 1) + (lane & 7), chunk));
  }

  // 4. Wait for the producer of q_nope / q_pe (no-op without PDL).
  pdl_wait();
  if constexpr (TRIG == 1) pdl_launch_dependents();

  // 5. Inputs: this thread's q_pe pair and this head's q_nope rows
  //    [8*MT][128] (16-byte loads, rows >= M zero), issued back to back; then
  //    the weight fragments, which need no input.  q_pe pair j (values 2j,
  //    2j+1 of the head's M x 64 q_pe block) belongs to thread j - kCta*tile.
  const int j_pe = tile * kCta + tid;
  const bool has_pe = j_pe < M * (kRope / 2);
  const int m_pe = j_pe >> 5;
  uint32_t pe = 0u;
  if (has_pe) pe = ld_u32((CH ? q_pe_c : p.q_pe) + m_pe * p.q_pe_ts + h * p.q_pe_hs + 2 * (j_pe & 31));
  constexpr int kQChunks = 8 * MT * KC;  // 16-byte chunks of the [8*MT][K] tile
  constexpr int QI = (kQChunks + kCta - 1) / kCta;
  uint4 qv[QI];
#pragma unroll
  for (int i = 0; i < QI; ++i) {
    const int c = tid + kCta * i;  // chunk c: token row c/KC, k chunk c%KC
    const int m = c / KC;
    qv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (c < kQChunks && m < M)
      qv[i] = ld_u128((CH ? q_nope_c : p.q_nope) + m * p.q_nope_ts + h * p.q_nope_hs + 8 * (c % KC));
  }

  if constexpr (WF == kWeightMXFP8) {
#pragma unroll
    for (int s = 0; s < KS; ++s) ldmatrix_x4_trans(a[s], s_a + sw128(16 * s + 8 * (mi >> 1) + (lane & 7), chunk));
  }

#pragma unroll
  for (int i = 0; i < QI; ++i) {
    const int c = tid + kCta * i;
    if (c < kQChunks) *reinterpret_cast<uint4*>(smem + L::Q + q_off<K>(c / KC, c % KC)) = qv[i];
  }
  __syncthreads();

  // 8. (ahead of the contraction, overlapping its latency) the q_pe append.
  if (has_pe) {
    const size_t off = static_cast<size_t>(CH ? m0 + m_pe : m_pe) * p.out_row_stride +
                       static_cast<size_t>(h) * kOutDim + kLatent + 2 * (j_pe & 31);
    if (OD == kOutBF16 || mul_ok) {
      write_pe_pair<OD, kE4m3MulExact>(p, off, pe, divtab, qs, rcp);
    } else if (table_ok) {
      write_pe_pair<OD, kE4m3Table>(p, off, pe, divtab, qs, rcp);
    } else {
      write_pe_pair<OD, kE4m3Divide>(p, off, pe, divtab, qs, rcp);
    }
  }

  // 6. Contraction, two independent accumulator chains (even / odd k-steps),
  //    over this warp's token tiles jt = wtok + TS*i.  B (q_nope): matrix L>>3
  //    of ldmatrix is k chunk 4*s2 + (L>>3) of tokens 8jt..8jt+7, giving
  //    b0/b1 of steps 2*s2 and 2*s2+1.
  const uint32_t s_q = smem_u32(smem + L::Q);
  bool tile_ok[MTW];
#pragma unroll
  for (int i = 0; i < MTW; ++i) tile_ok[i] = wtok + TS * i < MT;  // uniform per warp
  uint32_t b[KS / 2][MTW][4];
#pragma unroll
  for (int s2 = 0; s2 < KS / 2; ++s2)
#pragma unroll
    for (int i = 0; i < MTW; ++i)
      if (tile_ok[i]) ldmatrix_x4(b[s2][i], s_q + q_off<K>(8 * (wtok + TS * i) + (lane & 7), 4 * s2 + mi));
  float acc[2][MTW][4];
#pragma unroll
  for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
    for (int i = 0; i < MTW; ++i) acc[c2][i][0] = acc[c2][i][1] = acc[c2][i][2] = acc[c2][i][3] = 0.f;
#pragma unroll
  for (int s = 0; s < KS; ++s)
#pragma unroll
    for (int i = 0; i < MTW; ++i)
      if (tile_ok[i]) mma_bf16_16816(acc[s & 1][i], a[s], b[s >> 1][i][2 * (s & 1)], b[s >> 1][i][2 * (s & 1) + 1]);
#pragma unroll
  for (int i = 0; i < MTW; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[0][i][e] += acc[1][i][e];

  // 7. Epilogue; the E4M3 division form is chosen once per CTA so that the
  //    common path holds no call and no branch.
  if constexpr (OD == kOutBF16) {
    write_projection<OD, MTW, TS, kE4m3MulExact, CH>(p, acc[0], wcol, wtok, lane, h, n_cta, m0, M, divtab, qs, rcp);
  } else if (mul_ok) {
    write_projection<OD, MTW, TS, kE4m3MulExact, CH>(p, acc[0], wcol, wtok, lane, h, n_cta, m0, M, divtab, qs, rcp);
  } else if (table_ok) {
    write_projection<OD, MTW, TS, kE4m3Table, CH>(p, acc[0], wcol, wtok, lane, h, n_cta, m0, M, divtab, qs, rcp);
  } else {
    write_projection<OD, MTW, TS, kE4m3Divide, CH>(p, acc[0], wcol, wtok, lane, h, n_cta, m0, M, divtab, qs, rcp);
  }
}

// Host-side read (and optional clear) of this unit's device status word.
inline cudaError_t read_device_status(unsigned int* value, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_device_status, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace mlaqp
