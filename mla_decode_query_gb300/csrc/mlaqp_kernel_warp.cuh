// Fused MLA decode query projection + assembly, warp-tile form (M <= 32).
//
// Computes the same layer call as mlaqp_fused_query_kernel (SparkInfer PR #75
// "Add BF16 MLA query projection and assembly", sections What and Contract;
// vLLM PR #174 "Fuse MXFP8 and BF16 MLA query assembly", section What):
//   out[m,h,0:512]   = bf16(sum_k q_nope[m,h,k] * W_UK_T[h,k,:])  (FP32 sum)
//                      or e4m3_satfinite(that / q_scale)
//   out[m,h,512:576] = q_pe[m,h,:]  (bit copy, or the same E4M3 cast)
//
// Work split.  The unit of work is a warp tile: one head h and 16 latent
// columns [16c, 16c+16), all K and all M tokens; a head has 32 of them.  The
// grid has exactly one CTA per SM (G CTAs), split over the heads as evenly as
// it goes: head h owns CTAs [hG/H, (h+1)G/H), C_h of them (9 or 10 at H = 16,
// 13 or 14 at H = 11, 19 at H = 8 on 152 SMs), and its b-th CTA takes the
// head's tiles [32b/C_h, 32(b+1)/C_h): 3-4 tiles at H = 16, 2-3 at H = 11,
// 1-2 at H = 8.  With at most two CTAs per SM (the launch policy pads shared
// memory), the running layer and the layer launched after it then fill the
// SMs' slots exactly, one CTA of each per SM: no SM carries twice the
// post-wait work of another (a grid that leaves SMs free lets the block
// scheduler put two CTAs of one layer on them).  For M > 8 a second warp per
// tile takes every other 8-token MMA tile (TS = 2 token groups).
//
// Everything that does not depend on the previous kernel happens before the
// dependency wait: the weight tiles (one TMA box of 16 columns x K rows per
// warp tile, on one mbarrier), the MXFP8 dequantisation, the A fragments in
// registers, q_scale and the E4M3 conversion set-up.  After the wait the CTA
// stages its head's q_nope rows in shared memory once (16-byte loads, one
// barrier), appends its share of q_pe, and each warp runs its MMAs (B
// fragments by ldmatrix) and stores.
//
// A CUDA-core form of the same tile (ARM = kArmFma: FP32 FMAs over a K split
// across the lanes, then a shuffle reduction) is instantiated for M <= 8 and
// nope dim 128, so that the tensor-core choice can be measured against it.

#pragma once

#include "mlaqp_kernel.cuh"

namespace mlaqp {

constexpr int kWTileCols = 16;                         // latent columns per warp tile
constexpr int kWTilesPerHead = kLatent / kWTileCols;   // 32
constexpr int kWMaxTilesPerCta = 4;                    // H = 16 on >= 128 SMs

enum Arm : int { kArmMma = 0, kArmFma = 1 };

// Token groups of a warp-tile kernel: two for M > 8 (each warp then runs at
// most two of the four 8-token MMA tiles).
constexpr int wtoken_groups(int mt) { return mt >= 2 ? 2 : 1; }

struct WarpRunParams {
  CUtensorMap wmap;             // W_UK_T as [H*K rows][512 cols], box 16 cols x K rows
  const uint16_t* q_nope;       // BF16, element (m,h,k) at m*q_nope_ts + h*q_nope_hs + k
  const uint16_t* q_pe;         // BF16, element (m,h,j) at m*q_pe_ts + h*q_pe_hs + j
  int64_t q_nope_ts, q_nope_hs; // token / head strides (elements)
  int64_t q_pe_ts, q_pe_hs;
  const uint8_t* weight_scale;  // E8M0 [H,K,16] or null
  uint8_t* out;                 // element (m,h,j) at m*out_row_stride + h*576 + j
  int64_t out_row_stride;       // elements
  const float* q_scale;         // device scalar or null
  unsigned long long wait_limit_ns;  // bound on every mbarrier wait
  unsigned int extra_tx;        // test hook: bytes a barrier expects beyond its copy
  int M;
  int H;
  float inv_ctas;               // RN(1 / gridDim.x)
  float inv_heads;              // RN(1 / H)
};

// Dynamic shared memory of one CTA (offsets from a 1024-byte aligned base).
template <int K>
struct WSmem {
  static constexpr int kTileA = K * kWTileCols * 2;        // BF16 [K][16], 32-byte rows, 32B swizzle
  static constexpr int kTileRaw = K * kWTileCols;          // E4M3 [K][16], 16-byte rows
  static constexpr int A = 0;
  static constexpr int Raw = A + kWMaxTilesPerCta * kTileA;
  static constexpr int Q = Raw + kWMaxTilesPerCta * kTileRaw;    // BF16 [32][K], 16-byte chunks XOR-swizzled
  static constexpr int Div = Q + kMaxM * K * 2;                  // FP32 [128]: RN((128+f)/q_scale)
  static constexpr int Bar = Div + 128 * 4;                      // the weight barrier
  static constexpr int Bytes = Bar + 8 + 1024;                   // + slack for the alignment
};

// floor(a / d) for small non-negative integers without an integer division:
// `inv` = 1/d (within a few float ulps; the caller passes the host's RN(1/d)
// or a hardware reciprocal).  If a/d is not an integer it lies at least 1/d
// below the next integer, so for a, d < 2^11 the float error (about 2^-22
// relative) cannot cross it; if it is an integer the product may fall just
// short of it, which the 2^-12 bias (< 1/d) covers.
__device__ __forceinline__ int floor_div(int a, float inv) {
  return static_cast<int>(__fmaf_rn(static_cast<float>(a), inv, 0x1p-12f));
}


// Epilogue of the tensor-core arm for one warp: D rows g / g+8 of MMA tile i
// are latent columns n0+g / n0+g+8, its columns 2t, 2t+1 are tokens.  After
// movmatrix.trans a lane holds token 8*jt+g and columns n0+2t, +1 (first
// block) and n0+8+2t, +1 (second block).  BF16: two 4-byte stores per tile.
// E4M3: neighbouring lanes trade one value pair so that each lane makes one
// 4-byte store (the even lane columns 2t..2t+3, the odd lane 8+2t-2..8+2t+1).
template <int OD, int MTW, int TS, int MODE>
__device__ __forceinline__ void write_tile(const WarpRunParams& p, const float (&acc)[MTW][4], int grp, int lane,
                                           int h, int n0, const uint32_t* divtab, float qs, float rcp) {
  const int g = lane >> 2;
  const int t = lane & 3;
  uint32_t r[MTW][2];
#pragma unroll
  for (int i = 0; i < MTW; ++i) {
    r[i][0] = movmatrix_trans(pack_bf16x2(acc[i][1], acc[i][0]));
    r[i][1] = movmatrix_trans(pack_bf16x2(acc[i][3], acc[i][2]));
  }
  uint32_t w4[MTW];
  if constexpr (OD == kOutE4M3) {
#pragma unroll
    for (int i = 0; i < MTW; ++i) {
      const uint32_t lo = e4m3_pair<MODE>(r[i][0], divtab, qs, rcp) & 0xFFFFu;
      const uint32_t hi = e4m3_pair<MODE>(r[i][1], divtab, qs, rcp) & 0xFFFFu;
      const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, (t & 1) ? lo : hi, 1);
      w4[i] = (t & 1) ? (got | (hi << 16)) : (lo | (got << 16));
    }
  }
#pragma unroll
  for (int i = 0; i < MTW; ++i) {
    const int m = 8 * (grp + TS * i) + g;
    if (m < p.M) {
      const size_t off = static_cast<size_t>(m) * p.out_row_stride + static_cast<size_t>(h) * kOutDim + n0 + 2 * t;
      if constexpr (OD == kOutBF16) {
        uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + off;
        *reinterpret_cast<uint32_t*>(o) = r[i][0];
        *reinterpret_cast<uint32_t*>(o + 8) = r[i][1];
      } else {
        *reinterpret_cast<uint32_t*>(p.out + off + 6 * (t & 1)) = w4[i];
      }
    }
  }
}

// Epilogue of the CUDA-core arm: lane l holds column n0 + (l >> 1) (lanes 2j
// and 2j+1 hold the same sum).  BF16: lane 4j stores columns 2j, 2j+1 as one
// 4-byte store.  E4M3: lane 8j stores columns 4j..4j+3 as one 4-byte store.
template <int OD, int MODE>
__device__ __forceinline__ void write_fma_token(const WarpRunParams& p, float v, int m, int lane, int h, int n0,
                                                const uint32_t* divtab, float qs, float rcp) {
  const float v1 = __shfl_down_sync(0xFFFFFFFFu, v, 2);  // column +1
  const uint32_t pair = pack_bf16x2(v1, v);
  if constexpr (OD == kOutBF16) {
    if ((lane & 3) == 0 && m < p.M) {
      const size_t off = static_cast<size_t>(m) * p.out_row_stride + static_cast<size_t>(h) * kOutDim + n0 + (lane >> 1);
      *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + off) = pair;
    }
  } else {
    const uint32_t codes = e4m3_pair<MODE>(pair, divtab, qs, rcp) & 0xFFFFu;  // columns c, c+1
    const uint32_t next = __shfl_down_sync(0xFFFFFFFFu, codes, 4);             // columns c+2, c+3
    if ((lane & 7) == 0 && m < p.M) {
      const size_t off = static_cast<size_t>(m) * p.out_row_stride + static_cast<size_t>(h) * kOutDim + n0 + (lane >> 1);
      *reinterpret_cast<uint32_t*>(p.out + off) = codes | (next << 16);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.  Grid G (>= H).  MT = ceil(M/8) in 1..4, TRIG 0 = trigger the
// next kernel's launch at entry, 1 = right after the dependency wait.  ARM =
// kArmFma only with MT = 1 and K = 128.  blockDim.x = 32 * TS * (tiles per
// CTA, rounded up); warp w serves tile slot w / TS, token group w % TS.
// ---------------------------------------------------------------------------

template <int WF, int OD, int MT, int TRIG, int K, int ARM, int TS = wtoken_groups(MT)>
__global__ void __launch_bounds__(32 * TS * kWMaxTilesPerCta, 2) mlaqp_query_warp_kernel(
    const __grid_constant__ WarpRunParams p) {
  static_assert(K % 32 == 0 && K <= 256, "nope dim: multiple of 32, at most one TMA box (256 rows)");
  static_assert(ARM == kArmMma || (MT == 1 && K == 128 && TS == 1), "the FMA arm covers M <= 8 at nope 128");
  using L = WSmem<K>;
  constexpr int KS = K / 16;               // MMA k-steps
  constexpr int KC = K / 8;                // 16-byte chunks per q_nope row
  constexpr int MTW = (MT + TS - 1) / TS;  // MMA token tiles per warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int slot = warp / TS;
  const int grp = warp % TS;
  // CTA -> (head, tiles), without integer division (it measurably slowed
  // the layer that runs on the same SMs while this prologue executes).
  const int G = gridDim.x;
  const int h = floor_div((blockIdx.x + 1) * p.H - 1, p.inv_ctas);  // largest h with hG/H <= blockIdx.x
  const int cta0 = floor_div(h * G, p.inv_heads);                    // first CTA of head h
  const int C = floor_div((h + 1) * G, p.inv_heads) - cta0;          // CTAs of head h
  const float inv_c = __frcp_rn(static_cast<float>(C));
  const int b = blockIdx.x - cta0;
  const int c_begin = floor_div(b * kWTilesPerHead, inv_c);
  const int ntiles = floor_div((b + 1) * kWTilesPerHead, inv_c) - c_begin;
  const bool active = slot < ntiles;
  const int n0 = (c_begin + (active ? slot : 0)) * kWTileCols;
  const int M = p.M;
  const uint32_t s_bar = smem_u32(smem + L::Bar);
  const uint32_t s_tile = smem_u32(smem + L::A) + static_cast<uint32_t>(slot * L::kTileA);

  if constexpr (TRIG == 0) pdl_launch_dependents();

  float qs = 1.f;
  if constexpr (OD == kOutE4M3) qs = *p.q_scale;

  // 1. Weight tiles: one elected thread, one TMA box per tile, one barrier.
  if (tid == 0) {
    prefetch_tensormap(&p.wmap);
    mbar_init(s_bar, 1);
    fence_barrier_init();
    const int tile_bytes = WF == kWeightBF16 ? L::kTileA : L::kTileRaw;
    mbar_arrive_expect_tx(s_bar, ntiles * tile_bytes + p.extra_tx);
    for (int i = 0; i < ntiles; ++i) {
      const int x = (c_begin + i) * kWTileCols, y = h * K;
      if constexpr (WF == kWeightBF16) {
        tma_load_2d(smem_u32(smem + L::A) + i * L::kTileA, &p.wmap, x, y, s_bar);
      } else {
        tma_load_2d(smem_u32(smem + L::Raw) + i * L::kTileRaw, &p.wmap, x, y, s_bar);
      }
    }
  }

  // 2. Warm L2 with the head's q rows (L2 is the coherence point, so a line
  //    fetched before the producer writes it is updated by that write; the
  //    values are read only after the dependency wait), one prefetch per
  //    128-byte line.  (One bulk TMA-unit prefetch per q_nope row measured
  //    0.06-0.07 us per layer call faster at H = 16, M = 32 in a chain of
  //    this op, but 0.4-0.7 us slower behind a producer that has just
  //    written q.)  MXFP8: this lane's scale bytes (rows k = lane + 32i; the
  //    tile's 16 columns share one 32-column scale block).
  if (warp == 0 && lane < M) {
    const uint16_t* qrow = p.q_nope + lane * p.q_nope_ts + h * p.q_nope_hs;
#pragma unroll
    for (int o = 0; o < K; o += 64) prefetch_l2(qrow + o);
    prefetch_l2(p.q_pe + lane * p.q_pe_ts + h * p.q_pe_hs);
  }
  uint32_t sc[K / 32];
  if constexpr (WF == kWeightMXFP8) {
    if (active) {
      const uint8_t* srow = p.weight_scale + static_cast<size_t>(h) * K * (kLatent / kMxBlock) + n0 / kMxBlock;
#pragma unroll
      for (int i = 0; i < K / 32; ++i) sc[i] = srow[(lane + 32 * i) * (kLatent / kMxBlock)];
    }
  }
  __syncthreads();  // barrier initialised before anyone waits on it

  // 3. E4M3 output: the division table (one entry per thread and pass) and
  //    the per-significand check of the one-multiply form.
  uint32_t* divtab = reinterpret_cast<uint32_t*>(smem + L::Div);
  bool table_ok = false, mul_ok = false;
  float rcp = 1.f;
  if constexpr (OD == kOutE4M3) {
    table_ok = qs >= 0x1p-100f && qs <= 0x1p100f;  // uniform across the grid
    rcp = __frcp_rn(qs);
    bool mine = table_ok;
    if (table_ok)
      for (int f = tid; f < 128; f += nthreads) {
        divtab[f] = __float_as_uint(__fdiv_rn(static_cast<float>(128 + f), qs));
        mine = mine && e4m3_mul_exact_for(f, qs, rcp);
      }
    mul_ok = __syncthreads_and(mine);  // also publishes the table
  }

  // 4. The weight tiles: wait (bounded), MXFP8 dequantisation into the BF16
  //    tiles, then the A fragments (tensor-core arm) or the FP32 weights
  //    (CUDA-core arm) into registers.
  //    One thread polls the barrier; the others wait at the CTA barrier,
  //    which issues nothing (this prologue shares the SM with the post-wait
  //    path of the layer before), then observe the completed phase once.
  bool ok = true;
  if (tid == 0) ok = mbar_wait_bounded(s_bar, 0, p.wait_limit_ns);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
    pdl_wait();  // exit only after the previous kernel: later waits rely on it
    return;
  }
  if (tid != 0) ok = mbar_try_wait(s_bar, 0);  // completed: makes the tile's bytes visible to this thread
  if constexpr (WF == kWeightMXFP8) {
    if (active && grp == 0) {
      // Row k = lane + 32i: 16 E4M3 codes -> 16 BF16 values (exact, as two
      // power-of-two factors so that each stays inside BF16's range).
      const uint8_t* raw = smem + L::Raw + slot * L::kTileRaw;
      uint8_t* dst = smem + L::A + slot * L::kTileA;
#pragma unroll
      for (int i = 0; i < K / 32; ++i) {
        const int k = lane + 32 * i;
        const uint4 v = *reinterpret_cast<const uint4*>(raw + 16 * k);
        const uint32_t x = sc[i];
        const uint32_t s1 = pow2_bf16(min(x, 134u));
        const uint32_t f1 = s1 | (s1 << 16);
        const uint32_t s2 = x == 255u ? 0x7FC0u : pow2_bf16(max(x, 134u) - 127u);
        const uint32_t f2 = s2 | (s2 << 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          o[q] = mul_bf16x2(mul_bf16x2(e4m3x2_to_bf16x2_scaled(w[q >> 1] >> (16 * (q & 1))), f1), f2);
        *reinterpret_cast<uint4*>(dst + sw32(k, 0)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(dst + sw32(k, 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    __syncthreads();  // the token-group-1 warp of a tile reads what group 0 wrote
  }

  uint32_t a[ARM == kArmMma ? KS : 1][4];
  float wf[ARM == kArmFma ? 4 : 1][16];
  if (active) {
    if constexpr (ARM == kArmMma) {
      // ldmatrix.x4.trans: matrix mi = lane >> 3 holds k rows
      // 16s + 8*(mi>>1) .. +7 of the stored [K][16] tile and columns
      // 8*(mi&1) .. +7; lane L supplies the address of its matrix's row L & 7.
      const int mi = lane >> 3;
#pragma unroll
      for (int s = 0; s < KS; ++s)
        ldmatrix_x4_trans(a[s], s_tile + sw32(16 * s + 8 * (mi >> 1) + (lane & 7), mi & 1));
    } else {
      // Lane l owns k = 4l .. 4l+3 and all 16 columns.
      const uint8_t* tw = smem + L::A + slot * L::kTileA;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint4 lo = *reinterpret_cast<const uint4*>(tw + sw32(4 * lane + kk, 0));
        const uint4 hi = *reinterpret_cast<const uint4*>(tw + sw32(4 * lane + kk, 1));
        const uint32_t w8[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          wf[kk][2 * j] = bf16_lo(w8[j]);
          wf[kk][2 * j + 1] = bf16_hi(w8[j]);
        }
      }
    }
  }

  // 5. Wait for the producer of q_nope / q_pe (no-op without PDL).
  pdl_wait();
  if constexpr (TRIG == 1) pdl_launch_dependents();

  // 6. q_pe: the head's M x 32 value pairs, pair j handled by thread
  //    j - nthreads*b of the head's CTA b (coalesced rows).
  const int j_pe = b * nthreads + tid;
  const bool has_pe = j_pe < M * (kRope / 2);
  const int m_pe = j_pe >> 5;
  uint32_t pe = 0u;
  if (has_pe) pe = ld_u32(p.q_pe + m_pe * p.q_pe_ts + h * p.q_pe_hs + 2 * (j_pe & 31));
  const uint16_t* qh = p.q_nope + h * p.q_nope_hs;

  if constexpr (ARM == kArmMma) {
    // 7. The head's q_nope rows [8*MT][K] into the swizzled tile (rows >= M
    //    zero), up to four 16-byte loads per thread in flight at once (one
    //    pass covers every chunk unless the CTA has fewer than 8*MT*K/32
    //    threads); one barrier.
    constexpr int kQChunks = 8 * MT * KC;
    constexpr int QB = 4;
    for (int base = 0; base < kQChunks; base += QB * nthreads) {
      uint4 qv[QB];
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        const int c = base + tid + nthreads * i;
        const int m = c / KC;
        qv[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c < kQChunks && m < M) qv[i] = ld_u128(qh + m * p.q_nope_ts + 8 * (c % KC));
      }
#pragma unroll
      for (int i = 0; i < QB; ++i) {
        const int c = base + tid + nthreads * i;
        if (c < kQChunks) *reinterpret_cast<uint4*>(smem + L::Q + q_off<K>(c / KC, c % KC)) = qv[i];
      }
    }
    __syncthreads();

    // 8. The q_pe append, overlapping the MMA latency.
    if (has_pe) {
      const size_t off = static_cast<size_t>(m_pe) * p.out_row_stride + static_cast<size_t>(h) * kOutDim + kLatent +
                         2 * (j_pe & 31);
      if constexpr (OD == kOutBF16) {
        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + off) = pe;
      } else if (mul_ok) {
        *reinterpret_cast<uint16_t*>(p.out + off) = static_cast<uint16_t>(e4m3_pair<kE4m3MulExact>(pe, divtab, qs, rcp));
      } else if (table_ok) {
        *reinterpret_cast<uint16_t*>(p.out + off) = static_cast<uint16_t>(e4m3_pair<kE4m3Table>(pe, divtab, qs, rcp));
      } else {
        *reinterpret_cast<uint16_t*>(p.out + off) = static_cast<uint16_t>(e4m3_pair<kE4m3Divide>(pe, divtab, qs, rcp));
      }
    }
    if (!active) return;

    // 9. Contraction: B fragments by ldmatrix (matrix L>>3 = k chunk
    //    4*s2 + (L>>3) of tokens 8jt..8jt+7, giving b0/b1 of steps 2*s2 and
    //    2*s2+1), two accumulator chains per token tile (even / odd k-steps).
    const uint32_t s_q = smem_u32(smem + L::Q);
    const int mi = lane >> 3;
    bool tile_live[MTW];
#pragma unroll
    for (int i = 0; i < MTW; ++i) tile_live[i] = (grp + TS * i) < MT;  // uniform per warp
    uint32_t b[KS / 2][MTW][4];
#pragma unroll
    for (int s2 = 0; s2 < KS / 2; ++s2)
#pragma unroll
      for (int i = 0; i < MTW; ++i)
        if (tile_live[i]) ldmatrix_x4(b[s2][i], s_q + q_off<K>(8 * (grp + TS * i) + (lane & 7), 4 * s2 + mi));
    float acc[2][MTW][4];
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
      for (int i = 0; i < MTW; ++i) acc[c2][i][0] = acc[c2][i][1] = acc[c2][i][2] = acc[c2][i][3] = 0.f;
#pragma unroll
    for (int s = 0; s < KS; ++s)
#pragma unroll
      for (int i = 0; i < MTW; ++i)
        if (tile_live[i]) mma_bf16_16816(acc[s & 1][i], a[s], b[s >> 1][i][2 * (s & 1)], b[s >> 1][i][2 * (s & 1) + 1]);
#pragma unroll
    for (int i = 0; i < MTW; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[0][i][e] += acc[1][i][e];

    // 10. Epilogue (the E4M3 form is uniform across the grid).
    if constexpr (OD == kOutBF16) {
      write_tile<OD, MTW, TS, kE4m3Table>(p, acc[0], grp, lane, h, n0, divtab, qs, rcp);
    } else if (mul_ok) {
      write_tile<OD, MTW, TS, kE4m3MulExact>(p, acc[0], grp, lane, h, n0, divtab, qs, rcp);
    } else if (table_ok) {
      write_tile<OD, MTW, TS, kE4m3Table>(p, acc[0], grp, lane, h, n0, divtab, qs, rcp);
    } else {
      write_tile<OD, MTW, TS, kE4m3Divide>(p, acc[0], grp, lane, h, n0, divtab, qs, rcp);
    }
  } else {
    // CUDA-core arm: q[m][4l .. 4l+3] for every token straight into
    // registers, then per token 64 FMAs and a reduce-scatter over the lanes
    // (xor 16, 8, 4, 2 halve the columns each lane keeps; xor 1 completes
    // the sum), leaving column n0 + (lane >> 1) in lane `lane`.
    uint2 qv[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      qv[m] = make_uint2(0u, 0u);
      if (active && m < M) {
        const uint16_t* src = qh + m * p.q_nope_ts + 4 * lane;
        asm volatile("ld.global.v2.b32 {%0,%1}, [%2];" : "=r"(qv[m].x), "=r"(qv[m].y) : "l"(src));
      }
    }
    if (has_pe) {
      const size_t off = static_cast<size_t>(m_pe) * p.out_row_stride + static_cast<size_t>(h) * kOutDim + kLatent +
                         2 * (j_pe & 31);
      if constexpr (OD == kOutBF16) {
        *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + off) = pe;
      } else if (mul_ok) {
        *reinterpret_cast<uint16_t*>(p.out + off) = static_cast<uint16_t>(e4m3_pair<kE4m3MulExact>(pe, divtab, qs, rcp));
      } else if (table_ok) {
        *reinterpret_cast<uint16_t*>(p.out + off) = static_cast<uint16_t>(e4m3_pair<kE4m3Table>(pe, divtab, qs, rcp));
      } else {
        *reinterpret_cast<uint16_t*>(p.out + off) = static_cast<uint16_t>(e4m3_pair<kE4m3Divide>(pe, divtab, qs, rcp));
      }
    }
    if (!active) return;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (m >= M) break;  // uniform
      const float q0 = bf16_lo(qv[m].x), q1 = bf16_hi(qv[m].x), q2 = bf16_lo(qv[m].y), q3 = bf16_hi(qv[m].y);
      float v[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = fmaf(q3, wf[3][c], fmaf(q2, wf[2][c], fmaf(q1, wf[1][c], q0 * wf[0][c])));
      // reduce-scatter: after the step with offset 2^b (b = 4..1) a lane keeps
      // the half of its columns selected by bit b of its lane index.
#pragma unroll
      for (int b = 4, w = 8; b >= 1; --b, w >>= 1) {
        const bool upper = (lane >> b) & 1;
#pragma unroll
        for (int j = 0; j < w; ++j) {
          const float keep = upper ? v[w + j] : v[j];
          const float give = upper ? v[j] : v[w + j];
          v[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 1 << b);
        }
      }
      const float sum = v[0] + __shfl_xor_sync(0xFFFFFFFFu, v[0], 1);
      if constexpr (OD == kOutBF16) {
        write_fma_token<OD, kE4m3Table>(p, sum, m, lane, h, n0, divtab, qs, rcp);
      } else if (mul_ok) {
        write_fma_token<OD, kE4m3MulExact>(p, sum, m, lane, h, n0, divtab, qs, rcp);
      } else if (table_ok) {
        write_fma_token<OD, kE4m3Table>(p, sum, m, lane, h, n0, divtab, qs, rcp);
      } else {
        write_fma_token<OD, kE4m3Divide>(p, sum, m, lane, h, n0, divtab, qs, rcp);
      }
    }
  }
}

}  // namespace mlaqp
