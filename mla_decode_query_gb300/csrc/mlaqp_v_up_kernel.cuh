// V up-projection after attention over the latent cache, for GB300 (sm_103a):
//
//   out[m,h,d] = bf16_rne( sum_{c<512} x[m,h,c] * W_UV[h,c,d] )    d < 128, FP32 accumulation
//
// x is the attention output in the latent space (BF16), W_UV is BF16 or MXFP8
// (E4M3 + one E8M0 scale per 32 consecutive output elements of each (h,c)
// row), stored with the output axis fastest.  The pages name this step only
// as the downstream V up-projection (vLLM PR #174 "Fuse MXFP8 and BF16 MLA
// query assembly", section Safety scope); its weight formats follow the
// query side (section What).
//
// Used for M <= 64 (above that, mlaqp_v_up_kernel_large.cuh).  Work split:
// CTA (tile, h, z) owns head h, output columns [16*tile, 16*tile+16) and
// tokens [32z, 32z+32): 8 CTAs per head and 32-token chunk, each streaming a
// 512 x 16 weight tile (16 KB BF16; the second chunk finds it in L2).  Eight warps split the 512-long contraction, 64 each
// (four mma.sync m16n8k16 k-steps; swap-AB: the 16 output columns on the
// MMA's M side, tokens on its N side); the eight partial sums are added in
// shared memory, rounded to BF16 and stored as 4-byte column pairs.
//
// Steps of a CTA (the numbering of the query kernel where it matches):
//  1. thread 0: two 2-D TMA boxes of 16 columns x 256 rows (+ the head's
//     2 KB of E8M0 scales for MXFP8); x rows prefetched into L2;
//  3. MXFP8: dequantise into the BF16 tile before the dependency wait;
//  4. griddepcontrol.wait (everything above touches per-layer constants);
//  5. the head's x rows into a swizzled smem tile; weight fragments with
//     ldmatrix.trans;
//  6. MMAs over this warp's 64 contraction columns;
//  7. cross-warp sum, BF16 rounding, 4-byte stores of column pairs.
// Every mbarrier wait is bounded as in the query kernel.

#pragma once

#include "mlaqp_kernel.cuh"

namespace mlaqp {

constexpr int kVDim = 128;                            // v head dim (output columns)
constexpr int kVNTile = 16;                           // output columns per CTA
constexpr int kVTilesPerHead = kVDim / kVNTile;       // 8
constexpr int kVWarps = 8;
constexpr int kVThreads = 32 * kVWarps;               // 256
constexpr int kVKWarp = kLatent / kVWarps;            // 64 contraction columns per warp
constexpr int kVScaleRow = kVDim / kMxBlock;          // 4 E8M0 bytes per (h, c)
constexpr int kVChunk = 32;                           // tokens per CTA (two grid.z chunks for 32 < M <= 64)
// Row of the cross-warp partial-sum buffer: one warp's 32 values of one
// (token tile, D element), padded by 4 floats so that the two 16-lane halves
// of a summing warp (consecutive D elements) read disjoint banks.
constexpr int kVRedRow = 36;

struct VUpParams {
  CUtensorMap wmap;             // W_UV viewed as [H*512 rows][128 cols]; box 16 x 256 (64 x 128 for the cluster kernel)
  CUtensorMap xmap;             // multicast kernel only: x as [M][H][512], box 64 x 1 x 8*MT, 128B swizzle
  const uint16_t* x;            // BF16, element (m,h,c) at m*x_ts + h*x_hs + c
  int64_t x_ts, x_hs;           // token / head strides (elements)
  const uint8_t* weight_scale;  // E8M0 [H,512,4] or null
  uint16_t* out;                // BF16, element (m,h,d) at m*out_row_stride + h*128 + d
  int64_t out_row_stride;       // elements
  unsigned long long wait_limit_ns;
  unsigned int extra_tx;        // test hook, as in RunParams
  int M;
  int H;
};

// Shared memory layout for MT 8-token tiles (offsets from a 1024-byte aligned
// base).  The cross-warp partial sums reuse the E4M3 staging area, which is
// dead once the tile is dequantised (before the dependency wait).
template <int MT>
struct VSmem {
  static constexpr int W = 0;                              // BF16 [512][16], 32-byte rows, 32B swizzle
  static constexpr int Raw = W + kLatent * kVNTile * 2;    // E4M3 [512][16]; later FP32 partials
  static constexpr int RedBytes = kVWarps * MT * 4 * kVRedRow * 4;
  static constexpr int RawBytes = kLatent * kVNTile;
  static constexpr int Scale = Raw + (RedBytes > RawBytes ? RedBytes : RawBytes);  // E8M0 [512][4]
  static constexpr int X = Scale + kLatent * kVScaleRow;   // BF16 [8*MT][512], chunks XOR-swizzled
  static constexpr int Bar = X + 8 * MT * kLatent * 2;
  static constexpr int Bytes = Bar + 64 + 1024;
};

template <int WF, int MT, int TRIG>
__global__ void __launch_bounds__(kVThreads) mlaqp_v_up_kernel(const __grid_constant__ VUpParams p) {
  using L = VSmem<MT>;
  constexpr int KC = kLatent / 8;            // 16-byte chunks per x row (64)
  constexpr int kXChunks = 8 * MT * KC;      // chunks of the [8*MT][512] tile
  constexpr int XI = kXChunks / kVThreads;   // per thread (2*MT)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_w = smem_u32(smem + L::W);
  const uint32_t s_bar = smem_u32(smem + L::Bar);

  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int m0 = blockIdx.z * 8 * MT;    // this CTA's tokens: [m0, m0 + M) of an (8*MT)-token chunk
  const int M = min(8 * MT, p.M - m0);    // >= 1: the grid has ceil(M/(8*MT)) chunks
  const int d_cta = tile * kVNTile;
  const uint16_t* xh = p.x + m0 * p.x_ts + h * p.x_hs;
  uint16_t* const outc = p.out + m0 * p.out_row_stride;

  if constexpr (TRIG == 0) pdl_launch_dependents();

  // 1. Weight (and scale) stream: two boxes of 256 rows, one barrier phase.
  if (tid == 0) {
    prefetch_tensormap(&p.wmap);
    mbar_init(s_bar, 1);
    fence_barrier_init();
    if constexpr (WF == kWeightBF16) {
      mbar_arrive_expect_tx(s_bar, kLatent * kVNTile * 2 + p.extra_tx);
      tma_load_2d(s_w, &p.wmap, d_cta, h * kLatent, s_bar);
      tma_load_2d(s_w + 256 * kVNTile * 2, &p.wmap, d_cta, h * kLatent + 256, s_bar);
    } else {
      const uint32_t s_raw = smem_u32(smem + L::Raw);
      mbar_arrive_expect_tx(s_bar, kLatent * kVNTile + kLatent * kVScaleRow + p.extra_tx);
      tma_load_2d(s_raw, &p.wmap, d_cta, h * kLatent, s_bar);
      tma_load_2d(s_raw + 256 * kVNTile, &p.wmap, d_cta, h * kLatent + 256, s_bar);
      bulk_load_1d(smem_u32(smem + L::Scale), p.weight_scale + static_cast<size_t>(h) * kLatent * kVScaleRow,
                   kLatent * kVScaleRow, s_bar);
    }
  }
  // 2. Warm L2 with the head's x rows (eight 128-byte lines per row).
  if (tid < 8 * M) prefetch_l2(xh + (tid >> 3) * p.x_ts + 64 * (tid & 7));
  __syncthreads();  // barrier initialised before anyone waits on it

  // 3. MXFP8: dequantise into the BF16 tile (value = code * 2^(x-127) as
  //    two exact power-of-two factors).  Job (row r, half c): 1024 jobs.
  if constexpr (WF == kWeightMXFP8) {
    const bool ok = mbar_wait_bounded(s_bar, 0, p.wait_limit_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
      pdl_wait();  // exit only after the previous kernel: later waits rely on it
      return;
    }
    const uint8_t* raw = smem + L::Raw;
    const uint8_t* sc = smem + L::Scale;
    constexpr int kJobs = kLatent * 2 / kVThreads;  // 4
    uint2 v[kJobs];
    uint32_t xs[kJobs];
#pragma unroll
    for (int i = 0; i < kJobs; ++i) {
      const int j = tid + kVThreads * i;
      const int r = j >> 1;
      v[i] = *reinterpret_cast<const uint2*>(raw + r * kVNTile + 8 * (j & 1));
      xs[i] = sc[r * kVScaleRow + d_cta / kMxBlock];
    }
#pragma unroll
    for (int i = 0; i < kJobs; ++i) {
      const int j = tid + kVThreads * i;
      const uint32_t x = xs[i];
      const uint32_t s1 = pow2_bf16(min(x, 134u));
      const uint32_t f1 = s1 | (s1 << 16);
      const uint32_t s2 = x == 255u ? 0x7FC0u : pow2_bf16(max(x, 134u) - 127u);
      const uint32_t f2 = s2 | (s2 << 16);
      const uint32_t w[2] = {v[i].x, v[i].y};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o[q] = mul_bf16x2(mul_bf16x2(e4m3x2_to_bf16x2_scaled(w[q >> 1] >> (16 * (q & 1))), f1), f2);
      *reinterpret_cast<uint4*>(smem + L::W + sw32(j >> 1, j & 1)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();
  }

  // BF16 weights: their wait and the A fragments ahead of the dependency
  // wait (measured 0.005-0.03 us per layer call faster; for MXFP8 the same
  // order measured 0.05-0.09 us slower, so its fragments load after it).
  const int mi = lane >> 3;
  uint32_t a[4][4];
  if constexpr (WF == kWeightBF16) {
    const bool ok = mbar_wait_bounded(s_bar, 0, p.wait_limit_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
      pdl_wait();  // exit only after the previous kernel: later waits rely on it
      return;
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int row = 16 * (4 * warp + s) + 8 * (mi >> 1) + (lane & 7);
      ldmatrix_x4_trans(a[s], s_w + sw32(row, mi & 1));
    }
  }

  // 4. Wait for the producer of x (no-op without PDL).
  pdl_wait();
  if constexpr (TRIG == 1) pdl_launch_dependents();

  // 5. The head's x rows [8*MT][512] (16-byte loads, rows >= M zero).
  uint4 xv[XI];
#pragma unroll
  for (int i = 0; i < XI; ++i) {
    const int c = tid + kVThreads * i;
    const int m = c / KC;
    xv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (m < M) xv[i] = ld_u128(xh + m * p.x_ts + 8 * (c % KC));
  }
  // A fragments for the warp's four k-steps s = 4w..4w+3: matrices 0/1 =
  // rows 16s..+7 (columns 0-7 / 8-15), 2/3 = rows 16s+8..+15.  MXFP8: here,
  // after the dependency wait; BF16: before it (see there).
  if constexpr (WF == kWeightMXFP8) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int row = 16 * (4 * warp + s) + 8 * (mi >> 1) + (lane & 7);
      ldmatrix_x4_trans(a[s], s_w + sw32(row, mi & 1));
    }
  }
#pragma unroll
  for (int i = 0; i < XI; ++i) {
    const int c = tid + kVThreads * i;
    *reinterpret_cast<uint4*>(smem + L::X + q_off<kLatent>(c / KC, c % KC)) = xv[i];
  }
  __syncthreads();

  // 6. B fragments (x rows = tokens, 16-byte chunks = contraction) and MMAs:
  //    chunk 8w + 4*s2 + mi of tokens 8jt..8jt+7 gives b0/b1 of steps 2*s2
  //    and 2*s2+1 of this warp.
  const uint32_t s_x = smem_u32(smem + L::X);
  // Up to 16 tokens (MT <= 2) the even and odd k-steps accumulate in two
  // independent chains, added before the cross-warp sum (0.03-0.04 us per
  // layer call faster at M = 12-16; at MT = 3, 4 one chain measured faster).
  constexpr int NC = MT <= 2 ? 2 : 1;
  float acc[NC][MT][4];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int jt = 0; jt < MT; ++jt) acc[c][jt][0] = acc[c][jt][1] = acc[c][jt][2] = acc[c][jt][3] = 0.f;
#pragma unroll
  for (int s2 = 0; s2 < 2; ++s2) {
    uint32_t b[MT][4];
#pragma unroll
    for (int jt = 0; jt < MT; ++jt)
      ldmatrix_x4(b[jt], s_x + q_off<kLatent>(8 * jt + (lane & 7), 8 * warp + 4 * s2 + mi));
#pragma unroll
    for (int jt = 0; jt < MT; ++jt) {
      mma_bf16_16816(acc[0][jt], a[2 * s2], b[jt][0], b[jt][1]);
      mma_bf16_16816(acc[NC - 1][jt], a[2 * s2 + 1], b[jt][2], b[jt][3]);
    }
  }
  if constexpr (NC == 2) {
#pragma unroll
    for (int jt = 0; jt < MT; ++jt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[0][jt][e] += acc[1][jt][e];
  }

  // 7. Cross-warp sum: partial (jt, e, lane) of warp w at red[((w*MT+jt)*4+e)*kVRedRow+lane].
  //    D element e of lane ln is output column (ln>>2) + 8*(e>>1) and token
  //    8jt + 2*(ln&3) + (e&1); lanes ln and ln+4 hold adjacent columns.  Each
  //    thread below sums one such pair over the 8 warps, rounds it to BF16
  //    and writes it with one 4-byte store (64*MT pairs).
  float* red = reinterpret_cast<float*>(smem + L::Raw);
#pragma unroll
  for (int jt = 0; jt < MT; ++jt)
#pragma unroll
    for (int e = 0; e < 4; ++e) red[((warp * MT + jt) * 4 + e) * kVRedRow + lane] = acc[0][jt][e];
  __syncthreads();
  if (tid < 64 * MT) {
    const int t4 = tid & 3;           // lane & 3 of the pair
    const int gp = (tid >> 2) & 3;    // column pair: lanes 8*gp + t4 and 8*gp + 4 + t4
    const int e = (tid >> 4) & 3;
    const int jt = tid >> 6;
    const int ln = 8 * gp + t4;
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int w = 0; w < kVWarps; ++w) {
      v0 += red[((w * MT + jt) * 4 + e) * kVRedRow + ln];
      v1 += red[((w * MT + jt) * 4 + e) * kVRedRow + ln + 4];
    }
    const int col = 2 * gp + 8 * (e >> 1);   // even: columns col, col+1
    const int tok = 8 * jt + 2 * t4 + (e & 1);
    if (tok < M)
      *reinterpret_cast<uint32_t*>(outc + tok * p.out_row_stride + h * kVDim + d_cta + col) = pack_bf16x2(v1, v0);
  }
}

}  // namespace mlaqp
