// V up-projection for 9 <= M <= 64 with the attention output x brought in
// by one TMA multicast per CTA (sm_103a, mma.sync):
//
//   out[m,h,d] = bf16_rne( sum_{c<512} x[m,h,c] * W_UV[h,c,d] )    d < 128, FP32 accumulation
//
// (the downstream V up-projection the pages name, vLLM PR #174 "Fuse MXFP8
// and BF16 MLA query assembly", section Safety scope; weight formats as on
// the query side, section What).
//
// Work split as in mlaqp_v_up_kernel.cuh: CTA (tile, h, z) owns head h,
// output columns [16*tile, 16*tile+16) and tokens [32z, 32z+32); eight warps
// split the 512-long contraction, 64 each, and add their partial sums in
// shared memory.  Every CTA needs the chunk's whole x block [TT][512] (TT =
// 8*MT tokens).  Read with 16-byte loads after the dependency wait, that is
// M x 1 KB per CTA and eight copies of every x byte per head from L2.  Here
// the eight CTAs of (h, z) form a cluster, and CTA `tile` copies the
// 64-column box `tile` of the block (TT rows x 128 bytes, 128-byte swizzle)
// once into all eight CTAs (TMA multicast), so the contraction slice of
// warp w is box w.  Token rows at or beyond M lie outside the tensor map
// and arrive as zeros.
//
// Steps of a CTA:
//  1. thread 0: weight tile (two 2-D TMA boxes of 16 columns x 256 rows,
//     plus the E8M0 scales for MXFP8) on one barrier; the x barrier expects
//     the eight boxes; this CTA's box of x prefetched into L2;
//  2. cluster barrier, split: arrive here, wait just before the multicast
//     (every CTA's x barrier is initialised);
//  3. MXFP8: dequantise into the BF16 tile before the dependency wait;
//  4. griddepcontrol.wait;
//  5. thread 0 issues this CTA's x box to the whole cluster; the weight
//     fragments (ldmatrix.trans) load meanwhile; wait for the x barrier;
//  6. MMAs over this warp's 64 contraction columns;
//  7. cross-warp sum, BF16 rounding, 4-byte stores of column pairs.
//
// Failure handling: every mbarrier wait is bounded.  A CTA never returns
// before its x barrier wait: peers' multicasts write into its shared memory
// until then.  A CTA whose weight copy timed out still issues its x box and
// waits for the others; a CTA that gave up anywhere writes nothing and sets
// the device status.

#pragma once

#include "mlaqp_v_up_kernel_large.cuh"

namespace mlaqp {

// Shared memory layout for MT 8-token tiles (offsets from a 1024-byte
// aligned base).
template <int MT>
struct VMcSmem {
  static constexpr int TT = 8 * MT;
  static constexpr int W = 0;                                         // BF16 [512][16], 32B swizzle
  static constexpr int X = W + kLatent * kVNTile * 2;                // BF16 [8 boxes][TT][64], 128B swizzle
  static constexpr int Raw = X + 8 * TT * 128;                        // E4M3 [512][16]; later FP32 partials
  static constexpr int RedBytes = kVWarps * MT * 4 * kVRedRow * 4;
  static constexpr int RawBytes = kLatent * kVNTile;
  static constexpr int Scale = Raw + (RedBytes > RawBytes ? RedBytes : RawBytes);  // E8M0 [512][4]
  static constexpr int Bar = Scale + kLatent * kVScaleRow;           // weights, x
  static constexpr int Bytes = Bar + 16 + 1024;
  static_assert(X % 1024 == 0 && (TT * 128) % 1024 == 0, "128-byte swizzle atoms");
};

// 3-D TMA tile load multicast to the cluster's CTAs in `mask`: the same
// shared-memory offset `dst` and barrier offset `bar` in each of them.
__device__ __forceinline__ void tma_load_3d_multicast(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                                      uint32_t bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "h"(mask)
      : "memory");
}

template <int WF, int MT, int TRIG>
__global__ void __launch_bounds__(kVThreads) mlaqp_v_up_mc_kernel(const __grid_constant__ VUpParams p) {
  using L = VMcSmem<MT>;
  constexpr int TT = L::TT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_w = smem_u32(smem + L::W);
  const uint32_t s_x = smem_u32(smem + L::X);
  const uint32_t bar_w = smem_u32(smem + L::Bar);
  const uint32_t bar_x = bar_w + 8;

  const int tile = blockIdx.x;  // = rank in the (8, 1, 1) cluster
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int m0 = blockIdx.z * TT;       // this CTA's tokens: [m0, m0 + M) of a TT-token chunk
  const int M = min(TT, p.M - m0);      // >= 1
  const int d_cta = tile * kVNTile;
  uint16_t* const outc = p.out + m0 * p.out_row_stride;

  if constexpr (TRIG == 0) pdl_launch_dependents();

  // 1. Weight (and scale) stream; x barrier; this CTA's x box into L2.
  if (tid == 0) {
    prefetch_tensormap(&p.wmap);
    prefetch_tensormap(&p.xmap);
    mbar_init(bar_w, 1);
    mbar_init(bar_x, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar_x, 8 * TT * 128);
    if constexpr (WF == kWeightBF16) {
      mbar_arrive_expect_tx(bar_w, kLatent * kVNTile * 2 + p.extra_tx);
      tma_load_2d(s_w, &p.wmap, d_cta, h * kLatent, bar_w);
      tma_load_2d(s_w + 256 * kVNTile * 2, &p.wmap, d_cta, h * kLatent + 256, bar_w);
    } else {
      const uint32_t s_raw = smem_u32(smem + L::Raw);
      mbar_arrive_expect_tx(bar_w, kLatent * kVNTile + kLatent * kVScaleRow + p.extra_tx);
      tma_load_2d(s_raw, &p.wmap, d_cta, h * kLatent, bar_w);
      tma_load_2d(s_raw + 256 * kVNTile, &p.wmap, d_cta, h * kLatent + 256, bar_w);
      bulk_load_1d(smem_u32(smem + L::Scale), p.weight_scale + static_cast<size_t>(h) * kLatent * kVScaleRow,
                   kLatent * kVScaleRow, bar_w);
    }
  }
  if (tid < M) prefetch_l2(p.x + (m0 + tid) * p.x_ts + h * p.x_hs + 64 * tile);
  __syncthreads();           // barriers initialised before anyone waits on them
  cluster_arrive_relaxed();  // ... and, once every CTA has arrived, before any multicast lands

  // 3. MXFP8: dequantise into the BF16 tile (value = code * 2^(x-127) as two
  //    exact power-of-two factors).  Job (row r, half c): 1024 jobs.
  bool ok = true;  // uniform across the CTA
  if constexpr (WF == kWeightMXFP8) {
    ok = !__syncthreads_or(!mbar_wait_bounded(bar_w, 0, p.wait_limit_ns));
    if (ok) {
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
    }
    __syncthreads();  // the E4M3 staging area is free for the partial sums
  }

  // 4. Wait for the producer of x (no-op without PDL).
  pdl_wait();
  if constexpr (TRIG == 1) pdl_launch_dependents();

  // 5. This CTA's x box to every CTA of the cluster: columns [64*tile,
  //    64*tile+64) of tokens [m0, m0+TT) of head h (3-D map: column, head,
  //    token), into box `tile` of X.
  cluster_wait();  // every CTA's x barrier is initialised
  if (tid == 0) tma_load_3d_multicast(s_x + tile * (TT * 128), &p.xmap, 64 * tile, h, m0, bar_x, 0xFFu);
  if constexpr (WF == kWeightBF16) ok = !__syncthreads_or(!mbar_wait_bounded(bar_w, 0, p.wait_limit_ns));
  // A fragments for the warp's four k-steps s = 4w..4w+3: matrices 0/1 =
  // rows 16s..+7 (columns 0-7 / 8-15), 2/3 = rows 16s+8..+15.
  const int mi = lane >> 3;
  uint32_t a[4][4];
  if (ok) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int row = 16 * (4 * warp + s) + 8 * (mi >> 1) + (lane & 7);
      ldmatrix_x4_trans(a[s], s_w + sw32(row, mi & 1));
    }
  }
  // The x barrier is waited for on every path: until it completes, peers'
  // copies may still be landing in this CTA's shared memory.
  const bool xok = !__syncthreads_or(!mbar_wait_bounded(bar_x, 0, p.wait_limit_ns));
  if (!(ok && xok)) {
    if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
    return;
  }

  // 6. B fragments from box w (x rows = tokens; 16-byte chunk c of row m at
  //    m*128 + 16*(c ^ m%8)): chunk 4*s2 + mi of tokens 8jt..8jt+7 gives
  //    b0/b1 of steps 2*s2 and 2*s2+1 of this warp.
  const uint32_t s_box = s_x + warp * (TT * 128);
  constexpr int NC = MT <= 2 ? 2 : 1;  // accumulator chains, as in mlaqp_v_up_kernel.cuh
  float acc[NC][MT][4];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int jt = 0; jt < MT; ++jt) acc[c][jt][0] = acc[c][jt][1] = acc[c][jt][2] = acc[c][jt][3] = 0.f;
#pragma unroll
  for (int s2 = 0; s2 < 2; ++s2) {
    uint32_t b[MT][4];
#pragma unroll
    for (int jt = 0; jt < MT; ++jt) {
      const int m = 8 * jt + (lane & 7);
      ldmatrix_x4(b[jt], s_box + m * 128 + 16 * ((4 * s2 + mi) ^ (m & 7)));
    }
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

  // 7. Cross-warp sum (as in mlaqp_v_up_kernel.cuh): partial (jt, e, lane) of
  //    warp w at red[((w*MT+jt)*4+e)*kVRedRow+lane]; each thread below sums one
  //    pair of adjacent output columns over the 8 warps, rounds it to BF16
  //    and writes it with one 4-byte store.
  float* red = reinterpret_cast<float*>(smem + L::Raw);
#pragma unroll
  for (int jt = 0; jt < MT; ++jt)
#pragma unroll
    for (int e = 0; e < 4; ++e) red[((warp * MT + jt) * 4 + e) * kVRedRow + lane] = acc[0][jt][e];
  __syncthreads();
  if (tid < 64 * MT) {
    const int t4 = tid & 3;
    const int gp = (tid >> 2) & 3;
    const int e = (tid >> 4) & 3;
    const int jt = tid >> 6;
    const int ln = 8 * gp + t4;
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int w = 0; w < kVWarps; ++w) {
      v0 += red[((w * MT + jt) * 4 + e) * kVRedRow + ln];
      v1 += red[((w * MT + jt) * 4 + e) * kVRedRow + ln + 4];
    }
    const int col = 2 * gp + 8 * (e >> 1);
    const int tok = 8 * jt + 2 * t4 + (e & 1);
    if (tok < M)
      *reinterpret_cast<uint32_t*>(outc + tok * p.out_row_stride + h * kVDim + d_cta + col) = pack_bf16x2(v1, v0);
  }
}

}  // namespace mlaqp
