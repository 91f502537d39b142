// Fused MLA query projection for larger token counts (33 <= M <= 256: multi-
// token prediction and prefill-sized steps) on the 5th-generation tensor
// cores of sm_103a: tcgen05.mma with the accumulator in tensor memory (TMEM).
//
// Same operation as mlaqp_kernel.cuh (SparkInfer PR #75 "Add BF16 MLA query
// projection and assembly", sections What and Contract; vLLM PR #174 "Fuse
// MXFP8 and BF16 MLA query assembly", section What), different tiling:
//   CTA (tile, h, z) owns head h, latent columns [128*tile, 128*tile+128)
//   and tokens [TT*z, TT*z+TT).  One UMMA of shape M=128 (latent columns) x
//   N=ntok (the chunk's tokens rounded up to 16) x K=16 per k-step, K/16
//   k-steps issued by one thread:
//     A = W_UK_T tile, MN-major (latent columns contiguous), 128B swizzle:
//         two TMA boxes of 64 columns x K rows, which is the canonical
//         MN-major SW128 layout (64-element rows, 8-row core groups);
//     B = q_nope tile, K-major, 128B swizzle: for each 64-wide k slice a
//         block of TT rows of 128 bytes, written by the threads;
//     D = FP32 [128 lanes x ntok columns] in TMEM.
//   Warp w reads TMEM lanes 32w..32w+31 (one latent column per thread, all
//   tokens), rounds to BF16 (optionally divides by q_scale and converts to
//   E4M3), stages the [ntok][128] output tile in shared memory and stores it
//   with 16-byte writes; the chunk's q_pe is appended by the (h, z) CTAs.
//
// Tensor memory is allocated only after griddepcontrol.wait, so a CTA never
// holds TMEM while it waits for an earlier kernel, and the next kernel may
// launch only once every CTA of this one has its TMEM.  The host pads the
// shared memory so that the CTAs one SM can hold never ask for more than its
// 512 TMEM columns.  Every mbarrier wait is bounded; on expiry the CTA
// records the timeout, releases its TMEM and returns without writing.

#pragma once

#include "mlaqp_kernel.cuh"

namespace mlaqp {

constexpr int kLargeMaxM = 256;
constexpr int kLargeNTile = 128;                           // latent columns per CTA (UMMA M)
constexpr int kLargeTilesPerHead = kLatent / kLargeNTile;  // 4
// Threads per CTA for a token tile of tt tokens: groups of 4 warps, each
// group spanning the 128 TMEM lanes.  Tiles of 64 and 128 tokens convert
// 64 x 128 / 128 x 128 outputs per CTA with few CTAs per SM, so they get 4
// groups to keep more warps in flight (E4M3 output at M = 256: 5.38 -> 4.60
// us per layer); the 32-token tile gets 2.
__host__ __device__ constexpr int large_threads(int tt) { return tt >= 64 ? 512 : 256; }

// Shared memory layout of the large kernel for nope dim K, TT tokens per CTA
// and MXFP8 (mx) or BF16 weights (offsets from a 1024-byte aligned base).
// The E4M3 bytes of an MXFP8 tile share the q_nope region: they are consumed
// (dequantised into `a`) before the dependency wait, the q_nope rows written
// after it, with a CTA barrier in between.
struct LargeSmem {
  int a;          // BF16 weight tile: two [K][64] halves, 128B swizzle
  int b;          // q_nope tile: K/64 slices of [TT][64] BF16, 128B swizzle;
                  // after the MMAs, the [ntok][128] output stage
  int raw;        // MXFP8 only: E4M3 [2][K][64] as copied (= b)
  int scale;      // MXFP8 only: E8M0 [K][16] of the head
  int div;        // FP32 [128]: RN((128+f)/q_scale)
  int bar;        // two mbarriers: weights, MMA completion
  int tmem_slot;  // TMEM base address written by tcgen05.alloc
  int bytes;      // total, with slack for the 1024-byte alignment
};

__host__ __device__ constexpr LargeSmem large_smem_layout(int K, int TT, bool mx) {
  LargeSmem s{};
  s.a = 0;
  s.b = s.a + 2 * K * 128;
  s.raw = s.b;
  const int bq = TT * K * 2;
  const int braw = mx ? 2 * K * 64 : 0;
  s.scale = s.b + (bq > braw ? bq : braw);
  s.div = s.scale + (mx ? K * (kLatent / kMxBlock) : 0);
  s.bar = s.div + 128 * 4;
  s.tmem_slot = s.bar + 16;
  s.bytes = s.tmem_slot + 16 + 1024;
  return s;
}

// TMEM columns to allocate for ntok accumulator columns: a power of two >= 32.
__host__ __device__ constexpr uint32_t tmem_cols_for(int ntok) {
  return ntok <= 32 ? 32u : ntok <= 64 ? 64u : ntok <= 128 ? 128u : 256u;
}

// ---------------------------------------------------------------------------
// tcgen05 / TMEM helpers (documented PTX only)
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), the fixed descriptor version 1 of the sm_100
// family (bit 46) and the 128-byte swizzle mode (2 in bits 61..63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16: FP32 accumulator (bits 4..5 = 1),
// BF16 A and B (bits 7..9 = 1, 10..12 = 1), A MN-major (bit 15), B K-major
// (bit 16 clear), N/8 in bits 17..22, M/16 in bits 24..28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (tensor core) reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]; accumulate = 0 overwrites D.
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One arrival on `bar` once every tcgen05.mma this thread issued completes.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 16 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// The kernel.  Grid (4, H, ceil(M/TT)); large_threads(TT) threads.  EARLY = 1
// lets the next kernel launch at entry instead of after the TMEM allocation
// (the caller's opt-in: no later kernel may take TMEM before its own
// dependency wait, or it could hold the columns this one still needs).
// ---------------------------------------------------------------------------

template <int WF, int OD, int K, int TT, int EARLY = 0>
__global__ void __launch_bounds__(large_threads(TT)) mlaqp_fused_query_large_kernel(const __grid_constant__ RunParams p) {
  if constexpr (EARLY) pdl_launch_dependents();
  constexpr int kLargeThreads = large_threads(TT);
  constexpr int kLargeGroups = kLargeThreads / 128;
  static_assert(K % 64 == 0 && K <= 256, "nope dim: multiple of 64, at most one TMA box (256 rows)");
  static_assert(TT % 16 == 0 && TT <= 256 && (TT * K / 8) % kLargeThreads == 0, "token tile");
  constexpr LargeSmem L = large_smem_layout(K, TT, WF == kWeightMXFP8);
  constexpr int KS = K / 16;                          // UMMA k-steps
  constexpr int KC = K / 8;                           // 16-byte chunks per q_nope row
  constexpr int QI = TT * KC / kLargeThreads;         // q_nope chunks per thread
  constexpr int kScaleRow = kLatent / kMxBlock;       // E8M0 bytes per (h, k)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  const int m0 = blockIdx.z * TT;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int rows = min(TT, p.M - m0);  // >= 1: the grid has ceil(M/TT) chunks
  const int ntok = (rows + 15) & ~15;
  const uint32_t ncols = tmem_cols_for(ntok);
  const int n_cta = tile * kLargeNTile;
  const uint32_t s_a = smem_u32(smem + L.a);
  const uint32_t s_b = smem_u32(smem + L.b);
  const uint32_t bar_w = smem_u32(smem + L.bar);
  const uint32_t bar_mma = bar_w + 8;
  const uint16_t* q_nope = p.q_nope + m0 * p.q_nope_ts + h * p.q_nope_hs;
  const uint16_t* q_pe = p.q_pe + m0 * p.q_pe_ts + h * p.q_pe_hs;

  // q_scale is a per-tensor constant of the layer, read (and its division
  // table built) ahead of the dependency wait, like the weights.
  float qs = 1.f;
  if constexpr (OD == kOutE4M3) qs = *p.q_scale;

  // 1. Weight (and scale) stream: two TMA boxes of 64 columns x K rows.
  if (tid == 0) {
    prefetch_tensormap(&p.wmap);
    mbar_init(bar_w, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    if constexpr (WF == kWeightBF16) {
      mbar_arrive_expect_tx(bar_w, 2 * K * 128 + p.extra_tx);
      tma_load_2d(s_a, &p.wmap, n_cta, h * K, bar_w);
      tma_load_2d(s_a + K * 128, &p.wmap, n_cta + 64, h * K, bar_w);
    } else {
      const uint32_t s_raw = smem_u32(smem + L.raw);
      mbar_arrive_expect_tx(bar_w, 2 * K * 64 + K * kScaleRow + p.extra_tx);
      tma_load_2d(s_raw, &p.wmap, n_cta, h * K, bar_w);
      tma_load_2d(s_raw + K * 64, &p.wmap, n_cta + 64, h * K, bar_w);
      bulk_load_1d(smem_u32(smem + L.scale), p.weight_scale + static_cast<size_t>(h) * K * kScaleRow, K * kScaleRow,
                   bar_w);
    }
  }
  // 2. Warm L2 with the chunk's q rows (values are read after the wait).
  if (tid < rows) {
#pragma unroll
    for (int o = 0; o < K; o += 64) prefetch_l2(q_nope + tid * p.q_nope_ts + o);
  }
  if (tid >= kLargeThreads - 128 && tid - (kLargeThreads - 128) < rows) {
    prefetch_l2(q_pe + (tid - (kLargeThreads - 128)) * p.q_pe_ts);
  }
  uint32_t* divtab = reinterpret_cast<uint32_t*>(smem + L.div);
  bool table_ok = false, mul_ok = false;
  float rcp = 1.f;
  bool mine = true;
  if constexpr (OD == kOutE4M3) {
    table_ok = qs >= 0x1p-100f && qs <= 0x1p100f;  // uniform across the grid
    rcp = __frcp_rn(qs);
    mine = table_ok;
    if (table_ok && tid < 128) {
      divtab[tid] = __float_as_uint(__fdiv_rn(static_cast<float>(128 + tid), qs));
      mine = e4m3_mul_exact_for(tid, qs, rcp);
    }
  }
  mul_ok = __syncthreads_and(mine) && OD == kOutE4M3;  // barriers initialised, table visible

  // 3. MXFP8: dequantise both 64-column halves into the swizzled BF16 tile
  //    (value = code * 2^(x-127) as two exact power-of-two factors).  Job
  //    (half, row k, chunk c of 8 columns): 16K jobs, K/16 per thread.
  if constexpr (WF == kWeightMXFP8) {
    const bool ok = mbar_wait_bounded(bar_w, 0, p.wait_limit_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
      pdl_wait();  // exit only after the previous kernel: later waits rely on it
      return;
    }
    const uint8_t* raw = smem + L.raw;
    const uint8_t* sc = smem + L.scale;
    const int c = tid & 7;
#pragma unroll 4
    for (int i = 0; i < 16 * K / kLargeThreads; ++i) {
      const int row = (tid >> 3) + (kLargeThreads / 8) * i;  // half * K + k
      const int half = row >= K ? 1 : 0;
      const int k = row - half * K;
      const uint2 v = *reinterpret_cast<const uint2*>(raw + row * 64 + 8 * c);
      const uint32_t x = sc[k * kScaleRow + (n_cta + 64 * half + 8 * c) / kMxBlock];
      const uint32_t s1 = pow2_bf16(min(x, 134u));
      const uint32_t f1 = s1 | (s1 << 16);
      const uint32_t s2 = x == 255u ? 0x7FC0u : pow2_bf16(max(x, 134u) - 127u);
      const uint32_t f2 = s2 | (s2 << 16);
      const uint32_t w[2] = {v.x, v.y};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o[q] = mul_bf16x2(mul_bf16x2(e4m3x2_to_bf16x2_scaled(w[q >> 1] >> (16 * (q & 1))), f1), f2);
      *reinterpret_cast<uint4*>(smem + L.a + half * K * 128 + sw128(k, c)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    fence_proxy_async_smem();
    __syncthreads();  // every E4M3 byte read before the q_nope rows overwrite them
  }

  // 4. Wait for the producer of q_nope / q_pe (no-op without PDL).
  pdl_wait();

  // 5. Every input load of the CTA in flight at once: the chunk's q_nope
  //    rows (rows >= `rows` zero) and its share of the q_pe pairs (the
  //    chunk's rows*32 pairs dealt over the head's 4 CTAs).
  constexpr int kPe = (TT * (kRope / 2) + kLargeTilesPerHead * kLargeThreads - 1) / (kLargeTilesPerHead * kLargeThreads);
  uint4 qv[QI];
#pragma unroll
  for (int i = 0; i < QI; ++i) {
    const int c = tid + kLargeThreads * i;
    const int m = c / KC;
    qv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (m < rows) qv[i] = ld_u128(q_nope + m * p.q_nope_ts + 8 * (c % KC));
  }
  uint32_t pe[kPe];
#pragma unroll
  for (int i = 0; i < kPe; ++i) {
    const int j = tile * kLargeThreads + tid + kLargeTilesPerHead * kLargeThreads * i;
    pe[i] = 0u;
    if (j < rows * (kRope / 2)) pe[i] = ld_u32(q_pe + (j >> 5) * p.q_pe_ts + 2 * (j & 31));
  }
  // Accumulator columns in TMEM (warp 0) while the loads are in flight;
  // then the next kernel may launch.
  if (warp == 0) tmem_alloc(smem_u32(smem + L.tmem_slot), ncols);
  if constexpr (!EARLY) pdl_launch_dependents();

  // 6. q_nope into the B tile: k slice a of row m, 16-byte chunk cc at
  //    a*TT*128 + m*128 + 16*(cc ^ m%8).
#pragma unroll
  for (int i = 0; i < QI; ++i) {
    const int c = tid + kLargeThreads * i;
    const int kc = c % KC;
    *reinterpret_cast<uint4*>(smem + L.b + (kc >> 3) * (TT * 128) + sw128(c / KC, kc & 7)) = qv[i];
  }
  fence_proxy_async_smem();
  bool ok = true;
  if constexpr (WF == kWeightBF16) ok = mbar_wait_bounded(bar_w, 0, p.wait_limit_ns);
  tc_fence_before();
  const bool any_timeout = __syncthreads_or(!ok);
  tc_fence_after();
  const uint32_t taddr = *reinterpret_cast<volatile uint32_t*>(smem + L.tmem_slot);
  if (any_timeout) {
    if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
    if (warp == 0) tmem_dealloc(taddr, ncols);
    return;
  }

  // 7. One thread issues the K/16 MMAs and commits them to bar_mma.
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(kLargeNTile, ntok);
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      // A: k rows 16s..16s+15 = two 8-row core groups 1024 B apart (SBO);
      //    the second 64-column half is K*128 bytes further (LBO).
      const uint64_t ad = smem_desc_sw128(s_a + s * 2048, K * 128, 1024);
      // B: k slice s/4, 32-byte step s%4 inside its 128-byte rows; 8-row
      //    core groups 1024 B apart (SBO); LBO unused for this layout.
      const uint64_t bd = smem_desc_sw128(s_b + (s >> 2) * (TT * 128) + (s & 3) * 32, 16, 1024);
      umma_bf16(taddr, ad, bd, idesc, s > 0 ? 1u : 0u);
    }
    umma_commit(bar_mma);
  }

  // 8. q_pe append while the MMAs run (bit copy or E4M3 cast).
#pragma unroll
  for (int i = 0; i < kPe; ++i) {
    const int j = tile * kLargeThreads + tid + kLargeTilesPerHead * kLargeThreads * i;
    if (j < rows * (kRope / 2)) {
      const size_t off = static_cast<size_t>(m0 + (j >> 5)) * p.out_row_stride + static_cast<size_t>(h) * kOutDim +
                         kLatent + 2 * (j & 31);
      if (OD == kOutBF16 || mul_ok) {
        write_pe_pair<OD, kE4m3MulExact>(p, off, pe[i], divtab, qs, rcp);
      } else if (table_ok) {
        write_pe_pair<OD, kE4m3Table>(p, off, pe[i], divtab, qs, rcp);
      } else {
        write_pe_pair<OD, kE4m3Divide>(p, off, pe[i], divtab, qs, rcp);
      }
    }
  }

  // 9. Epilogue: wait for the accumulator.  Warp w reads TMEM lanes
  //    32*(w%4).. (latent column n_cta + 32*(w%4) + lane); the warp groups
  //    take the 16-token column chunks in turn.  Values are rounded to
  //    BF16 (optionally E4M3), staged as the [ntok][128] output tile in the
  //    (now free) B region, then stored row by row.
  const bool done = mbar_wait_bounded(bar_mma, 0, p.wait_limit_ns);
  tc_fence_after();
  if (__syncthreads_or(!done)) {
    if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(taddr, ncols);
    return;
  }
  constexpr int kEB = OD == kOutBF16 ? 2 : 1;  // output element bytes
  const int quarter = warp & 3;
  const int col = 32 * quarter + lane;         // latent column within the CTA tile
  uint8_t* stage = smem + L.b;                 // [ntok][128] output elements
  for (int c16 = warp >> 2; c16 < ntok / 16; c16 += kLargeGroups) {
    uint32_t r[16];
    tmem_ld16(taddr + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(16 * c16), r);
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = pack_bf16x2(__uint_as_float(r[2 * i + 1]), __uint_as_float(r[2 * i]));
    if constexpr (OD == kOutE4M3) {
      if (mul_ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = e4m3_pair<kE4m3MulExact>(v[i], divtab, qs, rcp);
      } else if (table_ok) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = e4m3_pair<kE4m3Table>(v[i], divtab, qs, rcp);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = e4m3_pair<kE4m3Divide>(v[i], divtab, qs, rcp);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = 16 * c16 + 2 * i;  // tokens j (low half / byte 0) and j+1
      if constexpr (OD == kOutBF16) {
        reinterpret_cast<uint16_t*>(stage)[j * kLargeNTile + col] = static_cast<uint16_t>(v[i]);
        reinterpret_cast<uint16_t*>(stage)[(j + 1) * kLargeNTile + col] = static_cast<uint16_t>(v[i] >> 16);
      } else {
        stage[j * kLargeNTile + col] = static_cast<uint8_t>(v[i]);
        stage[(j + 1) * kLargeNTile + col] = static_cast<uint8_t>(v[i] >> 8);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, ncols);
  // Row m of the tile is kLargeNTile*kEB contiguous bytes of output row m0+m.
  constexpr int kRowChunks = kLargeNTile * kEB / 16;
  for (int c = tid; c < rows * kRowChunks; c += kLargeThreads) {
    const int m = c / kRowChunks;
    const int part = c % kRowChunks;
    const uint4 v = *reinterpret_cast<const uint4*>(stage + m * (kLargeNTile * kEB) + 16 * part);
    const size_t off =
        (static_cast<size_t>(m0 + m) * p.out_row_stride + static_cast<size_t>(h) * kOutDim + n_cta) * kEB + 16 * part;
    *reinterpret_cast<uint4*>(p.out + off) = v;
  }
}

}  // namespace mlaqp
