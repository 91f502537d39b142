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
//  3. MXFP8: all threads wait for the copy and dequantise into the same
//     swizzled BF16 tile (e4m3 * 2^(e8m0-127), exact);
//  4. griddepcontrol.wait -- everything above is independent of the
//     previous kernel, so under programmatic dependent launch it overlaps
//     that kernel; everything below reads inputs it may have produced;
//  5. q_nope fragments straight from global memory into registers;
//  6. ldmatrix.trans of the weight fragments, mma.sync m16n8k16 BF16 -> FP32
//     with the latent axis on the MMA's M side and tokens on its N side
//     (swap-AB: M <= 32 tokens costs at most four 8-wide column tiles);
//  7. epilogue: round to BF16 (optionally divide by q_scale and convert to
//     E4M3 with saturation), transpose the 8x8 blocks with movmatrix so
//     each lane holds consecutive latent columns of one token, and store
//     straight into the caller's strided workspace; q_pe is appended by the
//     head's CTAs in 16-byte chunks.
//
// Every mbarrier wait is bounded by a wall-clock limit; on expiry the CTA
// records MLAQP_DEVSTATUS_WAIT_TIMEOUT in a device status word and returns
// without writing its outputs.

#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mlaqp {

constexpr int kNope = 128;
constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kOutDim = kLatent + kRope;
constexpr int kMxBlock = 32;
constexpr int kMaxM = 32;

constexpr int kNTile = 64;                       // latent columns per CTA
constexpr int kWarps = kNTile / 16;              // one 16-column MMA tile per warp
constexpr int kThreads = kWarps * 32;            // 128
constexpr int kTilesPerHead = kLatent / kNTile;  // 8

// Dynamic shared memory layout (offsets from a 1024-byte aligned base).
constexpr int kSmemA = 0;                            // BF16 [128][64], 128B swizzle: 16 KB
constexpr int kSmemRaw = kSmemA + kNope * kNTile * 2;  // E4M3 [128][64]: 8 KB
constexpr int kSmemScale = kSmemRaw + kNope * kNTile;  // E8M0 [128][16]: 2 KB
constexpr int kSmemBar = kSmemScale + kNope * (kLatent / kMxBlock);
constexpr int kSmemBytes = kSmemBar + 64 + 1024;  // + slack for the 1024-byte alignment

enum WeightFormat : int { kWeightBF16 = 0, kWeightMXFP8 = 1 };
enum OutDtype : int { kOutBF16 = 0, kOutE4M3 = 1 };

constexpr unsigned kDevStatusWaitTimeout = 1u;

struct RunParams {
  CUtensorMap wmap;             // 2-D map of W_UK_T viewed as [H*128 rows][512 cols], box 64 x 128
  const uint16_t* q_nope;       // BF16 [M,H,128]
  const uint16_t* q_pe;         // BF16 [M,H,64]
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

// E4M3 pair -> FP32 pair, exactly: every E4M3 value (subnormals included) is
// a normal FP16 value, so the E4M3x2 -> F16x2 conversion is exact, as is
// F16 -> F32.  Byte 0 of `pair16` gives `lo`.
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t pair16, float& lo, float& hi) {
  uint32_t h2;
  const uint16_t p16 = static_cast<uint16_t>(pair16);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(p16));
  const uint16_t h_lo = static_cast<uint16_t>(h2), h_hi = static_cast<uint16_t>(h2 >> 16);
  asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(h_lo));
  asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(h_hi));
}

// E8M0 byte -> 2^(x-127) as FP32 (x = 0 is the subnormal 2^-127, 255 NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t x) {
  const uint32_t bits = x == 0 ? 0x00400000u : (x == 255 ? 0x7FC00000u : (x << 23));
  return __uint_as_float(bits);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile of 128-byte
// rows stored with the TMA 128B swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------------------
// The kernel.  MT = number of 8-token column tiles, ceil(M/8) in 1..4.
// ---------------------------------------------------------------------------

template <int WF, int OD, int MT>
__global__ void __launch_bounds__(kThreads) mlaqp_fused_query_kernel(const __grid_constant__ RunParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_a = smem_u32(smem + kSmemA);
  const uint32_t s_bar = smem_u32(smem + kSmemBar);

  const int tile = blockIdx.x;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int H = p.H;
  const int M = p.M;
  const int n_cta = tile * kNTile;

  // The next kernel on the stream may start its independent prologue.
  pdl_launch_dependents();

  // 1. Weight (and scale) stream: one elected thread, one barrier phase.
  if (tid == 0) {
    prefetch_tensormap(&p.wmap);
    mbar_init(s_bar, 1);
    fence_barrier_init();
    if constexpr (WF == kWeightBF16) {
      mbar_arrive_expect_tx(s_bar, kNope * kNTile * 2 + p.extra_tx);
      tma_load_2d(s_a, &p.wmap, n_cta, h * kNope, s_bar);
    } else {
      mbar_arrive_expect_tx(s_bar, kNope * kNTile + kNope * (kLatent / kMxBlock) + p.extra_tx);
      tma_load_2d(smem_u32(smem + kSmemRaw), &p.wmap, n_cta, h * kNope, s_bar);
      bulk_load_1d(smem_u32(smem + kSmemScale), p.weight_scale + static_cast<size_t>(h) * kNope * (kLatent / kMxBlock),
                   kNope * (kLatent / kMxBlock), s_bar);
    }
  }

  // 2. Warm L2 with the head's q rows (L2 is the coherence point, so a line
  //    fetched before the producer writes it is updated by that write; the
  //    values themselves are read only after the dependency wait).
  if (warp == 0 && lane < M) {
    const uint16_t* qrow = p.q_nope + (static_cast<size_t>(lane) * H + h) * kNope;
    prefetch_l2(qrow);
    prefetch_l2(qrow + 64);
    prefetch_l2(p.q_pe + (static_cast<size_t>(lane) * H + h) * kRope);
  }
  __syncthreads();  // barrier initialised before anyone waits on it

  // 3. MXFP8: dequantise into the swizzled BF16 tile before the dependency
  //    wait.  Job (row k, chunk c of 8 columns); 1024 jobs, 8 per thread.
  if constexpr (WF == kWeightMXFP8) {
    const bool ok = mbar_wait_bounded(s_bar, 0, p.wait_limit_ns);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
      return;
    }
    const uint8_t* raw = smem + kSmemRaw;
    const uint8_t* sc = smem + kSmemScale;
    const int c = tid & 7;
    const int blk = (n_cta + 8 * c) / kMxBlock;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = (tid >> 3) + 16 * i;
      const uint2 v = *reinterpret_cast<const uint2*>(raw + k * kNTile + 8 * c);
      const float f = e8m0_to_f32(sc[k * (kLatent / kMxBlock) + blk]);
      uint32_t o[4];
      const uint32_t w[2] = {v.x, v.y};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float lo, hi;
        e4m3x2_to_f32(w[q >> 1] >> (16 * (q & 1)), lo, hi);
        o[q] = pack_bf16x2(__fmul_rn(hi, f), __fmul_rn(lo, f));
      }
      *reinterpret_cast<uint4*>(smem + kSmemA + sw128(k, c)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    __syncthreads();
  }

  // 4. Wait for the producer of q_nope / q_pe / q_scale (no-op without PDL).
  pdl_wait();

  // 5. B fragments: b0 = q[m][16s+2t .. +1], b1 = q[m][16s+8+2t .. +1],
  //    m = 8*jt + g (zero for m >= M).
  uint32_t bfrag[MT][8][2];
#pragma unroll
  for (int jt = 0; jt < MT; ++jt) {
    const int m = 8 * jt + g;
    if (m < M) {
      const uint16_t* q = p.q_nope + (static_cast<size_t>(m) * H + h) * kNope + 2 * t;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        bfrag[jt][s][0] = ld_u32(q + 16 * s);
        bfrag[jt][s][1] = ld_u32(q + 16 * s + 8);
      }
    } else {
#pragma unroll
      for (int s = 0; s < 8; ++s) bfrag[jt][s][0] = bfrag[jt][s][1] = 0u;
    }
  }
  float qs = 1.f;
  if constexpr (OD == kOutE4M3) qs = *p.q_scale;

  if constexpr (WF == kWeightBF16) {
    const bool ok = mbar_wait_bounded(s_bar, 0, p.wait_limit_ns);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      if (lane == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
      return;
    }
  }

  // 6. Contraction.  Lane L addresses row (L & 7) of 8x8 matrix L >> 3:
  //    matrices 0/1 = k 16s..16s+7, 2/3 = k 16s+8..+15; 0/2 = columns
  //    16w..16w+7, 1/3 = 16w+8..+15 -- the A fragment order of m16n8k16.
  float acc[MT][4];
#pragma unroll
  for (int jt = 0; jt < MT; ++jt) acc[jt][0] = acc[jt][1] = acc[jt][2] = acc[jt][3] = 0.f;
  const int mi = lane >> 3;
  const int chunk = 2 * warp + (mi & 1);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int k = 16 * s + 8 * (mi >> 1) + (lane & 7);
    uint32_t a[4];
    ldmatrix_x4_trans(a, s_a + sw128(k, chunk));
#pragma unroll
    for (int jt = 0; jt < MT; ++jt) mma_bf16_16816(acc[jt], a, bfrag[jt][s][0], bfrag[jt][s][1]);
  }

  // 7. Epilogue.  D rows g / g+8 are columns n_cta+16w+g / +8, columns 2t,
  //    2t+1 are tokens.  After movmatrix.trans a lane holds token 8jt+g and
  //    columns 16w+2t, +1 (first block) and 16w+8+2t, +1 (second block).
#pragma unroll
  for (int jt = 0; jt < MT; ++jt) {
    const uint32_t r0 = movmatrix_trans(pack_bf16x2(acc[jt][1], acc[jt][0]));
    const uint32_t r1 = movmatrix_trans(pack_bf16x2(acc[jt][3], acc[jt][2]));
    const int m = 8 * jt + g;
    if (m < M) {
      const size_t off =
          static_cast<size_t>(m) * p.out_row_stride + static_cast<size_t>(h) * kOutDim + n_cta + 16 * warp + 2 * t;
      if constexpr (OD == kOutBF16) {
        uint16_t* o = reinterpret_cast<uint16_t*>(p.out) + off;
        *reinterpret_cast<uint32_t*>(o) = r0;
        *reinterpret_cast<uint32_t*>(o + 8) = r1;
      } else {
        uint8_t* o = p.out + off;
        *reinterpret_cast<uint16_t*>(o) =
            static_cast<uint16_t>(pack_e4m3x2(__fdiv_rn(bf16_hi(r0), qs), __fdiv_rn(bf16_lo(r0), qs)));
        *reinterpret_cast<uint16_t*>(o + 8) =
            static_cast<uint16_t>(pack_e4m3x2(__fdiv_rn(bf16_hi(r1), qs), __fdiv_rn(bf16_lo(r1), qs)));
      }
    }
  }

  // 8. Append q_pe: 16-byte chunks (8 elements) spread over the head's CTAs.
  const int nchunks = M * (kRope / 8);
  for (int c = tile * kThreads + tid; c < nchunks; c += kTilesPerHead * kThreads) {
    const int m = c >> 3;
    const int part = c & 7;
    const uint4 x = ld_u128(p.q_pe + (static_cast<size_t>(m) * H + h) * kRope + 8 * part);
    const size_t off =
        static_cast<size_t>(m) * p.out_row_stride + static_cast<size_t>(h) * kOutDim + kLatent + 8 * part;
    if constexpr (OD == kOutBF16) {
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + off) = x;
    } else {
      const uint32_t in[4] = {x.x, x.y, x.z, x.w};
      uint32_t w[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t a = in[2 * i], b = in[2 * i + 1];
        const uint32_t lo = pack_e4m3x2(__fdiv_rn(bf16_hi(a), qs), __fdiv_rn(bf16_lo(a), qs));
        const uint32_t hi = pack_e4m3x2(__fdiv_rn(bf16_hi(b), qs), __fdiv_rn(bf16_lo(b), qs));
        w[i] = lo | (hi << 16);
      }
      *reinterpret_cast<uint2*>(p.out + off) = make_uint2(w[0], w[1]);
    }
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
