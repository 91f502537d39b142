// V up-projection for larger token counts (65 <= M <= 256) on the
// 5th-generation tensor cores of sm_103a, with the contraction split over a
// thread-block cluster:
//
//   out[m,h,d] = bf16_rne( sum_{c<512} x[m,h,c] * W_UV[h,c,d] )    d < 128
//
// (the step after attention that the pages name as the downstream V
// up-projection, vLLM PR #174 "Fuse MXFP8 and BF16 MLA query assembly",
// section Safety scope; weight formats as on the query side, section What).
//
// Tiling: CTA (kc, h, z) owns contraction rows [128*kc, 128*kc+128) of head
// h, all 128 output columns, and tokens [TT*z, TT*z+TT).  The four kc CTAs
// of one (h, z) form a cluster.  Each runs one UMMA chain of shape M=128
// (output columns) x N=ntok (the chunk's tokens rounded up to 16) x K=128:
//     A = W_UV rows of the slice, MN-major (output columns contiguous),
//         128B swizzle: two TMA boxes of 64 columns x 128 rows;
//     B = the chunk's x rows restricted to the slice, K-major, 128B swizzle;
//     D = FP32 [128 lanes x ntok columns] in TMEM.
//
// Token row m of the chunk belongs to CTA m mod 4.  Straight from TMEM, each
// CTA pushes its partial sums of every row into the owner's receive buffer
// (one slot per source CTA) with st.async, which also counts the bytes on
// the owner's receive mbarrier, and ends with a status word; the owner
// waits on that barrier alone, then adds the four partials of its rows from
// local shared memory in the fixed order kc = 0, 1, 2, 3, rounds to BF16 and
// stores 8 bytes per thread.  The only cluster-wide barrier (every receive
// mbarrier initialised before any push) is split: arrive at kernel entry,
// wait just before the first push, so its latency hides behind the weight
// copy, the dependency wait and the MMAs.  Measured on GB300, a full
// cluster barrier costs ~0.6 us inside a dependent-launch chain.
//
// Every weight byte is read once from HBM (the four CTAs of a cluster read
// disjoint slices; a head's second token chunk finds its slices in L2), and
// every x byte once; no global scratch is used.
//
// Failure handling: every mbarrier wait is bounded.  A CTA that gives up
// records the timeout and still passes the cluster barrier and pushes all
// its bytes (zeros) with a failure status, so no owner waits for bytes that
// never come and every CTA stays resident until all bytes meant for it have
// arrived (there is no early return in this kernel); an owner that sees a
// failed source writes nothing.  Tensor memory is allocated after
// griddepcontrol.wait and freed before the receive wait.

#pragma once

#include "mlaqp_kernel_large.cuh"
#include "mlaqp_v_up_kernel.cuh"

namespace mlaqp {

constexpr int kVLargeSplit = 4;                       // cluster size: contraction slices per (h, chunk)
constexpr int kVLargeK = kLatent / kVLargeSplit;      // 128 contraction rows per CTA
constexpr int kVLargeThreads = 256;

// Shared memory layout (offsets from a 1024-byte aligned base).  The E4M3
// bytes of an MXFP8 tile share the x region (dequantised before the
// dependency wait).  The receive buffer has a region of its own: peers may
// push into it while this CTA's MMAs still read A and B.
struct VLargeSmem {
  int a;          // BF16 W_UV slice: two [128][64] halves, 128B swizzle
  int b;          // x slice: two [TT][64] BF16 k-slices, 128B swizzle
  int raw;        // MXFP8 only: E4M3 [2][128][64] as copied (= b)
  int recv;       // FP32 partial sums of this CTA's rows: [4 sources][TT/4 rows][128]
  int scale;      // MXFP8 only: E8M0 [128][4] of the slice
  int bar;        // three mbarriers: weights, MMA completion, receive
  int tmem_slot;  // TMEM base address written by tcgen05.alloc
  int status;     // [4 sources]: 0 = that source's partials were pushed, 1 = it gave up
  int bytes;      // total, with slack for the 1024-byte alignment
};

__host__ __device__ constexpr VLargeSmem v_large_smem_layout(int TT, bool mx) {
  VLargeSmem s{};
  s.a = 0;
  s.b = s.a + 2 * kVLargeK * 128;
  s.raw = s.b;
  const int bx = TT * kVLargeK * 2;
  const int braw = mx ? 2 * kVLargeK * 64 : 0;
  s.recv = s.b + (bx > braw ? bx : braw);
  s.scale = s.recv + TT * kVDim * 4;
  s.bar = s.scale + (mx ? kVLargeK * kVScaleRow : 0);
  s.tmem_slot = s.bar + 32;
  s.status = s.tmem_slot + 16;
  s.bytes = s.status + 16 + 1024;
  return s;
}

// ---------------------------------------------------------------------------
// Cluster helpers (documented PTX only)
// ---------------------------------------------------------------------------

// Address of the same shared-memory offset in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

// Cluster barrier of all threads of all CTAs, in split form: arrive without
// ordering anything but the fence issued before it; wait with acquire.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// 4 bytes into a peer's shared memory; completes 4 bytes of the transaction
// count of the peer's mbarrier `bar` (both cluster addresses of that peer).
__device__ __forceinline__ void st_async_u32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(addr), "r"(v),
               "r"(bar)
               : "memory");
}

// One test, with cluster-scope acquire, of a barrier phase that peers
// complete (their st.async writes are visible once it returns true).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for that phase, as mbar_wait_bounded.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// The kernel.  Grid (4, H, ceil(M/TT)), cluster (4, 1, 1), 256 threads.
// ---------------------------------------------------------------------------

// EARLY = 1: the next kernel may launch at entry instead of after the TMEM
// allocation (the caller's opt-in, as for the tcgen05 query kernel).
template <int WF, int TT, int EARLY = 0>
__global__ void __launch_bounds__(kVLargeThreads) mlaqp_v_up_large_kernel(const __grid_constant__ VUpParams p) {
  if constexpr (EARLY) pdl_launch_dependents();
  constexpr int K = kVLargeK;
  static_assert(TT % 16 == 0 && TT <= 128 && (TT * K / 8) % kVLargeThreads == 0, "token tile");
  constexpr VLargeSmem L = v_large_smem_layout(TT, WF == kWeightMXFP8);
  constexpr int KS = K / 16;                      // UMMA k-steps (8)
  constexpr int KC = K / 8;                       // 16-byte chunks of an x row slice (16)
  constexpr int XI = TT * KC / kVLargeThreads;    // x chunks per thread
  constexpr int kGroups = kVLargeThreads / 128;   // warp groups spanning the 128 TMEM lanes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int kc = blockIdx.x;  // contraction slice = rank in the (4, 1, 1) cluster
  const int h = blockIdx.y;
  const int m0 = blockIdx.z * TT;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int rows = min(TT, p.M - m0);  // >= 1: the grid has ceil(M/TT) chunks
  const int ntok = (rows + 15) & ~15;
  const uint32_t ncols = tmem_cols_for(ntok);
  const int k0 = kc * K;
  const uint32_t s_a = smem_u32(smem + L.a);
  const uint32_t s_b = smem_u32(smem + L.b);
  const uint32_t bar_w = smem_u32(smem + L.bar);
  const uint32_t bar_mma = bar_w + 8;
  const uint32_t bar_recv = bar_w + 16;
  // Bytes pushed into this CTA by its three peers: ntok/4 rows of 128 FP32
  // values and one status word each.
  const uint32_t recv_tx = static_cast<uint32_t>(3 * ((ntok / 4) * kVDim * 4 + 4));
  const uint16_t* xs = p.x + m0 * p.x_ts + h * p.x_hs + k0;

  // 1. Weight (and scale) stream: two TMA boxes of 64 columns x 128 rows.
  if (tid == 0) {
    prefetch_tensormap(&p.wmap);
    mbar_init(bar_w, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_recv, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar_recv, recv_tx);
    const int row = h * kLatent + k0;
    if constexpr (WF == kWeightBF16) {
      mbar_arrive_expect_tx(bar_w, 2 * K * 128 + p.extra_tx);
      tma_load_2d(s_a, &p.wmap, 0, row, bar_w);
      tma_load_2d(s_a + K * 128, &p.wmap, 64, row, bar_w);
    } else {
      const uint32_t s_raw = smem_u32(smem + L.raw);
      mbar_arrive_expect_tx(bar_w, 2 * K * 64 + K * kVScaleRow + p.extra_tx);
      tma_load_2d(s_raw, &p.wmap, 0, row, bar_w);
      tma_load_2d(s_raw + K * 64, &p.wmap, 64, row, bar_w);
      bulk_load_1d(smem_u32(smem + L.scale), p.weight_scale + static_cast<size_t>(row) * kVScaleRow, K * kVScaleRow,
                   bar_w);
    }
  }
  // 2. Warm L2 with the chunk's x rows (two 128-byte lines per row slice).
  if (tid < 2 * rows) prefetch_l2(xs + (tid >> 1) * p.x_ts + 64 * (tid & 1));
  __syncthreads();  // barriers initialised before anyone waits on them
  cluster_arrive_relaxed();  // ... and, once every CTA has arrived, before any peer pushes

  // 3. MXFP8: dequantise both 64-column halves into the swizzled BF16 tile
  //    (value = code * 2^(x-127) as two exact power-of-two factors).  Job
  //    (half, row k, chunk c of 8 columns): 2048 jobs, 8 per thread.
  bool ok = true;  // uniform across the CTA
  if constexpr (WF == kWeightMXFP8) {
    const bool got = mbar_wait_bounded(bar_w, 0, p.wait_limit_ns);
    ok = !__syncthreads_or(!got);
    if (ok) {
      const uint8_t* raw = smem + L.raw;
      const uint8_t* sc = smem + L.scale;
      const int c = tid & 7;
#pragma unroll 4
      for (int i = 0; i < 16 * K / kVLargeThreads; ++i) {
        const int r = (tid >> 3) + (kVLargeThreads / 8) * i;  // half * K + k
        const int half = r >= K ? 1 : 0;
        const int k = r - half * K;
        const uint2 v = *reinterpret_cast<const uint2*>(raw + r * 64 + 8 * c);
        const uint32_t x = sc[k * kVScaleRow + (64 * half + 8 * c) / kMxBlock];
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
    }
    __syncthreads();  // every E4M3 byte read before the x rows overwrite them
  }

  // 4. Wait for the producer of x (no-op without PDL).
  pdl_wait();

  // 5. The chunk's x rows of this slice (rows >= `rows` zero), all loads in
  //    flight at once; the TMEM allocation overlaps them, then the next
  //    kernel may launch.
  uint4 xv[XI];
#pragma unroll
  for (int i = 0; i < XI; ++i) {
    const int c = tid + kVLargeThreads * i;
    const int m = c / KC;
    xv[i] = make_uint4(0u, 0u, 0u, 0u);
    if (m < rows) xv[i] = ld_u128(xs + m * p.x_ts + 8 * (c % KC));
  }
  if (warp == 0) tmem_alloc(smem_u32(smem + L.tmem_slot), ncols);
  if constexpr (!EARLY) pdl_launch_dependents();

  // 6. x into the B tile: k slice j of row m, 16-byte chunk cc at
  //    j*TT*128 + m*128 + 16*(cc ^ m%8).
#pragma unroll
  for (int i = 0; i < XI; ++i) {
    const int c = tid + kVLargeThreads * i;
    const int kq = c % KC;
    *reinterpret_cast<uint4*>(smem + L.b + (kq >> 3) * (TT * 128) + sw128(c / KC, kq & 7)) = xv[i];
  }
  fence_proxy_async_smem();
  bool wok = true;
  if constexpr (WF == kWeightBF16) wok = mbar_wait_bounded(bar_w, 0, p.wait_limit_ns);
  tc_fence_before();
  const bool w_fail = __syncthreads_or(!wok);
  tc_fence_after();
  ok = ok && !w_fail;
  const uint32_t taddr = *reinterpret_cast<volatile uint32_t*>(smem + L.tmem_slot);

  // 7. One thread issues the K/16 MMAs and commits them to bar_mma.
  if (ok && tid == 0) {
    const uint32_t idesc = idesc_bf16_f32(kVDim, ntok);
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      // A: k rows 16s..16s+15 = two 8-row core groups 1024 B apart (SBO);
      //    the second 64-column half is K*128 bytes further (LBO).
      const uint64_t ad = smem_desc_sw128(s_a + s * 2048, K * 128, 1024);
      // B: k slice s/4, 32-byte step s%4 inside its 128-byte rows.
      const uint64_t bd = smem_desc_sw128(s_b + (s >> 2) * (TT * 128) + (s & 3) * 32, 16, 1024);
      umma_bf16(taddr, ad, bd, idesc, s > 0 ? 1u : 0u);
    }
    umma_commit(bar_mma);
  }

  // 8. Wait for the accumulator, then push it: warp w reads TMEM lanes
  //    32*(w%4).. (output column 32*(w%4) + lane), the warp groups take the
  //    16-token column chunks in turn; token t = 16*c16 + i goes to CTA
  //    t mod 4 = i mod 4, row t/4 of the slot of source kc (a local store
  //    when that is this CTA).  One store instruction of a warp writes 128
  //    contiguous bytes of one peer.  A CTA that gave up pushes zeros.
  if (ok) {
    const bool done = mbar_wait_bounded(bar_mma, 0, p.wait_limit_ns);
    tc_fence_after();
    ok = !__syncthreads_or(!done);
  }
  const uint32_t s_recv = smem_u32(smem + L.recv);
  const uint32_t s_status = smem_u32(smem + L.status);
  float* recv = reinterpret_cast<float*>(smem + L.recv);
  uint32_t* status = reinterpret_cast<uint32_t*>(smem + L.status);
  cluster_wait();  // every peer's receive barrier is initialised
  {
    const int quarter = warp & 3;
    const int col = 32 * quarter + lane;
    const uint32_t slot = static_cast<uint32_t>((kc * (TT / 4) * kVDim + col) * 4);
    uint32_t dst[kVLargeSplit], rbar[kVLargeSplit];
#pragma unroll
    for (int r = 0; r < kVLargeSplit; ++r) {
      dst[r] = cluster_map(s_recv + slot, r);
      rbar[r] = cluster_map(bar_recv, r);
    }
    for (int c16 = warp >> 2; c16 < ntok / 16; c16 += kGroups) {
      uint32_t r[16];
      if (ok) {
        tmem_ld16(taddr + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(16 * c16), r);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = 0u;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int row = 4 * c16 + (i >> 2);
        if ((i & 3) == kc) {
          recv[(kc * (TT / 4) + row) * kVDim + col] = __uint_as_float(r[i]);
        } else {
          st_async_u32(dst[i & 3] + static_cast<uint32_t>(row * kVDim * 4), r[i], rbar[i & 3]);
        }
      }
    }
  }
  if (tid < kVLargeSplit) {
    if (tid == kc) {
      status[kc] = ok ? 0u : 1u;
    } else {
      st_async_u32(cluster_map(s_status + 4 * kc, tid), ok ? 0u : 1u, cluster_map(bar_recv, tid));
    }
  }
  if (tid == 0 && !ok) atomicOr(&g_device_status, kDevStatusWaitTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, ncols);

  // 9. Wait for the peers' pushes (the local ones are visible after the CTA
  //    barrier above).  CTA kc owns token rows m = kc, kc+4, ...; thread item
  //    (row j, q) adds output columns 4q..4q+3 of the four sources and stores
  //    them as four BF16 values.
  //    A CTA must not exit while a peer may still push into its shared
  //    memory.  Before pushing, a peer spends at most two bounded waits
  //    (weights, MMA commit) of wait_limit_ns each, so the receive wait is
  //    bounded by three of them plus a quarter: a live peer has always
  //    pushed (and its bytes have landed) before this CTA gives up.
  const unsigned long long recv_limit_ns = 3ull * p.wait_limit_ns + (p.wait_limit_ns >> 2);
  const bool got = mbar_wait_bounded_cluster(bar_recv, 0, recv_limit_ns);
  if (__syncthreads_or(!got)) {
    if (tid == 0) atomicOr(&g_device_status, kDevStatusWaitTimeout);
  } else if ((status[0] | status[1] | status[2] | status[3]) == 0u) {
    for (int i = tid;; i += kVLargeThreads) {
      const int j = i >> 5;
      const int m = kc + kVLargeSplit * j;
      if (m >= rows) break;
      const int q = i & 31;
      float4 s = *reinterpret_cast<const float4*>(recv + j * kVDim + 4 * q);
#pragma unroll
      for (int r = 1; r < kVLargeSplit; ++r) {
        const float4 v = *reinterpret_cast<const float4*>(recv + (r * (TT / 4) + j) * kVDim + 4 * q);
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
      }
      uint16_t* o = p.out + static_cast<size_t>(m0 + m) * p.out_row_stride + h * kVDim + 4 * q;
      *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(s.y, s.x), pack_bf16x2(s.w, s.z));
    }
  }
}

}  // namespace mlaqp
