// Host side of the C ABI declared in include/mlaqp.h: argument validation,
// capability gating, prewarm and the single kernel launch per layer call.
//
// The run path allocates nothing, never synchronises and issues exactly one
// cudaLaunchKernelExC on the caller's stream, so it can be captured into a
// CUDA graph (SparkInfer PR #75, section Validation: CUDA-graph replay with
// mutated inputs; vLLM PR #174, section Performance evidence: no extra
// hot-path synchronisation).

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "mlaqp.h"
#include "mlaqp_dispatch.h"
#include "mlaqp_kernel.cuh"
#include "mlaqp_kernel_large.cuh"
#include "mlaqp_kernel_warp.cuh"
#include "mlaqp_v_up_kernel.cuh"
#include "mlaqp_v_up_kernel_large.cuh"
#include "mlaqp_v_up_kernel_mc.cuh"

namespace {

// Diagnostic: a kernel with no work but the programmatic-launch protocol
// (trigger, dependency wait), to measure the floor a chain of dependent
// launches costs on this GPU.
__global__ void mlaqp_null_kernel() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// L2 warm-up of one layer's weights: CTA b asks the TMA unit of its SM to
// fetch bytes [b*chunk, (b+1)*chunk) of the weights (then the scales) into
// L2; nothing waits for the data.  It reads only the weights, so it lets the
// next kernel launch at once; it still waits for the previous kernel before
// it exits, because a later kernel's dependency wait covers only the kernel
// launched just before it: were this one to finish first, that wait would
// no longer imply that the kernels before it (the producer of q_nope, say)
// have finished.
__global__ void mlaqp_prefetch_kernel(const uint8_t* w, unsigned long long w_bytes, const uint8_t* sc,
                                      unsigned long long sc_bytes, unsigned int chunk) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    const unsigned long long w_chunks = (w_bytes + chunk - 1) / chunk;
    const unsigned long long b = blockIdx.x;
    const uint8_t* base = b < w_chunks ? w : sc;
    const unsigned long long total = b < w_chunks ? w_bytes : sc_bytes;
    const unsigned long long off = (b < w_chunks ? b : b - w_chunks) * chunk;
    if (off < total) {
      const unsigned long long n = total - off < chunk ? total - off : chunk;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + off), "r"(static_cast<unsigned>(n))
                   : "memory");
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

using mlaqp::KernelInfo;
using mlaqp::RunParams;

thread_local std::string g_last_error;

int fail(int status, const std::string& msg) {
  g_last_error = msg;
  return status;
}

int fail_cuda(const char* what, cudaError_t e) {
  return fail(MLAQP_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + ": " + cudaGetErrorString(e));
}

bool supported_heads(int h) { return h == 8 || h == 11 || h == 16; }

constexpr int kMaxDevices = 64;

// Per-device facts the launch policy needs, queried once.
struct DeviceInfo {
  std::atomic<int> state{0};  // 0 = not yet queried, 1 = sm_103 and set up, 2 = another architecture
  int smem_per_sm = 0;        // bytes of shared memory per SM
  int reserved_per_block = 0; // bytes the driver reserves per resident CTA
  int max_smem_optin = 0;     // largest dynamic shared memory a CTA may request
  int sm_count = 0;           // streaming multiprocessors
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;
// Bit (wf*2+od)*4 + (mt-1) set once that decode specialisation's images are
// loaded; bit 16 + wf*2+od for the M > 32 kernels (tcgen05 and the
// 32-token chunked CTA-tile form).
std::atomic<uint32_t> g_prewarmed[kMaxDevices];
std::mutex g_prewarm_mutex;

int resolve_device(int device, int* out) {
  if (device < 0) {
    const cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  }
  if (device >= kMaxDevices) return fail(MLAQP_ERR_UNSUPPORTED, "device ordinal out of range");
  *out = device;
  return MLAQP_OK;
}

// Raises every kernel's dynamic-shared-memory limit to what the launch
// policy may request on this device (current device must be `device`).
int setup_kernels(const DeviceInfo& d);

// MLAQP_OK if `device` is an sm_103 GPU (and its kernels are set up), else
// an error status + message.  The first call per device queries it and
// sets kernel attributes; it synchronises nothing and launches nothing.
int check_device(int device) {
  DeviceInfo& d = g_dev[device];
  int state = d.state.load(std::memory_order_acquire);
  if (state == 0) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    state = d.state.load(std::memory_order_acquire);
    if (state == 0) {
      int major = 0, minor = 0;
      cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.reserved_per_block, cudaDevAttrReservedSharedMemoryPerBlock, device);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
      if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute", e);
      state = (major == 10 && minor == 3) ? 1 : 2;
      if (state == 1) {
        int prev = -1;
        e = cudaGetDevice(&prev);
        if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
        if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return fail_cuda("cudaSetDevice", e);
        const int st = setup_kernels(d);
        if (prev != device) cudaSetDevice(prev);
        if (st != MLAQP_OK) return st;
      }
      d.state.store(state, std::memory_order_release);
    }
  }
  if (state != 1) return fail(MLAQP_ERR_UNSUPPORTED, "device is not an sm_103 (GB300) GPU");
  return MLAQP_OK;
}

// Default bound on every in-kernel mbarrier wait: far above any real copy
// latency, short enough that a lost completion surfaces as an error.
constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library needs no link-time dependency on libcuda.
EncodeTiledFn encode_tiled_fn(std::string* err) {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  static std::string init_err;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || ptr == nullptr)
      init_err = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorString(e);
    else
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  if (!fn) *err = init_err;
  return fn;
}

// 2-D tensor map over W_UK_T viewed as [H*K rows][512 columns]; one box is
// K rows x box_cols columns: the 64-column tile of a CTA of the CTA-tile
// kernels (BF16 128B-swizzled, the layout their ldmatrix addressing
// expects; E4M3 unswizzled), or the 16-column tile of a warp of the
// warp-tile kernel (BF16: 32-byte rows with the 32B swizzle; E4M3:
// unswizzled 16-byte rows).
int encode_weight_map(CUtensorMap* map, const void* weight, int H, int K, bool mx, int box_cols, bool swizzle,
                      bool swizzle32 = false) {
  std::string err;
  EncodeTiledFn fn = encode_tiled_fn(&err);
  if (!fn) return fail(MLAQP_ERR_CUDA, err);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(MLAQP_LATENT_DIM), static_cast<cuuint64_t>(H) * K};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(MLAQP_LATENT_DIM) * (mx ? 1 : 2)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(K)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(weight), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B
                                : (swizzle32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLAQP_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return MLAQP_OK;
}

// Launch policy of one call: where a PDL-launched CTA lets the next kernel
// start (see the kernel) and an optional cap on resident CTAs per SM,
// imposed by padding the dynamic shared memory.  Chosen from per-layer times
// of 128-layer CUDA-graph chains on GB300 (H = 16): the query kernel
// triggers at entry with at most 2 CTAs per SM at every M.  One layer then
// runs ahead with its weight copy (and MXFP8 dequantisation) overlapped,
// while no SM holds more than one early-launched CTA next to the running
// one.  Against the earlier mix (cap 3 up to M = 8, MXFP8 uncapped up to
// M = 4, trigger after the wait above M = 16), MXFP8->E4M3 went from
// 1.62 / 1.82 / 2.84 us to 1.38 / 1.52 / 2.54 us at M = 1 / 8 / 32.  The
// exception is BF16 weights with E4M3 output at M = 17..32, which trigger
// after the wait (2.16 against 2.61 us at M = 32).  The V up-projection
// (x-multicast kernel from M = 9) likewise triggers after the wait for BF16
// weights at 17 <= M <= 32 (2.12 against 2.37 us at M = 32), and drops the
// cap for MXFP8 weights above M = 32 (2.83 against 2.97 us at M = 64).
struct LaunchPolicy {
  int trig;     // 0 entry, 1 after the wait, 2 weights ready
  int cta_cap;  // 0: none, else resident CTAs per SM
};

// Smallest CTA cap any policy uses (the largest padded shared memory).
constexpr int kMinCtaCap = 2;

// Measurement override of the mma.sync kernels' launch policy
// (mlaqp_debug_set_policy): trig < 0 means none.
std::atomic<int> g_policy_trig{-1};
std::atomic<int> g_policy_cap{0};

LaunchPolicy launch_policy(int weight_format, int out_dtype, int M) {
  const int trig = g_policy_trig.load(std::memory_order_relaxed);
  if (trig >= 0) return LaunchPolicy{trig, g_policy_cap.load(std::memory_order_relaxed)};
  if (weight_format == MLAQP_WEIGHT_BF16 && out_dtype == MLAQP_OUT_E4M3 && M > 16 && M <= 32) return LaunchPolicy{1, 0};
  return LaunchPolicy{0, 2};
}

LaunchPolicy v_up_launch_policy(int weight_format, int M) {
  if (M > 32) return LaunchPolicy{0, weight_format == MLAQP_WEIGHT_BF16 ? 2 : 0};  // two 32-token chunks
  if (weight_format == MLAQP_WEIGHT_BF16 && M > 16) return LaunchPolicy{1, 0};
  return LaunchPolicy{0, 2};
}

// Dynamic shared memory that realises `cap` CTAs per SM for a kernel that
// needs `base` bytes.
int smem_for_cap(const DeviceInfo& d, int base, int cap) {
  if (cap <= 0) return base;
  const int bytes = d.smem_per_sm / cap - d.reserved_per_block;
  return bytes > base ? (bytes < d.max_smem_optin ? bytes : d.max_smem_optin) : base;
}


// Index of a supported nope dim in the kernel tables, or -1.
int nope_index(int K) {
  for (int i = 0; i < 2; ++i)
    if (mlaqp::kNopeDims[i] == K) return i;
  return -1;
}

// Above M = 32 the CTA-tile kernel runs in 32-token chunks (grid.z; the
// later chunks find the weight tile in L2) instead of the tcgen05 kernel:
// always up to M = 64, and up to kCtaMaxM while all its CTAs fit on the GPU
// at two, three or (nope dim 128) four per SM (cta_chunk_cap).  It needs no
// tensor memory, so it may trigger the next launch at entry.  Measured on GB300 (128/256-layer PDL chains, pdl = 1, us
// per layer call, tcgen05 / chunked): H = 16, BF16->BF16 2.43 / 2.08 at
// M = 33 and 2.51 / 2.28 at 64; MXFP8->E4M3 3.22 / 2.43 and 3.34 / 2.52;
// BF16->E4M3 2.46 / 2.12 and 2.55 / 2.27 (entry trigger, cap 2; after-wait
// trigger 2.68 / 2.74).  H = 8 (four chunks, 256 CTAs), M = 128: BF16->BF16
// 2.83 / 2.09, MXFP8->E4M3 3.27 / 2.39.  H = 16 with three or four chunks
// (384-512 CTAs, more than fit): 3.6-4.7 against 2.8-3.5.
constexpr int kCtaMaxM = MLAQP_MAX_M;
constexpr int kCtaAlwaysM = 64;

int cta_chunks(int M) { return (M + mlaqp::kMaxM - 1) / mlaqp::kMaxM; }

// CTAs per SM a chunked launch is capped at: 2 while its 8*H*chunks CTAs fit
// at two per SM, else 3 while they fit at three (H = 16, M = 65..96: BF16
// 2.42-2.52 us against 2.90 on tcgen05, MXFP8->E4M3 2.80-2.86 against
// 3.24-3.28); 0 when they do not fit at all (then the tcgen05 kernel runs;
// four chunks at H = 16 and cap 3 measured 4.0-4.6 us).  Above M = 128
// only H = 8 (to 224 tokens, up to 448 CTAs) and H = 11 (to 160) fit:
// H = 8, M = 192: BF16 3.64 / 2.42, MXFP8->E4M3 3.60 / 2.78; H = 11,
// M = 160: 3.74 / 2.65 and 3.62 / 3.02 (tcgen05 / chunks).
// A fourth tier (nope dim 128: 60-62 registers, so four 256-thread CTAs fit
// an SM; at 192, 80 registers allow three) caps at 4: H = 16, M = 97..128:
// BF16->E4M3 2.90-2.99 / 2.70-2.78, MXFP8->E4M3 3.32-3.44 / 3.26-3.33;
// H = 11, M = 161..192: BF16->BF16 3.70 / 2.84-2.90; H = 8, M = 225..256:
// BF16->BF16 3.64-3.67 / 2.83-2.85, MXFP8->E4M3 3.59-3.67 / 3.28-3.33.
int cta_chunk_cap(int M, int H, int K, int sm_count) {
  if (M <= kCtaAlwaysM) return 2;
  if (M > kCtaMaxM) return 0;
  const int ctas = mlaqp::kTilesPerHead * H * cta_chunks(M);
  if (ctas <= 2 * sm_count) return 2;
  if (ctas <= 3 * sm_count) return 3;
  return K == MLAQP_NOPE_DIM && ctas <= 4 * sm_count ? 4 : 0;
}

bool cta_chunks_fit(int M, int H, int K, int sm_count) { return cta_chunk_cap(M, H, K, sm_count) != 0; }

// Tokens per chunk of a CTA-tile launch: 32 above M = 32; for 9 <= M <= 32
// with nope dim 128, 8 (M <= 16) or 16 (MXFP8 weights, M = 17..32) where
// the two chunks' 16*H CTAs fit one per SM (H = 8 on 152 SMs); else 0, one
// launch over all tokens.  Measured on GB300 (128/256-layer PDL chains, us
// per layer call, H = 8, current choice / two chunks): M = 16: BF16->BF16
// 1.47 / 1.35, MXFP8->E4M3 1.53 / 1.38, BF16->E4M3 1.51 / 1.37; M = 32:
// MXFP8->E4M3 1.67 / 1.53, MXFP8->BF16 1.60 / 1.51.  With BF16 weights at
// M = 17..32 the chunks tie or lose (1.60-1.63 against 1.55-1.61), and at
// H = 16 (256 CTAs, two per SM) they lose at every M (0.2-0.5 us).
int cta_chunk_len(int weight_format, int M, int H, int K, int sm_count) {
  if (M > mlaqp::kMaxM) return mlaqp::kMaxM;
  if (M <= 8 || K != MLAQP_NOPE_DIM || 2 * mlaqp::kTilesPerHead * H > sm_count) return 0;
  if (M <= 16) return 8;
  return weight_format == MLAQP_WEIGHT_MXFP8 ? 16 : 0;
}

int cta_form(int M, int chunk) {
  if (chunk == 32) return mlaqp::kChunkedForm;
  if (chunk == 16) return mlaqp::kChunked16Form;
  if (chunk == 8) return mlaqp::kChunked8Form;
  return (M + 7) / 8 - 1;
}

// chunk < 0: the chunk length of a launch that splits only above M = 32.
const KernelInfo* lookup(int weight_format, int out_dtype, int M, int trig, int nope_idx, int chunk = -1) {
  if (M < 1) return nullptr;
  const int form = cta_form(M, chunk < 0 ? (M > mlaqp::kMaxM ? mlaqp::kMaxM : 0) : chunk);
  const mlaqp::KernelTable& table =
      weight_format == MLAQP_WEIGHT_BF16 ? mlaqp::kernels_bf16_weights() : mlaqp::kernels_mxfp8_weights();
  return &table[nope_idx][out_dtype][form][trig];
}

// Token tile (tokens per CTA) of a large-M call, as an index into
// kLargeTokTiles: 32 up to M = 64 (twice the CTAs of a 64-token tile), 64 up
// to M = 128, 128 above (at most 2 chunks, so one CTA per SM at H = 16).
int large_tile_index(int M) { return M <= 64 ? 0 : M <= 128 ? 1 : 2; }

const KernelInfo* lookup_large(int weight_format, int out_dtype, int nope_idx, int tile_idx, int early = 0) {
  return &mlaqp::kernels_large_m()[nope_idx][tile_idx][weight_format][out_dtype][early];
}

// Chunks of one token tile in a large-M call (grid.z).
int large_chunks(int M) {
  const int tt = mlaqp::kLargeTokTiles[large_tile_index(M)];
  return (M + tt - 1) / tt;
}

// Dynamic shared memory for a tcgen05 kernel of `base` bytes whose CTAs
// hold tmem_cols_for(ntok) TMEM columns each: the layout's size, padded when
// needed so that the CTAs one SM can hold never ask for more than its 512
// columns between them.
int tmem_safe_smem(const DeviceInfo& d, int base, int ntok) {
  const int cols = static_cast<int>(mlaqp::tmem_cols_for(ntok));
  const int max_ctas = 512 / cols;
  if (d.smem_per_sm / (base + d.reserved_per_block) <= max_ctas) return base;
  const int bytes = d.smem_per_sm / (max_ctas + 1) - d.reserved_per_block + 1;
  return bytes < d.max_smem_optin ? bytes : d.max_smem_optin;
}

// Dynamic shared memory of a large-M launch (a CTA of the largest chunk
// needs tmem_cols_for(chunk) columns).
int large_smem(const DeviceInfo& d, int base, int M) {
  const int tt = mlaqp::kLargeTokTiles[large_tile_index(M)];
  const int chunk = M < tt ? M : tt;
  return tmem_safe_smem(d, base, (chunk + 15) & ~15);
}

int setup_kernels(const DeviceInfo& d) {
  for (int wf = 0; wf < 2; ++wf)
    for (int mt = 0; mt < 4; ++mt)
      for (int trig = 0; trig < 2; ++trig) {
        const KernelInfo& k = mlaqp::kernels_v_up()[wf][mt][trig];
        cudaError_t e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_for_cap(d, k.smem_bytes, kMinCtaCap));
        if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute", e);
        const KernelInfo& km = mlaqp::kernels_v_up_mc()[wf][mt][trig];
        e = cudaFuncSetAttribute(km.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_for_cap(d, km.smem_bytes, kMinCtaCap));
        if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute", e);
      }
  for (int ki = 0; ki < 2; ++ki)
    for (int ti = 0; ti < 3; ++ti)
      for (int wf = 0; wf < 2; ++wf)
        for (int od = 0; od < 2; ++od) {
          for (int early = 0; early < 2; ++early) {
            const cudaError_t e = cudaFuncSetAttribute(lookup_large(wf, od, ki, ti, early)->fn,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_smem_optin);
            if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute", e);
          }
        }
  for (int wf = 0; wf < 2; ++wf)
    for (int ti = 0; ti < 2; ++ti) {
      for (int early = 0; early < 2; ++early) {
        const cudaError_t e = cudaFuncSetAttribute(mlaqp::kernels_v_up_large()[wf][ti][early].fn,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_smem_optin);
        if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute", e);
      }
    }
  for (int wf = 0; wf < 2; ++wf) {
    const mlaqp::WarpKernelSet& set = wf == 0 ? mlaqp::kernels_warp_bf16_weights() : mlaqp::kernels_warp_mxfp8_weights();
    for (int ki = 0; ki < 2; ++ki)
      for (int od = 0; od < 2; ++od)
        for (int mt = 0; mt < 4; ++mt)
          for (int trig = 0; trig < 2; ++trig) {
            const KernelInfo& k = set.mma[ki][od][mt][trig];
            const cudaError_t e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       smem_for_cap(d, k.smem_bytes, 1));
            if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute", e);
          }
    for (int od = 0; od < 2; ++od)
      for (int trig = 0; trig < 2; ++trig) {
        const KernelInfo& k = set.fma[od][trig];
        const cudaError_t e = cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   smem_for_cap(d, k.smem_bytes, 1));
        if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute", e);
      }
  }
  const int smem = smem_for_cap(d, mlaqp::Smem<192>::Bytes, 1);  // any cap the policy (or its override) uses
  for (int ki = 0; ki < 2; ++ki)
    for (int wf = 0; wf < 2; ++wf)
      for (int od = 0; od < 2; ++od)
        for (int form = 0; form <= mlaqp::kChunked16Form; ++form)
          for (int trig = 0; trig < mlaqp::kTrigVariants; ++trig) {
            const mlaqp::KernelTable& table = wf == 0 ? mlaqp::kernels_bf16_weights() : mlaqp::kernels_mxfp8_weights();
            const KernelInfo* k = &table[ki][od][form][trig];
            const cudaError_t e = cudaFuncSetAttribute(k->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute", e);
          }
  return MLAQP_OK;
}

bool valid_enums(int weight_format, int out_dtype) {
  return (weight_format == MLAQP_WEIGHT_BF16 || weight_format == MLAQP_WEIGHT_MXFP8) &&
         (out_dtype == MLAQP_OUT_BF16 || out_dtype == MLAQP_OUT_E4M3);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

Range span(const void* p, size_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{lo, lo + bytes};
}

// One layer call's arguments (pointers as given by the caller, strides in
// elements).
struct RunArgs {
  const void* q_nope;
  int64_t q_nope_ts, q_nope_hs;
  const void* q_pe;
  int64_t q_pe_ts, q_pe_hs;
  const void* weight;
  const void* weight_scale;
  void* out;
  int64_t out_row_stride;
  const float* q_scale;
  int M, H, K, weight_format, out_dtype;
};

RunArgs contiguous_args(const void* q_nope, const void* q_pe, const void* weight, const void* weight_scale, void* out,
                        int64_t out_row_stride, const float* q_scale, int M, int H, int weight_format, int out_dtype) {
  return RunArgs{q_nope, static_cast<int64_t>(H) * MLAQP_NOPE_DIM, MLAQP_NOPE_DIM,
                 q_pe, static_cast<int64_t>(H) * MLAQP_ROPE_DIM, MLAQP_ROPE_DIM,
                 weight, weight_scale, out, out_row_stride, q_scale, M, H, MLAQP_NOPE_DIM, weight_format, out_dtype};
}

// Which kernel serves a layer call.  kAuto is the library's choice
// (auto_arm: the CTA-tile kernel, whole or in token chunks, the warp-tile
// kernel, or the tcgen05 kernel); the others force one form, for
// measurement (mlaqp_debug_run_arm).
enum class Arm : int { kAuto = 0, kWarpMma = 1, kWarpFma = 2, kCtaMma = 3, kTcgen05 = 4 };

// The library's kernel choice for a decode call (M <= 32), from 128-layer
// PDL chains of every M = 1..32, H in {8, 11, 16}, all four format pairs
// (GB300): the CTA-tile kernel up to the crossover, the warp-tile kernel
// from it.  Below it the CTA-tile kernel's spare SM slots let the next
// layer's CTAs start (and stream weights) earlier, which pays while a
// layer's post-wait work is small; above it the warp-tile kernel's one CTA
// per SM keeps any SM from carrying two CTAs' contraction and epilogue.
// Measured crossovers (first M from which the warp-tile kernel is faster),
// nope dim 128: M = 17 at H = 11 and 16 for every format pair; at H = 8,
// M = 13 (MXFP8 -> BF16, BF16 -> E4M3), 15 (BF16 -> BF16), 16 (MXFP8 ->
// E4M3).  Nope dim 192 (H = 16): the warp-tile kernel from M = 17, but for
// M = 25..32 (four token tiles, 12 k-steps) only with BF16 weights and E4M3
// output.  Above 32 tokens: the chunked CTA-tile kernel while its CTAs fit,
// else the tcgen05 kernel (cta_chunk_cap).
int warp_crossover(int weight_format, int out_dtype, int H) {
  if (H > 8) return 17;
  if (weight_format == MLAQP_WEIGHT_BF16) return out_dtype == MLAQP_OUT_BF16 ? 15 : 13;
  return out_dtype == MLAQP_OUT_BF16 ? 13 : 16;
}

// sm_count: the device's SM count (the chunk rules depend on it).
Arm auto_arm(int weight_format, int out_dtype, int M, int H, int K, int sm_count) {
  if (M > MLAQP_MAX_M_DECODE) return cta_chunks_fit(M, H, K, sm_count) ? Arm::kCtaMma : Arm::kTcgen05;
  if (cta_chunk_len(weight_format, M, H, K, sm_count) != 0) return Arm::kCtaMma;
  if (M < warp_crossover(weight_format, out_dtype, H)) return Arm::kCtaMma;
  if (K != MLAQP_NOPE_DIM && M > 24 && !(weight_format == MLAQP_WEIGHT_BF16 && out_dtype == MLAQP_OUT_E4M3))
    return Arm::kCtaMma;
  return Arm::kWarpMma;
}

// Grid of a warp-tile launch: one CTA per SM, but at least 8 CTAs per head
// (at most kWMaxTilesPerCta tiles per CTA) and at most 32 (one tile each);
// the kernel splits the CTAs over the heads as evenly as it goes.
void warp_grid(int sm_count, int H, int* ctas, int* tiles_per_cta) {
  const int min_g = H * ((mlaqp::kWTilesPerHead + mlaqp::kWMaxTilesPerCta - 1) / mlaqp::kWMaxTilesPerCta);
  const int max_g = H * mlaqp::kWTilesPerHead;
  const int g = sm_count < min_g ? min_g : (sm_count > max_g ? max_g : sm_count);
  *ctas = g;
  *tiles_per_cta = (mlaqp::kWTilesPerHead + g / H - 1) / (g / H);  // the fewest CTAs a head gets is g / H
}

const KernelInfo* lookup_warp(int weight_format, int out_dtype, int M, int trig, int nope_idx, bool fma) {
  const mlaqp::WarpKernelSet& set =
      weight_format == MLAQP_WEIGHT_BF16 ? mlaqp::kernels_warp_bf16_weights() : mlaqp::kernels_warp_mxfp8_weights();
  if (fma) return &set.fma[out_dtype][trig];
  return &set.mma[nope_idx][out_dtype][(M + 7) / 8 - 1][trig];
}

// Launch policy of the warp-tile kernel: trigger at entry, at most 2 CTAs per
// SM (with one CTA per SM per launch, a running layer and the next one each
// hold one slot of every SM).
LaunchPolicy warp_launch_policy(int /*weight_format*/, int /*out_dtype*/, int /*M*/) {
  const int trig = g_policy_trig.load(std::memory_order_relaxed);
  if (trig >= 0) return LaunchPolicy{trig, g_policy_cap.load(std::memory_order_relaxed)};
  return LaunchPolicy{0, 2};
}

// Everything a query call launches, decided from the arguments and the SM
// count alone (no device access): run_impl, mlaqp_launch_shape and the
// mlaqp_debug_plan test hook share it.  forced = Arm::kAuto: the library's
// choice.  Returns MLAQP_ERR_UNSUPPORTED when a forced form does not cover
// the call.
struct QueryPlan {
  Arm arm = Arm::kAuto;
  const KernelInfo* k = nullptr;
  LaunchPolicy pol{0, 0};  // mma.sync kernels: trigger point, CTA cap (applied with PDL)
  int chunk = 0;           // CTA-tile kernel: tokens per grid.z chunk (0: one launch over all tokens)
  int grid = 0;            // CTAs
  int threads = 0;         // threads per CTA
  int tiles_per_cta = 1;   // warp-tile kernel: column tiles per CTA
};

int plan_query(int weight_format, int out_dtype, int M, int H, int K, int pdl, Arm forced, int sm_count,
               QueryPlan* q) {
  *q = QueryPlan{};
  const int ki = nope_index(K);
  const Arm arm = forced == Arm::kAuto ? auto_arm(weight_format, out_dtype, M, H, K, sm_count) : forced;
  if (arm == Arm::kWarpFma && (M > 8 || K != 128))
    return fail(MLAQP_ERR_UNSUPPORTED, "the CUDA-core arm covers M <= 8 at nope_dim 128");
  if (arm == Arm::kWarpMma && M > MLAQP_MAX_M_DECODE)
    return fail(MLAQP_ERR_UNSUPPORTED, "the warp-tile arm covers M <= 32");
  if (arm == Arm::kCtaMma && M > kCtaMaxM) return fail(MLAQP_ERR_UNSUPPORTED, "the CTA-tile arm covers M <= 256");
  q->arm = arm;
  if (arm == Arm::kWarpMma || arm == Arm::kWarpFma) {
    q->pol = warp_launch_policy(weight_format, out_dtype, M);
    q->k = lookup_warp(weight_format, out_dtype, M, q->pol.trig, ki, arm == Arm::kWarpFma);
    warp_grid(sm_count, H, &q->grid, &q->tiles_per_cta);
    q->threads = q->k->threads * q->tiles_per_cta;
  } else if (arm == Arm::kTcgen05) {
    q->k = lookup_large(weight_format, out_dtype, ki, large_tile_index(M), pdl == 2 ? 1 : 0);
    q->grid = q->k->tiles_per_head * H * large_chunks(M);
    q->threads = q->k->threads;
  } else {
    q->pol = launch_policy(weight_format, out_dtype, M);
    if (M > MLAQP_MAX_M_DECODE && g_policy_trig.load(std::memory_order_relaxed) < 0)
      q->pol.cta_cap = cta_chunk_cap(M, H, K, sm_count);
    q->chunk = cta_chunk_len(weight_format, M, H, K, sm_count);
    q->k = lookup(weight_format, out_dtype, M, q->pol.trig, ki, q->chunk);
    q->grid = q->k->tiles_per_head * H * (q->chunk ? (M + q->chunk - 1) / q->chunk : 1);
    q->threads = q->k->threads;
  }
  return MLAQP_OK;
}

int launch_warp(const RunArgs& a, mlaqp_stream_t stream, int pdl, unsigned long long wait_limit_ns, unsigned extra_tx,
                const QueryPlan& q, int device) {
  const int M = a.M, H = a.H, K = a.K;
  const bool mx = a.weight_format == MLAQP_WEIGHT_MXFP8;
  const LaunchPolicy pol = q.pol;
  const KernelInfo* k = q.k;
  const int ctas = q.grid, tpc = q.tiles_per_cta;
  mlaqp::WarpRunParams params;
  int st = encode_weight_map(&params.wmap, a.weight, H, K, mx, mlaqp::kWTileCols, false, !mx);
  if (st != MLAQP_OK) return st;
  params.q_nope = static_cast<const uint16_t*>(a.q_nope);
  params.q_pe = static_cast<const uint16_t*>(a.q_pe);
  params.q_nope_ts = a.q_nope_ts;
  params.q_nope_hs = a.q_nope_hs;
  params.q_pe_ts = a.q_pe_ts;
  params.q_pe_hs = a.q_pe_hs;
  params.weight_scale = static_cast<const uint8_t*>(a.weight_scale);
  params.out = static_cast<uint8_t*>(a.out);
  params.out_row_stride = a.out_row_stride;
  params.q_scale = a.q_scale;
  params.wait_limit_ns = wait_limit_ns;
  params.extra_tx = extra_tx;
  params.M = M;
  params.H = H;
  params.inv_ctas = 1.0f / static_cast<float>(ctas);
  params.inv_heads = 1.0f / static_cast<float>(H);

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(k->threads * tpc), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_for_cap(g_dev[device], k->smem_bytes, pdl ? pol.cta_cap : 0));
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[1] = {&params};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, k->fn, args);
  if (e != cudaSuccess) return fail_cuda("cudaLaunchKernelExC", e);
  return MLAQP_OK;
}

// pdl: 0 = ordinary launch, 1 = programmatic dependent launch, 2 = the same
// with the tcgen05 kernel's next-kernel trigger at entry (the caller's
// opt-in under the tensor-memory contract stated in the header).
int run_impl(const RunArgs& a, mlaqp_stream_t stream, int pdl, unsigned long long wait_limit_ns, unsigned extra_tx,
             Arm forced = Arm::kAuto) {
  if (pdl < 0 || pdl > 2) return fail(MLAQP_ERR_INVALID_ARG, "pdl must be 0, 1 or 2");
  const int M = a.M, H = a.H, K = a.K;
  if (!valid_enums(a.weight_format, a.out_dtype)) return fail(MLAQP_ERR_INVALID_ARG, "unknown weight_format or out_dtype");
  if (M < 0) return fail(MLAQP_ERR_INVALID_ARG, "M must be >= 0");
  if (!supported_heads(H)) return fail(MLAQP_ERR_UNSUPPORTED, "num_heads must be 8, 11 or 16");
  if (M > MLAQP_MAX_M) return fail(MLAQP_ERR_UNSUPPORTED, "M must be <= 256");
  const int ki = nope_index(K);
  if (ki < 0) return fail(MLAQP_ERR_UNSUPPORTED, "nope_dim must be 128 or 192");
  if (M == 0) return MLAQP_OK;

  const bool mx = a.weight_format == MLAQP_WEIGHT_MXFP8;
  const bool e4m3 = a.out_dtype == MLAQP_OUT_E4M3;
  if (!a.q_nope || !a.q_pe || !a.weight || !a.out)
    return fail(MLAQP_ERR_INVALID_ARG, "q_nope, q_pe, weight and out are required");
  if (mx && !a.weight_scale) return fail(MLAQP_ERR_INVALID_ARG, "MXFP8 weights require weight_scale");
  if (!mx && a.weight_scale) return fail(MLAQP_ERR_INVALID_ARG, "BF16 weights take no weight_scale (pass NULL)");
  if (e4m3 && !a.q_scale) return fail(MLAQP_ERR_INVALID_ARG, "E4M3 output requires q_scale");
  if (!e4m3 && a.q_scale) return fail(MLAQP_ERR_INVALID_ARG, "BF16 output takes no q_scale (pass NULL)");
  if (!aligned(a.q_nope, 16) || !aligned(a.weight, 16) || !aligned(a.out, 16) ||
      (a.weight_scale && !aligned(a.weight_scale, 16)))
    return fail(MLAQP_ERR_INVALID_ARG, "q_nope, weight, weight_scale and out must be 16-byte aligned");
  if (!aligned(a.q_pe, 4) || (a.q_scale && !aligned(a.q_scale, 4)))
    return fail(MLAQP_ERR_INVALID_ARG, "q_pe and q_scale must be 4-byte aligned");
  if (a.q_nope_ts < 0 || a.q_nope_hs < 0 || a.q_pe_ts < 0 || a.q_pe_hs < 0)
    return fail(MLAQP_ERR_INVALID_ARG, "input strides must be >= 0");
  if (a.q_nope_ts % 8 != 0 || a.q_nope_hs % 8 != 0)
    return fail(MLAQP_ERR_INVALID_ARG, "q_nope strides must be multiples of 8 elements (16 bytes)");
  if (a.q_pe_ts % 2 != 0 || a.q_pe_hs % 2 != 0)
    return fail(MLAQP_ERR_INVALID_ARG, "q_pe strides must be multiples of 2 elements (4 bytes)");
  const int64_t out_elem = e4m3 ? 1 : 2;
  if (a.out_row_stride < static_cast<int64_t>(MLAQP_OUT_DIM) * H)
    return fail(MLAQP_ERR_INVALID_ARG, "out_row_stride must be >= 576*H elements");
  if ((a.out_row_stride * out_elem) % 16 != 0)
    return fail(MLAQP_ERR_INVALID_ARG, "out_row_stride * element size must be a multiple of 16 bytes");

  const size_t out_bytes = static_cast<size_t>(
      (static_cast<int64_t>(M - 1) * a.out_row_stride + static_cast<int64_t>(MLAQP_OUT_DIM) * H) * out_elem);
  const Range o = span(a.out, out_bytes);
  const size_t w_elems = static_cast<size_t>(H) * K * MLAQP_LATENT_DIM;
  const Range inputs[5] = {
      span(a.q_nope, static_cast<size_t>((M - 1) * a.q_nope_ts + (H - 1) * a.q_nope_hs + K) * 2),
      span(a.q_pe, static_cast<size_t>((M - 1) * a.q_pe_ts + (H - 1) * a.q_pe_hs + MLAQP_ROPE_DIM) * 2),
      span(a.weight, w_elems * (mx ? 1 : 2)),
      span(a.weight_scale, mx ? w_elems / 32 : 0),
      span(a.q_scale, e4m3 ? sizeof(float) : 0),
  };
  for (const Range& r : inputs)
    if (r.hi > r.lo && overlaps(o, r)) return fail(MLAQP_ERR_INVALID_ARG, "out overlaps an input tensor");

  int device = 0;
  int st = resolve_device(-1, &device);
  if (st != MLAQP_OK) return st;
  st = check_device(device);
  if (st != MLAQP_OK) return st;

  QueryPlan q;
  st = plan_query(a.weight_format, a.out_dtype, M, H, K, pdl, forced, g_dev[device].sm_count, &q);
  if (st != MLAQP_OK) return st;
  if (q.arm == Arm::kWarpMma || q.arm == Arm::kWarpFma) return launch_warp(a, stream, pdl, wait_limit_ns, extra_tx, q, device);

  const bool large = q.arm == Arm::kTcgen05;
  const KernelInfo* k = q.k;
  const int smem_bytes = large ? large_smem(g_dev[device], k->smem_bytes, M)
                               : smem_for_cap(g_dev[device], k->smem_bytes, pdl ? q.pol.cta_cap : 0);
  RunParams params;
  st = encode_weight_map(&params.wmap, a.weight, H, K, mx, mlaqp::kNTile, !mx);
  if (st != MLAQP_OK) return st;
  params.q_nope = static_cast<const uint16_t*>(a.q_nope);
  params.q_pe = static_cast<const uint16_t*>(a.q_pe);
  params.q_nope_ts = a.q_nope_ts;
  params.q_nope_hs = a.q_nope_hs;
  params.q_pe_ts = a.q_pe_ts;
  params.q_pe_hs = a.q_pe_hs;
  params.weight_scale = static_cast<const uint8_t*>(a.weight_scale);
  params.out = static_cast<uint8_t*>(a.out);
  params.out_row_stride = a.out_row_stride;
  params.q_scale = a.q_scale;
  params.wait_limit_ns = wait_limit_ns;
  params.extra_tx = extra_tx;
  params.M = M;
  params.H = H;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(k->tiles_per_head), static_cast<unsigned>(H),
                     static_cast<unsigned>(large ? large_chunks(M) : (q.chunk ? (M + q.chunk - 1) / q.chunk : 1)));
  cfg.blockDim = dim3(static_cast<unsigned>(k->threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[1] = {&params};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, k->fn, args);
  if (e != cudaSuccess) return fail_cuda("cudaLaunchKernelExC", e);
  return MLAQP_OK;
}

// ---------------------------------------------------------------------------
// V up-projection
// ---------------------------------------------------------------------------

// 2-D tensor map over W_UV viewed as [H*512 rows][128 columns].  For the
// M <= 64 kernel one box is 16 columns x 256 rows (a CTA copies two), BF16
// with the 32-byte swizzle (conflict-free ldmatrix of its 32-byte rows),
// E4M3 unswizzled; for the cluster kernel 64 columns x 128 rows,
// 128B-swizzled for BF16 (the UMMA operand layout) and unswizzled for E4M3.
int encode_v_weight_map(CUtensorMap* map, const void* weight, int H, bool mx, bool large) {
  std::string err;
  EncodeTiledFn fn = encode_tiled_fn(&err);
  if (!fn) return fail(MLAQP_ERR_CUDA, err);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(MLAQP_V_HEAD_DIM),
                              static_cast<cuuint64_t>(H) * MLAQP_LATENT_DIM};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(MLAQP_V_HEAD_DIM) * (mx ? 1 : 2)};
  const cuuint32_t box[2] = {large ? 64u : static_cast<cuuint32_t>(mlaqp::kVNTile),
                             large ? static_cast<cuuint32_t>(mlaqp::kVLargeK) : 256u};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(weight), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        mx ? CU_TENSOR_MAP_SWIZZLE_NONE : (large ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MLAQP_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return MLAQP_OK;
}

// x of a V call as a 3-D tensor [M][H][512] (column fastest) for the
// multicast kernel: box 64 columns x 1 head x tt tokens, 128-byte swizzle;
// token rows at or beyond M read as zeros.  Returns false where the strides
// cannot form a tensor map (the caller then uses the kernel that reads x
// with plain loads).
bool encode_v_x_map(CUtensorMap* map, const void* x, int64_t x_ts, int64_t x_hs, int M, int H, int tt) {
  std::string err;
  EncodeTiledFn fn = encode_tiled_fn(&err);
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(MLAQP_LATENT_DIM), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(M)};
  if (x_hs <= 0) return false;
  // The token stride of a single token is never used; any valid value does.
  const int64_t ts = M == 1 && x_ts <= 0 ? x_hs * H : x_ts;
  if (ts <= 0) return false;
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(x_hs) * 2, static_cast<cuuint64_t>(ts) * 2};
  const cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(tt)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The mma.sync kernels run in 32-token chunks (grid.z) up to M = 64, and
// beyond while their 8*H*chunks CTAs fit the GPU (v_chunk_cap; BF16 capped
// accordingly, MXFP8 uncapped); otherwise (from M = kVLargeMinM) the
// tcgen05 cluster kernel (H = 16, M = 96: BF16 3.29 / 2.80 at cap 3, MXFP8
// 3.42 / 3.20).  Measured on GB300 (128-layer PDL chains, us per layer call,
// cluster kernel / chunks): H = 8, M = 128: BF16 3.01 / 2.25, MXFP8 3.24 /
// 2.76; H = 11, M = 96: BF16 3.03 / 2.32, MXFP8 3.25 / 2.79; H = 16 with
// three or four chunks at cap 2 (384-512 CTAs): BF16 3.23-3.35 / 4.02-4.37.  Before
// the x multicast the chunks took 3.0 / 5.8 / 9.4 at H = 16, M = 64 / 128
// / 256.
constexpr int kVLargeMinM = 65;

int v_up_chunks(int M) { return (M + mlaqp::kVChunk - 1) / mlaqp::kVChunk; }

// Tokens per chunk of a V launch at 9 <= M <= 32 where two chunks' 16*H
// CTAs fit one per SM (H = 8 on 152 SMs): 8 up to M = 16, 16 above for
// MXFP8 weights; 0 when one launch covers all tokens.  Measured on GB300
// (128/256-layer PDL chains, us per layer call, H = 8, one launch / two
// chunks): M = 16: BF16 1.72 / 1.48, MXFP8 1.73 / 1.53; M = 32: MXFP8 2.17
// / 1.69; BF16 at M = 17..32 1.82 / 1.85-1.87 (kept in one launch).
int v_small_chunk(int weight_format, int M, int H, int sm_count) {
  if (M <= 8 || M > mlaqp::kVChunk || 2 * mlaqp::kVTilesPerHead * H > sm_count) return 0;
  if (M <= 16) return 8;
  return weight_format == MLAQP_WEIGHT_MXFP8 ? 16 : 0;
}

// CTAs per SM the chunked V launch needs (2, or 3 where 2 do not hold all
// its CTAs), or 0 when it should not run.  The 8-CTA clusters place less
// freely than the query's CTAs: at 384 CTAs (H = 8, M = 192; H = 16, M = 96)
// the chunks still win (BF16 4.08 / 2.75 and 3.29 / 2.80 us, cluster kernel
// / chunks), at 440-448 (H = 11, M = 160; H = 8, M = 224) they lose (4.17 /
// 4.35, 4.11 / 4.42), so the three-per-SM tier stops at 2.6 CTAs per SM.
int v_chunk_cap(int M, int H, int sm_count) {
  if (M < kVLargeMinM) return 2;
  const int ctas = mlaqp::kVTilesPerHead * H * v_up_chunks(M);
  return ctas <= 2 * sm_count ? 2 : (5 * ctas <= 13 * sm_count ? 3 : 0);
}

bool v_chunks_fit(int M, int H, int sm_count) { return v_chunk_cap(M, H, sm_count) != 0; }

// From this M on the 8 CTAs of a (head, chunk) share x through a TMA
// multicast.  Measured on GB300 (128-layer PDL chains, us per layer call,
// plain loads against multicast): BF16 W_UV at H = 16 1.95 / 1.75 at M = 9,
// 2.03 / 1.77 at M = 16; MXFP8 1.71 / 1.75 at M = 9, equal at M = 12-13,
// 1.89 / 1.76 at M = 16.
int v_mc_min_m(int weight_format) { return weight_format == MLAQP_WEIGHT_BF16 ? 9 : 12; }

const KernelInfo* lookup_v_up_mc(int weight_format, int M, int trig) {
  const int m = M < mlaqp::kVChunk ? M : mlaqp::kVChunk;
  return &mlaqp::kernels_v_up_mc()[weight_format][(m + 7) / 8 - 1][trig];
}

const KernelInfo* lookup_v_up(int weight_format, int M, int trig) {
  const int m = M < mlaqp::kVChunk ? M : mlaqp::kVChunk;
  return &mlaqp::kernels_v_up()[weight_format][(m + 7) / 8 - 1][trig];
}

// Token tile of the cluster kernel (index into kVLargeTokTiles): 64 up to
// M = 128, 128 above (M = 256 with 64-token tiles: 5.27 / 6.44 us BF16 /
// MXFP8, against 5.07 / 5.75).
int v_large_tile_index(int M) { return M <= 128 ? 0 : 1; }

const KernelInfo* lookup_v_up_large(int weight_format, int M, int early) {
  return &mlaqp::kernels_v_up_large()[weight_format][v_large_tile_index(M)][early];
}

struct VUpArgs {
  const void* x;
  int64_t x_ts, x_hs;
  const void* weight;
  const void* weight_scale;
  void* out;
  int64_t out_row_stride;
  int M, H, weight_format;
};

// Everything a V call launches, decided from the arguments and the SM count
// alone (no device access): v_up_impl and the mlaqp_debug_v_plan test hook
// share it.  multicast_ok: whether x's strides form the tensor map the
// x-multicast kernel reads (v_up_impl plans again without it when not).
struct VPlan {
  int form = 0;            // 0 column-tile kernel, plain loads; 1 x multicast; 2 tcgen05 cluster kernel
  const KernelInfo* k = nullptr;
  LaunchPolicy pol{0, 0};  // column-tile kernels: trigger point, CTA cap (applied with PDL)
  int chunk = 0;           // tokens per grid.z chunk
  int chunks = 1;          // grid.z
  int tt = 0;              // token rows of a CTA's tile (multicast box height, cluster token tile)
};

void plan_v(int weight_format, int M, int H, int pdl, int sm_count, bool multicast_ok, VPlan* v) {
  *v = VPlan{};
  if (!v_chunks_fit(M, H, sm_count)) {
    v->form = 2;
    v->k = lookup_v_up_large(weight_format, M, pdl == 2 ? 1 : 0);
    v->tt = mlaqp::kVLargeTokTiles[v_large_tile_index(M)];
    v->chunk = v->tt;
    v->chunks = (M + v->tt - 1) / v->tt;
    return;
  }
  v->pol = v_up_launch_policy(weight_format, M);
  if (v->pol.cta_cap != 0 && M >= kVLargeMinM) v->pol.cta_cap = v_chunk_cap(M, H, sm_count);
  const int trig = v->pol.trig == 0 ? 0 : 1;
  const int vch = v_small_chunk(weight_format, M, H, sm_count);
  const int cm = vch ? vch : (M < mlaqp::kVChunk ? M : mlaqp::kVChunk);  // tokens per CTA chunk
  v->tt = 8 * ((cm + 7) / 8);
  // 8-token chunks read x with plain loads (x is 8 KB per CTA there)
  v->form = multicast_ok && vch != 8 && M >= v_mc_min_m(weight_format) ? 1 : 0;
  v->k = v->form == 1 ? lookup_v_up_mc(weight_format, cm, trig) : lookup_v_up(weight_format, cm, trig);
  v->chunk = vch ? vch : mlaqp::kVChunk;
  v->chunks = vch ? (M + vch - 1) / vch : v_up_chunks(M);
}

int v_up_impl(const VUpArgs& a, mlaqp_stream_t stream, int pdl, unsigned long long wait_limit_ns, unsigned extra_tx) {
  if (pdl < 0 || pdl > 2) return fail(MLAQP_ERR_INVALID_ARG, "pdl must be 0, 1 or 2");
  const int M = a.M, H = a.H;
  if (a.weight_format != MLAQP_WEIGHT_BF16 && a.weight_format != MLAQP_WEIGHT_MXFP8)
    return fail(MLAQP_ERR_INVALID_ARG, "unknown weight_format");
  if (M < 0) return fail(MLAQP_ERR_INVALID_ARG, "M must be >= 0");
  if (!supported_heads(H)) return fail(MLAQP_ERR_UNSUPPORTED, "num_heads must be 8, 11 or 16");
  if (M > MLAQP_MAX_M) return fail(MLAQP_ERR_UNSUPPORTED, "M must be <= 256");
  if (M == 0) return MLAQP_OK;
  const bool mx = a.weight_format == MLAQP_WEIGHT_MXFP8;
  if (!a.x || !a.weight || !a.out) return fail(MLAQP_ERR_INVALID_ARG, "x, weight and out are required");
  if (mx && !a.weight_scale) return fail(MLAQP_ERR_INVALID_ARG, "MXFP8 weights require weight_scale");
  if (!mx && a.weight_scale) return fail(MLAQP_ERR_INVALID_ARG, "BF16 weights take no weight_scale (pass NULL)");
  if (!aligned(a.x, 16) || !aligned(a.weight, 16) || !aligned(a.out, 16) ||
      (a.weight_scale && !aligned(a.weight_scale, 16)))
    return fail(MLAQP_ERR_INVALID_ARG, "x, weight, weight_scale and out must be 16-byte aligned");
  if (a.x_ts < 0 || a.x_hs < 0 || a.x_ts % 8 != 0 || a.x_hs % 8 != 0)
    return fail(MLAQP_ERR_INVALID_ARG, "x strides must be >= 0 and multiples of 8 elements (16 bytes)");
  if (a.out_row_stride < static_cast<int64_t>(MLAQP_V_HEAD_DIM) * H)
    return fail(MLAQP_ERR_INVALID_ARG, "out_row_stride must be >= 128*H elements");
  if (a.out_row_stride % 8 != 0) return fail(MLAQP_ERR_INVALID_ARG, "out_row_stride must be a multiple of 8 elements");

  const Range o = span(a.out, static_cast<size_t>(((M - 1) * a.out_row_stride + MLAQP_V_HEAD_DIM * H) * 2));
  const size_t w_elems = static_cast<size_t>(H) * MLAQP_LATENT_DIM * MLAQP_V_HEAD_DIM;
  const Range inputs[3] = {
      span(a.x, static_cast<size_t>((M - 1) * a.x_ts + (H - 1) * a.x_hs + MLAQP_LATENT_DIM) * 2),
      span(a.weight, w_elems * (mx ? 1 : 2)),
      span(a.weight_scale, mx ? w_elems / 32 : 0),
  };
  for (const Range& r : inputs)
    if (r.hi > r.lo && overlaps(o, r)) return fail(MLAQP_ERR_INVALID_ARG, "out overlaps an input tensor");

  int device = 0;
  int st = resolve_device(-1, &device);
  if (st != MLAQP_OK) return st;
  st = check_device(device);
  if (st != MLAQP_OK) return st;

  mlaqp::VUpParams params;
  const int sm_count = g_dev[device].sm_count;
  VPlan v;
  plan_v(a.weight_format, M, H, pdl, sm_count, true, &v);
  if (v.form == 1 && !encode_v_x_map(&params.xmap, a.x, a.x_ts, a.x_hs, M, H, v.tt))
    plan_v(a.weight_format, M, H, pdl, sm_count, false, &v);
  const bool large = v.form == 2;
  const bool mc = v.form == 1;
  const KernelInfo* k = v.k;
  const int chunks = v.chunks;
  const int smem_bytes = large ? tmem_safe_smem(g_dev[device], k->smem_bytes, ((M < v.tt ? M : v.tt) + 15) & ~15)
                               : smem_for_cap(g_dev[device], k->smem_bytes, pdl ? v.pol.cta_cap : 0);
  st = encode_v_weight_map(&params.wmap, a.weight, H, mx, large);
  if (st != MLAQP_OK) return st;
  params.x = static_cast<const uint16_t*>(a.x);
  params.x_ts = a.x_ts;
  params.x_hs = a.x_hs;
  params.weight_scale = static_cast<const uint8_t*>(a.weight_scale);
  params.out = static_cast<uint16_t*>(a.out);
  params.out_row_stride = a.out_row_stride;
  params.wait_limit_ns = wait_limit_ns;
  params.extra_tx = extra_tx;
  params.M = M;
  params.H = H;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(k->tiles_per_head), static_cast<unsigned>(H), static_cast<unsigned>(chunks));
  cfg.blockDim = dim3(static_cast<unsigned>(k->threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  unsigned n_attr = 0;
  if (large || mc) {  // the CTAs of one (head, chunk) form a cluster
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = static_cast<unsigned>(k->tiles_per_head);
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  if (pdl) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
    ++n_attr;
  }
  cfg.attrs = n_attr ? attr : nullptr;
  cfg.numAttrs = n_attr;
  void* args[1] = {&params};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, k->fn, args);
  if (e != cudaSuccess) return fail_cuda("cudaLaunchKernelExC", e);
  return MLAQP_OK;
}

}  // namespace

extern "C" {

int mlaqp_can_implement(int num_heads, int max_m, int nope_dim, int latent_dim, int rope_dim, int weight_format,
                        int out_dtype, int device) {
  if (!valid_enums(weight_format, out_dtype)) return fail(0, "unknown weight_format or out_dtype");
  if (!supported_heads(num_heads)) return fail(0, "num_heads must be 8, 11 or 16");
  if (max_m < 1 || max_m > MLAQP_MAX_M) return fail(0, "max_m must be in 1..256");
  if (nope_index(nope_dim) < 0 || latent_dim != MLAQP_LATENT_DIM || rope_dim != MLAQP_ROPE_DIM)
    return fail(0, "only nope_dim 128 or 192, latent_dim 512 and rope_dim 64 are implemented");
  int dev = 0;
  if (resolve_device(device, &dev) != MLAQP_OK) return 0;
  int count = 0;
  const cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return fail(0, std::string("no CUDA device: ") + cudaGetErrorString(e));
  if (dev >= count) return fail(0, "device ordinal out of range");
  if (check_device(dev) != MLAQP_OK) return 0;
  return 1;
}

int mlaqp_prewarm(int num_heads, int max_m, int weight_format, int out_dtype, int device) {
  if (!valid_enums(weight_format, out_dtype)) return fail(MLAQP_ERR_UNSUPPORTED, "unknown weight_format or out_dtype");
  if (!supported_heads(num_heads)) return fail(MLAQP_ERR_UNSUPPORTED, "num_heads must be 8, 11 or 16");
  if (max_m < 1 || max_m > MLAQP_MAX_M) return fail(MLAQP_ERR_UNSUPPORTED, "max_m must be in 1..256");
  int dev = 0;
  int st = resolve_device(device, &dev);
  if (st != MLAQP_OK) return st;
  st = check_device(dev);
  if (st != MLAQP_OK) return st;

  std::lock_guard<std::mutex> lock(g_prewarm_mutex);
  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  if (prev != dev && (e = cudaSetDevice(dev)) != cudaSuccess) return fail_cuda("cudaSetDevice", e);
  int status = MLAQP_OK;
  const int decode_m = max_m < MLAQP_MAX_M_DECODE ? max_m : MLAQP_MAX_M_DECODE;
  for (int mt = 1; mt <= (decode_m + 7) / 8 && status == MLAQP_OK; ++mt) {
    const uint32_t bit = 1u << (((weight_format * 2 + out_dtype) * 4) + (mt - 1));
    if (g_prewarmed[dev].load(std::memory_order_acquire) & bit) continue;
    for (int ki = 0; ki < 2 && status == MLAQP_OK; ++ki) {
      for (int trig = 0; trig < mlaqp::kTrigVariants && status == MLAQP_OK; ++trig) {
        const KernelInfo* k = lookup(weight_format, out_dtype, 8 * mt, trig, ki);
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, k->fn);  // forces the kernel image to load
        if (e == cudaSuccess && mt >= 2)           // and its 8- / 16-token chunked form
          e = cudaFuncGetAttributes(&attr, lookup(weight_format, out_dtype, 8 * mt, trig, ki, mt == 2 ? 8 : 16)->fn);
        if (e != cudaSuccess) status = fail_cuda("cudaFuncGetAttributes", e);
      }
      for (int trig = 0; trig < 2 && status == MLAQP_OK; ++trig) {
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, lookup_warp(weight_format, out_dtype, 8 * mt, trig, ki, false)->fn);
        if (e == cudaSuccess && mt == 1 && ki == 0)
          e = cudaFuncGetAttributes(&attr, lookup_warp(weight_format, out_dtype, 8, trig, 0, true)->fn);
        if (e != cudaSuccess) status = fail_cuda("cudaFuncGetAttributes", e);
      }
    }
    if (status != MLAQP_OK) break;
    g_prewarmed[dev].fetch_or(bit, std::memory_order_acq_rel);
  }
  const uint32_t large_bit = 1u << (16 + weight_format * 2 + out_dtype);
  if (status == MLAQP_OK && max_m > MLAQP_MAX_M_DECODE && !(g_prewarmed[dev].load(std::memory_order_acquire) & large_bit)) {
    for (int ki = 0; ki < 2 && status == MLAQP_OK; ++ki)
      for (int ti = 0; ti < 3 && status == MLAQP_OK; ++ti) {
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, lookup_large(weight_format, out_dtype, ki, ti, 0)->fn);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, lookup_large(weight_format, out_dtype, ki, ti, 1)->fn);
        if (e != cudaSuccess) status = fail_cuda("cudaFuncGetAttributes", e);
      }
    for (int ki = 0; ki < 2 && status == MLAQP_OK; ++ki)  // the 32-token chunked CTA-tile form
      for (int trig = 0; trig < mlaqp::kTrigVariants && status == MLAQP_OK; ++trig) {
        cudaFuncAttributes attr;
        e = cudaFuncGetAttributes(&attr, lookup(weight_format, out_dtype, mlaqp::kMaxM + 1, trig, ki)->fn);
        if (e != cudaSuccess) status = fail_cuda("cudaFuncGetAttributes", e);
      }
    if (status == MLAQP_OK) g_prewarmed[dev].fetch_or(large_bit, std::memory_order_acq_rel);
  }
  if (prev != dev) cudaSetDevice(prev);
  return status;
}

int mlaqp_run(const void* q_nope, const void* q_pe, const void* weight, const void* weight_scale, void* out,
              int64_t out_row_stride, const float* q_scale, int M, int H, int weight_format, int out_dtype,
              mlaqp_stream_t stream) {
  return run_impl(contiguous_args(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H,
                                  weight_format, out_dtype),
                  stream, 0, kDefaultWaitLimitNs, 0);
}

int mlaqp_run_pdl(const void* q_nope, const void* q_pe, const void* weight, const void* weight_scale, void* out,
                  int64_t out_row_stride, const float* q_scale, int M, int H, int weight_format, int out_dtype,
                  mlaqp_stream_t stream) {
  return run_impl(contiguous_args(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H,
                                  weight_format, out_dtype),
                  stream, 1, kDefaultWaitLimitNs, 0);
}

int mlaqp_run_strided(const void* q_nope, int64_t q_nope_token_stride, int64_t q_nope_head_stride, const void* q_pe,
                      int64_t q_pe_token_stride, int64_t q_pe_head_stride, const void* weight,
                      const void* weight_scale, void* out, int64_t out_row_stride, const float* q_scale, int M,
                      int H, int nope_dim, int weight_format, int out_dtype, int pdl, mlaqp_stream_t stream) {
  const RunArgs a{q_nope, q_nope_token_stride, q_nope_head_stride, q_pe, q_pe_token_stride, q_pe_head_stride,
                  weight, weight_scale, out, out_row_stride, q_scale, M, H, nope_dim, weight_format, out_dtype};
  return run_impl(a, stream, pdl, kDefaultWaitLimitNs, 0);
}

int mlaqp_launch_shape(int M, int H, int weight_format, int out_dtype, int* grid_ctas, int* threads_per_cta) {
  if (!valid_enums(weight_format, out_dtype)) return fail(MLAQP_ERR_UNSUPPORTED, "unknown weight_format or out_dtype");
  if (!supported_heads(H) || M < 1 || M > MLAQP_MAX_M) return fail(MLAQP_ERR_UNSUPPORTED, "unsupported H or M");
  int sm_count = 0;
  if (M > 8) {  // the choice depends on the device's SM count, except at 33..64
    int dev = 0;
    int st = resolve_device(-1, &dev);
    if (st == MLAQP_OK) st = check_device(dev);
    if (st == MLAQP_OK) {
      sm_count = g_dev[dev].sm_count;
    } else if (M <= MLAQP_MAX_M_DECODE || M > kCtaAlwaysM) {
      return st;
    }
  }
  QueryPlan q;
  const int st = plan_query(weight_format, out_dtype, M, H, MLAQP_NOPE_DIM, 1, Arm::kAuto, sm_count, &q);
  if (st != MLAQP_OK) return st;
  if (grid_ctas) *grid_ctas = q.grid;
  if (threads_per_cta) *threads_per_cta = q.threads;
  return MLAQP_OK;
}

int mlaqp_debug_plan(int M, int H, int nope_dim, int weight_format, int out_dtype, int pdl, int arm, int sm_count,
                     int* arm_out, int* chunk_tokens, int* trig, int* cta_cap, int* grid_ctas, int* threads_per_cta) {
  if (!valid_enums(weight_format, out_dtype)) return fail(MLAQP_ERR_INVALID_ARG, "unknown weight_format or out_dtype");
  if (!supported_heads(H) || M < 1 || M > MLAQP_MAX_M || nope_index(nope_dim) < 0)
    return fail(MLAQP_ERR_UNSUPPORTED, "unsupported H, M or nope_dim");
  if (pdl < 0 || pdl > 2 || arm < MLAQP_ARM_AUTO || arm > MLAQP_ARM_TCGEN05 || sm_count < 1)
    return fail(MLAQP_ERR_INVALID_ARG, "pdl must be 0..2, arm a MLAQP_ARM_* value and sm_count >= 1");
  QueryPlan q;
  const int st = plan_query(weight_format, out_dtype, M, H, nope_dim, pdl, static_cast<Arm>(arm), sm_count, &q);
  if (st != MLAQP_OK) return st;
  const bool tc = q.arm == Arm::kTcgen05;
  if (arm_out) *arm_out = static_cast<int>(q.arm);
  if (chunk_tokens) *chunk_tokens = q.chunk;
  if (trig) *trig = tc ? (pdl == 2 ? 0 : 1) : q.pol.trig;
  if (cta_cap) *cta_cap = (pdl && !tc) ? q.pol.cta_cap : 0;
  if (grid_ctas) *grid_ctas = q.grid;
  if (threads_per_cta) *threads_per_cta = q.threads;
  return MLAQP_OK;
}

int mlaqp_debug_v_plan(int M, int H, int weight_format, int pdl, int sm_count, int* form, int* chunk_tokens,
                       int* trig, int* cta_cap, int* grid_ctas, int* threads_per_cta, int* cluster) {
  if (weight_format != MLAQP_WEIGHT_BF16 && weight_format != MLAQP_WEIGHT_MXFP8)
    return fail(MLAQP_ERR_INVALID_ARG, "unknown weight_format");
  if (!supported_heads(H) || M < 1 || M > MLAQP_MAX_M) return fail(MLAQP_ERR_UNSUPPORTED, "unsupported H or M");
  if (pdl < 0 || pdl > 2 || sm_count < 1) return fail(MLAQP_ERR_INVALID_ARG, "pdl must be 0..2 and sm_count >= 1");
  VPlan v;
  plan_v(weight_format, M, H, pdl, sm_count, true, &v);
  const bool tc = v.form == 2;
  if (form) *form = v.form;
  if (chunk_tokens) *chunk_tokens = v.chunk;
  if (trig) *trig = tc ? (pdl == 2 ? 0 : 1) : v.pol.trig;
  if (cta_cap) *cta_cap = (pdl && !tc) ? v.pol.cta_cap : 0;
  if (grid_ctas) *grid_ctas = v.k->tiles_per_head * H * v.chunks;
  if (threads_per_cta) *threads_per_cta = v.k->threads;
  if (cluster) *cluster = v.form == 0 ? 1 : v.k->tiles_per_head;
  return MLAQP_OK;
}

int mlaqp_debug_run_bounded_wait(const void* q_nope, const void* q_pe, const void* weight, const void* weight_scale,
                                 void* out, int64_t out_row_stride, const float* q_scale, int M, int H,
                                 int weight_format, int out_dtype, unsigned long long wait_limit_ns,
                                 unsigned int extra_tx_bytes, mlaqp_stream_t stream) {
  if (wait_limit_ns == 0) return fail(MLAQP_ERR_INVALID_ARG, "wait_limit_ns must be > 0");
  if (extra_tx_bytes > (1u << 19)) return fail(MLAQP_ERR_INVALID_ARG, "extra_tx_bytes must be <= 2^19");
  return run_impl(contiguous_args(q_nope, q_pe, weight, weight_scale, out, out_row_stride, q_scale, M, H,
                                  weight_format, out_dtype),
                  stream, 0, wait_limit_ns, extra_tx_bytes);
}

int mlaqp_debug_run_arm(const void* q_nope, int64_t q_nope_token_stride, int64_t q_nope_head_stride, const void* q_pe,
                        int64_t q_pe_token_stride, int64_t q_pe_head_stride, const void* weight,
                        const void* weight_scale, void* out, int64_t out_row_stride, const float* q_scale, int M,
                        int H, int nope_dim, int weight_format, int out_dtype, int pdl, int arm,
                        mlaqp_stream_t stream) {
  if (arm < 0 || arm > 4) return fail(MLAQP_ERR_INVALID_ARG, "arm must be in 0..4");
  const RunArgs a{q_nope, q_nope_token_stride, q_nope_head_stride, q_pe, q_pe_token_stride, q_pe_head_stride,
                  weight, weight_scale, out, out_row_stride, q_scale, M, H, nope_dim, weight_format, out_dtype};
  return run_impl(a, stream, pdl, kDefaultWaitLimitNs, 0, static_cast<Arm>(arm));
}

int mlaqp_debug_set_policy(int trig, int cta_cap) {
  if (trig < -1 || trig > 1 || cta_cap < 0 || cta_cap > 8)
    return fail(MLAQP_ERR_INVALID_ARG, "trig must be -1, 0 or 1 and cta_cap in 0..8");
  g_policy_cap.store(cta_cap, std::memory_order_relaxed);
  g_policy_trig.store(trig, std::memory_order_relaxed);
  return MLAQP_OK;
}

int mlaqp_prefetch_weights(const void* weight, const void* weight_scale, int H, int nope_dim, int weight_format,
                           int pdl, mlaqp_stream_t stream) {
  if (weight_format != MLAQP_WEIGHT_BF16 && weight_format != MLAQP_WEIGHT_MXFP8)
    return fail(MLAQP_ERR_INVALID_ARG, "unknown weight_format");
  if (!supported_heads(H)) return fail(MLAQP_ERR_UNSUPPORTED, "num_heads must be 8, 11 or 16");
  if (nope_index(nope_dim) < 0) return fail(MLAQP_ERR_UNSUPPORTED, "nope_dim must be 128 or 192");
  const bool mx = weight_format == MLAQP_WEIGHT_MXFP8;
  if (!weight) return fail(MLAQP_ERR_INVALID_ARG, "weight is required");
  if (mx && !weight_scale) return fail(MLAQP_ERR_INVALID_ARG, "MXFP8 weights require weight_scale");
  if (!mx && weight_scale) return fail(MLAQP_ERR_INVALID_ARG, "BF16 weights take no weight_scale (pass NULL)");
  if (!aligned(weight, 16) || (weight_scale && !aligned(weight_scale, 16)))
    return fail(MLAQP_ERR_INVALID_ARG, "weight and weight_scale must be 16-byte aligned");
  int device = 0;
  int st = resolve_device(-1, &device);
  if (st != MLAQP_OK) return st;
  st = check_device(device);
  if (st != MLAQP_OK) return st;
  const unsigned long long w_bytes =
      static_cast<unsigned long long>(H) * nope_dim * MLAQP_LATENT_DIM * (mx ? 1 : 2);
  const unsigned long long sc_bytes = mx ? w_bytes / 32 : 0;
  constexpr unsigned kChunk = 64u << 10;  // per CTA (one TMA prefetch)
  const unsigned ctas = static_cast<unsigned>((w_bytes + kChunk - 1) / kChunk + (sc_bytes + kChunk - 1) / kChunk);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const uint8_t* w = static_cast<const uint8_t*>(weight);
  const uint8_t* sc = static_cast<const uint8_t*>(weight_scale);
  unsigned chunk = kChunk;
  void* args[5] = {&w, const_cast<unsigned long long*>(&w_bytes), &sc, const_cast<unsigned long long*>(&sc_bytes),
                   &chunk};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&mlaqp_prefetch_kernel), args);
  if (e != cudaSuccess) return fail_cuda("cudaLaunchKernelExC", e);
  return MLAQP_OK;
}

int mlaqp_device_status(unsigned int* status, int reset) {
  if (!status) return fail(MLAQP_ERR_INVALID_ARG, "status must not be NULL");
  unsigned int a = 0, b = 0, c = 0, v = 0, wa = 0, wb = 0;
  cudaError_t e = mlaqp::device_status_bf16_weights(&a, reset != 0);
  if (e == cudaSuccess) e = mlaqp::device_status_mxfp8_weights(&b, reset != 0);
  if (e == cudaSuccess) e = mlaqp::device_status_large_m(&c, reset != 0);
  if (e == cudaSuccess) e = mlaqp::device_status_v_up(&v, reset != 0);
  if (e == cudaSuccess) e = mlaqp::device_status_warp_bf16(&wa, reset != 0);
  if (e == cudaSuccess) e = mlaqp::device_status_warp_mxfp8(&wb, reset != 0);
  if (e != cudaSuccess) return fail_cuda("reading the device status word", e);
  *status = a | b | c | v | wa | wb;
  return MLAQP_OK;
}

int mlaqp_debug_launch_null(int ctas, int threads, int pdl, mlaqp_stream_t stream) {
  if (ctas < 1 || ctas > 65535 || threads < 1 || threads > 1024)
    return fail(MLAQP_ERR_INVALID_ARG, "ctas must be in 1..65535 and threads in 1..1024");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  void* args[1] = {nullptr};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&mlaqp_null_kernel), args);
  if (e != cudaSuccess) return fail_cuda("cudaLaunchKernelExC", e);
  return MLAQP_OK;
}

int mlaqp_v_up_run(const void* x, int64_t x_token_stride, int64_t x_head_stride, const void* weight,
                   const void* weight_scale, void* out, int64_t out_row_stride, int M, int H, int weight_format,
                   int pdl, mlaqp_stream_t stream) {
  const VUpArgs a{x, x_token_stride, x_head_stride, weight, weight_scale, out, out_row_stride, M, H, weight_format};
  return v_up_impl(a, stream, pdl, kDefaultWaitLimitNs, 0);
}

int mlaqp_debug_v_up_bounded_wait(const void* x, int64_t x_token_stride, int64_t x_head_stride, const void* weight,
                                  const void* weight_scale, void* out, int64_t out_row_stride, int M, int H,
                                  int weight_format, unsigned long long wait_limit_ns, unsigned int extra_tx_bytes,
                                  mlaqp_stream_t stream) {
  if (wait_limit_ns == 0) return fail(MLAQP_ERR_INVALID_ARG, "wait_limit_ns must be > 0");
  if (extra_tx_bytes > (1u << 19)) return fail(MLAQP_ERR_INVALID_ARG, "extra_tx_bytes must be <= 2^19");
  const VUpArgs a{x, x_token_stride, x_head_stride, weight, weight_scale, out, out_row_stride, M, H, weight_format};
  return v_up_impl(a, stream, 0, wait_limit_ns, extra_tx_bytes);
}

int mlaqp_v_up_can_implement(int num_heads, int max_m, int weight_format, int device) {
  if (weight_format != MLAQP_WEIGHT_BF16 && weight_format != MLAQP_WEIGHT_MXFP8)
    return fail(0, "unknown weight_format");
  if (!supported_heads(num_heads)) return fail(0, "num_heads must be 8, 11 or 16");
  if (max_m < 1 || max_m > MLAQP_MAX_M) return fail(0, "max_m must be in 1..256");
  int dev = 0;
  if (resolve_device(device, &dev) != MLAQP_OK) return 0;
  int count = 0;
  const cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return fail(0, std::string("no CUDA device: ") + cudaGetErrorString(e));
  if (dev >= count) return fail(0, "device ordinal out of range");
  if (check_device(dev) != MLAQP_OK) return 0;
  return 1;
}

int mlaqp_v_up_prewarm(int num_heads, int max_m, int weight_format, int device) {
  if (weight_format != MLAQP_WEIGHT_BF16 && weight_format != MLAQP_WEIGHT_MXFP8)
    return fail(MLAQP_ERR_UNSUPPORTED, "unknown weight_format");
  if (!supported_heads(num_heads)) return fail(MLAQP_ERR_UNSUPPORTED, "num_heads must be 8, 11 or 16");
  if (max_m < 1 || max_m > MLAQP_MAX_M) return fail(MLAQP_ERR_UNSUPPORTED, "max_m must be in 1..256");
  int dev = 0;
  int st = resolve_device(device, &dev);
  if (st != MLAQP_OK) return st;
  st = check_device(dev);
  if (st != MLAQP_OK) return st;
  std::lock_guard<std::mutex> lock(g_prewarm_mutex);
  int prev = -1;
  cudaError_t e = cudaGetDevice(&prev);
  if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  if (prev != dev && (e = cudaSetDevice(dev)) != cudaSuccess) return fail_cuda("cudaSetDevice", e);
  int status = MLAQP_OK;
  const int chunk_m = max_m < mlaqp::kVChunk ? max_m : mlaqp::kVChunk;
  for (int mt = 1; mt <= (chunk_m + 7) / 8 && status == MLAQP_OK; ++mt)
    for (int trig = 0; trig < 2 && status == MLAQP_OK; ++trig) {
      cudaFuncAttributes attr;
      e = cudaFuncGetAttributes(&attr, lookup_v_up(weight_format, 8 * mt, trig)->fn);
      if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, lookup_v_up_mc(weight_format, 8 * mt, trig)->fn);
      if (e != cudaSuccess) status = fail_cuda("cudaFuncGetAttributes", e);
    }
  if (max_m >= kVLargeMinM)
    for (int ti = 0; ti < 2 && status == MLAQP_OK; ++ti) {
      cudaFuncAttributes attr;
      e = cudaFuncGetAttributes(&attr, mlaqp::kernels_v_up_large()[weight_format][ti][0].fn);
      if (e == cudaSuccess) e = cudaFuncGetAttributes(&attr, mlaqp::kernels_v_up_large()[weight_format][ti][1].fn);
      if (e != cudaSuccess) status = fail_cuda("cudaFuncGetAttributes", e);
    }
  if (prev != dev) cudaSetDevice(prev);
  return status;
}

const char* mlaqp_last_error(void) { return g_last_error.c_str(); }

int mlaqp_version(void) { return 100; }

}  // extern "C"
