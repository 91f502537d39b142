// Internal kernel registry shared by the host-side C ABI and the
// per-weight-format instantiation units.
#pragma once

#include <cuda_runtime.h>

namespace mlaqp {

struct KernelInfo {
  const void* fn;      // __global__ function, launched with one RunParams argument
  int threads;         // threads per CTA
  int tiles_per_head;  // CTAs per head along the latent axis (grid.x)
  int smem_bytes;      // dynamic shared memory per CTA
};

// Table [nope][out_dtype][form][trig]: nope 0 = K 128, 1 = K 192; form
// mt-1 for mt = ceil(M/8) in 1..4 (one launch covers all tokens), and the
// chunked forms (grid.z chunks of 8*mt tokens): 4 = 32-token chunks (M > 32),
// 5 = 8-token chunks, 6 = 16-token chunks; trig = where the CTA triggers the next kernel's
// launch (0: at entry, 1: after the dependency wait, 2: once its weight
// tile is ready).
constexpr int kTrigVariants = 3;
constexpr int kNopeDims[2] = {128, 192};
constexpr int kChunkedForm = 4;
constexpr int kChunked8Form = 5;
constexpr int kChunked16Form = 6;
using KernelTable = KernelInfo[2][2][7][kTrigVariants];

const KernelTable& kernels_bf16_weights();
const KernelTable& kernels_mxfp8_weights();

// Warp-tile query kernels (M <= 32), per weight format: the tensor-core
// arm [nope][out_dtype][mt-1][trig] and the CUDA-core arm [out_dtype][trig]
// (M <= 8, nope 128); trig 0: at entry, 1: after the dependency wait.
// threads = 32 x token groups per tile slot (the launch multiplies it by the
// tile slots of a CTA); smem_bytes = the unpadded layout size.
struct WarpKernelSet {
  KernelInfo mma[2][2][4][2];
  KernelInfo fma[2][2];
};
const WarpKernelSet& kernels_warp_bf16_weights();
const WarpKernelSet& kernels_warp_mxfp8_weights();

// tcgen05 kernels for 32 < M <= 256, [nope][token tile][weight_format][out_dtype][early]
// with token tiles kLargeTokTiles (tokens per CTA); the grid is
// (tiles_per_head, H, ceil(M / token tile)) and smem_bytes the unpadded
// layout size.
constexpr int kLargeTokTiles[3] = {32, 64, 128};
// (early 1: the next kernel may launch at entry -- the caller's opt-in under
// the tensor-memory contract of mlaqp_run_strided's pdl = 2).
using LargeKernelTable = KernelInfo[2][3][2][2][2];
const LargeKernelTable& kernels_large_m();

// V up-projection kernels, [weight_format][mt-1][trig] (trig 0: at entry,
// 1: after the dependency wait); grid (tiles_per_head, H).
using VUpKernelTable = KernelInfo[2][4][2];
const VUpKernelTable& kernels_v_up();

// V up-projection with x multicast over the 8 column-tile CTAs of a head
// (cluster (8, 1, 1)), [weight_format][mt-1][trig], grid as kernels_v_up.
using VUpMcKernelTable = KernelInfo[2][4][2];
const VUpMcKernelTable& kernels_v_up_mc();

// V up-projection for 64 < M <= 256 (tcgen05, contraction split over a
// cluster of tiles_per_head CTAs), [weight_format][token tile] with the
// token tiles kVLargeTokTiles; grid (tiles_per_head, H, ceil(M / tile)).
constexpr int kVLargeTokTiles[2] = {64, 128};
using VUpLargeKernelTable = KernelInfo[2][2][2];  // [weight_format][token tile][early]
const VUpLargeKernelTable& kernels_v_up_large();

// Device status word of each instantiation unit (current device).
cudaError_t device_status_bf16_weights(unsigned int* value, bool reset);
cudaError_t device_status_mxfp8_weights(unsigned int* value, bool reset);
cudaError_t device_status_large_m(unsigned int* value, bool reset);
cudaError_t device_status_v_up(unsigned int* value, bool reset);
cudaError_t device_status_warp_bf16(unsigned int* value, bool reset);
cudaError_t device_status_warp_mxfp8(unsigned int* value, bool reset);

}  // namespace mlaqp
