// Instantiations of the V up-projection kernels: {BF16, MXFP8} W_UV x
// ceil(M/8) in 1..4 x trigger point {entry, after the wait} for M <= 64 (x
// read by every CTA, and x multicast over a cluster), and {BF16, MXFP8} x
// token tile {64, 128} of the tcgen05 cluster kernel above M = 64.
#include "mlaqp_dispatch.h"
#include "mlaqp_v_up_kernel.cuh"
#include "mlaqp_v_up_kernel_large.cuh"
#include "mlaqp_v_up_kernel_mc.cuh"

namespace mlaqp {
namespace {

template <int WF, int MT, int TRIG>
KernelInfo entry() {
  return KernelInfo{reinterpret_cast<const void*>(&mlaqp_v_up_kernel<WF, MT, TRIG>), kVThreads, kVTilesPerHead,
                    VSmem<MT>::Bytes};
}

template <int WF>
void fill(KernelInfo (&t)[4][2]) {
  t[0][0] = entry<WF, 1, 0>();
  t[0][1] = entry<WF, 1, 1>();
  t[1][0] = entry<WF, 2, 0>();
  t[1][1] = entry<WF, 2, 1>();
  t[2][0] = entry<WF, 3, 0>();
  t[2][1] = entry<WF, 3, 1>();
  t[3][0] = entry<WF, 4, 0>();
  t[3][1] = entry<WF, 4, 1>();
}

template <int WF, int MT, int TRIG>
KernelInfo mc_entry() {
  return KernelInfo{reinterpret_cast<const void*>(&mlaqp_v_up_mc_kernel<WF, MT, TRIG>), kVThreads, kVTilesPerHead,
                    VMcSmem<MT>::Bytes};
}

template <int WF>
void fill_mc(KernelInfo (&t)[4][2]) {
  t[0][0] = mc_entry<WF, 1, 0>();
  t[0][1] = mc_entry<WF, 1, 1>();
  t[1][0] = mc_entry<WF, 2, 0>();
  t[1][1] = mc_entry<WF, 2, 1>();
  t[2][0] = mc_entry<WF, 3, 0>();
  t[2][1] = mc_entry<WF, 3, 1>();
  t[3][0] = mc_entry<WF, 4, 0>();
  t[3][1] = mc_entry<WF, 4, 1>();
}

struct McTable {
  VUpMcKernelTable t;
  McTable() {
    fill_mc<kWeightBF16>(t[kWeightBF16]);
    fill_mc<kWeightMXFP8>(t[kWeightMXFP8]);
  }
};

struct Table {
  VUpKernelTable t;
  Table() {
    fill<kWeightBF16>(t[kWeightBF16]);
    fill<kWeightMXFP8>(t[kWeightMXFP8]);
  }
};

template <int WF, int TT, int EARLY>
KernelInfo large_entry() {
  return KernelInfo{reinterpret_cast<const void*>(&mlaqp_v_up_large_kernel<WF, TT, EARLY>), kVLargeThreads,
                    kVLargeSplit, v_large_smem_layout(TT, WF == kWeightMXFP8).bytes};
}

struct LargeTable {
  VUpLargeKernelTable t;
  LargeTable() {
    static_assert(kVLargeTokTiles[0] == 64 && kVLargeTokTiles[1] == 128, "token tiles");
    t[kWeightBF16][0][0] = large_entry<kWeightBF16, 64, 0>();
    t[kWeightBF16][1][0] = large_entry<kWeightBF16, 128, 0>();
    t[kWeightMXFP8][0][0] = large_entry<kWeightMXFP8, 64, 0>();
    t[kWeightMXFP8][1][0] = large_entry<kWeightMXFP8, 128, 0>();
    t[kWeightBF16][0][1] = large_entry<kWeightBF16, 64, 1>();
    t[kWeightBF16][1][1] = large_entry<kWeightBF16, 128, 1>();
    t[kWeightMXFP8][0][1] = large_entry<kWeightMXFP8, 64, 1>();
    t[kWeightMXFP8][1][1] = large_entry<kWeightMXFP8, 128, 1>();
  }
};

}  // namespace

const VUpKernelTable& kernels_v_up() {
  static const Table table;
  return table.t;
}

const VUpMcKernelTable& kernels_v_up_mc() {
  static const McTable table;
  return table.t;
}

const VUpLargeKernelTable& kernels_v_up_large() {
  static const LargeTable table;
  return table.t;
}

cudaError_t device_status_v_up(unsigned int* value, bool reset) { return read_device_status(value, reset); }

}  // namespace mlaqp
