// Instantiations of the warp-tile query kernel for MXFP8 W_UK_T.
#include "mlaqp_dispatch.h"
#include "mlaqp_kernel_warp.cuh"

namespace mlaqp {
namespace {
constexpr int kWF = kWeightMXFP8;

template <int K, int OD, int MT, int TRIG, int ARM>
KernelInfo entry() {
  return KernelInfo{reinterpret_cast<const void*>(&mlaqp_query_warp_kernel<kWF, OD, MT, TRIG, K, ARM>),
                    32 * wtoken_groups(MT), kWTilesPerHead, WSmem<K>::Bytes};
}

template <int K, int OD, int MT>
void fill(KernelInfo (&row)[2]) {
  row[0] = entry<K, OD, MT, 0, kArmMma>();
  row[1] = entry<K, OD, MT, 1, kArmMma>();
}

template <int K>
void fill_nope(KernelInfo (&t)[2][4][2]) {
  fill<K, kOutBF16, 1>(t[0][0]);
  fill<K, kOutBF16, 2>(t[0][1]);
  fill<K, kOutBF16, 3>(t[0][2]);
  fill<K, kOutBF16, 4>(t[0][3]);
  fill<K, kOutE4M3, 1>(t[1][0]);
  fill<K, kOutE4M3, 2>(t[1][1]);
  fill<K, kOutE4M3, 3>(t[1][2]);
  fill<K, kOutE4M3, 4>(t[1][3]);
}

struct Table {
  WarpKernelSet s;
  Table() {
    fill_nope<128>(s.mma[0]);
    fill_nope<192>(s.mma[1]);
    s.fma[0][0] = entry<128, kOutBF16, 1, 0, kArmFma>();
    s.fma[0][1] = entry<128, kOutBF16, 1, 1, kArmFma>();
    s.fma[1][0] = entry<128, kOutE4M3, 1, 0, kArmFma>();
    s.fma[1][1] = entry<128, kOutE4M3, 1, 1, kArmFma>();
  }
};
}  // namespace

const WarpKernelSet& kernels_warp_mxfp8_weights() {
  static const Table table;
  return table.s;
}

cudaError_t device_status_warp_mxfp8(unsigned int* value, bool reset) { return read_device_status(value, reset); }

}  // namespace mlaqp
