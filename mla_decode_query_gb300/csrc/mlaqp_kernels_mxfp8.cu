// Instantiations of the fused query kernel for MXFP8 W_UK_T (E4M3 values, E8M0 scales).
#include "mlaqp_dispatch.h"
#include "mlaqp_kernel.cuh"

namespace mlaqp {
namespace {
constexpr int kWF = kWeightMXFP8;

template <int OD, int MT>
KernelInfo entry() {
  return KernelInfo{reinterpret_cast<const void*>(&mlaqp_fused_query_kernel<kWF, OD, MT>), kThreads,
                    kTilesPerHead, kSmemBytes};
}
}  // namespace

const KernelTable& kernels_mxfp8_weights() {
  static const KernelTable table = {
      {entry<kOutBF16, 1>(), entry<kOutBF16, 2>(), entry<kOutBF16, 3>(), entry<kOutBF16, 4>()},
      {entry<kOutE4M3, 1>(), entry<kOutE4M3, 2>(), entry<kOutE4M3, 3>(), entry<kOutE4M3, 4>()},
  };
  return table;
}

cudaError_t device_status_mxfp8_weights(unsigned int* value, bool reset) { return read_device_status(value, reset); }

}  // namespace mlaqp
