// Instantiations of the fused query kernel for BF16 W_UK_T.
#include "mlaqp_dispatch.h"
#include "mlaqp_kernel.cuh"

namespace mlaqp {
namespace {
constexpr int kWF = kWeightBF16;

template <int OD, int MT, int TRIG>
KernelInfo entry() {
  return KernelInfo{reinterpret_cast<const void*>(&mlaqp_fused_query_kernel<kWF, OD, MT, TRIG>), kThreads * token_groups(MT),
                    kTilesPerHead, kSmemBytes};
}


}  // namespace

const KernelTable& kernels_bf16_weights() {
  static const KernelTable table = {
      {{entry<kOutBF16, 1, 0>(), entry<kOutBF16, 1, 1>(), entry<kOutBF16, 1, 2>()},
       {entry<kOutBF16, 2, 0>(), entry<kOutBF16, 2, 1>(), entry<kOutBF16, 2, 2>()},
       {entry<kOutBF16, 3, 0>(), entry<kOutBF16, 3, 1>(), entry<kOutBF16, 3, 2>()},
       {entry<kOutBF16, 4, 0>(), entry<kOutBF16, 4, 1>(), entry<kOutBF16, 4, 2>()}},
      {{entry<kOutE4M3, 1, 0>(), entry<kOutE4M3, 1, 1>(), entry<kOutE4M3, 1, 2>()},
       {entry<kOutE4M3, 2, 0>(), entry<kOutE4M3, 2, 1>(), entry<kOutE4M3, 2, 2>()},
       {entry<kOutE4M3, 3, 0>(), entry<kOutE4M3, 3, 1>(), entry<kOutE4M3, 3, 2>()},
       {entry<kOutE4M3, 4, 0>(), entry<kOutE4M3, 4, 1>(), entry<kOutE4M3, 4, 2>()}},
  };
  return table;
}

cudaError_t device_status_bf16_weights(unsigned int* value, bool reset) { return read_device_status(value, reset); }

}  // namespace mlaqp
