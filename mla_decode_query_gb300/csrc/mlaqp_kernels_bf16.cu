// Instantiations of the fused query kernel for BF16 W_UK_T.
#include "mlaqp_dispatch.h"
#include "mlaqp_kernel.cuh"

namespace mlaqp {
namespace {
constexpr int kWF = kWeightBF16;

template <int K, int OD, int MT, int TRIG, int CH>
KernelInfo entry() {
  return KernelInfo{
      reinterpret_cast<const void*>(&mlaqp_fused_query_kernel<kWF, OD, MT, TRIG, K, token_groups(MT), CH>),
      kThreads * token_groups(MT), kTilesPerHead, Smem<K>::Bytes};
}

template <int K, int OD, int MT, int CH = 0>
void fill(KernelInfo (&row)[kTrigVariants]) {
  row[0] = entry<K, OD, MT, 0, CH>();
  row[1] = entry<K, OD, MT, 1, CH>();
  row[2] = entry<K, OD, MT, 2, CH>();
}

template <int K>
void fill_nope(KernelInfo (&t)[2][7][kTrigVariants]) {
  fill<K, kOutBF16, 1>(t[0][0]);
  fill<K, kOutBF16, 2>(t[0][1]);
  fill<K, kOutBF16, 3>(t[0][2]);
  fill<K, kOutBF16, 4>(t[0][3]);
  fill<K, kOutE4M3, 1>(t[1][0]);
  fill<K, kOutE4M3, 2>(t[1][1]);
  fill<K, kOutE4M3, 3>(t[1][2]);
  fill<K, kOutE4M3, 4>(t[1][3]);
  fill<K, kOutBF16, 4, 1>(t[0][kChunkedForm]);  // M > 32: 32-token chunks
  fill<K, kOutE4M3, 4, 1>(t[1][kChunkedForm]);
  fill<K, kOutBF16, 1, 1>(t[0][kChunked8Form]);  // M = 9..32 on small H: 8- and 16-token chunks
  fill<K, kOutE4M3, 1, 1>(t[1][kChunked8Form]);
  fill<K, kOutBF16, 2, 1>(t[0][kChunked16Form]);
  fill<K, kOutE4M3, 2, 1>(t[1][kChunked16Form]);
}

struct Table {
  KernelTable t;
  Table() {
    fill_nope<128>(t[0]);
    fill_nope<192>(t[1]);
  }
};
}  // namespace

const KernelTable& kernels_bf16_weights() {
  static const Table table;
  return table.t;
}

cudaError_t device_status_bf16_weights(unsigned int* value, bool reset) { return read_device_status(value, reset); }

}  // namespace mlaqp
