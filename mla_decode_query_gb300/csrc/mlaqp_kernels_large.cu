// Instantiations of the tcgen05 query kernel for 33 <= M <= 256 (both weight
// formats, both output dtypes, nope dims 128 and 192, 32-, 64- and 128-token CTA tiles,
// trigger after the TMEM allocation or, opted in, at entry).
#include "mlaqp_dispatch.h"
#include "mlaqp_kernel_large.cuh"

namespace mlaqp {
namespace {

template <int K, int TT, int WF, int OD, int EARLY>
KernelInfo entry() {
  return KernelInfo{reinterpret_cast<const void*>(&mlaqp_fused_query_large_kernel<WF, OD, K, TT, EARLY>),
                    large_threads(TT), kLargeTilesPerHead, large_smem_layout(K, TT, WF == kWeightMXFP8).bytes};
}

template <int K, int TT>
void fill(KernelInfo (&t)[2][2][2]) {
  t[kWeightBF16][kOutBF16][0] = entry<K, TT, kWeightBF16, kOutBF16, 0>();
  t[kWeightBF16][kOutE4M3][0] = entry<K, TT, kWeightBF16, kOutE4M3, 0>();
  t[kWeightMXFP8][kOutBF16][0] = entry<K, TT, kWeightMXFP8, kOutBF16, 0>();
  t[kWeightMXFP8][kOutE4M3][0] = entry<K, TT, kWeightMXFP8, kOutE4M3, 0>();
  t[kWeightBF16][kOutBF16][1] = entry<K, TT, kWeightBF16, kOutBF16, 1>();
  t[kWeightBF16][kOutE4M3][1] = entry<K, TT, kWeightBF16, kOutE4M3, 1>();
  t[kWeightMXFP8][kOutBF16][1] = entry<K, TT, kWeightMXFP8, kOutBF16, 1>();
  t[kWeightMXFP8][kOutE4M3][1] = entry<K, TT, kWeightMXFP8, kOutE4M3, 1>();
}

struct Table {
  LargeKernelTable t;
  Table() {
    static_assert(kLargeTokTiles[0] == 32 && kLargeTokTiles[1] == 64 && kLargeTokTiles[2] == 128, "token tiles");
    fill<128, 32>(t[0][0]);
    fill<128, 64>(t[0][1]);
    fill<128, 128>(t[0][2]);
    fill<192, 32>(t[1][0]);
    fill<192, 64>(t[1][1]);
    fill<192, 128>(t[1][2]);
  }
};

}  // namespace

const LargeKernelTable& kernels_large_m() {
  static const Table table;
  return table.t;
}

cudaError_t device_status_large_m(unsigned int* value, bool reset) { return read_device_status(value, reset); }

}  // namespace mlaqp
