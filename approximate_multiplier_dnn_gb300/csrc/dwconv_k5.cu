// 5x5 variants of the depthwise tiled kernel (table products), compiled apart
// from dwconv.cu so the two build in parallel.
#include "dwconv_kernel.cuh"

namespace amsim {
namespace dw {
template int launch_tile<0, 0, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<1, 0, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<2, 0, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
}  // namespace dw
}  // namespace amsim
