// 5x5 variants of the depthwise tiled kernel with closed-form products
// (Mitchell, exact), compiled apart so the translation units build in parallel.
#include "dwconv_kernel.cuh"

namespace amsim {
namespace dw {
template int launch_tile<0, 1, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<1, 1, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<2, 1, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<0, 2, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<1, 2, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<2, 2, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
}  // namespace dw
}  // namespace amsim
