// Closed-form (Mitchell, exact) variants of the depthwise tiled kernel, compiled
// apart from the table variants in dwconv.cu so the two build in parallel.
#include "dwconv_kernel.cuh"

namespace amsim {
namespace dw {
template int launch_tile<0, 1>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<1, 1>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<2, 1>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<0, 2>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<1, 2>(int, const DwTileParams &, int, size_t, cudaStream_t);
template int launch_tile<2, 2>(int, const DwTileParams &, int, size_t, cudaStream_t);
}  // namespace dw
}  // namespace amsim
