// Instances of the TMA-fed LUT-GEMM kernel with the wide tile shape (128 x 256
// tiles, eight lane columns per thread) for 16-bit narrowed LUT entries.
#define AMSIM_WIDE_TILES 1
#include "gemm_tma.cuh"

namespace amsim {
namespace kern_wide {

int launch_tma_w16(const KParams &p, const TmaMaps &maps, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    return gl ? launch_tma_instance<16, true>(p, maps, grid, smem, st)
              : launch_tma_instance<16, false>(p, maps, grid, smem, st);
}

}  // namespace kern_wide
}  // namespace amsim
