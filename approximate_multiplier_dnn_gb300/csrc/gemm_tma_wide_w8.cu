// Instances of the TMA-fed LUT-GEMM kernel with the wide tile shape (128 x 256
// tiles, eight lane columns per thread) for 8-bit narrowed LUT entries, and the
// stream-K fixup of wide tiles.
#define AMSIM_WIDE_TILES 1
#include "gemm_tma.cuh"

namespace amsim {
namespace kern_wide {

int launch_fixup(const KParams &p, int boundaries, cudaStream_t st)
{
    if (boundaries <= 0) return AMSIM_OK;
    streamk_fixup<256><<<dim3(boundaries, BU * BL / kFixupChunk), 256, 0, st>>>(p);
    const int rc = cuda_status(cudaGetLastError());
    if (rc == AMSIM_OK) count_launch();
    return rc;
}

int launch_tma_w8(const KParams &p, const TmaMaps &maps, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    return gl ? launch_tma_instance<8, true>(p, maps, grid, smem, st)
              : launch_tma_instance<8, false>(p, maps, grid, smem, st);
}

}  // namespace kern_wide
}  // namespace amsim
