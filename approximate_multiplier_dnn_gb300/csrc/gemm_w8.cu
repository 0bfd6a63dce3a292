// Instances of the LUT-GEMM kernel for 8-bit narrowed LUT entries.
#include "gemm_ws.cuh"

namespace amsim {
namespace kern {

int launch_fixup(const KParams &p, int boundaries, cudaStream_t st)
{
    if (boundaries <= 0) return AMSIM_OK;
    streamk_fixup<256><<<dim3(boundaries, BU * BL / kFixupChunk), 256, 0, st>>>(p);
    const int rc = cuda_status(cudaGetLastError());
    if (rc == AMSIM_OK) count_launch();
    return rc;
}

int launch_ws_w8(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    return gl ? launch_ws_instance<8, true>(p, grid, smem, st) : launch_ws_instance<8, false>(p, grid, smem, st);
}

int launch_w8(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    return gl ? launch_instance<8, true>(p, grid, smem, st) : launch_instance<8, false>(p, grid, smem, st);
}

}  // namespace kern
}  // namespace amsim
