// Instances of the LUT-GEMM kernel for 16-bit narrowed LUT entries.
#include "gemm_ws.cuh"

namespace amsim {
namespace kern {

int launch_ws_w16(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    return gl ? launch_ws_instance<16, true>(p, grid, smem, st) : launch_ws_instance<16, false>(p, grid, smem, st);
}

int launch_w16(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    return gl ? launch_instance<16, true>(p, grid, smem, st) : launch_instance<16, false>(p, grid, smem, st);
}

}  // namespace kern
}  // namespace amsim
