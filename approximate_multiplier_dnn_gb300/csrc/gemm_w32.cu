// Instances of the LUT-GEMM kernel for 32-bit narrowed LUT entries.
#include "gemm_ws.cuh"

namespace amsim {
namespace kern {

int launch_ws_w32(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    return gl ? launch_ws_instance<32, true>(p, grid, smem, st) : launch_ws_instance<32, false>(p, grid, smem, st);
}

int launch_w32(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    return gl ? launch_instance<32, true>(p, grid, smem, st) : launch_instance<32, false>(p, grid, smem, st);
}

}  // namespace kern
}  // namespace amsim
