// Instances of the raw-tile TMA LUT-GEMM kernel for 32-bit narrowed LUT entries.
#include "gemm_raw.cuh"

namespace amsim {
namespace kern {

int launch_raw_w32(const KParams &p, const TmaMaps &maps, const PhaseTable *pt, bool gl, dim3 grid, size_t smem,
                  cudaStream_t st)
{
    if (p.nphase > 1)
        return gl || !pt ? AMSIM_EUNSUPPORTED : launch_raw_instance<32, false, true>(p, maps, pt, grid, smem, st);
    return gl ? launch_raw_instance<32, true>(p, maps, nullptr, grid, smem, st)
              : launch_raw_instance<32, false>(p, maps, nullptr, grid, smem, st);
}

}  // namespace kern
}  // namespace amsim
