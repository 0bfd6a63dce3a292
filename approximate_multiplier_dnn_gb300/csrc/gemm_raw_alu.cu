// Instances of the raw-tile LUT-GEMM kernel that compute each product's
// mantissa factor in registers instead of reading a table: W = 1 for
// Mitchell's logarithmic multiplier, W = 2 for the exact product of the
// truncated mantissas (the two built-in kinds of the ApproxTrain page,
// Sec. V-A; closed forms beside compute_stage).
#include "gemm_raw.cuh"

namespace amsim {
namespace kern {

template <int W>
static int launch_alu(const KParams &p, const TmaMaps &maps, const PhaseTable *pt, dim3 grid, size_t smem,
                      cudaStream_t st)
{
    if (p.nphase > 1)
        return pt ? launch_raw_instance<W, false, true>(p, maps, pt, grid, smem, st) : AMSIM_EUNSUPPORTED;
    return launch_raw_instance<W, false>(p, maps, nullptr, grid, smem, st);
}

int launch_raw_alu(const KParams &p, const TmaMaps &maps, const PhaseTable *pt, dim3 grid, size_t smem,
                   cudaStream_t st)
{
    if (p.table_bytes != 0) return AMSIM_EUNSUPPORTED;
    switch (p.alu) {
    case 1: return launch_alu<1>(p, maps, pt, grid, smem, st);
    case 2: return launch_alu<2>(p, maps, pt, grid, smem, st);
    default: return AMSIM_EUNSUPPORTED;
    }
}

}  // namespace kern
}  // namespace amsim
