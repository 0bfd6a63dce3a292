// Operand predecode pass of the TMA-fed LUT-GEMM: every dense operand of a
// launch is decoded once into (LUT offset, scale) planes that the GEMM copies
// tile by tile with the Tensor Memory Accelerator (ApproxTrain Sec. V-B,
// Algorithm 2, the per-operand half of the product).  Memory-bound: 4 bytes
// read and 4 (packed words) or 8 (two planes) written per element.  Operands stored row-fast are decoded in
// place order; k-fast ones go through a shared-memory transpose so that both
// reads and writes stay coalesced.
#include "decode_unit.cuh"

namespace amsim {
namespace kern {

namespace {

// The predecode pass as its own launch (used before data-parallel GEMM
// launches and when a cooperative launch is not available).
__global__ void __launch_bounds__(256) predecode_kernel(const __grid_constant__ DecodeParams p)
{
    // Sources may be outputs of the previous launch on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ uint32_t t_off[kDecodeTileK][kDecodePitch];
    __shared__ float t_scl[kDecodeTileK][kDecodePitch];
    for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x)
        decode_unit(p, t, t_off, t_scl, (int)threadIdx.x, [] { __syncthreads(); });
}

}  // namespace

int launch_predecode(const DecodeParams &p, int sms, cudaStream_t st)
{
    if (p.tiles <= 0) return AMSIM_OK;
    // The GEMM launches around this one run with the largest shared-memory
    // carve-out; asking for the same one spares the SMs a reconfiguration
    // between the launches.
    static bool carveout_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64 && !carveout_set[dev]) {
        cudaFuncSetAttribute(predecode_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        cudaGetLastError();
        carveout_set[dev] = true;
    }
    // one resident wave (four blocks per SM), so that every block has started,
    // and the dependent GEMM is launched, while the first blocks still run
    long long blocks = p.tiles;
    const long long cap = (long long)sms * 4;
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    for (int pdl = 1; pdl >= 0; --pdl) {
        cfg.attrs = pdl ? &attr : nullptr;
        cfg.numAttrs = pdl ? 1 : 0;
        cudaError_t e = cudaLaunchKernelEx(&cfg, predecode_kernel, p);
        if (e == cudaSuccess) {
            count_launch();
            return AMSIM_OK;
        }
        cudaGetLastError();
    }
    return AMSIM_ECUDA;
}

}  // namespace kern
}  // namespace amsim
