// Operand predecode pass of the TMA-fed LUT-GEMM: every dense operand of a
// launch is decoded once into (LUT offset, scale) planes that the GEMM copies
// tile by tile with the Tensor Memory Accelerator (ApproxTrain Sec. V-B,
// Algorithm 2, the per-operand half of the product).  Memory-bound: 4 bytes
// read and 8 written per element.  Operands stored row-fast are decoded in
// place order; k-fast ones go through a shared-memory transpose so that both
// reads and writes stay coalesced.
#include "gemm_kernel.cuh"
#include "predecode.h"

namespace amsim {
namespace kern {

namespace {

__global__ void __launch_bounds__(256) predecode_kernel(const __grid_constant__ DecodeParams p)
{
    // Sources may be outputs of the previous launch on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ uint32_t t_off[kDecodeTile][kDecodeTile + 1];
    __shared__ float t_scl[kDecodeTile][kDecodeTile + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;    // 32 x 8
    for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x) {
        int j = 0;
        while (j + 1 < p.njobs && t >= p.job[j + 1].tile0) ++j;
        const DecodeJob &d = p.job[j];
        const long long lt = t - d.tile0;
        const long long per_b = (long long)d.tiles_r * d.tiles_k;
        const int b = (int)(lt / per_b);
        const int rem = (int)(lt - (long long)b * per_b);
        const int r0 = (rem / d.tiles_k) * kDecodeTile, k0 = (rem % d.tiles_k) * kDecodeTile;
        const float *src = d.src + (long long)b * d.bs;
        uint32_t *po = d.plane + (size_t)b * 2 * d.K * d.rows_pad;
        float *ps = reinterpret_cast<float *>(po + (size_t)d.K * d.rows_pad);
        int big = 0;
        if (d.s_row == 1 && d.rdiv >= d.rows && d.kdiv >= d.K && d.roff == 0) {
            // row-fast dense source: lanes walk rows in both the read and the write
            const int r = r0 + tx;
#pragma unroll
            for (int i = 0; i < kDecodeTile / 8; ++i) {
                const int k = k0 + ty + 8 * i;
                if (r < d.rows && k < d.K) {
                    uint32_t o;
                    float s;
                    decode(__ldcs(src + r + (long long)k * d.s_k), p.M, d.offshift, o, s, big);
                    po[(size_t)k * d.rows_pad + r] = o;
                    ps[(size_t)k * d.rows_pad + r] = s;
                }
            }
        } else {
            // lanes walk k in the read, rows in the write
            const int k = k0 + tx;
            const long long koff = k < d.K ? (long long)(k / d.kdiv) * d.s_khi + (long long)(k % d.kdiv) * d.s_k : 0;
#pragma unroll
            for (int i = 0; i < kDecodeTile / 8; ++i) {
                const int rr = ty + 8 * i, r = r0 + rr;
                uint32_t o = 0;
                float s = 0.0f;
                if (r < d.rows && k < d.K) {
                    const int rl = r % d.rdiv + d.roff;
                    if (rl >= 0 && rl < d.rlim)   // else a zero operand: offset 0, scale +0
                        decode(__ldcs(src + (long long)(r / d.rdiv) * d.s_rhi + (long long)rl * d.s_row + koff),
                               p.M, d.offshift, o, s, big);
                }
                t_off[tx][rr] = o;
                t_scl[tx][rr] = s;
            }
            __syncthreads();
            const int r = r0 + tx;
#pragma unroll
            for (int i = 0; i < kDecodeTile / 8; ++i) {
                const int kk = ty + 8 * i, k2 = k0 + kk;
                if (r < d.rows && k2 < d.K) {
                    po[(size_t)k2 * d.rows_pad + r] = t_off[kk][tx];
                    ps[(size_t)k2 * d.rows_pad + r] = t_scl[kk][tx];
                }
            }
            __syncthreads();
        }
        // every thread of the warp takes part; one store per warp that saw a large element
        if (__any_sync(0xFFFFFFFFu, big) && tx == 0) *d.flag = p.epoch;
    }
}

}  // namespace

int launch_predecode(const DecodeParams &p, int sms, cudaStream_t st)
{
    if (p.tiles <= 0) return AMSIM_OK;
    long long blocks = p.tiles;
    const long long cap = (long long)sms * 8;
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
