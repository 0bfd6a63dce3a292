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
    constexpr int TR = kDecodeTileR, TK = kDecodeTileK, PITCH = TR + 1;   // odd pitch: conflict-free columns
    __shared__ uint32_t t_off[TK][PITCH];
    __shared__ float t_scl[TK][PITCH];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;    // 32 x 8
    for (long long t = blockIdx.x; t < p.tiles; t += gridDim.x) {
        int j = 0;
        while (j + 1 < p.njobs && t >= p.job[j + 1].tile0) ++j;
        const DecodeJob &d = p.job[j];
        const long long lt = t - d.tile0;
        const long long per_b = (long long)d.tiles_r * d.tiles_k;
        const int b = (int)(lt / per_b);
        const int rem = (int)(lt - (long long)b * per_b);
        const int r0 = (rem / d.tiles_k) * TR, k0 = (rem % d.tiles_k) * TK;
        const float *src = d.src + (long long)b * d.bs;
        uint32_t *po = d.plane + (size_t)b * 2 * d.K * d.rows_pad;
        float *ps = reinterpret_cast<float *>(po + (size_t)d.K * d.rows_pad);
        int big = 0;
        if (d.s_row == 1 && d.rdiv >= d.rows && d.kdiv >= d.K && d.roff == 0) {
            // row-fast dense source: lanes walk rows in both the read and the write
            float v[TR / 32][TK / 8];
#pragma unroll
            for (int h = 0; h < TR / 32; ++h)
#pragma unroll
                for (int i = 0; i < TK / 8; ++i) {
                    const int r = r0 + tx + 32 * h, k = k0 + ty + 8 * i;
                    v[h][i] = (r < d.rows && k < d.K) ? __ldcs(src + r + (long long)k * d.s_k) : 0.0f;
                }
#pragma unroll
            for (int h = 0; h < TR / 32; ++h)
#pragma unroll
                for (int i = 0; i < TK / 8; ++i) {
                    const int r = r0 + tx + 32 * h, k = k0 + ty + 8 * i;
                    if (r < d.rows && k < d.K) {
                        uint32_t o;
                        float s;
                        decode(v[h][i], p.M, d.offshift, o, s, big);
                        po[(size_t)k * d.rows_pad + r] = o;
                        ps[(size_t)k * d.rows_pad + r] = s;
                    }
                }
        } else {
            // lanes walk k in the read (rows ty, ty + 8, ...), rows in the write
            const int k = k0 + tx;
            const bool kok = k < d.K;
            const long long koff = kok ? (long long)(k / d.kdiv) * d.s_khi + (long long)(k % d.kdiv) * d.s_k : 0;
            int rh = (r0 + ty) / d.rdiv, rl = (r0 + ty) - rh * d.rdiv;     // (r / rdiv, r % rdiv), stepped by 8
            float v[TR / 8];
            bool ok[TR / 8];
#pragma unroll
            for (int i = 0; i < TR / 8; ++i) {
                const int r = r0 + ty + 8 * i;
                const int x = rl + d.roff;
                ok[i] = kok && r < d.rows && x >= 0 && x < d.rlim;   // else a zero operand: offset 0, scale +0
                v[i] = ok[i] ? __ldcs(src + (long long)rh * d.s_rhi + (long long)x * d.s_row + koff) : 0.0f;
                rl += 8;
                while (rl >= d.rdiv) { rl -= d.rdiv; ++rh; }
            }
#pragma unroll
            for (int i = 0; i < TR / 8; ++i) {
                uint32_t o = 0;
                float s = 0.0f;
                if (ok[i]) decode(v[i], p.M, d.offshift, o, s, big);
                t_off[tx][ty + 8 * i] = o;
                t_scl[tx][ty + 8 * i] = s;
            }
            __syncthreads();
            // each thread writes 4 consecutive rows of 2 reduction steps, 16-byte stores
            const int rq = (threadIdx.x & 15) * 4, r = r0 + rq;
#pragma unroll
            for (int h = 0; h < TK / 16; ++h) {
                const int kk = (threadIdx.x >> 4) + 16 * h, k2 = k0 + kk;
                if (k2 >= d.K || r >= d.rows) continue;
                const uint4 o4 = make_uint4(t_off[kk][rq], t_off[kk][rq + 1], t_off[kk][rq + 2], t_off[kk][rq + 3]);
                const float4 s4 = make_float4(t_scl[kk][rq], t_scl[kk][rq + 1], t_scl[kk][rq + 2], t_scl[kk][rq + 3]);
                uint32_t *od = po + (size_t)k2 * d.rows_pad + r;
                float *sd = ps + (size_t)k2 * d.rows_pad + r;
                if (r + 4 <= d.rows_pad) {      // rows_pad is a multiple of 4: the pad columns may be written
                    *reinterpret_cast<uint4 *>(od) = o4;
                    *reinterpret_cast<float4 *>(sd) = s4;
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
