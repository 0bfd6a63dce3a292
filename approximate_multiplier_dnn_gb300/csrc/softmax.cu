// Exact fp32 row softmax between the two attention contractions.  Not an
// approximate operation: it only carries the scores S = Q K^T / sqrt(d) to the
// probabilities P that the second contraction multiplies with V.
#include "amsim_internal.h"

namespace {

// One warp per row; three passes over the row (max, sum of exp, normalise).
__global__ void __launch_bounds__(256) softmax_rows_kernel(const float *S, float *P, long long rows, int cols)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const float *s = S + r * cols;
        float *o = P + r * cols;
        float m = -INFINITY;
        for (int c = lane; c < cols; c += 32) m = fmaxf(m, s[c]);
        for (int d = 16; d; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, d));
        float sum = 0.0f;
        for (int c = lane; c < cols; c += 32) sum += expf(s[c] - m);
        for (int d = 16; d; d >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, d);
        const float inv = 1.0f / sum;
        for (int c = lane; c < cols; c += 32) o[c] = expf(s[c] - m) * inv;
    }
}

// dS = P * (dP - sum_c P dP) per row: the gradient of the row softmax, one
// warp per row (two passes: the dot product, then the elementwise result).
__global__ void __launch_bounds__(256) softmax_rows_backward_kernel(const float *P, const float *dP, float *dS,
                                                                   long long rows, int cols)
{
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const float *p = P + r * cols, *g = dP + r * cols;
        float *o = dS + r * cols;
        float dot = 0.0f;
        for (int c = lane; c < cols; c += 32) dot = fmaf(p[c], g[c], dot);
        for (int d = 16; d; d >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, d);
        for (int c = lane; c < cols; c += 32) o[c] = p[c] * (g[c] - dot);
    }
}

int row_blocks(long long rows, long long *blocks)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AMSIM_ECUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return AMSIM_ECUDA;
    long long b = (rows + 7) / 8;
    if (b > (long long)sms * 16) b = (long long)sms * 16;
    *blocks = b;
    return AMSIM_OK;
}

}  // namespace

extern "C" int amsim_softmax_rows_backward(const float *P, const float *dP, float *dS, int64_t rows, int cols,
                                           amsim_stream_t stream)
{
    if (rows < 0 || cols < 0) return AMSIM_EINVAL;
    if (rows == 0 || cols == 0) return AMSIM_OK;
    if (!P || !dP || !dS) return AMSIM_EINVAL;
    long long blocks = 0;
    int rc = row_blocks(rows, &blocks);
    if (rc) return rc;
    softmax_rows_backward_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(P, dP, dS, rows,
                                                                                                  cols);
    rc = amsim::cuda_status(cudaGetLastError());
    if (rc == AMSIM_OK) amsim::count_launch();
    return rc;
}

extern "C" int amsim_softmax_rows(const float *S, float *P, int64_t rows, int cols, amsim_stream_t stream)
{
    if (rows < 0 || cols < 0) return AMSIM_EINVAL;
    if (rows == 0 || cols == 0) return AMSIM_OK;
    if (!S || !P) return AMSIM_EINVAL;
    long long blocks = 0;
    int rc = row_blocks(rows, &blocks);
    if (rc) return rc;
    softmax_rows_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(S, P, rows, cols);
    rc = amsim::cuda_status(cudaGetLastError());
    if (rc == AMSIM_OK) amsim::count_launch();
    return rc;
}
