// Elementwise AMSim products c[i] = AMSim(a[i], b[i]) (ApproxTrain Sec. V-B,
// Algorithm 2), bit-exact.  HBM-bound: 12 bytes per element; the narrowed LUT
// (<= 64 KB for M <= 7) stays in L1 through read-only loads.
#include <algorithm>

#include "amsim_internal.h"

namespace {

template <int W>
__device__ __forceinline__ uint32_t narrowed_at(const void *table, uint32_t idx)
{
    if constexpr (W == 8) return __ldg(static_cast<const uint8_t *>(table) + idx);
    else if constexpr (W == 16) return __ldg(static_cast<const uint16_t *>(table) + idx);
    else return __ldg(static_cast<const uint32_t *>(table) + idx);
}

// Algorithm 2 on bit patterns: sign XOR; index from the concatenated top-M
// fraction bits; zero if e0 = ea+eb-127 <= 0 or an input is zero/denormal;
// infinity if the exponent reaches 255 (before or through the carry); NaN
// propagation and Inf*0 as stated in the ABI header.
template <int W>
__device__ __forceinline__ uint32_t amsim_bits(uint32_t x, uint32_t y, const void *table, int M, int shift)
{
    const uint32_t s = (x ^ y) & 0x80000000u;
    const uint32_t ex = (x >> 23) & 0xFFu, ey = (y >> 23) & 0xFFu;
    const uint32_t fx = x & 0x7FFFFFu, fy = y & 0x7FFFFFu;
    const uint32_t idx = ((fx >> (23 - M)) << M) | (fy >> (23 - M));
    const uint32_t entry = narrowed_at<W>(table, idx) << shift;
    const bool nan_in = (ex == 255u && fx) || (ey == 255u && fy);
    const bool inf_in = (ex == 255u) || (ey == 255u);
    const bool zero_in = (ex == 0u) || (ey == 0u);
    const int e0 = (int)ex + (int)ey - 127;
    const int e = e0 + (int)(entry >> 23);
    if (nan_in || (inf_in && zero_in)) return 0x7FC00000u;
    if (inf_in) return s | 0x7F800000u;
    if (zero_in || e0 <= 0) return s;
    if (e >= 255) return s | 0x7F800000u;
    return s | ((uint32_t)e << 23) | (entry & 0x7FFFFFu);
}

// The same in a (1, E, M) format with E < 8 (Sec. V-B, last paragraph): each
// operand's exponent is cast first -- fp32 biased exponent e below f.lo is a
// zero, above f.hi an infinity, else re-biased to c = e - 127 + B -- and
// Algorithm 2 runs with bias B and all-ones exponent 2^E - 1; the result's
// exponent is re-biased back to fp32's.
template <int W>
__device__ __forceinline__ uint32_t amsim_bits_fmt(uint32_t x, uint32_t y, const void *table, int M, int shift,
                                                   const ExpFormat &f)
{
    const uint32_t s = (x ^ y) & 0x80000000u;
    const uint32_t ex = (x >> 23) & 0xFFu, ey = (y >> 23) & 0xFFu;
    const uint32_t fx = x & 0x7FFFFFu, fy = y & 0x7FFFFFu;
    const bool nan_in = (ex == 255u && fx) || (ey == 255u && fy);
    const bool inf_in = (int)ex > f.hi || (int)ey > f.hi;          // fp32 infinities included
    const bool zero_in = (int)ex < f.lo || (int)ey < f.lo;         // zero and denormal included
    if (nan_in || (inf_in && zero_in)) return 0x7FC00000u;
    if (inf_in) return s | 0x7F800000u;
    if (zero_in) return s;
    const uint32_t idx = ((fx >> (23 - M)) << M) | (fy >> (23 - M));
    const uint32_t entry = narrowed_at<W>(table, idx) << shift;
    const int e0 = ((int)ex - 127 + f.bias) + ((int)ey - 127 + f.bias) - f.bias;
    if (e0 <= 0) return s;
    if (e0 >= f.all_ones) return s | 0x7F800000u;
    const int e = e0 + (int)(entry >> 23);
    if (e >= f.all_ones) return s | 0x7F800000u;
    return s | ((uint32_t)(e - f.bias + 127) << 23) | (entry & 0x7FFFFFu);
}

template <int W>
__global__ void __launch_bounds__(256) amsim_mul_fmt_kernel(const float *__restrict__ a, const float *__restrict__ b,
                                                            float *c, int64_t n, const void *table, int M, int shift,
                                                            const ExpFormat f)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
        c[j] = __uint_as_float(amsim_bits_fmt<W>(__float_as_uint(a[j]), __float_as_uint(b[j]), table, M, shift, f));
}

template <int W>
__global__ void __launch_bounds__(256) amsim_mul_kernel(const float *__restrict__ a, const float *__restrict__ b,
                                                        float *c, int64_t n, const void *table, int M, int shift,
                                                        bool vec4)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (vec4) {
        const int64_t n4 = n >> 2;
        for (int64_t j = i; j < n4; j += stride) {
            uint4 x = __ldcs(reinterpret_cast<const uint4 *>(a) + j);
            uint4 y = __ldcs(reinterpret_cast<const uint4 *>(b) + j);
            uint4 r;
            r.x = amsim_bits<W>(x.x, y.x, table, M, shift);
            r.y = amsim_bits<W>(x.y, y.y, table, M, shift);
            r.z = amsim_bits<W>(x.z, y.z, table, M, shift);
            r.w = amsim_bits<W>(x.w, y.w, table, M, shift);
            __stcs(reinterpret_cast<uint4 *>(c) + j, r);
        }
        i += n4 << 2;
    }
    for (int64_t j = i; j < n; j += stride) {
        uint32_t r = amsim_bits<W>(__float_as_uint(a[j]), __float_as_uint(b[j]), table, M, shift);
        c[j] = __uint_as_float(r);
    }
}

}  // namespace

extern "C" int amsim_mul(const float *a, const float *b, float *c, int64_t n, amsim_lut_t lut,
                         amsim_stream_t stream)
{
    if (n < 0) return AMSIM_EINVAL;
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    if (n == 0) return AMSIM_OK;
    if (!a || !b || !c) return AMSIM_EINVAL;
    int dev = lut->device, sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return AMSIM_ECUDA;
    const bool vec4 = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                        reinterpret_cast<uintptr_t>(c)) & 15u) == 0;
    const int64_t work = vec4 ? (n + 3) / 4 : n;
    int64_t blocks = (work + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (lut->exp_bits != 8) {
        const ExpFormat f = exp_format(lut->exp_bits);
        blocks = std::min<int64_t>((n + 255) / 256, cap);
        if (lut->width_bits == 8)
            amsim_mul_fmt_kernel<8><<<(unsigned)blocks, 256, 0, st>>>(a, b, c, n, lut->d_narrow, lut->M, lut->shift, f);
        else if (lut->width_bits == 16)
            amsim_mul_fmt_kernel<16><<<(unsigned)blocks, 256, 0, st>>>(a, b, c, n, lut->d_narrow, lut->M, lut->shift, f);
        else
            amsim_mul_fmt_kernel<32><<<(unsigned)blocks, 256, 0, st>>>(a, b, c, n, lut->d_narrow, lut->M, lut->shift, f);
        rc = amsim::cuda_status(cudaGetLastError());
        if (rc == AMSIM_OK) amsim::count_launch();
        return rc;
    }
    switch (lut->width_bits) {
    case 8:
        amsim_mul_kernel<8><<<(unsigned)blocks, 256, 0, st>>>(a, b, c, n, lut->d_narrow, lut->M, lut->shift, vec4);
        break;
    case 16:
        amsim_mul_kernel<16><<<(unsigned)blocks, 256, 0, st>>>(a, b, c, n, lut->d_narrow, lut->M, lut->shift, vec4);
        break;
    default:
        amsim_mul_kernel<32><<<(unsigned)blocks, 256, 0, st>>>(a, b, c, n, lut->d_narrow, lut->M, lut->shift, vec4);
        break;
    }
    rc = amsim::cuda_status(cudaGetLastError());
    if (rc == AMSIM_OK) amsim::count_launch();
    return rc;
}
