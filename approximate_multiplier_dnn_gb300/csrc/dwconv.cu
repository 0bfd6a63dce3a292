// Depthwise Conv2D with AMSim products: forward, preceding-layer gradient and
// weight gradient (ApproxTrain Sec. III, Table I lists depthwise convolution
// among the layer types; every product is the AMSim product of Sec. V-B,
// Algorithm 2, accumulated in fp32).  The input has C channels and the filter
// w[r][s][c][d] a channel multiplier D, so there are K = C*D output channels
// and output channel k = c*D + d reads input channel c only:
//   y[n,p,q,c*D+d] = sum_{r,s}   AMSim(x[n, p*sh-ph+r*dh, q*sw-pw+s*dw, c], w[r,s,c,d])
//   dx[n,h,w,c]    = sum_{r,s,d} AMSim(dy[n,p,q,c*D+d], w[r,s,c,d]),
//                    p = (h+ph-r*dh)/sh, q = (w+pw-s*dw)/sw where integral and in range
//   dw[r,s,c,d]    = sum_{n,p,q} AMSim(x[n, p*sh-ph+r*dh, q*sw-pw+s*dw, c], dy[n,p,q,c*D+d])
// Operand order (first operand = high LUT index bits): (x, w), (dy, w), (x, dy).
//
// An output sums only R*S (or R*S*D) products, so this is a stencil, not a
// GEMM, and there is no contraction to tile for the tensor cores.  Kernels:
//  * dw_tile_kernel (dwconv_kernel.cuh; 3x3 filter, unit stride and dilation,
//    D = 1, channels a multiple of 4): a CTA stages a halo tile of 16 channels
//    of the activation (10 x 66 positions for an 8 x 64 output tile; narrower
//    layers take taller tiles of the same 512 outputs) in shared memory, each
//    element packed once into one word: sign and exponent bits (the signed
//    power-of-two scale, NaN kept as NaN), the rest the LUT byte offset of its
//    truncated mantissa.  In the forward and data-gradient passes a warp works
//    on one channel, so the filter tap is the same on all 32 lanes: every LUT
//    load of the warp reads one row of the table (the row-broadcast schedule
//    of the GEMM kernels).  A lane keeps a 2-column x 8-row block of outputs
//    and walks the 10 input rows once, so each staged word feeds up to 18
//    products.  Outputs go back through shared memory as 16-byte stores of
//    4 channels.  The weight gradient stages the output gradient too (8
//    channels per tile, one per warp, so that two CTAs fit on an SM) and
//    accumulates the 9 taps per lane across all tiles of its share; its
//    products have no uniform operand, so its lookups meet bank conflicts.
//    Thread 0 copies the next tile's raw boxes with a tensor copy (zero fill
//    outside the tensor) while the CTA computes the current tile.  Closed-form
//    variants (dwconv_alu.cu) compute the built-in multipliers in registers.
//  * dw_s2_kernel and dw_s2d_kernel (dwconv_s2.cu): the same scheme for 3x3
//    filters at stride 2 (the data gradient for padding 1).
//  * dw_direct_kernel (every other geometry): a warp takes one pixel and 32
//    consecutive channels, operands read as coalesced rows and decoded per
//    product, the LUT staged in shared memory when it fits.
// The weight gradient's reduction over N*P*Q is split into G shares written to
// scratch and added in share order by dw_sum_kernel, so results are
// deterministic for a given scratch size.
#include <algorithm>

#include "dwconv_kernel.cuh"

namespace {

using namespace amsim::dw;
using amsim::kern::expand;
using amsim::kern::lut_ld;
using amsim::kern::fmt_product;
using amsim::kern::fmt_scale_bits;

// ------------------------------------------------------------------ geometry
struct DwGeo {
    int N, H, W, C, D, K, R, S, sh, sw, ph, pw, dh, dw, P, Q;
};

int dw_geometry(const amsim_conv_desc *d, DwGeo *g)
{
    if (!d) return AMSIM_EINVAL;
    *g = {d->N, d->H, d->W, d->C, 0, d->K, d->R, d->S, d->stride_h, d->stride_w, d->pad_h, d->pad_w,
          d->dil_h, d->dil_w, 0, 0};
    if (g->N < 0 || g->H < 1 || g->W < 1 || g->C < 1 || g->K < 1 || g->R < 1 || g->S < 1) return AMSIM_EINVAL;
    if (g->K % g->C) return AMSIM_EINVAL;          // K = C * D
    if (g->sh < 1 || g->sw < 1 || g->ph < 0 || g->pw < 0 || g->dh < 1 || g->dw < 1) return AMSIM_EINVAL;
    g->D = g->K / g->C;
    const long long hh = (long long)g->H + 2LL * g->ph - (long long)g->dh * (g->R - 1) - 1;
    const long long ww = (long long)g->W + 2LL * g->pw - (long long)g->dw * (g->S - 1) - 1;
    if (hh < 0 || ww < 0) return AMSIM_EINVAL;
    g->P = (int)(hh / g->sh + 1);
    g->Q = (int)(ww / g->sw + 1);
    // coordinates are 32-bit inside the kernels, addresses 64-bit
    const long long px = (long long)g->N * std::max((long long)g->H * g->W, (long long)g->P * g->Q);
    if (px > 0x3FFFFFFFLL || (long long)g->R * g->S * g->K > 0x3FFFFFFFLL) return AMSIM_EUNSUPPORTED;
    if ((long long)g->R * g->dh > 0x3FFFFFFFLL || (long long)g->S * g->dw > 0x3FFFFFFFLL) return AMSIM_EUNSUPPORTED;
    return AMSIM_OK;
}

// ------------------------------------------------------------------ direct kernel
struct DwDirectParams {
    DwGeo g;
    const float *a, *b;
    float *out;
    const void *table;     // narrowed LUT, [first operand][second operand] of the pass
    int M, wlog;
    long long items;       // mode 0/1: pixels x channel groups; mode 2: taps x shares x channel groups
    int groups;            // 32-channel groups of the lanes' channel dimension
    int table_bytes;       // staged table bytes (0: read through the cache)
    int grid_taps;         // data gradient: unit dilation, so the taps on the stride grid can be enumerated
    int G;                 // mode 2: shares of the N*P*Q reduction
    ExpFormat fmt;         // (1, E, M) format with E < 8 when fmt.on
};

// Signed power-of-two scale of an operand (zero and denormal inputs a signed
// zero, infinity infinite, NaN a NaN).
__device__ __forceinline__ float dw_scale(uint32_t x)
{
    const bool nan = ((x >> 23) & 0xFFu) == 255u && (x & 0x7FFFFFu);
    return __uint_as_float(nan ? 0x7FC00000u : (x & 0xFF800000u));
}

// Whether v = u * s for an integer u in [0, lim) (u returned); s >= 1.
__device__ __forceinline__ bool dw_on_grid(int v, int s, int lim, int &u)
{
    if (v < 0) return false;
    if (s == 1) u = v;
    else if (s == 2) { if (v & 1) return false; u = v >> 1; }
    else { u = v / s; if (u * s != v) return false; }
    return u < lim;
}

// AMSim product from the staged (GL false) or global (GL true) narrowed table
// [first][second], rounded to fp32 before it is added; in a (1, E, M) format
// with E < 8 the operands are cast first and the product is the format's
// (fmt_product).
template <int W, bool GL>
__device__ __forceinline__ float dw_product_t(float first, float second, const uint8_t *lut, int M, int wlog,
                                              const ExpFormat &f)
{
    const uint32_t xa = __float_as_uint(first), xb = __float_as_uint(second);
    const uint32_t idx = ((((xa & 0x7FFFFFu) >> (23 - M)) << M) | ((xb & 0x7FFFFFu) >> (23 - M))) << wlog;
    const float v = expand<W>(lut_ld<W, GL>(lut, idx));
    if (f.on)
        return fmt_product(v, fmul_ftz(__uint_as_float(fmt_scale_bits(xa, f.lo, f.hi, f.off_u)),
                                       __uint_as_float(fmt_scale_bits(xb, f.lo, f.hi, f.off_l))), f);
    return __fmul_rn(v, fmul_ftz(dw_scale(xa), dw_scale(xb)));
}

// Whether an operand stays finite through the exponent cast (fp32 biased
// exponent at most hi; hi = 254 for fp32's own exponent: not Inf or NaN).
__device__ __forceinline__ bool dw_cast_finite(float v, int hi) { return (int)((__float_as_uint(v) >> 23) & 0xFFu) <= hi; }

// Direct kernel: a warp takes one pixel (or, for the weight gradient, one
// filter tap and one share of the pixels) and 32 consecutive channels, so both
// operands are read as coalesced rows; the table sits in shared memory unless
// it is wider than 16 bits or larger than 64 KB (then the read-only cache).
template <int W, int MODE, bool GL>
__global__ void __launch_bounds__(256) dw_direct_kernel(const __grid_constant__ DwDirectParams p)
{
    extern __shared__ __align__(16) uint8_t dsmem[];
    const DwGeo &g = p.g;
    const int lane = threadIdx.x & 31;
    const uint8_t *lut = static_cast<const uint8_t *>(p.table);
    if constexpr (!GL) {
        const uint4 *src = static_cast<const uint4 *>(p.table);
        uint4 *dst = reinterpret_cast<uint4 *>(dsmem);
        for (int i = threadIdx.x; i < (p.table_bytes + 15) >> 4; i += blockDim.x) dst[i] = __ldg(src + i);
        lut = dsmem;
    }
    // data gradient: per input channel, whether all its filter taps are finite
    // (then taps off the stride grid, whose products are signed zeros, need no visit)
    uint8_t *finite = dsmem + ((p.table_bytes + 15) & ~15);
    if constexpr (MODE == 1) {
        for (int c = threadIdx.x; c < g.C; c += blockDim.x) {
            bool ok = true;
            for (int t = 0; t < g.R * g.S * g.D; ++t) {
                const int tap = t / g.D, d = t - tap * g.D;
                ok = ok && dw_cast_finite(__ldg(p.b + ((long long)tap * g.C + c) * g.D + d), p.fmt.hi);
            }
            finite[c] = ok;
        }
    }
    __syncthreads();
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int warp0 = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if constexpr (MODE == 0) {
        // a warp takes output pixels warp0, warp0 + warps, ... (32-bit: N*P*Q < 2^30),
        // each for every 32-channel group; consecutive warps take neighbouring pixels
        const int npix = g.N * g.P * g.Q;
        for (int pix = warp0; pix < npix; pix += warps) {
            const int q = pix % g.Q, t = pix / g.Q;
            const int pp = t % g.P, n = t / g.P;
            for (int kg = 0; kg < p.groups; ++kg) {
                const int k = kg * 32 + lane;
                if (k >= g.K) continue;
                const int c = k / g.D, d = k - c * g.D;
                const float *xn = p.a + (long long)n * g.H * g.W * g.C + c;
                float acc = 0.0f;
                for (int r = 0; r < g.R; ++r) {
                    const int h = pp * g.sh - g.ph + r * g.dh;
                    const bool hin = (unsigned)h < (unsigned)g.H;
                    for (int s = 0; s < g.S; ++s) {
                        const int w = q * g.sw - g.pw + s * g.dw;
                        const float wv = __ldg(p.b + ((long long)(r * g.S + s) * g.C + c) * g.D + d);
                        const bool in = hin && (unsigned)w < (unsigned)g.W;
                        // a padded tap multiplies a zero operand: a signed zero, which leaves
                        // the sum unchanged, unless the weight is infinite or NaN (then NaN)
                        if (!in && dw_cast_finite(wv, p.fmt.hi)) continue;
                        const float xv = in ? __ldg(xn + ((long long)h * g.W + w) * g.C) : 0.0f;
                        acc = __fadd_rn(acc, dw_product_t<W, GL>(xv, wv, lut, p.M, p.wlog, p.fmt));
                    }
                }
                p.out[(long long)pix * g.K + k] = acc;
            }
        }
    } else if constexpr (MODE == 1) {
        // a warp takes input pixels warp0, warp0 + warps, ..., each for every 32-channel group
        const int npix = g.N * g.H * g.W;
        for (int pix = warp0; pix < npix; pix += warps) {
            const int w = pix % g.W, t = pix / g.W;
            const int h = t % g.H, n = t / g.H;
            for (int cg = 0; cg < p.groups; ++cg) {
                const int c = cg * 32 + lane;
                if (c >= g.C) continue;
                const float *dyn = p.a + (long long)n * g.P * g.Q * g.K + (long long)c * g.D;
                float acc = 0.0f;
                if (p.grid_taps && finite[c]) {
                    // unit dilation: the taps on the stride grid are r = r0, r0 + sh, ... with
                    // r0 = (h + ph) mod sh, and likewise s; the others add signed zeros
                    const int r0 = (h + g.ph) % g.sh, s0 = (w + g.pw) % g.sw;
                    for (int r = r0; r < g.R; r += g.sh) {
                        const int pr = (h + g.ph - r) / g.sh;
                        if (pr < 0 || pr >= g.P) continue;
                        for (int s = s0; s < g.S; s += g.sw) {
                            const int qs = (w + g.pw - s) / g.sw;
                            if (qs < 0 || qs >= g.Q) continue;
                            const float *dyp = dyn + ((long long)pr * g.Q + qs) * g.K;
                            const float *wp = p.b + ((long long)(r * g.S + s) * g.C + c) * g.D;
                            for (int d = 0; d < g.D; ++d)
                                acc = __fadd_rn(acc, dw_product_t<W, GL>(__ldg(dyp + d), __ldg(wp + d), lut, p.M,
                                                                         p.wlog, p.fmt));
                        }
                    }
                    p.out[(long long)pix * g.C + c] = acc;
                    continue;
                }
                for (int r = 0; r < g.R; ++r) {
                    int pr = 0;
                    const bool rin = dw_on_grid(h + g.ph - r * g.dh, g.sh, g.P, pr);
                    for (int s = 0; s < g.S; ++s) {
                        int qs = 0;
                        const bool in = rin && dw_on_grid(w + g.pw - s * g.dw, g.sw, g.Q, qs);
                        const float *dyp = dyn + ((long long)pr * g.Q + qs) * g.K;
                        for (int d = 0; d < g.D; ++d) {
                            const float wv = __ldg(p.b + ((long long)(r * g.S + s) * g.C + c) * g.D + d);
                            // a tap between stride positions or past the edge multiplies a zero
                            // operand: a signed zero, which leaves the sum unchanged, unless the
                            // weight is infinite or NaN (then NaN)
                            if (!in && dw_cast_finite(wv, p.fmt.hi)) continue;
                            const float dyv = in ? __ldg(dyp + d) : 0.0f;
                            acc = __fadd_rn(acc, dw_product_t<W, GL>(dyv, wv, lut, p.M, p.wlog, p.fmt));
                        }
                    }
                }
                p.out[(long long)pix * g.C + c] = acc;
            }
        }
    } else {
        for (long long it = warp0; it < p.items; it += warps) {
            // item: (filter tap, share of the N*P*Q pixels, 32-channel group); each lane
            // sums its channel over the share's pixels in order
            const int kg = (int)(it % p.groups);
            long long rest = it / p.groups;
            const int share = (int)(rest % p.G);
            const int tap = (int)(rest / p.G);
            const int r = tap / g.S, s = tap - r * g.S;
            const int k = kg * 32 + lane;
            if (k >= g.K) continue;
            const int c = k / g.D;
            const long long npq = (long long)g.N * g.P * g.Q;
            const long long b0 = npq * share / p.G, b1 = npq * (share + 1) / p.G;
            float acc = 0.0f;
            if (b0 < b1) {
                int q = (int)(b0 % g.Q);
                const long long t = b0 / g.Q;
                int pp = (int)(t % g.P), n = (int)(t / g.P);
                for (long long pix = b0; pix < b1; ++pix) {
                    const int h = pp * g.sh - g.ph + r * g.dh, w = q * g.sw - g.pw + s * g.dw;
                    const float dyv = __ldg(p.b + pix * g.K + k);
                    const bool in = (unsigned)h < (unsigned)g.H && (unsigned)w < (unsigned)g.W;
                    if (in || !dw_cast_finite(dyv, p.fmt.hi)) {
                        const float xv = in ? __ldg(p.a + (((long long)n * g.H + h) * g.W + w) * g.C + c) : 0.0f;
                        acc = __fadd_rn(acc, dw_product_t<W, GL>(xv, dyv, lut, p.M, p.wlog, p.fmt));
                    }
                    if (++q == g.Q) {
                        q = 0;
                        if (++pp == g.P) { pp = 0; ++n; }
                    }
                }
            }
            p.out[((long long)share * g.R * g.S + tap) * g.K + k] = acc;
        }
    }
}

// out[i] = sum over shares g = 0 .. G-1 of part[g*n + i], in share order (the
// loads of eight shares are issued together, the adds stay in order).
__global__ void __launch_bounds__(256) dw_sum_kernel(const float *__restrict__ part, float *__restrict__ out,
                                                     long long n, int G)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        float v = part[i];
        int g = 1;
        for (; g + 8 <= G; g += 8) {
            float t[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) t[u] = __ldg(part + (long long)(g + u) * n + i);
#pragma unroll
            for (int u = 0; u < 8; ++u) v += t[u];
        }
        for (; g < G; ++g) v += __ldg(part + (long long)g * n + i);
        out[i] = v;
    }
}

// ------------------------------------------------------------------ host side
int sm_count(int dev)
{
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    return sms;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kDwMaxTileLut = 64 * 1024;   // tables staged by the tiled kernel

// The tiled kernel covers 3x3 and 5x5 filters at unit stride and dilation
// with one filter per channel, channels a multiple of 4, 16-byte aligned
// tensors and a narrowed 8- or 16-bit LUT of at most 64 KB.
bool dw_tile_ok(const DwGeo &g, const amsim_lut_t lut, int which, const float *t0, const float *t1,
                const float *out)
{
    if (g.D != 1 || g.R != g.S || (g.R != 3 && g.R != 5) || g.sh != 1 || g.sw != 1 || g.dh != 1 || g.dw != 1)
        return false;
    if (g.C % 4 || lut->width_bits == 32 || (int)lut->narrow_bytes > kDwMaxTileLut) return false;
    if (lut->exp_bits != 8) return false;         // formats run on the direct kernel
    if (!aligned16(t0) || !aligned16(out)) return false;
    if (which == 2 && !aligned16(t1)) return false;
    return true;
}

// Tensor map of an NHWC fp32 tensor (C channels, H x W positions, N images)
// for boxes of 16 channels x bw columns x bh rows of one image.
bool dw_map(CUtensorMap *map, const float *base, int N, int H, int W, int C, int cb, int bw, int bh)
{
    amsim::TmaRawMap m{};
    m.base = base;
    m.rank = 4;
    m.dims[0] = (uint64_t)C;
    m.dims[1] = (uint64_t)W;
    m.dims[2] = (uint64_t)H;
    m.dims[3] = (uint64_t)std::max(N, 1);
    m.strides[0] = (uint64_t)C * 4;
    m.strides[1] = (uint64_t)W * C * 4;
    m.strides[2] = (uint64_t)H * W * C * 4;
    m.box[0] = (uint32_t)cb;
    m.box[1] = (uint32_t)bw;
    m.box[2] = (uint32_t)bh;
    m.box[3] = 1;
    m.swizzle64 = 0;
    return amsim::encode_tensor_map(map, m) == AMSIM_OK;
}

// The closed-form variants are compiled in dwconv_alu.cu, the 5x5 variants in
// dwconv_k5.cu, the stride-2 kernels in dwconv_s2.cu.
}  // namespace
namespace amsim {
namespace dw {
int launch_s2(int alu, int mode, int width, const DwTileParams &tp, int grid, size_t smem, cudaStream_t st);
size_t s2_smem_bytes(int table_bytes, int mode);
int launch_s2d(int alu, int width, const DwTileParams &tp, int grid, size_t smem, cudaStream_t st);
size_t s2d_smem_bytes(int table_bytes);
extern template int launch_tile<0, 1>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<1, 1>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<2, 1>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<0, 2>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<1, 2>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<2, 2>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<0, 0, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<1, 0, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<2, 0, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<0, 1, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<1, 1, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<2, 1, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<0, 2, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<1, 2, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
extern template int launch_tile<2, 2, 5>(int, const DwTileParams &, int, size_t, cudaStream_t);
}  // namespace dw
}  // namespace amsim
namespace {

template <int MODE>
int launch_tile_any(int alu, int ks, int width, const DwTileParams &tp, int grid, size_t smem, cudaStream_t st)
{
    if (ks == 5)
        return alu == 1   ? launch_tile<MODE, 1, 5>(width, tp, grid, smem, st)
               : alu == 2 ? launch_tile<MODE, 2, 5>(width, tp, grid, smem, st)
                          : launch_tile<MODE, 0, 5>(width, tp, grid, smem, st);
    if (alu == 1) return launch_tile<MODE, 1>(width, tp, grid, smem, st);
    if (alu == 2) return launch_tile<MODE, 2>(width, tp, grid, smem, st);
    return launch_tile<MODE, 0>(width, tp, grid, smem, st);
}

constexpr int kDwDirectMaxLut = 64 * 1024;   // tables the direct kernel stages in shared memory

template <int MODE>
int launch_direct(int width, const DwDirectParams &dp, int grid, cudaStream_t st)
{
    // the staged table, then (data gradient) one flag byte per input channel
    const size_t smem = (size_t)((dp.table_bytes + 15) & ~15) + (MODE == 1 ? (size_t)dp.g.C : 0);
    auto kfn = dp.table_bytes > 0 ? (width == 8 ? dw_direct_kernel<8, MODE, false> : dw_direct_kernel<16, MODE, false>)
             : width == 8          ? dw_direct_kernel<8, MODE, true>
             : width == 16         ? dw_direct_kernel<16, MODE, true>
                                   : dw_direct_kernel<32, MODE, true>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return amsim::cuda_status(e);
    }
    kfn<<<grid, 256, smem, st>>>(dp);
    return amsim::cuda_status(cudaGetLastError());
}

int wlog_of(int width_bits) { return width_bits == 8 ? 0 : width_bits == 16 ? 1 : 2; }

// Shares of the weight gradient's reduction: the count that fills the GPU,
// and the count that fits `ws_bytes` of scratch (at least 1: no scratch).
// The stride-2 tiled kernel covers 3x3 filters at stride 2 and unit dilation
// with one filter per channel, for the forward pass and the weight gradient,
// on the same conditions as the stride-1 kernel.
bool dw_s2_ok(const DwGeo &g, const amsim_lut_t lut, int which, const float *t0, const float *t1,
              const float *out)
{
    if (g.D != 1 || g.R != 3 || g.S != 3 || g.sh != 2 || g.sw != 2 || g.dh != 1 || g.dw != 1) return false;
    // the data gradient's kernel is written for padding 1 (each output parity
    // class then has fixed taps)
    if (which == 1 && (g.ph != 1 || g.pw != 1)) return false;
    if (g.C % 4 || lut->width_bits == 32 || (int)lut->narrow_bytes > kDwMaxTileLut) return false;
    if (lut->exp_bits != 8) return false;         // formats run on the direct kernel
    if (!aligned16(t0) || (which != 2 && !aligned16(out)) || (which == 2 && !aligned16(t1))) return false;
    return true;
}

int dw_staged_lut(const amsim_lut_t lut, int ks);

int s2_ctas_per_sm(const amsim_lut_t lut, int which)
{
    const int per = (int)amsim::dw::s2_smem_bytes(dw_staged_lut(lut, 3), which) + 1024;
    return std::max(1, std::min(2, (228 * 1024) / per));
}

constexpr int kS2Rows = 4, kS2Cols = 64, kS2Ch = 8;   // the stride-2 kernel's tile

struct DwFilterPlan {
    bool tiled;
    int tiles_p, tiles_q, cblocks, tiles;
    int G_want;
    long long outs;        // R*S*K
};

// Resident CTAs of the tiled kernel per SM, from its shared memory (each
// CTA also holds 1 KB of the SM's 228 KB for the system).
// Closed-form variant of the tiled kernel a handle selects for a ks x ks
// filter: 0 the table, 1 Mitchell, 2 exact (amsim_lut_set_closed_form on a
// built-in kind; 3x3 and 5x5 filters).
int dw_alu(const amsim_lut_t lut, int ks)
{
    if (!lut->closed_form || (ks != 3 && ks != 5)) return 0;
    return lut->kind == AMSIM_MITCHELL ? 1 : 2;
}

// Bytes of the LUT the tiled kernel stages (closed forms stage none).
int dw_staged_lut(const amsim_lut_t lut, int ks) { return dw_alu(lut, ks) ? 0 : (int)lut->narrow_bytes; }

int dw_tile_ctas_per_sm(const amsim_lut_t lut, int which, int ks)
{
    const int per = dw_tile_smem(dw_staged_lut(lut, ks), which, ks) + 1024;
    return std::max(1, std::min(2, (228 * 1024) / per));
}

// Tile shape of the tiled kernel for an OH x OW output grid: LQ lanes across
// (2 columns each) by 32 / LQ blocks of 8 rows.  The shape that computes the
// fewest outputs past the grid's edges wins; ties go to the smaller halo,
// then to the wider tile.
struct DwShape {
    int lq_shift, tp, tq, th, tw;
};

DwShape dw_shape(int OH, int OW, int ks)
{
    DwShape best{};
    long long best_cost = -1, best_halo = 0;
    for (int ls = 5; ls >= 2; --ls) {
        const int tq = 2 << ls, tp = kDwRB * (32 >> ls);
        const long long cost = (long long)((OH + tp - 1) / tp) * tp * ((OW + tq - 1) / tq) * tq;
        const long long halo = (long long)(tp + ks - 1) * (tq + ks - 1);
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && halo < best_halo)) {
            best = DwShape{ls, tp, tq, tp + ks - 1, tq + ks - 1};
            best_cost = cost;
            best_halo = halo;
        }
    }
    return best;
}

// kind: 0 direct kernel, 1 tiled kernel, 2 stride-2 tiled kernel.
DwFilterPlan filter_plan(const DwGeo &g, int kind, int sms, const amsim_lut_t lut)
{
    DwFilterPlan f{};
    f.tiled = kind != 0;
    f.outs = (long long)g.R * g.S * g.K;
    if (kind == 2) {
        f.tiles_p = (g.P + kS2Rows - 1) / kS2Rows;
        f.tiles_q = (g.Q + kS2Cols - 1) / kS2Cols;
        f.cblocks = (g.C + kS2Ch - 1) / kS2Ch;
        f.tiles = g.N * f.tiles_p * f.tiles_q;
        const int slots = s2_ctas_per_sm(lut, 2) * sms;
        f.G_want = std::max(1, std::min((slots + f.cblocks - 1) / f.cblocks, f.tiles));
    } else if (kind == 1) {
        const DwShape sh = dw_shape(g.P, g.Q, g.R);
        f.tiles_p = (g.P + sh.tp - 1) / sh.tp;
        f.tiles_q = (g.Q + sh.tq - 1) / sh.tq;
        f.cblocks = (g.C + dw_channel_block(2, g.R) - 1) / dw_channel_block(2, g.R);
        f.tiles = g.N * f.tiles_p * f.tiles_q;
        const int slots = dw_tile_ctas_per_sm(lut, 2, g.R) * sms;
        const int want = (slots + f.cblocks - 1) / f.cblocks;
        f.G_want = std::max(1, std::min(want, f.tiles));
    } else {
        const long long npq = (long long)g.N * g.P * g.Q;
        const long long items = (long long)g.R * g.S * ((g.K + 31) / 32);     // warps per share
        const long long want = (64LL * sms + items - 1) / items;              // about 64 warps per SM
        const long long cap = std::max(1LL, npq / 64);                        // at least 64 pixels a share
        f.G_want = (int)std::max(1LL, std::min(std::min(want, cap), 4096LL));
    }
    return f;
}

int shares_for(const DwFilterPlan &f, size_t ws_bytes)
{
    if (f.G_want <= 1 || f.outs == 0) return 1;
    const long long fit = (long long)(ws_bytes / (size_t)(f.outs * 4));
    return fit >= 2 ? (int)std::min<long long>(fit, f.G_want) : 1;
}

int dw_run(const amsim_conv_desc *desc, int which, const float *t0, const float *t1, float *out, amsim_lut_t lut,
           void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    DwGeo g;
    rc = dw_geometry(desc, &g);
    if (rc) return rc;
    amsim::set_last_path(0);
    const long long n_out = which == 0 ? (long long)g.N * g.P * g.Q * g.K
                          : which == 1 ? (long long)g.N * g.H * g.W * g.C
                                       : (long long)g.R * g.S * g.K;
    if (n_out == 0) return AMSIM_OK;       // N == 0 with the forward or data-gradient pass
    if (!out || (g.N > 0 && (!t0 || !t1))) return AMSIM_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int sms = sm_count(lut->device);
    const int width = lut->width_bits, wlog = wlog_of(width);
    bool tiled = dw_tile_ok(g, lut, which, t0, t1, out);
    int path = tiled ? AMSIM_PATH_DW_TILES : AMSIM_PATH_DW_DIRECT;
    // table orientation [high operand][low operand] of the kernel
    const void *tab_direct = lut->d_narrow;                  // direct kernel: [first][second]
    const void *tab_tiled = which == 2 ? lut->d_narrow : lut->d_narrow_t;   // tiled: [w][act] or [x][dy]

    if (which == 2 && g.N == 0) {
        // empty reduction: every filter gradient element is +0
        rc = amsim::cuda_status(cudaMemsetAsync(out, 0, (size_t)n_out * 4, st));
        if (rc == AMSIM_OK) amsim::set_last_path(path);
        return rc;
    }

    if (!tiled && dw_s2_ok(g, lut, which, t0, t1, out)) {
        // stride 2: forward or weight gradient on the stride-2 tiled kernel
        DwTileParams sp{};
        sp.table = tab_tiled;
        sp.table_bytes = (int)lut->narrow_bytes;
        sp.M = lut->M;
        sp.wlog = wlog;
        sp.N = g.N;
        sp.C = g.C;
        sp.a = t0;
        sp.b = t1;
        sp.expand_mul = 1u << (24 - width);
        sp.IH = g.H; sp.IW = g.W; sp.OH = g.P; sp.OW = g.Q;
        sp.oy = -g.ph; sp.ox = -g.pw;
        sp.tiles_p = (g.P + kS2Rows - 1) / kS2Rows;
        sp.tiles_q = (g.Q + kS2Cols - 1) / kS2Cols;
        sp.cblocks = (g.C + kS2Ch - 1) / kS2Ch;
        sp.tiles = g.N * sp.tiles_p * sp.tiles_q;
        const int alu = dw_alu(lut, 3);
        const int staged = dw_staged_lut(lut, 3);
        if (which == 1) {
            // data gradient: 8 x 64 dx tiles of 16 channels over 5 x 33 dy windows
            sp.IH = g.P; sp.IW = g.Q; sp.OH = g.H; sp.OW = g.W;
            sp.out = out;
            sp.tiles_p = (g.H + 7) / 8;
            sp.tiles_q = (g.W + 63) / 64;
            sp.cblocks = (g.C + 15) / 16;
            sp.tiles = g.N * sp.tiles_p * sp.tiles_q;
            if (dw_map(&sp.amap, t0, g.N, g.P, g.Q, g.C, 16, 33, 5)) {
                const long long total = (long long)sp.tiles * sp.cblocks;
                if (total > 0x7FFFFFFFLL) return AMSIM_EUNSUPPORTED;
                const size_t smem = amsim::dw::s2d_smem_bytes(staged);
                const int per_sm = std::max(1, std::min(2, (int)((228 * 1024) / (smem + 1024))));
                const int grid = (int)std::min<long long>(total, (long long)per_sm * sms);
                rc = amsim::dw::launch_s2d(alu, width, sp, grid, smem, st);
                if (rc == AMSIM_OK) {
                    amsim::count_launch();
                    amsim::set_last_path(AMSIM_PATH_DW_TILES | (alu ? AMSIM_PATH_CLOSED_FORM : 0));
                }
                return rc;
            }
        }
        const bool mapped = which != 1 &&
                            dw_map(&sp.amap, t0, g.N, g.H, g.W, g.C, kS2Ch, 2 * kS2Cols + 1, 2 * kS2Rows + 1) &&
                            (which == 0 || dw_map(&sp.bmap, t1, g.N, g.P, g.Q, g.C, kS2Ch, kS2Cols, kS2Rows));
        if (mapped) {
            const size_t smem = amsim::dw::s2_smem_bytes(staged, which);
            path = AMSIM_PATH_DW_TILES | (alu ? AMSIM_PATH_CLOSED_FORM : 0);
            if (which == 0) {
                sp.out = out;
                sp.G = 1;
                const long long total = (long long)sp.tiles * sp.cblocks;
                if (total > 0x7FFFFFFFLL) return AMSIM_EUNSUPPORTED;
                const int grid = (int)std::min<long long>(total, (long long)s2_ctas_per_sm(lut, 0) * sms);
                rc = amsim::dw::launch_s2(alu, 0, width, sp, grid, smem, st);
                if (rc == AMSIM_OK) amsim::count_launch();
            } else {
                const DwFilterPlan f = filter_plan(g, 2, sms, lut);
                sp.G = shares_for(f, ws_bytes);
                sp.out = sp.G > 1 ? static_cast<float *>(ws) : out;
                rc = amsim::dw::launch_s2(alu, 2, width, sp, sp.cblocks * sp.G, smem, st);
                if (rc == AMSIM_OK) amsim::count_launch();
                if (rc == AMSIM_OK && sp.G > 1) {
                    const int blocks = (int)std::min<long long>((n_out + 255) / 256, 4LL * sms);
                    dw_sum_kernel<<<blocks, 256, 0, st>>>(static_cast<const float *>(ws), out, n_out, sp.G);
                    rc = amsim::cuda_status(cudaGetLastError());
                    if (rc == AMSIM_OK) amsim::count_launch();
                    path |= AMSIM_PATH_STREAMK;
                }
            }
            if (rc == AMSIM_OK) amsim::set_last_path(path);
            return rc;
        }
    }

    DwTileParams tp{};
    if (tiled) {
        tp.table = tab_tiled;
        tp.table_bytes = (int)lut->narrow_bytes;
        tp.M = lut->M;
        tp.wlog = wlog;
        tp.N = g.N;
        tp.C = g.C;
        tp.a = t0;
        tp.expand_mul = 1u << (24 - width);
        // output grid: y (forward), dx (data gradient), dy (weight gradient)
        const int ks = g.R;
        const int cbk = dw_channel_block(which, ks);
        const DwShape sh = which == 1 ? dw_shape(g.H, g.W, ks) : dw_shape(g.P, g.Q, ks);
        tp.lq_shift = sh.lq_shift;
        tp.tp = sh.tp;
        tp.tq = sh.tq;
        tp.tq_shift = sh.lq_shift + 1;
        tp.th = sh.th;
        tp.tw = sh.tw;
        tp.raw_a_bytes = sh.th * sh.tw * cbk * 4;
        bool mapped;
        if (which == 0) {
            tp.IH = g.H; tp.IW = g.W;
            tp.b = t1; tp.out = out;
            tp.OH = g.P; tp.OW = g.Q;
            tp.oy = -g.ph; tp.ox = -g.pw;
            mapped = dw_map(&tp.amap, t0, g.N, g.H, g.W, g.C, cbk, sh.tw, sh.th);
        } else if (which == 1) {
            // dx[h][w] = sum_{r',s'} dy[h + ph - (ks-1) + r'][w + pw - (ks-1) + s'] * w[ks-1 - r'][ks-1 - s']
            tp.IH = g.P; tp.IW = g.Q;
            tp.b = t1; tp.out = out;
            tp.OH = g.H; tp.OW = g.W;
            tp.oy = g.ph - (ks - 1); tp.ox = g.pw - (ks - 1);
            mapped = dw_map(&tp.amap, t0, g.N, g.P, g.Q, g.C, cbk, sh.tw, sh.th);
        } else {
            tp.IH = g.H; tp.IW = g.W;
            tp.b = t1;
            tp.OH = g.P; tp.OW = g.Q;
            tp.oy = -g.ph; tp.ox = -g.pw;
            mapped = dw_map(&tp.amap, t0, g.N, g.H, g.W, g.C, cbk, sh.tw, sh.th) &&
                     dw_map(&tp.bmap, t1, g.N, g.P, g.Q, g.C, cbk, sh.tq, sh.tp);
        }
        if (!mapped) {               // the driver refused a tensor map: the direct kernel
            tiled = false;
            path = AMSIM_PATH_DW_DIRECT;
        }
    }
    if (tiled) {
        tp.tiles_p = (tp.OH + tp.tp - 1) / tp.tp;
        tp.tiles_q = (tp.OW + tp.tq - 1) / tp.tq;
        tp.cblocks = (g.C + dw_channel_block(which, g.R) - 1) / dw_channel_block(which, g.R);
        tp.tiles = g.N * tp.tiles_p * tp.tiles_q;
        const size_t smem = (size_t)dw_tile_smem(dw_staged_lut(lut, g.R), which, g.R);
        const int alu = dw_alu(lut, g.R);
        if (alu) path |= AMSIM_PATH_CLOSED_FORM;
        if (which < 2) {
            const long long total = (long long)tp.tiles * tp.cblocks;
            if (total > 0x7FFFFFFFLL) return AMSIM_EUNSUPPORTED;
            const int grid = (int)std::min<long long>(total, (long long)dw_tile_ctas_per_sm(lut, which, g.R) * sms);
            tp.G = 1;
            rc = which == 0 ? launch_tile_any<0>(alu, g.R, width, tp, grid, smem, st)
                            : launch_tile_any<1>(alu, g.R, width, tp, grid, smem, st);
            if (rc == AMSIM_OK) amsim::count_launch();
        } else {
            const DwFilterPlan f = filter_plan(g, 1, sms, lut);
            tp.G = shares_for(f, ws_bytes);
            tp.out = tp.G > 1 ? static_cast<float *>(ws) : out;
            const int grid = tp.cblocks * tp.G;
            rc = launch_tile_any<2>(alu, g.R, width, tp, grid, smem, st);
            if (rc == AMSIM_OK) amsim::count_launch();
            if (rc == AMSIM_OK && tp.G > 1) {
                const int blocks = (int)std::min<long long>((n_out + 255) / 256, 4LL * sms);
                dw_sum_kernel<<<blocks, 256, 0, st>>>(static_cast<const float *>(ws), out, n_out, tp.G);
                rc = amsim::cuda_status(cudaGetLastError());
                if (rc == AMSIM_OK) amsim::count_launch();
                path |= AMSIM_PATH_STREAMK;
            }
        }
    } else {
        DwDirectParams dp{};
        dp.g = g;
        dp.a = t0;
        dp.b = t1;
        dp.table = tab_direct;
        dp.M = lut->M;
        dp.wlog = wlog;
        dp.G = 1;
        dp.table_bytes = (width <= 16 && (int)lut->narrow_bytes <= kDwDirectMaxLut) ? (int)lut->narrow_bytes : 0;
        dp.grid_taps = g.dh == 1 && g.dw == 1;
        dp.fmt = exp_format(lut->exp_bits);
        if (which == 1 && (size_t)g.C + 16 + (size_t)dp.table_bytes > (size_t)amsim::kMaxSmemPerCta)
            return AMSIM_EUNSUPPORTED;     // the channel flags do not fit shared memory
        if (which == 0) {
            dp.groups = (g.K + 31) / 32;
            dp.items = (long long)g.N * g.P * g.Q * dp.groups;
            dp.out = out;
        } else if (which == 1) {
            dp.groups = (g.C + 31) / 32;
            dp.items = (long long)g.N * g.H * g.W * dp.groups;
            dp.out = out;
        } else {
            const DwFilterPlan f = filter_plan(g, 0, sms, lut);
            dp.G = shares_for(f, ws_bytes);
            dp.groups = (g.K + 31) / 32;
            dp.items = (long long)g.R * g.S * dp.G * dp.groups;
            dp.out = dp.G > 1 ? static_cast<float *>(ws) : out;
        }
        // persistent CTAs: each stages the table once
        const int grid = (int)std::max<long long>(1, std::min<long long>((dp.items + 7) / 8, 8LL * sms));
        rc = which == 0 ? launch_direct<0>(width, dp, grid, st)
           : which == 1 ? launch_direct<1>(width, dp, grid, st)
                        : launch_direct<2>(width, dp, grid, st);
        if (rc == AMSIM_OK) amsim::count_launch();
        if (rc == AMSIM_OK && which == 2 && dp.G > 1) {
            const int blocks = (int)std::min<long long>((n_out + 255) / 256, 4LL * sms);
            dw_sum_kernel<<<blocks, 256, 0, st>>>(static_cast<const float *>(ws), out, n_out, dp.G);
            rc = amsim::cuda_status(cudaGetLastError());
            if (rc == AMSIM_OK) amsim::count_launch();
            path |= AMSIM_PATH_STREAMK;
        }
    }
    if (rc == AMSIM_OK) amsim::set_last_path(path);
    return rc;
}

}  // namespace

extern "C" {

int amsim_dwconv2d_fwd(const amsim_conv_desc *desc, const float *x, const float *w, float *y, amsim_lut_t lut,
                       void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    return dw_run(desc, 0, x, w, y, lut, ws, ws_bytes, stream);
}

int amsim_dwconv2d_bwd_data(const amsim_conv_desc *desc, const float *dy, const float *w, float *dx,
                            amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    return dw_run(desc, 1, dy, w, dx, lut, ws, ws_bytes, stream);
}

int amsim_dwconv2d_bwd_filter(const amsim_conv_desc *desc, const float *x, const float *dy, float *dw,
                              amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream)
{
    return dw_run(desc, 2, x, dy, dw, lut, ws, ws_bytes, stream);
}

size_t amsim_dwconv2d_workspace_size(const amsim_conv_desc *desc, int which, amsim_lut_t lut)
{
    DwGeo g;
    if (which != 2 || !lut || dw_geometry(desc, &g) != AMSIM_OK) return 0;
    const int dev = lut->device;
    const int kind = dw_tile_ok(g, lut, 2, nullptr, nullptr, nullptr)  ? 1
                   : dw_s2_ok(g, lut, 2, nullptr, nullptr, nullptr) ? 2
                                                                     : 0;
    const DwFilterPlan f = filter_plan(g, kind, sm_count(dev), lut);
    if (f.G_want <= 1) return 0;
    return (size_t)f.G_want * (size_t)f.outs * 4;
}

}  // extern "C"
