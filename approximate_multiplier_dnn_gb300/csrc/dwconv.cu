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
// GEMM, and there is no contraction to tile for the tensor cores.  Two kernels:
//  * dw_tile_kernel (3x3 filter, unit stride and dilation, D = 1, channels a
//    multiple of 4): a CTA stages a halo tile of 16 channels of the activation
//    (10 x 66 positions for an 8 x 64 output tile) in shared memory, each
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
//    outside the tensor) while the CTA computes the current tile.
//  * dw_direct_kernel (every other geometry): one lane per output element,
//    operands loaded and decoded per product, the LUT read through the
//    read-only cache; the weight is still warp-uniform in the first two passes.
// The weight gradient's reduction over N*P*Q is split into G shares written to
// scratch and added in share order by dw_sum_kernel, so results are
// deterministic for a given scratch size.
#include <algorithm>

#include "gemm_tma.cuh"

namespace {

using amsim::kern::expand;
using amsim::kern::ffma2;
using amsim::kern::fmul2_ftz;
using amsim::kern::lut_ld;

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

// ------------------------------------------------------------------ operand packing
// One word per operand element: bits 31..23 sign and biased exponent (the
// element's signed power-of-two scale once the low bits are cleared; zero and
// denormal inputs give a signed zero, infinity an infinite scale), bit 22 set
// for NaN (so the cleared word is a NaN scale), bits 21..0 the byte offset of
// the truncated mantissa's LUT row (high operand) or column (low operand).
// `big` collects elements with biased exponent >= 191 (|x| >= 2^64, infinities
// and NaN): only products of such elements can overflow.
__device__ __forceinline__ uint32_t dw_pack(float v, int M, int offshift, int &big)
{
    const uint32_t x = __float_as_uint(v);
    const uint32_t e = (x >> 23) & 0xFFu;
    const uint32_t f = x & 0x7FFFFFu;
    uint32_t w = (x & 0xFF800000u) | ((f >> (23 - M)) << offshift);
    if (e == 255u && f) w |= 0x00400000u;
    big |= (e >= 191u);
    return w;
}

__device__ __forceinline__ uint32_t dw_scale_bits(uint32_t packed) { return packed & 0xFFC00000u; }

// The same packing without the NaN bit, for tiles whose elements all have
// |x| < 2^64: `big` is raised by any other element (|x| >= 2^64, infinity,
// NaN), and such a tile is packed again by dw_pack from global memory.
// k = 23 - M - offshift, offmask = (2^M - 1) << offshift.
__device__ __forceinline__ uint32_t dw_pack_fast(float v, int k, uint32_t offmask, bool &big)
{
    const uint32_t x = __float_as_uint(v);
    big |= !(fabsf(v) < 0x1p64f);
    return (x & 0xFF800000u) | ((x >> k) & offmask);
}

// v = 2^carry * 1.mantissa as fp32 bits from a narrowed entry: entry * 2^(24-W)
// + bits(1.0f).  `mul` is 2^(24-W) passed at run time, so the multiply-add
// stays an integer multiply-add on the FMA pipe, leaving the ALU pipe to the
// index adds.
__device__ __forceinline__ float dw_expand(uint32_t narrowed, uint32_t mul)
{
    uint32_t r;
    asm("mad.lo.u32 %0, %1, %2, 0x3F800000;" : "=r"(r) : "r"(narrowed), "r"(mul));
    return __uint_as_float(r);
}

// Scalar FTZ multiply: the page's "zero when the biased exponent sum is not above zero".
__device__ __forceinline__ float fmul_ftz(float a, float b)
{
    float d;
    asm("mul.rn.ftz.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// ------------------------------------------------------------------ tiled kernel
constexpr int kDwThreads = 256;       // 8 warps
constexpr int kDwTP = 8;              // output rows per tile
constexpr int kDwTQ = 64;             // output columns per tile (2 per lane)
constexpr int kDwTH = kDwTP + 2;      // halo rows (3x3 filter)
constexpr int kDwTW = kDwTQ + 2;      // halo columns
constexpr int kDwCP = 666;            // packed halo words per channel: >= 660, = 2 mod 8 (conflict-free packing)
constexpr int kDwOP = 514;            // packed output-gradient / output-tile words per channel: >= 512, = 2 mod 8
static_assert(kDwTH * kDwTW <= kDwCP && kDwTP * kDwTQ <= kDwOP, "tile pitches");
static_assert(kDwCP % 2 == 0 && kDwOP % 2 == 0 && kDwTW % 2 == 0, "8-byte aligned lane pairs");

__host__ __device__ constexpr int dw_lut_region(int table_bytes) { return (table_bytes + 127) & ~127; }

// Channels per tile: 16 (two per warp) in the forward and data-gradient
// passes; 8 (one per warp) in the weight gradient, whose two raw boxes and two
// packed tiles would otherwise leave room for one CTA per SM.
template <int MODE>
struct DwCfg {
    static constexpr int CB = MODE == 2 ? 8 : 16;
    static constexpr int CPW = CB / 8;                        // channels per warp
    static constexpr int RawA = kDwTH * kDwTW * CB * 4;       // raw halo box as the tensor copy lands: [row][col][c]
    static constexpr int RawB = kDwTP * kDwTQ * CB * 4;       // raw output-gradient box (weight gradient)
    static constexpr int Halo = (CB * kDwCP * 4 + 127) & ~127;   // packed halo [c][pos]
    static constexpr int Out = (CB * kDwOP * 4 + 127) & ~127;    // packed dy (weight gradient) / output tile
    static constexpr int WB = (2 * CB * 9 * 4 + 127) & ~127;     // packed filter taps
    static constexpr int Tail = MODE == 2 ? RawB + Out : WB;
    static_assert(Out <= Halo, "the output tile reuses the halo region");
    static_assert(RawA % 128 == 0 && RawB % 128 == 0 && Halo % 128 == 0 && Out % 128 == 0 && WB % 128 == 0,
                  "128-byte aligned regions");
};

// Shared memory of the tiled kernel: LUT, raw box(es), packed tiles, weights
// (forward / data gradient), one mbarrier.
__host__ __device__ constexpr int dw_tile_smem(int table_bytes, int mode)
{
    return dw_lut_region(table_bytes) +
           (mode == 2 ? DwCfg<2>::RawA + DwCfg<2>::Halo + DwCfg<2>::Tail
                      : DwCfg<0>::RawA + DwCfg<0>::Halo + DwCfg<0>::Tail) + 128;
}

__host__ __device__ constexpr int dw_channel_block(int mode) { return mode == 2 ? DwCfg<2>::CB : DwCfg<0>::CB; }

struct DwTileParams {
    CUtensorMap amap;      // activation: dims (C, IW, IH, N), box (16, kDwTW, kDwTH, 1)
    CUtensorMap bmap;      // weight gradient's dy: dims (C, OW, OH, N), box (16, kDwTQ, kDwTP, 1)
    const float *a;        // activation (for re-packing a tile with special values)
    const float *b;        // w [3][3][C] (modes 0, 1), dy (mode 2)
    float *out;            // y / dx (NHWC), or the weight gradient's shares [G][9][C]
    uint32_t expand_mul;   // 2^(24 - entry width)
    int IH, IW;            // activation height and width
    const void *table;     // narrowed LUT: [w][activation] (modes 0, 1), [x][dy] (mode 2)
    int table_bytes, M, wlog;
    int N, C;
    int OH, OW;            // output (modes 0, 1) or dy (mode 2) height and width
    int oy, ox;            // activation row/column of output (0, 0) at tap (0, 0)
    int tiles_p, tiles_q, cblocks;
    int tiles;             // N * tiles_p * tiles_q spatial tiles
    int G;                 // mode 2: shares of the spatial tiles
};

struct DwTile {
    int n, p0, q0, c0;
};

// Pack a raw box [pos][CB channels] (as the tensor copy wrote it) into
// [channel][pos] words with channel pitch `pitch`: 16-byte reads of 4
// channels, one word written per channel (fast packing, see dw_pack_fast).
template <int CB>
__device__ __forceinline__ void dw_pack_box(const float *raw, uint32_t *dst, int npos, int pitch, int k,
                                            uint32_t offmask, int tid, bool &big)
{
    constexpr int G4 = CB / 4;
#pragma unroll 4
    for (int e = tid; e < npos * G4; e += kDwThreads) {
        const int c4 = e % G4, pos = e / G4;
        const float4 v = *reinterpret_cast<const float4 *>(raw + pos * CB + 4 * c4);
        uint32_t *d = dst + 4 * c4 * pitch + pos;
        d[0] = dw_pack_fast(v.x, k, offmask, big);
        d[pitch] = dw_pack_fast(v.y, k, offmask, big);
        d[2 * pitch] = dw_pack_fast(v.z, k, offmask, big);
        d[3 * pitch] = dw_pack_fast(v.w, k, offmask, big);
    }
}

// Exact packing (NaN kept as NaN) of a box read straight from global memory:
// rows [r0, r0 + bh) x columns [w0, w0 + bw) of image n, channels c0 .. c0+CB-1
// of an NHWC tensor with dims (H, W, C); positions outside it are zeros.
template <int CB>
__device__ __forceinline__ void dw_repack(const float *src, uint32_t *dst, int pitch, int n, int H, int W, int C,
                                          int r0, int w0, int c0, int bh, int bw, int M, int offshift, int tid)
{
    const float *img = src + (long long)n * H * W * C;
    int unused = 0;
    constexpr int G4 = CB / 4;
    for (int e = tid; e < bh * bw * G4; e += kDwThreads) {
        const int c4 = e % G4, pos = e / G4;
        const int row = pos / bw, col = pos - row * bw;
        const int h = r0 + row, w = w0 + col, c = c0 + 4 * c4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if ((unsigned)h < (unsigned)H && (unsigned)w < (unsigned)W && c < C)
            v = __ldg(reinterpret_cast<const float4 *>(img + ((long long)h * W + w) * C + c));
        uint32_t *d = dst + 4 * c4 * pitch + pos;
        d[0] = dw_pack(v.x, M, offshift, unused);
        d[pitch] = dw_pack(v.y, M, offshift, unused);
        d[2 * pitch] = dw_pack(v.z, M, offshift, unused);
        d[3 * pitch] = dw_pack(v.w, M, offshift, unused);
    }
}

// One thread announces the tile's bytes and issues its box copies; channels
// past C and positions outside the tensor arrive as zeros.
template <int MODE>
__device__ __forceinline__ void dw_issue(const DwTileParams &p, const DwTile &t, float *rawA, float *rawB,
                                         uint64_t *bar)
{
    using amsim::kern::mbar_expect_tx;
    using amsim::kern::tma_load_4d;
    mbar_expect_tx(bar, MODE == 2 ? DwCfg<2>::RawA + DwCfg<2>::RawB : DwCfg<MODE>::RawA);
    tma_load_4d(rawA, &p.amap, t.c0, t.q0 + p.ox, t.p0 + p.oy, t.n, bar);
    if constexpr (MODE == 2) tma_load_4d(rawB, &p.bmap, t.c0, t.q0, t.p0, t.n, bar);
}

// Forward / data-gradient compute of one channel for one lane: acc[i] holds
// output row i at tile columns 2*lane (.x) and 2*lane + 1 (.y).
template <int W, bool SLOW>
__device__ __forceinline__ void dw_taps_channel(float2 (&acc)[kDwTP], const uint32_t *xr, const uint8_t *lut,
                                                const uint32_t (&woff)[9], const float (&wsc)[9], uint32_t mul)
{
#pragma unroll
    for (int i = 0; i < kDwTP; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int hh = 0; hh < kDwTH; ++hh) {
        const uint2 a01 = *reinterpret_cast<const uint2 *>(xr + hh * kDwTW);
        const uint2 a23 = *reinterpret_cast<const uint2 *>(xr + hh * kDwTW + 2);
        const uint32_t px[4] = {a01.x, a01.y, a23.x, a23.y};
        uint32_t sb[4];
        float sx[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sb[k] = dw_scale_bits(px[k]);
            sx[k] = __uint_as_float(sb[k]);
        }
#pragma unroll
        for (int r = 0; r < 3; ++r) {
            const int i = hh - r;
            if (i < 0 || i >= kDwTP) continue;
#pragma unroll
            for (int s = 0; s < 3; ++s) {
                const int t = r * 3 + s;
                const uint32_t i0 = px[s] - sb[s] + woff[t];
                const uint32_t i1 = px[s + 1] - sb[s + 1] + woff[t];
                const float2 v = make_float2(dw_expand(lut_ld<W, false>(lut, i0), mul),
                                             dw_expand(lut_ld<W, false>(lut, i1), mul));
                const float2 sc = fmul2_ftz(make_float2(wsc[t], wsc[t]), make_float2(sx[s], sx[s + 1]));
                if constexpr (SLOW) {
                    // product rounded to fp32 first (infinity on overflow), then added
                    acc[i].x = __fadd_rn(acc[i].x, __fmul_rn(v.x, sc.x));
                    acc[i].y = __fadd_rn(acc[i].y, __fmul_rn(v.y, sc.y));
                } else {
                    acc[i] = ffma2(v, sc, acc[i]);   // exact product, one rounding in the add
                }
            }
        }
    }
}

// Weight-gradient compute of one channel for one lane over one tile:
// acc[t] += products of tap t at output rows 0..7, tile columns 2*lane (.x)
// and 2*lane + 1 (.y).  In the slow form, positions outside the output
// gradient (past P or Q) are skipped, so an infinite activation there cannot
// meet a zero-filled gradient.
template <int W, bool SLOW>
__device__ __forceinline__ void dw_filter_channel(float2 (&acc)[9], const uint32_t *xr, const uint32_t *dr,
                                                  const uint8_t *lut, int rows_ok, bool ok0, bool ok1, uint32_t mul)
{
#pragma unroll
    for (int i = 0; i < kDwTP; ++i) {
        const uint2 d01 = *reinterpret_cast<const uint2 *>(dr + i * kDwTQ);
        const uint32_t db0 = dw_scale_bits(d01.x), db1 = dw_scale_bits(d01.y);
        const uint32_t od0 = d01.x - db0, od1 = d01.y - db1;
        const float2 sd = make_float2(__uint_as_float(db0), __uint_as_float(db1));
        const bool row_ok = i < rows_ok;
#pragma unroll
        for (int r = 0; r < 3; ++r) {
            const uint2 a01 = *reinterpret_cast<const uint2 *>(xr + (i + r) * kDwTW);
            const uint2 a23 = *reinterpret_cast<const uint2 *>(xr + (i + r) * kDwTW + 2);
            const uint32_t px[4] = {a01.x, a01.y, a23.x, a23.y};
            uint32_t sb[4];
            float sx[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                sb[k] = dw_scale_bits(px[k]);
                sx[k] = __uint_as_float(sb[k]);
            }
#pragma unroll
            for (int s = 0; s < 3; ++s) {
                const int t = r * 3 + s;
                const uint32_t i0 = px[s] - sb[s] + od0;
                const uint32_t i1 = px[s + 1] - sb[s + 1] + od1;
                const float2 v = make_float2(dw_expand(lut_ld<W, false>(lut, i0), mul),
                                             dw_expand(lut_ld<W, false>(lut, i1), mul));
                const float2 sc = fmul2_ftz(make_float2(sx[s], sx[s + 1]), sd);
                if constexpr (SLOW) {
                    if (row_ok && ok0) acc[t].x = __fadd_rn(acc[t].x, __fmul_rn(v.x, sc.x));
                    if (row_ok && ok1) acc[t].y = __fadd_rn(acc[t].y, __fmul_rn(v.y, sc.y));
                } else {
                    acc[t] = ffma2(v, sc, acc[t]);
                }
            }
        }
    }
}

// MODE 0: forward; 1: data gradient (the activation is dy, the filter flipped);
// 2: weight gradient (CTA = (channel block, share of the spatial tiles)).
// Thread 0 copies the next tile's raw boxes while the CTA computes the
// current one; every wait on the copy is bounded (a timeout is recorded and
// the CTA leaves its remaining tiles).
template <int W, int MODE>
__global__ void __launch_bounds__(kDwThreads, 2) dw_tile_kernel(const __grid_constant__ DwTileParams p)
{
    using amsim::kern::mbar_init;
    using amsim::kern::mbar_wait;
    extern __shared__ __align__(128) uint8_t smem[];
    using Cfg = DwCfg<MODE>;
    constexpr int CB = Cfg::CB, CPW = Cfg::CPW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t *lut = smem;
    float *rawA = reinterpret_cast<float *>(smem + dw_lut_region(p.table_bytes));
    uint32_t *xt = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(rawA) + Cfg::RawA);
    uint8_t *after = reinterpret_cast<uint8_t *>(xt) + Cfg::Halo;
    float *rawB = reinterpret_cast<float *>(after);                       // mode 2
    uint32_t *dyt = reinterpret_cast<uint32_t *>(after + Cfg::RawB);      // mode 2
    uint32_t *wt_off = reinterpret_cast<uint32_t *>(after);               // modes 0, 1
    float *wt_scl = reinterpret_cast<float *>(after + CB * 9 * 4);
    uint64_t *bar = reinterpret_cast<uint64_t *>(after + Cfg::Tail);

    // this CTA's tiles: [t_begin, t_end) step t_step of the launch's tile list
    int t_begin, t_end, t_step, cb_fixed = 0, g = 0;
    if constexpr (MODE == 2) {
        cb_fixed = blockIdx.x % p.cblocks;
        g = blockIdx.x / p.cblocks;
        t_begin = (int)((long long)p.tiles * g / p.G);
        t_end = (int)((long long)p.tiles * (g + 1) / p.G);
        t_step = 1;
    } else {
        t_begin = blockIdx.x;
        t_end = p.tiles * p.cblocks;
        t_step = gridDim.x;
    }
    auto tile_at = [&](int t) {
        DwTile d;
        int cb = cb_fixed, rest = t;
        if constexpr (MODE != 2) {
            cb = t % p.cblocks;
            rest = t / p.cblocks;
        }
        const int tq = rest % p.tiles_q;
        rest /= p.tiles_q;
        d.p0 = (rest % p.tiles_p) * kDwTP;
        d.n = rest / p.tiles_p;
        d.q0 = tq * kDwTQ;
        d.c0 = cb * CB;
        return d;
    };

    if (tid == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (t_begin < t_end) dw_issue<MODE>(p, tile_at(t_begin), rawA, rawB, bar);
    }
    {   // LUT -> shared memory (the device table is padded to 256 bytes)
        const uint4 *src = static_cast<const uint4 *>(p.table);
        uint4 *dst = reinterpret_cast<uint4 *>(lut);
        const int nvec = (p.table_bytes + 15) >> 4;
        for (int i = tid; i < nvec; i += kDwThreads) dst[i] = __ldg(src + i);
    }
    const int hi_shift = p.M + p.wlog, lo_shift = p.wlog;

    float2 facc[CPW][9];                    // mode 2: per-tap sums of this CTA's share
    if constexpr (MODE == 2) {
#pragma unroll
        for (int ci = 0; ci < CPW; ++ci)
#pragma unroll
            for (int t = 0; t < 9; ++t) facc[ci][t] = make_float2(0.0f, 0.0f);
    }
    uint32_t phase = 0;
    bool aborted = false;
    for (int t = t_begin; t < t_end; t += t_step) {
        const DwTile tl = tile_at(t);
        __syncthreads();                    // the previous tile's shared-memory reads are done
        mbar_wait(bar, phase, aborted);
        phase ^= 1;
        if (__syncthreads_or(aborted)) break;
        bool big = false;
        const int a_shift = MODE == 2 ? hi_shift : lo_shift;
        dw_pack_box<CB>(rawA, xt, kDwTH * kDwTW, kDwCP, 23 - p.M - a_shift, ((1u << p.M) - 1u) << a_shift, tid,
                        big);
        if constexpr (MODE == 2) {
            dw_pack_box<CB>(rawB, dyt, kDwTP * kDwTQ, kDwOP, 23 - p.M - lo_shift, ((1u << p.M) - 1u) << lo_shift,
                            tid, big);
        } else if (tid < CB * 9) {
            const int c = tid / 9, tap = tid % 9;
            const int src_t = MODE == 0 ? tap : 8 - tap;   // the data gradient reads the filter rotated by 180 degrees
            const float v = tl.c0 + c < p.C ? __ldg(p.b + (long long)src_t * p.C + tl.c0 + c) : 0.0f;
            int wbig = 0;
            const uint32_t pk = dw_pack(v, p.M, hi_shift, wbig);
            big |= wbig != 0;
            wt_off[tid] = pk - dw_scale_bits(pk);
            wt_scl[tid] = __uint_as_float(dw_scale_bits(pk));
        }
        const bool slow = __syncthreads_or(big);   // the raw boxes are consumed
        if (tid == 0 && t + t_step < t_end) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            dw_issue<MODE>(p, tile_at(t + t_step), rawA, rawB, bar);
        }
        if (slow) {
            // a tile with |x| >= 2^64, infinities or NaN: pack it again exactly
            // (NaN kept as NaN) from global memory, then take the slow products
            dw_repack<CB>(p.a, xt, kDwCP, tl.n, p.IH, p.IW, p.C, tl.p0 + p.oy, tl.q0 + p.ox, tl.c0, kDwTH, kDwTW, p.M,
                      a_shift, tid);
            if constexpr (MODE == 2)
                dw_repack<CB>(p.b, dyt, kDwOP, tl.n, p.OH, p.OW, p.C, tl.p0, tl.q0, tl.c0, kDwTP, kDwTQ, p.M, lo_shift,
                          tid);
            __syncthreads();
        }

        if constexpr (MODE == 2) {
            const int rows_ok = p.OH - tl.p0;
            const bool ok0 = tl.q0 + 2 * lane < p.OW, ok1 = tl.q0 + 2 * lane + 1 < p.OW;
#pragma unroll
            for (int ci = 0; ci < CPW; ++ci) {
                const int c = warp + 8 * ci;
                const uint32_t *xr = xt + c * kDwCP + 2 * lane;
                const uint32_t *dr = dyt + c * kDwOP + 2 * lane;
                if (slow) dw_filter_channel<W, true>(facc[ci], xr, dr, lut, rows_ok, ok0, ok1, p.expand_mul);
                else dw_filter_channel<W, false>(facc[ci], xr, dr, lut, rows_ok, ok0, ok1, p.expand_mul);
            }
        } else {
            float2 acc[CPW][kDwTP];
#pragma unroll
            for (int ci = 0; ci < CPW; ++ci) {
                const int c = warp + 8 * ci;
                uint32_t woff[9];
                float wsc[9];
#pragma unroll
                for (int k = 0; k < 9; ++k) {
                    woff[k] = wt_off[c * 9 + k];
                    wsc[k] = wt_scl[c * 9 + k];
                }
                const uint32_t *xr = xt + c * kDwCP + 2 * lane;
                if (slow) dw_taps_channel<W, true>(acc[ci], xr, lut, woff, wsc, p.expand_mul);
                else dw_taps_channel<W, false>(acc[ci], xr, lut, woff, wsc, p.expand_mul);
            }
            __syncthreads();                // every warp is done with the packed halo
            float *ot = reinterpret_cast<float *>(xt);
#pragma unroll
            for (int ci = 0; ci < CPW; ++ci) {
                float *o = ot + (warp + 8 * ci) * kDwOP + 2 * lane;
#pragma unroll
                for (int i = 0; i < kDwTP; ++i) *reinterpret_cast<float2 *>(o + i * kDwTQ) = acc[ci][i];
            }
            __syncthreads();
            float *dst = p.out + (long long)tl.n * p.OH * p.OW * p.C;
#pragma unroll 4
            for (int e = tid; e < kDwTP * kDwTQ * 4; e += kDwThreads) {
                const int c4 = e & 3, pos = e >> 2;
                const int i = pos / kDwTQ, j = pos % kDwTQ;
                const int pp = tl.p0 + i, qq = tl.q0 + j, c = tl.c0 + 4 * c4;
                if (pp < p.OH && qq < p.OW && c < p.C) {
                    const float *src = ot + 4 * c4 * kDwOP + pos;
                    const float4 v = make_float4(src[0], src[kDwOP], src[2 * kDwOP], src[3 * kDwOP]);
                    __stcs(reinterpret_cast<float4 *>(dst + ((long long)pp * p.OW + qq) * p.C + c), v);
                }
            }
        }
    }
    if constexpr (MODE == 2) {
        // lanes -> lane 0 in a fixed butterfly order; warp w owns channel w (and w + 8)
        const int c0 = cb_fixed * CB;
#pragma unroll
        for (int ci = 0; ci < CPW; ++ci) {
            const int c = c0 + warp + 8 * ci;
#pragma unroll
            for (int k = 0; k < 9; ++k) {
                float v = facc[ci][k].x + facc[ci][k].y;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                if (lane == 0 && c < p.C) p.out[((long long)g * 9 + k) * p.C + c] = v;
            }
        }
    }
}

// ------------------------------------------------------------------ direct kernel
struct DwDirectParams {
    DwGeo g;
    const float *a, *b;
    float *out;
    const void *table;     // narrowed LUT, [first operand][second operand] of the pass
    int M, wlog;
    long long items;       // mode 0/1: output channels x 32-position chunks; mode 2: R*S*K outputs x G shares
    long long chunks;      // mode 0/1: 32-position chunks per channel
    int G;                 // mode 2: shares of the N*P*Q reduction
};

// Signed power-of-two scale of an operand (zero and denormal inputs a signed
// zero, infinity infinite, NaN a NaN).
__device__ __forceinline__ float dw_scale(uint32_t x)
{
    const bool nan = ((x >> 23) & 0xFFu) == 255u && (x & 0x7FFFFFu);
    return __uint_as_float(nan ? 0x7FC00000u : (x & 0xFF800000u));
}

// AMSim product of two fp32 values (first operand = high index bits) from a
// narrowed table, rounded to fp32 before it is added (infinity on overflow).
template <int W>
__device__ __forceinline__ float dw_product(float first, float second, const void *table, int M, int wlog)
{
    const uint32_t xa = __float_as_uint(first), xb = __float_as_uint(second);
    const uint32_t idx = ((((xa & 0x7FFFFFu) >> (23 - M)) << M) | ((xb & 0x7FFFFFu) >> (23 - M))) << wlog;
    const float v = expand<W>(lut_ld<W, true>(static_cast<const uint8_t *>(table), idx));
    return __fmul_rn(v, fmul_ftz(dw_scale(xa), dw_scale(xb)));
}

template <int W, int MODE>
__global__ void __launch_bounds__(256) dw_direct_kernel(const __grid_constant__ DwDirectParams p)
{
    const DwGeo &g = p.g;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < p.items; it += warps) {
        if constexpr (MODE == 0) {
            // warp: output channel k (uniform filter tap), lanes: 32 consecutive output pixels
            const int k = (int)(it / p.chunks);
            const long long pix = (it % p.chunks) * 32 + lane;
            if (pix >= (long long)g.N * g.P * g.Q) continue;
            const int q = (int)(pix % g.Q);
            const int pp = (int)((pix / g.Q) % g.P);
            const int n = (int)(pix / ((long long)g.P * g.Q));
            const int c = k / g.D, d = k % g.D;
            float acc = 0.0f;
            for (int r = 0; r < g.R; ++r)
                for (int s = 0; s < g.S; ++s) {
                    const int h = pp * g.sh - g.ph + r * g.dh, w = q * g.sw - g.pw + s * g.dw;
                    float xv = 0.0f;
                    if ((unsigned)h < (unsigned)g.H && (unsigned)w < (unsigned)g.W)
                        xv = __ldg(p.a + (((long long)n * g.H + h) * g.W + w) * g.C + c);
                    const float wv = __ldg(p.b + ((long long)(r * g.S + s) * g.C + c) * g.D + d);
                    acc = __fadd_rn(acc, dw_product<W>(xv, wv, p.table, p.M, p.wlog));
                }
            p.out[pix * g.K + k] = acc;
        } else if constexpr (MODE == 1) {
            // warp: input channel c, lanes: 32 consecutive input pixels
            const int c = (int)(it / p.chunks);
            const long long pix = (it % p.chunks) * 32 + lane;
            if (pix >= (long long)g.N * g.H * g.W) continue;
            const int w = (int)(pix % g.W);
            const int h = (int)((pix / g.W) % g.H);
            const int n = (int)(pix / ((long long)g.H * g.W));
            float acc = 0.0f;
            for (int r = 0; r < g.R; ++r)
                for (int s = 0; s < g.S; ++s) {
                    const int hp = h + g.ph - r * g.dh, wq = w + g.pw - s * g.dw;
                    const bool in = hp >= 0 && wq >= 0 && hp % g.sh == 0 && wq % g.sw == 0 && hp / g.sh < g.P &&
                                    wq / g.sw < g.Q;
                    const long long base = in ? (((long long)n * g.P + hp / g.sh) * g.Q + wq / g.sw) * g.K : 0;
                    for (int d = 0; d < g.D; ++d) {
                        const float dyv = in ? __ldg(p.a + base + (long long)c * g.D + d) : 0.0f;
                        const float wv = __ldg(p.b + ((long long)(r * g.S + s) * g.C + c) * g.D + d);
                        acc = __fadd_rn(acc, dw_product<W>(dyv, wv, p.table, p.M, p.wlog));
                    }
                }
            p.out[pix * g.C + c] = acc;
        } else {
            // warp: one filter element (r,s,c,d) over one share of the N*P*Q pixels
            const long long RSK = (long long)g.R * g.S * g.K;
            const int share = (int)(it / RSK);
            const long long o = it % RSK;
            const int k = (int)(o % g.K);
            const int s = (int)((o / g.K) % g.S);
            const int r = (int)(o / ((long long)g.K * g.S));
            const int c = k / g.D;
            const long long npq = (long long)g.N * g.P * g.Q;
            const long long b0 = npq * share / p.G, b1 = npq * (share + 1) / p.G;
            float acc = 0.0f;
            for (long long pix = b0 + lane; pix < b1; pix += 32) {
                const int q = (int)(pix % g.Q);
                const int pp = (int)((pix / g.Q) % g.P);
                const int n = (int)(pix / ((long long)g.P * g.Q));
                const int h = pp * g.sh - g.ph + r * g.dh, w = q * g.sw - g.pw + s * g.dw;
                float xv = 0.0f;
                if ((unsigned)h < (unsigned)g.H && (unsigned)w < (unsigned)g.W)
                    xv = __ldg(p.a + (((long long)n * g.H + h) * g.W + w) * g.C + c);
                const float dyv = __ldg(p.b + pix * g.K + k);
                acc = __fadd_rn(acc, dw_product<W>(xv, dyv, p.table, p.M, p.wlog));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
            if (lane == 0) p.out[(long long)share * RSK + o] = acc;
        }
    }
}

// out[i] = sum over shares g = 0 .. G-1 of part[g*n + i], in share order.
__global__ void __launch_bounds__(256) dw_sum_kernel(const float *__restrict__ part, float *__restrict__ out,
                                                     long long n, int G)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        float v = part[i];
        for (int g = 1; g < G; ++g) v += part[(long long)g * n + i];
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

// The tiled kernel covers 3x3 filters at unit stride and dilation with one
// filter per channel, channels a multiple of 4, 16-byte aligned tensors and a
// narrowed 8- or 16-bit LUT of at most 64 KB.
bool dw_tile_ok(const DwGeo &g, const amsim_lut_t lut, int which, const float *t0, const float *t1,
                const float *out)
{
    if (g.D != 1 || g.R != 3 || g.S != 3 || g.sh != 1 || g.sw != 1 || g.dh != 1 || g.dw != 1) return false;
    if (g.C % 4 || lut->width_bits == 32 || (int)lut->narrow_bytes > kDwMaxTileLut) return false;
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

template <int W, int MODE>
int launch_tile_w(const DwTileParams &tp, int grid, size_t smem, cudaStream_t st)
{
    auto kfn = dw_tile_kernel<W, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return amsim::cuda_status(e);
    kfn<<<grid, kDwThreads, smem, st>>>(tp);
    return amsim::cuda_status(cudaGetLastError());
}

template <int MODE>
int launch_tile(int width, const DwTileParams &tp, int grid, size_t smem, cudaStream_t st)
{
    return width == 8 ? launch_tile_w<8, MODE>(tp, grid, smem, st) : launch_tile_w<16, MODE>(tp, grid, smem, st);
}

template <int MODE>
int launch_direct(int width, const DwDirectParams &dp, int grid, cudaStream_t st)
{
    if (width == 8) dw_direct_kernel<8, MODE><<<grid, 256, 0, st>>>(dp);
    else if (width == 16) dw_direct_kernel<16, MODE><<<grid, 256, 0, st>>>(dp);
    else dw_direct_kernel<32, MODE><<<grid, 256, 0, st>>>(dp);
    return amsim::cuda_status(cudaGetLastError());
}

int wlog_of(int width_bits) { return width_bits == 8 ? 0 : width_bits == 16 ? 1 : 2; }

// Shares of the weight gradient's reduction: the count that fills the GPU,
// and the count that fits `ws_bytes` of scratch (at least 1: no scratch).
struct DwFilterPlan {
    bool tiled;
    int tiles_p, tiles_q, cblocks, tiles;
    int G_want;
    long long outs;        // R*S*K
};

// Resident CTAs of the tiled kernel per SM, from its shared memory (each
// CTA also holds 1 KB of the SM's 228 KB for the system).
int dw_tile_ctas_per_sm(const amsim_lut_t lut, int which)
{
    const int per = dw_tile_smem((int)lut->narrow_bytes, which) + 1024;
    return std::max(1, std::min(2, (228 * 1024) / per));
}

DwFilterPlan filter_plan(const DwGeo &g, bool tiled, int sms, const amsim_lut_t lut)
{
    DwFilterPlan f{};
    f.tiled = tiled;
    f.outs = (long long)g.R * g.S * g.K;
    if (tiled) {
        f.tiles_p = (g.P + kDwTP - 1) / kDwTP;
        f.tiles_q = (g.Q + kDwTQ - 1) / kDwTQ;
        f.cblocks = (g.C + dw_channel_block(2) - 1) / dw_channel_block(2);
        f.tiles = g.N * f.tiles_p * f.tiles_q;
        const int slots = dw_tile_ctas_per_sm(lut, 2) * sms;
        const int want = (slots + f.cblocks - 1) / f.cblocks;
        f.G_want = std::max(1, std::min(want, f.tiles));
    } else {
        const long long npq = (long long)g.N * g.P * g.Q;
        const long long want = (64LL * sms + f.outs - 1) / f.outs;            // about 64 warps per SM
        const long long cap = std::max(1LL, npq / 256);                       // at least 256 pixels a share
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
        bool mapped;
        if (which == 0) {
            tp.IH = g.H; tp.IW = g.W;
            tp.b = t1; tp.out = out;
            tp.OH = g.P; tp.OW = g.Q;
            tp.oy = -g.ph; tp.ox = -g.pw;
            mapped = dw_map(&tp.amap, t0, g.N, g.H, g.W, g.C, dw_channel_block(0), kDwTW, kDwTH);
        } else if (which == 1) {
            // dx[h][w] = sum_{r',s'} dy[h + ph - 2 + r'][w + pw - 2 + s'] * w[2 - r'][2 - s']
            tp.IH = g.P; tp.IW = g.Q;
            tp.b = t1; tp.out = out;
            tp.OH = g.H; tp.OW = g.W;
            tp.oy = g.ph - 2; tp.ox = g.pw - 2;
            mapped = dw_map(&tp.amap, t0, g.N, g.P, g.Q, g.C, dw_channel_block(1), kDwTW, kDwTH);
        } else {
            tp.IH = g.H; tp.IW = g.W;
            tp.b = t1;
            tp.OH = g.P; tp.OW = g.Q;
            tp.oy = -g.ph; tp.ox = -g.pw;
            mapped = dw_map(&tp.amap, t0, g.N, g.H, g.W, g.C, dw_channel_block(2), kDwTW, kDwTH) &&
                     dw_map(&tp.bmap, t1, g.N, g.P, g.Q, g.C, dw_channel_block(2), kDwTQ, kDwTP);
        }
        if (!mapped) {               // the driver refused a tensor map: the direct kernel
            tiled = false;
            path = AMSIM_PATH_DW_DIRECT;
        }
    }
    if (tiled) {
        tp.tiles_p = (tp.OH + kDwTP - 1) / kDwTP;
        tp.tiles_q = (tp.OW + kDwTQ - 1) / kDwTQ;
        tp.cblocks = (g.C + dw_channel_block(which) - 1) / dw_channel_block(which);
        tp.tiles = g.N * tp.tiles_p * tp.tiles_q;
        const size_t smem = (size_t)dw_tile_smem((int)lut->narrow_bytes, which);
        if (which < 2) {
            const long long total = (long long)tp.tiles * tp.cblocks;
            if (total > 0x7FFFFFFFLL) return AMSIM_EUNSUPPORTED;
            const int grid = (int)std::min<long long>(total, (long long)dw_tile_ctas_per_sm(lut, which) * sms);
            tp.G = 1;
            rc = which == 0 ? launch_tile<0>(width, tp, grid, smem, st) : launch_tile<1>(width, tp, grid, smem, st);
            if (rc == AMSIM_OK) amsim::count_launch();
        } else {
            const DwFilterPlan f = filter_plan(g, true, sms, lut);
            tp.G = shares_for(f, ws_bytes);
            tp.out = tp.G > 1 ? static_cast<float *>(ws) : out;
            const int grid = tp.cblocks * tp.G;
            rc = launch_tile<2>(width, tp, grid, smem, st);
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
        if (which == 0) {
            dp.chunks = ((long long)g.N * g.P * g.Q + 31) / 32;
            dp.items = dp.chunks * g.K;
            dp.out = out;
        } else if (which == 1) {
            dp.chunks = ((long long)g.N * g.H * g.W + 31) / 32;
            dp.items = dp.chunks * g.C;
            dp.out = out;
        } else {
            const DwFilterPlan f = filter_plan(g, false, sms, lut);
            dp.G = shares_for(f, ws_bytes);
            dp.items = f.outs * dp.G;
            dp.out = dp.G > 1 ? static_cast<float *>(ws) : out;
        }
        const int grid = (int)std::max<long long>(1, std::min<long long>((dp.items + 7) / 8, 16LL * sms));
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
    const bool tiled = dw_tile_ok(g, lut, 2, nullptr, nullptr, nullptr);
    const DwFilterPlan f = filter_plan(g, tiled, sm_count(dev), lut);
    if (f.G_want <= 1) return 0;
    return (size_t)f.G_want * (size_t)f.outs * 4;
}

}  // extern "C"
