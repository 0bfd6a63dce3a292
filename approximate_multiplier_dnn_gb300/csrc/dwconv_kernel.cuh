// Depthwise Conv2D tiled kernel (internal header): the unit-stride kernel for
// 3x3 and 5x5 filters, shared by dwconv.cu (3x3 table variants),
// dwconv_alu.cu (3x3 closed forms), dwconv_k5.cu (5x5 table variants),
// dwconv_k5_alu.cu (5x5 closed forms) and dwconv_s2.cu (its packing helpers).  See dwconv.cu for the operation and the design.
#pragma once

#include "gemm_tma.cuh"

namespace amsim {
namespace dw {

using amsim::kern::fadd2;
using amsim::kern::ffma2;
using amsim::kern::fmul2_ftz;
using amsim::kern::lut_ld;

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
// Tile shapes: a lane owns 2 adjacent output columns of an 8-row block; a
// warp's 32 lanes are LQ = 32, 16, 8 or 4 lanes across by 32 / LQ row blocks,
// so a tile is (256 / LQ) rows x 2 LQ columns = 512 outputs per channel and
// its halo, for a KS x KS filter (KS = 3 or 5), (rows + KS - 1) x (columns +
// KS - 1), is at most 660 (KS = 3) or 816 (KS = 5) positions.  The host picks
// LQ per launch to waste the fewest computed outputs past the edges.
constexpr int kDwRB = 8;              // output rows per lane
constexpr int kDwTileOut = 512;       // outputs per tile and channel
constexpr int kDwOP = 514;            // packed output-gradient / output-tile words per channel: >= 512, = 2 mod 8
__host__ __device__ constexpr int dw_halo_max(int ks) { return ks == 3 ? 660 : 816; }
// packed halo words per channel: >= the halo, = 2 mod 8 (conflict-free packing)
__host__ __device__ constexpr int dw_cp(int ks) { return ks == 3 ? 666 : 818; }
static_assert(dw_halo_max(3) <= dw_cp(3) && dw_halo_max(5) <= dw_cp(5) && kDwTileOut <= kDwOP, "tile pitches");
static_assert(dw_cp(3) % 8 == 2 && dw_cp(5) % 8 == 2 && kDwOP % 2 == 0, "pitches");

__host__ __device__ constexpr int dw_lut_region(int table_bytes) { return (table_bytes + 127) & ~127; }

// Channels per tile: 16 (two per warp) in the forward and data-gradient
// passes of 3x3 filters; 8 (one per warp) in the weight gradient, whose two
// raw boxes and two packed tiles would otherwise leave room for one CTA per
// SM, and for 5x5 filters, whose halos are larger.
template <int MODE, int KS = 3>
struct DwCfg {
    static constexpr int CB = (MODE == 2 || KS == 5) ? 8 : 16;
    static constexpr int CPW = CB / 8;                        // channels per warp
    static constexpr int KK = KS * KS;                        // filter taps
    static constexpr int CP = dw_cp(KS);
    static constexpr int RawA = (dw_halo_max(KS) * CB * 4 + 127) & ~127;   // raw halo box as it lands: [row][col][c]
    static constexpr int RawB = kDwTileOut * CB * 4;          // raw output-gradient box (weight gradient)
    static constexpr int Halo = (CB * CP * 4 + 127) & ~127;   // packed halo [c][pos]
    static constexpr int Out = (CB * kDwOP * 4 + 127) & ~127;    // packed dy (weight gradient) / output tile
    static constexpr int WB = (3 * CB * KK * 4 + 127) & ~127;    // filter taps: offsets, scales, closed forms
    static constexpr int Tail = MODE == 2 ? RawB + Out : WB;
    static_assert(Out <= Halo, "the output tile reuses the halo region");
    static_assert(RawA % 128 == 0 && RawB % 128 == 0 && Halo % 128 == 0 && Out % 128 == 0 && WB % 128 == 0,
                  "128-byte aligned regions");
};

// Shared memory of the tiled kernel: LUT, raw box(es), packed tiles, weights
// (forward / data gradient), one mbarrier.
__host__ __device__ constexpr int dw_tile_smem(int table_bytes, int mode, int ks = 3)
{
    // table_bytes: the staged LUT (0 for closed forms, which read it only in slow tiles)
    return dw_lut_region(table_bytes) +
           (ks == 5 ? (mode == 2 ? DwCfg<2, 5>::RawA + DwCfg<2, 5>::Halo + DwCfg<2, 5>::Tail
                                 : DwCfg<0, 5>::RawA + DwCfg<0, 5>::Halo + DwCfg<0, 5>::Tail)
                    : (mode == 2 ? DwCfg<2>::RawA + DwCfg<2>::Halo + DwCfg<2>::Tail
                                 : DwCfg<0>::RawA + DwCfg<0>::Halo + DwCfg<0>::Tail)) + 128;
}

__host__ __device__ constexpr int dw_channel_block(int mode, int ks = 3)
{
    return ks == 5 ? 8 : mode == 2 ? DwCfg<2>::CB : DwCfg<0>::CB;
}

struct DwTileParams {
    CUtensorMap amap;      // activation: dims (C, IW, IH, N), box (CB, tw, th, 1)
    CUtensorMap bmap;      // weight gradient's dy: dims (C, OW, OH, N), box (CB, tq, tp, 1)
    const float *a;        // activation (for re-packing a tile with special values)
    const float *b;        // w [3][3][C] (modes 0, 1), dy (mode 2)
    float *out;            // y / dx (NHWC), or the weight gradient's shares [G][R*S][C]
    uint32_t expand_mul;   // 2^(24 - entry width)
    int IH, IW;            // activation height and width
    const void *table;     // narrowed LUT: [w][activation] (modes 0, 1), [x][dy] (mode 2)
    int table_bytes, M, wlog;
    int N, C;
    int OH, OW;            // output (modes 0, 1) or dy (mode 2) height and width
    int oy, ox;            // activation row/column of output (0, 0) at tap (0, 0)
    int tiles_p, tiles_q, cblocks;
    int lq_shift;          // log2 of the lanes across a row block (5, 4, 3, 2)
    int tp, tq, tq_shift;  // tile rows, tile columns (2 LQ) and log2(tq)
    int th, tw;            // halo rows and columns (tp + 2, tq + 2)
    int raw_a_bytes;       // bytes of one raw halo box (th * tw * CB * 4)
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
    mbar_expect_tx(bar, MODE == 2 ? p.raw_a_bytes + DwCfg<2>::RawB : p.raw_a_bytes);
    tma_load_4d(rawA, &p.amap, t.c0, t.q0 + p.ox, t.p0 + p.oy, t.n, bar);
    if constexpr (MODE == 2) tma_load_4d(rawB, &p.bmap, t.c0, t.q0, t.p0, t.n, bar);
}

// Forward / data-gradient compute of one channel for one lane: acc[i] holds
// output row i at tile columns 2*lane (.x) and 2*lane + 1 (.y).
// Load the lane's KS + 1 packed words of one halo row (two output columns
// and the KS - 1 columns past them) as 8-byte pairs.
template <int KS>
__device__ __forceinline__ void dw_row(const uint32_t *p, uint32_t (&px)[KS + 1])
{
#pragma unroll
    for (int k = 0; k < (KS + 1) / 2; ++k) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p + 2 * k);
        px[2 * k] = v.x;
        px[2 * k + 1] = v.y;
    }
}

template <int W, bool SLOW, bool GL = false, int KS = 3>
__device__ __forceinline__ void dw_taps_channel(float2 (&acc)[kDwRB], const uint32_t *xr, int tw, const uint8_t *lut,
                                                const uint32_t (&woff)[KS * KS], const float (&wsc)[KS * KS],
                                                uint32_t mul)
{
#pragma unroll
    for (int i = 0; i < kDwRB; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int hh = 0; hh < kDwRB + KS - 1; ++hh) {
        uint32_t px[KS + 1];
        dw_row<KS>(xr + hh * tw, px);
        uint32_t sb[KS + 1];
        float sx[KS + 1];
#pragma unroll
        for (int k = 0; k < KS + 1; ++k) {
            sb[k] = dw_scale_bits(px[k]);
            sx[k] = __uint_as_float(sb[k]);
        }
#pragma unroll
        for (int r = 0; r < KS; ++r) {
            const int i = hh - r;
            if (i < 0 || i >= kDwRB) continue;
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const int t = r * KS + s;
                const uint32_t i0 = px[s] - sb[s] + woff[t];
                const uint32_t i1 = px[s + 1] - sb[s + 1] + woff[t];
                const float2 v = make_float2(dw_expand(lut_ld<W, GL>(lut, i0), mul),
                                             dw_expand(lut_ld<W, GL>(lut, i1), mul));
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
template <int W, bool SLOW, bool GL = false, int KS = 3>
__device__ __forceinline__ void dw_filter_channel(float2 (&acc)[KS * KS], const uint32_t *xr, int tw,
                                                  const uint32_t *dr, int tq, const uint8_t *lut, int rows_ok,
                                                  bool ok0, bool ok1, uint32_t mul)
{
#pragma unroll
    for (int i = 0; i < kDwRB; ++i) {
        const uint2 d01 = *reinterpret_cast<const uint2 *>(dr + i * tq);
        const uint32_t db0 = dw_scale_bits(d01.x), db1 = dw_scale_bits(d01.y);
        const uint32_t od0 = d01.x - db0, od1 = d01.y - db1;
        const float2 sd = make_float2(__uint_as_float(db0), __uint_as_float(db1));
        const bool row_ok = i < rows_ok;
#pragma unroll
        for (int r = 0; r < KS; ++r) {
            uint32_t px[KS + 1];
            dw_row<KS>(xr + (i + r) * tw, px);
            uint32_t sb[KS + 1];
            float sx[KS + 1];
#pragma unroll
            for (int k = 0; k < KS + 1; ++k) {
                sb[k] = dw_scale_bits(px[k]);
                sx[k] = __uint_as_float(sb[k]);
            }
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const int t = r * KS + s;
                const uint32_t i0 = px[s] - sb[s] + od0;
                const uint32_t i1 = px[s + 1] - sb[s + 1] + od1;
                const float2 v = make_float2(dw_expand(lut_ld<W, GL>(lut, i0), mul),
                                             dw_expand(lut_ld<W, GL>(lut, i1), mul));
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

// ------------------------------------------------------------------ closed forms
// Closed-form packing: the operand truncated to its top M fraction bits
// (keep = their mask), sign and exponent kept, denormals flushed to signed
// zero.  `big` is raised by the values the fast closed forms must not see:
// |x| >= 2^64, infinities and NaN (as for the table), and nonzero magnitudes
// below 2^-63, whose products with each other can fall below the smallest
// normal, where the table path's scale product flushes them to zero.
__device__ __forceinline__ uint32_t dw_pack_alu(float v, uint32_t keep, bool &big)
{
    float f;
    asm("mul.rn.ftz.f32 %0, %1, 0f3F800000;" : "=f"(f) : "f"(v));
    const float a = fabsf(f);
    big |= !(a < 0x1p64f) || (a != 0.0f && a < 0x1p-63f);
    return __float_as_uint(f) & (0xFF800000u | keep);
}

template <int CB>
__device__ __forceinline__ void dw_pack_box_alu(const float *raw, uint32_t *dst, int npos, int pitch, uint32_t keep,
                                                int tid, bool &big)
{
    constexpr int G4 = CB / 4;
#pragma unroll 4
    for (int e = tid; e < npos * G4; e += kDwThreads) {
        const int c4 = e % G4, pos = e / G4;
        const float4 v = *reinterpret_cast<const float4 *>(raw + pos * CB + 4 * c4);
        uint32_t *d = dst + 4 * c4 * pitch + pos;
        d[0] = dw_pack_alu(v.x, keep, big);
        d[pitch] = dw_pack_alu(v.y, keep, big);
        d[2 * pitch] = dw_pack_alu(v.z, keep, big);
        d[3 * pitch] = dw_pack_alu(v.w, keep, big);
    }
}

// Forward / data-gradient products in closed form (ALU 1 Mitchell, 2 exact)
// for one channel and lane; wv: the filter taps' truncated values.
//  Mitchell: the bits of the tap's truncated value plus the activation's
//  truncated fraction field make tap_scale x Mitchell's factor (the fraction
//  sum's carry lands in the exponent exactly when the 2(x + y) branch
//  applies); times the activation's scale (flush to zero as in the table
//  path), then added.  Exact: one fp32 FMA of the two truncated values.
//  Both products are exact and equal the table path's v * s, and the
//  accumulation order is the table path's: results are bit-identical.
template <int ALU, int KS = 3>
__device__ __forceinline__ void dw_taps_alu(float2 (&acc)[kDwRB], const uint32_t *xr, int tw,
                                            const uint32_t (&wv)[KS * KS])
{
#pragma unroll
    for (int i = 0; i < kDwRB; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int hh = 0; hh < kDwRB + KS - 1; ++hh) {
        uint32_t px[KS + 1];
        dw_row<KS>(xr + hh * tw, px);
        uint32_t sb[KS + 1];
#pragma unroll
        for (int k = 0; k < KS + 1; ++k) sb[k] = px[k] & 0xFF800000u;
#pragma unroll
        for (int r = 0; r < KS; ++r) {
            const int i = hh - r;
            if (i < 0 || i >= kDwRB) continue;
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const int t = r * KS + s;
                if constexpr (ALU == 1) {
                    const float2 w = make_float2(__uint_as_float(wv[t] + px[s] - sb[s]),
                                                 __uint_as_float(wv[t] + px[s + 1] - sb[s + 1]));
                    acc[i] = fadd2(acc[i], fmul2_ftz(w, make_float2(__uint_as_float(sb[s]),
                                                                    __uint_as_float(sb[s + 1]))));
                } else {
                    const float b = __uint_as_float(wv[t]);
                    acc[i] = ffma2(make_float2(__uint_as_float(px[s]), __uint_as_float(px[s + 1])),
                                   make_float2(b, b), acc[i]);
                }
            }
        }
    }
}

// Weight-gradient products in closed form for one channel and lane (x the
// value operand, dy the fraction-and-scale operand for Mitchell).
template <int ALU, int KS = 3>
__device__ __forceinline__ void dw_filter_alu(float2 (&acc)[KS * KS], const uint32_t *xr, int tw, const uint32_t *dr,
                                              int tq)
{
#pragma unroll
    for (int i = 0; i < kDwRB; ++i) {
        const uint2 d01 = *reinterpret_cast<const uint2 *>(dr + i * tq);
        const uint32_t db0 = d01.x & 0xFF800000u, db1 = d01.y & 0xFF800000u;
        const uint32_t od0 = d01.x - db0, od1 = d01.y - db1;
        const float2 sd = make_float2(__uint_as_float(db0), __uint_as_float(db1));
        const float2 dv = make_float2(__uint_as_float(d01.x), __uint_as_float(d01.y));
#pragma unroll
        for (int r = 0; r < KS; ++r) {
            uint32_t px[KS + 1];
            dw_row<KS>(xr + (i + r) * tw, px);
#pragma unroll
            for (int s = 0; s < KS; ++s) {
                const int t = r * KS + s;
                if constexpr (ALU == 1) {
                    const float2 w = make_float2(__uint_as_float(px[s] + od0), __uint_as_float(px[s + 1] + od1));
                    acc[t] = fadd2(acc[t], fmul2_ftz(w, sd));
                } else {
                    acc[t] = ffma2(make_float2(__uint_as_float(px[s]), __uint_as_float(px[s + 1])), dv, acc[t]);
                }
            }
        }
    }
}

// MODE 0: forward; 1: data gradient (the activation is dy, the filter flipped);
// 2: weight gradient (CTA = (channel block, share of the spatial tiles)).
// ALU 0: products from the LUT staged in shared memory; 1 / 2: Mitchell /
// exact products in closed form, the LUT read from global memory only by
// tiles that take the slow computation.
// Thread 0 copies the next tile's raw boxes while the CTA computes the
// current one; every wait on the copy is bounded (a timeout is recorded and
// the CTA leaves its remaining tiles).
template <int W, int MODE, int ALU, bool WIDE, int KS = 3>
__global__ void __launch_bounds__(kDwThreads, 2) dw_tile_kernel(const __grid_constant__ DwTileParams p)
{
    using amsim::kern::mbar_init;
    using amsim::kern::mbar_wait;
    extern __shared__ __align__(128) uint8_t smem[];
    using Cfg = DwCfg<MODE, KS>;
    constexpr int CB = Cfg::CB, CPW = Cfg::CPW, KK = Cfg::KK, CP = Cfg::CP;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // tile shape: compile-time for the widest (8 x 64) tiles, else from the launch
    const int lq_shift = WIDE ? 5 : p.lq_shift, tq_shift = WIDE ? 6 : p.tq_shift;
    const int tq = WIDE ? 64 : p.tq, tw = WIDE ? 64 + KS - 1 : p.tw, th = WIDE ? 8 + KS - 1 : p.th;
    const int tpr = WIDE ? 8 : p.tp;
    uint8_t *lut = smem;
    const uint8_t *glut = static_cast<const uint8_t *>(p.table);         // slow closed-form tiles
    float *rawA = reinterpret_cast<float *>(smem + (ALU ? 0 : dw_lut_region(p.table_bytes)));
    uint32_t *xt = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(rawA) + Cfg::RawA);
    uint8_t *after = reinterpret_cast<uint8_t *>(xt) + Cfg::Halo;
    float *rawB = reinterpret_cast<float *>(after);                       // mode 2
    uint32_t *dyt = reinterpret_cast<uint32_t *>(after + Cfg::RawB);      // mode 2
    uint32_t *wt_off = reinterpret_cast<uint32_t *>(after);               // modes 0, 1
    float *wt_scl = reinterpret_cast<float *>(after + CB * KK * 4);
    uint32_t *wt_val = reinterpret_cast<uint32_t *>(after + 2 * CB * KK * 4);   // closed forms
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
        const int tqi = rest % p.tiles_q;
        rest /= p.tiles_q;
        d.p0 = (rest % p.tiles_p) * tpr;
        d.n = rest / p.tiles_p;
        d.q0 = tqi * tq;
        d.c0 = cb * CB;
        return d;
    };

    if (tid == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (t_begin < t_end) dw_issue<MODE>(p, tile_at(t_begin), rawA, rawB, bar);
    }
    if constexpr (ALU == 0) {   // LUT -> shared memory (the device table is padded to 256 bytes)
        const uint4 *src = static_cast<const uint4 *>(p.table);
        uint4 *dst = reinterpret_cast<uint4 *>(lut);
        const int nvec = (p.table_bytes + 15) >> 4;
        for (int i = tid; i < nvec; i += kDwThreads) dst[i] = __ldg(src + i);
    }
    // the barrier's initialisation (thread 0) and the staged table are visible to
    // every thread before any of them waits on the barrier or reads the table
    __syncthreads();
    const int hi_shift = p.M + p.wlog, lo_shift = p.wlog;

    float2 facc[CPW][MODE == 2 ? KK : 1];   // mode 2: per-tap sums of this CTA's share
    if constexpr (MODE == 2) {
#pragma unroll
        for (int ci = 0; ci < CPW; ++ci)
#pragma unroll
            for (int t = 0; t < KK; ++t) facc[ci][t] = make_float2(0.0f, 0.0f);
    }
    uint32_t phase = 0;
    bool aborted = false;
    for (int t = t_begin; t < t_end; t += t_step) {
        const DwTile tl = tile_at(t);
        mbar_wait(bar, phase, aborted);
        phase ^= 1;
        // also orders the previous tile's shared-memory reads before this tile's packing
        if (__syncthreads_or(aborted)) break;
        bool big = false;
        const int a_shift = MODE == 2 ? hi_shift : lo_shift;
        const uint32_t keep = ((1u << p.M) - 1u) << (23 - p.M);
        if constexpr (ALU != 0) {
            dw_pack_box_alu<CB>(rawA, xt, th * tw, CP, keep, tid, big);
            if constexpr (MODE == 2) dw_pack_box_alu<CB>(rawB, dyt, kDwTileOut, kDwOP, keep, tid, big);
        } else {
            dw_pack_box<CB>(rawA, xt, th * tw, CP, 23 - p.M - a_shift, ((1u << p.M) - 1u) << a_shift, tid,
                            big);
            if constexpr (MODE == 2)
                dw_pack_box<CB>(rawB, dyt, kDwTileOut, kDwOP, 23 - p.M - lo_shift, ((1u << p.M) - 1u) << lo_shift,
                                tid, big);
        }
        if (MODE != 2 && tid < CB * KK) {
            const int c = tid / KK, tap = tid % KK;
            const int src_t = MODE == 0 ? tap : KK - 1 - tap;   // the data gradient reads the filter rotated by 180 degrees
            const float v = tl.c0 + c < p.C ? __ldg(p.b + (long long)src_t * p.C + tl.c0 + c) : 0.0f;
            int wbig = 0;
            const uint32_t pk = dw_pack(v, p.M, hi_shift, wbig);
            big |= wbig != 0;
            wt_off[tid] = pk - dw_scale_bits(pk);
            wt_scl[tid] = __uint_as_float(dw_scale_bits(pk));
            if constexpr (ALU != 0) wt_val[tid] = dw_pack_alu(v, keep, big);
        }
        const bool slow = __syncthreads_or(big);   // the raw boxes are consumed
        if (tid == 0 && t + t_step < t_end) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            dw_issue<MODE>(p, tile_at(t + t_step), rawA, rawB, bar);
        }
        if (slow) {
            // a tile with |x| >= 2^64, infinities or NaN (closed forms: also
            // nonzero |x| < 2^-63): pack it again exactly for the table (NaN
            // kept as NaN) from global memory, then take the slow products
            dw_repack<CB>(p.a, xt, CP, tl.n, p.IH, p.IW, p.C, tl.p0 + p.oy, tl.q0 + p.ox, tl.c0, th, tw, p.M,
                      a_shift, tid);
            if constexpr (MODE == 2)
                dw_repack<CB>(p.b, dyt, kDwOP, tl.n, p.OH, p.OW, p.C, tl.p0, tl.q0, tl.c0, tpr, tq, p.M, lo_shift,
                          tid);
            __syncthreads();
        }

        // lane -> (row block rb of 8 output rows, column pair lc) of the tile
        const int rb = lane >> lq_shift, lc = lane & ((1 << lq_shift) - 1);
        if constexpr (MODE == 2) {
            const int rows_ok = p.OH - (tl.p0 + rb * kDwRB);
            const bool ok0 = tl.q0 + 2 * lc < p.OW, ok1 = tl.q0 + 2 * lc + 1 < p.OW;
#pragma unroll
            for (int ci = 0; ci < CPW; ++ci) {
                const int c = warp + 8 * ci;
                const uint32_t *xr = xt + c * CP + rb * kDwRB * tw + 2 * lc;
                const uint32_t *dr = dyt + c * kDwOP + rb * kDwRB * tq + 2 * lc;
                if constexpr (ALU != 0) {
                    if (slow)
                        dw_filter_channel<W, true, true, KS>(facc[ci], xr, tw, dr, tq, glut, rows_ok, ok0, ok1,
                                                             p.expand_mul);
                    else
                        dw_filter_alu<ALU, KS>(facc[ci], xr, tw, dr, tq);
                } else {
                    if (slow)
                        dw_filter_channel<W, true, false, KS>(facc[ci], xr, tw, dr, tq, lut, rows_ok, ok0, ok1,
                                                              p.expand_mul);
                    else
                        dw_filter_channel<W, false, false, KS>(facc[ci], xr, tw, dr, tq, lut, rows_ok, ok0, ok1,
                                                               p.expand_mul);
                }
            }
        } else {
            float2 acc[CPW][kDwRB];
#pragma unroll
            for (int ci = 0; ci < CPW; ++ci) {
                const int c = warp + 8 * ci;
                uint32_t woff[KK];
                float wsc[KK];
#pragma unroll
                for (int k = 0; k < KK; ++k) {
                    woff[k] = wt_off[c * KK + k];
                    wsc[k] = wt_scl[c * KK + k];
                }
                const uint32_t *xr = xt + c * CP + rb * kDwRB * tw + 2 * lc;
                if constexpr (ALU != 0) {
                    if (slow) {
                        dw_taps_channel<W, true, true, KS>(acc[ci], xr, tw, glut, woff, wsc, p.expand_mul);
                    } else {
                        uint32_t wv[KK];
#pragma unroll
                        for (int k = 0; k < KK; ++k) wv[k] = wt_val[c * KK + k];
                        dw_taps_alu<ALU, KS>(acc[ci], xr, tw, wv);
                    }
                } else {
                    if (slow)
                        dw_taps_channel<W, true, false, KS>(acc[ci], xr, tw, lut, woff, wsc, p.expand_mul);
                    else
                        dw_taps_channel<W, false, false, KS>(acc[ci], xr, tw, lut, woff, wsc, p.expand_mul);
                }
            }
            __syncthreads();                // every warp is done with the packed halo
            float *ot = reinterpret_cast<float *>(xt);
#pragma unroll
            for (int ci = 0; ci < CPW; ++ci) {
                float *o = ot + (warp + 8 * ci) * kDwOP + rb * kDwRB * tq + 2 * lc;
#pragma unroll
                for (int i = 0; i < kDwRB; ++i) *reinterpret_cast<float2 *>(o + i * tq) = acc[ci][i];
            }
            __syncthreads();
            float *dst = p.out + (long long)tl.n * p.OH * p.OW * p.C;
            constexpr int G4 = CB / 4;      // 4-channel groups of the tile
#pragma unroll 4
            for (int e = tid; e < kDwTileOut * G4; e += kDwThreads) {
                const int c4 = e % G4, pos = e / G4;
                const int i = pos >> tq_shift, j = pos & (tq - 1);
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
            for (int k = 0; k < KK; ++k) {
                float v = facc[ci][k].x + facc[ci][k].y;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                if (lane == 0 && c < p.C) p.out[((long long)g * KK + k) * p.C + c] = v;
            }
        }
    }
}

// Launch the tiled kernel for a narrowed table of `width` bits (8 or 16).
template <int MODE, int ALU, int KS = 3>
int launch_tile(int width, const DwTileParams &tp, int grid, size_t smem, cudaStream_t st)
{
    const bool wide = tp.lq_shift == 5;
    auto kfn = width == 8 ? (wide ? dw_tile_kernel<8, MODE, ALU, true, KS> : dw_tile_kernel<8, MODE, ALU, false, KS>)
                          : (wide ? dw_tile_kernel<16, MODE, ALU, true, KS>
                                  : dw_tile_kernel<16, MODE, ALU, false, KS>);
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return amsim::cuda_status(e);
    kfn<<<grid, kDwThreads, smem, st>>>(tp);
    return amsim::cuda_status(cudaGetLastError());
}

}  // namespace dw
}  // namespace amsim
