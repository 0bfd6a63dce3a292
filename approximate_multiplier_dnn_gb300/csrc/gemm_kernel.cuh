// LUT-GEMM kernel family: out[u][l] = sum_k AMSim(U[u][k], L[l][k]) with fp32
// accumulation (ApproxTrain Sec. V-B Algorithm 2 per product; Sec. VI-D GEMM
// kernel; Sec. VI-B Algorithms 3/4 as implicit GEMM through gather operands).
//
// Design (sm_103a, no tensor cores -- the multiply is not an IEEE multiply):
//  * The narrowed mantissa-product LUT sits in shared memory (global memory,
//    read-only path, when it does not fit).  Each warp owns TM "uniform" rows
//    (same U element for all 32 lanes in one lookup) and 32*TN lane columns, so
//    every LUT load of a warp reads one LUT row: with 8-bit entries a row of
//    128 entries is 32 words, one per bank, and the lookup is conflict-free.
//  * Operand tiles are staged through registers (loads for tile t+1 are in
//    flight while tile t is computed) and pre-decoded once per CTA into
//    (LUT byte offset, signed power-of-two scale): the decode applies the
//    denormal-as-zero, NaN and infinity rules of the ABI.
//  * Per product: one index add, one LUT load, one integer multiply-add that
//    rebuilds v = 1.mantissa * 2^carry as an fp32 bit pattern, and half of a
//    packed fp32x2 multiply (scale = sa*sb, flush-to-zero gives the page's
//    "zero when the biased exponent is not above zero") and half of a packed
//    fp32x2 FMA acc += v*scale.  v*scale is exact unless it overflows; tiles
//    holding an operand with |x| >= 2^64 take a slower path that rounds the
//    product to fp32 (infinity on overflow) before the add, exactly as
//    Algorithm 2 then an fp32 add would.
#pragma once

#include <cuda_runtime.h>

#include "amsim_internal.h"

#ifdef AMSIM_WIDE_TILES
#define AMSIM_KNS kern_wide
#else
#define AMSIM_KNS kern
#endif

namespace amsim {
namespace kern {

#ifndef AMSIM_NT
#define AMSIM_NT 256
#endif
#ifndef AMSIM_BU
#define AMSIM_BU 64
#endif
#ifndef AMSIM_BL
#define AMSIM_BL 256
#endif
#ifndef AMSIM_BK
#define AMSIM_BK 16
#endif
#ifndef AMSIM_TM
#define AMSIM_TM 16
#endif
#ifndef AMSIM_TN
#define AMSIM_TN 4
#endif
#ifndef AMSIM_KK_UNROLL
#define AMSIM_KK_UNROLL 1
#endif
// Tile shape of a LUT-GEMM kernel instance: BU uniform rows x BL lane columns
// per CTA tile, BK reduction steps per stage, TM uniform rows per warp and TN
// lane columns per thread.  Every kernel is built with the narrow shape; the
// predecoded (TMA) kernel is built with the wide one too, whose eight lane
// columns per thread halve the shared-memory wavefronts of the uniform
// operands' loads per lookup (1/TN of a lookup's).
struct TileCfg {
    int bu, bl, bk, tm, tn;
};
constexpr TileCfg kNarrowTiles = {AMSIM_BU, AMSIM_BL, AMSIM_BK, AMSIM_TM, AMSIM_TN};
constexpr TileCfg kWideTiles = {128, 256, 16, 16, 8};

struct RowInfo {
    int y, x;
    long long b;
};

constexpr int kMaxProblems = 10;     // contractions fused into one launch
constexpr int kMaxFixupParts = 1024;  // stream-K CTAs per launch (at most one per SM)
constexpr int kMaxPhases = 6;        // ordered phases of one launch (raw-tile kernel)
constexpr int kMaxPhasedCtas = 160;  // CTAs of a phased launch

// One contraction of a launch (see Problem in amsim_internal.h).
struct ProbParams {
    OperandDesc U, L;
    int K, batch;
    int tiles_u, tiles_l, kt_total;
    long long tiles;        // tiles_u * tiles_l * batch
    long long iter0;        // first iteration of this problem in the launch's iteration space
    long long tile0;        // first tile of this problem among the launch's tiles
    const void *table;      // LUT oriented [U mantissa][L mantissa]
    float *c_ptr;
    long long c_bs, c_su, c_sl;
    float alpha, beta;
    int u_kfast, l_kfast;
    // Predecoded operands (TMA kernel only): each plane's "holds an element
    // with |x| >= 2^64" flag, raised when it equals the launch epoch, and the
    // batch coordinate factor (0 when one plane serves every batch).
    const unsigned long long *u_big, *l_big;
    // ... its "holds an element with 0 < |x| < 2^-63" and "holds a zero (or a
    // denormal)" flags
    const unsigned long long *u_small, *l_small;
    int u_bsel, l_bsel;
    // Raw-tile kernel: the operand is read with plain loads by the decoders
    // (strides the copy engine cannot take) instead of a tensor box.
    int u_direct, l_direct;
};

// A launch: the (problem, tile, stage) iterations of all problems laid end to
// end.  Data-parallel mode: CTA c runs tile c whole.  Stream-K mode: CTA c
// runs iterations [c*W/G, (c+1)*W/G); a tile cut between CTAs leaves partial
// sums in per-CTA slots that a fixup kernel adds in CTA order.
struct KParams {
    ProbParams pr[kMaxProblems];
    int nprob;
    int streamk;
    long long iters;        // W
    int ctas;               // G (stream-K)
    int table_bytes;        // bytes staged to shared memory (0 when read from global)
    int M;
    int wlog;               // log2(entry bytes)
    float *ws;              // stream-K partial slots [G][2][BU*BL], then [G][2] epoch flags
    int fused;              // stream-K cut tiles are finished inside the kernel (cooperative launch)
    int stages;             // TMA kernel: stages in the shared-memory ring
    unsigned long long epoch;   // this launch's flag value (never reused)
    // Raw-tile kernel, convolution operands (one problem): conv 0 plain
    // operands, 1 whole-row L boxes per filter tap, 2 blocked-channel L boxes
    // (see ConvRaw); cv_u_tap: U boxes addressed (step in tap, row, tap)
    int conv, cv_u_tap;
    int direct;             // raw-tile kernel: some operand is read with plain loads
    int alu;                // raw-tile kernel: closed-form products, no table (1 Mitchell, 2 exact)
    // Phases (raw-tile kernel, fused stream-K): phase ph holds launch
    // iterations [ph_iter0[ph], ph_iter0[ph + 1]) -- whole problems; every CTA
    // takes a share of every phase (PhaseTable), in phase order, and loads
    // nothing of phase ph before phases 0 .. ph_after[ph] - 1 are complete on
    // every CTA.  nphase 0 or 1: an ordinary launch.
    int nphase;
    long long ph_iter0[kMaxPhases + 1];
    int ph_after[kMaxPhases];
    // Stream-K shares cut by stage cost (raw-tile kernel, ordinary launches):
    // when sk_n > 0, CTA c takes iterations [sk_bound[c], sk_bound[c + 1]),
    // strictly increasing; else the even split W * c / G.
    int sk_n;
    int sk_bound[kMaxPhasedCtas + 1];
    int cv_ch, cv_S, cv_tiles_img, cv_rows_tile, cv_ybase, cv_ystep, cv_xbase, cv_xstep, cv_N, cv_P, cv_Q, cv_rows;
    // (1, E, M) format with E < 8 (fmt.on): operands are cast and every stage
    // takes the rounding product path with the format's rescale and overflow
    // (in-kernel-decode and single-role kernels only; the host routes such
    // launches to them)
    ExpFormat fmt;
};

}  // namespace kern

// Everything below depends on the tile shape and is built once per shape: in
// namespace kern with the narrow shape, in kern_wide with the wide one (a
// translation unit that defines AMSIM_WIDE_TILES before including this file).
namespace AMSIM_KNS {

#ifdef AMSIM_WIDE_TILES
using namespace ::amsim::kern;
constexpr TileCfg kTiles = kWideTiles;
#else
constexpr TileCfg kTiles = kNarrowTiles;
#endif
constexpr int kKkUnroll = AMSIM_KK_UNROLL;   // reduction steps unrolled per loop iteration
constexpr int NT = AMSIM_NT;       // threads per CTA
constexpr int BU = kTiles.bu;       // uniform rows per CTA tile
constexpr int BL = kTiles.bl;       // lane columns per CTA tile
constexpr int BK = kTiles.bk;       // reduction depth per stage
constexpr int TM = kTiles.tm;       // uniform rows per warp (processed in pairs)
constexpr int TN = kTiles.tn;       // lane columns per thread
constexpr int WU = BU / TM;        // warps along U
constexpr int WL = BL / (32 * TN); // warps along L
constexpr int UST = BU + 4;        // decoded U row stride (words), 16-B aligned, few bank conflicts
constexpr int LST = BL + 4;        // decoded L row stride (words)
constexpr int NUE = BU * BK / NT;  // U elements loaded per thread per stage
constexpr int NLE = BL * BK / NT;  // L elements loaded per thread per stage
static_assert(TM % 4 == 0 && TN % 4 == 0, "micro-tile");
static_assert(NT % BK == 0 && (NT % BU == 0 || BU % NT == 0) && (NT % BL == 0 || BL % NT == 0), "loader mapping");
static_assert(WU * WL * 32 == NT, "warp layout");
// Lane columns: register column t of a lane is column lane*4 + col_of(t) of
// its warp's 32*TN-column span -- groups of four columns, the groups 128
// columns apart -- so each 128-bit load of one group reads 512 contiguous
// bytes across the warp (four wavefronts, no bank conflicts) whatever TN is.
constexpr int kColGroup = 128;
__host__ __device__ constexpr int col_of(int t) { return (t >> 2) * kColGroup + (t & 3); }
// Tail layout of the two-column-block shape: a tile whose real lane columns
// all lie in its first column block (at most 32 * TN of them) is computed by
// all the warps as WU * WL row blocks of TM / 2 rows over that block, instead
// of leaving the warps of the second block idle -- which, as they are every
// other warp and warps go to the SM's four schedulers by warp index modulo 4,
// would also leave two of the schedulers without a busy warp.  Each output's
// products are summed in the same order either way.
// A tile with at most 64 real lane columns takes the narrow tail layout: the
// same row blocks over 64 columns, two per lane (lane * 2, lane * 2 + 1).
constexpr bool kTailLayout = WL == 2 && (TM / 2) * WU * WL == BU && TM % 8 == 0;
constexpr int kTailRows = TM / 2;
constexpr int kNarrowTailCols = 2;
__host__ __device__ constexpr bool tail_tile(int l_tile0, int l_rows)
{
    return kTailLayout && l_tile0 + 32 * TN >= l_rows;
}
__host__ __device__ constexpr bool narrow_tail_tile(int l_tile0, int l_rows)
{
    return kTailLayout && l_tile0 + 32 * kNarrowTailCols >= l_rows;
}

// Shared-memory layout (bytes) after the LUT region.
constexpr int kUdecBytes = 2 * BK * UST * 4;   // one array (offsets or scales), 2 stages
constexpr int kLdecBytes = 2 * BK * LST * 4;
constexpr int kRowTabBytes = (BU + BL) * (int)sizeof(RowInfo);
constexpr int kFixedSmem = 2 * kUdecBytes + 2 * kLdecBytes + kRowTabBytes;

__host__ __device__ constexpr int lut_region_bytes(int table_bytes) { return (table_bytes + 127) & ~127; }

// This thread's warp index broadcast from lane 0: threadIdx.x / 32, as a value
// the compiler can see is the same across the warp, so that the uniform
// operands' shared-memory addresses and loads are treated as uniform.
// Measured on GB300 (predecoded 4096^3 GEMM): 2.6 % faster with two planes,
// and packed operand words cost 0.2 more instructions per lookup instead of
// 1.2.  Every lane of the warp must take part.
__device__ __forceinline__ int uniform_warp() { return __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0); }

// ------------------------------------------------------------------ fp32x2 helpers
__device__ __forceinline__ float2 fmul2_ftz(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.ftz.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// ------------------------------------------------------------------ LUT access
template <int W, bool GL>
__device__ __forceinline__ uint32_t lut_ld(const uint8_t *lut, uint32_t off)
{
    if constexpr (GL) {
        if constexpr (W == 8) return __ldg(lut + off);
        else if constexpr (W == 16) return __ldg(reinterpret_cast<const uint16_t *>(lut + off));
        else return __ldg(reinterpret_cast<const uint32_t *>(lut + off));
    } else {
        if constexpr (W == 8) return *(lut + off);
        else if constexpr (W == 16) return *reinterpret_cast<const uint16_t *>(lut + off);
        else return *reinterpret_cast<const uint32_t *>(lut + off);
    }
}

// v = 2^carry * 1.mantissa as fp32: the canonical entry (narrowed entry <<
// (24 - W) for 8/16-bit tables, the entry itself for 32-bit ones) plus the bit
// pattern of 1.0f.  A shift and an add keep this off the FMA pipes, which
// carry the scale multiply and the accumulation.
// v = 2^carry * 1.mantissa as fp32: the canonical entry (narrowed entry <<
// (24 - W) for 8/16-bit tables, the entry itself for 32-bit ones) plus the bit
// pattern of 1.0f.  (A shift-and-add or a multiply-add by 2^(24-W) compile to
// the same instruction.)
template <int W>
__device__ __forceinline__ float expand(uint32_t narrowed)
{
    uint32_t r;
    if constexpr (W == 32) {
        r = narrowed + 0x3F800000u;
    } else {
        asm("shl.b32 %0, %1, %2;\n\tadd.u32 %0, %0, 0x3F800000;" : "=r"(r) : "r"(narrowed), "n"(24 - W));
    }
    return __uint_as_float(r);
}

// Operand decode (once per element per CTA): byte offset of the mantissa's LUT
// row/column and the signed power-of-two scale 2^(e-127).  Zero and denormal
// inputs give a signed zero scale, infinities an infinite scale, NaN a NaN scale.
// zoff: for uniform (U) operands the byte offset of the table's zero row
// (uniform_zero_row), which zero and denormal elements take -- so that the
// folded form rebuilds a signed zero from them -- and 0 for lane operands.
__device__ __forceinline__ void decode(float v, int M, int offshift, uint32_t &off, float &s, int &big, uint32_t zoff)
{
    const uint32_t x = __float_as_uint(v);
    const uint32_t e = (x >> 23) & 0xFFu;
    const uint32_t f = x & 0x7FFFFFu;
    off = (e == 0u && zoff) ? zoff : (f >> (23 - M)) << offshift;
    uint32_t sb = x & 0xFF800000u;          // e == 0 leaves only the sign
    if (e == 255u && f) sb = 0x7FC00000u;
    s = __uint_as_float(sb);
    big |= (e >= 191u);
}

// Packed operand word (predecoded planes with the table in shared memory):
// the LUT byte offset in bits 10..31 and the top ten bits of the scale (sign,
// biased exponent, and the quiet bit that tells NaN from infinity; the scale's
// other bits are zero) in bits 0..9.  A zero word is offset 0 and scale +0.0,
// as an all-zero pair of plane words.  Offsets must stay below 2^22.
constexpr int kPackShift = 10;
__device__ __forceinline__ uint32_t pack_operand(uint32_t off, float s)
{
    return (off << kPackShift) | (__float_as_uint(s) >> (32 - kPackShift));
}
__device__ __forceinline__ uint32_t packed_off(uint32_t w) { return w >> kPackShift; }
// The scale's bit pattern: w * 2^22 (a multiply-add-pipe shift, which keeps
// the integer pipe that carries the index adds free).
__device__ __forceinline__ uint32_t packed_scale_bits(uint32_t w)
{
    uint32_t r;
    asm("mul.lo.u32 %0, %1, %2;" : "=r"(r) : "r"(w), "n"(1u << (32 - kPackShift)));
    return r;
}

// Byte offset of the zero row that every narrowed table carries after its 2^M
// rows (all entries zero): row 2^M of a table whose rows are 2^M entries of
// 2^(offshift - M) bytes, offshift being the uniform operand's offset shift.
// With it a zero uniform operand's folded entry is its scale bits alone, a
// signed zero, and the general form's entry is 1.0 times a zero scale.
__host__ __device__ __forceinline__ uint32_t uniform_zero_row(int M, int offshift)
{
    return (1u << M) << offshift;
}

// Scale bits of an operand after the exponent cast of a (1, E, M) format,
// re-biased by `off` (see ExpFormat): NaN stays NaN, fp32 infinities and
// operands above the format's range are signed infinities, zero, denormal and
// operands below its range signed zeros.  E = 8 (lo 1, hi 254, off 0) gives
// the fp32 scale of decode().
__device__ __forceinline__ uint32_t fmt_scale_bits(uint32_t x, int lo, int hi, int off)
{
    const uint32_t e = (x >> 23) & 0xFFu, sgn = x & 0x80000000u;
    if (e == 255u) return (x & 0x7FFFFFu) ? 0x7FC00000u : (sgn | 0x7F800000u);
    if ((int)e < lo) return sgn;
    if ((int)e > hi) return sgn | 0x7F800000u;
    return sgn | ((uint32_t)((int)e + off) << 23);
}

__device__ __forceinline__ void decode_fmt(float v, int M, int offshift, const ExpFormat &f, int off, uint32_t &o,
                                           float &s)
{
    const uint32_t x = __float_as_uint(v);
    o = ((x & 0x7FFFFFu) >> (23 - M)) << offshift;
    s = __uint_as_float(fmt_scale_bits(x, f.lo, f.hi, off));
}

// The product in a (1, E, M) format from the entry value v = 1.mant * 2^carry
// and the two cast scales: the flush-to-zero scale product is Algorithm 2's
// zero test, vscale undoes the scales' re-bias exactly, and products at or
// above 2^(B + 1) are Algorithm 2's overflow.  Rounded to fp32 (it is exact).
__device__ __forceinline__ float fmt_product(float v, float s, const ExpFormat &f)
{
    const float p = __fmul_rn(__fmul_rn(v, s), f.vscale);
    return fabsf(p) >= f.lim ? __uint_as_float((__float_as_uint(p) & 0x80000000u) | 0x7F800000u) : p;
}

// A nonzero operand whose magnitude is below 2^-63 (biased exponent 1 .. 63;
// zero and denormal excluded).  Stages whose operands are all zero or in
// [2^-63, 2^64) have every e0 = eA + eB - 127 of a nonzero pair in [1, 253]:
// no product meets Algorithm 2's zero test or its overflow.  A zero (or
// denormal) lane operand has a signed zero scale, and a zero uniform operand
// takes the table's zero row: both folded products are the signed zero
// Algorithm 2 gives.
__device__ __forceinline__ bool is_small_nonzero(float v) { return ((__float_as_uint(v) >> 23) & 0xFFu) - 1u < 63u; }

// v * sa for a uniform operand with scale bits ub = sign | eA << 23, straight
// from the narrowed entry: adding the entry's bits (carry at bit 23, mantissa
// below) to ub gives the fp32 bits of +-1.mant * 2^(eA - 127 + carry), exactly
// as expand() gives those of 1.mant * 2^carry for ub = bits(1.0f).  Valid while
// eA + carry <= 254 and eA >= 1: a stage whose operands are all in
// [2^-63, 2^64) (then eA is in [64, 190]).
template <int W>
__device__ __forceinline__ float expand_scaled(uint32_t narrowed, uint32_t ub)
{
    uint32_t r;
    if constexpr (W == 32) {
        r = narrowed + ub;
    } else {
        asm("shl.b32 %0, %1, %2;\n\tadd.u32 %0, %0, %3;" : "=r"(r) : "r"(narrowed), "n"(24 - W), "r"(ub));
    }
    return __uint_as_float(r);
}

// ------------------------------------------------------------------ gather state
struct KState {
    int k0, k1;
    int y, x;
    long long b;
};

__device__ __forceinline__ KState kstate_at(const OperandDesc &d, int k)
{
    KState s;
    int t = k / d.kD0;
    s.k0 = k - t * d.kD0;
    int k2 = t / d.kD1;
    s.k1 = t - k2 * d.kD1;
    s.y = s.k0 * d.kcy[0] + s.k1 * d.kcy[1] + k2 * d.kcy[2];
    s.x = s.k0 * d.kcx[0] + s.k1 * d.kcx[1] + k2 * d.kcx[2];
    s.b = (long long)s.k0 * d.kcb[0] + (long long)s.k1 * d.kcb[1] + (long long)k2 * d.kcb[2];
    return s;
}

// Advance by delta >= 0 with carries between levels (no division).
__device__ __forceinline__ void kstate_advance(const OperandDesc &d, KState &s, int delta)
{
    s.k0 += delta;
    s.y += delta * d.kcy[0];
    s.x += delta * d.kcx[0];
    s.b += (long long)delta * d.kcb[0];
    while (s.k0 >= d.kD0) {
        s.k0 -= d.kD0;
        s.y += d.kcy[1] - d.kD0 * d.kcy[0];
        s.x += d.kcx[1] - d.kD0 * d.kcx[0];
        s.b += d.kcb[1] - (long long)d.kD0 * d.kcb[0];
        if (++s.k1 >= d.kD1) {
            s.k1 = 0;
            s.y += d.kcy[2] - d.kD1 * d.kcy[1];
            s.x += d.kcx[2] - d.kD1 * d.kcx[1];
            s.b += d.kcb[2] - (long long)d.kD1 * d.kcb[1];
        }
    }
}

__device__ __forceinline__ RowInfo row_info(const OperandDesc &d, int r)
{
    RowInfo ri;
    if (r >= d.rows) {
        ri.y = -(1 << 29);     // never in range
        ri.x = 0;
        ri.b = 0;
        return ri;
    }
    int t = r / d.rE0;
    int r0 = r - t * d.rE0;
    int r2 = t / d.rE1;
    int r1 = t - r2 * d.rE1;
    ri.y = d.ry0 + r0 * d.rcy[0] + r1 * d.rcy[1] + r2 * d.rcy[2];
    ri.x = d.rx0 + r0 * d.rcx[0] + r1 * d.rcx[1] + r2 * d.rcx[2];
    ri.b = (long long)r0 * d.rcb[0] + (long long)r1 * d.rcb[1] + (long long)r2 * d.rcb[2];
    return ri;
}

__device__ __forceinline__ float gather_value(const OperandDesc &d, const float *base, const RowInfo &ri,
                                              const KState &ks)
{
    int y = ri.y + ks.y, x = ri.x + ks.x;
    if (d.sy > 1) {
        if (y < 0 || y % d.sy) return 0.0f;
        y /= d.sy;
    }
    if (d.sx > 1) {
        if (x < 0 || x % d.sx) return 0.0f;
        x /= d.sx;
    }
    if ((unsigned)y >= (unsigned)d.IH || (unsigned)x >= (unsigned)d.IW) return 0.0f;
    return __ldg(base + ri.b + ks.b + ((long long)y * d.IW + x) * d.Cs);
}

// ------------------------------------------------------------------ operand loader
// R rows per tile, N = R*BK/NTH elements per thread per stage (NTH loading
// threads).  "k-fast": thread t owns reduction slot t % BK and rows
// t/BK + (NTH/BK) e.  "row-fast": thread t owns row t % R (t + NTH*j when
// R > NTH) and the reduction slots left over.  The host picks the mapping that makes consecutive threads touch
// consecutive addresses.
template <int R, int N, int NTH = NT>
struct Loader {
    static constexpr int RRF = R > NTH ? R / NTH : 1;    // row repeats per thread (row-fast)
    static constexpr int KSF = R < NTH ? NTH / R : 1;    // reduction-slot stride (row-fast)
    static_assert(R * BK == N * NTH, "loader element count");
    bool kfast;
    int rsub, ksub0;
    int row0;               // global row of tile row 0
    const float *base;      // operand pointer + batch offset
    KState ks;              // gather state at k = stage*BK + ksub0
    float v[N];

    __device__ __forceinline__ int row_of(int e) const
    {
        return kfast ? rsub + (NTH / BK) * e : rsub + NTH * (e % RRF);
    }
    __device__ __forceinline__ int k_of(int e) const { return kfast ? ksub0 : ksub0 + KSF * (e / RRF); }

    __device__ __forceinline__ void init(const OperandDesc &d, bool kf, int tid, int row_tile0, int b, int kt_first)
    {
        kfast = kf;
        if (kfast) { rsub = tid / BK; ksub0 = tid % BK; }
        else if (R <= NTH) { rsub = tid % R; ksub0 = tid / R; }
        else { rsub = tid; ksub0 = 0; }
        row0 = row_tile0;
        base = d.ptr + (long long)b * d.batch_stride;
        if (d.gather) ks = kstate_at(d, kt_first * BK + ksub0);
    }

    __device__ __forceinline__ void load(const OperandDesc &d, const RowInfo *rowtab, int kt, int K)
    {
        const int kbase = kt * BK;
        if (!d.gather) {
#pragma unroll
            for (int e = 0; e < N; ++e) {
                const int r = row0 + row_of(e);
                const int k = kbase + k_of(e);
                v[e] = (r < d.rows && k < K) ? __ldg(base + (long long)r * d.s_row + (long long)k * d.s_k) : 0.0f;
            }
        } else {
            KState s = ks;
            int kprev = k_of(0);
#pragma unroll
            for (int e = 0; e < N; ++e) {
                const int kk = k_of(e);
                if (kk != kprev) { kstate_advance(d, s, kk - kprev); kprev = kk; }
                const RowInfo ri = rowtab[row_of(e)];
                v[e] = (kbase + kk < K) ? gather_value(d, base, ri, s) : 0.0f;
            }
            kstate_advance(d, ks, BK);
        }
    }

    // Decode into the stage buffers: off[k][row], scale[k][row] (row stride ST words).
    template <int ST>
    __device__ __forceinline__ void store(uint32_t *off, float *scl, int M, int offshift, int &big,
                                          uint32_t zoff) const
    {
#pragma unroll
        for (int e = 0; e < N; ++e) {
            const int r = row_of(e);
            const int k = k_of(e);
            uint32_t o;
            float s;
            decode(v[e], M, offshift, o, s, big, zoff);
            off[k * ST + r] = o;
            scl[k * ST + r] = s;
        }
    }
    // The same with the exponent cast of a (1, E, M) format.
    template <int ST>
    __device__ __forceinline__ void store_fmt(uint32_t *off, float *scl, int M, int offshift, const ExpFormat &f,
                                              int eoff) const
    {
#pragma unroll
        for (int e = 0; e < N; ++e) {
            uint32_t o;
            float s;
            decode_fmt(v[e], M, offshift, f, eoff, o, s);
            off[k_of(e) * ST + row_of(e)] = o;
            scl[k_of(e) * ST + row_of(e)] = s;
        }
    }
};

// ------------------------------------------------------------------ compute
// Accumulator of uniform row i, lane column t.
__device__ __forceinline__ float accv(const float2 (&acc)[TM / 2][TN], int i, int t)
{
    return (i & 1) ? acc[i >> 1][t].y : acc[i >> 1][t].x;
}

// One stage of BK reduction steps.  acc[p][t] holds rows (2p, 2p+1) of the
// warp's TM uniform rows for lane column t, so the U scales pair up straight
// from the vector loads and only the L scale is duplicated (once per column).
// FMT: a (1, E, M) format with E < 8 -- every product through fmt_product
// (rounded, then added), whatever the stage's magnitudes.
// FOLD: every uniform operand of the stage is in [2^-63, 2^64) and every lane
// operand too or zero -- the uniform
// operand's scale is folded into the rebuilt entry (expand_scaled), so a
// product is v' * sb with no scale product: the same exact value v * (sa * sb)
// the general form adds, one FMA per two products instead of a multiply and
// an FMA, and bit-identical sums.
// PU / PL: the stage holds packed operand words (pack_operand) in Uo / Lo,
// and Us / Ls are not read.  One 128-bit load brings four operands' offsets
// and scales: half the shared-memory wavefronts of two planes.
// ROWS / COLS: this warp's uniform rows and each lane's columns (TM and TN;
// the tail layouts' kTailRows with TN, or with kNarrowTailCols adjacent
// columns from lcol = lane * 2).
template <int W, bool GL, bool SLOW, int USTR = UST, int LSTR = LST, bool FMT = false, bool FOLD = false,
          bool PU = false, bool PL = false, int ROWS = TM, int COLS = TN>
__device__ __forceinline__ void compute_stage(float2 (&acc)[TM / 2][TN], const uint32_t *__restrict__ Uo,
                                              const float *__restrict__ Us, const uint32_t *__restrict__ Lo,
                                              const float *__restrict__ Ls, const uint8_t *lut, int urow, int lcol,
                                              const ExpFormat *fmt = nullptr)
{
    static_assert(COLS == TN || COLS == kNarrowTailCols, "lane columns");
#pragma unroll(kKkUnroll)
    for (int kk = 0; kk < BK; ++kk) {
        uint32_t lo[TN];
        float2 sb[TN];
        if constexpr (COLS == kNarrowTailCols) {
            uint2 o;
            float2 sc;
            if constexpr (PL) {
                const uint2 w = *reinterpret_cast<const uint2 *>(Lo + kk * LSTR + lcol);
                o = make_uint2(packed_off(w.x), packed_off(w.y));
                sc = make_float2(__uint_as_float(packed_scale_bits(w.x)), __uint_as_float(packed_scale_bits(w.y)));
            } else {
                o = *reinterpret_cast<const uint2 *>(Lo + kk * LSTR + lcol);
                sc = *reinterpret_cast<const float2 *>(Ls + kk * LSTR + lcol);
            }
            lo[0] = o.x; lo[1] = o.y;
            sb[0] = make_float2(sc.x, sc.x);
            sb[1] = make_float2(sc.y, sc.y);
        }
#pragma unroll
        for (int t4 = 0; t4 < (COLS == TN ? TN / 4 : 0); ++t4) {
            uint4 o;
            float4 sc;
            if constexpr (PL) {
                const uint4 w = *reinterpret_cast<const uint4 *>(Lo + kk * LSTR + lcol + kColGroup * t4);
                o = make_uint4(packed_off(w.x), packed_off(w.y), packed_off(w.z), packed_off(w.w));
                sc = make_float4(__uint_as_float(packed_scale_bits(w.x)), __uint_as_float(packed_scale_bits(w.y)),
                                 __uint_as_float(packed_scale_bits(w.z)), __uint_as_float(packed_scale_bits(w.w)));
            } else {
                o = *reinterpret_cast<const uint4 *>(Lo + kk * LSTR + lcol + kColGroup * t4);
                sc = *reinterpret_cast<const float4 *>(Ls + kk * LSTR + lcol + kColGroup * t4);
            }
            lo[4 * t4 + 0] = o.x; lo[4 * t4 + 1] = o.y; lo[4 * t4 + 2] = o.z; lo[4 * t4 + 3] = o.w;
            sb[4 * t4 + 0] = make_float2(sc.x, sc.x);
            sb[4 * t4 + 1] = make_float2(sc.y, sc.y);
            sb[4 * t4 + 2] = make_float2(sc.z, sc.z);
            sb[4 * t4 + 3] = make_float2(sc.w, sc.w);
        }
#pragma unroll
        for (int ig = 0; ig < ROWS / 4; ++ig) {
            uint4 uo;
            float4 us;
            if constexpr (PU) {
                const uint4 w = *reinterpret_cast<const uint4 *>(Uo + kk * USTR + urow + 4 * ig);
                uo = make_uint4(packed_off(w.x), packed_off(w.y), packed_off(w.z), packed_off(w.w));
                us = make_float4(__uint_as_float(packed_scale_bits(w.x)), __uint_as_float(packed_scale_bits(w.y)),
                                 __uint_as_float(packed_scale_bits(w.z)), __uint_as_float(packed_scale_bits(w.w)));
            } else {
                uo = *reinterpret_cast<const uint4 *>(Uo + kk * USTR + urow + 4 * ig);
                us = *reinterpret_cast<const float4 *>(Us + kk * USTR + urow + 4 * ig);
            }
            const uint32_t uov[4] = {uo.x, uo.y, uo.z, uo.w};
            const float2 sa[2] = {make_float2(us.x, us.y), make_float2(us.z, us.w)};
            if constexpr (FOLD) {
                const uint32_t ub[4] = {__float_as_uint(us.x), __float_as_uint(us.y), __float_as_uint(us.z),
                                        __float_as_uint(us.w)};
#pragma unroll
                for (int ip = 0; ip < 2; ++ip) {
#pragma unroll
                    for (int t = 0; t < COLS; ++t) {
                        const uint32_t ea = lut_ld<W, GL>(lut, uov[2 * ip] + lo[t]);
                        const uint32_t eb = lut_ld<W, GL>(lut, uov[2 * ip + 1] + lo[t]);
                        const float2 v =
                            make_float2(expand_scaled<W>(ea, ub[2 * ip]), expand_scaled<W>(eb, ub[2 * ip + 1]));
                        acc[2 * ig + ip][t] = ffma2(v, sb[t], acc[2 * ig + ip][t]);
                    }
                }
            } else {
#pragma unroll
                for (int ip = 0; ip < 2; ++ip) {
#pragma unroll
                    for (int t = 0; t < COLS; ++t) {
                        const uint32_t ea = lut_ld<W, GL>(lut, uov[2 * ip] + lo[t]);
                        const uint32_t eb = lut_ld<W, GL>(lut, uov[2 * ip + 1] + lo[t]);
                        const float2 v = make_float2(expand<W>(ea), expand<W>(eb));
                        const float2 s = fmul2_ftz(sa[ip], sb[t]);
                        float2 &a = acc[2 * ig + ip][t];
                        if constexpr (FMT) {
                            a.x = __fadd_rn(a.x, fmt_product(v.x, s.x, *fmt));
                            a.y = __fadd_rn(a.y, fmt_product(v.y, s.y, *fmt));
                        } else if constexpr (SLOW) {
                            // product rounded to fp32 first (infinity on overflow), then added;
                            // the _rn intrinsics are never contracted into an FMA
                            a.x = __fadd_rn(a.x, __fmul_rn(v.x, s.x));
                            a.y = __fadd_rn(a.y, __fmul_rn(v.y, s.y));
                        } else {
                            a = ffma2(v, s, a);
                        }
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------ the kernel
struct Smem {
    uint8_t *lut;
    uint32_t *Uoff;
    float *Uscl;
    uint32_t *Loff;
    float *Lscl;
    RowInfo *rowU, *rowL;
};

__device__ __forceinline__ float4 acc4(const float2 (&acc)[TM / 2][TN], int i, int t0)
{
    return make_float4(accv(acc, i, t0), accv(acc, i, t0 + 1), accv(acc, i, t0 + 2), accv(acc, i, t0 + 3));
}

// Write a finished tile: C = alpha*acc + beta*C with 128-bit stores when the
// output is contiguous along L (or along U, for transposed outputs).  ROWS /
// COLS: the rows and lane columns this warp holds (see compute_stage).
template <int ROWS = TM, int COLS = TN>
__device__ __forceinline__ void store_tile(const ProbParams &q, const float2 (&acc)[TM / 2][TN], int b, int u0,
                                           int l0)
{
    const int nU = q.U.rows, nL = q.L.rows;
    float *C = q.c_ptr + (long long)b * q.c_bs;
    const float alpha = q.alpha, beta = q.beta;
    const bool aligned = (reinterpret_cast<uintptr_t>(C) & 15) == 0;
    const bool vec_l = aligned && q.c_sl == 1 && (q.c_su & 3) == 0;
    const bool vec_u = aligned && q.c_su == 1 && (q.c_sl & 3) == 0;
    if (vec_l && l0 + col_of(COLS - 1) < nL) {
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            const int u = u0 + i;
            if (u >= nU) break;
            if constexpr (COLS == kNarrowTailCols) {
                float2 *dst = reinterpret_cast<float2 *>(C + (long long)u * q.c_su + l0);
                float2 r = make_float2(alpha * accv(acc, i, 0), alpha * accv(acc, i, 1));
                if (beta != 0.0f) {
                    const float2 o = *dst;
                    r.x = fmaf(beta, o.x, r.x); r.y = fmaf(beta, o.y, r.y);
                }
                *dst = r;
            }
#pragma unroll
            for (int t4 = 0; t4 < (COLS == TN ? TN / 4 : 0); ++t4) {
                float4 *dst = reinterpret_cast<float4 *>(C + (long long)u * q.c_su + l0 + kColGroup * t4);
                const float4 a = acc4(acc, i, 4 * t4);
                float4 r = make_float4(alpha * a.x, alpha * a.y, alpha * a.z, alpha * a.w);
                if (beta != 0.0f) {
                    const float4 o = *dst;
                    r.x = fmaf(beta, o.x, r.x); r.y = fmaf(beta, o.y, r.y);
                    r.z = fmaf(beta, o.z, r.z); r.w = fmaf(beta, o.w, r.w);
                }
                *dst = r;
            }
        }
    } else if (vec_u && u0 + ROWS <= nU) {
#pragma unroll
        for (int t = 0; t < COLS; ++t) {
            const int l = l0 + col_of(t);
            if (l >= nL) break;
            float *col = C + (long long)l * q.c_sl + u0;
#pragma unroll
            for (int i4 = 0; i4 < ROWS / 4; ++i4) {
                float4 r = make_float4(alpha * accv(acc, 4 * i4, t), alpha * accv(acc, 4 * i4 + 1, t),
                                       alpha * accv(acc, 4 * i4 + 2, t), alpha * accv(acc, 4 * i4 + 3, t));
                float4 *dst = reinterpret_cast<float4 *>(col + 4 * i4);
                if (beta != 0.0f) {
                    const float4 o = *dst;
                    r.x = fmaf(beta, o.x, r.x); r.y = fmaf(beta, o.y, r.y);
                    r.z = fmaf(beta, o.z, r.z); r.w = fmaf(beta, o.w, r.w);
                }
                *dst = r;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            const int u = u0 + i;
            if (u >= nU) break;
#pragma unroll
            for (int t = 0; t < COLS; ++t) {
                const int l = l0 + col_of(t);
                if (l >= nL) break;
                float *dst = C + (long long)u * q.c_su + (long long)l * q.c_sl;
                float r = alpha * accv(acc, i, t);
                if (beta != 0.0f) r = fmaf(beta, *dst, r);
                *dst = r;
            }
        }
    }
}

// Stages [s0, s1) of tile `tile` of problem q; returns with acc holding the
// partial (or full) sum of those stages.
template <int W, bool GL>
__device__ __forceinline__ void run_stages(const KParams &p, const ProbParams &q, const Smem &sm, int b, int u_tile0,
                                           int l_tile0, int s0, int s1, float2 (&acc)[TM / 2][TN])
{
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = uniform_warp();
    const int wu = warp / WL, wl = warp % WL;
    const int offU = p.M + p.wlog, offL = p.wlog;
    const uint8_t *lut = GL ? static_cast<const uint8_t *>(q.table) : sm.lut;

    Loader<BU, NUE> ldU;
    Loader<BL, NLE> ldL;
    ldU.init(q.U, q.u_kfast, tid, u_tile0, b, s0);
    ldL.init(q.L, q.l_kfast, tid, l_tile0, b, s0);
    ldU.load(q.U, sm.rowU, s0, q.K);
    ldL.load(q.L, sm.rowL, s0, q.K);
    int big = 0;
    if (p.fmt.on) {
        ldU.template store_fmt<UST>(sm.Uoff, sm.Uscl, p.M, offU, p.fmt, p.fmt.off_u);
        ldL.template store_fmt<LST>(sm.Loff, sm.Lscl, p.M, offL, p.fmt, p.fmt.off_l);
    } else {
        ldU.template store<UST>(sm.Uoff, sm.Uscl, p.M, offU, big, uniform_zero_row(p.M, offU));
        ldL.template store<LST>(sm.Loff, sm.Lscl, p.M, offL, big, 0u);
    }
    int slow = __syncthreads_or(big);

    const int urow = wu * TM;
    const int lcol = wl * 32 * TN + lane * 4;
    for (int kt = s0; kt < s1; ++kt) {
        const int buf = (kt - s0) & 1;
        const bool more = kt + 1 < s1;
        if (more) {
            ldU.load(q.U, sm.rowU, kt + 1, q.K);
            ldL.load(q.L, sm.rowL, kt + 1, q.K);
        }
        const uint32_t *Uo = sm.Uoff + buf * BK * UST;
        const float *Us = sm.Uscl + buf * BK * UST;
        const uint32_t *Lo = sm.Loff + buf * BK * LST;
        const float *Ls = sm.Lscl + buf * BK * LST;
        if (p.fmt.on) compute_stage<W, GL, true, UST, LST, true>(acc, Uo, Us, Lo, Ls, lut, urow, lcol, &p.fmt);
        else if (slow) compute_stage<W, GL, true>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
        else compute_stage<W, GL, false>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
        int nbig = 0;
        if (more) {
            const int nb = buf ^ 1;
            if (p.fmt.on) {
                ldU.template store_fmt<UST>(sm.Uoff + nb * BK * UST, sm.Uscl + nb * BK * UST, p.M, offU, p.fmt,
                                            p.fmt.off_u);
                ldL.template store_fmt<LST>(sm.Loff + nb * BK * LST, sm.Lscl + nb * BK * LST, p.M, offL, p.fmt,
                                            p.fmt.off_l);
            } else {
                ldU.template store<UST>(sm.Uoff + nb * BK * UST, sm.Uscl + nb * BK * UST, p.M, offU, nbig,
                                        uniform_zero_row(p.M, offU));
                ldL.template store<LST>(sm.Loff + nb * BK * LST, sm.Lscl + nb * BK * LST, p.M, offL, nbig, 0u);
            }
        }
        slow = __syncthreads_or(nbig);
    }
}

// First launch iteration of stream-K CTA c (c = ctas: the launch's end).
__device__ __forceinline__ long long sk_begin(const KParams &p, int c)
{
    return p.sk_n > 0 ? (long long)p.sk_bound[c] : p.iters * c / p.ctas;
}

__device__ __forceinline__ int n_phases(const KParams &p) { return p.nphase > 1 ? p.nphase : 1; }

// Share boundaries of a phased launch: CTA c takes iterations
// [bound[ph][c], bound[ph][c + 1]) of phase ph, counted from the phase's first
// iteration (computed by the host from a cost model of the phase's tiles).
struct PhaseTable {
    int bound[kMaxPhases][kMaxPhasedCtas + 1];
};

template <int W, bool GL>
__global__ void __launch_bounds__(NT, 1) lutgemm_kernel(const __grid_constant__ KParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int wu = warp / WL, wl = warp % WL;

    const int lut_bytes = GL ? 0 : lut_region_bytes(p.table_bytes);
    Smem sm;
    sm.lut = smem;
    sm.Uoff = reinterpret_cast<uint32_t *>(smem + lut_bytes);
    sm.Uscl = reinterpret_cast<float *>(smem + lut_bytes + kUdecBytes);
    sm.Loff = reinterpret_cast<uint32_t *>(smem + lut_bytes + 2 * kUdecBytes);
    sm.Lscl = reinterpret_cast<float *>(smem + lut_bytes + 2 * kUdecBytes + kLdecBytes);
    sm.rowU = reinterpret_cast<RowInfo *>(smem + lut_bytes + 2 * kUdecBytes + 2 * kLdecBytes);
    sm.rowL = sm.rowU + BU;

    long long it, it_end;
    if (p.streamk) {
        it = sk_begin(p, blockIdx.x);
        it_end = sk_begin(p, blockIdx.x + 1);
    } else {
        // data parallel: CTA x runs the x-th tile of the launch whole
        long long t = blockIdx.x;
        int pi = 0;
        while (pi + 1 < p.nprob && t >= p.pr[pi].tiles) t -= p.pr[pi++].tiles;
        it = p.pr[pi].iter0 + t * p.pr[pi].kt_total;
        it_end = it + p.pr[pi].kt_total;
    }

    const void *staged = nullptr;
    bool first_segment = true;
    while (it < it_end) {
        int pi = 0;
        while (pi + 1 < p.nprob && it >= p.pr[pi + 1].iter0) ++pi;
        const ProbParams &q = p.pr[pi];
        const long long local = it - q.iter0;
        const int S = q.kt_total;
        const long long tile = local / S;
        const int s0 = (int)(local - tile * S);
        const int s1 = (int)min((long long)S, s0 + (it_end - it));
        const int per_batch = q.tiles_u * q.tiles_l;
        const int b = (int)(tile / per_batch);
        const int rem = (int)(tile - (long long)b * per_batch);
        const int u_tile0 = (rem / q.tiles_l) * BU, l_tile0 = (rem % q.tiles_l) * BL;

        if (!first_segment) __syncthreads();      // previous segment done with shared memory
        if constexpr (!GL) {
            if (q.table != staged) {
                // LUT -> shared memory (the device allocation is padded to 256
                // bytes, so whole 16-byte vectors stay inside it)
                const uint4 *src = static_cast<const uint4 *>(q.table);
                uint4 *dst = reinterpret_cast<uint4 *>(sm.lut);
                const int nvec = (p.table_bytes + 15) >> 4;
                for (int i = tid; i < nvec; i += NT) dst[i] = __ldg(src + i);
                staged = q.table;
            }
        }
        if (q.U.gather)
            for (int r = tid; r < BU; r += NT) sm.rowU[r] = row_info(q.U, u_tile0 + r);
        if (q.L.gather)
            for (int r = tid; r < BL; r += NT) sm.rowL[r] = row_info(q.L, l_tile0 + r);
        __syncthreads();

        float2 acc[TM / 2][TN];
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
        run_stages<W, GL>(p, q, sm, b, u_tile0, l_tile0, s0, s1, acc);

        const int u0 = u_tile0 + wu * TM;
        const int l0 = l_tile0 + wl * 32 * TN + lane * 4;
        if (s0 == 0 && s1 == S) {
            store_tile(q, acc, b, u0, l0);
        } else {
            // partial tile: slot 0 holds the CTA's first segment, slot 1 its last
            float *slot = p.ws + ((long long)blockIdx.x * 2 + (first_segment ? 0 : 1)) * (BU * BL);
            const int ur = wu * TM, lr = wl * 32 * TN + lane * 4;
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int t4 = 0; t4 < TN / 4; ++t4)
                    *reinterpret_cast<float4 *>(slot + (ur + i) * BL + lr + kColGroup * t4) = acc4(acc, i, 4 * t4);
        }
        first_segment = false;
        it += s1 - s0;
    }
}

// Adds the partial slots of every tile that stream-K cut between CTAs, in CTA
// order (deterministic), and writes alpha*sum + beta*C.  blockIdx.x = c-1 for
// the boundary before stream-K CTA c (the first boundary inside a tile owns
// it); blockIdx.y = a chunk of kFixupChunk elements of that tile, so every cut
// tile is spread over many CTAs and the partial loads overlap.
constexpr int kFixupChunk = 1024;
template <int kThreads>
__global__ void __launch_bounds__(kThreads) streamk_fixup(const __grid_constant__ KParams p)
{
    static_assert(kThreads * 4 == kFixupChunk, "one float4 per thread");
    const int c = blockIdx.x + 1;                     // boundary before CTA c
    if (c >= p.ctas) return;
    const long long W = p.iters;
    const int G = p.ctas;
    const long long bpos = sk_begin(p, c);
    if (bpos >= W) return;
    int pi = 0;
    while (pi + 1 < p.nprob && bpos >= p.pr[pi + 1].iter0) ++pi;
    const ProbParams &q = p.pr[pi];
    const int S = q.kt_total;
    const long long local = bpos - q.iter0;
    const long long tile = local / S;
    const long long tstart = q.iter0 + tile * S, tend = tstart + S;
    if (bpos == tstart) return;                       // boundary on a tile edge: nothing cut
    if (sk_begin(p, c - 1) > tstart) return;          // an earlier boundary in this tile owns it
    const int c_lo = c - 1;
    int c_hi = c;
    while (c_hi + 1 < G && sk_begin(p, c_hi + 1) < tend) ++c_hi;

    // slot offsets of the contributing CTAs, in CTA order (G <= kMaxFixupParts)
    __shared__ long long slot_off[kMaxFixupParts];
    const int nparts = min(c_hi - c_lo + 1, kMaxFixupParts);
    for (int i = threadIdx.x; i < nparts; i += kThreads) {
        const int cc = c_lo + i;
        const bool first_is_this = sk_begin(p, cc) >= tstart;
        slot_off[i] = ((long long)cc * 2 + (first_is_this ? 0 : 1)) * (BU * BL);
    }
    __syncthreads();

    const int e0 = blockIdx.y * kFixupChunk + threadIdx.x * 4;   // 4 consecutive elements along L
    const int ur = e0 / BL, lr = e0 % BL;
    const float *src = p.ws + e0;
    float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    int i = 0;
    for (; i + 4 <= nparts; i += 4) {          // loads first, adds in CTA order
        const float4 a = *reinterpret_cast<const float4 *>(src + slot_off[i]);
        const float4 b = *reinterpret_cast<const float4 *>(src + slot_off[i + 1]);
        const float4 cv = *reinterpret_cast<const float4 *>(src + slot_off[i + 2]);
        const float4 d = *reinterpret_cast<const float4 *>(src + slot_off[i + 3]);
        sum.x += a.x; sum.y += a.y; sum.z += a.z; sum.w += a.w;
        sum.x += b.x; sum.y += b.y; sum.z += b.z; sum.w += b.w;
        sum.x += cv.x; sum.y += cv.y; sum.z += cv.z; sum.w += cv.w;
        sum.x += d.x; sum.y += d.y; sum.z += d.z; sum.w += d.w;
    }
    for (; i < nparts; ++i) {
        const float4 a = *reinterpret_cast<const float4 *>(src + slot_off[i]);
        sum.x += a.x; sum.y += a.y; sum.z += a.z; sum.w += a.w;
    }

    const int per_batch = q.tiles_u * q.tiles_l;
    const int b = (int)(tile / per_batch);
    const int rem = (int)(tile - (long long)b * per_batch);
    const int u = (rem / q.tiles_l) * BU + ur;
    const int l = (rem % q.tiles_l) * BL + lr;
    if (u >= q.U.rows) return;
    float *C = q.c_ptr + (long long)b * q.c_bs;
    const float v[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        if (l + t >= q.L.rows) break;
        float *dst = C + (long long)u * q.c_su + (long long)(l + t) * q.c_sl;
        float r = q.alpha * v[t];
        if (q.beta != 0.0f) r = fmaf(q.beta, *dst, r);
        *dst = r;
    }
}

}  // namespace AMSIM_KNS
}  // namespace amsim

namespace amsim {
namespace AMSIM_KNS {

// Host-side launcher for one instance; sets the dynamic shared-memory limit
// once per device.
template <int W, bool GL>
int launch_instance(const KParams &p, dim3 grid, size_t smem, cudaStream_t st)
{
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AMSIM_ECUDA;
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(lutgemm_kernel<W, GL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kMaxSmemPerCta);
        if (e != cudaSuccess) return cuda_status(e);
        attr_done[dev] = true;
    }
    lutgemm_kernel<W, GL><<<grid, NT, smem, st>>>(p);
    const int rc = cuda_status(cudaGetLastError());
    if (rc == AMSIM_OK) count_launch();
    return rc;
}

int launch_fixup(const KParams &p, int boundaries, cudaStream_t st);
int launch_w8(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);
int launch_w16(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);
int launch_w32(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);

}  // namespace AMSIM_KNS
}  // namespace amsim
