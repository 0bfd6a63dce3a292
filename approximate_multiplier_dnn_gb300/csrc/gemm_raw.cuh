// LUT-GEMM fed with raw operand tiles by the Tensor Memory Accelerator and
// decoded in shared memory (ApproxTrain Sec. V-B Algorithm 2 per product,
// Sec. VI-D GEMM kernel).
//
// One producer thread copies each stage's fp32 tiles -- BU (or BL) rows x BK
// reduction steps of each operand, straight from the caller's tensors -- as
// tensor boxes into a raw ring.  Unit-stride convolutions read their im2col
// tiles the same way: a box of 16 channels of the NHWC activation at the
// stage's filter tap covers whole output rows (the tap's row and column
// offsets are box coordinates; out-of-range pixels arrive as zeros), and the
// filter gradient's tile is four boxes of 64 channels.  The producer warpgroup (128 threads) then
// decodes a landed stage into (LUT byte offset, scale) [k][row] arrays, which
// the eight consumer warps use exactly as in the predecoded kernel.  Operands
// stored k-fast arrive [row][k] with the copy engine's 64-byte swizzle, so the
// decoders' transposing reads are free of bank conflicts.  No operand planes
// and no separate decode launch are needed; each CTA decodes its own tiles.
//
// A tile whose real lane columns all fit in its first 128 (or 64) is
// computed in a tail layout (kTailLayout: every consumer warp on 8 rows), and
// its decoders skip the columns that layout never reads; the host cuts an
// ordinary launch's stream-K shares by each tile's stage cost.  Phased
// launches keep the regular layout.
//
// Barriers: raw_full (copy bytes), raw_empty (decoders done with a raw slot),
// full (decoded stage ready), empty (consumers done).  Every wait is bounded
// by the global timer; copies still in flight at an abort are waited for.
#pragma once

#include "gemm_tma.cuh"

#ifdef AMSIM_WIDE_TILES
#error "the raw-tile kernel is built with the narrow tile shape only"
#endif

namespace amsim {
namespace kern {

constexpr int kRawDecoders = 128;                       // the producer warpgroup
constexpr int kRawThreads = kTmaConsumerThreads + kRawDecoders;
static_assert(kRawThreads == kTmaThreads, "same block shape as the predecoded kernel");
// Register split of the decoder warpgroup and the consumers: the decoders'
// dispatch over full and tail-tile decodes spilled at 56 registers.
constexpr int kRawProducerRegs = 72;
constexpr int kRawConsumerRegs =
    ((kRawThreads * kTmaLaunchRegs - kRawDecoders * kRawProducerRegs) / kTmaConsumerThreads) & ~7;
static_assert(kRawConsumerRegs <= 256 &&
                  kTmaConsumerThreads * kRawConsumerRegs + kRawDecoders * kRawProducerRegs <= kRawThreads * kTmaLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kRawUBytes = BU * BK * 4;                 // raw fp32 tile of U
constexpr int kRawLBytes = BL * BK * 4;
constexpr int kRawStageBytes = kRawUBytes + kRawLBytes; // 20 KB
constexpr int kRawRing = 3;                             // raw stages
constexpr int kRawDec = 3;                              // decoded stages
constexpr int kRawBarBytes = 256;                       // barriers and big-operand flags
static_assert(kRawUBytes % 1024 == 0 && kRawLBytes % 1024 == 0, "swizzled boxes start 1024-byte aligned");
static_assert(BL % 64 == 0 && (BL / 64) * BK * 64 * 4 == kRawLBytes, "blocked L boxes fill the L stage");
static_assert((2 * kRawRing + 2 * kRawDec + 2) * 8 + (kRawDec * (kRawDecoders / 32) + 1) * 4 <= kRawBarBytes,
              "barrier block");
static_assert(kRawDec * kTmaStageBytes + kRawRing * kRawStageBytes >= (BU * BL + 1024 * 4) * 4,
              "the rings hold the stream-K reduction buffer");

__host__ __device__ constexpr int raw_lut_region(int lut_bytes) { return (lut_bytes + 1023) & ~1023; }

// Shared memory of the raw-tile kernel beside a LUT of lut_bytes (1 KB for alignment).
__host__ __device__ constexpr int raw_smem_bytes(int lut_bytes)
{
    return 1024 + raw_lut_region(lut_bytes) + kRawDec * kTmaStageBytes + kRawRing * kRawStageBytes + kRawBarBytes;
}

// Box (x, y, z) of a 3-D tensor map into shared memory; completes on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// What a decoder thread saw in a stage that the fast stage computations must
// not see: the table decode's flag (|x| >= 2^64, infinities, NaN), and for
// closed forms the largest magnitude and the smallest nonzero magnitude
// (minus one) as bit patterns.  Closed forms send to the slow computation the
// values the table's does (magnitudes of 2^64 and up, infinities, NaN) and
// nonzero magnitudes below 2^-63, whose products with each other can fall
// below the smallest normal, where the table path's scale product flushes them.
struct StageFlags {
    int big = 0;
    int small = 0;          // table decode: an element that blocks the folded form (see bits())
    uint32_t amax = 0u, aminm1 = 0xFFFFFFFFu;
    __device__ __forceinline__ int any() const
    {
        return big | (amax >= 0x5F800000u) | (aminm1 < 0x1FFFFFFFu);
    }
    // bit 0: the stage takes the rounding slow products; bit 1: it may not
    // fold the uniform scale into the entry -- an operand below 2^-63 but not
    // zero (zero uniform operands take the table's zero row and zero lane
    // operands a zero scale: both give the exact signed zero product folded)
    __device__ __forceinline__ int bits() const { return (any() ? 1 : 0) | (small ? 2 : 0); }
};

// v * 1 with denormals flushed to signed zero (NaN stays NaN with its
// fraction's top bit set).
__device__ __forceinline__ uint32_t ftz_bits(float v)
{
    float r;
    asm("mul.rn.ftz.f32 %0, %1, 0f3F800000;" : "=f"(r) : "f"(v));
    return __float_as_uint(r);
}

// Closed-form operand decode (no table): without FRAC, off is the operand
// truncated to the M fraction bits keep masks, sign and exponent kept and
// denormals as signed zero (no scale is stored: the slow computation takes it
// from off); with FRAC, off is that truncated fraction field alone and s the
// signed power-of-two scale.
template <bool FRAC>
__device__ __forceinline__ void decode_alu(float v, uint32_t keep, uint32_t &off, float &s, StageFlags &fl)
{
    const uint32_t y = ftz_bits(v);
    const uint32_t ax = y & 0x7FFFFFFFu;
    fl.amax = max(fl.amax, ax);
    fl.aminm1 = min(fl.aminm1, ax - 1u);
    if constexpr (FRAC) {
        off = y & keep;
        s = __uint_as_float(y & 0xFF800000u);
    } else {
        off = y & (0xFF800000u | keep);
    }
}

// Decode mode DM: 0 the table's (offset, scale), 3 the same packed into one
// word (pack_operand; tables in shared memory, whose offsets stay below
// 2^18), 1 the closed-form truncated value (no scale), 2 the closed-form
// truncated fraction and scale; aux is the table offset's shift (DM 0, 3) or
// the mask of the kept fraction bits.  Modes 1 and 3 store no scale array.
template <int DM, bool LANE = false>
__device__ __forceinline__ void decode_as(float v, int M, uint32_t aux, uint32_t &off, float &s, StageFlags &fl)
{
    if constexpr (DM == 0 || DM == 3) {
        decode(v, M, (int)aux, off, s, fl.big, LANE ? 0u : uniform_zero_row(M, (int)aux));
        fl.small |= is_small_nonzero(v);
        if constexpr (DM == 3) off = pack_operand(off, s);
    } else {
        decode_alu<DM == 2>(v, aux, off, s, fl);
    }
}

// Decode a raw R-row tile into off/scl [BK][R].  k-fast tiles are [R][BK]
// fp32 rows of 64 bytes whose 16-byte chunks the copy engine swizzled as
// chunk ^ ((row >> 1) & 3); row-fast tiles are [BK][R].  Only rows 0 .. NR - 1
// are decoded (a tail tile's consumers read no others).
template <int R, int DM, bool LANE = false, int NR = R>
__device__ __forceinline__ void raw_decode(const uint8_t *raw, bool kfast, uint32_t *off, float *scl, int M,
                                           uint32_t aux, int d, StageFlags &fl)
{
    static_assert(NR <= R && NR % 4 == 0, "decoded rows");
    if (kfast) {
#pragma unroll 2
        for (int task = d; task < NR * (BK / 4); task += kRawDecoders) {
            const int r = task % NR, c = task / NR;
            const float4 v = *reinterpret_cast<const float4 *>(raw + r * (BK * 4) + ((c ^ ((r >> 1) & 3)) << 4));
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t o;
                float s;
                decode_as<DM, LANE>(e[i], M, aux, o, s, fl);
                off[(4 * c + i) * R + r] = o;
                if constexpr (DM != 1 && DM != 3) scl[(4 * c + i) * R + r] = s;
            }
        }
    } else {
#pragma unroll 2
        for (int task = d; task < BK * (NR / 4); task += kRawDecoders) {
            const int k = task / (NR / 4), r4 = (task % (NR / 4)) * 4;
            const float4 v = *reinterpret_cast<const float4 *>(raw + (k * R + r4) * 4);
            uint4 o;
            float4 s;
            decode_as<DM, LANE>(v.x, M, aux, o.x, s.x, fl);
            decode_as<DM, LANE>(v.y, M, aux, o.y, s.y, fl);
            decode_as<DM, LANE>(v.z, M, aux, o.z, s.z, fl);
            decode_as<DM, LANE>(v.w, M, aux, o.w, s.w, fl);
            *reinterpret_cast<uint4 *>(off + k * R + r4) = o;
            if constexpr (DM != 1 && DM != 3) *reinterpret_cast<float4 *>(scl + k * R + r4) = s;
        }
    }
}

// Decode four row-fast 64-row blocks ([BK][64] each, the filter gradient's
// L tile) into columns 64 b .. 64 b + 63 of off/scl [BK][BL]; only the first
// NB blocks (a tail tile's consumers read no others).
template <int DM, int NB = BL / 64>
__device__ __forceinline__ void raw_decode_blocks(const uint8_t *raw, uint32_t *off, float *scl, int M,
                                                  uint32_t aux, int d, StageFlags &fl)
{
#pragma unroll 2
    for (int task = d; task < NB * BK * 16; task += kRawDecoders) {
        const int b = task / (BK * 16), rem = task % (BK * 16);
        const int k = rem / 16, r4 = (rem % 16) * 4;
        const float4 v = *reinterpret_cast<const float4 *>(raw + ((b * BK + k) * 64 + r4) * 4);
        uint4 o;
        float4 s;
        decode_as<DM, true>(v.x, M, aux, o.x, s.x, fl);
        decode_as<DM, true>(v.y, M, aux, o.y, s.y, fl);
        decode_as<DM, true>(v.z, M, aux, o.z, s.z, fl);
        decode_as<DM, true>(v.w, M, aux, o.w, s.w, fl);
        *reinterpret_cast<uint4 *>(off + k * BL + 64 * b + r4) = o;
        if constexpr (DM != 1 && DM != 3) *reinterpret_cast<float4 *>(scl + k * BL + 64 * b + r4) = s;
    }
}

// Convolution boxes of stage kt (see ConvRaw): U from the filter or dy, L from
// the activation at the stage's filter tap.
__device__ __forceinline__ void conv_raw_boxes(const KParams &p, const TmaMaps &maps, const ProbParams &q,
                                               int u_tile0, int l_tile0, int kt, uint8_t *st, uint64_t *bar)
{
    const int k0 = kt * BK;
    if (p.cv_u_tap) {
        const int rs = k0 / p.cv_ch;
        tma_load_3d(st, &maps.u[0], k0 - rs * p.cv_ch, u_tile0, rs, bar);
    } else if (q.u_kfast) {
        tma_load_3d(st, &maps.u[0], k0, u_tile0, 0, bar);
    } else {
        tma_load_3d(st, &maps.u[0], u_tile0, k0, 0, bar);
    }
    uint8_t *dl = st + kRawUBytes;
    if (p.conv == 1) {
        // whole output rows y0 .. of image n; channels ch0 .. ch0 + 15 of tap (r, s)
        const int t = l_tile0 / BL;
        const int n = t / p.cv_tiles_img, y0 = (t - n * p.cv_tiles_img) * p.cv_rows_tile;
        const int rs = k0 / p.cv_ch, ch0 = k0 - rs * p.cv_ch;
        const int r = rs / p.cv_S, s = rs - r * p.cv_S;
        tma_load_4d(dl, &maps.l[0], ch0, p.cv_xbase + s * p.cv_xstep, y0 + p.cv_ybase + r * p.cv_ystep, n, bar);
    } else {
        // 16 output pixels (n, pp, q0 ..) of one row; four blocks of 64 rows
        // (tap, channel), each 64 channels at the tap's input position; rows
        // past the end get a box wholly outside the tensor (zeros), so every
        // stage carries the same bytes
        const int pq = p.cv_P * p.cv_Q;
        const int n = k0 / pq, rem = k0 - n * pq;
        const int pp = rem / p.cv_Q, q0 = rem - pp * p.cv_Q;
#pragma unroll
        for (int blk = 0; blk < BL / 64; ++blk) {
            const int row = l_tile0 + 64 * blk;
            int c0 = 0, h = 0, w = 0, nn = p.cv_N;
            if (row < p.cv_rows) {
                const int rs = row / p.cv_ch;
                const int r = rs / p.cv_S, s = rs - r * p.cv_S;
                c0 = row - rs * p.cv_ch;
                h = pp + p.cv_ybase + r * p.cv_ystep;
                w = q0 + p.cv_xbase + s * p.cv_xstep;
                nn = n;
            }
            tma_load_4d(dl + blk * (BK * 64 * 4), &maps.l[0], c0, w, h, nn, bar);
        }
    }
}

// Decode an R-row tile of an operand read with plain loads (rows row0 ..,
// steps k0 .., batch b; zeros outside the operand) into off/scl [BK][R].
// Lanes walk the operand's unit-stride dimension when it has one.
// Operands whose strides the copy engine cannot take (a leading dimension that
// is not a multiple of 4 elements, or a base address off a 16-byte boundary)
// are read with plain loads.  Only the tile's in-range elements are loaded,
// spread over all decoders so that each issues as few dependent loads as
// possible; the rest of the tile is the decode of zero.
struct DirectTile {
    const float *base;
    long long sr, sk;         // element strides of rows and steps
    int vr, vk;               // in-range rows and steps of the tile
    bool rows_fast;           // consecutive tasks walk rows (unit row stride, or neither stride unit)
};

__device__ __forceinline__ DirectTile direct_tile(const OperandDesc &od, int K, int b, int bsel, int row0, int k0,
                                                  int R)
{
    DirectTile t;
    t.sr = od.s_row;
    t.sk = od.s_k;
    t.base = od.ptr + (long long)b * bsel * od.batch_stride + (long long)row0 * t.sr + (long long)k0 * t.sk;
    t.vr = max(0, min(R, od.rows - row0));
    t.vk = max(0, min(BK, K - k0));
    t.rows_fast = od.s_row == 1 || od.s_k != 1;
    return t;
}

__device__ __forceinline__ void direct_task(const DirectTile &t, int task, int &rr, int &kk)
{
    if (t.rows_fast) {
        kk = task / t.vr;
        rr = task - kk * t.vr;
    } else {
        rr = task / t.vk;
        kk = task - rr * t.vk;
    }
}

// Pull a later stage's in-range elements toward L2 (no destination, no wait).
template <int R>
__device__ __forceinline__ void direct_prefetch(const OperandDesc &od, int K, int b, int bsel, int row0, int k0, int d)
{
    const DirectTile t = direct_tile(od, K, b, bsel, row0, k0, R);
    const int n = t.vr * t.vk;
#pragma unroll 1
    for (int task = d; task < n; task += kRawDecoders) {
        int rr, kk;
        direct_task(t, task, rr, kk);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(t.base + rr * t.sr + kk * t.sk));
    }
}

// Copy a tile of a plainly-read operand into its raw slot with asynchronous
// 4-byte copies (every copy of the tile in flight at once; zero-filled out of
// range), in the layout a tensor copy would have produced: [k][row] for an
// operand with unit row stride, otherwise the swizzled [row][k] boxes.  The
// caller waits for the copies and syncs the decoders before decoding.
template <int R>
__device__ __forceinline__ void direct_copy(const OperandDesc &od, int K, int b, int bsel, int row0, int k0,
                                            uint8_t *raw, int d)
{
    const DirectTile t = direct_tile(od, K, b, bsel, row0, k0, R);
    float *dst = reinterpret_cast<float *>(raw);
    if (od.s_row == 1) {
#pragma unroll 1
        for (int task = d; task < R * BK; task += kRawDecoders) {
            const int rr = task % R, kk = task / R;
            const bool ok = rr < t.vr && kk < t.vk;
            cp_async4(dst + kk * R + rr, ok ? t.base + rr + kk * t.sk : od.ptr, ok);
        }
    } else {
#pragma unroll 1
        for (int task = d; task < R * BK; task += kRawDecoders) {
            const int kk = task % BK, rr = task / BK;
            const bool ok = rr < t.vr && kk < t.vk;
            float *e = reinterpret_cast<float *>(raw + rr * (BK * 4) + ((((kk >> 2) ^ ((rr >> 1) & 3))) << 4)) + (kk & 3);
            cp_async4(e, ok ? t.base + rr * t.sr + kk * t.sk : od.ptr, ok);
        }
    }
}

__device__ __forceinline__ void decoder_bar() { asm volatile("bar.sync 3, %0;" ::"n"(kRawDecoders) : "memory"); }

struct RawSmem {
    uint8_t *dec;          // kRawDec decoded stages of kTmaStageBytes
    uint8_t *raw;          // kRawRing raw stages of kRawStageBytes
    uint64_t *raw_full, *raw_empty, *full, *empty;
    int *flags;            // [kRawDec][decoder warps]: the stage needs the slow computation (StageFlags)
};

// Signed power-of-two scale of a truncated value (sign | exponent | fraction
// bits): zero for a zero, infinity for an infinity, NaN for a NaN.
__device__ __forceinline__ float trunc_scale(uint32_t t)
{
    return __uint_as_float((t & 0x7FFFFFFFu) > 0x7F800000u ? 0x7FC00000u : (t & 0xFF800000u));
}

// One decoded stage with closed-form products (KIND 1 Mitchell, 2 exact),
// same accumulator layout and summation order as compute_stage, so that the
// sums equal the table path's bit for bit.  Uo holds truncated values
// (sign | exponent | M fraction bits), Lo truncated values (exact) or
// fractions in place (Mitchell).
//  - Fast stages (every nonzero operand in [2^-63, 2^64)): Mitchell's product
//    is the float whose bits are a's truncated value plus b's fraction --
//    a's scale times Mitchell's factor, the fraction carry landing in the
//    exponent exactly when the 2 (x + y) branch applies -- times b's scale;
//    a zero a gives a denormal, which the multiply flushes to a signed zero.
//    The exact product is the fp32 FMA of the two truncated values.  Each
//    is exact and normal (exponent sum >= 1), as the table path's v * s is.
//  - Other stages rebuild the table path's (v, s) and round the product
//    before adding it, as compute_stage's slow stages do.
template <int KIND, bool SLOW, int ROWS = TM, int COLS = TN>
__device__ __forceinline__ void compute_stage_alu(float2 (&acc)[TM / 2][TN], const uint32_t *__restrict__ Uo,
                                                  const float *__restrict__ Us, const uint32_t *__restrict__ Lo,
                                                  const float *__restrict__ Ls, int urow, int lcol)
{
#pragma unroll(kKkUnroll)
    for (int kk = 0; kk < BK; ++kk) {
        uint32_t lo[TN];
        float2 sb[TN];
        if constexpr (COLS == kNarrowTailCols) {
            const uint2 o = *reinterpret_cast<const uint2 *>(Lo + kk * BL + lcol);
            lo[0] = o.x; lo[1] = o.y;
            if constexpr (KIND == 1) {
                const float2 sc = *reinterpret_cast<const float2 *>(Ls + kk * BL + lcol);
                sb[0] = make_float2(sc.x, sc.x);
                sb[1] = make_float2(sc.y, sc.y);
            }
            if constexpr (SLOW) {
#pragma unroll
                for (int t = 0; t < COLS; ++t) {
                    const float b = KIND == 1 ? trunc_scale(__float_as_uint(sb[t].x) | lo[t]) : trunc_scale(lo[t]);
                    sb[t] = make_float2(b, b);
                }
            }
        }
#pragma unroll
        for (int t4 = 0; t4 < (COLS == TN ? TN / 4 : 0); ++t4) {
            const uint4 o = *reinterpret_cast<const uint4 *>(Lo + kk * BL + lcol + kColGroup * t4);
            lo[4 * t4 + 0] = o.x; lo[4 * t4 + 1] = o.y; lo[4 * t4 + 2] = o.z; lo[4 * t4 + 3] = o.w;
            if constexpr (KIND == 1) {
                const float4 sc = *reinterpret_cast<const float4 *>(Ls + kk * BL + lcol + kColGroup * t4);
                sb[4 * t4 + 0] = make_float2(sc.x, sc.x);
                sb[4 * t4 + 1] = make_float2(sc.y, sc.y);
                sb[4 * t4 + 2] = make_float2(sc.z, sc.z);
                sb[4 * t4 + 3] = make_float2(sc.w, sc.w);
            }
            if constexpr (SLOW) {
                // the scales, NaN included, from the truncated values (Mitchell's
                // L scale and fraction together make one)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = 4 * t4 + i;
                    const float b = KIND == 1 ? trunc_scale(__float_as_uint(sb[t].x) | lo[t]) : trunc_scale(lo[t]);
                    sb[t] = make_float2(b, b);
                }
            }
        }
#pragma unroll
        for (int ig = 0; ig < ROWS / 4; ++ig) {
            const uint4 uo = *reinterpret_cast<const uint4 *>(Uo + kk * BU + urow + 4 * ig);
            const uint32_t uov[4] = {uo.x, uo.y, uo.z, uo.w};
            float2 sa[2];
            if constexpr (SLOW) {
                sa[0] = make_float2(trunc_scale(uo.x), trunc_scale(uo.y));
                sa[1] = make_float2(trunc_scale(uo.z), trunc_scale(uo.w));
            }
#pragma unroll
            for (int ip = 0; ip < 2; ++ip) {
#pragma unroll
                for (int t = 0; t < COLS; ++t) {
                    float2 &a = acc[2 * ig + ip][t];
                    const uint32_t u0 = uov[2 * ip], u1 = uov[2 * ip + 1];
                    if constexpr (SLOW) {
                        float2 v;
                        if constexpr (KIND == 1) {
                            v = make_float2(__uint_as_float(0x3F800000u + (u0 & 0x7FFFFFu) + lo[t]),
                                            __uint_as_float(0x3F800000u + (u1 & 0x7FFFFFu) + lo[t]));
                        } else {
                            const float vb = __uint_as_float(0x3F800000u | (lo[t] & 0x7FFFFFu));
                            v = make_float2(__fmul_rn(__uint_as_float(0x3F800000u | (u0 & 0x7FFFFFu)), vb),
                                            __fmul_rn(__uint_as_float(0x3F800000u | (u1 & 0x7FFFFFu)), vb));
                        }
                        const float2 s = fmul2_ftz(sa[ip], sb[t]);
                        a.x = __fadd_rn(a.x, __fmul_rn(v.x, s.x));
                        a.y = __fadd_rn(a.y, __fmul_rn(v.y, s.y));
                    } else if constexpr (KIND == 1) {
                        const float2 w = make_float2(__uint_as_float(u0 + lo[t]), __uint_as_float(u1 + lo[t]));
                        a = fadd2(a, fmul2_ftz(w, sb[t]));
                    } else {
                        const float b = __uint_as_float(lo[t]);
                        a = ffma2(make_float2(__uint_as_float(u0), __uint_as_float(u1)), make_float2(b, b), a);
                    }
                }
            }
        }
    }
}

// A decoded stage of the raw-tile kernel: table entries (W = 8, 16, 32; packed
// operand words with the table in shared memory) or closed forms (W = 1
// Mitchell, 2 exact), over this warp's ROWS uniform rows and each lane's
// COLS columns.
template <int W, bool GL, bool SLOW, bool FOLD = false, int ROWS = TM, int COLS = TN>
__device__ __forceinline__ void raw_stage(float2 (&acc)[TM / 2][TN], const uint32_t *Uo, const float *Us,
                                          const uint32_t *Lo, const float *Ls, const uint8_t *lut, int urow,
                                          int lcol)
{
    if constexpr (W <= 2) compute_stage_alu<W, SLOW, ROWS, COLS>(acc, Uo, Us, Lo, Ls, urow, lcol);
    else compute_stage<W, GL, SLOW, BU, BL, false, FOLD, !GL, !GL, ROWS, COLS>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
}

// One stage of a consumer: the rounding slow products when a decoder flagged
// bit 0, the folded-scale form when no decoder flagged bit 1 (tables in
// shared memory only), else the general form.
template <int W, bool GL, int ROWS = TM, int COLS = TN>
__device__ __forceinline__ void raw_stage_by_flags(int fl, float2 (&acc)[TM / 2][TN], const uint32_t *Uo,
                                                   const float *Us, const uint32_t *Lo, const float *Ls,
                                                   const uint8_t *lut, int urow, int lcol)
{
    if (fl & 1) raw_stage<W, GL, true, false, ROWS, COLS>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
    else if (W > 2 && !GL && !(fl & 2))
        raw_stage<W, GL, false, (W > 2 && !GL), ROWS, COLS>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
    else raw_stage<W, GL, false, false, ROWS, COLS>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
}

// This warp's rows, lane columns and column block of a tile in the regular
// layout (ROWS = TM, COLS = TN) or a tail layout (ROWS = kTailRows; COLS = TN,
// or kNarrowTailCols adjacent columns per lane).
template <int ROWS, int COLS>
__device__ __forceinline__ void warp_span(int warp, int lane, int &urow, int &lcol, int &lblock)
{
    if constexpr (ROWS == TM) {
        urow = (warp / WL) * TM;
        lblock = (warp % WL) * 32 * TN;
        lcol = lblock + lane * 4;
    } else {
        urow = warp * ROWS;
        lblock = 0;
        lcol = lane * (COLS == TN ? 4 : COLS);
    }
}

// The producer warpgroup: thread 0 also issues the copies, kRawRing - 1 stages
// ahead.  ALU: 0 table offsets, 1 / 2 Mitchell's / the exact closed form.
// PK: table offsets and scales packed into one word (table in shared memory).
template <int ALU, bool PK>
__device__ __forceinline__ void raw_producer(const KParams &p, const TmaMaps &maps, const RawSmem &sm)
{
    const int d = threadIdx.x - kTmaConsumerThreads;
    const int lane = d & 31, dw = d >> 5;
    // decode modes and their shift / fraction mask (closed forms: U keeps its
    // sign and exponent; L keeps them for the exact product, not for Mitchell's)
    constexpr int DT = PK ? 3 : 0;
    constexpr int DU = ALU ? 1 : DT, DL = ALU == 1 ? 2 : ALU ? 1 : DT;
    const uint32_t keep = ((1u << p.M) - 1u) << (23 - p.M);
    const uint32_t offU = ALU ? keep : (uint32_t)(p.M + p.wlog), offL = ALU ? keep : (uint32_t)p.wlog;
    long long it0, it1;
    cta_range(p, it0, it1);
    bool aborted = false;
    long long issued = 0;
    auto issue = [&](long long it) {
        const long long g = it - it0;
        const int rs = (int)(g % kRawRing);
        if (!mbar_wait(&sm.raw_empty[rs], (uint32_t)(((g / kRawRing) & 1) ^ 1), aborted)) return;
        const StagePos sp = stage_pos(p, it);
        const ProbParams &q = p.pr[sp.pi];
        uint8_t *st = sm.raw + (size_t)rs * kRawStageBytes;
        const int k0 = sp.kt * BK;
        if (p.conv) {
            mbar_expect_tx(&sm.raw_full[rs], kRawStageBytes);
            conv_raw_boxes(p, maps, q, sp.u_tile0, sp.l_tile0, sp.kt, st, &sm.raw_full[rs]);
        } else {
            // operands read with plain loads contribute no copy bytes (an all-plain
            // stage is a bare arrival)
            const uint32_t bytes = (q.u_direct ? 0 : kRawUBytes) + (q.l_direct ? 0 : kRawLBytes);
            if (bytes) mbar_expect_tx(&sm.raw_full[rs], bytes);
            else mbar_arrive(&sm.raw_full[rs]);
            if (q.u_direct) {
            } else if (q.u_kfast) {
                tma_load_3d(st, &maps.u[sp.pi], k0, sp.u_tile0, sp.b * q.u_bsel, &sm.raw_full[rs]);
            } else {
                tma_load_3d(st, &maps.u[sp.pi], sp.u_tile0, k0, sp.b * q.u_bsel, &sm.raw_full[rs]);
            }
            if (q.l_direct) {
            } else if (q.l_kfast) {
                tma_load_3d(st + kRawUBytes, &maps.l[sp.pi], k0, sp.l_tile0, sp.b * q.l_bsel, &sm.raw_full[rs]);
            } else {
                tma_load_3d(st + kRawUBytes, &maps.l[sp.pi], sp.l_tile0, k0, sp.b * q.l_bsel, &sm.raw_full[rs]);
            }
        }
        ++issued;
    };
    if (d == 0)
        for (long long it = it0; it < it1 && it < it0 + kRawRing - 1; ++it) issue(it);
    for (long long it = it0; it < it1; ++it) {
        const long long g = it - it0;
        if (d == 0 && it + kRawRing - 1 < it1 && !aborted) issue(it + kRawRing - 1);
        const int rs = (int)(g % kRawRing), ds = (int)(g % kRawDec);
        mbar_wait(&sm.raw_full[rs], (uint32_t)((g / kRawRing) & 1), aborted);
        mbar_wait(&sm.empty[ds], (uint32_t)(((g / kRawDec) & 1) ^ 1), aborted);
        const StagePos sp = stage_pos(p, it);
        const ProbParams &q = p.pr[sp.pi];
        const uint8_t *raw = sm.raw + (size_t)rs * kRawStageBytes;
        uint8_t *st = sm.dec + (size_t)ds * kTmaStageBytes;
        StageFlags big;
        if (q.u_direct || q.l_direct) {
            uint8_t *rw = sm.raw + (size_t)rs * kRawStageBytes;
            if (q.u_direct) direct_copy<BU>(q.U, q.K, sp.b, q.u_bsel, sp.u_tile0, sp.kt * BK, rw, d);
            if (q.l_direct) direct_copy<BL>(q.L, q.K, sp.b, q.l_bsel, sp.l_tile0, sp.kt * BK, rw + kRawUBytes, d);
            cp_async_commit();
            cp_async_wait<0>();
            decoder_bar();          // every decoder's copies have landed
        }
        raw_decode<BU, DU>(raw, q.u_kfast, reinterpret_cast<uint32_t *>(st),
                       reinterpret_cast<float *>(st + BK * BU * 4), p.M, offU, d, big);
        // the L columns the tile's consumers read: all, or those of a tail layout
        const int lcols = narrow_tail_tile(sp.l_tile0, q.L.rows) ? 32 * kNarrowTailCols
                          : tail_tile(sp.l_tile0, q.L.rows)      ? 32 * TN
                                                                 : BL;
        uint32_t *lo = reinterpret_cast<uint32_t *>(st + kTmaUBytes);
        float *ls = reinterpret_cast<float *>(st + kTmaUBytes + BK * BL * 4);
        if (p.conv == 2) {
            if (lcols == 32 * kNarrowTailCols)
                raw_decode_blocks<DL, 32 * kNarrowTailCols / 64>(raw + kRawUBytes, lo, ls, p.M, offL, d, big);
            else if (lcols == 32 * TN)
                raw_decode_blocks<DL, 32 * TN / 64>(raw + kRawUBytes, lo, ls, p.M, offL, d, big);
            else
                raw_decode_blocks<DL>(raw + kRawUBytes, lo, ls, p.M, offL, d, big);
        } else {
            if (lcols == 32 * kNarrowTailCols)
                raw_decode<BL, DL, true, 32 * kNarrowTailCols>(raw + kRawUBytes, q.l_kfast, lo, ls, p.M, offL, d,
                                                               big);
            else if (lcols == 32 * TN)
                raw_decode<BL, DL, true, 32 * TN>(raw + kRawUBytes, q.l_kfast, lo, ls, p.M, offL, d, big);
            else
                raw_decode<BL, DL, true>(raw + kRawUBytes, q.l_kfast, lo, ls, p.M, offL, d, big);
        }
        mbar_arrive(&sm.raw_empty[rs]);
        const int any = __reduce_or_sync(0xFFFFFFFFu, big.bits());
        if (lane == 0) sm.flags[ds * (kRawDecoders / 32) + dw] = any;
        mbar_arrive(&sm.full[ds]);
        if (p.direct && it + kRawRing < it1) {
            const StagePos np = stage_pos(p, it + kRawRing);
            const ProbParams &nq = p.pr[np.pi];
            if (nq.u_direct) direct_prefetch<BU>(nq.U, nq.K, np.b, nq.u_bsel, np.u_tile0, np.kt * BK, d);
            if (nq.l_direct) direct_prefetch<BL>(nq.L, nq.K, np.b, nq.l_bsel, np.l_tile0, np.kt * BK, d);
        }
    }
    if (d == 0 && aborted) {
        // copies issued into raw slots nobody waited for may still be landing
        bool gave_up = false;
        const long long n = issued < kRawRing ? issued : kRawRing;
        for (long long j = issued - n; j < issued; ++j)
            mbar_wait(&sm.raw_full[j % kRawRing], (uint32_t)((j / kRawRing) & 1), gave_up);
    }
}

// Stages [s0, s1) of one segment of a tile for one consumer warp in the
// layout ROWS (TM, or kTailRows for a tail tile); `g` counts decoded stages.
template <int W, bool GL, int ROWS, int COLS>
__device__ __forceinline__ void raw_segment(const KParams &p, const ProbParams &q, const uint8_t *lut,
                                            const RawSmem &sm, int b, int u_tile0, int l_tile0, int s0, int s1,
                                            bool first, uint32_t &g, bool &aborted, CutTile &cut0, CutTile &cut1,
                                            int &ncut)
{
    int urow, lcol, lblock;
    warp_span<ROWS, COLS>(uniform_warp(), threadIdx.x & 31, urow, lcol, lblock);
    float2 acc[TM / 2][TN];
#pragma unroll
    for (int i = 0; i < TM / 2; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
    const bool idle = u_tile0 + urow >= q.U.rows || l_tile0 + lblock >= q.L.rows;
    for (int kt = s0; kt < s1; ++kt, ++g) {
        const int ds = g % kRawDec;
        mbar_wait(&sm.full[ds], (g / kRawDec) & 1, aborted);
        if (!idle) {
            const uint8_t *st = sm.dec + (size_t)ds * kTmaStageBytes;
            const uint32_t *Uo = reinterpret_cast<const uint32_t *>(st);
            const float *Us = reinterpret_cast<const float *>(st + BK * BU * 4);
            const uint32_t *Lo = reinterpret_cast<const uint32_t *>(st + kTmaUBytes);
            const float *Ls = reinterpret_cast<const float *>(st + kTmaUBytes + BK * BL * 4);
            int fl = 0;
#pragma unroll
            for (int w = 0; w < kRawDecoders / 32; ++w) fl |= sm.flags[ds * (kRawDecoders / 32) + w];
            raw_stage_by_flags<W, GL, ROWS, COLS>(fl, acc, Uo, Us, Lo, Ls, lut, urow, lcol);
        }
        mbar_arrive(&sm.empty[ds]);
    }
    segment_epilogue<ROWS, COLS>(p, q, acc, b, u_tile0, l_tile0, s0, s1, first, cut0, cut1, ncut);
}

template <int W, bool GL>
__device__ __forceinline__ void raw_consumer(const KParams &p, const uint8_t *lut, const RawSmem &sm, int red_bytes)
{
    uint32_t g = 0;
    bool aborted = false;
    CutTile cut0, cut1;
    int ncut = 0;
    for_each_segment(p, [&](const ProbParams &q, int b, int u_tile0, int l_tile0, int s0, int s1, bool first) {
        if (narrow_tail_tile(l_tile0, q.L.rows))
            raw_segment<W, GL, kTailRows, kNarrowTailCols>(p, q, lut, sm, b, u_tile0, l_tile0, s0, s1, first, g,
                                                           aborted, cut0, cut1, ncut);
        else if (tail_tile(l_tile0, q.L.rows))
            raw_segment<W, GL, kTailRows, TN>(p, q, lut, sm, b, u_tile0, l_tile0, s0, s1, first, g, aborted, cut0,
                                              cut1, ncut);
        else
            raw_segment<W, GL, TM, TN>(p, q, lut, sm, b, u_tile0, l_tile0, s0, s1, first, g, aborted, cut0, cut1,
                                       ncut);
    });
    // the rings (decoded, then raw, contiguous) hold the reduction's copies
    finish_cut_tiles(p, cut0, cut1, ncut, reinterpret_cast<float *>(sm.dec), red_bytes, sm.raw_full + 2 * kRawRing +
                     2 * kRawDec, aborted);
}

// Scratch of a phased launch: completion flags [phase][cta]; per tile of the
// launch an arrival ticket (launch epoch in the high half, stages arrived in
// the low half) and a spare word; then, 256-byte aligned, two partial-sum
// slots [phase][cta][2][BU * BL] per CTA and phase (slot 0 for the first
// segment of the CTA's share of the phase, slot 1 for its last).
__device__ __forceinline__ unsigned long long *phase_done(const KParams &p)
{
    return reinterpret_cast<unsigned long long *>(p.ws);
}

__device__ __forceinline__ unsigned long long *tile_ticket(const KParams &p, long long tile)
{
    return phase_done(p) + (long long)n_phases(p) * p.ctas + 2 * tile;
}

__device__ __forceinline__ float *phased_slot(const KParams &p, long long total_tiles, int ph, int cta, int slot)
{
    const long long words = (long long)n_phases(p) * p.ctas + 2 * total_tiles;
    const long long off = ((words * 8 + 255) & ~255LL) / 4;
    return p.ws + off + (((long long)ph * p.ctas + cta) * 2 + slot) * (BU * BL);
}

// Add this part's stages to a cut tile's ticket; true for the part that
// brings the count to the tile's stage count (the last to arrive).
__device__ __forceinline__ bool last_arrival(const KParams &p, long long tile, int stages, int kt_total)
{
    unsigned long long *t = tile_ticket(p, tile);
    const unsigned long long ep = (p.epoch & 0xFFFFFFFFull) << 32;
    unsigned long long v = *reinterpret_cast<volatile unsigned long long *>(t);
    for (;;) {
        const unsigned long long nv =
            (v & 0xFFFFFFFF00000000ull) == ep ? v + (unsigned)stages : ep | (unsigned)stages;
        const unsigned long long old = atomicCAS(t, v, nv);
        if (old == v) return (nv & 0xFFFFFFFFull) == (unsigned long long)kt_total;
        v = old;
    }
}

// First launch iteration of CTA c's share of phase ph (c = ctas: the phase's end).
__device__ __forceinline__ long long ph_begin(const KParams &p, const PhaseTable &pt, int ph, int c)
{
    return p.ph_iter0[ph] + pt.bound[ph][c];
}

// The CTA whose share of phase ph holds launch iteration `it` (the largest c
// with ph_begin(c) <= it: CTAs with empty shares are passed over).
__device__ __forceinline__ int ph_owner(const KParams &p, const PhaseTable &pt, int ph, long long it)
{
    int lo = 0, hi = p.ctas - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ph_begin(p, pt, ph, mid) <= it) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// This CTA's launch iterations in order: its share of every phase.  `it` runs
// through [it, end) of phase `ph`, then moves to the next phase with a
// non-empty share.
struct IterCursor {
    int ph;
    int it, end;               // the raw-tile kernel runs launches of fewer than 2^31 iterations
};

__device__ __forceinline__ void cursor_settle(const KParams &p, const PhaseTable &pt, IterCursor &c)
{
    const int nph = n_phases(p);
    while (c.it >= c.end && c.ph + 1 < nph) {
        ++c.ph;
        c.it = (int)ph_begin(p, pt, c.ph, blockIdx.x);
        c.end = (int)ph_begin(p, pt, c.ph, blockIdx.x + 1);
    }
}

__device__ __forceinline__ IterCursor cursor_start(const KParams &p, const PhaseTable &pt)
{
    IterCursor c;
    c.ph = 0;
    c.it = (int)ph_begin(p, pt, 0, blockIdx.x);
    c.end = (int)ph_begin(p, pt, 0, blockIdx.x + 1);
    cursor_settle(p, pt, c);
    return c;
}

__device__ __forceinline__ void cursor_next(const KParams &p, const PhaseTable &pt, IterCursor &c)
{
    ++c.it;
    cursor_settle(p, pt, c);
}

// Before the first copy of a phase that reads earlier phases' outputs: every
// decoder waits for a part of the completion flags of phases 0 .. nreq - 1
// (one per CTA and phase), then they sync, so that the copies issued or made
// after this see those outputs.
__device__ __forceinline__ void wait_phases(const KParams &p, int nreq, int d, bool &aborted)
{
    const unsigned long long *done = phase_done(p);
    for (int i = d; i < nreq * p.ctas; i += kRawDecoders) flag_wait(done + i, p.epoch, aborted, AMSIM_WAIT_PHASE);
    decoder_bar();
}

// The producer warpgroup of a phased launch: thread 0 also issues the copies;
// every decoder tracks the issue position, so that they can wait for a
// phase's inputs together.
template <int ALU>
__device__ __forceinline__ void raw_producer_phased(const KParams &p, const TmaMaps &maps, const PhaseTable &pt,
                                                   const RawSmem &sm)
{
    const int d = threadIdx.x - kTmaConsumerThreads;
    const int lane = d & 31, dw = d >> 5;
    // decode modes and their shift / fraction mask (closed forms: U keeps its
    // sign and exponent; L keeps them for the exact product, not for Mitchell's);
    // phased launches keep the table in shared memory: packed table words
    constexpr int DU = ALU ? 1 : 3, DL = ALU == 1 ? 2 : ALU ? 1 : 3;
    const uint32_t keep = ((1u << p.M) - 1u) << (23 - p.M);
    const uint32_t offU = ALU ? keep : (uint32_t)(p.M + p.wlog), offL = ALU ? keep : (uint32_t)p.wlog;
    IterCursor cur = cursor_start(p, pt), iss = cur;
    bool aborted = false;
    int issued = 0, gi = 0;    // stages copied, stages passed by the issue position
    int waited_ph = 0;          // phases up to this one have had their inputs awaited
    auto issue = [&]() {
        if (p.nphase > 1 && iss.ph > waited_ph) {
            waited_ph = iss.ph;
            if (p.ph_after[iss.ph] > 0) {
                wait_phases(p, p.ph_after[iss.ph], d, aborted);
                // outputs written through the generic proxy, read by tensor copies
                if (d == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
            }
        }
        const int it = iss.it;
        const int g = gi++;
        cursor_next(p, pt, iss);
        if (d != 0 || aborted) return;
        const int rs = g % kRawRing;
        if (!mbar_wait(&sm.raw_empty[rs], (uint32_t)(((g / kRawRing) & 1) ^ 1), aborted)) return;
        const StagePos sp = stage_pos(p, it);
        const ProbParams &q = p.pr[sp.pi];
        uint8_t *st = sm.raw + (size_t)rs * kRawStageBytes;
        const int k0 = sp.kt * BK;
        if (p.conv) {
            mbar_expect_tx(&sm.raw_full[rs], kRawStageBytes);
            conv_raw_boxes(p, maps, q, sp.u_tile0, sp.l_tile0, sp.kt, st, &sm.raw_full[rs]);
        } else {
            // operands read with plain loads contribute no copy bytes (an all-plain
            // stage is a bare arrival)
            const uint32_t bytes = (q.u_direct ? 0 : kRawUBytes) + (q.l_direct ? 0 : kRawLBytes);
            if (bytes) mbar_expect_tx(&sm.raw_full[rs], bytes);
            else mbar_arrive(&sm.raw_full[rs]);
            if (q.u_direct) {
            } else if (q.u_kfast) {
                tma_load_3d(st, &maps.u[sp.pi], k0, sp.u_tile0, sp.b * q.u_bsel, &sm.raw_full[rs]);
            } else {
                tma_load_3d(st, &maps.u[sp.pi], sp.u_tile0, k0, sp.b * q.u_bsel, &sm.raw_full[rs]);
            }
            if (q.l_direct) {
            } else if (q.l_kfast) {
                tma_load_3d(st + kRawUBytes, &maps.l[sp.pi], k0, sp.l_tile0, sp.b * q.l_bsel, &sm.raw_full[rs]);
            } else {
                tma_load_3d(st + kRawUBytes, &maps.l[sp.pi], sp.l_tile0, k0, sp.b * q.l_bsel, &sm.raw_full[rs]);
            }
        }
        ++issued;
    };
    // Copies run up to kRawRing stages ahead of the decode, except into a
    // phase that reads earlier phases: its first copy waits until every
    // earlier stage of this CTA is decoded, so that the wait for other CTAs
    // never holds back this CTA's own part of the phases it waits for.
    auto may_issue = [&](int g) {
        if (iss.it >= iss.end || gi >= g + kRawRing) return false;
        return !(iss.ph > waited_ph && cur.ph < iss.ph && p.ph_after[iss.ph] > 0);
    };
    for (int g = 0; cur.it < cur.end; cursor_next(p, pt, cur), ++g) {
        while (may_issue(g)) issue();
        const int rs = g % kRawRing, ds = g % kRawDec;
        mbar_wait(&sm.raw_full[rs], (uint32_t)((g / kRawRing) & 1), aborted);
        mbar_wait(&sm.empty[ds], (uint32_t)(((g / kRawDec) & 1) ^ 1), aborted);
        const StagePos sp = stage_pos(p, cur.it);
        const ProbParams &q = p.pr[sp.pi];
        const uint8_t *raw = sm.raw + (size_t)rs * kRawStageBytes;
        uint8_t *st = sm.dec + (size_t)ds * kTmaStageBytes;
        StageFlags big;
        if (q.u_direct || q.l_direct) {
            uint8_t *rw = sm.raw + (size_t)rs * kRawStageBytes;
            if (q.u_direct) direct_copy<BU>(q.U, q.K, sp.b, q.u_bsel, sp.u_tile0, sp.kt * BK, rw, d);
            if (q.l_direct) direct_copy<BL>(q.L, q.K, sp.b, q.l_bsel, sp.l_tile0, sp.kt * BK, rw + kRawUBytes, d);
            cp_async_commit();
            cp_async_wait<0>();
            decoder_bar();          // every decoder's copies have landed
        }
        raw_decode<BU, DU>(raw, q.u_kfast, reinterpret_cast<uint32_t *>(st),
                       reinterpret_cast<float *>(st + BK * BU * 4), p.M, offU, d, big);
        if (p.conv == 2)
            raw_decode_blocks<DL>(raw + kRawUBytes, reinterpret_cast<uint32_t *>(st + kTmaUBytes),
                              reinterpret_cast<float *>(st + kTmaUBytes + BK * BL * 4), p.M, offL, d, big);
        else
            raw_decode<BL, DL, true>(raw + kRawUBytes, q.l_kfast, reinterpret_cast<uint32_t *>(st + kTmaUBytes),
                           reinterpret_cast<float *>(st + kTmaUBytes + BK * BL * 4), p.M, offL, d, big);
        mbar_arrive(&sm.raw_empty[rs]);
        const int any = __reduce_or_sync(0xFFFFFFFFu, big.bits());
        if (lane == 0) sm.flags[ds * (kRawDecoders / 32) + dw] = any;
        mbar_arrive(&sm.full[ds]);
        // the tile after the issue position is the next to be copied: pull its
        // plainly-read operands toward L2 (its phase's inputs may not be ready
        // yet; a prefetch only warms the cache)
        if (p.direct && iss.it < iss.end) {
            const StagePos np = stage_pos(p, iss.it);
            const ProbParams &nq = p.pr[np.pi];
            if (nq.u_direct) direct_prefetch<BU>(nq.U, nq.K, np.b, nq.u_bsel, np.u_tile0, np.kt * BK, d);
            if (nq.l_direct) direct_prefetch<BL>(nq.L, nq.K, np.b, nq.l_bsel, np.l_tile0, np.kt * BK, d);
        }
    }
    if (d == 0 && aborted) {
        // copies issued into raw slots nobody waited for may still be landing
        bool gave_up = false;
        const int n = issued < kRawRing ? issued : kRawRing;
        for (int j = issued - n; j < issued; ++j)
            mbar_wait(&sm.raw_full[j % kRawRing], (uint32_t)((j / kRawRing) & 1), gave_up);
    }
}

// The consumers of a phased launch (LUT in shared memory).  A tile that the
// share boundaries cut is finished without any CTA waiting for another: each
// part leaves its partial sum in its CTA's slot and adds its stage count to
// the tile's ticket; the part that completes the count (the last to arrive)
// adds every part's partial sum in CTA order -- the order of their stages --
// and stores alpha * sum + beta * C.  Results are therefore the same from run
// to run.
// One segment of a phased launch for one consumer warp in the layout ROWS
// (TM, or kTailRows for a tail tile): its stages, then the tile's store, or
// this part's partial sum and, for the last part to arrive, the sum of all
// parts in CTA order.
template <int W, int ROWS>
__device__ __forceinline__ void phased_segment(const KParams &p, const PhaseTable &pt, const ProbParams &q,
                                               const uint8_t *lut, const RawSmem &sm, long long total_tiles, int ph,
                                               int b, int u_tile0, int l_tile0, int s0, int s1, bool first,
                                               uint32_t &g, bool &aborted)
{
    volatile int *last_flag = sm.flags + kRawDec * (kRawDecoders / 32);   // the ticket's verdict
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    int urow, lcol, lblock;
    warp_span<ROWS, TN>(uniform_warp(), lane, urow, lcol, lblock);
    float2 acc[TM / 2][TN];
#pragma unroll
    for (int i = 0; i < TM / 2; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
    const bool idle = u_tile0 + urow >= q.U.rows || l_tile0 + lblock >= q.L.rows;
    for (int kt = s0; kt < s1; ++kt, ++g) {
        const int ds = g % kRawDec;
        mbar_wait(&sm.full[ds], (g / kRawDec) & 1, aborted);
        if (!idle) {
            const uint8_t *st = sm.dec + (size_t)ds * kTmaStageBytes;
            const uint32_t *Uo = reinterpret_cast<const uint32_t *>(st);
            const float *Us = reinterpret_cast<const float *>(st + BK * BU * 4);
            const uint32_t *Lo = reinterpret_cast<const uint32_t *>(st + kTmaUBytes);
            const float *Ls = reinterpret_cast<const float *>(st + kTmaUBytes + BK * BL * 4);
            int fl = 0;
#pragma unroll
            for (int w = 0; w < kRawDecoders / 32; ++w) fl |= sm.flags[ds * (kRawDecoders / 32) + w];
            raw_stage_by_flags<W, false, ROWS>(fl, acc, Uo, Us, Lo, Ls, lut, urow, lcol);
        }
        mbar_arrive(&sm.empty[ds]);
    }
    if (s0 == 0 && s1 == q.kt_total) {
        store_tile<ROWS>(q, acc, b, u_tile0 + urow, l_tile0 + lcol);
        return;
    }
    const long long lt = (long long)b * q.tiles_u * q.tiles_l + (long long)(u_tile0 / BU) * q.tiles_l +
                         l_tile0 / BL;
    float *mine = phased_slot(p, total_tiles, ph, blockIdx.x, first ? 0 : 1);
    if (!idle) {
#pragma unroll
        for (int i = 0; i < ROWS; ++i)
#pragma unroll
            for (int t4 = 0; t4 < TN / 4; ++t4)
                __stcg(reinterpret_cast<float4 *>(mine + (urow + i) * BL + lcol + kColGroup * t4), acc4(acc, i, 4 * t4));
    }
    // every consumer's slot writes precede the barrier; thread 0's
    // fence and ticket update then publish them (cumulative release)
    consumer_bar();
    if (tid == 0) {
        __threadfence();
        const bool last = last_arrival(p, q.tile0 + lt, s1 - s0, q.kt_total);
        __threadfence();
        *last_flag = last ? 1 : 0;
    }
    consumer_bar();
    const bool last = *last_flag != 0;
    consumer_bar();         // everyone has read the ticket's verdict
    if (!last || idle) return;
    const long long tbeg = q.iter0 + lt * q.kt_total, tend = tbeg + q.kt_total;
    const int c_lo = ph_owner(p, pt, ph, tbeg), c_hi = ph_owner(p, pt, ph, tend - 1);
    float2 sum[TM / 2][TN];
#pragma unroll
    for (int i = 0; i < TM / 2; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) sum[i][j] = make_float2(0.0f, 0.0f);
    for (int c = c_lo; c <= c_hi; ++c) {
        const long long cb = ph_begin(p, pt, ph, c);
        if (cb == ph_begin(p, pt, ph, c + 1)) continue;          // empty share
        const float *part = phased_slot(p, total_tiles, ph, c, cb >= tbeg ? 0 : 1);
#pragma unroll
        for (int i = 0; i < ROWS; ++i)
#pragma unroll
            for (int t4 = 0; t4 < TN / 4; ++t4) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(part + (urow + i) * BL + lcol + kColGroup * t4));
                float2 &lo = sum[i >> 1][4 * t4], &l1 = sum[i >> 1][4 * t4 + 1];
                float2 &l2 = sum[i >> 1][4 * t4 + 2], &l3 = sum[i >> 1][4 * t4 + 3];
                if (i & 1) { lo.y += v.x; l1.y += v.y; l2.y += v.z; l3.y += v.w; }
                else { lo.x += v.x; l1.x += v.y; l2.x += v.z; l3.x += v.w; }
            }
    }
    store_tile<ROWS>(q, sum, b, u_tile0 + urow, l_tile0 + lcol);
}

template <int W>
__device__ __forceinline__ void raw_consumer_phased(const KParams &p, const PhaseTable &pt, const uint8_t *lut,
                                                   const RawSmem &sm)
{
    const int tid = threadIdx.x;
    const long long total_tiles = p.pr[p.nprob - 1].tile0 + p.pr[p.nprob - 1].tiles;
    uint32_t g = 0;
    bool aborted = false;
    const int nph = n_phases(p);
    for (int ph = 0; ph < nph; ++ph) {
        const long long it0 = ph_begin(p, pt, ph, blockIdx.x), it1 = ph_begin(p, pt, ph, blockIdx.x + 1);
        // (phased launches keep the regular layout on tail tiles: with a
        // second instance of the stage loops in this kernel the MLP step,
        // which has no tail tiles, ran about 1 % slower)
        walk_segments(p, it0, it1,
                      [&](const ProbParams &q, int b, int u_tile0, int l_tile0, int s0, int s1, bool first) {
            phased_segment<W, TM>(p, pt, q, lut, sm, total_tiles, ph, b, u_tile0, l_tile0, s0, s1, first, g,
                                  aborted);
        });
        // every consumer's stores of the phase precede the flag
        consumer_bar();
        if (tid == 0) flag_store(phase_done(p) + (long long)ph * p.ctas + blockIdx.x, p.epoch);
    }
}

// All problems of a launch read the same LUT orientation (staged once).  PH:
// a phased launch (its own kernel, so that plain launches keep the lean
// single-range loops and their parameter size; the LUT is then in shared
// memory).
template <int W, bool GL, bool PH>
__device__ __forceinline__ void raw_kernel_body(const KParams &p, const TmaMaps &maps, const PhaseTable *pt)
{
    static_assert(!(PH && GL), "phased launches stage the LUT in shared memory");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    // swizzled copies want their boxes 1024-byte aligned: align the base at run time
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int lut_bytes = GL ? 0 : raw_lut_region(p.table_bytes);
    RawSmem sm;
    sm.dec = smem + lut_bytes;
    sm.raw = sm.dec + kRawDec * kTmaStageBytes;
    sm.raw_full = reinterpret_cast<uint64_t *>(sm.raw + kRawRing * kRawStageBytes);
    sm.raw_empty = sm.raw_full + kRawRing;
    sm.full = sm.raw_empty + kRawRing;
    sm.empty = sm.full + kRawDec;
    uint64_t *red = sm.empty + kRawDec;                    // the stream-K reduction's barrier
    uint64_t *lut_bar = red + 1;                           // the LUT's copy into shared memory
    sm.flags = reinterpret_cast<int *>(red + 2);

    if (tid == 0) {
        for (int s = 0; s < kRawRing; ++s) {
            mbar_init(&sm.raw_full[s], 1);
            mbar_init(&sm.raw_empty[s], kRawDecoders);
        }
        for (int s = 0; s < kRawDec; ++s) {
            mbar_init(&sm.full[s], kRawDecoders);
            mbar_init(&sm.empty[s], kTmaConsumerThreads);
        }
        mbar_init(red, 1);
        mbar_init(lut_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!GL && p.table_bytes > 0) {
            // one bulk copy of the table (written when the LUT was built, before
            // any launch; its allocation is padded to 256 bytes), overlapping the
            // first tile copies; the consumers wait for it before their first stage
            const uint32_t bytes = (uint32_t)((p.table_bytes + 15) & ~15);
            mbar_expect_tx(lut_bar, bytes);
            bulk_g2s(smem, p.pr[0].table, bytes, lut_bar);
        }
    }
    if (tid == kTmaConsumerThreads) {
        for (int i = 0; i < p.nprob; ++i) {
            // operands read with plain loads have no tensor map
            if (!p.pr[i].u_direct) tma_prefetch_map(&maps.u[i]);
            if (!p.pr[i].l_direct) tma_prefetch_map(&maps.l[i]);
        }
    }
    __syncthreads();
    // Operands, outputs and scratch may belong to the previous launch on the
    // stream: wait for it to complete before any of them is touched.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const uint8_t *lut = GL ? static_cast<const uint8_t *>(p.pr[0].table) : smem;
    if (tid >= kTmaConsumerThreads) {
        reg_dealloc<kRawProducerRegs>();
        constexpr int ALU = W <= 2 ? W : 0;
        if constexpr (PH) raw_producer_phased<ALU>(p, maps, *pt, sm);
        else raw_producer<ALU, ALU == 0 && !GL>(p, maps, sm);
    } else {
        reg_alloc<kRawConsumerRegs>();
        if (!GL && p.table_bytes > 0) {
            bool gave_up = false;
            mbar_wait(lut_bar, 0, gave_up);
        }
        if constexpr (PH) raw_consumer_phased<W>(p, *pt, lut, sm);
        else raw_consumer<W, GL>(p, lut, sm, kRawDec * kTmaStageBytes + kRawRing * kRawStageBytes);
    }
}

template <int W, bool GL>
__global__ void __launch_bounds__(kRawThreads, 1)
    lutgemm_raw_kernel(const __grid_constant__ KParams p, const __grid_constant__ TmaMaps maps)
{
    raw_kernel_body<W, GL, false>(p, maps, nullptr);
}

template <int W>
__global__ void __launch_bounds__(kRawThreads, 1)
    lutgemm_raw_phased_kernel(const __grid_constant__ KParams p, const __grid_constant__ TmaMaps maps,
                              const __grid_constant__ PhaseTable pt)
{
    raw_kernel_body<W, false, true>(p, maps, &pt);
}

template <int W, bool GL, bool PH = false>
int launch_raw_instance(const KParams &p, const TmaMaps &maps, const PhaseTable *pt, dim3 grid, size_t smem,
                        cudaStream_t st)
{
    auto kernel = [] {
        if constexpr (PH) return lutgemm_raw_phased_kernel<W>;
        else return lutgemm_raw_kernel<W, GL>;
    }();
    static int checked[64] = {};   // 0 unknown, 1 usable, -1 register split not satisfiable
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AMSIM_ECUDA;
    if (dev >= 64) return AMSIM_EUNSUPPORTED;
    if (checked[dev] == 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return cuda_status(e);
        if (fa.numRegs * kRawThreads < kTmaConsumerThreads * kRawConsumerRegs + kRawDecoders * kRawProducerRegs) {
            checked[dev] = -1;
        } else {
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSmemPerCta);
            if (e != cudaSuccess) return cuda_status(e);
            checked[dev] = 1;
        }
    }
    if (checked[dev] < 0) return AMSIM_EUNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kRawThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    for (int pdl = 1; pdl >= 0; --pdl) {
        int na = 0;
        if (pdl) {
            attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attrs[na].val.programmaticStreamSerializationAllowed = 1;
            ++na;
        }
        if (p.fused) {
            attrs[na].id = cudaLaunchAttributeCooperative;
            attrs[na].val.cooperative = 1;
            ++na;
        }
        cfg.attrs = attrs;
        cfg.numAttrs = na;
        cudaError_t e;
        if constexpr (PH) e = cudaLaunchKernelEx(&cfg, kernel, p, maps, *pt);
        else e = cudaLaunchKernelEx(&cfg, kernel, p, maps);
        if (e == cudaSuccess) {
            count_launch();
            return AMSIM_OK;
        }
        cudaGetLastError();
    }
    return p.fused ? AMSIM_ENOTCOOP : AMSIM_ECUDA;
}

// pt: the share boundaries of a phased launch (p.nphase > 1), else null.
int launch_raw_w8(const KParams &p, const TmaMaps &maps, const PhaseTable *pt, bool gl, dim3 grid, size_t smem,
                  cudaStream_t st);
int launch_raw_w16(const KParams &p, const TmaMaps &maps, const PhaseTable *pt, bool gl, dim3 grid, size_t smem,
                   cudaStream_t st);
int launch_raw_w32(const KParams &p, const TmaMaps &maps, const PhaseTable *pt, bool gl, dim3 grid, size_t smem,
                   cudaStream_t st);
// Closed-form products (p.alu: 1 Mitchell, 2 exact), no table.
int launch_raw_alu(const KParams &p, const TmaMaps &maps, const PhaseTable *pt, dim3 grid, size_t smem,
                   cudaStream_t st);

}  // namespace kern
}  // namespace amsim
