// Depthwise Conv2D tiled kernel for 3x3 filters at stride 2 (unit dilation, one
// filter per channel): the forward pass and the weight gradient, table products
// (ApproxTrain Sec. III, Table I; every product per Sec. V-B, Algorithm 2).
//
// A tile is 4 output rows x 64 output columns x 8 channels (one per warp; a
// lane owns 2 adjacent output columns of all 4 rows).  Its input window,
// 9 rows x 129 columns, arrives by one tensor copy and is packed (as in the
// stride-1 kernel: scale bits and LUT offset per word) into four parity
// planes -- even or odd input row x even or odd input column -- so that the
// taps of one parity class read unit-stride columns of one plane:
//   output (i, j), tap (r, s) reads input (2i + r, 2j + s), i.e. plane
//   (r & 1, s & 1) at row i + (r >> 1), column j + (s >> 1).
// In the forward pass the filter tap is warp-uniform, so every lookup of a
// warp reads one table row.  Tiles holding |x| >= 2^64, infinities or NaN are
// packed again from global memory with NaN kept, and take the rounding slow
// products, as in the stride-1 kernel.
#include "dwconv_kernel.cuh"

namespace amsim {
namespace dw {

constexpr int kS2TP = 4;                  // output rows per tile (and per lane)
constexpr int kS2TQ = 64;                 // output columns per tile
constexpr int kS2CB = 8;                  // channels per tile, one per warp
constexpr int kS2HR = 2 * kS2TP + 1;      // input rows of the window
constexpr int kS2HC = 2 * kS2TQ + 1;      // input columns of the window
constexpr int kS2PW = 66;                 // packed plane row pitch (65 columns used at most)
// plane (a, b) offsets within a channel: rows 5 (a = 0) or 4 (a = 1) of kS2PW words
__host__ __device__ constexpr int s2_plane_off(int a, int b) { return a * 2 * 5 * kS2PW + b * (5 - a) * kS2PW; }
constexpr int kS2CP = 2 * 5 * kS2PW + 2 * 4 * kS2PW;   // 1188 packed words per channel
constexpr int kS2OP = kS2TP * kS2TQ + 2;               // output / dy tile words per channel (258)
constexpr int kS2RawA = (kS2HR * kS2HC * kS2CB * 4 + 127) & ~127;
constexpr int kS2RawB = kS2TP * kS2TQ * kS2CB * 4;
constexpr int kS2Halo = (kS2CB * kS2CP * 4 + 127) & ~127;
constexpr int kS2Out = (kS2CB * kS2OP * 4 + 127) & ~127;
constexpr int kS2WB = (3 * kS2CB * 9 * 4 + 127) & ~127;   // tap offsets, scales, closed-form values
static_assert(kS2Out <= kS2Halo, "the output tile reuses the packed window");
static_assert(s2_plane_off(1, 1) + 4 * kS2PW == kS2CP, "plane layout");

__host__ __device__ constexpr int s2_smem(int table_bytes, int mode)
{
    return dw_lut_region(table_bytes) + kS2RawA + kS2Halo + (mode == 2 ? kS2RawB + kS2Out : kS2WB) + 128;
}

// Packed-plane index of window position (row, col) of one channel.
__device__ __forceinline__ int s2_index(int row, int col)
{
    return s2_plane_off(row & 1, col & 1) + (row >> 1) * kS2PW + (col >> 1);
}

// Fast packing of the raw window [pos][8 channels] into the channels' planes.
__device__ __forceinline__ void s2_pack_window(const float *raw, uint32_t *xt, int k, uint32_t offmask, int tid,
                                               bool &big)
{
#pragma unroll 4
    for (int e = tid; e < kS2HR * kS2HC * 2; e += kDwThreads) {
        const int c4 = e & 1, pos = e >> 1;
        const int row = pos / kS2HC, col = pos - row * kS2HC;
        const float4 v = *reinterpret_cast<const float4 *>(raw + pos * kS2CB + 4 * c4);
        uint32_t *d = xt + 4 * c4 * kS2CP + s2_index(row, col);
        d[0] = dw_pack_fast(v.x, k, offmask, big);
        d[kS2CP] = dw_pack_fast(v.y, k, offmask, big);
        d[2 * kS2CP] = dw_pack_fast(v.z, k, offmask, big);
        d[3 * kS2CP] = dw_pack_fast(v.w, k, offmask, big);
    }
}

// Exact packing (NaN kept) of the window straight from global memory.
__device__ __forceinline__ void s2_repack_window(const float *x, uint32_t *xt, int n, int H, int W, int C, int r0,
                                                 int w0, int c0, int M, int offshift, int tid)
{
    const float *img = x + (long long)n * H * W * C;
    int unused = 0;
    for (int e = tid; e < kS2HR * kS2HC * 2; e += kDwThreads) {
        const int c4 = e & 1, pos = e >> 1;
        const int row = pos / kS2HC, col = pos - row * kS2HC;
        const int h = r0 + row, w = w0 + col, c = c0 + 4 * c4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if ((unsigned)h < (unsigned)H && (unsigned)w < (unsigned)W && c < C)
            v = __ldg(reinterpret_cast<const float4 *>(img + ((long long)h * W + w) * C + c));
        uint32_t *d = xt + 4 * c4 * kS2CP + s2_index(row, col);
        d[0] = dw_pack(v.x, M, offshift, unused);
        d[kS2CP] = dw_pack(v.y, M, offshift, unused);
        d[2 * kS2CP] = dw_pack(v.z, M, offshift, unused);
        d[3 * kS2CP] = dw_pack(v.w, M, offshift, unused);
    }
}

// Forward products of one channel for one lane (xc: the channel's planes,
// offset by the lane's column pair).
template <int W, bool SLOW, bool GL = false>
__device__ __forceinline__ void s2_taps(float2 (&acc)[kS2TP], const uint32_t *xc, const uint8_t *lut,
                                        const uint32_t (&woff)[9], const float (&wsc)[9], uint32_t mul)
{
#pragma unroll
    for (int i = 0; i < kS2TP; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int pr = 0; pr < 5 - a; ++pr) {
                const uint32_t *row = xc + s2_plane_off(a, b) + pr * kS2PW;
                const uint2 a01 = *reinterpret_cast<const uint2 *>(row);
                const uint32_t px[3] = {a01.x, a01.y, b == 0 ? row[2] : 0u};
                uint32_t sb[3];
                float sx[3];
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    sb[k] = dw_scale_bits(px[k]);
                    sx[k] = __uint_as_float(sb[k]);
                }
#pragma unroll
                for (int ro = 0; ro < 2; ++ro) {
                    const int r = 2 * ro + a, i = pr - ro;
                    if (r > 2 || i < 0 || i >= kS2TP) continue;
#pragma unroll
                    for (int so = 0; so < 2; ++so) {
                        const int s = 2 * so + b;
                        if (s > 2) continue;
                        const int t = r * 3 + s;
                        const uint32_t i0 = px[so] - sb[so] + woff[t];
                        const uint32_t i1 = px[so + 1] - sb[so + 1] + woff[t];
                        const float2 v = make_float2(dw_expand(lut_ld<W, GL>(lut, i0), mul),
                                                     dw_expand(lut_ld<W, GL>(lut, i1), mul));
                        const float2 sc = fmul2_ftz(make_float2(wsc[t], wsc[t]), make_float2(sx[so], sx[so + 1]));
                        if constexpr (SLOW) {
                            acc[i].x = __fadd_rn(acc[i].x, __fmul_rn(v.x, sc.x));
                            acc[i].y = __fadd_rn(acc[i].y, __fmul_rn(v.y, sc.y));
                        } else {
                            acc[i] = ffma2(v, sc, acc[i]);
                        }
                    }
                }
            }
}

// Weight-gradient products of one channel for one lane over one tile (dr: the
// channel's dy tile at the lane's column pair).  In the slow form, positions
// past the output gradient's edge are skipped.
template <int W, bool SLOW, bool GL = false>
__device__ __forceinline__ void s2_filter(float2 (&acc)[9], const uint32_t *xc, const uint32_t *dr,
                                          const uint8_t *lut, int rows_ok, bool ok0, bool ok1, uint32_t mul)
{
    uint32_t od[kS2TP][2];
    float2 sd[kS2TP];
#pragma unroll
    for (int i = 0; i < kS2TP; ++i) {
        const uint2 d01 = *reinterpret_cast<const uint2 *>(dr + i * kS2TQ);
        const uint32_t db0 = dw_scale_bits(d01.x), db1 = dw_scale_bits(d01.y);
        od[i][0] = d01.x - db0;
        od[i][1] = d01.y - db1;
        sd[i] = make_float2(__uint_as_float(db0), __uint_as_float(db1));
    }
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int pr = 0; pr < 5 - a; ++pr) {
                const uint32_t *row = xc + s2_plane_off(a, b) + pr * kS2PW;
                const uint2 a01 = *reinterpret_cast<const uint2 *>(row);
                const uint32_t px[3] = {a01.x, a01.y, b == 0 ? row[2] : 0u};
                uint32_t sb[3];
                float sx[3];
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    sb[k] = dw_scale_bits(px[k]);
                    sx[k] = __uint_as_float(sb[k]);
                }
#pragma unroll
                for (int ro = 0; ro < 2; ++ro) {
                    const int r = 2 * ro + a, i = pr - ro;
                    if (r > 2 || i < 0 || i >= kS2TP) continue;
                    const bool row_ok = i < rows_ok;
#pragma unroll
                    for (int so = 0; so < 2; ++so) {
                        const int s = 2 * so + b;
                        if (s > 2) continue;
                        const int t = r * 3 + s;
                        const uint32_t i0 = px[so] - sb[so] + od[i][0];
                        const uint32_t i1 = px[so + 1] - sb[so + 1] + od[i][1];
                        const float2 v = make_float2(dw_expand(lut_ld<W, GL>(lut, i0), mul),
                                                     dw_expand(lut_ld<W, GL>(lut, i1), mul));
                        const float2 sc = fmul2_ftz(make_float2(sx[so], sx[so + 1]), sd[i]);
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
// Closed-form products (amsim_lut_set_closed_form; ALU 1 Mitchell, 2 exact) on
// words packed by dw_pack_alu (the truncated value itself), as in the
// stride-1 kernel: Mitchell adds the other operand's fraction field to the
// truncated value's bits and multiplies by its scale; exact takes one FMA of
// the two truncated values.  Same products and accumulation order as the
// table path, so results are bit-identical.
__device__ __forceinline__ void s2_pack_window_alu(const float *raw, uint32_t *xt, uint32_t keep, int tid, bool &big)
{
#pragma unroll 4
    for (int e = tid; e < kS2HR * kS2HC * 2; e += kDwThreads) {
        const int c4 = e & 1, pos = e >> 1;
        const int row = pos / kS2HC, col = pos - row * kS2HC;
        const float4 v = *reinterpret_cast<const float4 *>(raw + pos * kS2CB + 4 * c4);
        uint32_t *d = xt + 4 * c4 * kS2CP + s2_index(row, col);
        d[0] = dw_pack_alu(v.x, keep, big);
        d[kS2CP] = dw_pack_alu(v.y, keep, big);
        d[2 * kS2CP] = dw_pack_alu(v.z, keep, big);
        d[3 * kS2CP] = dw_pack_alu(v.w, keep, big);
    }
}

template <int ALU>
__device__ __forceinline__ void s2_taps_alu(float2 (&acc)[kS2TP], const uint32_t *xc, const uint32_t (&wv)[9])
{
#pragma unroll
    for (int i = 0; i < kS2TP; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int pr = 0; pr < 5 - a; ++pr) {
                const uint32_t *row = xc + s2_plane_off(a, b) + pr * kS2PW;
                const uint2 a01 = *reinterpret_cast<const uint2 *>(row);
                const uint32_t px[3] = {a01.x, a01.y, b == 0 ? row[2] : 0u};
                uint32_t sb[3];
#pragma unroll
                for (int k = 0; k < 3; ++k) sb[k] = px[k] & 0xFF800000u;
#pragma unroll
                for (int ro = 0; ro < 2; ++ro) {
                    const int r = 2 * ro + a, i = pr - ro;
                    if (r > 2 || i < 0 || i >= kS2TP) continue;
#pragma unroll
                    for (int so = 0; so < 2; ++so) {
                        const int s = 2 * so + b;
                        if (s > 2) continue;
                        const int t = r * 3 + s;
                        if constexpr (ALU == 1) {
                            const float2 w = make_float2(__uint_as_float(wv[t] + px[so] - sb[so]),
                                                         __uint_as_float(wv[t] + px[so + 1] - sb[so + 1]));
                            acc[i] = fadd2(acc[i], fmul2_ftz(w, make_float2(__uint_as_float(sb[so]),
                                                                            __uint_as_float(sb[so + 1]))));
                        } else {
                            const float wf = __uint_as_float(wv[t]);
                            acc[i] = ffma2(make_float2(__uint_as_float(px[so]), __uint_as_float(px[so + 1])),
                                           make_float2(wf, wf), acc[i]);
                        }
                    }
                }
            }
}

template <int ALU>
__device__ __forceinline__ void s2_filter_alu(float2 (&acc)[9], const uint32_t *xc, const uint32_t *dr)
{
    uint32_t od[kS2TP][2];
    float2 sd[kS2TP], dv[kS2TP];
#pragma unroll
    for (int i = 0; i < kS2TP; ++i) {
        const uint2 d01 = *reinterpret_cast<const uint2 *>(dr + i * kS2TQ);
        const uint32_t db0 = d01.x & 0xFF800000u, db1 = d01.y & 0xFF800000u;
        od[i][0] = d01.x - db0;
        od[i][1] = d01.y - db1;
        sd[i] = make_float2(__uint_as_float(db0), __uint_as_float(db1));
        dv[i] = make_float2(__uint_as_float(d01.x), __uint_as_float(d01.y));
    }
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int pr = 0; pr < 5 - a; ++pr) {
                const uint32_t *row = xc + s2_plane_off(a, b) + pr * kS2PW;
                const uint2 a01 = *reinterpret_cast<const uint2 *>(row);
                const uint32_t px[3] = {a01.x, a01.y, b == 0 ? row[2] : 0u};
#pragma unroll
                for (int ro = 0; ro < 2; ++ro) {
                    const int r = 2 * ro + a, i = pr - ro;
                    if (r > 2 || i < 0 || i >= kS2TP) continue;
#pragma unroll
                    for (int so = 0; so < 2; ++so) {
                        const int s = 2 * so + b;
                        if (s > 2) continue;
                        const int t = r * 3 + s;
                        if constexpr (ALU == 1) {
                            const float2 w = make_float2(__uint_as_float(px[so] + od[i][0]),
                                                         __uint_as_float(px[so + 1] + od[i][1]));
                            acc[t] = fadd2(acc[t], fmul2_ftz(w, sd[i]));
                        } else {
                            acc[t] = ffma2(make_float2(__uint_as_float(px[so]), __uint_as_float(px[so + 1])), dv[i],
                                           acc[t]);
                        }
                    }
                }
            }
}

// MODE 0: forward (grid-stride over the tiles); 2: weight gradient (CTA =
// (channel block, share of the spatial tiles)).  ALU 0: table products from
// the staged LUT; 1 / 2: closed forms (the LUT read from global memory only by
// slow tiles).  p.tiles_p / p.tiles_q count
// 4-row / 64-column tiles of the output (or dy) grid.
template <int W, int MODE, int ALU>
__global__ void __launch_bounds__(kDwThreads, 2) dw_s2_kernel(const __grid_constant__ DwTileParams p)
{
    using amsim::kern::mbar_expect_tx;
    using amsim::kern::mbar_init;
    using amsim::kern::mbar_wait;
    using amsim::kern::tma_load_4d;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t *lut = smem;
    const uint8_t *glut = static_cast<const uint8_t *>(p.table);         // slow closed-form tiles
    float *rawA = reinterpret_cast<float *>(smem + (ALU ? 0 : dw_lut_region(p.table_bytes)));
    uint32_t *xt = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(rawA) + kS2RawA);
    uint8_t *after = reinterpret_cast<uint8_t *>(xt) + kS2Halo;
    float *rawB = reinterpret_cast<float *>(after);                      // mode 2
    uint32_t *dyt = reinterpret_cast<uint32_t *>(after + kS2RawB);       // mode 2
    uint32_t *wt_off = reinterpret_cast<uint32_t *>(after);              // mode 0
    float *wt_scl = reinterpret_cast<float *>(after + kS2CB * 9 * 4);
    uint32_t *wt_val = reinterpret_cast<uint32_t *>(after + 2 * kS2CB * 9 * 4);   // closed forms
    uint64_t *bar = reinterpret_cast<uint64_t *>(after + (MODE == 2 ? kS2RawB + kS2Out : kS2WB));

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
        d.p0 = (rest % p.tiles_p) * kS2TP;
        d.n = rest / p.tiles_p;
        d.q0 = tqi * kS2TQ;
        d.c0 = cb * kS2CB;
        return d;
    };
    auto issue = [&](const DwTile &t) {
        mbar_expect_tx(bar, MODE == 2 ? kS2HR * kS2HC * kS2CB * 4 + kS2RawB : kS2HR * kS2HC * kS2CB * 4);
        tma_load_4d(rawA, &p.amap, t.c0, 2 * t.q0 + p.ox, 2 * t.p0 + p.oy, t.n, bar);
        if constexpr (MODE == 2) tma_load_4d(rawB, &p.bmap, t.c0, t.q0, t.p0, t.n, bar);
    };

    if (tid == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (t_begin < t_end) issue(tile_at(t_begin));
    }
    if constexpr (ALU == 0) {   // LUT -> shared memory (the device table is padded to 256 bytes)
        const uint4 *src = static_cast<const uint4 *>(p.table);
        uint4 *dst = reinterpret_cast<uint4 *>(lut);
        const int nvec = (p.table_bytes + 15) >> 4;
        for (int i = tid; i < nvec; i += kDwThreads) dst[i] = __ldg(src + i);
    }
    // the barrier's initialisation and the staged table are visible to every
    // thread before any of them waits on the barrier or reads the table
    __syncthreads();
    const int hi_shift = p.M + p.wlog, lo_shift = p.wlog;

    float2 facc[9];
#pragma unroll
    for (int t = 0; t < 9; ++t) facc[t] = make_float2(0.0f, 0.0f);
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
            s2_pack_window_alu(rawA, xt, keep, tid, big);
            if constexpr (MODE == 2) dw_pack_box_alu<kS2CB>(rawB, dyt, kS2TP * kS2TQ, kS2OP, keep, tid, big);
        } else {
            s2_pack_window(rawA, xt, 23 - p.M - a_shift, ((1u << p.M) - 1u) << a_shift, tid, big);
            if constexpr (MODE == 2)
                dw_pack_box<kS2CB>(rawB, dyt, kS2TP * kS2TQ, kS2OP, 23 - p.M - lo_shift,
                                   ((1u << p.M) - 1u) << lo_shift, tid, big);
        }
        if (MODE != 2 && tid < kS2CB * 9) {
            const int c = tid / 9, tap = tid % 9;
            const float v = tl.c0 + c < p.C ? __ldg(p.b + (long long)tap * p.C + tl.c0 + c) : 0.0f;
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
            issue(tile_at(t + t_step));
        }
        if (slow) {
            s2_repack_window(p.a, xt, tl.n, p.IH, p.IW, p.C, 2 * tl.p0 + p.oy, 2 * tl.q0 + p.ox, tl.c0, p.M, a_shift,
                             tid);
            if constexpr (MODE == 2)
                dw_repack<kS2CB>(p.b, dyt, kS2OP, tl.n, p.OH, p.OW, p.C, tl.p0, tl.q0, tl.c0, kS2TP, kS2TQ, p.M,
                                 lo_shift, tid);
            __syncthreads();
        }

        const uint32_t *xc = xt + warp * kS2CP + 2 * lane;
        if constexpr (MODE == 2) {
            const int rows_ok = p.OH - tl.p0;
            const bool ok0 = tl.q0 + 2 * lane < p.OW, ok1 = tl.q0 + 2 * lane + 1 < p.OW;
            const uint32_t *dr = dyt + warp * kS2OP + 2 * lane;
            if constexpr (ALU != 0) {
                if (slow) s2_filter<W, true, true>(facc, xc, dr, glut, rows_ok, ok0, ok1, p.expand_mul);
                else s2_filter_alu<ALU>(facc, xc, dr);
            } else {
                if (slow) s2_filter<W, true>(facc, xc, dr, lut, rows_ok, ok0, ok1, p.expand_mul);
                else s2_filter<W, false>(facc, xc, dr, lut, rows_ok, ok0, ok1, p.expand_mul);
            }
        } else {
            uint32_t woff[9];
            float wsc[9];
#pragma unroll
            for (int k = 0; k < 9; ++k) {
                woff[k] = wt_off[warp * 9 + k];
                wsc[k] = wt_scl[warp * 9 + k];
            }
            float2 acc[kS2TP];
            if constexpr (ALU != 0) {
                if (slow) {
                    s2_taps<W, true, true>(acc, xc, glut, woff, wsc, p.expand_mul);
                } else {
                    uint32_t wv[9];
#pragma unroll
                    for (int k = 0; k < 9; ++k) wv[k] = wt_val[warp * 9 + k];
                    s2_taps_alu<ALU>(acc, xc, wv);
                }
            } else {
                if (slow) s2_taps<W, true>(acc, xc, lut, woff, wsc, p.expand_mul);
                else s2_taps<W, false>(acc, xc, lut, woff, wsc, p.expand_mul);
            }
            __syncthreads();                // every warp is done with the packed window
            float *ot = reinterpret_cast<float *>(xt);
            float *o = ot + warp * kS2OP + 2 * lane;
#pragma unroll
            for (int i = 0; i < kS2TP; ++i) *reinterpret_cast<float2 *>(o + i * kS2TQ) = acc[i];
            __syncthreads();
            float *dst = p.out + (long long)tl.n * p.OH * p.OW * p.C;
#pragma unroll 4
            for (int e = tid; e < kS2TP * kS2TQ * 2; e += kDwThreads) {
                const int c4 = e & 1, pos = e >> 1;
                const int i = pos / kS2TQ, j = pos % kS2TQ;
                const int pp = tl.p0 + i, qq = tl.q0 + j, c = tl.c0 + 4 * c4;
                if (pp < p.OH && qq < p.OW && c < p.C) {
                    const float *src = ot + 4 * c4 * kS2OP + pos;
                    const float4 v = make_float4(src[0], src[kS2OP], src[2 * kS2OP], src[3 * kS2OP]);
                    __stcs(reinterpret_cast<float4 *>(dst + ((long long)pp * p.OW + qq) * p.C + c), v);
                }
            }
        }
    }
    if constexpr (MODE == 2) {
        // lanes -> lane 0 in a fixed butterfly order; warp w owns channel w of the block
        const int c = cb_fixed * kS2CB + warp;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            float v = facc[k].x + facc[k].y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
            if (lane == 0 && c < p.C) p.out[((long long)g * 9 + k) * p.C + c] = v;
        }
    }
}

// ------------------------------------------------------------------ data gradient
// Stride 2, padding 1: dx(2I + a, 2J + b) = sum over the taps whose parity fits:
//   rows: a = 0 -> tap row 1 at dy row I; a = 1 -> tap rows 0 and 2 at dy rows I + 1 and I
//   columns likewise (b = 0 -> tap column 1 at dy column J; b = 1 -> tap columns 0 and 2
//   at dy columns J + 1 and J).
// A tile is 8 dx rows x 64 dx columns x 16 channels (two per warp); a lane owns
// dx columns 2J, 2J + 1 (J = lane) of all 8 rows and reads dy columns J, J + 1
// of the tile's 5 x 33 dy window.  The tap is warp-uniform, so lookups read one
// table row.  Tiles with |x| >= 2^64, infinities or NaN take a slow computation
// that rounds every product before the add and also visits the off-parity taps
// of every output (as zero operands, as the page's zero-operand rule has them),
// after the on-parity taps, which it adds in the fast branch's order.
constexpr int kSdRows = 8, kSdCols = 64, kSdCB = 16;
constexpr int kSdWR = kSdRows / 2 + 1;        // dy window rows
constexpr int kSdWC = kSdCols / 2 + 1;        // dy window columns
constexpr int kSdPW = kSdWC;                  // packed window row pitch (scalar loads)
constexpr int kSdCP = 170;                    // words per channel: >= 5 x 33, = 2 mod 8
static_assert(kSdWR * kSdPW <= kSdCP, "window pitch");
constexpr int kSdRaw = (kSdWR * kSdWC * kSdCB * 4 + 127) & ~127;
constexpr int kSdWin = (kSdCB * kSdCP * 4 + 127) & ~127;
constexpr int kSdOut = (kSdCB * kDwOP * 4 + 127) & ~127;
constexpr int kSdWB = (3 * kSdCB * 9 * 4 + 127) & ~127;

__host__ __device__ constexpr int sd_smem(int table_bytes)
{
    return dw_lut_region(table_bytes) + kSdRaw + kSdWin + kSdOut + kSdWB + 128;
}

template <int W, bool SLOW, bool GL = false>
__device__ __forceinline__ void sd_channel(float2 (&acc)[kSdRows], const uint32_t *wr, const uint8_t *lut,
                                           const uint32_t (&woff)[9], const float (&wsc)[9], uint32_t mul)
{
#pragma unroll
    for (int i = 0; i < kSdRows; ++i) acc[i] = make_float2(0.0f, 0.0f);
    if constexpr (!SLOW) {
#pragma unroll
        for (int ww = 0; ww < kSdWR; ++ww) {
            const uint32_t d0 = wr[ww * kSdPW], d1 = wr[ww * kSdPW + 1];
            const uint32_t b0 = dw_scale_bits(d0), b1 = dw_scale_bits(d1);
            const float2 sd = make_float2(__uint_as_float(b0), __uint_as_float(b1));
            // (dx row, tap row) pairs this window row feeds
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int row = k == 0 ? 2 * ww : k == 1 ? 2 * ww - 1 : 2 * ww + 1;   // dx row of the lane
                const int r = k == 0 ? 1 : k == 1 ? 0 : 2;
                if (row < 0 || row >= kSdRows) continue;
                // column pair: dx 2J (tap column 1, dy J) and 2J + 1 (tap column 0, dy J + 1)
                const int t1 = r * 3 + 1, t0 = r * 3 + 0, t2 = r * 3 + 2;
                const uint32_t i0 = d0 - b0 + woff[t1], i1 = d1 - b1 + woff[t0];
                const float2 v = make_float2(dw_expand(lut_ld<W, GL>(lut, i0), mul),
                                             dw_expand(lut_ld<W, GL>(lut, i1), mul));
                const float2 sc = fmul2_ftz(make_float2(wsc[t1], wsc[t0]), sd);
                acc[row] = ffma2(v, sc, acc[row]);
                // dx 2J + 1 again: tap column 2 at dy J
                const float v2 = dw_expand(lut_ld<W, GL>(lut, d0 - b0 + woff[t2]), mul);
                acc[row].y = fmaf(v2, fmul_ftz(wsc[t2], sd.x), acc[row].y);
            }
        }
    } else {
        // every product rounded before the add: first the on-parity taps in the
        // fast branch's order (so finite tiles sum exactly as it does), then the
        // off-parity taps of each output as zero operands (a signed zero, or NaN
        // when the tap is infinite or NaN, as the page's zero-operand rule has it)
#pragma unroll
        for (int ww = 0; ww < kSdWR; ++ww) {
            const uint32_t d0 = wr[ww * kSdPW], d1 = wr[ww * kSdPW + 1];
            const uint32_t b0 = dw_scale_bits(d0), b1 = dw_scale_bits(d1);
            const float2 sd = make_float2(__uint_as_float(b0), __uint_as_float(b1));
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int row = k == 0 ? 2 * ww : k == 1 ? 2 * ww - 1 : 2 * ww + 1;
                const int r = k == 0 ? 1 : k == 1 ? 0 : 2;
                if (row < 0 || row >= kSdRows) continue;
                const int t1 = r * 3 + 1, t0 = r * 3 + 0, t2 = r * 3 + 2;
                const float v0 = dw_expand(lut_ld<W, GL>(lut, d0 - b0 + woff[t1]), mul);
                const float v1 = dw_expand(lut_ld<W, GL>(lut, d1 - b1 + woff[t0]), mul);
                const float2 sc = fmul2_ftz(make_float2(wsc[t1], wsc[t0]), sd);
                acc[row].x = __fadd_rn(acc[row].x, __fmul_rn(v0, sc.x));
                acc[row].y = __fadd_rn(acc[row].y, __fmul_rn(v1, sc.y));
                const float v2 = dw_expand(lut_ld<W, GL>(lut, d0 - b0 + woff[t2]), mul);
                acc[row].y = __fadd_rn(acc[row].y, __fmul_rn(v2, fmul_ftz(wsc[t2], sd.x)));
            }
        }
#pragma unroll
        for (int row = 0; row < kSdRows; ++row)
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
                for (int r = 0; r < 3; ++r)
#pragma unroll
                    for (int s = 0; s < 3; ++s) {
                        // on-parity: row + 1 - r and b + 1 - s both even (added above)
                        if (((row + 1 - r) & 1) == 0 && ((b + 1 - s) & 1) == 0) continue;
                        const int t = r * 3 + s;
                        const float v = dw_expand(lut_ld<W, GL>(lut, woff[t]), mul);
                        const float z = __fmul_rn(v, fmul_ftz(wsc[t], 0.0f));
                        if (b == 0) acc[row].x = __fadd_rn(acc[row].x, z);
                        else acc[row].y = __fadd_rn(acc[row].y, z);
                    }
    }
}

// The fast branch of sd_channel in closed form (ALU 1 Mitchell, 2 exact), same
// pairing and order; wv: the channel's nine truncated tap values.
template <int ALU>
__device__ __forceinline__ void sd_channel_alu(float2 (&acc)[kSdRows], const uint32_t *wr, const uint32_t (&wv)[9])
{
#pragma unroll
    for (int i = 0; i < kSdRows; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int ww = 0; ww < kSdWR; ++ww) {
        const uint32_t d0 = wr[ww * kSdPW], d1 = wr[ww * kSdPW + 1];
        const uint32_t b0 = d0 & 0xFF800000u, b1 = d1 & 0xFF800000u;
        const float2 sd = make_float2(__uint_as_float(b0), __uint_as_float(b1));
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int row = k == 0 ? 2 * ww : k == 1 ? 2 * ww - 1 : 2 * ww + 1;
            const int r = k == 0 ? 1 : k == 1 ? 0 : 2;
            if (row < 0 || row >= kSdRows) continue;
            const int t1 = r * 3 + 1, t0 = r * 3 + 0, t2 = r * 3 + 2;
            if constexpr (ALU == 1) {
                const float2 w = make_float2(__uint_as_float(wv[t1] + d0 - b0), __uint_as_float(wv[t0] + d1 - b1));
                acc[row] = fadd2(acc[row], fmul2_ftz(w, sd));
                acc[row].y = __fadd_rn(acc[row].y, fmul_ftz(__uint_as_float(wv[t2] + d0 - b0), sd.x));
            } else {
                acc[row] = ffma2(make_float2(__uint_as_float(d0), __uint_as_float(d1)),
                                 make_float2(__uint_as_float(wv[t1]), __uint_as_float(wv[t0])), acc[row]);
                acc[row].y = fmaf(__uint_as_float(d0), __uint_as_float(wv[t2]), acc[row].y);
            }
        }
    }
}

template <int W, int ALU>
__global__ void __launch_bounds__(kDwThreads, 2) dw_s2d_kernel(const __grid_constant__ DwTileParams p)
{
    using amsim::kern::mbar_expect_tx;
    using amsim::kern::mbar_init;
    using amsim::kern::mbar_wait;
    using amsim::kern::tma_load_4d;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t *lut = smem;
    const uint8_t *glut = static_cast<const uint8_t *>(p.table);         // slow closed-form tiles
    float *raw = reinterpret_cast<float *>(smem + (ALU ? 0 : dw_lut_region(p.table_bytes)));
    uint32_t *win = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(raw) + kSdRaw);
    float *ot = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(win) + kSdWin);
    uint32_t *wt_off = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(ot) + kSdOut);
    float *wt_scl = reinterpret_cast<float *>(wt_off + kSdCB * 9);
    uint32_t *wt_val = wt_off + 2 * kSdCB * 9;   // closed forms
    uint64_t *bar = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(wt_off) + kSdWB);

    const int total = p.tiles * p.cblocks;
    auto tile_at = [&](int t) {
        DwTile d;
        const int cb = t % p.cblocks;
        int rest = t / p.cblocks;
        const int tqi = rest % p.tiles_q;
        rest /= p.tiles_q;
        d.p0 = (rest % p.tiles_p) * kSdRows;     // first dx row
        d.n = rest / p.tiles_p;
        d.q0 = tqi * kSdCols;                    // first dx column
        d.c0 = cb * kSdCB;
        return d;
    };
    auto issue = [&](const DwTile &t) {
        mbar_expect_tx(bar, kSdWR * kSdWC * kSdCB * 4);
        tma_load_4d(raw, &p.amap, t.c0, t.q0 / 2, t.p0 / 2, t.n, bar);
    };
    if (tid == 0) {
        mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if ((int)blockIdx.x < total) issue(tile_at(blockIdx.x));
    }
    if constexpr (ALU == 0) {
        const uint4 *src = static_cast<const uint4 *>(p.table);
        uint4 *dst = reinterpret_cast<uint4 *>(lut);
        const int nvec = (p.table_bytes + 15) >> 4;
        for (int i = tid; i < nvec; i += kDwThreads) dst[i] = __ldg(src + i);
    }
    // the barrier's initialisation and the staged table are visible to every
    // thread before any of them waits on the barrier or reads the table
    __syncthreads();
    const int hi_shift = p.M + p.wlog, lo_shift = p.wlog;
    uint32_t phase = 0;
    bool aborted = false;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const DwTile tl = tile_at(t);
        mbar_wait(bar, phase, aborted);
        phase ^= 1;
        // also orders the previous tile's shared-memory reads before this tile's packing
        if (__syncthreads_or(aborted)) break;
        bool big = false;
        const uint32_t keep = ((1u << p.M) - 1u) << (23 - p.M);
        if constexpr (ALU != 0)
            dw_pack_box_alu<kSdCB>(raw, win, kSdWR * kSdWC, kSdCP, keep, tid, big);
        else
            dw_pack_box<kSdCB>(raw, win, kSdWR * kSdWC, kSdCP, 23 - p.M - lo_shift, ((1u << p.M) - 1u) << lo_shift,
                               tid, big);
        if (tid < kSdCB * 9) {
            const int c = tid / 9, tap = tid % 9;
            const float v = tl.c0 + c < p.C ? __ldg(p.b + (long long)tap * p.C + tl.c0 + c) : 0.0f;
            int wbig = 0;
            const uint32_t pk = dw_pack(v, p.M, hi_shift, wbig);
            big |= wbig != 0;
            wt_off[tid] = pk - dw_scale_bits(pk);
            wt_scl[tid] = __uint_as_float(dw_scale_bits(pk));
            if constexpr (ALU != 0) wt_val[tid] = dw_pack_alu(v, keep, big);
        }
        const bool slow = __syncthreads_or(big);   // the raw window is consumed
        if (tid == 0 && t + (int)gridDim.x < total) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(tile_at(t + gridDim.x));
        }
        if (slow) {
            dw_repack<kSdCB>(p.a, win, kSdCP, tl.n, p.IH, p.IW, p.C, tl.p0 / 2, tl.q0 / 2, tl.c0, kSdWR, kSdWC, p.M,
                             lo_shift, tid);
            __syncthreads();
        }
        float2 acc[2][kSdRows];
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
            const int c = warp + 8 * ci;
            uint32_t woff[9];
            float wsc[9];
#pragma unroll
            for (int k = 0; k < 9; ++k) {
                woff[k] = wt_off[c * 9 + k];
                wsc[k] = wt_scl[c * 9 + k];
            }
            const uint32_t *wr = win + c * kSdCP + lane;
            if constexpr (ALU != 0) {
                if (slow) {
                    sd_channel<W, true, true>(acc[ci], wr, glut, woff, wsc, p.expand_mul);
                } else {
                    uint32_t wv[9];
#pragma unroll
                    for (int k = 0; k < 9; ++k) wv[k] = wt_val[c * 9 + k];
                    sd_channel_alu<ALU>(acc[ci], wr, wv);
                }
            } else {
                if (slow) sd_channel<W, true>(acc[ci], wr, lut, woff, wsc, p.expand_mul);
                else sd_channel<W, false>(acc[ci], wr, lut, woff, wsc, p.expand_mul);
            }
        }
#pragma unroll
        for (int ci = 0; ci < 2; ++ci) {
            float *o = ot + (warp + 8 * ci) * kDwOP + 2 * lane;
#pragma unroll
            for (int i = 0; i < kSdRows; ++i) *reinterpret_cast<float2 *>(o + i * kSdCols) = acc[ci][i];
        }
        __syncthreads();
        float *dst = p.out + (long long)tl.n * p.OH * p.OW * p.C;
#pragma unroll 4
        for (int e = tid; e < kSdRows * kSdCols * 4; e += kDwThreads) {
            const int c4 = e & 3, pos = e >> 2;
            const int i = pos / kSdCols, j = pos % kSdCols;
            const int hh = tl.p0 + i, wq = tl.q0 + j, c = tl.c0 + 4 * c4;
            if (hh < p.OH && wq < p.OW && c < p.C) {
                const float *src = ot + 4 * c4 * kDwOP + pos;
                const float4 v = make_float4(src[0], src[kDwOP], src[2 * kDwOP], src[3 * kDwOP]);
                __stcs(reinterpret_cast<float4 *>(dst + ((long long)hh * p.OW + wq) * p.C + c), v);
            }
        }
    }
}

// alu 0: table products (narrowed width 8 or 16); 1 / 2: closed forms.
int launch_s2d(int alu, int width, const DwTileParams &tp, int grid, size_t smem, cudaStream_t st)
{
    void (*kfn)(DwTileParams);
    if (alu == 1) kfn = width == 8 ? dw_s2d_kernel<8, 1> : dw_s2d_kernel<16, 1>;
    else if (alu == 2) kfn = width == 8 ? dw_s2d_kernel<8, 2> : dw_s2d_kernel<16, 2>;
    else kfn = width == 8 ? dw_s2d_kernel<8, 0> : dw_s2d_kernel<16, 0>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return amsim::cuda_status(e);
    kfn<<<grid, kDwThreads, smem, st>>>(tp);
    return amsim::cuda_status(cudaGetLastError());
}

// table_bytes: the staged table's size, 0 for closed forms.
size_t s2d_smem_bytes(int table_bytes) { return (size_t)sd_smem(table_bytes); }

// Launch for mode 0 or 2; alu and width as for launch_s2d.
int launch_s2(int alu, int mode, int width, const DwTileParams &tp, int grid, size_t smem, cudaStream_t st)
{
    void (*kfn)(DwTileParams);
    if (alu == 1)
        kfn = mode == 0 ? (width == 8 ? dw_s2_kernel<8, 0, 1> : dw_s2_kernel<16, 0, 1>)
                        : (width == 8 ? dw_s2_kernel<8, 2, 1> : dw_s2_kernel<16, 2, 1>);
    else if (alu == 2)
        kfn = mode == 0 ? (width == 8 ? dw_s2_kernel<8, 0, 2> : dw_s2_kernel<16, 0, 2>)
                        : (width == 8 ? dw_s2_kernel<8, 2, 2> : dw_s2_kernel<16, 2, 2>);
    else
        kfn = mode == 0 ? (width == 8 ? dw_s2_kernel<8, 0, 0> : dw_s2_kernel<16, 0, 0>)
                        : (width == 8 ? dw_s2_kernel<8, 2, 0> : dw_s2_kernel<16, 2, 0>);
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return amsim::cuda_status(e);
    kfn<<<grid, kDwThreads, smem, st>>>(tp);
    return amsim::cuda_status(cudaGetLastError());
}

size_t s2_smem_bytes(int table_bytes, int mode) { return (size_t)s2_smem(table_bytes, mode); }

}  // namespace dw
}  // namespace amsim
