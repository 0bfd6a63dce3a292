// One unit of the operand predecode pass (internal), shared by the
// predecode kernel and the fused first phase of the cooperative TMA LUT-GEMM.
// A unit is 64 rows x 64 reduction steps of one batch of one job, decoded by
// 256 threads (16 elements each): row-fast sources are read and written along
// rows (4 rows per thread, 16-byte loads and stores where aligned), the others
// are read along k and transposed through shared memory.
#pragma once

#include "gemm_kernel.cuh"
#include "predecode.h"

namespace amsim {
namespace kern {

constexpr int kDecodePitch = kDecodeTileR + 1;   // odd pitch: conflict-free transposes
constexpr int kDecodeSmemBytes = 2 * kDecodeTileK * kDecodePitch * 4;

// Offset of element (r, k) of a job's batch, and whether it is inside the operand.
__device__ __forceinline__ bool elem_at(const DecodeJob &d, int rh, int rl, int k, long long &off)
{
    const int x = rl + d.roff;
    off = (long long)rh * d.s_rhi + (long long)x * d.s_row + (long long)(k / d.kdiv) * d.s_khi +
          (long long)(k % d.kdiv) * d.s_k;
    return x >= 0 && x < d.rlim;
}

// Four decoded elements at word i of the job's planes: packed words, or
// offsets and scales.
__device__ __forceinline__ void store_quad(const DecodeJob &d, uint32_t *po, float *ps, size_t i, const uint4 &o4,
                                           const float4 &s4)
{
    if (d.packed) {
        *reinterpret_cast<uint4 *>(po + i) = make_uint4(pack_operand(o4.x, s4.x), pack_operand(o4.y, s4.y),
                                                        pack_operand(o4.z, s4.z), pack_operand(o4.w, s4.w));
    } else {
        *reinterpret_cast<uint4 *>(po + i) = o4;
        *reinterpret_cast<float4 *>(ps + i) = s4;
    }
}

// Decode unit t of p.  tid in [0, 256); sync() synchronises those 256 threads;
// t_off / t_scl: kDecodeTileK rows of kDecodePitch words of shared memory each.
template <class Sync>
__device__ __forceinline__ void decode_unit(const DecodeParams &p, long long t, uint32_t (*t_off)[kDecodePitch],
                                            float (*t_scl)[kDecodePitch], int tid, Sync sync)
{
    constexpr int TR = kDecodeTileR, TK = kDecodeTileK;
    const int lane4 = (tid & 15) * 4, grp = tid >> 4;          // 16 groups of 16 threads
    int j = 0;
    while (j + 1 < p.njobs && t >= p.job[j + 1].tile0) ++j;
    const DecodeJob &d = p.job[j];
    const int lt = (int)(t - d.tile0);
    const int per_b = d.tiles_r * d.tiles_k;
    const int b = lt / per_b;
    const int rem = lt - b * per_b;
    const int r0 = (rem / d.tiles_k) * TR, k0 = (rem % d.tiles_k) * TK;
    const float *src = d.src + (long long)b * d.bs;
    uint32_t *po = d.plane + (size_t)b * (d.packed ? 1 : 2) * d.K * d.rows_pad;
    float *ps = reinterpret_cast<float *>(po + (size_t)d.K * d.rows_pad);   // two-plane layout only
    int big = 0, small = 0;
    if (d.rowfast) {
        // rows r .. r + 3 at reduction steps k0 + grp + 16 i
        const int r = r0 + lane4;
        if (r < d.rows) {
#pragma unroll
            for (int i = 0; i < TK / 16; ++i) {
                const int k = k0 + grp + 16 * i;
                if (k >= d.K) break;
                const float *a = src + r + (long long)k * d.s_k;
                float v[4];
                if (d.vec && r + 4 <= d.rows) {
                    const float4 q = __ldcs(reinterpret_cast<const float4 *>(a));
                    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = r + e < d.rows ? __ldcs(a + e) : 0.0f;
                }
                uint4 o4;
                float4 s4;
                decode(v[0], p.M, d.offshift, o4.x, s4.x, big, d.zero_off);
                decode(v[1], p.M, d.offshift, o4.y, s4.y, big, d.zero_off);
                decode(v[2], p.M, d.offshift, o4.z, s4.z, big, d.zero_off);
                decode(v[3], p.M, d.offshift, o4.w, s4.w, big, d.zero_off);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    small |= r + e < d.rows && is_small_nonzero(v[e]);
                }
                // rows_pad is a multiple of 4: the pad columns of a partial quad may be written
                store_quad(d, po, ps, (size_t)k * d.rows_pad + r, o4, s4);
            }
        }
    } else {
        // read steps k0 + lane4 .. + 3 of rows r0 + grp + 16 i, transpose, write rows
        const int k = k0 + lane4;
        int rr0 = r0 + grp;
        int rh = rr0 / d.rdiv, rl = rr0 - rh * d.rdiv;
#pragma unroll
        for (int i = 0; i < TR / 16; ++i) {
            const int r = rr0 + 16 * i;
            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            bool ok[4] = {false, false, false, false};
            if (r < d.rows) {
                long long off;
                const bool in = elem_at(d, rh, rl, k < d.K ? k : 0, off);
                if (d.vec && k + 4 <= d.K) {
                    // k .. k + 3 contiguous and 16-byte aligned
                    if (in) {
                        const float4 q = __ldcs(reinterpret_cast<const float4 *>(src + off));
                        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
                    }
                    ok[0] = ok[1] = ok[2] = ok[3] = in;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (k + e >= d.K) break;
                        long long oe;
                        ok[e] = elem_at(d, rh, rl, k + e, oe);
                        if (ok[e]) v[e] = __ldcs(src + oe);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t o = 0;
                float sc = 0.0f;                 // outside the operand: offset 0, scale +0
                if (ok[e]) {
                    decode(v[e], p.M, d.offshift, o, sc, big, d.zero_off);
                    small |= is_small_nonzero(v[e]);
                }
                t_off[lane4 + e][grp + 16 * i] = o;
                t_scl[lane4 + e][grp + 16 * i] = sc;
            }
            rl += 16;
            while (rl >= d.rdiv) { rl -= d.rdiv; ++rh; }
        }
        sync();
        // each thread writes rows r0 + lane4 .. + 3 of steps k0 + grp + 16 i
        const int r = r0 + lane4;
        if (r < d.rows) {
#pragma unroll
            for (int i = 0; i < TK / 16; ++i) {
                const int kk = grp + 16 * i, k2 = k0 + kk;
                if (k2 >= d.K) break;
                const uint4 o4 = make_uint4(t_off[kk][lane4], t_off[kk][lane4 + 1], t_off[kk][lane4 + 2],
                                            t_off[kk][lane4 + 3]);
                const float4 s4 = make_float4(t_scl[kk][lane4], t_scl[kk][lane4 + 1], t_scl[kk][lane4 + 2],
                                              t_scl[kk][lane4 + 3]);
                store_quad(d, po, ps, (size_t)k2 * d.rows_pad + r, o4, s4);
            }
        }
        sync();
    }
    // every thread of the warp takes part; one store per warp that saw a large
    // (or a small) element
    if (__any_sync(0xFFFFFFFFu, big) && (tid & 31) == 0) *d.flag = p.epoch;
    if (__any_sync(0xFFFFFFFFu, small) && (tid & 31) == 0) *d.flag_small = p.epoch;
}

}  // namespace kern
}  // namespace amsim
