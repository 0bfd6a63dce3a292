// LUT-GEMM over predecoded operands, fed by the Tensor Memory Accelerator.
//
// A separate pass (decode.cu) turns every dense operand into two planes once
// per launch -- the byte offset of the element's LUT row/column and its signed
// power-of-two scale, laid out [batch][plane][k][row] -- so that a stage of a
// tile is one 4-D box per operand: BU (or BL) rows x BK reduction steps x both
// planes.  One thread issues the two bulk tensor copies of a stage and the
// copies complete on the stage's "full" mbarrier (transaction bytes); eight
// consumer warps run the LUT lookups exactly as in the warp-specialised kernel
// (ApproxTrain Sec. V-B Algorithm 2 per product, Sec. VI-D GEMM kernel) and
// release the stage on its "empty" mbarrier.  Out-of-range rows and reduction
// steps arrive as zero words, which decode as offset 0 and scale +0.0: the
// product of +0.0 adds nothing.
//
// Every wait is bounded by the global timer (2 s): a thread that gives up
// records it in a device flag and skips its remaining waits, and the copy
// thread waits (again bounded) for its copies still in flight before the CTA
// ends.
#pragma once

#include <cuda.h>

#include "gemm_ws.cuh"

namespace amsim {
namespace kern {

// Shape-independent parts, seen by the host for both tile shapes.
constexpr int kTmaMaxStages = 8;
constexpr int kTmaBarBytes = (2 * kTmaMaxStages + 1) * 8;      // full, empty, reduction
// One ring stage: BK reduction steps of the tile's U rows, then of its L rows,
// [plane][k][row]: one plane of packed operand words (pack_operand) with the
// table in shared memory, two (offsets, then scales) with the table in global
// memory, whose offsets reach 2^23.  Measured on GB300 (4096^3 Mitchell M = 7,
// wide tiles): packed words take the shared-memory wavefronts per lookup from
// 1.25 to 1.125 for 0.2 more instructions: 2.2 % faster with both operands
// packed; packing only the uniform operand gained nothing.
__host__ __device__ constexpr int tma_u_planes(bool gl) { return gl ? 2 : 1; }
__host__ __device__ constexpr int tma_l_planes(bool gl) { return gl ? 2 : 1; }
// `planes` encodes both operands' plane counts: U planes + 4 * L planes.
__host__ __device__ constexpr int tma_planes(bool gl) { return tma_u_planes(gl) + 4 * tma_l_planes(gl); }
__host__ __device__ constexpr int tma_stage_bytes(TileCfg c, int planes)
{
    return c.bk * ((planes & 3) * c.bu + (planes >> 2) * c.bl) * 4;
}
// The ring doubles as the stream-K reduction buffer: one tile plus 16 bytes
// per participant (up to 1024).
__host__ __device__ constexpr int tma_red_bytes(TileCfg c) { return (c.bu * c.bl + 1024 * 4) * 4; }
__host__ __device__ constexpr int tma_min_stages(TileCfg c, int planes)
{
    return (tma_red_bytes(c) + tma_stage_bytes(c, planes) - 1) / tma_stage_bytes(c, planes) < 2
               ? 2 : (tma_red_bytes(c) + tma_stage_bytes(c, planes) - 1) / tma_stage_bytes(c, planes);
}
// Shared memory of the TMA kernel for a ring of `stages` and a LUT region of `lut_bytes`.
__host__ __device__ constexpr int tma_cfg_smem_bytes(TileCfg c, int planes, int lut_bytes, int stages)
{
    return 128 + lut_bytes + stages * tma_stage_bytes(c, planes) + kTmaBarBytes;
}

// Tensor maps of the operand planes of every problem of a launch.
struct TmaMaps {
    CUtensorMap u[kMaxProblems];
    CUtensorMap l[kMaxProblems];
};

}  // namespace kern

// The wide-shape instances (built in their own translation units).
namespace kern_wide {
int launch_tma_w8(const kern::KParams &p, const kern::TmaMaps &maps, bool gl, dim3 grid, size_t smem,
                  cudaStream_t st);
int launch_tma_w16(const kern::KParams &p, const kern::TmaMaps &maps, bool gl, dim3 grid, size_t smem,
                   cudaStream_t st);
int launch_tma_w32(const kern::KParams &p, const kern::TmaMaps &maps, bool gl, dim3 grid, size_t smem,
                   cudaStream_t st);
// stream-K fixup of wide tiles (see launch_fixup)
int launch_fixup(const kern::KParams &p, int boundaries, cudaStream_t st);
}  // namespace kern_wide

namespace AMSIM_KNS {

// The copy thread lives in one extra warp; with AMSIM_TMA_PWARPS=4 it gets a
// whole warpgroup that gives its registers to the consumers (setmaxnreg).
#ifndef AMSIM_TMA_PWARPS
#define AMSIM_TMA_PWARPS 4
#endif
constexpr int kTmaConsumerThreads = WU * WL * 32;              // 256
constexpr int kTmaProducerWarps = AMSIM_TMA_PWARPS;
constexpr int kTmaThreads = kTmaConsumerThreads + 32 * kTmaProducerWarps;
constexpr int kTmaLaunchRegs = (65536 / kTmaThreads) & ~7;
constexpr int kTmaProducerRegs = 56;
constexpr int kTmaConsumerRegs =
    ((kTmaThreads * kTmaLaunchRegs - 32 * kTmaProducerWarps * kTmaProducerRegs) / kTmaConsumerThreads) & ~7;
static_assert(kTmaProducerWarps == 1 || kTmaProducerWarps == 4, "one copy warp or one warpgroup");
static_assert(kTmaProducerWarps == 1 || (kTmaConsumerRegs <= 256 && kTmaConsumerThreads * kTmaConsumerRegs +
                                         128 * kTmaProducerRegs <= kTmaThreads * kTmaLaunchRegs),
              "register split exceeds the launch allocation");
// A stage of two planes (offsets then scales, [k][row]), also the decoded
// stage of the raw-tile kernel.
constexpr int kTmaUBytes = 2 * BK * BU * 4;
constexpr int kTmaLBytes = 2 * BK * BL * 4;
constexpr int kTmaStageBytes = kTmaUBytes + kTmaLBytes;        // 40 KB narrow
static_assert(kTmaStageBytes == tma_stage_bytes(kTiles, 2 + 4 * 2), "stage layout");
static_assert(kTmaStageBytes % 128 == 0 && kTmaUBytes % 128 == 0, "stage alignment");
// The TMA kernel's stage for its table placement: packed words with the
// table in shared memory (20 KB narrow, 24 KB wide), two planes with it in
// global memory.
template <bool GL> constexpr int kTmaStage = tma_stage_bytes(kTiles, tma_planes(GL));
template <bool GL> constexpr int kTmaStageU = tma_u_planes(GL) * BK * BU * 4;
static_assert(kTmaStage<false> % 128 == 0 && kTmaStageU<false> % 128 == 0, "packed stage alignment");

// Box (x, y, z, w) of the 4-D tensor map into shared memory; completes on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z, int w,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// The copy thread: for every iteration of this CTA, wait for the ring slot to
// be released, announce the stage's bytes and issue the two box copies.
template <bool GL>
__device__ __forceinline__ void tma_producer(const KParams &p, const TmaMaps &maps, uint8_t *ring, uint64_t *full,
                                             uint64_t *empty)
{
    long long it0, it1;
    cta_range(p, it0, it1);
    const int S = p.stages;
    int slot = 0;
    uint32_t phase = 0;
    bool aborted = false;
    long long issued = 0;
    for (long long it = it0; it < it1; ++it) {
        if (!mbar_wait(&empty[slot], phase ^ 1, aborted)) break;
        const StagePos sp = stage_pos(p, it);
        const ProbParams &q = p.pr[sp.pi];
        uint8_t *st = ring + (size_t)slot * kTmaStage<GL>;
        mbar_expect_tx(&full[slot], kTmaStage<GL>);
        tma_load_4d(st, &maps.u[sp.pi], sp.u_tile0, sp.kt * BK, 0, sp.b * q.u_bsel, &full[slot]);
        tma_load_4d(st + kTmaStageU<GL>, &maps.l[sp.pi], sp.l_tile0, sp.kt * BK, 0, sp.b * q.l_bsel, &full[slot]);
        ++issued;
        if (++slot == S) { slot = 0; phase ^= 1; }
    }
    if (aborted) {
        // copies issued into slots the consumers never waited for may still
        // be landing: let them finish before the CTA's shared memory goes away
        bool gave_up = false;
        const long long n = issued < S ? issued : S;
        for (long long j = issued - n; j < issued; ++j) {
            const int sl = (int)(j % S);
            mbar_wait(&full[sl], (uint32_t)((j / S) & 1), gave_up);
        }
    }
}

template <int W, bool GL>
__device__ __forceinline__ void tma_consumer(const KParams &p, const uint8_t *lut, uint8_t *ring, uint64_t *full,
                                             uint64_t *empty, uint64_t *red)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = uniform_warp();
    const int wu = warp / WL, wl = warp % WL;
    const int urow = wu * TM;
    const int lcol = wl * 32 * TN + lane * 4;
    const int S = p.stages;
    int slot = 0;
    uint32_t phase = 0;
    bool aborted = false;
    CutTile cut0, cut1;
    int ncut = 0;
    for_each_segment(p, [&](const ProbParams &q, int b, int u_tile0, int l_tile0, int s0, int s1, bool first) {
        // a problem with an operand of magnitude >= 2^64 rounds every product before adding it
        const bool slow = __ldcg(q.u_big) == p.epoch || __ldcg(q.l_big) == p.epoch;
        // a problem whose operands are zero or lie in [2^-63, 2^64) folds the
        // uniform scale into the entry -- with the table in shared memory;
        // gathers from a table in global memory are bound by their misses, and
        // measured slower in the folded form
        const bool fold = !GL && !slow && __ldcg(q.u_small) != p.epoch && __ldcg(q.l_small) != p.epoch;
        float2 acc[TM / 2][TN];
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
        // a warp whose rows or columns all lie past the problem's edge has nothing to add
        const bool idle = u_tile0 + urow >= q.U.rows || l_tile0 + wl * 32 * TN >= q.L.rows;
        for (int kt = s0; kt < s1; ++kt) {
            mbar_wait(&full[slot], phase, aborted);
            if (idle) {
                mbar_arrive(&empty[slot]);
                if (++slot == S) { slot = 0; phase ^= 1; }
                continue;
            }
            // (the scale planes exist only in the two-plane stages of global-memory tables)
            const uint8_t *st = ring + (size_t)slot * kTmaStage<GL>;
            const uint32_t *Uo = reinterpret_cast<const uint32_t *>(st);
            const float *Us = reinterpret_cast<const float *>(st + BK * BU * 4);
            const uint32_t *Lo = reinterpret_cast<const uint32_t *>(st + kTmaStageU<GL>);
            const float *Ls = reinterpret_cast<const float *>(st + kTmaStageU<GL> + BK * BL * 4);
            constexpr bool PU = tma_u_planes(GL) == 1, PL = tma_l_planes(GL) == 1;
            if (slow)
                compute_stage<W, GL, true, BU, BL, false, false, PU, PL>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
            else if (fold)
                compute_stage<W, GL, false, BU, BL, false, true, PU, PL>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
            else
                compute_stage<W, GL, false, BU, BL, false, false, PU, PL>(acc, Uo, Us, Lo, Ls, lut, urow, lcol);
            mbar_arrive(&empty[slot]);
            if (++slot == S) { slot = 0; phase ^= 1; }
        }
        segment_epilogue(p, q, acc, b, u_tile0, l_tile0, s0, s1, first, cut0, cut1, ncut);
    });
    // the ring (at least the reduction buffer's bytes, tma_min_stages) holds the reduction's copies
    finish_cut_tiles(p, cut0, cut1, ncut, reinterpret_cast<float *>(ring), S * kTmaStage<GL>, red, aborted);
}

// All problems of a launch read the same LUT orientation (staged once).
template <int W, bool GL>
__global__ void __launch_bounds__(kTmaThreads, 1)
    lutgemm_tma_kernel(const __grid_constant__ KParams p, const __grid_constant__ TmaMaps maps)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // The next launch on the stream may begin its own set-up as our CTAs retire.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    uint8_t *smem = smem_raw + ((128 - (smem_u32(smem_raw) & 127)) & 127);
    const int lut_bytes = GL ? 0 : lut_region_bytes(p.table_bytes);
    uint8_t *ring = smem + lut_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)p.stages * kTmaStage<GL>);
    uint64_t *empty = full + kTmaMaxStages;

    if constexpr (!GL) {
        // the table was written when the LUT was built, before any launch
        const uint4 *src = static_cast<const uint4 *>(p.pr[0].table);
        uint4 *dst = reinterpret_cast<uint4 *>(smem);
        const int nvec = (p.table_bytes + 15) >> 4;
        for (int i = tid; i < nvec; i += kTmaThreads) dst[i] = __ldg(src + i);
    }
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kTmaConsumerThreads);
        }
        mbar_init(empty + kTmaMaxStages, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid == kTmaConsumerThreads) {
        for (int i = 0; i < p.nprob; ++i) {
            tma_prefetch_map(&maps.u[i]);
            tma_prefetch_map(&maps.l[i]);
        }
    }
    __syncthreads();
    // Planes, flags, outputs and scratch belong to earlier launches on the
    // stream: wait for them to complete before any of them is touched.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const uint8_t *lut = GL ? static_cast<const uint8_t *>(p.pr[0].table) : smem;
    if (tid >= kTmaConsumerThreads) {
        if constexpr (kTmaProducerWarps == 4) reg_dealloc<kTmaProducerRegs>();
        if (tid == kTmaConsumerThreads) tma_producer<GL>(p, maps, ring, full, empty);
    } else {
        if constexpr (kTmaProducerWarps == 4) reg_alloc<kTmaConsumerRegs>();
        tma_consumer<W, GL>(p, lut, ring, full, empty, empty + kTmaMaxStages);
    }
}

template <int W, bool GL>
int launch_tma_instance(const KParams &p, const TmaMaps &maps, dim3 grid, size_t smem, cudaStream_t st)
{
    static int checked[64] = {};   // 0 unknown, 1 usable, -1 register split not satisfiable
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AMSIM_ECUDA;
    if (dev >= 64) return AMSIM_EUNSUPPORTED;
    if (checked[dev] == 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, lutgemm_tma_kernel<W, GL>);
        if (e != cudaSuccess) return cuda_status(e);
        // setmaxnreg.inc waits for registers released from the launch
        // allocation; only launch when the split provably fits in it
        if (kTmaProducerWarps == 4 &&
            fa.numRegs * kTmaThreads < kTmaConsumerThreads * kTmaConsumerRegs + 128 * kTmaProducerRegs) {
            checked[dev] = -1;
        } else {
            e = cudaFuncSetAttribute(lutgemm_tma_kernel<W, GL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSmemPerCta);
            if (e != cudaSuccess) return cuda_status(e);
            checked[dev] = 1;
        }
    }
    if (checked[dev] < 0) return AMSIM_EUNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTmaThreads);
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
        cudaError_t e = cudaLaunchKernelEx(&cfg, lutgemm_tma_kernel<W, GL>, p, maps);
        if (e == cudaSuccess) {
            count_launch();
            return AMSIM_OK;
        }
        cudaGetLastError();
    }
    return p.fused ? AMSIM_ENOTCOOP : AMSIM_ECUDA;
}

int launch_tma_w8(const KParams &p, const TmaMaps &maps, bool gl, dim3 grid, size_t smem, cudaStream_t st);
int launch_tma_w16(const KParams &p, const TmaMaps &maps, bool gl, dim3 grid, size_t smem, cudaStream_t st);
int launch_tma_w32(const KParams &p, const TmaMaps &maps, bool gl, dim3 grid, size_t smem, cudaStream_t st);

}  // namespace AMSIM_KNS
}  // namespace amsim
