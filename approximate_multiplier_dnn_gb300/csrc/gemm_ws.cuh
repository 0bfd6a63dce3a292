// Warp-specialised LUT-GEMM: four producer warps stream the operand tiles from
// global memory, decode them (LUT byte offset, power-of-two scale) and fill a
// two-stage shared-memory ring; eight consumer warps only run the LUT lookups
// and the fp32x2 accumulation (ApproxTrain Sec. V-B Algorithm 2 per product,
// Sec. VI-D GEMM kernel, Sec. VI-B implicit-GEMM convolution).
//
// The two roles hand stages over through mbarriers (full: producers arrive,
// consumers wait; empty: the reverse).  Every wait is bounded by the global
// timer: after kWaitLimitNs a thread records the timeout in a device flag,
// stops waiting and still arrives on every barrier, so the CTA always runs to
// its end.  Register budgets are rebalanced with setmaxnreg: producers give
// registers back, consumers take them for deeper instruction-level parallelism.
#pragma once

#include "gemm_kernel.cuh"

namespace amsim {
namespace kern {

constexpr int kConsumerWarps = WU * WL;                 // 8
constexpr int kProducerWarps = 4;                       // one warpgroup
constexpr int kWsThreads = (kConsumerWarps + kProducerWarps) * 32;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kStages = 2;
constexpr int kLaunchRegs = 168;                        // 65536 / 384 rounded down to 8
constexpr int kProducerRegs = 88;
constexpr int kConsumerRegs = 208;                      // 256*208 + 128*88 == 384*168
static_assert(kConsumerWarps * 32 * kConsumerRegs + kProducerThreads * kProducerRegs <=
                  kWsThreads * kLaunchRegs, "register split exceeds the launch allocation");
static_assert(kConsumerWarps % 4 == 0, "consumer warps must form whole warpgroups");

constexpr long long kWaitLimitNs = 2000000000LL;        // 2 s

constexpr int kStageBytes = 2 * BK * UST * 4 + 2 * BK * LST * 4;
constexpr int kWsFixedSmem = kStages * kStageBytes + kRowTabBytes + 128;

// Set when a bounded wait gave up (one flag per translation unit).
static __device__ unsigned int g_ws_wait_timeouts;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with parity `parity`; false (and `aborted`) on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, bool &aborted)
{
    if (aborted) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > (unsigned long long)kWaitLimitNs) {
            aborted = true;
            atomicOr(&g_ws_wait_timeouts, 1u);
            return false;
        }
    }
    return true;
}

template <int N>
__device__ __forceinline__ void reg_alloc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N));
}

template <int N>
__device__ __forceinline__ void reg_dealloc()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N));
}

__device__ __forceinline__ void producer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kProducerThreads) : "memory");
}

struct WsSmem {
    uint8_t *lut;
    uint8_t *stage;        // kStages x kStageBytes
    RowInfo *rowU, *rowL;
    uint64_t *full, *empty;
    int *flags;            // [kStages][kProducerWarps]: a stage holds |x| >= 2^64
};

__device__ __forceinline__ uint32_t *st_Uoff(const WsSmem &s, int slot)
{
    return reinterpret_cast<uint32_t *>(s.stage + slot * kStageBytes);
}
__device__ __forceinline__ float *st_Uscl(const WsSmem &s, int slot)
{
    return reinterpret_cast<float *>(s.stage + slot * kStageBytes + BK * UST * 4);
}
__device__ __forceinline__ uint32_t *st_Loff(const WsSmem &s, int slot)
{
    return reinterpret_cast<uint32_t *>(s.stage + slot * kStageBytes + 2 * BK * UST * 4);
}
__device__ __forceinline__ float *st_Lscl(const WsSmem &s, int slot)
{
    return reinterpret_cast<float *>(s.stage + slot * kStageBytes + 2 * BK * UST * 4 + BK * LST * 4);
}

// Segment walk shared by both roles: calls f(q, b, u_tile0, l_tile0, s0, s1, first).
template <typename F>
__device__ __forceinline__ void for_each_segment(const KParams &p, F &&f)
{
    long long it, it_end;
    if (p.streamk) {
        it = sk_begin(p.iters, p.ctas, blockIdx.x);
        it_end = sk_begin(p.iters, p.ctas, blockIdx.x + 1);
    } else {
        long long t = blockIdx.x;
        int pi = 0;
        while (pi + 1 < p.nprob && t >= p.pr[pi].tiles) t -= p.pr[pi++].tiles;
        it = p.pr[pi].iter0 + t * p.pr[pi].kt_total;
        it_end = it + p.pr[pi].kt_total;
    }
    bool first = true;
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
        f(q, b, (rem / q.tiles_l) * BU, (rem % q.tiles_l) * BL, s0, s1, first);
        first = false;
        it += s1 - s0;
    }
}

template <int W, bool GL>
__device__ __forceinline__ void ws_producer(const KParams &p, const WsSmem &sm)
{
    const int ptid = threadIdx.x - kConsumerWarps * 32;
    const int pwarp = ptid >> 5, lane = ptid & 31;
    const int offU = p.M + p.wlog, offL = p.wlog;
    uint32_t g = 0;
    bool aborted = false;
    for_each_segment(p, [&](const ProbParams &q, int b, int u_tile0, int l_tile0, int s0, int s1, bool) {
        if (q.U.gather || q.L.gather) {
            producer_bar();     // every producer is done reading the previous segment's row tables
            if (q.U.gather)
                for (int r = ptid; r < BU; r += kProducerThreads) sm.rowU[r] = row_info(q.U, u_tile0 + r);
            if (q.L.gather)
                for (int r = ptid; r < BL; r += kProducerThreads) sm.rowL[r] = row_info(q.L, l_tile0 + r);
            producer_bar();
        }
        Loader<BU, BU * BK / kProducerThreads, kProducerThreads> ldU;
        Loader<BL, BL * BK / kProducerThreads, kProducerThreads> ldL;
        ldU.init(q.U, q.u_kfast, ptid, u_tile0, b, s0);
        ldL.init(q.L, q.l_kfast, ptid, l_tile0, b, s0);
        for (int kt = s0; kt < s1; ++kt) {
            ldU.load(q.U, sm.rowU, kt, q.K);
            ldL.load(q.L, sm.rowL, kt, q.K);
            const int slot = g % kStages;
            mbar_wait(&sm.empty[slot], ((g / kStages) & 1) ^ 1, aborted);
            int big = 0;
            ldU.template store<UST>(st_Uoff(sm, slot), st_Uscl(sm, slot), p.M, offU, big);
            ldL.template store<LST>(st_Loff(sm, slot), st_Lscl(sm, slot), p.M, offL, big);
            const int any = __any_sync(0xFFFFFFFFu, big);
            if (lane == 0) sm.flags[slot * kProducerWarps + pwarp] = any;
            mbar_arrive(&sm.full[slot]);
            ++g;
        }
    });
}

template <int W, bool GL>
__device__ __forceinline__ void ws_consumer(const KParams &p, const WsSmem &sm)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int wu = warp / WL, wl = warp % WL;
    const int urow = wu * TM;
    const int lcol = wl * 32 * TN + lane * TN;
    const uint8_t *lut = GL ? static_cast<const uint8_t *>(p.pr[0].table) : sm.lut;
    uint32_t g = 0;
    bool aborted = false;
    for_each_segment(p, [&](const ProbParams &q, int b, int u_tile0, int l_tile0, int s0, int s1, bool first) {
        float2 acc[TM / 2][TN];
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
        for (int kt = s0; kt < s1; ++kt) {
            const int slot = g % kStages;
            mbar_wait(&sm.full[slot], (g / kStages) & 1, aborted);
            const int *fl = sm.flags + slot * kProducerWarps;
            const bool slow = (fl[0] | fl[1] | fl[2] | fl[3]) != 0;
            if (slow)
                compute_stage<W, GL, true>(acc, st_Uoff(sm, slot), st_Uscl(sm, slot), st_Loff(sm, slot),
                                           st_Lscl(sm, slot), lut, urow, lcol);
            else
                compute_stage<W, GL, false>(acc, st_Uoff(sm, slot), st_Uscl(sm, slot), st_Loff(sm, slot),
                                            st_Lscl(sm, slot), lut, urow, lcol);
            mbar_arrive(&sm.empty[slot]);
            ++g;
        }
        const int u0 = u_tile0 + wu * TM;
        const int l0 = l_tile0 + wl * 32 * TN + lane * TN;
        if (s0 == 0 && s1 == q.kt_total) {
            store_tile(q, acc, b, u0, l0);
        } else {
            float *slotp = p.ws + ((long long)blockIdx.x * 2 + (first ? 0 : 1)) * (BU * BL);
            const int ur = wu * TM, lr = wl * 32 * TN + lane * TN;
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int t4 = 0; t4 < TN / 4; ++t4)
                    *reinterpret_cast<float4 *>(slotp + (ur + i) * BL + lr + 4 * t4) = acc4(acc, i, 4 * t4);
        }
    });
}

// All problems of a launch must read the same LUT orientation (the host splits
// launches otherwise): the table is staged once.
template <int W, bool GL>
__global__ void __launch_bounds__(kWsThreads, 1) lutgemm_ws_kernel(const __grid_constant__ KParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lut_bytes = GL ? 0 : lut_region_bytes(p.table_bytes);
    WsSmem sm;
    sm.lut = smem;
    sm.stage = smem + lut_bytes;
    sm.rowU = reinterpret_cast<RowInfo *>(smem + lut_bytes + kStages * kStageBytes);
    sm.rowL = sm.rowU + BU;
    uint8_t *tail = smem + lut_bytes + kStages * kStageBytes + kRowTabBytes;
    sm.full = reinterpret_cast<uint64_t *>(tail);
    sm.empty = sm.full + kStages;
    sm.flags = reinterpret_cast<int *>(sm.empty + kStages);

    if constexpr (!GL) {
        const uint4 *src = static_cast<const uint4 *>(p.pr[0].table);
        uint4 *dst = reinterpret_cast<uint4 *>(sm.lut);
        const int nvec = (p.table_bytes + 15) >> 4;
        for (int i = tid; i < nvec; i += kWsThreads) dst[i] = __ldg(src + i);
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], kProducerThreads);
            mbar_init(&sm.empty[s], kConsumerWarps * 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (tid >= kConsumerWarps * 32) {
        reg_dealloc<kProducerRegs>();
        ws_producer<W, GL>(p, sm);
    } else {
        reg_alloc<kConsumerRegs>();
        ws_consumer<W, GL>(p, sm);
    }
}

template <int W, bool GL>
int launch_ws_instance(const KParams &p, dim3 grid, size_t smem, cudaStream_t st)
{
    static int checked[64] = {};   // 0 unknown, 1 usable, -1 register split not satisfiable
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AMSIM_ECUDA;
    if (dev >= 64) return AMSIM_EUNSUPPORTED;
    if (checked[dev] == 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, lutgemm_ws_kernel<W, GL>);
        if (e != cudaSuccess) return cuda_status(e);
        // setmaxnreg.inc waits for registers released from the launch
        // allocation; only launch when the split provably fits in it.
        if (fa.numRegs * kWsThreads < kConsumerWarps * 32 * kConsumerRegs + kProducerThreads * kProducerRegs) {
            checked[dev] = -1;
        } else {
            e = cudaFuncSetAttribute(lutgemm_ws_kernel<W, GL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSmemPerCta);
            if (e != cudaSuccess) return cuda_status(e);
            checked[dev] = 1;
        }
    }
    if (checked[dev] < 0) return AMSIM_EUNSUPPORTED;
    lutgemm_ws_kernel<W, GL><<<grid, kWsThreads, smem, st>>>(p);
    return cuda_status(cudaGetLastError());
}

int launch_ws_w8(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);
int launch_ws_w16(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);
int launch_ws_w32(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);

}  // namespace kern
}  // namespace amsim
