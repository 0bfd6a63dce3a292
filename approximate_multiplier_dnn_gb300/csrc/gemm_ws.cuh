// Warp-specialised LUT-GEMM: eight producer warps stream the operand tiles from
// global memory, decode them (LUT byte offset, power-of-two scale) and fill a
// two-stage shared-memory ring; eight consumer warps only run the LUT lookups
// and the fp32x2 accumulation (ApproxTrain Sec. V-B Algorithm 2 per product,
// Sec. VI-D GEMM kernel, Sec. VI-B implicit-GEMM convolution).
//
// The two roles hand stages over through mbarriers (full: producers arrive,
// consumers wait; empty: the reverse).  Every wait is bounded by the global
// timer: after kWaitLimitNs (waits on another CTA's flag: the settable
// g_flag_wait_limit_ns) a thread records the timeout in a device status word
// that amsim_device_errors reads, stops waiting and still arrives on every
// barrier, so the CTA always runs to its end.  Register budgets are rebalanced with setmaxnreg: producers give
// registers back, consumers take them for deeper instruction-level parallelism.
#pragma once

#include "gemm_kernel.cuh"

namespace amsim {
namespace AMSIM_KNS {

#ifndef AMSIM_WS_PWARPS
#define AMSIM_WS_PWARPS 8
#endif
constexpr int kConsumerWarps = WU * WL;                 // 8
constexpr int kProducerWarps = AMSIM_WS_PWARPS;         // whole warpgroups
constexpr int kWsThreads = (kConsumerWarps + kProducerWarps) * 32;
constexpr int kProducerThreads = kProducerWarps * 32;
#ifndef AMSIM_WS_STAGES
#define AMSIM_WS_STAGES 2
#endif
constexpr int kStages = AMSIM_WS_STAGES;                // decoded stages in the ring
// Register budget: the launch gets 65536 / threads (rounded down to 8) per
// thread; producers release down to kProducerRegs and consumers grow to
// kConsumerRegs, which must fit in what the launch holds.
constexpr int kLaunchRegs = (65536 / kWsThreads) & ~7;
constexpr int kProducerRegs = kProducerWarps == 4 ? 88 : 56;
constexpr int kConsumerRegs =
    ((kWsThreads * kLaunchRegs - kProducerThreads * kProducerRegs) / (kConsumerWarps * 32)) & ~7;
static_assert(kConsumerWarps * 32 * kConsumerRegs + kProducerThreads * kProducerRegs <=
                  kWsThreads * kLaunchRegs, "register split exceeds the launch allocation");
static_assert(kConsumerRegs <= 256 && kConsumerRegs >= kLaunchRegs, "consumer register count");
static_assert(kProducerWarps % 4 == 0, "producer warps must form whole warpgroups");
static_assert(kConsumerWarps % 4 == 0, "consumer warps must form whole warpgroups");

constexpr long long kWaitLimitNs = 2000000000LL;        // 2 s
constexpr int AMSIM_ENOTCOOP = -100;                    // internal: cooperative launch refused

#ifndef AMSIM_WS_RAW
#define AMSIM_WS_RAW 2
#endif
constexpr int kRawStages = AMSIM_WS_RAW;                // raw (undecoded) stages in flight
constexpr int kStageBytes = 2 * BK * UST * 4 + 2 * BK * LST * 4;
constexpr int kRawBytes = (BU + BL) * BK * 4;           // one raw stage: U then L elements
constexpr int kWsFixedSmem = kStages * kStageBytes + kRawStages * kRawBytes + kRowTabBytes + 128;
// the decoded and raw rings (contiguous) double as the stream-K reduction buffer
static_assert(kStages * kStageBytes + kRawStages * kRawBytes >= (BU * BL + 1024 * 4) * 4,
              "stream-K reduction buffer");
static_assert(2 * kStages * 8 + 8 + kStages * kProducerWarps * 4 <= 128, "barrier block");

// Wait status of this translation unit's kernels on the current device: the
// AMSIM_WAIT_* bits of the waits that gave up.  Every translation unit that
// includes this header has its own copy of the two words below (device code
// cannot name another unit's variables without relocatable device code), and
// registers a reader and a writer for them with the library's registry at
// load time, so amsim_device_errors and amsim_set_flag_wait_limit reach all
// of them.
static __device__ unsigned int g_ws_wait_timeouts;
// Limit of the waits on flags that other CTAs raise (stream-K partial sums,
// phase dependencies); copy waits keep kWaitLimitNs.
static __device__ long long g_flag_wait_limit_ns = kWaitLimitNs;

namespace {
int tu_wait_status(unsigned int *bits, int clear)
{
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_ws_wait_timeouts, sizeof(v)) != cudaSuccess) return AMSIM_ECUDA;
    *bits |= v;
    if (clear && v) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_ws_wait_timeouts, &zero, sizeof(zero)) != cudaSuccess) return AMSIM_ECUDA;
    }
    return AMSIM_OK;
}
int tu_flag_wait_limit(long long ns)
{
    return cudaMemcpyToSymbol(g_flag_wait_limit_ns, &ns, sizeof(ns)) == cudaSuccess ? AMSIM_OK : AMSIM_ECUDA;
}
[[maybe_unused]] const bool g_tu_wait_words = register_wait_words(&tu_wait_status, &tu_flag_wait_limit);
}  // namespace

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

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
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
            atomicOr(&g_ws_wait_timeouts, (unsigned)AMSIM_WAIT_COPY);
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
    float *raw;            // kRawStages x (BU + BL) x BK floats, element e of producer t at [e * threads + t]
    RowInfo *rowU, *rowL;
    uint64_t *full, *empty;
    uint64_t *red;         // completion of the stream-K reduction's bulk copies
    int *flags;            // [kStages][kProducerWarps]: bit 0 a stage holds |x| >= 2^64, bit 1 no folded form
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

// Segment walk of launch iterations [it, it_end): calls
// f(q, b, u_tile0, l_tile0, s0, s1, first) per tile segment.
template <typename F>
__device__ __forceinline__ void walk_segments(const KParams &p, long long it, long long it_end, F &&f)
{
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

// Segment walk of this CTA's iterations, shared by both roles.
template <typename F>
__device__ __forceinline__ void for_each_segment(const KParams &p, F &&f)
{
    long long it, it_end;
    if (p.streamk) {
        it = sk_begin(p, blockIdx.x);
        it_end = sk_begin(p, blockIdx.x + 1);
    } else {
        long long t = blockIdx.x;
        int pi = 0;
        while (pi + 1 < p.nprob && t >= p.pr[pi].tiles) t -= p.pr[pi++].tiles;
        it = p.pr[pi].iter0 + t * p.pr[pi].kt_total;
        it_end = it + p.pr[pi].kt_total;
    }
    walk_segments(p, it, it_end, f);
}

// ------------------------------------------------------------------ producer
// Element mapping of a producer thread (same scheme as Loader): "k-fast"
// thread t owns reduction slot t % BK and rows t/BK + (NTH/BK) e; "row-fast"
// owns row t % R (t + NTH*j when R > NTH) and the reduction slots left over.
template <int R>
struct PMap {
    static constexpr int NTH = kProducerThreads;
    static constexpr int N = R * BK / NTH;
    static constexpr int RRF = R > NTH ? R / NTH : 1;
    static constexpr int KSF = R < NTH ? NTH / R : 1;
    static constexpr int CH = N < 8 ? N : 8;             // elements per chunk
    static_assert(R * BK == N * NTH && N % CH == 0, "producer element count");
    bool kfast;
    int rsub, ksub0;
    __device__ __forceinline__ PMap(bool kf, int tid) : kfast(kf)
    {
        if (kfast) { rsub = tid / BK; ksub0 = tid % BK; }
        else if (R <= NTH) { rsub = tid % R; ksub0 = tid / R; }
        else { rsub = tid; ksub0 = 0; }
    }
    __device__ __forceinline__ int row_of(int e) const
    {
        return kfast ? rsub + (NTH / BK) * e : rsub + NTH * (e % RRF);
    }
    __device__ __forceinline__ int k_of(int e) const { return kfast ? ksub0 : ksub0 + KSF * (e / RRF); }
};

__device__ __forceinline__ void cp_async4(float *dst, const float *src, bool valid)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Issue-side state of one operand: asynchronous 4-byte copies of this
// thread's elements of a stage into the raw ring (zero-filled when out of
// range), with the gather's reduction-index counter carried across stages.
template <int R>
struct PIssue {
    PMap<R> map;
    int row0;
    const float *base;
    KState ks;

    __device__ __forceinline__ PIssue() : map(false, 0) {}

    __device__ __forceinline__ void init(const OperandDesc &d, bool kf, int tid, int row_tile0, int b, int kt)
    {
        map = PMap<R>(kf, tid);
        row0 = row_tile0;
        base = d.ptr + (long long)b * d.batch_stride;
        if (d.gather) ks = kstate_at(d, kt * BK + map.ksub0);
    }

    __device__ __forceinline__ void issue(const OperandDesc &d, const RowInfo *rowtab, int kt, int K, float *raw,
                                          int tid)
    {
        constexpr int N = PMap<R>::N, CH = PMap<R>::CH;
        const int kbase = kt * BK;
        if (!d.gather) {
#pragma unroll 1
            for (int c = 0; c < N; c += CH) {
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    const int e = c + j;
                    const int r = row0 + map.row_of(e);
                    const int k = kbase + map.k_of(e);
                    const bool ok = r < d.rows && k < K;
                    const float *src = ok ? base + (long long)r * d.s_row + (long long)k * d.s_k : d.ptr;
                    cp_async4(raw + e * kProducerThreads + tid, src, ok);
                }
            }
        } else {
            KState s = ks;
            int kprev = map.k_of(0);
#pragma unroll 1
            for (int c = 0; c < N; c += CH) {
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    const int e = c + j;
                    const int kk = map.k_of(e);
                    if (kk != kprev) { kstate_advance(d, s, kk - kprev); kprev = kk; }
                    const RowInfo ri = rowtab[map.row_of(e)];
                    int y = ri.y + s.y, x = ri.x + s.x;
                    bool ok = kbase + kk < K;
                    if (d.sy > 1) { ok = ok && y >= 0 && y % d.sy == 0; y /= d.sy; }
                    if (d.sx > 1) { ok = ok && x >= 0 && x % d.sx == 0; x /= d.sx; }
                    ok = ok && (unsigned)y < (unsigned)d.IH && (unsigned)x < (unsigned)d.IW;
                    const float *src = ok ? base + ri.b + s.b + ((long long)y * d.IW + x) * d.Cs : d.ptr;
                    cp_async4(raw + e * kProducerThreads + tid, src, ok);
                }
            }
            kstate_advance(d, ks, BK);
        }
    }
};

// Decode this thread's landed elements of a stage into the consumer layout
// (fmt: with the exponent cast of a (1, E, M) format, scale re-bias eoff).
// nofold collects the elements that keep the stage in the general form: a
// nonzero operand below 2^-63 (zero uniform operands take the table's zero
// row, zero lane operands a zero scale; both fold).
template <int R, int ST, bool LANE>
__device__ __forceinline__ void pdecode(const PMap<R> &map, const float *raw, int tid, uint32_t *off, float *scl,
                                        int M, int offshift, int &big, int &nofold, const ExpFormat &fmt, int eoff)
{
    constexpr int N = PMap<R>::N, CH = PMap<R>::CH;
#pragma unroll 1
    for (int c = 0; c < N; c += CH) {
        float v[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) v[j] = raw[(c + j) * kProducerThreads + tid];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int e = c + j;
            uint32_t o;
            float sc;
            if (fmt.on) {
                decode_fmt(v[j], M, offshift, fmt, eoff, o, sc);
            } else {
                decode(v[j], M, offshift, o, sc, big, LANE ? 0u : uniform_zero_row(M, offshift));
                nofold |= is_small_nonzero(v[j]);
            }
            off[map.k_of(e) * ST + map.row_of(e)] = o;
            scl[map.k_of(e) * ST + map.row_of(e)] = sc;
        }
    }
}

// Where iteration `it` of the launch falls: problem, batch, tile origin, stage.
struct StagePos {
    int pi, b, u_tile0, l_tile0, kt;
};

__device__ __forceinline__ StagePos stage_pos(const KParams &p, long long it)
{
    StagePos sp;
    int pi = 0;
    while (pi + 1 < p.nprob && it >= p.pr[pi + 1].iter0) ++pi;
    const ProbParams &q = p.pr[pi];
    const long long local = it - q.iter0;
    const long long tile = local / q.kt_total;
    sp.pi = pi;
    sp.kt = (int)(local - tile * q.kt_total);
    const int per_batch = q.tiles_u * q.tiles_l;
    sp.b = (int)(tile / per_batch);
    const int rem = (int)(tile - (long long)sp.b * per_batch);
    sp.u_tile0 = (rem / q.tiles_l) * BU;
    sp.l_tile0 = (rem % q.tiles_l) * BL;
    return sp;
}

__device__ __forceinline__ void cta_range(const KParams &p, long long &it, long long &it_end)
{
    if (p.streamk) {
        it = sk_begin(p, blockIdx.x);
        it_end = sk_begin(p, blockIdx.x + 1);
    } else {
        long long t = blockIdx.x;
        int pi = 0;
        while (pi + 1 < p.nprob && t >= p.pr[pi].tiles) t -= p.pr[pi++].tiles;
        it = p.pr[pi].iter0 + t * p.pr[pi].kt_total;
        it_end = it + p.pr[pi].kt_total;
    }
}

template <int W, bool GL>
__device__ __forceinline__ void ws_producer(const KParams &p, const WsSmem &sm)
{
    const int ptid = threadIdx.x - kConsumerWarps * 32;
    const int pwarp = ptid >> 5, lane = ptid & 31;
    const int offU = p.M + p.wlog, offL = p.wlog;
    long long it0, it1;
    cta_range(p, it0, it1);

    PIssue<BU> isU;
    PIssue<BL> isL;
    // Issue the copies of iteration `it` into raw slot `rs`, starting a new
    // segment (row tables, counters) at a tile's first stage or the CTA's first.
    auto issue = [&](long long it, int rs) {
        const StagePos sp = stage_pos(p, it);
        const ProbParams &q = p.pr[sp.pi];
        if (it == it0 || sp.kt == 0) {
            if (q.U.gather || q.L.gather) {
                producer_bar();     // all producers are done with the previous row tables
                if (q.U.gather)
                    for (int r = ptid; r < BU; r += kProducerThreads) sm.rowU[r] = row_info(q.U, sp.u_tile0 + r);
                if (q.L.gather)
                    for (int r = ptid; r < BL; r += kProducerThreads) sm.rowL[r] = row_info(q.L, sp.l_tile0 + r);
                producer_bar();
            }
            isU.init(q.U, q.u_kfast, ptid, sp.u_tile0, sp.b, sp.kt);
            isL.init(q.L, q.l_kfast, ptid, sp.l_tile0, sp.b, sp.kt);
        }
        float *raw = sm.raw + (size_t)rs * ((BU + BL) * BK);
        isU.issue(q.U, sm.rowU, sp.kt, q.K, raw, ptid);
        isL.issue(q.L, sm.rowL, sp.kt, q.K, raw + BU * BK, ptid);
    };

    long long iti = it0;
    for (int r = 0; r < kRawStages - 1; ++r, ++iti) {
        if (iti < it1) issue(iti, r);
        cp_async_commit();
    }
    uint32_t g = 0;
    bool aborted = false;
    for (long long itd = it0; itd < it1; ++itd, ++iti, ++g) {
        if (iti < it1) issue(iti, (int)((g + kRawStages - 1) % kRawStages));
        cp_async_commit();
        cp_async_wait<kRawStages - 1>();        // this thread's copies of stage g have landed
        const ProbParams &q = p.pr[stage_pos(p, itd).pi];
        const int slot = g % kStages;
        mbar_wait(&sm.empty[slot], ((g / kStages) & 1) ^ 1, aborted);
        const float *raw = sm.raw + (size_t)(g % kRawStages) * ((BU + BL) * BK);
        int big = 0, nofold = 0;
        pdecode<BU, UST, false>(PMap<BU>(q.u_kfast, ptid), raw, ptid, st_Uoff(sm, slot), st_Uscl(sm, slot), p.M, offU,
                                big, nofold, p.fmt, p.fmt.off_u);
        pdecode<BL, LST, true>(PMap<BL>(q.l_kfast, ptid), raw + BU * BK, ptid, st_Loff(sm, slot), st_Lscl(sm, slot),
                               p.M, offL, big, nofold, p.fmt, p.fmt.off_l);
        // bit 0: rounding slow products; bit 1: no folded-scale form
        const int any = __reduce_or_sync(0xFFFFFFFFu, (big ? 1 : 0) | (nofold ? 2 : 0));
        if (lane == 0) sm.flags[slot * kProducerWarps + pwarp] = any;
        mbar_arrive(&sm.full[slot]);
    }
    cp_async_wait<0>();
}

__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 2, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ unsigned long long *sk_flags(const KParams &p)
{
    return reinterpret_cast<unsigned long long *>(p.ws + (long long)p.ctas * 2 * (BU * BL));
}

__device__ __forceinline__ void flag_store(unsigned long long *f, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long flag_load(const unsigned long long *f)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}

// Wait until *f == v (another CTA of this cooperative launch raised it);
// `bit` is the AMSIM_WAIT_* kind recorded if the wait gives up.
__device__ __forceinline__ void flag_wait(const unsigned long long *f, unsigned long long v, bool &aborted,
                                          unsigned int bit = AMSIM_WAIT_PARTIAL)
{
    if (aborted) return;
    if (flag_load(f) == v) return;
    const unsigned long long limit = (unsigned long long)*(volatile long long *)&g_flag_wait_limit_ns;
    const unsigned long long t0 = global_ns();
    while (flag_load(f) != v) {
        if (global_ns() - t0 > limit) {
            aborted = true;
            atomicOr(&g_ws_wait_timeouts, bit);
            return;
        }
    }
}

// One past the last launch iteration of the tile with origin (b, u_tile0, l_tile0).
__device__ __forceinline__ long long stage_tile_end(const KParams &p, const ProbParams &q, int b, int u_tile0,
                                                    int l_tile0)
{
    const long long tile = (long long)b * q.tiles_u * q.tiles_l + (long long)(u_tile0 / BU) * q.tiles_l +
                           l_tile0 / BL;
    return q.iter0 + (tile + 1) * q.kt_total;
}

// A tile cut between CTAs (stream-K): its problem, batch and origin, and its
// first launch iteration.
struct CutTile {
    int pi, b, u_tile0, l_tile0;
    long long tstart;
};

// Finish a segment of tile (b, u_tile0, l_tile0) covering stages [s0, s1):
// store a whole tile, or leave the partial sum of a cut tile in this CTA's
// slot (0 for its first segment, 1 for its last) -- for the separate fixup
// kernel, or (fused stream-K) raising the slot's flag and recording the tile
// in `cut` so that finish_cut_tiles reduces it.  Called by all consumer threads.
// ROWS / COLS: TM and TN for the regular warp layout; kTailRows with TN or
// kNarrowTailCols for the tail layouts.
template <int ROWS = TM, int COLS = TN>
__device__ __forceinline__ void segment_epilogue(const KParams &p, const ProbParams &q, float2 (&acc)[TM / 2][TN],
                                                 int b, int u_tile0, int l_tile0, int s0, int s1, bool first,
                                                 CutTile &cut0, CutTile &cut1, int &ncut)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int wu = warp / WL, wl = warp % WL;
    const int ur = ROWS == TM ? wu * TM : warp * ROWS;
    const int lr = ROWS == TM ? wl * 32 * TN + lane * 4 : lane * (COLS == TN ? 4 : COLS);
    const int u0 = u_tile0 + ur, l0 = l_tile0 + lr;
    if (s0 == 0 && s1 == q.kt_total) {
        store_tile<ROWS, COLS>(q, acc, b, u0, l0);
        return;
    }
    const int slot = first ? 0 : 1;
    float *slotp = p.ws + ((long long)blockIdx.x * 2 + slot) * (BU * BL);
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
        if constexpr (COLS == kNarrowTailCols)
            *reinterpret_cast<float2 *>(slotp + (ur + i) * BL + lr) = make_float2(accv(acc, i, 0), accv(acc, i, 1));
#pragma unroll
        for (int t4 = 0; t4 < (COLS == TN ? TN / 4 : 0); ++t4)
            *reinterpret_cast<float4 *>(slotp + (ur + i) * BL + lr + kColGroup * t4) = acc4(acc, i, 4 * t4);
    }
    if (!p.fused) return;
    // every consumer's slot writes precede the barrier; the release store of
    // one thread then publishes all of them (release is cumulative)
    consumer_bar();
    if (threadIdx.x == 0) flag_store(sk_flags(p) + 2 * blockIdx.x + slot, p.epoch);
    CutTile c;
    c.pi = (int)(&q - p.pr);
    c.b = b;
    c.u_tile0 = u_tile0;
    c.l_tile0 = l_tile0;
    c.tstart = stage_tile_end(p, q, b, u_tile0, l_tile0) - q.kt_total;
    if (ncut++ == 0) cut0 = c;
    else cut1 = c;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Fused stream-K: every CTA that holds part of a cut tile reduces an equal
// share of the tile's elements once all of them have left their partial sums.
// One thread pulls the share of every participant's partial into shared
// memory (`red`, free once the main loop is over) with bulk copies; then the
// consumers add the partials in CTA order (the order the separate fixup
// kernel uses), scale by alpha, add beta*C and store.
struct CutShare {
    int c_lo, n;        // participants c_lo .. c_lo + n - 1
    int lo_slot;        // slot of the first participant's partial (the others use slot 0)
    int e_lo, m;        // this CTA's float4 units of the tile
};

__device__ __forceinline__ CutShare cut_share(const KParams &p, const CutTile &ct)
{
    constexpr int kUnits = BU * BL / 4;
    const int G = p.ctas;
    const long long tstart = ct.tstart, tend = tstart + p.pr[ct.pi].kt_total;
    int c_lo = blockIdx.x, c_hi = blockIdx.x;
    while (c_lo > 0 && sk_begin(p, c_lo) > tstart) --c_lo;
    while (c_hi + 1 < G && sk_begin(p, c_hi + 1) < tend) ++c_hi;
    CutShare sh;
    sh.c_lo = c_lo;
    sh.n = c_hi - c_lo + 1;
    // the first participant began before the tile unless it began exactly at
    // its start (then the tile was its first segment); every later one began
    // inside the tile, so the tile was its first segment
    sh.lo_slot = sk_begin(p, c_lo) == tstart ? 0 : 1;
    const int j = blockIdx.x - c_lo;
    sh.e_lo = (int)((long long)j * kUnits / sh.n);
    sh.m = (int)((long long)(j + 1) * kUnits / sh.n) - sh.e_lo;
    return sh;
}

// Consumer thread i waits for the flags of participants i, i + 256, ...
__device__ __forceinline__ void wait_participants(const KParams &p, const CutShare &sh, bool &aborted)
{
    for (int i = threadIdx.x; i < sh.n; i += kConsumerWarps * 32)
        flag_wait(sk_flags(p) + 2 * (sh.c_lo + i) + (i == 0 ? sh.lo_slot : 0), p.epoch, aborted);
}

// One thread: copy every participant's part of this CTA's share into red.
__device__ __forceinline__ void copy_share(const KParams &p, const CutShare &sh, float *red, uint64_t *bar)
{
    for (int i = 0; i < sh.n; ++i) {
        const float *src = p.ws + ((long long)(sh.c_lo + i) * 2 + (i == 0 ? sh.lo_slot : 0)) * (BU * BL) + 4 * sh.e_lo;
        bulk_g2s(red + (size_t)4 * sh.m * i, src, (uint32_t)(16 * sh.m), bar);
    }
}

__device__ __forceinline__ void store_share(const KParams &p, const CutTile &ct, const CutShare &sh, const float *red)
{
    const ProbParams &q = p.pr[ct.pi];
    float *C = q.c_ptr + (long long)ct.b * q.c_bs;
    for (int e = (int)threadIdx.x; e < sh.m; e += kConsumerWarps * 32) {
        const int ur = (4 * (sh.e_lo + e)) / BL, lr = (4 * (sh.e_lo + e)) % BL;
        const int u = ct.u_tile0 + ur, l = ct.l_tile0 + lr;
        float4 sum = *reinterpret_cast<const float4 *>(red + 4 * e);
        for (int i = 1; i < sh.n; ++i) {
            const float4 v = *reinterpret_cast<const float4 *>(red + (size_t)4 * sh.m * i + 4 * e);
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
        }
        if (u >= q.U.rows) continue;
        const float v4[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (l + k >= q.L.rows) break;
            float *dst = C + (long long)u * q.c_su + (long long)(l + k) * q.c_sl;
            float r = q.alpha * v4[k];
            if (q.beta != 0.0f) r = fmaf(q.beta, *dst, r);
            *dst = r;
        }
    }
}

// Reduce this CTA's cut tiles (at most two: its first and its last segment),
// both in one round of copies when `red_bytes` holds both shares.
__device__ __forceinline__ void finish_cut_tiles(const KParams &p, const CutTile &cut0, const CutTile &cut1,
                                                 int ncut, float *red, int red_bytes, uint64_t *bar, bool &aborted)
{
    if (ncut == 0) return;
    const CutShare sh0 = cut_share(p, cut0);
    CutShare sh1 = sh0;
    if (ncut > 1) sh1 = cut_share(p, cut1);
    const int bytes0 = 16 * sh0.m * sh0.n, bytes1 = ncut > 1 ? 16 * sh1.m * sh1.n : 0;
    const bool together = ncut > 1 && bytes0 + bytes1 <= red_bytes;
    uint32_t phase = 0;
    for (int round = 0; round < (ncut > 1 && !together ? 2 : 1); ++round) {
        const bool first_tile = round == 0;
        const bool second_tile = round == 1 || together;
        if (first_tile) wait_participants(p, sh0, aborted);
        if (second_tile) wait_participants(p, sh1, aborted);
        consumer_bar();         // every consumer is past the main loop and has seen the flags
        float *red1 = first_tile ? red + bytes0 / 4 : red;
        if (threadIdx.x == 0) {
            asm volatile("fence.proxy.async;" ::: "memory");
            mbar_expect_tx(bar, (uint32_t)((first_tile ? bytes0 : 0) + (second_tile ? bytes1 : 0)));
            if (first_tile) copy_share(p, sh0, red, bar);
            if (second_tile) copy_share(p, sh1, red1, bar);
        }
        // wait for the copies even after an earlier wait gave up: they land in
        // this CTA's shared memory and must complete before it is released
        bool copies_timed_out = false;
        mbar_wait(bar, phase, copies_timed_out);
        if (first_tile) store_share(p, cut0, sh0, red);
        if (second_tile) store_share(p, cut1, sh1, red1);
        consumer_bar();         // the shared buffer is free again
        phase ^= 1;
    }
}

template <int W, bool GL>
__device__ __forceinline__ void ws_consumer(const KParams &p, const WsSmem &sm)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = uniform_warp();
    const int wu = warp / WL, wl = warp % WL;
    const int urow = wu * TM;
    const int lcol = wl * 32 * TN + lane * 4;
    const uint8_t *lut = GL ? static_cast<const uint8_t *>(p.pr[0].table) : sm.lut;
    uint32_t g = 0;
    bool aborted = false;
    CutTile cut0, cut1;
    int ncut = 0;
    for_each_segment(p, [&](const ProbParams &q, int b, int u_tile0, int l_tile0, int s0, int s1, bool first) {
        float2 acc[TM / 2][TN];
#pragma unroll
        for (int i = 0; i < TM / 2; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
        // a warp whose rows or columns all lie past the problem's edge has nothing to add
        const bool idle = u_tile0 + urow >= q.U.rows || l_tile0 + wl * 32 * TN >= q.L.rows;
        for (int kt = s0; kt < s1; ++kt) {
            const int slot = g % kStages;
            mbar_wait(&sm.full[slot], (g / kStages) & 1, aborted);
            if (idle) {
                mbar_arrive(&sm.empty[slot]);
                ++g;
                continue;
            }
            const int *fl = sm.flags + slot * kProducerWarps;
            int fb = 0;
#pragma unroll
            for (int w = 0; w < kProducerWarps; ++w) fb |= fl[w];
            const bool slow = (fb & 1) != 0;
            if (!p.fmt.on && !GL && fb == 0)
                compute_stage<W, GL, false, UST, LST, false, true>(acc, st_Uoff(sm, slot), st_Uscl(sm, slot),
                                                                   st_Loff(sm, slot), st_Lscl(sm, slot), lut, urow,
                                                                   lcol);
            else if (p.fmt.on)
                compute_stage<W, GL, true, UST, LST, true>(acc, st_Uoff(sm, slot), st_Uscl(sm, slot),
                                                           st_Loff(sm, slot), st_Lscl(sm, slot), lut, urow, lcol,
                                                           &p.fmt);
            else if (slow)
                compute_stage<W, GL, true>(acc, st_Uoff(sm, slot), st_Uscl(sm, slot), st_Loff(sm, slot),
                                           st_Lscl(sm, slot), lut, urow, lcol);
            else
                compute_stage<W, GL, false>(acc, st_Uoff(sm, slot), st_Uscl(sm, slot), st_Loff(sm, slot),
                                            st_Lscl(sm, slot), lut, urow, lcol);
            mbar_arrive(&sm.empty[slot]);
            ++g;
        }
        segment_epilogue(p, q, acc, b, u_tile0, l_tile0, s0, s1, first, cut0, cut1, ncut);
    });
    finish_cut_tiles(p, cut0, cut1, ncut, reinterpret_cast<float *>(sm.stage),
                     kStages * kStageBytes + kRawStages * kRawBytes, sm.red, aborted);
}

// All problems of a launch must read the same LUT orientation (the host splits
// launches otherwise): the table is staged once.
template <int W, bool GL>
__global__ void __launch_bounds__(kWsThreads, 1) lutgemm_ws_kernel(const __grid_constant__ KParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    // The next launch on the stream may begin its own set-up as our CTAs
    // retire (it waits for our results before touching global data).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int lut_bytes = GL ? 0 : lut_region_bytes(p.table_bytes);
    WsSmem sm;
    sm.lut = smem;
    sm.stage = smem + lut_bytes;
    sm.raw = reinterpret_cast<float *>(smem + lut_bytes + kStages * kStageBytes);
    sm.rowU = reinterpret_cast<RowInfo *>(smem + lut_bytes + kStages * kStageBytes + kRawStages * kRawBytes);
    sm.rowL = sm.rowU + BU;
    uint8_t *tail = smem + lut_bytes + kStages * kStageBytes + kRawStages * kRawBytes + kRowTabBytes;
    sm.full = reinterpret_cast<uint64_t *>(tail);
    sm.empty = sm.full + kStages;
    sm.red = sm.empty + kStages;
    sm.flags = reinterpret_cast<int *>(sm.red + 1);

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
        mbar_init(sm.red, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Operands, outputs and scratch may belong to the previous launch on the
    // stream: wait for it to complete before any of them is touched.
    asm volatile("griddepcontrol.wait;" ::: "memory");

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
    // Programmatic stream serialisation lets this launch overlap the tail of
    // the previous one; a cut tile finished inside the kernel needs every CTA
    // resident (cooperative).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kWsThreads);
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
        cudaError_t e = cudaLaunchKernelEx(&cfg, lutgemm_ws_kernel<W, GL>, p);
        if (e == cudaSuccess) {
            count_launch();
            return AMSIM_OK;
        }
        cudaGetLastError();
    }
    return p.fused ? AMSIM_ENOTCOOP : AMSIM_ECUDA;
}

int launch_ws_w8(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);
int launch_ws_w16(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);
int launch_ws_w32(const KParams &p, bool gl, dim3 grid, size_t smem, cudaStream_t st);

}  // namespace AMSIM_KNS
}  // namespace amsim
