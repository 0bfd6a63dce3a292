// Host planning for the LUT-GEMM kernels (tile counts, split-K, LUT residency,
// operand roles), the deterministic split-K reduction, and the GEMM ABI
// (ApproxTrain Sec. VI-D GEMM kernel; Sec. VI-C AMDENSE forward and gradients).
#include <algorithm>
#include <atomic>

#include "gemm_ws.cuh"

namespace amsim {

namespace {

using kern::BK;
using kern::BL;
using kern::BU;

constexpr int kMaxSmemLut = 160 * 1024;   // LUTs up to this size are staged in shared memory

// Stream-K flag values: every launch gets a fresh one, so flags left in
// scratch by earlier launches never match.
std::atomic<unsigned long long> g_epoch{0x5EED0001ULL};

int device_sms(int dev)
{
    static std::atomic<int> cache[64];
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    if (dev >= 0 && dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Launch plan for a group of problems sharing one LUT.
struct Plan {
    int tiles_u[kern::kMaxProblems], tiles_l[kern::kMaxProblems], kt[kern::kMaxProblems];
    long long tiles[kern::kMaxProblems], iter0[kern::kMaxProblems];
    long long total_tiles, iters;
    bool streamk;
    int ctas;
    size_t ws_bytes;   // scratch the chosen plan uses
    size_t sk_bytes;   // scratch stream-K would use
};

Plan make_plan(const Problem *p, int n, int sms, size_t ws_avail)
{
    Plan pl = {};
    for (int i = 0; i < n; ++i) {
        const bool empty = p[i].U.rows == 0 || p[i].L.rows == 0 || p[i].batch == 0;
        pl.tiles_u[i] = std::max(1, ceil_div(p[i].U.rows, BU));
        pl.tiles_l[i] = std::max(1, ceil_div(p[i].L.rows, BL));
        pl.kt[i] = std::max(1, ceil_div(p[i].K, BK));
        pl.tiles[i] = empty ? 0 : (long long)pl.tiles_u[i] * pl.tiles_l[i] * p[i].batch;
        pl.iter0[i] = pl.iters;
        pl.iters += pl.tiles[i] * pl.kt[i];
        pl.total_tiles += pl.tiles[i];
    }
    pl.ctas = (int)std::min<long long>(std::min(sms, kern::kMaxFixupParts), pl.iters);
    pl.sk_bytes = (size_t)2 * pl.ctas * BU * BL * sizeof(float) + (size_t)pl.ctas * sizeof(unsigned long long);
    // Data parallel (one CTA per tile) when the tiles fill the SMs in nearly
    // whole waves; otherwise stream-K over (tile, stage) iterations.
    const long long waves = (pl.total_tiles + sms - 1) / std::max(1, sms);
    const double dp_eff = pl.total_tiles > 0 ? (double)pl.total_tiles / (double)(waves * sms) : 1.0;
    pl.streamk = pl.ctas > 1 && dp_eff < 0.9 && pl.sk_bytes <= ws_avail;
    pl.ws_bytes = pl.streamk ? pl.sk_bytes : 0;
    return pl;
}

int launch_ws(int width, const kern::KParams &kp, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    switch (width) {
    case 8: return kern::launch_ws_w8(kp, gl, grid, smem, st);
    case 16: return kern::launch_ws_w16(kp, gl, grid, smem, st);
    default: return kern::launch_ws_w32(kp, gl, grid, smem, st);
    }
}

int launch_w(int width, const kern::KParams &kp, bool gl, dim3 grid, size_t smem, cudaStream_t st)
{
    switch (width) {
    case 8: return kern::launch_w8(kp, gl, grid, smem, st);
    case 16: return kern::launch_w16(kp, gl, grid, smem, st);
    default: return kern::launch_w32(kp, gl, grid, smem, st);
    }
}

}  // namespace

size_t problems_workspace(const Problem *p, int n, amsim_lut_t lut)
{
    if (n <= 0 || n > kern::kMaxProblems) return 0;
    const int dev = lut ? lut->device : 0;
    const int sms = device_sms(dev);
    Plan pl = make_plan(p, n, sms, (size_t)-1);
    return pl.ws_bytes;
}

size_t problem_workspace(const Problem &p, amsim_lut_t lut) { return problems_workspace(&p, 1, lut); }

namespace {

// One launch for problems that all read the same LUT orientation.
int run_same_table(const Problem *p, int n, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (n <= 0) return AMSIM_OK;
    if (n > kern::kMaxProblems) return AMSIM_EINVAL;
    const int sms = device_sms(lut->device);
    const Plan pl = make_plan(p, n, sms, ws ? ws_bytes : 0);
    if (pl.total_tiles == 0) return AMSIM_OK;

    // Shared-memory LUT when it fits beside the warp-specialised kernel's
    // rings; else beside the single-role kernel's stages; else read from global.
    const size_t lut_smem = kern::lut_region_bytes((int)lut->narrow_bytes);
    bool use_ws = true, gl = false;
    if (lut->narrow_bytes > (size_t)kMaxSmemLut) gl = true;
    else if ((size_t)kern::kWsFixedSmem + lut_smem <= (size_t)kMaxSmemPerCta) gl = false;
    else if ((size_t)kern::kFixedSmem + lut_smem <= (size_t)kMaxSmemPerCta) use_ws = false;
    else gl = true;
    kern::KParams kp = {};
    int np = 0;
    for (int i = 0; i < n; ++i) {
        if (pl.tiles[i] == 0) continue;
        kern::ProbParams &q = kp.pr[np++];
        q.U = p[i].U;
        q.L = p[i].L;
        q.K = p[i].K;
        q.batch = p[i].batch;
        q.tiles_u = pl.tiles_u[i];
        q.tiles_l = pl.tiles_l[i];
        q.kt_total = pl.kt[i];
        q.tiles = pl.tiles[i];
        q.iter0 = pl.iter0[i];
        q.table = p[i].u_is_first ? lut->d_narrow : lut->d_narrow_t;
        q.c_ptr = p[i].c_ptr;
        q.c_bs = p[i].c_bs;
        q.c_su = p[i].c_su;
        q.c_sl = p[i].c_sl;
        q.alpha = p[i].alpha;
        q.beta = p[i].beta;
        q.u_kfast = p[i].U.gather ? (p[i].U.kcb[0] == 1) : (p[i].U.s_k == 1 && p[i].U.s_row != 1);
        q.l_kfast = p[i].L.gather ? (p[i].L.kcb[0] == 1) : (p[i].L.s_k == 1 && p[i].L.s_row != 1);
    }
    kp.nprob = np;
    kp.streamk = pl.streamk ? 1 : 0;
    kp.iters = pl.iters;
    kp.ctas = pl.ctas;
    kp.table_bytes = gl ? 0 : (int)lut->narrow_bytes;
    kp.M = lut->M;
    kp.wlog = lut->width_bits == 8 ? 0 : lut->width_bits == 16 ? 1 : 2;
    kp.ws = static_cast<float *>(ws);

    const size_t lutb = gl ? 0 : kern::lut_region_bytes(kp.table_bytes);
    const long long blocks = pl.streamk ? pl.ctas : pl.total_tiles;
    if (blocks > 0x7FFFFFFFLL) return AMSIM_EUNSUPPORTED;
    // warp-specialised kernel first; the single-role kernel if its register
    // split cannot be honoured on this device
    int rc = AMSIM_EUNSUPPORTED;
    if (use_ws) {
        // stream-K: finish cut tiles inside the kernel when a cooperative
        // launch is possible, else run the separate fixup kernel afterwards
        kp.fused = pl.streamk ? 1 : 0;
        kp.epoch = g_epoch.fetch_add(1, std::memory_order_relaxed);
        rc = launch_ws(lut->width_bits, kp, gl, dim3((unsigned)blocks), (size_t)kern::kWsFixedSmem + lutb, stream);
        if (rc == kern::AMSIM_ENOTCOOP) {
            kp.fused = 0;
            rc = launch_ws(lut->width_bits, kp, gl, dim3((unsigned)blocks), (size_t)kern::kWsFixedSmem + lutb, stream);
        }
        if (rc == AMSIM_OK && kp.fused) return AMSIM_OK;
    }
    if (rc == AMSIM_EUNSUPPORTED) {
        kp.fused = 0;
        rc = launch_w(lut->width_bits, kp, gl, dim3((unsigned)blocks), (size_t)kern::kFixedSmem + lutb, stream);
    }
    if (rc || !pl.streamk) return rc;
    return kern::launch_fixup(kp, pl.ctas - 1, stream);
}

}  // namespace

int run_problems(const Problem *p, int n, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (n <= 0) return AMSIM_OK;
    if (n > kern::kMaxProblems) return AMSIM_EINVAL;
    if (lut->symmetric) return run_same_table(p, n, lut, ws, ws_bytes, stream);
    // an asymmetric LUT read in both orientations: one launch per orientation
    Problem part[kern::kMaxProblems];
    for (int orient = 0; orient < 2; ++orient) {
        int m = 0;
        for (int i = 0; i < n; ++i)
            if ((int)p[i].u_is_first == orient) part[m++] = p[i];
        int rc = run_same_table(part, m, lut, ws, ws_bytes, stream);
        if (rc) return rc;
    }
    return AMSIM_OK;
}

int run_problem(const Problem &p, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    return run_problems(&p, 1, lut, ws, ws_bytes, stream);
}

}  // namespace amsim

// ------------------------------------------------------------------ GEMM ABI
namespace {

using amsim::OperandDesc;
using amsim::Problem;
using amsim::kern::BL;
using amsim::kern::BU;

OperandDesc dense(const float *ptr, int rows, long long s_row, long long s_k, long long batch_stride)
{
    OperandDesc d = {};
    d.ptr = ptr;
    d.rows = rows;
    d.gather = 0;
    d.s_row = s_row;
    d.s_k = s_k;
    d.batch_stride = batch_stride;
    d.kD0 = d.kD1 = d.rE0 = d.rE1 = 1;
    d.IH = d.IW = 1;
    d.sy = d.sx = 1;
    return d;
}

bool trans_flag(char t, bool *out)
{
    if (t == 'N' || t == 'n') { *out = false; return true; }
    if (t == 'T' || t == 't') { *out = true; return true; }
    return false;
}

// Padded tile area if U = first operand's rows (a) and L = second's (b).
long long padded_area(int u_rows, int l_rows)
{
    return (long long)((u_rows + BU - 1) / BU) * BU * ((long long)((l_rows + BL - 1) / BL) * BL);
}

int build_gemm(char transA, char transB, int m, int n, int k, float alpha, const float *A, int lda,
               long long strideA, const float *B, int ldb, long long strideB, float beta, float *C, int ldc,
               long long strideC, int batch, Problem *pr)
{
    bool ta, tb;
    if (!trans_flag(transA, &ta) || !trans_flag(transB, &tb)) return AMSIM_EINVAL;
    if (m < 0 || n < 0 || k < 0 || batch < 0) return AMSIM_EINVAL;
    if (strideA < 0 || strideB < 0 || strideC < 0) return AMSIM_EINVAL;
    if (lda < std::max(1, ta ? m : k) || ldb < std::max(1, tb ? k : n) || ldc < std::max(1, n)) return AMSIM_EINVAL;
    if (batch > 0 && m > 0 && n > 0) {
        if (!C) return AMSIM_EINVAL;
        if (k > 0 && (!A || !B)) return AMSIM_EINVAL;
    }
    const OperandDesc a = dense(A, m, ta ? 1 : lda, ta ? lda : 1, strideA);
    const OperandDesc b = dense(B, n, tb ? ldb : 1, tb ? 1 : ldb, strideB);
    const bool swap = padded_area(n, m) < padded_area(m, n);
    pr->U = swap ? b : a;
    pr->L = swap ? a : b;
    pr->u_is_first = !swap;
    pr->K = k;
    pr->batch = batch;
    pr->c_ptr = C;
    pr->c_bs = strideC;
    pr->c_su = swap ? 1 : ldc;
    pr->c_sl = swap ? ldc : 1;
    pr->alpha = alpha;
    pr->beta = beta;
    return AMSIM_OK;
}

}  // namespace

extern "C" {

int amsim_gemm_strided_batched(char transA, char transB, int m, int n, int k, float alpha, const float *A, int lda,
                               int64_t strideA, const float *B, int ldb, int64_t strideB, float beta, float *C,
                               int ldc, int64_t strideC, int batch, amsim_lut_t lut, void *ws, size_t ws_bytes,
                               amsim_stream_t stream)
{
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    Problem pr;
    rc = build_gemm(transA, transB, m, n, k, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC, batch,
                    &pr);
    if (rc) return rc;
    return amsim::run_problem(pr, lut, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

int amsim_gemm(char transA, char transB, int m, int n, int k, float alpha, const float *A, int lda, const float *B,
               int ldb, float beta, float *C, int ldc, amsim_lut_t lut, void *ws, size_t ws_bytes,
               amsim_stream_t stream)
{
    return amsim_gemm_strided_batched(transA, transB, m, n, k, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1, lut,
                                      ws, ws_bytes, stream);
}

static int grouped_build(const amsim_gemm_problem *g, Problem *pr)
{
    return build_gemm(g->transA, g->transB, g->m, g->n, g->k, g->alpha, g->A, g->lda, g->strideA, g->B, g->ldb,
                      g->strideB, g->beta, g->C, g->ldc, g->strideC, g->batch, pr);
}

int amsim_gemm_grouped(int count, const amsim_gemm_problem *problems, amsim_lut_t lut, void *ws, size_t ws_bytes,
                       amsim_stream_t stream)
{
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    if (count < 0 || (count > 0 && !problems)) return AMSIM_EINVAL;
    Problem pr[amsim::kern::kMaxProblems];
    for (int i = 0; i < count; ++i) {           // validate everything before enqueuing anything
        rc = grouped_build(&problems[i], &pr[0]);
        if (rc) return rc;
    }
    for (int base = 0; base < count; base += amsim::kern::kMaxProblems) {
        const int n = std::min(count - base, amsim::kern::kMaxProblems);
        for (int i = 0; i < n; ++i) grouped_build(&problems[base + i], &pr[i]);
        rc = amsim::run_problems(pr, n, lut, ws, ws_bytes, static_cast<cudaStream_t>(stream));
        if (rc) return rc;
    }
    return AMSIM_OK;
}

size_t amsim_gemm_grouped_workspace_size(int count, const amsim_gemm_problem *problems, amsim_lut_t lut)
{
    if (!lut || count <= 0 || !problems) return 0;
    Problem pr[amsim::kern::kMaxProblems];
    size_t best = 0;
    for (int base = 0; base < count; base += amsim::kern::kMaxProblems) {
        const int n = std::min(count - base, amsim::kern::kMaxProblems);
        for (int i = 0; i < n; ++i)
            if (grouped_build(&problems[base + i], &pr[i])) return 0;
        best = std::max(best, amsim::problems_workspace(pr, n, lut));
    }
    return best;
}

size_t amsim_gemm_workspace_size(char transA, char transB, int m, int n, int k, int batch, amsim_lut_t lut)
{
    if (!lut) return 0;
    Problem pr;
    static const float dummy = 0.0f;
    float *dc = const_cast<float *>(&dummy);
    bool ta, tb;
    if (!trans_flag(transA, &ta) || !trans_flag(transB, &tb) || m < 0 || n < 0 || k < 0 || batch < 1) return 0;
    if (build_gemm(transA, transB, m, n, k, 1.0f, &dummy, std::max(1, ta ? m : k), 0, &dummy,
                   std::max(1, tb ? k : n), 0, 0.0f, dc, std::max(1, n), 0, batch, &pr))
        return 0;
    return amsim::problem_workspace(pr, lut);
}

}  // extern "C"
