// Host planning for the LUT-GEMM kernels (tile counts, split-K, LUT residency,
// operand roles), the deterministic split-K reduction, and the GEMM ABI
// (ApproxTrain Sec. VI-D GEMM kernel; Sec. VI-C AMDENSE forward and gradients).
#include <algorithm>
#include <atomic>

#include "gemm_kernel.cuh"

namespace amsim {

namespace {

using kern::BK;
using kern::BL;
using kern::BU;

constexpr int kMaxSmemLut = 160 * 1024;   // LUTs up to this size are staged in shared memory

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

struct Plan {
    int tiles_u, tiles_l, kt_total, splits, kt_per_split, ws_ld;
    size_t ws_bytes;
};

Plan make_plan(const Problem &p, int sms, size_t ws_avail)
{
    Plan pl;
    pl.tiles_u = std::max(1, ceil_div(p.U.rows, BU));
    pl.tiles_l = std::max(1, ceil_div(p.L.rows, BL));
    pl.kt_total = ceil_div(p.K, BK);
    pl.ws_ld = (p.L.rows + 3) & ~3;
    pl.splits = 1;
    pl.kt_per_split = std::max(1, pl.kt_total);
    pl.ws_bytes = 0;
    const long long tiles = (long long)pl.tiles_u * pl.tiles_l * p.batch;
    // Split the reduction only when the output tiles leave SMs idle: as many
    // splits as fit in one wave, at least two stages per split.
    if (tiles < sms && pl.kt_total >= 4) {
        int want = (int)std::min<long long>(sms / tiles, pl.kt_total / 2);
        want = std::min(want, 65535);
        if (want > 1) {
            int kps = ceil_div(pl.kt_total, want);
            int splits = ceil_div(pl.kt_total, kps);
            size_t need = (size_t)p.batch * splits * (size_t)p.U.rows * pl.ws_ld * sizeof(float);
            if (splits > 1 && need <= ws_avail) {
                pl.splits = splits;
                pl.kt_per_split = kps;
                pl.ws_bytes = need;
            }
        }
    }
    return pl;
}

__global__ void splitk_reduce(const float *__restrict__ ws, int splits, int nU, int nL, int ws_ld, int batch,
                              float *C, long long c_bs, long long c_su, long long c_sl, float alpha, float beta,
                              bool u_fastest)
{
    const long long total = (long long)batch * nU * nL;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        int u, l;
        long long b;
        if (u_fastest) {
            u = (int)(i % nU);
            long long t = i / nU;
            l = (int)(t % nL);
            b = t / nL;
        } else {
            l = (int)(i % nL);
            long long t = i / nL;
            u = (int)(t % nU);
            b = t / nU;
        }
        const float *src = ws + ((b * splits) * nU + u) * (long long)ws_ld + l;
        const long long sstride = (long long)nU * ws_ld;
        float s = 0.0f;
        for (int sp = 0; sp < splits; ++sp) s += src[sp * sstride];
        float *dst = C + b * c_bs + (long long)u * c_su + (long long)l * c_sl;
        float r = alpha * s;
        if (beta != 0.0f) r = fmaf(beta, *dst, r);
        *dst = r;
    }
}

}  // namespace

size_t problem_workspace(const Problem &p, amsim_lut_t lut)
{
    int dev = lut ? lut->device : 0;
    return make_plan(p, device_sms(dev), (size_t)-1).ws_bytes;
}

int run_problem(const Problem &p, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (p.U.rows == 0 || p.L.rows == 0 || p.batch == 0) return AMSIM_OK;
    const int sms = device_sms(lut->device);
    const Plan pl = make_plan(p, sms, ws ? ws_bytes : 0);

    kern::KParams kp;
    kp.U = p.U;
    kp.L = p.L;
    kp.K = p.K;
    kp.batch = p.batch;
    kp.tiles_u = pl.tiles_u;
    kp.tiles_l = pl.tiles_l;
    kp.splits = pl.splits;
    kp.kt_per_split = pl.kt_per_split;
    kp.kt_total = pl.kt_total;
    kp.table = p.u_is_first ? lut->d_narrow : lut->d_narrow_t;
    const bool gl = lut->narrow_bytes > (size_t)kMaxSmemLut ||
                    (size_t)kern::kFixedSmem + kern::lut_region_bytes((int)lut->narrow_bytes) > (size_t)kMaxSmemPerCta;
    kp.table_bytes = gl ? 0 : (int)lut->narrow_bytes;
    kp.M = lut->M;
    kp.mul = 1u << lut->shift;
    kp.wlog = lut->width_bits == 8 ? 0 : lut->width_bits == 16 ? 1 : 2;
    kp.c_ptr = p.c_ptr;
    kp.c_bs = p.c_bs;
    kp.c_su = p.c_su;
    kp.c_sl = p.c_sl;
    kp.alpha = p.alpha;
    kp.beta = p.beta;
    kp.ws = static_cast<float *>(ws);
    kp.ws_ld = pl.ws_ld;
    kp.u_kfast = p.U.gather ? 1 : (p.U.s_k == 1 && p.U.s_row != 1);
    kp.l_kfast = p.L.gather ? 1 : (p.L.s_k == 1 && p.L.s_row != 1);
    if (p.U.gather && p.U.kcb[0] != 1) kp.u_kfast = 0;
    if (p.L.gather && p.L.kcb[0] != 1) kp.l_kfast = 0;

    const size_t smem = (size_t)kern::kFixedSmem + (gl ? 0 : kern::lut_region_bytes(kp.table_bytes));
    if (smem > (size_t)kMaxSmemPerCta) return AMSIM_EUNSUPPORTED;
    const long long tiles = (long long)pl.tiles_u * pl.tiles_l;
    if (tiles > 0x7FFFFFFFLL || p.batch > 65535) return AMSIM_EUNSUPPORTED;
    dim3 grid((unsigned)tiles, (unsigned)pl.splits, (unsigned)p.batch);
    int rc;
    switch (lut->width_bits) {
    case 8: rc = kern::launch_w8(kp, gl, grid, smem, stream); break;
    case 16: rc = kern::launch_w16(kp, gl, grid, smem, stream); break;
    default: rc = kern::launch_w32(kp, gl, grid, smem, stream); break;
    }
    if (rc || pl.splits == 1) return rc;

    const long long total = (long long)p.batch * p.U.rows * p.L.rows;
    long long blocks = std::min<long long>((total + 255) / 256, (long long)sms * 16);
    const bool u_fastest = p.c_su == 1 && p.c_sl != 1;
    splitk_reduce<<<(unsigned)std::max(1LL, blocks), 256, 0, stream>>>(
        kp.ws, pl.splits, p.U.rows, p.L.rows, pl.ws_ld, p.batch, p.c_ptr, p.c_bs, p.c_su, p.c_sl, p.alpha, p.beta,
        u_fastest);
    return cuda_status(cudaGetLastError());
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
