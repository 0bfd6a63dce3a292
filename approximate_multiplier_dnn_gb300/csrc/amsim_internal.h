// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "amsim.h"

struct CUtensorMap_st;   // cuda.h's tensor map (CUtensorMap)

struct amsim_lut_s {
    int M = 0;
    int device = -1;
    int width_bits = 32;   // narrowed entry width: 8, 16 or 32
    int shift = 0;         // canonical entry = narrowed << shift
    bool symmetric = false;
    void *d_base = nullptr;       // one allocation holding everything below
    const uint32_t *d_canon = nullptr;   // 2^(2M) canonical entries, index p<<M|q
    const void *d_narrow = nullptr;      // narrowed, index [first operand][second operand]
    const void *d_narrow_t = nullptr;    // narrowed, index [second operand][first operand]
    size_t narrow_bytes = 0;             // 2^(2M) narrowed entries (each copy is followed by a zero row)
    int kind = -1;              // AMSIM_EXACT / AMSIM_MITCHELL when built from a kind, else -1
    bool closed_form = false;   // raw-tile launches compute products in registers (kinds only)
    int exp_bits = 8;           // exponent bits E of the simulated (1, E, M) format
};

// The exponent cast of a (1, E, M) format with E < 8 (ApproxTrain Sec. V-B,
// last paragraph), as the kernels apply it.  Bias B = 2^(E-1) - 1; an fp32
// operand with biased exponent e is zero below lo = 128 - B, infinite above
// hi = 127 + B, else kept.  Its power-of-two scale is re-biased by `off`
// (off_u + off_l = B - 127), so that the flush-to-zero scale product sa * sb
// is zero exactly when Algorithm 2's e0 = eA + eB - B is not above zero; the
// product v * sa * sb is then multiplied by vscale = 2^(127 - B) (exactly) and
// becomes an infinity at or above lim = 2^(B + 1), Algorithm 2's overflow.
// E = 8 gives lo = 1, hi = 254, no offsets, vscale 1 and lim = infinity: the
// ordinary fp32 path.
struct ExpFormat {
    int on;                  // E < 8
    int lo, hi;
    int off_u, off_l;        // scale re-bias of the U and L operands (or first and second)
    int bias, all_ones;      // B and 2^E - 1 (elementwise bit logic)
    float vscale, lim;
};

inline ExpFormat exp_format(int E)
{
    ExpFormat f{};
    const int B = (1 << (E - 1)) - 1;
    f.on = E < 8;
    f.bias = B;
    f.all_ones = (1 << E) - 1;
    f.lo = 128 - B;
    f.hi = 127 + B;
    f.off_u = (B - 127) / 2;                 // (B - 127) is even for E >= 2
    f.off_l = (B - 127) - f.off_u;
    uint32_t vb = (uint32_t)(127 + 127 - B) << 23, lb = E < 8 ? (uint32_t)(127 + B + 1) << 23 : 0x7F800000u;
    __builtin_memcpy(&f.vscale, &vb, 4);
    __builtin_memcpy(&f.lim, &lb, 4);
    return f;
}

// Bytes of a narrowed table as the LUT-GEMM kernels stage and read it: its
// 2^(2M) entries, then one row of 2^M zero entries, the row zero uniform
// operands index (kern::uniform_zero_row).
inline size_t gemm_table_bytes(const amsim_lut_s *L)
{
    return L->narrow_bytes + ((size_t)1 << L->M) * (size_t)(L->width_bits / 8);
}

namespace amsim {

// Maximum dynamic shared memory a CTA may use on sm_100-family parts.
constexpr int kMaxSmemPerCta = 227 * 1024;

int check_lut(amsim_lut_t lut);   // AMSIM_OK if usable on the current device
// Each translation unit with bounded device waits registers a reader of its
// wait-status word (OR its AMSIM_WAIT_* bits into *bits, clear when asked)
// and a writer of its flag-wait limit; both act on the current device.
using WaitStatusFn = int (*)(unsigned int *bits, int clear);
using WaitLimitFn = int (*)(long long ns);
bool register_wait_words(WaitStatusFn status, WaitLimitFn limit);
void count_launch();              // one kernel enqueued by the library
int cuda_status(cudaError_t e);   // maps to AMSIM_OK / AMSIM_ECUDA / AMSIM_ENOMEM
void set_last_path(int bits);     // the calling thread's amsim_last_path() value

// One GEMM operand in the kernel's terms: element (row r, reduction index k).
// Dense: value at ptr[batch*batch_stride + r*s_row + k*s_k].
// Gather (implicit im2col): k = (k2*kD1 + k1)*kD0 + k0 and r = (r2*rE1 + r1)*rE0 + r0
// contribute y = ry + ky, x = rx + kx, base = rb + kb (per-level linear coefficients);
// the value is ptr[base + (y/sy * IW + x/sx) * Cs] when y, x are divisible by
// sy, sx and in [0, IH*sy) x [0, IW*sx) after division, else a zero operand.
struct OperandDesc {
    const float *ptr;
    int64_t batch_stride;
    int rows;
    int gather;          // 0 dense, 1 gather
    int64_t s_row, s_k;  // dense strides
    // gather geometry
    int kD0, kD1;
    int kcy[3], kcx[3];
    int64_t kcb[3];
    int rE0, rE1;
    int rcy[3], rcx[3];
    int64_t rcb[3];
    int ry0, rx0;        // constant offsets added to the row part
    int IH, IW, Cs, sy, sx;
    int64_t extent;      // gather: elements of the source tensor (dense operands: computed by the planner)
};

// A convolution's operands read in place by the raw-tile TMA kernel (built in
// conv.cu): a tensor map over each caller tensor (dims[0] innermost, strides
// in bytes for dims 1.., 64-byte swizzle for boxes that arrive [row][k]).
struct TmaRawMap {
    const float *base;
    int rank;
    uint64_t dims[5], strides[4];
    uint32_t box[5];
    int swizzle64;
};
// Encode a tiled fp32 tensor map (zero fill out of bounds) into `map` (a
// CUtensorMap); AMSIM_EUNSUPPORTED when the driver refuses it.
int encode_tensor_map(::CUtensorMap_st *map, const TmaRawMap &m);
struct ConvRaw {
    // 1: the L tile is whole output rows of one image; a stage is one box of
    //    16 channels of the activation at the filter tap's offset (forward,
    //    data gradient); 2: the L tile is four 64-channel blocks of filter taps
    //    over 16 output pixels of one row (filter gradient)
    int mode;
    TmaRawMap umap, lmap;
    int u_kfast;     // the U box arrives [row][k]
    int u_tap;       // U box coordinates (step within the tap, row, tap): the data gradient's filter
    // box coordinates (see the raw-tile kernel's copy thread)
    int ch, S, tiles_img, rows_tile, ybase, ystep, xbase, xstep, N, P, Q, rows;
};

// A contraction as the kernels see it: out[u][l] = sum_k AMSim-product of the
// U operand's (u,k) and the L operand's (l,k) element, where the LUT index has
// the U element's mantissa in the high bits when `u_is_first` (the original
// first operand), else in the low bits (the kernel then reads the transposed
// table).  Output element (u,l) of batch b lives at c_ptr + b*c_bs + u*c_su + l*c_sl.
struct Problem {
    OperandDesc U, L;
    int K;               // reduction length
    int batch;
    bool u_is_first;
    float *c_ptr;
    int64_t c_bs, c_su, c_sl;
    float alpha, beta;
    const ConvRaw *conv = nullptr;  // convolution operands as tensor boxes, if they qualify
};

// Launch the LUT-GEMM for a problem.  ws may be null; the stream-K schedule
// (partial tiles in scratch) is used only if ws_bytes allows it.
int run_problem(const Problem &p, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream);
size_t problem_workspace(const Problem &p, amsim_lut_t lut);
// Up to ten independent problems in one launch (one LUT for all).
int run_problems(const Problem *p, int n, amsim_lut_t lut, void *ws, size_t ws_bytes, cudaStream_t stream);
size_t problems_workspace(const Problem *p, int n, amsim_lut_t lut);
// Ordered phases of problems in one launch (see amsim_gemm_phased); n <= kMaxProblems.
int run_phased(const Problem *p, int n, int nphase, const int *first, const int *after, amsim_lut_t lut, void *ws,
               size_t ws_bytes, cudaStream_t stream);
size_t phased_workspace(const Problem *p, int n, int nphase, const int *first, amsim_lut_t lut);
// The part of the above that the stream-K schedule alone needs.
size_t problems_workspace_streamk(const Problem *p, int n, amsim_lut_t lut);
// Workspace of a (batched) GEMM call: the fastest plan's, or the stream-K part only.
size_t gemm_workspace(char transA, char transB, int m, int n, int k, int batch, amsim_lut_t lut, bool streamk_only);

}  // namespace amsim
