// Operand predecode pass of the TMA-fed LUT-GEMM (internal).
//
// Each job turns one operand into planes laid out [b][plane][k][row] with a
// row pitch of rows_pad words: two planes, or one of packed words.  Element (b, r, k) of the operand is
//   src[b*bs + (r / rdiv)*s_rhi + (r % rdiv + roff)*s_row + (k / kdiv)*s_khi + (k % kdiv)*s_k]
// and reads as zero when r % rdiv + roff falls outside [0, rlim) -- a dense
// matrix (rdiv = rows, kdiv = K), a filter read with its channel axes
// swapped, or an activation shifted along its width for one filter column.
// Plane 0 holds the byte offset of the
// element's LUT row (U operands) or column (L operands), plane 1 its signed
// power-of-two scale (ApproxTrain Sec. V-B Algorithm 2: the operand half of
// the product -- sign, biased exponent, top-M fraction bits, with denormals
// as zero and NaN kept); a packed job writes both in one word per element
// (pack_operand: offset << 10 | the scale's top ten bits).  Zero and denormal
// elements of a uniform (U) operand take the table's zero row (zero_off; 0
// for lane operands).  A job raises *flag to the launch epoch when an element
// has |x| >= 2^64, the magnitude above which a product may overflow, and
// *flag_small when one has 0 < |x| < 2^-63 (a product may meet Algorithm 2's
// zero test): a plane with neither holds only zeros and magnitudes in
// [2^-63, 2^64).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace amsim {
namespace kern {

constexpr int kMaxDecodeJobs = 20;
constexpr int kDecodeTileR = 64;                 // rows per tile
constexpr int kDecodeTileK = 64;                 // reduction steps per tile

struct DecodeJob {
    const float *src;
    long long bs, s_row, s_k;                    // element strides
    long long s_rhi, s_khi;                      // strides of r / rdiv and k / kdiv
    int rdiv, roff, rlim, kdiv;
    int rows, K, batch;                          // batch: planes written (1 for a broadcast operand)
    int rows_pad;                                // row pitch of a plane, multiple of 4
    int offshift;                                // offset = top-M fraction bits << offshift
    int packed;                                  // one plane of packed words (offsets below 2^22)
    uint32_t *plane;                             // [batch][packed ? 1 : 2][K][rows_pad]
    unsigned long long *flag, *flag_small;
    uint32_t zero_off;                           // U planes: the zero row's byte offset; L planes: 0
    int tiles_r, tiles_k;                        // 64 x 64 tiles per batch
    // row-fast: a dense operand with unit row stride (read and written along
    // rows); vec: 16-byte loads of 4 consecutive rows (row-fast) or steps
    // (otherwise) start aligned wherever they lie inside the operand
    int rowfast, vec;
    long long tile0;                             // first tile of this job in the launch
};

struct DecodeParams {
    DecodeJob job[kMaxDecodeJobs];
    int njobs;
    long long tiles;
    int M;
    unsigned long long epoch;
};

// Enqueue the predecode of all jobs (programmatic dependent launch: the kernel
// waits for the previous launch on the stream before reading any source).
int launch_predecode(const DecodeParams &p, int sms, cudaStream_t st);

}  // namespace kern
}  // namespace amsim
