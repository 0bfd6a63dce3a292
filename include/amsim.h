/*
 * amsim.h -- C ABI of the GB300 (sm_103a) library that simulates approximate
 * floating-point multipliers inside DNN contractions with a mantissa-product
 * lookup table, after "ApproxTrain: Fast Simulation of Approximate Multipliers
 * for DNN Training and Inference" (arXiv 2209.04161).
 *
 * Every scalar product a*b inside the contractions below is replaced by the
 * AMSim product of Sec. V-B, Algorithm 2:
 *   sign      = sign(a) XOR sign(b)
 *   index     = (top-M fraction bits of a) << M | (top-M fraction bits of b)
 *   entry     = LUT[index] = carry << 23 | 23-bit mantissa     (Sec. V-A, fn. 2)
 *   e0        = biased exp(a) + biased exp(b) - 127
 *   result    = signed zero      if e0 <= 0 or an input is zero,
 *               signed infinity  if e0 >= 255,
 *               sign | (e0 + carry) << 23 | mantissa   otherwise.
 * Readings of points the page leaves open (the design notes list them):
 *   denormal inputs count as zero; NaN in -> NaN; infinity times zero or a
 *   denormal -> NaN; infinity times anything else -> signed infinity; an
 *   exponent that reaches 255 through the carry -> signed infinity; the zero
 *   test precedes the carry adjustment.  Accumulation is IEEE fp32; alpha and
 *   beta are IEEE fp32 scalings, not simulated.
 *
 * Conventions for every call:
 *   - All tensors are fp32, dense, row-major (C order), owned by the caller.
 *     Pointers named "host_*" are host memory; all others are device memory
 *     of the device that was current when the LUT handle was built.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work: they do not synchronise, do not allocate device memory and
 *     do not copy to or from the host (the LUT build calls excepted).
 *   - `ws`/`ws_bytes` is optional caller-owned device scratch (256-byte
 *     aligned).  With less than the size the matching *_workspace_size query
 *     returns, a call still runs correctly with a plan that needs less
 *     scratch (possibly slower).  A call never reads scratch contents left by
 *     an earlier call; calls sharing one scratch buffer must be ordered on the
 *     GPU (same stream or events).
 *   - Return value: AMSIM_OK or an amsim_status code.  Arguments are checked
 *     on the host before anything is enqueued; on error nothing is enqueued
 *     and outputs are untouched.  A failed launch returns AMSIM_ECUDA.
 *     Kernels contain no device-side asserts or traps.  Every wait inside a
 *     kernel (for a copy, or for a flag another CTA raises) is bounded; a wait
 *     that gives up leaves that call's outputs wrong and is recorded on the
 *     device, where amsim_device_errors reads it (AMSIM_ETIMEOUT).
 *   - Results are deterministic: the same call on the same inputs with the
 *     same scratch size gives bit-identical outputs.
 */
#ifndef AMSIM_H
#define AMSIM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct amsim_lut_s *amsim_lut_t;  /* opaque; owns its device table */
typedef void *amsim_stream_t;             /* a cudaStream_t */

enum amsim_kind {
    AMSIM_EXACT = 0,     /* exact product of the M-bit-truncated mantissas: (1+x)(1+y) */
    AMSIM_MITCHELL = 1   /* Mitchell logarithmic multiplier: 1+x+y if x+y<1, else 2(x+y) */
};

enum amsim_status {
    AMSIM_OK = 0,
    AMSIM_EINVAL = 1,        /* bad argument (null pointer, negative size, bad stride, wrong device) */
    AMSIM_EUNSUPPORTED = 2,  /* M outside [1,11], unknown kind, a LUT entry outside carry 0/1 */
    AMSIM_ENOMEM = 3,        /* the LUT's device (or host) allocation failed */
    AMSIM_ECUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    AMSIM_ETIMEOUT = 5       /* a bounded device-side wait gave up (amsim_device_errors) */
};

/* Human-readable text for a status code (static storage). */
const char *amsim_status_string(int status);

/* Number of kernels this library has enqueued in the process so far (all
 * devices, all calls); a diagnostic for counting launches around a region. */
unsigned long long amsim_kernel_launches(void);

/* Kernel paths of the calling host thread's most recent GEMM or convolution
 * (ordinary or depthwise) call (a diagnostic; 0 before any, or when the call enqueued nothing): */
enum amsim_path {
    AMSIM_PATH_PLANES = 1,          /* operands decoded once into planes, copied by TMA */
    AMSIM_PATH_INKERNEL_DECODE = 4, /* operands decoded inside the warp-specialised GEMM */
    AMSIM_PATH_SINGLE_ROLE = 8,     /* the single-role fallback kernel */
    AMSIM_PATH_STREAMK = 16,        /* reduction split across CTAs (stream-K) */
    AMSIM_PATH_FIXUP = 32,          /* cut tiles finished by the separate fixup kernel */
    AMSIM_PATH_CONV_BOXES = 64,     /* convolution operands as shifted or blocked tensor boxes */
    AMSIM_PATH_RAW_TILES = 128,     /* operand tiles copied in place by TMA, decoded in shared memory */
    AMSIM_PATH_PHASED = 256,        /* every phase of amsim_gemm_phased in one launch */
    AMSIM_PATH_CLOSED_FORM = 512,   /* products computed in registers (amsim_lut_set_closed_form) */
    AMSIM_PATH_DW_TILES = 1024,     /* depthwise: halo tiles in shared memory, one channel per warp */
    AMSIM_PATH_DW_DIRECT = 2048,    /* depthwise: one lane per output element, operands read directly */
    AMSIM_PATH_WIDE_TILES = 4096    /* with AMSIM_PATH_PLANES: 128 x 256 tiles, eight lane columns per thread */
};
int amsim_last_path(void);

/*
 * Kinds of device-side waits (bits of amsim_device_errors' *flags):
 *   AMSIM_WAIT_COPY     a CTA waited for its own asynchronous copies or for
 *                       another warp of its CTA (limit 2 s);
 *   AMSIM_WAIT_PARTIAL  a CTA waited for another CTA's partial sums of a
 *                       tile split across CTAs (stream-K);
 *   AMSIM_WAIT_PHASE    a CTA of an amsim_gemm_phased launch waited for the
 *                       earlier phases its phase reads.
 * The last two wait on other CTAs of the same launch, with the limit that
 * amsim_set_flag_wait_limit sets (2 s by default).
 */
enum amsim_wait_bits { AMSIM_WAIT_COPY = 1, AMSIM_WAIT_PARTIAL = 2, AMSIM_WAIT_PHASE = 4 };

/*
 * Which bounded waits of the library's kernels have given up on the current
 * device since the last clear: synchronises the device (so every call enqueued
 * before it has finished), ORs the AMSIM_WAIT_* bits of every kernel family
 * into *flags, and clears them when `clear` is nonzero.  A set bit means some
 * call since the last clear produced wrong outputs (its kernels still ran to
 * their end and the context stays usable).  Returns AMSIM_OK when no wait gave
 * up, AMSIM_ETIMEOUT when one did, AMSIM_EINVAL for a null `flags`,
 * AMSIM_ECUDA when the device cannot be read.  Not for use during stream
 * capture.  The paper has no counterpart; it is the library's error report.
 */
int amsim_device_errors(unsigned int *flags, int clear);

/*
 * Limit, in nanoseconds, of the device-side waits on flags that other CTAs of
 * the same launch raise (AMSIM_WAIT_PARTIAL, AMSIM_WAIT_PHASE), for launches
 * enqueued after the call on the current device; 0 <= ns <= 10 s, default
 * 2 s.  Those waits normally last microseconds; a watchdog that wants a hung
 * launch reported sooner can lower it (0 gives up at the first flag not yet
 * raised, which is how the tests provoke a timeout).  Copy waits keep 2 s.
 * Synchronising; not for use during stream capture.  Errors: AMSIM_EINVAL
 * for ns outside the range, AMSIM_ECUDA.  The paper has no counterpart.
 */
int amsim_set_flag_wait_limit(long long ns);

/*
 * Cooperative launches on (1, the default) or off (0), for calls made after
 * it from any thread.  On: a stream-K GEMM finishes the tiles it cuts between
 * CTAs inside its own (cooperative) launch, and amsim_gemm_phased runs all of
 * its phases in one launch.  Off: cut tiles are finished by a second kernel,
 * the fixup kernel, which adds the same partial sums in the same CTA order,
 * so the results are bit-identical (AMSIM_PATH_FIXUP in amsim_last_path); and
 * a phased call runs its phases as consecutive grouped launches.  For hosts
 * where a launch must not hold every SM until all its CTAs are resident (a
 * context shared with other work).  A cooperative launch the driver refuses
 * takes the same route on its own.  Errors: AMSIM_EINVAL for a value other
 * than 0 or 1.  The paper has no counterpart.
 */
int amsim_set_cooperative_launches(int on);

/* ------------------------------------------------------------------ LUTs */

/*
 * Algorithm 1 (Sec. V-A) on the host: for every mantissa pair (p, q) in
 * [0,2^M)^2, form A = 1.p and B = 1.q with non-special exponents, multiply them
 * with the closed-form model of `kind`, compare the product's exponent with the
 * unnormalised one to find the carry, and store carry << 23 | mantissa at
 * index p << M | q.  `host_entries` receives 2^(2M) uint32 values (4 B each, as
 * fn. 2 prescribes: M=7 -> 65,536 B, M=11 -> 16,777,216 B).  No device work.
 * Errors: AMSIM_EUNSUPPORTED for M outside [1,11] or an unknown kind,
 * AMSIM_EINVAL for a null pointer.
 */
int amsim_lut_generate(int kind, int M, uint32_t *host_entries);

/*
 * Algorithm 1 with a user-supplied multiplier model `approx_mul` (the "C/C++
 * approximate multiplication function" of Sec. V-A / Fig. 7).  The function is
 * called with normal operands in [1,2) and must return a positive normal
 * product in [1,4).  An entry whose exponent moves by anything but 0 or +1
 * yields AMSIM_EUNSUPPORTED.  Host only.
 */
typedef float (*amsim_approx_mul_fn)(float a, float b);
int amsim_lut_generate_from_fn(amsim_approx_mul_fn approx_mul, int M, uint32_t *host_entries);

/*
 * Build a device-resident LUT handle on the current device from Algorithm 1
 * for `kind` (host generation + one synchronous upload; call once, outside any
 * timed or captured region).  The handle keeps the canonical 4-byte entries and
 * a losslessly narrowed copy (8, 16 or 32 bits per entry, whichever is the
 * narrowest that holds every entry exactly) in both index orders, which the
 * contraction kernels stage in shared memory when it fits.
 */
int amsim_lut_build(int kind, int M, amsim_lut_t *out);

/*
 * Same as amsim_lut_build for an arbitrary table of 2^(2M) canonical entries
 * (carry << 23 | mantissa, carry in {0,1}), e.g. produced by
 * amsim_lut_generate_from_fn or loaded from a file at run time (Sec. VI, Fig. 5:
 * generated tables are handed to the operator library when the program
 * runs, not compiled into it).  The table need
 * not be symmetric.  Errors: AMSIM_EUNSUPPORTED if an entry has bits above 23.
 */
int amsim_lut_build_from_entries(const uint32_t *host_entries, int M, amsim_lut_t *out);

/*
 * Algorithm 1 over a user's approx_mul and the device upload in one call: the
 * page's flow in which the designer writes the multiplier as a C/C++ function
 * and its generated table is handed to the operator library when the program
 * runs (Sec. V-A, Algorithm 1; Sec. VI, Figs. 5 and 7).
 * Equivalent to amsim_lut_generate_from_fn followed by
 * amsim_lut_build_from_entries: `approx_mul` is called 2^(2M) times on the
 * host, with normal operands 1.p and 1.q in [1,2), and must return a positive
 * normal product in [1,4).  The handle belongs to the current device.
 * Errors: AMSIM_EINVAL for a null function or output, AMSIM_EUNSUPPORTED for
 * M outside [1,11] or a product whose exponent moves by anything but 0 or +1
 * (or that is negative), AMSIM_ENOMEM / AMSIM_ECUDA from the upload.
 */
int amsim_lut_build_from_fn(amsim_approx_mul_fn approx_mul, int M, amsim_lut_t *out);

/* Copy the 2^(2M) canonical entries of a handle back to host memory (synchronous). */
int amsim_lut_entries(amsim_lut_t lut, uint32_t *host_dst);

/* M, narrowed entry width in bits, and the left shift that restores an entry. */
int amsim_lut_info(amsim_lut_t lut, int *M, int *width_bits, int *shift);

/*
 * Closed-form products for a handle built by amsim_lut_build (on != 0), or
 * the table again (on == 0).  With it on, GEMM and convolution launches that
 * take the raw-tile kernel (AMSIM_PATH_RAW_TILES, including phased launches)
 * compute each product's mantissa factor in registers instead of reading the
 * table -- the direct simulation the ApproxTrain page compares its LUT with
 * (Sec. VII, Fig. 6):
 *   AMSIM_MITCHELL: the fp32 whose bits are 1.0f + (qa + qb) << (23 - M),
 *                   qa, qb the operands' truncated M-bit fractions (the sum's
 *                   carry into the exponent is Mitchell's 2(x+y) branch);
 *   AMSIM_EXACT:    (1 + qa/2^M) * (1 + qb/2^M) rounded to fp32 (exact, M <= 11).
 * Both equal the table's entries bit for bit, so results are identical to the
 * table's for the same plan.  Depthwise launches on the tiled kernels
 * (AMSIM_PATH_DW_TILES: 3x3 at stride 1 or 2, 5x5 at stride 1) use them too;
 * launches on other kernel paths keep reading the table.  Such launches add AMSIM_PATH_CLOSED_FORM to the path bits.  The
 * setting belongs to the handle: calls enqueued after it changes see the new
 * setting.  Errors: AMSIM_EINVAL for a null handle; AMSIM_EUNSUPPORTED when
 * on != 0 and the handle was built from entries or a function, or simulates
 * an exponent narrower than 8 bits (amsim_lut_set_exponent_bits).
 */
int amsim_lut_set_closed_form(amsim_lut_t lut, int on);

/*
 * The exponent width E of the simulated (1, E, M) multiplier (Sec. V-B, last
 * paragraph: E from 1 to 8 with an exponent casting function); 8, the
 * default, is fp32's own exponent.  Casting function taken for E < 8 (IEEE
 * convention, bias B = 2^(E-1) - 1, biased exponent 0 = zero, 2^E - 1 =
 * Inf/NaN): an fp32 operand's exponent is re-biased to B; an operand below
 * the format's smallest normal 2^(1-B) becomes a signed zero and one of
 * magnitude 2^(B+1) or more a signed infinity; Algorithm 2 runs with bias B
 * (zero when eA + eB - B <= 0, infinity when it or the carried exponent
 * reaches 2^E - 1); the product returns as fp32 (exact: B + 1 <= 64) and
 * accumulation stays fp32.  E = 1 leaves no normal magnitudes: |x| < 2
 * casts to zero and |x| >= 2 to infinity.  The setting belongs to the
 * handle and applies to every call enqueued after it: elementwise products,
 * GEMMs (all variants; phased calls then run phase by phase), Conv2D and
 * depthwise Conv2D.  Such calls run on the in-kernel-decode GEMM kernels and
 * the direct depthwise kernel, with every product rounded before it is
 * added (AMSIM_PATH_INKERNEL_DECODE or AMSIM_PATH_SINGLE_ROLE, or
 * AMSIM_PATH_DW_DIRECT).  Errors: AMSIM_EINVAL for a null handle,
 * AMSIM_EUNSUPPORTED for E outside [1,8] or E < 8 on a handle with closed
 * forms on (amsim_lut_set_closed_form then also refuses while E < 8).
 */
int amsim_lut_set_exponent_bits(amsim_lut_t lut, int E);

/* Free the handle's device memory.  NULL is ignored. */
void amsim_lut_destroy(amsim_lut_t lut);

/* ------------------------------------------------------------------ elementwise */

/*
 * c[i] = AMSim(a[i], b[i]) for i < n (Sec. V-B, Algorithm 2), bit-exact, NaN
 * results canonical (0x7FC00000).  a, b, c: device fp32 arrays of n elements;
 * c may alias a or b.  n == 0 is a no-op.
 */
int amsim_mul(const float *a, const float *b, float *c, int64_t n, amsim_lut_t lut,
              amsim_stream_t stream);

/* ------------------------------------------------------------------ GEMM */

/*
 * C = alpha * op(A) op(B) + beta * C with every product an AMSim product whose
 * first operand (high LUT index bits) is the element of A (Sec. VI-D, "GEMM
 * kernel"; Sec. VI-C AMDENSE forward and gradients).  Row-major:
 *   op(A) is m x k: A is m x k (lda >= k) for transA 'N', k x m (lda >= m) for 'T';
 *   op(B) is k x n: B is k x n (ldb >= n) for transB 'N', n x k (ldb >= k) for 'T';
 *   C is m x n with ldc >= n.
 * beta == 0 does not read C.  m, n or k == 0 is allowed (k == 0 gives beta*C).
 * Scratch: see amsim_gemm_workspace_size.
 */
int amsim_gemm(char transA, char transB, int m, int n, int k, float alpha,
               const float *A, int lda, const float *B, int ldb, float beta,
               float *C, int ldc, amsim_lut_t lut, void *ws, size_t ws_bytes,
               amsim_stream_t stream);

/*
 * `batch` independent GEMMs as above; problem i uses A + i*strideA,
 * B + i*strideB, C + i*strideC (element strides, >= 0).  Used for the two
 * contractions of attention (S = Q K^T with transB 'T', O = P V).
 */
int amsim_gemm_strided_batched(char transA, char transB, int m, int n, int k, float alpha,
                               const float *A, int lda, int64_t strideA,
                               const float *B, int ldb, int64_t strideB, float beta,
                               float *C, int ldc, int64_t strideC, int batch,
                               amsim_lut_t lut, void *ws, size_t ws_bytes,
                               amsim_stream_t stream);

/*
 * Bytes of scratch with which the GEMM calls above run their fastest plan:
 * the split-K (stream-K) partial sums, when the problem needs them, plus the
 * operands decoded once into LUT-offset and scale planes, when the plan uses
 * them (4 bytes per operand element for tables that fit shared memory, 8 for
 * larger ones; per batch unless the batch stride is 0).  Less scratch selects
 * a plan that decodes operands inside the GEMM; none selects one without
 * split-K.  All plans give results within the contraction tolerance; a
 * given scratch size always gives the same plan.
 */
size_t amsim_gemm_workspace_size(char transA, char transB, int m, int n, int k, int batch,
                                 amsim_lut_t lut);

/*
 * One GEMM of a group: the arguments of amsim_gemm_strided_batched as a struct
 * (element strides; transA/transB 'N' or 'T').
 */
typedef struct amsim_gemm_problem {
    const float *A;
    const float *B;
    float *C;
    int64_t strideA, strideB, strideC;
    int m, n, k, lda, ldb, ldc, batch;
    float alpha, beta;
    char transA, transB;
} amsim_gemm_problem;

/*
 * `count` independent GEMMs sharing one LUT, scheduled together so that the
 * work of all of them is spread evenly over the SMs (up to ten per launch;
 * larger groups run as consecutive launches).  This is how a Dense layer's
 * forward and both gradients (Sec. VI-C) -- or the independent contractions of
 * several layers -- fill the GPU when each alone is too small.  No problem may
 * read another's output or write memory another touches.  `problems` is host
 * memory, read during the call.  Results equal the separate amsim_gemm calls'
 * up to fp32 summation order.
 */
int amsim_gemm_grouped(int count, const amsim_gemm_problem *problems, amsim_lut_t lut, void *ws,
                       size_t ws_bytes, amsim_stream_t stream);

/* Bytes of scratch with which amsim_gemm_grouped runs its fastest plan. */
size_t amsim_gemm_grouped_workspace_size(int count, const amsim_gemm_problem *problems, amsim_lut_t lut);

/*
 * Ordered phases of GEMMs sharing one LUT -- for example the forward and
 * backward contractions of a stack of Dense layers (Sec. VI-C), where a
 * layer's forward GEMM reads the previous layer's output.  Problems
 * problems[phase_first[ph]] .. problems[phase_first[ph + 1] - 1] form phase ph
 * (the last phase ends at `count`); phase_first[0] == 0 and phase_first is
 * non-decreasing (a phase may be empty).  The result equals that of
 * amsim_gemm_grouped called on each phase in turn on `stream`, up to fp32
 * summation order, provided that:
 *   - phase ph reads (as A or B) outputs of phases 0 .. phase_after[ph] - 1
 *     only, 0 <= phase_after[ph] <= ph;
 *   - no problem's C is read or written by any other problem of the call
 *     except as just allowed (in particular, C with beta != 0 is not another
 *     problem's output);
 *   - within a phase, the rules of amsim_gemm_grouped hold.
 * Phases that need nothing of the phase just before them let the SMs carry
 * straight on from one phase to the next: with up to ten problems, six
 * phases, operands the raw-tile path reads, one LUT orientation, a LUT that
 * fits shared memory and at least amsim_gemm_phased_workspace_size bytes of
 * 256-byte-aligned scratch, every phase runs in one cooperative launch
 * (AMSIM_PATH_PHASED): each SM takes a share of every phase in order and
 * waits, before it loads a phase's operands, until every SM has finished
 * phases 0 .. phase_after[ph] - 1.  A tile that the shares cut is finished by
 * the last of its parts to arrive, which adds every part's partial sum (kept
 * in scratch) in the parts' order, so repeated calls give identical bits.
 * Otherwise the phases run as consecutive grouped launches.  Host arrays are
 * read during the call.
 * Errors: AMSIM_EINVAL for an invalid phase layout or problem, as
 * amsim_gemm_grouped otherwise.
 */
int amsim_gemm_phased(int count, const amsim_gemm_problem *problems, int nphase, const int *phase_first,
                      const int *phase_after, amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream);

/* Bytes of scratch with which amsim_gemm_phased runs its fastest plan (0 for
 * an invalid phase layout). */
size_t amsim_gemm_phased_workspace_size(int count, const amsim_gemm_problem *problems, int nphase,
                                        const int *phase_first, const int *phase_after, amsim_lut_t lut);

/*
 * amsim_gemm without a workspace argument and without any allocation: for
 * callers that cannot allocate device memory at call time -- a serving loop
 * that must not allocate after start-up (cudaMalloc can stall the device and
 * can fail under memory pressure), a plugin host whose own allocator holds the
 * memory budget, or an interface with nowhere to keep a workspace.  The ApproxTrain
 * page has no counterpart; this is a library convenience.
 *
 * Same arguments and results as amsim_gemm.  The stream-K partial sums go to a
 * fixed device array of AMSIM_NOALLOC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library reserves until the process exits.  The
 * first call on a device looks up that array's address (cudaGetSymbolAddress)
 * with the device current; make that first call before any stream capture.
 * All calls on a device share the array and leave their partial sums in it;
 * nothing needs clearing between calls, but calls that may overlap on the GPU
 * (unordered streams) race on it and must not be made.  The array holds the
 * stream-K partial sums of one wave on up to 159 SMs; on a larger device the
 * plan amsim_gemm picks for a workspace of that size is used instead (a
 * multi-wave problem then runs without stream-K).  Errors as amsim_gemm.
 */
#define AMSIM_NOALLOC_SCRATCH_BYTES ((size_t)20 << 20)
int amsim_gemm_noalloc(char transA, char transB, int m, int n, int k, float alpha,
                       const float *A, int lda, const float *B, int ldb, float beta,
                       float *C, int ldc, amsim_lut_t lut, amsim_stream_t stream);

/* ------------------------------------------------------------------ Conv2D */

/*
 * Convolution geometry.  Activations are NHWC, filters RSCK (TF's HWIO, the
 * layout of the TensorFlow ops ApproxTrain replaces), outputs NPQK with
 *   P = (H + 2 pad_h - dil_h (R-1) - 1) / stride_h + 1, Q likewise.
 * The operation is cross-correlation; padded taps are zero operands.
 */
typedef struct amsim_conv_desc {
    int N, H, W, C;     /* input batch, height, width, channels */
    int K, R, S;        /* output channels, filter height, filter width */
    int stride_h, stride_w, pad_h, pad_w, dil_h, dil_w;
} amsim_conv_desc;

/* Output height/width of a descriptor; AMSIM_EINVAL if the geometry is empty. */
int amsim_conv2d_out_hw(const amsim_conv_desc *desc, int *P, int *Q);

/*
 * Forward (Sec. VI-B, Algorithm 3, Fig. 8a, IM2COL + GEMM, here an implicit
 * GEMM with the im2col addressing fused into the operand loads):
 *   y[n,p,q,k] = sum_{r,s,c} AMSim(x[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c], w[r,s,c,k]).
 * x: N*H*W*C, w: R*S*C*K, y: N*P*Q*K (written, not accumulated).
 */
int amsim_conv2d_fwd(const amsim_conv_desc *desc, const float *x, const float *w, float *y,
                     amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream);

/*
 * Preceding-layer gradient (Algorithm 4 lines 6-8: IM2COL_PLG over the
 * padded-dilated errors and TransposeAndReverse of the filter, here folded into
 * the operand addressing):
 *   dx[n,h,w,c] = sum_{r,s,k} AMSim(dy[n,p,q,k], w[r,s,c,k]),
 *   p = (h + ph - r*dh)/sh, q = (w + pw - s*dw)/sw where integral and in range.
 * dy: N*P*Q*K, w: R*S*C*K, dx: N*H*W*C (written).
 */
int amsim_conv2d_bwd_data(const amsim_conv_desc *desc, const float *dy, const float *w, float *dx,
                          amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream);

/*
 * Weight gradient (Algorithm 4 lines 4-5: IM2COL_Weight + GEMM):
 *   dw[r,s,c,k] = sum_{n,p,q} AMSim(x[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c], dy[n,p,q,k]).
 * x: N*H*W*C, dy: N*P*Q*K, dw: R*S*C*K (written).  The long reduction over
 * N*P*Q is split across CTAs when scratch allows, reduced in a fixed order.
 */
int amsim_conv2d_bwd_filter(const amsim_conv_desc *desc, const float *x, const float *dy, float *dw,
                            amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream);

/*
 * which: 0 forward, 1 bwd_data, 2 bwd_filter.  Bytes of scratch for the
 * fastest plan: the split-K (stream-K) partial sums (unit-stride passes copy
 * their operands as tensor boxes and others gather them inside the GEMM, so
 * no operand planes are kept; a 1x1 filter at stride 1 without padding is a
 * plain GEMM and may also take planes, as amsim_gemm_workspace_size says).
 * Less scratch selects a plan without split-K.
 */
size_t amsim_conv2d_workspace_size(const amsim_conv_desc *desc, int which, amsim_lut_t lut);

/* ------------------------------------------------------------------ depthwise Conv2D */

/*
 * Depthwise convolution (Sec. III, Table I: depthwise Conv2D is one of the
 * layer types ApproxTrain simulates), every product an AMSim product, fp32
 * accumulation.  The descriptor is the Conv2D one with K = C * D output
 * channels for a channel multiplier D >= 1 (K not a multiple of C is
 * AMSIM_EINVAL).  The filter is w[r][s][c][d] (R*S*C*D floats, TF's
 * depthwise HWC-multiplier layout) and output channel k = c*D + d reads input
 * channel c only:
 *   y[n,p,q,c*D+d] = sum_{r,s} AMSim(x[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c], w[r,s,c,d]).
 * x: N*H*W*C, w: R*S*C*D, y: N*P*Q*K (written).  Padded taps are zero
 * operands.  3x3 filters with unit dilation at stride 1 or 2 and 5x5 filters
 * at stride 1, D = 1, C a multiple of 4, 16-byte aligned x and y and an 8- or
 * 16-bit narrowed LUT of at most 64 KB take a tiled kernel
 * (AMSIM_PATH_DW_TILES); everything else the direct kernel
 * (AMSIM_PATH_DW_DIRECT).  Scratch is not used.
 */
int amsim_dwconv2d_fwd(const amsim_conv_desc *desc, const float *x, const float *w, float *y,
                       amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream);

/*
 * Preceding-layer gradient of the depthwise convolution (Algorithm 4's
 * IM2COL_PLG / TransposeAndReverse reading, per channel):
 *   dx[n,h,w,c] = sum_{r,s,d} AMSim(dy[n,p,q,c*D+d], w[r,s,c,d]),
 *   p = (h + ph - r*dh)/sh, q = (w + pw - s*dw)/sw where integral and in range
 *   (zero operands elsewhere).
 * dy: N*P*Q*K, w: R*S*C*D, dx: N*H*W*C (written).  Kernel choice as for the
 * forward pass (dy and dx 16-byte aligned), at stride 2 for padding 1 only.
 * Scratch is not used.
 */
int amsim_dwconv2d_bwd_data(const amsim_conv_desc *desc, const float *dy, const float *w, float *dx,
                            amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream);

/*
 * Weight gradient of the depthwise convolution:
 *   dw[r,s,c,d] = sum_{n,p,q} AMSim(x[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c], dy[n,p,q,c*D+d]).
 * x: N*H*W*C, dy: N*P*Q*K, dw: R*S*C*D (written; all +0 when N == 0).  The
 * reduction over N*P*Q is split into shares when scratch allows
 * (amsim_dwconv2d_workspace_size), whose partial sums a second kernel adds in
 * share order (AMSIM_PATH_STREAMK is then set); without scratch one share per
 * channel block runs, more slowly.  Results are deterministic for a given
 * scratch size.  Kernel choice as for the forward pass (x and dy 16-byte
 * aligned).
 */
int amsim_dwconv2d_bwd_filter(const amsim_conv_desc *desc, const float *x, const float *dy, float *dw,
                              amsim_lut_t lut, void *ws, size_t ws_bytes, amsim_stream_t stream);

/*
 * which: 0 forward, 1 bwd_data, 2 bwd_filter.  Bytes of scratch with which the
 * call splits its reduction over every SM (0 for the first two passes, and
 * for an invalid descriptor).
 */
size_t amsim_dwconv2d_workspace_size(const amsim_conv_desc *desc, int which, amsim_lut_t lut);

/* ------------------------------------------------------------------ glue */

/*
 * Exact fp32 row softmax P[r,:] = exp(S[r,:] - max) / sum(...) for `rows` rows of
 * `cols` contiguous values (ld = cols).  Not simulated: attention's softmax
 * sits between its two approximate contractions.  P may alias S.
 */
int amsim_softmax_rows(const float *S, float *P, int64_t rows, int cols, amsim_stream_t stream);

/*
 * Gradient of amsim_softmax_rows: dS[r,c] = P[r,c] * (dP[r,c] - sum_j P[r,j] dP[r,j])
 * for `rows` rows of `cols` contiguous values, in exact fp32 (the backward of
 * attention's softmax, between its approximate gradient contractions).  dS may
 * alias dP.  Device pointers; asynchronous on `stream`.
 */
int amsim_softmax_rows_backward(const float *P, const float *dP, float *dS, int64_t rows, int cols,
                                amsim_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AMSIM_H */
