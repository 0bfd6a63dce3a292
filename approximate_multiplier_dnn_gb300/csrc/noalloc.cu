// amsim_gemm_noalloc: the LUT-GEMM with its stream-K scratch in a fixed,
// file-scope device array instead of caller-provided memory.
//
// Some callers cannot allocate device memory when they call into the library:
// a serving loop that must not allocate after start-up (cudaMalloc can stall
// the device and can fail under memory pressure), a plugin host whose own
// allocator has claimed the memory budget, or an interface with nowhere to
// keep a workspace between calls.  This entry point needs no workspace from
// them and allocates nothing itself.
//
// The array below is reserved on every GPU that loads the library, for as long
// as the process lives.  Every call on a device shares it and leaves its
// contents behind; the kernels write each partial-sum slot before they read it,
// so nothing needs clearing between calls.  Calls that can overlap on the GPU
// (different streams without ordering) race on the array and must not be made.
#include <mutex>

#include "amsim_internal.h"

namespace {

constexpr size_t kScratchBytes = AMSIM_NOALLOC_SCRATCH_BYTES;   // stream-K slots for up to 159 SMs

static __device__ __align__(256) unsigned char amsim_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (with that device current).
int scratch_on_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return AMSIM_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return AMSIM_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, amsim_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return AMSIM_ECUDA;
        }
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return AMSIM_OK;
}

}  // namespace

extern "C" int amsim_gemm_noalloc(char transA, char transB, int m, int n, int k, float alpha, const float *A,
                                  int lda, const float *B, int ldb, float beta, float *C, int ldc,
                                  amsim_lut_t lut, amsim_stream_t stream)
{
    int rc = amsim::check_lut(lut);
    if (rc) return rc;
    // amsim_gemm plans for the array's size: operand planes that do not fit
    // are not used, and a stream-K plan whose partial sums do not fit (more
    // SMs than the array has slots for) gives way to the plan without them.
    void *scratch = nullptr;
    rc = scratch_on_current_device(&scratch);
    if (rc) return rc;
    return amsim_gemm(transA, transB, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, lut, scratch, kScratchBytes,
                      stream);
}
