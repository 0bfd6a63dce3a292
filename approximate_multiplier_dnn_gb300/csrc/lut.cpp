// Mantissa-product LUT: host generation (ApproxTrain Sec. V-A, Algorithm 1),
// lossless narrowing, device upload, and the handle's ABI entry points.
#include <cmath>
#include <new>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <vector>

#include "amsim_internal.h"

namespace {

uint32_t bits_of(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
float float_of(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// Closed-form multiplier models evaluated on operands 1.p and 1.q (M fraction
// bits each), returning the fp32 product.  exact: (1+x)(1+y) with at most
// 2M+2 <= 24 significant bits, so the fp32 result is exact.  mitchell:
// 1+x+y below 2, else 2(x+y) (Mitchell's log-add-antilog), also exact.
float model_exact(float a, float b) { return a * b; }

float model_mitchell(float a, float b)
{
    // a, b in [1,2): x = a-1, y = b-1 are exact in fp32.
    float x = a - 1.0f, y = b - 1.0f;
    float s = x + y;                  // exact: both have <= 11 fraction bits
    return s < 1.0f ? 1.0f + s : 2.0f * s;
}

// Algorithm 1 for a generic model: fix the operands' biased exponent at 127,
// fill the mantissas from the loop indices, compare exponents for the carry.
int generate(amsim_approx_mul_fn fn, int M, uint32_t *out)
{
    if (M < 1 || M > 11) return AMSIM_EUNSUPPORTED;
    if (!fn || !out) return AMSIM_EINVAL;
    const uint32_t n = 1u << M;
    const int unnormalised_exp = 127 + 127 - 127;
    for (uint32_t p = 0; p < n; ++p) {
        float A = float_of((127u << 23) | (p << (23 - M)));
        for (uint32_t q = 0; q < n; ++q) {
            float B = float_of((127u << 23) | (q << (23 - M)));
            uint32_t c = bits_of(fn(A, B));
            int e = (int)((c >> 23) & 0xFF);
            if (c >> 31) return AMSIM_EUNSUPPORTED;
            int carry = e - unnormalised_exp;
            if (carry != 0 && carry != 1) return AMSIM_EUNSUPPORTED;
            out[(p << M) | q] = ((uint32_t)carry << 23) | (c & 0x7FFFFFu);
        }
    }
    return AMSIM_OK;
}

// Narrowest lossless width.  Entries are < 2^24 (carry bit 23 + mantissa), so
// 8-bit storage holds bits 16..23 and 16-bit storage bits 8..23: a table
// narrows when every entry's bits below that are zero (Mitchell for M <= 7
// and exact for M <= 3 fit 8 bits; exact for M <= 7 fits 16 bits).  The
// fixed shifts let the kernels rebuild an entry with a constant shift.
void choose_width(const uint32_t *e, size_t n, int *width, int *shift)
{
    uint32_t all_or = 0;
    for (size_t i = 0; i < n; ++i) all_or |= e[i];
    if ((all_or & 0xFFFFu) == 0) { *width = 8; *shift = 16; return; }
    if ((all_or & 0xFFu) == 0) { *width = 16; *shift = 8; return; }
    *width = 32; *shift = 0;
}

void narrow_into(const uint32_t *e, int M, int width, int shift, bool transpose, void *dst)
{
    const uint32_t n = 1u << M;
    for (uint32_t r = 0; r < n; ++r)
        for (uint32_t c = 0; c < n; ++c) {
            uint32_t v = transpose ? e[(c << M) | r] : e[(r << M) | c];
            v >>= shift;
            size_t i = ((size_t)r << M) | c;
            if (width == 8) static_cast<uint8_t *>(dst)[i] = (uint8_t)v;
            else if (width == 16) static_cast<uint16_t *>(dst)[i] = (uint16_t)v;
            else static_cast<uint32_t *>(dst)[i] = v;
        }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int build_from_entries(const uint32_t *entries, int M, amsim_lut_t *out)
{
    if (!entries || !out) return AMSIM_EINVAL;
    if (M < 1 || M > 11) return AMSIM_EUNSUPPORTED;
    const size_t n = size_t(1) << (2 * M);
    for (size_t i = 0; i < n; ++i)
        if (entries[i] >> 24) return AMSIM_EUNSUPPORTED;
    int width, shift;
    choose_width(entries, n, &width, &shift);
    bool symmetric = true;
    const uint32_t side = 1u << M;
    for (uint32_t r = 0; r < side && symmetric; ++r)
        for (uint32_t c = r + 1; c < side; ++c)
            if (entries[(r << M) | c] != entries[(c << M) | r]) { symmetric = false; break; }

    const size_t canon_bytes = n * 4;
    const size_t narrow_bytes = n * (width / 8);
    // each narrowed copy is followed by a row of zero entries (the host buffer
    // is zero-filled), which zero uniform operands index in the GEMM kernels
    const size_t zero_row = side * (width / 8);
    const size_t off_narrow = align256(canon_bytes);
    const size_t off_narrow_t = align256(off_narrow + narrow_bytes + zero_row);
    const size_t total = symmetric ? off_narrow_t : align256(off_narrow_t + narrow_bytes + zero_row);

    std::vector<uint8_t> host(total, 0);
    std::memcpy(host.data(), entries, canon_bytes);
    narrow_into(entries, M, width, shift, false, host.data() + off_narrow);
    if (!symmetric) narrow_into(entries, M, width, shift, true, host.data() + off_narrow_t);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AMSIM_ECUDA;
    void *d = nullptr;
    cudaError_t err = cudaMalloc(&d, total);
    if (err != cudaSuccess) { cudaGetLastError(); return AMSIM_ENOMEM; }
    err = cudaMemcpy(d, host.data(), total, cudaMemcpyHostToDevice);
    if (err != cudaSuccess) { cudaFree(d); return AMSIM_ECUDA; }

    amsim_lut_s *L = new (std::nothrow) amsim_lut_s();
    if (!L) { cudaFree(d); return AMSIM_ENOMEM; }
    L->M = M;
    L->device = dev;
    L->width_bits = width;
    L->shift = shift;
    L->symmetric = symmetric;
    L->d_base = d;
    L->d_canon = static_cast<const uint32_t *>(d);
    L->d_narrow = static_cast<const uint8_t *>(d) + off_narrow;
    L->d_narrow_t = symmetric ? L->d_narrow : static_cast<const uint8_t *>(d) + off_narrow_t;
    L->narrow_bytes = narrow_bytes;
    *out = L;
    return AMSIM_OK;
}

}  // namespace

namespace amsim {

namespace {
std::atomic<unsigned long long> g_launches{0};
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return AMSIM_OK;
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? AMSIM_ENOMEM : AMSIM_ECUDA;
}

int check_lut(amsim_lut_t lut)
{
    if (!lut || !lut->d_base) return AMSIM_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return AMSIM_ECUDA;
    return dev == lut->device ? AMSIM_OK : AMSIM_EINVAL;
}

}  // namespace amsim

extern "C" {

const char *amsim_status_string(int status)
{
    switch (status) {
    case AMSIM_OK: return "ok";
    case AMSIM_EINVAL: return "invalid argument";
    case AMSIM_EUNSUPPORTED: return "unsupported mantissa width, kind or LUT entry";
    case AMSIM_ENOMEM: return "out of memory";
    case AMSIM_ECUDA: return "CUDA runtime error";
    case AMSIM_ETIMEOUT: return "a device-side wait gave up (outputs of some call are wrong)";
    default: return "unknown status";
    }
}

int amsim_lut_generate(int kind, int M, uint32_t *host_entries)
{
    if (kind == AMSIM_EXACT) return generate(model_exact, M, host_entries);
    if (kind == AMSIM_MITCHELL) return generate(model_mitchell, M, host_entries);
    return AMSIM_EUNSUPPORTED;
}

int amsim_lut_generate_from_fn(amsim_approx_mul_fn approx_mul, int M, uint32_t *host_entries)
{
    return generate(approx_mul, M, host_entries);
}

int amsim_lut_build(int kind, int M, amsim_lut_t *out)
{
    if (!out) return AMSIM_EINVAL;
    if (M < 1 || M > 11) return AMSIM_EUNSUPPORTED;
    std::vector<uint32_t> e(size_t(1) << (2 * M));
    int rc = amsim_lut_generate(kind, M, e.data());
    if (rc) return rc;
    rc = build_from_entries(e.data(), M, out);
    if (rc == AMSIM_OK) (*out)->kind = kind;
    return rc;
}

int amsim_lut_set_closed_form(amsim_lut_t lut, int on)
{
    if (!lut) return AMSIM_EINVAL;
    if (on && lut->kind != AMSIM_EXACT && lut->kind != AMSIM_MITCHELL) return AMSIM_EUNSUPPORTED;
    if (on && lut->exp_bits != 8) return AMSIM_EUNSUPPORTED;
    lut->closed_form = on != 0;
    return AMSIM_OK;
}

int amsim_lut_set_exponent_bits(amsim_lut_t lut, int E)
{
    if (!lut) return AMSIM_EINVAL;
    if (E < 1 || E > 8) return AMSIM_EUNSUPPORTED;
    if (E != 8 && lut->closed_form) return AMSIM_EUNSUPPORTED;
    lut->exp_bits = E;
    return AMSIM_OK;
}

int amsim_lut_build_from_entries(const uint32_t *host_entries, int M, amsim_lut_t *out)
{
    return build_from_entries(host_entries, M, out);
}

int amsim_lut_build_from_fn(amsim_approx_mul_fn approx_mul, int M, amsim_lut_t *out)
{
    if (!out || !approx_mul) return AMSIM_EINVAL;
    if (M < 1 || M > 11) return AMSIM_EUNSUPPORTED;
    std::vector<uint32_t> e(size_t(1) << (2 * M));
    int rc = generate(approx_mul, M, e.data());
    if (rc) return rc;
    return build_from_entries(e.data(), M, out);
}

int amsim_lut_entries(amsim_lut_t lut, uint32_t *host_dst)
{
    if (!lut || !host_dst) return AMSIM_EINVAL;
    size_t bytes = (size_t(1) << (2 * lut->M)) * 4;
    return amsim::cuda_status(cudaMemcpy(host_dst, lut->d_canon, bytes, cudaMemcpyDeviceToHost));
}

int amsim_lut_info(amsim_lut_t lut, int *M, int *width_bits, int *shift)
{
    if (!lut) return AMSIM_EINVAL;
    if (M) *M = lut->M;
    if (width_bits) *width_bits = lut->width_bits;
    if (shift) *shift = lut->shift;
    return AMSIM_OK;
}

unsigned long long amsim_kernel_launches(void) { return amsim::g_launches.load(std::memory_order_relaxed); }

void amsim_lut_destroy(amsim_lut_t lut)
{
    if (!lut) return;
    if (lut->d_base) cudaFree(lut->d_base);
    delete lut;
}

}  // extern "C"
