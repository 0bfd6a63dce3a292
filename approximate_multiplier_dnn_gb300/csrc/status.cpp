// Device-side wait status: the registry of every translation unit's wait words
// and the ABI calls that read them (amsim_device_errors) and set the limit of
// waits on other CTAs' flags (amsim_set_flag_wait_limit).
#include <mutex>
#include <vector>

#include "amsim_internal.h"

namespace amsim {

namespace {

struct WaitWords {
    WaitStatusFn status;
    WaitLimitFn limit;
};

std::mutex &registry_mutex()
{
    static std::mutex m;
    return m;
}

std::vector<WaitWords> &registry()
{
    static std::vector<WaitWords> r;
    return r;
}

}  // namespace

bool register_wait_words(WaitStatusFn status, WaitLimitFn limit)
{
    std::lock_guard<std::mutex> lock(registry_mutex());
    registry().push_back({status, limit});
    return true;
}

}  // namespace amsim

extern "C" int amsim_device_errors(unsigned int *flags, int clear)
{
    if (!flags) return AMSIM_EINVAL;
    *flags = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return AMSIM_ECUDA;
    }
    std::lock_guard<std::mutex> lock(amsim::registry_mutex());
    unsigned int bits = 0;
    for (const auto &w : amsim::registry()) {
        const int rc = w.status(&bits, clear);
        if (rc) {
            cudaGetLastError();
            return rc;
        }
    }
    *flags = bits;
    return bits ? AMSIM_ETIMEOUT : AMSIM_OK;
}

extern "C" int amsim_set_flag_wait_limit(long long ns)
{
    if (ns < 0 || ns > 10000000000LL) return AMSIM_EINVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return AMSIM_ECUDA;
    }
    std::lock_guard<std::mutex> lock(amsim::registry_mutex());
    for (const auto &w : amsim::registry()) {
        const int rc = w.limit(ns);
        if (rc) {
            cudaGetLastError();
            return rc;
        }
    }
    return AMSIM_OK;
}
