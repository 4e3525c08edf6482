// Host-side plumbing of libbiv: status strings, the thread-local CUDA error
// record, the device error word readers and the SM count.
#include <atomic>
#include <mutex>
#include <vector>

#include "biv_common.cuh"

namespace biv {

namespace {
thread_local int t_last_cuda_error = 0;

std::vector<err_reader_fn>& readers() {
    static std::vector<err_reader_fn> r;   // constructed on first use (static-init safe)
    return r;
}
std::mutex& readers_mu() {
    static std::mutex m;
    return m;
}
}  // namespace

void set_cuda_error(cudaError_t e) { t_last_cuda_error = static_cast<int>(e); }

void register_err_reader(err_reader_fn fn) {
    std::lock_guard<std::mutex> g(readers_mu());
    readers().push_back(fn);
}

int num_sms() {
    static std::atomic<int> cached[kMaxDevices];   // 0 = not yet queried (static storage: zero)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev < 0 || dev >= kMaxDevices) return 1;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

}  // namespace biv

extern "C" const char* biv_status_string(int status) {
    switch (status) {
        case BIV_OK: return "ok";
        case BIV_ERR_NULL: return "a required pointer is NULL";
        case BIV_ERR_SHAPE: return "a size is negative, inconsistent or out of range";
        case BIV_ERR_ALIGN: return "a pointer or leading dimension is not 16-byte aligned";
        case BIV_ERR_VALUE: return "a scalar argument is outside its domain";
        case BIV_ERR_UNSUPPORTED: return "valid arguments, but this configuration is not built";
        case BIV_ERR_CUDA: return "a CUDA runtime call failed (see biv_last_cuda_error)";
        case BIV_ERR_DEVICE: return "no usable device for this call";
        case BIV_ERR_SCRATCH: return "the problem needs more scratch than the no-alloc entry point holds";
        default: return "unknown status";
    }
}

extern "C" int biv_last_cuda_error(void) { return biv::t_last_cuda_error; }

extern "C" int biv_version(void) { return 100; }

extern "C" int biv_device_error(uint32_t* bits_out) {
    BIV_TRACE_CALL();
    if (!bits_out) return BIV_ERR_NULL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return biv::cuda_status(e);
    uint32_t bits = 0;
    std::lock_guard<std::mutex> g(biv::readers_mu());
    for (auto fn : biv::readers()) {
        e = fn(&bits, true);
        if (e != cudaSuccess) return biv::cuda_status(e);
    }
    *bits_out = bits;
    return BIV_OK;
}
