// host_common.cu -- error reporting, device properties, the device status word,
// and the diagnostics entry points of the C ABI.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "host_common.cuh"
#include "ptx.cuh"

namespace sdt {

static thread_local std::string t_last_error;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

void clear_error() { t_last_error.clear(); }

// The status word: first bounded wait that gives up writes its site code here.
__device__ int g_sdt_status = 0;

static constexpr int kMaxDevices = 64;
static std::mutex g_dev_mu;
static DeviceInfo g_dev[kMaxDevices];
static bool g_dev_ok[kMaxDevices];
static int *g_status_ptr[kMaxDevices];

int current_device(DeviceInfo *out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return fail(SDT_ERR_UNSUPPORTED_DEVICE, "no CUDA device available (%s)", cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_dev_ok[dev]) {
        DeviceInfo d;
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
            cudaGetLastError();
            return fail(SDT_ERR_CUDA, "cudaDeviceGetAttribute failed on device %d", dev);
        }
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    const DeviceInfo &d = g_dev[dev];
    if (!(d.cc_major == 10 && d.cc_minor == 3))
        return fail(SDT_ERR_UNSUPPORTED_DEVICE,
                    "device %d is compute capability %d.%d; this library is built for sm_103a only", dev,
                    d.cc_major, d.cc_minor);
    if (out) *out = d;
    return SDT_OK;
}

int status_word(int **out) {
    DeviceInfo d;
    int rc = current_device(&d);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_status_ptr[d.device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_sdt_status);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SDT_ERR_CUDA, "cudaGetSymbolAddress(status) failed: %s", cudaGetErrorString(e));
        }
        g_status_ptr[d.device] = static_cast<int *>(p);
    }
    *out = g_status_ptr[d.device];
    return SDT_OK;
}

unsigned long long wait_timeout_ns() {
    static unsigned long long v = [] {
        const char *s = getenv("SDT_WAIT_TIMEOUT_MS");
        long long ms = s ? atoll(s) : 2000;
        if (ms < 1) ms = 1;
        if (ms > 60000) ms = 60000;
        return static_cast<unsigned long long>(ms) * 1000000ull;
    }();
    return v;
}

bool env_flag(const char *name) {
    const char *s = getenv(name);
    if (!s) return false;
    return !strcmp(s, "1") || !strcasecmp(s, "on") || !strcasecmp(s, "true") || !strcasecmp(s, "yes");
}

// One thread waits on an mbarrier that nothing arrives at, until the deadline.
__global__ void timeout_probe_kernel(unsigned long long limit_ns, int *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    const uint64_t deadline = global_timer_ns() + limit_ns;
    if (!mbar_wait_sleepy(b, 0, deadline)) atomicCAS(status, 0, static_cast<int>(kSiteProbe));
}

}  // namespace sdt

using namespace sdt;

extern "C" {

const char *sdt_last_error(void) { return t_last_error.c_str(); }

int sdt_abi_version(void) { return SDT_ABI_VERSION; }

int sdt_device_sm_count(void) {
    DeviceInfo d;
    int rc = current_device(&d);
    return rc ? rc : d.sm_count;
}

int sdt_device_smem_optin(void) {
    DeviceInfo d;
    int rc = current_device(&d);
    return rc ? rc : d.smem_optin;
}

int sdt_check_device_status(sdt_stream_t stream, int *where) {
    clear_error();
    if (where) *where = 0;
    int *st = nullptr;
    int rc = status_word(&st);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int host = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&host, g_sdt_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SDT_ERR_CUDA, "reading the device status failed: %s", cudaGetErrorString(e));
    }
    if (host != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_sdt_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SDT_ERR_CUDA, "clearing the device status failed: %s", cudaGetErrorString(e));
        }
        if (where) *where = host;
        return fail(SDT_ERR_TIMEOUT, "a kernel gave up a bounded wait (site %d)", host);
    }
    return SDT_OK;
}

int sdt_debug_timeout_probe(sdt_stream_t stream, int64_t limit_us) {
    clear_error();
    if (limit_us < 1 || limit_us > 10000000)
        return fail(SDT_ERR_ARG, "limit_us must be in 1 .. 10,000,000 (got %lld)", (long long)limit_us);
    int *st = nullptr;
    int rc = status_word(&st);
    if (rc) return rc;
    timeout_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<unsigned long long>(limit_us) * 1000ull, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SDT_ERR_LAUNCH, "probe launch failed: %s", cudaGetErrorString(e));
    return SDT_OK;
}

}  // extern "C"
