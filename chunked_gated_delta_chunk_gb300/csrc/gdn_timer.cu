// Host-side launch bookkeeping.  Launch timing: every kernel launch of the
// library can be bracketed by a pair of CUDA events on its stream, so a
// caller can read the device time of each launch (the bench reports the
// dominant kernel's own duration this way); recording is off unless started.
// Kernel attributes: the dynamic shared-memory limit of each kernel is
// raised once per device instead of on every launch.

#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "gdn_common.cuh"

namespace gdn {
namespace {

struct Record {
    const char* kernel;
    int pair;         // index into the event pool
    bool closed;      // stop event recorded
};

std::mutex g_mu;
std::atomic<bool> g_on{false};
std::vector<cudaEvent_t> g_start, g_stop;
std::vector<Record> g_records;
int g_dropped = 0;
thread_local int t_open = -1;   // pair opened by timer_begin on this thread

void destroy_pool() {
    for (cudaEvent_t e : g_start) cudaEventDestroy(e);
    for (cudaEvent_t e : g_stop) cudaEventDestroy(e);
    g_start.clear();
    g_stop.clear();
}

}  // namespace

void timer_begin(cudaStream_t s, const char* kernel) {
    t_open = -1;
    if (!g_on.load(std::memory_order_acquire)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_on.load(std::memory_order_relaxed)) return;
    if (g_records.size() >= g_start.size()) {
        ++g_dropped;
        return;
    }
    const int pair = int(g_records.size());
    g_records.push_back({kernel, pair, false});
    cudaEventRecord(g_start[pair], s);
    t_open = pair;
}

void timer_end(cudaStream_t s) {
    if (t_open < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (t_open < int(g_records.size()) && g_records[t_open].pair == t_open) {
        cudaEventRecord(g_stop[t_open], s);
        g_records[t_open].closed = true;
    }
    t_open = -1;
}

namespace {
std::mutex g_attr_mu;
std::vector<std::pair<std::pair<int, const void*>, int>> g_attr;   // (device, kernel) -> bytes set
}  // namespace

cudaError_t ensure_smem(const void* kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    for (auto& a : g_attr)
        if (a.first.first == dev && a.first.second == kernel) {
            if (a.second >= bytes) return cudaSuccess;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e == cudaSuccess) a.second = bytes;
            return e;
        }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_attr.push_back({{dev, kernel}, bytes});
    return e;
}

}  // namespace gdn

extern "C" {

int gdn_launch_timer_start(int capacity) {
    if (capacity < 1 || capacity > 1000000) return GDN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(gdn::g_mu);
    gdn::g_on.store(false, std::memory_order_release);
    gdn::destroy_pool();
    gdn::g_records.clear();
    gdn::g_dropped = 0;
    gdn::g_start.reserve(capacity);
    gdn::g_stop.reserve(capacity);
    for (int i = 0; i < capacity; ++i) {
        cudaEvent_t a = nullptr, b = nullptr;
        if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
            if (a) cudaEventDestroy(a);
            gdn::destroy_pool();
            return GDN_ERR_CUDA;
        }
        gdn::g_start.push_back(a);
        gdn::g_stop.push_back(b);
    }
    gdn::g_on.store(true, std::memory_order_release);
    return GDN_OK;
}

int gdn_launch_timer_stop(void) {
    gdn::g_on.store(false, std::memory_order_release);
    return GDN_OK;
}

int gdn_launch_timer_read(const char** names, float* ms, int max, int* dropped) {
    std::lock_guard<std::mutex> lk(gdn::g_mu);
    const int n = int(gdn::g_records.size());
    if (dropped) *dropped = gdn::g_dropped;
    for (int i = 0; i < n && i < max; ++i) {
        const gdn::Record& r = gdn::g_records[i];
        if (names) names[i] = r.kernel;
        if (ms && !r.closed) {
            ms[i] = -1.f;                  // launch not made (e.g. rejected)
        } else if (ms) {
            if (cudaEventSynchronize(gdn::g_stop[r.pair]) != cudaSuccess) return -GDN_ERR_CUDA;
            float t = 0.f;
            if (cudaEventElapsedTime(&t, gdn::g_start[r.pair], gdn::g_stop[r.pair]) != cudaSuccess)
                return -GDN_ERR_CUDA;
            ms[i] = t;
        }
    }
    return n;
}

}  // extern "C"
