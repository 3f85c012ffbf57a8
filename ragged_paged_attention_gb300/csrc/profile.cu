// Per-kernel timing for diagnostics: when enabled, each library launch is bracketed
// by two CUDA events recorded on the launch stream, and rpa_profile_read() turns the
// pairs into launches and milliseconds per kernel.  When disabled it costs one
// atomic load per launch.
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "profile.h"

namespace rpa {
namespace {
std::atomic<int> g_on{0};
std::atomic<long long> g_launches{0};
struct Rec {
    const char* name;
    cudaEvent_t a, b;
};
std::mutex g_mu;
std::vector<Rec> g_pending;
std::vector<cudaEvent_t> g_pool;
std::map<std::string, std::pair<long long, double>> g_acc;

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}
}  // namespace

bool prof_enabled() { return g_on.load(std::memory_order_relaxed) != 0; }

ProfScope::ProfScope(const char* name, cudaStream_t s) : name_(name), stream_(s), a_(nullptr), b_(nullptr) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    a_ = take_event();
    b_ = take_event();
    if (a_ && b_) cudaEventRecord(static_cast<cudaEvent_t>(a_), stream_);
}

ProfScope::~ProfScope() {
    if (!a_ || !b_) return;
    cudaEventRecord(static_cast<cudaEvent_t>(b_), stream_);
    std::lock_guard<std::mutex> lk(g_mu);
    g_pending.push_back({name_, static_cast<cudaEvent_t>(a_), static_cast<cudaEvent_t>(b_)});
}

}  // namespace rpa

using namespace rpa;

extern "C" {

int64_t rpa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int rpa_profile_enable(int on) {
    g_on.store(on ? 1 : 0);
    return RPA_OK;
}

int rpa_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& r : g_pending) {
        cudaEventSynchronize(r.b);
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_pending.clear();
    g_acc.clear();
    return RPA_OK;
}

int rpa_profile_read(rpa_kernel_time* out, int max_entries, int* n_entries) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& r : g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
            return RPA_ERR_CUDA;
        auto& acc = g_acc[r.name];
        acc.first += 1;
        acc.second += ms;
        g_pool.push_back(r.a);
        g_pool.push_back(r.b);
    }
    g_pending.clear();
    int i = 0;
    for (auto& kv : g_acc) {
        if (out && i < max_entries) {
            memset(&out[i], 0, sizeof out[i]);
            strncpy(out[i].name, kv.first.c_str(), sizeof(out[i].name) - 1);
            out[i].launches = kv.second.first;
            out[i].total_ms = kv.second.second;
        }
        ++i;
    }
    if (n_entries) *n_entries = i;
    return RPA_OK;
}

}  // extern "C"
