// Launch counter and profiling sessions behind nha_launch_count /
// nha_profile_begin / nha_profile_end (include/nha.h).
#include <atomic>
#include <mutex>
#include <string.h>
#include <vector>

#include "nha.h"
#include "nha_prof.h"

namespace {

std::atomic<unsigned long long> g_launches{0};
std::atomic<bool> g_profiling{false};
std::mutex g_mu;

struct Rec {
    const char* name;
    cudaEvent_t start, stop;
};
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;  // events reused across sessions

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

namespace nha {

LaunchScope::LaunchScope(const char* name, cudaStream_t s) : name_(name), s_(s), slot_(-1) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!g_profiling.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_mu);
    Rec r{name, take_event(), take_event()};
    if (r.start == nullptr || r.stop == nullptr) return;
    cudaEventRecord(r.start, s);
    g_recs.push_back(r);
    slot_ = (int)g_recs.size() - 1;
}

LaunchScope::~LaunchScope() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEventRecord(g_recs[slot_].stop, s_);
}

}  // namespace nha

extern "C" {

unsigned long long nha_launch_count(void) { return g_launches.load(); }

nha_status_t nha_profile_begin(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& r : g_recs) {
        g_pool.push_back(r.start);
        g_pool.push_back(r.stop);
    }
    g_recs.clear();
    g_profiling.store(true);
    return NHA_OK;
}

int nha_profile_end(nha_profile_record_t* out, int cap) {
    g_profiling.store(false);
    std::lock_guard<std::mutex> lk(g_mu);
    std::vector<nha_profile_record_t> agg;
    int status = 0;
    for (auto& r : g_recs) {
        float ms = 0.0f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
            status = -1;
            continue;
        }
        nha_profile_record_t* hit = nullptr;
        for (auto& a : agg)
            if (strcmp(a.name, r.name) == 0) hit = &a;
        if (!hit) {
            nha_profile_record_t n;
            memset(&n, 0, sizeof(n));
            strncpy(n.name, r.name, sizeof(n.name) - 1);
            agg.push_back(n);
            hit = &agg.back();
        }
        hit->launches += 1;
        hit->total_ms += ms;
    }
    for (auto& r : g_recs) {
        g_pool.push_back(r.start);
        g_pool.push_back(r.stop);
    }
    g_recs.clear();
    if (status != 0) return -1;
    int n = (int)agg.size();
    for (int i = 0; i < n && i < cap; i++) out[i] = agg[i];
    return n;
}

}  // extern "C"
