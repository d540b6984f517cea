// Kernel timing hook (see cpr_profile_begin / cpr_profile_end in cpr_gdn.h).
#include "profile.h"

#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "cpr_gdn.h"

namespace cpr {
namespace {

struct Record {
    const char* name;
    cudaEvent_t start, stop;
};

std::mutex g_mu;
std::atomic<bool> g_on{false};
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_pool;

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

ProfScope::ProfScope(const char* name, cudaStream_t stream) : slot_(-1), stream_(stream) {
    if (!g_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_mu);
    Record r{name, take_event(), take_event()};
    if (!r.start || !r.stop) return;
    cudaEventRecord(r.start, stream);
    g_records.push_back(r);
    slot_ = (int)g_records.size() - 1;
}

ProfScope::~ProfScope() {
    if (slot_ < 0) return;
    std::lock_guard<std::mutex> lock(g_mu);
    if (slot_ < (int)g_records.size()) cudaEventRecord(g_records[slot_].stop, stream_);
}

}  // namespace cpr

extern "C" int cpr_profile_begin(void) {
    std::lock_guard<std::mutex> lock(cpr::g_mu);
    for (auto& r : cpr::g_records) {
        cpr::g_pool.push_back(r.start);
        cpr::g_pool.push_back(r.stop);
    }
    cpr::g_records.clear();
    cpr::g_on = true;
    return CPR_OK;
}

extern "C" int cpr_profile_end(cpr_kernel_time* out, int max_entries, int* n_entries) {
    cpr::g_on = false;
    if (cudaDeviceSynchronize() != cudaSuccess) return CPR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(cpr::g_mu);
    std::map<std::string, std::pair<uint32_t, double>> agg;
    std::vector<std::string> order;
    for (auto& r : cpr::g_records) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) return CPR_ERR_CUDA;
        auto it = agg.find(r.name);
        if (it == agg.end()) {
            order.push_back(r.name);
            agg[r.name] = {1u, (double)ms};
        } else {
            it->second.first += 1;
            it->second.second += ms;
        }
    }
    if (n_entries) *n_entries = (int)order.size();
    for (int i = 0; i < (int)order.size() && i < max_entries && out; ++i) {
        std::memset(out[i].name, 0, sizeof(out[i].name));
        std::strncpy(out[i].name, order[i].c_str(), sizeof(out[i].name) - 1);
        out[i].launches = agg[order[i]].first;
        out[i].total_ms = agg[order[i]].second;
    }
    return CPR_OK;
}
