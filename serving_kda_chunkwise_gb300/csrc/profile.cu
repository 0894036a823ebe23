// profile.cu -- optional per-kernel timing: between kda_profile_begin() and
// kda_profile_end() every kernel the library launches is bracketed by a pair of CUDA
// events recorded on the stream it is launched on; kda_profile_end() waits for them and
// returns, per kernel name, the number of launches and their summed device time.
#include <cstring>
#include <mutex>
#include <vector>

#include "kda.h"
#include "kda_internal.h"

namespace kda {
namespace {

struct Rec {
    const char* name;
    int ev;  // index of the start event; the stop event is ev + 1
};

constexpr size_t kMaxRecs = 1 << 16;

std::mutex g_mu;
bool g_on = false;
std::vector<cudaEvent_t> g_events;
std::vector<Rec> g_recs;

}  // namespace

int prof_kernel_begin(const char* name, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_on || g_recs.size() >= kMaxRecs) return -1;
    const size_t need = 2 * (g_recs.size() + 1);
    while (g_events.size() < need) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return -1;
        g_events.push_back(e);
    }
    const int ev = (int)(2 * g_recs.size());
    if (cudaEventRecord(g_events[ev], s) != cudaSuccess) return -1;
    g_recs.push_back({name, ev});
    return ev;
}

void prof_kernel_end(int ev, cudaStream_t s) {
    if (ev < 0) return;
    std::lock_guard<std::mutex> lock(g_mu);
    cudaEventRecord(g_events[ev + 1], s);
}

}  // namespace kda

extern "C" {

kda_status_t kda_profile_begin(void) {
    std::lock_guard<std::mutex> lock(kda::g_mu);
    kda::g_recs.clear();
    kda::g_on = true;
    return KDA_OK;
}

int kda_profile_end(kda_profile_entry_t* entries, int max_entries) {
    std::lock_guard<std::mutex> lock(kda::g_mu);
    kda::g_on = false;
    int n = 0;
    for (const kda::Rec& r : kda::g_recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(kda::g_events[r.ev + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, kda::g_events[r.ev], kda::g_events[r.ev + 1]) !=
                cudaSuccess)
            return -1;
        int i = 0;
        while (i < n && strncmp(entries[i].name, r.name, sizeof entries[i].name) != 0) ++i;
        if (i == n) {
            if (n == max_entries || entries == nullptr) continue;
            memset(&entries[n], 0, sizeof entries[n]);
            strncpy(entries[n].name, r.name, sizeof entries[n].name - 1);
            ++n;
        }
        entries[i].launches += 1;
        entries[i].total_ms += ms;
    }
    kda::g_recs.clear();
    return n;
}

}  // extern "C"
