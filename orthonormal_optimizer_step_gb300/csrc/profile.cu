// profile.cu -- optional CUDA-event timing of every kernel libdion launches.
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"

namespace dion {
namespace {

struct Rec { const char* name; cudaEvent_t a, b; };
struct State {
    bool on = false;
    int cap = 0, used = 0, dropped = 0;
    std::vector<Rec> recs;
    // aggregated results (filled by dion_profile_count)
    std::vector<const char*> names;
    std::vector<int> launches;
    std::vector<double> ms;
};
State g;

void release()
{
    for (auto& r : g.recs) {
        if (r.a) cudaEventDestroy(r.a);
        if (r.b) cudaEventDestroy(r.b);
    }
    g.recs.clear();
    g.cap = g.used = g.dropped = 0;
}

}  // namespace

int prof_begin(const char* name, cudaStream_t s)
{
    if (!g.on) return -1;
    if (g.used >= g.cap) {
        ++g.dropped;
        return -1;
    }
    const int slot = g.used++;
    g.recs[slot].name = name;
    cudaEventRecord(g.recs[slot].a, s);
    return slot;
}

void prof_end(int slot, cudaStream_t s)
{
    if (slot >= 0) cudaEventRecord(g.recs[slot].b, s);
}

}  // namespace dion

using namespace dion;

extern "C" dion_status dion_profile_begin(int max_launches)
{
    if (max_launches <= 0) return DION_ERR_INVALID_ARG;
    release();
    g.recs.assign(max_launches, Rec{nullptr, nullptr, nullptr});
    for (auto& r : g.recs) {
        if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) {
            release();
            return DION_ERR_CUDA;
        }
    }
    g.cap = max_launches;
    g.used = 0;
    g.dropped = 0;
    g.names.clear(); g.launches.clear(); g.ms.clear();
    g.on = true;
    return DION_OK;
}

extern "C" dion_status dion_profile_end(void)
{
    g.on = false;
    return DION_OK;
}

extern "C" int dion_profile_count(void)
{
    g.names.clear(); g.launches.clear(); g.ms.clear();
    for (int i = 0; i < g.used; ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g.recs[i].a, g.recs[i].b) != cudaSuccess) continue;
        size_t k = 0;
        for (; k < g.names.size(); ++k)
            if (std::strcmp(g.names[k], g.recs[i].name) == 0) break;
        if (k == g.names.size()) { g.names.push_back(g.recs[i].name); g.launches.push_back(0); g.ms.push_back(0.0); }
        g.launches[k] += 1;
        g.ms[k] += t;
    }
    return (int)g.names.size();
}

extern "C" dion_status dion_profile_entry(int i, const char** name, int* launches, double* total_ms)
{
    if (i < 0 || i >= (int)g.names.size() || !name || !launches || !total_ms) return DION_ERR_INVALID_ARG;
    *name = g.names[i];
    *launches = g.launches[i];
    *total_ms = g.ms[i];
    return DION_OK;
}

extern "C" int dion_profile_dropped(void) { return g.dropped; }
