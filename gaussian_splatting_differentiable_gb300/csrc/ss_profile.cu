// Per-kernel timing, off by default ("从 8.6 KB 到 4.2 KB ...", section
// 亲手验证: SS_PROFILE=1 gives per-kernel segment timings).  When enabled
// (environment SS_PROFILE=1 at load, or ss_profile_enable(1)), every kernel
// the library launches is bracketed by two CUDA events recorded on its own
// stream; ss_profile_collect waits for them and returns, per kernel name,
// the launch count and total / min / max milliseconds.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ss_internal.h"
#include "ss_profile.h"

namespace ss {

namespace {
struct Rec {
    const char *name;
    cudaEvent_t a, b;
};
std::mutex g_mu;
std::vector<Rec> g_pending;
std::vector<cudaEvent_t> g_pool;
bool g_on = [] {
    const char *e = std::getenv("SS_PROFILE");
    return e && e[0] == '1';
}();

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

bool profile_on() { return g_on; }

ProfScope::ProfScope(const char *name, cudaStream_t s) : name_(name), s_(s), a_(nullptr) {
    if (!g_on) return;
    std::lock_guard<std::mutex> lk(g_mu);
    a_ = take_event();
    if (a_) cudaEventRecord(a_, s_);
}

ProfScope::~ProfScope() {
    if (!a_) return;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t b = take_event();
    if (!b) return;
    cudaEventRecord(b, s_);
    g_pending.push_back(Rec{name_, a_, b});
}

}  // namespace ss

using namespace ss;

extern "C" void ss_profile_enable(int32_t on) { g_on = on != 0; }

extern "C" int64_t ss_profile_collect(char *buf, size_t len) {
    std::vector<Rec> recs;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        recs.swap(g_pending);
    }
    struct Agg {
        std::string name;
        int64_t count;
        double total, mn, mx;
    };
    std::vector<Agg> agg;
    for (const Rec &r : recs) {
        float ms = 0.f;
        cudaEventSynchronize(r.b);
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) ms = -1.f;
        Agg *a = nullptr;
        for (Agg &x : agg)
            if (x.name == r.name) a = &x;
        if (!a) {
            agg.push_back(Agg{r.name, 0, 0.0, 1e30, 0.0});
            a = &agg.back();
        }
        a->count += 1;
        a->total += ms;
        a->mn = ms < a->mn ? ms : a->mn;
        a->mx = ms > a->mx ? ms : a->mx;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (const Rec &r : recs) {
            g_pool.push_back(r.a);
            g_pool.push_back(r.b);
        }
    }
    std::string out;
    char line[256];
    for (const Agg &a : agg) {
        snprintf(line, sizeof line, "%s %lld %.6f %.6f %.6f\n", a.name.c_str(), (long long)a.count,
                 a.total, a.mn, a.mx);
        out += line;
    }
    if (buf && len) {
        const size_t n = out.size() < len - 1 ? out.size() : len - 1;
        memcpy(buf, out.data(), n);
        buf[n] = 0;
    }
    return int64_t(out.size());
}
