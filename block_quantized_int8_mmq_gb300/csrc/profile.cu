// Per-kernel device timing: when enabled, every kernel launch of the library is
// bracketed by two CUDA events on its stream; mmq_profile_read folds the finished
// pairs into per-kernel launch counts and total device time.  Under stream capture the
// records are external event-record nodes of the graph; those events stay owned by the
// graph (never recycled), and their pair is read once, after the graph has run.
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace mmq {
namespace {

struct Pending {
    const char* name;
    cudaEvent_t a, b;
    bool captured;
};
struct Total {
    int64_t launches = 0;
    double ms = 0.0;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free;
std::vector<cudaEvent_t> g_graph_owned;  // referenced by captured graphs: never reused
std::map<std::string, Total> g_totals;

cudaEvent_t take_event() {
    if (!g_free.empty()) {
        cudaEvent_t e = g_free.back();
        g_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return e;
}

}  // namespace

bool profiling() { return g_on.load(std::memory_order_relaxed); }

int prof_begin(const char* name, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    const bool captured = cs != cudaStreamCaptureStatusNone;
    std::lock_guard<std::mutex> lk(g_mu);
    cudaEvent_t a = take_event(), b = take_event();
    if (!a || !b) {
        if (a) g_free.push_back(a);
        if (b) g_free.push_back(b);
        return -1;
    }
    if (cudaEventRecordWithFlags(a, s, captured ? cudaEventRecordExternal : cudaEventRecordDefault) != cudaSuccess) {
        cudaGetLastError();
        g_free.push_back(a);
        g_free.push_back(b);
        return -1;
    }
    g_pending.push_back({name, a, b, captured});
    return (int)g_pending.size() - 1;
}

void prof_end(int slot, cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (slot < 0 || slot >= (int)g_pending.size()) return;
    const Pending& p = g_pending[slot];
    if (cudaEventRecordWithFlags(p.b, s, p.captured ? cudaEventRecordExternal : cudaEventRecordDefault) !=
        cudaSuccess)
        cudaGetLastError();
}

}  // namespace mmq

using namespace mmq;

extern "C" {

int mmq_profile_enable(int on) { return g_on.exchange(on != 0) ? 1 : 0; }

int mmq_profile_read(mmq_kernel_time* out, int capacity, int reset) {
    std::lock_guard<std::mutex> lk(g_mu);
    int status = MMQ_OK;
    for (const Pending& p : g_pending) {
        float ms = 0.f;
        if (cudaEventSynchronize(p.b) == cudaSuccess && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
            Total& t = g_totals[p.name];
            t.launches += 1;
            t.ms += ms;
        } else {
            cudaGetLastError();
            status = MMQ_ERR_CUDA;
        }
        std::vector<cudaEvent_t>& dst = p.captured ? g_graph_owned : g_free;
        dst.push_back(p.a);
        dst.push_back(p.b);
    }
    g_pending.clear();
    if (status != MMQ_OK) {
        fprintf(stderr, "libmmq: mmq_profile_read: a timing event could not be read\n");
        return status;
    }
    int n = 0;
    for (const auto& kv : g_totals) {
        if (out && n < capacity) {
            memset(&out[n], 0, sizeof(out[n]));
            strncpy(out[n].name, kv.first.c_str(), sizeof(out[n].name) - 1);
            out[n].launches = kv.second.launches;
            out[n].total_ms = kv.second.ms;
        }
        ++n;
    }
    if (reset) g_totals.clear();
    return n;
}

}  // extern "C"
