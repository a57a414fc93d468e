// Kernel trace: the device time of each kernel the library launches, measured with a pair of
// CUDA timing events recorded on the kernel's own stream just before and just after its
// launch. Opt-in per host thread (moe_trace_begin .. moe_trace_end); a launch on a stream
// that is being captured into a graph is not traced. The events make the traced kernel wait
// for its predecessor to finish (no dependent-launch overlap), so each duration is the
// kernel's own, as it would be launched back to back.
#include <cxxabi.h>

#include <cstdlib>
#include <string>
#include <vector>

#include "internal.cuh"

namespace moe {

thread_local bool t_trace_on = false;

namespace {

struct TraceRec {
    const void* fn;
    int ev;          // index of its start event; the end event follows it
};

struct TraceState {
    std::vector<cudaEvent_t> events;
    std::vector<TraceRec> recs;
    std::vector<std::string> names;
    std::vector<float> ms;
    int max_launches = 0;
    int dropped = 0;
    bool failed = false;
};

thread_local TraceState t_trace;

void destroy_events(TraceState& st) {
    for (cudaEvent_t e : st.events) cudaEventDestroy(e);
    st.events.clear();
}

// "void moe::route_tc_kernel<2>(moe::RouteParams, ...)" -> "route_tc_kernel<2>"
std::string kernel_name(const void* fn) {
    const char* raw = nullptr;
    if (cudaFuncGetName(&raw, fn) != cudaSuccess || !raw) return "unknown";
    int status = 0;
    char* dem = abi::__cxa_demangle(raw, nullptr, nullptr, &status);
    std::string s = (status == 0 && dem) ? std::string(dem) : std::string(raw);
    std::free(dem);
    const std::string anon = "(anonymous namespace)::";
    for (size_t at; (at = s.find(anon)) != std::string::npos;) s.erase(at, anon.size());
    // drop the parameter list (the first '(' outside template brackets) and the return type
    int depth = 0;
    size_t end = s.size();
    for (size_t i = 0; i < s.size(); ++i) {
        if (s[i] == '<') ++depth;
        else if (s[i] == '>') --depth;
        else if (s[i] == '(' && depth == 0) { end = i; break; }
    }
    s = s.substr(0, end);
    if (s.rfind("void ", 0) == 0) s = s.substr(5);
    for (size_t at; (at = s.find("moe::")) != std::string::npos;) s.erase(at, 5);
    return s.empty() ? std::string("unknown") : s;
}

}  // namespace

int trace_before(const void* fn, cudaStream_t s) {
    TraceState& st = t_trace;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return -1;
    if ((int)st.recs.size() >= st.max_launches) {
        ++st.dropped;
        return -1;
    }
    const int slot = (int)st.recs.size();
    if (cudaEventRecord(st.events[2 * slot], s) != cudaSuccess) {
        st.failed = true;
        return -1;
    }
    st.recs.push_back({fn, 2 * slot});
    return slot;
}

void trace_after(int slot, cudaStream_t s) {
    if (cudaEventRecord(t_trace.events[2 * slot + 1], s) != cudaSuccess) t_trace.failed = true;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_trace_begin(int32_t max_launches) {
    if (max_launches < 1 || max_launches > (1 << 16)) return MOE_ERR_INVALID_ARG;
    TraceState& st = t_trace;
    t_trace_on = false;
    destroy_events(st);
    st.recs.clear();
    st.names.clear();
    st.ms.clear();
    st.dropped = 0;
    st.failed = false;
    st.events.reserve(2 * (size_t)max_launches);
    for (int i = 0; i < 2 * max_launches; ++i) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) {
            destroy_events(st);
            return MOE_ERR_CUDA;
        }
        st.events.push_back(e);
    }
    st.max_launches = max_launches;
    t_trace_on = true;
    return MOE_OK;
}

int32_t moe_trace_end(void) {
    TraceState& st = t_trace;
    if (!t_trace_on) return MOE_ERR_INVALID_ARG;
    t_trace_on = false;
    bool ok = !st.failed;
    for (const TraceRec& r : st.recs) {
        float ms = 0.f;
        if (ok && (cudaEventSynchronize(st.events[r.ev + 1]) != cudaSuccess ||
                   cudaEventElapsedTime(&ms, st.events[r.ev], st.events[r.ev + 1]) != cudaSuccess))
            ok = false;
        st.names.push_back(kernel_name(r.fn));
        st.ms.push_back(ms);
    }
    destroy_events(st);
    if (!ok) return MOE_ERR_CUDA;
    return (int32_t)st.recs.size();
}

moe_status_t moe_trace_record(int32_t i, const char** name, float* ms) {
    TraceState& st = t_trace;
    if (t_trace_on || !name || !ms || i < 0 || i >= (int32_t)st.names.size()) return MOE_ERR_INVALID_ARG;
    *name = st.names[i].c_str();
    *ms = st.ms[i];
    return MOE_OK;
}

int32_t moe_trace_dropped(void) { return t_trace.dropped; }

}  // extern "C"
