// bh_api.cu -- the C ABI (include/orrery_bh.h): argument checks, the
// per-device grow-only workspace, phase events, and the one blocking
// read-back of the status word at the end of each call.
//
// The phase order follows the pages' force evaluation ("sycl_tree_solver.hpp",
// SyclTreeTimings and "Where the tree comes from"; docs/performance/
// sycl_tree.md, "Where one evaluation goes"): sort, gather, build, node
// staging, walk, scatter. Here every phase runs on the device; the node
// staging step has no counterpart because the build writes the walk's node
// format directly, and the int32 bounds check it carried moves to the
// argument checks below (node count bound against INT32_MAX).
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/orrery_bh.h"
#include "bh_common.cuh"

namespace obh {

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int64_t node_bound(int64_t n, int32_t cap)
{
    return n + 21 * (n / ((int64_t)cap + 1)) + 1;
}

static int bbox_blocks_for(int64_t n)
{
    int64_t b = (n + 255) / 256;
    if (b > 1216) b = 1216;  // 8 blocks per SM on 152 SMs
    return (int)(b < 1 ? 1 : b);
}

// Lays the buffers of (n, nodes) out over one allocation; returns its size.
// Both entry points (the grow-only workspace and the fixed no-allocation
// scratch) lay their buffers out with this one function.
size_t carve(Buffers &b, char *base, int64_t n, int64_t nodes)
{
    size_t off = 0;
    auto take = [&](size_t bytes) -> char * {
        char *p = base ? base + off : nullptr;
        off += align256(bytes);
        return p;
    };
    b.n = n;
    b.max_nodes = nodes;
    b.bbox_blocks = bbox_blocks_for(n);
    const size_t n1 = (size_t)n + 1;
    b.bbox_partial = (float *)take(sizeof(float) * 8 * (size_t)b.bbox_blocks);
    b.params = (DeviceParams *)take(sizeof(DeviceParams));
    b.keys_a = (uint64_t *)take(sizeof(uint64_t) * (size_t)n);
    b.keys_b = (uint64_t *)take(sizeof(uint64_t) * (size_t)n);
    b.idx_a = (uint32_t *)take(sizeof(uint32_t) * (size_t)n);
    b.idx_b = (uint32_t *)take(sizeof(uint32_t) * (size_t)n);
    b.sort_ctl = (uint32_t *)take(sizeof(uint32_t) * (size_t)sort_ctl_words());
    b.sort_look = (uint32_t *)take(sizeof(uint32_t) * (size_t)sort_look_words(n));
    b.ps = (float4 *)take(sizeof(float4) * (size_t)n);
    b.lev_d = (int8_t *)take(n1);
    b.ncount = (uint8_t *)take(n1);
    b.pstart = (int32_t *)take(sizeof(int32_t) * n1);
    b.node_start = (uint32_t *)take(sizeof(uint32_t) * n1);
    b.scan_partial = (uint32_t *)take(sizeof(uint32_t) * (size_t)scan_partial_count((int64_t)n1));
    b.meta = (int4 *)take(sizeof(int4) * (size_t)nodes);
    b.parent = (int32_t *)take(sizeof(int32_t) * (size_t)nodes);
    b.arrive = (int32_t *)take(sizeof(int32_t) * (size_t)nodes);
    b.sums = (float4 *)take(sizeof(float4) * (size_t)nodes);
    b.wnode = (WalkNode *)take(sizeof(WalkNode) * ((size_t)nodes + 1));  // + the sentinel
    return off;
}

namespace {

constexpr int64_t kMaxN = int64_t(1) << 30;
constexpr int kMaxDevices = 64;

enum Ev {
    EV_H2D0,
    EV_START,
    EV_BBOX,
    EV_MORTON,
    EV_SORT,
    EV_GATHER,
    EV_BUILD,
    EV_MOMENTS,
    EV_WALK,
    EV_SCATTER,
    EV_D2H,
    EV_COUNT
};

// One replayable evaluation: every argument that the captured launches bake
// in, plus the workspace base they point into.
struct GraphKey {
    const void *pos, *mass, *base;
    void *acc, *inter, *visits;
    int64_t n, t_begin, t_end;
    float theta, eps;
    int32_t cap, traversal;
    bool operator==(const GraphKey &o) const
    {
        return pos == o.pos && mass == o.mass && base == o.base && acc == o.acc &&
               inter == o.inter && visits == o.visits && n == o.n && t_begin == o.t_begin &&
               t_end == o.t_end && theta == o.theta && eps == o.eps && cap == o.cap &&
               traversal == o.traversal;
    }
};

struct GraphEntry {
    GraphKey key;
    cudaGraphExec_t exec;
    uint64_t launches;  // kernels in the graph
    uint64_t last_use;
};

constexpr size_t kGraphCache = 8;

struct Workspace {
    int device = -1;
    void *base = nullptr;
    size_t bytes = 0;
    int64_t cap_n = -1;
    int64_t cap_nodes = -1;
    Buffers b{};
    DeviceParams *host_params = nullptr;  // page-locked read-back slot
    cudaEvent_t ev[EV_COUNT] = {};
    // device staging for orrery_bh_forces_host
    void *io = nullptr;
    int64_t io_n = -1;
    // captured evaluations, replayed when a call repeats its arguments
    cudaStream_t capture_stream = nullptr;
    std::vector<GraphEntry> graphs;
    // argument sets seen once and not captured yet: a graph is captured on
    // the second call with the same arguments, so one-off calls (new output
    // buffers every time) never pay for a capture they cannot reuse
    std::vector<GraphKey> seen;
    uint64_t tick = 0;
};

void drop_graphs(Workspace *w)
{
    for (auto &g : w->graphs) cudaGraphExecDestroy(g.exec);
    w->graphs.clear();
    w->seen.clear();
}

bool graphs_enabled()
{
    static const bool on = [] {
        const char *v = getenv("ORRERY_GRAPHS");
        return !(v && v[0] == '0');
    }();
    return on;
}

// Calls on one device are serialised (they share its workspace and graphs);
// calls on different devices run concurrently.
std::mutex g_dev_mu[kMaxDevices];
std::mutex g_last_mu;  // guards g_last / g_have_last
Workspace *g_ws[kMaxDevices] = {};
orrery_bh_timings g_last{};
bool g_have_last = false;

void free_workspace(Workspace *w)
{
    if (!w) return;
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(w->device);
    drop_graphs(w);
    if (w->capture_stream) cudaStreamDestroy(w->capture_stream);
    if (w->base) cudaFree(w->base);
    if (w->io) cudaFree(w->io);
    if (w->host_params) cudaFreeHost(w->host_params);
    for (int e = 0; e < EV_COUNT; ++e)
        if (w->ev[e]) cudaEventDestroy(w->ev[e]);
    if (prev >= 0) cudaSetDevice(prev);
    delete w;
}

// The calling thread's current device, or -1.
int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}

// The calling thread's current device's workspace, grown to (n, nodes).
int get_workspace(int64_t n, int64_t nodes, Workspace **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ORRERY_ECUDA;
    Workspace *w = g_ws[dev];
    if (!w) {
        w = new Workspace();
        w->device = dev;
        for (int e = 0; e < EV_COUNT; ++e)
            if (cudaEventCreate(&w->ev[e]) != cudaSuccess) {
                free_workspace(w);
                return ORRERY_ECUDA;
            }
        if (cudaMallocHost((void **)&w->host_params, sizeof(DeviceParams)) != cudaSuccess) {
            free_workspace(w);
            return ORRERY_ENOMEM;
        }
        g_ws[dev] = w;
    }
    if (n > w->cap_n || nodes > w->cap_nodes) {
        const int64_t cn = n > w->cap_n ? n : w->cap_n;
        const int64_t cm = nodes > w->cap_nodes ? nodes : w->cap_nodes;
        drop_graphs(w);  // they point into the old allocation
        if (w->base) cudaFree(w->base);
        w->base = nullptr;
        w->cap_n = w->cap_nodes = -1;
        Buffers probe{};
        size_t bytes = carve(probe, nullptr, cn, cm);
        // ORRERY_FAIL_ALLOC=1 makes this allocation fail (failure-path tests)
        const char *fail = getenv("ORRERY_FAIL_ALLOC");
        if ((fail && fail[0] == '1') || cudaMalloc(&w->base, bytes) != cudaSuccess) {
            cudaGetLastError();
            w->base = nullptr;
            return ORRERY_ENOMEM;
        }
        w->bytes = bytes;
        w->cap_n = cn;
        w->cap_nodes = cm;
    }
    carve(w->b, (char *)w->base, n, nodes);
    *out = w;
    return ORRERY_OK;
}

int check_args(int64_t n, float theta, float eps, int32_t leaf_cap, int32_t traversal)
{
    if (n < 0 || n > kMaxN) return ORRERY_EINVAL;
    if (!(theta >= 0.0f) || !(eps >= 0.0f)) return ORRERY_EINVAL;  // also rejects NaN
    if (leaf_cap < 1) return ORRERY_EINVAL;
    const int walk = traversal & kTraversalMask;
    if ((traversal & ~(kTraversalMask | kFastTermFlag)) != 0) return ORRERY_EINVAL;
    if (walk < ORRERY_INDEPENDENT || walk > ORRERY_COHERENT_BALLOT) return ORRERY_EINVAL;
    if (node_bound(n, leaf_cap) > (int64_t)INT32_MAX) return ORRERY_ERANGE;
    return ORRERY_OK;
}

// Records a phase event. Under stream capture a plain record only orders
// streams; the external flag makes it a node of the graph, so replays record
// it as well.
void record_event(cudaEvent_t ev, cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(st, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
    else
        cudaEventRecord(ev, st);
}

float ms_between(cudaEvent_t a, cudaEvent_t b)
{
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) {
        cudaGetLastError();
        return -1.0f;
    }
    return ms;
}

// Phases a1..a6 (through the moments). Returns the sorted keys / perm.
void run_tree(Workspace &w, const float *pos, const float *mass, int32_t cap, cudaStream_t st,
              uint64_t **keys_sorted, uint32_t **perm)
{
    const Buffers &b = w.b;
    record_event(w.ev[EV_START], st);
    launch_bbox(pos, mass, b, st);
    record_event(w.ev[EV_BBOX], st);
    launch_morton(pos, b, st);
    record_event(w.ev[EV_MORTON], st);
    launch_sort(b, st, keys_sorted, perm);
    record_event(w.ev[EV_SORT], st);
    launch_gather(pos, mass, *perm, b, st);
    record_event(w.ev[EV_GATHER], st);
    launch_build(*keys_sorted, cap, b, st);
    record_event(w.ev[EV_BUILD], st);
    launch_moments(*keys_sorted, cap, b, st);
    record_event(w.ev[EV_MOMENTS], st);
}

int collect(Workspace &w, cudaStream_t st);

int finish(Workspace &w, cudaStream_t st)
{
    cudaMemcpyAsync(w.host_params, w.b.params, sizeof(DeviceParams), cudaMemcpyDeviceToHost, st);
    return collect(w, st);
}

// Host destinations of orrery_bh_forces_host.
struct HostOut {
    float *acc;
    uint32_t *inter;
    uint32_t *visits;
};

// Enqueues phases a1..a8, for the host entry point the result copies, and
// the read-back of the status word.
void enqueue_forces(Workspace &w, const float *pos, const float *mass, int64_t n, float theta,
                    float eps, int32_t cap, int32_t traversal, int64_t t_begin, int64_t t_end,
                    float *acc, uint32_t *inter, uint32_t *visits, cudaStream_t st,
                    const HostOut *host)
{
    uint64_t *keys_sorted = nullptr;
    uint32_t *perm = nullptr;
    run_tree(w, pos, mass, cap, st, &keys_sorted, &perm);
    launch_walk(traversal, theta, eps, perm, w.b, t_begin, t_end, acc, inter, visits, st);
    record_event(w.ev[EV_WALK], st);
    record_event(w.ev[EV_SCATTER], st);  // the scatter is fused into the walk
    if (host) {  // outputs the walk wrote straight to host memory have no copy
        if (host->acc)
            cudaMemcpyAsync(host->acc, acc, 12 * (size_t)n, cudaMemcpyDeviceToHost, st);
        if (host->inter)
            cudaMemcpyAsync(host->inter, inter, 8 * (size_t)n, cudaMemcpyDeviceToHost, st);
        if (host->visits)
            cudaMemcpyAsync(host->visits, visits, 4 * (size_t)n, cudaMemcpyDeviceToHost, st);
        record_event(w.ev[EV_D2H], st);
    }
    cudaMemcpyAsync(w.host_params, w.b.params, sizeof(DeviceParams), cudaMemcpyDeviceToHost, st);
}

// Blocks on the stream and turns the status word into a status code.
int collect(Workspace &w, cudaStream_t st)
{
    if (cudaStreamSynchronize(st) != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return ORRERY_ECUDA;
    const int s = w.host_params->status;
    if (s & kStatusNonFinite) return ORRERY_ENONFINITE;
    if (s & kStatusNodeBound) return ORRERY_ERANGE;
    if (s & kStatusWalkBound) return ORRERY_EWALK;
    if (s & kStatusInternal) return ORRERY_EINTERNAL;
    return ORRERY_OK;
}

// The cached graph of this call, captured on first use; nullptr when capture
// is off or fails (the caller then launches directly). Capture runs on the
// workspace's own stream, so it never touches the caller's stream.
GraphEntry *graph_for(Workspace &w, const GraphKey &key, const float *pos, const float *mass,
                      int64_t n, float theta, float eps, int32_t cap, int32_t traversal,
                      int64_t t_begin, int64_t t_end, float *acc, uint32_t *inter,
                      uint32_t *visits)
{
    if (!graphs_enabled()) return nullptr;
    for (auto &g : w.graphs)
        if (g.key == key) {
            g.last_use = ++w.tick;
            return &g;
        }
    bool repeat = false;
    for (size_t i = 0; i < w.seen.size(); ++i)
        if (w.seen[i] == key) {
            repeat = true;
            w.seen.erase(w.seen.begin() + (long)i);
            break;
        }
    if (!repeat) {  // first sight: remember it, launch directly
        if (w.seen.size() >= kGraphCache * 2) w.seen.erase(w.seen.begin());
        w.seen.push_back(key);
        return nullptr;
    }
    if (!w.capture_stream &&
        cudaStreamCreateWithFlags(&w.capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        w.capture_stream = nullptr;
        return nullptr;
    }
    prepare_sort();  // function attributes are set outside the capture
    prepare_walk();
    const uint64_t before = g_launches.load();
    if (cudaStreamBeginCapture(w.capture_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    enqueue_forces(w, pos, mass, n, theta, eps, cap, traversal, t_begin, t_end, acc, inter, visits,
                   w.capture_stream, nullptr);
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(w.capture_stream, &graph);
    const uint64_t launches = g_launches.load() - before;
    g_launches -= launches;  // captured, not launched
    cudaGraphExec_t exec = nullptr;
    const bool ok = ec == cudaSuccess && graph &&
                    cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
    if (graph) cudaGraphDestroy(graph);
    if (!ok) {
        cudaGetLastError();
        return nullptr;
    }
    if (w.graphs.size() >= kGraphCache) {  // evict the least recently used
        size_t old = 0;
        for (size_t i = 1; i < w.graphs.size(); ++i)
            if (w.graphs[i].last_use < w.graphs[old].last_use) old = i;
        cudaGraphExecDestroy(w.graphs[old].exec);
        w.graphs.erase(w.graphs.begin() + (long)old);
    }
    w.graphs.push_back(GraphEntry{key, exec, launches, ++w.tick});
    return &w.graphs.back();
}

// Runs one evaluation: replays its captured graph when the call repeats the
// arguments of an earlier one (device buffers only), else launches directly;
// then blocks once and records the phase timings.
int forces_device(Workspace &w, const float *pos, const float *mass, int64_t n, float theta,
                  float eps, int32_t cap, int32_t traversal, int64_t t_begin, int64_t t_end,
                  float *acc, uint32_t *inter, uint32_t *visits, cudaStream_t st,
                  const HostOut *host)
{
    const uint64_t launches0 = g_launches.load();
    GraphEntry *g = nullptr;
    // host outputs that are all page-locked need no copy after the walk, so
    // the call is the device path's and may replay its graph too
    const bool copies = host && (host->acc || host->inter || host->visits);
    if (!copies) {
        const GraphKey key{pos, mass, w.base, acc, inter, visits, n, t_begin, t_end,
                           theta, eps, cap, traversal};
        g = graph_for(w, key, pos, mass, n, theta, eps, cap, traversal, t_begin, t_end, acc, inter,
                      visits);
    }
    if (g && cudaGraphLaunch(g->exec, st) == cudaSuccess) {
        g_launches += g->launches;
    } else {
        if (g) cudaGetLastError();
        enqueue_forces(w, pos, mass, n, theta, eps, cap, traversal, t_begin, t_end, acc, inter,
                       visits, st, host);
    }
    const int rc = collect(w, st);
    if (rc != ORRERY_OK) return rc;
    orrery_bh_timings t{};
    t.bbox_ms = ms_between(w.ev[EV_START], w.ev[EV_BBOX]);
    t.morton_ms = ms_between(w.ev[EV_BBOX], w.ev[EV_MORTON]);
    t.sort_ms = ms_between(w.ev[EV_MORTON], w.ev[EV_SORT]);
    t.gather_ms = ms_between(w.ev[EV_SORT], w.ev[EV_GATHER]);
    t.build_ms = ms_between(w.ev[EV_GATHER], w.ev[EV_BUILD]);
    t.moments_ms = ms_between(w.ev[EV_BUILD], w.ev[EV_MOMENTS]);
    t.walk_ms = ms_between(w.ev[EV_MOMENTS], w.ev[EV_WALK]);
    t.scatter_ms = ms_between(w.ev[EV_WALK], w.ev[EV_SCATTER]);
    t.total_ms = ms_between(w.ev[EV_START], w.ev[EV_SCATTER]);
    if (host) {
        t.h2d_ms = ms_between(w.ev[EV_H2D0], w.ev[EV_START]);
        t.d2h_ms = copies ? ms_between(w.ev[EV_SCATTER], w.ev[EV_D2H]) : 0.0f;
        t.total_ms = ms_between(w.ev[EV_H2D0], w.ev[copies ? EV_D2H : EV_SCATTER]);
    }
    t.traversal = traversal;
    t.depth = w.host_params->depth;
    t.n = n;
    t.num_nodes = w.host_params->num_nodes;
    t.launches = g_launches.load() - launches0;
    std::lock_guard<std::mutex> last(g_last_mu);
    g_last = t;
    g_have_last = true;
    return ORRERY_OK;
}

}  // namespace
}  // namespace obh

using namespace obh;

extern "C" {

int orrery_bh_forces(const float *pos_d, const float *mass_d, int64_t n, float theta, float eps,
                     int32_t leaf_cap, int32_t traversal, float *acc_d, uint32_t *interactions_d,
                     uint32_t *visits_d, void *stream)
{
    int rc = check_args(n, theta, eps, leaf_cap, traversal);
    if (rc != ORRERY_OK) return rc;
    if (n == 0) return ORRERY_OK;
    if (!pos_d || !mass_d || !acc_d) return ORRERY_EINVAL;
    const int dev = current_device();
    if (dev < 0) return ORRERY_ECUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu[dev]);
    Workspace *w = nullptr;
    rc = get_workspace(n, node_bound(n, leaf_cap), &w);
    if (rc != ORRERY_OK) return rc;
    return forces_device(*w, pos_d, mass_d, n, theta, eps, leaf_cap, traversal, 0, n, acc_d,
                         interactions_d, visits_d, (cudaStream_t)stream, nullptr);
}

int orrery_bh_forces_range(const float *pos_d, const float *mass_d, int64_t n, float theta,
                           float eps, int32_t leaf_cap, int32_t traversal, int64_t begin,
                           int64_t end, float *acc_d, uint32_t *interactions_d, uint32_t *visits_d,
                           void *stream)
{
    int rc = check_args(n, theta, eps, leaf_cap, traversal);
    if (rc != ORRERY_OK) return rc;
    if (begin < 0 || end < begin || end > n) return ORRERY_EINVAL;
    if (n == 0) return ORRERY_OK;
    if (!pos_d || !mass_d || !acc_d) return ORRERY_EINVAL;
    const int dev = current_device();
    if (dev < 0) return ORRERY_ECUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu[dev]);
    Workspace *w = nullptr;
    rc = get_workspace(n, node_bound(n, leaf_cap), &w);
    if (rc != ORRERY_OK) return rc;
    return forces_device(*w, pos_d, mass_d, n, theta, eps, leaf_cap, traversal, begin, end, acc_d,
                         interactions_d, visits_d, (cudaStream_t)stream, nullptr);
}

// The device address of host memory [p, p + bytes) when all of it is
// page-locked (cudaHostAlloc, cudaHostRegister), else null.
static void *mapped(void *p, size_t bytes)
{
    if (!p || bytes == 0) return nullptr;
    cudaPointerAttributes first{}, last{};
    if (cudaPointerGetAttributes(&first, p) != cudaSuccess ||
        cudaPointerGetAttributes(&last, (char *)p + bytes - 1) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (first.type != cudaMemoryTypeHost || last.type != cudaMemoryTypeHost || !first.devicePointer ||
        !last.devicePointer || (char *)last.devicePointer - (char *)first.devicePointer != (ptrdiff_t)(bytes - 1))
        return nullptr;
    return first.devicePointer;
}

int orrery_bh_forces_host(const float *pos, const float *mass, int64_t n, float theta, float eps,
                          int32_t leaf_cap, int32_t traversal, float *acc, uint32_t *interactions,
                          uint32_t *visits, void *stream)
{
    int rc = check_args(n, theta, eps, leaf_cap, traversal);
    if (rc != ORRERY_OK) return rc;
    if (n == 0) return ORRERY_OK;
    if (!pos || !mass || !acc) return ORRERY_EINVAL;
    const int dev = current_device();
    if (dev < 0) return ORRERY_ECUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu[dev]);
    Workspace *w = nullptr;
    rc = get_workspace(n, node_bound(n, leaf_cap), &w);
    if (rc != ORRERY_OK) return rc;
    // device staging: pos [3n] | mass [n] | acc [3n] | inter [2n] | visits [n]
    if (n > w->io_n) {
        if (w->io) cudaFree(w->io);
        w->io = nullptr;
        w->io_n = -1;
        if (cudaMalloc(&w->io, align256(12 * (size_t)n) * 2 + align256(4 * (size_t)n) * 2 +
                                   align256(8 * (size_t)n)) != cudaSuccess) {
            cudaGetLastError();
            w->io = nullptr;
            return ORRERY_ENOMEM;
        }
        w->io_n = n;
    }
    char *p = (char *)w->io;
    float *pos_d = (float *)p;
    p += align256(12 * (size_t)w->io_n);
    float *mass_d = (float *)p;
    p += align256(4 * (size_t)w->io_n);
    float *acc_d = (float *)p;
    p += align256(12 * (size_t)w->io_n);
    uint32_t *inter_d = (uint32_t *)p;
    p += align256(8 * (size_t)w->io_n);
    uint32_t *vis_d = (uint32_t *)p;
    cudaStream_t st = (cudaStream_t)stream;
    // the inputs' copies first: they start while the outputs are looked up
    record_event(w->ev[EV_H2D0], st);
    cudaMemcpyAsync(pos_d, pos, 12 * (size_t)n, cudaMemcpyHostToDevice, st);
    cudaMemcpyAsync(mass_d, mass, 4 * (size_t)n, cudaMemcpyHostToDevice, st);
    // page-locked outputs are written by the walk itself, over the host link
    // while it runs, instead of copied after it (0.15 ms less at 1M)
    HostOut host{acc, interactions, visits};
    if (float *a = (float *)mapped(acc, 12 * (size_t)n)) {
        acc_d = a;
        host.acc = nullptr;
    }
    if (uint32_t *c = (uint32_t *)mapped(interactions, 8 * (size_t)n)) {
        inter_d = c;
        host.inter = nullptr;
    }
    if (uint32_t *v = (uint32_t *)mapped(visits, 4 * (size_t)n)) {
        vis_d = v;
        host.visits = nullptr;
    }
    return forces_device(*w, pos_d, mass_d, n, theta, eps, leaf_cap, traversal, 0, n, acc_d,
                         interactions ? inter_d : nullptr, visits ? vis_d : nullptr, st, &host);
}

int orrery_bh_tree(const float *pos_d, const float *mass_d, int64_t n, int32_t leaf_cap,
                   float *cube_d, uint64_t *keys_d, uint32_t *perm_d, int32_t *nodes_d,
                   float *com_d, int64_t max_nodes, int64_t *num_nodes, void *stream)
{
    int rc = check_args(n, 0.0f, 0.0f, leaf_cap, ORRERY_COHERENT);
    if (rc != ORRERY_OK) return rc;
    if (!num_nodes || max_nodes < 0) return ORRERY_EINVAL;
    *num_nodes = 0;
    if (n == 0) return ORRERY_OK;
    if (!pos_d || !mass_d) return ORRERY_EINVAL;
    const int dev = current_device();
    if (dev < 0) return ORRERY_ECUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu[dev]);
    Workspace *w = nullptr;
    rc = get_workspace(n, node_bound(n, leaf_cap), &w);
    if (rc != ORRERY_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    uint64_t *keys_sorted = nullptr;
    uint32_t *perm = nullptr;
    run_tree(*w, pos_d, mass_d, leaf_cap, st, &keys_sorted, &perm);
    rc = finish(*w, st);
    if (rc != ORRERY_OK) return rc;
    const int64_t nn = w->host_params->num_nodes;
    *num_nodes = nn;
    if (cube_d) cudaMemcpyAsync(cube_d, w->b.params, 5 * sizeof(float), cudaMemcpyDeviceToDevice, st);
    if (keys_d) cudaMemcpyAsync(keys_d, keys_sorted, 8 * (size_t)n, cudaMemcpyDeviceToDevice, st);
    if (perm_d) cudaMemcpyAsync(perm_d, perm, 4 * (size_t)n, cudaMemcpyDeviceToDevice, st);
    const int64_t nc = nn < max_nodes ? nn : max_nodes;
    if (nodes_d && nc > 0)
        cudaMemcpyAsync(nodes_d, w->b.meta, 16 * (size_t)nc, cudaMemcpyDeviceToDevice, st);
    if (com_d && nc > 0)  // the {CoM, M} half of each 32-byte walk node
        cudaMemcpy2DAsync(com_d, sizeof(float4), &w->b.wnode[0].c, sizeof(WalkNode),
                          sizeof(float4), (size_t)nc, cudaMemcpyDeviceToDevice, st);
    if (cudaStreamSynchronize(st) != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return ORRERY_ECUDA;
    return nn > max_nodes ? ORRERY_ERANGE : ORRERY_OK;
}

int orrery_direct_forces(const float *pos_d, const float *mass_d, int64_t n, float eps,
                         float *acc_d, void *stream)
{
    if (n < 0 || n > kMaxN || !(eps >= 0.0f)) return ORRERY_EINVAL;
    if (n == 0) return ORRERY_OK;
    if (!pos_d || !mass_d || !acc_d) return ORRERY_EINVAL;
    const int dev = current_device();
    if (dev < 0) return ORRERY_ECUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu[dev]);
    Workspace *w = nullptr;
    int rc = get_workspace(1, node_bound(1, 1), &w);  // only the status word is used
    if (rc != ORRERY_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    cudaMemsetAsync(&w->b.params->status, 0, sizeof(int), st);
    launch_direct(pos_d, mass_d, n, eps, acc_d, &w->b.params->status, st);
    cudaMemcpyAsync(w->host_params, w->b.params, sizeof(DeviceParams), cudaMemcpyDeviceToHost, st);
    if (cudaStreamSynchronize(st) != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return ORRERY_ECUDA;
    return (w->host_params->status & kStatusNonFinite) ? ORRERY_ENONFINITE : ORRERY_OK;
}

int64_t orrery_bh_max_nodes(int64_t n, int32_t leaf_cap)
{
    if (n < 0 || n > kMaxN || leaf_cap < 1) return -1;
    return node_bound(n, leaf_cap);
}

int orrery_bh_last_timings(orrery_bh_timings *out)
{
    if (!out) return ORRERY_EINVAL;
    std::lock_guard<std::mutex> lock(g_last_mu);
    if (!g_have_last) return ORRERY_EINVAL;
    *out = g_last;
    return ORRERY_OK;
}

uint64_t orrery_bh_kernel_launches(void) { return g_launches.load(); }

const char *orrery_bh_strerror(int status)
{
    switch (status) {
    case ORRERY_OK: return "ok";
    case ORRERY_EINVAL: return "invalid argument";
    case ORRERY_ENONFINITE: return "non-finite position or mass";
    case ORRERY_ERANGE: return "node count or size beyond the int32 range";
    case ORRERY_ECUDA: return "CUDA runtime error";
    case ORRERY_EWALK: return "walk exceeded its iteration bound";
    case ORRERY_ENOMEM: return "workspace allocation failed";
    case ORRERY_EINTERNAL: return "internal consistency check failed";
    case ORRERY_ESCRATCH: return "problem too large for the fixed no-allocation scratch";
    default: return "unknown status";
    }
}

void orrery_bh_release(void)
{
    for (int d = 0; d < kMaxDevices; ++d) {
        std::lock_guard<std::mutex> lock(g_dev_mu[d]);
        free_workspace(g_ws[d]);
        g_ws[d] = nullptr;
    }
    std::lock_guard<std::mutex> last(g_last_mu);
    g_have_last = false;
}

}  // extern "C"
