// C ABI of the solver (declared in include/jacobi.h): argument checking,
// TMA tensor maps, one CUDA graph per check interval, and the convergence
// loop of "Synchronous vs block-async Jacobi on one RTX 5050", sections
// 01-02.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <map>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/jacobi.h"
#include "jacobi_kernels.cuh"

using namespace tbj;

struct jacobi_handle {
    GridDesc g;
    jacobi_config_t cfg;
    float *u = nullptr, *u_alt = nullptr, *b = nullptr;  // caller-owned
    float *g_copy = nullptr;  // library-owned copy of g (unfused rhs only)
    int b_mode = -1;          // rhs mode b was last prepared for (-1: none)
    cudaStream_t stream = nullptr;   // caller's stream: all work goes here
    cudaStream_t capture = nullptr;  // private stream used to record graphs

    // Library-owned device state.
    ResidualOut *dev_out = nullptr;
    ResidualOut *host_out = nullptr;  // pinned
    LoopState *loop = nullptr;        // device-side loop state
    LoopState *loop_host = nullptr;   // pinned copy read after each step

    // Tiled strategies.
    TileConf tc{};
    CUtensorMap map_u{}, map_alt{}, map_b{};
    int *etbs_work = nullptr;  // column-streamed ETB: its work list (device)

    // Host-buffer runs (jacobi_run_host), allocated on first use: a twin
    // handle over a second pair of fields (hb_tu, hb_tualt; it shares b and
    // the stream), the source of each handle's problems (hb_g[0] for this
    // handle, hb_g[1] for the twin), a stream for the copies and, per pair,
    // an event marking its next problem's inputs in place.
    jacobi_handle_t *hb_twin = nullptr;
    float *hb_tu = nullptr, *hb_tualt = nullptr;
    float *hb_g[2] = {nullptr, nullptr};
    cudaStream_t hb_copy = nullptr;
    cudaEvent_t hb_staged[2] = {nullptr, nullptr};

    // Sweeps per launch, launches per check, sweeps per check.
    int per_launch = 1;
    long long launches_per_check = 8;
    long long interval = 8;

    // Host control: graph for a check interval starting from u (index 0)
    // and from u_alt (index 1; only when launches_per_check is odd).
    cudaGraphExec_t batch[2] = {nullptr, nullptr};
    // Device control: one graph per time step (conditional WHILE loop), and
    // one graph for a whole jacobi_run of run_steps steps with source run_g.
    cudaGraphExec_t step = nullptr;
    cudaGraphExec_t run = nullptr;
    const float *run_g = nullptr;
    int run_steps = 0;
    LoopState *run_states = nullptr;       // device, run_cap entries
    LoopState *run_states_host = nullptr;  // pinned copy
    int run_cap = 0;
    // The run graph's steps start with a sweep launch that forms b itself
    // (rhs_first_launch) instead of k_rhs and k_bnorm, each from the buffer
    // that holds the previous step's answer (record_run_rhs_first).
    bool run_rhs_first = false;
    int cur = 0;  // 0: the iterate is in u; 1: in u_alt

    // Adaptive depth (BLOCK_ASYNC with a depth controller): one fixed-depth
    // handle per D = 1, 2, 4, ... cfg.depth over the same buffers and stream,
    // each with check graphs from both buffers.
    jacobi_handle_t *level[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
    int nlevels = 0;
    cudaEvent_t ev[2] = {nullptr, nullptr};  // times each check interval

    // Checks of the last solve_step (host control).
    std::vector<jacobi_check_record_t> trace;

    long long launches = 0;  // kernels launched so far
    char err[512] = {0};
};

namespace {

thread_local char g_create_err[512];

int fail(jacobi_handle_t *h, int status, const char *fmt, ...) {
    char *dst = h ? h->err : g_create_err;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(dst, 512, fmt, ap);
    va_end(ap);
    return status;
}

#define TBJ_CUDA(h, call)                                                     \
    do {                                                                      \
        cudaError_t e_ = (call);                                              \
        if (e_ != cudaSuccess)                                                \
            return fail((h), JACOBI_ERR_CUDA, "%s: %s", #call,                \
                        cudaGetErrorString(e_));                              \
    } while (0)

bool aligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool is_device_pointer(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// The driver's tensor-map encoder, looked up once per process (a local
// static, so handles created on several threads at once do not race).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p,
                                             12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
        return PFN_cuTensorMapEncodeTiled_v12000{nullptr};
    }();
    return fn;
}

int make_map(jacobi_handle_t *h, CUtensorMap *map, const float *ptr) {
    auto fn = encode_fn();
    if (!fn) return fail(h, JACOBI_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {(cuuint64_t)h->g.n, (cuuint64_t)h->g.n};
    const cuuint64_t strides[1] = {(cuuint64_t)h->g.ld * sizeof(float)};
    const cuuint32_t box[2] = {(cuuint32_t)h->tc.box_x,
                               (cuuint32_t)h->tc.box_y};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                    const_cast<float *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(h, JACOBI_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)",
                    (int)r);
    return JACOBI_OK;
}

long long gcd_ll(long long a, long long b) {
    while (b) {
        long long t = a % b;
        a = b;
        b = t;
    }
    return a;
}

int check_config(jacobi_handle_t *h, const jacobi_config_t &c) {
    if (c.rhs != JACOBI_RHS_FUSED && c.rhs != JACOBI_RHS_UNFUSED)
        return fail(h, JACOBI_ERR_INVALID_ARG, "unknown rhs mode %d", c.rhs);
    if (c.rhs == JACOBI_RHS_UNFUSED && c.strategy != JACOBI_SYNC)
        return fail(h, JACOBI_ERR_UNSUPPORTED,
                    "the unfused right-hand side is provided for SYNC only");
    if (c.adapt < JACOBI_ADAPT_NONE || c.adapt > JACOBI_ADAPT_G_FB)
        return fail(h, JACOBI_ERR_INVALID_ARG, "unknown adapt %d", c.adapt);
    if (c.adapt != JACOBI_ADAPT_NONE) {
        if (c.strategy != JACOBI_BLOCK_ASYNC)
            return fail(h, JACOBI_ERR_INVALID_ARG,
                        "a depth controller needs BLOCK_ASYNC");
        if (c.depth != 2 && c.depth != 4 && c.depth != 8 && c.depth != 16)
            return fail(h, JACOBI_ERR_INVALID_ARG,
                        "a depth controller takes depth 2, 4, 8 or 16 (the "
                        "largest D)");
        if (c.control != JACOBI_CONTROL_HOST)
            return fail(h, JACOBI_ERR_UNSUPPORTED,
                        "a depth controller runs under JACOBI_CONTROL_HOST");
    }
    if (c.division != JACOBI_DIVISION_AUTO && c.division != JACOBI_DIVISION_IEEE)
        return fail(h, JACOBI_ERR_INVALID_ARG, "unknown division %d", c.division);
    if (c.check_every < 1)
        return fail(h, JACOBI_ERR_INVALID_ARG, "check_every must be >= 1");
    if (!(c.tol >= 0.0) || !std::isfinite(c.tol))
        return fail(h, JACOBI_ERR_INVALID_ARG, "tol must be finite and >= 0");
    if (c.max_sweeps < 1)
        return fail(h, JACOBI_ERR_INVALID_ARG, "max_sweeps must be >= 1");
    if (c.control != JACOBI_CONTROL_HOST && c.control != JACOBI_CONTROL_DEVICE &&
        c.control != JACOBI_CONTROL_PERSISTENT)
        return fail(h, JACOBI_ERR_INVALID_ARG, "unknown control %d", c.control);
    if (c.control == JACOBI_CONTROL_PERSISTENT &&
        c.strategy != JACOBI_EXACT_TEMPORAL_BLOCKED)
        return fail(h, JACOBI_ERR_UNSUPPORTED,
                    "JACOBI_CONTROL_PERSISTENT is provided for "
                    "EXACT_TEMPORAL_BLOCKED only");
    switch (c.strategy) {
        case JACOBI_SYNC:
            if (c.depth != 1)
                return fail(h, JACOBI_ERR_INVALID_ARG, "SYNC takes depth 1");
            break;
        case JACOBI_EXACT_TEMPORAL_BLOCKED:
            if (c.depth != 2 && c.depth != 4 && c.depth != 8 && c.depth != 16)
                return fail(h, JACOBI_ERR_INVALID_ARG,
                            "EXACT_TEMPORAL_BLOCKED takes depth 2, 4, 8 or 16");
            break;
        case JACOBI_BLOCK_ASYNC:
            if (c.depth != 1 && c.depth != 2 && c.depth != 4 && c.depth != 8 &&
                c.depth != 16 && c.depth != 32)
                return fail(h, JACOBI_ERR_INVALID_ARG,
                            "BLOCK_ASYNC takes depth 1, 2, 4, 8, 16 or 32");
            break;
        default:
            return fail(h, JACOBI_ERR_INVALID_ARG, "unknown strategy %d",
                        c.strategy);
    }
    if (c.tile_x < 0 || c.tile_y < 0)
        return fail(h, JACOBI_ERR_INVALID_ARG, "tile sizes must be >= 0");
    if (c.overlap_x || c.overlap_y) {
        if (c.strategy != JACOBI_BLOCK_ASYNC)
            return fail(h, JACOBI_ERR_INVALID_ARG,
                        "overlapping subdomains need BLOCK_ASYNC");
        if (c.overlap_x < 0 || c.overlap_y < 0 || c.overlap_x % 2 ||
            c.overlap_y % 2)
            return fail(h, JACOBI_ERR_INVALID_ARG,
                        "overlaps must be even and >= 0");
    }
    return JACOBI_OK;
}

// Plain launch control: no stop flag, no fused residual.
LaunchCtl plain_ctl() {
    LaunchCtl c;
    std::memset(&c, 0, sizeof c);
    return c;
}

// Control of a launch inside the device-side loop: honours the stop flag;
// a fused launch also reduces the residual of its input and decides.
LaunchCtl loop_ctl(jacobi_handle_t *h, LoopState *st, bool fused,
                   int src_is_alt, cudaGraphConditionalHandle cond) {
    LaunchCtl c = plain_ctl();
    c.stop = &st->stop;
    c.fused = fused;
    c.lp.state = st;
    c.lp.d = h->g.d;
    c.lp.tol = h->cfg.tol;
    c.lp.max_sweeps = h->cfg.max_sweeps;
    c.lp.interval = h->interval;
    c.lp.cond = cond;
    c.lp.src_is_alt = src_is_alt;
    return c;
}

// Enqueue one launch of the configured strategy: src -> dst.
cudaError_t enqueue_launch(jacobi_handle_t *h, int src_is_alt,
                           cudaStream_t s, const LaunchCtl &ctl) {
    const float *src = src_is_alt ? h->u_alt : h->u;
    float *dst = src_is_alt ? h->u : h->u_alt;
    const CUtensorMap *map_src = src_is_alt ? &h->map_alt : &h->map_u;
    if (kBoundsChecked) {
        // The launch must write every interior cell of dst.
        cudaError_t e = launch_poison_interior(h->g, dst, ctl.stop, s);
        if (e != cudaSuccess) return e;
    }
    switch (h->cfg.strategy) {
        case JACOBI_SYNC:
            return launch_sweep_sync(h->g, src, h->b, dst, ctl, s);
        case JACOBI_EXACT_TEMPORAL_BLOCKED:
            return launch_sweep_etb(h->g, h->tc, map_src, &h->map_b, src,
                                    h->b, dst, h->dev_out, ctl, s);
        default:
            return launch_sweep_ba(h->g, h->tc, map_src, &h->map_b, src,
                                   h->b, dst, h->dev_out, ctl, s);
    }
}

cudaError_t enqueue_launch(jacobi_handle_t *h, int src_is_alt,
                           cudaStream_t s) {
    return enqueue_launch(h, src_is_alt, s, plain_ctl());
}

void destroy_levels(jacobi_handle_t *h) {
    for (auto &l : h->level) {
        if (l) jacobi_destroy(l);
        l = nullptr;
    }
    h->nlevels = 0;
}

void destroy_graphs(jacobi_handle_t *h) {
    for (auto &e : h->batch) {
        if (e) cudaGraphExecDestroy(e);
        e = nullptr;
    }
    if (h->step) cudaGraphExecDestroy(h->step);
    h->step = nullptr;
    if (h->run) cudaGraphExecDestroy(h->run);
    h->run = nullptr;
    h->run_g = nullptr;
    h->run_steps = 0;
}

// Record the check interval starting from buffer `start` (0 = u, 1 = u_alt):
// launches_per_check launches, the residual of the resulting iterate, and a
// copy of the result block to pinned host memory.
int record_batch(jacobi_handle_t *h, int start, cudaGraphExec_t *exec) {
    TBJ_CUDA(h, cudaStreamBeginCapture(h->capture,
                                       cudaStreamCaptureModeThreadLocal));
    int src = start;
    cudaError_t e = cudaSuccess;
    for (long long l = 0; l < h->launches_per_check && e == cudaSuccess; ++l) {
        e = enqueue_launch(h, src, h->capture);
        src ^= 1;
    }
    if (e == cudaSuccess)
        e = launch_residual(h->g, src ? h->u_alt : h->u, h->b, h->dev_out,
                            h->capture);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(h->host_out, h->dev_out, sizeof(ResidualOut),
                            cudaMemcpyDeviceToHost, h->capture);
    cudaGraph_t graph = nullptr;
    cudaError_t e2 = cudaStreamEndCapture(h->capture, &graph);
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess) e = cudaGraphInstantiate(exec, graph, 0);
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess)
        return fail(h, JACOBI_ERR_CUDA, "recording the check graph: %s",
                    cudaGetErrorString(e));
    return JACOBI_OK;
}

// Check intervals per iteration of the device-side loop. A loop iteration
// costs a few launches' worth of time, so an iteration runs about `target`
// launches (those after the stop return at entry, so some are wasted per
// time step): 16 from N = 1024 on, where launches are long enough for the
// saved iterations to win, 8 below (measured on GB300). Even when an
// interval has an odd number of launches, so that the body ends in u.
long long intervals_per_iteration(long long launches_per_check, int n) {
    const long long target = n >= 1024 ? 16 : 8;
    const long long k =
        launches_per_check >= target ? 1 : target / launches_per_check;
    return (launches_per_check % 2 == 1 && k % 2 == 1) ? k + 1 : k;
}

// The body of the device-side loop for the step whose state is `st`, into
// the stream being captured: intervals_per_iteration() check intervals
// starting from u, each with a fused first launch and the rest honouring the
// stop flag, then the kernel that ends the loop once the step has stopped.
cudaError_t capture_body(jacobi_handle_t *h, LoopState *st,
                         cudaGraphConditionalHandle cond, int start = 0) {
    const long long L = h->launches_per_check;
    const long long halves = intervals_per_iteration(L, h->g.n);
    int src = start;
    cudaError_t e = cudaSuccess;
    for (long long half = 0; half < halves && e == cudaSuccess; ++half)
        for (long long l = 0; l < L && e == cudaSuccess; ++l) {
            e = enqueue_launch(h, src, h->capture,
                               loop_ctl(h, st, l == 0, src, cond));
            src ^= 1;
        }
    if (e == cudaSuccess) e = launch_loop_condition(st, cond, h->capture);
    return e;
}

// Persistent control: the one cooperative launch that runs the step whose
// state is `st`, from u (its answer lands in u or u_alt, LoopState::where).
cudaError_t enqueue_persistent(jacobi_handle_t *h, LoopState *st,
                               cudaStream_t s) {
    const LaunchCtl c = loop_ctl(h, st, true, 0, cudaGraphConditionalHandle{});
    return launch_etb_persistent(h->g, h->tc, &h->map_u, &h->map_alt, &h->map_b,
                                 h->u, h->u_alt, c.lp, h->launches_per_check, s);
}

// Persistent control: record the graph of one time step,
//   reset(LoopState) -> bmax of b -> persistent step -> copy LoopState to
//   the host.
int record_step_persistent(jacobi_handle_t *h) {
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(h->capture, cudaStreamCaptureModeThreadLocal);
    auto check = [&](cudaError_t err) {
        if (e == cudaSuccess) e = err;
        return e == cudaSuccess;
    };
    if (e == cudaSuccess) {
        check(launch_loop_reset(h->loop, nullptr, h->capture));
        check(launch_bnorm(h->g, h->u, h->b, h->loop, h->capture));
        check(enqueue_persistent(h, h->loop, h->capture));
        check(cudaMemcpyAsync(h->loop_host, h->loop, sizeof(LoopState),
                              cudaMemcpyDeviceToHost, h->capture));
        cudaError_t e2 = cudaStreamEndCapture(h->capture, &graph);
        check(e2);
    }
    if (e == cudaSuccess) check(cudaGraphInstantiate(&h->step, graph, 0));
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, JACOBI_ERR_CUDA, "recording the persistent step graph: %s",
                    cudaGetErrorString(e));
    }
    return JACOBI_OK;
}

// Device control: record the graph of one time step,
//   reset(LoopState) -> bmax of b -> WHILE(cond) { body } -> copy LoopState
//   to the host,
// where the body is intervals_per_iteration() check intervals starting from u,
// each with a fused first launch and the rest honouring the stop flag.
int record_step(jacobi_handle_t *h) {
    if (h->cfg.control == JACOBI_CONTROL_PERSISTENT) return record_step_persistent(h);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaGraphCreate(&graph, 0);
    cudaGraphConditionalHandle cond{};
    cudaGraphNode_t head_node = nullptr, loop_node = nullptr;
    auto check = [&](cudaError_t err) {
        if (e == cudaSuccess) e = err;
        return e == cudaSuccess;
    };
    if (check(e) &&
        check(cudaGraphConditionalHandleCreate(&cond, graph, 1,
                                               cudaGraphCondAssignDefault)) &&
        check(cudaStreamBeginCaptureToGraph(h->capture, graph, nullptr, nullptr,
                                            0, cudaStreamCaptureModeThreadLocal))) {
        check(launch_loop_reset(h->loop, nullptr, h->capture));
        // bmax of the step's right-hand side, once per step (b is fixed).
        check(launch_bnorm(h->g, h->u, h->b, h->loop, h->capture));
        // The loop node follows the last node captured so far.
        cudaStreamCaptureStatus cs;
        const cudaGraphNode_t *deps = nullptr;
        size_t ndeps = 0;
        if (check(cudaStreamGetCaptureInfo(h->capture, &cs, nullptr, nullptr,
                                           &deps, nullptr, &ndeps))) {
            if (ndeps == 1) head_node = deps[0];
            else check(cudaErrorStreamCaptureUnmatched);
        }
        cudaGraph_t g2 = nullptr;
        check(cudaStreamEndCapture(h->capture, &g2));
    }
    cudaGraph_t body = nullptr;
    if (e == cudaSuccess) {
        cudaGraphNodeParams p = {};
        p.type = cudaGraphNodeTypeConditional;
        p.conditional.handle = cond;
        p.conditional.type = cudaGraphCondTypeWhile;
        p.conditional.size = 1;
        if (check(cudaGraphAddNode(&loop_node, graph, &head_node, nullptr, 1, &p)))
            body = p.conditional.phGraph_out[0];
    }
    if (e == cudaSuccess &&
        check(cudaStreamBeginCaptureToGraph(h->capture, body, nullptr, nullptr,
                                            0, cudaStreamCaptureModeThreadLocal))) {
        check(capture_body(h, h->loop, cond));
        cudaGraph_t g2 = nullptr;
        check(cudaStreamEndCapture(h->capture, &g2));
    }
    if (e == cudaSuccess &&
        check(cudaStreamBeginCaptureToGraph(h->capture, graph, &loop_node,
                                            nullptr, 1,
                                            cudaStreamCaptureModeThreadLocal))) {
        check(cudaMemcpyAsync(h->loop_host, h->loop, sizeof(LoopState),
                              cudaMemcpyDeviceToHost, h->capture));
        cudaGraph_t g2 = nullptr;
        check(cudaStreamEndCapture(h->capture, &g2));
    }
    if (e == cudaSuccess) check(cudaGraphInstantiate(&h->step, graph, 0));
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, JACOBI_ERR_CUDA, "recording the device-loop graph: %s",
                    cudaGetErrorString(e));
    }
    return JACOBI_OK;
}

// Device control, whole run: one graph for `steps` time steps with source g
// (section 01: a run is successive backward-Euler steps). Step s is
//   right-hand side -> reset(state s) -> bmax -> WHILE(cond s) { body }
//   [-> settle: answer back into u, when intervals have an odd launch count]
// and a single copy of all steps' states to pinned memory ends the graph.
// A step whose predecessor did not converge is skipped on the device.
// Persistent control, whole run: per step the right-hand side, the reset of
// that step's state (skipped after a failed step), bmax, the persistent
// step and the settle kernel (the answer may sit in u_alt), then one copy of
// all step states to pinned memory.
int record_run_persistent(jacobi_handle_t *h, const float *g, int steps) {
    if (h->run) cudaGraphExecDestroy(h->run);
    h->run = nullptr;
    h->run_g = nullptr;
    h->run_steps = 0;
    if (steps > h->run_cap) {
        if (h->run_states) cudaFree(h->run_states);
        if (h->run_states_host) cudaFreeHost(h->run_states_host);
        h->run_states = nullptr;
        h->run_states_host = nullptr;
        h->run_cap = 0;
        TBJ_CUDA(h, cudaMalloc(&h->run_states, sizeof(LoopState) * steps));
        TBJ_CUDA(h, cudaMallocHost(&h->run_states_host, sizeof(LoopState) * steps));
        h->run_cap = steps;
    }
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(h->capture, cudaStreamCaptureModeThreadLocal);
    auto check = [&](cudaError_t err) {
        if (e == cudaSuccess) e = err;
        return e == cudaSuccess;
    };
    if (e == cudaSuccess) {
        for (int s = 0; s < steps && e == cudaSuccess; ++s) {
            LoopState *st = h->run_states + s;
            check(launch_rhs(h->g, h->u, g, h->b, h->capture));
            check(launch_loop_reset(st, s ? st - 1 : nullptr, h->capture));
            check(launch_bnorm(h->g, h->u, h->b, st, h->capture));
            check(enqueue_persistent(h, st, h->capture));
            check(launch_settle(h->g, st, h->u_alt, h->u, h->capture));
        }
        check(cudaMemcpyAsync(h->run_states_host, h->run_states,
                              sizeof(LoopState) * steps, cudaMemcpyDeviceToHost,
                              h->capture));
        cudaError_t e2 = cudaStreamEndCapture(h->capture, &graph);
        check(e2);
    }
    if (e == cudaSuccess) check(cudaGraphInstantiate(&h->run, graph, 0));
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, JACOBI_ERR_CUDA, "recording the persistent run graph: %s",
                    cudaGetErrorString(e));
    }
    h->run_g = g;
    h->run_steps = steps;
    return JACOBI_OK;
}

// Whether a device-controlled run starts each step with a sweep launch that
// forms the right-hand side b = u^n + g itself (and the cells of bmax
// without ring neighbours) from the u^n it reads, in place of k_rhs and
// k_bnorm: the column-streamed ETB kernel, with one launch per check
// interval (that first launch is the step's first interval, which has no
// check: section 01, the first check comes after M sweeps).
bool rhs_first_launch(const jacobi_handle_t *h) {
    return h->cfg.control == JACOBI_CONTROL_DEVICE &&
           h->cfg.rhs == JACOBI_RHS_FUSED &&
           h->cfg.strategy == JACOBI_EXACT_TEMPORAL_BLOCKED &&
           h->tc.variant == kEtbsVariant && h->launches_per_check == 1;
}

// Capture what `fn` enqueues on the capture stream into graph `gr`, after
// node `dep` (null: none); *last receives the one node it ends in.
template <class F>
cudaError_t capture_into(jacobi_handle_t *h, cudaGraph_t gr, cudaGraphNode_t dep,
                         F fn, cudaGraphNode_t *last) {
    cudaError_t e = cudaStreamBeginCaptureToGraph(
        h->capture, gr, dep ? &dep : nullptr, nullptr, dep ? 1 : 0,
        cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return e;
    e = fn();
    if (e == cudaSuccess && last) {
        cudaStreamCaptureStatus cs;
        const cudaGraphNode_t *deps = nullptr;
        size_t ndeps = 0;
        e = cudaStreamGetCaptureInfo(h->capture, &cs, nullptr, nullptr, &deps,
                                     nullptr, &ndeps);
        if (e == cudaSuccess) {
            if (ndeps == 1) *last = deps[0];
            else e = cudaErrorStreamCaptureUnmatched;
        }
    }
    cudaGraph_t g2 = nullptr;
    cudaError_t e2 = cudaStreamEndCapture(h->capture, &g2);
    return e != cudaSuccess ? e : e2;
}

// One way through a step of a run that starts each step with the launch
// that forms b (rhs_first_launch), into graph `gr` after `dep`, for u^n in
// buffer `sb` (0: u, 1: u_alt): bmax of the ring-adjacent cells -> the first
// launch, sb -> the other buffer -> WHILE(cond) { loop body from there }.
cudaError_t add_rhs_first_step(jacobi_handle_t *h, cudaGraph_t gr,
                               cudaGraphNode_t dep, LoopState *st,
                               const float *g, int sb,
                               cudaGraphNode_t *loop_out) {
    cudaGraphConditionalHandle cond{};
    cudaError_t e = cudaGraphConditionalHandleCreate(&cond, gr, 1,
                                                     cudaGraphCondAssignDefault);
    cudaGraphNode_t head = nullptr;
    if (e == cudaSuccess)
        e = capture_into(h, gr, dep, [&]() {
            cudaError_t r = launch_bnorm_ring(h->g, sb ? h->u_alt : h->u, g, st,
                                              h->capture);
            if (r != cudaSuccess) return r;
            LaunchCtl c = loop_ctl(h, st, false, sb, cond);
            c.rhs_g = g;
            c.rhs_b = h->b;
            return enqueue_launch(h, sb, h->capture, c);
        }, &head);
    cudaGraph_t body = nullptr;
    if (e == cudaSuccess) {
        cudaGraphNodeParams p = {};
        p.type = cudaGraphNodeTypeConditional;
        p.conditional.handle = cond;
        p.conditional.type = cudaGraphCondTypeWhile;
        p.conditional.size = 1;
        cudaGraphNode_t loop_node = nullptr;
        e = cudaGraphAddNode(&loop_node, gr, &head, nullptr, 1, &p);
        if (e == cudaSuccess) body = p.conditional.phGraph_out[0];
        if (loop_out) *loop_out = loop_node;
    }
    if (e == cudaSuccess)
        e = capture_into(h, body, nullptr,
                         [&]() { return capture_body(h, st, cond, 1 - sb); }, nullptr);
    return e;
}

// Device control, whole run, each step starting with the launch that forms
// b. A step's answer stays in whichever buffer holds it, and the next step
// starts from there: step s > 0 is an if/else node on the previous step's
// LoopState::where whose two branches are add_rhs_first_step from u and
// from u_alt (step 0 starts from u). Only the run's answer is moved into u,
// at the end:
//   [reset(s) -> choose branch -> IF { from u } ELSE { from u_alt }] x steps
//   -> settle (u_alt -> u when the last answer is there) -> states to host
int record_run_rhs_first(jacobi_handle_t *h, const float *g, int steps) {
    if (steps < 1)
        return fail(h, JACOBI_ERR_INVALID_ARG, "a run graph needs steps >= 1");
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaGraphCreate(&graph, 0);
    cudaGraphNode_t prev = nullptr;
    for (int s = 0; s < steps && e == cudaSuccess; ++s) {
        LoopState *st = h->run_states + s;
        LoopState *pst = s ? st - 1 : nullptr;
        cudaGraphConditionalHandle ifc{};
        if (s > 0)
            e = cudaGraphConditionalHandleCreate(&ifc, graph, 0,
                                                 cudaGraphCondAssignDefault);
        cudaGraphNode_t head = nullptr;
        if (e == cudaSuccess)
            e = capture_into(h, graph, prev, [&]() {
                cudaError_t r = launch_loop_reset(st, pst, h->capture,
                                                  h->interval, true);
                if (r == cudaSuccess && s > 0)
                    r = launch_branch_on_where(pst, ifc, h->capture);
                return r;
            }, &head);
        if (e != cudaSuccess) break;
        if (s == 0) {
            e = add_rhs_first_step(h, graph, head, st, g, 0, &prev);
        } else {
            cudaGraphNodeParams p = {};
            p.type = cudaGraphNodeTypeConditional;
            p.conditional.handle = ifc;
            p.conditional.type = cudaGraphCondTypeIf;
            p.conditional.size = 2;
            cudaGraphNode_t if_node = nullptr;
            e = cudaGraphAddNode(&if_node, graph, &head, nullptr, 1, &p);
            if (e == cudaSuccess)
                e = add_rhs_first_step(h, p.conditional.phGraph_out[0], nullptr,
                                       st, g, 0, nullptr);
            if (e == cudaSuccess)
                e = add_rhs_first_step(h, p.conditional.phGraph_out[1], nullptr,
                                       st, g, 1, nullptr);
            prev = if_node;
        }
    }
    LoopState *last_st = h->run_states + (steps - 1);
    if (e == cudaSuccess)
        e = capture_into(h, graph, prev, [&]() {
            cudaError_t r = launch_settle(h->g, last_st, h->u_alt, h->u, h->capture);
            if (r == cudaSuccess)
                r = cudaMemcpyAsync(h->run_states_host, h->run_states,
                                    sizeof(LoopState) * steps,
                                    cudaMemcpyDeviceToHost, h->capture);
            return r;
        }, nullptr);
    if (e == cudaSuccess) e = cudaGraphInstantiate(&h->run, graph, 0);
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, JACOBI_ERR_CUDA, "recording the run graph: %s",
                    cudaGetErrorString(e));
    }
    h->run_rhs_first = true;
    h->run_g = g;
    h->run_steps = steps;
    return JACOBI_OK;
}

int record_run(jacobi_handle_t *h, const float *g, int steps) {
    h->run_rhs_first = false;
    if (h->cfg.control == JACOBI_CONTROL_PERSISTENT)
        return record_run_persistent(h, g, steps);
    if (h->run) cudaGraphExecDestroy(h->run);
    h->run = nullptr;
    h->run_g = nullptr;
    h->run_steps = 0;
    if (steps > h->run_cap) {
        if (h->run_states) cudaFree(h->run_states);
        if (h->run_states_host) cudaFreeHost(h->run_states_host);
        h->run_states = nullptr;
        h->run_states_host = nullptr;
        h->run_cap = 0;
        TBJ_CUDA(h, cudaMalloc(&h->run_states, sizeof(LoopState) * steps));
        TBJ_CUDA(h, cudaMallocHost(&h->run_states_host, sizeof(LoopState) * steps));
        h->run_cap = steps;
    }
    if (rhs_first_launch(h)) return record_run_rhs_first(h, g, steps);
    const bool settle_needed = h->launches_per_check % 2 == 1;
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaGraphCreate(&graph, 0);
    auto check = [&](cudaError_t err) {
        if (e == cudaSuccess) e = err;
        return e == cudaSuccess;
    };
    cudaGraphNode_t prev = nullptr;  // last node of the previous step
    for (int s = 0; s < steps && e == cudaSuccess; ++s) {
        LoopState *st = h->run_states + s;
        cudaGraphConditionalHandle cond{};
        cudaGraphNode_t head = nullptr, loop_node = nullptr;
        check(cudaGraphConditionalHandleCreate(&cond, graph, 1,
                                               cudaGraphCondAssignDefault));
        if (e == cudaSuccess &&
            check(cudaStreamBeginCaptureToGraph(
                h->capture, graph, prev ? &prev : nullptr, nullptr,
                prev ? 1 : 0, cudaStreamCaptureModeThreadLocal))) {
            if (h->cfg.rhs == JACOBI_RHS_UNFUSED) {
                if (s == 0) check(launch_copy_interior(h->g, g, h->g_copy, h->capture));
                check(launch_copy_interior(h->g, h->u, h->b, h->capture));
            } else {
                check(launch_rhs(h->g, h->u, g, h->b, h->capture));
            }
            check(launch_loop_reset(st, s ? st - 1 : nullptr, h->capture));
            check(launch_bnorm(h->g, h->u, h->b, st, h->capture));
            cudaStreamCaptureStatus cs;
            const cudaGraphNode_t *deps = nullptr;
            size_t ndeps = 0;
            if (check(cudaStreamGetCaptureInfo(h->capture, &cs, nullptr, nullptr,
                                               &deps, nullptr, &ndeps))) {
                if (ndeps == 1) head = deps[0];
                else check(cudaErrorStreamCaptureUnmatched);
            }
            cudaGraph_t g2 = nullptr;
            check(cudaStreamEndCapture(h->capture, &g2));
        }
        cudaGraph_t body = nullptr;
        if (e == cudaSuccess) {
            cudaGraphNodeParams p = {};
            p.type = cudaGraphNodeTypeConditional;
            p.conditional.handle = cond;
            p.conditional.type = cudaGraphCondTypeWhile;
            p.conditional.size = 1;
            if (check(cudaGraphAddNode(&loop_node, graph, &head, nullptr, 1, &p)))
                body = p.conditional.phGraph_out[0];
        }
        if (e == cudaSuccess &&
            check(cudaStreamBeginCaptureToGraph(h->capture, body, nullptr, nullptr,
                                                0, cudaStreamCaptureModeThreadLocal))) {
            check(capture_body(h, st, cond));
            cudaGraph_t g2 = nullptr;
            check(cudaStreamEndCapture(h->capture, &g2));
        }
        prev = loop_node;
        if (settle_needed && e == cudaSuccess &&
            check(cudaStreamBeginCaptureToGraph(h->capture, graph, &loop_node,
                                                nullptr, 1,
                                                cudaStreamCaptureModeThreadLocal))) {
            check(launch_settle(h->g, st, h->u_alt, h->u, h->capture));
            cudaStreamCaptureStatus cs;
            const cudaGraphNode_t *deps = nullptr;
            size_t ndeps = 0;
            if (check(cudaStreamGetCaptureInfo(h->capture, &cs, nullptr, nullptr,
                                               &deps, nullptr, &ndeps))) {
                if (ndeps == 1) prev = deps[0];
                else check(cudaErrorStreamCaptureUnmatched);
            }
            cudaGraph_t g2 = nullptr;
            check(cudaStreamEndCapture(h->capture, &g2));
        }
    }
    if (e == cudaSuccess &&
        check(cudaStreamBeginCaptureToGraph(h->capture, graph, &prev, nullptr, 1,
                                            cudaStreamCaptureModeThreadLocal))) {
        check(cudaMemcpyAsync(h->run_states_host, h->run_states,
                              sizeof(LoopState) * steps, cudaMemcpyDeviceToHost,
                              h->capture));
        cudaGraph_t g2 = nullptr;
        check(cudaStreamEndCapture(h->capture, &g2));
    }
    if (e == cudaSuccess) check(cudaGraphInstantiate(&h->run, graph, 0));
    if (graph) cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, JACOBI_ERR_CUDA, "recording the run graph: %s",
                    cudaGetErrorString(e));
    }
    h->run_g = g;
    h->run_steps = steps;
    return JACOBI_OK;
}

// Is the fixed-divisor division bit-identical to IEEE division for every
// finite numerator with this d? Checked exhaustively on the device once per
// distinct d per process.
std::mutex g_fastdiv_mutex;
std::map<unsigned, bool> g_fastdiv_ok;

int fast_division_ok(jacobi_handle_t *h, bool *ok) {
    unsigned key;
    std::memcpy(&key, &h->g.d, sizeof key);
    {
        std::lock_guard<std::mutex> lock(g_fastdiv_mutex);
        auto it = g_fastdiv_ok.find(key);
        if (it != g_fastdiv_ok.end()) {
            *ok = it->second;
            return JACOBI_OK;
        }
    }
    unsigned long long *count = nullptr, host = ~0ull;
    cudaError_t e = cudaMalloc(&count, sizeof *count);
    if (e == cudaSuccess) e = cudaMemsetAsync(count, 0, sizeof *count, h->stream);
    if (e == cudaSuccess) e = fastdiv_verify_launch(h->g.d, h->g.y, count, h->stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(&host, count, sizeof host, cudaMemcpyDeviceToHost,
                            h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    if (count) cudaFree(count);
    if (e != cudaSuccess)
        return fail(h, JACOBI_ERR_CUDA, "checking the fixed-divisor division: %s",
                    cudaGetErrorString(e));
    *ok = (host == 0);
    std::lock_guard<std::mutex> lock(g_fastdiv_mutex);
    g_fastdiv_ok[key] = *ok;
    return JACOBI_OK;
}

// Column-streamed exact temporal blocking: the device work list of the
// prepared shape (counters at zero, then the row bands).
int setup_etbs_work(jacobi_handle_t *h) {
    if (h->etbs_work) {
        cudaFree(h->etbs_work);
        h->etbs_work = nullptr;
    }
    std::vector<int> list(2 + (size_t)h->g.n + 1, 0);
    const int ints = etbs_schedule(h->tc, h->g.n, list.data() + 2,
                                   (int)list.size() - 2);
    if (ints < 3)
        return fail(h, JACOBI_ERR_CUDA, "no work list for the streamed kernel");
    TBJ_CUDA(h, cudaMalloc(&h->etbs_work, sizeof(int) * ints));
    TBJ_CUDA(h, cudaMemcpy(h->etbs_work, list.data(), sizeof(int) * ints,
                           cudaMemcpyHostToDevice));
    h->tc.work = h->etbs_work;
    h->tc.bands = ints - 3;
    return JACOBI_OK;
}

// Apply a (validated) configuration: tiles, tensor maps, graphs.
int create_levels(jacobi_handle_t *h, const jacobi_config_t &c);

int apply_config(jacobi_handle_t *h, const jacobi_config_t &c) {
    destroy_graphs(h);
    destroy_levels(h);
    h->cfg = c;
    h->g.fast = false;
    if (c.division == JACOBI_DIVISION_AUTO) {
        bool ok = false;
        int rc = fast_division_ok(h, &ok);
        if (rc) return rc;
        h->g.fast = ok;
    }
    if (c.rhs == JACOBI_RHS_UNFUSED) {
        if (!h->g_copy)
        {
            const size_t bytes = sizeof(float) * (size_t)h->g.n * (size_t)h->g.ld;
            TBJ_CUDA(h, cudaMalloc(&h->g_copy, bytes));
            // Ring and padding are read (never used) by the sweeps.
            TBJ_CUDA(h, cudaMemsetAsync(h->g_copy, 0, bytes, h->stream));
        }
        h->g.g2 = h->g_copy;
    } else {
        h->g.g2 = nullptr;
    }
    int rc = 0;
    if (c.strategy == JACOBI_EXACT_TEMPORAL_BLOCKED)
        rc = etb_configure(h->g.n, c.depth, c.tile_x, c.tile_y, &h->tc,
                           c.control != JACOBI_CONTROL_PERSISTENT);
    else if (c.strategy == JACOBI_BLOCK_ASYNC)
        rc = ba_configure(h->g.n, c.depth, c.tile_x, c.tile_y, c.overlap_x,
                          c.overlap_y, &h->tc);
    if (rc == -1)
        return fail(h, JACOBI_ERR_INVALID_ARG,
                    "tile %dx%d (overlap %dx%d) not valid for this strategy "
                    "(tile_x a multiple of 4, overlaps smaller than the tile)",
                    c.tile_x, c.tile_y, c.overlap_x, c.overlap_y);
    if (rc)
        return fail(h, JACOBI_ERR_UNSUPPORTED,
                    "tile %dx%d with depth %d needs a TMA box over 256 or more "
                    "shared memory than a block can have",
                    c.tile_x, c.tile_y, c.depth);
    if (c.strategy != JACOBI_SYNC) {
        if ((rc = make_map(h, &h->map_u, h->u)) ||
            (rc = make_map(h, &h->map_alt, h->u_alt)) ||
            (rc = make_map(h, &h->map_b, h->b)))
            return rc;
        TBJ_CUDA(h, c.strategy == JACOBI_EXACT_TEMPORAL_BLOCKED
                        ? prepare_sweep_etb(h->tc, h->g.n)
                        : prepare_sweep_ba(h->tc));
        if (c.strategy == JACOBI_EXACT_TEMPORAL_BLOCKED &&
            h->tc.variant == kEtbsVariant && (rc = setup_etbs_work(h)))
            return rc;
    }
    if (c.control == JACOBI_CONTROL_PERSISTENT) {
        if (!etb_persistent_ok(h->tc))
            return fail(h, JACOBI_ERR_UNSUPPORTED,
                        "JACOBI_CONTROL_PERSISTENT needs a tile shape held in "
                        "registers (the default tile of D = 4, 8 or 16)");
        TBJ_CUDA(h, prepare_etb_persistent(h->tc, h->g.n));
    }
    h->per_launch = c.strategy == JACOBI_SYNC ? 1 : c.depth;
    h->interval = (long long)c.check_every /
                  gcd_ll(c.check_every, h->per_launch) * h->per_launch;
    h->launches_per_check = h->interval / h->per_launch;
    if (c.control != JACOBI_CONTROL_HOST) return record_step(h);
    if ((rc = record_batch(h, 0, &h->batch[0]))) return rc;
    if (h->launches_per_check % 2 == 1)
        if ((rc = record_batch(h, 1, &h->batch[1]))) return rc;
    if (c.adapt != JACOBI_ADAPT_NONE) return create_levels(h, c);
    return JACOBI_OK;
}

// The fixed-depth handles an adaptive handle switches between. Each one's
// check graphs exist for both start buffers, since the iterate may sit in
// either when the controller picks its depth.
int create_levels(jacobi_handle_t *h, const jacobi_config_t &c) {
    jacobi_config_t lc = c;
    lc.adapt = JACOBI_ADAPT_NONE;
    lc.control = JACOBI_CONTROL_HOST;
    int k = 0;
    for (int d = 1; d <= c.depth; d *= 2, ++k) {
        lc.depth = d;
        jacobi_handle_t *l = nullptr;
        int rc = jacobi_create(&l, h->g.n, h->g.ld, h->g.r, &lc, h->u,
                               h->u_alt, h->b, h->stream);
        if (rc) {
            fail(h, rc, "creating the depth-%d solver: %s", d,
                 jacobi_last_error(nullptr));
            destroy_levels(h);
            return rc;
        }
        h->level[k] = l;
        h->nlevels = k + 1;
        for (int start = 0; start < 2; ++start) {
            if (l->batch[start]) continue;
            if ((rc = record_batch(l, start, &l->batch[start]))) {
                fail(h, rc, "depth-%d solver: %s", d, l->err);
                destroy_levels(h);
                return rc;
            }
        }
    }
    for (auto &e : h->ev)
        if (!e) TBJ_CUDA(h, cudaEventCreate(&e));
    return JACOBI_OK;
}

// Bring the iterate back into u if it sits in u_alt.
int settle(jacobi_handle_t *h) {
    if (h->cur == 1) {
        TBJ_CUDA(h, launch_copy_interior(h->g, h->u_alt, h->u, h->stream));
        h->launches += 1;
        h->cur = 0;
    }
    return JACOBI_OK;
}

// What the error bits a kernel left in its status word mean.
const char *device_error_text(unsigned err) {
    if (err & ERR_BOUNDS)
        return "bounds check: a kernel access fell outside its buffer (checked "
               "build; the access was not performed)";
    if (err & ERR_TMA_TIMEOUT)
        return "a TMA load did not complete within its wait limit";
    if (err & ERR_SYNC_TIMEOUT)
        return "a grid barrier of the persistent step did not complete within "
               "its wait limit";
    return "a kernel reported an error";
}

int check_device_status(jacobi_handle_t *h, unsigned err) {
    if (err) {
        // Clear the word so the handle stays usable, then report.
        cudaMemsetAsync(&h->dev_out->err, 0, sizeof(unsigned), h->stream);
        return fail(h, JACOBI_ERR_CUDA, "%s", device_error_text(err));
    }
    return JACOBI_OK;
}

}  // namespace

extern "C" {

int jacobi_config_default(jacobi_config_t *cfg) {
    if (!cfg) return JACOBI_ERR_INVALID_ARG;
    std::memset(cfg, 0, sizeof(*cfg));
    cfg->strategy = JACOBI_SYNC;
    cfg->depth = 1;
    cfg->check_every = 8;
    cfg->tol = 1e-5;
    cfg->max_sweeps = 1ll << 22;
    cfg->control = JACOBI_CONTROL_HOST;
    cfg->division = JACOBI_DIVISION_AUTO;
    return JACOBI_OK;
}

int jacobi_create(jacobi_handle_t **out, int n, long long ld, float r,
                  const jacobi_config_t *cfg, float *u, float *u_alt,
                  float *b, void *cuda_stream) {
    if (!out) return fail(nullptr, JACOBI_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    g_create_err[0] = 0;
    if (n < 3) return fail(nullptr, JACOBI_ERR_INVALID_ARG, "n must be >= 3");
    if (ld < n || ld % 4 != 0)
        return fail(nullptr, JACOBI_ERR_INVALID_ARG,
                    "ld must be >= n and a multiple of 4 (got %lld)", ld);
    if (!std::isfinite(r) || r < 0.f)
        return fail(nullptr, JACOBI_ERR_INVALID_ARG, "r must be finite and >= 0");
    if (!u || !u_alt || !b || u == u_alt || u == b || u_alt == b)
        return fail(nullptr, JACOBI_ERR_INVALID_ARG,
                    "u, u_alt and b must be distinct non-NULL buffers");
    if (!aligned16(u) || !aligned16(u_alt) || !aligned16(b))
        return fail(nullptr, JACOBI_ERR_INVALID_ARG,
                    "u, u_alt and b must be 16-byte aligned");
    if (!is_device_pointer(u) || !is_device_pointer(u_alt) ||
        !is_device_pointer(b))
        return fail(nullptr, JACOBI_ERR_INVALID_ARG,
                    "u, u_alt and b must be device memory");
    jacobi_config_t c;
    if (cfg)
        c = *cfg;
    else
        jacobi_config_default(&c);
    int rc = check_config(nullptr, c);
    if (rc) return rc;

    jacobi_handle_t *h = new (std::nothrow) jacobi_handle_t();
    if (!h) return fail(nullptr, JACOBI_ERR_CUDA, "out of host memory");
    h->g.n = n;
    h->g.ld = ld;
    h->g.r = r;
    {
        // d = fl(1 + fl(4 r)) in float32 (host code, -ffp-contract=off).
        volatile float four_r = 4.0f * r;
        h->g.d = 1.0f + four_r;
        h->g.y = reciprocal_rn(h->g.d);
        h->g.fast = false;
    }
    h->u = u;
    h->u_alt = u_alt;
    h->b = b;
    h->stream = static_cast<cudaStream_t>(cuda_stream);
    auto bail = [&](int status) {
        std::snprintf(g_create_err, sizeof g_create_err, "%s", h->err);
        jacobi_destroy(h);
        return status;
    };
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&h->capture, cudaStreamNonBlocking)) ||
        (e = cudaMalloc(&h->dev_out, sizeof(ResidualOut))) ||
        (e = cudaMallocHost(&h->host_out, sizeof(ResidualOut))) ||
        (e = cudaMalloc(&h->loop, sizeof(LoopState))) ||
        (e = cudaMallocHost(&h->loop_host, sizeof(LoopState))) ||
        (e = cudaMemsetAsync(h->loop, 0, sizeof(LoopState), h->stream)) ||
        (e = cudaMemsetAsync(h->dev_out, 0, sizeof(ResidualOut), h->stream)) ||
        // Both ping-pong buffers carry the same Dirichlet ring.
        (e = cudaMemcpyAsync(u_alt, u, sizeof(float) * (size_t)n * (size_t)ld,
                             cudaMemcpyDeviceToDevice, h->stream))) {
        fail(h, JACOBI_ERR_CUDA, "allocating solver state: %s",
             cudaGetErrorString(e));
        return bail(JACOBI_ERR_CUDA);
    }
    std::memset(h->host_out, 0, sizeof(ResidualOut));
    std::memset(h->loop_host, 0, sizeof(LoopState));
    if ((rc = apply_config(h, c))) return bail(rc);
    *out = h;
    return JACOBI_OK;
}

int jacobi_rhs(jacobi_handle_t *h, const float *g) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    if (!g || !aligned16(g))
        return fail(h, JACOBI_ERR_INVALID_ARG, "g must be a 16-byte aligned buffer");
    int rc = settle(h);
    if (rc) return rc;
    if (h->cfg.rhs == JACOBI_RHS_UNFUSED) {
        TBJ_CUDA(h, launch_copy_interior(h->g, h->u, h->b, h->stream));
        TBJ_CUDA(h, launch_copy_interior(h->g, g, h->g_copy, h->stream));
        h->launches += 2;
    } else {
        TBJ_CUDA(h, launch_rhs(h->g, h->u, g, h->b, h->stream));
        h->launches += 1;
    }
    h->b_mode = h->cfg.rhs;
    return JACOBI_OK;
}

// b must have been prepared by jacobi_rhs for the current rhs mode.
static int check_b_mode(jacobi_handle_t *h) {
    if (h->b_mode != -1 && h->b_mode != h->cfg.rhs)
        return fail(h, JACOBI_ERR_INVALID_ARG,
                    "the right-hand side was prepared for the other rhs mode; "
                    "call jacobi_rhs again");
    return JACOBI_OK;
}

// One time step with the device-side loop: one graph launch, one sync.
// Kernels one device-side step ran: reset + bmax, then per loop iteration
// the body (no-op launches after the stop included) and its condition
// kernel. A skipped step runs one iteration of no-ops.
static long long device_step_launches(const jacobi_handle_t *h,
                                      const LoopState &st,
                                      bool rhs_first = false) {
    // persistent: reset, bmax and the one cooperative launch
    if (h->cfg.control == JACOBI_CONTROL_PERSISTENT) return 3;
    const long long per_body = intervals_per_iteration(h->launches_per_check, h->g.n);
    // Intervals the loop ran: one per check up to the deciding one, plus
    // the unchecked first interval unless the step's first launch (with
    // the reset and the ring part of bmax) ran ahead of the loop.
    const long long checks = st.status == kStepSkipped
                                 ? 1
                                 : st.result_k / h->interval + (rhs_first ? 0 : 1);
    const long long iters = (checks + per_body - 1) / per_body;
    return (rhs_first ? 3 : 2) + iters * (per_body * h->launches_per_check + 1);
}

// Outcome of a device-side step from its final state: sweeps or a status.
static long long device_step_outcome(jacobi_handle_t *h, const LoopState &st) {
    if (!st.stop)
        return fail(h, JACOBI_ERR_CUDA, "device loop ended without a decision");
    if (st.err) return fail(h, JACOBI_ERR_CUDA, "%s", device_error_text(st.err));
    switch (st.status) {
        case 0:
            return st.result_k;
        case JACOBI_ERR_NONFINITE:
            return fail(h, JACOBI_ERR_NONFINITE,
                        "residual norms not finite (rmax=%g, bmax=%g) after "
                        "%lld sweeps",
                        (double)st.rmax, (double)st.bmax, st.result_k);
        case JACOBI_ERR_NOT_CONVERGED:
            return fail(h, JACOBI_ERR_NOT_CONVERGED,
                        "not converged after %lld sweeps (rho=%g)", st.result_k,
                        st.bmax > 0 ? (double)st.rmax / st.bmax : (double)st.rmax);
        default:
            return fail(h, JACOBI_ERR_CUDA, "device loop failed (%d)", st.status);
    }
}

static long long solve_step_device(jacobi_handle_t *h) {
    TBJ_CUDA(h, cudaGraphLaunch(h->step, h->stream));
    TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
    const LoopState st = *h->loop_host;
    h->launches += device_step_launches(h, st);
    if (st.stop) {
        h->cur = st.where;
        int rc = settle(h);
        if (rc) return rc;
        TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
    }
    return device_step_outcome(h, st);
}

// A whole run under device control: one graph launch, one synchronisation.
static long long run_device(jacobi_handle_t *h, const float *g, int steps,
                            long long *sweeps_per_step) {
    int rc = settle(h);
    if (rc) return rc;
    if (!h->run || h->run_g != g || h->run_steps != steps)
        if ((rc = record_run(h, g, steps))) return rc;
    TBJ_CUDA(h, cudaGraphLaunch(h->run, h->stream));
    TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
    h->b_mode = h->cfg.rhs;
    const bool rf = h->run_rhs_first;
    const bool settle_each = !rf && (h->launches_per_check % 2 == 1 ||
                                     h->cfg.control == JACOBI_CONTROL_PERSISTENT);
    // Kernels step s ran: its own (device_step_launches) plus, when steps
    // start with the launch that forms b, the branch choice of steps > 0;
    // otherwise the right-hand side (two copies for the first unfused step)
    // and the per-step settle where intervals have an odd launch count.
    auto step_launches = [&](int s, const LoopState &st) {
        long long n = device_step_launches(h, st, rf);
        if (rf) return n + (s > 0 ? 1 : 0);
        return n + ((h->cfg.rhs == JACOBI_RHS_UNFUSED && s == 0) ? 2 : 1) +
               (settle_each ? 1 : 0);
    };
    long long total = 0;
    for (int s = 0; s < steps; ++s) {
        const LoopState st = h->run_states_host[s];
        h->launches += step_launches(s, st);
        const long long k = device_step_outcome(h, st);
        if (sweeps_per_step) sweeps_per_step[s] = k;
        if (k < 0) {
            // later steps were skipped on the device: count their kernels
            for (int q = s + 1; q < steps; ++q)
                h->launches += step_launches(q, h->run_states_host[q]);
            if (rf) h->launches += 1;  // the run's final settle
            return k;
        }
        total += k;
    }
    if (rf) h->launches += 1;  // the run's final settle
    return total;
}

// Stopping rule at a check (section 01), shared by the host-driven loops:
// 1 = stop (converged), 0 = continue, < 0 = a status to return.
static int decide(jacobi_handle_t *h, const ResidualOut &ro, long long k) {
    const double rm = (double)ro.rmax, bm = (double)ro.bmax;
    if (!std::isfinite(rm) || !std::isfinite(bm))
        return fail(h, JACOBI_ERR_NONFINITE,
                    "residual norms not finite (rmax=%g, bmax=%g) after %lld "
                    "sweeps",
                    rm, bm, k);
    if (rm == 0.0 || rm < h->cfg.tol * bm) return 1;
    if (k >= h->cfg.max_sweeps)
        return fail(h, JACOBI_ERR_NOT_CONVERGED,
                    "not converged after %lld sweeps (rho=%g)", k,
                    bm > 0 ? rm / bm : rm);
    return 0;
}

static jacobi_check_record_t check_record(int depth, long long k,
                                          const ResidualOut &ro, float ms) {
    jacobi_check_record_t rec;
    std::memset(&rec, 0, sizeof rec);
    rec.depth = depth;
    rec.sweeps = k;
    rec.rmax = ro.rmax;
    rec.bmax = ro.bmax;
    rec.ms = ms;
    return rec;
}

// One time step under a depth controller (section 02, G-asc / G-desc /
// G-fb): each check interval runs the check graph of the fixed-depth handle
// for the controller's current D, timed with CUDA events; the controller
// then sees that check's rho and time.
static long long solve_step_adaptive(jacobi_handle_t *h) {
    jacobi_adapt_state_t st;
    if (jacobi_adapt_init(&st, h->cfg.adapt, h->cfg.depth) != JACOBI_OK)
        return fail(h, JACOBI_ERR_INVALID_ARG, "bad depth controller");
    long long k = 0;
    int status = JACOBI_OK;
    for (;;) {
        int li = 0;
        while ((1 << li) < st.depth) ++li;
        if (li >= h->nlevels || !h->level[li])
            return fail(h, JACOBI_ERR_INVALID_ARG, "no solver for depth %d",
                        st.depth);
        jacobi_handle_t *l = h->level[li];
        TBJ_CUDA(h, cudaEventRecord(h->ev[0], h->stream));
        TBJ_CUDA(h, cudaGraphLaunch(l->batch[h->cur], h->stream));
        TBJ_CUDA(h, cudaEventRecord(h->ev[1], h->stream));
        TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
        h->launches += l->launches_per_check + 1;
        if (l->launches_per_check % 2 == 1) h->cur ^= 1;
        k += l->interval;
        float ms = 0.f;
        TBJ_CUDA(h, cudaEventElapsedTime(&ms, h->ev[0], h->ev[1]));
        const ResidualOut ro = *l->host_out;
        h->trace.push_back(check_record(st.depth, k, ro, ms));
        if (check_device_status(l, ro.err)) {
            status = fail(h, JACOBI_ERR_CUDA, "%s", l->err);
            break;
        }
        const int dec = decide(h, ro, k);
        if (dec < 0) {
            status = dec;
            break;
        }
        if (dec == 1) break;
        const double rm = (double)ro.rmax, bm = (double)ro.bmax;
        const double rho = bm > 0.0 ? rm / bm : INFINITY;
        if (jacobi_adapt_next(&st, rho, (double)ms) < 0)
            return fail(h, JACOBI_ERR_INVALID_ARG, "depth controller failed");
    }
    int rc = settle(h);
    if (rc) return rc;
    TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
    return status ? status : k;
}

long long jacobi_solve_step(jacobi_handle_t *h) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    if (int rc = check_b_mode(h)) return rc;
    h->trace.clear();
    if (h->nlevels > 0) {
        int rc = settle(h);
        if (rc) return rc;
        return solve_step_adaptive(h);
    }
    if (h->cfg.control != JACOBI_CONTROL_HOST) {
        int rc = settle(h);
        if (rc) return rc;
        return solve_step_device(h);
    }
    long long k = 0;
    int status = JACOBI_OK;
    for (;;) {
        const int start = h->cur;
        TBJ_CUDA(h, cudaGraphLaunch(h->batch[start], h->stream));
        TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
        h->launches += h->launches_per_check + 1;
        if (h->launches_per_check % 2 == 1) h->cur ^= 1;
        k += h->interval;
        const ResidualOut ro = *h->host_out;
        h->trace.push_back(check_record(h->per_launch, k, ro, 0.f));
        if ((status = check_device_status(h, ro.err))) break;
        const int dec = decide(h, ro, k);
        if (dec < 0) {
            status = dec;
            break;
        }
        if (dec == 1) break;
    }
    int rc = settle(h);
    if (rc) return rc;
    TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
    return status ? status : k;
}

long long jacobi_sweeps(jacobi_handle_t *h, long long launches) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    if (launches < 0)
        return fail(h, JACOBI_ERR_INVALID_ARG, "launches must be >= 0");
    if (int rc = check_b_mode(h)) return rc;
    for (long long l = 0; l < launches; ++l) {
        TBJ_CUDA(h, enqueue_launch(h, h->cur, h->stream));
        h->cur ^= 1;
        h->launches += 1;
    }
    int rc = settle(h);
    if (rc) return rc;
    return launches * h->per_launch;
}

int jacobi_residual(jacobi_handle_t *h, float *rmax, float *bmax) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    if (!rmax || !bmax)
        return fail(h, JACOBI_ERR_INVALID_ARG, "rmax and bmax must be non-NULL");
    if (int rc0 = check_b_mode(h)) return rc0;
    int rc = settle(h);
    if (rc) return rc;
    TBJ_CUDA(h, launch_residual(h->g, h->u, h->b, h->dev_out, h->stream));
    h->launches += 1;
    TBJ_CUDA(h, cudaMemcpyAsync(h->host_out, h->dev_out, sizeof(ResidualOut),
                                cudaMemcpyDeviceToHost, h->stream));
    TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
    *rmax = h->host_out->rmax;
    *bmax = h->host_out->bmax;
    return check_device_status(h, h->host_out->err);
}

int jacobi_set_strategy(jacobi_handle_t *h, const jacobi_config_t *cfg) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    if (!cfg) return fail(h, JACOBI_ERR_INVALID_ARG, "cfg is NULL");
    int rc = check_config(h, *cfg);
    if (rc) return rc;
    if ((rc = settle(h))) return rc;
    TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
    return apply_config(h, *cfg);
}

long long jacobi_run(jacobi_handle_t *h, const float *g, int steps,
                     long long *sweeps_per_step) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    if (steps < 0) return fail(h, JACOBI_ERR_INVALID_ARG, "steps must be >= 0");
    if (steps > 0 && h->cfg.control != JACOBI_CONTROL_HOST && h->nlevels == 0) {
        if (!g || !aligned16(g))
            return fail(h, JACOBI_ERR_INVALID_ARG,
                        "g must be a 16-byte aligned buffer");
        h->trace.clear();
        return run_device(h, g, steps, sweeps_per_step);
    }
    long long total = 0;
    for (int s = 0; s < steps; ++s) {
        int rc = jacobi_rhs(h, g);
        if (rc) return rc;
        long long k = jacobi_solve_step(h);
        if (sweeps_per_step) sweeps_per_step[s] = k;
        if (k < 0) return k;
        total += k;
    }
    return total;
}

int jacobi_division_mode(const jacobi_handle_t *h) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    return h->g.fast ? 1 : 0;
}

long long jacobi_launch_count(const jacobi_handle_t *h) {
    return h ? h->launches : 0;
}

long long jacobi_check_trace(const jacobi_handle_t *h,
                             jacobi_check_record_t *rec, long long cap) {
    if (!h || cap < 0 || (cap > 0 && !rec)) return JACOBI_ERR_INVALID_ARG;
    const long long n = (long long)h->trace.size();
    for (long long i = 0; i < n && i < cap; ++i) rec[i] = h->trace[(size_t)i];
    return n;
}

void jacobi_destroy(jacobi_handle_t *h) {
    if (!h) return;
    if (h->stream || h->capture) cudaStreamSynchronize(h->stream);
    destroy_graphs(h);
    destroy_levels(h);
    if (h->run_states) cudaFree(h->run_states);
    if (h->run_states_host) cudaFreeHost(h->run_states_host);
    for (auto &e : h->ev)
        if (e) cudaEventDestroy(e);
    if (h->capture) cudaStreamDestroy(h->capture);
    if (h->etbs_work) cudaFree(h->etbs_work);
    if (h->dev_out) cudaFree(h->dev_out);
    if (h->host_out) cudaFreeHost(h->host_out);
    if (h->loop) cudaFree(h->loop);
    if (h->loop_host) cudaFreeHost(h->loop_host);
    if (h->g_copy) cudaFree(h->g_copy);
    if (h->hb_copy) cudaStreamSynchronize(h->hb_copy);
    if (h->hb_twin) jacobi_destroy(h->hb_twin);
    for (float *p : {h->hb_tu, h->hb_tualt, h->hb_g[0], h->hb_g[1]})
        if (p) cudaFree(p);
    for (cudaEvent_t e : h->hb_staged)
        if (e) cudaEventDestroy(e);
    if (h->hb_copy) cudaStreamDestroy(h->hb_copy);
    delete h;
}

long long jacobi_run_host(jacobi_handle_t *h, int count,
                          const float *const *u0_host,
                          const float *const *g_host, float *const *u_host,
                          int steps, long long *sweeps) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    if (count < 1 || steps < 1 || !u0_host || !g_host || !u_host)
        return fail(h, JACOBI_ERR_INVALID_ARG,
                    "count and steps must be >= 1 and the pointer arrays non-NULL");
    for (int i = 0; i < count; ++i)
        if (!u0_host[i] || !g_host[i] || !u_host[i])
            return fail(h, JACOBI_ERR_INVALID_ARG, "problem %d has a NULL buffer", i);
    const size_t bytes = sizeof(float) * (size_t)h->g.n * (size_t)h->g.ld;
    if (!h->hb_copy) {  // first use: the twin's fields, the sources, copy stream, events
        TBJ_CUDA(h, cudaMalloc(&h->hb_tu, bytes));
        TBJ_CUDA(h, cudaMalloc(&h->hb_tualt, bytes));
        TBJ_CUDA(h, cudaMalloc(&h->hb_g[0], bytes));
        TBJ_CUDA(h, cudaMalloc(&h->hb_g[1], bytes));
        TBJ_CUDA(h, cudaMemsetAsync(h->hb_tu, 0, bytes, h->stream));
        for (cudaEvent_t &e : h->hb_staged)
            TBJ_CUDA(h, cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        TBJ_CUDA(h, cudaStreamCreateWithFlags(&h->hb_copy, cudaStreamNonBlocking));
    }
    // The twin solves the odd problems, on its own fields and with this
    // handle's configuration, b and stream.
    if (!h->hb_twin) {
        int rc = jacobi_create(&h->hb_twin, h->g.n, h->g.ld, h->g.r, &h->cfg,
                               h->hb_tu, h->hb_tualt, h->b, h->stream);
        if (rc) {
            h->hb_twin = nullptr;
            return fail(h, rc, "creating the second solver of jacobi_run_host: %s",
                        jacobi_last_error(nullptr));
        }
    } else if (std::memcmp(&h->hb_twin->cfg, &h->cfg, sizeof h->cfg) != 0) {
        if (int rc = jacobi_set_strategy(h->hb_twin, &h->cfg))
            return fail(h, rc, "%s", jacobi_last_error(h->hb_twin));
    }
    jacobi_handle_t *hs[2] = {h, h->hb_twin};
    cudaStream_t cs = h->hb_copy;
    int rc = settle(h);  // this handle's iterate back in u before its buffers are reused
    if (rc) return rc;
    // Problem i runs on hs[i % 2]. Its inputs go straight into that
    // handle's u (and the Dirichlet ring into its u_alt) and into
    // hb_g[i % 2], on the copy stream, while problem i - 1 runs; its result
    // leaves from that u while problem i + 1 runs. The copy stream takes
    // things in order, so a pair's next inputs come in only after its last
    // result has gone out.
    TBJ_CUDA(h, cudaEventRecord(h->hb_staged[0], h->stream));
    TBJ_CUDA(h, cudaStreamWaitEvent(cs, h->hb_staged[0], 0));
    auto stage = [&](int i) -> int {
        jacobi_handle_t *t = hs[i % 2];
        TBJ_CUDA(h, cudaMemcpyAsync(t->u, u0_host[i], bytes, cudaMemcpyHostToDevice, cs));
        TBJ_CUDA(h, cudaMemcpyAsync(h->hb_g[i % 2], g_host[i], bytes,
                                    cudaMemcpyHostToDevice, cs));
        TBJ_CUDA(h, launch_copy_ring(h->g, t->u, t->u_alt, cs));
        h->launches += 1;
        TBJ_CUDA(h, cudaEventRecord(h->hb_staged[i % 2], cs));
        return JACOBI_OK;
    };
    if ((rc = stage(0))) return rc;
    long long total = 0, status = 0;
    for (int i = 0; i < count; ++i) {
        jacobi_handle_t *t = hs[i % 2];
        if (i + 1 < count && (rc = stage(i + 1))) return rc;
        TBJ_CUDA(h, cudaStreamWaitEvent(h->stream, h->hb_staged[i % 2], 0));
        t->cur = 0;
        const long long before = t->launches;
        const long long k = jacobi_run(t, h->hb_g[i % 2], steps,
                                       sweeps ? sweeps + (size_t)i * steps : nullptr);
        if (t != h) h->launches += t->launches - before;
        if (k < 0) {
            status = t == h ? k : fail(h, (int)k, "%s", jacobi_last_error(t));
            break;
        }
        total += k;
        // jacobi_run returned with the stream idle: problem i's result is in
        // t->u; it leaves on the copy stream while problem i + 1 runs.
        TBJ_CUDA(h, cudaMemcpyAsync(u_host[i], t->u, bytes, cudaMemcpyDeviceToHost, cs));
    }
    TBJ_CUDA(h, cudaStreamSynchronize(cs));
    // As documented: u holds the last problem's result (u_alt its ring).
    const int last = status ? -1 : count - 1;
    if (last >= 0 && hs[last % 2] != h) {
        TBJ_CUDA(h, cudaMemcpyAsync(h->u, h->hb_tu, bytes, cudaMemcpyDeviceToDevice,
                                    h->stream));
        TBJ_CUDA(h, launch_copy_ring(h->g, h->u, h->u_alt, h->stream));
        h->launches += 1;
        h->cur = 0;
    }
    TBJ_CUDA(h, cudaStreamSynchronize(h->stream));
    return status ? status : total;
}

int jacobi_tile(const jacobi_handle_t *h, int *tile_x, int *tile_y) {
    if (!h || !tile_x || !tile_y) return JACOBI_ERR_INVALID_ARG;
    const bool tiled = h->cfg.strategy != JACOBI_SYNC;
    *tile_x = tiled ? h->tc.tile_x : 0;
    *tile_y = tiled ? h->tc.tile_y : 0;
    return JACOBI_OK;
}

int jacobi_bounds_checked(void) { return kBoundsChecked ? 1 : 0; }

int jacobi_bounds_selftest(jacobi_handle_t *h) {
    if (!h) return JACOBI_ERR_INVALID_ARG;
    if (!kBoundsChecked)
        return fail(h, JACOBI_ERR_UNSUPPORTED,
                    "the bounds self-test needs the bounds-checked library");
    constexpr int kChecks = 5;
    unsigned *flags = nullptr;
    TBJ_CUDA(h, cudaMalloc(&flags, kChecks * sizeof(unsigned)));
    unsigned host[kChecks] = {0};
    cudaError_t e = cudaMemsetAsync(flags, 0, sizeof host, h->stream);
    if (e == cudaSuccess)
        e = launch_bounds_selftest(h->u, h->g.n, h->g.ld, flags, h->stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(host, flags, sizeof host, cudaMemcpyDeviceToHost,
                            h->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(h->stream);
    cudaFree(flags);
    if (e != cudaSuccess)
        return fail(h, JACOBI_ERR_CUDA, "bounds self-test: %s",
                    cudaGetErrorString(e));
    int mask = 0;
    for (int k = 0; k < kChecks; ++k)
        if (host[k] & ERR_BOUNDS) mask |= 1 << k;
    return mask;
}

const char *jacobi_last_error(const jacobi_handle_t *h) {
    return h ? h->err : g_create_err;
}

const char *jacobi_status_string(int status) {
    switch (status) {
        case JACOBI_OK: return "JACOBI_OK";
        case JACOBI_ERR_INVALID_ARG: return "JACOBI_ERR_INVALID_ARG";
        case JACOBI_ERR_CUDA: return "JACOBI_ERR_CUDA";
        case JACOBI_ERR_NOT_CONVERGED: return "JACOBI_ERR_NOT_CONVERGED";
        case JACOBI_ERR_NONFINITE: return "JACOBI_ERR_NONFINITE";
        case JACOBI_ERR_UNSUPPORTED: return "JACOBI_ERR_UNSUPPORTED";
        default: return "JACOBI_STATUS_UNKNOWN";
    }
}

}  // extern "C"
