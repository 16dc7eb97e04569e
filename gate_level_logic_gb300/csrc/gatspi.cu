// Host side of the GB300 gate-level re-simulator: the C ABI of include/gatspi.h.
//
// It validates and uploads the levelised netlist, owns the window index, the
// toggle statistics and the scan state on the device, borrows the caller's
// waveform pool, and enqueues one level kernel per logic level (GATSPI, Section 3,
// Fig. 5) -- captured once into a CUDA graph and replayed.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <unordered_set>
#include <vector>

#include "gatspi_internal.cuh"
#include "testbench.cuh"

using namespace gatspi;

namespace {

thread_local std::string g_err;

gatspi_status fail(gatspi_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
gatspi_status fail(gatspi_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

gatspi_status cuda_fail(cudaError_t e, const char *what) {
    if (e == cudaErrorMemoryAllocation) return fail(GATSPI_ENOMEM, "%s: %s", what, cudaGetErrorString(e));
    return fail(GATSPI_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CUDA_TRY(call, what)                     \
    do {                                         \
        cudaError_t e_ = (call);                 \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

template <class T>
cudaError_t dev_alloc(T **p, size_t n) {
    return cudaMalloc((void **)p, std::max<size_t>(n, 1) * sizeof(T));
}

}  // namespace

void gatspi_set_last_error(const char *msg) { g_err = msg ? msg : ""; }

struct gatspi_ctx {
    int device = 0;
    int32_t P = 0, G = 0, L = 0, W = 0;
    int32_t ngroups = 1, lpg_log2 = 0, slots_per_gate = 1;
    long long max_level_gates = 0;
    long long num_nets = 0;
    int32_t *pool = nullptr;
    long long pool_words = 0;
    uint32_t flags = 0;
    int32_t pulse_percent = 100;

    // device arrays owned by the context
    int4 *gate_desc = nullptr;
    int32_t *dly = nullptr;
    int32_t *gate_order = nullptr;   // W < 32: every level's gates by pin count
    int32_t *heavy_order = nullptr;  // W <= 16: a level's gates, heaviest first (level_chunk_kernel)
    uint32_t *seg_items = nullptr, *seg_count = nullptr, *seg_cnt = nullptr;   // W = 1: segments of heavy gates
    int32_t *seg_counter = nullptr;
    int32_t resident_warps = 0;
    bool compact = false;            // GATSPI_FLAG_COMPACT
    bool long_windows = false;       // the loaded inputs average kLongWindowWords words or more per window
    bool split_windows = false;      // one window of kSplitWindowWords words or more per input: segments
    bool dense_windows = false;      // kDenseWindowWords words or more per input window
    uint32_t *gexact = nullptr;      // compaction: exact words per (gate, group) of a level
    long long *old_base = nullptr;   // compaction: a level's bound-sized regions
    long long *level_bound = nullptr, *level_need = nullptr;   // compaction: [L]
    long long *net_base = nullptr;
    uint32_t *wstart = nullptr;
    uint32_t *wend = nullptr;
    uint8_t *wlen8 = nullptr;
    uint16_t *perm = nullptr;
    uint32_t *goff = nullptr;
    int32_t *window_len = nullptr;
    unsigned long long *tc = nullptr, *t1 = nullptr;
    unsigned long long *tile_status = nullptr;
    int32_t *tickets = nullptr;
    long long *level_base = nullptr;
    int32_t *status = nullptr;
    long long *load_off = nullptr;
    int32_t *max_time = nullptr;
    long long *win_start = nullptr;   // [W+1] start of every window on the testbench's time axis
    unsigned long long *tc_in = nullptr, *t1_in = nullptr;   // [P] input statistics of the last load
    std::vector<unsigned long long> tc_in_host, t1_in_host;

    // host copies
    std::vector<int32_t> level_offsets;
    std::vector<LevelLaunch> launches;
    std::vector<LevelLaunch> exact_launches;   // compaction: the scans of the exact sizes
    long long total_tiles = 0;
    long long sum_window_len = 0;
    long long path_delay_bound = 0;   // levels * (max wire delay + max gate delay)
    long long max_window_len = 0;
    bool loaded = false;
    bool simulated = false;
    bool timed_last = false;   // the last simulate recorded level events
    int32_t stall_level = -1;          // gatspi_inject_scan_stall: the level whose scan stalls in the next simulate
    long long stall_wait_ns = 0;       // and the wait limit of that simulate
    cudaStream_t last_stream = nullptr;

    // TC/T1 copied to pinned host memory level by level while later levels run
    unsigned long long *tc_host = nullptr, *t1_host = nullptr;
    cudaStream_t dump_stream = nullptr;
    std::vector<cudaEvent_t> dump_events;   // [L] after each level's simulation kernel
    cudaEvent_t dump_done = nullptr;

    // replayed level sequence
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t graph_exec = nullptr;
    cudaStream_t capture_stream = nullptr;
    std::vector<cudaEvent_t> events;

    DevParams params() const {
        DevParams p{};
        p.gate_desc = gate_desc;
        p.dly_data = dly;
        p.gate_order = gate_order;
        p.heavy_order = heavy_order;
        // segments of one window: when its windows are cut and very long, or cut by force
        const bool seg = chunks_per_window(W, flags, long_windows) > 1 &&
                         (split_windows || (flags & GATSPI_FLAG_CUT_WINDOWS));
        p.seg_items = seg ? seg_items : nullptr;
        p.seg_kernel = seg || (W >= 2 && dense_windows) ? 1 : 0;
        p.seg_count = seg_count;
        p.seg_cnt = seg_cnt;
        p.seg_counter = seg_counter;
        p.resident_warps = resident_warps;
        p.pool = pool;
        p.pool_words = pool_words;
        p.net_base = net_base;
        p.wstart = wstart;
        p.wend = wend;
        p.wlen8 = wlen8;
        p.w8stride = (W + 3) & ~3;
        p.plan_words = plan_words(W);
        p.perm = perm;
        p.goff = goff;
        p.window_len = window_len;
        p.tc = tc;
        p.t1 = t1;
        p.tile_status = tile_status;
        p.tickets = tickets;
        p.level_base = level_base;
        p.status = status;
        p.num_inputs = P;
        p.W = W;
        p.ngroups = ngroups;
        p.ngroups_m = 0xffffffffu / (uint32_t)ngroups;
        p.lpg_log2 = lpg_log2;
        p.slots_per_gate = slots_per_gate;
        p.pulse_percent = pulse_percent;
        p.ranked = windows_ranked(W) ? 1 : 0;
        p.chunks = chunks_per_window(W, flags, long_windows);
        p.compact = compact ? 1 : 0;
        p.gexact = gexact;
        p.old_base = old_base;
        p.level_bound = level_bound;
        p.level_need = level_need;
        p.spin_limit_ns = stall_level >= 0 ? (unsigned long long)stall_wait_ns : kSpinLimitNs;
        return p;
    }
};

namespace {

gatspi_status validate(const gatspi_netlist *nl, const gatspi_config *cfg, long long *path_bound) {
    if (!nl || !cfg) return fail(GATSPI_EINVAL, "netlist and config are required");
    const long long P = nl->num_inputs, G = nl->num_gates, L = nl->num_levels, T = nl->num_types;
    if (P < 0 || G < 0 || L < 0 || T < 0 || P + G > INT32_MAX)
        return fail(GATSPI_EINVAL, "negative or too large netlist sizes");
    if (G > 0 && (L < 1 || T < 1)) return fail(GATSPI_EINVAL, "gates need at least one level and one type");
    if (cfg->num_windows < 1 || cfg->num_windows > GATSPI_MAX_WINDOWS)
        return fail(GATSPI_EINVAL, "num_windows must be 1 .. %d", GATSPI_MAX_WINDOWS);
    if (!cfg->window_len) return fail(GATSPI_EINVAL, "window_len is required");
    for (int w = 0; w < cfg->num_windows; ++w)
        if (cfg->window_len[w] < 1 || cfg->window_len[w] > (1ll << 30))
            return fail(GATSPI_EINVAL, "window %d: length must be in 1 .. 2^30", w);
    if ((cfg->flags & GATSPI_FLAG_PULSE_PERCENT) && (cfg->pulse_percent < 0 || cfg->pulse_percent > 100))
        return fail(GATSPI_EINVAL, "pulse_percent must be 0 .. 100");
    if ((cfg->flags & GATSPI_FLAG_WHOLE_WINDOWS) && (cfg->flags & GATSPI_FLAG_CUT_WINDOWS))
        return fail(GATSPI_EINVAL, "GATSPI_FLAG_WHOLE_WINDOWS and GATSPI_FLAG_CUT_WINDOWS exclude each other");
    if (G == 0) {
        *path_bound = 0;
        return GATSPI_OK;
    }
    if (!nl->level_offsets || !nl->gate_type || !nl->type_num_pins || !nl->type_tt_off || !nl->tt_data ||
        !nl->fanin_off || !nl->fanin_net || !nl->pin_weight || !nl->wire_rise || !nl->wire_fall ||
        !nl->gate_dly_off || !nl->dly_data)
        return fail(GATSPI_EINVAL, "a netlist array is missing");
    if (nl->level_offsets[0] != 0 || nl->level_offsets[L] != G)
        return fail(GATSPI_EINVAL, "level_offsets must run from 0 to num_gates");
    for (long long l = 0; l < L; ++l)
        if (nl->level_offsets[l + 1] < nl->level_offsets[l]) return fail(GATSPI_EINVAL, "level %lld: negative size", l);
    for (long long t = 0; t < T; ++t) {
        const int n = nl->type_num_pins[t];
        if (n < 1 || n > GATSPI_MAX_PINS) return fail(GATSPI_EINVAL, "type %lld: %d pins (1 .. %d)", t, n, GATSPI_MAX_PINS);
        if (nl->type_tt_off[t] < 0 || nl->type_tt_off[t] + (1ll << n) > nl->tt_len)
            return fail(GATSPI_EINVAL, "type %lld: truth table out of range", t);
        for (int k = 0; k < (1 << n); ++k)
            if (nl->tt_data[nl->type_tt_off[t] + k] > 1) return fail(GATSPI_EINVAL, "type %lld: truth-table entry not 0/1", t);
    }
    if (nl->fanin_off[0] != 0) return fail(GATSPI_EINVAL, "fanin_off[0] must be 0");
    int max_wire = 0, max_gate = 0;
    long long lvl = 0;
    for (long long g = 0; g < G; ++g) {
        while (g >= nl->level_offsets[lvl + 1]) ++lvl;
        const long long level_first_net = P + nl->level_offsets[lvl];
        const int t = nl->gate_type[g];
        if (t < 0 || t >= T) return fail(GATSPI_EINVAL, "gate %lld: type %d out of range", g, t);
        const int n = nl->type_num_pins[t];
        const long long e0 = nl->fanin_off[g];
        if (nl->fanin_off[g + 1] - e0 != n) return fail(GATSPI_EINVAL, "gate %lld: %d pins expected", g, n);
        unsigned seen = 0;
        for (int i = 0; i < n; ++i) {
            const long long s = nl->fanin_net[e0 + i];
            if (s < 0 || s >= level_first_net)
                return fail(GATSPI_EINVAL, "gate %lld pin %d: net %lld is not an input or a gate of a lower level", g, i, s);
            const int wt = nl->pin_weight[e0 + i];
            if (wt <= 0 || wt >= (1 << n) || (wt & (wt - 1)) || (seen & (unsigned)wt))
                return fail(GATSPI_EINVAL, "gate %lld: pin weights must be the distinct powers 2^0 .. 2^(n-1)", g);
            seen |= (unsigned)wt;
            const int wr = nl->wire_rise[e0 + i], wf = nl->wire_fall[e0 + i];
            if (wr < 0 || wr > 0xffff || wf < 0 || wf > 0xffff)
                return fail(GATSPI_EINVAL, "gate %lld pin %d: interconnect delay out of 0 .. 65535", g, i);
            max_wire = std::max(max_wire, std::max(wr, wf));
        }
        const long long d0 = nl->gate_dly_off[g];
        const long long dn = 4ll * n * (1ll << (n - 1));
        if (d0 < 0 || d0 + dn > nl->dly_len) return fail(GATSPI_EINVAL, "gate %lld: delay table out of range", g);
        for (long long k = 0; k < dn; ++k) {
            const int d = nl->dly_data[d0 + k];
            if (d == GATSPI_NO_ARC) continue;
            if (d < 0 || d >= (1 << 24)) return fail(GATSPI_EINVAL, "gate %lld: delay %d out of 0 .. 2^24-1", g, d);
            max_gate = std::max(max_gate, d);
        }
    }
    *path_bound = L * ((long long)max_wire + max_gate);
    return GATSPI_OK;
}

// The level kernel's delay-table layout: the entry of Fig. 4's row 4*i + 2*e_in +
// e_out and column c (the other pins' values, first pin most significant) moves to
// ((2*i + e_out) << n) | v, v being all n pin values after the switch (pin j at bit
// n-1-j), so that the kernel indexes with the pin values it already holds.  Same size
// (4n * 2^(n-1) = 2n * 2^n); tables shared by several gates are moved once.
void layout_delay_tables(const gatspi_netlist *nl, std::vector<int32_t> &out) {
    out.assign(nl->dly_data, nl->dly_data + nl->dly_len);
    std::unordered_set<long long> done;
    for (long long g = 0; g < nl->num_gates; ++g) {
        const long long off = nl->gate_dly_off[g];
        if (!done.insert(off).second) continue;
        const int n = nl->type_num_pins[nl->gate_type[g]];
        const int cols = 1 << (n - 1);
        const int32_t *src = nl->dly_data + off;
        int32_t *dst = out.data() + off;
        for (int i = 0; i < n; ++i)
            for (int e_out = 0; e_out < 2; ++e_out)
                for (uint32_t v = 0; v < (1u << n); ++v) {
                    const int b = n - 1 - i;
                    const int e_in = ((v >> b) & 1u) ? 0 : 1;   // the pin's new value 1: a rising input
                    const uint32_t col = ((v >> (b + 1)) << b) | (v & ((1u << b) - 1u));
                    dst[(((uint32_t)i << 1 | (uint32_t)e_out) << n) | v] = src[(4 * i + 2 * e_in + e_out) * cols + col];
                }
    }
}

// After a load: whether its windows are long (level_chunk_kernel's rule) and, with one
// window, long enough for segments; a change of the kernel that simulates them makes
// the captured level graph stale.
void set_long_windows(gatspi_ctx *c, long long window_words) {
    const long long n = (long long)c->P * c->W;
    const bool lw = n > 0 && window_words >= kLongWindowWords * n;
    const bool sw = n > 0 && c->W == 1 && window_words >= kSplitWindowWords * n;
    const bool dw = n > 0 && window_words >= kDenseWindowWords * n;
    if (lw == c->long_windows && sw == c->split_windows && dw == c->dense_windows) return;
    c->long_windows = lw;
    c->split_windows = sw;
    c->dense_windows = dw;
    if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
    if (c->graph) cudaGraphDestroy(c->graph);
    c->graph_exec = nullptr;
    c->graph = nullptr;
}

void free_all(gatspi_ctx *c) {
    if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
    if (c->graph) cudaGraphDestroy(c->graph);
    if (c->capture_stream) cudaStreamDestroy(c->capture_stream);
    for (cudaEvent_t e : c->events) cudaEventDestroy(e);
    for (cudaEvent_t e : c->dump_events) cudaEventDestroy(e);
    if (c->dump_done) cudaEventDestroy(c->dump_done);
    if (c->dump_stream) cudaStreamDestroy(c->dump_stream);
    if (c->tc_host) cudaFreeHost(c->tc_host);
    if (c->t1_host) cudaFreeHost(c->t1_host);
    void *ptrs[] = {c->gexact, c->old_base, c->level_bound, c->level_need, c->gate_desc, c->dly, c->gate_order, c->heavy_order, c->seg_items, c->seg_count, c->seg_cnt, c->seg_counter, c->net_base, c->wstart, c->wend, c->wlen8, c->perm, c->goff,
                    c->window_len, c->tc, c->t1,
                    c->tile_status, c->tickets, c->level_base, c->status, c->load_off, c->max_time,
                    c->win_start, c->tc_in, c->t1_in};
    for (void *p : ptrs)
        if (p) cudaFree(p);
}

gatspi_status read_status(gatspi_ctx *c) {
    int32_t st[kStatusWords];
    CUDA_TRY(cudaMemcpy(st, c->status, sizeof st, cudaMemcpyDeviceToHost), "reading the device status");
    switch (st[0]) {
        case GATSPI_OK: return GATSPI_OK;
        case GATSPI_EPOOL_OVERFLOW:
            return fail(GATSPI_EPOOL_OVERFLOW, "waveform pool too small (%lld words) at level %d", c->pool_words, st[1]);
        case GATSPI_EBADWAVE:
            return fail(GATSPI_EBADWAVE, "malformed waveform (net %d, window %d)", st[1], st[2]);
        case GATSPI_EBADLUT:
            return fail(GATSPI_EBADLUT, "gate %d window %d: every switching arc of an output change has no delay", st[1], st[2]);
        case GATSPI_ETIMEOUT:
            return fail(GATSPI_ETIMEOUT, "scan look-back stalled at level %d tile %d (waiting on tile %d)", st[1], st[2], st[3]);
        case GATSPI_EINTERNAL:
            return fail(GATSPI_EINTERNAL, "library fault: a chunk of gate %d window %d (lane %d) outgrew its bound",
                        st[1], st[2], st[3]);
        default: return fail((gatspi_status)st[0], "device error %d", st[0]);
    }
}

gatspi_status sync_ctx(gatspi_ctx *c) {
    CUDA_TRY(cudaSetDevice(c->device), "cudaSetDevice");
    CUDA_TRY(cudaStreamSynchronize(c->last_stream), "synchronising the stream");
    CUDA_TRY(cudaGetLastError(), "pending CUDA error");
    return read_status(c);
}

// Statistics of the loaded inputs (their window index has been checked): computed on
// the device, kept on the host.
gatspi_status input_stats(gatspi_ctx *c, cudaStream_t s) {
    c->tc_in_host.assign(c->P, 0);
    c->t1_in_host.assign(c->P, 0);
    if (c->P == 0) return GATSPI_OK;
    CUDA_TRY(launch_input_stats(c->params(), c->tc_in, c->t1_in, s), "input statistics");
    CUDA_TRY(cudaStreamSynchronize(s), "input statistics");
    CUDA_TRY(cudaMemcpy(c->tc_in_host.data(), c->tc_in, sizeof(unsigned long long) * c->P, cudaMemcpyDeviceToHost),
             "reading input statistics");
    CUDA_TRY(cudaMemcpy(c->t1_in_host.data(), c->t1_in, sizeof(unsigned long long) * c->P, cudaMemcpyDeviceToHost),
             "reading input statistics");
    return GATSPI_OK;
}

// Enqueue the whole level sequence on stream s.
gatspi_status enqueue_levels(gatspi_ctx *c, cudaStream_t s) {
    CUDA_TRY(cudaMemsetAsync(c->tc, 0, sizeof(unsigned long long) * std::max(c->G, 1), s), "clearing TC");
    CUDA_TRY(cudaMemsetAsync(c->t1, 0, sizeof(unsigned long long) * std::max(c->G, 1), s), "clearing T1");
    const int scans = c->compact ? 2 : 1;   // compaction scans every level twice
    if (c->seg_counter)   // a run that stopped on an error may have left segments uncounted
        CUDA_TRY(cudaMemsetAsync(c->seg_counter, 0, sizeof(int32_t) * (size_t)std::max<long long>(c->max_level_gates, 1), s),
                 "clearing the segment counters");
    CUDA_TRY(cudaMemsetAsync(c->tile_status, 0, sizeof(unsigned long long) * std::max<long long>(scans * c->total_tiles, 1),
                             s), "clearing the scan state");
    CUDA_TRY(cudaMemsetAsync(c->tickets, 0, sizeof(int32_t) * std::max(scans * c->L, 1), s), "clearing the tile tickets");
    // an injected stall: the level's first ticket becomes 1 (its low byte set), so no
    // block ever takes tile 0 and the tiles after it wait for a flag nobody sets
    if (c->stall_level >= 0)
        CUDA_TRY(cudaMemsetAsync(c->tickets + c->stall_level, 1, 1, s), "injecting a scan stall");
    CUDA_TRY(cudaMemsetAsync(c->status, 0, sizeof(int32_t) * kStatusWords, s), "clearing the status");
    const DevParams p = c->params();
    const bool timing = (c->flags & GATSPI_FLAG_LEVEL_TIMING) != 0;
    // events: [2l] before the bounds kernels of level l, [2l+1] between them and the
    // simulation kernel, [2l+2] after the simulation kernel
    for (int l = 0; l < c->L; ++l) {
        if (timing) CUDA_TRY(cudaEventRecord(c->events[2 * l], s), "recording a level event");
        // compaction: the previous level is packed before this one is planned (its
        // time counts with this level's bounds kernels)
        if (c->compact && l > 0)
            CUDA_TRY(launch_level_compact(p, c->launches[l - 1], c->exact_launches[l - 1], s), "packing a level");
        CUDA_TRY(launch_level_bounds(p, c->launches[l], s), "launching a bounds kernel");
        if (timing) CUDA_TRY(cudaEventRecord(c->events[2 * l + 1], s), "recording a level event");
        CUDA_TRY(launch_level_sim(p, c->launches[l], s), "launching a level kernel");
        // the level's TC/T1 are final: copy them out on the side stream while the
        // next levels run
        const long long gb = c->level_offsets[l], ng = c->level_offsets[l + 1] - gb;
        if (ng > 0) {
            CUDA_TRY(cudaEventRecord(c->dump_events[l], s), "recording a dump event");
            CUDA_TRY(cudaStreamWaitEvent(c->dump_stream, c->dump_events[l], 0), "ordering the dump");
            CUDA_TRY(cudaMemcpyAsync(c->tc_host + gb, c->tc + gb, sizeof(unsigned long long) * ng,
                                     cudaMemcpyDeviceToHost, c->dump_stream), "dumping TC");
            CUDA_TRY(cudaMemcpyAsync(c->t1_host + gb, c->t1 + gb, sizeof(unsigned long long) * ng,
                                     cudaMemcpyDeviceToHost, c->dump_stream), "dumping T1");
        }
    }
    if (timing && c->L > 0) CUDA_TRY(cudaEventRecord(c->events[2 * c->L], s), "recording a level event");
    if (c->compact && c->L > 0)
        CUDA_TRY(launch_level_compact(p, c->launches[c->L - 1], c->exact_launches[c->L - 1], s), "packing a level");
    if (c->G > 0) {   // the stream's later work waits for the dump
        CUDA_TRY(cudaEventRecord(c->dump_done, c->dump_stream), "recording the dump's end");
        CUDA_TRY(cudaStreamWaitEvent(s, c->dump_done, 0), "joining the dump");
    }
    return GATSPI_OK;
}

}  // namespace

extern "C" {

const char *gatspi_last_error(void) { return g_err.c_str(); }

int32_t gatspi_lanes_per_window(const gatspi_ctx *c) {
    if (!c) return 0;
    const int k = chunks_per_window(c->W, c->flags, c->long_windows);
    return k > 1 ? k : 1;
}

const char *gatspi_status_name(gatspi_status s) {
    switch (s) {
        case GATSPI_OK: return "GATSPI_OK";
        case GATSPI_EINVAL: return "GATSPI_EINVAL";
        case GATSPI_ENOMEM: return "GATSPI_ENOMEM";
        case GATSPI_EPOOL_OVERFLOW: return "GATSPI_EPOOL_OVERFLOW";
        case GATSPI_EBADWAVE: return "GATSPI_EBADWAVE";
        case GATSPI_ECUDA: return "GATSPI_ECUDA";
        case GATSPI_ESTATE: return "GATSPI_ESTATE";
        case GATSPI_EBADLUT: return "GATSPI_EBADLUT";
        case GATSPI_ETIMEOUT: return "GATSPI_ETIMEOUT";
        case GATSPI_EINTERNAL: return "GATSPI_EINTERNAL";
    }
    return "GATSPI_UNKNOWN";
}

gatspi_status gatspi_create(const gatspi_netlist *nl, const gatspi_config *cfg, int32_t *d_pool, size_t pool_words,
                            gatspi_ctx **out) {
    g_err.clear();
    if (!out) return fail(GATSPI_EINVAL, "out is NULL");
    *out = nullptr;
    long long path_bound = 0;
    gatspi_status st = validate(nl, cfg, &path_bound);
    if (st != GATSPI_OK) return st;
    if (!d_pool || pool_words == 0 || (pool_words & 3) || ((uintptr_t)d_pool & 15))
        return fail(GATSPI_EINVAL, "the pool must be a non-empty, 16-byte aligned device buffer of 4k words");

    gatspi_ctx *c = new (std::nothrow) gatspi_ctx();
    if (!c) return fail(GATSPI_ENOMEM, "host allocation failed");
    st = [&]() -> gatspi_status {
        CUDA_TRY(cudaGetDevice(&c->device), "cudaGetDevice");
        c->P = nl->num_inputs;
        c->G = nl->num_gates;
        c->L = nl->num_gates > 0 ? nl->num_levels : 0;
        c->W = cfg->num_windows;
        c->pool = d_pool;
        c->pool_words = (long long)pool_words;
        c->flags = cfg->flags;
        c->pulse_percent = (cfg->flags & GATSPI_FLAG_PULSE_PERCENT) ? cfg->pulse_percent : 100;
        c->num_nets = (long long)c->P + c->G;
        c->ngroups = (c->W + 31) / 32;
        int lpg = 32;
        if (c->W < 32) {
            lpg = 1;
            while (lpg < c->W) lpg <<= 1;
        }
        while ((1 << c->lpg_log2) < lpg) ++c->lpg_log2;
        c->slots_per_gate = c->ngroups << c->lpg_log2;
        c->path_delay_bound = path_bound;
        for (int w = 0; w < c->W; ++w) c->sum_window_len += cfg->window_len[w];

        // gate records: descriptor, source nets, wire delays (unused pins: 0)
        std::vector<int4> gd(3 * std::max(c->G, 1), make_int4(0, 0, 0, 0));
        for (long long g = 0; g < c->G; ++g) {
            const int t = nl->gate_type[g];
            const int n = nl->type_num_pins[t];
            // truth table re-indexed by the pin values (first pin most significant):
            // entry v is the page's entry at the sum of the weights of the pins at 1
            uint32_t mask = 0;
            const long long e0 = nl->fanin_off[g];
            for (int v = 0; v < (1 << n); ++v) {
                int k = 0;
                for (int i = 0; i < n; ++i)
                    if ((v >> (n - 1 - i)) & 1) k += nl->pin_weight[e0 + i];
                mask |= (uint32_t)nl->tt_data[nl->type_tt_off[t] + k] << v;
            }
            const long long d0 = nl->gate_dly_off[g];
            int src[4] = {0, 0, 0, 0}, drf[4] = {0, 0, 0, 0};
            for (int i = 0; i < n; ++i) {
                src[i] = nl->fanin_net[e0 + i];
                drf[i] = (int)((uint32_t)nl->wire_rise[e0 + i] | ((uint32_t)nl->wire_fall[e0 + i] << 16));
            }
            gd[3 * g] = make_int4(0, (int)(n | (mask << 8)), (int)(uint32_t)(d0 & 0xffffffffll), (int)(d0 >> 32));
            gd[3 * g + 1] = make_int4(src[0], src[1], src[2], src[3]);
            gd[3 * g + 2] = make_int4(drf[0], drf[1], drf[2], drf[3]);
        }

        // levels and tiles
        c->level_offsets.assign(nl->level_offsets, nl->level_offsets + c->L + 1);
        for (int l = 0; l < c->L; ++l) {
            LevelLaunch ll{};
            ll.level = l;
            ll.gate_begin = c->level_offsets[l];
            ll.num_gates = c->level_offsets[l + 1] - c->level_offsets[l];
            const long long slots = (long long)ll.num_gates * c->slots_per_gate;
            const long long tiles = std::max<long long>(1, (slots + kTileSlots - 1) / kTileSlots);
            const long long scan = std::max<long long>(1, ((long long)ll.num_gates + kPlaceTile - 1) / kPlaceTile);
            if (tiles > INT32_MAX / kTileSlots)
                return fail(GATSPI_EINVAL, "level %d has too many (gate, window) slots", l);
            ll.num_tiles = (int32_t)tiles;
            ll.scan_tiles = (int32_t)scan;
            c->max_level_gates = std::max<long long>(c->max_level_gates, ll.num_gates);
            ll.tile_base = c->total_tiles;
            ll.ticket = l;
            c->total_tiles += scan;
            c->launches.push_back(ll);
        }
        c->compact = (cfg->flags & GATSPI_FLAG_COMPACT) != 0;
        if (c->compact)
            for (int l = 0; l < c->L; ++l) {   // the exact scans: their own tickets and look-back words
                LevelLaunch ex = c->launches[l];
                ex.tile_base += c->total_tiles;
                ex.ticket = c->L + l;
                c->exact_launches.push_back(ex);
            }

        const long long dly_len = c->G > 0 ? nl->dly_len : 0;
        CUDA_TRY(dev_alloc(&c->gate_desc, gd.size()), "allocating gate descriptors");
        if (c->lpg_log2 < 5 && c->G > 0) {
            // several gates share a warp: take every level's gates by pin count (stable)
            std::vector<int32_t> order((size_t)c->G);
            for (int l = 0; l < c->L; ++l) {
                size_t k = (size_t)c->level_offsets[l];
                for (int n = 1; n <= GATSPI_MAX_PINS; ++n)
                    for (int32_t g = c->level_offsets[l]; g < c->level_offsets[l + 1]; ++g)
                        if (nl->type_num_pins[nl->gate_type[g]] == n) order[k++] = g;
            }
            CUDA_TRY(dev_alloc(&c->gate_order, order.size()), "allocating the gate order");
            if (c->W <= 16)
                CUDA_TRY(dev_alloc(&c->heavy_order, (size_t)std::max<long long>(c->max_level_gates, 1)),
                         "allocating the gate order");
            if (c->W == 1) {
                const size_t mg = (size_t)std::max<long long>(c->max_level_gates, 1);
                CUDA_TRY(dev_alloc(&c->seg_items, mg + kExtraSegments), "allocating the segment list");
                CUDA_TRY(dev_alloc(&c->seg_count, (size_t)1), "allocating the segment list");
                CUDA_TRY(dev_alloc(&c->seg_cnt, mg * kMaxSegments), "allocating the segment list");
                CUDA_TRY(dev_alloc(&c->seg_counter, mg), "allocating the segment list");
                CUDA_TRY(cudaMemset(c->seg_counter, 0, mg * sizeof(int32_t)), "clearing the segment counters");
                // 8 blocks of 4 warps per SM (level_chunk_kernel's occupancy)
                int sms = 0;
                CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device), "reading the SM count");
                c->resident_warps = std::max(sms, 1) * 32;
            }
            CUDA_TRY(cudaMemcpy(c->gate_order, order.data(), order.size() * sizeof(int32_t), cudaMemcpyHostToDevice),
                     "uploading the gate order");
        }
        CUDA_TRY(dev_alloc(&c->dly, (size_t)dly_len), "allocating delay tables");
        CUDA_TRY(dev_alloc(&c->net_base, (size_t)std::max<long long>(c->num_nets, 1)), "allocating the window index");
        CUDA_TRY(dev_alloc(&c->wstart, (size_t)(c->num_nets * c->W)), "allocating the window index");
        CUDA_TRY(dev_alloc(&c->wend, (size_t)(c->num_nets * c->W)), "allocating the window index");
        CUDA_TRY(dev_alloc(&c->wlen8, (size_t)std::max<long long>(c->num_nets * ((c->W + 3) & ~3), 4)),
                 "allocating the window index");
        CUDA_TRY(dev_alloc(&c->perm, (size_t)(windows_ranked(c->W) ? std::max<long long>(c->max_level_gates * c->W, 1) : 1)),
                 "allocating the plan");
        CUDA_TRY(dev_alloc(&c->goff, (size_t)std::max<long long>(c->max_level_gates * (c->ngroups + 1), 1)),
                 "allocating the plan");
        CUDA_TRY(dev_alloc(&c->window_len, (size_t)c->W), "allocating window lengths");
        CUDA_TRY(dev_alloc(&c->tc, (size_t)c->G), "allocating TC");
        CUDA_TRY(dev_alloc(&c->t1, (size_t)c->G), "allocating T1");
        const int scans = c->compact ? 2 : 1;
        CUDA_TRY(dev_alloc(&c->tile_status, (size_t)(scans * c->total_tiles)), "allocating the scan state");
        CUDA_TRY(dev_alloc(&c->tickets, (size_t)(scans * c->L)), "allocating tile tickets");
        if (c->compact) {
            CUDA_TRY(dev_alloc(&c->gexact, (size_t)std::max<long long>(c->max_level_gates * c->ngroups, 1)),
                     "allocating the compaction state");
            CUDA_TRY(dev_alloc(&c->old_base, (size_t)std::max<long long>(c->max_level_gates, 1)),
                     "allocating the compaction state");
            CUDA_TRY(dev_alloc(&c->level_bound, (size_t)std::max(c->L, 1)), "allocating the compaction state");
            CUDA_TRY(dev_alloc(&c->level_need, (size_t)std::max(c->L, 1)), "allocating the compaction state");
        }
        CUDA_TRY(dev_alloc(&c->level_base, (size_t)c->L + 1), "allocating level bases");
        CUDA_TRY(dev_alloc(&c->status, (size_t)kStatusWords), "allocating the status word");
        CUDA_TRY(dev_alloc(&c->load_off, (size_t)((long long)c->P * c->W + 1)), "allocating load offsets");
        CUDA_TRY(dev_alloc(&c->max_time, 1), "allocating the load scratch");
        CUDA_TRY(dev_alloc(&c->win_start, (size_t)c->W + 1), "allocating window starts");
        CUDA_TRY(dev_alloc(&c->tc_in, (size_t)std::max(c->P, 1)), "allocating input statistics");
        CUDA_TRY(dev_alloc(&c->t1_in, (size_t)std::max(c->P, 1)), "allocating input statistics");

        std::vector<int32_t> wl(c->W);
        std::vector<long long> ws(c->W + 1, 0);
        for (int w = 0; w < c->W; ++w) {
            wl[w] = (int32_t)cfg->window_len[w];
            ws[w + 1] = ws[w] + cfg->window_len[w];
            c->max_window_len = std::max(c->max_window_len, (long long)cfg->window_len[w]);
        }
        CUDA_TRY(cudaMemcpy(c->win_start, ws.data(), ws.size() * sizeof(long long), cudaMemcpyHostToDevice),
                 "uploading window starts");
        CUDA_TRY(cudaMemcpy(c->gate_desc, gd.data(), gd.size() * sizeof(int4), cudaMemcpyHostToDevice), "uploading gates");
        if (dly_len > 0) {
            std::vector<int32_t> packed;
            layout_delay_tables(nl, packed);
            CUDA_TRY(cudaMemcpy(c->dly, packed.data(), (size_t)dly_len * sizeof(int32_t), cudaMemcpyHostToDevice),
                     "uploading delay tables");
        }
        CUDA_TRY(cudaMemcpy(c->window_len, wl.data(), wl.size() * sizeof(int32_t), cudaMemcpyHostToDevice),
                 "uploading window lengths");
        CUDA_TRY(cudaMemset(c->status, 0, sizeof(int32_t) * kStatusWords), "clearing the status");
        CUDA_TRY(cudaMemset(c->tc, 0, sizeof(unsigned long long) * std::max(c->G, 1)), "clearing TC");
        CUDA_TRY(cudaMemset(c->t1, 0, sizeof(unsigned long long) * std::max(c->G, 1)), "clearing T1");
        CUDA_TRY(set_level_smem_limit(), "configuring shared memory");
        c->events.resize(2 * c->L + 1, nullptr);   // level timing can be switched on later
        for (auto &e : c->events) CUDA_TRY(cudaEventCreate(&e), "creating level events");
        if (c->G > 0) {
            CUDA_TRY(cudaHostAlloc((void **)&c->tc_host, sizeof(unsigned long long) * c->G, cudaHostAllocDefault),
                     "allocating pinned TC");
            CUDA_TRY(cudaHostAlloc((void **)&c->t1_host, sizeof(unsigned long long) * c->G, cudaHostAllocDefault),
                     "allocating pinned T1");
            CUDA_TRY(cudaStreamCreateWithFlags(&c->dump_stream, cudaStreamNonBlocking), "creating the dump stream");
            c->dump_events.resize(c->L, nullptr);
            for (auto &e : c->dump_events)
                CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "creating dump events");
            CUDA_TRY(cudaEventCreateWithFlags(&c->dump_done, cudaEventDisableTiming), "creating dump events");
        }
        return GATSPI_OK;
    }();
    if (st != GATSPI_OK) {
        free_all(c);
        delete c;
        return st;
    }
    *out = c;
    return GATSPI_OK;
}

gatspi_status gatspi_load_waveforms(gatspi_ctx *c, const int64_t *off, const int32_t *words, size_t nwords, int where,
                                    void *stream) {
    g_err.clear();
    if (!c || !off || (!words && nwords)) return fail(GATSPI_EINVAL, "ctx, off and words are required");
    if (where != GATSPI_HOST && where != GATSPI_DEVICE) return fail(GATSPI_EINVAL, "where must be HOST or DEVICE");
    if ((long long)nwords > c->pool_words)
        return fail(GATSPI_EPOOL_OVERFLOW, "%zu input words exceed the pool (%lld words)", nwords, c->pool_words);
    CUDA_TRY(cudaSetDevice(c->device), "cudaSetDevice");
    cudaStream_t s = (cudaStream_t)stream;
    const long long n = (long long)c->P * c->W + 1;
    const cudaMemcpyKind kind = where == GATSPI_HOST ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    if (where == GATSPI_HOST && off[n - 1] != (long long)nwords)
        return fail(GATSPI_EINVAL, "off[num_inputs * W] (%lld) must equal nwords (%zu)", (long long)off[n - 1], nwords);
    c->loaded = false;
    c->last_stream = s;
    CUDA_TRY(cudaMemcpyAsync(c->load_off, off, (size_t)n * sizeof(long long), kind, s), "copying input offsets");
    if (nwords) CUDA_TRY(cudaMemcpyAsync(c->pool, words, nwords * sizeof(int32_t), kind, s), "copying input words");
    CUDA_TRY(cudaMemsetAsync(c->status, 0, sizeof(int32_t) * kStatusWords, s), "clearing the status");
    CUDA_TRY(cudaMemsetAsync(c->max_time, 0, sizeof(int32_t), s), "clearing the load scratch");
    CUDA_TRY(launch_load_index(c->params(), c->load_off, (long long)nwords, c->max_time, s), "indexing the inputs");
    CUDA_TRY(cudaStreamSynchronize(s), "loading waveforms");
    int32_t st[kStatusWords];
    int32_t tmax = 0;
    CUDA_TRY(cudaMemcpy(st, c->status, sizeof st, cudaMemcpyDeviceToHost), "reading the load status");
    CUDA_TRY(cudaMemcpy(&tmax, c->max_time, sizeof tmax, cudaMemcpyDeviceToHost), "reading the load status");
    if (st[0] == GATSPI_EBADWAVE)
        return fail(GATSPI_EBADWAVE, "input %d window %d: malformed waveform or offsets", st[1], st[2]);
    if (st[0] != 0) return read_status(c);
    if ((long long)tmax + c->path_delay_bound >= (long long)GATSPI_EOW)
        return fail(GATSPI_EINVAL, "latest input time %d plus the longest path delay bound %lld reaches EOW", tmax,
                    c->path_delay_bound);
    gatspi_status ist = input_stats(c, s);
    if (ist != GATSPI_OK) return ist;
    set_long_windows(c, (long long)nwords);
    c->loaded = true;
    return GATSPI_OK;
}

gatspi_status gatspi_load_testbench(gatspi_ctx *c, const int64_t *off, const int32_t *words, size_t nwords, int where,
                                    void *stream) {
    g_err.clear();
    if (!c || !off || (!words && nwords)) return fail(GATSPI_EINVAL, "ctx, off and words are required");
    if (where != GATSPI_HOST && where != GATSPI_DEVICE) return fail(GATSPI_EINVAL, "where must be HOST or DEVICE");
    const long long P = c->P, W = c->W;
    // the windows of input p take at most (its transitions) + 3 W words
    const long long region = (long long)nwords + 3 * W * P;
    const long long stage_at = where == GATSPI_HOST ? ((c->pool_words - (long long)nwords) & ~3ll) : c->pool_words;
    if (stage_at < 0 || region > stage_at)
        return fail(GATSPI_EPOOL_OVERFLOW,
                    "%zu testbench words need %lld pool words for the windows%s (pool: %lld words)", nwords, region,
                    where == GATSPI_HOST ? " plus the staged testbench" : "", c->pool_words);
    if (where == GATSPI_HOST) {
        if (off[0] != 0 || off[P] != (long long)nwords)
            return fail(GATSPI_EINVAL, "off[0] must be 0 and off[num_inputs] (%lld) must equal nwords (%zu)",
                        (long long)off[P], nwords);
        for (long long p = 0; p < P; ++p)
            if (off[p + 1] < off[p]) return fail(GATSPI_EINVAL, "off must be non-decreasing (input %lld)", p);
    }
    if (c->max_window_len - 1 + c->path_delay_bound >= (long long)GATSPI_EOW)
        return fail(GATSPI_EINVAL, "the longest window plus the longest path delay bound %lld reaches EOW",
                    c->path_delay_bound);
    CUDA_TRY(cudaSetDevice(c->device), "cudaSetDevice");
    cudaStream_t s = (cudaStream_t)stream;
    const cudaMemcpyKind kind = where == GATSPI_HOST ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    c->loaded = false;
    c->last_stream = s;
    // a host testbench is staged at the far end of the pool, behind the windows' regions
    const int32_t *tb = where == GATSPI_HOST ? c->pool + stage_at : words;
    if (where == GATSPI_HOST && nwords)
        CUDA_TRY(cudaMemcpyAsync(c->pool + stage_at, words, nwords * sizeof(int32_t), kind, s), "copying the testbench");
    CUDA_TRY(cudaMemcpyAsync(c->load_off, off, (size_t)(P + 1) * sizeof(long long), kind, s),
             "copying testbench offsets");
    CUDA_TRY(cudaMemsetAsync(c->status, 0, sizeof(int32_t) * kStatusWords, s), "clearing the status");
    if (P == 0) CUDA_TRY(cudaMemsetAsync(c->level_base, 0, sizeof(long long), s), "setting the first level base");
    CUDA_TRY(launch_testbench_cut(c->params(), c->load_off, tb, (long long)nwords, c->win_start, s),
             "cutting the testbench into windows");
    CUDA_TRY(cudaStreamSynchronize(s), "loading the testbench");
    int32_t st[kStatusWords];
    CUDA_TRY(cudaMemcpy(st, c->status, sizeof st, cudaMemcpyDeviceToHost), "reading the load status");
    if (st[0] == GATSPI_EBADWAVE)
        return fail(GATSPI_EBADWAVE, "input %d: malformed testbench waveform or offsets", st[1]);
    if (st[0] != 0) return read_status(c);
    gatspi_status ist = input_stats(c, s);
    if (ist != GATSPI_OK) return ist;
    set_long_windows(c, (long long)nwords + 2 * W * P);   // transitions, plus a head and an EOW per window
    c->loaded = true;
    return GATSPI_OK;
}

gatspi_status gatspi_simulate(gatspi_ctx *c, void *stream) {
    g_err.clear();
    if (!c) return fail(GATSPI_EINVAL, "ctx is NULL");
    if (!c->loaded) return fail(GATSPI_ESTATE, "load the input waveforms first");
    CUDA_TRY(cudaSetDevice(c->device), "cudaSetDevice");
    cudaStream_t s = (cudaStream_t)stream;
    c->last_stream = s;
    c->simulated = true;
    c->timed_last = (c->flags & GATSPI_FLAG_LEVEL_TIMING) != 0;
    // per-level events are recorded on the caller's stream: they cannot be read back
    // from a replayed graph, so timing runs launch the levels directly
    if (c->stall_level >= 0) {   // an injected stall runs once, launched directly
        const gatspi_status st = enqueue_levels(c, s);
        c->stall_level = -1;
        return st;
    }
    if (c->flags & (GATSPI_FLAG_NO_GRAPH | GATSPI_FLAG_LEVEL_TIMING)) return enqueue_levels(c, s);
    if (!c->graph_exec) {
        if (!c->capture_stream)
            CUDA_TRY(cudaStreamCreateWithFlags(&c->capture_stream, cudaStreamNonBlocking), "creating the capture stream");
        CUDA_TRY(cudaStreamBeginCapture(c->capture_stream, cudaStreamCaptureModeThreadLocal), "beginning capture");
        gatspi_status st = enqueue_levels(c, c->capture_stream);
        cudaGraph_t g = nullptr;
        cudaError_t e = cudaStreamEndCapture(c->capture_stream, &g);
        if (st != GATSPI_OK) {
            if (g) cudaGraphDestroy(g);
            return st;
        }
        if (e != cudaSuccess) return cuda_fail(e, "ending capture");
        c->graph = g;
        CUDA_TRY(cudaGraphInstantiate(&c->graph_exec, c->graph, 0), "instantiating the level graph");
    }
    CUDA_TRY(cudaGraphLaunch(c->graph_exec, s), "launching the level graph");
    return GATSPI_OK;
}

gatspi_status gatspi_sync(gatspi_ctx *c) {
    g_err.clear();
    if (!c) return fail(GATSPI_EINVAL, "ctx is NULL");
    return sync_ctx(c);
}

gatspi_status gatspi_toggle_stats(gatspi_ctx *c, int64_t *tc, int64_t *t0, int64_t *t1) {
    g_err.clear();
    if (!c) return fail(GATSPI_EINVAL, "ctx is NULL");
    if (!c->simulated) return fail(GATSPI_ESTATE, "simulate first");
    gatspi_status st = sync_ctx(c);
    if (st != GATSPI_OK) return st;
    if (c->G == 0) return GATSPI_OK;
    // simulate copied the statistics to pinned host memory level by level; the
    // stream it ran on has finished, and with it the copies
    if (tc) std::memcpy(tc, c->tc_host, sizeof(int64_t) * c->G);
    for (int g = 0; g < c->G; ++g) {
        if (t1) t1[g] = (int64_t)c->t1_host[g];
        if (t0) t0[g] = c->sum_window_len - (int64_t)c->t1_host[g];
    }
    return GATSPI_OK;
}

gatspi_status gatspi_toggle_stats_host(gatspi_ctx *c, const uint64_t **tc, const uint64_t **t1, int64_t *window_sum) {
    g_err.clear();
    if (!c || !tc || !t1) return fail(GATSPI_EINVAL, "ctx, tc and t1 are required");
    if (!c->simulated) return fail(GATSPI_ESTATE, "simulate first");
    gatspi_status st = sync_ctx(c);
    if (st != GATSPI_OK) return st;
    *tc = c->G > 0 ? (const uint64_t *)c->tc_host : nullptr;
    *t1 = c->G > 0 ? (const uint64_t *)c->t1_host : nullptr;
    if (window_sum) *window_sum = c->sum_window_len;
    return GATSPI_OK;
}

gatspi_status gatspi_input_stats(gatspi_ctx *c, int64_t *tc, int64_t *t0, int64_t *t1) {
    g_err.clear();
    if (!c) return fail(GATSPI_EINVAL, "ctx is NULL");
    if (!c->loaded) return fail(GATSPI_ESTATE, "load the inputs first");
    for (int p = 0; p < c->P; ++p) {
        if (tc) tc[p] = (int64_t)c->tc_in_host[p];
        if (t1) t1[p] = (int64_t)c->t1_in_host[p];
        if (t0) t0[p] = c->sum_window_len - (int64_t)c->t1_in_host[p];
    }
    return GATSPI_OK;
}

gatspi_status gatspi_write_saif(gatspi_ctx *c, const char *path, const char *design, const char *timescale,
                                const char *const *net_names) {
    g_err.clear();
    if (!c || !path) return fail(GATSPI_EINVAL, "ctx and path are required");
    if (!c->loaded || !c->simulated) return fail(GATSPI_ESTATE, "simulate first");
    gatspi_status st = sync_ctx(c);
    if (st != GATSPI_OK) return st;
    FILE *f = std::fopen(path, "w");
    if (!f) return fail(GATSPI_EINVAL, "cannot open %s for writing", path);
    const char *top = design && *design ? design : "top";
    std::fprintf(f, "(SAIFILE\n(SAIFVERSION \"2.0\")\n(DIRECTION \"backward\")\n(DESIGN \"%s\")\n", top);
    std::fprintf(f, "(PROGRAM_NAME \"gate_level_logic_gb300\")\n(DIVIDER / )\n(TIMESCALE %s)\n(DURATION %lld)\n",
                 timescale && *timescale ? timescale : "1 ps", c->sum_window_len);
    std::fprintf(f, "(INSTANCE %s\n  (NET\n", top);
    std::string name;
    for (long long n = 0; n < c->num_nets; ++n) {
        name.clear();
        if (net_names && net_names[n]) {
            for (const char *q = net_names[n]; *q; ++q) {   // escape what is not an identifier character
                const char ch = *q;
                const bool plain = (ch >= 'a' && ch <= 'z') || (ch >= 'A' && ch <= 'Z') || (ch >= '0' && ch <= '9') ||
                                   ch == '_';
                if (!plain) name.push_back('\\');
                name.push_back(ch);
            }
        } else {
            name = "n" + std::to_string(n);
        }
        const bool in = n < c->P;
        const long long tc = in ? (long long)c->tc_in_host[n] : (long long)c->tc_host[n - c->P];
        const long long t1 = in ? (long long)c->t1_in_host[n] : (long long)c->t1_host[n - c->P];
        std::fprintf(f, "    (%s\n      (T0 %lld) (T1 %lld) (TX 0)\n      (TC %lld) (IG 0)\n    )\n", name.c_str(),
                     c->sum_window_len - t1, t1, tc);
    }
    std::fprintf(f, "  )\n)\n)\n");
    const bool bad = std::ferror(f) != 0;
    if (std::fclose(f) != 0 || bad) return fail(GATSPI_EINVAL, "writing %s failed", path);
    return GATSPI_OK;
}

gatspi_status gatspi_get_waveform(gatspi_ctx *c, int32_t net, int32_t window, int32_t *buf, size_t cap, size_t *len) {
    g_err.clear();
    if (!c || !len) return fail(GATSPI_EINVAL, "ctx and len are required");
    if (net < 0 || net >= c->num_nets || window < 0 || window >= c->W)
        return fail(GATSPI_EINVAL, "net %d / window %d out of range", net, window);
    if (!c->loaded || (net >= c->P && !c->simulated)) return fail(GATSPI_ESTATE, "waveform not computed yet");
    gatspi_status st = sync_ctx(c);
    if (st != GATSPI_OK) return st;
    long long base = 0;
    uint32_t end = 0, start = 0;
    const long long k = (long long)net * c->W + window;
    CUDA_TRY(cudaMemcpy(&base, c->net_base + net, sizeof base, cudaMemcpyDeviceToHost), "reading the window index");
    CUDA_TRY(cudaMemcpy(&start, c->wstart + k, sizeof start, cudaMemcpyDeviceToHost), "reading the window index");
    CUDA_TRY(cudaMemcpy(&end, c->wend + k, sizeof end, cudaMemcpyDeviceToHost), "reading the window index");
    *len = (size_t)(end - start);
    if (*len > cap || !buf) return fail(GATSPI_EINVAL, "buffer of %zu words too small for %zu", cap, *len);
    CUDA_TRY(cudaMemcpy(buf, c->pool + base + start, *len * sizeof(int32_t), cudaMemcpyDeviceToHost), "reading a waveform");
    return GATSPI_OK;
}

gatspi_status gatspi_export_offsets(gatspi_ctx *c, int64_t *start, int32_t *len, size_t n) {
    g_err.clear();
    if (!c || (!start && !len)) return fail(GATSPI_EINVAL, "ctx and start or len are required");
    if ((long long)n != c->num_nets * c->W) return fail(GATSPI_EINVAL, "the arrays need num_nets * W entries");
    if (!c->loaded || !c->simulated) return fail(GATSPI_ESTATE, "simulate first");
    gatspi_status st = sync_ctx(c);
    if (st != GATSPI_OK) return st;
    std::vector<long long> base((size_t)c->num_nets);
    std::vector<uint32_t> ws((size_t)(c->num_nets * c->W)), we((size_t)(c->num_nets * c->W));
    CUDA_TRY(cudaMemcpy(base.data(), c->net_base, base.size() * sizeof(long long), cudaMemcpyDeviceToHost), "reading the window index");
    CUDA_TRY(cudaMemcpy(ws.data(), c->wstart, ws.size() * sizeof(uint32_t), cudaMemcpyDeviceToHost), "reading the window index");
    CUDA_TRY(cudaMemcpy(we.data(), c->wend, we.size() * sizeof(uint32_t), cudaMemcpyDeviceToHost), "reading the window index");
    for (long long net = 0; net < c->num_nets; ++net)
        for (int w = 0; w < c->W; ++w) {
            const long long k = net * c->W + w;
            if (start) start[k] = base[net] + ws[k];
            if (len) len[k] = (int32_t)(we[k] - ws[k]);
        }
    return GATSPI_OK;
}

gatspi_status gatspi_export_windows(gatspi_ctx *c, const int32_t *windows, int32_t nsel, int64_t *off, int32_t *words,
                                    size_t cap) {
    g_err.clear();
    if (!c || !windows || !off || nsel < 1) return fail(GATSPI_EINVAL, "ctx, windows (nsel >= 1) and off are required");
    for (int s = 0; s < nsel; ++s)
        if (windows[s] < 0 || windows[s] >= c->W) return fail(GATSPI_EINVAL, "window %d out of range", windows[s]);
    if (!c->loaded || !c->simulated) return fail(GATSPI_ESTATE, "simulate first");
    gatspi_status st = sync_ctx(c);
    if (st != GATSPI_OK) return st;
    const long long n = c->num_nets * nsel;
    int32_t *d_sel = nullptr;
    long long *d_len = nullptr;
    int32_t *d_words = nullptr;
    st = [&]() -> gatspi_status {
        CUDA_TRY(dev_alloc(&d_sel, (size_t)nsel), "allocating export scratch");
        CUDA_TRY(dev_alloc(&d_len, (size_t)n + 1), "allocating export scratch");
        CUDA_TRY(cudaMemcpy(d_sel, windows, sizeof(int32_t) * nsel, cudaMemcpyHostToDevice), "copying windows");
        const DevParams p = c->params();
        CUDA_TRY(launch_window_lengths(p, c->num_nets, d_sel, nsel, d_len, nullptr), "measuring waveforms");
        std::vector<long long> len((size_t)n);
        CUDA_TRY(cudaMemcpy(len.data(), d_len, sizeof(long long) * n, cudaMemcpyDeviceToHost), "reading lengths");
        long long acc = 0;
        for (long long k = 0; k < n; ++k) {
            off[k] = acc;
            acc += len[k];
        }
        off[n] = acc;
        if (!words) return GATSPI_OK;
        if ((long long)cap < acc) return fail(GATSPI_EINVAL, "words buffer of %zu too small for %lld", cap, acc);
        CUDA_TRY(cudaMemcpy(d_len, off, sizeof(long long) * (n + 1), cudaMemcpyHostToDevice), "copying offsets");
        CUDA_TRY(dev_alloc(&d_words, (size_t)acc), "allocating export scratch");
        CUDA_TRY(launch_window_gather(p, c->num_nets, d_sel, nsel, d_len, d_words, nullptr), "gathering waveforms");
        CUDA_TRY(cudaMemcpy(words, d_words, sizeof(int32_t) * acc, cudaMemcpyDeviceToHost), "reading waveforms");
        return GATSPI_OK;
    }();
    if (d_sel) cudaFree(d_sel);
    if (d_len) cudaFree(d_len);
    if (d_words) cudaFree(d_words);
    return st;
}

gatspi_status gatspi_net_digests(gatspi_ctx *c, int64_t net_begin, int64_t num_nets, uint64_t *digest,
                                 int64_t *words) {
    g_err.clear();
    if (!c || (!digest && num_nets)) return fail(GATSPI_EINVAL, "ctx and digest are required");
    if (net_begin < 0 || num_nets < 0 || net_begin + num_nets > c->num_nets)
        return fail(GATSPI_EINVAL, "nets [%lld, %lld) outside 0 .. %lld", (long long)net_begin,
                    (long long)(net_begin + num_nets), c->num_nets);
    if (!c->loaded) return fail(GATSPI_ESTATE, "load the inputs first");
    if (net_begin + num_nets > c->P && !c->simulated) return fail(GATSPI_ESTATE, "simulate before digesting gates");
    gatspi_status st = sync_ctx(c);
    if (st != GATSPI_OK || num_nets == 0) return st;
    unsigned long long *d_out = nullptr;
    long long *d_words = nullptr;
    st = [&]() -> gatspi_status {
        CUDA_TRY(dev_alloc(&d_out, (size_t)num_nets), "allocating digest scratch");
        CUDA_TRY(dev_alloc(&d_words, (size_t)num_nets), "allocating digest scratch");
        CUDA_TRY(launch_net_digests(c->params(), net_begin, num_nets, d_out, d_words, nullptr), "digesting waveforms");
        CUDA_TRY(cudaMemcpy(digest, d_out, sizeof(uint64_t) * num_nets, cudaMemcpyDeviceToHost), "reading digests");
        if (words)
            CUDA_TRY(cudaMemcpy(words, d_words, sizeof(int64_t) * num_nets, cudaMemcpyDeviceToHost), "reading counts");
        return GATSPI_OK;
    }();
    if (d_out) cudaFree(d_out);
    if (d_words) cudaFree(d_words);
    return st;
}

gatspi_status gatspi_device_views(gatspi_ctx *c, gatspi_views *v) {
    g_err.clear();
    if (!c || !v) return fail(GATSPI_EINVAL, "ctx and out are required");
    v->pool = c->pool;
    v->pool_words = c->pool_words;
    v->pool_used = 0;
    if (c->loaded) {
        gatspi_status st = sync_ctx(c);
        if (st != GATSPI_OK) return st;
        long long used = 0;
        CUDA_TRY(cudaMemcpy(&used, c->level_base + (c->simulated ? c->L : 0), sizeof used, cudaMemcpyDeviceToHost),
                 "reading the pool size");
        if (c->compact && c->simulated && c->L > 0) {   // the most any level needed with its scratch
            std::vector<long long> need((size_t)c->L);
            CUDA_TRY(cudaMemcpy(need.data(), c->level_need, sizeof(long long) * c->L, cudaMemcpyDeviceToHost),
                     "reading the pool size");
            for (long long n : need) used = std::max(used, n);
        }
        v->pool_used = used;
    }
    v->net_base = (const int64_t *)c->net_base;
    v->wstart = c->wstart;
    v->wend = c->wend;
    v->tc = c->tc;
    v->t1 = c->t1;
    v->num_nets = (int32_t)c->num_nets;
    v->num_windows = c->W;
    return GATSPI_OK;
}

gatspi_status gatspi_level_times(gatspi_ctx *c, float *sim_ms, float *bounds_ms, int32_t n) {
    g_err.clear();
    if (!c || (!sim_ms && !bounds_ms)) return fail(GATSPI_EINVAL, "ctx and an output array are required");
    if (n != c->L) return fail(GATSPI_EINVAL, "ms needs num_levels entries");
    if (!c->simulated) return fail(GATSPI_ESTATE, "simulate first");
    if (!c->timed_last) return fail(GATSPI_ESTATE, "the last simulate ran without GATSPI_FLAG_LEVEL_TIMING");
    gatspi_status st = sync_ctx(c);
    if (st != GATSPI_OK) return st;
    for (int l = 0; l < c->L; ++l) {
        if (bounds_ms)
            CUDA_TRY(cudaEventElapsedTime(&bounds_ms[l], c->events[2 * l], c->events[2 * l + 1]), "reading level events");
        if (sim_ms)
            CUDA_TRY(cudaEventElapsedTime(&sim_ms[l], c->events[2 * l + 1], c->events[2 * l + 2]), "reading level events");
    }
    return GATSPI_OK;
}

gatspi_status gatspi_set_level_timing(gatspi_ctx *c, int32_t on) {
    g_err.clear();
    if (!c) return fail(GATSPI_EINVAL, "ctx is NULL");
    if (on)
        c->flags |= GATSPI_FLAG_LEVEL_TIMING;
    else
        c->flags &= ~GATSPI_FLAG_LEVEL_TIMING;
    return GATSPI_OK;
}

gatspi_status gatspi_inject_scan_stall(gatspi_ctx *c, int32_t level, int64_t wait_ns) {
    g_err.clear();
    if (!c) return fail(GATSPI_EINVAL, "ctx is NULL");
    if (level < 0 || level >= c->L) return fail(GATSPI_EINVAL, "level %d out of range", level);
    if (c->launches[level].scan_tiles < 2)
        return fail(GATSPI_EINVAL, "level %d has %d gates: a stall needs more than %d", level,
                    c->launches[level].num_gates, kPlaceTile);
    if (wait_ns < 1000 || wait_ns > 10000000000ll) return fail(GATSPI_EINVAL, "wait_ns must be 1 us .. 10 s");
    c->stall_level = level;
    c->stall_wait_ns = wait_ns;
    return GATSPI_OK;
}

void gatspi_destroy(gatspi_ctx *c) {
    if (!c) return;
    cudaSetDevice(c->device);
    if (c->loaded || c->simulated) cudaStreamSynchronize(c->last_stream);
    free_all(c);
    delete c;
}

}  // extern "C"
