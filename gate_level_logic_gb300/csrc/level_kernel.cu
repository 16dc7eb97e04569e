// Level kernels of the GB300 gate-level re-simulator.
//
// Three launches per logic level (GATSPI, Section 3, Fig. 5, whose two passes they
// replace): planning, placement, simulation.
//
// level_plan_kernel plans the level before anything is simulated, one warp per
// gate.  An output window can hold at most 3 + sum over pins of (input length - 2)
// words: every stored toggle needs an iteration of the event loop and every
// iteration consumes at least one input transition.  The warp computes this bound
// for each of the gate's windows from the window index of its sources, ranks the
// windows by bound, largest first (a stable counting sort: equal bounds keep window
// order, so the layout depends only on the inputs), and sums the bounds of every
// group of 32 ranks.  The gate's region is the sum of all its bounds;
// level_place_kernel scans the region sizes in gate order (a decoupled look-back
// over tiles of 32 gates) into pool offsets.  The page sizes its outputs with a full
// counting pass instead; the bound replaces that pass and leaves a gap after each
// window (its size is the only cost).  The ranking is for load
// balance: a warp runs as long as its slowest lane, and the bound follows a window's
// event count closely, so a warp that gets 32 windows of similar bound keeps its
// lanes busy.
//
// level_kernel simulates.  A warp owns 32 slots: one gate and 32 consecutive ranks
// (or, for W < 32, several gates with all W windows each), so that a warp's lanes
// run the same cell as in the page's mapping.  Each lane runs Algorithm 1 of the page
// for its (gate, window): merge the fanin waveforms with interconnect inertial
// filtering, resolve simultaneous switching, look up the truth table by summed pin
// weights, pick the conditional delay (row = switching pin and edges, column = the
// other pins' values) and apply the gate's inertial filter.  The kernel comes in two
// variants: PATHPULSEPERCENT = 100, the page's setting, where the filter cancels
// exactly the output entries that have not matured and at most one is ever pending;
// and any other percentage q, where both filters compare against the reject limit
// floor(d * q / 100), several output entries can be pending and a cancel re-reads
// the entry before the one it exposes from the lane's own output.  Before
// simulating, each lane turns its inputs' lengths into its window's bound and a warp
// scan gives the window its slot, bound-sized, in the group's part of the region;
// the lane writes its output words straight there, and the gap after them (bound
// minus length) stays unused.  Every (gate, window) is simulated once and no word is
// moved afterwards.  The window index records each window's start and end relative
// to its net's region, since windows are stored in rank order.  TC and T1 are
// reduced per warp and added with one 64-bit atomic each.  The pins of a multi-pin
// cell live in a small shared-memory table per warp (see PinTab), so that the event
// loop keeps only the pins' next arrivals in registers and most of the SM's L1 is
// left to the source waveforms.  No warp waits for another.
//
// With 16 windows or fewer and long windows, level_chunk_kernel (chunk_kernel.cu)
// replaces level_kernel: one warp per gate, each window cut at quiet times of the gate
// into stretches that the lanes simulate in parallel; level_order_kernel orders the
// gates heaviest first and, with one window, splits the heaviest into segments of
// several warps.  The per-(gate, window) machinery both use is in lane.cuh.
//
// No kernel traps: a missing delay arc, pool overflow or a stalled look-back sets the
// device status word and the kernels carry on without writing out of bounds.  Input
// waveforms are checked when they are loaded (load_index_kernel, the testbench cut);
// every later waveform is this kernel's own output.
#include "gatspi_internal.cuh"
#include "lane.cuh"

namespace gatspi {

namespace {

// Exclusive prefix of this warp's tile within the level (decoupled look-back over
// warp tiles).  All 32 lanes take part: each probe reads the look-back words of 32
// predecessors at once, closest first, and stops at the first inclusive prefix.
// Publishes the tile's aggregate before looking back and its inclusive prefix
// after.  Waits are bounded: a stalled predecessor raises GATSPI_ETIMEOUT.
__device__ long long look_back(const DevParams &P, const LevelLaunch &L, int tile, long long total, int lane) {
    unsigned long long *st = P.tile_status + L.tile_base;
    if (tile == 0) {
        if (lane == 0) st_relaxed(st, kFlagIncl | (unsigned long long)total);
        return 0;
    }
    if (lane == 0) st_relaxed(st + tile, kFlagAgg | (unsigned long long)total);
    long long excl = 0;
    int k = tile - 1;
    const unsigned long long t0 = global_ns();
    unsigned sleep = 32;
    for (;;) {
        const int idx = k - lane;
        unsigned long long v = idx >= 0 ? ld_relaxed(st + idx) : kFlagIncl;
        const unsigned incl = __ballot_sync(0xffffffffu, (v >> 62) == 2);
        const unsigned busy = __ballot_sync(0xffffffffu, (v >> 62) == 0);
        const unsigned need = incl ? ((incl & (0u - incl)) << 1) - 1u : 0xffffffffu;  // lanes up to the first inclusive
        if (busy & need) {
            bool stop = false;
            if (lane == 0) {
                if (ld_status(P.status) != 0) {
                    stop = true;                                       // another warp failed: stop waiting
                } else if (global_ns() - t0 > P.spin_limit_ns) {
                    raise_error(P.status, GATSPI_ETIMEOUT, L.level, tile, k);
                    stop = true;
                }
            }
            if (__shfl_sync(0xffffffffu, (int)stop, 0)) break;
            __nanosleep(sleep);
            if (sleep < 1024) sleep <<= 1;
            continue;
        }
        long long part = (need >> lane) & 1u ? (long long)(v & kValueMask) : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        excl += part;
        if (incl) break;
        k -= 32;
    }
    if (lane == 0) st_relaxed(st + tile, kFlagIncl | (unsigned long long)(excl + total));
    return excl;
}

// Output bounds of a gate's W windows into bnd[], from the one-byte window lengths of
// its N sources: four consecutive windows per lane and load, summed over the pins
// in 16-bit halves (two windows per register); a length of 255 or more is read
// exactly from the index and added as a correction.  Returns this lane's sum.
template <int N>
__device__ __forceinline__ long long plan_bounds(const DevParams &P, int4 sv, int lane, uint32_t *bnd) {
    const int W = P.W;
    const int s4[GATSPI_MAX_PINS] = {sv.x, sv.y, sv.z, sv.w};
    long long lane_sum = 0;
    for (int w0 = 4 * lane; w0 < W; w0 += 4 * 32) {
        uint32_t even = 0, odd = 0;            // windows w0, w0 + 2 and w0 + 1, w0 + 3 in 16-bit halves
        uint32_t fix[4] = {0, 0, 0, 0};        // lengths beyond 255
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const long long src = s4[i];
            const uint32_t four = __ldg((const uint32_t *)(P.wlen8 + src * P.w8stride + w0));
            even += four & 0x00ff00ffu;
            odd += (four >> 8) & 0x00ff00ffu;
            if (__vcmpeq4(four, 0xffffffffu)) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int w = w0 + u;
                    if (((four >> (8 * u)) & 0xffu) == 0xffu && w < W)
                        fix[u] += __ldg(P.wend + src * W + w) - __ldg(P.wstart + src * W + w) - 255u;
                }
            }
        }
        const uint32_t base = 3u - 2u * (uint32_t)N;
        const uint32_t b[4] = {base + (even & 0xffffu) + fix[0], base + (odd & 0xffffu) + fix[1],
                               base + (even >> 16) + fix[2], base + (odd >> 16) + fix[3]};
        // the four bounds in one 16-byte store (padding words past W included): the
        // lanes' stores do not share banks
        *reinterpret_cast<uint4 *>(bnd + w0) = make_uint4(b[0], b[1], b[2], b[3]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (w0 + u < W) lane_sum += b[u];
    }
    return lane_sum;
}

// The plan of one gate per warp: window bounds, their ranking (largest first,
// stable), the offset of every group of 32 ranks and the region's size, stored
// after the group offsets (goff row of ngroups + 1 entries).  Shared memory per
// warp: the bounds of the gate's windows, the bucket counters of the counting sort,
// the group sums.  level_place_kernel then scans the sizes into pool offsets.
__global__ void __launch_bounds__(kPlanWarps * 32, kPlanMinBlocks) level_plan_kernel(const DevParams P, const LevelLaunch L) {
    extern __shared__ __align__(16) uint32_t psm[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    // every array starts 16-byte aligned, so four words move in one access
    uint32_t *bnd = psm + (size_t)warp * P.plan_words;
    uint32_t *hist = bnd + P.w8stride;
    uint32_t *gsum = hist + kSortBuckets;
    const int gl = blockIdx.x * (blockDim.x >> 5) + warp;   // the gate of this warp
    if (gl >= L.num_gates) return;
    const int g = L.gate_begin + gl;
    const int W = P.W;
    long long total = 0;
    {
        for (int k = lane; k < kSortBuckets; k += 32) hist[k] = 0;
        for (int k = lane; k < P.ngroups; k += 32) gsum[k] = 0;
        const int4 gd = __ldg(P.gate_desc + 3 * (long long)g);
        const int4 sv = __ldg(P.gate_desc + 3 * (long long)g + 1);
        __syncwarp();
        long long lane_sum = 0;
        switch (gd.y & 7) {   // warp-uniform: one gate per warp
            case 1: lane_sum = plan_bounds<1>(P, sv, lane, bnd); break;
            case 2: lane_sum = plan_bounds<2>(P, sv, lane, bnd); break;
            case 3: lane_sum = plan_bounds<3>(P, sv, lane, bnd); break;
            default: lane_sum = plan_bounds<4>(P, sv, lane, bnd); break;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) lane_sum += __shfl_xor_sync(0xffffffffu, lane_sum, o);
        total = lane_sum;
        __syncwarp();
    }
    {
        // bucket counts (bucket 0 = the largest bounds; bounds above 255 share it)
        for (int w = lane; w < W; w += 32)
            atomicAdd(&hist[kSortBuckets - 1 - min(bnd[w], (uint32_t)(kSortBuckets - 1))], 1u);
        __syncwarp();
        {   // exclusive scan of the bucket counts: the first rank of every bucket
            constexpr int kPer = kSortBuckets / 32;   // 8 buckets per lane, two 16-byte accesses
            static_assert(kPer == 8, "the scan moves a lane's buckets as two uint4");
            uint4 *mine = reinterpret_cast<uint4 *>(hist + lane * kPer);
            uint4 lo = mine[0], hi = mine[1];
            const uint32_t slo = lo.x + lo.y + lo.z + lo.w;
            uint32_t run = warp_incl_scan(slo + hi.x + hi.y + hi.z + hi.w, lane) - (slo + hi.x + hi.y + hi.z + hi.w);
            // exclusive prefix of the lane's eight buckets, in place
            uint32_t t = lo.x; lo.x = run; run += t;
            t = lo.y; lo.y = run; run += t;
            t = lo.z; lo.z = run; run += t;
            t = lo.w; lo.w = run; run += t;
            t = hi.x; hi.x = run; run += t;
            t = hi.y; hi.y = run; run += t;
            t = hi.z; hi.z = run; run += t;
            hi.w = run;
            mine[0] = lo;
            mine[1] = hi;
        }
        __syncwarp();
        // ranks, windows in order so that equal bounds keep window order
        for (int w0 = 0; w0 < W; w0 += 32) {
            const int w = w0 + lane;
            const bool act = w < W;
            const uint32_t b = act ? bnd[w] : 0u;
            const int key = act ? kSortBuckets - 1 - (int)min(b, (uint32_t)(kSortBuckets - 1)) : kSortBuckets + lane;
            const unsigned same = __match_any_sync(0xffffffffu, key);
            const uint32_t first = act ? hist[key] : 0u;
            __syncwarp();
            if (act && lane == __ffs(same) - 1) hist[key] = first + (uint32_t)__popc(same);
            __syncwarp();
            if (act) {
                const uint32_t rank = first + (uint32_t)__popc(same & ((1u << lane) - 1u));
                P.perm[(long long)gl * W + rank] = (uint16_t)w;
                atomicAdd(&gsum[rank >> 5], b);
            }
        }
        __syncwarp();
        // group offsets inside the gate's region
        long long run = 0;
        for (int j0 = 0; j0 < P.ngroups; j0 += 32) {
            const int j = j0 + lane;
            const uint32_t v = j < P.ngroups ? gsum[j] : 0u;
            const uint32_t incl = warp_incl_scan(v, lane);
            if (j < P.ngroups) P.goff[(long long)gl * (P.ngroups + 1) + j] = (uint32_t)(run + incl - v);
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            if (total >= (1ll << 32)) raise_error(P.status, GATSPI_EPOOL_OVERFLOW, L.level, g, 1);
            P.goff[(long long)gl * (P.ngroups + 1) + P.ngroups] = (uint32_t)total;   // the region's size
        }
    }
}

// The plan of one gate per warp when the windows are not ranked (many short
// windows): the windows' output bounds, 128 consecutive windows per step (four per
// lane from one 4-byte load of the byte lengths per pin, the bounds summed in 16-bit
// halves as in plan_bounds), each group of 32 windows (eight lanes) summed by a
// segmented warp reduction into the group offsets and the region's size.  No shared
// memory, no ranks.
template <int N>
__device__ __forceinline__ void plan_window_order(const DevParams &P, const LevelLaunch &L, int gl, int4 sv, int lane) {
    const int W = P.W;
    const int s4[GATSPI_MAX_PINS] = {sv.x, sv.y, sv.z, sv.w};
    uint32_t *goff = P.goff + (long long)gl * (P.ngroups + 1);
    long long run = 0;
    // kAhead steps' length words are loaded before any of them is summed, so that a
    // lane has that many loads per pin in flight instead of one
    constexpr int kAhead = 4;
    const int steps = (W + 127) / 128;
    for (int s0 = 0; s0 < steps; s0 += kAhead) {
        uint32_t fours[kAhead][N];
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            const int w0 = (s0 + u) * 128 + 4 * lane;
#pragma unroll
            for (int i = 0; i < N; ++i)
                fours[u][i] = w0 < W ? __ldg((const uint32_t *)(P.wlen8 + (long long)s4[i] * P.w8stride + w0)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            if (s0 + u >= steps) break;                  // warp-uniform
            const int w0 = (s0 + u) * 128 + 4 * lane;
            long long part = 0;   // this lane's four windows
            if (w0 < W) {
                uint32_t even = 0, odd = 0;        // windows w0, w0 + 2 and w0 + 1, w0 + 3 in 16-bit halves
                uint32_t fix[4] = {0, 0, 0, 0};    // lengths beyond 255
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    const long long src = s4[i];
                    const uint32_t four = fours[u][i];
                    even += four & 0x00ff00ffu;
                    odd += (four >> 8) & 0x00ff00ffu;
                    if (__vcmpeq4(four, 0xffffffffu)) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const int w = w0 + v;
                            if (((four >> (8 * v)) & 0xffu) == 0xffu && w < W)
                                fix[v] += __ldg(P.wend + src * W + w) - __ldg(P.wstart + src * W + w) - 255u;
                        }
                    }
                }
                const uint32_t base = 3u - 2u * (uint32_t)N;
                const uint32_t b[4] = {base + (even & 0xffffu) + fix[0], base + (odd & 0xffffu) + fix[1],
                                       base + (even >> 16) + fix[2], base + (odd >> 16) + fix[3]};
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (w0 + v < W) part += b[v];
            }
            // the group of 32 windows of this step that holds lane's windows: lanes 8k .. 8k+7
            long long gsum = part;
#pragma unroll
            for (int o = 4; o >= 1; o >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
            // the four groups' sums (lanes 0, 8, 16, 24) and their running offsets
            const long long g0 = __shfl_sync(0xffffffffu, gsum, 0), g1 = __shfl_sync(0xffffffffu, gsum, 8);
            const long long g2 = __shfl_sync(0xffffffffu, gsum, 16), g3 = __shfl_sync(0xffffffffu, gsum, 24);
            const int grp = (s0 + u) * 4;                    // first group of this step
            if (lane < 4 && grp + lane < P.ngroups) {
                const long long before = lane == 0 ? 0 : lane == 1 ? g0 : lane == 2 ? g0 + g1 : g0 + g1 + g2;
                goff[grp + lane] = (uint32_t)(run + before);
            }
            run += g0 + g1 + g2 + g3;
        }
    }
    if (lane == 0) {
        if (run >= (1ll << 32)) raise_error(P.status, GATSPI_EPOOL_OVERFLOW, L.level, L.gate_begin + gl, 1);
        goff[P.ngroups] = (uint32_t)run;   // the region's size
    }
}

__global__ void __launch_bounds__(kPlanWarps * 32) level_plan_window_order_kernel(const DevParams P, const LevelLaunch L) {
    const int lane = threadIdx.x & 31;
    const int gl = blockIdx.x * kPlanWarps + (threadIdx.x >> 5);
    if (gl >= L.num_gates) return;
    const int g = L.gate_begin + gl;
    const int4 gd = __ldg(P.gate_desc + 3 * (long long)g);
    const int4 sv = __ldg(P.gate_desc + 3 * (long long)g + 1);
    switch (gd.y & 7) {   // warp-uniform: one gate per warp
        case 1: plan_window_order<1>(P, L, gl, sv, lane); break;
        case 2: plan_window_order<2>(P, L, gl, sv, lane); break;
        case 3: plan_window_order<3>(P, L, gl, sv, lane); break;
        default: plan_window_order<4>(P, L, gl, sv, lane); break;
    }
}

// Pool offsets of the level's gate regions: their sizes (from the plan) scanned in
// gate order, one thread per gate and one tile of kPlaceTile gates per block (warp
// shuffles, then the warps' totals), and a decoupled look-back over the tiles; the
// values are ready when this kernel starts, so the waits are short and few.
// kMode: kPlaceFront -- the regions of the bounds from the front of the free pool;
// kPlaceTop -- the same regions placed down from the top of the pool (compaction:
// the level's scratch); kPlaceExact -- regions of the exact output sizes from the
// front (compaction: where the packing copy puts the level).
enum { kPlaceFront = 0, kPlaceTop = 1, kPlaceExact = 2 };

template <int kMode>
__global__ void __launch_bounds__(kPlaceTile) level_place_kernel(const DevParams P, const LevelLaunch L) {
    __shared__ long long warp_sum[kPlaceTile / 32];
    __shared__ int tile_id, stop;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        tile_id = atomicAdd(P.tickets + L.ticket, 1);
        stop = ld_status(P.status) != 0;
    }
    __syncthreads();
    const int tile = tile_id;
    if (tile >= L.scan_tiles) return;                      // spare blocks
    const int gl = tile * kPlaceTile + threadIdx.x;
    const bool valid = !stop && gl < L.num_gates;
    long long size = 0;
    if (valid) {
        if (kMode == kPlaceExact) {
            const uint32_t *ge = P.gexact + (long long)gl * P.ngroups;
            for (int c = 0; c < P.ngroups; ++c) size += __ldg(ge + c);
        } else {
            size = (long long)__ldg(P.goff + (long long)gl * (P.ngroups + 1) + P.ngroups);
        }
    }
    long long incl = size;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        // the warps' totals scanned, then the tile's offset from the look-back
        const long long t = warp_sum[lane];
        long long ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += v;
        }
        const long long total = __shfl_sync(0xffffffffu, ti, 31);
        const long long front = kMode == kPlaceTop ? 0 : P.level_base[L.level];
        const long long base = front + look_back(P, L, tile, total, lane);
        warp_sum[lane] = base + ti - t;                    // the first word of each warp's gates
        if (lane == 0 && tile == L.scan_tiles - 1) {
            if (kMode == kPlaceFront) {
                P.level_base[L.level + 1] = base + total;
                if (base + total > P.pool_words) raise_error(P.status, GATSPI_EPOOL_OVERFLOW, L.level, 0, 0);
            } else if (kMode == kPlaceTop) {
                // the level's scratch [pool top - total, pool top) must stay above the packed front
                P.level_bound[L.level] = base + total;
                if (P.level_base[L.level] + base + total > P.pool_words)
                    raise_error(P.status, GATSPI_EPOOL_OVERFLOW, L.level, 0, 0);
            } else {
                // the packed level must end below the scratch it is copied from
                const long long bound = P.level_bound[L.level];
                P.level_base[L.level + 1] = base + total;
                P.level_need[L.level] = base + total + bound;
                if (base + total + bound > P.pool_words) raise_error(P.status, GATSPI_EPOOL_OVERFLOW, L.level, 0, 0);
            }
        }
    }
    __syncthreads();
    if (valid) {
        const long long net = (long long)P.num_inputs + L.gate_begin + gl;
        if (kMode == kPlaceTop) {
            const long long b = P.pool_words - (warp_sum[warp] + incl);   // down from the top
            P.net_base[net] = b;
            P.old_base[gl] = b;
        } else {
            P.net_base[net] = warp_sum[warp] + incl - size;
        }
    }
}

// One warp = 32 slots of the level: a gate and 32 of its ranks.  Warps share nothing
// and never wait for each other.  kFull: PATHPULSEPERCENT = 100.
template <bool kFull>
__global__ void __launch_bounds__(kLevelBlock, kLevelMinBlocks) level_kernel(const DevParams P, const LevelLaunch L) {
    __shared__ int2 pin_hot[kLevelWarps][GATSPI_MAX_PINS * 32];       // [pin][lane] per warp
    __shared__ uint32_t pin_end[kLevelWarps][GATSPI_MAX_PINS * 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int tile = blockIdx.x * kLevelWarps + warp;
    if (tile >= L.num_tiles) return;                       // spare warps of the last block
    // the status word is read now but waited for only before the first store: after
    // an error the warp loads in bounds and writes nothing
    const int32_t st = lane == 0 ? ld_status(P.status) : 0;

    // slot -> (gate, group, rank): W >= 32 gives one (gate, group of 32 ranks) per
    // warp, W < 32 gives 32 >> lpg_log2 gates of lpg lanes each; the plan maps the
    // rank to a window
    int gl, c, j;
    if (P.lpg_log2 == 5) {
        // tile / ngroups: the multiply-high estimate is at most two below the quotient
        gl = (int)__umulhi((uint32_t)tile, P.ngroups_m);
        c = tile - gl * P.ngroups;
        if (c >= P.ngroups) { ++gl; c -= P.ngroups; }
        if (c >= P.ngroups) { ++gl; c -= P.ngroups; }
        j = lane;
    } else {
        // several gates per warp: the level's gates are taken by pin count, so that the
        // gates sharing a warp run the same code
        const int slot = tile * 32 + lane;
        gl = slot >> P.lpg_log2;
        if (P.gate_order && gl < L.num_gates) gl = __ldg(P.gate_order + L.gate_begin + gl) - L.gate_begin;
        c = 0;
        j = slot & ((1 << P.lpg_log2) - 1);
    }
    const int rank = c * 32 + j;
    const bool in_level = gl < L.num_gates;
    const bool loaded = in_level && rank < P.W;
    const int g = L.gate_begin + gl;
    const int w = loaded ? (P.ranked ? (int)__ldg(P.perm + (long long)gl * P.W + rank) : rank) : 0;

    const int seg_lead = lane & ~((1 << P.lpg_log2) - 1);  // first lane of this (gate, group) segment
    const long long net = (long long)P.num_inputs + g;

    // Slot of this window inside its group's part of the gate's region: the window's
    // own bound, 3 + sum over pins of (input length - 2), scanned over the segment in
    // rank order.  These bounds add up to what the plan reserved.
    // Pins of the gate in window w: source waveforms from the window index.
    int4 gd = make_int4(0, 0, 0, 0);
    int32_t Lw = 0;
    uint32_t bound = 0;
    uint32_t gofs = 0;      // the group's offset inside the gate's region
    long long base = 0;     // the group's first pool word
    Pin pins[GATSPI_MAX_PINS];
    if (loaded) {
        gd = __ldg(P.gate_desc + 3 * (long long)g);
        const int4 sv = __ldg(P.gate_desc + 3 * (long long)g + 1);
        const int4 dv = __ldg(P.gate_desc + 3 * (long long)g + 2);
        Lw = __ldg(P.window_len + w);
        switch (gd.y & 7) {   // warp-uniform when a warp holds one gate
            case 1: bound = load_pins<1>(P, sv, dv, w, pins); break;
            case 2: bound = load_pins<2>(P, sv, dv, w, pins); break;
            case 3: bound = load_pins<3>(P, sv, dv, w, pins); break;
            default: bound = load_pins<4>(P, sv, dv, w, pins); break;
        }
        gofs = __ldg(P.goff + (long long)gl * (P.ngroups + 1) + c);
        base = __ldg(P.net_base + net) + gofs;
    }
    const uint32_t bincl = warp_incl_scan(bound, lane);
    const uint32_t bexcl = bincl - bound;
    const uint32_t rel = bexcl - __shfl_sync(0xffffffffu, bexcl, seg_lead);
    const bool skip = __shfl_sync(0xffffffffu, st, 0) != 0;
    const bool gate_ok = in_level && !skip;
    const bool valid = loaded && !skip;

    LaneResult res{0, 0, 0, 0};
    if (valid) {
        const PinTab tab{&pin_hot[warp][lane], &pin_end[warp][lane]};
        res = dispatch<kFull>(P, gd, pins, tab, Lw, P.pool + base + rel);
        if (res.err) {
            raise_error(P.status, res.err, g, w, 0);
            res.len = 0;
        }
    }

    // TC and T1 per (gate, group): reduce over the segment's lanes, one atomic each
    long long tcs = res.tc, t1s = res.t1;
    if (P.lpg_log2 == 5) {
        // one gate per warp: exact 64-bit sums of the 32-bit counts from 16-bit halves
        const uint32_t tcu = (uint32_t)res.tc, t1u = (uint32_t)res.t1;
        tcs = ((long long)__reduce_add_sync(0xffffffffu, tcu >> 16) << 16) + __reduce_add_sync(0xffffffffu, tcu & 0xffffu);
        t1s = ((long long)__reduce_add_sync(0xffffffffu, t1u >> 16) << 16) + __reduce_add_sync(0xffffffffu, t1u & 0xffffu);
    } else {
        for (int o = (1 << P.lpg_log2) >> 1; o >= 1; o >>= 1) {
            tcs += __shfl_xor_sync(0xffffffffu, tcs, o);
            t1s += __shfl_xor_sync(0xffffffffu, t1s, o);
        }
    }
    if (gate_ok && j == 0) {
        atomicAdd(P.tc + g, (unsigned long long)tcs);
        atomicAdd(P.t1 + g, (unsigned long long)t1s);
    }
    if (P.compact) {   // the (gate, group)'s output words, for the packing
        uint32_t lsum = (uint32_t)res.len;
        if (P.lpg_log2 == 5) {
            lsum = __reduce_add_sync(0xffffffffu, lsum);
        } else {
            for (int o = (1 << P.lpg_log2) >> 1; o >= 1; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        }
        if (gate_ok && j == 0) P.gexact[(long long)gl * P.ngroups + c] = lsum;
    }

    if (valid) {
        P.wstart[net * P.W + w] = gofs + rel;
        P.wend[net * P.W + w] = gofs + rel + (uint32_t)res.len;
        P.wlen8[net * P.w8stride + w] = (uint8_t)min(res.len, 255);
    }
}

// Packing of a level's outputs (compaction): every window moves from its bound-sized
// slot in the level's scratch to its place in the gate's exact region, windows in
// rank order and back to back; the window index is rewritten relative to the packed
// region.  Same tiling as level_kernel (one (gate, group of 32 ranks) per warp, or
// several gates per warp below 32 windows); a group's first word is the sum of the
// gate's earlier groups' exact sizes.  The warp copies every segment's run of words
// across its lanes: stores contiguous, each word's window found by a search of fixed
// steps over the lanes' run offsets, so that every lane takes part in every shuffle.
__global__ void __launch_bounds__(kLevelBlock) level_pack_kernel(const DevParams P, const LevelLaunch L) {
    const int lane = threadIdx.x & 31;
    const int tile = blockIdx.x * kLevelWarps + (threadIdx.x >> 5);
    if (tile >= L.num_tiles) return;
    const bool stop = __shfl_sync(0xffffffffu, lane == 0 ? ld_status(P.status) : 0, 0) != 0;
    int gl, c, j;
    if (P.lpg_log2 == 5) {
        gl = (int)__umulhi((uint32_t)tile, P.ngroups_m);
        c = tile - gl * P.ngroups;
        if (c >= P.ngroups) { ++gl; c -= P.ngroups; }
        if (c >= P.ngroups) { ++gl; c -= P.ngroups; }
        j = lane;
    } else {
        const int slot = tile * 32 + lane;
        gl = slot >> P.lpg_log2;
        if (P.gate_order && gl < L.num_gates) gl = __ldg(P.gate_order + L.gate_begin + gl) - L.gate_begin;
        c = 0;
        j = slot & ((1 << P.lpg_log2) - 1);
    }
    const int rank = c * 32 + j;
    const bool in_level = gl < L.num_gates;
    const bool loaded = !stop && in_level && rank < P.W;
    const long long net = (long long)P.num_inputs + L.gate_begin + gl;
    const int w = loaded ? (P.ranked ? (int)__ldg(P.perm + (long long)gl * P.W + rank) : rank) : 0;
    const long long k = net * P.W + w;
    uint32_t ws = 0, len = 0;
    if (loaded) {
        ws = P.wstart[k];
        len = P.wend[k] - ws;
    }
    // the gate's earlier groups
    long long before = 0;
    if (P.lpg_log2 == 5 && in_level) {
        const uint32_t *ge = P.gexact + (long long)gl * P.ngroups;
        for (int cc = lane; cc < c; cc += 32) before += ge[cc];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    }
    // this window's place in its segment (rank order)
    const int seg_lead = lane & ~((1 << P.lpg_log2) - 1);
    const uint32_t incl = warp_incl_scan(len, lane);
    const uint32_t excl = incl - len - (__shfl_sync(0xffffffffu, incl, seg_lead) - __shfl_sync(0xffffffffu, len, seg_lead));
    const uint32_t rel = (uint32_t)before + excl;
    const long long src0 = loaded ? P.old_base[gl] + ws : 0;      // this window's first word (scratch)
    const long long dst0 = loaded ? P.net_base[net] + rel : 0;    // and its packed place
    const int seg_n = 1 << P.lpg_log2;
    for (int s0 = 0; s0 < 32; s0 += seg_n) {
        const uint32_t run = __shfl_sync(0xffffffffu, excl + len, s0 + seg_n - 1);   // the segment's words
        const long long dbase = __shfl_sync(0xffffffffu, dst0, s0);
        // four words per lane per round, their loads issued before their stores
        for (uint32_t x0 = 0; x0 < run; x0 += 128) {
            int32_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t x = x0 + 32u * u + lane;
                int lo = s0;   // last lane of the segment whose window starts at or before word x
                for (int step = seg_n >> 1; step >= 1; step >>= 1) {
                    const uint32_t e = __shfl_sync(0xffffffffu, excl, lo + step);
                    if (e <= x) lo += step;
                }
                const uint32_t e = __shfl_sync(0xffffffffu, excl, lo);
                const long long sb = __shfl_sync(0xffffffffu, src0, lo);
                v[u] = x < run ? __ldcg(P.pool + sb + (x - e)) : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t x = x0 + 32u * u + lane;
                if (x < run) P.pool[dbase + x] = v[u];
            }
        }
    }
    if (!loaded) return;
    P.wstart[k] = rel;
    P.wend[k] = rel + len;
}

// Window index of the loaded input waveforms and a format check of every one of
// them (Fig. 3): head [0] or [-1, 0], timestamps strictly increasing in 1 .. 2^30,
// EOW last.  One thread per (input, window).
__global__ void load_index_kernel(const DevParams P, const long long *__restrict__ off, long long nwords,
                                  int32_t *max_time) {
    const long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long n = (long long)P.num_inputs * P.W;
    if (k == 0) P.level_base[0] = nwords;
    if (k >= n) return;
    const int w = (int)(k % P.W);
    const long long pi = k / P.W;
    const long long s = off[k], e = off[k + 1];
    const long long c0 = off[k - w];                   // first word of the input's windows
    bool ok = s >= 0 && e <= nwords && e - s >= 2 && e - c0 < (1ll << 32) && c0 <= s && (k > 0 || s == 0);
    int32_t tmax = 0;
    if (ok) {
        const int32_t *x = P.pool + s;
        long long q = 0;
        if (x[0] == -1) {
            ok = x[1] == 0;
            q = 1;
        } else {
            ok = x[0] == 0;
        }
        int32_t prev = 0;
        for (long long i = q + 1; ok && i < e - s - 1; ++i) {
            ok = x[i] > prev && x[i] <= (1 << 30);
            prev = x[i];
        }
        ok = ok && x[e - s - 1] == kEOW;
        tmax = prev;
    }
    if (!ok) {
        raise_error(P.status, GATSPI_EBADWAVE, (int)pi, w, 0);
        return;
    }
    atomicMax(max_time, tmax);
    if (w == 0) P.net_base[pi] = c0;
    P.wstart[k] = (uint32_t)(s - c0);
    P.wend[k] = (uint32_t)(e - c0);
    P.wlen8[pi * P.w8stride + w] = (uint8_t)min(e - s, 255ll);
}

// Length of waveform (net, sel[s]) for an export of selected windows.
__global__ void window_lengths_kernel(const DevParams P, long long num_nets, const int32_t *__restrict__ sel, int nsel,
                                      long long *__restrict__ len) {
    const long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= num_nets * nsel) return;
    const long long net = k / nsel;
    const int w = sel[k % nsel];
    len[k] = (long long)(P.wend[net * P.W + w] - P.wstart[net * P.W + w]);
}

// Copy of waveform (net, sel[s]) to words[off[k] ..], one warp per waveform.
__global__ void window_gather_kernel(const DevParams P, long long num_nets, const int32_t *__restrict__ sel, int nsel,
                                     const long long *__restrict__ off, int32_t *__restrict__ words) {
    const long long k = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (k >= num_nets * nsel) return;
    const long long net = k / nsel;
    const int w = sel[k % nsel];
    const int32_t *src = P.pool + P.net_base[net] + P.wstart[net * P.W + w];
    const long long n = off[k + 1] - off[k];
    for (long long i = lane; i < n; i += 32) words[off[k] + i] = src[i];
}

// Digest of every net of [net0, net0 + n): 64-bit FNV-1a, a byte at a time, over the
// little-endian bytes of the net's waveforms in window order (each with its head and
// EOW), one thread per net.  For comparing runs without moving their waveforms.
__global__ void net_digest_kernel(const DevParams P, long long net0, long long n, unsigned long long *__restrict__ out,
                                  long long *__restrict__ words) {
    const long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= n) return;
    const long long net = net0 + k;
    const int32_t *base = P.pool + P.net_base[net];
    unsigned long long h = 14695981039346656037ull;
    long long count = 0;
    for (int w = 0; w < P.W; ++w) {
        const uint32_t s = P.wstart[net * P.W + w], e = P.wend[net * P.W + w];
        count += e - s;
        for (uint32_t i = s; i < e; ++i) {
            const uint32_t u = (uint32_t)base[i];
#pragma unroll
            for (int b = 0; b < 4; ++b) h = (h ^ ((u >> (8 * b)) & 0xffu)) * 1099511628211ull;
        }
    }
    out[k] = h;
    words[k] = count;
}

}  // namespace

cudaError_t launch_window_lengths(const DevParams &p, long long num_nets, const int32_t *sel, int nsel, long long *len,
                                  cudaStream_t s) {
    const long long n = num_nets * nsel;
    window_lengths_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p, num_nets, sel, nsel, len);
    return cudaGetLastError();
}

cudaError_t launch_window_gather(const DevParams &p, long long num_nets, const int32_t *sel, int nsel,
                                 const long long *off, int32_t *words, cudaStream_t s) {
    const long long n = num_nets * nsel;
    window_gather_kernel<<<(unsigned)((n * 32 + 255) / 256), 256, 0, s>>>(p, num_nets, sel, nsel, off, words);
    return cudaGetLastError();
}


cudaError_t launch_net_digests(const DevParams &p, long long net0, long long n, unsigned long long *out,
                               long long *words, cudaStream_t s) {
    if (n > 0) net_digest_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p, net0, n, out, words);
    return cudaGetLastError();
}

int plan_gates_per_tile(int) { return kPlanWarps; }

int plan_words(int W) {   // per warp: W bounds, the buckets, the group sums, each padded to 4 words
    return windows_ranked(W) ? ((W + 3) & ~3) + kSortBuckets + (((W + 31) / 32 + 3) & ~3) : 0;
}

size_t plan_smem_bytes(int W) {
    return (size_t)plan_gates_per_tile(W) * (size_t)plan_words(W) * sizeof(uint32_t);
}

cudaError_t launch_level_bounds(const DevParams &p, const LevelLaunch &l, cudaStream_t s) {
    const int wpb = plan_gates_per_tile(p.W);
    if (l.num_gates > 0) {
        const unsigned blocks = (unsigned)((l.num_gates + wpb - 1) / wpb);
        if (p.ranked)
            level_plan_kernel<<<blocks, wpb * 32, plan_smem_bytes(p.W), s>>>(p, l);
        else
            level_plan_window_order_kernel<<<blocks, kPlanWarps * 32, 0, s>>>(p, l);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.compact)
        level_place_kernel<kPlaceTop><<<(unsigned)l.scan_tiles, kPlaceTile, 0, s>>>(p, l);
    else
        level_place_kernel<kPlaceFront><<<(unsigned)l.scan_tiles, kPlaceTile, 0, s>>>(p, l);
    return cudaGetLastError();
}

cudaError_t launch_level_compact(const DevParams &p, const LevelLaunch &l, const LevelLaunch &exact, cudaStream_t s) {
    level_place_kernel<kPlaceExact><<<(unsigned)exact.scan_tiles, kPlaceTile, 0, s>>>(p, exact);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((l.num_tiles + kLevelWarps - 1) / kLevelWarps);
    level_pack_kernel<<<blocks, kLevelBlock, 0, s>>>(p, l);
    return cudaGetLastError();
}

cudaError_t launch_level_sim(const DevParams &p, const LevelLaunch &l, cudaStream_t s) {
    if (p.chunks > 1) return launch_level_chunks(p, l, s);   // chunk_kernel.cu
    const unsigned blocks = (unsigned)((l.num_tiles + kLevelWarps - 1) / kLevelWarps);
    if (p.pulse_percent == 100)
        level_kernel<true><<<blocks, kLevelBlock, 0, s>>>(p, l);
    else
        level_kernel<false><<<blocks, kLevelBlock, 0, s>>>(p, l);
    return cudaGetLastError();
}

cudaError_t launch_level(const DevParams &p, const LevelLaunch &l, cudaStream_t s) {
    const cudaError_t e = launch_level_bounds(p, l, s);
    return e != cudaSuccess ? e : launch_level_sim(p, l, s);
}

cudaError_t set_level_smem_limit() {
    // The simulation kernel's pin table takes 6 KB per block (7 KB with the driver's
    // reserve): 9 blocks fit the 64 KB shared-memory configuration, which leaves the
    // rest of the SM's 256 KB to L1 for the source waveforms.  The preference is a
    // percentage that the driver rounds up to a configuration: 20 gives 64 KB on
    // GB300 (28 already gives 100 KB; 0 gives 8 KB and a single block per SM).
    cudaError_t e = cudaFuncSetAttribute(level_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout, 20);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(level_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout, 20);
    if (e == cudaSuccess) e = set_chunk_smem_limit();
    // The planning kernel's dynamic shared memory limit is an attribute of the kernel,
    // shared by every context of the process: it is always set to what the largest
    // window count needs, so that no context lowers it below another's launches.
    size_t most = 0;
    for (int w = 1; w <= GATSPI_MAX_WINDOWS; ++w) most = plan_smem_bytes(w) > most ? plan_smem_bytes(w) : most;
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(level_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
    return e;
}

cudaError_t launch_load_index(const DevParams &p, const long long *off, long long nwords, int32_t *max_time,
                              cudaStream_t s) {
    const long long n = (long long)p.num_inputs * p.W;
    const int threads = 256;
    const long long blocks = n > 0 ? (n + threads - 1) / threads : 1;
    load_index_kernel<<<(unsigned)blocks, threads, 0, s>>>(p, off, nwords, max_time);
    return cudaGetLastError();
}

}  // namespace gatspi
