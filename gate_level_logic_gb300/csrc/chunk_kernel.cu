// Level kernels for windows cut into time chunks (16 windows or fewer, long windows,
// any PATHPULSEPERCENT): the cut search, the heaviest-first gate order (with the
// segments of one window's heavy gates), the moves that join the stretches, and
// level_chunk_kernel itself.  The per-lane simulation is lane.cuh's run_lane.
#include "gatspi_internal.cuh"
#include "lane.cuh"

namespace gatspi {

namespace {

// Windows cut into time chunks (16 windows or fewer, any PATHPULSEPERCENT): with
// few windows a lane runs its gate through a long stretch of the testbench and a level
// lasts as long as its busiest gate's serial chain.  Here a warp takes one gate and
// gives each of its windows K = 32 / W lanes; lane k of a window simulates the window
// from its k-th cut to the next.  A cut T is a time at which the gate is quiet: no
// pin has a transition in [T - M1, T + M2), M1 = the largest wire delay of its pins +
// its largest gate delay, M2 = that wire delay + 1.  Then, whatever happened before,
// every pin's entry in effect at T is its last transition before T (a pulse around T
// is wider than any reject limit, so none is swallowed across it), every arrival
// before T comes from a transition before T - M1 and every arrival at or after T from
// one at or after T + M2, and every output entry made before T lies before T, so no
// later event can cancel it (at q = 100 an entry is cancelled only by an event
// earlier than the entry; at any q an event after T makes an entry at least
// M2 + 1 + its delay d after every entry before T, more than the reject limit of d,
// so none of those is cancelled either).  The simulation from T on therefore needs only the pins'
// entries in effect and the output value at T (the truth table of the pins' values),
// and yields exactly the entries, toggles and time at 1 of the whole window's run.
// Lane k looks for its cut from k * Lw / K on (the first quiet time, within a few
// dozen transitions and before the next lane's start); a lane that finds none leaves
// its stretch to the lane before.  Each chunk writes its entries into its own part of
// the window's slot (as many words as its pins have transitions in the chunk); after
// the event loops the warp moves the entries of every chunk after the first down
// behind the previous one's, in ascending order (each word moves to a lower or equal
// address, so no word is overwritten before it is read), and closes the window with
// its EOW.
constexpr int kCutSteps = 64;   // transitions a cut search may pass before it gives up

// First index in [lo, hi] whose word is >= v; w[hi] >= v must hold (the EOW does).
__device__ __forceinline__ uint32_t lower_bound_words(const int32_t *w, uint32_t lo, uint32_t hi, long long v) {
    while (lo < hi) {
        const uint32_t mid = lo + ((hi - lo) >> 1);
        if ((long long)__ldg(w + mid) < v) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// The first quiet time at or after T0 (see above) and every pin's entry in effect
// there, or false when none is found before Tnext or within kCutSteps transitions.
template <int N>
__device__ __forceinline__ bool find_cut(Pin (&pins)[GATSPI_MAX_PINS], long long T0, long long Tnext, int32_t M1,
                                         int32_t M2, int32_t &T, uint32_t (&pos)[GATSPI_MAX_PINS]) {
    long long cur = T0 - M1 > 1 ? T0 - M1 : 1;   // where the quiet stretch would start
    if (cur + M1 >= Tnext) return false;
    uint32_t q[N];
    long long v[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        q[i] = lower_bound_words(pins[i].w, 1u, pins[i].len - 1u, cur);   // transitions are >= 1
        v[i] = __ldg(pins[i].w + q[i]);
    }
    for (int step = 0; step < kCutSteps; ++step) {
        long long m = v[0];
#pragma unroll
        for (int i = 1; i < N; ++i) m = m < v[i] ? m : v[i];
        if (m >= cur + M1 + M2) {                    // [cur, cur + M1 + M2) holds no transition
            T = (int32_t)(cur + M1);
#pragma unroll
            for (int i = 0; i < N; ++i) pos[i] = q[i] - 1u;
            return true;
        }
        cur = m + 1;
        if (cur + M1 >= Tnext) return false;
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (v[i] == m) {                         // m < EOW here, so q[i] + 1 is in the window
                ++q[i];
                v[i] = __ldg(pins[i].w + q[i]);
            }
    }
    return false;
}

// 8 blocks per SM: 64 registers, which the cut search and the moves use (9 blocks at
// 56 registers spill and run 2-8 % slower)
constexpr int kChunkMinBlocks = 8;
// The order in which level_chunk_kernel takes a level's gates: heaviest first (by the
// size of the gate's output region, the sum of its windows' bounds, in power-of-two
// classes), so that the longest warps start in the first wave and the light ones fill
// in around them instead of a heavy gate starting last and holding the level up.  One
// block; the order within a class is whatever the atomics give (it changes nothing in
// the results, only which warp runs when).
//
// With one window, a gate whose region exceeds the level's share per resident warp
// also gets up to kMaxSegments warps, one per segment of its window (see
// level_chunk_kernel), at least kSegmentMinWords bound words each (the join of the
// segments is one warp's serial work, which a short segment does not repay), while the
// level's budget of kExtraSegments extra warps lasts, heaviest gates first; seg_items
// then lists the warps' (gate, segment, segments).
constexpr int kOrderThreads = 1024;

__device__ __forceinline__ uint32_t pack_item(int gl, int q, int Q) {
    return (uint32_t)gl | ((uint32_t)q << 24) | ((uint32_t)(Q - 1) << 28);
}

__global__ void __launch_bounds__(kOrderThreads) level_order_kernel(const DevParams P, const LevelLaunch L) {
    __shared__ uint32_t cursor[33];
    __shared__ unsigned long long wtot[kOrderThreads / 32];
    __shared__ uint32_t wsum[kOrderThreads / 32];
    __shared__ unsigned long long total_s;
    __shared__ uint32_t carry;
    const int n = L.num_gates;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x < 33) cursor[threadIdx.x] = 0;
    __syncthreads();
    auto size_of = [&](int gl) { return __ldg(P.goff + (long long)gl * (P.ngroups + 1) + P.ngroups); };
    auto cls = [&](int gl) {   // 0 for the largest regions
        const uint32_t size = size_of(gl);
        return size ? __clz(size) : 32;
    };
    for (int gl = threadIdx.x; gl < n; gl += kOrderThreads) atomicAdd(&cursor[cls(gl)], 1u);
    __syncthreads();
    // the classes that may be split hold regions of 2 kSegmentMinWords words or more
    constexpr int kSplitClasses = __builtin_clzll(2 * kSegmentMinWords) - 32 + 1;
    __shared__ uint32_t splittable;
    if (threadIdx.x == 0) {
        uint32_t run = 0;
        for (int c = 0; c < 33; ++c) {
            if (c == kSplitClasses) splittable = run;
            const uint32_t v = cursor[c];
            cursor[c] = run;
            run += v;
        }
    }
    __syncthreads();
    for (int gl = threadIdx.x; gl < n; gl += kOrderThreads) P.heavy_order[atomicAdd(&cursor[cls(gl)], 1u)] = gl;
    if (!P.seg_items) return;
    __syncthreads();
    const int h = (int)splittable;   // the gates at the front of the order that may be split
    if (h == 0 || n >= (1 << 24)) {   // nothing to split: the chunk kernel takes heavy_order
        if (threadIdx.x == 0) *P.seg_count = 0;
        return;
    }

    // the level's total work, then the segments of the splittable gates in heavy-first
    // order (a block scan), the other gates one warp each
    unsigned long long t = 0;
    for (int gl = threadIdx.x; gl < n; gl += kOrderThreads) t += size_of(gl);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) wtot[wid] = t;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long sum = 0;
        for (int i = 0; i < kOrderThreads / 32; ++i) sum += wtot[i];
        total_s = sum;
    }
    __syncthreads();
    const unsigned long long total = total_s;
    const bool split = total > 0;
    for (int p0 = 0; p0 < h; p0 += kOrderThreads) {
        const int p = p0 + threadIdx.x;
        int gl = 0;
        uint32_t extra = 0;   // segments wanted beyond the first
        if (p < h) {
            gl = P.heavy_order[p];
            if (split) {
                const unsigned long long size = size_of(gl);
                unsigned long long want = (size * (unsigned)P.resident_warps + total - 1) / total;
                const unsigned long long most = size / kSegmentMinWords;   // long enough to pay for the join
                want = want > most ? most : want;
                want = want < 1 ? 1 : (want > kMaxSegments ? kMaxSegments : want);
                extra = (uint32_t)want - 1u;
            }
        }
        const uint32_t incl = warp_incl_scan(extra, lane);
        if (lane == 31) wsum[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            const uint32_t v = wsum[lane];
            const uint32_t vi = warp_incl_scan(v, lane);
            wsum[lane] = vi - v;
        }
        __syncthreads();
        const uint32_t excl = carry + wsum[wid] + incl - extra;
        if (p < h) {
            const uint32_t before = min(excl, (uint32_t)kExtraSegments);
            const uint32_t after = min(excl + extra, (uint32_t)kExtraSegments);
            const int Q = 1 + (int)(after - before);
            for (int q = 0; q < Q; ++q) P.seg_items[p + before + q] = pack_item(gl, q, Q);
        }
        __syncthreads();
        if (threadIdx.x == kOrderThreads - 1) carry = excl + extra;
        __syncthreads();
    }
    const uint32_t extras = min(carry, (uint32_t)kExtraSegments);
    for (int p = h + threadIdx.x; p < n; p += kOrderThreads) P.seg_items[p + extras] = pack_item(P.heavy_order[p], 0, 1);
    if (threadIdx.x == 0) *P.seg_count = (uint32_t)n + extras;
}

// Moves runs of words down inside the pool, all 32 lanes taking part: lane c owns a
// run of m words from p[dst + shift] to p[dst] (shift >= 0); the runs are listed in
// lane order and word i of the list belongs to the lane whose run starts last at or
// before i.  The caller guarantees that, within each region written, the list
// ascends by destination and no word's destination lies above its source, so that
// no word is overwritten before it is read; kMoveWords words per lane and round, all
// loads of a round before its stores (8: 0-3 % faster than 4, 2 % faster than 2).
__device__ __forceinline__ void move_runs(int32_t *p, uint32_t dst, uint32_t shift, uint32_t m, int lane) {
    constexpr int kMoveWords = 8;
    const uint32_t mincl = warp_incl_scan(m, lane);
    const uint32_t M = mincl - m;
    const uint32_t total = __shfl_sync(0xffffffffu, mincl, 31);
    __syncwarp();
    for (uint32_t i0 = 0; i0 < total; i0 += 32u * kMoveWords) {
        int32_t v[kMoveWords];
        uint32_t d[kMoveWords];
#pragma unroll
        for (int u = 0; u < kMoveWords; ++u) {
            const uint32_t i = i0 + 32u * u + (uint32_t)lane;
            int c = 0;
#pragma unroll
            for (int stp = 16; stp >= 1; stp >>= 1)
                if (__shfl_sync(0xffffffffu, M, c + stp) <= i) c += stp;
            d[u] = __shfl_sync(0xffffffffu, dst, c) + (i - __shfl_sync(0xffffffffu, M, c));
            const uint32_t sh = __shfl_sync(0xffffffffu, shift, c);
            v[u] = i < total ? __ldcg(p + d[u] + sh) : 0;
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < kMoveWords; ++u)
            if (i0 + 32u * u + (uint32_t)lane < total) p[d[u]] = v[u];
        __syncwarp();
    }
}

// With one window, a heavy gate's window is first split into Q segments at quiet
// times S_1 < ... < S_{Q-1} (searched from j * Lw / Q on, the same rule as the chunk
// cuts; every warp of the gate finds the same ones), and warp q takes segment q: its
// 32 lanes cut it into stretches as above, simulate them, and pack them in the
// segment's own part of the slot (from the head for segment 0, from 2 + the
// transitions before S_q otherwise).  Each warp then adds its toggles and signed
// time-at-1 sums to the gate's statistics, records its entry count, and increments
// the gate's counter (after a fence); the warp that takes it to Q moves segments 1 ..
// Q-1 down behind each other, writes the EOW and the window index, and adds the final
// time at 1.  No warp waits for another.  A segment whose quiet time is not found is
// empty, and the segment before it runs on to the next found one.
// kFull: PATHPULSEPERCENT = 100 (else the reject-limit filter, see run_lane).
// kSeg: the instantiation that can split a gate's one window into segments.  Its
// code generation also happens to run windows that are not split a little faster at
// high activity (1-2 % at 20 and 50 %, 2-16 windows) and a little slower at low (about
// 3 % at 5 %), so the host picks the instantiation by the loaded inputs' words per
// window (DevParams::seg_kernel).
template <bool kSeg, bool kFull>
__global__ void __launch_bounds__(kLevelBlock, kChunkMinBlocks) level_chunk_kernel(const DevParams P,
                                                                                  const LevelLaunch L) {
    __shared__ int2 pin_hot[kLevelWarps][GATSPI_MAX_PINS * 32];
    __shared__ uint32_t pin_end[kLevelWarps][GATSPI_MAX_PINS * 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int tile = blockIdx.x * kLevelWarps + warp;      // heaviest first
    int gl, q = 0, Q = 1;
    const int items = kSeg && P.seg_items ? (int)__ldg(P.seg_count) : 0;   // 0: no gate of the level is split
    if (items > 0) {
        if (tile >= items) return;
        const uint32_t it = __ldg(P.seg_items + tile);
        gl = (int)(it & 0xffffffu);
        q = (int)((it >> 24) & 15u);
        Q = (int)(it >> 28) + 1;
    } else {
        if (tile >= L.num_gates) return;
        gl = __ldg(P.heavy_order + tile);
    }
    // after an error (read now) the warp reads no waveform and writes nothing: the
    // window index of this level's sources may then never have been written
    const bool skip = __shfl_sync(0xffffffffu, lane == 0 ? ld_status(P.status) : 0, 0) != 0;
    const int K = P.chunks;
    const int W = P.W;
    const int rank = lane / K;
    const int k = lane - rank * K;
    const int lead = rank * K < 32 ? rank * K : 31;         // the window's first lane
    const bool loaded = rank < W;
    const int g = L.gate_begin + gl;
    const long long net = (long long)P.num_inputs + g;
    const int w = loaded ? (P.ranked ? (int)__ldg(P.perm + (long long)gl * W + rank) : rank) : 0;

    const int4 gd = __ldg(P.gate_desc + 3 * (long long)g);
    const int4 sv = __ldg(P.gate_desc + 3 * (long long)g + 1);
    const int4 dv = __ldg(P.gate_desc + 3 * (long long)g + 2);
    const int n = gd.y & 7;
    const int32_t Lw = loaded ? __ldg(P.window_len + w) : 0;
    Pin pins[GATSPI_MAX_PINS];
    uint32_t bound = 0;
    if (loaded) {
        switch (n) {
            case 1: bound = load_pins<1>(P, sv, dv, w, pins); break;
            case 2: bound = load_pins<2>(P, sv, dv, w, pins); break;
            case 3: bound = load_pins<3>(P, sv, dv, w, pins); break;
            default: bound = load_pins<4>(P, sv, dv, w, pins); break;
        }
    }
    const uint32_t gofs = __ldg(P.goff + (long long)gl * (P.ngroups + 1));
    const long long base = __ldg(P.net_base + net) + gofs;

    // the window's slot: a scan of the windows' bounds in rank order
    const uint32_t bw = loaded && k == 0 ? bound : 0u;
    const uint32_t bexcl = warp_incl_scan(bw, lane) - bw;
    const uint32_t slotrel = __shfl_sync(0xffffffffu, bexcl, lead);
    int32_t *slot = P.pool + base + slotrel;

    // the margins of a quiet time: the largest wire delay of the pins and the largest
    // finite delay of the gate's table (read by the whole warp)
    int32_t wdmax = 0;
    {
        const int d4[GATSPI_MAX_PINS] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
        for (int i = 0; i < GATSPI_MAX_PINS; ++i)
            if (i < n) wdmax = max(wdmax, max(d4[i] & 0xffff, (int)((uint32_t)d4[i] >> 16)));
    }
    uint32_t dgmax = 0;
    {
        const long long dly = (long long)(uint32_t)gd.z | ((long long)gd.w << 32);
        const int entries = (2 * n) << n;
        for (int e = lane; e < entries; e += 32) {
            const int32_t d = __ldg(P.dly_data + dly + e);
            if (d != kNoArc) dgmax = max(dgmax, (uint32_t)d);
        }
        dgmax = __reduce_max_sync(0xffffffffu, dgmax);
    }
    const int32_t M1 = wdmax + (int32_t)dgmax, M2 = wdmax + 1;
    auto cut = [&](long long T0, long long Tn, int32_t &T, uint32_t (&pos)[GATSPI_MAX_PINS]) {
        switch (n) {
            case 1: return find_cut<1>(pins, T0, Tn, M1, M2, T, pos);
            case 2: return find_cut<2>(pins, T0, Tn, M1, M2, T, pos);
            case 3: return find_cut<3>(pins, T0, Tn, M1, M2, T, pos);
            default: return find_cut<4>(pins, T0, Tn, M1, M2, T, pos);
        }
    };
    // every pin's entry in effect at the window's start
    uint32_t pos0[GATSPI_MAX_PINS] = {0, 0, 0, 0};
    if (loaded && !skip) {
#pragma unroll
        for (int i = 0; i < GATSPI_MAX_PINS; ++i)
            if (i < n) pos0[i] = __ldg(pins[i].w) == -1 ? 1u : 0u;
    }

    // The segment of this warp (one window: all lanes hold it): from S_q to the next
    // quiet time found after it, or to the window's end.
    bool seg_ok = true;
    int32_t segS = 0, segE = kEOW;
    uint32_t posS[GATSPI_MAX_PINS] = {pos0[0], pos0[1], pos0[2], pos0[3]};
    uint32_t posE[GATSPI_MAX_PINS] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < GATSPI_MAX_PINS; ++i)
        if (loaded && i < n) posE[i] = pins[i].len - 2u;
    uint32_t Rj = 2;          // lane j: first word of segment j's part of the slot
    if (kSeg && Q > 1) {
        bool ok = lane == 0;
        int32_t Sj = 0;
        uint32_t pj[GATSPI_MAX_PINS] = {pos0[0], pos0[1], pos0[2], pos0[3]};
        if (!skip && lane >= 1 && lane < Q) {
            const long long T0 = (long long)lane * Lw / Q;
            const long long Tn = lane + 1 < Q ? (long long)(lane + 1) * Lw / Q : (long long)Lw;
            ok = cut(T0, Tn, Sj, pj);
        }
#pragma unroll
        for (int i = 0; i < GATSPI_MAX_PINS; ++i)
            if (i < n) Rj += pj[i] - pos0[i];
        const unsigned smask = __ballot_sync(0xffffffffu, ok) & ((1u << Q) - 1u);
        seg_ok = (smask >> q) & 1u;
        const unsigned after = smask & ~((2u << q) - 1u);
        const int e = after ? __ffs(after) - 1 : q;
        segS = __shfl_sync(0xffffffffu, Sj, q);
        const int32_t Se = __shfl_sync(0xffffffffu, Sj, e);
        if (after) segE = Se;
#pragma unroll
        for (int i = 0; i < GATSPI_MAX_PINS; ++i) {
            posS[i] = __shfl_sync(0xffffffffu, pj[i], q);
            const uint32_t pe = __shfl_sync(0xffffffffu, pj[i], e);
            if (after) posE[i] = pe;
        }
    }
    const uint32_t segR = kSeg ? __shfl_sync(0xffffffffu, Rj, q & 31) : 2u;   // this segment's part of the slot (q >= 1)

    // this lane's cut and every pin's entry in effect there (lane 0 of a window: its
    // start, or the segment's)
    bool valid = false;
    int32_t T = 0;
    uint32_t pos[GATSPI_MAX_PINS] = {0, 0, 0, 0};
    if (loaded && !skip && seg_ok) {
        if (k == 0) {
            valid = true;
            T = segS;
#pragma unroll
            for (int i = 0; i < GATSPI_MAX_PINS; ++i) pos[i] = posS[i];
        } else {
            const long long s0 = segS, span = (segE == kEOW ? (long long)Lw : (long long)segE) - s0;
            const long long T0 = s0 + (long long)k * span / K;
            const long long Tn = s0 + (k + 1 < K ? (long long)(k + 1) * span / K : span);
            valid = cut(T0, Tn, T, pos);
        }
    }
    // the chunk runs to the next valid cut of the segment (or to the segment's end)
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    const unsigned seg = (K == 32 ? 0xffffffffu : ((1u << K) - 1u)) << (lead & 31);
    const unsigned above = lane == 31 ? 0u : ~((2u << lane) - 1u);
    const unsigned later = vmask & seg & above;
    const int nxt = later ? __ffs(later) - 1 : lane;
    const int32_t tend_n = __shfl_sync(0xffffffffu, T, nxt);
    const int32_t tend = later ? tend_n : segE;
    uint32_t cb = 0;   // transitions of the chunk over its pins: a bound on its entries
#pragma unroll
    for (int i = 0; i < GATSPI_MAX_PINS; ++i) {
        const uint32_t pe_n = __shfl_sync(0xffffffffu, pos[i], nxt);
        if (valid && i < n) cb += (later ? pe_n : posE[i]) - pos[i];
    }
    // chunk regions inside the slot: chunk 0 of the window from word 0 (head and
    // entries), the next chunks from word 2 + the bounds of the chunks before them; a
    // later segment's chunks from its own first word on
    const uint32_t cbx = valid ? cb : 0u;
    const uint32_t cexcl = warp_incl_scan(cbx, lane) - cbx;
    const uint32_t off = (q == 0 ? 2u : segR) + cexcl - __shfl_sync(0xffffffffu, cexcl, lead);
    const bool from_start = k == 0 && q == 0;

    LaneResult res{0, 0, 0, 0};
    if (valid) {
        const PinTab tab{&pin_hot[warp][lane], &pin_end[warp][lane]};
#pragma unroll
        for (int i = 0; i < GATSPI_MAX_PINS; ++i) pins[i].p = pos[i];
        res = dispatch<kFull, true>(P, gd, pins, tab, Lw, from_start ? slot : slot + off - 1, from_start, tend,
                                   (int32_t)cb);
        if (res.err) raise_error(P.status, res.err, g, w, k);
    }
    // exact places: chunk k's entries follow the head (or the segment's start) and the
    // entries of the chunks before it (never more than the chunk's bound, even after a
    // recorded fault)
    const int32_t cnt = valid ? min(res.tc, (int32_t)cb) : 0;
    const int32_t y0w = __shfl_sync(0xffffffffu, res.len - res.tc, lead);   // the window's initial value (q = 0)
    const uint32_t first = q == 0 ? (uint32_t)y0w + 1u : segR;
    const uint32_t incl = warp_incl_scan((uint32_t)cnt, lane);
    const uint32_t E = first + (incl - (uint32_t)cnt) - (__shfl_sync(0xffffffffu, incl, lead) -
                                                         (uint32_t)__shfl_sync(0xffffffffu, cnt, lead));
    const uint32_t Eend = __shfl_sync(0xffffffffu, E + (uint32_t)cnt, (lead + K - 1) & 31);

    // every chunk after the first moved behind the one before it, as one list over all
    // the warp's windows
    if (!skip) move_runs(P.pool + base, slotrel + E, (k == 0 ? E : off) - E, loaded && k > 0 ? (uint32_t)cnt : 0u, lane);

    long long tcs = cnt;
    long long t1s = valid ? (long long)res.t1 : 0;
    if (!kSeg || Q == 1) {
        const bool head = loaded && k == 0 && !skip;
        if (head) {
            slot[Eend] = kEOW;
            const uint32_t len = Eend + 1u;
            P.wstart[net * W + w] = gofs + slotrel;
            P.wend[net * W + w] = gofs + slotrel + len;
            P.wlen8[net * P.w8stride + w] = (uint8_t)min(len, 255u);
        }
        // TC and T1 of the gate: every chunk's entries and signed sums, and each
        // window's final value over its length
        t1s += head && ((Eend - 1u) & 1u) ? (long long)Lw : 0;
        long long ws_len = head ? (long long)Eend + 1 : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            tcs += __shfl_xor_sync(0xffffffffu, tcs, o);
            t1s += __shfl_xor_sync(0xffffffffu, t1s, o);
            ws_len += __shfl_xor_sync(0xffffffffu, ws_len, o);
        }
        if (lane == 0 && !skip) {
            atomicAdd(P.tc + g, (unsigned long long)tcs);
            atomicAdd(P.t1 + g, (unsigned long long)t1s);
            if (P.compact) P.gexact[(long long)gl * P.ngroups] = (uint32_t)ws_len;
        }
        return;
    }

    // a segment of a split window (one window): its statistics, its entry count, then
    // the join by the last of the gate's warps to finish
    if constexpr (kSeg) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            tcs += __shfl_xor_sync(0xffffffffu, tcs, o);
            t1s += __shfl_xor_sync(0xffffffffu, t1s, o);
        }
        if (lane == 0) {
            if (!skip) {
                atomicAdd(P.tc + g, (unsigned long long)tcs);
                atomicAdd(P.t1 + g, (unsigned long long)t1s);
            }
            P.seg_cnt[(long long)gl * kMaxSegments + q] = (Eend - first) | (q == 0 && y0w ? 0x80000000u : 0u);
        }
        __threadfence();   // this warp's words and count before its arrival
        __syncwarp();
        int arrived = 0;
        if (lane == 0) arrived = atomicAdd(P.seg_counter + gl, 1);
        const bool last = __shfl_sync(0xffffffffu, arrived, 0) == Q - 1;
        if (!last) return;
        __threadfence();
        const bool bad = __shfl_sync(0xffffffffu, lane == 0 ? ld_status(P.status) : 0, 0) != 0;
        if (lane == 0) P.seg_counter[gl] = 0;   // ready for the next level
        if (bad) return;
        const uint32_t cj = lane < Q ? __ldcg(P.seg_cnt + (long long)gl * kMaxSegments + lane) : 0u;
        const uint32_t y0 = __shfl_sync(0xffffffffu, cj, 0) >> 31;
        const uint32_t nj = cj & 0x7fffffffu;
        const uint32_t jincl = warp_incl_scan(nj, lane);
        const uint32_t Ej = y0 + 1u + jincl - nj;               // segment j's exact first word
        const uint32_t Sj = lane == 0 ? Ej : Rj;                // where its entries are now
        move_runs(P.pool + base, slotrel + Ej, Sj - Ej, lane >= 1 && lane < Q ? nj : 0u, lane);
        const uint32_t Ew = y0 + 1u + __shfl_sync(0xffffffffu, jincl, 31);   // the window's EOW word
        if (lane == 0) {
            slot[Ew] = kEOW;
            P.wstart[net * W + w] = gofs + slotrel;
            P.wend[net * W + w] = gofs + slotrel + Ew + 1u;
            P.wlen8[net * P.w8stride + w] = (uint8_t)min(Ew + 1u, 255u);
            if ((Ew - 1u) & 1u) atomicAdd(P.t1 + g, (unsigned long long)Lw);
            if (P.compact) P.gexact[(long long)gl * P.ngroups] = Ew + 1u;
        }
    }
}

}  // namespace

cudaError_t launch_level_chunks(const DevParams &p, const LevelLaunch &l, cudaStream_t s) {
    // one warp per gate (or segment of one window), heaviest first
    if (l.num_gates > 0) {
        const long long warps = (long long)l.num_gates + (p.seg_items ? kExtraSegments : 0);
        const unsigned blocks = (unsigned)((warps + kLevelWarps - 1) / kLevelWarps);
        level_order_kernel<<<1, kOrderThreads, 0, s>>>(p, l);
        const bool full = p.pulse_percent == 100;
        if (p.seg_kernel && full)
            level_chunk_kernel<true, true><<<blocks, kLevelBlock, 0, s>>>(p, l);
        else if (p.seg_kernel)
            level_chunk_kernel<true, false><<<blocks, kLevelBlock, 0, s>>>(p, l);
        else if (full)
            level_chunk_kernel<false, true><<<blocks, kLevelBlock, 0, s>>>(p, l);
        else
            level_chunk_kernel<false, false><<<blocks, kLevelBlock, 0, s>>>(p, l);
    }
    return cudaGetLastError();
}

cudaError_t set_chunk_smem_limit() {
    // the same pin table and shared-memory configuration as level_kernel
    const cudaFuncAttribute a = cudaFuncAttributePreferredSharedMemoryCarveout;
    cudaError_t e = cudaFuncSetAttribute(level_chunk_kernel<false, true>, a, 20);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(level_chunk_kernel<true, true>, a, 20);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(level_chunk_kernel<false, false>, a, 20);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(level_chunk_kernel<true, false>, a, 20);
    return e;
}

}  // namespace gatspi
