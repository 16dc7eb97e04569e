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
// With 16 windows or fewer and long windows, level_chunk_kernel replaces level_kernel:
// one warp per gate, each window cut at quiet times of the gate into stretches that
// the lanes simulate in parallel (see there); level_order_kernel orders the gates
// heaviest first and, with one window, splits the heaviest into segments of several
// warps.
//
// No kernel traps: a missing delay arc, pool overflow or a stalled look-back sets the
// device status word and the kernels carry on without writing out of bounds.  Input
// waveforms are checked when they are loaded (load_index_kernel, the testbench cut);
// every later waveform is this kernel's own output.
#include "gatspi_internal.cuh"

namespace gatspi {

namespace {

__device__ __forceinline__ unsigned long long ld_relaxed(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ int ld_status(const int32_t *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ void raise_error(int32_t *status, int code, int a, int b, int c) {
    if (atomicCAS(status, 0, code) == 0) {
        status[1] = a;
        status[2] = b;
        status[3] = c;
    }
}

// One fanin pin of a lane.
struct Pin {
    const int32_t *w;  // the source net's waveform for this window
    uint32_t len;      // its length in words, EOW included
    uint32_t p;        // index of the entry in effect (value = p & 1)
    int32_t a;         // arrival time of the next transition at the pin, or EOW
    int32_t nx;        // w[p + 1]: the next transition's time, kept from the previous step
    uint32_t drf;      // interconnect delays: rise | fall << 16
};

// Reject limit of delay d at PATHPULSEPERCENT q (d * q < 2^31 for every delay the
// library accepts).
__device__ __forceinline__ int32_t reject_limit(int32_t d, int32_t q) {
    return (int32_t)((uint32_t)d * (uint32_t)q / 100u);
}

// Next arrival of a pin: skip every pulse narrower than the interconnect delay of
// its first edge (the fall delay when the pin is at 1, the rise delay when at 0),
// or than that delay's reject limit when kFull is false; the arrival is the next
// timestamp plus the delay.  On entry s.nx holds w[p + 1] (the word after the
// previous pulse test), so a step loads one word.  The common step is straight-line
// code, so that lanes advancing different pins stay together; only a swallowed
// pulse takes the loop.  The waves are well formed: inputs are checked when they are
// loaded and every output is written by this kernel; whatever a wave holds, the
// reads stay inside it (len bounds them) and the loop ends.
// p and len may be offsets from any base w (the entry is w[p], the window ends at
// w[len]); par is the pin's value in entry p (p's parity when p counts from the
// window's start).  t2pre: w[p + 2] when the caller has it already (a wave's first
// words are loaded together), else unused.
template <bool kFull, bool kPre = false>
__device__ __forceinline__ void next_arrival(uint32_t &p, int32_t &a, int32_t &nx, const int32_t *__restrict__ w,
                                             uint32_t len, uint32_t drf, uint32_t par, int32_t q, int32_t t2pre = 0) {
    bool last = p + 2 >= len;                      // p + 1 is the EOW slot: no further transition
    int32_t t1 = nx;
    int32_t t2 = kPre ? t2pre : (last ? kEOW : __ldg(w + p + 2));
    // a long window: on entering a new 32-byte sector, ask L1 for the next one, so that
    // a lane running through hundreds of words does not wait for every sector in turn
    if (!kPre && (((uintptr_t)(w + p + 2) & 31u) == 0) && p + 10 < len)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(w + p + 10));
    const int32_t d = par ? (int32_t)(drf >> 16) : (int32_t)(drf & 0xffffu);
    const int32_t lim = kFull ? d : reject_limit(d, q);
    if (!last && t2 - t1 < lim) {                   // the pulse [t1, t2) never reaches the pin
        for (;;) {
            p += 2;                                 // same parity: same delay
            last = p + 2 >= len;
            if (last) break;
            t1 = __ldg(w + p + 1);
            t2 = __ldg(w + p + 2);
            if (t2 - t1 >= lim) break;
        }
    }
    a = last ? kEOW : t1 + d;
    nx = t2;                                        // w[p + 2]: the next transition once this one is taken
}

// A pin of a multi-pin cell in the event loop lives in shared memory (one column per
// lane, 12 bytes): the offset of its entry in effect and the word after the next
// transition in one 8-byte entry, the offset one past its window's last word in a
// 4-byte one, offsets counted in words from the lowest of the lane's waveform
// pointers.  Only the pins' next arrivals and wire delays stay in registers (the loop
// takes the arrivals' minimum every step), so a step reads the switching pin with two
// shared loads and writes it back with one store instead of moving every field
// through per-pin selects, and the table is small enough to leave most of the SM's
// L1 to the source waveforms.  A lane whose waveforms lie 2^32 words apart or more
// (pools beyond 16 GiB) counts each pin's offsets from its own window instead, and the
// step selects the switching pin's window pointer (kPinsFar).
struct PinTab {
    int2 *hot;          // [pin * 32 + lane]: {entry offset, next word}
    uint32_t *end;      // [pin * 32 + lane]
};

struct LaneResult {
    int32_t len;   // output words, EOW included
    int32_t tc;    // output toggles
    int32_t t1;    // time at 1 within [0, Lw)
    int32_t err;   // 0 or a gatspi_status
};

// Delay of the arc of switching pin i to output edge e_out.  The table was laid out
// at create so that the Fig. 4 entry for row 4*i + 2*e_in + e_out and the column of
// the other pins' values sits at ((2*i + e_out) << N) | vbits, vbits holding every
// pin's new value (pin j at bit N-1-j; pin i's bit gives e_in).
template <int N>
__device__ __forceinline__ int32_t arc_delay(const int32_t *__restrict__ D, uint32_t vbits, int i, int e_out) {
    return __ldg(D + ((((uint32_t)i << 1) | (uint32_t)e_out) << N | vbits));
}

// Where a multi-pin lane's pin table counts its offsets from (kPins): kPinsNear, from
// the lowest of the lane's waveform pointers, one pointer for every pin (the lane's
// waveforms lie within 2^32 words); kPinsFar, from each pin's own window, whose
// pointer the step selects among the pins' (a few more instructions, no limit on how
// far apart the sources lie).  A one-pin cell keeps its pin in registers (kPinsOne).
enum { kPinsOne = 0, kPinsNear = 1, kPinsFar = 2 };

// Take the transition of pin k (chosen per lane) that has just arrived and find the
// pin's next arrival.  vbits holds every pin's value after the step.
template <int N, bool kFull, int kPins>
__device__ __forceinline__ void advance_pin(Pin (&pin)[N], const int32_t *lb, const PinTab &tab, int k,
                                            uint32_t vbits, int32_t q) {
    if constexpr (N == 1) {
        ++pin[0].p;
        next_arrival<kFull>(pin[0].p, pin[0].a, pin[0].nx, pin[0].w, pin[0].len, pin[0].drf, pin[0].p & 1u, q);
    } else {
        const int2 h = tab.hot[k * 32];
        const uint32_t end = tab.end[k * 32];
        uint32_t drf = pin[0].drf;
        const int32_t *base = kPins == kPinsNear ? lb : pin[0].w;
#pragma unroll
        for (int i = 1; i < N; ++i)
            if (k == i) {
                drf = pin[i].drf;
                if constexpr (kPins == kPinsFar) base = pin[i].w;
            }
        uint32_t off = (uint32_t)h.x + 1u;
        int32_t nx = h.y, a;
        next_arrival<kFull>(off, a, nx, base, end, drf, (vbits >> (N - 1 - k)) & 1u, q);
        tab.hot[k * 32] = make_int2((int32_t)off, nx);
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (k == i) pin[i].a = a;
    }
}

// Whether a lane's pins can use 32-bit offsets from the lowest of their waveform
// pointers (that pointer in lb): kPinsNear, else kPinsFar.
template <int N>
__device__ __forceinline__ bool table_fits(const Pin (&pin)[N], const int32_t *&lb) {
    lb = pin[0].w;
#pragma unroll
    for (int i = 1; i < N; ++i) lb = pin[i].w < lb ? pin[i].w : lb;
    bool fits = true;
#pragma unroll
    for (int i = 0; i < N; ++i) fits &= (unsigned long long)(pin[i].w - lb) + pin[i].len < 0xfffffff0ull;
    return fits;
}

// Algorithm 1 for one (gate, window).  The output words go to gout, the window's
// slot in the pool.
// The loop body is written so that a warp's lanes stay together: the switching
// pins form a bit mask, the delay lookup and the pin advance serve the first
// switching pin through a lane-selected pin state, and only simultaneous
// switching of several pins takes an extra (rare) loop.
// kChunk: one time chunk of the window (level_chunk_kernel).  A chunk that does not
// start the window starts from each pin's entry in effect at its cut (pin[i].p, set
// by the caller), with no output entry pending, and writes no head: its entries go to
// gout[1], gout[2], ... (gout is moved down by the output value at the cut, so that
// the parity of an entry's index stays its value).  Every chunk stops before the
// first arrival at or after tend, writes no EOW, and returns in len the index of its
// last entry, in tc its entries (stores less cancels) and in t1 its signed sum of
// clipped entries, without the final adjustment.
template <int N, bool kFull, int kPins, bool kChunk = false>
__device__ __forceinline__ LaneResult run_lane(Pin (&pin)[N], const int32_t *lb, const PinTab &tab, uint32_t tt,
                                               const int32_t *__restrict__ D, int32_t Lw, int32_t *__restrict__ gout,
                                               int32_t q, bool from_start = true, int32_t tend = kEOW,
                                               int32_t cap = 0) {
    LaneResult r{0, 0, 0, 0};
    // a chunk holds at most cap entries (its pins' transitions): a write past them
    // would be a fault of the library's bound, so it is recorded instead of made
    int32_t wcap = 0;
    bool over = false;
    auto put = [&](int32_t k, int32_t v) {
        if (!kChunk || k <= wcap) gout[k] = v;
        else over = true;
    };
    auto get = [&](int32_t k) { return gout[k]; };   // this lane's own words

    uint32_t vbits = 0;
    int32_t t2first[N];
    if (!kChunk || from_start) {
        // initial values: pin index 1 when the waveform starts with -1.  The truth
        // table was re-indexed at create by the pin weights, so its index is the pin
        // values read as a binary number, first pin most significant.
        // every pin's first four words are loaded at once (the head, the first
        // transition and the word after it, whichever head the wave has); a wave
        // holds at least its head and EOW, so words 0 and 1 always exist
        int32_t x[N][4];
#pragma unroll
        for (int i = 0; i < N; ++i) {
            x[i][0] = __ldg(pin[i].w);
            x[i][1] = __ldg(pin[i].w + 1);
            x[i][2] = pin[i].len > 2 ? __ldg(pin[i].w + 2) : kEOW;
            x[i][3] = pin[i].len > 3 ? __ldg(pin[i].w + 3) : kEOW;
        }
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const bool one = x[i][0] == -1;
            pin[i].p = one ? 1u : 0u;
            vbits |= pin[i].p << (N - 1 - i);
            pin[i].nx = one ? x[i][2] : x[i][1];          // w[p + 1]
            t2first[i] = one ? x[i][3] : x[i][2];         // w[p + 2]
        }
    } else {
        // a cut: every pin's entry in effect is given, and entry p + 1 exists (at
        // worst the EOW)
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const uint32_t p = pin[i].p;
            vbits |= (p & 1u) << (N - 1 - i);
            pin[i].nx = __ldg(pin[i].w + p + 1);
            t2first[i] = p + 2 < pin[i].len ? __ldg(pin[i].w + p + 2) : kEOW;
        }
    }
    const int32_t y0 = (tt >> vbits) & 1;
    int32_t po = y0;        // index of the last output entry
    int32_t top = 0;        // O[po]
    int32_t second = 0;     // O[po - 1] (read only after a store, or after a cancel when kFull is false)
    int32_t t1acc = 0;      // signed sum of clipped entries: time at 1 before the final adjustment
    wcap = y0 + cap;
    if (!kChunk || from_start) {
        put(0, y0 ? -1 : 0);
        if (y0) put(1, 0);
    } else {
        gout -= y0;
    }

    bool lutbad = false;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        next_arrival<kFull, true>(pin[i].p, pin[i].a, pin[i].nx, pin[i].w, pin[i].len, pin[i].drf,
                                        pin[i].p & 1u, q, t2first[i]);
        if constexpr (N > 1) {
            const uint32_t o = kPins == kPinsNear ? (uint32_t)(pin[i].w - lb) : 0u;
            tab.hot[i * 32] = make_int2((int32_t)(o + pin[i].p), pin[i].nx);
            tab.end[i * 32] = o + pin[i].len;
        }
    }

    for (;;) {
        int32_t t = pin[0].a;
#pragma unroll
        for (int i = 1; i < N; ++i) t = min(t, pin[i].a);
        if (kChunk ? t >= tend : t == kEOW) break;

        // every pin arriving at t switches together (bit N-1-i = pin i); each one's
        // entry index moves on when the pin is advanced below
        uint32_t swb = 0;
#pragma unroll
        for (int i = 0; i < N; ++i) swb |= (pin[i].a == t ? 1u : 0u) << (N - 1 - i);
        vbits ^= swb;
        const int hb = 31 - __clz(swb);
        const int k = N - 1 - hb;                       // first switching pin
        const uint32_t more = swb & ~(1u << hb);        // any others (simultaneous switching)
        // output update as selects, not branches, so that the lanes stay together:
        // chg = the truth table changes the output; then the inertial filter either
        // cancels the last entry or stores a new one
        const int32_t y = (tt >> vbits) & 1;
        const int e_out = y ^ 1;
        // smallest finite conditional delay among the switching pins
        int32_t d = arc_delay<N>(D, vbits, k, e_out);
        for (uint32_t m = more; m; m &= m - 1u) d = min(d, arc_delay<N>(D, vbits, N - __ffs(m), e_out));
        bool chg = y != (po & 1);
        lutbad |= chg && d == kNoArc;
        // At q = 100 a missing arc only taints this lane's output, which the error
        // then discards: its entry (t + the no-arc value wraps below t) is never
        // cancelled, so the output index stays within the window's slot, and the
        // filter decision does not have to wait for the delay load.  Below 100 the
        // reject limit of such a delay is meaningless, so the change is dropped.
        if (!kFull) chg = chg && d != kNoArc;
        const int32_t to = (int32_t)((uint32_t)t + (uint32_t)d);   // used only when chg
        // inertial filter: at q = 100, to - top < d exactly when the last entry
        // has not matured (top > t); otherwise the reject limit decides
        const bool cancel = chg && (kFull ? top > t : to - top < reject_limit(d, q));
        const bool store = chg && !cancel;
        // time at 1: a cancelled entry gives back what it added, a stored one adds
        // its clipped time with the sign of its parity; both come to this
        const int32_t c = min(cancel ? top : to, Lw);
        t1acc += (chg ? 2 * (po & 1) - 1 : 0) * c;
        po += store ? 1 : (cancel ? -1 : 0);
        if (store) put(po, to);
        if (kFull) {
            const int32_t ntop = cancel ? second : (store ? to : top);
            second = store ? top : second;
            top = ntop;
        } else if (cancel) {
            top = second;
            second = po > 0 ? get(po - 1) : 0;           // the exposed entry may be pending too
        } else if (store) {
            second = top;
            top = to;
        }
        advance_pin<N, kFull, kPins>(pin, lb, tab, k, vbits, q);
        for (uint32_t mm = more; mm; mm &= mm - 1u)   // lowest bit first
            advance_pin<N, kFull, kPins>(pin, lb, tab, N - __ffs(mm), vbits, q);
    }
    if (lutbad) r.err = GATSPI_EBADLUT;
    if (kChunk && over) r.err = GATSPI_EINTERNAL;
    if constexpr (kChunk) {
        r.len = po;
        r.tc = po - y0;
        r.t1 = t1acc;
    } else {
        put(po + 1, kEOW);
        r.len = po + 2;
        r.tc = po - y0;
        r.t1 = t1acc + ((po & 1) ? Lw : 0);
    }
    return r;
}

template <int N, bool kFull, bool kChunk = false>
__device__ __forceinline__ LaneResult simulate_gate(const DevParams &P, int4 gd, Pin (&pins)[GATSPI_MAX_PINS],
                                                 const PinTab &tab, int32_t Lw, int32_t *gout, bool from_start = true,
                                                 int32_t tend = kEOW, int32_t cap = 0) {
    Pin pin[N];
#pragma unroll
    for (int i = 0; i < N; ++i) pin[i] = pins[i];
    const uint32_t tt = (uint32_t)gd.y >> 8;
    const long long dly = (long long)(uint32_t)gd.z | ((long long)gd.w << 32);
    if constexpr (N == 1) {
        return run_lane<N, kFull, kPinsOne, kChunk>(pin, pin[0].w, tab, tt, P.dly_data + dly, Lw, gout,
                                                    P.pulse_percent, from_start, tend, cap);
    } else {
        const int32_t *lb;
        if (table_fits<N>(pin, lb))
            return run_lane<N, kFull, kPinsNear, kChunk>(pin, lb, tab, tt, P.dly_data + dly, Lw, gout,
                                                         P.pulse_percent, from_start, tend, cap);
        return run_lane<N, kFull, kPinsFar, kChunk>(pin, lb, tab, tt, P.dly_data + dly, Lw, gout, P.pulse_percent,
                                                    from_start, tend, cap);
    }
}

template <bool kFull, bool kChunk = false>
__device__ __forceinline__ LaneResult dispatch(const DevParams &P, int4 gd, Pin (&pins)[GATSPI_MAX_PINS],
                                               const PinTab &tab, int32_t Lw, int32_t *gout, bool from_start = true,
                                               int32_t tend = kEOW, int32_t cap = 0) {
    switch (gd.y & 7) {
        case 1: return simulate_gate<1, kFull, kChunk>(P, gd, pins, tab, Lw, gout, from_start, tend, cap);
        case 2: return simulate_gate<2, kFull, kChunk>(P, gd, pins, tab, Lw, gout, from_start, tend, cap);
        case 3: return simulate_gate<3, kFull, kChunk>(P, gd, pins, tab, Lw, gout, from_start, tend, cap);
        default: return simulate_gate<4, kFull, kChunk>(P, gd, pins, tab, Lw, gout, from_start, tend, cap);
    }
}

// The N pins of a gate in window w from the window index: source waveform, length
// and wire delays; returns the window's output bound, 3 + sum over pins of
// (input length - 2).
template <int N>
__device__ __forceinline__ uint32_t load_pins(const DevParams &P, int4 sv, int4 dv, int w,
                                              Pin (&pins)[GATSPI_MAX_PINS]) {
    const int s4[GATSPI_MAX_PINS] = {sv.x, sv.y, sv.z, sv.w};
    const int d4[GATSPI_MAX_PINS] = {dv.x, dv.y, dv.z, dv.w};
    uint32_t bound = 3u - 2u * (uint32_t)N;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const long long src = s4[i];
        const uint32_t end = __ldg(P.wend + src * P.W + w);
        const uint32_t start = __ldg(P.wstart + src * P.W + w);
        pins[i].w = P.pool + __ldg(P.net_base + src) + start;
        pins[i].len = end - start;
        pins[i].drf = (uint32_t)d4[i];
        bound += end - start;
    }
    return bound;
}

// Inclusive warp scan.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += v;
    }
    return x;
}

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
    for (int w0 = 4 * lane; w0 - 4 * lane < W; w0 += 4 * 32) {
        long long part = 0;   // this lane's four windows
        if (w0 < W) {
            uint32_t even = 0, odd = 0;        // windows w0, w0 + 2 and w0 + 1, w0 + 3 in 16-bit halves
            uint32_t fix[4] = {0, 0, 0, 0};    // lengths beyond 255
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
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (w0 + u < W) part += b[u];
        }
        // the group of 32 windows of this step that holds lane's windows: lanes 8k .. 8k+7
        long long gsum = part;
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
        // the four groups' sums (lanes 0, 8, 16, 24) and their running offsets
        const long long g0 = __shfl_sync(0xffffffffu, gsum, 0), g1 = __shfl_sync(0xffffffffu, gsum, 8);
        const long long g2 = __shfl_sync(0xffffffffu, gsum, 16), g3 = __shfl_sync(0xffffffffu, gsum, 24);
        const int grp = (w0 - 4 * lane) >> 5;            // first group of this step
        if (lane < 4 && grp + lane < P.ngroups) {
            const long long before = lane == 0 ? 0 : lane == 1 ? g0 : lane == 2 ? g0 + g1 : g0 + g1 + g2;
            goff[grp + lane] = (uint32_t)(run + before);
        }
        run += g0 + g1 + g2 + g3;
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

// Windows cut into time chunks (16 windows or fewer, PATHPULSEPERCENT = 100): with
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
// earlier than the entry).  The simulation from T on therefore needs only the pins'
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
// kSeg: the instantiation that can split a gate's one window into segments.  Its
// code generation also happens to run windows that are not split 2-9 % faster at 2-16
// windows of 100 words or more per input, and 4-6 % slower on shorter ones, so the
// host picks the instantiation by the loaded inputs (DevParams::seg_kernel).
template <bool kSeg>
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
        res = dispatch<true, true>(P, gd, pins, tab, Lw, from_start ? slot : slot + off - 1, from_start, tend,
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
    if (p.chunks > 1 && p.pulse_percent == 100) {   // one warp per gate (or segment), heaviest first
        if (l.num_gates > 0) {
            const long long warps = (long long)l.num_gates + (p.seg_items ? kExtraSegments : 0);
            const unsigned blocks = (unsigned)((warps + kLevelWarps - 1) / kLevelWarps);
            level_order_kernel<<<1, kOrderThreads, 0, s>>>(p, l);
            if (p.seg_kernel)
                level_chunk_kernel<true><<<blocks, kLevelBlock, 0, s>>>(p, l);
            else
                level_chunk_kernel<false><<<blocks, kLevelBlock, 0, s>>>(p, l);
        }
        return cudaGetLastError();
    }
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
    if (e == cudaSuccess) e = cudaFuncSetAttribute(level_chunk_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout, 20);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(level_chunk_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout, 20);
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
