// The per-(gate, window) machinery of the level kernels (level_kernel.cu and
// chunk_kernel.cu): GATSPI Algorithm 1 for one lane -- the fanin waveforms merged with
// interconnect inertial filtering, simultaneous switching resolved, the truth table
// looked up by the pins' values, the conditional delay picked (row = switching pin
// and edges, column = the other pins' values), the gate's inertial filter applied --
// and the helpers around it (status word, pin loading, warp scans).  Included by each
// kernel file into its own anonymous namespace.
#pragma once

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
// clipped entries, without the final adjustment.  The entry in effect at the cut
// (index y0) lies before the cut and is never cancelled: any event after the cut
// makes an entry more than its delay's reject limit after it.  The chunk does not
// hold that entry and stands in time 0 for it, which gives the same filter decisions
// (it too lies at least that far before every later entry).
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
            // the exposed entry may be pending too; below a chunk's first entry lies
            // the entry in effect at its cut, which another lane wrote (stand-in 0)
            second = po > (kChunk && !from_start ? y0 + 1 : 0) ? get(po - 1) : 0;
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

}  // namespace

}  // namespace gatspi
