/*
 * gatspi.h -- C ABI of the GB300 gate-level re-simulator.
 *
 * The library re-simulates a levelised gate-level netlist, cycle window by cycle
 * window, from known primary / pseudo-primary input waveforms, as described in
 * "GATSPI: GPU-Accelerated Gate-Level Simulation for Power Improvement" (DAC '22):
 *   - Section 3, Fig. 3: the waveform array format;
 *   - Section 3, Fig. 4: truth-table lookup by summed pin weights and the
 *     conditional (SDF COND) delay table indexed by switching arc and the weights
 *     of the non-switching pins;
 *   - Section 3, Fig. 5: one device-resident waveform pool, levels simulated in
 *     order, each gate/cycle-window re-simulated by one GPU thread;
 *   - Section 3, Algorithm 1: per (gate, window) the merge of the fanin waveforms,
 *     interconnect inertial filtering, multiple-simultaneous-input-switching
 *     resolution, delay selection and gate inertial filtering with
 *     PATHPULSEPERCENT = 100.  The page sizes every output with a first counting
 *     pass; here an upper bound computed from the input lengths takes its place.
 *   - Section 3, the prose after Algorithm 1: other PATHPULSEPERCENT values come
 *     from editing the filter comparison.  With GATSPI_FLAG_PULSE_PERCENT and a
 *     percentage q, the delay d in both inertial comparisons (the interconnect
 *     pulse test and the gate filter) becomes the reject limit floor(d * q / 100):
 *     a fanin pulse narrower than the limit of its first edge's wire delay never
 *     reaches the pin, and the last output entry is cancelled when the new output
 *     time minus that entry is below the limit of the new event's delay.  Below
 *     100 several output events can be pending; a cancel exposes the entry before
 *     it.  q = 0 is transport delay: nothing is filtered, and only an output
 *     event scheduled before the last scheduled one replaces it.
 *
 * Conventions for every call:
 *   - every call returns a gatspi_status; nothing throws across this ABI, nothing
 *     exits, no kernel traps;
 *   - gatspi_last_error() returns a message about the calling thread's last failure;
 *   - host arrays passed in are copied during the call; the caller keeps ownership;
 *   - the waveform pool is borrowed: a device buffer the caller allocates (for
 *     example a torch int32 tensor) and keeps alive until gatspi_destroy;
 *   - asynchronous failures (pool overflow, missing delay arc, a stalled scan) are
 *     latched in a device status word and reported by the next
 *     synchronising call (gatspi_sync, gatspi_toggle_stats, gatspi_get_waveform,
 *     gatspi_export_offsets);
 *   - a context is used by one host thread at a time.
 *
 * Waveform format (Fig. 3): int32 timestamps of signal toggles; the index parity
 * is the logic value (even = 0, odd = 1); a waveform that starts at 1 begins with
 * -1, 0 and one that starts at 0 begins with 0; the array ends with
 * GATSPI_EOW = INT32_MAX.  Timestamps are relative to the start of their window.
 *
 * Windows (cycle parallelism, Section 1 and Section 4): the testbench is cut into
 * W independent windows; every window starts from the zero-delay steady state of
 * its input values and is simulated to completion (events scheduled past the
 * window's end are kept in the waveform and counted in TC; T1/T0 count only
 * [0, window_len)).  With few, long windows the library also splits each window at
 * times when the gate is quiet and simulates the stretches in parallel, which gives
 * exactly the window's result (see gatspi_simulate).
 */
#ifndef GATSPI_H
#define GATSPI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GATSPI_EOW 2147483647
#define GATSPI_NO_ARC 2147483647   /* delay-table entry of an arc that cannot occur */
#define GATSPI_MAX_PINS 4
#define GATSPI_MAX_WINDOWS 16384   /* cycle windows of one context */

typedef enum {
    GATSPI_OK = 0,
    GATSPI_EINVAL = 1,          /* invalid argument or netlist                       */
    GATSPI_ENOMEM = 2,          /* a device allocation failed                        */
    GATSPI_EPOOL_OVERFLOW = 3,  /* the waveform pool is too small for the outputs    */
    GATSPI_EBADWAVE = 4,        /* an input waveform breaks the Fig. 3 format        */
    GATSPI_ECUDA = 5,           /* a CUDA runtime call failed                        */
    GATSPI_ESTATE = 6,          /* call out of order (e.g. simulate before load)     */
    GATSPI_EBADLUT = 7,         /* every switching arc of an output change is NO_ARC */
    GATSPI_ETIMEOUT = 8,        /* a device-side wait gave up (scan look-back)       */
    GATSPI_EINTERNAL = 9        /* a kernel found one of the library's own bounds
                                   broken (a library fault); the access was not made  */
} gatspi_status;

/* Where a buffer passed to gatspi_load_waveforms lives. */
enum { GATSPI_HOST = 0, GATSPI_DEVICE = 1 };

/* gatspi_config.flags */
#define GATSPI_FLAG_LEVEL_TIMING 0x1u  /* record CUDA events around every level kernel (no graph) */
#define GATSPI_FLAG_NO_GRAPH 0x2u      /* launch level kernels directly, no CUDA graph  */
#define GATSPI_FLAG_PULSE_PERCENT 0x4u /* apply pulse_percent (else PATHPULSEPERCENT = 100) */
#define GATSPI_FLAG_COMPACT 0x8u       /* pack every level to its exact size (see gatspi_simulate) */
#define GATSPI_FLAG_WHOLE_WINDOWS 0x10u /* never cut a window into time chunks (see gatspi_simulate) */
#define GATSPI_FLAG_CUT_WINDOWS 0x20u   /* cut windows into time chunks whatever their length (one
                                           window: heavy gates also split into segments) */

/*
 * Levelised netlist (all host arrays, copied by gatspi_create).
 *
 * Nets 0 .. num_inputs-1 are primary / pseudo-primary inputs; gate g drives net
 * num_inputs + g.  Gates are numbered in level order: level l holds gates
 * [level_offsets[l], level_offsets[l+1]); every fanin of a gate in level l is an
 * input or a gate of a lower level.
 *
 *   gate_type[G]          cell type of every gate, 0 .. num_types-1
 *   type_num_pins[T]      pins of every type, 1 .. GATSPI_MAX_PINS
 *   type_tt_off[T], tt_data[tt_len]
 *                         truth table of type t: tt_data[type_tt_off[t] + k], k < 2^n,
 *                         entries 0/1; k is the sum of pin_weight over the pins at 1
 *                         (Fig. 4: NAND2 with A = 2^1, B = 2^0 has Y = [1, 1, 1, 0])
 *   fanin_off[G+1], fanin_net[E], pin_weight[E], wire_rise[E], wire_fall[E]
 *                         pins of gate g are edges fanin_off[g] .. fanin_off[g+1]-1 in pin
 *                         order: driving net, truth-table weight (the weights of one gate
 *                         are the distinct powers 2^0 .. 2^(n-1)), interconnect rise / fall
 *                         delay (0 .. 65535)
 *   gate_dly_off[G], dly_data[dly_len]
 *                         per-instance conditional delay table of gate g at
 *                         dly_data[gate_dly_off[g]], laid out [4n][2^(n-1)] int32:
 *                         row = 4*pin + 2*e_in + e_out (RISE = 0, FALL = 1; e_in is the
 *                         switching pin's new edge, e_out the output's), column = the
 *                         values of the other pins, in pin order with the first one most
 *                         significant (Fig. 4: for AOI21 B->Y, A1 = 2^1 and A2 = 2^0);
 *                         entries are 0 .. 2^24-1 or GATSPI_NO_ARC.  Instances may share
 *                         a table.
 */
typedef struct {
    int32_t num_inputs;
    int32_t num_gates;
    int32_t num_levels;
    int32_t num_types;
    const int32_t *level_offsets;
    const int32_t *gate_type;
    const int32_t *type_num_pins;
    const int32_t *type_tt_off;
    int64_t tt_len;
    const uint8_t *tt_data;
    const int32_t *fanin_off;
    const int32_t *fanin_net;
    const int32_t *pin_weight;
    const int32_t *wire_rise;
    const int32_t *wire_fall;
    const int64_t *gate_dly_off;
    int64_t dly_len;
    const int32_t *dly_data;
} gatspi_netlist;

/*
 * Run configuration.
 *   num_windows   W independent cycle windows, 1 .. GATSPI_MAX_WINDOWS
 *   window_len    host array [W] of window lengths in time units (1 .. 2^30)
 *   flags         GATSPI_FLAG_*
 *   pulse_percent PATHPULSEPERCENT q, 0 .. 100, read only with
 *                 GATSPI_FLAG_PULSE_PERCENT (a zeroed config means 100).
 */
typedef struct {
    int32_t num_windows;
    const int64_t *window_len;
    uint32_t flags;
    int32_t pulse_percent;
} gatspi_config;

typedef struct gatspi_ctx gatspi_ctx;

/*
 * Device views of the simulation state (valid until gatspi_destroy).
 *
 * The pool holds first the input waveforms as loaded, then the gates' outputs level
 * by level; every net has one region.  A gate's region is sized by upper bounds of
 * its windows' outputs (see gatspi_simulate); its windows are stored in rank order
 * (windows ordered by bound, largest first; window order beyond 1024 windows), each
 * in a slot as long as its bound, so
 * a gap may follow every window.  Waveform k = (net, w), k = net * W + w,
 * is pool[net_base[net] + wstart[k] .. net_base[net] + wend[k]) (EOW included).  The
 * layout depends only on the inputs: every run gives the same pool.
 */
typedef struct {
    const int32_t *pool;
    int64_t pool_words;            /* capacity                                       */
    int64_t pool_used;             /* words written by the last load + simulate      */
    const int64_t *net_base;       /* [num_nets] first pool word of the net's region */
    const uint32_t *wstart;        /* [num_nets * num_windows] relative to net_base  */
    const uint32_t *wend;          /* [num_nets * num_windows] relative to net_base  */
    const unsigned long long *tc;  /* [num_gates] output toggles summed over windows */
    const unsigned long long *t1;  /* [num_gates] time at 1 summed over windows      */
    int32_t num_nets;
    int32_t num_windows;
} gatspi_views;

/*
 * Create a simulator for one netlist and window configuration.
 *   d_pool      device int32 buffer of pool_words words, 16-byte aligned, borrowed
 *   pool_words  capacity, a multiple of 4 words
 * Validates the netlist (EINVAL with a message naming the first offending gate),
 * copies it to the device and allocates the context's own device arrays (ENOMEM).
 * Fig. 5 / Algorithm 1 inputs.
 */
gatspi_status gatspi_create(const gatspi_netlist *nl, const gatspi_config *cfg, int32_t *d_pool,
                            size_t pool_words, gatspi_ctx **out);

/*
 * Load the input waveforms of every (input, window).
 *   off    int64 [num_inputs * W + 1] offsets into words, input-major and window-minor,
 *          non-decreasing (CSR)
 *   words  int32 [nwords] waveform words (Fig. 3 format)
 *   where  GATSPI_HOST (pageable or pinned host memory) or GATSPI_DEVICE
 * Copies the words to the front of the pool on `stream`, checks the format of every
 * waveform on the device (timestamps after the head strictly increasing, 1 .. 2^30)
 * and builds the window index.  Synchronises `stream` before returning: EBADWAVE
 * names the first malformed (input, window); EPOOL_OVERFLOW if nwords exceeds the
 * pool; EINVAL if the longest path could carry a timestamp to EOW.
 */
gatspi_status gatspi_load_waveforms(gatspi_ctx *ctx, const int64_t *off, const int32_t *words, size_t nwords,
                                    int where, void *stream);

/*
 * Load the inputs from whole-testbench waveforms and cut them into the windows on
 * the device.  GATSPI re-simulates cycle windows from known input waveforms
 * (Sections 1 and 4) and restructures its inputs into that per-window format on the
 * host, most of its set-up time (Section 5, Table 5); this call does it on the GPU.
 *   off    int64 [num_inputs + 1] offsets into words (off[0] = 0, off[num_inputs] =
 *          nwords, non-decreasing)
 *   words  int32 [nwords]: one Fig. 3 waveform per input with times from the start
 *          of the testbench (head [0] or [-1, 0], times strictly increasing from 1,
 *          GATSPI_EOW last)
 *   where  GATSPI_HOST (pageable or pinned) or GATSPI_DEVICE (off and words both in
 *          device memory, outside the first nwords + 3 * W * num_inputs words of the
 *          pool)
 * Window w covers [S_w, S_w + window_len[w]) of the testbench, S_w being the sum of
 * the lengths of the windows before it.  Its waveform starts at the input's value at
 * S_w (a transition exactly at S_w folds into it) and holds the transitions inside
 * the window minus S_w; transitions at or after the end of the last window belong
 * to no window.  The windows of input p go to a region of the pool bounded by its
 * transitions + 3 * W words (gaps between regions, as for gate outputs); a host
 * testbench is first staged at the far end of the pool.  Synchronises `stream`
 * before returning: EBADWAVE names the first malformed input; EPOOL_OVERFLOW when
 * nwords + 3 * W * num_inputs words (plus nwords staged, from the host) exceed the
 * pool; EINVAL for bad offsets or when the longest window plus the longest path
 * could carry a timestamp to EOW.  Replaces gatspi_load_waveforms for the run.
 */
gatspi_status gatspi_load_testbench(gatspi_ctx *ctx, const int64_t *off, const int32_t *words, size_t nwords,
                                    int where, void *stream);

/*
 * Re-simulate every level, in order, on `stream` (a cudaStream_t; NULL = legacy
 * default stream).  Asynchronous: returns after enqueueing.  Clears TC/T1 and the
 * device status first.  Per level three kernels run, in place of the page's
 * counting and writing passes.  The first plans the level: it bounds every (gate,
 * window) output (an output window holds at most 3 + the sum over its pins of (input
 * length - 2) words, since each stored toggle takes an event-loop iteration and each
 * iteration consumes an input transition) and ranks each gate's windows by bound so
 * that a warp gets 32 windows of similar work (up to 1024 windows; beyond, the windows
 * are short and are taken in window order).  The second scans the gates' bound sums
 * into pool offsets.  The third runs Algorithm 1 for every (gate, window) of the level
 * and stores the output waveforms, the window index and TC/T1 per gate.  Windows cut
 * into time chunks (below) add a kernel that orders the gates, packing two more.  The
 * level sequence is captured once into a CUDA graph and replayed by later calls,
 * unless GATSPI_FLAG_NO_GRAPH or GATSPI_FLAG_LEVEL_TIMING is set (then the level
 * kernels are launched directly on `stream`).
 */
gatspi_status gatspi_simulate(gatspi_ctx *ctx, void *stream);

/*
 * (continuation of gatspi_simulate) With GATSPI_FLAG_COMPACT every level is simulated
 * into bound-sized regions placed down from the top of the pool, then a scan of the
 * exact sizes and a copy pack it to exact size at the front, windows back to back,
 * before the next level is planned: the pool then holds the waveforms themselves
 * (exact sizes, as the page's counting pass gives, Section 3, Fig. 5) plus room for
 * one level's bound-sized regions, at the cost of copying every level once.
 * gatspi_views.pool_used then reports the most words any level needed (the packed
 * front plus its bound-sized regions); EPOOL_OVERFLOW when that exceeds the pool.
 *
 * After each level's simulation kernel, that
 * level's TC and T1 are copied to pinned host memory on a side stream while the
 * later levels run (the page dumps its statistics asynchronously as well, Section 3);
 * `stream` waits for the copies at the end, so the statistics are on the host once
 * the stream has finished and gatspi_toggle_stats reads no device memory.
 *
 * With 16 windows or fewer, at any PATHPULSEPERCENT, when the windows are long (the
 * last load averaged 32 words or more per (input, window); always with
 * GATSPI_FLAG_CUT_WINDOWS, never with GATSPI_FLAG_WHOLE_WINDOWS; the two flags
 * exclude each other: EINVAL at create), a lane would run its gate through a long
 * window alone, so each gate takes one warp and each of its windows 32 / W lanes,
 * every lane simulating the window between two cuts: times at which none of the
 * gate's pins has a transition within its largest wire delay after, nor within that
 * wire delay plus its largest gate delay before.  At such a time every pin's entry
 * in effect is its last transition, no pulse spans it, and no output entry made
 * before it can be cancelled by an event after it (below 100 %, every entry an
 * event after it makes lies more than that delay's reject limit later), so the
 * stretches simulate independently and give exactly the whole window's waveform,
 * toggles and time at 1 (the page runs windows, not stretches of one, in parallel:
 * Section 4, cycle parallelism).  A lane that finds no cut near its share leaves
 * its stretch to the lane before.  The warp then moves the stretches' entries
 * together inside the window's slot.  Each level's gates are taken heaviest first.
 * With one window of 4096 words or more per input (or with
 * GATSPI_FLAG_CUT_WINDOWS), a gate whose work exceeds its level's share per warp
 * the GPU holds takes up to 8 warps, each a segment of the window between two such
 * times, and the last warp to finish moves the segments together.  A load that
 * changes whether the windows are long makes the next simulate capture its graph
 * again.
 */

/*
 * Wait for the last simulate / load and report a latched device error.  The page's
 * host waits for the level loop before dumping the statistics (Section 3, Fig. 5);
 * this is that wait, plus the report of the device status word.
 */
gatspi_status gatspi_sync(gatspi_ctx *ctx);

/*
 * Lanes the next gatspi_simulate gives each window: 32 / num_windows when it cuts the
 * windows into time chunks (see gatspi_simulate), else 1; 0 for a NULL ctx.  Decided
 * by the flags, the window count and the last load.  The page has no counterpart: it
 * runs windows, not stretches of one window, in parallel (Section 4, cycle
 * parallelism).
 */
int32_t gatspi_lanes_per_window(const gatspi_ctx *ctx);

/*
 * SAIF-style toggle statistics per gate, summed over windows (host arrays [G]; any
 * may be NULL): tc = output toggles, t1 = time at 1, t0 = time at 0, with
 * t0 + t1 = sum of window_len -- the per-net activity the page's re-simulation
 * produces for power analysis (Section 3, Fig. 2).  Synchronises first.
 */
gatspi_status gatspi_toggle_stats(gatspi_ctx *ctx, int64_t *tc, int64_t *t0, int64_t *t1);

/*
 * The same statistics without a copy (the page dumps its statistics while the GPU
 * works, Section 3): *tc and *t1 point at the library's pinned host
 * copies (uint64 [num_gates], gate order) that simulate filled level by level, valid
 * until the next simulate or destroy; t0 = sum of window_len - t1 (*window_sum).
 * Synchronises first.  GATSPI_ESTATE before the first simulate; NULL pointers for a
 * netlist without gates.
 */
gatspi_status gatspi_toggle_stats_host(gatspi_ctx *ctx, const uint64_t **tc, const uint64_t **t1,
                                       int64_t *window_sum);

/*
 * The same statistics for the inputs, from the loaded windows (host arrays
 * [num_inputs]; any may be NULL): computed on the device by every load.  A SAIF
 * file covers every net, inputs included (Section 3, Fig. 2).
 */
gatspi_status gatspi_input_stats(gatspi_ctx *ctx, int64_t *tc, int64_t *t0, int64_t *t1);

/*
 * Write the toggle statistics of every net (inputs, then gate outputs) as a SAIF 2.0
 * file, the output format the GATSPI page produces for power analysis (Section 3,
 * Fig. 2): (DURATION) = the sum of the window lengths; per net (T0) (T1) (TX 0)
 * (TC) (IG 0), summed over the windows.
 *   path       file to write (overwritten)
 *   design     design / top instance name (NULL: "top")
 *   timescale  the time unit of the waveforms, e.g. "1 ps" (NULL: "1 ps")
 *   net_names  NULL (nets named n<index>) or num_inputs + num_gates C strings;
 *              characters other than letters, digits and '_' are escaped with '\'
 * Synchronises first.  EINVAL if the file cannot be written.
 */
gatspi_status gatspi_write_saif(gatspi_ctx *ctx, const char *path, const char *design, const char *timescale,
                                const char *const *net_names);

/*
 * Copy one (net, window) waveform to host memory (the page spot-checks waveforms
 * against a reference simulator's, Section 4).  *len receives its length in
 * words (EOW included) even when it exceeds cap, in which case nothing is copied
 * and EINVAL is returned.  Synchronises first.
 */
gatspi_status gatspi_get_waveform(gatspi_ctx *ctx, int32_t net, int32_t window, int32_t *buf, size_t cap,
                                  size_t *len);

/*
 * Write the pool position and length (EOW included) of every (net, window)
 * waveform, net-major and window-minor, to host memory (the offsets into the Fig. 5
 * waveform pool that the page's scan produces): waveform k = net * W + w
 * occupies pool[start[k] .. start[k] + len[k]) (n = num_nets * W entries; either
 * array may be NULL).  Synchronises first.
 */
gatspi_status gatspi_export_offsets(gatspi_ctx *ctx, int64_t *start, int32_t *len, size_t n);

/*
 * Export the waveforms of selected windows for every net, as CSR in host memory:
 *   windows  host int32 [nsel], each 0 .. W-1 (any order, repeats allowed)
 *   off      host int64 [num_nets * nsel + 1]: waveform (net, windows[s]) occupies
 *            words[off[net * nsel + s] .. off[net * nsel + s + 1])
 *   words    host int32 [cap], or NULL to query the size (off is still filled)
 * Windows are independent re-simulations (cycle parallelism, Sections 1 and 4), so
 * this is the natural unit to check or dump a slice of a large run.  Allocates and
 * frees device scratch; synchronises.
 * EINVAL if cap < off[num_nets * nsel] (off is filled either way).
 */
gatspi_status gatspi_export_windows(gatspi_ctx *ctx, const int32_t *windows, int32_t nsel, int64_t *off,
                                    int32_t *words, size_t cap);

/*
 * Digest of every net's waveforms, for checking a run against a reference without
 * moving its waveforms (the page checks its results by comparing the SAIF files and
 * spot-checking waveforms, Section 4).  digest[k] (host uint64 [num_nets]) is the
 * 64-bit FNV-1a hash (offset basis 14695981039346656037, prime 1099511628211, one
 * byte at a time) of the little-endian bytes of net (net_begin + k)'s waveforms
 * concatenated in window order, each window's Fig. 3 array with its head and its
 * GATSPI_EOW; words[k] (host int64 [num_nets], or NULL) the number of words hashed.
 * Inputs need a load, gates a simulate (GATSPI_ESTATE otherwise).  Allocates and
 * frees device scratch; synchronises first.  EINVAL when the range leaves
 * 0 .. num_inputs + num_gates.
 */
gatspi_status gatspi_net_digests(gatspi_ctx *ctx, int64_t net_begin, int64_t num_nets, uint64_t *digest,
                                 int64_t *words);

/* Device views of the pool, window index and statistics (see gatspi_views): the
 * Fig. 5 pool and offsets for callers that keep working on the device. */
gatspi_status gatspi_device_views(gatspi_ctx *ctx, gatspi_views *out);

/*
 * Per-level kernel times in milliseconds of the last simulate (the page profiles the
 * kernel level by level, Section 5, Table 6), which must have run
 * with GATSPI_FLAG_LEVEL_TIMING: sim_ms[l] for the simulation kernel of level l,
 * bounds_ms[l] for the kernels that plan and place its output regions (either may
 * be NULL; n = num_levels).  Synchronises first.  GATSPI_ESTATE when the last
 * simulate was not timed.
 */
gatspi_status gatspi_level_times(gatspi_ctx *ctx, float *sim_ms, float *bounds_ms, int32_t n);

/*
 * Switch GATSPI_FLAG_LEVEL_TIMING (per-level times, Section 5, Table 6) on (on != 0)
 * or off for the following simulate calls.  Timed runs launch the levels directly with a CUDA event between every two
 * kernels; untimed runs replay the captured level graph (unless
 * GATSPI_FLAG_NO_GRAPH).  GATSPI_EINVAL when ctx is NULL.
 */
gatspi_status gatspi_set_level_timing(gatspi_ctx *ctx, int32_t on);

/*
 * Buffers of one logic level for gatspi_simulate_level_static (all device memory,
 * owned by the caller).  The layouts are the library's own:
 *   gate_desc   int32 [12 * num_gates of the netlist], 16-byte aligned; gate g's
 *               record is the 12 words at 12 * g:
 *               {0, n | truth-table bits << 8, low and high 32 bits of the
 *               delay-table offset}, {the net driving pin 0, 1, 2, 3},
 *               {wire rise | wire fall << 16 of pin 0, 1, 2, 3}, pins past n being 0;
 *               truth-table bit v is the output when the pin values, read as a
 *               binary number with the first pin most significant, equal v (the
 *               page's table re-indexed by pin weight)
 *   dly_data    the delay tables of gatspi_netlist laid out for the kernel: the entry
 *               of row 4*i + 2*e_in + e_out and column c of gate g's table sits at
 *               dly_data[gate_dly_off[g] + (((2*i + e_out) << n) | v)], v being all n
 *               pin values after the switch (pin j at bit n-1-j, so pin i's bit gives
 *               e_in and the others give c); the same size as the Fig. 4 table
 *   window_len  int32 [num_windows]
 *   pool, net_base, wstart, wend, wlen8
 *               the waveform store of gatspi_views (pool_words = capacity); the
 *               sources of this level must already be in it, well formed (the regular
 *               path checks every input when it loads it; from a malformed source this
 *               call writes unspecified words, but reads and writes stay inside the
 *               source's window and the output's slot); wlen8 (uint8, 4-byte
 *               aligned) holds min(length, 255) of waveform (net, w) at
 *               net * W4 + w, W4 = num_windows rounded up to a multiple of 4
 *   perm, goff  the level's plan (scratch, written then read by this call):
 *               uint16 [num_gates * num_windows] (unused beyond 1024 windows, which
 *               are taken in window order) and uint32 [num_gates * (ceil(W / 32) + 1)]
 *   tc, t1      per-gate toggle count and time at 1, accumulated (not cleared)
 *   level_base  int64 [2]: [0] = first pool word of this level's outputs (read),
 *               [1] = one past its last word (written)
 *   flags, pulse_percent
 *               GATSPI_FLAG_PULSE_PERCENT selects pulse_percent as in gatspi_config
 *               (other flags are ignored); zeroed fields mean PATHPULSEPERCENT = 100
 */
typedef struct {
    const int32_t *gate_desc;
    const int32_t *dly_data;
    const int32_t *window_len;
    int32_t *pool;
    int64_t pool_words;
    int64_t *net_base;
    uint32_t *wstart;
    uint32_t *wend;
    uint8_t *wlen8;
    uint16_t *perm;
    uint32_t *goff;
    unsigned long long *tc;
    unsigned long long *t1;
    int64_t *level_base;
    int32_t num_inputs;
    int32_t num_windows;
    int32_t gate_begin;   /* first gate of the level */
    int32_t num_gates;    /* gates in the level */
    uint32_t flags;
    int32_t pulse_percent;
} gatspi_level_args;

/*
 * Re-simulate one logic level without allocating any memory.  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate device
 * memory -- code running under a framework that owns all of the device memory
 * through its own allocator, or code that must not allocate once it has started.
 * The caller passes every input and output buffer (gatspi_level_args); the only
 * scratch, the look-back flags of the output-region scan, its tile ticket and the
 * status word, lives in a file-scope device array of 8192 tile flags plus 32
 * bytes (about 64 KiB) that every GPU which loads the library holds until the
 * process exits.
 *
 *   - No cudaMalloc, cudaFree or allocating library call is made.
 *   - A level may have at most 8192 x 1024 = 8388608 gates (one look-back flag per
 *     1024); a larger level returns GATSPI_EINVAL before anything runs.  The caller
 *     also makes sure the gates exist.
 *   - The first call on a device looks up the device address of the scratch array
 *     (with that device current); make that first call before any stream capture.
 *   - Every call shares the one array and clears the part it uses before its
 *     kernel runs; calls that overlap on the GPU (other streams, other threads)
 *     race on it and must be serialised by the caller.
 *   - Synchronous: enqueues on `stream`, waits for it, and returns the kernel's
 *     status (GATSPI_EPOOL_OVERFLOW, GATSPI_EBADLUT, ...).
 *   - Every window runs whole, one lane each: the time-chunk form of few long
 *     windows (GATSPI_FLAG_CUT_WINDOWS) needs per-level scratch that this call
 *     does not have.  That form gives the same words, so only the speed differs.
 * Results are identical to the level kernels gatspi_simulate runs.
 */
gatspi_status gatspi_simulate_level_static(const gatspi_level_args *args, void *stream);

/*
 * SDF -> delay tables.  GATSPI translates SDF IOPATH and COND statements into the
 * Fig. 4 arrays with no calibration run (Section 3, Fig. 4); this is that translator,
 * on the host.  The design names what the SDF text refers to:
 *   type_names[T]       CELLTYPE of every cell type
 *   type_num_pins[T]    its input pins (1 .. GATSPI_MAX_PINS)
 *   pin_names[]         the input pin names of every type in pin order, types one
 *                       after another
 *   out_pin             the output pin name of every cell (e.g. "Y")
 *   gate_type[G], instance_names[G]
 *                       every gate's type and SDF instance name (unique)
 *   fanin_off[G+1]      gate g's fanin edges fanin_off[g] .. fanin_off[g+1]-1, in pin
 *                       order (for INTERCONNECT destinations inst/pin)
 *   gate_dly_off[G], dly_len
 *                       where gate g's [4n][2^(n-1)] table goes in dly_data
 *   unit_fs             the simulator's time unit in femtoseconds (1000 = 1 ps)
 * Writes dly_data[dly_len] (every gate's table: rows 4*pin + 2*e_in + e_out, RISE = 0,
 * FALL = 1; columns the other pins' values, first pin most significant; entries no
 * statement sets are GATSPI_NO_ARC; words outside every table 0) and, if not NULL,
 * wire_rise/wire_fall[fanin_off[G]] (0 where no INTERCONNECT names the pin).
 * Rules: (posedge P) / (negedge P) / bare P select the input edge(s); the first
 * value is the output-rise delay and the second the output-fall delay (one value
 * serves both); () is no arc; min:typ:max gives typ; an unconditional IOPATH sets
 * every column and a COND IOPATH the columns where its condition holds for the other
 * pins, over the unconditional one (the last COND written wins where several hold);
 * values are converted from the TIMESCALE (1 ns when absent) exactly and rounded to
 * the nearest unit, halves up.  Conditions: Verilog == === != !== ! ~ & | ^ && ||,
 * parentheses, 0, 1, 1'b0, 1'b1, 'b0, 'b1.  Only ABSOLUTE delays are read.
 * EINVAL (message with the offending item) on malformed text, an unknown instance or
 * pin, a CELLTYPE that does not match, a condition on the switching pin or a negative
 * delay; the outputs are then unspecified.  Host memory only; no GPU is used.
 */
typedef struct {
    int32_t num_types;
    const char *const *type_names;
    const int32_t *type_num_pins;
    const char *const *pin_names;
    const char *out_pin;
    int32_t num_gates;
    const int32_t *gate_type;
    const char *const *instance_names;
    const int32_t *fanin_off;
    const int64_t *gate_dly_off;
    int64_t dly_len;
    int64_t unit_fs;
} gatspi_sdf_design;

gatspi_status gatspi_sdf_annotate(const gatspi_sdf_design *design, const char *text, size_t len, int32_t *dly_data,
                                  int32_t *wire_rise, int32_t *wire_fall);

/*
 * Failure injection for the bounded device waits (the page has no counterpart).  The
 * only place a kernel waits for another block is the decoupled look-back of the
 * output-region scan (see gatspi_simulate); every such wait gives up after a time
 * limit with GATSPI_ETIMEOUT instead of hanging.  This call arms the next
 * gatspi_simulate (launched directly, not from the graph) to stall the scan of
 * `level`: its first tile is never taken, so the tiles after it wait for a flag that
 * nothing sets, give up after wait_ns (1 us .. 10 s) and latch GATSPI_ETIMEOUT; the
 * following kernels see the status and write nothing, and the context stays usable
 * (the simulate after it runs normally).  The level must have more than 1024 gates
 * (two tiles); EINVAL otherwise.
 */
gatspi_status gatspi_inject_scan_stall(gatspi_ctx *ctx, int32_t level, int64_t wait_ns);

/* Release the context's device arrays (not the borrowed pool).  NULL is allowed.
 * The page has no counterpart (a library lifetime call). */
void gatspi_destroy(gatspi_ctx *ctx);

/* Message about the calling thread's last failed call ("" if none).  The page has
 * no counterpart (error reporting of this ABI). */
const char *gatspi_last_error(void);

/* Name of a status code.  The page has no counterpart. */
const char *gatspi_status_name(gatspi_status s);

#ifdef __cplusplus
}
#endif

#endif /* GATSPI_H */
