/*
 * TEST INFRASTRUCTURE ONLY: the CPU oracle of the gate-level re-simulator.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load it.
 * It shares no code with the CUDA library and is deliberately plain and slow.
 *
 * What it computes (GATSPI: GPU-Accelerated Gate-Level Simulation for Power
 * Improvement, Section 3, Algorithm 1 and the prose after it; Fig. 3 for the
 * waveform format; Fig. 4 for the truth-table and conditional-delay lookups):
 * every gate, in logic-level order, is re-simulated independently in every cycle
 * window.  For one (gate, window):
 *
 *   init: each pin's index starts at 1 if its waveform
 *     starts with -1 (initial value 1), else at 0; the truth-table index is the
 *     sum of the weights of the pins at 1; the output starts as [0] or [-1, 0].
 *   loop, until no pin has a next transition:
 *     - next arrival: for every pin, skip every pulse narrower than the wire delay
 *       of its first edge (the delay is the fall delay when the pin is at 1, the
 *       rise delay when at 0); the pin's next arrival is its next timestamp plus
 *       that delay; t is the earliest arrival.
 *     - switching: every pin whose arrival equals t switches (multiple
 *       simultaneous input switching is resolved together); the truth table
 *       gives the new output value y.
 *     - output: if y differs from the value of the last output entry, the
 *       gate delay d is looked up in the conditional delay table and t_o = t + d;
 *       if t_o - O[last] < d the last entry has not matured yet and is cancelled
 *       (inertial filter, PATHPULSEPERCENT = 100), otherwise t_o is appended.
 *   finish: EOW is appended.  TC = number of output toggles; T1 = time at 1
 *   within [0, window length).
 *
 * Readings where the extracted page is silent or garbled (variable names of
 * Algorithm 1 are lost in the extraction):
 *   - the interconnect pulse skip repeats until the next pulse is wide enough
 *     (a loop, not a single test), and the comparison is strict (< 0);
 *   - the right-hand side of the gate's inertial test is the selected gate delay d;
 *   - when several pins switch together and the output changes, d is the
 *     smallest finite delay among the switching pins' arcs; if every arc is
 *     INT32_MAX the run fails with ORACLE_EBADLUT;
 *   - delay row = 4*pin + 2*e_in + e_out with RISE = 0, FALL = 1 (e_in is the
 *     switching pin's new edge, e_out the output's); column = the values (after
 *     the switch) of the other pins in pin order, first pin most significant;
 *   - each window starts from the zero-delay steady state of its input values.
 *
 * Other pulse limits.  The page fixes PATHPULSEPERCENT at 100 and notes that other
 * values come from editing the inertial comparison.  With a percentage q (0..100)
 * the delay in both comparisons -- the interconnect pulse test and the gate's
 * filter -- is replaced by its reject limit r = floor(d * q / 100): a pulse on a
 * fanin whose width is below r of its first edge's wire delay is skipped, and the
 * last output entry is cancelled when t_o - O[last] < r.  q = 100 gives the rules
 * above.  Below 100 several output entries can be pending at once; a cancel then
 * exposes the entry before it, which a later event may cancel in turn.  q = 0 is
 * transport delay: no pulse is filtered, and only an output event scheduled before
 * the last scheduled one replaces it.
 *
 * Study variant (off unless oracle_set_literal_skip(1) is called): the interconnect
 * pulse test written in Algorithm 1 as a single test, taken literally -- each pin
 * skips at most one narrow pulse per iteration of the event loop, so the first edge
 * of a second narrow pulse right behind it can be taken in that iteration.  The
 * reading above (skip until the next pulse is wide enough) is what every other
 * part of this project computes.
 */
#include <pthread.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "oracle_abi.h"

#define EOW 2147483647LL
#define NO_ARC 2147483647LL
#define MAXP 8
#define RISE 0
#define FALL 1

/* study variant of the interconnect pulse test (see the header); set before a run */
static int g_literal_skip = 0;
void oracle_set_literal_skip(int on) { g_literal_skip = on != 0; }

/* reject limit of a delay d at PATHPULSEPERCENT q */
static int64_t reject_limit(int64_t d, int32_t q) { return d * q / 100; }

typedef struct {
    int32_t *w;
    int64_t len, cap;
} wbuf;

static int wbuf_reserve(wbuf *b, int64_t need) {
    if (need <= b->cap) return 0;
    int64_t cap = b->cap ? b->cap : 64;
    while (cap < need) cap *= 2;
    int32_t *nw = (int32_t *)realloc(b->w, (size_t)cap * sizeof(int32_t));
    if (!nw) return -1;
    b->w = nw;
    b->cap = cap;
    return 0;
}

/* One gate in one window: Algorithm 1.  Win[i] is pin i's input waveform.
 * The output waveform is written to O (O->len set); *tc and *t1 receive the
 * window's toggle count and time at 1. */
static int simulate_task(int n, const int32_t *const *Win, const int32_t *wire_rise,
                         const int32_t *wire_fall, const int32_t *weight, const uint8_t *T,
                         const int32_t *D, int64_t Lw, int32_t q, wbuf *O, int64_t *tc, int64_t *t1) {
    int64_t p[MAXP];
    int64_t a[MAXP];
    int sw[MAXP];
    const int ncol = 1 << (n - 1);

    /* init: pin indices, truth-table index and initial output value */
    int64_t idx = 0;
    for (int i = 0; i < n; ++i) {
        p[i] = (Win[i][0] == -1) ? 1 : 0;
        idx += (p[i] % 2) * weight[i];
    }
    const int y0 = T[idx];

    /* init: output starts as [0] or [-1, 0]; po indexes its last entry */
    if (wbuf_reserve(O, 4)) return ORACLE_ENOMEM;
    int64_t po;
    if (y0 == 0) {
        O->w[0] = 0;
        po = 0;
    } else {
        O->w[0] = -1;
        O->w[1] = 0;
        po = 1;
    }

    /* event loop */
    for (;;) {
        int64_t t = EOW;
        for (int i = 0; i < n; ++i) {
            int64_t d;
            for (int skipped = 0;; ) {
                d = (p[i] % 2) ? wire_fall[i] : wire_rise[i]; /* edge leaving the current value */
                if (Win[i][p[i] + 1] == EOW) break;
                if (g_literal_skip && skipped) break;          /* study variant: one test only */
                /* interconnect inertial filter: a pulse narrower than the reject limit
                 * of d never reaches the pin (the limit is d itself at q = 100) */
                if ((int64_t)Win[i][p[i] + 2] - reject_limit(d, q) - (int64_t)Win[i][p[i] + 1] < 0) {
                    p[i] += 2;
                    skipped = 1;
                } else {
                    break;
                }
            }
            a[i] = (Win[i][p[i] + 1] == EOW) ? EOW : (int64_t)Win[i][p[i] + 1] + d;
            if (a[i] < t) t = a[i];
        }
        if (t == EOW) break;

        /* switching: every pin arriving at t switches together */
        for (int i = 0; i < n; ++i) {
            sw[i] = (a[i] == t);
            if (sw[i]) p[i] += 1;
        }
        idx = 0;
        for (int i = 0; i < n; ++i) idx += (p[i] % 2) * weight[i];
        const int y = T[idx];

        if (y != (int)(po % 2)) { /* output change */
            const int e_out = y ? RISE : FALL;
            int64_t d = NO_ARC;
            for (int i = 0; i < n; ++i) {
                if (!sw[i]) continue;
                const int e_in = (p[i] % 2) ? RISE : FALL;
                int64_t col = 0;
                for (int j = 0; j < n; ++j)
                    if (j != i) col = col * 2 + (p[j] % 2);
                const int64_t row = 4 * i + 2 * e_in + e_out;
                const int64_t dd = D[row * ncol + col];
                if (dd != NO_ARC && dd < d) d = dd;
            }
            if (d == NO_ARC) return ORACLE_EBADLUT;
            const int64_t t_o = t + d;
            if (t_o >= EOW) return ORACLE_EINVAL;
            if (t_o - (int64_t)O->w[po] < reject_limit(d, q)) { /* gate inertial filter */
                po -= 1;                        /* cancel the unmatured entry */
            } else {
                po += 1;
                if (wbuf_reserve(O, po + 2)) return ORACLE_ENOMEM;
                O->w[po] = (int32_t)t_o;
            }
        }
    }
    if (wbuf_reserve(O, po + 2)) return ORACLE_ENOMEM;
    O->w[po + 1] = (int32_t)EOW;
    O->len = po + 2;

    /* statistics: toggles after the initial entries; time spent at 1 in [0, Lw) */
    *tc = po - (y0 ? 1 : 0);
    int64_t ones = 0;
    for (int64_t k = 1; k <= po; k += 2) {
        int64_t s = O->w[k], e = (k < po) ? O->w[k + 1] : Lw;
        if (s < 0) s = 0;
        if (e > Lw) e = Lw;
        if (e > s) ones += e - s;
    }
    *t1 = ones;
    return ORACLE_OK;
}

/* ---- checks of the input waveforms (Fig. 3 format) ------------------------ */
static int check_wave(const int32_t *w, int64_t len) {
    int64_t k = 0;
    if (len < 2) return 0;
    if (w[0] == -1) {
        if (w[1] != 0) return 0;
        k = 1;
    } else if (w[0] != 0) {
        return 0;
    }
    for (int64_t j = k + 1; j < len - 1; ++j)
        if (w[j] <= w[j - 1] || w[j] == EOW) return 0;
    return w[len - 1] == EOW;
}

/* ---- windows-parallel driver ---------------------------------------------- */
typedef struct {
    const oracle_netlist *nl;
    int32_t W;
    const int64_t *window_len;
    const int64_t *pi_off;
    const int32_t *pi_words;
    int32_t pulse_percent;
    int32_t w0, w1;         /* window range of this worker */
    wbuf pool;              /* gate outputs of this worker, task order (gate, window) */
    int64_t *start;         /* [G * nw] start of each (gate, local window) in pool */
    int64_t *len;           /* [G * nw] */
    int64_t *tc, *t1;       /* [G] partial sums */
    int status;
    char msg[256];
} worker;

static void *worker_run(void *arg) {
    worker *wk = (worker *)arg;
    const oracle_netlist *nl = wk->nl;
    const int32_t P = nl->num_inputs, G = nl->num_gates, W = wk->W;
    const int32_t nw = wk->w1 - wk->w0;
    wbuf O = {0, 0, 0};
    const int32_t *Win[MAXP];
    int32_t wr[MAXP], wf[MAXP], wt[MAXP];
    for (int32_t g = 0; g < G; ++g) {
        const int32_t ty = nl->gate_type[g];
        const int n = nl->type_num_pins[ty];
        const uint8_t *T = nl->tt_data + nl->type_tt_off[ty];
        const int32_t *D = nl->dly_data + nl->gate_dly_off[g];
        const int32_t e0 = nl->fanin_off[g];
        for (int i = 0; i < n; ++i) {
            wr[i] = nl->wire_rise[e0 + i];
            wf[i] = nl->wire_fall[e0 + i];
            wt[i] = nl->pin_weight[e0 + i];
        }
        for (int32_t lw = 0; lw < nw; ++lw) {
            const int32_t w = wk->w0 + lw;
            for (int i = 0; i < n; ++i) {
                const int32_t s = nl->fanin_net[e0 + i];
                if (s < P)
                    Win[i] = wk->pi_words + wk->pi_off[(int64_t)s * W + w];
                else
                    Win[i] = wk->pool.w + wk->start[(int64_t)(s - P) * nw + lw];
            }
            int64_t tc = 0, t1 = 0;
            int st = simulate_task(n, Win, wr, wf, wt, T, D, wk->window_len[w], wk->pulse_percent, &O, &tc, &t1);
            if (st != ORACLE_OK) {
                wk->status = st;
                snprintf(wk->msg, sizeof wk->msg, "gate %d window %d: %s", g, w,
                         st == ORACLE_EBADLUT ? "every switching arc has no delay"
                         : st == ORACLE_EINVAL ? "timestamp reaches EOW" : "out of memory");
                free(O.w);
                return NULL;
            }
            const int64_t at = wk->pool.len;
            if (wbuf_reserve(&wk->pool, at + O.len)) {
                wk->status = ORACLE_ENOMEM;
                snprintf(wk->msg, sizeof wk->msg, "out of memory");
                free(O.w);
                return NULL;
            }
            memcpy(wk->pool.w + at, O.w, (size_t)O.len * sizeof(int32_t));
            wk->pool.len = at + O.len;
            wk->start[(int64_t)g * nw + lw] = at;
            wk->len[(int64_t)g * nw + lw] = O.len;
            wk->tc[g] += tc;
            wk->t1[g] += t1;
        }
    }
    free(O.w);
    return NULL;
}

static int validate(const oracle_netlist *nl, int32_t W, const int64_t *pi_off, const int32_t *pi_words,
                    char *err, int errlen) {
    const int32_t P = nl->num_inputs, G = nl->num_gates;
    if (P < 0 || G < 0 || W < 1) {
        snprintf(err, errlen, "bad sizes");
        return ORACLE_EINVAL;
    }
    for (int32_t g = 0; g < G; ++g) {
        const int32_t ty = nl->gate_type[g];
        if (ty < 0 || ty >= nl->num_types) {
            snprintf(err, errlen, "gate %d: bad type", g);
            return ORACLE_EINVAL;
        }
        const int n = nl->type_num_pins[ty];
        if (n < 1 || n > MAXP || nl->fanin_off[g + 1] - nl->fanin_off[g] != n) {
            snprintf(err, errlen, "gate %d: bad pin count", g);
            return ORACLE_EINVAL;
        }
        for (int i = 0; i < n; ++i) {
            const int32_t s = nl->fanin_net[nl->fanin_off[g] + i];
            if (s < 0 || s >= P + g) {
                snprintf(err, errlen, "gate %d: fanin net %d is not an earlier net", g, s);
                return ORACLE_EINVAL;
            }
        }
    }
    for (int64_t k = 0; k < (int64_t)P * W; ++k) {
        if (!check_wave(pi_words + pi_off[k], pi_off[k + 1] - pi_off[k])) {
            snprintf(err, errlen, "input waveform %lld (net %lld, window %lld) is malformed", (long long)k,
                     (long long)(k / W), (long long)(k % W));
            return ORACLE_EBADWAVE;
        }
    }
    return ORACLE_OK;
}

/* Simulate the whole netlist in every window.  out_off receives the CSR offsets
 * of all (net, window) waveforms, net-major and window-minor, over a pool that
 * holds the input waveforms followed by the gate outputs in (gate, window)
 * order.  *out_pool is malloc'd and must be released with oracle_free. */
int oracle_simulate(const oracle_netlist *nl, int32_t W, const int64_t *window_len, const int64_t *pi_off,
                    const int32_t *pi_words, int32_t pulse_percent, int nthreads, int64_t *out_off,
                    int32_t **out_pool, int64_t *out_pool_words, int64_t *tc, int64_t *t1, char *err,
                    int errlen) {
    if (pulse_percent < 0 || pulse_percent > 100) {
        snprintf(err, errlen, "PATHPULSEPERCENT must be 0 .. 100");
        return ORACLE_EINVAL;
    }
    int st = validate(nl, W, pi_off, pi_words, err, errlen);
    if (st) return st;
    const int32_t P = nl->num_inputs, G = nl->num_gates;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > W) nthreads = W;
    worker *wk = (worker *)calloc((size_t)nthreads, sizeof(worker));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!wk || !th) {
        free(wk);
        free(th);
        snprintf(err, errlen, "out of memory");
        return ORACLE_ENOMEM;
    }
    for (int k = 0; k < nthreads; ++k) {
        worker *x = &wk[k];
        x->nl = nl;
        x->W = W;
        x->window_len = window_len;
        x->pi_off = pi_off;
        x->pi_words = pi_words;
        x->pulse_percent = pulse_percent;
        x->w0 = (int32_t)((int64_t)W * k / nthreads);
        x->w1 = (int32_t)((int64_t)W * (k + 1) / nthreads);
        const int64_t nw = x->w1 - x->w0;
        x->start = (int64_t *)calloc((size_t)(G * nw + 1), sizeof(int64_t));
        x->len = (int64_t *)calloc((size_t)(G * nw + 1), sizeof(int64_t));
        x->tc = (int64_t *)calloc((size_t)G + 1, sizeof(int64_t));
        x->t1 = (int64_t *)calloc((size_t)G + 1, sizeof(int64_t));
        if (!x->start || !x->len || !x->tc || !x->t1) st = ORACLE_ENOMEM;
    }
    if (st == ORACLE_OK) {
        if (nthreads == 1) {
            worker_run(&wk[0]);
        } else {
            for (int k = 0; k < nthreads; ++k) pthread_create(&th[k], NULL, worker_run, &wk[k]);
            for (int k = 0; k < nthreads; ++k) pthread_join(th[k], NULL);
        }
        for (int k = 0; k < nthreads && st == ORACLE_OK; ++k)
            if (wk[k].status) {
                st = wk[k].status;
                snprintf(err, errlen, "%s", wk[k].msg);
            }
    } else {
        snprintf(err, errlen, "out of memory");
    }
    if (st == ORACLE_OK) {
        /* lengths in (net, window) order, then their exclusive prefix sum */
        int64_t acc = 0;
        for (int64_t k = 0; k < (int64_t)P * W; ++k) {
            out_off[k] = acc;
            acc += pi_off[k + 1] - pi_off[k];
        }
        for (int32_t g = 0; g < G; ++g)
            for (int k = 0; k < nthreads; ++k) {
                const int64_t nw = wk[k].w1 - wk[k].w0;
                for (int64_t lw = 0; lw < nw; ++lw) {
                    out_off[(int64_t)(P + g) * W + wk[k].w0 + lw] = acc;
                    acc += wk[k].len[(int64_t)g * nw + lw];
                }
            }
        out_off[(int64_t)(P + G) * W] = acc;
        int32_t *pool = (int32_t *)malloc((size_t)(acc > 0 ? acc : 1) * sizeof(int32_t));
        if (!pool) {
            st = ORACLE_ENOMEM;
            snprintf(err, errlen, "out of memory");
        } else {
            memcpy(pool, pi_words + pi_off[0], (size_t)(pi_off[(int64_t)P * W] - pi_off[0]) * sizeof(int32_t));
            for (int32_t g = 0; g < G; ++g) {
                tc[g] = 0;
                t1[g] = 0;
                for (int k = 0; k < nthreads; ++k) {
                    const int64_t nw = wk[k].w1 - wk[k].w0;
                    for (int64_t lw = 0; lw < nw; ++lw) {
                        const int64_t dst = out_off[(int64_t)(P + g) * W + wk[k].w0 + lw];
                        memcpy(pool + dst, wk[k].pool.w + wk[k].start[(int64_t)g * nw + lw],
                               (size_t)wk[k].len[(int64_t)g * nw + lw] * sizeof(int32_t));
                    }
                    tc[g] += wk[k].tc[g];
                    t1[g] += wk[k].t1[g];
                }
            }
            *out_pool = pool;
            *out_pool_words = acc;
        }
    }
    for (int k = 0; k < nthreads; ++k) {
        free(wk[k].pool.w);
        free(wk[k].start);
        free(wk[k].len);
        free(wk[k].tc);
        free(wk[k].t1);
    }
    free(wk);
    free(th);
    return st;
}

void oracle_free(void *p) { free(p); }

/* ---- digests of every net's waveforms (level-parallel driver) -------------- */
/*
 * For checking runs too large to keep or compare word by word.  A net's digest is
 * the 64-bit FNV-1a hash (offset basis 14695981039346656037, prime 1099511628211,
 * one byte at a time) of the little-endian bytes of its waveforms concatenated in
 * window order, each window's array with its head and its EOW.  The caller passes
 * every net's running hash in and gets it back continued, so windows can be
 * simulated in consecutive batches (windows are independent) with the digest of the
 * whole run at the end.
 *
 * The driver processes the levels in order; inside a level every (gate, window) is
 * independent, so the level's tasks, gate-major, are split into one contiguous
 * range per thread.  Each task is simulate_task() above, unchanged.
 */
static uint64_t fnv1a_words(uint64_t h, const int32_t *w, int64_t n) {
    for (int64_t k = 0; k < n; ++k) {
        const uint32_t u = (uint32_t)w[k];
        for (int b = 0; b < 4; ++b) {
            h ^= (u >> (8 * b)) & 0xffu;
            h *= 1099511628211ULL;
        }
    }
    return h;
}

uint64_t oracle_fnv1a64(uint64_t h, const uint8_t *bytes, int64_t n) {
    for (int64_t k = 0; k < n; ++k) {
        h ^= bytes[k];
        h *= 1099511628211ULL;
    }
    return h;
}

typedef struct {
    const oracle_netlist *nl;
    int32_t W;
    const int64_t *window_len;
    const int64_t *pi_off;
    const int32_t *pi_words;
    int32_t pulse_percent;
    int32_t g0;               /* first gate of the level */
    int64_t k0, k1;           /* task range [k0, k1): task k = (g0 + k / W, k % W) */
    const int32_t **wave;     /* [G * W] output of (gate, window), once its level is done */
    int32_t *wlen;            /* [G * W] */
    wbuf out;                 /* this thread's outputs of this level, task order */
    int64_t *start;           /* [k1 - k0] start of each task's output in out */
    int64_t *tc, *t1;         /* [gates of the level] partial sums */
    int status;
    char msg[256];
} lvl_worker;

static void *lvl_worker_run(void *arg) {
    lvl_worker *wk = (lvl_worker *)arg;
    const oracle_netlist *nl = wk->nl;
    const int32_t P = nl->num_inputs, W = wk->W;
    wbuf O = {0, 0, 0};
    const int32_t *Win[MAXP];
    int32_t wr[MAXP], wf[MAXP], wt[MAXP];
    for (int64_t k = wk->k0; k < wk->k1; ++k) {
        const int32_t g = wk->g0 + (int32_t)(k / W), w = (int32_t)(k % W);
        const int32_t ty = nl->gate_type[g];
        const int n = nl->type_num_pins[ty];
        const int32_t e0 = nl->fanin_off[g];
        for (int i = 0; i < n; ++i) {
            const int32_t s = nl->fanin_net[e0 + i];
            wr[i] = nl->wire_rise[e0 + i];
            wf[i] = nl->wire_fall[e0 + i];
            wt[i] = nl->pin_weight[e0 + i];
            Win[i] = s < P ? wk->pi_words + wk->pi_off[(int64_t)s * W + w] : wk->wave[(int64_t)(s - P) * W + w];
        }
        int64_t tc = 0, t1 = 0;
        const int st = simulate_task(n, Win, wr, wf, wt, nl->tt_data + nl->type_tt_off[ty],
                                     nl->dly_data + nl->gate_dly_off[g], wk->window_len[w], wk->pulse_percent, &O,
                                     &tc, &t1);
        if (st != ORACLE_OK) {
            wk->status = st;
            snprintf(wk->msg, sizeof wk->msg, "gate %d window %d: %s", g, w,
                     st == ORACLE_EBADLUT ? "every switching arc has no delay"
                     : st == ORACLE_EINVAL ? "timestamp reaches EOW" : "out of memory");
            break;
        }
        const int64_t at = wk->out.len;
        if (wbuf_reserve(&wk->out, at + O.len)) {
            wk->status = ORACLE_ENOMEM;
            snprintf(wk->msg, sizeof wk->msg, "out of memory");
            break;
        }
        memcpy(wk->out.w + at, O.w, (size_t)O.len * sizeof(int32_t));
        wk->out.len = at + O.len;
        wk->start[k - wk->k0] = at;
        wk->wlen[(int64_t)g * W + w] = (int32_t)O.len;
        wk->tc[g - wk->g0] += tc;
        wk->t1[g - wk->g0] += t1;
    }
    free(O.w);
    return NULL;
}

typedef struct {
    const int32_t *const *wave;   /* per (net, window) first word */
    const int64_t *len;           /* per (net, window) words */
    int32_t W;
    int64_t n0, n1;               /* net range */
    uint64_t *hash;               /* [nets], continued */
    int64_t *words;               /* [nets], accumulated */
} hash_worker;

static void *hash_worker_run(void *arg) {
    hash_worker *hw = (hash_worker *)arg;
    for (int64_t net = hw->n0; net < hw->n1; ++net)
        for (int32_t w = 0; w < hw->W; ++w) {
            const int64_t k = net * hw->W + w;
            hw->hash[net] = fnv1a_words(hw->hash[net], hw->wave[k], hw->len[k]);
            hw->words[net] += hw->len[k];
        }
    return NULL;
}

/* Simulate every gate in every window and continue each net's digest (net_hash,
 * [P + G], in/out) and word count (net_words, in/out) over this run's windows in
 * window order; TC and T1 of every gate are added to tc[G] and t1[G]. */
int oracle_digest(const oracle_netlist *nl, int32_t W, const int64_t *window_len, const int64_t *pi_off,
                  const int32_t *pi_words, int32_t pulse_percent, int nthreads, uint64_t *net_hash,
                  int64_t *net_words, int64_t *tc, int64_t *t1, char *err, int errlen) {
    if (pulse_percent < 0 || pulse_percent > 100) {
        snprintf(err, errlen, "PATHPULSEPERCENT must be 0 .. 100");
        return ORACLE_EINVAL;
    }
    int st = validate(nl, W, pi_off, pi_words, err, errlen);
    if (st) return st;
    const int32_t P = nl->num_inputs, G = nl->num_gates, L = nl->num_levels;
    if (nthreads < 1) nthreads = 1;
    const int64_t NW = (int64_t)(P + G) * W;
    const int32_t **wave = (const int32_t **)calloc((size_t)(NW + 1), sizeof(int32_t *));
    int64_t *len = (int64_t *)calloc((size_t)(NW + 1), sizeof(int64_t));
    int32_t *glen = (int32_t *)calloc((size_t)((int64_t)G * W + 1), sizeof(int32_t));
    wbuf *bufs = (wbuf *)calloc((size_t)L * nthreads + 1, sizeof(wbuf));   /* [level][thread] */
    lvl_worker *wk = (lvl_worker *)calloc((size_t)nthreads, sizeof(lvl_worker));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!wave || !len || !glen || !bufs || !wk || !th) {
        st = ORACLE_ENOMEM;
        snprintf(err, errlen, "out of memory");
    }
    for (int64_t k = 0; st == ORACLE_OK && k < (int64_t)P * W; ++k) {
        wave[k] = pi_words + pi_off[k];
        len[k] = pi_off[k + 1] - pi_off[k];
    }
    /* gate outputs, level by level; wave[] of a level's gates is set once it is done */
    const int32_t **gwave = wave + (int64_t)P * W;
    for (int32_t l = 0; st == ORACLE_OK && l < L; ++l) {
        const int32_t g0 = nl->level_offsets[l], ng = nl->level_offsets[l + 1] - g0;
        const int64_t ntask = (int64_t)ng * W;
        for (int k = 0; k < nthreads; ++k) {
            lvl_worker *x = &wk[k];
            memset(x, 0, sizeof *x);
            x->nl = nl;
            x->W = W;
            x->window_len = window_len;
            x->pi_off = pi_off;
            x->pi_words = pi_words;
            x->pulse_percent = pulse_percent;
            x->g0 = g0;
            x->k0 = ntask * k / nthreads;
            x->k1 = ntask * (k + 1) / nthreads;
            x->wave = gwave;
            x->wlen = glen;
            x->start = (int64_t *)calloc((size_t)(x->k1 - x->k0 + 1), sizeof(int64_t));
            x->tc = (int64_t *)calloc((size_t)ng + 1, sizeof(int64_t));
            x->t1 = (int64_t *)calloc((size_t)ng + 1, sizeof(int64_t));
            if (!x->start || !x->tc || !x->t1) st = ORACLE_ENOMEM;
        }
        if (st == ORACLE_OK) {
            if (nthreads == 1) {
                lvl_worker_run(&wk[0]);
            } else {
                for (int k = 0; k < nthreads; ++k) pthread_create(&th[k], NULL, lvl_worker_run, &wk[k]);
                for (int k = 0; k < nthreads; ++k) pthread_join(th[k], NULL);
            }
            for (int k = 0; k < nthreads && st == ORACLE_OK; ++k)
                if (wk[k].status) {
                    st = wk[k].status;
                    snprintf(err, errlen, "%s", wk[k].msg);
                }
        } else {
            snprintf(err, errlen, "out of memory");
        }
        for (int k = 0; k < nthreads; ++k) {
            lvl_worker *x = &wk[k];
            if (st == ORACLE_OK) {
                for (int64_t t = x->k0; t < x->k1; ++t) {
                    const int64_t gk = (int64_t)g0 * W + t;      /* (gate, window) index */
                    gwave[gk] = x->out.w + x->start[t - x->k0];
                    len[(int64_t)P * W + gk] = glen[gk];
                }
                for (int32_t j = 0; j < ng; ++j) {
                    tc[g0 + j] += x->tc[j];
                    t1[g0 + j] += x->t1[j];
                }
            }
            bufs[(int64_t)l * nthreads + k] = x->out;      /* kept: later levels read it */
            free(x->start);
            free(x->tc);
            free(x->t1);
        }
    }
    if (st == ORACLE_OK) {
        const int64_t nets = (int64_t)P + G;
        hash_worker *hw = (hash_worker *)calloc((size_t)nthreads, sizeof(hash_worker));
        if (!hw) {
            st = ORACLE_ENOMEM;
            snprintf(err, errlen, "out of memory");
        } else {
            for (int k = 0; k < nthreads; ++k) {
                hw[k].wave = wave;
                hw[k].len = len;
                hw[k].W = W;
                hw[k].n0 = nets * k / nthreads;
                hw[k].n1 = nets * (k + 1) / nthreads;
                hw[k].hash = net_hash;
                hw[k].words = net_words;
            }
            if (nthreads == 1) {
                hash_worker_run(&hw[0]);
            } else {
                for (int k = 0; k < nthreads; ++k) pthread_create(&th[k], NULL, hash_worker_run, &hw[k]);
                for (int k = 0; k < nthreads; ++k) pthread_join(th[k], NULL);
            }
            free(hw);
        }
    }
    if (bufs)
        for (int64_t k = 0; k < (int64_t)L * nthreads; ++k) free(bufs[k].w);
    free(bufs);
    free(wave);
    free(len);
    free(glen);
    free(wk);
    free(th);
    return st;
}
