/*
 * TEST INFRASTRUCTURE ONLY: a brute-force unit-time-step simulator that pins the
 * event-driven oracle on tiny netlists.  It shares no code with the oracle's
 * event loop nor with the CUDA library.
 *
 * Model (inertial delays as in Verilog-style gate and interconnect delays with a
 * pulse reject limit of q percent of the delay, q = PATHPULSEPERCENT; the GATSPI
 * page's Algorithm 1 implements q = 100):
 *   - every fanin edge (interconnect) and every gate is an inertial element with
 *     an output value and a queue of pending events (value, due time, the time it
 *     was scheduled, its delay), oldest first;
 *   - time advances one unit per step; within a step, elements are visited in
 *     topological order (wires of a gate, then the gate, gates in level order);
 *   - at each step an element first lets the pending events due now take effect,
 *     then applies the input changes of this step one after another; a net can
 *     change more than once in one step (zero-width pulses) and its k-th change is
 *     applied at the k-th sub-step;
 *   - delays: rise delay for a new value 1, fall delay for 0 on a wire; on a gate,
 *     the smallest finite conditional delay among the pins that changed in this
 *     sub-step, looked up at row 4*pin + 2*e_in + e_out, RISE = 0, FALL = 1, and at
 *     the column formed by the other pins' values, first pin most significant;
 *     r(d) = floor(d * q / 100) is the reject limit of delay d;
 *   - a wire input change at time now withdraws the newest pending event when that
 *     event was scheduled less than r(its delay) ago (the pulse it starts is too
 *     narrow); otherwise it schedules (v, now + d);
 *   - a gate compares its new value with its last scheduled value (the newest
 *     pending value, else its output) and does nothing when equal; otherwise it
 *     withdraws the newest pending event when the output pulse between that event
 *     and now + d would be narrower than r(d), else schedules (v, now + d);
 *   - with q = 100 both withdrawal tests mean "not yet due", so at most one event
 *     is ever pending; a zero delay with nothing pending takes effect at once;
 *   - an element whose events would fall due out of order (a wire whose rise and
 *     fall delays differ by more than a pulse it lets through) is outside this
 *     model: the run fails with ORACLE_EINVAL;
 *   - each window starts from the zero-delay steady state of the inputs' values.
 * Output waveforms are written in the Fig. 3 array format: [0] or [-1, 0], then
 * one timestamp per change, then EOW.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "oracle_abi.h"

#define BF_EOW 2147483647
#define BF_NONE 2147483647
#define BF_MAXP 8

typedef struct {
    int val;
    long long due, at, d;   /* due time, time scheduled, delay */
} event;

typedef struct {
    int out;
    int n, cap;     /* pending events q[0 .. n), oldest first */
    event *q;
} element;

static long long bf_reject(long long d, int32_t q) { return d * q / 100; }

static int el_push(element *x, int v, long long now, long long d) {
    if (x->n > 0 && now + d < x->q[x->n - 1].due) return -2; /* out of order */
    if (x->n == x->cap) {
        int c = x->cap ? 2 * x->cap : 4;
        event *nq = (event *)realloc(x->q, (size_t)c * sizeof(event));
        if (!nq) return -1;
        x->q = nq;
        x->cap = c;
    }
    x->q[x->n].val = v;
    x->q[x->n].due = now + d;
    x->q[x->n].at = now;
    x->q[x->n].d = d;
    x->n += 1;
    return 0;
}

/* Let the events due now take effect; returns how many did. */
static int el_mature(element *x, long long now) {
    int k = 0;
    while (k < x->n && x->q[k].due == now) x->out = x->q[k++].val;
    if (k) {
        memmove(x->q, x->q + k, (size_t)(x->n - k) * sizeof(event));
        x->n -= k;
    }
    return k;
}

typedef struct {
    int32_t *t;
    long long n, cap;
} tlist;

static int tl_push(tlist *l, int32_t v) {
    if (l->n == l->cap) {
        long long c = l->cap ? 2 * l->cap : 16;
        int32_t *nt = (int32_t *)realloc(l->t, (size_t)c * sizeof(int32_t));
        if (!nt) return -1;
        l->t = nt;
        l->cap = c;
    }
    l->t[l->n++] = v;
    return 0;
}

static int bf_lookup(const uint8_t *tt, const int32_t *wt, const int *v, int n) {
    long long k = 0;
    for (int i = 0; i < n; ++i)
        if (v[i]) k += wt[i];
    return tt[k];
}

/* Simulate one window; fills per-gate change lists and initial values. */
static int bf_window(const oracle_netlist *nl, int32_t W, int32_t w, long long Lw, const int64_t *pi_off,
                     const int32_t *pi_words, int32_t q, tlist *changes, int *init, long long *ones, char *err,
                     int errlen) {
    const int32_t P = nl->num_inputs, G = nl->num_gates, N = P + G;
    const int32_t E = nl->fanin_off[G];
    int *val = (int *)calloc((size_t)N + 1, sizeof(int));      /* value at the end of the step */
    int *prev = (int *)calloc((size_t)N + 1, sizeof(int));     /* value at the start of the step */
    int *cnt = (int *)calloc((size_t)N + 1, sizeof(int));      /* number of changes in this step */
    long long *cur = (long long *)calloc((size_t)P + 1, sizeof(long long));
    element *wire = (element *)calloc((size_t)E + 1, sizeof(element));
    element *gate = (element *)calloc((size_t)G + 1, sizeof(element));
    int *wcnt = (int *)calloc((size_t)E + 1, sizeof(int));
    int *wprev = (int *)calloc((size_t)E + 1, sizeof(int));
    int rc = ORACLE_OK;
    if (!val || !prev || !cnt || !cur || !wire || !gate || !wcnt || !wprev) {
        rc = ORACLE_ENOMEM;
        goto done;
    }

    /* steady state at time 0 */
    long long last_input = 0;
    for (int32_t s = 0; s < P; ++s) {
        const int32_t *x = pi_words + pi_off[(int64_t)s * W + w];
        const long long len = pi_off[(int64_t)s * W + w + 1] - pi_off[(int64_t)s * W + w];
        val[s] = (x[0] == -1);
        cur[s] = (x[0] == -1) ? 2 : 1;
        if (len >= 2 && len - 2 >= cur[s] && x[len - 2] > last_input) last_input = x[len - 2];
    }
    for (int32_t g = 0; g < G; ++g) {
        const int32_t ty = nl->gate_type[g];
        const int n = nl->type_num_pins[ty];
        int v[BF_MAXP];
        for (int i = 0; i < n; ++i) {
            const int32_t e = nl->fanin_off[g] + i;
            wire[e].out = val[nl->fanin_net[e]];
            v[i] = wire[e].out;
        }
        gate[g].out = bf_lookup(nl->tt_data + nl->type_tt_off[ty], nl->pin_weight + nl->fanin_off[g], v, n);
        val[P + g] = gate[g].out;
        init[g] = gate[g].out;
    }
    for (int32_t g = 0; g < G; ++g) ones[g] = 0;

    for (long long now = 0;; ++now) {
        if (now > 0) {
            int busy = now <= last_input;
            for (int32_t e = 0; e < E && !busy; ++e) busy = wire[e].n > 0;
            for (int32_t g = 0; g < G && !busy; ++g) busy = gate[g].n > 0;
            if (!busy && now >= Lw) break;
            /* input changes at this step */
            for (int32_t s = 0; s < P; ++s) {
                const int32_t *x = pi_words + pi_off[(int64_t)s * W + w];
                prev[s] = val[s];
                cnt[s] = 0;
                while (x[cur[s]] != BF_EOW && x[cur[s]] == now) {
                    val[s] ^= 1;
                    cnt[s] += 1;
                    cur[s] += 1;
                }
                if (x[cur[s]] != BF_EOW && x[cur[s]] < now) {
                    snprintf(err, errlen, "input %d window %d: timestamps not increasing", s, w);
                    rc = ORACLE_EBADWAVE;
                    goto done;
                }
            }
            for (int32_t g = 0; g < G; ++g) {
                const int32_t ty = nl->gate_type[g];
                const int n = nl->type_num_pins[ty];
                const int32_t e0 = nl->fanin_off[g];
                const uint8_t *tt = nl->tt_data + nl->type_tt_off[ty];
                const int32_t *D = nl->dly_data + nl->gate_dly_off[g];
                const int ncol = 1 << (n - 1);
                int maxk = 0;
                /* the gate's interconnects */
                for (int i = 0; i < n; ++i) {
                    const int32_t e = e0 + i;
                    const int32_t s = nl->fanin_net[e];
                    element *x = &wire[e];
                    wprev[e] = x->out;
                    wcnt[e] = 0;
                    wcnt[e] += el_mature(x, now);
                    for (int k = 1; k <= cnt[s]; ++k) {
                        const int sv = prev[s] ^ (k & 1);
                        const int last = x->n ? x->q[x->n - 1].val : x->out;
                        if (x->n && now - x->q[x->n - 1].at < bf_reject(x->q[x->n - 1].d, q)) {
                            x->n -= 1; /* the pulse the newest event starts is too narrow */
                        } else if (sv != last) {
                            const long long d = sv ? nl->wire_rise[e] : nl->wire_fall[e];
                            if (d == 0 && x->n == 0) {
                                x->out = sv;
                                wcnt[e] += 1;
                            } else {
                                const int pr = el_push(x, sv, now, d);
                                if (pr) {
                                    snprintf(err, errlen, "wire %d window %d: %s", e, w,
                                             pr == -2 ? "events fall due out of order" : "out of memory");
                                    rc = pr == -2 ? ORACLE_EINVAL : ORACLE_ENOMEM;
                                    goto done;
                                }
                            }
                        }
                    }
                    if (wcnt[e] > maxk) maxk = wcnt[e];
                }
                /* the gate */
                element *y = &gate[g];
                prev[P + g] = y->out;
                cnt[P + g] = 0;
                for (int k = el_mature(y, now); k > 0; --k) {
                    cnt[P + g] += 1;
                    if (tl_push(&changes[g], (int32_t)now)) {
                        rc = ORACLE_ENOMEM;
                        goto done;
                    }
                }
                int pv[BF_MAXP];
                for (int i = 0; i < n; ++i) pv[i] = wprev[e0 + i];
                for (int k = 1; k <= maxk; ++k) {
                    int changed[BF_MAXP];
                    for (int i = 0; i < n; ++i) {
                        changed[i] = wcnt[e0 + i] >= k;
                        if (changed[i]) pv[i] ^= 1;
                    }
                    const int nv = bf_lookup(tt, nl->pin_weight + e0, pv, n);
                    const int last = y->n ? y->q[y->n - 1].val : y->out;
                    if (nv == last) continue;
                    long long d = BF_NONE;
                    for (int i = 0; i < n; ++i) {
                        if (!changed[i]) continue;
                        int row = 4 * i + 2 * (pv[i] ? 0 : 1) + (nv ? 0 : 1);
                        int col = 0;
                        for (int j = 0; j < n; ++j) {
                            if (j == i) continue;
                            col = (col << 1) | pv[j];
                        }
                        const long long dd = D[row * ncol + col];
                        if (dd != BF_NONE && dd < d) d = dd;
                    }
                    if (d == BF_NONE) {
                        snprintf(err, errlen, "gate %d window %d: every switching arc has no delay", g, w);
                        rc = ORACLE_EBADLUT;
                        goto done;
                    }
                    if (y->n && now + d - y->q[y->n - 1].due < bf_reject(d, q)) {
                        y->n -= 1; /* the output pulse would be too narrow */
                    } else if (d == 0 && y->n == 0) {
                        y->out = nv;
                        cnt[P + g] += 1;
                        if (tl_push(&changes[g], (int32_t)now)) {
                            rc = ORACLE_ENOMEM;
                            goto done;
                        }
                    } else {
                        const int pr = el_push(y, nv, now, d);
                        if (pr) {
                            snprintf(err, errlen, "gate %d window %d: %s", g, w,
                                     pr == -2 ? "events fall due out of order" : "out of memory");
                            rc = pr == -2 ? ORACLE_EINVAL : ORACLE_ENOMEM;
                            goto done;
                        }
                    }
                }
                val[P + g] = y->out;
            }
        }
        if (now < Lw)
            for (int32_t g = 0; g < G; ++g) ones[g] += gate[g].out;
    }
done:
    if (wire)
        for (int32_t e = 0; e < E; ++e) free(wire[e].q);
    if (gate)
        for (int32_t g = 0; g < G; ++g) free(gate[g].q);
    free(val);
    free(prev);
    free(cnt);
    free(cur);
    free(wire);
    free(gate);
    free(wcnt);
    free(wprev);
    return rc;
}

/* Same output layout as oracle_simulate: CSR offsets over (net, window), net-major. */
int brute_simulate(const oracle_netlist *nl, int32_t W, const int64_t *window_len, const int64_t *pi_off,
                   const int32_t *pi_words, int32_t pulse_percent, int64_t *out_off, int32_t **out_pool, int64_t *out_pool_words,
                   int64_t *tc, int64_t *t1, char *err, int errlen) {
    const int32_t P = nl->num_inputs, G = nl->num_gates;
    tlist *ch = (tlist *)calloc((size_t)G * W + 1, sizeof(tlist));
    int *init = (int *)calloc((size_t)G * W + 1, sizeof(int));
    long long *ones = (long long *)calloc((size_t)G * W + 1, sizeof(long long));
    int rc = ORACLE_OK;
    if (!ch || !init || !ones) {
        rc = ORACLE_ENOMEM;
        goto out;
    }
    {
        tlist *tmp = (tlist *)calloc((size_t)G + 1, sizeof(tlist));
        int *ini = (int *)calloc((size_t)G + 1, sizeof(int));
        long long *on = (long long *)calloc((size_t)G + 1, sizeof(long long));
        for (int32_t w = 0; w < W && rc == ORACLE_OK; ++w) {
            for (int32_t g = 0; g < G; ++g) tmp[g].n = 0;
            rc = bf_window(nl, W, w, window_len[w], pi_off, pi_words, pulse_percent, tmp, ini, on, err, errlen);
            for (int32_t g = 0; g < G && rc == ORACLE_OK; ++g) {
                tlist *dst = &ch[(int64_t)g * W + w];
                for (long long k = 0; k < tmp[g].n; ++k) tl_push(dst, tmp[g].t[k]);
                init[(int64_t)g * W + w] = ini[g];
                ones[(int64_t)g * W + w] = on[g];
            }
        }
        for (int32_t g = 0; g < G; ++g) free(tmp[g].t);
        free(tmp);
        free(ini);
        free(on);
    }
    if (rc != ORACLE_OK) goto out;
    {
        int64_t acc = 0;
        for (int64_t k = 0; k < (int64_t)P * W; ++k) {
            out_off[k] = acc;
            acc += pi_off[k + 1] - pi_off[k];
        }
        for (int64_t k = 0; k < (int64_t)G * W; ++k) {
            out_off[(int64_t)P * W + k] = acc;
            acc += (init[k] ? 2 : 1) + ch[k].n + 1;
        }
        out_off[(int64_t)(P + G) * W] = acc;
        int32_t *pool = (int32_t *)malloc((size_t)(acc > 0 ? acc : 1) * sizeof(int32_t));
        if (!pool) {
            rc = ORACLE_ENOMEM;
            goto out;
        }
        memcpy(pool, pi_words + pi_off[0], (size_t)(pi_off[(int64_t)P * W] - pi_off[0]) * sizeof(int32_t));
        for (int32_t g = 0; g < G; ++g) {
            tc[g] = 0;
            t1[g] = 0;
            for (int32_t w = 0; w < W; ++w) {
                const int64_t k = (int64_t)g * W + w;
                int32_t *o = pool + out_off[(int64_t)P * W + k];
                int64_t j = 0;
                if (init[k]) o[j++] = -1;
                o[j++] = 0;
                for (long long q = 0; q < ch[k].n; ++q) o[j++] = ch[k].t[q];
                o[j++] = BF_EOW;
                tc[g] += ch[k].n;
                t1[g] += ones[k];
            }
        }
        *out_pool = pool;
        *out_pool_words = acc;
    }
out:
    if (ch)
        for (int64_t k = 0; k < (int64_t)G * W; ++k) free(ch[k].t);
    free(ch);
    free(init);
    free(ones);
    return rc;
}
