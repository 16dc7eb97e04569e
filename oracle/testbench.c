/*
 * TEST INFRASTRUCTURE ONLY: the CPU oracle of the testbench restructuring.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load it.
 * It shares no code with the CUDA library and is deliberately plain and slow.
 *
 * What it computes (GATSPI: GPU-Accelerated Gate-Level Simulation for Power
 * Improvement -- Section 1 and Section 4 on cycle parallelism with known input
 * waveforms; Section 5, Table 5, where restructuring the input waveforms into the
 * cycle-parallel format takes most of the application's set-up time): every
 * input's waveform over the whole testbench (Fig. 3 format, times from the start
 * of the testbench) is cut into the cycle windows, each window becoming an
 * independent waveform that starts at its own time 0.
 *
 * Readings where the page is silent:
 *   - window w covers [S_w, S_w + L_w) with S_w the sum of the lengths of the
 *     windows before it;
 *   - the window's initial value is the input's value at S_w, so a transition
 *     exactly at S_w folds into it (a window waveform has no transition at its
 *     time 0); a transition inside (S_w, S_w + L_w) becomes t - S_w;
 *   - transitions at or after the end of the last window belong to no window.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "oracle_abi.h"

#define TB_EOW 2147483647

typedef struct {
    int32_t *w;
    int64_t n, cap;
} tbuf;

static int tb_push(tbuf *b, int32_t v) {
    if (b->n == b->cap) {
        int64_t c = b->cap ? 2 * b->cap : 1024;
        int32_t *nw = (int32_t *)realloc(b->w, (size_t)c * sizeof(int32_t));
        if (!nw) return -1;
        b->w = nw;
        b->cap = c;
    }
    b->w[b->n++] = v;
    return 0;
}

/* Fig. 3 format over the whole testbench: [0] or [-1, 0], strictly increasing
 * times from 1, EOW last. */
static int tb_wave_ok(const int32_t *x, int64_t len) {
    int64_t k;
    if (len < 2) return 0;
    if (x[0] == -1) {
        if (x[1] != 0) return 0;
        k = 2;
    } else if (x[0] == 0) {
        k = 1;
    } else {
        return 0;
    }
    for (int64_t j = k; j < len - 1; ++j) {
        if (x[j] == TB_EOW) return 0;
        if (x[j] <= (j == k ? 0 : x[j - 1])) return 0;
    }
    return x[len - 1] == TB_EOW;
}

/* Cut the testbench of P inputs (CSR tb_off[P + 1] over tb_words) into W windows of
 * window_len[w] time units.  out_off[P * W + 1] receives the CSR offsets of the
 * (input, window) waveforms, input-major and window-minor; *out_words is malloc'd
 * and released with oracle_free. */
int oracle_restructure(int32_t P, const int64_t *tb_off, const int32_t *tb_words, int32_t W,
                       const int64_t *window_len, int64_t *out_off, int32_t **out_words, int64_t *out_nwords,
                       char *err, int errlen) {
    if (P < 0 || W < 1) {
        snprintf(err, errlen, "bad sizes");
        return ORACLE_EINVAL;
    }
    for (int32_t w = 0; w < W; ++w)
        if (window_len[w] < 1) {
            snprintf(err, errlen, "window %d: length must be positive", w);
            return ORACLE_EINVAL;
        }
    tbuf out = {0, 0, 0};
    int64_t k = 0;
    for (int32_t p = 0; p < P; ++p) {
        const int32_t *x = tb_words + tb_off[p];
        const int64_t len = tb_off[p + 1] - tb_off[p];
        if (!tb_wave_ok(x, len)) {
            snprintf(err, errlen, "input %d: malformed testbench waveform", p);
            free(out.w);
            return ORACLE_EBADWAVE;
        }
        int value = (x[0] == -1);
        int64_t i = value ? 2 : 1; /* next transition */
        int64_t start = 0;
        for (int32_t w = 0; w < W; ++w) {
            const int64_t end = start + window_len[w];
            /* value at the window's start: transitions up to and including it */
            while (x[i] != TB_EOW && x[i] <= start) {
                value ^= 1;
                ++i;
            }
            out_off[k++] = out.n;
            int bad = value ? (tb_push(&out, -1) || tb_push(&out, 0)) : tb_push(&out, 0);
            /* transitions inside the window, relative to its start */
            while (!bad && x[i] != TB_EOW && x[i] < end) {
                bad = tb_push(&out, (int32_t)(x[i] - start));
                value ^= 1;
                ++i;
            }
            if (bad || tb_push(&out, TB_EOW)) {
                snprintf(err, errlen, "out of memory");
                free(out.w);
                return ORACLE_ENOMEM;
            }
            start = end;
        }
    }
    out_off[k] = out.n;
    *out_words = out.w ? out.w : (int32_t *)malloc(sizeof(int32_t));
    *out_nwords = out.n;
    return ORACLE_OK;
}
