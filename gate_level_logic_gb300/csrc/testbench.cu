// Testbench restructuring on the device: whole-testbench input waveforms cut into
// the cycle windows.
//
// GATSPI (Sections 1 and 4) re-simulates cycle windows in parallel from known input
// waveforms; the page restructures the inputs into that per-window format on the
// host, and its application profile (Section 5, Table 5) shows this restructuring
// is most of the set-up time.  Here it is two kernels over device-resident data:
//
// tb_check_kernel: one warp per input checks the Fig. 3 format of its testbench
// waveform (head [0] or [-1, 0], times strictly increasing from 1, EOW last) and
// its offsets.
//
// tb_cut_kernel: one warp per (input, chunk of 32 consecutive windows); lane j takes window
// w = 32c + j, which covers [S_w, S_w + L_w).  Two binary searches give the window's
// transitions (after S_w, before S_w + L_w) and its initial value (the parity of the
// last entry at or before S_w: a transition exactly at S_w folds into it).  A warp
// scan places the chunk's windows; each lane writes its head, its transitions minus
// S_w and EOW, and its window-index entry.  No scan over inputs is needed: input p's
// windows take at most (its transitions) + 3 W words, so its region starts at
// (tb_off[p] - tb_off[0]) + 3 W p, and chunk c of it at that plus (transitions before
// S_32c) + 96 c -- the same bound-and-gap layout as the gates' outputs.
// Transitions at or after the end of the last window belong to no window.
#include "gatspi_internal.cuh"
#include "testbench.cuh"

namespace gatspi {

namespace {

__device__ __forceinline__ int tb_status(const int32_t *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ void tb_raise(int32_t *status, int code, int a, int b, int c) {
    if (atomicCAS(status, 0, code) == 0) {
        status[1] = a;
        status[2] = b;
        status[3] = c;
    }
}

// first index k in [lo, hi) with x[k] > v (hi if none); x sorted ascending
__device__ __forceinline__ long long upper_bound(const int32_t *x, long long lo, long long hi, long long v) {
    while (lo < hi) {
        const long long mid = (lo + hi) >> 1;
        if ((long long)x[mid] <= v)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// first index k in [lo, hi) with x[k] >= v (hi if none)
__device__ __forceinline__ long long lower_bound(const int32_t *x, long long lo, long long hi, long long v) {
    while (lo < hi) {
        const long long mid = (lo + hi) >> 1;
        if ((long long)x[mid] < v)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

__global__ void tb_check_kernel(const DevParams P, const long long *__restrict__ tb_off,
                                const int32_t *__restrict__ tb, long long nwords) {
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= P.num_inputs) return;
    const int p = (int)warp;
    const long long s = tb_off[p], e = tb_off[p + 1];
    const long long len = e - s;
    bool ok = s >= 0 && s <= e && e <= nwords && len >= 2 && len < (1ll << 31);
    if (ok) {
        const int32_t *x = tb + s;
        long long h = 1;
        if (x[0] == -1) {
            ok = x[1] == 0;
            h = 2;
        } else {
            ok = x[0] == 0;
        }
        if (ok) {
            for (long long j = h + lane; j < len - 1; j += 32) {
                const int32_t prev = j == h ? 0 : x[j - 1];
                if (x[j] <= prev || x[j] == kEOW) ok = false;
            }
            if (lane == 0 && x[len - 1] != kEOW) ok = false;
        }
    }
    const bool bad = __any_sync(0xffffffffu, !ok);
    if (bad && lane == 0) tb_raise(P.status, GATSPI_EBADWAVE, p, -1, 0);
}

__global__ void tb_cut_kernel(const DevParams P, const long long *__restrict__ tb_off, const int32_t *__restrict__ tb,
                              const long long *__restrict__ wstart) {
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nch = (P.W + 31) / 32;
    if (warp >= (long long)P.num_inputs * nch) return;
    if (__shfl_sync(0xffffffffu, lane == 0 ? tb_status(P.status) : 0, 0) != 0) return;   // malformed input
    const int p = (int)(warp / nch);
    const int c = (int)(warp - (long long)p * nch);
    const int w = c * 32 + lane;
    const bool valid = w < P.W;

    const long long s = tb_off[p];
    const int32_t *x = tb + s;
    const long long eow = tb_off[p + 1] - s - 1;          // index of EOW
    const long long h = x[0] == -1 ? 2 : 1;               // first transition
    long long lo = h, hi = h;
    long long S = 0;
    int v0 = 0;
    uint32_t wl = 0;
    if (valid) {
        S = wstart[w];
        lo = upper_bound(x, h, eow, S);
        hi = lower_bound(x, lo, eow, wstart[w + 1]);
        v0 = (int)((lo - 1) & 1);
        wl = (uint32_t)(1 + v0 + (hi - lo) + 1);
    }
    uint32_t incl = wl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - wl;
    // the input's region starts at (tb_off[p] - tb_off[0]) + 3 W p; chunk c of it at
    // (transitions before S_32c) + 96 c further
    const long long region = (s - tb_off[0]) + 3ll * P.W * p;
    uint32_t rel = 0;
    if (lane == 0) rel = (uint32_t)(lower_bound(x, h, eow, wstart[c * 32]) - h + 96ll * c);
    rel = __shfl_sync(0xffffffffu, rel, 0);
    if (c == 0 && lane == 0) P.net_base[p] = region;
    if (valid) {
        int32_t *dst = P.pool + region + rel + excl;
        int k = 0;
        if (v0) dst[k++] = -1;
        dst[k++] = 0;
        for (long long i = lo; i < hi; ++i) dst[k++] = (int32_t)((long long)x[i] - S);
        dst[k] = kEOW;
        P.wstart[(long long)p * P.W + w] = rel + excl;
        P.wend[(long long)p * P.W + w] = rel + incl;
        P.wlen8[(long long)p * P.w8stride + w] = (uint8_t)min(wl, 255u);
    }
    if (warp == 0 && lane == 0) P.level_base[0] = (tb_off[P.num_inputs] - tb_off[0]) + 3ll * P.W * P.num_inputs;
}

// Toggle count and time at 1 of every input, summed over its windows (the inputs'
// part of the SAIF statistics): one warp per input, a lane per window.
__global__ void input_stats_kernel(const DevParams P, unsigned long long *__restrict__ tc,
                                   unsigned long long *__restrict__ t1) {
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= P.num_inputs) return;
    const long long p = warp;
    long long toggles = 0, ones = 0;
    for (int w = lane; w < P.W; w += 32) {
        const uint32_t end = P.wend[p * P.W + w];
        const uint32_t start = P.wstart[p * P.W + w];
        const int32_t *x = P.pool + P.net_base[p] + start;
        const int len = (int)(end - start);
        const long long Lw = P.window_len[w];
        const int h = x[0] == -1 ? 2 : 1;
        int v = h - 1;               // value from time 0
        long long from = 0;          // start of the current interval, clipped to Lw
        for (int k = h; k < len - 1; ++k) {
            const long long t = min((long long)x[k], Lw);
            if (v) ones += t - from;
            from = t;
            v ^= 1;
        }
        if (v) ones += Lw - from;
        toggles += len - h - 1;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        toggles += __shfl_xor_sync(0xffffffffu, toggles, o);
        ones += __shfl_xor_sync(0xffffffffu, ones, o);
    }
    if (lane == 0) {
        tc[p] = (unsigned long long)toggles;
        t1[p] = (unsigned long long)ones;
    }
}

}  // namespace

cudaError_t launch_input_stats(const DevParams &p, unsigned long long *tc, unsigned long long *t1, cudaStream_t s) {
    if (p.num_inputs == 0) return cudaSuccess;
    const int threads = 256;
    const long long warps = p.num_inputs;
    input_stats_kernel<<<(unsigned)((warps * 32 + threads - 1) / threads), threads, 0, s>>>(p, tc, t1);
    return cudaGetLastError();
}

cudaError_t launch_testbench_cut(const DevParams &p, const long long *tb_off, const int32_t *tb, long long nwords,
                                 const long long *wstart, cudaStream_t s) {
    if (p.num_inputs == 0) return cudaSuccess;
    const int threads = 256;
    const long long check_warps = p.num_inputs;
    tb_check_kernel<<<(unsigned)((check_warps * 32 + threads - 1) / threads), threads, 0, s>>>(p, tb_off, tb, nwords);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long cut_warps = (long long)p.num_inputs * ((p.W + 31) / 32);
    tb_cut_kernel<<<(unsigned)((cut_warps * 32 + threads - 1) / threads), threads, 0, s>>>(p, tb_off, tb, wstart);
    return cudaGetLastError();
}

}  // namespace gatspi
