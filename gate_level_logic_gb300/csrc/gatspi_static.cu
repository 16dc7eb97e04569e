// Allocation-free entry point: one logic level re-simulated with caller-owned
// buffers only.
//
// Some callers cannot allocate device memory: code that runs inside a framework
// which owns the whole device memory through its own allocator, or code that is
// not allowed to allocate once it has started.  gatspi_create allocates the
// context's arrays; this entry point instead takes every input and output buffer
// from the caller (the level's plan included) and keeps the only scratch the
// level's kernels need -- the look-back flags of the output-region scan, its tile
// ticket and the status word -- in a file-scope device array of fixed size.  Every GPU that loads the library holds
// that array until the process exits.
#include <cstdio>
#include <mutex>

#include "gatspi_internal.cuh"

using namespace gatspi;

namespace {

constexpr int kStaticTiles = 1 << 13;                     // placement tiles (1024 gates each) of one level at most
constexpr int kTicketWord = kStaticTiles;                 // index of the ticket word
constexpr int kStatusWord = kStaticTiles + 1;             // index of the status words (2 x 8 bytes)
constexpr int kScratchWords = kStaticTiles + 4;

// Look-back flags, then the tile ticket, then the 4-int status word.  Shared by
// every call on a device; a call clears what it uses before its kernel runs.
static __device__ __align__(256) unsigned long long g_level_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

thread_local char g_msg[256];

}  // namespace

// Defined in gatspi.cu: routes a message to gatspi_last_error().
void gatspi_set_last_error(const char *msg);

extern "C" gatspi_status gatspi_simulate_level_static(const gatspi_level_args *a, void *stream) {
    auto err = [](gatspi_status s, const char *m) {
        gatspi_set_last_error(m);
        return s;
    };
    if (!a) return err(GATSPI_EINVAL, "args are required");
    if (!a->gate_desc || !a->dly_data || !a->window_len || !a->pool || !a->net_base ||
        !a->wstart || !a->wend || !a->wlen8 || !a->perm || !a->goff || !a->tc || !a->t1 || !a->level_base)
        return err(GATSPI_EINVAL, "every buffer of gatspi_level_args is required");
    if ((uintptr_t)a->gate_desc & 15) return err(GATSPI_EINVAL, "gate_desc must be 16-byte aligned");
    if ((uintptr_t)a->wlen8 & 3) return err(GATSPI_EINVAL, "wlen8 must be 4-byte aligned");
    if (a->num_inputs < 0 || a->num_windows < 1 || a->gate_begin < 0 || a->num_gates < 0 || a->pool_words < 0)
        return err(GATSPI_EINVAL, "negative sizes");
    if (a->num_windows > GATSPI_MAX_WINDOWS) return err(GATSPI_EINVAL, "too many windows");
    const bool own_percent = (a->flags & GATSPI_FLAG_PULSE_PERCENT) != 0;
    if (own_percent && (a->pulse_percent < 0 || a->pulse_percent > 100))
        return err(GATSPI_EINVAL, "pulse_percent must be 0 .. 100");

    DevParams p{};
    p.W = a->num_windows;
    p.ngroups = (p.W + 31) / 32;
    p.ngroups_m = 0xffffffffu / (uint32_t)p.ngroups;
    int lpg = 32;
    if (p.W < 32) {
        lpg = 1;
        while (lpg < p.W) lpg <<= 1;
    }
    p.lpg_log2 = 0;
    while ((1 << p.lpg_log2) < lpg) ++p.lpg_log2;
    p.slots_per_gate = p.ngroups << p.lpg_log2;
    const long long slots = (long long)a->num_gates * p.slots_per_gate;
    const long long tiles = slots > 0 ? (slots + kTileSlots - 1) / kTileSlots : 1;
    const long long scan = a->num_gates > 0 ? ((long long)a->num_gates + kPlaceTile - 1) / kPlaceTile : 1;
    if (scan > kStaticTiles)
        return err(GATSPI_EINVAL, "level too large for the static scratch (at most 8192 x 1024 gates)");
    if (tiles > INT32_MAX / kTileSlots) return err(GATSPI_EINVAL, "level has too many (gate, window) slots");

    // once per device, with that device current: the device address of the scratch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return err(GATSPI_ECUDA, "no current CUDA device");
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_scratch_addr[dev]) {
            void *ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&ptr, g_level_scratch);
            if (e != cudaSuccess || !ptr) {
                snprintf(g_msg, sizeof g_msg, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
                return err(GATSPI_ECUDA, g_msg);
            }
            g_scratch_addr[dev] = ptr;
        }
        scratch = g_scratch_addr[dev];
    }
    unsigned long long *words = (unsigned long long *)scratch;

    p.gate_desc = (const int4 *)a->gate_desc;
    p.dly_data = a->dly_data;
    p.pool = a->pool;
    p.pool_words = a->pool_words;
    p.net_base = (long long *)a->net_base;
    p.wstart = a->wstart;
    p.wend = a->wend;
    p.wlen8 = a->wlen8;
    p.w8stride = (a->num_windows + 3) & ~3;
    p.plan_words = plan_words(a->num_windows);
    p.perm = a->perm;
    p.goff = a->goff;
    p.window_len = a->window_len;
    p.tc = a->tc;
    p.t1 = a->t1;
    p.tile_status = words;
    p.tickets = (int32_t *)(words + kTicketWord);
    p.level_base = (long long *)a->level_base;
    p.status = (int32_t *)(words + kStatusWord);
    p.num_inputs = a->num_inputs;
    p.pulse_percent = own_percent ? a->pulse_percent : 100;
    p.ranked = windows_ranked(a->num_windows) ? 1 : 0;
    p.spin_limit_ns = kSpinLimitNs;

    LevelLaunch l{};
    l.level = 0;
    l.gate_begin = a->gate_begin;
    l.num_gates = a->num_gates;
    l.num_tiles = (int32_t)tiles;
    l.scan_tiles = (int32_t)scan;
    l.tile_base = 0;

    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = set_level_smem_limit();
    // clear the flags of the tiles this call uses, the ticket and the status
    if (e == cudaSuccess) e = cudaMemsetAsync(words, 0, sizeof(unsigned long long) * (size_t)scan, s);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(words + kTicketWord, 0, sizeof(unsigned long long) * (kScratchWords - kTicketWord), s);
    if (e == cudaSuccess) e = launch_level(p, l, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        snprintf(g_msg, sizeof g_msg, "level kernel: %s", cudaGetErrorString(e));
        return err(GATSPI_ECUDA, g_msg);
    }
    int32_t st[kStatusWords] = {0, 0, 0, 0};
    e = cudaMemcpy(st, words + kStatusWord, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return err(GATSPI_ECUDA, "reading the status word");
    if (st[0] != GATSPI_OK) {
        snprintf(g_msg, sizeof g_msg, "device error %d (detail %d, %d, %d)", st[0], st[1], st[2], st[3]);
        return err((gatspi_status)st[0], g_msg);
    }
    gatspi_set_last_error("");
    return GATSPI_OK;
}
