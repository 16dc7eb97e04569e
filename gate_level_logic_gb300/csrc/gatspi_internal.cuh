// Internal declarations shared by the host code (gatspi.cu) and the level kernel
// (level_kernel.cu) of the GB300 gate-level re-simulator.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gatspi.h"

namespace gatspi {

constexpr int kBlock = 256;               // threads per block of the light kernels
constexpr int kWarps = kBlock / 32;
constexpr int kPlaceTile = 1024;          // gates per block (and look-back tile) of the placement scan
#ifndef GATSPI_LEVEL_WARPS
#define GATSPI_LEVEL_WARPS 4
#endif
#ifndef GATSPI_LEVEL_MIN_BLOCKS
#define GATSPI_LEVEL_MIN_BLOCKS (36 / GATSPI_LEVEL_WARPS)
#endif
constexpr int kLevelWarps = GATSPI_LEVEL_WARPS;   // warps per level-kernel block (independent warps)
constexpr int kLevelBlock = 32 * kLevelWarps;
constexpr int kLevelMinBlocks = GATSPI_LEVEL_MIN_BLOCKS;  // resident blocks per SM the registers must allow
constexpr int kTileSlots = 32;            // (gate, rank) slots per warp of the level kernel
constexpr int kPlanWarps = 4;             // warps per block of the planning kernel (one gate each)
constexpr int kPlanMinBlocks = 12;        // planning blocks per SM the registers must allow (40 registers)
constexpr int kSortBuckets = 256;         // counting-sort buckets of the window bounds
// Up to this many windows a gate's windows are ranked by bound for the simulation
// warps (load balance); beyond it the windows are short (few cycles each), set-up
// dominates and they are taken in window order, with no plan of ranks.
constexpr int kRankMaxWindows = 1024;
inline bool windows_ranked(int W) { return W <= kRankMaxWindows; }
constexpr int32_t kEOW = GATSPI_EOW;
constexpr int32_t kNoArc = GATSPI_NO_ARC;

// Look-back status words: flag in the top two bits, inclusive/aggregate value below.
constexpr unsigned long long kFlagAgg = 1ull << 62;
constexpr unsigned long long kFlagIncl = 2ull << 62;
constexpr unsigned long long kValueMask = (1ull << 62) - 1;
constexpr unsigned long long kSpinLimitNs = 2000000000ull;   // default: 2 s without progress -> ETIMEOUT

// Device status word: [0] first error code, [1..3] details (gate / net, window, extra).
constexpr int kStatusWords = 4;

// Everything a level kernel reads or writes, by value in the kernel parameters.
struct DevParams {
    // netlist
    const int4 *gate_desc;     // [3G] per gate: {0, n | truth table << 8, delay-table offset lo/hi},
                               //     {source net of pin 0..3}, {wire rise | fall << 16 of pin 0..3};
                               //     truth-table bit k = output for pin values k (first pin most significant)
    const int32_t *dly_data;   // per-instance conditional delay tables
    int32_t *heavy_order;      // [gates of the level]: level_chunk_kernel's gate order, heaviest first
    // one window cut into time chunks: a heavy gate's window split into segments, one
    // warp each (null unless W = 1)
    uint32_t *seg_items;       // [gates of the level + kExtraSegments]: gate | segment << 24 | (segments - 1) << 28
    uint32_t *seg_count;       // [1]: items of the level
    uint32_t *seg_cnt;         // [gates of the level * kMaxSegments]: entries of every segment (bit 31: y0)
    int32_t *seg_counter;      // [gates of the level]: segments finished (reset by the last)
    int32_t resident_warps;    // warps the GPU holds at once in level_chunk_kernel
    int32_t seg_kernel;        // level_chunk_kernel<true> (segments possible) instead of <false>
    const int32_t *gate_order; // [G] or null: with W < 32 (several gates per warp) the gates of every
                               //     level in the order the simulation kernel takes them, by pin count
    // waveform store: waveform (net, w) is pool[net_base[net] + wstart[k] .. net_base[net] + wend[k]),
    // k = net * W + w, EOW included
    int32_t *pool;
    long long pool_words;
    long long *net_base;       // [num_nets] first pool word of the net's region
    uint32_t *wstart;          // [num_nets * W] relative to net_base
    uint32_t *wend;            // [num_nets * W] relative to net_base
    uint8_t *wlen8;            // [num_nets * w8stride] min(window length, 255), for the plan
    const int32_t *window_len; // [W]
    // the level's plan: per gate, its windows by rank (largest output bound first) and
    // the offset of every group of 32 ranks inside the gate's region
    uint16_t *perm;            // [gates of the level * W] (ranked windows only)
    uint32_t *goff;            // [gates of the level * (ngroups + 1)]: group offsets, then the region's size
    // toggle statistics
    unsigned long long *tc;    // [G]
    unsigned long long *t1;    // [G]
    // scan state
    unsigned long long *tile_status;  // [total look-back tiles: kPlaceTile gates each], zeroed per simulate
    int32_t *tickets;                 // [L], zeroed per simulate
    long long *level_base;            // [L+1]; [0] = words of the input waveforms
    int32_t *status;                  // [kStatusWords]
    // shape
    int32_t num_inputs;
    int32_t W;
    int32_t w8stride;         // W rounded up to a multiple of 4 (rows of wlen8 start 4-byte aligned)
    int32_t plan_words;       // shared words per warp of the planning kernel (plan_words(W))
    int32_t ngroups;          // ceil(W / 32): groups of 32 ranks per gate
    uint32_t ngroups_m;       // floor((2^32 - 1) / ngroups): tile / ngroups by a multiply-high
    int32_t lpg_log2;         // log2(lanes per (gate, group) segment)
    int32_t slots_per_gate;   // ngroups << lpg_log2
    int32_t pulse_percent;    // PATHPULSEPERCENT, 0 .. 100
    int32_t ranked;           // windows_ranked(W): perm holds the ranks; else rank = window
    int32_t chunks;           // > 1: lanes per window of level_chunk_kernel (W <= 16); else 0
    // compaction (GATSPI_FLAG_COMPACT): every level is simulated into bound-sized regions
    // placed down from the top of the pool, then packed to exact size at the front
    int32_t compact;
    uint32_t *gexact;         // [gates of the level * ngroups] output words of every (gate, group)
    long long *old_base;      // [gates of the level] the gate's bound-sized region before packing
    long long *level_bound;   // [L] words of the level's bound-sized regions
    long long *level_need;    // [L] pool words the level needed: packed front + its bound-sized regions
    unsigned long long spin_limit_ns;   // how long a look-back wait may see no progress before ETIMEOUT
};

struct LevelLaunch {
    int32_t level;
    int32_t gate_begin;
    int32_t num_gates;
    int32_t num_tiles;      // warps of the level kernel: ceil(gates * slots_per_gate / 32)
    int32_t scan_tiles;     // blocks of the placement scan: max(1, ceil(gates / kPlaceTile))
    long long tile_base;    // first look-back word of this level's scan
    int32_t ticket;         // this scan's tile ticket (level, or L + level for the exact scan)
};

int plan_words(int W);
// Lanes per window of level_chunk_kernel: 32 / W with 16 windows or fewer, at any
// PATHPULSEPERCENT, when the windows are long (the loaded inputs average
// kLongWindowWords words or more per (input, window): shorter windows lose more to
// finding cuts and moving the chunks together than they gain), or always with
// GATSPI_FLAG_CUT_WINDOWS; never with GATSPI_FLAG_WHOLE_WINDOWS.  0: every window in
// one lane.
constexpr long long kLongWindowWords = 32;
constexpr int kMaxSegments = 8;        // warps one gate's window may take (one window)
constexpr int kExtraSegments = 4096;   // segments beyond one per gate, per level
constexpr unsigned long long kSegmentMinWords = 16384;  // bound words a segment needs at least
// One window is split into segments (several warps per heavy gate) when the loaded
// inputs average this many words or more per input, or whenever windows are cut by
// GATSPI_FLAG_CUT_WINDOWS; shorter windows gain less than the segment code costs.
constexpr long long kSplitWindowWords = 4096;
// From this many words per input window on, cut windows of 2 .. 16 run faster in the
// segment-capable instantiation of level_chunk_kernel (measured; nothing is split).
constexpr long long kDenseWindowWords = 100;
inline int chunks_per_window(int W, uint32_t flags, bool long_windows) {
    const bool cut = (flags & GATSPI_FLAG_CUT_WINDOWS) || (long_windows && !(flags & GATSPI_FLAG_WHOLE_WINDOWS));
    return W >= 1 && W <= 16 && cut ? 32 / W : 0;
}
size_t plan_smem_bytes(int W);
int plan_gates_per_tile(int W);   // gates (warps) of one planning block
cudaError_t set_level_smem_limit();
// chunk_kernel.cu: the level's simulation with windows cut into time chunks
// (DevParams::chunks > 1), and its kernels' shared-memory configuration.
cudaError_t launch_level_chunks(const DevParams &p, const LevelLaunch &l, cudaStream_t s);
cudaError_t set_chunk_smem_limit();   // the planning kernel's shared memory (largest W), the simulation kernels' L1
cudaError_t launch_level_bounds(const DevParams &p, const LevelLaunch &l, cudaStream_t s);   // plan + placement
cudaError_t launch_level_sim(const DevParams &p, const LevelLaunch &l, cudaStream_t s);      // the simulation
cudaError_t launch_level_compact(const DevParams &p, const LevelLaunch &l, const LevelLaunch &exact,
                                 cudaStream_t s);  // compaction: exact scan + packing copy
cudaError_t launch_level(const DevParams &p, const LevelLaunch &l, cudaStream_t s);          // both, in order
cudaError_t launch_window_lengths(const DevParams &p, long long num_nets, const int32_t *sel, int nsel,
                                  long long *len, cudaStream_t s);
cudaError_t launch_window_gather(const DevParams &p, long long num_nets, const int32_t *sel, int nsel,
                                 const long long *off, int32_t *words, cudaStream_t s);
cudaError_t launch_net_digests(const DevParams &p, long long net0, long long n, unsigned long long *out,
                               long long *words, cudaStream_t s);
cudaError_t launch_load_index(const DevParams &p, const long long *off, long long nwords, int32_t *max_time,
                              cudaStream_t s);

}  // namespace gatspi
