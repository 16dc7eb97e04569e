// Device-side testbench restructuring (testbench.cu).
#pragma once

#include "gatspi_internal.cuh"

namespace gatspi {

// Check the whole-testbench waveforms (tb_off[num_inputs + 1] over tb, nwords words,
// device memory) and cut them into the windows starting at wstart[0 .. W] (int64,
// wstart[W] = end of the last window): writes every input's windows into the pool,
// the window index of the inputs and level_base[0].  A malformed waveform sets the
// status word (GATSPI_EBADWAVE, input) and nothing is written.
cudaError_t launch_testbench_cut(const DevParams &p, const long long *tb_off, const int32_t *tb, long long nwords,
                                 const long long *wstart, cudaStream_t s);

// Toggle count and time at 1 (within each window) of every input, summed over its
// windows, from the loaded inputs' window index: tc[num_inputs], t1[num_inputs].
cudaError_t launch_input_stats(const DevParams &p, unsigned long long *tc, unsigned long long *t1, cudaStream_t s);

}  // namespace gatspi
