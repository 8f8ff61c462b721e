// scan_tm_chunk.cu -- the tensor-memory scan kernel instantiated for the two
// passes of the decay-truncated chunked scan (long sequences; freeguideonline
// tutorial §5.1, the recurrence as a scan of composable step transforms, and
// the chunking of long sequences in mlqm.cn §6.2): MODE_FULL_STATES, y of every
// chunk from a zero state together with the chunk's end state and sum of
// Delta, and MODE_CORR, which adds to y the contribution of the state a chunk
// actually enters with (the carry of the end states), decaying step by step
// with no input, and stops where that contribution has decayed below fp32
// resolution.  Its bounded-wait timeouts go to the device error word of this
// file.
#include <cuda.h>

#include "../../include/mamba_scan.h"
#include "internal.h"

namespace mamba {
static __device__ unsigned int g_device_error = 0;
}  // namespace mamba

#include "scan_tm.cuh"

namespace mamba {

template <typename T, int S>
static cudaError_t launch_chunk_s(int mode, const ScanArgs &a, const TmMaps &maps, int warps, long long Bsz, int gc,
                                  cudaStream_t st) {
    if (mode == MODE_FULL_STATES)
        return a.z != nullptr ? launch_tm_one<T, MODE_FULL_STATES, true, S>(a, maps, warps, Bsz, gc, st)
                              : launch_tm_one<T, MODE_FULL_STATES, false, S>(a, maps, warps, Bsz, gc, st);
    return a.z != nullptr ? launch_tm_one<T, MODE_CORR, true, S>(a, maps, warps, Bsz, gc, st)
                          : launch_tm_one<T, MODE_CORR, false, S>(a, maps, warps, Bsz, gc, st);
}

cudaError_t launch_tm_chunk(int dtype, int S, int mode, const ScanArgs &a, const TmMaps &maps, int warps,
                            long long Bsz, int gc, cudaStream_t st) {
    if (dtype != 1) return launch_chunk_s<float, 4>(mode, a, maps, warps, Bsz, gc, st);
    switch (S) {
        case 4: return launch_chunk_s<bf16_t, 4>(mode, a, maps, warps, Bsz, gc, st);
        case 8: return launch_chunk_s<bf16_t, 8>(mode, a, maps, warps, Bsz, gc, st);
        default: return launch_chunk_s<bf16_t, 16>(mode, a, maps, warps, Bsz, gc, st);
    }
}

int tm_chunk_read_clear_error(unsigned int *v) { return read_clear_word(g_device_error, v); }

}  // namespace mamba
