// scan_tm_rev.cu -- the tensor-memory scan kernel instantiated for the reverse-time scan (MAMBA_FLAG_REVERSE:
// t = L-1 .. 0, the reverse SSM of the fsdata.site explainer §7 table).
// Compiled apart from the plain instantiations (scan_tm.cu) so that the files
// compile in parallel and the plain kernels carry no flag code; its
// bounded-wait timeouts go to the device error word of this file.
#include <cuda.h>

#include "../../include/mamba_scan.h"
#include "internal.h"

namespace mamba {
static __device__ unsigned int g_device_error = 0;
}  // namespace mamba

#include "scan_tm.cuh"

namespace mamba {

cudaError_t launch_tm_rev(int dtype, int S, int mode, const ScanArgs &a, const TmMaps &maps, int warps,
                          long long Bsz, int gc, cudaStream_t st) {
    return launch_tm_variant<FL_REV>(dtype, S, mode, a, maps, warps, Bsz, gc, st);
}

int tm_rev_read_clear_error(unsigned int *v) { return read_clear_word(g_device_error, v); }

}  // namespace mamba
