// scan_tm_ckpt.cu -- the tensor-memory scan kernel instantiated for the plain direct scan that also writes
// the backward pass's checkpoints (mamba_selective_scan_fwd_save).  Compiled apart from the plain
// instantiations (scan_tm.cu) so that those carry no checkpoint code; its bounded-wait timeouts go to
// the device error word of this file.
#include <cuda.h>

#include "../../include/mamba_scan.h"
#include "internal.h"

namespace mamba {
static __device__ unsigned int g_device_error = 0;
}  // namespace mamba

#include "scan_tm.cuh"

namespace mamba {

cudaError_t launch_tm_ckpt(int dtype, int S, const ScanArgs &a, const TmMaps &maps, int warps, bool lean,
                           long long Bsz, cudaStream_t st) {
    if (dtype != 1) {
        return a.z != nullptr ? launch_tm_one<float, MODE_FULL, true, 4, false, FL_CKPT>(a, maps, warps, Bsz, 1, st)
                              : launch_tm_one<float, MODE_FULL, false, 4, false, FL_CKPT>(a, maps, warps, Bsz, 1, st);
    }
    if (lean) {
        switch (S) {
            case 4: return launch_tm_lean<4, FL_CKPT>(a, maps, warps, Bsz, st);
            case 8: return launch_tm_lean<8, FL_CKPT>(a, maps, warps, Bsz, st);
            default: return launch_tm_lean<16, FL_CKPT>(a, maps, warps, Bsz, st);
        }
    }
    switch (S) {
        case 4:
            return a.z != nullptr ? launch_tm_one<bf16_t, MODE_FULL, true, 4, false, FL_CKPT>(a, maps, warps, Bsz, 1, st)
                                  : launch_tm_one<bf16_t, MODE_FULL, false, 4, false, FL_CKPT>(a, maps, warps, Bsz, 1, st);
        case 8:
            return a.z != nullptr ? launch_tm_one<bf16_t, MODE_FULL, true, 8, false, FL_CKPT>(a, maps, warps, Bsz, 1, st)
                                  : launch_tm_one<bf16_t, MODE_FULL, false, 8, false, FL_CKPT>(a, maps, warps, Bsz, 1, st);
        default:
            return a.z != nullptr ? launch_tm_one<bf16_t, MODE_FULL, true, 16, false, FL_CKPT>(a, maps, warps, Bsz, 1, st)
                                  : launch_tm_one<bf16_t, MODE_FULL, false, 16, false, FL_CKPT>(a, maps, warps, Bsz, 1, st);
    }
}

int tm_ckpt_read_clear_error(unsigned int *v) { return read_clear_word(g_device_error, v); }

}  // namespace mamba
