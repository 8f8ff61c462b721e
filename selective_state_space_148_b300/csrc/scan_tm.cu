// scan_tm.cu -- instantiations and launch of the tensor-memory scan kernel, and
// the device error word it reports bounded-wait timeouts in.
#include "../../include/mamba_scan.h"
#include "internal.h"

namespace mamba {
__device__ unsigned int g_device_error = 0;
}  // namespace mamba

#include "scan_tm.cuh"

namespace mamba {

template <typename T, int MODE>
static cudaError_t launch_tm_one(const ScanArgs &a, long long Bsz, int grid_chunks, cudaStream_t st) {
    using Sh = TmShape<T, MODE>;
    auto kern = scan_tm_kernel<T, MODE>;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) attr_set[dev] = true;
    }
    dim3 grid((unsigned)((a.Dch + Sh::CH - 1) / Sh::CH), (unsigned)Bsz, (unsigned)grid_chunks);
    kern<<<grid, Sh::NTHR, Sh::SMEM_BYTES, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_scan_tm(int dtype, int mode, const ScanArgs &a, long long Bsz, int grid_chunks, cudaStream_t st) {
    if (dtype == 1)
        return mode == MODE_FULL ? launch_tm_one<bf16_t, MODE_FULL>(a, Bsz, grid_chunks, st)
                                 : launch_tm_one<bf16_t, MODE_STATES>(a, Bsz, grid_chunks, st);
    return mode == MODE_FULL ? launch_tm_one<float, MODE_FULL>(a, Bsz, grid_chunks, st)
                             : launch_tm_one<float, MODE_STATES>(a, Bsz, grid_chunks, st);
}

}  // namespace mamba

extern "C" int mamba_device_error(void) {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, mamba::g_device_error, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_DEVICE;
    }
    if (v != 0 && cudaMemcpyToSymbol(mamba::g_device_error, &zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_DEVICE;
    }
    return v != 0 ? MAMBA_ERR_DEVICE_TIMEOUT : MAMBA_OK;
}
