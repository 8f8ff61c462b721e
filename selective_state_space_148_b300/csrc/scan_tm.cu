// scan_tm.cu -- instantiations and launch of the tensor-memory scan kernel
// (TMA descriptors, launch geometry), and the device error word its
// instantiations here report bounded-wait timeouts in (the instantiations that
// honour the scan flags live in scan_tm_rev.cu and scan_tm_zoh.cu, with words of
// their own).
#include <cstdlib>

#include <cuda.h>

#include "../../include/mamba_scan.h"
#include "internal.h"

namespace mamba {
static __device__ unsigned int g_device_error = 0;
}  // namespace mamba

#include "scan_tm.cuh"

namespace mamba {

long long tm_launch_cost(long long Bsz, long long Dch, int grid_chunks, int sms, int S, int *warps) {
    using Sh = TmShape<float, MODE_FULL>;
    int best = Sh::MAX_WARPS;
    long long best_cost = -1;
    for (int w = Sh::MIN_WARPS; w <= Sh::MAX_WARPS; ++w) {
        const long long cw = 32LL * w / S;  // channels per CTA
        const long long ctas = Bsz * ((Dch + cw - 1) / cw) * grid_chunks;
        const long long waves = sms > 0 ? (ctas + sms - 1) / sms : 1;
        const long long cost = waves * ((w + 1 + 3) / 4);  // + the producer warp, over 4 sub-partitions
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = w;
        }
    }
    if (warps != nullptr) *warps = best;
    return best_cost;
}

namespace {

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point so
// that the library does not link the driver library itself
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<EncodeTiledFn>(nullptr);
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// [outer][mid][inner] tensor, box of box_inner x box_mid x 1 elements
bool encode_3d(CUtensorMap *m, const void *ptr, bool bf16, long long inner, long long mid, long long outer,
               unsigned box_mid, bool swizzle, unsigned box_inner = 32) {
    const EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t es = bf16 ? 2 : 4;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)mid, (cuuint64_t)outer};
    const cuuint64_t strides[2] = {(cuuint64_t)inner * es, (cuuint64_t)inner * (cuuint64_t)mid * es};
    const cuuint32_t box[3] = {box_inner, box_mid, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapSwizzle sw =
        !swizzle ? CU_TENSOR_MAP_SWIZZLE_NONE : (bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(ptr),
              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sms() {
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

// CTA width in warps (32 / S channels each): the one tm_launch_cost picks.
int choose_warps(long long Bsz, long long Dch, int grid_chunks, int sms, int S) {
    int w = 0;
    tm_launch_cost(Bsz, Dch, grid_chunks, sms, S, &w);
    return w;
}

long long waves_of(long long Bsz, long long Dch, int sms, int S, int w) {
    const long long cw = 32LL * w / S;
    const long long ctas = Bsz * ((Dch + cw - 1) / cw);
    return sms > 0 ? (ctas + sms - 1) / sms : 1;
}

// The lean form (12..18 compute warps, fewer registers per thread) of a direct scan: the narrowest
// width with the fewest waves, taken when that is fewer waves than the regular width needs (its
// channels then run with more warps per SM sub-partition).  MAMBA_TM_LEAN=0 / 1 (read on every call)
// never / always takes it.  Returns 0 for the regular form.
int choose_lean_warps(long long Bsz, long long Dch, int sms, int S, int regular_warps) {
    using Sh = TmShape<bf16_t, MODE_FULL, 4, false, true>;
    const char *v = std::getenv("MAMBA_TM_LEAN");
    if (v != nullptr && v[0] == '0' && v[1] == '\0') return 0;
    const bool force = v != nullptr && v[0] == '1' && v[1] == '\0';
    int best = 0;
    long long best_waves = force ? (1LL << 62) : waves_of(Bsz, Dch, sms, S, regular_warps);
    for (int w = Sh::MIN_WARPS; w <= Sh::MAX_WARPS; ++w) {
        const long long wv = waves_of(Bsz, Dch, sms, S, w);
        if (wv < best_waves) {
            best_waves = wv;
            best = w;
        }
    }
    return best;
}

}  // namespace

// The kernel's pipeline waits are bounded by time (about a second); MAMBA_TEST_WAIT_POLLS=0, a host-side
// test hook, makes them give up after one test so that the abort path and the device error word can be
// exercised without any fault.  Any other value keeps the normal bound.
static unsigned pipeline_wait_polls() {
    const char *v = std::getenv("MAMBA_TEST_WAIT_POLLS");
    if (v == nullptr || *v == '\0') return 1u << 24;
    char *end = nullptr;
    const unsigned long n = std::strtoul(v, &end, 10);
    return (end != nullptr && *end == '\0' && n < (1ul << 24)) ? (unsigned)n : (1u << 24);
}

cudaError_t launch_scan_tm(int dtype, int mode, const ScanArgs &args, long long Bsz, int grid_chunks,
                           cudaStream_t st) {
    ScanArgs a = args;
    a.wait_polls = pipeline_wait_polls();
    // TMA coordinates are 32-bit: the time axis and the channel axis must fit
    if (a.L >= (1LL << 31) - 64 || a.Dch >= (1LL << 31) - 128 || Bsz >= (1LL << 31)) return cudaErrorNotSupported;
    const bool bf16 = dtype == 1;
    // lanes per channel: each lane owns 4 states; fp32 B/C (three bf16 parts per
    // value) fit the selector's K = 16 for 4 lanes only
    const int S = a.N <= 16 ? 4 : a.N <= 32 ? 8 : 16;
    if (a.N > 64 || (!bf16 && S != 4)) return cudaErrorNotSupported;
    // the convolution-fed variant is built for bf16, N <= 16, with the gate
    const bool conv = a.conv_w != nullptr;
    if (conv && (!bf16 || S != 4 || (mode == MODE_FULL && a.z == nullptr))) return cudaErrorNotSupported;
    int warps = choose_warps(Bsz, a.Dch, grid_chunks, device_sms(), S);
    // the plain direct bf16 scan may take the lean form (more warps per CTA)
    const int lean_warps = (bf16 && !conv && mode == MODE_FULL && a.flags == 0 && grid_chunks == 1)
                               ? choose_lean_warps(Bsz, a.Dch, device_sms(), S, warps)
                               : 0;
    if (lean_warps > 0) warps = lean_warps;
    const unsigned ch = 32u * (unsigned)warps / (unsigned)S;
    TmMaps maps;
    const bool ok = (conv ? encode_3d(&maps.u, a.u, bf16, a.L, a.Dch, Bsz, ch, false, TmShape<bf16_t, MODE_FULL, 4, true>::XSTEPS)
                          : encode_3d(&maps.u, a.u, bf16, a.L, a.Dch, Bsz, ch, true)) &&
                    encode_3d(&maps.delta, a.delta, bf16, a.L, a.Dch, Bsz, ch, true) &&
                    encode_3d(&maps.z, a.z != nullptr ? a.z : a.u, bf16, a.L, a.Dch, Bsz, ch, true) &&
                    encode_3d(&maps.B, a.Bm, bf16, a.L, a.N, Bsz, 4u * S, false) &&
                    encode_3d(&maps.C, a.Cm, bf16, a.L, a.N, Bsz, 4u * S, false);
    if (!ok) return cudaErrorNotSupported;
    if (a.ckpt != nullptr) {  // the direct scan that also writes the backward's checkpoints
        if (mode != MODE_FULL || grid_chunks != 1 || conv || a.flags != 0) return cudaErrorNotSupported;
        return launch_tm_ckpt(dtype, S, a, maps, warps, lean_warps > 0, Bsz, st);
    }
    if (mode == MODE_FULL_STATES || mode == MODE_CORR) {
        if (conv || a.flags != 0) return cudaErrorNotSupported;
        return launch_tm_chunk(dtype, S, mode, a, maps, warps, Bsz, grid_chunks, st);
    }
    if (a.flags & SCAN_FLAG_ZOH) return launch_tm_zoh(dtype, S, mode, a, maps, warps, Bsz, grid_chunks, st);
    if (a.flags & SCAN_FLAG_REVERSE) return launch_tm_rev(dtype, S, mode, a, maps, warps, Bsz, grid_chunks, st);
    if (conv)
        return mode == MODE_STATES
                   ? launch_tm_one<bf16_t, MODE_STATES, false, 4, true>(a, maps, warps, Bsz, grid_chunks, st)
                   : launch_tm_one<bf16_t, MODE_FULL, true, 4, true>(a, maps, warps, Bsz, grid_chunks, st);
    if (!bf16) return launch_tm_s<float, 4>(mode, a, maps, warps, Bsz, grid_chunks, st);
    if (lean_warps > 0) {
        switch (S) {
            case 4: return launch_tm_lean<4>(a, maps, warps, Bsz, st);
            case 8: return launch_tm_lean<8>(a, maps, warps, Bsz, st);
            default: return launch_tm_lean<16>(a, maps, warps, Bsz, st);
        }
    }
    switch (S) {
        case 4: return launch_tm_s<bf16_t, 4>(mode, a, maps, warps, Bsz, grid_chunks, st);
        case 8: return launch_tm_s<bf16_t, 8>(mode, a, maps, warps, Bsz, grid_chunks, st);
        default: return launch_tm_s<bf16_t, 16>(mode, a, maps, warps, Bsz, grid_chunks, st);
    }
}

}  // namespace mamba

namespace mamba {
int tm_read_clear_error(unsigned int *v) { return read_clear_word(g_device_error, v); }
int tm_ckpt_read_clear_error(unsigned int *v);  // scan_tm_ckpt.cu
}  // namespace mamba

extern "C" int mamba_device_error(void) {
    unsigned int v = 0, r = 0, z = 0, c = 0, k = 0;
    if (mamba::tm_read_clear_error(&v) != MAMBA_OK || mamba::tm_rev_read_clear_error(&r) != MAMBA_OK ||
        mamba::tm_zoh_read_clear_error(&z) != MAMBA_OK || mamba::tm_chunk_read_clear_error(&c) != MAMBA_OK ||
        mamba::tm_ckpt_read_clear_error(&k) != MAMBA_OK)
        return MAMBA_ERR_DEVICE;
    return (v | r | z | c | k) != 0 ? MAMBA_ERR_DEVICE_TIMEOUT : MAMBA_OK;
}
