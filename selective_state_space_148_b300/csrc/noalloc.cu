// noalloc.cu -- chunked selective scan that allocates no device memory.
//
// The chunked scan needs scratch for the per-chunk end states and step sums.
// mamba_selective_scan_fwd / _ex either take it from the caller or allocate it
// stream-ordered.  Some callers can do neither: a framework that hands the
// library only the tensors of one call and owns every other byte of device
// memory, or host code running where device allocation is not allowed (a
// real-time loop with a fixed memory budget, or any caller that must not
// synchronise with the allocator).  This entry point serves them: its scratch
// is one file-scope __device__ array, created with the module on every GPU that
// loads the library and kept until the process exits.
#include <atomic>

#include "../../include/mamba_scan.h"
#include "internal.h"

using namespace mamba;

namespace {

constexpr size_t kScratchBytes = MAMBA_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  In host code `g_scratch` names a host-side stand-in,
// not a device address: only the address returned by cudaGetSymbolAddress on
// the current device may be handed to a kernel.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::atomic<void *> g_scratch_addr[kMaxDevices];

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Device address of g_scratch on the current device, looked up once per device.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return MAMBA_ERR_DEVICE;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MAMBA_ERR_DEVICE;
        }
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return MAMBA_OK;
}

}  // namespace

extern "C" int mamba_selective_scan_fwd_noalloc(const void *u, const void *delta, const float *A, const void *B,
                                                const void *C, const float *D, const void *z,
                                                const float *delta_bias, int softplus_flag, void *y,
                                                float *last_state, const float *h0, int64_t Bsz, int64_t Dch,
                                                int64_t L, int64_t N, int dtype, int64_t chunk_len,
                                                mamba_stream_t stream) {
    if (!u || !delta || !A || !B || !C || !y) return MAMBA_ERR_NULL_ARG;
    if (dtype != MAMBA_F32 && dtype != MAMBA_BF16) return MAMBA_ERR_BAD_DTYPE;
    if (Bsz <= 0 || Dch <= 0 || L <= 0 || N <= 0 || chunk_len <= 0) return MAMBA_ERR_BAD_SHAPE;
    if (N > 64) return MAMBA_ERR_UNSUPPORTED_N;
    constexpr int64_t kMax = 1LL << 40;
    if (Bsz > 65535 || Dch > kMax || L > kMax || Bsz * Dch > kMax / L || Bsz * Dch > kMax / N ||
        Bsz * N > kMax / L)
        return MAMBA_ERR_BAD_SHAPE;

    const ScanGeom g = scan_geom(N);
    const int64_t cl = (chunk_len + g.TT - 1) / g.TT * g.TT;  // chunk starts on tile boundaries
    const int64_t K = (L + cl - 1) / cl;
    if (K > 65535) return MAMBA_ERR_BAD_SHAPE;
    const size_t h_bytes = round_up256((size_t)Bsz * K * Dch * N * sizeof(float));
    const size_t s_bytes = round_up256((size_t)Bsz * K * Dch * sizeof(float));
    if (K > 1 && h_bytes + s_bytes > kScratchBytes) return MAMBA_ERR_SCRATCH_LIMIT;

    const bool vec = ((reinterpret_cast<uintptr_t>(u) | reinterpret_cast<uintptr_t>(delta) |
                       reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C) |
                       reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(z)) & 15u) == 0 &&
                     (L * (dtype == MAMBA_BF16 ? 2 : 4)) % 16 == 0;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    ScanArgs a{};
    a.u = u;
    a.delta = delta;
    a.z = z;
    a.Bm = B;
    a.Cm = C;
    a.A = A;
    a.D = D;
    a.bias = delta_bias;
    a.y = y;
    a.last_state = last_state;
    a.Dch = Dch;
    a.L = L;
    a.N = N;
    a.softplus = softplus_flag ? 1 : 0;

    if (K == 1) {  // one chunk covers the sequence: the direct scan, no scratch
        a.hin = h0;
        a.chunk_len = L;
        a.nchunks = 1;
        return launch_scan(dtype, MODE_FULL, vec, a, Bsz, 1, st) == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
    }

    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != MAMBA_OK) return rc;
    // The first pass writes every chunk end state and step sum it covers before
    // the carry reads them, and the carry writes every chunk's initial state
    // before the last pass reads it, so the stale contents of earlier calls are
    // never read.
    float *ws_h = reinterpret_cast<float *>(scratch);
    float *ws_sdt = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(scratch) + h_bytes);
    a.chunk_len = cl;
    a.nchunks = (int)K;
    return run_chunked(dtype, vec, a, Bsz, ws_h, ws_sdt, h0, st) == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}
