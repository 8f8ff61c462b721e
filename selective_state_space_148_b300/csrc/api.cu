// api.cu -- the C ABI (include/mamba_scan.h): argument validation, choice
// between the direct and the chunked scan, stream-ordered workspace, and
// mapping of CUDA errors to status codes.  No C++ exception leaves this file.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "../../include/mamba_scan.h"
#include "internal.h"

using namespace mamba;

namespace {

constexpr long long kMaxDim = 1LL << 40;  // sizes beyond this are rejected (index overflow guard)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int io_bytes(int dtype) { return dtype == MAMBA_BF16 ? 2 : 4; }

// Host-side fault injection for tests: MAMBA_FAULT_INJECT=alloc makes the
// workspace allocation report failure without calling the allocator.
bool inject_alloc_failure() {
    const char *v = std::getenv("MAMBA_FAULT_INJECT");
    return v != nullptr && std::strcmp(v, "alloc") == 0;
}

bool u_ok_args(const void *delta, const float *A, const void *B, const void *C, const void *y) {
    return delta && A && B && C && y;
}

int sm_count(int *out) {
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_DEVICE;
    }
    if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) {
        *out = cache[dev];
        return MAMBA_OK;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return MAMBA_ERR_DEVICE;
    }
    if (dev >= 0 && dev < kMaxDevices) cache[dev] = n;
    *out = n;
    return MAMBA_OK;
}

int check_sizes(long long Bsz, long long Dch, long long L, long long N, int dtype) {
    if (dtype != MAMBA_F32 && dtype != MAMBA_BF16) return MAMBA_ERR_BAD_DTYPE;
    if (Bsz <= 0 || Dch <= 0 || L <= 0 || N <= 0) return MAMBA_ERR_BAD_SHAPE;
    if (N > 64) return MAMBA_ERR_UNSUPPORTED_N;
    if (Bsz > 65535) return MAMBA_ERR_BAD_SHAPE;  // batch is the grid's y dimension
    if (Bsz > kMaxDim || Dch > kMaxDim || L > kMaxDim) return MAMBA_ERR_BAD_SHAPE;
    if (Bsz * Dch > kMaxDim || (Bsz * Dch) > kMaxDim / L || (Bsz * Dch) > kMaxDim / N) return MAMBA_ERR_BAD_SHAPE;
    if (Bsz * N > kMaxDim / L) return MAMBA_ERR_BAD_SHAPE;
    return MAMBA_OK;
}

// Chunk plan: chunk_len steps per chunk, K chunks (K == 1: direct scan).
struct Plan {
    long long chunk_len;
    int K;
};

int make_plan(long long Bsz, long long Dch, long long L, long long N, int dtype, long long chunk_len_req, Plan *plan) {
    const ScanGeom g = scan_geom(N);
    if (chunk_len_req < 0) {
        *plan = Plan{L, 1};
        return MAMBA_OK;
    }
    long long cl = 0;
    if (chunk_len_req > 0) {
        cl = chunk_len_req;
    } else {
        // Automatic: the direct scan keeps Bsz*Dch*S lanes busy.  When that is
        // well under what the GPU holds and the sequence is long, cut the time
        // axis into chunks; the chunked scan pays a second exp pass, so only
        // do it when the direct scan would leave most of the GPU idle.
        int sms = 0;
        const int st = sm_count(&sms);
        if (st != MAMBA_OK) return st;
        if (tm_kernel_for(dtype, N) && L >= 16LL * g.TT) {
            // The tensor-memory kernel runs one CTA per SM: a launch costs whole waves.  The chunked
            // scan runs K - 1 chunks (end states) and then K chunks (outputs), each pass costing its
            // waves times the chunk length; take the K (narrower chunks only when strictly cheaper)
            // that minimises (cost(K - 1) + cost(K)) * chunk_len, against cost(1) * L for the direct scan.
            // Narrower chunks must be at least 3 % cheaper: long chunks pay fewer CTA set-ups, and the
            // correction pass of the decay-truncated scan stops at a fixed number of steps, a smaller
            // share of a long chunk.
            const int S = N <= 16 ? 4 : N <= 32 ? 8 : 16;
            double best = (double)tm_launch_cost(Bsz, Dch, 1, sms, S, nullptr) * (double)L;
            long long best_cl = L;
            const long long kmax = std::min<long long>(L / (8LL * g.TT), 1024);  // chunks of at least 8 tiles
            for (long long K = 2; K <= kmax; ++K) {
                const long long c = ((L + K - 1) / K + g.TT - 1) / g.TT * g.TT;
                const long long Kr = (L + c - 1) / c;
                if (Kr < 2) continue;
                const double t = (double)(tm_launch_cost(Bsz, Dch, (int)(Kr - 1), sms, S, nullptr) +
                                          tm_launch_cost(Bsz, Dch, (int)Kr, sms, S, nullptr)) * (double)c;
                if (t < best * (best_cl >= L ? 1.0 - 1e-9 : 0.97)) {
                    best = t;
                    best_cl = c;
                }
            }
            if (best_cl >= L) {
                *plan = Plan{L, 1};
                return MAMBA_OK;
            }
            *plan = Plan{best_cl, (int)((L + best_cl - 1) / best_cl)};
            return MAMBA_OK;
        }
        const long long lanes = Bsz * Dch * g.S;
        const long long target = (long long)sms * 1024;  // lanes the GPU can keep in flight
        if (lanes * 4 >= target || L < 16LL * g.TT) {
            *plan = Plan{L, 1};
            return MAMBA_OK;
        }
        long long K = (target + lanes - 1) / lanes;
        const long long kmax = L / (8LL * g.TT);  // keep chunks at least 8 tiles long
        if (K > kmax) K = kmax;
        if (K <= 1) {
            *plan = Plan{L, 1};
            return MAMBA_OK;
        }
        cl = (L + K - 1) / K;
    }
    cl = (cl + g.TT - 1) / g.TT * g.TT;  // chunk starts must fall on tile (and 16-byte) boundaries
    long long K = (L + cl - 1) / cl;
    if (K > 65535) return MAMBA_ERR_BAD_SHAPE;
    *plan = Plan{cl, (int)K};
    return MAMBA_OK;
}

size_t workspace_bytes_for(long long Bsz, long long Dch, long long N, int K) {
    if (K <= 1) return 0;
    const size_t h = round_up((size_t)Bsz * K * Dch * N * sizeof(float), 256);
    const size_t s = round_up((size_t)Bsz * K * Dch * sizeof(float), 256);
    return h + s;
}

// Internal status of scan_impl with conv taps: the convolution-fed kernel
// declined the problem before anything was launched (the caller falls back).
constexpr int kNotFused = 1;

int scan_impl(const void *u, const void *delta, const float *A, const void *B, const void *C, const float *D,
              const void *z, const float *delta_bias, int softplus_flag, void *y, float *last_state,
              const float *h0, long long Bsz, long long Dch, long long L, long long N, int dtype, int flags,
              long long chunk_len, void *workspace, size_t workspace_bytes, cudaStream_t stream,
              const float *conv_w = nullptr, const float *conv_b = nullptr) {
    if (!u || !delta || !A || !B || !C || !y) return MAMBA_ERR_NULL_ARG;
    int st = check_sizes(Bsz, Dch, L, N, dtype);
    if (st != MAMBA_OK) return st;
    if (flags & ~(MAMBA_FLAG_ZOH | MAMBA_FLAG_REVERSE)) return MAMBA_ERR_BAD_FLAGS;

    Plan plan;
    st = make_plan(Bsz, Dch, L, N, dtype, chunk_len, &plan);
    if (st != MAMBA_OK) return st;

    const bool vec = aligned16(u) && aligned16(delta) && aligned16(B) && aligned16(C) && aligned16(y) &&
                     (z == nullptr || aligned16(z)) && ((L * io_bytes(dtype)) % 16 == 0);

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
    a.flags = flags;
    a.conv_w = conv_w;
    a.conv_b = conv_b;

    if (plan.K == 1) {
        a.hin = h0;
        a.chunk_len = L;
        a.nchunks = 1;
        const cudaError_t e = launch_scan(dtype, MODE_FULL, vec, a, Bsz, 1, stream);
        if (e == cudaErrorNotSupported && conv_w != nullptr) return kNotFused;
        return e == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
    }

    // chunked scan: pass A (chunk end states), carry, pass B (seeded rescan)
    const size_t need = workspace_bytes_for(Bsz, Dch, N, plan.K);
    void *ws = workspace;
    bool owned = false;
    if (ws != nullptr) {
        if (workspace_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MAMBA_ERR_WORKSPACE;
    } else {
        if (inject_alloc_failure()) return MAMBA_ERR_ALLOC;
        if (cudaMallocAsync(&ws, need, stream) != cudaSuccess) {
            cudaGetLastError();
            return MAMBA_ERR_ALLOC;
        }
        owned = true;
    }
    float *ws_h = reinterpret_cast<float *>(ws);
    float *ws_sdt = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) +
                                              round_up((size_t)Bsz * plan.K * Dch * N * sizeof(float), 256));
    a.chunk_len = plan.chunk_len;
    a.nchunks = plan.K;
    int rc = MAMBA_OK;
    const cudaError_t e = run_chunked(dtype, vec, a, Bsz, ws_h, ws_sdt, h0, stream);
    if (e == cudaErrorNotSupported && conv_w != nullptr) {  // nothing launched yet
        if (owned) cudaFreeAsync(ws, stream);
        return kNotFused;
    }
    if (e != cudaSuccess) rc = MAMBA_ERR_LAUNCH;
    if (owned && cudaFreeAsync(ws, stream) != cudaSuccess) {
        cudaGetLastError();
        if (rc == MAMBA_OK) rc = MAMBA_ERR_LAUNCH;
    }
    return rc;
}

}  // namespace

extern "C" {

int mamba_selective_scan_fwd(const void *u, const void *delta, const float *A, const void *B, const void *C,
                             const float *D, const void *z, const float *delta_bias, int softplus_flag, void *y,
                             float *last_state, int64_t Bsz, int64_t Dch, int64_t L, int64_t N, int dtype,
                             mamba_stream_t stream) {
    return scan_impl(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, nullptr, Bsz, Dch, L, N,
                     dtype, 0, 0, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
}

int mamba_selective_scan_fwd_ex(const void *u, const void *delta, const float *A, const void *B, const void *C,
                                const float *D, const void *z, const float *delta_bias, int softplus_flag,
                                void *y, float *last_state, const float *h0, int64_t Bsz, int64_t Dch, int64_t L,
                                int64_t N, int dtype, int flags, int64_t chunk_len, void *workspace,
                                size_t workspace_bytes, mamba_stream_t stream) {
    return scan_impl(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, h0, Bsz, Dch, L, N, dtype,
                     flags, chunk_len, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t mamba_scan_workspace_size(int64_t Bsz, int64_t Dch, int64_t L, int64_t N, int64_t chunk_len, int dtype) {
    if (check_sizes(Bsz, Dch, L, N, dtype) != MAMBA_OK) return (size_t)-1;
    Plan plan;
    if (make_plan(Bsz, Dch, L, N, dtype, chunk_len, &plan) != MAMBA_OK) return (size_t)-1;
    return workspace_bytes_for(Bsz, Dch, N, plan.K);
}

int mamba_state_update(float *state, const void *u, const void *delta, const float *A, const void *B,
                       const void *C, const float *D, const void *z, const float *delta_bias, int softplus_flag,
                       void *y, int64_t Bsz, int64_t Dch, int64_t N, int dtype, mamba_stream_t stream) {
    if (!state || !u || !delta || !A || !B || !C || !y) return MAMBA_ERR_NULL_ARG;
    const int st = check_sizes(Bsz, Dch, 1, N, dtype);
    if (st != MAMBA_OK) return st;
    StepArgs a{};
    a.state = state;
    a.u = u;
    a.delta = delta;
    a.z = z;
    a.Bm = B;
    a.Cm = C;
    a.A = A;
    a.D = D;
    a.bias = delta_bias;
    a.y = y;
    a.Bsz = Bsz;
    a.Dch = Dch;
    a.N = N;
    a.softplus = softplus_flag ? 1 : 0;
    // the aligned kernel reads V = 8 or 4 consecutive states of state, A, B and C per lane with
    // 16-byte (and, for bf16 B/C with V = 4, 8-byte) loads
    auto aligned_to = [](const void *p, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(p) & (bytes - 1u)) == 0; };
    const uintptr_t eb = (uintptr_t)io_bytes(dtype);
    const bool rows_ok = aligned16(state) && aligned16(A) && Bsz * Dch < (1LL << 31);
    int lane_states = 0;
    if (rows_ok && N % 8 == 0 && aligned_to(B, 8 * eb) && aligned_to(C, 8 * eb))
        lane_states = 8;
    else if (rows_ok && N % 4 == 0 && aligned_to(B, 4 * eb) && aligned_to(C, 4 * eb))
        lane_states = 4;
    return launch_state_update(dtype, lane_states, a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MAMBA_OK
               : MAMBA_ERR_LAUNCH;
}

const char *mamba_status_string(int status) {
    switch (status) {
        case MAMBA_OK: return "ok";
        case MAMBA_ERR_NULL_ARG: return "a required pointer argument is NULL";
        case MAMBA_ERR_BAD_SHAPE: return "a size argument is out of range";
        case MAMBA_ERR_UNSUPPORTED_N: return "state size N must be in 1..64";
        case MAMBA_ERR_BAD_DTYPE: return "dtype must be MAMBA_F32 or MAMBA_BF16";
        case MAMBA_ERR_ALLOC: return "workspace allocation failed";
        case MAMBA_ERR_LAUNCH: return "kernel launch failed";
        case MAMBA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait expired";
        case MAMBA_ERR_BAD_FLAGS: return "unknown or unsupported flag bits";
        case MAMBA_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
        case MAMBA_ERR_DEVICE: return "no usable CUDA device";
        case MAMBA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the no-allocation entry point holds";
        default: return "unknown status";
    }
}

int mamba_causal_conv1d_silu(const void *x, const float *conv_w, const float *conv_bias, int silu_flag, void *u,
                             int64_t Bsz, int64_t Dch, int64_t L, int dtype, mamba_stream_t stream) {
    if (!x || !conv_w || !u) return MAMBA_ERR_NULL_ARG;
    if (dtype != MAMBA_F32 && dtype != MAMBA_BF16) return MAMBA_ERR_BAD_DTYPE;
    if (Bsz <= 0 || Dch <= 0 || L <= 0 || Bsz > kMaxDim || Dch > kMaxDim || L > kMaxDim || Bsz * Dch > kMaxDim / L)
        return MAMBA_ERR_BAD_SHAPE;
    const bool vec = aligned16(x) && aligned16(u) && aligned16(conv_w) && (L * io_bytes(dtype)) % 16 == 0;
    return launch_conv1d(dtype, vec, x, conv_w, conv_bias, silu_flag ? 1 : 0, u, Bsz * Dch, Dch, L,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MAMBA_OK
               : MAMBA_ERR_LAUNCH;
}

int mamba_selective_scan_fwd_conv(const void *x, const float *conv_w, const float *conv_bias, const void *delta,
                                  const float *A, const void *B, const void *C, const float *D, const void *z,
                                  const float *delta_bias, int softplus_flag, void *y, float *last_state,
                                  int64_t Bsz, int64_t Dch, int64_t L, int64_t N, int dtype,
                                  mamba_stream_t stream) {
    if (!x || !conv_w) return MAMBA_ERR_NULL_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (z != nullptr) {  // the fused kernel is built with the gate
        const int rc = scan_impl(x, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, nullptr, Bsz,
                                 Dch, L, N, dtype, 0, 0, nullptr, 0, st, conv_w, conv_bias);
        if (rc != kNotFused) return rc;
    } else {
        const int chk = check_sizes(Bsz, Dch, L, N, dtype);
        if (chk != MAMBA_OK) return chk;
        if (!u_ok_args(delta, A, B, C, y)) return MAMBA_ERR_NULL_ARG;
    }
    // two steps: the convolution into a stream-ordered temporary, then the scan
    void *u = nullptr;
    if (inject_alloc_failure()) return MAMBA_ERR_ALLOC;
    if (cudaMallocAsync(&u, (size_t)(Bsz * Dch * L) * io_bytes(dtype), st) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_ALLOC;
    }
    int rc = mamba_causal_conv1d_silu(x, conv_w, conv_bias, 1, u, Bsz, Dch, L, dtype, stream);
    if (rc == MAMBA_OK)
        rc = scan_impl(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, nullptr, Bsz, Dch, L, N,
                       dtype, 0, 0, nullptr, 0, st);
    if (cudaFreeAsync(u, st) != cudaSuccess) {
        cudaGetLastError();
        if (rc == MAMBA_OK) rc = MAMBA_ERR_LAUNCH;
    }
    return rc;
}

int mamba_bench_ex2(int64_t *cycles, float *sink, int64_t iters, int blocks, int threads, mamba_stream_t stream) {
    if (!cycles || !sink) return MAMBA_ERR_NULL_ARG;
    if (iters <= 0 || blocks <= 0 || threads <= 0 || threads > 1024) return MAMBA_ERR_BAD_SHAPE;
    return launch_bench_ex2(reinterpret_cast<long long *>(cycles), sink, iters, blocks, threads,
                            reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MAMBA_OK
               : MAMBA_ERR_LAUNCH;
}

}  // extern "C"
