// state_update.cu -- one-token recurrent step (selective_state_update).
//
// The selective_step of the fsdata.site explainer §3.2 applied to a stored
// state: Delta = softplus(Delta_raw + bias), h = exp(Delta A) h + Delta B u,
// y = (C . h + D u) * SiLU(z).  The state [Bsz][Dch][N] fp32 is read and
// written once per call, so the kernel is bound by HBM bandwidth on the state
// bytes.  On 16-byte aligned rows (state_update_rows_kernel) every lane owns
// V = 8 (or 4) consecutive states of a (b, d) row, moves them with 16-byte
// loads and stores and reads B and C with vector loads; the NP/V lanes of a
// row reduce C . h with butterfly shuffles and the first of them writes y.
// Otherwise one (b, d) row is spread over NP/4 lanes with scalar accesses
// (state_update_kernel).
#include "internal.h"

namespace mamba {

template <typename T, int NP, bool VEC>
__global__ void __launch_bounds__(256)
state_update_kernel(const StepArgs a) {
    using IO = Io<T>;
    constexpr int G = NP / 4;  // lanes per (b, d)
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long ch = gid / G;  // b * Dch + d
    const int q = (int)(gid % G);
    const long long nch = a.Bsz * a.Dch;
    const bool valid = ch < nch;
    const long long cc = valid ? ch : 0;
    const long long b = cc / a.Dch, d = cc % a.Dch;
    const long long N = a.N;
    const long long n0 = 4LL * q;

    float h[4] = {0.f, 0.f, 0.f, 0.f}, A2[4] = {0.f, 0.f, 0.f, 0.f};
    float Bv[4] = {0.f, 0.f, 0.f, 0.f}, Cv[4] = {0.f, 0.f, 0.f, 0.f};
    if (valid) {
        if (VEC && n0 < N) {  // N % 4 == 0 and 16-byte aligned rows
            const float4 hv = __ldcs(reinterpret_cast<const float4 *>(a.state + cc * N + n0));
            const float4 av = __ldg(reinterpret_cast<const float4 *>(a.A + d * N + n0));
            h[0] = hv.x; h[1] = hv.y; h[2] = hv.z; h[3] = hv.w;
            A2[0] = av.x; A2[1] = av.y; A2[2] = av.z; A2[3] = av.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (n0 + j < N) {
                    h[j] = a.state[cc * N + n0 + j];
                    A2[j] = a.A[d * N + n0 + j];
                }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            A2[j] *= kLog2e;
            if (n0 + j < N) {
                Bv[j] = IO::load(a.Bm, b * N + n0 + j);
                Cv[j] = IO::load(a.Cm, b * N + n0 + j);
            }
        }
    }
    const float uu = valid ? IO::load(a.u, cc) : 0.f;
    const float raw = (valid ? IO::load(a.delta, cc) : 0.f) + (a.bias != nullptr && valid ? a.bias[d] : 0.f);
    const float dl = a.softplus ? softplus_f(raw) : raw;
    const float du = dl * uu;
    float p = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        h[j] = fmaf(ex2_approx(dl * A2[j]), h[j], du * Bv[j]);
        p = fmaf(Cv[j], h[j], p);
    }
#pragma unroll
    for (int off = 1; off < G; off <<= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
    if (!valid) return;
    if (VEC && n0 < N) {
        __stcs(reinterpret_cast<float4 *>(a.state + cc * N + n0), make_float4(h[0], h[1], h[2], h[3]));
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (n0 + j < N) a.state[cc * N + n0 + j] = h[j];
    }
    if (q == 0) {
        float y = fmaf(a.D != nullptr ? a.D[d] : 0.f, uu, p);
        if (a.z != nullptr) y *= silu_f(IO::load(a.z, cc));
        IO::store(a.y, cc, y);
    }
}

// elements i..i+V-1 (V = 4 or 8) of a bf16 or fp32 array with 8- or 16-byte loads (i a multiple of
// V and the array aligned to V elements), or zeros
template <typename T, int V>
__device__ __forceinline__ void loadv(float (&v)[V], const void *p, long long i, bool ok) {
    if constexpr (sizeof(T) == 2) {
        const uint16_t *q = reinterpret_cast<const uint16_t *>(p) + i;
        uint32_t w[V / 2];
        if constexpr (V >= 8) {
#pragma unroll
            for (int k = 0; k < V / 8; ++k) {
                const uint4 x = ok ? __ldg(reinterpret_cast<const uint4 *>(q) + k) : make_uint4(0u, 0u, 0u, 0u);
                w[4 * k] = x.x; w[4 * k + 1] = x.y; w[4 * k + 2] = x.z; w[4 * k + 3] = x.w;
            }
        } else {
            const uint2 x = ok ? __ldg(reinterpret_cast<const uint2 *>(q)) : make_uint2(0u, 0u);
            w[0] = x.x; w[1] = x.y;
        }
#pragma unroll
        for (int k = 0; k < V / 2; ++k) {
            v[2 * k] = bf16_lo(w[k]);
            v[2 * k + 1] = bf16_hi(w[k]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < V / 4; ++k) {
            const float4 x = ok ? __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p) + i) + k)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            v[4 * k] = x.x;
            v[4 * k + 1] = x.y;
            v[4 * k + 2] = x.z;
            v[4 * k + 3] = x.w;
        }
    }
}

// 16-byte aligned state rows with N % V == 0, B and C aligned to V elements, and fewer than 2^31
// rows: each lane owns V = 4 or 8 consecutive states of a (b, d) row (NP / V lanes per row) and
// issues all its loads (state, A, B, C, u, Delta, z, D, bias) before any arithmetic.  Row r of warp
// w covers channels w * R * (32 / G) + r * (32 / G) + lane / G, so every state load instruction of
// the warp reads one contiguous span.  Measured on the B300 decode workload (B256 D5120 N16, bf16):
// V = 4 with scalar B/C loads 4.45 TB/s, with vector B/C loads 5.04, V = 8 5.40, V = 16 (one lane
// per row) 4.00; with V = 4, R = 2 and R = 4 rows per lane cost more occupancy than they add loads
// in flight.
template <typename T, int NP, int R, int V = 4>
__global__ void __launch_bounds__(256)
state_update_rows_kernel(const StepArgs a) {
    using IO = Io<T>;
    constexpr int G = NP / V;   // lanes per channel
    constexpr int CPI = 32 / G; // channels per warp instruction
    constexpr int NV = V / 4;   // 16-byte state vectors per lane
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int q = lane % G;
    const long long N = a.N, nch = a.Bsz * a.Dch;
    const long long n0 = (long long)V * q;
    const bool live = n0 < N;  // lanes past N (N < NP) carry no states

    long long chan[R];
    bool valid[R];
    float4 hv[R][NV], av[R][NV];
    float Bv[R][V], Cv[R][V], uu[R], raw[R], zz[R], Dd[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        chan[r] = warp * (R * CPI) + r * CPI + lane / G;
        valid[r] = chan[r] < nch;
        // the host sends this kernel fewer than 2^31 rows: 32-bit division
        const unsigned cc32 = valid[r] ? (unsigned)chan[r] : 0u, dch32 = (unsigned)a.Dch;
        const unsigned b32 = cc32 / dch32;
        const long long cc = cc32, b = b32, d = cc32 - b32 * dch32;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            hv[r][k] = make_float4(0.f, 0.f, 0.f, 0.f);
            av[r][k] = hv[r][k];
            if (valid[r] && live) {
                hv[r][k] = __ldcs(reinterpret_cast<const float4 *>(a.state + cc * N + n0) + k);
                av[r][k] = __ldg(reinterpret_cast<const float4 *>(a.A + d * N + n0) + k);
            }
        }
        loadv<T, V>(Bv[r], a.Bm, b * N + n0, valid[r] && live);
        loadv<T, V>(Cv[r], a.Cm, b * N + n0, valid[r] && live);
        uu[r] = valid[r] ? IO::load(a.u, cc) : 0.f;
        raw[r] = (valid[r] ? IO::load(a.delta, cc) : 0.f) + (a.bias != nullptr && valid[r] ? a.bias[d] : 0.f);
        zz[r] = (a.z != nullptr && valid[r]) ? IO::load(a.z, cc) : 0.f;
        Dd[r] = (a.D != nullptr && valid[r]) ? a.D[d] : 0.f;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float dl = a.softplus ? softplus_f(raw[r]) : raw[r];
        const float du = dl * uu[r];
        float p = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            float h[4] = {hv[r][k].x, hv[r][k].y, hv[r][k].z, hv[r][k].w};
            const float A[4] = {av[r][k].x, av[r][k].y, av[r][k].z, av[r][k].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                h[j] = fmaf(ex2_approx(dl * (A[j] * kLog2e)), h[j], du * Bv[r][4 * k + j]);
                p = fmaf(Cv[r][4 * k + j], h[j], p);
            }
            hv[r][k] = make_float4(h[0], h[1], h[2], h[3]);
        }
#pragma unroll
        for (int off = 1; off < G; off <<= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
        if (valid[r] && live)
#pragma unroll
            for (int k = 0; k < NV; ++k) __stcs(reinterpret_cast<float4 *>(a.state + chan[r] * N + n0) + k, hv[r][k]);
        if (valid[r] && q == 0) {
            float y = fmaf(Dd[r], uu[r], p);
            if (a.z != nullptr) y *= silu_f(zz[r]);
            IO::store(a.y, chan[r], y);
        }
    }
}

// rows per lane of the aligned kernel (0: one row per lane, state_update_kernel)
#ifndef MAMBA_STATE_ROWS
#define MAMBA_STATE_ROWS 1
#endif

template <typename T, int NP>
static cudaError_t launch_np(int lane_states, const StepArgs &a, cudaStream_t st) {
    const int threads = 256;
    const bool vec = lane_states > 0;
    if (MAMBA_STATE_ROWS == 0 && vec) {
        const long long total = a.Bsz * a.Dch * (NP / 4);
        state_update_kernel<T, NP, true><<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(a);
        return cudaGetLastError();
    }
    if (vec) {
        constexpr int R = MAMBA_STATE_ROWS > 0 ? MAMBA_STATE_ROWS : 1;
        if (NP >= 8 && lane_states == 8) {
            constexpr int V = NP >= 8 ? 8 : 4;
            const long long per_block = (long long)(threads / 32) * R * (32 / (NP / V));
            const long long blocks = (a.Bsz * a.Dch + per_block - 1) / per_block;
            state_update_rows_kernel<T, NP, R, V><<<(unsigned)blocks, threads, 0, st>>>(a);
        } else {
            const long long per_block = (long long)(threads / 32) * R * (32 / (NP / 4));
            const long long blocks = (a.Bsz * a.Dch + per_block - 1) / per_block;
            state_update_rows_kernel<T, NP, R, 4><<<(unsigned)blocks, threads, 0, st>>>(a);
        }
        return cudaGetLastError();
    }
    const long long total = a.Bsz * a.Dch * (NP / 4);
    const long long blocks = (total + threads - 1) / threads;
    state_update_kernel<T, NP, false><<<(unsigned)blocks, threads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_t(int lane_states, const StepArgs &a, cudaStream_t st) {
    if (a.N <= 4) return launch_np<T, 4>(lane_states, a, st);
    if (a.N <= 8) return launch_np<T, 8>(lane_states, a, st);
    if (a.N <= 16) return launch_np<T, 16>(lane_states, a, st);
    if (a.N <= 32) return launch_np<T, 32>(lane_states, a, st);
    return launch_np<T, 64>(lane_states, a, st);
}

cudaError_t launch_state_update(int dtype, int lane_states, const StepArgs &a, cudaStream_t st) {
    return dtype == 1 ? launch_t<bf16_t>(lane_states, a, st) : launch_t<float>(lane_states, a, st);
}

}  // namespace mamba
