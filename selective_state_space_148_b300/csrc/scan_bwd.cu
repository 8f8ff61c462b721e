// scan_bwd.cu -- backward pass of the selective scan (simple discretisation,
// forward time, zero initial state): gradients of sum(dy * y) for u, Delta_raw,
// A, B, C, D, z and the Delta bias.
//
// The pages measure training throughput but print no backward pass; this is
// the chain rule of the forward step (fsdata.site explainer §3.2 selective_step)
// with, per (b, d, n), a sweep from t = L-1 down to 0 that carries
// dh = dLoss/dh_t:
//   dyh = dy_t g_t (g = SiLU(z_t), or 1),  dz_t = dy_t yhat_t SiLU'(z_t)
//   dC_{t,n} += dyh h_t;  dh += dyh C_{t,n}
//   a = exp(Delta A_n):  dB_{t,n} += dh Delta u_t,  du_t += dh Delta B_{t,n},
//     dDelta_t += dh (B_{t,n} u_t + A_n a h_{t-1}),  dA_n += dh Delta a h_{t-1},  dh *= a
//   du_t += D dyh,  dD += dyh u_t,  dDelta_raw_t = dDelta_t sigmoid(Delta_raw_t + bias),  dbias += dDelta_raw_t
//
// One CTA holds 32 channels of one batch row, 4 lanes per channel and NS
// states per lane, and walks the whole sequence: a forward sweep writes the
// state at every chunk start (TC = 64 / NS steps apart) to a checkpoint
// workspace; then, chunk by chunk from the end, the chunk's states are
// recomputed from its checkpoint into shared memory and swept in reverse.
//
// Per chunk, the work that depends only on (channel, step) -- Delta, sigmoid of
// the Delta pre-activation, the gate and its derivative -- is done once, by the
// channel's 4 lanes taking TC / 4 steps each, and read back by all 4 lanes from
// shared memory; those lanes also write the chunk's du, ddelta, dz.  The sums
// over the 4 lanes of a channel (du, ddelta and yhat for dz) and over the 8
// channels of a warp (dB, dC) are transposed shuffle reductions: every lane
// ends with a different total, so no lane waits on a chain of shuffles of one
// value.  The 4 warps' dB, dC partials are added in shared memory and sent to
// memory with one vector atomic add per 4 steps.  dA, dD and dbias (sums over
// batch rows and steps) stay in registers and are added atomically at the end.
// Steps past L and channels past Dch run as steps with Delta = 0 and dy = 0,
// which change neither the state nor any gradient, so the sweeps have no
// per-step branches.  No device-side waits.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <type_traits>

#include "../../include/mamba_scan.h"
#include "internal.h"

namespace mamba {

struct BwdArgs {
    const void *u, *delta, *z, *Bm, *Cm, *dy;
    const float *A, *D, *bias;
    void *du, *ddelta, *dz;
    float *dA, *dB, *dC, *dD, *dbias;
    float *ckpt;  // [Bsz][Dch][K][NP]: the state before step k * TC (entry 0 unused)
    long long Dch, L, N;
    int softplus;
    int vec;  // L % 4 == 0 and every row pointer 16-byte aligned: vector loads, stores and atomics
    int ckpt_given;  // 1: the checkpoints were saved by the forward pass (no checkpoint sweep here)
    int sweep_only;  // 1: only the checkpoint sweep, writing every entry 1 .. K-1, then return
};

template <int NS>
struct BwdShape {
    static constexpr int S = 4, CH = 32, NTHR = S * CH, NWARP = NTHR / 32;
    static constexpr int TC = 64 / NS;  // steps per chunk: TC * NS = 64 recomputed states per lane
    static constexpr int NP = S * NS;   // padded state count
    static constexpr int G = TC / S;    // steps per lane in the per-(channel, step) work
    static constexpr int NQ = NS / 4;   // float4 per lane per step of states
    // shared memory, floats: states [TC][NQ][NTHR] float4 (lane innermost; h, then dh); per (step,
    // channel) float4s [TC][CH]: {Delta, Delta u, dy g, u}, {sigmoid, dz factor, -, -} and the lane sums
    // {q, sum_n A_n w_n / ln2, C.h, -}; B, C rows [TC][2][NP]; dB, dC channel sums [TC][2][NP]
    static constexpr int OFF_H = 0, OFF_R = OFF_H + TC * NS * NTHR, OFF_E = OFF_R + 4 * TC * CH;
    static constexpr int OFF_Q = OFF_E + 4 * TC * CH, OFF_BC = OFF_Q + 4 * TC * CH;
    static constexpr int OFF_O = OFF_BC + 2 * TC * NP, FLOATS = OFF_O + 2 * TC * NP;
    static constexpr size_t SMEM_BYTES = (size_t)FLOATS * sizeof(float);
    static_assert(2 * NP * (TC / 4) == NTHR, "one thread per (B or C row, 4 steps)");
    static_assert(NS % 4 == 0 && TC % 4 == 0, "float4 state groups, 4-step row groups");
    static_assert(TC * NQ == 16 && CH == 32, "channel sums: 128 threads = 16 (step, state quad) x 4 lanes x 2 parities");
};

// M consecutive elements of storage type T: loaded with one vector access where the caller says the
// whole group is in range and aligned, element by element (zero past `nvalid`) otherwise.
template <typename T, int M>
struct Pack {
    static constexpr int BYTES = M * (int)sizeof(T), W = BYTES >= 4 ? BYTES / 4 : 1;
    uint32_t w[W];
    __device__ __forceinline__ void load(const void *base, long long idx, int nvalid, bool vec) {
        const T *p = reinterpret_cast<const T *>(base) + idx;
        if (vec && nvalid >= M && BYTES >= 4) {
            if constexpr (BYTES == 16) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else if constexpr (BYTES == 8) {
                const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
                w[0] = v.x; w[1] = v.y;
            } else if constexpr (BYTES == 4) {
                w[0] = __ldg(reinterpret_cast<const uint32_t *>(p));
            }
            return;
        }
#pragma unroll
        for (int e = 0; e < M; ++e) set(e, e < nvalid ? Io<T>::load(base, idx + e) : 0.f);
    }
    __device__ __forceinline__ float get(int e) const {
        if constexpr (sizeof(T) == 4) return __uint_as_float(w[e]);
        else return (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
    }
    __device__ __forceinline__ void set(int e, float f) {
        if constexpr (sizeof(T) == 4) {
            w[e] = __float_as_uint(f);
        } else {
            const uint32_t h = pack_bf16x2(f, 0.f) & 0xffffu;  // round to nearest even
            w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0x0000ffffu) | (h << 16)) : ((w[e >> 1] & 0xffff0000u) | h);
        }
    }
    __device__ __forceinline__ void store(void *base, long long idx, int nvalid, bool vec) const {
        T *p = reinterpret_cast<T *>(base) + idx;
        if (vec && nvalid >= M && BYTES >= 4) {
            if constexpr (BYTES == 16) *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
            else if constexpr (BYTES == 8) *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
            else if constexpr (BYTES == 4) *reinterpret_cast<uint32_t *>(p) = w[0];
            return;
        }
#pragma unroll
        for (int e = 0; e < M; ++e)
            if (e < nvalid) Io<T>::store(base, idx + e, get(e));
    }
};

__device__ __forceinline__ void red_add_v4(float *p, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// One level of a transposed butterfly: lanes l and l ^ X exchange halves of v[0 .. 2H); afterwards
// v[0 .. H) holds the pair's sums of the half selected by bit X of the lane (upper half where set).
template <int H, int X, int V>
__device__ __forceinline__ void transpose_level(float (&v)[V], int lane) {
    const bool hi = (lane & X) != 0;
#pragma unroll
    for (int k = 0; k < H; ++k) {
        const float keep = hi ? v[H + k] : v[k], send = hi ? v[k] : v[H + k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, X);
    }
}

template <typename T, int NS, bool HAS_Z>
__global__ void __launch_bounds__(128, 3)
scan_bwd_kernel(const BwdArgs a, int K) {
    using Sh = BwdShape<NS>;
    constexpr int CH = Sh::CH, NTHR = Sh::NTHR, TC = Sh::TC, NP = Sh::NP, G = Sh::G;
    constexpr int NQ = Sh::NQ, NH = NS / 2;
    extern __shared__ float4 smem_f4[];
    float *const smem = reinterpret_cast<float *>(smem_f4);
    float4 *const sH = reinterpret_cast<float4 *>(smem + Sh::OFF_H);  // [TC][NQ][NTHR]: h, then dh
    float4 *const sR = reinterpret_cast<float4 *>(smem + Sh::OFF_R);  // [TC][CH]: Delta, Delta u, dy g, u
    float4 *const sE = reinterpret_cast<float4 *>(smem + Sh::OFF_E);  // [TC][CH]: sigmoid, dz factor
    float4 *const sQ = reinterpret_cast<float4 *>(smem + Sh::OFF_Q);  // [TC][CH]: q, wa / ln2, C.h
    float *const sBC = smem + Sh::OFF_BC;                             // [TC][2][NP]: B, C rows
    float *const sO = smem + Sh::OFF_O;                               // [TC][2][NP]: dB, dC channel sums

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, s = tid & 3, c = tid >> 2;
    const long long d = (long long)blockIdx.x * CH + c;
    const bool valid = d < a.Dch;
    const long long dd = valid ? d : 0;
    const long long b = blockIdx.y;
    const long long N = a.N, L = a.L;
    const bool vec = a.vec != 0;
    const long long row = (b * a.Dch + dd) * L;  // this channel's (b, d) row of u, Delta, z, dy
    // B/C rows and dB/dC sums: thread -> (which = B or C, state n, 4-step group rg)
    const int rg = tid % (TC / 4), rrow = tid / (TC / 4), rwhich = rrow / NP, rn = rrow % NP;
    const long long bcrow = (b * N + (rn < N ? rn : 0)) * L;
    // [TC][CH] arrays: the column of channel c at step i is c ^ 2 f(i), f(i) = (i / G xor i) mod 4 (i mod 4
    // for G = 1): the 4 lanes of a channel, which take consecutive groups of G steps, and the 4 steps that
    // a warp's channel sums read at once fall on distinct banks
    auto swz = [](int i) { return 2 * (((i / G) ^ (G == 1 ? 0 : i)) & 3); };
    auto sw = [&](int i, int cc) { return i * CH + (cc ^ swz(i)); };

    // per-state constants in pairs of adjacent states (f32x2): A log2 e
    float2 A2[NH];
#pragma unroll
    for (int jp = 0; jp < NH; ++jp) {
        float v[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const long long n = (long long)s * NS + 2 * jp + k;
            v[k] = (valid && n < N) ? a.A[dd * N + n] * kLog2e : 0.f;
        }
        A2[jp] = f2(v[0], v[1]);
    }
    const float Dd = (a.D != nullptr && valid) ? a.D[dd] : 0.f;
    const float bias = (a.bias != nullptr && valid) ? a.bias[dd] : 0.f;
    float *const ck = a.ckpt + ((b * a.Dch + dd) * K) * NP + s * NS;

    // this lane's G steps of the chunk starting at t0: how many are in range
    auto lane_valid = [&](long long t0) {
        const long long r = L - (t0 + s * G);
        return valid ? (int)(r < 0 ? 0 : r > G ? G : r) : 0;
    };
    auto row_valid = [&](long long t0) {
        const long long r = L - (t0 + 4 * rg);
        return rn < N ? (int)(r < 0 ? 0 : r > 4 ? 4 : r) : 0;
    };
    auto softplus_of = [&](float x) { return a.softplus ? softplus_f(x) : x; };

    // Sums over the CTA's 32 channels, for every (step, state) of the chunk, of w[c][t] X[c][t][n]:
    // X = sH (h for dC, dh for dB), w = dy g (dC) or Delta u (dB); into sO[t][WHICH][n].  Thread: step t,
    // state quad q of state-lane ls, and the channels of one parity (c = 2j + half), which keeps the 8
    // lanes of a quarter-warp on distinct banks; the parities meet in one shuffle.
    const int ls = lane & 3, half = (lane >> 2) & 1, qt = (lane >> 3) + 4 * warp;
    const int sq = qt % NQ, st = qt / NQ;
    const int kx = swz(st) / 2;  // the swizzle of step st, in channel pairs
    const float4 *const hcol = sH + (st * NQ + sq) * NTHR + ls + 4 * half;
    const float *wcol[4];  // row st of sR at channels 2 (jj ^ kx) + half, jj = 0..3 (then + 8 jj' float4)
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) wcol[jj] = reinterpret_cast<const float *>(sR + st * CH + 2 * (jj ^ kx) + half);
    auto channel_sums = [&](auto which_tag) {
        constexpr int WHICH = decltype(which_tag)::value;  // 0: dB (w = Delta u), 1: dC (w = dy g)
        float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < CH / 2; ++j) {
            // channel 2j + half: its states at hcol[8 j], its weight in swizzled column 2 (j ^ kx) + half
            const float4 x = hcol[8 * j];
            const float w = wcol[j & 3][32 * (j >> 2) + 1 + WHICH];
            acc0 = __ffma2_rn(f2(w, w), f2(x.x, x.y), acc0);
            acc1 = __ffma2_rn(f2(w, w), f2(x.z, x.w), acc1);
        }
        acc0.x += __shfl_xor_sync(0xffffffffu, acc0.x, 4);
        acc0.y += __shfl_xor_sync(0xffffffffu, acc0.y, 4);
        acc1.x += __shfl_xor_sync(0xffffffffu, acc1.x, 4);
        acc1.y += __shfl_xor_sync(0xffffffffu, acc1.y, 4);
        if (half == 0)
            *reinterpret_cast<float4 *>(sO + (st * 2 + WHICH) * NP + ls * NS + 4 * sq) =
                make_float4(acc0.x, acc0.y, acc1.x, acc1.y);
    };
    // dB, dC of the chunk at t0 (in sO): this thread's (B or C row, 4 steps), one vector atomic add
    auto flush_sums = [&](long long t0) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = sO[((4 * rg + e) * 2 + rwhich) * NP + rn];
        const int nv = row_valid(t0);
        float *const dst = (rwhich ? a.dC : a.dB) + bcrow + t0 + 4 * rg;
        if (vec && nv == 4) {
            red_add_v4(dst, v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nv) atomicAdd(dst + e, v[e]);
        }
    };

    Pack<T, G> pu, pr, pz, pdy;  // this lane's steps of u, Delta_raw, z, dy (one chunk ahead)
    Pack<T, 4> pbc;              // this thread's 4 steps of its B or C row (one chunk ahead)

    // ---- forward sweep over chunks 0 .. K-2: the state before each chunk k >= 1 goes to the checkpoints
    // (skipped when the forward pass saved them)
    float2 h2[NH];
#pragma unroll
    for (int jp = 0; jp < NH; ++jp) h2[jp] = f2(0.f, 0.f);
    if (a.ckpt_given) {
        if (K > 1 && valid) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4 v = *reinterpret_cast<const float4 *>(ck + (long long)(K - 1) * NP + 4 * q);
                h2[2 * q] = f2(v.x, v.y);
                h2[2 * q + 1] = f2(v.z, v.w);
            }
        }
    } else if (K > 1) {
        pu.load(a.u, row + s * G, lane_valid(0), vec);
        pr.load(a.delta, row + s * G, lane_valid(0), vec);
        if (rwhich == 0) pbc.load(a.Bm, bcrow + 4 * rg, row_valid(0), vec);
    }
    for (int k = 0; !a.ckpt_given && k + 1 < K; ++k) {
        const long long t0 = (long long)k * TC;
        __syncthreads();  // the previous chunk's readers are done
#pragma unroll
        for (int e = 0; e < G; ++e) {
            const int i = s * G + e;
            const bool in = e < lane_valid(t0);
            const float dl = in ? softplus_of(pr.get(e) + bias) : 0.f;
            *reinterpret_cast<float2 *>(sR + sw(i, c)) = f2(dl, dl * pu.get(e));
        }
        if (rwhich == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sBC[(4 * rg + e) * 2 * NP + rn] = pbc.get(e);
        }
        __syncthreads();
        if (k + 2 < K) {  // the next chunk's inputs, in flight during this one
            pu.load(a.u, row + t0 + TC + s * G, lane_valid(t0 + TC), vec);
            pr.load(a.delta, row + t0 + TC + s * G, lane_valid(t0 + TC), vec);
            if (rwhich == 0) pbc.load(a.Bm, bcrow + t0 + TC + 4 * rg, row_valid(t0 + TC), vec);
        }
        if (k > 0 && valid) {
#pragma unroll
            for (int q = 0; q < NQ; ++q)
                *reinterpret_cast<float4 *>(ck + (long long)k * NP + 4 * q) =
                    make_float4(h2[2 * q].x, h2[2 * q].y, h2[2 * q + 1].x, h2[2 * q + 1].y);
        }
#pragma unroll
        for (int i = 0; i < TC; ++i) {
            const float2 r = *reinterpret_cast<const float2 *>(sR + sw(i, c));
            const float2 dl2 = f2(r.x, r.x), du2 = f2(r.y, r.y);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4 bq = *reinterpret_cast<const float4 *>(sBC + i * 2 * NP + s * NS + 4 * q);
                const float2 bb[2] = {f2(bq.x, bq.y), f2(bq.z, bq.w)};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int jp = 2 * q + h;
                    const float2 x = __fmul2_rn(dl2, A2[jp]);
                    h2[jp] = __ffma2_rn(f2(ex2_approx(x.x), ex2_approx(x.y)), h2[jp], __fmul2_rn(du2, bb[h]));
                }
            }
        }
    }
    // h2 now holds the state before the last chunk
    if (a.sweep_only) {  // (uniform over the grid: every thread returns here)
        if (K > 1 && valid) {
#pragma unroll
            for (int q = 0; q < NQ; ++q)
                *reinterpret_cast<float4 *>(ck + (long long)(K - 1) * NP + 4 * q) =
                    make_float4(h2[2 * q].x, h2[2 * q].y, h2[2 * q + 1].x, h2[2 * q + 1].y);
        }
        return;
    }

    // ---- reverse sweep, chunk by chunk
    float2 dh2[NH], dA2[NH];
#pragma unroll
    for (int jp = 0; jp < NH; ++jp) dh2[jp] = dA2[jp] = f2(0.f, 0.f);
    float dDacc = 0.f, dbacc = 0.f;
    {
        const long long t0 = (long long)(K - 1) * TC;
        pu.load(a.u, row + t0 + s * G, lane_valid(t0), vec);
        pr.load(a.delta, row + t0 + s * G, lane_valid(t0), vec);
        if (HAS_Z) pz.load(a.z, row + t0 + s * G, lane_valid(t0), vec);
        pdy.load(a.dy, row + t0 + s * G, lane_valid(t0), vec);
        pbc.load(rwhich ? a.Cm : a.Bm, bcrow + t0 + 4 * rg, row_valid(t0), vec);
    }
    float4 hnext[NQ];  // the checkpoint of the next chunk to process, loaded one chunk ahead
#pragma unroll
    for (int q = 0; q < NQ; ++q)
        hnext[q] = make_float4(h2[2 * q].x, h2[2 * q].y, h2[2 * q + 1].x, h2[2 * q + 1].y);
    for (int k = K - 1; k >= 0; --k) {
        const long long t0 = (long long)k * TC;
        __syncthreads();  // the previous chunk's readers are done
        if (k + 1 < K) flush_sums(t0 + TC);
        // per (channel, step) values of this chunk, this lane's G steps
#pragma unroll
        for (int e = 0; e < G; ++e) {
            const int i = s * G + e;
            float dl = 0.f, uu = 0.f, dyh = 0.f, sig = 0.f, gz = 0.f;
            if (e < lane_valid(t0)) {
                const float raw = pr.get(e) + bias;
                uu = pu.get(e);
                dl = softplus_of(raw);
                sig = a.softplus ? rcp_approx(1.f + ex2_approx(-raw * kLog2e)) : 1.f;
                const float dy = pdy.get(e);
                if (HAS_Z) {
                    const float zt = pz.get(e);
                    const float sz = rcp_approx(1.f + ex2_approx(-zt * kLog2e));
                    dyh = dy * zt * sz;
                    gz = dy * sz * fmaf(zt, 1.f - sz, 1.f);
                } else {
                    dyh = dy;
                }
            }
            sR[sw(i, c)] = make_float4(dl, dl * uu, dyh, uu);
            sE[sw(i, c)] = make_float4(sig, gz, 0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sBC[((4 * rg + e) * 2 + rwhich) * NP + rn] = pbc.get(e);
        __syncthreads();
        float4 hstart[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) hstart[q] = hnext[q];
        if (k > 0) {  // the next chunk's inputs and checkpoint, in flight during this one
            const long long tn = t0 - TC;
            pu.load(a.u, row + tn + s * G, lane_valid(tn), vec);
            pr.load(a.delta, row + tn + s * G, lane_valid(tn), vec);
            if (HAS_Z) pz.load(a.z, row + tn + s * G, lane_valid(tn), vec);
            pdy.load(a.dy, row + tn + s * G, lane_valid(tn), vec);
            pbc.load(rwhich ? a.Cm : a.Bm, bcrow + tn + 4 * rg, row_valid(tn), vec);
#pragma unroll
            for (int q = 0; q < NQ; ++q)
                hnext[q] = (k > 1 && valid) ? *reinterpret_cast<const float4 *>(ck + (long long)(k - 1) * NP + 4 * q)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // recompute the chunk's states h_t into sH
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            h2[2 * q] = f2(hstart[q].x, hstart[q].y);
            h2[2 * q + 1] = f2(hstart[q].z, hstart[q].w);
        }
        float2 hreg[TC][NH];  // the chunk's states, also kept in registers for the reverse sweep
#pragma unroll
        for (int i = 0; i < TC; ++i) {
            const float2 r = *reinterpret_cast<const float2 *>(sR + sw(i, c));
            const float2 dl2 = f2(r.x, r.x), du2 = f2(r.y, r.y);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4 bq = *reinterpret_cast<const float4 *>(sBC + i * 2 * NP + s * NS + 4 * q);
                const float2 bb[2] = {f2(bq.x, bq.y), f2(bq.z, bq.w)};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int jp = 2 * q + h;
                    const float2 x = __fmul2_rn(dl2, A2[jp]);
                    h2[jp] = __ffma2_rn(f2(ex2_approx(x.x), ex2_approx(x.y)), h2[jp], __fmul2_rn(du2, bb[h]));
                    hreg[i][jp] = h2[jp];
                }
                sH[(i * NQ + q) * NTHR + tid] = make_float4(h2[2 * q].x, h2[2 * q].y, h2[2 * q + 1].x, h2[2 * q + 1].y);
            }
        }
        __syncthreads();
        channel_sums(std::integral_constant<int, 1>{});  // dC = sum_c dy g h
        __syncthreads();  // sH is rewritten with dh below
        // reverse sweep over the chunk; dh_t goes to sH in place of h_t once h_t has been used
        float2 ht[NH];  // h_t of the step being swept
#pragma unroll
        for (int jp = 0; jp < NH; ++jp) ht[jp] = h2[jp];
#pragma unroll
        for (int i = TC - 1; i >= 0; --i) {
            const float4 r = sR[sw(i, c)];  // Delta, Delta u, dy g, u
            const float2 dl2 = f2(r.x, r.x), dyh2 = f2(r.z, r.z);
            float2 q2 = f2(0.f, 0.f), wa2 = f2(0.f, 0.f), ch2 = f2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float4 bq = *reinterpret_cast<const float4 *>(sBC + i * 2 * NP + s * NS + 4 * q);
                const float4 cq = *reinterpret_cast<const float4 *>(sBC + (i * 2 + 1) * NP + s * NS + 4 * q);
                const float4 hv = i > 0 ? make_float4(hreg[i - 1][2 * q].x, hreg[i - 1][2 * q].y, hreg[i - 1][2 * q + 1].x,
                                                      hreg[i - 1][2 * q + 1].y)
                                        : hstart[q];  // h_{t-1}
                const float2 bb[2] = {f2(bq.x, bq.y), f2(bq.z, bq.w)}, cc2[2] = {f2(cq.x, cq.y), f2(cq.z, cq.w)};
                const float2 hp[2] = {f2(hv.x, hv.y), f2(hv.z, hv.w)};
                float2 dht[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int jp = 2 * q + h;
                    dht[h] = __ffma2_rn(dyh2, cc2[h], dh2[jp]);
                    q2 = __ffma2_rn(dht[h], bb[h], q2);
                    if (HAS_Z) ch2 = __ffma2_rn(cc2[h], ht[jp], ch2);
                    const float2 x = __fmul2_rn(dl2, A2[jp]);
                    const float2 e = f2(ex2_approx(x.x), ex2_approx(x.y));
                    const float2 w = __fmul2_rn(dht[h], __fmul2_rn(e, hp[h]));
                    dA2[jp] = __ffma2_rn(dl2, w, dA2[jp]);
                    wa2 = __ffma2_rn(A2[jp], w, wa2);
                    dh2[jp] = __fmul2_rn(dht[h], e);
                    ht[jp] = hp[h];
                }
                sH[(i * NQ + q) * NTHR + tid] = make_float4(dht[0].x, dht[0].y, dht[1].x, dht[1].y);
            }
            // sums over the channel's 4 lanes: lane s keeps the total of entry 2 (s & 1) + (s >> 1)
            float *const qrow = reinterpret_cast<float *>(sQ + sw(i, c));
            if (HAS_Z) {
                float v[4] = {q2.x + q2.y, wa2.x + wa2.y, ch2.x + ch2.y, 0.f};
                transpose_level<2, 1>(v, lane);
                transpose_level<1, 2>(v, lane);
                qrow[2 * (s & 1) + (s >> 1)] = v[0];
            } else {
                float v[2] = {q2.x + q2.y, wa2.x + wa2.y};
                transpose_level<1, 1>(v, lane);
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
                qrow[s & 1] = v[0];
            }
        }
        __syncthreads();
        channel_sums(std::integral_constant<int, 0>{});  // dB = sum_c Delta u dh
        // du, ddelta, dz of this lane's G steps
        {
            Pack<T, G> odu, odd, odz;
#pragma unroll
            for (int e = 0; e < G; ++e) {
                const int i = s * G + e;
                const float4 r = sR[sw(i, c)];
                const float4 ex = sE[sw(i, c)];
                const float4 qv = sQ[sw(i, c)];  // q, wa / ln2, C.h
                const float ddt = fmaf(r.w, qv.x, qv.y * kLn2);
                const float draw = ddt * ex.x;
                odu.set(e, fmaf(r.x, qv.x, Dd * r.z));
                odd.set(e, draw);
                if (HAS_Z) odz.set(e, ex.y * fmaf(Dd, r.w, qv.z));
                if (e < lane_valid(t0)) {
                    dDacc = fmaf(r.z, r.w, dDacc);
                    dbacc += draw;
                }
            }
            const int nv = lane_valid(t0);
            const long long o = row + t0 + s * G;
            odu.store(a.du, o, nv, vec);
            odd.store(a.ddelta, o, nv, vec);
            if (HAS_Z) odz.store(a.dz, o, nv, vec);
        }
    }
    __syncthreads();
    flush_sums(0);
    // dA, dD, dbias
#pragma unroll
    for (int jp = 0; jp < NH; ++jp) {
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            const long long n = (long long)s * NS + 2 * jp + k2;
            if (valid && n < N) atomicAdd(a.dA + dd * N + n, k2 ? dA2[jp].y : dA2[jp].x);
        }
    }
    dDacc += __shfl_xor_sync(0xffffffffu, dDacc, 1);
    dDacc += __shfl_xor_sync(0xffffffffu, dDacc, 2);
    dbacc += __shfl_xor_sync(0xffffffffu, dbacc, 1);
    dbacc += __shfl_xor_sync(0xffffffffu, dbacc, 2);
    if (valid && s == 0) {
        if (a.dD != nullptr) atomicAdd(a.dD + dd, dDacc);
        if (a.dbias != nullptr) atomicAdd(a.dbias + dd, dbacc);
    }
}

template <typename T, int NS, bool HAS_Z>
static cudaError_t launch_bwd_ns(const BwdArgs &a, long long Bsz, int K, cudaStream_t st) {
    using Sh = BwdShape<NS>;
    auto kern = scan_bwd_kernel<T, NS, HAS_Z>;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sh::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) attr_set[dev] = true;
    }
    dim3 grid((unsigned)((a.Dch + Sh::CH - 1) / Sh::CH), (unsigned)Bsz, 1);
    kern<<<grid, Sh::NTHR, Sh::SMEM_BYTES, st>>>(a, K);
    return cudaGetLastError();
}

template <typename T, int NS>
static cudaError_t launch_bwd_z(const BwdArgs &a, long long Bsz, int K, cudaStream_t st) {
    return a.z != nullptr ? launch_bwd_ns<T, NS, true>(a, Bsz, K, st) : launch_bwd_ns<T, NS, false>(a, Bsz, K, st);
}

// states per lane, steps per checkpoint chunk and padded state count for N states
static int bwd_ns(long long N) { return N <= 16 ? 4 : N <= 32 ? 8 : 16; }
int bwd_chunk_steps(long long N) { return 64 / bwd_ns(N); }

cudaError_t launch_scan_bwd(int dtype, const BwdArgs &a, long long Bsz, cudaStream_t st) {
    const int K = (int)((a.L + bwd_chunk_steps(a.N) - 1) / bwd_chunk_steps(a.N));
    switch (bwd_ns(a.N) + (dtype == 1 ? 100 : 0)) {
        case 104: return launch_bwd_z<bf16_t, 4>(a, Bsz, K, st);
        case 108: return launch_bwd_z<bf16_t, 8>(a, Bsz, K, st);
        case 116: return launch_bwd_z<bf16_t, 16>(a, Bsz, K, st);
        case 4: return launch_bwd_z<float, 4>(a, Bsz, K, st);
        case 8: return launch_bwd_z<float, 8>(a, Bsz, K, st);
        default: return launch_bwd_z<float, 16>(a, Bsz, K, st);
    }
}

}  // namespace mamba

// ---------------------------------------------------------------------------- C ABI

namespace {

using namespace mamba;

// Shape checks shared by the entry points (the checkpoint chunks are at least 4 steps).
int check_bwd_shape(int64_t Bsz, int64_t Dch, int64_t L, int64_t N, int dtype) {
    if (dtype != MAMBA_F32 && dtype != MAMBA_BF16) return MAMBA_ERR_BAD_DTYPE;
    constexpr long long kMax = 1LL << 40;
    const long long Kc = (L + 3) / 4;
    if (Bsz <= 0 || Dch <= 0 || L <= 0 || N <= 0 || Bsz > 65535 || Dch > kMax || L > kMax ||
        Bsz * Dch > kMax / L || Bsz * N > kMax / L || Bsz * Dch > kMax / (Kc * 64) || Kc > (1LL << 30))
        return MAMBA_ERR_BAD_SHAPE;
    if (N > 64) return MAMBA_ERR_UNSUPPORTED_N;
    return MAMBA_OK;
}

size_t ckpt_bytes(int64_t Bsz, int64_t Dch, int64_t L, int64_t N) {
    const long long K = (L + bwd_chunk_steps(N) - 1) / bwd_chunk_steps(N);
    return (size_t)(Bsz * Dch) * (size_t)K * (size_t)(4LL * bwd_ns(N)) * sizeof(float);
}

bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The backward kernel over caller-provided (given = 1) or call-owned checkpoints.
int run_bwd(const void *u, const void *delta, const float *A, const void *B, const void *C, const float *D,
            const void *z, const float *delta_bias, int softplus_flag, const void *dy, void *du, void *ddelta,
            float *dA, float *dB, float *dC, float *dD, void *dz, float *ddelta_bias, int64_t Bsz, int64_t Dch,
            int64_t L, int64_t N, int dtype, cudaStream_t st, float *ck, int given) {
    // the sums start from zero
    if (cudaMemsetAsync(dA, 0, (size_t)(Dch * N) * sizeof(float), st) != cudaSuccess ||
        cudaMemsetAsync(dB, 0, (size_t)(Bsz * N * L) * sizeof(float), st) != cudaSuccess ||
        cudaMemsetAsync(dC, 0, (size_t)(Bsz * N * L) * sizeof(float), st) != cudaSuccess ||
        (dD != nullptr && cudaMemsetAsync(dD, 0, (size_t)Dch * sizeof(float), st) != cudaSuccess) ||
        (ddelta_bias != nullptr && cudaMemsetAsync(ddelta_bias, 0, (size_t)Dch * sizeof(float), st) != cudaSuccess))
        return MAMBA_ERR_LAUNCH;
    BwdArgs a{};
    a.u = u;
    a.delta = delta;
    a.z = z;
    a.Bm = B;
    a.Cm = C;
    a.dy = dy;
    a.A = A;
    a.D = D;
    a.bias = delta_bias;
    a.du = du;
    a.ddelta = ddelta;
    a.dz = dz;
    a.dA = dA;
    a.dB = dB;
    a.dC = dC;
    a.dD = dD;
    a.dbias = ddelta_bias;
    a.ckpt = ck;
    a.ckpt_given = given;
    a.Dch = Dch;
    a.L = L;
    a.N = N;
    a.softplus = softplus_flag ? 1 : 0;
    a.vec = (L % 4 == 0 && aligned16(u) && aligned16(delta) && aligned16(z) && aligned16(B) && aligned16(C) &&
             aligned16(dy) && aligned16(du) && aligned16(ddelta) && aligned16(dz) && aligned16(dB) && aligned16(dC))
                ? 1
                : 0;
    return launch_scan_bwd(dtype, a, Bsz, st) == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}

}  // namespace

extern "C" size_t mamba_scan_bwd_ckpt_size(int64_t Bsz, int64_t Dch, int64_t L, int64_t N) {
    if (check_bwd_shape(Bsz, Dch, L, N, MAMBA_F32) != MAMBA_OK) return 0;
    return ckpt_bytes(Bsz, Dch, L, N);
}

extern "C" int mamba_selective_scan_bwd(const void *u, const void *delta, const float *A, const void *B,
                                        const void *C, const float *D, const void *z, const float *delta_bias,
                                        int softplus_flag, const void *dy, void *du, void *ddelta, float *dA,
                                        float *dB, float *dC, float *dD, void *dz, float *ddelta_bias, int64_t Bsz,
                                        int64_t Dch, int64_t L, int64_t N, int dtype, mamba_stream_t stream) {
    if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC) return MAMBA_ERR_NULL_ARG;
    if (z != nullptr && dz == nullptr) return MAMBA_ERR_NULL_ARG;
    int rc = check_bwd_shape(Bsz, Dch, L, N, dtype);
    if (rc != MAMBA_OK) return rc;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *ck = nullptr;
    const char *inject = std::getenv("MAMBA_FAULT_INJECT");  // host-side test hook, as in the forward scan
    if (inject != nullptr && std::strcmp(inject, "alloc") == 0) return MAMBA_ERR_ALLOC;
    if (cudaMallocAsync(&ck, ckpt_bytes(Bsz, Dch, L, N), st) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_ALLOC;
    }
    rc = run_bwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta, dA, dB, dC, dD, dz,
                 ddelta_bias, Bsz, Dch, L, N, dtype, st, static_cast<float *>(ck), 0);
    if (cudaFreeAsync(ck, st) != cudaSuccess) {
        cudaGetLastError();
        if (rc == MAMBA_OK) rc = MAMBA_ERR_LAUNCH;
    }
    return rc;
}

extern "C" int mamba_selective_scan_bwd_from_ckpt(const void *u, const void *delta, const float *A, const void *B,
                                                  const void *C, const float *D, const void *z,
                                                  const float *delta_bias, int softplus_flag, const void *dy,
                                                  const float *ckpt, void *du, void *ddelta, float *dA, float *dB,
                                                  float *dC, float *dD, void *dz, float *ddelta_bias, int64_t Bsz,
                                                  int64_t Dch, int64_t L, int64_t N, int dtype,
                                                  mamba_stream_t stream) {
    if (!u || !delta || !A || !B || !C || !dy || !ckpt || !du || !ddelta || !dA || !dB || !dC)
        return MAMBA_ERR_NULL_ARG;
    if (z != nullptr && dz == nullptr) return MAMBA_ERR_NULL_ARG;
    const int rc = check_bwd_shape(Bsz, Dch, L, N, dtype);
    if (rc != MAMBA_OK) return rc;
    if (!aligned16(ckpt)) return MAMBA_ERR_BAD_SHAPE;
    // the kernel only reads the checkpoints in this mode
    return run_bwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, dy, du, ddelta, dA, dB, dC, dD, dz,
                   ddelta_bias, Bsz, Dch, L, N, dtype, reinterpret_cast<cudaStream_t>(stream),
                   const_cast<float *>(ckpt), 1);
}

extern "C" int mamba_selective_scan_fwd_save(const void *u, const void *delta, const float *A, const void *B,
                                             const void *C, const float *D, const void *z,
                                             const float *delta_bias, int softplus_flag, void *y,
                                             float *last_state, float *ckpt, int64_t Bsz, int64_t Dch, int64_t L,
                                             int64_t N, int dtype, mamba_stream_t stream) {
    if (!u || !delta || !A || !B || !C || !y || !ckpt) return MAMBA_ERR_NULL_ARG;
    const int rc = check_bwd_shape(Bsz, Dch, L, N, dtype);
    if (rc != MAMBA_OK) return rc;
    if (!aligned16(ckpt)) return MAMBA_ERR_BAD_SHAPE;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int es = dtype == MAMBA_BF16 ? 2 : 4;
    const bool vec = aligned16(u) && aligned16(delta) && aligned16(B) && aligned16(C) && aligned16(y) &&
                     aligned16(z) && (L * es) % 16 == 0;
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
    a.chunk_len = L;
    a.nchunks = 1;
    // the direct scan on the tensor-memory kernel writes the checkpoints as it goes
    if (vec && tm_kernel_for(dtype, N)) {
        a.ckpt = ckpt;
        a.ckpt_k = (int)((L + bwd_chunk_steps(N) - 1) / bwd_chunk_steps(N));
        const cudaError_t e = launch_scan_tm(dtype, MODE_FULL, a, Bsz, 1, st);
        if (e == cudaSuccess) return MAMBA_OK;
        if (e != cudaErrorNotSupported) return MAMBA_ERR_LAUNCH;
        a.ckpt = nullptr;
    }
    // otherwise: the direct scan, then the backward kernel's own checkpoint sweep
    if (launch_scan(dtype, MODE_FULL, vec, a, Bsz, 1, st) != cudaSuccess) return MAMBA_ERR_LAUNCH;
    BwdArgs b{};
    b.u = u;
    b.delta = delta;
    b.Bm = B;
    b.Cm = C;
    b.A = A;
    b.bias = delta_bias;
    b.ckpt = ckpt;
    b.Dch = Dch;
    b.L = L;
    b.N = N;
    b.softplus = softplus_flag ? 1 : 0;
    b.vec = (L % 4 == 0 && aligned16(u) && aligned16(delta) && aligned16(B)) ? 1 : 0;
    b.sweep_only = 1;
    return launch_scan_bwd(dtype, b, Bsz, st) == cudaSuccess ? MAMBA_OK : MAMBA_ERR_LAUNCH;
}
