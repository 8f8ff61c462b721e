// scan_kernels.cuh -- the selective-scan kernel (direct scan, chunk-state pass
// and seeded rescan of the chunked scan) for sm_103a.
//
// Method: per (b, d, n), Delta_t = softplus(Delta_raw + bias_d),
// A_bar = exp(Delta_t A_{d,n}), h_t = A_bar h_{t-1} + Delta_t B_{t,n} u_t,
// y_t = sum_n C_{t,n} h_t + D_d u_t, times SiLU(z_t)
// (fsdata.site explainer §3.2 selective_step; freeguideonline tutorial §4.2,
// §4.3, §5.2 "fuse discretisation and scan, keep the state on chip").
//
// Mapping (B300: 148 SMs, fp32 FMA + f32x2 paired FMA, 16 MUFU lanes/SM/clk
// nominal):
//   * a CTA owns CH channels of one batch b and one time range (the whole
//     sequence, or one chunk of the chunked scan);
//   * each channel is split over S = NP/NS lanes of one warp; every lane keeps
//     NS fp32 states in registers for the whole time range;
//   * time advances in tiles of TT steps.  Per tile:
//       - B/C [N][TT] (shared by all CH channels) are loaded by a few threads,
//         converted to fp32 and transposed into shared memory sBC[t][n-group]
//         (double buffered: tile i+1's global loads are in flight while tile i
//         is computed);
//       - every lane loads TT/S consecutive steps of u, Delta_raw and z of its
//         channel with 16-byte loads (also one tile ahead), computes
//         Delta = softplus(.) and Delta*u for those steps only, and publishes
//         them in sDU[channel][t] so the S lanes of the channel share one
//         softplus per (b, d, t);
//       - the serial loop: per step one ex2 per state, f32x2 paired FMAs for
//         h = A_bar*h + (Delta*u)*B and the partial C.h over the lane's states;
//       - partial sums go to sP; afterwards each lane sums the S partials of
//         its own TT/S steps, adds D*u, applies the gate and stores y with
//         16-byte stores.
//   No inter-CTA communication, no spin waits.
#pragma once

#include "common.cuh"

namespace mamba {

// MODE_FULL: y (and last_state) of a chunk from its initial state.  MODE_STATES: a chunk's end state
// from zero and its sum of Delta (no y).  The tensor-memory kernel also has MODE_FULL_STATES (y from a
// zero initial state and the end state and sum of Delta) and MODE_CORR (y += the contribution of the
// chunk's entering state, decaying with no input), the two passes of the decay-truncated chunked scan.
enum { MODE_FULL = 0, MODE_STATES = 1, MODE_FULL_STATES = 2, MODE_CORR = 3 };

struct ScanArgs {
    const void *u, *delta, *z, *Bm, *Cm;
    const float *A, *D, *bias;
    void *y;
    float *last_state;
    const float *hin;  // [Bsz][K][Dch][N] initial state of every chunk (K = 1: plain h0), may be null
    float *ws_h;       // MODE_STATES: chunk end states [Bsz][K][Dch][N]
    float *ws_sdt;     // MODE_STATES: per chunk sum of Delta [Bsz][K][Dch]
    long long Dch, L, N;
    long long chunk_len;  // steps per chunk (multiple of TT); L for the direct scan
    int nchunks;          // K
    int softplus;
    // tensor-memory kernel: 0 makes a pipeline wait (loads landed, MMA done, buffer free) give up after
    // one test (test hook), anything else bounds it at about a second; the drain waits before TMEM is
    // freed keep their own limit
    unsigned wait_polls;
    int flags;            // MAMBA_FLAG_ZOH (1) | MAMBA_FLAG_REVERSE (2); honoured by the GEN instantiation only
    // non-null: `u` holds x and u = SiLU(causal width-4 conv of x) is formed in
    // the kernel (tensor-memory kernel only): taps [Dch][4], bias [Dch] or null
    const float *conv_w, *conv_b;
    int chunk0;  // MODE_CORR: chunk of blockIdx.z == 0
    // tensor-memory kernel, plain direct scan: non-null = also write the backward pass's checkpoints,
    // [Bsz][Dch][ckpt_k][4 S] (S lanes per channel): entry k >= 1 is the state before step k * 64 / S
    float *ckpt;
    int ckpt_k;
};

enum { SCAN_FLAG_ZOH = 1, SCAN_FLAG_REVERSE = 2 };

// Exact zero-order-hold weight f = (e^{Delta A} - 1) / A (Delta where A = 0)
// (freeguideonline tutorial §2.2: B_bar = (Delta A)^{-1} (exp(Delta A) - I) Delta B,
// which for a diagonal A is (exp(Delta A_n) - 1) / A_n B_n).  e = 2^{x2} is
// the decay already computed from x2 = Delta A log2 e.  e - 1 cancels for small
// |Delta A|, so there expm1 is the Taylor series to the x^7 term (truncation
// below 2e-7 relative for |x| < 1/2).  inv_a = 1/A_n (0 where A_n = 0), a_zero =
// 1 where A_n = 0 (0 elsewhere).
__device__ __forceinline__ float zoh_weight(float e, float x2, float dl, float inv_a, float a_zero) {
    const float x = x2 * kLn2;
    float p = fmaf(x, 1.0f / 5040.0f, 1.0f / 720.0f);
    p = fmaf(x, p, 1.0f / 120.0f);
    p = fmaf(x, p, 1.0f / 24.0f);
    p = fmaf(x, p, 1.0f / 6.0f);
    p = fmaf(x, p, 0.5f);
    p = fmaf(x, p, 1.0f);
    const float em1 = fabsf(x) < 0.5f ? x * p : e - 1.0f;
    return fmaf(a_zero, dl, em1 * inv_a);
}

// The same weight for a pair of steps of one state, in packed arithmetic:
// f = Delta phi(Delta A), phi(y) = (e^y - 1) / y.  x = Delta A log2 e (the
// decay's exponent), e = 2^x.  Where |Delta A| < 1/64, phi is its Taylor series
// to the y^2 term (the first dropped term, y^3/24, is below 2e-7 relative),
// written in x (coefficient k is ln2^k / (k+1)!), so that A = 0 gives f = Delta
// with no special case.  Elsewhere f = (e - 1) / A in one fused multiply-add
// (e * inv_a - inv_a): there |e - 1| > 0.0155, so the ex2 error (about 2^-22
// relative to e) is below 1.6e-5 of e - 1.  inv_a = 1/A_n (anything finite where
// A_n = 0).
__device__ __forceinline__ float2 zoh_weight2(float2 e, float2 x, float2 dl, float inv_a) {
    constexpr double l = 0.6931471805599453;
    constexpr float c1 = (float)(l / 2), c2 = (float)(l * l / 6);
    float2 p = __ffma2_rn(x, f2(c2, c2), f2(c1, c1));
    p = __ffma2_rn(x, p, f2(1.f, 1.f));
    const float2 small = __fmul2_rn(dl, p);
    const float2 big = __ffma2_rn(e, f2(inv_a, inv_a), f2(-inv_a, -inv_a));
    constexpr float xmax = (float)(1.0 / 64.0 / l);  // |Delta A| < 1/64 in units of x
    return f2(fabsf(x.x) < xmax ? small.x : big.x, fabsf(x.y) < xmax ? small.y : big.y);
}

template <int NP, int NS, int TT, int NWARPS, int MODE, int IOBYTES>
struct ScanShape {
    static constexpr int S = NP / NS;         // lanes per channel
    static constexpr int CPW = 32 / S;        // channels per warp
    static constexpr int CH = NWARPS * CPW;   // channels per CTA
    static constexpr int SEG = TT / S;        // steps per lane segment
    static constexpr int PER16 = 16 / IOBYTES;
    static constexpr int W = SEG / PER16;     // 16-byte vectors per lane segment
    static constexpr int NG = NP / 4;         // groups of 4 states
    static constexpr int TPT = PER16;         // steps per B/C staging task
    static constexpr int NTASK = (TT / TPT) * NG * 2;
    static constexpr int NTHR = NWARPS * 32;
    static constexpr int MAXT = (NTASK + NTHR - 1) / NTHR;
    static constexpr int DU_STRIDE = TT * 2 + 4;  // floats per channel row of sDU
    static constexpr int P_STRIDE = TT + 4;       // floats per (channel, lane) row of sP
    static constexpr int SMEM_FLOATS =
        2 * TT * NG * 8 + CH * DU_STRIDE + (MODE == MODE_FULL ? CH * S * P_STRIDE : 0);
    static constexpr size_t SMEM_BYTES = SMEM_FLOATS * sizeof(float);
    static_assert(NP % NS == 0 && 32 % S == 0, "lanes per channel must divide a warp");
    static_assert(NS % 4 == 0, "states per lane must be a multiple of 4");
    static_assert(W >= 1 && SEG % PER16 == 0, "lane segment must be whole 16-byte vectors");
    static_assert(SEG % 4 == 0, "lane segment must be a multiple of 4 steps");
};

// GEN: the general instantiation (scalar loads only, VEC = false) that honours
// a.flags: ZOH weights, and the reverse scan, which walks logical step tau at
// physical index L - 1 - tau (chunks, carries and h0 are all in logical order).
template <typename T, int NP, int NS, int TT, int NWARPS, int MODE, bool VEC, bool GEN = false>
__global__ void __launch_bounds__(NWARPS * 32)
scan_kernel(const ScanArgs a) {
    using Sh = ScanShape<NP, NS, TT, NWARPS, MODE, (int)sizeof(T)>;
    using IO = Io<T>;
    constexpr int S = Sh::S, CPW = Sh::CPW, CH = Sh::CH, SEG = Sh::SEG, PER16 = Sh::PER16;
    constexpr int W = Sh::W, NG = Sh::NG, TPT = Sh::TPT, NTASK = Sh::NTASK, NTHR = Sh::NTHR;
    constexpr int MAXT = Sh::MAXT, DU_STRIDE = Sh::DU_STRIDE, P_STRIDE = Sh::P_STRIDE;

    extern __shared__ float4 smem_f4[];
    float *const sBC = reinterpret_cast<float *>(smem_f4);  // [2][TT][NG][8]
    float *const sDU = sBC + 2 * TT * NG * 8;               // [CH][DU_STRIDE]
    float *const sP = sDU + CH * DU_STRIDE;                 // [CH][S][P_STRIDE]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = lane % S, cw = lane / S;
    const int c = warp * CPW + cw;
    const long long d = (long long)blockIdx.x * CH + c;
    const bool valid = d < a.Dch;
    const long long b = blockIdx.y;
    const int k = blockIdx.z;
    const long long N = a.N, L = a.L;
    const long long t_begin = (long long)k * a.chunk_len;
    const long long t_end = min(L, t_begin + a.chunk_len);
    const int ntiles = (int)((t_end - t_begin + TT - 1) / TT);
    const long long dd = valid ? d : 0;
    const long long row = (b * a.Dch + dd) * L;  // element offset of this channel's time row
    const long long bc_row0 = b * N * L;         // B/C rows of batch b
    const bool has_z = a.z != nullptr;
    static_assert(!(GEN && VEC), "the general instantiation uses scalar loads");
    const bool rev = GEN && (a.flags & SCAN_FLAG_REVERSE);
    const bool zoh = GEN && (a.flags & SCAN_FLAG_ZOH);
    auto ph = [&](long long t) { return rev ? (L - 1 - t) : t; };  // physical index of logical step t

    // ---- per-lane constants and state (states n = s*NS + j)
    float2 A2[NS / 2];  // A * log2(e), so A_bar = 2^(Delta * A2)
    float2 h[NS / 2];
    float2 invA[GEN ? NS / 2 : 1], aZero[GEN ? NS / 2 : 1];  // ZOH: 1/A (0 at A = 0), [A = 0]
#pragma unroll
    for (int j = 0; j < NS; j += 2) {
        const long long n0 = (long long)s * NS + j;
        float a0 = 0.f, a1 = 0.f, h0 = 0.f, h1 = 0.f;
        if (valid && n0 < N) a0 = a.A[dd * N + n0] * kLog2e;
        if (valid && n0 + 1 < N) a1 = a.A[dd * N + n0 + 1] * kLog2e;
        if (a.hin != nullptr) {
            const long long base = ((b * a.nchunks + k) * a.Dch + dd) * N;
            if (valid && n0 < N) h0 = a.hin[base + n0];
            if (valid && n0 + 1 < N) h1 = a.hin[base + n0 + 1];
        }
        A2[j / 2] = make_float2(a0, a1);
        h[j / 2] = make_float2(h0, h1);
        if constexpr (GEN) {
            invA[j / 2] = make_float2(a0 != 0.f ? kLog2e / a0 : 0.f, a1 != 0.f ? kLog2e / a1 : 0.f);
            aZero[j / 2] = make_float2(a0 == 0.f ? 1.f : 0.f, a1 == 0.f ? 1.f : 0.f);
        }
    }
    const float Dd = (a.D != nullptr && valid) ? a.D[dd] : 0.f;
    const float bias = (a.bias != nullptr && valid) ? a.bias[dd] : 0.f;

    // ---- B/C staging: task q -> (which, g, tq); consecutive q read consecutive 16 B of a row
    uint4 rbc[MAXT][4];
    auto bc_load = [&](int tile) {
        const long long t0 = t_begin + (long long)tile * TT;
#pragma unroll
        for (int m = 0; m < MAXT; ++m) {
            const int q = tid + m * NTHR;
            if (q < NTASK) {
                const int tq = q % (TT / TPT);
                const int g = (q / (TT / TPT)) % NG;
                const int which = q / ((TT / TPT) * NG);
                const void *base = which ? a.Cm : a.Bm;
                const long long tt = t0 + (long long)tq * TPT;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const long long n = 4LL * g + j;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (n < N) {
                        const long long off = bc_row0 + n * L;
                        if (VEC && tt + TPT <= t_end) {
                            v = ldg16(reinterpret_cast<const T *>(base) + off + tt);
                        } else {
#pragma unroll
                            for (int i = 0; i < TPT; ++i)
                                if (tt + i < t_end) IO::set(v, i, IO::load(base, off + ph(tt + i)));
                        }
                    }
                    rbc[m][j] = v;
                }
            }
        }
    };
    auto bc_store = [&](int buf) {
#pragma unroll
        for (int m = 0; m < MAXT; ++m) {
            const int q = tid + m * NTHR;
            if (q < NTASK) {
                const int tq = q % (TT / TPT);
                const int g = (q / (TT / TPT)) % NG;
                const int which = q / ((TT / TPT) * NG);
#pragma unroll
                for (int i = 0; i < TPT; ++i) {
                    const float4 v = make_float4(IO::get(rbc[m][0], i), IO::get(rbc[m][1], i),
                                                 IO::get(rbc[m][2], i), IO::get(rbc[m][3], i));
                    *reinterpret_cast<float4 *>(sBC + ((buf * TT + tq * TPT + i) * NG + g) * 8 + which * 4) = v;
                }
            }
        }
    };

    // ---- per-lane segment of u, Delta_raw, z: steps [tile*TT + s*SEG, +SEG)
    uint4 ru[W], rd[W], rz[W];
    auto seg_load = [&](int tile, uint4 (&xu)[W], uint4 (&xd)[W], uint4 (&xz)[W]) {
        const long long t0 = t_begin + (long long)tile * TT + (long long)s * SEG;
        const T *pu = reinterpret_cast<const T *>(a.u) + row + t0;
        const T *pd = reinterpret_cast<const T *>(a.delta) + row + t0;
        const T *pz = reinterpret_cast<const T *>(a.z) + row + t0;
        if (VEC && valid && t0 + SEG <= t_end) {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                xu[w] = ldg16(pu + w * PER16);
                xd[w] = ldg16(pd + w * PER16);
                xz[w] = has_z ? ldg16(pz + w * PER16) : make_uint4(0u, 0u, 0u, 0u);
            }
        } else {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                uint4 vu = make_uint4(0u, 0u, 0u, 0u), vd = vu, vz = vu;
#pragma unroll
                for (int i = 0; i < PER16; ++i) {
                    const long long t = t0 + w * PER16 + i;
                    if (valid && t < t_end) {
                        IO::set(vu, i, IO::load(a.u, row + ph(t)));
                        IO::set(vd, i, IO::load(a.delta, row + ph(t)));
                        if (has_z) IO::set(vz, i, IO::load(a.z, row + ph(t)));
                    }
                }
                xu[w] = vu;
                xd[w] = vd;
                xz[w] = vz;
            }
        }
    };

    float sdt_acc = 0.f;  // MODE_STATES: this lane's share of sum(Delta) over the chunk
    float *const du_row = sDU + c * DU_STRIDE;

    // ---- prologue: tile 0 staged
    bc_load(0);
    seg_load(0, ru, rd, rz);
    bc_store(0);
    __syncthreads();

    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        const bool has_next = tile + 1 < ntiles;
        uint4 nu[W], nd[W], nz[W];
        if (has_next) {
            bc_load(tile + 1);
            seg_load(tile + 1, nu, nd, nz);
        }

        // Delta and Delta*u for this lane's steps, shared with the other lanes of the channel
        {
            const long long t0 = t_begin + (long long)tile * TT + (long long)s * SEG;
#pragma unroll
            for (int i = 0; i < SEG; i += 2) {
                float o[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int ii = i + e;
                    const float raw = IO::get(rd[ii / PER16], ii % PER16) + bias;
                    float dl = a.softplus ? softplus_f(raw) : raw;
                    if (!(valid && t0 + ii < t_end)) dl = 0.f;  // masked step: state unchanged
                    o[2 * e] = dl;
                    // ZOH keeps u itself: its weight depends on the state
                    o[2 * e + 1] = zoh ? (dl != 0.f ? IO::get(ru[ii / PER16], ii % PER16) : 0.f)
                                       : dl * IO::get(ru[ii / PER16], ii % PER16);
                    sdt_acc += dl;
                }
                *reinterpret_cast<float4 *>(du_row + (s * SEG + i) * 2) = make_float4(o[0], o[1], o[2], o[3]);
            }
        }
        __syncwarp();

        // the serial recurrence over the tile
        {
            const float *bc = sBC + buf * TT * NG * 8 + (s * (NS / 4)) * 8;
            float *prow = sP + (c * S + s) * P_STRIDE;
            float pq[4];
#pragma unroll
            for (int t = 0; t < TT; t += 2) {
                const float4 du2 = *reinterpret_cast<const float4 *>(du_row + t * 2);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float dl = e ? du2.z : du2.x;
                    const float du = e ? du2.w : du2.y;
                    const float *bct = bc + (t + e) * NG * 8;
                    const float2 dl2 = make_float2(dl, dl);
                    const float2 du2v = make_float2(du, du);
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int g = 0; g < NS / 4; ++g) {
                        const float4 Bv = *reinterpret_cast<const float4 *>(bct + g * 8);
                        const float2 x01 = __fmul2_rn(dl2, A2[2 * g]);
                        const float2 x23 = __fmul2_rn(dl2, A2[2 * g + 1]);
                        const float2 a01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
                        const float2 a23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
                        float2 bu01 = __fmul2_rn(du2v, make_float2(Bv.x, Bv.y));
                        float2 bu23 = __fmul2_rn(du2v, make_float2(Bv.z, Bv.w));
                        if constexpr (GEN) {
                            if (zoh) {  // du2v holds u: B_bar u = f_n u B_n
                                const float2 iA01 = invA[2 * g], iA23 = invA[2 * g + 1];
                                const float2 z01 = aZero[2 * g], z23 = aZero[2 * g + 1];
                                const float2 f01 = make_float2(zoh_weight(a01.x, x01.x, dl, iA01.x, z01.x),
                                                               zoh_weight(a01.y, x01.y, dl, iA01.y, z01.y));
                                const float2 f23 = make_float2(zoh_weight(a23.x, x23.x, dl, iA23.x, z23.x),
                                                               zoh_weight(a23.y, x23.y, dl, iA23.y, z23.y));
                                bu01 = __fmul2_rn(__fmul2_rn(f01, du2v), make_float2(Bv.x, Bv.y));
                                bu23 = __fmul2_rn(__fmul2_rn(f23, du2v), make_float2(Bv.z, Bv.w));
                            }
                        }
                        h[2 * g] = __ffma2_rn(a01, h[2 * g], bu01);
                        h[2 * g + 1] = __ffma2_rn(a23, h[2 * g + 1], bu23);
                        if (MODE == MODE_FULL) {
                            const float4 Cv = *reinterpret_cast<const float4 *>(bct + g * 8 + 4);
                            acc0 = __ffma2_rn(make_float2(Cv.x, Cv.y), h[2 * g], acc0);
                            acc1 = __ffma2_rn(make_float2(Cv.z, Cv.w), h[2 * g + 1], acc1);
                        }
                    }
                    if (MODE == MODE_FULL) {
                        const float2 acc = __fadd2_rn(acc0, acc1);
                        pq[(t + e) & 3] = acc.x + acc.y;
                    }
                }
                if (MODE == MODE_FULL && (t & 3) == 2)
                    *reinterpret_cast<float4 *>(prow + t - 2) = make_float4(pq[0], pq[1], pq[2], pq[3]);
            }
        }

        if (MODE == MODE_FULL) {
            __syncwarp();
            // y for this lane's own steps: sum the S partials, add D*u, gate, store
            const long long t0 = t_begin + (long long)tile * TT + (long long)s * SEG;
            float yv[SEG];
#pragma unroll
            for (int i = 0; i < SEG; ++i) yv[i] = 0.f;
#pragma unroll
            for (int s2 = 0; s2 < S; ++s2) {
                const float *pr = sP + (c * S + s2) * P_STRIDE + s * SEG;
#pragma unroll
                for (int i = 0; i < SEG; i += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(pr + i);
                    yv[i] += v.x;
                    yv[i + 1] += v.y;
                    yv[i + 2] += v.z;
                    yv[i + 3] += v.w;
                }
            }
#pragma unroll
            for (int i = 0; i < SEG; ++i) {
                const float uu = IO::get(ru[i / PER16], i % PER16);
                float yy = fmaf(Dd, uu, yv[i]);
                if (has_z) yy *= silu_f(IO::get(rz[i / PER16], i % PER16));
                yv[i] = yy;
            }
            T *py = reinterpret_cast<T *>(a.y) + row + t0;
            if (VEC && valid && t0 + SEG <= t_end) {
#pragma unroll
                for (int w = 0; w < W; ++w) stg16(py + w * PER16, IO::pack(yv + w * PER16));
            } else if (valid) {
#pragma unroll
                for (int i = 0; i < SEG; ++i)
                    if (t0 + i < t_end) IO::store(a.y, row + ph(t0 + i), yv[i]);
            }
        }

        if (has_next) bc_store(buf ^ 1);
        __syncthreads();
        if (has_next) {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                ru[w] = nu[w];
                rd[w] = nd[w];
                rz[w] = nz[w];
            }
        }
    }

    // ---- epilogue
    if (MODE == MODE_STATES) {
#pragma unroll
        for (int off = 1; off < S; off <<= 1) sdt_acc += __shfl_xor_sync(0xffffffffu, sdt_acc, off);
        if (valid) {
            const long long base = (b * a.nchunks + k) * a.Dch + d;
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                const long long n = (long long)s * NS + j;
                if (n < N) a.ws_h[base * N + n] = (j & 1) ? h[j / 2].y : h[j / 2].x;
            }
            if (s == 0) a.ws_sdt[base] = sdt_acc;
        }
    } else if (a.last_state != nullptr && valid && k == a.nchunks - 1) {
#pragma unroll
        for (int j = 0; j < NS; ++j) {
            const long long n = (long long)s * NS + j;
            if (n < N) a.last_state[(b * a.Dch + d) * N + n] = (j & 1) ? h[j / 2].y : h[j / 2].x;
        }
    }
}

}  // namespace mamba
