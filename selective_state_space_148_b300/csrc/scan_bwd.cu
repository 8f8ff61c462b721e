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
// h_{t-1} is needed in reverse order, so states are recomputed by chunks: a
// forward sweep writes the state at every chunk start (TC steps apart) to a
// checkpoint workspace; then, chunk by chunk from the end, the chunk's states
// are recomputed into shared memory from its checkpoint and swept in reverse.
// Mapping: 4 lanes per channel, NS states per lane (N <= 4 NS), 32 channels
// per CTA.  Each chunk's inputs (u, Delta_raw, z, dy rows of the CTA's
// channels, B and C rows) are staged in shared memory with coalesced loads, and
// its du, ddelta, dz rows leave through shared memory the same way.  B and C
// are shared by every channel of a batch, so dB and dC are
// sums over channels: each lane writes its per-step terms to shared memory,
// the CTA sums them over its 32 channels at the end of a chunk and adds the
// sums to dB, dC with one atomic add per CTA and element.  dA, dD and dbias
// (sums over batches and steps) are kept in registers and added atomically at
// the end.  No device-side waits.
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
    float *ckpt;  // [Bsz][Dch][K][N]: state before step k * TC
    long long Dch, L, N;
    int softplus;
};

template <typename T, int NS>
struct BwdShape {
    static constexpr int S = 4, CH = 32, NTHR = S * CH;
    static constexpr int TC = 32 / NS;  // steps per chunk: TC * NS = 32 states kept per lane
    static constexpr int NP = S * NS;   // padded state count
    // shared memory, floats: recomputed states [TC][NS][NTHR]; the dB, dC terms [TC][NP][CHP] each (channel
    // innermost, padded to 33 so that the sum over channels reads distinct banks; a term of channel c and
    // state slice s goes to column (c + ROT s) mod 32, which puts the 32 lanes of a warp's store in 32
    // banks, and the sum over a row does not depend on the column order); the chunk's inputs u, Delta_raw,
    // z, dy [4][CH][TCP] and B, C [2][TC][NP]; outputs du, ddelta, dz [3][CH][TCP] (rows padded to TCP =
    // TC + 1 so that the 8 channels of a warp read distinct banks)
    static constexpr int CHP = CH + 1, TCP = TC + 1, ROT = (8 - NS) & 31;
    static constexpr int SH_FLOATS = TC * NS * NTHR, SD_FLOATS = TC * NP * CHP;
    static constexpr int IN_FLOATS = 4 * CH * TCP, BC_FLOATS = 2 * TC * NP, OUT_FLOATS = 3 * CH * TCP;
    static_assert(CH == 32, "the column rotation permutes 32 channels");
    static constexpr size_t SMEM_BYTES =
        (SH_FLOATS + 2 * SD_FLOATS + IN_FLOATS + BC_FLOATS + OUT_FLOATS) * sizeof(float);
};

// NS consecutive floats of shared memory (16-byte aligned) into registers with 16-byte loads
template <int NS>
__device__ __forceinline__ void load_vec(float (&v)[NS], const float *p) {
#pragma unroll
    for (int k = 0; k < NS; k += 4) {
        const float4 q = *reinterpret_cast<const float4 *>(p + k);
        v[k] = q.x;
        v[k + 1] = q.y;
        v[k + 2] = q.z;
        v[k + 3] = q.w;
    }
}

template <typename T, int NS>
__global__ void __launch_bounds__(128)
scan_bwd_kernel(const BwdArgs a, long long K) {
    using Sh = BwdShape<T, NS>;
    using IO = Io<T>;
    constexpr int CH = Sh::CH, NTHR = Sh::NTHR, TC = Sh::TC, NP = Sh::NP;
    extern __shared__ float4 smem_f4[];
    float *const sH = reinterpret_cast<float *>(smem_f4);  // [TC][NS][NTHR]
    float *const sdB = sH + Sh::SH_FLOATS;     // [TC][NP][CHP]
    float *const sdC = sdB + Sh::SD_FLOATS;
    float *const sIn = sdC + Sh::SD_FLOATS;    // [4][CH][TC]: u, Delta_raw, z, dy
    float *const sBC = sIn + Sh::IN_FLOATS;    // [2][TC][NP]: B, C
    float *const sOut = sBC + Sh::BC_FLOATS;   // [3][CH][TC]: du, ddelta, dz

    const int tid = threadIdx.x, s = tid & 3, c = tid >> 2;
    const long long d = (long long)blockIdx.x * CH + c;
    const bool valid = d < a.Dch;
    const long long dd = valid ? d : 0;
    const long long b = blockIdx.y;
    const long long N = a.N, L = a.L;
    const long long bc0 = b * N * L;
    const bool has_z = a.z != nullptr;

    // per-state values in pairs of adjacent states (f32x2 arithmetic)
    constexpr int NH = NS / 2;
    float2 Anp[NH], A2p[NH], h2[NH];
    bool live[NS];
#pragma unroll
    for (int jp = 0; jp < NH; ++jp) {
        float v[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int j = 2 * jp + k;
            const long long n = (long long)s * NS + j;
            live[j] = valid && n < N;
            v[k] = live[j] ? a.A[dd * N + n] : 0.f;
        }
        Anp[jp] = f2(v[0], v[1]);
        A2p[jp] = f2(v[0] * kLog2e, v[1] * kLog2e);
        h2[jp] = f2(0.f, 0.f);
    }
    const float Dd = (a.D != nullptr && valid) ? a.D[dd] : 0.f;
    const float bias = (a.bias != nullptr && valid) ? a.bias[dd] : 0.f;
    float *const ck = a.ckpt + ((b * a.Dch + dd) * K) * N + (long long)s * NS;
    constexpr int TCP = Sh::TCP;
    const float *const in_u = sIn + c * TCP, *const in_r = sIn + (CH + c) * TCP;
    const float *const in_z = sIn + (2 * CH + c) * TCP, *const in_dy = sIn + (3 * CH + c) * TCP;
    const int dcol = (c + Sh::ROT * s) & 31;  // this lane's column in the dB/dC term rows

    // Inputs of steps t0 .. t0 + nt - 1 (zero past the end, past Dch, past N): loaded into registers one
    // chunk ahead (load_chunk), written to shared memory when the chunk starts (store_chunk).  ntens = 2: u
    // and Delta_raw with B (the forward sweep); 4: also z and dy, with B and C.
    constexpr int PT = TC, PB = 2;  // elements per thread: 4 * CH * TC / NTHR and 2 * NP * TC / NTHR
    static_assert(4 * CH * TC == PT * NTHR && 2 * NP * TC == PB * NTHR, "staging splits evenly");
    float pt[PT], pb[PB];
    auto load_chunk = [&](long long t0, int nt, int ntens) {
#pragma unroll
        for (int r = 0; r < PT; ++r) {
            const int q = tid + r * NTHR;
            const int tens = q / (CH * TC), cc = (q / TC) % CH, i = q % TC;
            const long long dch = (long long)blockIdx.x * CH + cc;
            const void *p = tens == 0 ? a.u : tens == 1 ? a.delta : tens == 2 ? a.z : a.dy;
            float v = 0.f;
            if (tens < ntens && i < nt && dch < a.Dch && p != nullptr) v = IO::load(p, (b * a.Dch + dch) * L + t0 + i);
            pt[r] = v;
        }
#pragma unroll
        for (int r = 0; r < PB; ++r) {
            const int q = tid + r * NTHR;
            const int which = q / (NP * TC), n = (q / TC) % NP, i = q % TC;
            float v = 0.f;
            if ((which == 0 || ntens == 4) && i < nt && n < N)
                v = IO::load(which ? a.Cm : a.Bm, bc0 + (long long)n * L + t0 + i);
            pb[r] = v;
        }
    };
    auto store_chunk = [&]() {
#pragma unroll
        for (int r = 0; r < PT; ++r) {
            const int q = tid + r * NTHR;  // (tensor, channel) row q / TC, step q % TC
            sIn[(q / TC) * TCP + q % TC] = pt[r];
        }
#pragma unroll
        for (int r = 0; r < PB; ++r) {
            const int q = tid + r * NTHR;
            const int which = q / (NP * TC), n = (q / TC) % NP, i = q % TC;
            sBC[(which * TC + i) * NP + n] = pb[r];
        }
    };
    auto softplus_of = [&](float raw) { return a.softplus ? softplus_f(raw) : raw; };

    auto chunk_len = [&](long long k) { return (int)min((long long)TC, L - k * TC); };
    // ---- forward sweep: checkpoint the state before every chunk.  It stages FW chunks (TW steps) of u,
    // Delta_raw and B at a time, one window ahead, in the dB/dC scratch, which is idle until the reverse sweep.
    constexpr int FW = 4, TW = FW * TC;
    constexpr int FT = 2 * CH * TW / NTHR, FB = NP * TW / NTHR;  // elements per thread: u/Delta_raw, B
    static_assert(2 * CH * TW == FT * NTHR && NP * TW == FB * NTHR, "window staging splits evenly");
    constexpr int TWP = TW + 1;  // padded rows: the 8 channels of a warp read distinct banks
    static_assert(2 * CH * TWP + NP * TW <= 2 * Sh::SD_FLOATS, "the window fits the dB/dC scratch");
    float *const wIn = sdB;                // [2][CH][TWP]: u, Delta_raw
    float *const wB = sdB + 2 * CH * TWP;  // [TW][NP]
    float ft[FT], fb[FB];
    auto load_window = [&](long long t0) {
#pragma unroll
        for (int r = 0; r < FT; ++r) {
            const int q = tid + r * NTHR;
            const int tens = q / (CH * TW), cc = (q / TW) % CH, i = q % TW;
            const long long dch = (long long)blockIdx.x * CH + cc;
            ft[r] = (t0 + i < L && dch < a.Dch) ? IO::load(tens ? a.delta : a.u, (b * a.Dch + dch) * L + t0 + i) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < FB; ++r) {
            const int q = tid + r * NTHR;
            const int n = q / TW, i = q % TW;
            fb[r] = (t0 + i < L && n < N) ? IO::load(a.Bm, bc0 + (long long)n * L + t0 + i) : 0.f;
        }
    };
    auto store_window = [&]() {
#pragma unroll
        for (int r = 0; r < FT; ++r) {
            const int q = tid + r * NTHR;
            wIn[(q / TW) * TWP + q % TW] = ft[r];
        }
#pragma unroll
        for (int r = 0; r < FB; ++r) {
            const int q = tid + r * NTHR;
            wB[(q % TW) * NP + q / TW] = fb[r];
        }
    };
    const long long nwin = (L + TW - 1) / TW;
    load_window(0);
    for (long long w = 0; w < nwin; ++w) {
        __syncthreads();
        store_window();
        __syncthreads();
        if (w + 1 < nwin) load_window((w + 1) * TW);  // in flight during this window
#pragma unroll
        for (int i = 0; i < TW; ++i) {
            const long long t = w * TW + i;
            if (t < L) {  // uniform
                if (i % TC == 0) {
#pragma unroll
                    for (int j = 0; j < NS; ++j)
                        if (live[j]) ck[(t / TC) * N + j] = (j & 1) ? h2[j / 2].y : h2[j / 2].x;
                }
                const float dl = softplus_of(wIn[(CH + c) * TWP + i] + bias);
                const float du = dl * wIn[c * TWP + i];
                const float2 dl2 = f2(dl, dl), du2 = f2(du, du);
                const float2 *wb = reinterpret_cast<const float2 *>(wB + i * NP + s * NS);
#pragma unroll
                for (int jp = 0; jp < NH; ++jp) {
                    const float2 x = __fmul2_rn(dl2, A2p[jp]);
                    h2[jp] = __ffma2_rn(f2(ex2_approx(x.x), ex2_approx(x.y)), h2[jp], __fmul2_rn(du2, wb[jp]));
                }
            }
        }
    }

    // ---- reverse sweep, chunk by chunk
    float2 dh2[NH], dA2[NH];
#pragma unroll
    for (int jp = 0; jp < NH; ++jp) dh2[jp] = dA2[jp] = f2(0.f, 0.f);
    float dDacc = 0.f, dbacc = 0.f;
    float hnext[NS];  // checkpoint of the next chunk to process, loaded one chunk ahead
    load_chunk((K - 1) * TC, chunk_len(K - 1), 4);
#pragma unroll
    for (int j = 0; j < NS; ++j) hnext[j] = live[j] ? ck[(K - 1) * N + j] : 0.f;
    for (long long k = K - 1; k >= 0; --k) {
        const long long t0 = k * TC;
        const int nt = chunk_len(k);
        __syncthreads();
        store_chunk();
        __syncthreads();
        float hstart[NS], dlr[TC];
#pragma unroll
        for (int j = 0; j < NS; ++j) hstart[j] = hnext[j];
#pragma unroll
        for (int jp = 0; jp < NH; ++jp) h2[jp] = f2(hnext[2 * jp], hnext[2 * jp + 1]);
        if (k > 0) {  // in flight during this chunk
            load_chunk((k - 1) * TC, TC, 4);
#pragma unroll
            for (int j = 0; j < NS; ++j) hnext[j] = live[j] ? ck[(k - 1) * N + j] : 0.f;
        }
        // the chunk body, without per-step length tests for whole chunks (all but possibly the last)
        auto sweep = [&](auto full_tag) {
            constexpr bool FULLC = decltype(full_tag)::value;
#pragma unroll
            for (int i = 0; i < TC; ++i) {  // recompute the chunk's states (private to this lane)
                dlr[i] = 0.f;
                if (FULLC || i < nt) {
                    const float dl = softplus_of(in_r[i] + bias);
                    dlr[i] = dl;
                    const float du = dl * in_u[i];
                    const float2 dl2 = f2(dl, dl), du2 = f2(du, du);
                    const float2 *bp = reinterpret_cast<const float2 *>(sBC + i * NP + s * NS);
#pragma unroll
                    for (int jp = 0; jp < NH; ++jp) {
                        const float2 x = __fmul2_rn(dl2, A2p[jp]);
                        h2[jp] = __ffma2_rn(f2(ex2_approx(x.x), ex2_approx(x.y)), h2[jp], __fmul2_rn(du2, bp[jp]));
                        sH[(i * NS + 2 * jp) * NTHR + tid] = h2[jp].x;
                        sH[(i * NS + 2 * jp + 1) * NTHR + tid] = h2[jp].y;
                    }
                }
            }
            float hcur[NS];  // h_t of the step being swept (h_{t-1} of the step after it)
#pragma unroll
            for (int j = 0; j < NS; ++j) hcur[j] = sH[((FULLC ? TC - 1 : nt - 1) * NS + j) * NTHR + tid];
#pragma unroll
            for (int i = TC - 1; i >= 0; --i) {
                if (!FULLC && i >= nt) continue;
                const float dl = dlr[i];
                const float raw = in_r[i] + bias;
                const float uu = in_u[i], dyt = in_dy[i];
                float Bt[NS], Ct[NS], hprev[NS];
                load_vec<NS>(Bt, sBC + i * NP + s * NS);
                load_vec<NS>(Ct, sBC + (TC + i) * NP + s * NS);
#pragma unroll
                for (int j = 0; j < NS; ++j) hprev[j] = i > 0 ? sH[((i - 1) * NS + j) * NTHR + tid] : hstart[j];
                float g = 1.f, dzt = 0.f;
                if (has_z) {  // yhat = C . h_t + D u, the C . h part summed over the 4 lanes
                    float2 ch2 = f2(0.f, 0.f);
#pragma unroll
                    for (int jp = 0; jp < NH; ++jp)
                        ch2 = __ffma2_rn(f2(Ct[2 * jp], Ct[2 * jp + 1]), f2(hcur[2 * jp], hcur[2 * jp + 1]), ch2);
                    float ch = ch2.x + ch2.y;
                    ch += __shfl_xor_sync(0xffffffffu, ch, 1);
                    ch += __shfl_xor_sync(0xffffffffu, ch, 2);
                    const float zt = in_z[i];
                    const float sg = rcp_approx(1.f + ex2_approx(-zt * kLog2e));
                    g = zt * sg;
                    dzt = dyt * fmaf(Dd, uu, ch) * sg * fmaf(zt, 1.f - sg, 1.f);
                }
                const float dyh = dyt * g;
                // with dh_n after the C term and w_n = dh_n a_n h_{t-1,n}:  du gets Delta q, dDelta gets u q +
                // sum_n A_n w_n (q = sum_n dh_n B_n), dA_n gets Delta w_n
                const float dluu = dl * uu;
                const float2 dl2 = f2(dl, dl), dluu2 = f2(dluu, dluu), dyh2 = f2(dyh, dyh);
                float2 q2 = f2(0.f, 0.f), wa2 = f2(0.f, 0.f);
#pragma unroll
                for (int jp = 0; jp < NH; ++jp) {
                    const int j = 2 * jp;
                    const float2 ht = f2(hcur[j], hcur[j + 1]), hp = f2(hprev[j], hprev[j + 1]);
                    hcur[j] = hp.x;
                    hcur[j + 1] = hp.y;
                    const float2 tc = __fmul2_rn(dyh2, ht);
                    sdC[(i * NP + s * NS + j) * Sh::CHP + dcol] = tc.x;
                    sdC[(i * NP + s * NS + j + 1) * Sh::CHP + dcol] = tc.y;
                    const float2 dhj = __ffma2_rn(dyh2, f2(Ct[j], Ct[j + 1]), dh2[jp]);
                    const float2 x = __fmul2_rn(dl2, A2p[jp]);
                    const float2 e = f2(ex2_approx(x.x), ex2_approx(x.y));
                    const float2 tb = __fmul2_rn(dhj, dluu2);
                    sdB[(i * NP + s * NS + j) * Sh::CHP + dcol] = tb.x;
                    sdB[(i * NP + s * NS + j + 1) * Sh::CHP + dcol] = tb.y;
                    q2 = __ffma2_rn(dhj, f2(Bt[j], Bt[j + 1]), q2);  // (Bt, Ct from the chunk's B/C rows)
                    const float2 w = __fmul2_rn(dhj, __fmul2_rn(e, hp));
                    dA2[jp] = __ffma2_rn(dl2, w, dA2[jp]);
                    wa2 = __ffma2_rn(Anp[jp], w, wa2);
                    dh2[jp] = __fmul2_rn(dhj, e);
                }
                const float q = q2.x + q2.y, wa = wa2.x + wa2.y;
                float dup = dl * q, ddt = fmaf(uu, q, wa);
                dup += __shfl_xor_sync(0xffffffffu, dup, 1);
                dup += __shfl_xor_sync(0xffffffffu, dup, 2);
                ddt += __shfl_xor_sync(0xffffffffu, ddt, 1);
                ddt += __shfl_xor_sync(0xffffffffu, ddt, 2);
                if (s == 0) {
                    const float draw = a.softplus ? ddt * rcp_approx(1.f + ex2_approx(-raw * kLog2e)) : ddt;
                    sOut[c * TCP + i] = fmaf(Dd, dyh, dup);
                    sOut[(CH + c) * TCP + i] = draw;
                    sOut[(2 * CH + c) * TCP + i] = dzt;
                    if (valid) {
                        dDacc = fmaf(dyh, uu, dDacc);
                        dbacc += draw;
                    }
                }
            }
        };
        if (nt == TC)
            sweep(std::true_type{});
        else
            sweep(std::false_type{});
        __syncthreads();
        // this chunk's du, ddelta, dz rows, and dB, dC summed over the CTA's channels (one atomic add
        // per CTA and element)
        for (int q = tid; q < (has_z ? 3 : 2) * CH * TC; q += NTHR) {
            const int tens = q / (CH * TC), cc = (q / TC) % CH, i = q % TC;
            const long long dch = (long long)blockIdx.x * CH + cc;
            if (i < nt && dch < a.Dch)
                IO::store(tens == 0 ? a.du : tens == 1 ? a.ddelta : a.dz, (b * a.Dch + dch) * L + t0 + i,
                          sOut[(q / TC) * TCP + i]);
        }
        for (int q = tid; q < nt * NP; q += NTHR) {
            const int i = q / NP, n = q % NP;
            if (n < N) {
                const float *pb = sdB + (i * NP + n) * Sh::CHP, *pc = sdC + (i * NP + n) * Sh::CHP;
                float sb4[4] = {0.f, 0.f, 0.f, 0.f}, sc4[4] = {0.f, 0.f, 0.f, 0.f};  // four independent chains
#pragma unroll
                for (int cc = 0; cc < CH; ++cc) {
                    sb4[cc & 3] += pb[cc];
                    sc4[cc & 3] += pc[cc];
                }
                const float sb = (sb4[0] + sb4[1]) + (sb4[2] + sb4[3]), sc = (sc4[0] + sc4[1]) + (sc4[2] + sc4[3]);
                atomicAdd(a.dB + bc0 + (long long)n * L + t0 + i, sb);
                atomicAdd(a.dC + bc0 + (long long)n * L + t0 + i, sc);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NS; ++j)
        if (live[j]) atomicAdd(a.dA + dd * N + (long long)s * NS + j, (j & 1) ? dA2[j / 2].y : dA2[j / 2].x);
    if (valid && s == 0) {
        if (a.dD != nullptr) atomicAdd(a.dD + dd, dDacc);
        if (a.dbias != nullptr) atomicAdd(a.dbias + dd, dbacc);
    }
}

template <typename T, int NS>
static cudaError_t launch_bwd_ns(const BwdArgs &a, long long Bsz, long long K, cudaStream_t st) {
    using Sh = BwdShape<T, NS>;
    auto kern = scan_bwd_kernel<T, NS>;
    if (Sh::SMEM_BYTES > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sh::SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)((a.Dch + Sh::CH - 1) / Sh::CH), (unsigned)Bsz, 1);
    kern<<<grid, Sh::NTHR, Sh::SMEM_BYTES, st>>>(a, K);
    return cudaGetLastError();
}

// steps per checkpoint chunk for N states
int bwd_chunk_steps(long long N) { return N <= 16 ? 8 : N <= 32 ? 4 : 2; }

cudaError_t launch_scan_bwd(int dtype, const BwdArgs &a, long long Bsz, cudaStream_t st) {
    const long long K = (a.L + bwd_chunk_steps(a.N) - 1) / bwd_chunk_steps(a.N);
    if (dtype == 1) {
        if (a.N <= 16) return launch_bwd_ns<bf16_t, 4>(a, Bsz, K, st);
        if (a.N <= 32) return launch_bwd_ns<bf16_t, 8>(a, Bsz, K, st);
        return launch_bwd_ns<bf16_t, 16>(a, Bsz, K, st);
    }
    if (a.N <= 16) return launch_bwd_ns<float, 4>(a, Bsz, K, st);
    if (a.N <= 32) return launch_bwd_ns<float, 8>(a, Bsz, K, st);
    return launch_bwd_ns<float, 16>(a, Bsz, K, st);
}

}  // namespace mamba

// ---------------------------------------------------------------------------- C ABI

extern "C" int mamba_selective_scan_bwd(const void *u, const void *delta, const float *A, const void *B,
                                        const void *C, const float *D, const void *z, const float *delta_bias,
                                        int softplus_flag, const void *dy, void *du, void *ddelta, float *dA,
                                        float *dB, float *dC, float *dD, void *dz, float *ddelta_bias, int64_t Bsz,
                                        int64_t Dch, int64_t L, int64_t N, int dtype, mamba_stream_t stream) {
    using namespace mamba;
    if (!u || !delta || !A || !B || !C || !dy || !du || !ddelta || !dA || !dB || !dC) return MAMBA_ERR_NULL_ARG;
    if (z != nullptr && dz == nullptr) return MAMBA_ERR_NULL_ARG;
    if (dtype != MAMBA_F32 && dtype != MAMBA_BF16) return MAMBA_ERR_BAD_DTYPE;
    constexpr long long kMax = 1LL << 40;
    if (Bsz <= 0 || Dch <= 0 || L <= 0 || N <= 0 || Bsz > 65535 || Dch > kMax || L > kMax ||
        Bsz * Dch > kMax / L || Bsz * N > kMax / L)
        return MAMBA_ERR_BAD_SHAPE;
    if (N > 64) return MAMBA_ERR_UNSUPPORTED_N;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const long long K = (L + bwd_chunk_steps(N) - 1) / bwd_chunk_steps(N);
    const size_t ck_bytes = (size_t)(Bsz * Dch) * (size_t)K * (size_t)N * sizeof(float);
    void *ck = nullptr;
    const char *inject = std::getenv("MAMBA_FAULT_INJECT");  // host-side test hook, as in the forward scan
    if (inject != nullptr && std::strcmp(inject, "alloc") == 0) return MAMBA_ERR_ALLOC;
    if (cudaMallocAsync(&ck, ck_bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_ALLOC;
    }
    int rc = MAMBA_OK;
    // the sums start from zero
    if (cudaMemsetAsync(dA, 0, (size_t)(Dch * N) * sizeof(float), st) != cudaSuccess ||
        cudaMemsetAsync(dB, 0, (size_t)(Bsz * N * L) * sizeof(float), st) != cudaSuccess ||
        cudaMemsetAsync(dC, 0, (size_t)(Bsz * N * L) * sizeof(float), st) != cudaSuccess ||
        (dD != nullptr && cudaMemsetAsync(dD, 0, (size_t)Dch * sizeof(float), st) != cudaSuccess) ||
        (ddelta_bias != nullptr && cudaMemsetAsync(ddelta_bias, 0, (size_t)Dch * sizeof(float), st) != cudaSuccess))
        rc = MAMBA_ERR_LAUNCH;
    if (rc == MAMBA_OK) {
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
        a.ckpt = static_cast<float *>(ck);
        a.Dch = Dch;
        a.L = L;
        a.N = N;
        a.softplus = softplus_flag ? 1 : 0;
        if (launch_scan_bwd(dtype, a, Bsz, st) != cudaSuccess) rc = MAMBA_ERR_LAUNCH;
    }
    if (cudaFreeAsync(ck, st) != cudaSuccess) {
        cudaGetLastError();
        if (rc == MAMBA_OK) rc = MAMBA_ERR_LAUNCH;
    }
    return rc;
}
