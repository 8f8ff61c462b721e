// scan_tm.cuh -- selective scan for N <= 16 with B/C broadcast through tensor memory.
//
// Same arithmetic as scan_kernel (fsdata.site explainer §3.2 selective_step;
// freeguideonline tutorial §4.2, §4.3, §5.2), different operand delivery.
//
// Why: on B300 the MUFU pipe issues 32 ex2 per SM per clock, while a 16-byte
// shared-memory load costs four L1 wavefronts (one per quarter warp) even when
// every lane of a quarter reads the same address.  Feeding B_t and C_t (8
// floats per lane and step) through shared memory therefore costs more issue
// and L1 bandwidth than the exps themselves.  Tensor memory has its own path
// to the registers, and the tensor core can write it: one MMA with a constant
// one-hot "selector" matrix replicates each state slice's B/C values into the
// TMEM lane of every thread that owns that slice.
//
//   D[m][col] = sum_k Sel[m][k] * X[col][k],   Sel[m][k] = 1 iff k selects slice (m mod 4)
//
// X holds, per pair of steps (t, t+1), 16 columns j: B_{4s+j/2} at step t+j%2
// for j < 8, C_{4s+(j-8)/2} at step t+j%2 for j >= 8, with the four slices'
// values along K (bf16 storage: one bf16 each, exact; fp32 storage: each value
// split into three bf16 parts hi+mid+lo whose fp32 sum reproduces it, K rows
// 3s..3s+2).  D lands in TMEM as fp32; thread m reads its lane with
// tcgen05.ld.  One MMA (M=128, N=64, K=16) covers 8 steps.  Pairing the columns
// by time lets the f32x2 instructions take (Delta_t, Delta_t+1) against a
// duplicated (A_n, A_n) and (Delta u) pairs against (B_n(t), B_n(t+1)) without
// register moves; the h recurrence stays scalar.
//
// Mapping: 128 threads = 128 TMEM lanes; thread m owns channel m/4 (32
// channels per CTA) and states 4*(m%4)..+3.  Time advances in super-tiles of
// 32 steps (u/Delta_raw/z loads, one softplus per (b,d,t) shared through
// shared memory, the y output) made of 4 MMA tiles of 8 steps; TMEM holds two
// tiles (double buffer, 128 columns), the X operand two super-tiles.  Every
// mbarrier wait is bounded; a timeout is agreed block-wide, recorded in the
// device error word, and the CTA frees its TMEM and returns.
#pragma once

#include "scan_kernels.cuh"
#include "tcgen05.cuh"

namespace mamba {

// Device error word (defined by the one translation unit that includes this
// header, scan_tm.cu, before the include).  Bit 0: an mbarrier wait of the
// tensor-memory scan timed out.

template <typename T, int MODE>
struct TmShape {
    static constexpr int NTHR = 128, CH = 32, S = 4, NS = 4;
    static constexpr int TT = 32;              // super-tile (steps)
    static constexpr int TB = 8;               // MMA tile (steps)
    static constexpr int NTILE = TT / TB;      // MMA tiles per super-tile
    static constexpr int COLS = 8 * TB;        // TMEM columns per tile (B[4], C[4] per step)
    static constexpr int TMEM_COLS = 2 * COLS; // double buffered
    static constexpr int SEG = TT / S;         // steps per lane segment (Delta, u, z, y)
    static constexpr int PER16 = 16 / (int)sizeof(T);
    static constexpr int W = SEG / PER16;      // 16-byte vectors per lane segment
    static constexpr bool SPLIT = sizeof(T) == 4;
    static constexpr int CPR = TT * (int)sizeof(T) / 16;  // 16-byte chunks per B/C row and super-tile
    static constexpr int NCHUNK = 2 * 16 * CPR;            // B and C, 16 rows
    static constexpr int RAW_PER_THR = NCHUNK / NTHR;      // 1 (bf16) or 2 (fp32)
    static constexpr int A_BYTES = 128 * 16 * 2;
    static constexpr int X_STEP = 256;         // bytes per step: 8 columns x 16 K bf16 (one 8-row group)
    static constexpr int X_BYTES = TT * X_STEP;
    static constexpr int RAW_BYTES = 2 * 16 * TT * (int)sizeof(T);
    static constexpr int DU_STRIDE = TT * 2 + 4;
    static constexpr int P_STRIDE = TT + 4;
    static constexpr int OFF_X = A_BYTES;
    static constexpr int OFF_RAW = OFF_X + 2 * X_BYTES;
    static constexpr int OFF_DU = OFF_RAW + RAW_BYTES;
    static constexpr int OFF_P = OFF_DU + CH * DU_STRIDE * 4;
    static constexpr int OFF_BAR = OFF_P + (MODE == MODE_FULL ? CH * S * P_STRIDE * 4 : 0);
    static constexpr int USED = OFF_BAR + 32;
    // at most four CTAs per SM: four x 128 TMEM columns is the whole of TMEM, so
    // the dynamic shared memory is padded until a fifth CTA cannot be resident
    static constexpr int SMEM_BYTES = USED > 47 * 1024 ? USED : 47 * 1024;
    static_assert(NCHUNK % NTHR == 0, "B/C staging must split evenly over the CTA");
    static_assert(W >= 1, "lane segment must be whole 16-byte vectors");
};

template <typename T, int MODE>
__global__ void __launch_bounds__(128, 3)
scan_tm_kernel(const ScanArgs a) {
    using Sh = TmShape<T, MODE>;
    using IO = Io<T>;
    constexpr bool FAST = sizeof(T) == 2;
    constexpr int S = Sh::S, SEG = Sh::SEG, PER16 = Sh::PER16, W = Sh::W, TT = Sh::TT, TB = Sh::TB;
    constexpr int NTILE = Sh::NTILE, COLS = Sh::COLS, CPR = Sh::CPR;
    constexpr uint32_t kWaitPolls = 1u << 24;
    constexpr uint32_t kIdesc = tc::umma_idesc_bf16_f32(128, COLS);

    extern __shared__ __align__(1024) unsigned char smem[];
    uint16_t *const sA = reinterpret_cast<uint16_t *>(smem);
    unsigned char *const sX = smem + Sh::OFF_X;
    unsigned char *const sRaw = smem + Sh::OFF_RAW;
    float *const sDU = reinterpret_cast<float *>(smem + Sh::OFF_DU);
    float *const sP = reinterpret_cast<float *>(smem + Sh::OFF_P);
    uint64_t *const mbar = reinterpret_cast<uint64_t *>(smem + Sh::OFF_BAR);
    uint32_t *const taddr_s = reinterpret_cast<uint32_t *>(smem + Sh::OFF_BAR + 16);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int s = tid & 3, c = tid >> 2;
    const long long d = (long long)blockIdx.x * Sh::CH + c;
    const bool valid = d < a.Dch;
    const long long b = blockIdx.y;
    const int kch = blockIdx.z;
    const long long N = a.N, L = a.L;
    const long long t_begin = (long long)kch * a.chunk_len;
    const long long t_end = min(L, t_begin + a.chunk_len);
    const int nsup = (int)((t_end - t_begin + TT - 1) / TT);
    const int ntile = nsup * NTILE;
    const long long dd = valid ? d : 0;
    const long long row = (b * a.Dch + dd) * L;
    const long long bc_row0 = b * N * L;
    const bool has_z = a.z != nullptr;

    // ---------------------------------------------------------------- one-time set-up
    if (warp == 0) {
        tc::tmem_alloc(taddr_s, Sh::TMEM_COLS);
        tc::tmem_relinquish();
    }
    // selector: element (m, k) of the 128 x 16 K-major operand
    for (int i = tid; i < 128 * 16; i += Sh::NTHR) {
        const int m = i >> 4, kk = i & 15;
        const bool one = Sh::SPLIT ? (kk < 12 && kk / 3 == (m & 3)) : (kk == (m & 3));
        sA[((m >> 3) * 256 + (kk >> 3) * 128 + (m & 7) * 16 + (kk & 7) * 2) >> 1] = one ? 0x3F80u : 0u;
    }
    for (int i = tid; i < 2 * Sh::X_BYTES / 16; i += Sh::NTHR)
        reinterpret_cast<uint4 *>(sX)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        tc::mbar_init(&mbar[0], 1);
        tc::mbar_init(&mbar[1], 1);
        tc::fence_mbar_init();
    }

    // per-lane constants and state (states n = 4s + j); A2d[j] = (A_n log2 e, A_n log2 e)
    float2 A2d[4];
    float h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const long long n = 4LL * s + j;
        float an = 0.f, hn = 0.f;
        if (valid && n < N) an = a.A[dd * N + n] * kLog2e;
        if (a.hin != nullptr && valid && n < N) hn = a.hin[((b * a.nchunks + kch) * a.Dch + dd) * N + n];
        A2d[j] = f2(an, an);
        h[j] = hn;
    }
    const float Dd = (a.D != nullptr && valid) ? a.D[dd] : 0.f;
    const float bias = (a.bias != nullptr && valid) ? a.bias[dd] : 0.f;

    // ---- B/C staging: raw rows of one super-tile (chunk q -> tensor, state row, 16-byte chunk)
    uint4 rraw[Sh::RAW_PER_THR];
    auto raw_load = [&](int sup) {
        const long long t0 = t_begin + (long long)sup * TT;
#pragma unroll
        for (int r = 0; r < Sh::RAW_PER_THR; ++r) {
            const int q = tid + r * Sh::NTHR;
            const int chunk = q % CPR, n = (q / CPR) & 15, which = q / (16 * CPR);
            const void *base = which ? a.Cm : a.Bm;
            const long long tt = t0 + (long long)chunk * PER16;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (n < N && tt < t_end) {
                const long long off = bc_row0 + n * L + tt;
                if (tt + PER16 <= t_end) {
                    v = ldg16(reinterpret_cast<const T *>(base) + off);
                } else {
#pragma unroll
                    for (int i = 0; i < PER16; ++i)
                        if (tt + i < t_end) IO::set(v, i, IO::load(base, off + i));
                }
            }
            rraw[r] = v;
        }
    };
    auto raw_store = [&]() {
#pragma unroll
        for (int r = 0; r < Sh::RAW_PER_THR; ++r)
            reinterpret_cast<uint4 *>(sRaw)[tid + r * Sh::NTHR] = rraw[r];
    };
    // X for one super-tile from sRaw: column n = 16 * pair + j (see the column order above)
    auto x_build = [&](int xb) {
        const T *raw = reinterpret_cast<const T *>(sRaw);  // [which][16][TT]
        unsigned char *xbase = sX + xb * Sh::X_BYTES;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int n = tid + r * Sh::NTHR;  // 256 columns
            const int j = n & 15;
            const int t = 2 * (n >> 4) + (j & 1);
            const int which = j >> 3, col = (j & 7) >> 1;
            float v[4];
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) {
                const T *p = raw + (which * 16 + 4 * sl + col) * TT + t;
                v[sl] = Sh::SPLIT ? *reinterpret_cast<const float *>(p)
                                  : __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(p)) << 16);
            }
            unsigned char *dst = xbase + (n >> 3) * 256 + (n & 7) * 16;
            if (!Sh::SPLIT) {
                // bf16 inputs are exact in bf16: K rows 0..3
                *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
            } else {
                // fp32: value = hi + mid + lo, three bf16 parts, K rows 3*sl .. 3*sl+2
                uint32_t hb[12];
#pragma unroll
                for (int sl = 0; sl < 4; ++sl) {
                    const uint32_t hi = pack_bf16x2(v[sl], 0.f) & 0xffffu;
                    const float r1 = v[sl] - __uint_as_float(hi << 16);
                    const uint32_t mid = pack_bf16x2(r1, 0.f) & 0xffffu;
                    const float r2 = r1 - __uint_as_float(mid << 16);
                    const uint32_t lo = pack_bf16x2(r2, 0.f) & 0xffffu;
                    hb[3 * sl] = hi;
                    hb[3 * sl + 1] = mid;
                    hb[3 * sl + 2] = lo;
                }
                *reinterpret_cast<uint4 *>(dst) = make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16),
                                                             hb[4] | (hb[5] << 16), hb[6] | (hb[7] << 16));
                *reinterpret_cast<uint2 *>(dst + 128) = make_uint2(hb[8] | (hb[9] << 16), hb[10] | (hb[11] << 16));
            }
        }
    };

    // ---- per-lane segment of u, Delta_raw, z
    uint4 ru[W], rd[W], rz[W];
    auto seg_load = [&](int sup, uint4 (&xu)[W], uint4 (&xd)[W], uint4 (&xz)[W]) {
        const long long t0 = t_begin + (long long)sup * TT + (long long)s * SEG;
        const T *pu = reinterpret_cast<const T *>(a.u) + row + t0;
        const T *pd = reinterpret_cast<const T *>(a.delta) + row + t0;
        const T *pz = reinterpret_cast<const T *>(a.z) + row + t0;
        if (valid && t0 + SEG <= t_end) {
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
                        IO::set(vu, i, IO::load(a.u, row + t));
                        IO::set(vd, i, IO::load(a.delta, row + t));
                        if (has_z) IO::set(vz, i, IO::load(a.z, row + t));
                    }
                }
                xu[w] = vu;
                xd[w] = vd;
                xz[w] = vz;
            }
        }
    };

    // ---- prologue: X of super-tile 0 built, the first two MMA tiles issued
    raw_load(0);
    seg_load(0, ru, rd, rz);
    raw_store();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_base = *taddr_s;
    const uint32_t tmem_lane = tmem_base + (static_cast<uint32_t>(warp * 32) << 16);
    x_build(0);
    if (nsup > 1) raw_load(1);
    tc::fence_proxy_async();
    __syncthreads();
    const uint64_t descA = tc::umma_desc(tc::smem_addr(sA), 128, 256);
    auto issue = [&](int i) {  // MMA tile i -> TMEM buffer i & 1, completion on mbar[i & 1]
        const uint32_t xaddr = tc::smem_addr(sX + ((i / NTILE) & 1) * Sh::X_BYTES + (i % NTILE) * TB * Sh::X_STEP);
        tc::umma_bf16(tmem_base + (i & 1) * COLS, descA, tc::umma_desc(xaddr, 128, 256), kIdesc, 0u);
        tc::umma_commit(&mbar[i & 1]);
    };
    if (tid == 0) {
        tc::fence_after_sync();
        issue(0);
        if (ntile > 1) issue(1);
    }

    float sdt_acc = 0.f;
    float *const du_c = sDU + c * Sh::DU_STRIDE;
    const float2 bias2 = f2(bias, bias);
    const float2 D2 = f2(Dd, Dd);
    bool failed = false;

    for (int sup = 0; sup < nsup && !failed; ++sup) {
        const bool has_next = sup + 1 < nsup;
        // X of the next super-tile (its raw rows were loaded one super-tile ago)
        if (has_next) {
            raw_store();
            __syncthreads();
            x_build((sup + 1) & 1);
            tc::fence_proxy_async();
            if (sup + 2 < nsup) raw_load(sup + 2);
        }
        uint4 nu[W], nd[W], nz[W];
        if (has_next) seg_load(sup + 1, nu, nd, nz);

        // Delta and Delta*u for this lane's 8 steps, shared with the channel's other lanes
        const long long tseg = t_begin + (long long)sup * TT + (long long)s * SEG;
        const bool seg_full = valid && tseg + SEG <= t_end;
#pragma unroll
        for (int i = 0; i < SEG; i += 2) {
            const float2 raw = __fadd2_rn(f2(IO::get(rd[i / PER16], i % PER16),
                                             IO::get(rd[(i + 1) / PER16], (i + 1) % PER16)), bias2);
            float2 dl = a.softplus ? softplus2<FAST>(raw) : raw;
            if (!seg_full) {
                if (!(valid && tseg + i < t_end)) dl.x = 0.f;
                if (!(valid && tseg + i + 1 < t_end)) dl.y = 0.f;
            }
            const float2 du = __fmul2_rn(dl, f2(IO::get(ru[i / PER16], i % PER16),
                                                IO::get(ru[(i + 1) / PER16], (i + 1) % PER16)));
            *reinterpret_cast<float4 *>(du_c + (s * SEG + i) * 2) = make_float4(dl.x, dl.y, du.x, du.y);
            if (MODE == MODE_STATES) sdt_acc += dl.x + dl.y;
        }
        __syncwarp();

        float *const prow = sP + (c * S + s) * Sh::P_STRIDE;
#pragma unroll
        for (int q = 0; q < NTILE; ++q) {
            const int i = sup * NTILE + q;
            // warp-uniform outcome: tcgen05.ld below is .sync.aligned
            const bool ok = __all_sync(0xffffffffu, tc::mbar_wait_bounded(&mbar[i & 1], (i >> 1) & 1, kWaitPolls));
            tc::fence_after_sync();
            float bc[64];
            if (ok) {
                float *b0 = bc, *b1 = bc + 32;
                tc::tmem_ld32_wait(tmem_lane + (i & 1) * COLS, *reinterpret_cast<float(*)[32]>(b0));
                tc::tmem_ld32_wait(tmem_lane + (i & 1) * COLS + 32, *reinterpret_cast<float(*)[32]>(b1));
            }
            tc::fence_before_sync();
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
            if (tid == 0 && i + 2 < ntile) {
                tc::fence_after_sync();
                issue(i + 2);
            }
            // all of the tile's shared-memory inputs first: (Delta, Delta', du, du') per step pair
            float4 dd[TB / 2];
#pragma unroll
            for (int p = 0; p < TB / 2; ++p) dd[p] = *reinterpret_cast<const float4 *>(du_c + (q * TB / 2 + p) * 4);
            float pq[TB];
#pragma unroll
            for (int p = 0; p < TB / 2; ++p) {
                const float2 dl = f2(dd[p].x, dd[p].y);
                const float2 du = f2(dd[p].z, dd[p].w);
                const float *bcp = bc + 16 * p;
                float2 hp[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x = __fmul2_rn(dl, A2d[j]);
                    const float2 bu = __fmul2_rn(du, f2(bcp[2 * j], bcp[2 * j + 1]));
                    const float ht = fmaf(ex2_approx(x.x), h[j], bu.x);
                    h[j] = fmaf(ex2_approx(x.y), ht, bu.y);
                    hp[j] = f2(ht, h[j]);
                }
                if (MODE == MODE_FULL) {
                    float2 P = __fmul2_rn(f2(bcp[8], bcp[9]), hp[0]);
                    P = __ffma2_rn(f2(bcp[10], bcp[11]), hp[1], P);
                    P = __ffma2_rn(f2(bcp[12], bcp[13]), hp[2], P);
                    P = __ffma2_rn(f2(bcp[14], bcp[15]), hp[3], P);
                    pq[2 * p] = P.x;
                    pq[2 * p + 1] = P.y;
                }
            }
            if (MODE == MODE_FULL) {
#pragma unroll
                for (int t = 0; t < TB; t += 4)
                    *reinterpret_cast<float4 *>(prow + q * TB + t) = make_float4(pq[t], pq[t + 1], pq[t + 2], pq[t + 3]);
            }
        }
        if (failed) break;

        if (MODE == MODE_FULL) {
            __syncwarp();
            float2 ys[SEG / 2];
#pragma unroll
            for (int i = 0; i < SEG / 2; ++i) ys[i] = f2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < S; ++r) {
                const float *pr = sP + (c * S + r) * Sh::P_STRIDE + s * SEG;
#pragma unroll
                for (int i = 0; i < SEG; i += 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(pr + i);
                    ys[i / 2] = __fadd2_rn(ys[i / 2], f2(v.x, v.y));
                    ys[i / 2 + 1] = __fadd2_rn(ys[i / 2 + 1], f2(v.z, v.w));
                }
            }
            float yv[SEG];
#pragma unroll
            for (int i = 0; i < SEG; i += 2) {
                const float2 u2 = f2(IO::get(ru[i / PER16], i % PER16), IO::get(ru[(i + 1) / PER16], (i + 1) % PER16));
                float2 yy = __ffma2_rn(D2, u2, ys[i / 2]);
                if (has_z)
                    yy = gate2<FAST>(yy, f2(IO::get(rz[i / PER16], i % PER16),
                                            IO::get(rz[(i + 1) / PER16], (i + 1) % PER16)));
                yv[i] = yy.x;
                yv[i + 1] = yy.y;
            }
            T *py = reinterpret_cast<T *>(a.y) + row + tseg;
            if (seg_full) {
#pragma unroll
                for (int w = 0; w < W; ++w) stg16(py + w * PER16, IO::pack(yv + w * PER16));
            } else if (valid) {
#pragma unroll
                for (int i = 0; i < SEG; ++i)
                    if (tseg + i < t_end) IO::store(a.y, row + tseg + i, yv[i]);
            }
        }
        if (has_next) {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                ru[w] = nu[w];
                rd[w] = nd[w];
                rz[w] = nz[w];
            }
        }
        __syncwarp();
    }

    if (failed) {
        if (tid == 0) {
            atomicOr(&g_device_error, 1u);
            // give MMAs already issued a bounded chance to finish before TMEM is freed
            tc::mbar_wait_bounded(&mbar[0], 0, kWaitPolls);
            tc::mbar_wait_bounded(&mbar[1], 0, kWaitPolls);
        }
    } else if (MODE == MODE_STATES) {
        float sdt = sdt_acc;
#pragma unroll
        for (int off = 1; off < S; off <<= 1) sdt += __shfl_xor_sync(0xffffffffu, sdt, off);
        if (valid) {
            const long long base = (b * a.nchunks + kch) * a.Dch + d;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const long long n = 4LL * s + j;
                if (n < N) a.ws_h[base * N + n] = h[j];
            }
            if (s == 0) a.ws_sdt[base] = sdt;
        }
    } else if (a.last_state != nullptr && valid && kch == a.nchunks - 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const long long n = 4LL * s + j;
            if (n < N) a.last_state[(b * a.Dch + d) * N + n] = h[j];
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem_base, Sh::TMEM_COLS);
    }
}

}  // namespace mamba
