// scan_tm.cuh -- selective scan for N <= 16 with B/C broadcast through tensor memory.
//
// Same arithmetic as scan_kernel (fsdata.site explainer §3.2 selective_step;
// freeguideonline tutorial §4.2, §4.3, §5.2), different operand delivery and
// schedule.
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
// for j < 8, C_{4s+(j-8)/2} at step t+j%2 for j >= 8 (the end-state pass of
// the chunked scan, which reads no C, orders each 8-step sub-tile's 64 columns
// as its 32 B columns then its 32 C columns and loads only the first half),
// with the four slices'
// values along K (bf16 storage: one bf16 each, exact; fp32 storage: each value
// split into three bf16 parts hi+mid+lo whose fp32 sum reproduces it, K rows
// 3s..3s+2).  D lands in TMEM as fp32; thread m reads its lane with
// tcgen05.ld.  Pairing the columns by time lets the f32x2 instructions take
// (Delta_t, Delta_t+1) against a duplicated (A_n, A_n), (Delta u) pairs
// against (B_n(t), B_n(t+1)) and (C_n(t), C_n(t+1)) against the state pair
// (h_n(t), h_n(t+1)), which the recurrence writes in place.
//
// B and C do not depend on the channel, so all warps of a CTA read the same
// TMEM columns.  A channel is spread over S = 4, 8 or 16 lanes (N <= 4 S), lane
// m % S owning states 4(m % S)..+3 (warp w reads TMEM lanes 32(w % 4)..+31, and
// the selector picks K row m % S, so a lane always receives its own 4 states'
// B and C: 8 columns per step for every S).  A CTA of W compute warps (32 W / S
// channels) and one producer warp takes the whole of TMEM (512 columns, one
// CTA per SM) as two buffers of one 32-step super-tile each.  W (8..11) is
// chosen per problem so that the CTAs fill the SMs in whole waves.  Per
// super-tile the producer warp does, once: five tiled TMA loads (u, Delta_raw,
// z boxes of 32 steps x 32 W / S channels, B and C boxes of 32 steps x 4 S
// states; out-of-range rows and steps read as zero), one X build and one MMA
// (M=128, N=256, K=16).  The compute warps never wait for one another: each
// waits for its super-tile's MMA (mbarrier full[buffer]) and, when done with
// the buffer and its input stage, arrives on empty[buffer]; the producer waits
// for all W arrivals before it rebuilds that buffer two super-tiles later.  The
// input ring has 3 stages; u/Delta_raw/z use the TMA's 16-byte-chunk swizzle so
// that the channels of a warp hit distinct banks.
//
// Per 8-step sub-tile i each lane loads its 64 TMEM columns, then in one
// branch-free block computes Delta = softplus(.), Delta*u, D*u and SiLU(z) for
// step pair s % 4 of sub-tile i+1 (Delta, Delta*u go to shared memory for the
// channel's lanes; D*u, SiLU(z) stay in registers), finishes y for that pair
// of sub-tile i-1 (sum of the channel's S C.h partials, + D*u, * SiLU(z),
// predicated store by lanes s < 4) and runs the recurrence over sub-tile i's
// 8 steps.
//
// Every mbarrier wait is bounded (about a second); a timeout sets a shared abort flag that
// every later wait honours and that stops further loads and MMAs, is recorded
// in the device error word, and the CTA still walks its loop (its results are
// then meaningless), waits (bounded) for its issued MMAs and loads, frees its
// TMEM and returns.
#pragma once

#include <cuda.h>

#include "scan_kernels.cuh"
#include "tcgen05.cuh"

namespace mamba {

// Device error word: each translation unit that includes this header defines
// its own g_device_error (static, before the include) and reports it through
// mamba_device_error.  Bit 0: an mbarrier wait of the tensor-memory scan
// timed out.

// TMA descriptors of one call: u, Delta_raw, z as [Bsz][Dch][L] with boxes of
// 32 steps x 8W channels (swizzled); B, C as [Bsz][N][L] with boxes of 32
// steps x 16 states (plain).
struct TmMaps {
    CUtensorMap u, delta, z, B, C;
};

// flag variants of the kernel (template argument FLAGS); FL_CKPT: the plain direct scan that also writes
// the backward pass's checkpoints (ScanArgs::ckpt)
enum { FL_REV = 1, FL_ZOH = 2, FL_CKPT = 4 };

// S = lanes per channel (4, 8 or 16: N <= 4 S), each lane owning 4 states.
// CONV: the first input tile is x with an 8-step halo (40 steps from t0 - 8,
// unswizzled) from which u = SiLU(causal conv(x)) is formed.
// LEAN: each lane loads one step pair's 16 TMEM columns at a time instead of a
// sub-tile's 64, which brings the kernel to 96 registers per thread, so a
// CTA can run 12..18 compute warps (one CTA per SM still): problems whose
// channels would need two or more waves of 8..11-warp CTAs fit in fewer.
template <typename T, int MODE, int S_ = 4, bool CONV = false, bool LEAN = false>
struct TmShape {
    static constexpr int S = S_;
    static constexpr int MIN_WARPS = LEAN ? 12 : 8, MAX_WARPS = LEAN ? 18 : 11;  // compute warps, 32 / S channels each
    static constexpr int MAX_THR = 32 * MAX_WARPS, MAX_CH = MAX_THR / S;
    static constexpr int LAUNCH_THR = MAX_THR + 32;       // + the producer warp
    static constexpr int TT = 32;                  // steps per super-tile
    static constexpr int TB = 8;                   // steps per sub-tile
    static constexpr int NSUB = TT / TB;
    static constexpr int COLS = 8 * TT;            // TMEM columns per super-tile (B[4], C[4] per step)
    static constexpr int TMEM_COLS = 2 * COLS;     // 512: all of TMEM, one CTA per SM
    static constexpr int NST = 3;                  // input stages
    static constexpr bool SPLIT = sizeof(T) == 4;
    static constexpr int ROW = TT * (int)sizeof(T);  // bytes of one row of a box
    static constexpr int SWZ = ROW / 16;             // 16-byte chunks per swizzle span (64 B or 128 B)
    static constexpr int IO_TILE = (MAX_CH * ROW + 1023) / 1024 * 1024;  // slot of u, Delta_raw or z (box: 32 W / S rows)
    static constexpr int BC_TILE = 4 * S * ROW;      // one of B, C (box: 4 S state rows)
    static constexpr int XSTEPS = TT + 8;            // CONV: steps of the x box (8 of halo)
    static constexpr int X0_TILE = CONV ? (MAX_CH * XSTEPS * (int)sizeof(T) + 1023) / 1024 * 1024 : IO_TILE;
    static constexpr int OFF_BC = X0_TILE + 2 * IO_TILE;  // B then C, after u (or x), Delta_raw, z
    static constexpr int STAGE_BYTES = OFF_BC + 2 * BC_TILE;
    static constexpr int A_BYTES = 128 * 16 * 2;
    static constexpr int X_BYTES = COLS * 16 * 2;
    static constexpr int DU_BYTES = MAX_CH * 4 * 16;           // per sub-tile: (Delta, Delta', du, du') per step pair
    static constexpr int P_STRIDE = TB + 4;                    // floats per lane row of partials
    static constexpr int P_BYTES = MAX_THR * P_STRIDE * 4;     // per sub-tile
    static constexpr int OFF_ST = 0;
    static constexpr int OFF_A = OFF_ST + NST * STAGE_BYTES;
    static constexpr int OFF_X = OFF_A + A_BYTES;
    static constexpr int OFF_DU = OFF_X + 2 * X_BYTES;
    static constexpr int OFF_P = OFF_DU + 2 * DU_BYTES;
    static constexpr int OFF_BAR = OFF_P + (MODE != MODE_STATES ? 2 * P_BYTES : 0);
    static constexpr int OFF_VOTE = OFF_BAR + 128;  // MODE_CORR: super-tile at which each compute warp's
                                                    // states had decayed below the stopping bound
    static constexpr int SMEM_BYTES = OFF_VOTE + 4 * MAX_WARPS + 1024;  // + room to align the base to 1024 bytes
    static_assert(5 + NST <= 8, "full[2], empty[2], done and io[NST] in the first 64 bytes of the barrier block");
    static_assert(IO_TILE % 1024 == 0 && BC_TILE % 1024 == 0, "swizzled boxes need 1024-byte aligned tiles");
    static_assert(SWZ == 4 || SWZ == 8, "rows of 64 or 128 bytes");
    static_assert(S == 4 || S == 8 || S == 16, "4, 8 or 16 lanes per channel");
    static_assert(!SPLIT || S == 4, "fp32 B/C take 3 K rows per slice: 4 slices fill K = 16");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// HAS_Z: the gate z is given (MODE_FULL only).  S lanes per channel.  CONV:
// a.u holds x and u = SiLU(a.conv_b + causal width-4 conv with a.conv_w) is
// formed here (ai.xwebgame.com summary, "running it in PyTorch" block).
// FLAGS (compile time): 0 the plain scan; FL_REV the scan over t = L-1 .. 0
// (SCAN_FLAG_REVERSE; fsdata.site explainer §7 table, the reverse SSM);
// FL_ZOH the exact zero-order-hold input weight (freeguideonline tutorial
// §2.2), forwards or, with SCAN_FLAG_REVERSE, in reverse.
// blockDim.x = 32 (W + 1): W compute warps (8..11, lean form 12..18) and one producer warp.
template <typename T, int MODE, bool HAS_Z, int S_, bool CONV, int FLAGS, bool LEAN>
__device__ __forceinline__ void scan_tm_body(const ScanArgs &a, const TmMaps &maps) {
    using Sh = TmShape<T, MODE, S_, CONV, LEAN>;
    static_assert(!LEAN || (MODE == MODE_FULL && !CONV && (FLAGS == 0 || FLAGS == FL_CKPT)),
                  "the lean form serves the plain direct scan");
    static_assert(FLAGS != FL_CKPT || (MODE == MODE_FULL && !CONV), "checkpoints come from the plain direct scan");
    constexpr bool FAST = sizeof(T) == 2;
    constexpr bool HASY = MODE != MODE_STATES;                             // forms y (and reads C)
    constexpr bool ENDS = MODE == MODE_STATES || MODE == MODE_FULL_STATES;  // writes end states, sum of Delta
    constexpr bool CORR = MODE == MODE_CORR;
    constexpr int S = Sh::S, TT = Sh::TT, TB = Sh::TB, NSUB = Sh::NSUB, COLS = Sh::COLS, MAX_CH = Sh::MAX_CH;
    constexpr int NST = Sh::NST;
    constexpr uint32_t kWaitPolls = 1u << 24;  // drain waits before TMEM and shared memory are released
    constexpr uint32_t kIdesc = tc::umma_idesc_bf16_f32(128, COLS);
    using Word = typename std::conditional<Sh::SPLIT, float2, uint32_t>::type;  // one step pair

    extern __shared__ unsigned char smem_raw[];
    unsigned char *const smem = smem_raw + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u);
    unsigned char *const sSt = smem + Sh::OFF_ST;
    uint16_t *const sA = reinterpret_cast<uint16_t *>(smem + Sh::OFF_A);
    unsigned char *const sX = smem + Sh::OFF_X;
    float4 *const sDU = reinterpret_cast<float4 *>(smem + Sh::OFF_DU);  // [2][MAX_CH][4 pairs]
    float *const sP = reinterpret_cast<float *>(smem + Sh::OFF_P);      // [2][MAX_THR][P_STRIDE]
    uint64_t *const full = reinterpret_cast<uint64_t *>(smem + Sh::OFF_BAR);  // [2] MMA of a super-tile done
    uint64_t *const empty = full + 2;  // [2] every compute warp is done with a super-tile's TMEM buffer and stage
    uint64_t *const done = full + 4;   // abort path: all MMAs done
    uint64_t *const io = full + 5;     // [NST] stage loads landed
    uint32_t *const taddr_s = reinterpret_cast<uint32_t *>(smem + Sh::OFF_BAR + 64);
    volatile int *const first_small = reinterpret_cast<volatile int *>(smem + Sh::OFF_VOTE);  // [MAX_WARPS]
    volatile int *const abort_flag = reinterpret_cast<volatile int *>(smem + Sh::OFF_BAR + 68);

    const int nthr = blockDim.x, ncw = nthr / 32 - 1, ch = 32 * ncw / S;  // compute warps, channels of this CTA
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool producer = warp == ncw;  // the last warp loads, builds X and issues the MMAs
    const int s = tid % S, c = tid / S;  // state slice, channel within the CTA
    // the 4 step pairs of a sub-tile: lane s handles pair ps for its channel's
    // Delta and y (lanes s >= 4 of a wider channel repeat lane s % 4's work and
    // store nothing)
    const int ps = s & 3;
    const bool pair_owner = s < 4;
    const long long d0 = (long long)blockIdx.x * ch;
    const long long d = d0 + c;
    const bool valid = !producer && d < a.Dch;
    const long long b = blockIdx.y;
    const int kch = blockIdx.z + (CORR ? a.chunk0 : 0);
    const long long N = a.N, L = a.L;
    const long long t_begin = (long long)kch * a.chunk_len;
    const int len = (int)(min(L, t_begin + a.chunk_len) - t_begin);  // steps of this chunk (< 2^31)
    const int nsup = (len + TT - 1) / TT;
    const long long dd = valid ? d : 0;
    // a step pair of this lane at offset r (from t_begin) is in range iff (unsigned) r < lenv
    const unsigned lenv = valid ? (unsigned)len : 0u;

    // ---------------------------------------------------------------- one-time set-up
    if (warp == 0) {
        tc::tmem_alloc(taddr_s, Sh::TMEM_COLS);
        tc::tmem_relinquish();
    }
    // selector: element (m, k) of the 128 x 16 K-major operand
    for (int i = tid; i < 128 * 16; i += nthr) {
        const int m = i >> 4, kk = i & 15;
        const bool one = Sh::SPLIT ? (kk < 12 && kk / 3 == (m & 3)) : (kk == m % S);
        sA[((m >> 3) * 256 + (kk >> 3) * 128 + (m & 7) * 16 + (kk & 7) * 2) >> 1] = one ? 0x3F80u : 0u;
    }
    for (int i = tid; i < 2 * Sh::X_BYTES / 16; i += nthr)
        reinterpret_cast<uint4 *>(sX)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        tc::mbar_init(&full[0], 1);
        tc::mbar_init(&full[1], 1);
        tc::mbar_init(&empty[0], ncw);
        tc::mbar_init(&empty[1], ncw);
        tc::mbar_init(done, 1);
        for (int k = 0; k < NST; ++k) tc::mbar_init(&io[k], 1);
        *abort_flag = 0;
        for (int w = 0; w < Sh::MAX_WARPS; ++w) first_small[w] = 0x7fffffff;
        tc::fence_mbar_init();
    }

    // per-lane constants and state (states n = 4s + j).  A2d[j] = (A_n log2 e, A_n log2 e);
    // hh[j] = (h_n(t), h_n(t+1)) of the last step pair, .y the current state.
    float2 A2d[4], hh[4];
    constexpr bool zoh = FLAGS == FL_ZOH;
    float invA[zoh ? 4 : 1];  // ZOH: 1/A_n (0 where A_n = 0)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const long long n = 4LL * s + j;
        float an = 0.f, hn = 0.f;
        if (valid && n < N) an = a.A[dd * N + n] * kLog2e;
        if (a.hin != nullptr && valid && n < N) hn = a.hin[((b * a.nchunks + kch) * a.Dch + dd) * N + n];
        A2d[j] = f2(an, an);
        hh[j] = f2(0.f, hn);
        if constexpr (zoh) invA[j] = an != 0.f ? kLog2e / an : 0.f;
    }
    // FL_REV is launched only for reverse scans; FL_ZOH serves both directions
    const bool rev = FLAGS == FL_REV || (FLAGS == FL_ZOH && (a.flags & SCAN_FLAG_REVERSE) != 0);
    const float Dd = (a.D != nullptr && valid && !CORR) ? a.D[dd] : 0.f;  // the correction has no input
    const float bias = (a.bias != nullptr && valid) ? a.bias[dd] : 0.f;
    const float2 bias2 = f2(bias, bias);
    const float2 D2 = f2(Dd, Dd);
    const bool softplus = a.softplus != 0;
    float4 cw = make_float4(0.f, 0.f, 0.f, 0.f);  // CONV: taps on x_{t-3}, ..., x_t
    float cb = 0.f;
    if constexpr (CONV) {
        if (valid) {
            cw = make_float4(a.conv_w[dd * 4], a.conv_w[dd * 4 + 1], a.conv_w[dd * 4 + 2], a.conv_w[dd * 4 + 3]);
            cb = a.conv_b != nullptr ? a.conv_b[dd] : 0.f;
        }
    }
    // y of the (logical) step at offset r from t_begin in this lane's channel: ylane[r] forwards, the
    // physical row mirrored in reverse (logical step tau sits at L - 1 - tau)
    T *const yrow = reinterpret_cast<T *>(a.y) + (b * a.Dch + dd) * L;
    T *const ylane = yrow + t_begin;

    // Bounded wait that gives up at once when another warp has already given up: a non-blocking test,
    // then try_wait calls that suspend the thread in hardware until the phase completes (at most 20 us
    // each; a waiting warp spends no issue slots) until one second of the global timer has passed.  With
    // a.wait_polls == 0 (test hook) the wait gives up after the first test.
    auto wait_or_abort = [&](uint64_t *bar, uint32_t parity, bool) -> bool {
        if (tc::mbar_test_wait(bar, parity)) return true;
        if (a.wait_polls == 0 || *abort_flag != 0) return false;
        const uint64_t t0 = tc::globaltimer_ns();
        for (;;) {
            if (tc::mbar_try_wait(bar, parity, 20000u)) return true;
            if (*abort_flag != 0 || tc::globaltimer_ns() - t0 > 1000000000ull) return false;
        }
    };

    // ---- inputs of super-tile sn -> stage sn % NST (thread 0).  The time
    // coordinate is a multiple of 32 steps, so x * element size is a multiple
    // of 16 bytes.
    auto stage_of = [&](int k) { return sSt + k * Sh::STAGE_BYTES; };
    auto load_stage = [&](int sn) {
        unsigned char *st = stage_of(sn % NST);
        uint64_t *bar = &io[sn % NST];
        // forwards: the box of logical steps tau0 .. tau0 + 31 starts at tau0; reverse: it covers physical
        // steps L - 32 - tau0 .. L - 1 - tau0 (a negative start of the last one reads zeros)
        const long long tau0 = t_begin + (long long)sn * TT;
        const int x = (int)(rev ? L - TT - tau0 : tau0);
        const uint32_t first = CONV ? (uint32_t)(ch * Sh::XSTEPS * (int)sizeof(T)) : (uint32_t)(ch * Sh::ROW);
        tc::mbar_arrive_expect_tx(bar, first + (uint32_t)((HAS_Z ? 2 : 1) * ch * Sh::ROW + 2 * Sh::BC_TILE));
        // CONV: x from 8 steps back (a negative start reads zeros: the causal padding)
        tc::tma_load_3d(st, &maps.u, CONV ? x - 8 : x, (int)d0, (int)b, bar);
        tc::tma_load_3d(st + Sh::X0_TILE, &maps.delta, x, (int)d0, (int)b, bar);
        if (HAS_Z) tc::tma_load_3d(st + Sh::X0_TILE + Sh::IO_TILE, &maps.z, x, (int)d0, (int)b, bar);
        tc::tma_load_3d(st + Sh::OFF_BC, &maps.B, x, 0, (int)b, bar);  // 4 S state rows, zero past N
        tc::tma_load_3d(st + Sh::OFF_BC + Sh::BC_TILE, &maps.C, x, 0, (int)b, bar);
    };

    // X of one super-tile from its stage: column n = 16 * pair + j (MODE_FULL) or
    // 64 * sub-tile + 32 * (B or C) + 8 * pair-in-sub-tile + j (MODE_STATES), the
    // column orders above; K row k = slice k's value (bf16), or K rows 3k..3k+2
    // its three bf16 parts (fp32, S = 4)
    auto x_build = [&](int xb, const unsigned char *st) {  // by the producer warp
        const T *raw = reinterpret_cast<const T *>(st + Sh::OFF_BC);  // [which][4 S][TT]
        unsigned char *xbase = sX + xb * Sh::X_BYTES;
        for (int n = lane; n < COLS; n += 32) {
            int t, which, col;
            if constexpr (HASY) {
                const int j = n & 15;
                t = 2 * (n >> 4) + (j & 1);
                which = j >> 3;
                col = (j & 7) >> 1;
            } else {
                const int j = n & 7;
                t = 8 * (n >> 6) + 2 * ((n >> 3) & 3) + (j & 1);
                which = (n >> 5) & 1;
                col = j >> 1;
            }
            if (rev) t = TT - 1 - t;  // logical step t of the super-tile sits at box position 31 - t
            float v[S];
#pragma unroll
            for (int sl = 0; sl < S; ++sl) {
                const T *p = raw + (which * 4 * S + 4 * sl + col) * TT + t;
                v[sl] = Sh::SPLIT ? *reinterpret_cast<const float *>(p)
                                  : __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(p)) << 16);
            }
            unsigned char *dst = xbase + (n >> 3) * 256 + (n & 7) * 16;
            if constexpr (!Sh::SPLIT) {
                // bf16 inputs are exact in bf16; K rows 0..7 at dst, 8..15 at dst + 128
                uint32_t w[S / 2];
#pragma unroll
                for (int k = 0; k < S / 2; ++k) w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
                if constexpr (S == 4) {
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
                } else {
                    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                    if constexpr (S == 16)
                        *reinterpret_cast<uint4 *>(dst + 128) = make_uint4(w[4], w[5], w[6], w[7]);
                }
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

    // ---- this lane's step pair of sub-tile q of a stage: steps 8q + 2s, +1 of
    // the super-tile.  The box rows are swizzled: byte offset o of the
    // 1024-byte aligned box sits at o ^ (((o >> 7) % SWZ) << 4).
    auto unpack = [](Word w) -> float2 {
        if constexpr (Sh::SPLIT) return w;
        else return f2(bf16_lo(w), bf16_hi(w));
    };
    int sw_off[NSUB];  // swizzled byte offset of this lane's pair in sub-tile q
#pragma unroll
    for (int q = 0; q < NSUB; ++q) {
        // reverse: logical steps i, i + 1 sit at box positions 31 - i, 30 - i, i.e. in the word at 30 - i
        const int pos = rev ? TT - 2 - (q * TB + 2 * ps) : q * TB + 2 * ps;
        const int o = c * Sh::ROW + pos * (int)sizeof(T);
        sw_off[q] = o ^ (((o >> 7) & (Sh::SWZ - 1)) << 4);
    }
    auto order = [&](float2 v) { return rev ? f2(v.y, v.x) : v; };  // box pair -> (step i, step i + 1)
    // tensor 0 = u (or x), 1 = Delta_raw, 2 = z
    auto stage_word = [&](const unsigned char *st, int tensor, int q) -> Word {
        return *reinterpret_cast<const Word *>(st + (tensor == 0 ? 0 : Sh::X0_TILE + (tensor - 1) * Sh::IO_TILE) +
                                               sw_off[q]);
    };
    // CONV: u of this lane's pair of sub-tile q, SiLU of the causal convolution
    // of x; the x box holds steps t0 - 8 .. t0 + 31 of the super-tile unswizzled
    auto conv_u = [&](const unsigned char *st, int q) -> float2 {
        const T *xr = reinterpret_cast<const T *>(st) + c * Sh::XSTEPS + 8 + q * TB + 2 * ps;  // step t of the pair
        const float2 m4 = unpack(*reinterpret_cast<const Word *>(xr - 4));  // x_{t-4}, x_{t-3}
        const float2 m2 = unpack(*reinterpret_cast<const Word *>(xr - 2));  // x_{t-2}, x_{t-1}
        const float2 m0 = unpack(*reinterpret_cast<const Word *>(xr));      // x_t, x_{t+1}
        const float p0 = fmaf(cw.w, m0.x, fmaf(cw.z, m2.y, fmaf(cw.y, m2.x, fmaf(cw.x, m4.y, cb))));
        const float p1 = fmaf(cw.w, m0.y, fmaf(cw.z, m0.x, fmaf(cw.y, m2.y, fmaf(cw.x, m2.x, cb))));
        // u feeds the fp32 state, so it takes the accurate SiLU (z / (1 + e^-z), ~1e-6 relative), not
        // the one-MUFU tanh form whose ~2^-11 error would carry into last_state
        return silu2<false>(f2(p0, p1));
    };
    float4 *const du_chan = sDU + c * 4;  // + (i & 1) * MAX_CH * 4 + pair
    // Delta, Delta * u of this lane's pair at offset r (sub-tile parity par) ->
    // sDU; D * u and SiLU(z) stay in this lane's registers until y of the pair is formed
    float sdt_acc = 0.f;  // MODE_STATES: this lane's share of sum(Delta) over the chunk
    auto side_pair = [&](const unsigned char *st, int q, int r, int par, float2 &Du, float2 &g) {
        const bool in = (unsigned)r < lenv;
        float2 u;
        if constexpr (CONV) u = conv_u(st, q);
        else u = order(unpack(stage_word(st, 0, q)));
        const float2 raw = __fadd2_rn(order(unpack(stage_word(st, 1, q))), bias2);
        float2 dl = softplus ? softplus2<FAST>(raw) : raw;
        dl = in ? dl : f2(0.f, 0.f);
        // the input factor of the state update: Delta u (ZOH: u, the weight being formed per state)
        // (the correction pass carries the entering state only: no input)
        const float2 du = CORR ? f2(0.f, 0.f) : zoh ? (in ? u : f2(0.f, 0.f)) : __fmul2_rn(dl, u);
        if (pair_owner) du_chan[par * MAX_CH * 4 + ps] = make_float4(dl.x, dl.y, du.x, du.y);
        if (ENDS && pair_owner) sdt_acc += dl.x + dl.y;
        if (HASY) {
            Du = __fmul2_rn(D2, u);
            if (HAS_Z) g = silu2<FAST>(order(unpack(stage_word(st, 2, q))));
        }
    };
    // partial sums of this lane's group of 4 lanes (lanes 4 (s / 4) .. + 3 of the channel)
    const float *const p_chan = sP + (c * S + (s & ~3)) * Sh::P_STRIDE + 2 * ps;  // + (i & 1) * MAX_THR * P_STRIDE
    // y of this lane's pair at offset r from the channel's S partial sums: each lane adds its group's
    // 4 partials, the S / 4 groups are combined with shuffles
    auto output_pair = [&](int r, int par, float2 Du, float2 g) {
        if (!HASY) return;
        const float *pp = p_chan + par * Sh::MAX_THR * Sh::P_STRIDE;
        float2 ys = *reinterpret_cast<const float2 *>(pp);
#pragma unroll
        for (int k = 1; k < 4; ++k) ys = __fadd2_rn(ys, *reinterpret_cast<const float2 *>(pp + k * Sh::P_STRIDE));
#pragma unroll
        for (int off = 4; off < S; off <<= 1)
            ys = __fadd2_rn(ys, f2(__shfl_xor_sync(0xffffffffu, ys.x, off), __shfl_xor_sync(0xffffffffu, ys.y, off)));
        float2 yy = __fadd2_rn(ys, Du);
        if (HAS_Z) yy = __fmul2_rn(yy, g);
        const bool st = pair_owner && (unsigned)r < lenv;
        // reverse: logical steps tau, tau + 1 (tau = t_begin + r) are physical L - 1 - tau, L - 2 - tau
        T *const dst = rev ? yrow + (L - 2 - (t_begin + r)) : ylane + r;
        yy = order(yy);
        if constexpr (CORR) {  // y += the entering state's contribution
            if constexpr (Sh::SPLIT) {
                if (st) yy = __fadd2_rn(yy, *reinterpret_cast<const float2 *>(dst));
            } else {
                if (st) {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(dst);
                    yy = __fadd2_rn(yy, f2(bf16_lo(w), bf16_hi(w)));
                }
            }
        }
        if constexpr (Sh::SPLIT)
            st_f32x2_if(dst, yy, st);
        else
            st_b32_if(dst, pack_bf16x2(yy.x, yy.y), st);
    };

    const uint64_t descA = tc::umma_desc(tc::smem_addr(sA), 128, 256);
    auto issue_mma = [&](int sn) {  // producer lane 0: MMA of super-tile sn -> TMEM buffer sn & 1, completion on full[sn & 1]
        const uint32_t xaddr = tc::smem_addr(sX + (sn & 1) * Sh::X_BYTES);
        tc::fence_after_sync();
        tc::umma_bf16(*taddr_s + (sn & 1) * COLS, descA, tc::umma_desc(xaddr, 128, 256), kIdesc, 0u);
        tc::umma_commit(&full[sn & 1]);
    };

    // ---- the producer warp runs ahead of the compute warps by up to two
    // super-tiles (the two TMEM buffers): stage loads, X builds and MMAs.  The
    // compute warps never wait for one another.
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem_lane = *taddr_s + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    int last_loaded = -1;  // producer lane 0: latest super-tile whose loads were issued
    int mma_issued = 0;    // producer lane 0: MMAs issued
    bool stopped = false;  // producer: MODE_CORR stopped before the end of the chunk
    // MODE_CORR: stop at super-tile sup once every compute warp's states had decayed by the end of
    // super-tile sup - 2 (the same answer for every warp: entries up to sup - 2 are final)
    auto corr_done = [&](int sup) {
        int m = lane < ncw ? first_small[lane] : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        return m <= sup - 2;
    };
    // MODE_CORR: the bound below which a state's contribution is dropped, and whether its decay is monotone
    float thr[CORR ? 4 : 1];
    bool monotone = CORR && softplus;
    if constexpr (CORR) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            thr[j] = fabsf(hh[j].y) * (FAST ? 0x1p-16f : 0x1p-30f);
            monotone = monotone && A2d[j].x <= 0.f;
        }
    }
    if (producer) {
        if (lane == 0)
            for (int sn = 0; sn < NST && sn < nsup; ++sn) {
                load_stage(sn);
                last_loaded = sn;
            }
        for (int sn = 0; sn < nsup; ++sn) {
            // the stage of sn has landed; for sn >= 2 every compute warp is done
            // with super-tile sn - 2, so TMEM buffer sn & 1, X buffer sn & 1 (its
            // MMA was waited for) and the stage of sn - 2 are free
            bool ok = __all_sync(0xffffffffu, wait_or_abort(&io[sn % NST], (sn / NST) & 1, true));
            if (ok && sn >= 2)
                ok = __all_sync(0xffffffffu, wait_or_abort(&empty[sn & 1], ((sn - 2) >> 1) & 1, true));
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            if (CORR && sn >= 2 && corr_done(sn)) {  // the compute warps stop at the same super-tile
                stopped = true;
                break;
            }
            tc::fence_after_sync();
            x_build(sn & 1, stage_of(sn % NST));
            tc::fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                issue_mma(sn);
                mma_issued = sn + 1;
                const int m = sn + NST - 2;  // into the stage of super-tile sn - 2
                if (sn >= 2 && m < nsup) {
                    load_stage(m);
                    last_loaded = m;
                }
            }
            __syncwarp();
        }
    } else {
        // (D u, SiLU z) of the step pairs whose y is still open, by sub-tile parity
        float2 Du_r[2], g_r[2];
        if (!__all_sync(0xffffffffu, wait_or_abort(&io[0], 0, false))) *abort_flag = 1;
        side_pair(stage_of(0), 0, 2 * ps, 0, Du_r[0], g_r[0]);
        __syncwarp();

        int k_cur = 0;  // stage of super-tile sup
        int last_sup = nsup - 1;  // the last super-tile processed
        bool recorded = false;    // MODE_CORR: this warp's decay point is in first_small
        for (int sup = 0; sup < nsup; ++sup) {
            const int k_nxt = k_cur == NST - 1 ? 0 : k_cur + 1;
            if (CORR && sup >= 2) {
                // every compute warp is done with super-tile sup - 2 (the producer waited for that before
                // the MMA of sup); this acquire makes their first_small entries visible
                if (!__all_sync(0xffffffffu, wait_or_abort(&empty[sup & 1], ((sup - 2) >> 1) & 1, false))) *abort_flag = 1;
                if (corr_done(sup)) {
                    last_sup = sup - 1;
                    break;
                }
            }
            // this super-tile's B/C are in TMEM buffer sup & 1 (after an abort the
            // loads below still read allocated TMEM; the results are then discarded)
            if (!__all_sync(0xffffffffu, wait_or_abort(&full[sup & 1], (sup >> 1) & 1, false))) *abort_flag = 1;
            tc::fence_after_sync();
            const unsigned char *st_cur = stage_of(k_cur);
            const unsigned char *st_nxt = stage_of(k_nxt);
            const int r0 = sup * TT + 2 * ps;  // this lane's pair offset in sub-tile 0 of this super-tile
#pragma unroll
            for (int q = 0; q < NSUB; ++q) {
                // MODE_FULL: step pairs 0, 1 in bcu[0] and 2, 3 in bcu[1], 16 columns each;
                // MODE_STATES: B of the 4 step pairs in bcu[0] (8 columns each), no C.
                // LEAN: each pair's 16 columns are loaded in the recurrence below.
                uint32_t bcu[LEAN ? 1 : 2][32];
                float4 dq[LEAN ? 1 : TB / 2];
                if constexpr (!LEAN) {
                    tc::tmem_ld32_nowait(tmem_lane + (sup & 1) * COLS + q * 64, bcu[0]);
                    if constexpr (HASY) {
                        tc::tmem_ld32_nowait(tmem_lane + (sup & 1) * COLS + q * 64 + 32, bcu[1]);
                        tc::tmem_wait_ld_tied(bcu[0], bcu[1]);
                    } else {
                        tc::tmem_wait_ld_tied(bcu[0]);
                    }
                    // one block: y of sub-tile i-1, Delta etc. of sub-tile i+1 and the recurrence of
                    // sub-tile i (i = 4 sup + q, so i & 1 == q & 1)
#pragma unroll
                    for (int p = 0; p < TB / 2; ++p) dq[p] = du_chan[(q & 1) * MAX_CH * 4 + p];
                }
                // Delta etc. of sub-tile i+1 (into the Du, g registers of parity (i+1) & 1, which held those
                // of sub-tile i-1)
                auto side_only = [&]() {
                    if (q + 1 < NSUB) {
                        side_pair(st_cur, q + 1, r0 + (q + 1) * TB, (q + 1) & 1, Du_r[(q + 1) & 1], g_r[(q + 1) & 1]);
                    } else {
                        if (sup + 1 < nsup && !__all_sync(0xffffffffu, wait_or_abort(&io[k_nxt], ((sup + 1) / NST) & 1, false)))
                            *abort_flag = 1;
                        side_pair(st_nxt, 0, r0 + TT, 0, Du_r[0], g_r[0]);
                    }
                };
                // the regular form: the side work first, then y of sub-tile i-1 from its Du, g saved before the
                // side work reuses their registers; measured 1.4 % faster than the other order (130M layer
                // 0.1334 -> 0.1315 ms), as was splitting the recurrence around y
                if constexpr (!LEAN) {
                    const float2 Du_prev = Du_r[(q + 1) & 1], g_prev = g_r[(q + 1) & 1];
                    side_only();
                    output_pair(r0 + (q - 1) * TB, (q + 1) & 1, Du_prev, g_prev);
                }
                float pq[TB];
#pragma unroll
                for (int p = 0; p < TB / 2; ++p) {
                    // the lean form does its side work and y of sub-tile i-1 before the sub-tile's last step
                    // pair.  On the 2.8B layer (S = 4): 0.4246 ms before the recurrence, 0.4130 after it,
                    // 0.4085 with y then the side work before the last pair, 0.4009 with the side work then y
                    // (Du, g saved first); with N = 64 (S = 16) the last order measured 1.6 % slower than
                    // y first, so S = 16 keeps y first.  These places measured 1-12 % slower in the regular form.
                    if constexpr (LEAN) {
                        if (p == TB / 2 - 1) {
                            if constexpr (S == 16) {
                                output_pair(r0 + (q - 1) * TB, (q + 1) & 1, Du_r[(q + 1) & 1], g_r[(q + 1) & 1]);
                                side_only();
                            } else {
                                const float2 Du_prev = Du_r[(q + 1) & 1], g_prev = g_r[(q + 1) & 1];
                                side_only();
                                output_pair(r0 + (q - 1) * TB, (q + 1) & 1, Du_prev, g_prev);
                            }
                        }
                    }
                    uint32_t bcl[LEAN ? 16 : 1];
                    float4 dqp;
                    const uint32_t *bcp;
                    if constexpr (LEAN) {
                        // this pair's B and C columns, and its Delta, Delta u (written in the previous
                        // sub-tile, before the last __syncwarp)
                        tc::tmem_ld16_nowait(tmem_lane + (sup & 1) * COLS + q * 64 + 16 * p, bcl);
                        dqp = du_chan[(q & 1) * MAX_CH * 4 + p];
                        tc::tmem_wait_ld_tied(bcl);
                        bcp = bcl;
                    } else {
                        dqp = dq[p];
                        bcp = HASY ? bcu[p >> 1] + 16 * (p & 1) : bcu[0] + 8 * p;
                    }
                    const float2 dl = f2(dqp.x, dqp.y);
                    const float2 du = f2(dqp.z, dqp.w);
                    const uint32_t *ccp = bcp + 8;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 x = __fmul2_rn(dl, A2d[j]);
                        const float2 Bt = f2(__uint_as_float(bcp[2 * j]), __uint_as_float(bcp[2 * j + 1]));
                        const float2 e = f2(ex2_approx(x.x), ex2_approx(x.y));
                        float2 bu;
                        if constexpr (zoh) {  // du holds u: B_bar u = (e^{Delta A} - 1) / A * B * u
                            bu = __fmul2_rn(__fmul2_rn(zoh_weight2(e, x, dl, invA[j]), du), Bt);
                        } else {
                            bu = __fmul2_rn(du, Bt);
                        }
                        hh[j].x = fmaf(e.x, hh[j].y, bu.x);
                        hh[j].y = fmaf(e.y, hh[j].x, bu.y);
                    }
                    // the backward pass's checkpoint: the state before step k * TCK, every TCK = 64 / S steps
                    // (the chunk length of the backward kernel for this state count)
                    if constexpr (FLAGS == FL_CKPT) {
                        if ((q * TB + 2 * p + 2) % (64 / S) == 0 && valid) {  // q, p unrolled: compile time
                            const long long kc = ((long long)sup * TT + q * TB + 2 * p + 2) / (64 / S);
                            if (kc < a.ckpt_k)
                                *reinterpret_cast<float4 *>(a.ckpt + ((b * a.Dch + d) * a.ckpt_k + kc) * (4 * S) + 4 * s) =
                                    make_float4(hh[0].y, hh[1].y, hh[2].y, hh[3].y);
                        }
                    }
                    if (HASY) {
                        float2 P = __fmul2_rn(f2(__uint_as_float(ccp[0]), __uint_as_float(ccp[1])), hh[0]);
                        P = __ffma2_rn(f2(__uint_as_float(ccp[2]), __uint_as_float(ccp[3])), hh[1], P);
                        P = __ffma2_rn(f2(__uint_as_float(ccp[4]), __uint_as_float(ccp[5])), hh[2], P);
                        P = __ffma2_rn(f2(__uint_as_float(ccp[6]), __uint_as_float(ccp[7])), hh[3], P);
                        pq[2 * p] = P.x;
                        pq[2 * p + 1] = P.y;
                    }
                }
                if (HASY) {
                    float *prow = sP + ((q & 1) * Sh::MAX_THR + tid) * Sh::P_STRIDE;
                    *reinterpret_cast<float4 *>(prow) = make_float4(pq[0], pq[1], pq[2], pq[3]);
                    *reinterpret_cast<float4 *>(prow + 4) = make_float4(pq[4], pq[5], pq[6], pq[7]);
                }
                __syncwarp();  // partials of sub-tile i and Delta of sub-tile i+1 visible to the channel's lanes
            }
            if constexpr (CORR) {
                // Once every state of the warp has decayed below 2^-16 (bf16 y) or 2^-30 (fp32 y) of the
                // state it entered the chunk with, it stays there (softplus Delta > 0 and A <= 0: each step
                // multiplies it by exp(Delta A) <= 1), and what it would still add to y is 2^7 (bf16: 2^-16
                // against the 2^-9 rounding of the stored y) or 2^6 (fp32) times below the rounding of the
                // entering state's contribution: record the super-tile, once.
                bool small = monotone;
#pragma unroll
                for (int j = 0; j < 4; ++j) small = small && fabsf(hh[j].y) <= thr[j];
                if (__all_sync(0xffffffffu, small) && !recorded) {
                    if (lane == 0) first_small[warp] = sup;
                    recorded = true;
                }
            }
            // this warp is done with TMEM buffer sup & 1 and with the stage of sup
            tc::fence_before_sync();
            __syncwarp();
            tc::mbar_arrive_if(&empty[sup & 1], lane == 0);
            k_cur = k_nxt;
        }

        output_pair(last_sup * TT + 3 * TB + 2 * ps, 1, Du_r[1], g_r[1]);  // the last sub-tile is odd
        if (ENDS) {
            float sdt = sdt_acc;
#pragma unroll
            for (int off = 1; off < S; off <<= 1) sdt += __shfl_xor_sync(0xffffffffu, sdt, off);
            if (valid) {
                const long long base = (b * a.nchunks + kch) * a.Dch + d;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const long long n = 4LL * s + j;
                    if (n < N) a.ws_h[base * N + n] = hh[j].y;
                }
                if (s == 0) a.ws_sdt[base] = sdt;
            }
        } else if (MODE == MODE_FULL && a.last_state != nullptr && valid && kch == a.nchunks - 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const long long n = 4LL * s + j;
                if (n < N) a.last_state[(b * a.Dch + d) * N + n] = hh[j].y;
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (producer && lane == 0 && *abort_flag != 0) atomicOr(&g_device_error, 1u);
    if (producer && lane == 0 && (*abort_flag != 0 || stopped)) {
        // the MMAs and loads this CTA started must finish before its TMEM and
        // shared memory are released (each stage has at most its latest
        // issued phase open)
        if (mma_issued > 0) {
            tc::umma_commit(done);
            tc::mbar_wait_bounded(done, 0, kWaitPolls);
        }
        for (int sn = max(0, last_loaded - NST + 1); sn <= last_loaded; ++sn)
            tc::mbar_wait_bounded(&io[sn % NST], (sn / NST) & 1, kWaitPolls);
    }
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(*taddr_s, Sh::TMEM_COLS);
    }
}


// The kernel: blockDim.x = 32 (W + 1), W = 8..11 compute warps and the producer warp.
template <typename T, int MODE, bool HAS_Z, int S_, bool CONV = false, int FLAGS = 0>
__global__ void __launch_bounds__(TmShape<T, MODE, S_, CONV>::LAUNCH_THR, 1)
scan_tm_kernel(const ScanArgs a, const __grid_constant__ TmMaps maps) {
    scan_tm_body<T, MODE, HAS_Z, S_, CONV, FLAGS, false>(a, maps);
}

// The lean form: W = 12..18 compute warps and the producer warp; at most 96 registers per thread.  A
// CTA's warps are spread over the SM's 4 sub-partitions, each with a quarter of the register file
// (16 384 registers): 19 warps put 5 warps on a sub-partition, 5 x 32 x 96 = 15 360.
template <typename T, int MODE, bool HAS_Z, int S_, int FLAGS = 0>
__global__ void __maxnreg__(96) scan_tm_lean_kernel(const ScanArgs a, const __grid_constant__ TmMaps maps) {
    scan_tm_body<T, MODE, HAS_Z, S_, false, FLAGS, true>(a, maps);
}

// Launch of one instantiation: grid (ceil(Dch / channels per CTA), Bsz, grid_chunks), W compute warps
// plus the producer warp, one CTA per SM.
template <typename T, int MODE, bool HAS_Z, int S, bool CONV = false, int FLAGS = 0, bool LEAN = false>
cudaError_t launch_tm_one(const ScanArgs &a, const TmMaps &maps, int warps, long long Bsz, int grid_chunks,
                          cudaStream_t st) {
    using Sh = TmShape<T, MODE, S, CONV, LEAN>;
    // registers of a full-width CTA: the warps on the busiest sub-partition fit its quarter of the file
    static_assert((Sh::MAX_WARPS + 1 + 3) / 4 * 32 * (LEAN ? 96 : 168) <= 16384, "registers of a full-width CTA");
    void (*kern)(const ScanArgs, const TmMaps) = nullptr;
    if constexpr (LEAN) kern = scan_tm_lean_kernel<T, MODE, HAS_Z, S, FLAGS>;
    else kern = scan_tm_kernel<T, MODE, HAS_Z, S, CONV, FLAGS>;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) attr_set[dev] = true;
    }
    const long long ch = 32LL * warps / S;
    dim3 grid((unsigned)((a.Dch + ch - 1) / ch), (unsigned)Bsz, (unsigned)grid_chunks);
    kern<<<grid, 32 * (warps + 1), Sh::SMEM_BYTES, st>>>(a, maps);  // + the producer warp
    return cudaGetLastError();
}

// The lean form (12..18 compute warps) of the plain direct scan, bf16 storage (FLAGS 0 or FL_CKPT).
template <int S, int FLAGS = 0>
cudaError_t launch_tm_lean(const ScanArgs &a, const TmMaps &maps, int warps, long long Bsz, cudaStream_t st) {
    return a.z != nullptr ? launch_tm_one<bf16_t, MODE_FULL, true, S, false, FLAGS, true>(a, maps, warps, Bsz, 1, st)
                          : launch_tm_one<bf16_t, MODE_FULL, false, S, false, FLAGS, true>(a, maps, warps, Bsz, 1, st);
}

// The direct scan that also writes the backward pass's checkpoints (scan_tm_ckpt.cu): the regular form
// (lean_warps == 0) or the lean form; dtype 1 = bf16, S lanes per channel.
cudaError_t launch_tm_ckpt(int dtype, int S, const ScanArgs &a, const TmMaps &maps, int warps, bool lean,
                           long long Bsz, cudaStream_t st);

template <typename T, int S, int FLAGS = 0>
cudaError_t launch_tm_s(int mode, const ScanArgs &a, const TmMaps &maps, int warps, long long Bsz, int gc,
                        cudaStream_t st) {
    if (mode == MODE_STATES) return launch_tm_one<T, MODE_STATES, false, S, false, FLAGS>(a, maps, warps, Bsz, gc, st);
    return a.z != nullptr ? launch_tm_one<T, MODE_FULL, true, S, false, FLAGS>(a, maps, warps, Bsz, gc, st)
                          : launch_tm_one<T, MODE_FULL, false, S, false, FLAGS>(a, maps, warps, Bsz, gc, st);
}

// The two passes of the decay-truncated chunked scan (scan_tm_chunk.cu): MODE_FULL_STATES and MODE_CORR.
cudaError_t launch_tm_chunk(int dtype, int S, int mode, const ScanArgs &a, const TmMaps &maps, int warps,
                            long long Bsz, int gc, cudaStream_t st);

// The instantiations that honour the scan flags: the reverse scan (scan_tm_rev.cu) and the exact
// zero-order hold, forwards or reverse (scan_tm_zoh.cu); dtype 1 = bf16, S lanes per channel.
cudaError_t launch_tm_rev(int dtype, int S, int mode, const ScanArgs &a, const TmMaps &maps, int warps,
                          long long Bsz, int gc, cudaStream_t st);
cudaError_t launch_tm_zoh(int dtype, int S, int mode, const ScanArgs &a, const TmMaps &maps, int warps,
                          long long Bsz, int gc, cudaStream_t st);

// Instantiate the kernels of one flag variant for every storage type and lane count.
template <int FL>
cudaError_t launch_tm_variant(int dtype, int S, int mode, const ScanArgs &a, const TmMaps &maps, int warps,
                              long long Bsz, int gc, cudaStream_t st) {
    if (dtype != 1) return launch_tm_s<float, 4, FL>(mode, a, maps, warps, Bsz, gc, st);
    switch (S) {
        case 4: return launch_tm_s<bf16_t, 4, FL>(mode, a, maps, warps, Bsz, gc, st);
        case 8: return launch_tm_s<bf16_t, 8, FL>(mode, a, maps, warps, Bsz, gc, st);
        default: return launch_tm_s<bf16_t, 16, FL>(mode, a, maps, warps, Bsz, gc, st);
    }
}

// Read and clear a device error word (MAMBA_OK, or MAMBA_ERR_DEVICE if the copy fails).
inline int read_clear_word(const unsigned int &word, unsigned int *v) {
    unsigned int zero = 0;
    *v = 0;
    if (cudaMemcpyFromSymbol(v, word, sizeof(*v)) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_DEVICE;
    }
    if (*v != 0 && cudaMemcpyToSymbol(word, &zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return MAMBA_ERR_DEVICE;
    }
    return MAMBA_OK;
}

}  // namespace mamba
