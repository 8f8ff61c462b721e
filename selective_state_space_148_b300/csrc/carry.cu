// carry.cu -- carry pass of the sequence-parallel (chunked) scan.
//
// Within one channel and state the step h_t = a_t h_{t-1} + x_t is the affine
// map h -> a_t h + x_t.  Composing two consecutive maps gives
//   (a1, x1) then (a2, x2)  =  (a1 a2, a2 x1 + x2),
// an associative operator (freeguideonline tutorial §5.1: the recurrence as a
// scan under a binary operator that combines step transforms).  Pass A of the
// chunked scan reduced every chunk k to its pair (prod_t a_t, end state from
// zero) = (exp(A * sum_t Delta_t), h_end[k]).  This kernel folds the pairs in
// chunk order, starting from h0, and leaves in ws_h[k] the state that enters
// chunk k; pass B rescans each chunk from it.  In the decay-truncated scheme
// every chunk (the last one too) comes with its pair, and the fold also
// yields the state after the last chunk.  K is small (tens to a few
// hundred), so one thread per (b, d, n) walks the chunks; its loads do not
// depend on the running value and are issued ahead by the unrolled loop.
#include "internal.h"

namespace mamba {

__global__ void __launch_bounds__(256)
carry_kernel(const float *__restrict__ A, const float *__restrict__ h0, float *ws_h,
             const float *__restrict__ ws_sdt, long long Bsz, long long Dch, long long N, int K,
             int all_chunks, float *last_state) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (b, d, n), n fastest
    if (i >= Bsz * Dch * N) return;
    const long long n = i % N, bd = i / N, d = bd % Dch, b = bd / Dch;
    const float an = A[d * N + n];
    const int kend = all_chunks ? K : K - 1;  // chunks with an end state
    float carry = h0 != nullptr ? h0[i] : 0.f;
#pragma unroll 8
    for (int k = 0; k < K; ++k) {
        const long long base = (b * K + k) * Dch + d;
        float e = 0.f, sdt = 0.f;
        if (k < kend) {
            e = ws_h[base * N + n];
            sdt = ws_sdt[base];
        }
        ws_h[base * N + n] = carry;  // state entering chunk k
        carry = fmaf(expf(an * sdt), carry, e);
    }
    if (all_chunks && last_state != nullptr) last_state[i] = carry;  // the state after the last chunk
}

cudaError_t launch_carry(const float *A, const float *h0, float *ws_h, const float *ws_sdt, long long Bsz,
                         long long Dch, long long N, int K, cudaStream_t st, bool all_chunks, float *last_state) {
    const long long total = Bsz * Dch * N;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    carry_kernel<<<(unsigned)blocks, threads, 0, st>>>(A, h0, ws_h, ws_sdt, Bsz, Dch, N, K, all_chunks ? 1 : 0,
                                                       last_state);
    return cudaGetLastError();
}

}  // namespace mamba
