// internal.h -- host-side launch interface between the C ABI (api.cu) and the
// kernels.  Not installed; the public interface is include/mamba_scan.h.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "scan_kernels.cuh"

namespace mamba {

constexpr int kMaxDevices = 64;

// Tile geometry of the scan kernel for a padded state count NP (4..64).
struct ScanGeom {
    int NP;      // padded state count (power of two >= N, >= 4)
    int TT;      // time steps per tile; chunk lengths are multiples of it
    int S;       // lanes per channel
    int CH;      // channels per CTA
    int threads; // threads per CTA
};
ScanGeom scan_geom(long long N);

// Cost of one launch of the tensor-memory scan kernel in units of one CTA's time: waves of CTAs (one
// CTA per SM) times the warps of the busiest SM sub-partition (W compute warps and the producer warp
// over 4 sub-partitions set the pace of a CTA).  *warps (if not null) receives the width W that
// minimises it, the narrower one on ties.  S = lanes per channel (4, 8 or 16).
long long tm_launch_cost(long long Bsz, long long Dch, int grid_chunks, int sms, int S, int *warps);

// Whether the tensor-memory kernel is the one that serves problems of this storage type and state
// count (on 16-byte aligned data without flags).
bool tm_kernel_for(int dtype, long long N);

// Launch the scan kernel: grid (ceil(Dch/CH), Bsz, grid_chunks).
cudaError_t launch_scan(int dtype, int mode, bool vec, const ScanArgs &a, long long Bsz, int grid_chunks,
                        cudaStream_t st);

// Tensor-memory variant of the scan kernel (N <= 16, 16-byte aligned rows):
// B/C reach the registers through TMEM instead of shared memory, inputs arrive
// by TMA.  Returns cudaErrorNotSupported, launching nothing, when the problem
// does not fit its TMA descriptors (the caller then uses the other kernel).
cudaError_t launch_scan_tm(int dtype, int mode, const ScanArgs &a, long long Bsz, int grid_chunks, cudaStream_t st);

// Carry pass of the chunked scan: per (b, d, n) an exclusive combine over the
// chunk (decay, end-state) pairs; writes every chunk's initial state into ws_h
// in place (hin[k] = prod decay * h0 + ...).  all_chunks false: ws_h and
// ws_sdt hold chunks 0..K-2 (the two-pass scan).  True: they hold all K chunks
// (the decay-truncated scan) and the state after the last chunk goes to
// last_state (if not null).
cudaError_t launch_carry(const float *A, const float *h0, float *ws_h, const float *ws_sdt, long long Bsz,
                         long long Dch, long long N, int K, cudaStream_t st, bool all_chunks = false,
                         float *last_state = nullptr);

// Whether the decay-truncated chunked scan (tensor-memory kernel) serves these sizes and flags.
bool tm_chunked_for(int dtype, long long N, int flags, bool vec, bool conv);

// The chunked scan after its workspace is in hand: the decay-truncated scan where tm_chunked_for holds
// (unless MAMBA_CHUNKED_SCAN=two-pass), else the two-pass scan (chunk end states, carry, seeded rescan).  a.chunk_len and a.nchunks
// set; ws_h [Bsz][K][Dch][N] and ws_sdt [Bsz][K][Dch]; h0 may be null.
cudaError_t run_chunked(int dtype, bool vec, ScanArgs a, long long Bsz, float *ws_h, float *ws_sdt,
                        const float *h0, cudaStream_t st);

// Read and clear the device error words of the tensor-memory scan's translation units (its plain, reverse
// and zero-order-hold instantiations); MAMBA_OK or MAMBA_ERR_DEVICE.
int tm_read_clear_error(unsigned int *v);
int tm_rev_read_clear_error(unsigned int *v);
int tm_zoh_read_clear_error(unsigned int *v);
int tm_chunk_read_clear_error(unsigned int *v);

struct StepArgs {
    float *state;
    const void *u, *delta, *z, *Bm, *Cm;
    const float *A, *D, *bias;
    void *y;
    long long Bsz, Dch, N;
    int softplus;
};
// lane_states: 8 or 4 for the aligned kernel with that many states per lane (16-byte aligned
// state and A rows, N and the B/C alignment multiples of it), 0 for the scalar kernel.
cudaError_t launch_state_update(int dtype, int lane_states, const StepArgs &a, cudaStream_t st);

// Depthwise causal conv (width 4) + optional SiLU over rows of length L
// (row r uses taps w[r % Dch]); vec: 16-byte aligned x, u, w and 16-byte rows.
cudaError_t launch_conv1d(int dtype, bool vec, const void *x, const float *w, const float *bias, int silu, void *u,
                          long long rows, long long Dch, long long L, cudaStream_t st);

cudaError_t launch_bench_ex2(long long *cycles, float *sink, long long iters, int blocks, int threads,
                             cudaStream_t st);

}  // namespace mamba
