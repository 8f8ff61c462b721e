// conv1d.cu -- depthwise causal convolution of width 4 followed by SiLU, the
// branch that produces the scan's input u from x (ai.xwebgame.com summary,
// "running it in PyTorch" block: Conv1d(d_inner, d_inner, kernel_size=4,
// groups=d_inner, padding=3), first L outputs, then SiLU):
//   pre_t = bias_d + sum_{k=0..3} w[d][k] x_{t-3+k}   (x_s = 0 for s < 0),  u_t = SiLU(pre_t)
//
// HBM-bound (one read of x, one write of u).  Vector path: a warp covers 256
// consecutive steps of one row, 8 per lane (one 16-byte load for bf16, two for
// fp32); the three steps before a lane's first come from the previous lane by
// shuffle, lane 0 reads them itself.  Scalar path otherwise: one step per thread.
#include "../../include/mamba_scan.h"
#include "internal.h"

namespace mamba {

template <typename T>
__device__ __forceinline__ float conv_out(const float4 w, float b, float x0, float x1, float x2, float x3, bool silu) {
    const float pre = fmaf(w.w, x3, fmaf(w.z, x2, fmaf(w.y, x1, fmaf(w.x, x0, b))));
    return silu ? silu_f(pre) : pre;
}

template <typename T>
__global__ void __launch_bounds__(256)
conv1d_vec_kernel(const void *x, const float *w, const float *bias, int silu, void *u, long long rows, long long Dch,
                  long long L) {
    using IO = Io<T>;
    constexpr int PER16 = 16 / (int)sizeof(T);
    constexpr int NV = 8 / PER16;  // 16-byte vectors per lane (1 for bf16, 2 for fp32)
    const int lane = threadIdx.x & 31;
    const long long segs = (L + 255) / 256;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (warp >= rows * segs) return;  // whole warps exit together
    const long long r = warp / segs, seg = warp % segs;
    const long long d = r % Dch;
    const long long t0 = seg * 256 + 8LL * lane;
    const T *xr = reinterpret_cast<const T *>(x) + r * L;
    const float4 wv = __ldg(reinterpret_cast<const float4 *>(w + d * 4));
    const float bv = bias != nullptr ? __ldg(bias + d) : 0.f;

    float v[8];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        uint4 q = make_uint4(0u, 0u, 0u, 0u);
        if (t0 + (k + 1) * PER16 <= L) q = ldg16(xr + t0 + k * PER16);  // L is a multiple of PER16
#pragma unroll
        for (int i = 0; i < PER16; ++i) v[k * PER16 + i] = IO::get(q, i);
    }
    // the three steps before t0: the previous lane's last three, or loaded by lane 0
    float p5 = __shfl_up_sync(0xffffffffu, v[5], 1);
    float p6 = __shfl_up_sync(0xffffffffu, v[6], 1);
    float p7 = __shfl_up_sync(0xffffffffu, v[7], 1);
    if (lane == 0) {
        p5 = t0 >= 3 ? IO::load(x, r * L + t0 - 3) : 0.f;
        p6 = t0 >= 2 ? IO::load(x, r * L + t0 - 2) : 0.f;
        p7 = t0 >= 1 ? IO::load(x, r * L + t0 - 1) : 0.f;
    }
    const bool s = silu != 0;
    float o[8];
    o[0] = conv_out<T>(wv, bv, p5, p6, p7, v[0], s);
    o[1] = conv_out<T>(wv, bv, p6, p7, v[0], v[1], s);
    o[2] = conv_out<T>(wv, bv, p7, v[0], v[1], v[2], s);
#pragma unroll
    for (int i = 3; i < 8; ++i) o[i] = conv_out<T>(wv, bv, v[i - 3], v[i - 2], v[i - 1], v[i], s);
    T *ur = reinterpret_cast<T *>(u) + r * L;
#pragma unroll
    for (int k = 0; k < NV; ++k)
        if (t0 + (k + 1) * PER16 <= L) stg16(ur + t0 + k * PER16, IO::pack(o + k * PER16));
}

template <typename T>
__global__ void __launch_bounds__(256)
conv1d_scalar_kernel(const void *x, const float *w, const float *bias, int silu, void *u, long long rows,
                     long long Dch, long long L) {
    using IO = Io<T>;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * L) return;
    const long long r = i / L, t = i % L, d = r % Dch;
    float xs[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) xs[k] = t - 3 + k >= 0 ? IO::load(x, r * L + t - 3 + k) : 0.f;
    const float4 wv = make_float4(w[d * 4], w[d * 4 + 1], w[d * 4 + 2], w[d * 4 + 3]);
    IO::store(u, i, conv_out<T>(wv, bias != nullptr ? bias[d] : 0.f, xs[0], xs[1], xs[2], xs[3], silu != 0));
}

cudaError_t launch_conv1d(int dtype, bool vec, const void *x, const float *w, const float *bias, int silu, void *u,
                          long long rows, long long Dch, long long L, cudaStream_t st) {
    const int threads = 256;
    if (vec) {
        const long long warps = rows * ((L + 255) / 256);
        const long long blocks = (warps * 32 + threads - 1) / threads;
        if (dtype == 1)
            conv1d_vec_kernel<bf16_t><<<(unsigned)blocks, threads, 0, st>>>(x, w, bias, silu, u, rows, Dch, L);
        else
            conv1d_vec_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(x, w, bias, silu, u, rows, Dch, L);
    } else {
        const long long blocks = (rows * L + threads - 1) / threads;
        if (dtype == 1)
            conv1d_scalar_kernel<bf16_t><<<(unsigned)blocks, threads, 0, st>>>(x, w, bias, silu, u, rows, Dch, L);
        else
            conv1d_scalar_kernel<float><<<(unsigned)blocks, threads, 0, st>>>(x, w, bias, silu, u, rows, Dch, L);
    }
    return cudaGetLastError();
}

}  // namespace mamba
