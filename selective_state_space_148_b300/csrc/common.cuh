// common.cuh -- device helpers shared by the selective-scan kernels.
//
// Storage types: fp32 or bf16 (kept as raw 16-bit patterns).  Arithmetic is
// always fp32.  The special-function instructions are used as functions
// (ex2/lg2/rcp .approx); nothing here re-implements CUDA's math library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mamba {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- MUFU wrappers
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// softplus(x) = log(1 + e^x), for Delta = softplus(Delta_raw + bias)
// (fsdata.site explainer §3.2; freeguideonline tutorial §4.2 step 2).
//   x > 15            : x                      (log1p(e^-x) < 3.1e-7 absolute)
//   e = e^x < 1/16    : e - e^2/2 + e^3/3 - e^4/4 + e^5/5  (Taylor series of
//                       log1p, truncation < e^6/6, i.e. < 2e-7 relative)
//   otherwise         : log2(1 + e) * ln 2     (1 + e >= 17/16 keeps the
//                       lg2 error relative, not absolute)
// The series branch matters: the workloads draw Delta_raw + bias around -2..-9,
// where 1 + e rounds away most digits of e.
__device__ __forceinline__ float softplus_f(float x) {
    const float e = ex2_approx(x * kLog2e);
    const float big = lg2_approx(1.0f + e) * kLn2;
    float p = fmaf(e, 0.2f, -0.25f);
    p = fmaf(e, p, 0.33333334f);
    p = fmaf(e, p, -0.5f);
    p = fmaf(e, p, 1.0f);
    const float small = e * p;
    const float r = (e < 0.0625f) ? small : big;
    return (x > 15.0f) ? x : r;
}

// SiLU(z) = z * sigmoid(z) = z / (1 + e^-z)  (nn.SiLU of the gate branch).
// For z -> -inf, e^-z -> inf and the result tends to -0 as it should.
__device__ __forceinline__ float silu_f(float z) {
    return z * rcp_approx(1.0f + ex2_approx(-z * kLog2e));
}

// Pairwise forms used by the scan kernel (two time steps at a time, f32x2).
// FAST selects the forms used for bf16 storage, whose output rounding (2^-9
// relative) dwarfs their error:
//   softplus(x) = max(x, ln2 * log2(1 + 2^(min(x, 15) * log2 e)))  -- two MUFU ops;
//     the lg2 of a value near 1 carries ~2^-22 absolute error, i.e. ~1e-4
//     relative error on the smallest Delta of the workloads;
//   y * SiLU(z) = (y z / 2) (1 + tanh(z / 2))                        -- one MUFU op;
//     tanh.approx has ~2^-11 relative error.
// The fp32-storage path keeps the accurate scalar forms above.
template <bool FAST>
__device__ __forceinline__ float2 softplus2(float2 x) {
    if (FAST) {
        const float2 xm = f2(fminf(x.x, 15.0f), fminf(x.y, 15.0f));
        const float2 sc = __fmul2_rn(xm, f2(kLog2e, kLog2e));
        const float2 e1 = __fadd2_rn(f2(ex2_approx(sc.x), ex2_approx(sc.y)), f2(1.0f, 1.0f));
        const float2 r = __fmul2_rn(f2(lg2_approx(e1.x), lg2_approx(e1.y)), f2(kLn2, kLn2));
        return f2(fmaxf(r.x, x.x), fmaxf(r.y, x.y));
    }
    return f2(softplus_f(x.x), softplus_f(x.y));
}
template <bool FAST>
__device__ __forceinline__ float2 gate2(float2 y, float2 z) {
    if (FAST) {
        const float2 g = __fmul2_rn(z, f2(0.5f, 0.5f));
        const float2 th = f2(tanh_approx(g.x), tanh_approx(g.y));
        const float2 yg = __fmul2_rn(y, g);
        return __ffma2_rn(yg, th, yg);
    }
    return f2(y.x * silu_f(z.x), y.y * silu_f(z.y));
}

// SiLU of a pair: FAST (bf16 storage) as (z / 2) (1 + tanh(z / 2)), one MUFU op
// per element; otherwise the accurate scalar form above.
template <bool FAST>
__device__ __forceinline__ float2 silu2(float2 z) {
    if (FAST) {
        const float2 hz = __fmul2_rn(z, f2(0.5f, 0.5f));
        return __ffma2_rn(hz, f2(tanh_approx(hz.x), tanh_approx(hz.y)), hz);
    }
    return f2(z.x * rcp_approx(1.0f + ex2_approx(-z.x * kLog2e)), z.y * rcp_approx(1.0f + ex2_approx(-z.y * kLog2e)));
}

// global stores that happen only where pred holds, without a branch around them
__device__ __forceinline__ void st_b32_if(void *p, uint32_t v, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q st.global.b32 [%0], %1;\n\t}\n" ::"l"(p), "r"(v),
                 "r"((uint32_t)pred)
                 : "memory");
}
__device__ __forceinline__ void st_f32x2_if(void *p, float2 v, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %3, 0;\n\t@q st.global.v2.f32 [%0], {%1, %2};\n\t}\n" ::"l"(p),
                 "f"(v.x), "f"(v.y), "r"((uint32_t)pred)
                 : "memory");
}

// ---------------------------------------------------------------- storage types
struct bf16_t {  // tag type: 16-bit brain float stored as its bit pattern
    uint16_t bits;
};

template <typename T>
struct Io;

template <>
struct Io<float> {
    static constexpr int kPer16 = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static float load(const void *p, long long i) {
        return __ldg(reinterpret_cast<const float *>(p) + i);
    }
    __device__ __forceinline__ static void store(void *p, long long i, float v) {
        reinterpret_cast<float *>(p)[i] = v;
    }
    // element j (0..3) of a 16-byte vector
    __device__ __forceinline__ static float get(const uint4 &v, int j) {
        const uint32_t w = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
        return __uint_as_float(w);
    }
    __device__ __forceinline__ static void set(uint4 &v, int j, float f) {
        const uint32_t w = __float_as_uint(f);
        if (j == 0) v.x = w;
        else if (j == 1) v.y = w;
        else if (j == 2) v.z = w;
        else v.w = w;
    }
    // pack 4 values into one 16-byte vector (for 4-element stores)
    __device__ __forceinline__ static uint4 pack(const float *f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// two fp32 -> packed bf16x2, round to nearest even (lo in the low half)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <>
struct Io<bf16_t> {
    static constexpr int kPer16 = 8;
    __device__ __forceinline__ static float load(const void *p, long long i) {
        const uint16_t h = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    __device__ __forceinline__ static void store(void *p, long long i, float v) {
        reinterpret_cast<uint16_t *>(p)[i] = static_cast<uint16_t>(pack_bf16x2(v, 0.0f) & 0xffffu);
    }
    __device__ __forceinline__ static float get(const uint4 &v, int j) {
        const int k = j >> 1;
        const uint32_t w = k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
        return (j & 1) ? bf16_hi(w) : bf16_lo(w);
    }
    __device__ __forceinline__ static void set(uint4 &v, int j, float f) {
        const uint32_t h = __float_as_uint(f) >> 16;  // exact for values read from bf16
        const int k = j >> 1;
        uint32_t *w = k == 0 ? &v.x : k == 1 ? &v.y : k == 2 ? &v.z : &v.w;
        *w = (j & 1) ? ((*w & 0x0000ffffu) | (h << 16)) : ((*w & 0xffff0000u) | h);
    }
    __device__ __forceinline__ static uint4 pack(const float *f) {
        return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                          pack_bf16x2(f[6], f[7]));
    }
};

__device__ __forceinline__ uint4 ldg16(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void stg16(void *p, const uint4 &v) { *reinterpret_cast<uint4 *>(p) = v; }

}  // namespace mamba
