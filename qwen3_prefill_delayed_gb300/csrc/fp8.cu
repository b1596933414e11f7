// fp8.cu -- E4M3 quantization for the static-FP8 variant of the prefill projections.
//
// The variant ("flashrt-structures 0.2.0, prefill_tower/fp8_chain.py" page, its description: RMSNorm then FP8, merged-QKV / output / gate-up /
// down FP8 GEMMs with static activation scales; "Stabilize Higgs Audio termination and prefill",
// Summary: the activation scales come from a fixed calibration prompt):
//   weights     w8 = e4m3(w / s_w), s_w = max|w| / 448 (1 for an all-zero tensor), once;
//   activations x8 = e4m3(x / s_a) before each projection, s_a static per layer and projection
//               (calibration: s_a = max|x| / 448 over a bf16 prefill of the calibration batch);
//   the GEMM multiplies its fp32 accumulators by s_a * s_w.
// e4m3() is the round-to-nearest-even, saturating (finite overflow -> +-448) conversion.
#include <cuda_fp8.h>

#include <algorithm>

#include "internal.h"

namespace hra {

namespace {

__device__ __forceinline__ uint8_t to_e4m3(float v) {
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// out[i] = e4m3(x[i] / *scale) (IEEE division), 8 elements per thread; n a multiple of 8.
__global__ void fp8_quantize_kernel(const bf16* __restrict__ x, long long n, const float* __restrict__ scale,
                                    uint8_t* __restrict__ out) {
    pdl_launch();
    pdl_wait();
    const float s = *scale;
    const long long n8 = n >> 3;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (long long)gridDim.x * blockDim.x) {
        float f[8];
        unpack8(reinterpret_cast<const uint4*>(x)[i], f);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) lo |= (uint32_t)to_e4m3(__fdiv_rn(f[j], s)) << (8 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j) hi |= (uint32_t)to_e4m3(__fdiv_rn(f[4 + j], s)) << (8 * j);
        reinterpret_cast<uint2*>(out)[i] = make_uint2(lo, hi);
    }
}

// *amax = max(*amax, max |x[i]|); the bits of non-negative floats order like the floats.
__global__ void absmax_kernel(const bf16* __restrict__ x, long long n, float* amax) {
    pdl_launch();
    pdl_wait();
    float m = 0.f;
    const long long n8 = n >> 3;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
         i += (long long)gridDim.x * blockDim.x) {
        float f[8];
        unpack8(reinterpret_cast<const uint4*>(x)[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float s_m[32];
    if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, s_m[w]);
        atomicMax(reinterpret_cast<int*>(amax), __float_as_int(m));
    }
}

// ---------------------------------------------------------------- NVFP4 (E2M1 + block scales)
// The FP4 band of the prefill chain (same page, its precision bands: the output projection and the
// FFN pair run in NVFP4 with per-block scales computed on the fly), in NVIDIA's published NVFP4 format: E2M1 elements, one
// E4M3 scale per 16 consecutive elements along K, one fp32 global scale g per tensor.

// value of a finite E4M3 code: (8 + M) 2^(E - 10) for E > 0, M 2^-9 for E = 0
__device__ __forceinline__ float e4m3_value(uint8_t c) {
    const int E = (c >> 3) & 15, M = c & 7;
    const float v = E == 0 ? ldexpf((float)M, -9) : ldexpf((float)(8 + M), E - 10);
    return (c & 0x80) ? -v : v;
}

// FP4 E2M1 code (sign in bit 3) of x: the nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6; at a midpoint
// the value with the even mantissa (even code); beyond 6 (and NaN) saturates to 6
__device__ __forceinline__ uint32_t to_e2m1(float x) {
    const uint32_t sgn = signbit(x) ? 8u : 0u;
    const float a = fabsf(x);
    if (!(a < 6.0f)) return sgn | 7u;
    uint32_t c;
    if (a <= 0.25f) c = 0;        // 0.25 lies between 0 and 0.5: 0
    else if (a < 0.75f) c = 1;    // 0.75 lies between 0.5 and 1: 1
    else if (a <= 1.25f) c = 2;   // 1.25: 1
    else if (a < 1.75f) c = 3;    // 1.75: 2
    else if (a <= 2.5f) c = 4;    // 2.5: 2
    else if (a < 3.5f) c = 5;     // 3.5: 4
    else if (a <= 5.0f) c = 6;    // 5: 4
    else c = 7;
    return sgn | c;
}

// One thread per 16-element block of x [rows][K]: s = e4m3(amax / (6 g)); codes =
// e2m1(x / (g dec(s))) (0 when g dec(s) is 0); every operation a single fp32 rounding.
__global__ void nvfp4_quantize_kernel(const bf16* __restrict__ x, int rows, int K, const float* __restrict__ g_ptr,
                                      uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    pdl_launch();
    pdl_wait();
    const int nb = K >> 4;
    const long long nblk = (long long)rows * nb;
    const float g = *g_ptr;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nblk;
         i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / nb;
        const int b = (int)(i - r * nb);
        const uint4* src = reinterpret_cast<const uint4*>(x + r * K + 16 * b);
        float f0[8], f1[8], f[16];
        unpack8(src[0], f0);
        unpack8(src[1], f1);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            f[j] = f0[j];
            f[8 + j] = f1[j];
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
        const uint8_t sc = to_e4m3(__fdiv_rn(amax, __fmul_rn(6.0f, g)));
        scales[i] = sc;
        const float step = __fmul_rn(g, e4m3_value(sc));
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            w[q] = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[q] |= (step > 0.f ? to_e2m1(__fdiv_rn(f[4 * q + e], step)) : 0u) << (8 * e);
        }
        *reinterpret_cast<uint4*>(codes + r * K + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// v[i] = 0 (the amax accumulators)
__global__ void zero_floats_kernel(float* v, int n) {
    pdl_launch();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) v[i] = 0.f;
}

// scale[i] = amax[i] > 0 ? amax[i] / 448 : 1
__global__ void amax_to_scale_kernel(const float* amax, float* scale, int n) {
    pdl_launch();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float a = amax[i];
        scale[i] = a > 0.f ? a / 448.0f : 1.0f;
    }
}

unsigned grid_for(long long n8) {
    const long long b = (n8 + 255) / 256;
    const long long cap = 8LL * device_sm_count();
    return (unsigned)std::max<long long>(1, std::min(b, cap));
}

}  // namespace

cudaError_t launch_nvfp4_quantize(const bf16* x, int rows, int K, const float* g, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t st) {
    const long long nblk = (long long)rows * (K / 16);
    const int threads = 256;
    const unsigned grid = (unsigned)std::min<long long>((nblk + threads - 1) / threads, 4LL * device_sm_count());
    HRA_LAUNCH(nvfp4_quantize_kernel, dim3(grid), dim3(threads), 0, st, x, rows, K, g, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_fp8_quantize(const bf16* x, long long n, const float* scale, uint8_t* out, cudaStream_t st) {
    HRA_LAUNCH(fp8_quantize_kernel, dim3(grid_for(n >> 3)), dim3(256), 0, st, x, n, scale, out);
    return cudaGetLastError();
}

cudaError_t launch_absmax(const bf16* x, long long n, float* amax, cudaStream_t st) {
    HRA_LAUNCH(absmax_kernel, dim3(grid_for(n >> 3)), dim3(256), 0, st, x, n, amax);
    return cudaGetLastError();
}

cudaError_t launch_zero_floats(float* v, int n, cudaStream_t st) {
    HRA_LAUNCH(zero_floats_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, v, n);
    return cudaGetLastError();
}

cudaError_t launch_amax_to_scale(const float* amax, float* scale, int n, cudaStream_t st) {
    HRA_LAUNCH(amax_to_scale_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, amax, scale, n);
    return cudaGetLastError();
}

}  // namespace hra
