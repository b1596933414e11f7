// nvfp4.cu -- the NVFP4 projection GEMM of the prefill chain's FP4 band.
//
// Source: the "flashrt-structures 0.2.0, prefill_tower/fp8_chain.py" page, its precision bands (the
// output projection and the FFN pair in NVFP4, per-block scales computed from the data), in
// NVIDIA's published NVFP4 format: E2M1 elements (one code per byte here, sign in bit 3), one E4M3
// scale per 16 consecutive elements along K, one fp32 global scale per tensor.
//
//   y[m][n] = (g_a g_w) * sum_k (e2m1(a[m][k]) dec(sa[m][k/16])) (e2m1(w[n][k]) dec(sw[n][k/16]))
//
// Every factor e2m1(.) dec(s) is exactly an f16 number (at most 5 significant bits, exponent inside
// f16's normal range), and so is every product of two of them in fp32: the kernel expands each
// E2M1 code times its block scale to f16 in shared memory and runs kind::f16 tcgen05 MMAs (f16
// operands, fp32 accumulation in TMEM), so the result is the NVFP4 product sum up to the order of
// fp32 additions.
//
// One CTA per 128 x 256 output tile (SwiGLU: 128 gate + the 128 matching up columns):
//   warp 0     TMA of the E2M1 code tiles (64 K x 128 rows boxes, no swizzle) into a 3-stage ring;
//   warps 2-9  expand codes x block scales into 128-byte-swizzled f16 tiles (a 3-stage ring; the
//              hardware's E2M1 and E4M3 conversions to f16, then one f16 multiply each), then,
//              after the last k-block, the epilogue from TMEM (two warps per lane quarter);
//   warp 1     TMEM allocation and the MMA issue (one lane), 4 x (128 x 256 x 16) per k-block.
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"

namespace hra {

namespace {

constexpr int kNvThreads = 320;
constexpr int kNvDeq = 256;          // expanding threads (warps 2-9)
constexpr int kNvBN = 256;
constexpr int kCodeStages = 3;
constexpr int kHalfStages = 3;
constexpr int kACodes = 128 * 64;    // bytes
constexpr int kWCodes = kNvBN * 64;
constexpr int kCodeStage = kACodes + kWCodes;
constexpr int kAHalf = 128 * 128;    // 128 rows x 64 f16
constexpr int kWHalf = kNvBN * 128;
constexpr int kHalfStage = kAHalf + kWHalf;
constexpr int kNvSmem = kCodeStages * kCodeStage + kHalfStages * kHalfStage + 1024 + 256;

enum NvMode : int { NV_STORE = 0, NV_RESIDUAL = 1, NV_SWIGLU = 2, NV_F32 = 3 };

struct NvArgs {
    const uint8_t* a_scales;   // [M][K/16]
    const uint8_t* w_scales;   // [w_rows][K/16]
    const float* g_a;          // device scalars
    const float* g_w;
    void* out;
    unsigned int* err;
    int M, N, K;               // N: output columns (F for SwiGLU)
    int w_rows;                // rows of the weight (2F for SwiGLU)
    int mode;
    int mt;
};

// kind::f16 instruction descriptor with A and B f16 (type code 0), D fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Two E2M1 codes in the low bytes of w (one code per byte, sign in bit 3) -> f16x2 (the first code
// in the low half), exactly: the codes are packed into one byte and converted by the hardware.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t w) {
    const uint32_t packed = (w & 0x0Fu) | ((w >> 4) & 0xF0u);
    uint32_t d;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(d) : "r"(packed));
    return d;
}

// Two E4M3 codes in the low 16 bits of w -> f16x2 (exact).
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t w) {
    uint32_t d;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(d) : "r"(w));
    return *reinterpret_cast<__half2*>(&d);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, __half2 s) {
    __half2 x = *reinterpret_cast<__half2*>(&a);
    x = __hmul2(x, s);
    return *reinterpret_cast<uint32_t*>(&x);
}

__device__ __forceinline__ float silu_nv(float x) { return x / (1.0f + expf(-x)); }

__global__ void __launch_bounds__(kNvThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW,
                      const NvArgs p) {
    pdl_launch();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* halfs = smem;                                           // f16 ring (1024-aligned stages)
    uint8_t* codes = smem + kHalfStages * kHalfStage;                // code ring
    uint64_t* bars = reinterpret_cast<uint64_t*>(codes + kCodeStages * kCodeStage);
    // bars: code_full[3], code_empty[3], half_full[3], half_empty[3], tfull
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kCodeStages + 2 * kHalfStages + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued_slot = reinterpret_cast<int*>(tmem_slot + 2);
    int* committed_slot = reinterpret_cast<int*>(tmem_slot + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_blk = blockIdx.x % p.mt, n_blk = blockIdx.x / p.mt;
    const int m0 = m_blk * 128;
    const bool swiglu = p.mode == NV_SWIGLU;
    const int wrow0 = swiglu ? n_blk * 128 : n_blk * kNvBN;               // first row of the tile's first half
    const int wrow1 = swiglu ? p.N + n_blk * 128 : n_blk * kNvBN + 128;   // first row of the second half
    const int n_kb = p.K / 64, nb16 = p.K / 16;

    auto code_full = [&](int s) { return smem_u32(bars + s); };
    auto code_empty = [&](int s) { return smem_u32(bars + kCodeStages + s); };
    auto half_full = [&](int s) { return smem_u32(bars + 2 * kCodeStages + s); };
    auto half_empty = [&](int s) { return smem_u32(bars + 2 * kCodeStages + kHalfStages + s); };
    const uint32_t tfull = smem_u32(bars + 2 * kCodeStages + 2 * kHalfStages);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kCodeStages; ++s) {
            mbar_init(code_full(s), 1);
            mbar_init(code_empty(s), kNvDeq / 32);
        }
        for (int s = 0; s < kHalfStages; ++s) {
            mbar_init(half_full(s), kNvDeq / 32);
            mbar_init(half_empty(s), 1);
        }
        mbar_init(tfull, 1);
        *abort_flag = 0;
        *issued_slot = 0;
        *committed_slot = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmW);
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            // weight codes of the first stages before waiting for the kernels ahead (weights are
            // constant; the activation codes are written by the quantizer just before)
            const int pre = min(kCodeStages, n_kb);
            for (int i = 0; i < pre; ++i) {
                mbar_expect_tx(code_full(i), kCodeStage);
                const uint32_t wdst = smem_u32(codes + i * kCodeStage + kACodes);
                tma_load_2d(wdst, &tmW, code_full(i), i * 64, wrow0);
                tma_load_2d(wdst + 128 * 64, &tmW, code_full(i), i * 64, wrow1);
            }
            pdl_wait();
            int s = 0, i = 0;
            uint32_t ph = 0;
            for (; i < n_kb; ++i) {
                uint8_t* st = codes + s * kCodeStage;
                if (i >= pre) {
                    if (!mbar_wait(code_empty(s), ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                    mbar_expect_tx(code_full(s), kCodeStage);
                    tma_load_2d(smem_u32(st + kACodes), &tmW, code_full(s), i * 64, wrow0);
                    tma_load_2d(smem_u32(st + kACodes + 128 * 64), &tmW, code_full(s), i * 64, wrow1);
                }
                tma_load_2d(smem_u32(st), &tmA, code_full(s), i * 64, m0);
                if (++s == kCodeStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            *issued_slot = max(i, pre);
        }
    } else if (warp == 1) {
        pdl_wait();
        tmem_alloc(smem_u32(tmem_slot), kNvBN);
        tmem_relinquish();
        tc_fence_before();
        asm volatile("bar.sync 2, 288;" ::: "memory");
        tc_fence_after();
        const uint32_t tmem = *tmem_slot;
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(128, kNvBN);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int i = 0; i < n_kb; ++i) {
                if (!mbar_wait(half_full(s), ph, abort_flag)) {
                    *abort_flag = 1;
                    raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sdesc_sw128(smem_u32(halfs + s * kHalfStage));
                const uint64_t bd = sdesc_sw128(smem_u32(halfs + s * kHalfStage + kAHalf));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc_mma_bf16(tmem, ad + 2ull * k, bd + 2ull * k, idesc, (i > 0 || k > 0) ? 1u : 0u);
                tc_commit(half_empty(s));
                if (++s == kHalfStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok) {
                tc_commit(tfull);
                *committed_slot = 1;
            }
        }
    } else {
        // ---- expansion: block q = td + 256 j (j < 6) of the k-block -- 16 codes sharing one scale --
        // A rows 0..127, then W rows 0..255, four 16-element blocks per 64-element row
        pdl_wait();
        asm volatile("bar.sync 2, 288;" ::: "memory");
        const int td = threadIdx.x - 64;
        constexpr int kBlocks = (kACodes + kWCodes) / 16 / kNvDeq;   // 6
        const uint8_t* srow[kBlocks];   // the block's scale in k-block 0, or null past the matrix
        uint32_t src_off[kBlocks], dst0[kBlocks], dst1[kBlocks];
#pragma unroll
        for (int j = 0; j < kBlocks; ++j) {
            const int q = td + kNvDeq * j;
            const bool is_a = q < 512;
            const int r = is_a ? (q >> 2) : ((q - 512) >> 2);
            const int blk = q & 3;
            if (is_a) {
                const int m = m0 + r;
                srow[j] = m < p.M ? p.a_scales + (long long)m * nb16 + blk : nullptr;
            } else {
                const int wr = r < 128 ? wrow0 + r : wrow1 + r - 128;
                srow[j] = wr < p.w_rows ? p.w_scales + (long long)wr * nb16 + blk : nullptr;
            }
            src_off[j] = (is_a ? 0u : (uint32_t)kACodes) + (uint32_t)(r * 64 + blk * 16);
            const uint32_t base = (is_a ? 0u : (uint32_t)kAHalf) + (uint32_t)(r * 128);
            dst0[j] = base + (uint32_t)(((2 * blk) ^ (r & 7)) << 4);
            dst1[j] = base + (uint32_t)(((2 * blk + 1) ^ (r & 7)) << 4);
        }
        int cs = 0, hs = 0;
        uint32_t cph = 0, hph = 0;
        bool ok = true;
        uint32_t sc[kBlocks];
#pragma unroll
        for (int j = 0; j < kBlocks; ++j) sc[j] = srow[j] ? __ldg(srow[j]) : 0u;
        for (int i = 0; i < n_kb; ++i) {
            uint32_t scn[kBlocks];   // next k-block's scales, requested before this one is expanded
#pragma unroll
            for (int j = 0; j < kBlocks; ++j) scn[j] = (srow[j] && i + 1 < n_kb) ? __ldg(srow[j] + 4 * (i + 1)) : 0u;
            if (!mbar_wait(code_full(cs), cph, abort_flag) || !mbar_wait(half_empty(hs), hph ^ 1u, abort_flag)) {
                *abort_flag = 1;
                raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                ok = false;
                break;
            }
            const uint8_t* cst = codes + cs * kCodeStage;
            uint8_t* hst = halfs + hs * kHalfStage;
#pragma unroll
            for (int j = 0; j < kBlocks; ++j) {
                const uint4 cw = *reinterpret_cast<const uint4*>(cst + src_off[j]);   // 16 codes
                const __half2 s2 = e4m3x2_to_half2(sc[j] | (sc[j] << 8));
                uint4 o0, o1;
                o0.x = hmul2_u32(e2m1x2_to_f16x2(cw.x), s2);
                o0.y = hmul2_u32(e2m1x2_to_f16x2(cw.x >> 16), s2);
                o0.z = hmul2_u32(e2m1x2_to_f16x2(cw.y), s2);
                o0.w = hmul2_u32(e2m1x2_to_f16x2(cw.y >> 16), s2);
                o1.x = hmul2_u32(e2m1x2_to_f16x2(cw.z), s2);
                o1.y = hmul2_u32(e2m1x2_to_f16x2(cw.z >> 16), s2);
                o1.z = hmul2_u32(e2m1x2_to_f16x2(cw.w), s2);
                o1.w = hmul2_u32(e2m1x2_to_f16x2(cw.w >> 16), s2);
                *reinterpret_cast<uint4*>(hst + dst0[j]) = o0;
                *reinterpret_cast<uint4*>(hst + dst1[j]) = o1;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(half_full(hs));
                mbar_arrive(code_empty(cs));
            }
#pragma unroll
            for (int j = 0; j < kBlocks; ++j) sc[j] = scn[j];
            if (++cs == kCodeStages) {
                cs = 0;
                cph ^= 1u;
            }
            if (++hs == kHalfStages) {
                hs = 0;
                hph ^= 1u;
            }
        }
        // ---- epilogue: two warps per TMEM lane quarter split the tile's columns
        ok = __all_sync(0xffffffffu, ok);
        if (ok && !__all_sync(0xffffffffu, mbar_wait(tfull, 0u, abort_flag))) {
            *abort_flag = 1;
            raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
            ok = false;
        }
        if (ok) {
            tc_fence_after();
            const int quad = warp & 3, half = (warp - 2) >> 2;
            const int row = quad * 32 + lane;
            const int m = m0 + row;
            const uint32_t tq = *tmem_slot + ((uint32_t)(quad * 32) << 16);
            const float g = *p.g_a * *p.g_w;
            if (swiglu) {
#pragma unroll 1
                for (int c = 0; c < 64; c += 32) {
                    float vg[32], vu[32];
                    tmem_ld32(tq + (uint32_t)(64 * half + c), vg);
                    tmem_ld32(tq + (uint32_t)(128 + 64 * half + c), vu);
                    const int n = n_blk * 128 + 64 * half + c;
                    if (m < p.M) {
                        bf16* o = reinterpret_cast<bf16*>(p.out) + (long long)m * p.N + n;
#pragma unroll
                        for (int i = 0; i < 32; i += 8) {
                            if (n + i >= p.N) break;
                            float f[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                f[e] = silu_nv(round_bf(vg[i + e] * g)) * round_bf(vu[i + e] * g);
                            *reinterpret_cast<uint4*>(o + i) = pack8(f);
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    float v[32];
                    tmem_ld32(tq + (uint32_t)(128 * half + c), v);
                    const int n = n_blk * kNvBN + 128 * half + c;
                    if (m < p.M) {
                        if (p.mode == NV_F32) {
                            float* o = reinterpret_cast<float*>(p.out) + (long long)m * p.N + n;
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                if (n + i < p.N)
                                    *reinterpret_cast<float4*>(o + i) =
                                        make_float4(v[i] * g, v[i + 1] * g, v[i + 2] * g, v[i + 3] * g);
                        } else {
                            bf16* o = reinterpret_cast<bf16*>(p.out) + (long long)m * p.N + n;
#pragma unroll
                            for (int i = 0; i < 32; i += 8) {
                                if (n + i >= p.N) break;
                                float f[8];
                                if (p.mode == NV_RESIDUAL) {
                                    float r8[8];
                                    unpack8(*reinterpret_cast<const uint4*>(o + i), r8);
#pragma unroll
                                    for (int e = 0; e < 8; ++e) f[e] = r8[e] + v[i + e] * g;
                                } else {
#pragma unroll
                                    for (int e = 0; e < 8; ++e) f[e] = v[i + e] * g;
                                }
                                *reinterpret_cast<uint4*>(o + i) = pack8(f);
                            }
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == 0 && lane == 0) {
        // a wait gave up: let every copy and MMA already issued land before the memory goes away
        volatile int never = 0;
        const int issued = *issued_slot;
        for (int i = max(0, issued - kCodeStages); i < issued; ++i)
            (void)mbar_wait(code_full(i % kCodeStages), (uint32_t)(i / kCodeStages) & 1u, &never);
        if (*committed_slot) (void)mbar_wait(tfull, 0u, &never);
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(*tmem_slot, kNvBN);
    }
}

// out[i] = amax[i] > 0 ? amax[i] / div : 1
__global__ void amax_div_kernel(const float* amax, float* out, int n, float div) {
    pdl_launch();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float a = amax[i];
        out[i] = a > 0.f ? a / div : 1.0f;
    }
}

// Static input scales of the NVFP4 band from the calibration amax [n_layers][4]: the QKV input's
// E4M3 scale amax / 448, the other three inputs' NVFP4 global scale amax / (6 * 448); 1 where amax
// is 0.
__global__ void nvfp4_band_scales_kernel(const float* amax, float* scale, int n) {
    pdl_launch();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float a = amax[i];
        scale[i] = a > 0.f ? a / ((i & 3) == 0 ? 448.0f : 6.0f * 448.0f) : 1.0f;
    }
}

}  // namespace

cudaError_t launch_nvfp4_band_scales(const float* amax, float* scale, int n_layers, cudaStream_t st) {
    const int n = 4 * n_layers;
    HRA_LAUNCH(nvfp4_band_scales_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, amax, scale, n);
    return cudaGetLastError();
}

cudaError_t launch_amax_div(const float* amax, float* out, int n, float div, cudaStream_t st) {
    HRA_LAUNCH(amax_div_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, amax, out, n, div);
    return cudaGetLastError();
}

cudaError_t launch_linear_nvfp4(const Nvfp4Call& c, cudaStream_t st) {
    if (c.M < 1 || c.N < 8 || c.N % 8 != 0 || c.K < 64 || c.K % 64 != 0) return cudaErrorInvalidValue;
    const bool sw = c.epi == EPI_SWIGLU;
    const int w_rows = sw ? 2 * c.N : c.N;
    CUtensorMap ma, mw;
    if (!make_map_u8(&ma, c.a_codes, c.M, c.K, 128)) return cudaErrorInvalidValue;
    if (!make_map_u8(&mw, c.w_codes, w_rows, c.K, 128)) return cudaErrorInvalidValue;
    NvArgs p{};
    p.a_scales = c.a_scales;
    p.w_scales = c.w_scales;
    p.g_a = c.g_a;
    p.g_w = c.g_w;
    p.out = c.out;
    p.err = c.err;
    p.M = c.M;
    p.N = c.N;
    p.K = c.K;
    p.w_rows = w_rows;
    p.mode = c.epi == EPI_STORE ? NV_STORE : c.epi == EPI_RESIDUAL ? NV_RESIDUAL : sw ? NV_SWIGLU : NV_F32;
    p.mt = (c.M + 127) / 128;
    const int nt = sw ? (c.N + 127) / 128 : (c.N + kNvBN - 1) / kNvBN;
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(gemm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kNvSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    HRA_LAUNCH(gemm_nvfp4_kernel, dim3((unsigned)(p.mt * nt)), dim3(kNvThreads), kNvSmem, st, ma, mw, p);
    return cudaGetLastError();
}

}  // namespace hra
