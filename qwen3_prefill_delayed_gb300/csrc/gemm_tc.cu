// gemm_tc.cu -- BF16 projection GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Computes D[m, n] = sum_k A[m, k] * W[n, k] for A = activations [M, K] and W = weight rows
// [N, K] (both K-major, bf16), fp32 accumulation in tensor memory, with the epilogue fused:
// plain bf16 store, in-place residual add (r = bf16(r + acc)), SwiGLU over the gate and up rows
// of a merged [2F, K] weight (h = bf16(silu(bf16(g)) * bf16(u))), or fp32 store.  These are the
// projection GEMMs of the batched prefill ("Stabilize Higgs Audio termination and prefill",
// Summary: "projection GEMMs"; merged QKV and merged gate/up as in "fp8_chain.py", run()) and the
// audio-head projection.
//
// One CTA owns a 128 x BN output tile (M = 128 rows of A per tcgen05.mma, N = BN weight rows):
//   warp 0     TMA producer: streams 128x64 A boxes and BNx64 W boxes (128-byte swizzle) into a
//              STAGES-deep shared-memory ring, one mbarrier pair per stage;
//   warp 1     allocates BN TMEM columns; one elected lane issues 4 tcgen05.mma (K = 16 each) per
//              64-wide K block and commits each stage back to the producer;
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane TMEM quadrant (one output row per thread),
//              fused epilogue math, 16-byte vector stores.
// Small-M calls (decode rows, the last prefill layer, the audio head) split K across CTAs so the
// weight stream covers every SM; the fp32 partials are summed in split order by a second kernel
// that then applies the epilogue.
#include <algorithm>
#include <cudaTypedefs.h>
#include <mutex>

#include "internal.h"

namespace hra {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;

enum KMode : int { KM_STORE = 0, KM_RESIDUAL = 1, KM_SWIGLU = 2, KM_F32 = 3, KM_PARTIAL = 4 };

struct GemmArgs {
    void* out;
    unsigned int* err;
    long long split_stride;   // elements between split partial planes (KM_PARTIAL)
    int M;
    int n_valid;              // valid output columns (N, or F for SwiGLU)
    int ldo;                  // output row stride in elements
    int n_kb;                 // K / 64
    int kb_per_split;
    int up_row0;              // SwiGLU: first up row in W (= F)
    int mode;
    int mt, nt, splits;       // tile grid: M tiles, N tiles, K splits
    int group;                // N tiles per raster band
};

template <int BN>
struct Cfg {
    static constexpr int STAGES = BN >= 256 ? 4 : 6;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
    // two fp32 accumulators of BN columns each: the epilogue drains one while the MMA fills the other
    static constexpr uint32_t TMEM_COLS = 2 * BN;
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// Store 32 fp32 values of one output row starting at column `col`; `nv` columns are valid
// (multiple of 8 for bf16, of 4 for fp32).
__device__ __forceinline__ void store_row_chunk(int mode, void* out, long long off, const float (&v)[32],
                                                int nv) {
    if (mode == KM_F32 || mode == KM_PARTIAL) {
        float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + off);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (4 * i < nv) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        return;
    }
    uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(out) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (8 * i >= nv) break;
        float f[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = v[8 * i + j];
        if (mode == KM_RESIDUAL) {
            float r[8];
            unpack8(p[i], r);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = r[j] + f[j];
        }
        p[i] = pack8(f);
    }
}

// Work unit u -> (M tile, N tile, K split).  Tiles are rastered in bands of `group` N tiles with
// the M tile varying fastest inside a band, so the CTAs resident at one time share a few weight
// tiles (and the activation tiles stay in L2 across bands when they fit).
__device__ __forceinline__ void unit_coords(int u, const GemmArgs& p, int& m_blk, int& n_blk, int& split) {
    const int tiles = p.mt * p.nt;
    split = u / tiles;
    const int t = u - split * tiles;
    const int band_units = p.group * p.mt;
    const int band = t / band_units;
    const int within = t - band * band_units;
    m_blk = within % p.mt;
    n_blk = band * p.group + within / p.mt;
}

// Persistent: each CTA walks work units blockIdx.x, blockIdx.x + gridDim.x, ...
template <int BN, bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs p) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    // bars: full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued_slot = reinterpret_cast<int*>(tmem_slot + 2);
    int* committed_slot = reinterpret_cast<int*>(tmem_slot + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = p.mt * p.nt * p.splits;

    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + C::STAGES + s); };
    auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * C::STAGES + b); };
    auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * C::STAGES + 2 + b); };
    auto a_tile = [&](int s) { return smem_u32(smem + s * C::STAGE_BYTES); };
    auto b_tile = [&](int s) { return smem_u32(smem + s * C::STAGE_BYTES + C::A_BYTES); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4);   // one arrival per epilogue warp
        }
        *abort_flag = 0;
        *issued_slot = 0;
        *committed_slot = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: one continuous stage ring across all of this CTA's units
        int it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
            int mb, nb, sp;
            unit_coords(u, p, mb, nb, sp);
            const int kb0 = sp * p.kb_per_split;
            const int kb1 = min(p.n_kb, kb0 + p.kb_per_split);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
                if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                mbar_expect_tx(full_bar(s), C::STAGE_BYTES);
                const int kx = kb * BK;
                tma_load_2d(a_tile(s), &tmA, full_bar(s), kx, mb * BM);
                if (SWIGLU) {
                    const int j0 = nb * (BN / 2);
                    tma_load_2d(b_tile(s), &tmB, full_bar(s), kx, j0);
                    tma_load_2d(b_tile(s) + C::B_BYTES / 2, &tmB, full_bar(s), kx, p.up_row0 + j0);
                } else {
                    tma_load_2d(b_tile(s), &tmB, full_bar(s), kx, nb * BN);
                }
            }
        }
        *issued_slot = it;
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer: accumulator buffer j % 2 for this CTA's j-th unit
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
        int it = 0, j = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++j) {
            int mb, nb, sp;
            unit_coords(u, p, mb, nb, sp);
            const int kb0 = sp * p.kb_per_split;
            const int kb1 = min(p.n_kb, kb0 + p.kb_per_split);
            const int buf = j & 1;
            const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
            if (!mbar_wait(tempty_bar(buf), ((uint32_t)(j >> 1) & 1u) ^ 1u, abort_flag)) {
                *abort_flag = 1;
                raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                break;
            }
            tc_fence_after();
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
                if (!mbar_wait(full_bar(s), ph, abort_flag)) {
                    *abort_flag = 1;
                    raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sdesc_sw128(a_tile(s));
                const uint64_t bd = sdesc_sw128(b_tile(s));
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)
                    tc_mma_bf16(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                tc_commit(empty_bar(s));
            }
            tc_commit(tfull_bar(buf));
            *committed_slot = j + 1;
        }
    } else if (warp >= 2) {
        // ---------------- epilogue: warp w drains TMEM lanes 32*(w%4) .. +31 (one row per thread)
        const int quad = warp & 3;
        int j = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
            int mb, nb, sp;
            unit_coords(u, p, mb, nb, sp);
            const int buf = j & 1;
            // warp-uniform decision: tcgen05.ld below is a .sync.aligned warp instruction
            const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), (uint32_t)(j >> 1) & 1u, abort_flag));
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN);
            const int row = mb * BM + quad * 32 + lane;
            const bool row_ok = row < p.M;
            const long long split_off = (long long)sp * p.split_stride;
            if (!SWIGLU) {
                const int n0 = nb * BN;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float v[32];
                    tmem_ld32(tq + c, v);
                    const int col = n0 + c;
                    if (row_ok && col < p.n_valid)
                        store_row_chunk(p.mode, p.out, split_off + (long long)row * p.ldo + col, v,
                                        min(32, p.n_valid - col));
                }
            } else {
                const int j0 = nb * (BN / 2);
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    float g[32], uu[32];
                    tmem_ld32(tq + c, g);
                    tmem_ld32(tq + BN / 2 + c, uu);
                    const int col = j0 + c;
                    if (row_ok && col < p.n_valid) {
                        const int nv = min(32, p.n_valid - col);
                        if (p.mode == KM_PARTIAL) {
                            const long long base = split_off + (long long)row * p.ldo;
                            store_row_chunk(KM_PARTIAL, p.out, base + col, g, nv);
                            store_row_chunk(KM_PARTIAL, p.out, base + p.up_row0 + col, uu, nv);
                        } else {
#pragma unroll
                            for (int q = 0; q < 32; ++q) g[q] = silu_f(round_bf(g[q])) * round_bf(uu[q]);
                            store_row_chunk(KM_STORE, p.out, (long long)row * p.ldo + col, g, nv);
                        }
                    }
                }
            }
            // this warp is done reading accumulator `buf`: hand it back to the MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(buf));
        }
    }

    // ---------------- teardown
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == 0 && lane == 0) {
        // Let every TMA load and MMA this CTA issued land before its shared memory and TMEM go.
        volatile int never = 0;
        const int issued = *issued_slot;
        for (int i = max(0, issued - C::STAGES); i < issued; ++i)
            (void)mbar_wait(full_bar(i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u, &never);
        const int committed = *committed_slot;
        for (int jj = max(0, committed - 2); jj < committed; ++jj)
            (void)mbar_wait(tfull_bar(jj & 1), (uint32_t)(jj >> 1) & 1u, &never);
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Sum of split partials in split order, then the epilogue.  One thread per 8 output columns.
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, long long split_stride,
                                     int M, int n_out, int ldp, int up_off, int mode, void* out, int ldo) {
    const int groups = n_out >> 3;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)M * groups) return;
    const int row = (int)(idx / groups);
    const int col = (int)(idx % groups) * 8;
    float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float u[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int s = 0; s < splits; ++s) {
        const float* p = part + s * split_stride + (long long)row * ldp + col;
        const float4 x0 = *reinterpret_cast<const float4*>(p);
        const float4 x1 = *reinterpret_cast<const float4*>(p + 4);
        a[0] += x0.x; a[1] += x0.y; a[2] += x0.z; a[3] += x0.w;
        a[4] += x1.x; a[5] += x1.y; a[6] += x1.z; a[7] += x1.w;
        if (mode == KM_SWIGLU) {
            const float4 y0 = *reinterpret_cast<const float4*>(p + up_off);
            const float4 y1 = *reinterpret_cast<const float4*>(p + up_off + 4);
            u[0] += y0.x; u[1] += y0.y; u[2] += y0.z; u[3] += y0.w;
            u[4] += y1.x; u[5] += y1.y; u[6] += y1.z; u[7] += y1.w;
        }
    }
    const long long o = (long long)row * ldo + col;
    if (mode == KM_F32) {
        float4* q = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o);
        q[0] = make_float4(a[0], a[1], a[2], a[3]);
        q[1] = make_float4(a[4], a[5], a[6], a[7]);
        return;
    }
    uint4* q = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(out) + o);
    if (mode == KM_SWIGLU) {
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = silu_f(round_bf(a[j])) * round_bf(u[j]);
    } else if (mode == KM_RESIDUAL) {
        float r[8];
        unpack8(*q, r);
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = r[j] + a[j];
    }
    *q = pack8(a);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// Row-major bf16 matrix [rows, cols] viewed as a 2-D tensor (cols innermost), boxes of 64 x box_rows.
bool make_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
    int bn;
    int splits;
    int kbps;
    int mt, nt;
};

// Choose the tile width and K split.  The kernel is persistent (one CTA per SM walking work
// units), so the grid runs in ceil(units / SMs) rounds; per-unit time ~ (K blocks) x BN (bytes
// streamed and MMA work both scale with BN) plus a fixed tile overhead.  Splitting K is allowed
// for a single M tile only and costs a reduction pass.
Plan make_plan(int M, int N, int K, int epi, int split_req, int nsm) {
    const int n_kb = K / BK;
    const int mt = (M + BM - 1) / BM;
    const int dcols = epi == EPI_SWIGLU ? 2 * N : N;
    Plan best{256, 1, n_kb, mt, 0};
    double best_cost = 1e30;
    const int bns[2] = {256, 128};
    for (int bi = 0; bi < 2; ++bi) {
        const int bn = bns[bi];
        const int nt = (dcols + bn - 1) / bn;
        const int max_split = (mt == 1) ? std::min(8, n_kb) : 1;
        for (int s = 1; s <= max_split; ++s) {
            if (split_req > 0 && s != std::min(split_req, max_split)) continue;
            const int kbps = (n_kb + s - 1) / s;
            const int splits = (n_kb + kbps - 1) / kbps;
            const long long units = (long long)mt * nt * splits;
            const long long rounds = (units + nsm - 1) / nsm;
            double cost = (double)rounds * (kbps * (bn / 256.0) + 0.5);
            if (splits > 1) cost += 2.0;
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best = Plan{bn, splits, kbps, mt, nt};
            }
        }
    }
    return best;
}

template <int BN, bool SW>
cudaError_t launch_tile(const CUtensorMap& ma, const CUtensorMap& mb, const GemmArgs& g, const Plan& pl,
                        cudaStream_t st) {
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(gemm_bf16_tc_kernel<BN, SW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<BN>::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const long long units = (long long)pl.mt * pl.nt * pl.splits;
    const int nsm = device_sm_count();
    dim3 grid((unsigned)std::min<long long>(units, nsm));
    gemm_bf16_tc_kernel<BN, SW><<<grid, kThreads, Cfg<BN>::SMEM, st>>>(ma, mb, g);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

size_t linear_partial_bytes(int M, int N, int K, int epi, int split_req) {
    const Plan pl = make_plan(M, N, K, epi, split_req, device_sm_count());
    if (pl.splits <= 1) return 0;
    const size_t ldp = epi == EPI_SWIGLU ? 2 * (size_t)N : (size_t)N;
    return (size_t)pl.splits * (size_t)M * ldp * sizeof(float);
}

size_t linear_partial_bound(int m_max, int N, int K, int epi) {
    if (m_max > BM) m_max = BM;
    const size_t ldp = epi == EPI_SWIGLU ? 2 * (size_t)N : (size_t)N;
    return 8 * (size_t)m_max * ldp * sizeof(float);
}

cudaError_t launch_linear(const LinearCall& c, cudaStream_t st) {
    if (!get_encoder()) return cudaErrorNotSupported;
    const int nsm = device_sm_count();
    const Plan pl = make_plan(c.M, c.N, c.K, c.epi, c.split_req, nsm);
    const bool sw = c.epi == EPI_SWIGLU;
    const int w_rows = sw ? 2 * c.N : c.N;

    CUtensorMap ma, mb;
    if (!make_map(&ma, c.a, c.M, c.K, BM)) return cudaErrorInvalidValue;
    if (!make_map(&mb, c.w, w_rows, c.K, sw ? pl.bn / 2 : pl.bn)) return cudaErrorInvalidValue;

    GemmArgs g;
    g.err = c.err;
    g.M = c.M;
    g.n_valid = c.N;
    g.n_kb = c.K / BK;
    g.kb_per_split = pl.kbps;
    g.up_row0 = c.N;
    g.mt = pl.mt;
    g.nt = pl.nt;
    g.splits = pl.splits;
    g.group = 8;
    if (pl.splits > 1) {
        g.out = c.partial;
        g.mode = KM_PARTIAL;
        g.ldo = sw ? 2 * c.N : c.N;
        g.split_stride = (long long)c.M * g.ldo;
    } else {
        g.out = c.out;
        g.mode = c.epi == EPI_STORE ? KM_STORE : c.epi == EPI_RESIDUAL ? KM_RESIDUAL : c.epi == EPI_SWIGLU ? KM_SWIGLU : KM_F32;
        g.ldo = c.N;
        g.split_stride = 0;
    }

    cudaError_t e;
    if (pl.bn == 256)
        e = sw ? launch_tile<256, true>(ma, mb, g, pl, st) : launch_tile<256, false>(ma, mb, g, pl, st);
    else
        e = sw ? launch_tile<128, true>(ma, mb, g, pl, st) : launch_tile<128, false>(ma, mb, g, pl, st);
    if (c.splits_used) *c.splits_used = pl.splits;
    if (e != cudaSuccess || pl.splits <= 1 || c.partial_only) return e;

    const int mode = c.epi == EPI_STORE ? KM_STORE : c.epi == EPI_RESIDUAL ? KM_RESIDUAL : c.epi == EPI_SWIGLU ? KM_SWIGLU : KM_F32;
    const long long items = (long long)c.M * (c.N / 8);
    const int threads = 256;
    splitk_reduce_kernel<<<(unsigned)((items + threads - 1) / threads), threads, 0, st>>>(
        c.partial, pl.splits, (long long)c.M * g.ldo, c.M, c.N, g.ldo, c.N, mode, c.out, c.N);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace hra
