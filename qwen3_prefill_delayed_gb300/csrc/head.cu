// head.cu -- weight-streaming projections over at most 128 activation rows: the audio head of the
// delayed-codebook step, and every projection of a backbone pass over at most 64 token rows (the
// decode pass; launch_linear_small_head in gemm_tc.cu adds the split reduction and its epilogue).
//
// Source: "Stabilize Higgs Audio termination and prefill" (FlashRT PR #141), Summary (per-frame
// argmax over the audio head's codebook logits) and Performance (the AR decode time per frame); the
// argmax, delay state machine and embedding sum that follow the audio head run in codebook.cu.
//
// logits[b][n] = sum_k hidden[b][k] * head_w[n][k] for the n = K * Vc head rows.  With at most 128
// activation rows this is a stream of the 42 MB head through the tensor cores, and the tensor core
// is fed so that each instruction does as much of that stream as it can: one tcgen05.mma of
// kind::f16 (K = 16) costs about the same issue time for N = 16 as for N = 256, so the weight rows
// are the N = 256 side and the activation rows the M = 128 side (rows past the batch only feed
// accumulator rows that are never read).  A
// CTA owns one 256-row tile of the head over one of `splits` K ranges; the fp32 partial of each
// range goes to its own plane partial[split][b][n], and the finalize sums the planes in split
// order (so the result does not depend on which CTA finishes first).  The weight tiles of the
// first ring stages are requested before the kernel waits for the kernels ahead of it in the
// stream: the head is constant, so one step's weight stream starts while the previous step ends.
//
// Roles (192 threads): warp 0 TMA producer (128-byte swizzled boxes: activations 64 K x B rows,
// weights 64 K x 256 rows, 4 ring stages), warp 1 TMEM allocation + MMA issue (one lane), warps 2-5 epilogue
// (tcgen05.ld of their 32-lane quarter: one activation row per thread, 256 fp32 columns).
#include <algorithm>

#include "internal.h"

namespace hra {

namespace {

constexpr int kHeadThreads = 192;
constexpr int kHeadBN = 256;        // weight rows per tile (MMA N)

// Ring stage = activation tile (128 rows, NBX of them loaded) + weight tile.
template <int NBX>
struct HeadCfg {
    static constexpr int A_BYTES = 128 * 64 * 2;       // activation tile
    static constexpr int B_BYTES = kHeadBN * 64 * 2;   // weight tile
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = 4;
    static constexpr int SMEM = STAGES * STAGE + 1024 /*align*/ + 256 /*barriers*/;
    static constexpr uint32_t TMEM_COLS = kHeadBN;
    static_assert(128 * (kHeadBN + 4) * 4 <= STAGES * STAGE, "the staging tile must fit in the ring");
    static_assert(A_BYTES % 1024 == 0 && STAGE % 1024 == 0, "tiles stay 1024-byte aligned (128-byte swizzle)");
};

struct HeadArgs {
    int N;                    // head rows (K * Vc)
    int B;                    // activation rows
    int n_kb;                 // H / 64
    int nt, splits, kbps;     // tiles of 256 rows, K splits, k-blocks per split
    float* partial;           // [splits][B][N]
    long long split_stride;   // B * N
    unsigned int* err;
    unsigned int* zero_ptr;   // CTA 0 clears zero_words words here once earlier kernels are done
    int zero_words;
    int l2_prefetch;          // send the CTA's later weight tiles towards L2 before waiting
};

// OR of `v` over the four epilogue warps (named barrier 1, 128 threads); all of them get the answer.
__device__ __forceinline__ bool epilogue_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, 1, 128, pi;\n"
        " selp.u32 %0, 1, 0, po;\n}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

template <int NBX>
__global__ void __launch_bounds__(kHeadThreads, 1)
    audio_head_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const HeadArgs p) {
    using C = HeadCfg<NBX>;
    constexpr int S = C::STAGES;
    pdl_launch();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued_slot = reinterpret_cast<int*>(tmem_slot + 2);
    int* committed_slot = reinterpret_cast<int*>(tmem_slot + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x % p.nt, split = blockIdx.x / p.nt;
    const int kb0 = split * p.kbps, kb1 = min(p.n_kb, kb0 + p.kbps);
    const int nkb = kb1 - kb0;
    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + S + s); };
    const uint32_t tfull = smem_u32(bars + 2 * S);
    auto a_tile = [&](int s) { return smem_u32(smem + s * C::STAGE); };
    auto b_tile = [&](int s) { return smem_u32(smem + s * C::STAGE + C::A_BYTES); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull, 1);
        *abort_flag = 0;
        *issued_slot = 0;
        *committed_slot = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmW);
        tma_prefetch_map(&tmX);
    }
    // Activation rows [NBX, 128) of the A tiles are never loaded: they only feed accumulator rows
    // (TMEM lanes) that are never read, so they are left as they are.
    __syncthreads();
    constexpr int stage_tx = NBX * 128 + C::B_BYTES;

    if (warp == 0) {
        if (lane == 0) {
            // weight tiles of the first stages before waiting for the kernels ahead in the stream
            const int pre = min(S, nkb);
            for (int i = 0; i < pre; ++i) {
                mbar_expect_tx(full_bar(i), stage_tx);
                tma_load_2d(b_tile(i), &tmW, full_bar(i), (kb0 + i) * 64, tile * kHeadBN);
            }
            // and the rest of this CTA's weight tiles towards L2, so the whole head is in flight
            // while the kernels ahead finish
            if (p.l2_prefetch)
                for (int i = pre; i < nkb; ++i) tma_prefetch_l2_2d(&tmW, (kb0 + i) * 64, tile * kHeadBN);
            pdl_wait();
            int s = 0, i = 0;
            uint32_t ph = 0;
            for (; i < nkb; ++i) {
                const int kx = (kb0 + i) * 64;
                if (i >= pre) {
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                    mbar_expect_tx(full_bar(s), stage_tx);
                    tma_load_2d(b_tile(s), &tmW, full_bar(s), kx, tile * kHeadBN);
                }
                tma_load_2d(a_tile(s), &tmX, full_bar(s), kx, 0);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            *issued_slot = max(i, pre);
        }
    } else if (warp == 1) {
        // TMEM is taken only once the kernels ahead have finished, so that a kernel ahead that still
        // has to allocate its own columns on this SM is never kept waiting by this one.
        pdl_wait();
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
        asm volatile("bar.sync 2, 160;" ::: "memory");
        tc_fence_after();
        const uint32_t tmem = *tmem_slot;
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, kHeadBN);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
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
                for (int k = 0; k < 4; ++k)
                    tc_mma_bf16(tmem, ad + 2ull * k, bd + 2ull * k, idesc, (i > 0 || k > 0) ? 1u : 0u);
                tc_commit(empty_bar(s));
                if (++s == S) {
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
        pdl_wait();
        if (blockIdx.x == 0 && warp == 2)
            for (int i = lane; i < p.zero_words; i += 32) p.zero_ptr[i] = 0u;
        asm volatile("bar.sync 2, 160;" ::: "memory");
        // the four epilogue warps agree on the outcome, since they meet at a named barrier below
        const bool ok = !epilogue_any(!__all_sync(0xffffffffu, mbar_wait(tfull, 0u, abort_flag)));
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
        } else {
            // TMEM lane b = activation row b: each thread moves its row's 256 sums into a staging
            // tile (rows padded to 260 floats against bank conflicts; the ring is free by now),
            // then every warp writes whole rows with coalesced 16-byte stores.
            tc_fence_after();
            float* stage = reinterpret_cast<float*>(smem);
            constexpr int kLd = kHeadBN + 4;
            const int quad = warp & 3;
            if (quad * 32 < p.B) {
                const uint32_t tq = *tmem_slot + ((uint32_t)(quad * 32) << 16);
                const int b = quad * 32 + lane;
#pragma unroll 1
                for (int c = 0; c < kHeadBN; c += 32) {
                    float v[32];
                    tmem_ld32(tq + (uint32_t)c, v);
                    if (b < p.B) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            *reinterpret_cast<float4*>(stage + b * kLd + c + 4 * i) =
                                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    }
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const int ncol = min(kHeadBN, p.N - tile * kHeadBN);
            for (int b = warp - 2; b < p.B; b += 4) {
                float* out = p.partial + (long long)split * p.split_stride + (long long)b * p.N + tile * kHeadBN;
#pragma unroll
                for (int h = 0; h < kHeadBN / 128; ++h) {
                    const int col = 128 * h + 4 * lane;
                    if (col < ncol)
                        *reinterpret_cast<float4*>(out + col) = *reinterpret_cast<const float4*>(stage + b * kLd + col);
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
        for (int i = max(0, issued - S); i < issued; ++i)
            (void)mbar_wait(full_bar(i % S), (uint32_t)(i / S) & 1u, &never);
        if (*committed_slot) (void)mbar_wait(tfull, 0u, &never);
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(*tmem_slot, C::TMEM_COLS);
    }
}

template <int NBX>
cudaError_t launch_head_nb(const CUtensorMap& mw, const CUtensorMap& mx, const HeadArgs& p, int grid,
                           cudaStream_t st) {
    using C = HeadCfg<NBX>;
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(audio_head_kernel<NBX>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    HRA_LAUNCH(audio_head_kernel<NBX>, dim3(grid), dim3(kHeadThreads), C::SMEM, st, mw, mx, p);
    return cudaGetLastError();
}

}  // namespace

HeadPlan head_plan(int N, int H, int max_splits, int split_req) {
    HeadPlan pl;
    const int nsm = device_sm_count();
    const int n_kb = H / 64;
    pl.nt = (N + kHeadBN - 1) / kHeadBN;
    int s = split_req > 0 ? std::min(split_req, n_kb) : std::max(1, std::min({nsm / pl.nt, n_kb, max_splits}));
    pl.kbps = (n_kb + s - 1) / s;
    pl.splits = (n_kb + pl.kbps - 1) / pl.kbps;
    return pl;
}

cudaError_t launch_audio_head(const HeadCall& c, cudaStream_t st) {
    if (c.B < 1 || c.B > kHeadMaxBatch) return cudaErrorInvalidValue;
    const HeadPlan pl = head_plan(c.N, c.H, c.max_splits > 0 ? c.max_splits : kHeadMaxSplits, c.split_req);
    const int nbx = c.B <= 16 ? 16 : c.B <= 32 ? 32 : c.B <= 64 ? 64 : 128;
    CUtensorMap mw, mx;
    if (!make_map_2d(&mw, c.head_w, c.N, c.H, kHeadBN)) return cudaErrorInvalidValue;
    if (!make_map_2d(&mx, c.hidden, c.B, c.H, nbx)) return cudaErrorInvalidValue;
    HeadArgs p{};
    p.N = c.N;
    p.B = c.B;
    p.n_kb = c.H / 64;
    p.nt = pl.nt;
    p.splits = pl.splits;
    p.kbps = pl.kbps;
    p.partial = c.partial;
    p.split_stride = (long long)c.B * c.N;
    p.err = c.err;
    p.zero_ptr = c.zero_ptr;
    p.zero_words = c.zero_ptr ? c.zero_words : 0;
    p.l2_prefetch = c.no_l2_prefetch ? 0 : 1;
    if (c.splits_used) *c.splits_used = pl.splits;
    const int grid = pl.nt * pl.splits;
    if (nbx == 16) return launch_head_nb<16>(mw, mx, p, grid, st);
    if (nbx == 32) return launch_head_nb<32>(mw, mx, p, grid, st);
    if (nbx == 64) return launch_head_nb<64>(mw, mx, p, grid, st);
    return launch_head_nb<128>(mw, mx, p, grid, st);
}

}  // namespace hra
