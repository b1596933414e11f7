// gemm_tc.cu -- BF16 projection GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Computes D[m, n] = sum_k A[m, k] * W[n, k] for A = activations [M, K] and W = weight rows
// [N, K] (both K-major, bf16), fp32 accumulation in tensor memory, with the epilogue fused:
// plain bf16 store, in-place residual add (r = bf16(r + acc)), SwiGLU over the gate and up rows
// of a merged [2F, K] weight (h = bf16(silu(bf16(g)) * bf16(u))), or fp32 store.  These are the
// projection GEMMs of the batched prefill ("Stabilize Higgs Audio termination and prefill",
// Summary: the projection GEMMs; merged QKV and merged gate/up as in the "flashrt-structures 0.2.0,
// prefill_tower/fp8_chain.py" page, its per-layer chain) and the
// audio-head projection.
//
// Persistent kernel, one CTA per SM walking 128 x BN output tiles (M = 128 rows of A per
// tcgen05.mma, N = BN weight rows), or -- from 512 rows, the default -- 2-CTA clusters walking
// 256 x 256 tiles with one cta_group::2 MMA of M = 256 per K step (each CTA stages its 128 rows of
// A and half of the weight rows):
//   warp 0     TMA producer: streams 128x64 A boxes and W boxes (128-byte swizzle) into a
//              STAGES-deep shared-memory ring, one mbarrier pair per stage;
//   warp 1     allocates two accumulators of BN TMEM columns; one elected lane issues 4
//              tcgen05.mma (K = 16 each) per 64-wide K block and commits each stage back to the
//              producer (for a pair: rank 0 only, committing to both CTAs);
//   warps 2-9  epilogue: tcgen05.ld of their 32-lane TMEM quadrant (one output row per thread),
//              fused epilogue math, 32-byte (else 16-byte) vector stores, while the MMA fills the
//              other accumulator.
// A last round of tiles that would leave most SMs idle runs as K pieces summed by a fix-up kernel.
// Calls of at most 64 rows take the head-form kernel of head.cu through launch_linear_small_head.
#include <algorithm>
#include <cudaTypedefs.h>
#include <mutex>
#include <unordered_map>

#include "internal.h"

namespace hra {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kMaxTailPieces = 4;   // K pieces of a last-round tile
constexpr int kTileThreads = 320;   // tile kernel: TMA warp, MMA warp, 8 epilogue warps

enum KMode : int { KM_STORE = 0, KM_RESIDUAL = 1, KM_SWIGLU = 2, KM_F32 = 3, KM_PARTIAL = 4, KM_QKROPE = 5 };

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
    // last-round split: tiles [head_units, mt*nt) run as tail_splits K pieces each, written as fp32
    // tile partials [piece][tile - head_units][BM][BN] to tail_part (0 tail tiles = off)
    int head_units, tail_tiles, tail_splits, kb_per_tail;
    float* tail_part;
    unsigned int* zero_ptr;   // CTA 0 clears zero_words words here once earlier kernels are done
    int zero_words;
    int v8;                   // outputs 32-byte aligned (rows and base): epilogues move 32 bytes an instruction
    QkRopeArgs qk;            // KM_QKROPE: per-head q/k norm + RoPE + K/V cache write in the epilogue
    // FP8 operands: the accumulators are multiplied by (*a_scale) * (*w_scale) (device scalars)
    const float* a_scale;
    const float* w_scale;
};

// PAIR: two CTAs (a 2-CTA cluster) share each 256 x BN tile through one M = 256 MMA; each CTA
// stages its 128 rows of A and half of the BN weight rows, so a stage is 32 KB instead of 48 KB and
// the same shared memory holds six stages (1.6x the loads in flight per byte consumed).
template <int BN, bool PAIR = false>
struct Cfg {
    static constexpr int STAGES = PAIR ? 6 : (BN >= 256 ? 4 : 6);
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;   // this CTA's weight rows
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
    // two fp32 accumulators of BN columns each: the epilogue drains one while the MMA fills the other
    static constexpr uint32_t TMEM_COLS = 2 * BN;
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// Store 32 fp32 values of one output row starting at column `col`; `nv` columns are valid
// (multiple of 8 for bf16, of 4 for fp32).  v8: the chunk is 32-byte aligned (whole chunks move in
// 32-byte accesses).
__device__ __forceinline__ void store_row_chunk(int mode, void* out, long long off, const float (&v)[32],
                                                int nv, bool v8) {
    if (v8 && nv == 32) {
        if (mode == KM_F32 || mode == KM_PARTIAL) {
            float* p = reinterpret_cast<float*>(out) + off;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                st_global_32(p + 8 * i, f4_as_u4(v[8 * i], v[8 * i + 1], v[8 * i + 2], v[8 * i + 3]),
                             f4_as_u4(v[8 * i + 4], v[8 * i + 5], v[8 * i + 6], v[8 * i + 7]));
            return;
        }
        bf16* p = reinterpret_cast<bf16*>(out) + off;
        uint4 r[4];
        if (mode == KM_RESIDUAL) {
            ld_global_32(p, r[0], r[1]);
            ld_global_32(p + 16, r[2], r[3]);
        }
        uint4 o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = v[8 * i + j];
            if (mode == KM_RESIDUAL) {
                float rr[8];
                unpack8(r[i], rr);
#pragma unroll
                for (int j = 0; j < 8; ++j) f[j] = rr[j] + f[j];
            }
            o[i] = pack8(f);
        }
        st_global_32(p, o[0], o[1]);
        st_global_32(p + 16, o[2], o[3]);
        return;
    }
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

// KM_QKROPE epilogue: the tile's columns [n0, n0 + BN) are whole heads of the merged QKV row
// (BN a multiple of HD).  Per head: round the fp32 accumulators to bf16 (the QKV output rounding),
// then V heads go to the cache as is; q / k heads get RMSNorm over HD (compensated sum of squares,
// shared gains) and rotate-half RoPE at the row's position, rounded once, to q_out or the K cache.
// One row (token) per thread; the RoPE partner i + HD/2 is in the same thread.
template <int BN, int HD>
__device__ __forceinline__ void qk_rope_epilogue_hd(uint32_t tq, int n0, int half, int row, bool row_ok,
                                                    const QkRopeArgs& a, bool v8) {
    constexpr int HALF = HD / 2;
    const int seq = row_ok ? a.row_seq[row] : 0;
    const int pos = row_ok ? a.row_pos[row] : 0;
    const float2* cs = a.rope + (a.rope_row_is_pos ? pos : row);   // pair i at cs[i * rope_rows]
    const long long head_stride = (long long)a.n_slots * HD;
    // Two passes over each head's TMEM columns keep at most 64 values in registers: the first
    // writes V heads and takes the sum of squares of q / k heads, the second applies the norm and
    // RoPE to the pairs (c, c + HD/2).  tcgen05.ld is a warp instruction: every lane issues it.
#pragma unroll 1
    for (int h0 = half * HD; h0 < BN; h0 += 2 * HD) {   // this warp's heads: every other one of the tile
        const int hh = (n0 + h0) / HD;   // head index in the merged row (uniform over the warp)
        if (hh >= a.nq + 2 * a.nkv) break;
        const bool is_v = hh >= a.nq + a.nkv;
        bf16* vdst = a.kv_layer + ((long long)(seq * 2 + 1) * a.nkv + (hh - a.nq - a.nkv)) * head_stride +
                     (long long)pos * HD;
        // four interleaved compensated sums (short dependency chains), combined compensated
        float s4[4] = {0.f, 0.f, 0.f, 0.f}, c4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < HD; c += 32) {
            float v[32];
            tmem_ld32(tq + h0 + c, v);
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = round_bf(v[q]);
            if (is_v) {
                if (row_ok) {
                    if (v8) {
#pragma unroll
                        for (int e = 0; e < 32; e += 16) st_global_32(vdst + c + e, pack8(v + e), pack8(v + e + 8));
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; e += 8) *reinterpret_cast<uint4*>(vdst + c + e) = pack8(v + e);
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < 32; ++q) csum_add(s4[q & 3], c4[q & 3], __fmul_rn(v[q], v[q]));
            }
        }
        if (is_v) continue;
        float ss = s4[0], sc = c4[0];
#pragma unroll
        for (int q = 1; q < 4; ++q) {
            float t, er;
            two_sum(ss, s4[q], t, er);
            ss = t;
            sc = __fadd_rn(__fadd_rn(sc, c4[q]), er);
        }
        ss = __fadd_rn(ss, sc);
        const float inv = 1.0f / sqrtf(ss / (float)HD + a.eps);
        const bool is_q = hh < a.nq;
        const bf16* gain = is_q ? a.q_norm : a.k_norm;
        bf16* dst = is_q ? a.q_out + ((long long)row * a.nq + hh) * HD
                         : a.kv_layer + ((long long)(seq * 2) * a.nkv + (hh - a.nq)) * head_stride + (long long)pos * HD;
#pragma unroll
        for (int c = 0; c < HALF; c += 32) {
            float xl[32], xh[32];
            tmem_ld32(tq + h0 + c, xl);
            tmem_ld32(tq + h0 + HALF + c, xh);
            if (!row_ok) continue;
#pragma unroll
            for (int e16 = 0; e16 < 32; e16 += 16) {
                float lo[16], hi[16];
#pragma unroll
                for (int e8 = 0; e8 < 16; e8 += 8) {
                    float g_lo[8], g_hi[8];
                    unpack8(*reinterpret_cast<const uint4*>(gain + c + e16 + e8), g_lo);
                    unpack8(*reinterpret_cast<const uint4*>(gain + HALF + c + e16 + e8), g_hi);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int k = e16 + e8 + e;
                        const float xa = __fmul_rn(__fmul_rn(round_bf(xl[k]), inv), g_lo[e]);
                        const float xb = __fmul_rn(__fmul_rn(round_bf(xh[k]), inv), g_hi[e]);
                        const float2 t = cs[(long long)(c + k) * a.rope_rows];   // (cos, sin)
                        lo[e8 + e] = __fsub_rn(__fmul_rn(xa, t.x), __fmul_rn(xb, t.y));
                        hi[e8 + e] = __fadd_rn(__fmul_rn(xb, t.x), __fmul_rn(xa, t.y));
                    }
                }
                if (v8) {
                    st_global_32(dst + c + e16, pack8(lo), pack8(lo + 8));
                    st_global_32(dst + HALF + c + e16, pack8(hi), pack8(hi + 8));
                } else {
                    *reinterpret_cast<uint4*>(dst + c + e16) = pack8(lo);
                    *reinterpret_cast<uint4*>(dst + c + e16 + 8) = pack8(lo + 8);
                    *reinterpret_cast<uint4*>(dst + HALF + c + e16) = pack8(hi);
                    *reinterpret_cast<uint4*>(dst + HALF + c + e16 + 8) = pack8(hi + 8);
                }
            }
        }
    }
}

template <int BN>
__device__ __forceinline__ void qk_rope_epilogue(uint32_t tq, int n0, int half, int row, bool row_ok,
                                                 const QkRopeArgs& a, bool v8) {
    if (a.hd == 128) qk_rope_epilogue_hd<BN, 128>(tq, n0, half, row, row_ok, a, v8);
    else qk_rope_epilogue_hd<BN, 64>(tq, n0, half, row, row_ok, a, v8);
}

// Linear tile index of (mb, nb) in the raster order of unit_coords.
__device__ __forceinline__ int tile_linear(int mb, int nb, const GemmArgs& p) {
    const int band = nb / p.group;
    return band * p.group * p.mt + (nb - band * p.group) * p.mt + mb;
}
__device__ __forceinline__ int tail_index(int mb, int nb, const GemmArgs& p) {
    return tile_linear(mb, nb, p) - p.head_units;
}

// Work unit u -> tile, K-block range and (for last-round pieces) the piece index (-1 otherwise).
__device__ __forceinline__ void unit_work(int u, const GemmArgs& p, int& mb, int& nb, int& kb0, int& kb1,
                                          int& piece) {
    if (p.tail_tiles > 0 && u >= p.head_units) {
        const int v = u - p.head_units;
        piece = v / p.tail_tiles;
        int sp;
        unit_coords(p.head_units + (v - piece * p.tail_tiles), p, mb, nb, sp);
        kb0 = piece * p.kb_per_tail;
        kb1 = min(p.n_kb, kb0 + p.kb_per_tail);
        return;
    }
    int sp;
    unit_coords(u, p, mb, nb, sp);
    piece = -1;
    kb0 = sp * p.kb_per_split;
    kb1 = min(p.n_kb, kb0 + p.kb_per_split);
}

// Persistent: each CTA walks work units blockIdx.x, blockIdx.x + gridDim.x, ...
// F8: both operands E4M3 (kind::f8f6f4): a 128-byte stage row holds 128 elements instead of 64,
// and every accumulator is scaled by the two per-tensor scales before any store.
// PAIR: the grid is 2-CTA clusters and cluster c walks units c, c + gridDim.x / 2, ...; a unit is
// a 256 x BN tile, CTA rank r owns its rows [128 r, 128 r + 128).  Both CTAs load their A rows and
// their half of the weight rows (SwiGLU: rank 0 the gate rows, rank 1 the up rows), and both
// loads complete on rank 0's stage barrier; rank 0 issues the M = 256 MMAs and commits each stage
// and each accumulator to both CTAs' barriers; each CTA's epilogue drains its own tensor memory
// and arrives on rank 0's accumulator-free barrier.
template <int BN, bool SWIGLU, bool F8, bool PAIR>
__global__ void __launch_bounds__(kTileThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs p) {
    static_assert(!PAIR || BN == 256, "CTA pairs: 256-wide tiles");
    using C = Cfg<BN, PAIR>;
    constexpr int KE = F8 ? 2 * BK : BK;   // elements per K block (one 128-byte row)
    constexpr int BMU = PAIR ? 2 * BM : BM;   // rows of a work unit's tile
    pdl_launch();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    // bars: full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* issued_slot = reinterpret_cast<int*>(tmem_slot + 2);
    int* committed_slot = reinterpret_cast<int*>(tmem_slot + 3);
    int* peer_slot = reinterpret_cast<int*>(tmem_slot + 4);   // PAIR, rank 0: rank 1's issued count, abort flag

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = p.tail_tiles > 0 ? p.head_units + p.tail_tiles * p.tail_splits : p.mt * p.nt * p.splits;
    const uint32_t rank = PAIR ? cta_rank_in_cluster() : 0u;
    const int walker = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;   // this CTA's (pair's) first unit
    const int walkers = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

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
            mbar_init(tempty_bar(b), PAIR ? 16 : 8);   // one arrival per epilogue warp (of both CTAs)
        }
        *abort_flag = 0;
        *issued_slot = 0;
        *committed_slot = 0;
        peer_slot[0] = 0;
        peer_slot[1] = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    // PAIR: the peer's barriers are initialised before any load or commit can reach them
    if constexpr (PAIR) cluster_barrier_sync();
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: one continuous stage ring across all of this CTA's units
        // PAIR: this CTA's boxes complete on rank 0's barrier, which rank 0 arms for both CTAs' bytes
        auto load = [&](uint32_t dst, const CUtensorMap* map, int s, int x, int y) {
            if constexpr (PAIR) tma_load_2d_pair(dst, map, smem_in_cta(full_bar(s), 0), x, y);
            else tma_load_2d(dst, map, full_bar(s), x, y);
        };
        constexpr uint32_t kStageTx = PAIR ? 2 * C::STAGE_BYTES : C::STAGE_BYTES;
        const bool arms = !PAIR || rank == 0;
        auto load_w = [&](int s, int kx, int nb) {
            if (SWIGLU) {
                const int j0 = nb * (BN / 2);
                if constexpr (PAIR) {
                    load(b_tile(s), &tmB, s, kx, rank == 0 ? j0 : p.up_row0 + j0);
                } else {
                    load(b_tile(s), &tmB, s, kx, j0);
                    load(b_tile(s) + C::B_BYTES / 2, &tmB, s, kx, p.up_row0 + j0);
                }
            } else {
                load(b_tile(s), &tmB, s, kx, nb * BN + (int)rank * (BN / 2));
            }
        };
        // Weight tiles of the first ring stages do not depend on earlier kernels: fetch them before
        // waiting for those kernels (the activation half of each stage follows after the wait).
        int pre = 0;
        for (int u = walker; u < units && pre < C::STAGES; u += walkers) {
            int mb, nb, kb0, kb1, piece;
            unit_work(u, p, mb, nb, kb0, kb1, piece);
            for (int kb = kb0; kb < kb1 && pre < C::STAGES; ++kb, ++pre) {
                if (arms) mbar_expect_tx(full_bar(pre), kStageTx);
                load_w(pre, kb * KE, nb);
            }
        }
        pdl_wait();
        int it = 0;
        bool ok = true;
        for (int u = walker; u < units && ok; u += walkers) {
            int mb, nb, kb0, kb1, piece;
            unit_work(u, p, mb, nb, kb0, kb1, piece);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % C::STAGES;
                const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
                const int kx = kb * KE;
                if (it >= pre) {
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) {
                        *abort_flag = 1;
                        raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                        ok = false;
                        break;
                    }
                    if (arms) mbar_expect_tx(full_bar(s), kStageTx);
                    load_w(s, kx, nb);
                }
                load(a_tile(s), &tmA, s, kx, mb * BMU + (int)rank * BM);
            }
        }
        *issued_slot = ok ? it : max(it, pre);
    } else if (warp == 1 && lane == 0 && (!PAIR || rank == 0)) {
        // ---------------- MMA issuer: accumulator buffer j % 2 for this CTA's j-th unit
        constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(BMU, BN) : idesc_bf16_f32(BMU, BN);
        int it = 0, j = 0;
        bool ok = true;
        for (int u = walker; u < units && ok; u += walkers, ++j) {
            int mb, nb, kb0, kb1, piece;
            unit_work(u, p, mb, nb, kb0, kb1, piece);
            const int buf = j & 1;
            const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
            const uint32_t tpar = ((uint32_t)(j >> 1) & 1u) ^ 1u;
            if (!(PAIR ? mbar_wait_cluster(tempty_bar(buf), tpar, abort_flag) : mbar_wait(tempty_bar(buf), tpar, abort_flag))) {
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
                for (int k = 0; k < 4; ++k) {   // 4 x 32 bytes of each 128-byte row
                    if constexpr (F8 && PAIR)
                        tc_mma_f8_pair(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    else if constexpr (F8)
                        tc_mma_f8(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    else if constexpr (PAIR)
                        tc_mma_bf16_pair(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    else
                        tc_mma_bf16(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                }
                if constexpr (PAIR) tc_commit_pair(empty_bar(s), 0x3);
                else tc_commit(empty_bar(s));
            }
            if constexpr (PAIR) tc_commit_pair(tfull_bar(buf), 0x3);
            else tc_commit(tfull_bar(buf));
            *committed_slot = j + 1;
        }
    } else if (warp >= 2) {
        // ---------------- epilogue: warp w drains TMEM lanes 32*(w%4) .. +31 (one row per thread);
        // warps 2-5 take the first half of the tile's columns (QKV: its even heads), warps 6-9 the
        // second half (odd heads)
        pdl_wait();
        if (blockIdx.x == 0 && warp == 2)
            for (int i = lane; i < p.zero_words; i += 32) p.zero_ptr[i] = 0u;
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        constexpr int HC = BN / 2;   // columns of a half (SwiGLU: gate + up columns of a half: HC / 2 each)
        float scale = 1.f;
        if constexpr (F8) scale = (*p.a_scale) * (*p.w_scale);
        auto scaled = [&](float (&v)[32]) {
            if constexpr (F8) {
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] *= scale;
            }
        };
        int j = 0;
        for (int u = walker; u < units; u += walkers, ++j) {
            int mb, nb, kb0, kb1, piece;
            unit_work(u, p, mb, nb, kb0, kb1, piece);
            const int sp = piece < 0 ? u / (p.mt * p.nt) : 0;
            const int buf = j & 1;
            const int trow = (int)rank * BM + quad * 32 + lane;   // row within the unit's tile
            const int row = mb * BMU + trow;
            const bool row_ok = row < p.M;
            // While the MMAs of this unit run, pull the residual row segment its epilogue reads into L2.
            if (!SWIGLU && piece < 0 && p.mode == KM_RESIDUAL && row_ok) {
                const int n0 = nb * BN + half * HC;
                for (int c = 0; c < HC && n0 + c < p.n_valid; c += 64)
                    prefetch_l2(reinterpret_cast<const bf16*>(p.out) + (long long)row * p.ldo + n0 + c);
            }
            // warp-uniform decision: tcgen05.ld below is a .sync.aligned warp instruction
            const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), (uint32_t)(j >> 1) & 1u, abort_flag));
            if (!ok) {
                *abort_flag = 1;
                raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                break;
            }
            tc_fence_after();
            const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * BN);
            const long long split_off = (long long)sp * p.split_stride;
            if (piece >= 0) {
                // last-round K piece: raw fp32 tile [BM][BN] for the fix-up pass
                float* dst = p.tail_part +
                             ((long long)piece * p.tail_tiles + tail_index(mb, nb, p)) * (BMU * BN) +
                             (long long)trow * BN;
#pragma unroll 1
                for (int c = half * HC; c < half * HC + HC; c += 32) {
                    float v[32];
                    tmem_ld32(tq + c, v);
                    scaled(v);
#pragma unroll
                    for (int q = 0; q < 4; ++q)   // tail planes are 256-byte aligned, rows BN floats
                        st_global_32(dst + c + 8 * q, f4_as_u4(v[8 * q], v[8 * q + 1], v[8 * q + 2], v[8 * q + 3]),
                                     f4_as_u4(v[8 * q + 4], v[8 * q + 5], v[8 * q + 6], v[8 * q + 7]));
                }
            } else if (!SWIGLU && !F8 && p.mode == KM_QKROPE) {
                qk_rope_epilogue<BN>(tq, nb * BN, half, row, row_ok, p.qk, p.v8 != 0);
            } else if (!SWIGLU && p.mode == KM_RESIDUAL) {
                // out += acc: the chunk's residual loads are issued before its TMEM read
                const int n0 = nb * BN;
#pragma unroll 1
                for (int c = half * HC; c < half * HC + HC; c += 32) {
                    const int col = n0 + c;
                    const int nv = row_ok ? max(0, min(32, p.n_valid - col)) : 0;
                    uint4* o4 = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(p.out) + (long long)row * p.ldo + col);
                    const bool wide = p.v8 != 0 && nv == 32;
                    uint4 r4[4];
                    if (wide) {
                        ld_global_32(o4, r4[0], r4[1]);
                        ld_global_32(o4 + 2, r4[2], r4[3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) r4[i] = 8 * i < nv ? o4[i] : make_uint4(0u, 0u, 0u, 0u);
                    }
                    float v[32];
                    tmem_ld32(tq + c, v);
                    scaled(v);
                    uint4 w4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float r[8];
                        unpack8(r4[i], r);
#pragma unroll
                        for (int e = 0; e < 8; ++e) r[e] = r[e] + v[8 * i + e];
                        w4[i] = pack8(r);
                    }
                    if (wide) {
                        st_global_32(o4, w4[0], w4[1]);
                        st_global_32(o4 + 2, w4[2], w4[3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (8 * i < nv) o4[i] = w4[i];
                    }
                }
            } else if (!SWIGLU) {
                const int n0 = nb * BN;
#pragma unroll 1
                for (int c = half * HC; c < half * HC + HC; c += 32) {
                    float v[32];
                    tmem_ld32(tq + c, v);
                    scaled(v);
                    const int col = n0 + c;
                    if (row_ok && col < p.n_valid)
                        store_row_chunk(p.mode, p.out, split_off + (long long)row * p.ldo + col, v,
                                        min(32, p.n_valid - col), p.v8 != 0);
                }
            } else {
                // gate columns [0, BN/2), up columns [BN/2, BN): this half takes output columns
                // [half * BN/4, half * BN/4 + BN/4) of the tile's BN/2
                const int j0 = nb * (BN / 2);
#pragma unroll 1
                for (int c = half * (HC / 2); c < half * (HC / 2) + HC / 2; c += 32) {
                    float g[32], uu[32];
                    tmem_ld32(tq + c, g);
                    tmem_ld32(tq + BN / 2 + c, uu);
                    scaled(g);
                    scaled(uu);
                    const int col = j0 + c;
                    if (row_ok && col < p.n_valid) {
                        const int nv = min(32, p.n_valid - col);
                        if (p.mode == KM_PARTIAL) {
                            const long long base = split_off + (long long)row * p.ldo;
                            store_row_chunk(KM_PARTIAL, p.out, base + col, g, nv, p.v8 != 0);
                            store_row_chunk(KM_PARTIAL, p.out, base + p.up_row0 + col, uu, nv, p.v8 != 0);
                        } else {
#pragma unroll
                            for (int q = 0; q < 32; ++q) g[q] = silu_f(round_bf(g[q])) * round_bf(uu[q]);
                            store_row_chunk(KM_STORE, p.out, (long long)row * p.ldo + col, g, nv, p.v8 != 0);
                        }
                    }
                }
            }
            // this warp is done reading accumulator `buf`: hand it back to the MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_remote(smem_in_cta(tempty_bar(buf), 0));
                else mbar_arrive(tempty_bar(buf));
            }
        }
    }

    // ---------------- teardown
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) {
        // Rank 1's loads complete on rank 0's barriers, so rank 0 does the waiting for both: rank 1
        // reports how far its loads went and whether it gave up a wait.
        if (rank == 1 && threadIdx.x == 0) {
            st_shared_cluster(smem_in_cta(smem_u32(peer_slot), 0), (uint32_t)*issued_slot);
            st_shared_cluster(smem_in_cta(smem_u32(peer_slot + 1), 0), (uint32_t)*abort_flag);
        }
        cluster_barrier_sync();
    }
    if ((*abort_flag || (PAIR && peer_slot[1])) && rank == 0 && warp == 0 && lane == 0) {
        // Let every TMA load and MMA issued land before the shared memory and TMEM go.
        volatile int never = 0;
        const int issued = max(*issued_slot, peer_slot[0]);
        for (int i = max(0, issued - C::STAGES); i < issued; ++i)
            (void)mbar_wait(full_bar(i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u, &never);
        const int committed = *committed_slot;
        for (int jj = max(0, committed - 2); jj < committed; ++jj)
            (void)mbar_wait(tfull_bar(jj & 1), (uint32_t)(jj >> 1) & 1u, &never);
    }
    if constexpr (PAIR) cluster_barrier_sync();   // rank 1 stays until rank 0 has seen every copy land
    else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem, C::TMEM_COLS);
        else tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Fix-up of the last-round K pieces: sum the pieces of each tail tile in piece order, then apply
// the tile's epilogue.  One thread per 8 D-columns of one row (SwiGLU: 8 gate + the 8 matching up).
// Tiles are BMt x BNt (BMt = 256 when CTA pairs computed them).
__global__ void tail_fixup_kernel(const float* __restrict__ tp, int pieces, int tail_tiles, int head_units,
                                  int mt, int group, int BMt, int BNt, int swiglu, int M, int n_valid, int ldo,
                                  int mode, void* out) {
    pdl_launch();
    pdl_wait();
    const int gw = swiglu ? BNt / 16 : BNt / 8;
    const long long per_tile = (long long)BMt * gw;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= per_tile * tail_tiles) return;
    const int t = (int)(idx / per_tile);
    const int rem = (int)(idx - (long long)t * per_tile);
    const int r = rem / gw, cg = (rem - r * gw) * 8;
    // tile (mb, nb) from the raster order
    const int lin = head_units + t;
    const int band_units = group * mt;
    const int band = lin / band_units;
    const int within = lin - band * band_units;
    const int mb = within % mt, nb = band * group + within / mt;
    const int row = mb * BMt + r;
    if (row >= M) return;
    float a[8] = {0, 0, 0, 0, 0, 0, 0, 0}, u[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int pc = 0; pc < pieces; ++pc) {
        const float* src = tp + ((long long)pc * tail_tiles + t) * ((long long)BMt * BNt) + (long long)r * BNt + cg;
        const float4 x0 = *reinterpret_cast<const float4*>(src), x1 = *reinterpret_cast<const float4*>(src + 4);
        a[0] += x0.x; a[1] += x0.y; a[2] += x0.z; a[3] += x0.w; a[4] += x1.x; a[5] += x1.y; a[6] += x1.z; a[7] += x1.w;
        if (swiglu) {
            const float4 y0 = *reinterpret_cast<const float4*>(src + BNt / 2);
            const float4 y1 = *reinterpret_cast<const float4*>(src + BNt / 2 + 4);
            u[0] += y0.x; u[1] += y0.y; u[2] += y0.z; u[3] += y0.w; u[4] += y1.x; u[5] += y1.y; u[6] += y1.z; u[7] += y1.w;
        }
    }
    const int col = swiglu ? nb * (BNt / 2) + cg : nb * BNt + cg;
    if (col >= n_valid) return;
    const long long o = (long long)row * ldo + col;
    if (mode == KM_F32) {
        float4* q = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o);
        q[0] = make_float4(a[0], a[1], a[2], a[3]);
        q[1] = make_float4(a[4], a[5], a[6], a[7]);
        return;
    }
    uint4* q = reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(out) + o);
    if (swiglu) {
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = silu_f(round_bf(a[j])) * round_bf(u[j]);
    } else if (mode == KM_RESIDUAL) {
        float rr[8];
        unpack8(*q, rr);
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = rr[j] + a[j];
    }
    *q = pack8(a);
}

// Last-round K pieces of a residual GEMM fused with the RMSNorm that follows it: one warp per row
// (the whole row in registers, NC 16-byte chunks per lane, N = 256 * NC).  A chunk that lies in a
// tail tile gets r = bf16(r + sum of its pieces in piece order), as tail_fixup_kernel computes it;
// the other chunks already hold the GEMM's residual sum.  Then y = RMSNorm(r) * g over the rounded
// row, with the compensated sum of squares of the row norm kernel.
template <int NC>
__global__ void __launch_bounds__(256, 2) tail_fixup_norm_kernel(const float* __restrict__ tp, int pieces, int tail_tiles, int head_units,
                                       int mt, int group, int BMt, int BNt, int M, int N, bf16* __restrict__ r,
                                       const bf16* __restrict__ g, bf16* __restrict__ y, float eps) {
    pdl_launch();
    pdl_wait();
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    const int mb = row / BMt, rr = row - mb * BMt;
    uint4* rrow = reinterpret_cast<uint4*>(r + (long long)row * N);
    const uint4* gv = reinterpret_cast<const uint4*>(g);
    // the row, and the gains, requested before anything waits for them
    uint4 u[NC], gw[NC];
#pragma unroll
    for (int q = 0; q < NC; ++q) u[q] = rrow[lane + 32 * q];
#pragma unroll
    for (int q = 0; q < NC; ++q) gw[q] = gv[lane + 32 * q];
#pragma unroll
    for (int q = 0; q < NC; ++q) {
        const int col = (lane + 32 * q) * 8;
        const int nb = col / BNt;
        const int band = nb / group;
        const int lin = band * group * mt + (nb - band * group) * mt + mb;
        if (lin < head_units) continue;
        const int t = lin - head_units;
        // every piece of the chunk requested before the first is added (piece order kept)
        float4 x0[kMaxTailPieces], x1[kMaxTailPieces];
#pragma unroll
        for (int pc = 0; pc < kMaxTailPieces; ++pc) {
            if (pc < pieces) {
                const float* src = tp + ((long long)pc * tail_tiles + t) * ((long long)BMt * BNt) + (long long)rr * BNt + (col - nb * BNt);
                x0[pc] = *reinterpret_cast<const float4*>(src);
                x1[pc] = *reinterpret_cast<const float4*>(src + 4);
            }
        }
        float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int pc = 0; pc < kMaxTailPieces; ++pc) {
            if (pc < pieces) {
                a[0] += x0[pc].x; a[1] += x0[pc].y; a[2] += x0[pc].z; a[3] += x0[pc].w;
                a[4] += x1[pc].x; a[5] += x1[pc].y; a[6] += x1[pc].z; a[7] += x1[pc].w;
            }
        }
        float f[8];
        unpack8(u[q], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = f[j] + a[j];
        u[q] = pack8(a);
        rrow[lane + 32 * q] = u[q];
    }
    float ss = 0.f, sc = 0.f;
#pragma unroll
    for (int q = 0; q < NC; ++q) {
        float f[8];
        unpack8(u[q], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) csum_add(ss, sc, __fmul_rn(f[j], f[j]));
    }
    ss = csum_warp(ss, sc);
    const float inv = 1.0f / sqrtf(ss / (float)N + eps);
    uint4* dy = reinterpret_cast<uint4*>(y + (long long)row * N);
#pragma unroll
    for (int q = 0; q < NC; ++q) {
        float f[8], w[8];
        unpack8(u[q], f);
        unpack8(gw[q], w);
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = (f[j] * inv) * w[j];
        dy[lane + 32 * q] = pack8(f);
    }
}

// Sum of split partials in split order, then the epilogue.  One thread per 8 output columns.
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, long long split_stride,
                                     int M, int n_out, int ldp, int up_off, int mode, void* out, int ldo) {
    pdl_launch();
    pdl_wait();
    const int groups = n_out >> 3;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)M * groups) return;
    const int row = (int)(idx / groups);
    const int col = (int)(idx % groups) * 8;
    float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float u[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    constexpr int kBatch = 4;   // split partials loaded together before they are added
    const bool sw = mode == KM_SWIGLU;
    for (int s0 = 0; s0 < splits; s0 += kBatch) {
        float4 x[kBatch][4];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const float* p = part + (s0 + b) * split_stride + (long long)row * ldp + col;
            const bool ok = s0 + b < splits;
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            x[b][0] = ok ? *reinterpret_cast<const float4*>(p) : z;
            x[b][1] = ok ? *reinterpret_cast<const float4*>(p + 4) : z;
            x[b][2] = ok && sw ? *reinterpret_cast<const float4*>(p + up_off) : z;
            x[b][3] = ok && sw ? *reinterpret_cast<const float4*>(p + up_off + 4) : z;
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            if (s0 + b < splits) {
                a[0] += x[b][0].x; a[1] += x[b][0].y; a[2] += x[b][0].z; a[3] += x[b][0].w;
                a[4] += x[b][1].x; a[5] += x[b][1].y; a[6] += x[b][1].z; a[7] += x[b][1].w;
                if (sw) {
                    u[0] += x[b][2].x; u[1] += x[b][2].y; u[2] += x[b][2].z; u[3] += x[b][2].w;
                    u[4] += x[b][3].x; u[5] += x[b][3].y; u[6] += x[b][3].z; u[7] += x[b][3].w;
                }
            }
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

// Split-K reduction fused with the residual add and the RMSNorm that follows it (small M): one CTA
// per row, one thread per group of 8 columns (blockDim = groups rounded up to a warp), all split
// loads issued before the sum (split order kept); writes r = bf16(r + acc), then y = RMSNorm(r) * g
// with the compensated sum of squares of the rounded residual.
constexpr int kNormMaxThreads = 512;   // hidden sizes up to 4096; 128 registers a thread (no spill)
constexpr int kNormMaxSplits = 16;
constexpr int kNormSplitBatch = 8;      // split partials loaded together before they are added
__global__ void __launch_bounds__(kNormMaxThreads) splitk_residual_norm_kernel(
    const float* __restrict__ part, int splits, long long split_stride, int N, bf16* __restrict__ r,
    const bf16* __restrict__ gain, bf16* __restrict__ y, float eps) {
    pdl_launch();
    pdl_wait();
    const int row = blockIdx.x;
    const int groups = N >> 3;
    const int gi = threadIdx.x;
    const bool active = gi < groups;
    const int col = gi * 8;
    float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float ss = 0.f, sc = 0.f;
    if (active) {
        uint4* rp = reinterpret_cast<uint4*>(r + (long long)row * N + col);
        float rr[8];
        unpack8(*rp, rr);
        float a[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
        for (int s0 = 0; s0 < kNormMaxSplits; s0 += kNormSplitBatch) {
            if (s0 < splits) {
                float4 x0[kNormSplitBatch], x1[kNormSplitBatch];
#pragma unroll
                for (int b = 0; b < kNormSplitBatch; ++b) {
                    if (s0 + b < splits) {
                        const float* p = part + (s0 + b) * split_stride + (long long)row * N + col;
                        x0[b] = *reinterpret_cast<const float4*>(p);
                        x1[b] = *reinterpret_cast<const float4*>(p + 4);
                    }
                }
#pragma unroll
                for (int b = 0; b < kNormSplitBatch; ++b) {
                    if (s0 + b < splits) {
                        a[0] += x0[b].x; a[1] += x0[b].y; a[2] += x0[b].z; a[3] += x0[b].w;
                        a[4] += x1[b].x; a[5] += x1[b].y; a[6] += x1[b].z; a[7] += x1[b].w;
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = rr[e] + a[e];
        const uint4 packed = pack8(a);
        *rp = packed;
        unpack8(packed, v);   // the bf16-rounded residual is what the norm sees
#pragma unroll
        for (int e = 0; e < 8; ++e) csum_add(ss, sc, __fmul_rn(v[e], v[e]));
    }
    const float tot = csum_block(ss, sc);
    const float inv = 1.0f / sqrtf(tot / (float)N + eps);
    if (active) {
        float w[8];
        unpack8(*reinterpret_cast<const uint4*>(gain + col), w);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (v[e] * inv) * w[e];
        *reinterpret_cast<uint4*>(y + (long long)row * N + col) = pack8(v);
    }
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

// Row-major matrix [rows, cols] of bf16 (esize 2) or one-byte E4M3 (esize 1) viewed as a 2-D
// tensor (cols innermost), boxes of 128 bytes x box_rows.
bool encode_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int esize) {
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
    cuuint32_t box[2] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps describe only (address, shape, box), so an encoded map is reused whenever the same
// matrix is seen again (weights every call, workspace buffers every layer).
struct MapKey {
    const void* base;
    int rows, cols, box_rows, esize;
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && cols == o.cols && box_rows == o.box_rows && esize == o.esize;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        size_t h = std::hash<const void*>()(k.base);
        h ^= (size_t)k.rows * 0x9E3779B97F4A7C15ull + (size_t)k.cols * 0xC2B2AE3D27D4EB4Full + (size_t)k.box_rows +
             ((size_t)k.esize << 40);
        return h;
    }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

bool make_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows, int esize = 2) {
    const MapKey key{base, rows, cols, box_rows, esize};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *m = it->second;
            return true;
        }
    }
    if (!encode_map(m, base, rows, cols, box_rows, esize)) return false;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() > 8192) g_maps.clear();
    g_maps.emplace(key, *m);
    return true;
}

struct Plan {
    int bn;
    int splits;
    int kbps;
    int mt, nt;
    int head_units = 0, tail_tiles = 0, tail_splits = 1, kb_per_tail = 0;
    bool pair = false;   // 2-CTA clusters on 256 x 256 tiles
    int bmt = BM;        // rows of a tile
};

// Last-round split: when the final round of tiles fills at most half the SMs, each of its tiles is
// cut into up to kMaxTailPieces K pieces that run on the SMs that would otherwise idle.
void plan_tail(Plan& pl, int n_kb, int nsm) {
    const long long units = (long long)pl.mt * pl.nt;
    const long long rounds = (units + nsm - 1) / nsm;
    const long long tail = units - (rounds - 1) * nsm;
    if (pl.splits != 1 || rounds < 2 || tail * 2 > nsm) return;
    int S = (int)std::min<long long>(kMaxTailPieces, nsm / tail);
    while (S > 1 && n_kb < 2 * S) --S;
    if (S < 2) return;
    pl.head_units = (int)((rounds - 1) * nsm);
    pl.tail_tiles = (int)tail;
    pl.tail_splits = S;
    pl.kb_per_tail = (n_kb + S - 1) / S;
}

// Choose the tile width and K split.  The kernel is persistent (one CTA per SM walking work
// units), so the grid runs in ceil(units / SMs) rounds; per-unit time ~ (K blocks) x BN (bytes
// streamed and MMA work both scale with BN) plus a fixed tile overhead.  Splitting K is allowed
// for a single M tile only and costs a reduction pass.
Plan make_plan(int M, int N, int K, int epi, int split_req, int nsm, int ke = BK) {
    const int n_kb = K / ke;
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
            // K-block cost relative to a 256-wide tile: with one M tile the unit streams weights
            // (cost ~ BN); with several, the 128-wide tile is bound by operand traffic into shared
            // memory (measured 0.83 of the 256-wide tile's time for half its MMA work).
            const double c_kb = bn == 256 ? 1.0 : (mt == 1 ? 0.5 : 0.83);
            Plan cand{bn, splits, kbps, mt, nt};
            plan_tail(cand, n_kb, nsm);
            const double eff_rounds = cand.tail_tiles > 0 ? (double)(rounds - 1) + 1.0 / cand.tail_splits + 0.1
                                                          : (double)rounds;
            double cost = eff_rounds * (kbps * c_kb + 0.5);
            if (splits > 1) cost += 2.0;
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best = cand;
            }
        }
    }
    return best;
}

// Rows from which the projection GEMM runs on CTA pairs (at least two 256-row tiles).
constexpr int kPairMinM = 512;

template <int BN, bool SW, bool F8, bool PAIR>
cudaError_t configure_tile() {
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(gemm_bf16_tc_kernel<BN, SW, F8, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<BN, PAIR>::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    return cudaSuccess;
}

// CTA pairs that can be resident at once (one CTA per SM; a pair needs two SMs of one GPC).
int pair_walkers() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return device_sm_count() / 2;
    if (cached[dev] == 0) {
        int n = 0;
        if (configure_tile<256, false, false, true>() == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * device_sm_count());
            cfg.blockDim = dim3(kTileThreads);
            cfg.dynamicSmemBytes = Cfg<256, true>::SMEM;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, gemm_bf16_tc_kernel<256, false, false, true>, &cfg) != cudaSuccess)
                n = 0;
            (void)cudaGetLastError();
        }
        cached[dev] = n > 0 ? std::min(n, device_sm_count() / 2) : device_sm_count() / 2;
    }
    return cached[dev];
}

// 256 x 256 tiles over CTA pairs: no K split; a last round that leaves more than half of the pairs
// idle runs as K pieces, as on single CTAs.
Plan make_plan_pair(int M, int N, int K, int epi, int npairs, int ke = BK) {
    const int n_kb = K / ke;
    const int dcols = epi == EPI_SWIGLU ? 2 * N : N;
    Plan pl{256, 1, n_kb, (M + 2 * BM - 1) / (2 * BM), (dcols + 255) / 256};
    pl.pair = true;
    pl.bmt = 2 * BM;
    plan_tail(pl, n_kb, npairs);
    return pl;
}

bool use_pairs(int M, int split_req, bool partial_only) {
    return g_gemm_pairs && !partial_only && M >= kPairMinM && split_req <= 1;
}

template <int BN, bool SW, bool F8, bool PAIR>
cudaError_t launch_tile(const CUtensorMap& ma, const CUtensorMap& mb, const GemmArgs& g, const Plan& pl,
                        cudaStream_t st) {
    cudaError_t e = configure_tile<BN, SW, F8, PAIR>();
    if (e != cudaSuccess) return e;
    const long long units = (long long)pl.mt * pl.nt * pl.splits;
    if constexpr (PAIR) {
        const int pairs = (int)std::min<long long>(units, pair_walkers());
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * pairs);
        cfg.blockDim = dim3(kTileThreads);
        cfg.dynamicSmemBytes = Cfg<BN, PAIR>::SMEM;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        count_launches(1);
        e = cudaLaunchKernelEx(&cfg, gemm_bf16_tc_kernel<BN, SW, F8, PAIR>, ma, mb, g);
        if (e != cudaSuccess) return e;
    } else {
        const int nsm = device_sm_count();
        dim3 grid((unsigned)std::min<long long>(units, nsm));
        HRA_LAUNCH(gemm_bf16_tc_kernel<BN, SW, F8, PAIR>, dim3(grid), dim3(kTileThreads), Cfg<BN, PAIR>::SMEM, st, ma,
                   mb, g);
    }
    return cudaGetLastError();
}


constexpr int kSmallM = 64;   // at most this many rows take the head-form path below

// Reduction / epilogue pass shared by both GEMM paths once fp32 partials exist.
cudaError_t reduce_partials(const LinearCall& c, int splits, int ldp, cudaStream_t st) {
    const int mode = c.epi == EPI_STORE ? KM_STORE : c.epi == EPI_RESIDUAL ? KM_RESIDUAL : c.epi == EPI_SWIGLU ? KM_SWIGLU : KM_F32;
    if (mode == KM_RESIDUAL && c.norm_out != nullptr && c.N <= 8 * kNormMaxThreads && splits <= kNormMaxSplits) {
        const int threads = ((c.N / 8 + 31) / 32) * 32;
        HRA_LAUNCH(splitk_residual_norm_kernel, dim3(c.M), dim3(threads), 0, st, c.partial, splits, (long long)c.M * ldp, c.N,
                                                              reinterpret_cast<bf16*>(c.out), c.norm_gain,
                                                              c.norm_out, c.norm_eps);
        if (c.norm_done) *c.norm_done = true;
        return cudaGetLastError();
    }
    const long long items = (long long)c.M * (c.N / 8);
    const int threads = 256;
    HRA_LAUNCH(splitk_reduce_kernel, dim3((unsigned)((items + threads - 1) / threads)), dim3(threads), 0, st, 
        c.partial, splits, (long long)c.M * ldp, c.M, c.N, ldp, c.N, mode, c.out, c.N);
    return cudaGetLastError();
}

// At most 64 BF16 rows: the audio-head kernel's form (head.cu) -- 256 weight rows a tile as the
// MMA's N side, so that one instruction consumes 256 rows x 16 K of weights -- over tiles x K splits
// (up to kSmallHeadSplits), fp32 partial planes [split][M][ldp], then the epilogue's reduction.
constexpr int kSmallHeadSplits = 16;

cudaError_t launch_linear_small_head(const LinearCall& c, cudaStream_t st) {
    const bool sw = c.epi == EPI_SWIGLU;
    const int ldp = sw ? 2 * c.N : c.N;   // gate/up: gate columns then up columns, as the weight's rows
    HeadCall h{};
    h.hidden = c.a;
    h.head_w = c.w;
    h.partial = c.partial;
    h.err = c.err;
    h.zero_ptr = c.zero_ptr;
    h.zero_words = c.zero_ptr ? c.zero_words : 0;
    int splits = 1;
    h.splits_used = &splits;
    h.B = c.M;
    h.N = ldp;
    h.H = c.K;
    h.max_splits = kSmallHeadSplits;
    h.split_req = c.split_req;
    h.no_l2_prefetch = true;
    cudaError_t e = launch_audio_head(h, st);
    if (c.splits_used) *c.splits_used = splits;
    if (e != cudaSuccess || c.partial_only) return e;
    if (c.qk != nullptr && c.epi == EPI_STORE && c.M == c.qk->rows && c.N == (c.qk->nq + 2 * c.qk->nkv) * c.qk->hd) {
        // merged QKV: the split reduction happens inside the q/k norm + RoPE + cache-write kernel
        QkRopeArgs qa = *c.qk;
        qa.part = c.partial;
        qa.splits = splits;
        qa.split_stride = (long long)c.M * ldp;
        qa.ldp = ldp;
        e = launch_qk_rope_kv(qa, st);
        if (e == cudaSuccess && c.qk_done) *c.qk_done = true;
        return e;
    }
    return reduce_partials(c, splits, ldp, st);
}

}  // namespace

bool make_map_u8(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    if (!get_encoder()) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_2d(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    return get_encoder() && make_map(m, base, rows, cols, box_rows, 2);
}

bool encode_tensor_map(void* map, int rank, const void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                       const uint32_t* box) {
    if (!get_encoder() || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    return g_encode(reinterpret_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                    const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool g_gemm_pairs = true;

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

size_t linear_partial_bytes(int M, int N, int K, int epi, int split_req, bool partial_only) {
    if (M <= kSmallM) {   // the head-form path always writes its partial planes
        const size_t ldp = epi == EPI_SWIGLU ? 2 * (size_t)N : (size_t)N;
        const HeadPlan hp = head_plan((int)ldp, K, kSmallHeadSplits, split_req);
        return (size_t)hp.splits * (size_t)M * ldp * sizeof(float);
    }
    const Plan pl = use_pairs(M, split_req, partial_only) ? make_plan_pair(M, N, K, epi, pair_walkers())
                                                                   : make_plan(M, N, K, epi, split_req, device_sm_count());
    if (pl.tail_tiles > 0) return (size_t)pl.tail_splits * pl.tail_tiles * pl.bmt * pl.bn * sizeof(float);
    if (pl.splits <= 1) return 0;
    const size_t ldp = epi == EPI_SWIGLU ? 2 * (size_t)N : (size_t)N;
    return (size_t)pl.splits * (size_t)M * ldp * sizeof(float);
}

// Tail pieces x tail tiles stay within the walkers (SMs, or pairs of 256-row tiles): either way at
// most SMs x 128 rows x 256 columns of fp32.
size_t linear_tail_bound() { return (size_t)device_sm_count() * BM * 256 * sizeof(float); }

size_t linear_partial_bound(int m_max, int N, int K, int epi) {
    if (m_max > BM) m_max = BM;
    const size_t ldp = epi == EPI_SWIGLU ? 2 * (size_t)N : (size_t)N;
    const size_t splits = m_max <= kSmallM ? kSmallHeadSplits : 8;
    return splits * (size_t)m_max * ldp * sizeof(float);
}

cudaError_t launch_linear(const LinearCall& c, cudaStream_t st) {
    if (!get_encoder()) return cudaErrorNotSupported;
    if (c.M <= kSmallM && !c.fp8) return launch_linear_small_head(c, st);   // FP8 always takes the tile path
    const int nsm = device_sm_count();
    const int ke = c.fp8 ? 2 * BK : BK;
    if (c.fp8 && (c.K % ke != 0 || c.a_scale == nullptr || c.w_scale == nullptr)) return cudaErrorInvalidValue;
    Plan pl = use_pairs(c.M, c.split_req, c.partial_only) ? make_plan_pair(c.M, c.N, c.K, c.epi, pair_walkers(), ke)
                                                         : make_plan(c.M, c.N, c.K, c.epi, c.split_req, nsm, ke);
    if (c.partial_only) pl.tail_tiles = 0;   // the caller reads one output plane from the partial buffer
    const bool fuse_qk =
        !c.fp8 && c.qk != nullptr && c.epi == EPI_STORE && pl.splits == 1 && pl.bn % c.qk->hd == 0;
    if (fuse_qk) pl.tail_tiles = 0;
    const bool sw = c.epi == EPI_SWIGLU;
    const int w_rows = sw ? 2 * c.N : c.N;
    const int esize = c.fp8 ? 1 : 2;

    CUtensorMap ma, mb;
    if (!make_map(&ma, c.a, c.M, c.K, BM, esize)) return cudaErrorInvalidValue;
    if (!make_map(&mb, c.w, w_rows, c.K, (sw || pl.pair) ? pl.bn / 2 : pl.bn, esize)) return cudaErrorInvalidValue;

    GemmArgs g{};
    g.err = c.err;
    g.M = c.M;
    g.n_valid = c.N;
    g.n_kb = c.K / ke;
    g.a_scale = c.a_scale;
    g.w_scale = c.w_scale;
    g.kb_per_split = pl.kbps;
    g.up_row0 = c.N;
    g.mt = pl.mt;
    g.nt = pl.nt;
    g.splits = pl.splits;
    g.group = 8;
    g.head_units = pl.head_units;
    g.tail_tiles = pl.tail_tiles;
    g.tail_splits = pl.tail_splits;
    g.kb_per_tail = pl.kb_per_tail;
    g.tail_part = c.partial;
    g.zero_ptr = c.zero_ptr;
    g.zero_words = c.zero_ptr ? c.zero_words : 0;
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
    if (fuse_qk) {
        g.mode = KM_QKROPE;
        g.qk = *c.qk;
        if (c.qk_done) *c.qk_done = true;
    }
    // 32-byte epilogue accesses when every output row starts 32-byte aligned
    {
        const size_t esz = g.mode == KM_F32 || g.mode == KM_PARTIAL ? 4 : 2;
        const auto a32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
        bool ok = a32(g.out) && ((size_t)g.ldo * esz) % 32 == 0 && (g.split_stride * (long long)esz) % 32 == 0;
        if (g.mode == KM_QKROPE) ok = a32(g.qk.q_out) && a32(g.qk.kv_layer);
        g.v8 = ok ? 1 : 0;
    }

    cudaError_t e;
    if (pl.pair && c.fp8) {
        e = sw ? launch_tile<256, true, true, true>(ma, mb, g, pl, st)
               : launch_tile<256, false, true, true>(ma, mb, g, pl, st);
    } else if (pl.pair) {
        e = sw ? launch_tile<256, true, false, true>(ma, mb, g, pl, st)
               : launch_tile<256, false, false, true>(ma, mb, g, pl, st);
    } else if (c.fp8) {
        if (pl.bn == 256)
            e = sw ? launch_tile<256, true, true, false>(ma, mb, g, pl, st)
                   : launch_tile<256, false, true, false>(ma, mb, g, pl, st);
        else
            e = sw ? launch_tile<128, true, true, false>(ma, mb, g, pl, st)
                   : launch_tile<128, false, true, false>(ma, mb, g, pl, st);
    } else if (pl.bn == 256) {
        e = sw ? launch_tile<256, true, false, false>(ma, mb, g, pl, st)
               : launch_tile<256, false, false, false>(ma, mb, g, pl, st);
    } else {
        e = sw ? launch_tile<128, true, false, false>(ma, mb, g, pl, st)
               : launch_tile<128, false, false, false>(ma, mb, g, pl, st);
    }
    if (c.splits_used) *c.splits_used = pl.splits;
    if (e == cudaSuccess && pl.tail_tiles > 0 && g.mode == KM_RESIDUAL && c.norm_out != nullptr &&
        (c.N == 2560 || c.N == 256)) {
        // the tail pieces and the RMSNorm that follows in one pass over each row
        const int warps = 8;
        const dim3 grid((unsigned)((c.M + warps - 1) / warps));
        if (c.N == 2560)
            HRA_LAUNCH(tail_fixup_norm_kernel<10>, grid, dim3(32 * warps), 0, st, c.partial, pl.tail_splits,
                       pl.tail_tiles, pl.head_units, pl.mt, 8, pl.bmt, pl.bn, c.M, c.N, reinterpret_cast<bf16*>(c.out),
                       c.norm_gain, c.norm_out, c.norm_eps);
        else
            HRA_LAUNCH(tail_fixup_norm_kernel<1>, grid, dim3(32 * warps), 0, st, c.partial, pl.tail_splits,
                       pl.tail_tiles, pl.head_units, pl.mt, 8, pl.bmt, pl.bn, c.M, c.N, reinterpret_cast<bf16*>(c.out),
                       c.norm_gain, c.norm_out, c.norm_eps);
        if (c.norm_done) *c.norm_done = true;
        return cudaGetLastError();
    }
    if (e == cudaSuccess && pl.tail_tiles > 0) {
        const int gw = sw ? pl.bn / 16 : pl.bn / 8;
        const long long items = (long long)pl.tail_tiles * pl.bmt * gw;
        HRA_LAUNCH(tail_fixup_kernel, dim3((unsigned)((items + 255) / 256)), dim3(256), 0, st,
            c.partial, pl.tail_splits, pl.tail_tiles, pl.head_units, pl.mt, 8, pl.bmt, pl.bn, sw ? 1 : 0, c.M, c.N,
            c.N, g.mode, c.out);
        return cudaGetLastError();
    }
    if (e != cudaSuccess || pl.splits <= 1 || c.partial_only) return e;

    const int mode = c.epi == EPI_STORE ? KM_STORE : c.epi == EPI_RESIDUAL ? KM_RESIDUAL : c.epi == EPI_SWIGLU ? KM_SWIGLU : KM_F32;
    if (mode == KM_RESIDUAL && c.norm_out != nullptr && c.N <= 8 * kNormMaxThreads && pl.splits <= kNormMaxSplits) {
        const int threads = ((c.N / 8 + 31) / 32) * 32;
        HRA_LAUNCH(splitk_residual_norm_kernel, dim3(c.M), dim3(threads), 0, st, c.partial, pl.splits, (long long)c.M * g.ldo, c.N,
                                                              reinterpret_cast<bf16*>(c.out), c.norm_gain,
                                                              c.norm_out, c.norm_eps);
        if (c.norm_done) *c.norm_done = true;
        return cudaGetLastError();
    }
    const long long items = (long long)c.M * (c.N / 8);
    const int threads = 256;
    HRA_LAUNCH(splitk_reduce_kernel, dim3((unsigned)((items + threads - 1) / threads)), dim3(threads), 0, st, 
        c.partial, pl.splits, (long long)c.M * g.ldo, c.M, c.N, g.ldo, c.N, mode, c.out, c.N);
    return cudaGetLastError();
}

}  // namespace hra
