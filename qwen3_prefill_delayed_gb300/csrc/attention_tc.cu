// attention_tc.cu -- causal GQA prefill attention on the 5th-generation tensor cores.
//
// Semantics: row i of sequence b (position start_b + i) with
// q head h attends cache slots 0 .. start_b + i of kv head h / (n_q / n_kv) with
// softmax(q.k / sqrt(hd)) ("flashrt-structures 0.2.0, prefill_tower/fp8_chain.py" page, its description: attention runs over the used keys only;
// causal because the backbone is a decoder).
//
// A work item = one kv head of one sequence and QT = 128 / G consecutive query positions, for all
// G = n_q / n_kv q heads of that kv head: the 128 rows of every tcgen05.mma are (position, head)
// pairs, row r = (position r / G, head r % G), so each K/V tile is loaded once for the G heads.
// The kernel is persistent (two CTAs per SM) and its pipelines run across items.  The items come
// from a work list built once per call (attn_schedule_kernel): the non-empty (query tile, sequence)
// pairs sorted by their key-tile count, heaviest first, each for every kv head; CTA c takes list
// entries in snake order (c, 2 grid - 1 - c, 2 grid + c, ...), so every round pairs a heavier and
// a lighter item and all CTAs finish close together (a single sequence needs no list: its query
// tiles, last first).  Within a CTA, the next item's Q and K/V stream in while this one's softmax and PV finish, and O
// alternates between two TMEM accumulators so one item's epilogue overlaps the next item's MMAs.
//   warp 0     TMA: lane 0 the Q tile (a 3-D box of 64 dims x G heads x QT positions per 64-dim
//              half) and a 3-stage ring of 64-key K tiles, lane 1 the V ring, straight from the
//              cache (K stages come free once S has read them, V stages once PV has);
//   warp 1     allocates TMEM (S: two 64-column buffers, O: two hd-column accumulators) and issues
//              the MMAs:
//              S_j = Q K_j^T (K-major operands), then O += P_j V_j with P_j from shared memory
//              (K-major) and V_j as the MN-major B operand;
//   warps 2-5  one row per thread: online softmax of S_j in fp32 (scores in log2 units, causal and
//              length mask on the tiles that need it), P_j written to one of two shared-memory buffers
//              as a bf16 hi + lo pair (hi the top 16 bits, lo = bf16(p - hi), so the probabilities
//              enter PV with about 16 significant bits), the O accumulator rescaled in TMEM only
//              when a row's reference max moves by more than 2^8 (only then does the softmax wait for
//              the previous PV), and the final O / l stored as bf16.
// Key slots past the last valid key of a tile are zeroed in the V tile before PV, so stale cache
// contents never reach the output (0 x NaN).
#include <cudaTypedefs.h>

#include <algorithm>
#include <math.h>

#include "internal.h"

namespace hra {

namespace {

constexpr int TROWS = 128;         // MMA rows: G heads x QT positions
constexpr int kTcThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyLog2 = 8.0f;   // reference-max slack of the online softmax (log2 units)

// TK keys per K/V tile, NS stages in each of the K and V rings, OB TMEM accumulators for O.
//   <32, 2, 1> (launched): ~97 KB of shared memory and 256 TMEM columns, so two CTAs share an SM and
//               hide each other's per-item latency; P rows are 64 bytes (64-byte swizzle).
//   <64, 3, 2>: one CTA per SM (198 KB, 512 TMEM columns); O alternates between items so an item's
//               epilogue overlaps the next.  Kept as a configuration; measured slower.
template <int HD, int TK, int NS, int OB>
struct AttnCfg {
    static constexpr int NSUB = HD / 64;                 // 64-dim (128-byte) halves of a head
    static constexpr int Q_BYTES = NSUB * TROWS * 128;   // Q tile
    static constexpr int KV_SUB = TK * 128;              // one TK-key x 64-dim sub-tile
    static constexpr int K_BYTES = NSUB * KV_SUB;
    static constexpr int P_ROW = TK * 2;                 // bytes of one P row (bf16)
    static constexpr int P_BYTES = TROWS * P_ROW;
    // Q | K stages | V stages | P buffer 0 (hi, lo) | P buffer 1 (hi, lo) | barriers
    static constexpr int OFF_K = Q_BYTES;
    static constexpr int OFF_V = OFF_K + NS * K_BYTES;
    static constexpr int OFF_P = OFF_V + NS * K_BYTES;
    static constexpr int OFF_BAR = OFF_P + 4 * P_BYTES;
    static constexpr int SMEM = OFF_BAR + 256 + 1024;
    // S buffers at columns [0, TK) and [TK, 2 TK), O accumulator ob at 2 TK + 128 ob
    static constexpr uint32_t TMEM_COLS = 2 * TK + 128 * OB <= 256 ? 256u : 512u;
    // barriers: q_full, q_empty, k_full[NS], v_full[NS], k_empty[NS], v_empty[NS], s_full[2],
    // s_free[2], p_full[2], pv_done[2], o_free[OB], mma_idle
    static constexpr int B_QF = 0, B_QE = 1, B_KF = 2, B_VF = 2 + NS, B_KE = 2 + 2 * NS, B_VE = 2 + 3 * NS;
    static constexpr int B_SF = 2 + 4 * NS, B_SFREE = B_SF + 2, B_PF = B_SFREE + 2, B_PV = B_PF + 2;
    static constexpr int B_OF = B_PV + 2, B_IDLE = B_OF + OB, NBARS = B_IDLE + 1;
    static_assert(NBARS * 8 + 5 * 4 <= 256, "barrier area");
};

struct TcAttnArgs {
    const int32_t* cu;      // [batch + 1]
    const int32_t* start;   // [batch]
    bf16* out;              // [T, nq * hd]
    unsigned int* err;
    int batch, max_len, n_slots, nq, nkv, G, QT;
    long long kv_rows_per_seq;   // 2 * nkv * n_slots: rows of one sequence in the cache's row view
    float scale_log2;
    const int32_t* sched;        // [0] = pairs; pair i's record at sched + 8 (i + 1): sequence, first
                                 // packed row, length, first query position in it, start position,
                                 // keys (start + min(length, t0 + QT)); heaviest first.  Null for one
                                 // sequence: pair i is its query tile n_qt - 1 - i
    int v8;                      // out 32-byte aligned: O rows leave in 32-byte stores
};

// Work-list builder: one CTA.  Pair (q tile qt, sequence b) is non-empty when qt * QT < len_b; its
// weight is its key-tile count ceil((start_b + min(len_b, (qt + 1) QT)) / TK).  Counting sort by
// weight, heaviest first (the order inside one weight is immaterial: items are independent).  Each
// entry is the pair's whole record (32 bytes), so an item's set-up is one load, not a chain.
constexpr int kSchedBins = 1024;
constexpr int kLaunchedTK = 32;   // keys per tile of the launched configuration (the list's weights)
__global__ void __launch_bounds__(1024) attn_schedule_kernel(const int32_t* __restrict__ cu,
                                                             const int32_t* __restrict__ start, int batch, int n_qt,
                                                             int QT, int TK, int32_t* __restrict__ sched) {
    pdl_launch();
    pdl_wait();
    __shared__ int hist[kSchedBins];
    __shared__ int total;
    for (int i = threadIdx.x; i < kSchedBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int n_pairs = n_qt * batch;
    auto bin_of = [&](int pr, int& code) -> int {   // -1: empty pair
        const int qt = pr / batch, b = pr - qt * batch;
        const int len = cu[b + 1] - cu[b];
        const int t0 = qt * QT;
        if (t0 >= len) return -1;
        const int kv = (start ? start[b] : 0) + min(len, t0 + QT);
        code = (qt << 16) | b;
        return kSchedBins - 1 - min(kSchedBins - 1, (kv + TK - 1) / TK);   // heaviest first
    };
    for (int pr = threadIdx.x; pr < n_pairs; pr += blockDim.x) {
        int code;
        const int bin = bin_of(pr, code);
        if (bin >= 0) atomicAdd(&hist[bin], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {   // exclusive scan of the histogram: 32 bins a lane, then across lanes
        constexpr int per = kSchedBins / 32;
        int s = 0;
        for (int i = 0; i < per; ++i) s += hist[threadIdx.x * per + i];
        int incl = s;
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if ((int)threadIdx.x >= o) incl += v;
        }
        int run = incl - s;
        for (int i = 0; i < per; ++i) {
            const int h = hist[threadIdx.x * per + i];
            hist[threadIdx.x * per + i] = run;
            run += h;
        }
        if (threadIdx.x == 31) total = incl;
    }
    __syncthreads();
    for (int pr = threadIdx.x; pr < n_pairs; pr += blockDim.x) {
        int code;
        const int bin = bin_of(pr, code);
        if (bin >= 0) {
            const int b = code & 0xFFFF, qt = code >> 16;
            const int c0 = cu[b], len = cu[b + 1] - c0, t0 = qt * QT, s0 = start ? start[b] : 0;
            int4* rec = reinterpret_cast<int4*>(sched + 8 * (1 + atomicAdd(&hist[bin], 1)));
            rec[0] = make_int4(b, c0, len, t0);
            rec[1] = make_int4(s0, s0 + min(len, t0 + QT), 0, 0);
        }
    }
    if (threadIdx.x == 0) sched[0] = total;
}

// List entry s: pair s / nkv of the work list, kv head s % nkv.  Returns the item's key-tile count.
__device__ __forceinline__ int attn_item(const TcAttnArgs& p, int s, int tk, int& b, int& j, int& cu0, int& len,
                                         int& t0, int& s0, int& kv_len) {
    const int pi = s / p.nkv;
    j = s - pi * p.nkv;
    if (p.sched != nullptr) {   // the pair's record, both halves requested together
        const int4* rec = reinterpret_cast<const int4*>(p.sched + 8 * (1 + pi));
        const int4 r0 = rec[0], r1 = rec[1];
        b = r0.x;
        cu0 = r0.y;
        len = r0.z;
        t0 = r0.w;
        s0 = r1.x;
        kv_len = r1.y;
        return (kv_len + tk - 1) / tk;
    }
    // one sequence: its query tiles, last (heaviest) first
    b = 0;
    const int qt = (p.max_len + p.QT - 1) / p.QT - 1 - pi;
    cu0 = p.cu[b];
    len = p.cu[b + 1] - cu0;
    t0 = qt * p.QT;
    if (t0 >= len) return 0;
    s0 = p.start ? p.start[b] : 0;
    kv_len = s0 + min(len, t0 + p.QT);
    return (kv_len + tk - 1) / tk;
}

// The k-th list entry of this CTA: snake order over the grid.
__device__ __forceinline__ int snake_entry(int k) {
    return k * (int)gridDim.x + ((k & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// Persistent: each CTA walks list entries snake_entry(0), snake_entry(1), ...  Every role walks
// the same items and numbers the key tiles it handles across items (g), which fixes the K/V ring
// stage (g % NS), the S and P buffer (g & 1) and each barrier's phase.  Every barrier's consecutive
// completions are gated by the other side having seen the previous one, so no waiter can fall two
// phases behind.
template <int HD, int TK, int NS, int OB>
__global__ void __launch_bounds__(kTcThreads, (TK == 32 ? 2 : 1))
    prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                           const TcAttnArgs p) {
    using C = AttnCfg<HD, TK, NS, OB>;
    pdl_launch();
    pdl_wait();   // the row map, Q and this layer's K/V all come from earlier kernels
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* slots = reinterpret_cast<uint32_t*>(bars + C::NBARS);   // tmem, abort, issued K, V, Q
    volatile int* abort_flag = reinterpret_cast<volatile int*>(slots + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const uint32_t sQ = smem_u32(smem), sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
    const uint32_t sP0 = smem_u32(smem + C::OFF_P);   // buffer q: hi at sP0 + 2q P_BYTES, lo right after

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = (p.sched != nullptr ? p.sched[0] : (p.max_len + p.QT - 1) / p.QT) * p.nkv;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NBARS; ++i) {
            const bool four = (i >= C::B_SFREE && i < C::B_PV) || (i >= C::B_OF && i < C::B_IDLE);
            mbar_init(bar(i), four ? 4 : 1);   // s_free, p_full, o_free: one arrival per softmax warp
        }
        *abort_flag = 0;
        slots[2] = slots[3] = slots[4] = 0;
        mbar_fence_init();
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmKV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(slots), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = slots[0];
    int b, j, cu0, len, t0, s0, kv_len;

    if (warp == 0 && lane < 2) {
        // lane 0: Q and the K ring; lane 1: the V ring
        const bool is_k = lane == 0;
        const int full0 = is_k ? C::B_KF : C::B_VF, empty0 = is_k ? C::B_KE : C::B_VE;
        const uint32_t ring = is_k ? sK : sV;
        int g = 0, it = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int i = snake_entry(k);
            if (i >= n_items) break;
            const int n_kt = attn_item(p, i, TK, b, j, cu0, len, t0, s0, kv_len);
            if (n_kt == 0) continue;
            if (is_k) {
                if (it >= 1 && !mbar_wait(bar(C::B_QE), (uint32_t)(it - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(bar(C::B_QF), C::Q_BYTES);
#pragma unroll
                for (int h = 0; h < C::NSUB; ++h)
                    tma_load_3d(sQ + h * TROWS * 128, &tmQ, bar(C::B_QF), 64 * h, j * p.G, cu0 + t0);
                reinterpret_cast<volatile int*>(slots)[4] = it + 1;
            }
            const long long row0 = (long long)b * p.kv_rows_per_seq + (long long)j * p.n_slots +
                                   (is_k ? 0LL : (long long)p.nkv * p.n_slots);
            for (int t = 0; t < n_kt; ++t, ++g) {
                const int st = g % NS;
                if (g >= NS && !mbar_wait(bar(empty0 + st), (uint32_t)(g / NS - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(bar(full0 + st), C::K_BYTES);
#pragma unroll
                for (int h = 0; h < C::NSUB; ++h)
                    tma_load_2d(ring + st * C::K_BYTES + h * C::KV_SUB, &tmKV, bar(full0 + st), 64 * h,
                                (int)(row0 + (long long)t * TK));
                reinterpret_cast<volatile int*>(slots)[2 + lane] = g + 1;
            }
            ++it;
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
        }
    } else if (warp == 1 && lane == 0) {
        constexpr uint32_t idesc_s = idesc_bf16_f32(TROWS, TK);
        // PV: B = V is MN-major (transpose bit 16), N = HD
        constexpr uint32_t idesc_o = idesc_bf16_f32(TROWS, HD) | (1u << 16);
        auto issue_s = [&](int gs) -> bool {
            const int sb = gs & 1, ks = gs % NS;
            if (!mbar_wait(bar(C::B_KF + ks), (uint32_t)(gs / NS) & 1u, abort_flag)) return false;
            if (gs >= 2 && !mbar_wait(bar(C::B_SFREE + sb), (uint32_t)((gs >> 1) - 1) & 1u, abort_flag)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * TROWS * 128) + 2ull * (kk & 3);
                const uint64_t bd = sdesc_sw128(sK + ks * C::K_BYTES + (kk >> 2) * C::KV_SUB) + 2ull * (kk & 3);
                tc_mma_bf16(tmem + sb * TK, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(bar(C::B_SF + sb));   // S ready for the softmax
            tc_commit(bar(C::B_KE + ks));   // K stage free again
            return true;
        };
        int g = 0, it = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int i = snake_entry(k);
            if (i >= n_items) break;
            const int n_kt = attn_item(p, i, TK, b, j, cu0, len, t0, s0, kv_len);
            if (n_kt == 0) continue;
            const int ob = it % OB;
            const uint32_t tO = tmem + 2 * TK + (uint32_t)(ob * 128);
            if (!mbar_wait(bar(C::B_QF), (uint32_t)it & 1u, abort_flag) || !issue_s(g)) {
                ok = false;
                break;
            }
            if (n_kt == 1) tc_commit(bar(C::B_QE));   // Q read by the item's last S
            for (int t = 0; t < n_kt; ++t) {
                const int gt = g + t;
                if (t + 1 < n_kt) {
                    if (!issue_s(gt + 1)) {
                        ok = false;
                        break;
                    }
                    if (t + 2 == n_kt) tc_commit(bar(C::B_QE));
                }
                // O buffer ob was last read by the epilogue of item it - OB
                if (!mbar_wait(bar(C::B_PF + (gt & 1)), (uint32_t)(gt >> 1) & 1u, abort_flag) ||
                    !mbar_wait(bar(C::B_VF + gt % NS), (uint32_t)(gt / NS) & 1u, abort_flag) ||
                    (t == 0 && it >= OB &&
                     !mbar_wait(bar(C::B_OF + ob), (uint32_t)((it / OB) - 1) & 1u, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t v_base = sV + (gt % NS) * C::K_BYTES;
                const uint32_t ph = sP0 + (uint32_t)(2 * (gt & 1) * C::P_BYTES), pl = ph + C::P_BYTES;
#pragma unroll
                for (int ks = 0; ks < TK / 16; ++ks) {
                    const uint64_t bd = sdesc_sw128_mn(v_base + ks * 16 * 128, C::KV_SUB, 1024);
                    const uint64_t adh = (TK == 64 ? sdesc_sw128(ph) : sdesc_sw64(ph)) + 2ull * ks;
                    const uint64_t adl = (TK == 64 ? sdesc_sw128(pl) : sdesc_sw64(pl)) + 2ull * ks;
                    tc_mma_bf16(tO, adh, bd, idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
                    tc_mma_bf16(tO, adl, bd, idesc_o, 1u);
                }
                tc_commit(bar(C::B_PV + (gt & 1)));   // P buffer gt & 1 (and O) free again
                tc_commit(bar(C::B_VE + gt % NS));    // V stage free again
            }
            g += n_kt;
            ++it;
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
        }
        tc_commit(bar(C::B_IDLE));   // completes once every MMA this thread issued has finished
    } else if (warp >= 2) {
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                 // MMA row = TMEM lane
        const int tl = r / p.G, hg = r - (r / p.G) * p.G;
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        int g = 0, it = 0, pv_seen = 0;   // PV(0) .. PV(pv_seen - 1) are known to be complete
        bool ok = true;
        auto wait_pv = [&](int need) {   // PV(x) completes barrier B_PV + (x & 1) for the (x >> 1)-th time
            while (ok && pv_seen <= need) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_PV + (pv_seen & 1)), (uint32_t)(pv_seen >> 1) & 1u,
                                                       abort_flag));
                ++pv_seen;
            }
        };
        for (int k = 0; ok; ++k) {
            const int i = snake_entry(k);
            if (i >= n_items) break;
            const int n_kt = attn_item(p, i, TK, b, j, cu0, len, t0, s0, kv_len);
            if (n_kt == 0) continue;
            const bool row_ok = t0 + tl < len;
            const int qpos = s0 + t0 + tl;
            const int ob = it % OB;
            const uint32_t tO = lane_base + 2 * TK + (uint32_t)(ob * 128);
            float m = -INFINITY, l = 0.f;
            for (int t = 0; t < n_kt && ok; ++t) {
                const int gt = g + t;
                const int sb = gt & 1;
                ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SF + sb), (uint32_t)(gt >> 1) & 1u, abort_flag));
                if (!ok) break;
                tc_fence_after();
                float sv[TK];
#pragma unroll
                for (int c0 = 0; c0 < TK; c0 += 32) {
                    float a[32];
                    tmem_ld32(lane_base + sb * TK + c0, a);
#pragma unroll
                    for (int q = 0; q < 32; ++q) sv[c0 + q] = a[q];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_SFREE + sb));   // S buffer may be reused
                const int j0 = t * TK;
                // causal / length mask only where this tile reaches past a row's position or the
                // keys' end (the item's first row has the smallest position, s0 + t0)
                if (j0 + TK > s0 + t0 + 1 || j0 + TK > kv_len) {
#pragma unroll
                    for (int q = 0; q < TK; ++q) {
                        const int key = j0 + q;
                        if (key > qpos || key >= kv_len) sv[q] = -INFINITY;
                    }
                }
                // row max in four independent chains (max is exact in any order), in log2 units
                float mx4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
                for (int q = 4; q < TK; ++q) mx4[q & 3] = fmaxf(mx4[q & 3], sv[q]);
                const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
                // Lazy reference max: it moves (and O is rescaled) only when this tile's max exceeds it
                // by more than kLazyLog2, so p = 2^(s * scale - mref) <= 2^kLazyLog2.  O / l is
                // unchanged; the softmax of tile t then waits only for PV(t - 2), not PV(t - 1).
                const float mn = mx > m + kLazyLog2 ? mx : m;
                const float mref = mn == -INFINITY ? 0.f : mn;
                const float alpha = exp2f(m - mref);   // exactly 1 while the reference stays
                // p = 2^(s * scale - mref) (one rounding of the exponent), summed in four chains
                float rs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < TK; ++q) {
                    sv[q] = exp2f(fmaf(sv[q], p.scale_log2, -mref));
                    rs4[q & 3] += sv[q];
                }
                l = l * alpha + ((rs4[0] + rs4[1]) + (rs4[2] + rs4[3]));
                m = mn;
                // P buffer gt & 1 was last read by PV(gt - 2); O needs PV(gt - 1) done only when it is
                // rescaled
                const bool rescale = t > 0 && !__all_sync(0xffffffffu, alpha == 1.f);
                wait_pv(rescale ? gt - 1 : gt - 2);
                if (!ok) break;
                tc_fence_after();
                if (rescale) {
#pragma unroll 1
                    for (int c = 0; c < HD; c += 32) {
                        float o[32];
                        tmem_ld32(tO + c, o);
#pragma unroll
                        for (int q = 0; q < 32; ++q) o[q] *= alpha;
                        tmem_st32(tO + c, o);
                    }
                }
                // the item's last tile: zero the V rows of slots past the valid keys (stale cache)
                const int valid_in_tile = kv_len - j0;
                if (valid_in_tile < TK) {
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_VF + gt % NS), (uint32_t)(gt / NS) & 1u, abort_flag));
                    if (!ok) break;
                    const int z_rows = TK - valid_in_tile;
                    uint8_t* vt = smem + C::OFF_V + (gt % NS) * C::K_BYTES;
                    for (int idx = r; idx < C::NSUB * z_rows * 8; idx += TROWS) {
                        const int h = idx / (z_rows * 8), rem = idx - h * z_rows * 8;
                        const int row = valid_in_tile + rem / 8, chunk = rem & 7;
                        *reinterpret_cast<uint4*>(vt + h * C::KV_SUB + row * 128 + ((chunk ^ (row & 7)) << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                // P as bf16 hi + lo, K-major: 128-byte rows (TK 64) with chunk c of row r at c ^ (r & 7),
                // or 64-byte rows (TK 32) with chunk c at c ^ ((r >> 1) & 3)
                {
                    uint8_t* ph = smem + C::OFF_P + 2 * (gt & 1) * C::P_BYTES + r * C::P_ROW;
                    uint8_t* pl = ph + C::P_BYTES;
#pragma unroll
                    for (int c = 0; c < TK / 8; ++c) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // hi = the top 16 bits (p truncated to bf16), lo = bf16(p - hi): p - hi is exact
                            const uint32_t u0 = __float_as_uint(sv[c * 8 + 2 * e]) & 0xFFFF0000u;
                            const uint32_t u1 = __float_as_uint(sv[c * 8 + 2 * e + 1]) & 0xFFFF0000u;
                            hw[e] = (u0 >> 16) | u1;
                            lw[e] = pack_bf2(sv[c * 8 + 2 * e] - __uint_as_float(u0),
                                             sv[c * 8 + 2 * e + 1] - __uint_as_float(u1));
                        }
                        const int off = (TK == 64 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3))) << 4;
                        *reinterpret_cast<uint4*>(ph + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        *reinterpret_cast<uint4*>(pl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                }
                fence_proxy_async_smem();   // generic-proxy writes (P, zeroed V rows) before the MMA reads them
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_PF + (gt & 1)));
            }
            // the item's output: O / l once its last PV is done
            wait_pv(g + n_kt - 1);
            if (!ok) break;
            tc_fence_after();
            const float il = 1.0f / l;
            bf16* dst = p.out + ((long long)(cu0 + t0 + tl) * p.nq + (long long)j * p.G + hg) * HD;
#pragma unroll 1
            for (int c = 0; c < HD; c += 32) {
                float o[32];
                tmem_ld32(tO + c, o);
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 32; e += 16) {
                        float f[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q) f[q] = o[e + q] * il;
                        if (p.v8) {
                            st_global_32(dst + c + e, pack8(f), pack8(f + 8));
                        } else {
                            *reinterpret_cast<uint4*>(dst + c + e) = pack8(f);
                            *reinterpret_cast<uint4*>(dst + c + e + 8) = pack8(f + 8);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_OF + ob));   // O buffer free for item it + OB
            g += n_kt;
            ++it;
        }
        if (!ok) {
            *abort_flag = 1;
            raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
        }
    }

    // ---------------- teardown: on abort, let every issued TMA load and MMA land first
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && warp == 0 && lane < 2) {
        volatile int never = 0;
        if (lane == 0) {
            const int qi = reinterpret_cast<volatile int*>(slots)[4];
            if (qi > 0) (void)mbar_wait(bar(C::B_QF), (uint32_t)(qi - 1) & 1u, &never);
        }
        const int issued = reinterpret_cast<volatile int*>(slots)[2 + lane];
        const int full0 = lane == 0 ? C::B_KF : C::B_VF;
        for (int t = max(0, issued - NS); t < issued; ++t)
            (void)mbar_wait(bar(full0 + t % NS), (uint32_t)(t / NS) & 1u, &never);
    }
    if (warp == 1 && lane == 0) {
        volatile int never = 0;
        (void)mbar_wait(bar(C::B_IDLE), 0u, &never);
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int HD, int TK, int NS, int OB>
cudaError_t launch_tc_cfg(const PrefillAttnArgs& a, cudaStream_t st) {
    using C = AttnCfg<HD, TK, NS, OB>;
    constexpr int kCtasPerSm = TK == 32 ? 2 : 1;
    const int G = a.nq / a.nkv;
    const int QT = TROWS / G;
    alignas(64) CUtensorMap mq, mkv;
    // q [T, nq, hd] as (hd, nq, T); one box = 64 dims x G heads x QT positions (zero past T)
    const uint64_t qdims[3] = {(uint64_t)HD, (uint64_t)a.nq, (uint64_t)a.total_rows};
    const uint64_t qstr[2] = {(uint64_t)HD * 2, (uint64_t)a.nq * HD * 2};
    const uint32_t qbox[3] = {64u, (uint32_t)G, (uint32_t)QT};
    if (!encode_tensor_map(&mq, 3, a.q, qdims, qstr, qbox)) return cudaErrorInvalidValue;
    // the layer's cache as rows of hd: [cache_batch * 2 * nkv * n_slots, hd]; box 64 dims x TK keys
    const uint64_t kvdims[2] = {(uint64_t)HD, (uint64_t)a.cache_batch * 2 * a.nkv * a.n_slots};
    const uint64_t kvstr[1] = {(uint64_t)HD * 2};
    const uint32_t kvbox[2] = {64u, (uint32_t)TK};
    if (!encode_tensor_map(&mkv, 2, a.kv_layer, kvdims, kvstr, kvbox)) return cudaErrorInvalidValue;
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(prefill_attn_tc_kernel<HD, TK, NS, OB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    TcAttnArgs p{};
    p.cu = a.cu;
    p.start = a.start;
    p.out = a.out;
    p.err = a.err;
    p.batch = a.batch;
    p.max_len = a.max_len;
    p.n_slots = a.n_slots;
    p.nq = a.nq;
    p.nkv = a.nkv;
    p.G = G;
    p.QT = QT;
    p.kv_rows_per_seq = 2LL * a.nkv * a.n_slots;
    p.scale_log2 = (1.0f / sqrtf((float)HD)) * kLog2e;
    p.sched = a.sched;
    p.v8 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0 ? 1 : 0;   // rows (nq hd bf16) and heads are 32-byte multiples
    const long long items = (long long)((a.max_len + QT - 1) / QT) * a.nkv * a.batch;
    const int grid = (int)std::min<long long>(items, (long long)device_sm_count() * kCtasPerSm);
    HRA_LAUNCH((prefill_attn_tc_kernel<HD, TK, NS, OB>), dim3(grid), dim3(kTcThreads), C::SMEM, st, mq, mkv, p);
    return cudaGetLastError();
}

// The two-CTAs-per-SM configuration is the one launched: measured on the 36-layer ragged batch
// (53 against 61 us per layer) and on 4 prompts of 1024-2048 tokens (422 against 438 us per
// layer) it beats <64, 3, 2>.
template <int HD>
cudaError_t launch_tc_hd(const PrefillAttnArgs& a, cudaStream_t st) {
    return launch_tc_cfg<HD, kLaunchedTK, 2, 1>(a, st);
}

}  // namespace

size_t attention_schedule_bytes(int rows, int batch) {
    // pairs <= sum_b ceil(len_b / QT) <= rows / QT + batch, QT >= 16; a 32-byte record each after
    // a 32-byte head holding the count
    return ((size_t)rows / 16 + (size_t)batch + 2) * 8 * sizeof(int32_t);
}

cudaError_t launch_attention_schedule(const int32_t* cu, const int32_t* start, int batch, int max_len, int nq,
                                      int nkv, int32_t* sched, cudaStream_t st) {
    const int G = nkv > 0 ? nq / nkv : 0;
    if ((G != 1 && G != 2 && G != 4 && G != 8) || batch < 1 || batch > 65535 || sched == nullptr)
        return cudaErrorInvalidValue;
    const int QT = TROWS / G;
    const int n_qt = (max_len + QT - 1) / QT;
    HRA_LAUNCH(attn_schedule_kernel, dim3(1), dim3(1024), 0, st, cu, start, batch, n_qt, QT, kLaunchedTK, sched);
    return cudaGetLastError();
}

cudaError_t launch_prefill_attention_tc(const PrefillAttnArgs& a, cudaStream_t st) {
    const int G = a.nkv > 0 ? a.nq / a.nkv : 0;
    if (G != 1 && G != 2 && G != 4 && G != 8) return cudaErrorInvalidValue;
    if (a.sched == nullptr && a.batch != 1) return cudaErrorInvalidValue;
    if (a.hd == 128) return launch_tc_hd<128>(a, st);
    if (a.hd == 64) return launch_tc_hd<64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace hra
