// codebook.cu -- finalize of the per-frame delayed-codebook step.
//
// One CTA per (codebook, row) sums the audio-head logit partials (split order) and takes the argmax
// (lowest index on ties) after adding the optional EOC bias; the K CTAs of a row form a thread-block
// cluster, whose rank 0 runs the delay-pattern state machine, after which every CTA writes 1/K of
// next = bf16(sum over k ascending of fp32 code_emb[k][code_k]) with 16-byte loads.  Source: "Stabilize Higgs Audio termination and prefill" (FlashRT PR #141),
// Summary (one shared helper takes the per-frame argmax, applies the delays and sums the codebook
// embeddings) and Root cause
// (EOC on any codebook must end the stream, not only on the first).
//
// The sampled variant (codebook_sample_kernel, one CTA per (codebook, row)) replaces the argmax with
// temperature / top-k / top-p sampling by an exponential race on per-row seeded Philox noise; the
// last of a row's CTAs to finish runs the same per-row tail.
//
// Delay rule per row (t = frame, e = eoc_frame, codebook k lags k frames):
//   t < k -> BOS; e >= 0 and t - k >= e -> EOC; otherwise argmax.  If e < 0 and an argmaxed
//   codebook chose EOC, e = min over those k of (t - k) and every codebook with t >= k and
//   t - k >= e emits EOC in this frame.  done |= e >= 0 and t >= e + K - 1; t += 1.
#include <limits.h>
#include <math.h>

#include "internal.h"

namespace hra {

namespace {

constexpr int kMaxCodebooks = 16;
constexpr int kMaxSplits = 8;   // the audio-head GEMM splits K at most 8 ways

__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

// The per-row tail once all K candidates of row b are known (in shared memory `s_cand`, or else in
// cand[b][*], written by other CTAs), with st = the row's state as read before any CTA of this step
// could advance it: the delay state machine on the K candidates, then
// next = bf16(sum_k fp32 code_emb[k][code_k]), k ascending.
template <int J>
__device__ void finish_row(const CodebookArgs& a, int b, int tid, int nthreads, int* s_code, const int* s_cand,
                           int4 st) {
    if (tid == 0) {
        int am[kMaxCodebooks];   // the K candidates, all requested at once (from L2 when in cand[])
#pragma unroll
        for (int kk = 0; kk < kMaxCodebooks; ++kk)
            if (kk < a.K) am[kk] = s_cand ? s_cand[kk] : __ldcg(a.cand + b * a.K + kk);
        const int t = st.x;
        int e = st.y, done = st.z;
        bool forced[kMaxCodebooks];
        int code[kMaxCodebooks];
        for (int kk = 0; kk < a.K; ++kk) {
            if (t < kk) {
                code[kk] = a.bos;
                forced[kk] = true;
            } else if (e >= 0 && t - kk >= e) {
                code[kk] = a.eoc;
                forced[kk] = true;
            } else {
                code[kk] = am[kk];
                forced[kk] = false;
            }
        }
    if (e < 0) {
            int cand = INT_MAX;
            for (int kk = 0; kk < a.K; ++kk)
                if (!forced[kk] && code[kk] == a.eoc && t - kk < cand) cand = t - kk;
            if (cand != INT_MAX) {
                e = cand;
                for (int kk = 0; kk < a.K; ++kk)
                    if (t >= kk && t - kk >= e) code[kk] = a.eoc;
            }
        }
        if (e >= 0 && t >= e + a.K - 1) done = 1;
        for (int kk = 0; kk < a.K; ++kk) {
            s_code[kk] = code[kk];
            a.codes[b * a.K + kk] = code[kk];
        }
        a.state[b] = make_int4(t + 1, e, done, 0);
        a.done[b] = done;
    }
    __syncthreads();

    // next = bf16(sum_k fp32(code_emb[k][code_k])), k ascending
    const int nc = a.H >> 3;
    for (int c0 = tid; c0 < nc; c0 += J * nthreads) {
        // J 8-column chunks per thread and eight rows at a time: 8 J rows requested before the
        // first is added
        float acc[J][8];
#pragma unroll
        for (int j = 0; j < J; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] = 0.f;
        for (int k0 = 0; k0 < a.K; k0 += 8) {
            uint4 u[J][8];
#pragma unroll
            for (int j = 0; j < J; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = c0 + j * nthreads;
                    if (k0 + i < a.K && c < nc)
                        u[j][i] = reinterpret_cast<const uint4*>(
                            a.code_emb + ((long long)(k0 + i) * a.Vc + s_code[k0 + i]) * a.H)[c];
                }
#pragma unroll
            for (int j = 0; j < J; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (k0 + i < a.K && c0 + j * nthreads < nc) {
                        float f[8];
                        unpack8(u[j][i], f);
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[j][q] += f[q];
                    }
                }
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int c = c0 + j * nthreads;
            if (c < nc) reinterpret_cast<uint4*>(a.next_emb + (long long)b * a.H)[c] = pack8(acc[j]);
        }
    }
}

// Thread-block cluster helpers: the K CTAs of a row form one cluster and exchange the K argmax
// results and the codes through distributed shared memory, with hardware cluster barriers.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of `p` (this CTA's variable) in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_cluster(uint32_t addr) {
    int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Cluster of K CTAs per row b; CTA k (cluster rank k) takes codebook k.  Its logits are the split
// partials summed in split order (all of a thread's partials are requested before the first is
// added); the argmax (lowest index on ties, EOC bias included) goes into rank 0's shared memory.
// After a cluster barrier rank 0 runs the delay state machine and writes the codes, state and done;
// after a second barrier every CTA reads the codes from rank 0 and gathers 1/K of the hidden columns
// of next = bf16(sum_k fp32 code_emb[k][code_k]), k ascending.  No global atomics, fences or
// hand-offs through memory: spreading a row over K CTAs keeps each CTA's share of the partials
// small, and the cluster keeps the row's tail on chip.
constexpr int kFinThreads = 256;
constexpr int kFinPer = 5;   // entries per thread in one pass (codebook_size <= 1280 in one pass)
__global__ void __launch_bounds__(kFinThreads, 4) codebook_finalize_kernel(const CodebookArgs a) {
    pdl_launch();
    pdl_wait();
    __shared__ float s_bv[kFinThreads / 32];
    __shared__ int s_bi[kFinThreads / 32];
    __shared__ int s_am[kMaxCodebooks];     // rank 0: argmax of every codebook
    __shared__ int s_code[kMaxCodebooks];   // rank 0: the codes; elsewhere: a copy
    const int k = (int)cluster_rank(), b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KV = a.K * a.Vc;
    const long long split_stride = (long long)a.batch * KV;
    const float* base = a.partial + (long long)b * KV + (long long)k * a.Vc;
    const float bias = a.eoc_bias ? a.eoc_bias[b * a.K + k] : 0.f;
    const int4 st = k == 0 ? a.state[b] : make_int4(0, 0, 0, 0);

    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int v0 = 0; v0 < a.Vc; v0 += kFinThreads * kFinPer) {
        float x[kFinPer];
#pragma unroll
        for (int i = 0; i < kFinPer; ++i) x[i] = 0.f;
        for (int s0 = 0; s0 < a.splits; s0 += 4) {
            float part[4][kFinPer];
#pragma unroll
            for (int h = 0; h < 4; ++h)
#pragma unroll
                for (int i = 0; i < kFinPer; ++i) {
                    const int v = v0 + tid + i * kFinThreads;
                    part[h][i] = (s0 + h < a.splits && v < a.Vc) ? base[(s0 + h) * split_stride + v] : 0.f;
                }
#pragma unroll
            for (int h = 0; h < 4; ++h)
#pragma unroll
                for (int i = 0; i < kFinPer; ++i)
                    if (s0 + h < a.splits) x[i] += part[h][i];
        }
#pragma unroll
        for (int i = 0; i < kFinPer; ++i) {
            const int v = v0 + tid + i * kFinThreads;
            if (v < a.Vc) {
                if (a.logits_out) a.logits_out[((long long)b * a.K + k) * a.Vc + v] = x[i];
                const float y = (v == a.eoc && a.eoc_bias) ? x[i] + bias : x[i];
                better(bv, bi, y, v);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        better(bv, bi, ov, oi);
    }
    if (lane == 0) {
        s_bv[warp] = bv;
        s_bi[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
        float fv = s_bv[0];
        int fi = s_bi[0];
        for (int w = 1; w < kFinThreads / 32; ++w) better(fv, fi, s_bv[w], s_bi[w]);
        if (fi < 0 || fi >= a.Vc) {   // only when every logit was NaN
            raise_error(a.err, HRA_DEVERR_CODE_RANGE);
            fi = 0;
        }
        st_cluster(cluster_addr(&s_am[k], 0), fi);
    }
    cluster_sync();
    if (k == 0 && tid == 0) {
        const int t = st.x;
        int e = st.y, done = st.z;
        bool forced[kMaxCodebooks];
        int code[kMaxCodebooks];
        for (int kk = 0; kk < a.K; ++kk) {
            if (t < kk) {
                code[kk] = a.bos;
                forced[kk] = true;
            } else if (e >= 0 && t - kk >= e) {
                code[kk] = a.eoc;
                forced[kk] = true;
            } else {
                code[kk] = s_am[kk];
                forced[kk] = false;
            }
        }
        if (e < 0) {
            int cand = INT_MAX;
            for (int kk = 0; kk < a.K; ++kk)
                if (!forced[kk] && code[kk] == a.eoc && t - kk < cand) cand = t - kk;
            if (cand != INT_MAX) {
                e = cand;
                for (int kk = 0; kk < a.K; ++kk)
                    if (t >= kk && t - kk >= e) code[kk] = a.eoc;
            }
        }
        if (e >= 0 && t >= e + a.K - 1) done = 1;
        for (int kk = 0; kk < a.K; ++kk) {
            s_code[kk] = code[kk];
            a.codes[b * a.K + kk] = code[kk];
        }
        a.state[b] = make_int4(t + 1, e, done, 0);
        a.done[b] = done;
    }
    cluster_sync();
    if (k != 0 && tid < a.K) s_code[tid] = ld_cluster(cluster_addr(&s_code[tid], 0));
    cluster_sync();   // rank 0's shared memory is not read after this point
    // this CTA's share of the hidden columns: chunks [c0, c1) of 8 columns
    const int nc = a.H >> 3;
    const int per = (nc + a.K - 1) / a.K;
    const int c0 = k * per, c1 = min(nc, c0 + per);
    for (int c = c0 + tid; c < c1; c += kFinThreads) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; k0 < a.K; k0 += 8) {
            uint4 u[8];   // eight rows requested before the first is added
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (k0 + i < a.K)
                    u[i] = reinterpret_cast<const uint4*>(a.code_emb +
                                                          ((long long)(k0 + i) * a.Vc + s_code[k0 + i]) * a.H)[c];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (k0 + i < a.K) {
                    float f[8];
                    unpack8(u[i], f);
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[q] += f[q];
                }
            }
        }
        reinterpret_cast<uint4*>(a.next_emb + (long long)b * a.H)[c] = pack8(acc);
    }
}

// ------------------------------------------------------------------ sampled step
//
// Sampling rule (vLLM-Omni PR #8226, Purpose and Test Plan: temperature / top-k / top-p with
// per-request seeded exponential noise): z_v = (logit_v (+ EOC bias)) / T; order the entries by z
// descending, ties by ascending index; top-k keeps every entry at or above the top_k-th largest z;
// top-p keeps an entry while the probability of the kept entries before it is below top_p; the
// sample is the kept entry whose exponential clock E_v / exp(z_v - z_max) rings first (lowest
// index on ties).  E_v = -log(u), u = (word >> 8 + 1) / 2^24 in (0, 1] from Philox4x32-10 at
// counter (v >> 2, k, frame, 0) under the row's 64-bit seed, word v & 3.

constexpr int kSampleThreads = 1024;
constexpr int kSortN = 2048;   // entries sorted per codebook (codebook_size <= kSortN)
constexpr int kFastKeep = 256; // top-k sets up to this size are sorted alone (no full sort)

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC 2011): ten rounds of (c0, c1, c2, c3) <- (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1,
// lo(M0 c0)), the key bumped by the Weyl constants between rounds.  Returns output word `word`.
__device__ __forceinline__ uint32_t philox_word(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, int word) {
    uint32_t x0 = c0, x1 = c1, x2 = c2, x3 = 0u;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, x0), lo0 = 0xD2511F53u * x0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, x2), lo1 = 0xCD9E8D57u * x2;
        const uint32_t n0 = hi1 ^ x1 ^ k0, n2 = hi0 ^ x3 ^ k1;
        x0 = n0;
        x1 = lo1;
        x2 = n2;
        x3 = lo0;
    }
    return word == 0 ? x0 : word == 1 ? x1 : word == 2 ? x2 : x3;
}

// Order-preserving map of a float to a uint32 (and back).
__device__ __forceinline__ uint32_t sortable(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unsortable(uint32_t s) {
    return __uint_as_float((s & 0x80000000u) ? (s & 0x7fffffffu) : ~s);
}
// Sort key: ascending keys = z descending, then index ascending.
__device__ __forceinline__ float key_z(unsigned long long key) { return unsortable(~(uint32_t)(key >> 32)); }
__device__ __forceinline__ int key_v(unsigned long long key) { return (int)(uint32_t)key; }

__device__ __forceinline__ float block_sum_1024(float x, float* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    x = warp_sum(x);
    __syncthreads();
    if (lane == 0) s_red[warp] = x;
    __syncthreads();
    float y = s_red[lane];
    y = warp_sum(y);
    return y;
}

// CTA (k, b) with 1024 threads: the sampled choice of codebook k of row b goes to cand[b][k]; the
// row's last CTA then runs the same state machine and embedding sum as the greedy step.
__global__ void __launch_bounds__(kSampleThreads) codebook_sample_kernel(const CodebookArgs a) {
    pdl_launch();
    pdl_wait();
    const int k = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ unsigned long long s_key[kSortN];
    __shared__ unsigned long long s_list[kFastKeep];
    __shared__ unsigned int s_hist[256];
    __shared__ int s_sel[2];
    __shared__ int s_cnt;
    __shared__ float s_red[32];
    __shared__ int s_redi[32];
    __shared__ int s_last;
    __shared__ int s_code[kMaxCodebooks];
    const int KV = a.K * a.Vc;
    const long long split_stride = (long long)a.batch * KV;
    const float* base = a.partial + (long long)b * KV + (long long)k * a.Vc;
    const float bias = a.eoc_bias ? a.eoc_bias[b * a.K + k] : 0.f;
    const int4 st0 = a.state[b];      // read before the row's last CTA advances the state
    const int frame = st0.x;
    const uint64_t seed = a.seeds[b];

    // z and the sort keys: ascending keys = z descending, then index ascending (padding sorts last)
    uint32_t mine[2] = {0u, 0u};   // order-preserving bits of z of entries tid, tid + 1024 (0: none)
    float xs[2] = {0.f, 0.f};      // the two entries' logits: all partials requested before any is added
    for (int s0 = 0; s0 < a.splits; s0 += 4) {
        float part[4][2];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = tid + h * kSampleThreads;
                part[q][h] = (s0 + q < a.splits && v < a.Vc) ? base[(s0 + q) * split_stride + v] : 0.f;
            }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (s0 + q < a.splits) xs[h] += part[q][h];
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int v = tid + h * kSampleThreads;
        unsigned long long key = ~0ull;
        if (v < a.Vc) {
            float x = xs[h];
            if (a.logits_out) a.logits_out[((long long)b * a.K + k) * a.Vc + v] = x;
            if (v == a.eoc && a.eoc_bias) x = x + bias;
            float z = x / a.temperature;
            if (z != z) z = -INFINITY;
            if (z == 0.f) z = 0.f;   // -0 sorts with +0 (equal values tie on the index)
            mine[h] = sortable(z);
            key = ((unsigned long long)(~mine[h]) << 32) | (uint32_t)v;
        }
        s_key[v] = key;
    }
    __syncthreads();
    // Top-k without sorting every entry: select the top_k-th largest z by its bits, eight at a time
    // (a 256-bin histogram of the entries that match the bits chosen so far), keep every entry at
    // or above it, and sort only those.  The kept prefix is then exactly the one a full sort gives.
    // Top-k off, or more than kFastKeep entries at or above the threshold: the full sort below.
    bool sorted = false;
    if (a.top_k > 0 && a.top_k < a.Vc) {
        uint32_t prefix = 0u, pmask = 0u;
        int need = a.top_k;
        for (int shift = 24; shift >= 0; shift -= 8) {
            if (tid < 256) s_hist[tid] = 0u;
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (mine[h] != 0u && (mine[h] & pmask) == prefix) atomicAdd(&s_hist[(mine[h] >> shift) & 255u], 1u);
            __syncthreads();
            if (warp == 0) {
                // lane l holds bins 8l .. 8l + 7; `above` = entries in the bins above a bin
                unsigned int c[8], tot = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    c[i] = s_hist[8 * lane + i];
                    tot += c[i];
                }
                unsigned int suf = tot;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned int y = __shfl_down_sync(0xffffffffu, suf, o);
                    if (lane + o < 32) suf += y;
                }
                unsigned int above = suf - tot;
#pragma unroll
                for (int i = 7; i >= 0; --i) {
                    if (above < (unsigned)need && (unsigned)need <= above + c[i]) {
                        s_sel[0] = 8 * lane + i;
                        s_sel[1] = need - (int)above;
                    }
                    above += c[i];
                }
            }
            __syncthreads();
            prefix |= (uint32_t)s_sel[0] << shift;
            pmask |= 255u << shift;
            need = s_sel[1];
        }
        const int n_keep = __syncthreads_count(mine[0] >= prefix) + __syncthreads_count(mine[1] >= prefix);
        if (n_keep <= kFastKeep) {
            if (tid == 0) s_cnt = 0;
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (mine[h] >= prefix)
                    s_list[atomicAdd(&s_cnt, 1)] =
                        ((unsigned long long)(~mine[h]) << 32) | (uint32_t)(tid + h * kSampleThreads);
            __syncthreads();
            s_key[tid] = ~0ull;
            s_key[tid + kSampleThreads] = ~0ull;
            __syncthreads();
            if (tid < n_keep) {
                const unsigned long long me = s_list[tid];
                int rank = 0;
                for (int j = 0; j < n_keep; ++j) rank += s_list[j] < me ? 1 : 0;
                s_key[rank] = me;
            }
            __syncthreads();
            sorted = true;
        }
    }
    if (!sorted) {
        // bitonic sort, ascending keys; thread t compares the pair (i, i + stride)
        for (int size = 2; size <= kSortN; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                const int i = 2 * tid - (tid & (stride - 1));
                const int j = i + stride;
                const bool up = (i & size) == 0;
                const unsigned long long x = s_key[i], y = s_key[j];
                if ((x > y) == up) {
                    s_key[i] = y;
                    s_key[j] = x;
                }
                __syncthreads();
            }
        }
    }
    const float z0 = key_z(s_key[0]);
    const int i0 = 2 * tid, i1 = i0 + 1;   // this thread's sorted positions
    // top-k: every entry at or above the top_k-th largest z (a prefix of the sorted order)
    int n = a.Vc;
    if (a.top_k > 0 && a.top_k < a.Vc) {
        const float zk = key_z(s_key[a.top_k - 1]);
        const int c0 = __syncthreads_count(i0 >= a.top_k && i0 < a.Vc && key_z(s_key[i0]) >= zk);
        const int c1 = __syncthreads_count(i1 >= a.top_k && i1 < a.Vc && key_z(s_key[i1]) >= zk);
        n = a.top_k + c0 + c1;
    }
    const bool valid = z0 > -INFINITY;
    float q0 = i0 < n && valid ? expf(key_z(s_key[i0]) - z0) : 0.f;
    float q1 = i1 < n && valid ? expf(key_z(s_key[i1]) - z0) : 0.f;
    bool keep0 = i0 < n, keep1 = i1 < n;
    if (a.top_p < 1.f) {
        // exclusive prefix of p = q / S over the sorted order
        const float S = block_sum_1024(q0 + q1, s_red);
        const float p0 = q0 / S, p1 = q1 / S;
        const float mine = p0 + p1;
        float incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncthreads();
        if (lane == 31) s_red[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            float w = s_red[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            s_red[lane] = w;   // inclusive prefix of the warp totals
        }
        __syncthreads();
        const float before = (warp > 0 ? s_red[warp - 1] : 0.f) + incl - mine;
        keep0 = keep0 && (i0 == 0 || before < a.top_p);
        keep1 = keep1 && (before + p0 < a.top_p);
    }
    // the exponential race over the kept entries
    float bt = INFINITY;
    int bv = INT_MAX;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const bool keep = h == 0 ? keep0 : keep1;
        const float q = h == 0 ? q0 : q1;
        if (keep && q > 0.f) {
            const int v = key_v(s_key[h == 0 ? i0 : i1]);
            const uint32_t w = philox_word(seed, (uint32_t)v >> 2, (uint32_t)k, (uint32_t)frame, v & 3);
            const float u = (float)((w >> 8) + 1u) * (1.0f / 16777216.0f);
            const float tv = -logf(u) / q;
            if (tv < bt || (tv == bt && v < bv)) {
                bt = tv;
                bv = v;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ot = __shfl_xor_sync(0xffffffffu, bt, o);
        const int ov = __shfl_xor_sync(0xffffffffu, bv, o);
        if (ot < bt || (ot == bt && ov < bv)) {
            bt = ot;
            bv = ov;
        }
    }
    __syncthreads();
    if (lane == 0) {
        s_red[warp] = bt;
        s_redi[warp] = bv;
    }
    __syncthreads();
    if (tid == 0) {
        float ft = s_red[0];
        int fv = s_redi[0];
        for (int w = 1; w < 32; ++w)
            if (s_red[w] < ft || (s_red[w] == ft && s_redi[w] < fv)) {
                ft = s_red[w];
                fv = s_redi[w];
            }
        if (fv < 0 || fv >= a.Vc) {   // every logit NaN or -inf
            raise_error(a.err, HRA_DEVERR_CODE_RANGE);
            fv = 0;
        }
        a.cand[b * a.K + k] = fv;
        __threadfence();
        s_last = atomicAdd(&a.counters[b], 1) == a.K - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    finish_row<1>(a, b, tid, kSampleThreads, s_code, nullptr, st0);
}

}  // namespace

cudaError_t launch_codebook_finalize(const CodebookArgs& a, cudaStream_t st) {
    if (a.K > kMaxCodebooks || a.splits > kMaxSplits) return cudaErrorInvalidValue;
    if (a.seeds != nullptr) {
        if (a.Vc > kSortN) return cudaErrorInvalidValue;
        HRA_LAUNCH(codebook_sample_kernel, dim3(a.K, a.batch), dim3(kSampleThreads), 0, st, a);
    } else {
        // one cluster of K CTAs per row (K <= 8 portable; up to 16 with the non-portable opt-in)
        static bool configured[64] = {false};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (a.K > 8 && (dev < 0 || dev >= 64 || !configured[dev])) {
            e = cudaFuncSetAttribute(codebook_finalize_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) configured[dev] = true;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(a.K, a.batch);
        cfg.blockDim = dim3(kFinThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = a.K;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        count_launches(1);
        e = cudaLaunchKernelEx(&cfg, codebook_finalize_kernel, a);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace hra
