// codebook.cu -- finalize of the per-frame delayed-codebook step.
//
// One CTA per (codebook, row) sums the audio-head logit partials (split order) and takes the argmax
// (lowest index on ties) after adding the optional EOC bias; the last CTA of each row runs the
// delay-pattern state machine and writes next = bf16(sum over k ascending of fp32
// code_emb[k][code_k]) with 16-byte loads.  Source: "Stabilize Higgs Audio termination and prefill" (FlashRT PR #141), Summary
// ("per-frame argmax, delay handling, and codebook embedding accumulation") and Root cause (EOC on
// any codebook must end the stream, not only on the first).
//
// The sampled variant (codebook_sample_kernel) replaces the argmax with temperature / top-k /
// top-p sampling by an exponential race on per-row seeded Philox noise; the per-row tail is shared.
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
constexpr int kThreads = 256;
constexpr int kMaxSplits = 8;   // the audio-head GEMM splits K at most 8 ways

__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

// The last CTA of row b to finish (all K candidates are in cand[b][*]): the delay state machine on
// the K candidates, then next = bf16(sum_k fp32 code_emb[k][code_k]), k ascending.
__device__ void finish_row(const CodebookArgs& a, int b, int tid, int nthreads, int* s_code) {
    if (tid == 0) {
        const int4 st = a.state[b];
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
                code[kk] = reinterpret_cast<volatile int*>(a.cand)[b * a.K + kk];
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
    for (int c = tid; c < nc; c += nthreads) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int kk = 0; kk < a.K; ++kk) {
            const uint4 u = reinterpret_cast<const uint4*>(a.code_emb + ((long long)kk * a.Vc + s_code[kk]) * a.H)[c];
            float f[8];
            unpack8(u, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += f[j];
        }
        reinterpret_cast<uint4*>(a.next_emb + (long long)b * a.H)[c] = pack8(acc);
    }
}

// CTA (k, b): codebook k of row b.  The logits of that codebook are the split partials summed in
// split order; the argmax (lowest index on ties, EOC bias included) goes to cand[b][k].  The last of
// the row's K CTAs to finish (an atomic count, no waiting) runs the delay state machine on the K
// candidates and writes next = bf16(sum_k fp32 code_emb[k][code_k]), k ascending.
__global__ void __launch_bounds__(kThreads) codebook_finalize_kernel(const CodebookArgs a) {
    pdl_launch();
    pdl_wait();
    const int k = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KV = a.K * a.Vc;
    const long long split_stride = (long long)a.batch * KV;
    const float* base = a.partial + (long long)b * KV + (long long)k * a.Vc;
    const float bias = a.eoc_bias ? a.eoc_bias[b * a.K + k] : 0.f;

    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int v = tid; v < a.Vc; v += kThreads) {
        float part[kMaxSplits];
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) part[s] = s < a.splits ? base[s * split_stride + v] : 0.f;
        float x = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s)
            if (s < a.splits) x += part[s];
        if (a.logits_out) a.logits_out[((long long)b * a.K + k) * a.Vc + v] = x;
        if (v == a.eoc && a.eoc_bias) x = x + bias;
        better(bv, bi, x, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        better(bv, bi, ov, oi);
    }
    __shared__ float s_bv[kThreads / 32];
    __shared__ int s_bi[kThreads / 32];
    __shared__ int s_last;
    __shared__ int s_code[kMaxCodebooks];
    if (lane == 0) {
        s_bv[warp] = bv;
        s_bi[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
        float fv = s_bv[0];
        int fi = s_bi[0];
        for (int w = 1; w < kThreads / 32; ++w) better(fv, fi, s_bv[w], s_bi[w]);
        if (fi < 0 || fi >= a.Vc) {   // only when every logit was NaN
            raise_error(a.err, HRA_DEVERR_CODE_RANGE);
            fi = 0;
        }
        a.cand[b * a.K + k] = fi;
        __threadfence();
        s_last = atomicAdd(&a.counters[b], 1) == a.K - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    finish_row(a, b, tid, kThreads, s_code);
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
    __shared__ float s_red[32];
    __shared__ int s_redi[32];
    __shared__ int s_last;
    __shared__ int s_code[kMaxCodebooks];
    const int KV = a.K * a.Vc;
    const long long split_stride = (long long)a.batch * KV;
    const float* base = a.partial + (long long)b * KV + (long long)k * a.Vc;
    const float bias = a.eoc_bias ? a.eoc_bias[b * a.K + k] : 0.f;
    const int frame = a.state[b].x;   // read before the row's last CTA advances the state
    const uint64_t seed = a.seeds[b];

    // z and the sort keys (padding sorts last)
    for (int v = tid; v < kSortN; v += kSampleThreads) {
        unsigned long long key = ~0ull;
        if (v < a.Vc) {
            float x = 0.f;
            for (int sp = 0; sp < a.splits; ++sp) x += base[sp * split_stride + v];
            if (a.logits_out) a.logits_out[((long long)b * a.K + k) * a.Vc + v] = x;
            if (v == a.eoc && a.eoc_bias) x = x + bias;
            float z = x / a.temperature;
            if (z != z) z = -INFINITY;
            key = ((unsigned long long)(~sortable(z)) << 32) | (uint32_t)v;
        }
        s_key[v] = key;
    }
    __syncthreads();
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
    finish_row(a, b, tid, kSampleThreads, s_code);
}

}  // namespace

cudaError_t launch_codebook_finalize(const CodebookArgs& a, cudaStream_t st) {
    if (a.K > kMaxCodebooks || a.splits > kMaxSplits) return cudaErrorInvalidValue;
    if (a.seeds != nullptr) {
        if (a.Vc > kSortN) return cudaErrorInvalidValue;
        HRA_LAUNCH(codebook_sample_kernel, dim3(a.K, a.batch), dim3(kSampleThreads), 0, st, a);
    } else {
        HRA_LAUNCH(codebook_finalize_kernel, dim3(a.K, a.batch), dim3(kThreads), 0, st, a);
    }
    return cudaGetLastError();
}

}  // namespace hra
