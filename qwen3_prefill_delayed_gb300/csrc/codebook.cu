// codebook.cu -- finalize of the per-frame delayed-codebook step.
//
// One CTA per (codebook, row) sums the audio-head logit partials (split order) and takes the argmax
// (lowest index on ties) after adding the optional EOC bias; the last CTA of each row runs the
// delay-pattern state machine and writes next = bf16(sum over k ascending of fp32
// code_emb[k][code_k]) with 16-byte loads.  Source: "Stabilize Higgs Audio termination and prefill" (FlashRT PR #141), Summary
// ("per-frame argmax, delay handling, and codebook embedding accumulation") and Root cause (EOC on
// any codebook must end the stream, not only on the first).
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
    for (int c = tid; c < nc; c += kThreads) {
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

}  // namespace

cudaError_t launch_codebook_finalize(const CodebookArgs& a, cudaStream_t st) {
    if (a.K > kMaxCodebooks || a.splits > kMaxSplits) return cudaErrorInvalidValue;
    HRA_LAUNCH(codebook_finalize_kernel, dim3(a.K, a.batch), dim3(kThreads), 0, st, a);
    return cudaGetLastError();
}

}  // namespace hra
