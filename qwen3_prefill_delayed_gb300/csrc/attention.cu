// attention.cu -- causal GQA attention over the used keys of the KV cache.
//
// Semantics: row i of sequence b (position p_i) with q head h attends cache slots 0..p_i of kv head
// h / (n_q / n_kv) with softmax(q.k / sqrt(hd)); slots past the sequence's length carry zero
// weight and are never used ("flashrt-structures 0.2.0, prefill_tower/fp8_chain.py" page, its
// description: attention covers only the used keys, and since pads trail, a count of used keys
// stands for the mask; causal here because the backbone is a decoder).
//
// decode_attn_kernel   one query per row (decode pass, last prefill layer): the keys are split
//                      across CTAs and stream through a 3-stage cp.async ring; the G = n_q / n_kv
//                      q heads of a kv head are the rows of one MMA tile, so they share every K/V
//                      load; partial (m, l, o) go to scratch and a combine kernel merges the
//                      splits (skipped when a row takes one split).
#include <math.h>

#include "internal.h"

namespace hra {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Prefill (many queries per kv head) runs on the tensor-core kernel in attention_tc.cu.

// (a, b) -> bf16 pairs hi = bf16(a, b) and lo = bf16(a - hi_a, b - hi_b).
__device__ __forceinline__ void split_bf2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_bf2(a - hf.x, b - hf.y);
}
constexpr int PK = 64;    // keys per tile

template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    // byte offset of 16-byte chunk `chunk` of row `row` in a [rows][HD] bf16 tile
    return (uint32_t)(row * HD * 2 + ((chunk ^ (row & 7)) << 4));
}

// ROWS rows of HD bf16 into a swizzled tile, rows past rows_valid zero-filled (128 threads).
template <int HD, int ROWS = PK>
__device__ __forceinline__ void load_tile(uint32_t sbase, const bf16* gbase, long long row_stride, int rows_valid,
                                          int tid) {
    constexpr int CH = HD / 8;   // 16-byte chunks per row
    for (int idx = tid; idx < ROWS * CH; idx += 128) {
        const int r = idx / CH, c = idx % CH;
        const bool ok = r < rows_valid;
        const bf16* src = gbase + (ok ? (long long)r * row_stride + c * 8 : 0);
        cp_async16(sbase + swz<HD>(r, c), src, ok ? 16u : 0u);
    }
}

// ------------------------------------------------------------------ single-query decode

constexpr int DS = 3;     // K/V stages in flight per CTA

// One CTA = one (row, kv head, key split); 4 warps.  The split's keys stream through a ring of DS
// shared-memory stages of PK keys (coalesced cp.async, zero-filled past the last key).  The G q
// heads of the kv head are the rows of a 16-row MMA tile (rows G..15 are zero), so S = QK^T and
// O += PV run on the same m16n8k16 fragments as the prefill kernel.  Warp w owns keys
// w*16 .. w*16+15 of every stage and keeps its own online-softmax state; the four warps merge
// through shared memory at the end.
template <int HD, int G>
__global__ void __launch_bounds__(128) decode_attn_kernel(const DecodeAttnArgs a, float scale_log2) {
    static_assert(G <= 8, "the q heads of one kv head fill at most the upper half of the MMA tile");
    pdl_launch();
    pdl_wait();
    constexpr int KS = HD / 16;
    constexpr int DN = HD / 8;
    constexpr uint32_t TILE = PK * HD * 2;   // bytes of one K (or V) stage
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sQ = smem_u32(sm);
    const uint32_t sK0 = sQ + 16 * HD * 2;
    const uint32_t sV0 = sK0 + DS * TILE;

    const int i = blockIdx.z, j = blockIdx.y, sp = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qr = a.q_row ? a.q_row[i] : i;
    const int seq = a.seq[qr], pos = a.pos[qr];
    const int nkeys = pos + 1;
    const int per = (nkeys + a.splits - 1) / a.splits;
    const int chunk = (per + PK - 1) / PK * PK;
    const int k0 = sp * chunk, k1 = min(nkeys, k0 + chunk);
    const int n_t = k1 > k0 ? (k1 - k0 + PK - 1) / PK : 0;

    const long long hstride = (long long)a.n_slots * HD;
    const bf16* kbase = a.kv_layer + ((long long)(seq * 2) * a.nkv + j) * hstride + (long long)k0 * HD;
    const bf16* vbase = a.kv_layer + ((long long)(seq * 2 + 1) * a.nkv + j) * hstride + (long long)k0 * HD;
    const bf16* qbase = a.q + ((long long)qr * a.nq + j * G) * HD;

    // q rows 0..G-1 (the G heads), rows G..15 zero-filled
    for (int idx = tid; idx < 16 * (HD / 8); idx += 128) {
        const int r = idx / (HD / 8), c = idx % (HD / 8);
        const bool ok = r < G;
        cp_async16(sQ + swz<HD>(r, c), qbase + (ok ? (long long)r * HD + c * 8 : 0), ok ? 16u : 0u);
    }
#pragma unroll
    for (int t = 0; t < DS - 1; ++t) {
        if (t < n_t) {
            const int rv = min(PK, k1 - k0 - t * PK);
            load_tile<HD>(sK0 + t * TILE, kbase + (long long)t * PK * HD, HD, rv, tid);
            load_tile<HD>(sV0 + t * TILE, vbase + (long long)t * PK * HD, HD, rv, tid);
        }
        cp_async_commit();
    }

    uint32_t qf[KS][4];
    float o[DN][4];
#pragma unroll
    for (int d = 0; d < DN; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    float m_a = -INFINITY, l_a = 0.f;
    const int tig = lane & 3;

    for (int t = 0; t < n_t; ++t) {
        {
            const int tn = t + DS - 1;
            if (tn < n_t) {
                const int rv = min(PK, k1 - k0 - tn * PK);
                load_tile<HD>(sK0 + (tn % DS) * TILE, kbase + (long long)tn * PK * HD, HD, rv, tid);
                load_tile<HD>(sV0 + (tn % DS) * TILE, vbase + (long long)tn * PK * HD, HD, rv, tid);
            }
            cp_async_commit();
        }
        cp_async_wait<DS - 1>();
        __syncthreads();
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldmatrix_x4(qf[ks], sQ + swz<HD>(lane & 15, ks * 2 + (lane >> 4)));
        }
        const uint32_t sK = sK0 + (t % DS) * TILE;
        const uint32_t sV = sV0 + (t % DS) * TILE;
        const int kw = k0 + t * PK + warp * 16;   // first key of this warp's 16

        float s[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t kb[4];
            ldmatrix_x4(kb, sK + swz<HD>(warp * 16 + (lane & 7) + ((lane >> 4) << 3), ks * 2 + ((lane >> 3) & 1)));
            mma_bf16_16816(s[0], qf[ks], kb[0], kb[1]);
            mma_bf16_16816(s[1], qf[ks], kb[2], kb[3]);
        }
        // rows 8..15 are padding: their probabilities are zero.  Keys past k1 get zero weight.
        float mx = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int key = kw + n * 8 + 2 * tig + c;
                const float v = key < k1 ? s[n][c] * scale_log2 : -INFINITY;
                s[n][c] = v;
                mx = fmaxf(mx, v);
            }
            s[n][2] = s[n][3] = 0.f;
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m_a, mx);
        const float mref = mn == -INFINITY ? 0.f : mn;   // a warp with no key yet keeps p = 0
        const float al = exp2f(m_a - mref);
        m_a = mn;
        float rs = 0.f;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            s[n][0] = exp2f(s[n][0] - mref);
            s[n][1] = exp2f(s[n][1] - mref);
            rs += s[n][0] + s[n][1];
        }
        l_a = l_a * al + rs;
#pragma unroll
        for (int d = 0; d < DN; ++d) {
            o[d][0] *= al;
            o[d][1] *= al;
        }
        uint32_t ph[4], pl[4];
        split_bf2(s[0][0], s[0][1], ph[0], pl[0]);
        split_bf2(s[0][2], s[0][3], ph[1], pl[1]);
        split_bf2(s[1][0], s[1][1], ph[2], pl[2]);
        split_bf2(s[1][2], s[1][3], ph[3], pl[3]);
#pragma unroll
        for (int dp = 0; dp < DN / 2; ++dp) {
            uint32_t vb[4];
            ldmatrix_x4_trans(vb, sV + swz<HD>(warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), dp * 2 + (lane >> 4)));
            mma_bf16_16816(o[2 * dp], ph, vb[0], vb[1]);
            mma_bf16_16816(o[2 * dp + 1], ph, vb[2], vb[3]);
            mma_bf16_16816(o[2 * dp], pl, vb[0], vb[1]);
            mma_bf16_16816(o[2 * dp + 1], pl, vb[2], vb[3]);
        }
        __syncthreads();   // the stage is refilled by the next iteration's loads
    }
    cp_async_wait<0>();
    __syncthreads();

    // merge the four warps: per warp and head, (m, l) and the unnormalised o row
    float* s_o = reinterpret_cast<float*>(sm + 16 * HD * 2);   // [4][G][HD], over the stages
    float* s_ml = s_o + 4 * G * HD;                             // [4][G][2]
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    const int g = lane >> 2;
    if (g < G) {
        float* dst = s_o + (warp * G + g) * HD + 2 * tig;
#pragma unroll
        for (int d = 0; d < DN; ++d) {
            dst[d * 8] = o[d][0];
            dst[d * 8 + 1] = o[d][1];
        }
        if (tig == 0) {
            s_ml[(warp * G + g) * 2] = m_a;
            s_ml[(warp * G + g) * 2 + 1] = l_a;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < G * HD; idx += 128) {
        const int hg = idx / HD, dc = idx % HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w)
            if (s_ml[(w * G + hg) * 2 + 1] > 0.f) M = fmaxf(M, s_ml[(w * G + hg) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float lw = s_ml[(w * G + hg) * 2 + 1];
            if (lw > 0.f) {
                const float f = exp2f(s_ml[(w * G + hg) * 2] - M);
                L += lw * f;
                O += s_o[(w * G + hg) * HD + dc] * f;
            }
        }
        if (a.splits == 1) {
            a.out[((long long)i * a.nq + j * G + hg) * HD + dc] = f2bf(O / L);
        } else {
            float* dst = a.part + (((long long)sp * a.rows + i) * a.nq + j * G + hg) * (HD + 2);
            dst[dc] = O;
            if (dc == 0) {
                dst[HD] = M;
                dst[HD + 1] = L;
            }
        }
    }
}

template <int HD>
__global__ void decode_combine_kernel(const DecodeAttnArgs a) {
    pdl_launch();
    pdl_wait();
    const int i = blockIdx.y, h = blockIdx.x;
    const int stride = HD + 2;
    for (int d = threadIdx.x; d < HD; d += blockDim.x) {
        float M = -INFINITY;
        for (int s = 0; s < a.splits; ++s) {
            const float* p = a.part + (((long long)s * a.rows + i) * a.nq + h) * stride;
            if (p[HD + 1] > 0.f) M = fmaxf(M, p[HD]);
        }
        float L = 0.f, O = 0.f;
        for (int s = 0; s < a.splits; ++s) {
            const float* p = a.part + (((long long)s * a.rows + i) * a.nq + h) * stride;
            if (p[HD + 1] > 0.f) {
                const float f = exp2f(p[HD] - M);
                L += p[HD + 1] * f;
                O += p[d] * f;
            }
        }
        a.out[((long long)i * a.nq + h) * HD + d] = f2bf(O / L);
    }
}

template <int HD, int G>
cudaError_t launch_decode_hd(const DecodeAttnArgs& a, cudaStream_t st) {
    constexpr int smem = 16 * HD * 2 + 2 * DS * PK * HD * 2;
    static_assert(4 * G * HD * 4 + 4 * G * 2 * 4 <= 2 * DS * PK * HD * 2, "merge area fits over the stages");
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(decode_attn_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    dim3 grid(a.splits, a.nkv, a.rows);
    const float scale_log2 = (1.0f / sqrtf((float)HD)) * kLog2e;
    HRA_LAUNCH(decode_attn_kernel<HD, G>, dim3(grid), dim3(128), smem, st, a, scale_log2);
    if (a.splits == 1) return cudaSuccess;
    HRA_LAUNCH(decode_combine_kernel<HD>, dim3(dim3(a.nq, a.rows)), dim3(HD), 0, st, a);
    return cudaGetLastError();
}

template <int HD>
cudaError_t launch_decode_g(const DecodeAttnArgs& a, cudaStream_t st) {
    switch (a.nq / a.nkv) {
        case 1: return launch_decode_hd<HD, 1>(a, st);
        case 2: return launch_decode_hd<HD, 2>(a, st);
        case 4: return launch_decode_hd<HD, 4>(a, st);
        case 8: return launch_decode_hd<HD, 8>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// At most one wave of (row, kv head, split) CTAs (two per SM), with at least 128 keys per split:
// short rows take one split and skip the combine.
int decode_attention_splits(int rows, int nkv, int max_pos) {
    const int target = 2 * device_sm_count();
    int s = target / max(1, rows * nkv);
    s = min(s, (max_pos + 1) / 128);
    s = min(s, 32);
    return max(s, 1);
}

size_t decode_attention_scratch_bytes(int rows, int nq, int hd, int splits) {
    return (size_t)splits * rows * nq * (hd + 2) * sizeof(float);
}

cudaError_t launch_decode_attention(const DecodeAttnArgs& a, cudaStream_t st) {
    if (a.hd == 128) return launch_decode_g<128>(a, st);
    if (a.hd == 64) return launch_decode_g<64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace hra
