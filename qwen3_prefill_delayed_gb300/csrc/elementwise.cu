// elementwise.cu -- bandwidth-bound kernels of the prefill / decode chain.
//
//   build_rowmap      packed-row bookkeeping (sequence + position of each row) from the host lengths
//   rope_table        cos/sin of pos * theta^(-2i/hd), evaluated in double, rounded to fp32
//   embed_rmsnorm     embedding gather fused with the first RMSNorm ("Stabilize Higgs Audio
//                     termination and prefill", Summary: embedding lookup)
//   rmsnorm           RMSNorm of rows (optionally gathered), or a plain row gather
//   qk_rope_kv        per-head q/k RMSNorm + rotate-half RoPE, q to scratch, K/V into the cache
//                     (half a warp per head)
//                     (same page: q/k norm, RoPE and the KV writes; the fp8_chain page: keys in
//                     the host rotate-half layout in the cache)
// One warp per row (a CTA per row for q/k/v heads); 16-byte vector loads; shuffle reductions.
#include <algorithm>

#include "internal.h"

namespace hra {

namespace {

__global__ void build_rowmap_kernel(const SeqMeta meta, int T, int32_t* row_seq, int32_t* row_pos,
                                    int32_t* cu, int32_t* last_row, int32_t* seq_start, unsigned int* err,
                                    unsigned int* zero_ptr, int zero_words) {
    pdl_launch();
    pdl_wait();
    if (err != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *err = 0u;   // first kernel of a call
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < zero_words; i += blockDim.x) zero_ptr[i] = 0u;
    __shared__ int32_t s_vals[kMaxBatch + 1];
    const int B = meta.batch;
    const int nvals = meta.mode == 0 ? B + 1 : B;
    for (int i = threadIdx.x; i < nvals; i += blockDim.x) s_vals[i] = meta.vals[i];
    __syncthreads();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (meta.mode == 0) {
        if (r < T) {
            int lo = 0, hi = B - 1;   // largest b with cu[b] <= r
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_vals[mid] <= r) lo = mid; else hi = mid - 1;
            }
            row_seq[r] = lo;
            row_pos[r] = meta.start[lo] + r - s_vals[lo];
        }
        if (blockIdx.x == 0)
            for (int b = threadIdx.x; b <= B; b += blockDim.x) {
                cu[b] = s_vals[b];
                if (b < B) {
                    last_row[b] = s_vals[b + 1] - 1;
                    if (seq_start != nullptr) seq_start[b] = meta.start[b];
                }
            }
    } else if (meta.mode == 2) {
        // one CTA (the launcher makes it so): the error word was cleared above, before the barrier
        for (int i = threadIdx.x; i < T; i += blockDim.x) {
            const int p = meta.pos_dev[i];
            int pc = p;
            if (p < 0 || p >= meta.n_slots) {
                raise_error(err, HRA_DEVERR_POS_RANGE);
                pc = p < 0 ? 0 : meta.n_slots - 1;
            }
            row_seq[i] = i;
            row_pos[i] = pc;
            if (meta.advance) meta.pos_dev[i] = p + 1;
        }
        for (int b = threadIdx.x; b < B; b += blockDim.x) {
            cu[b] = b;
            last_row[b] = b;
        }
    } else {
        if (r < T) {
            row_seq[r] = r;
            row_pos[r] = s_vals[r];
        }
        if (blockIdx.x == 0)
            for (int b = threadIdx.x; b < B; b += blockDim.x) {
                cu[b] = b;
                last_row[b] = b;
            }
    }
}

__global__ void rope_table_kernel(int n_rows, const int32_t* __restrict__ pos_of_row, int hd, double theta,
                                  float2* __restrict__ table) {
    pdl_launch();
    pdl_wait();
    const int half = hd / 2;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n_rows * half) return;
    const int i = idx / n_rows, r = idx % n_rows;   // transposed: entry (r, i) at i * n_rows + r
    const int pos = pos_of_row ? pos_of_row[r] : r;
    const double inv_freq = pow(theta, -(2.0 * (double)i) / (double)hd);
    double s, c;
    sincos((double)pos * inv_freq, &s, &c);
    table[idx] = make_float2((float)c, (float)s);
}

// Row RMSNorm: a warp holds its whole row in registers (NC 16-byte chunks per lane, H = 256 * NC),
// so every load of the row is in flight at once; NC = 0 takes H at run time in two passes.
template <int NC>
__device__ __forceinline__ void norm_row(const uint4* __restrict__ src, uint4* __restrict__ copy, int lane,
                                         const bf16* __restrict__ g, bf16* __restrict__ yrow, int H, float eps) {
    const uint4* gv = reinterpret_cast<const uint4*>(g);
    uint4* dy = reinterpret_cast<uint4*>(yrow);
    float ss = 0.f, sc = 0.f;
    if constexpr (NC > 0) {
        uint4 u[NC];
#pragma unroll
        for (int q = 0; q < NC; ++q) u[q] = src[lane + 32 * q];
#pragma unroll
        for (int q = 0; q < NC; ++q) {
            if (copy) copy[lane + 32 * q] = u[q];
            float f[8];
            unpack8(u[q], f);
#pragma unroll
            for (int j = 0; j < 8; ++j) csum_add(ss, sc, __fmul_rn(f[j], f[j]));
        }
        ss = csum_warp(ss, sc);
        if (g == nullptr) return;
        const float inv = 1.0f / sqrtf(ss / (float)H + eps);
#pragma unroll
        for (int q = 0; q < NC; ++q) {
            float f[8], w[8];
            unpack8(u[q], f);
            unpack8(gv[lane + 32 * q], w);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = (f[j] * inv) * w[j];
            dy[lane + 32 * q] = pack8(f);
        }
    } else {
        const int nc = H >> 3;
        for (int c = lane; c < nc; c += 32) {
            const uint4 u = src[c];
            if (copy) copy[c] = u;
            float f[8];
            unpack8(u, f);
#pragma unroll
            for (int j = 0; j < 8; ++j) csum_add(ss, sc, __fmul_rn(f[j], f[j]));
        }
        ss = csum_warp(ss, sc);
        if (g == nullptr) return;
        const float inv = 1.0f / sqrtf(ss / (float)H + eps);
        for (int c = lane; c < nc; c += 32) {
            float f[8], w[8];
            unpack8(src[c], f);
            unpack8(gv[c], w);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = (f[j] * inv) * w[j];
            dy[c] = pack8(f);
        }
    }
}

template <int NC>
__global__ void embed_rmsnorm_kernel(const int32_t* __restrict__ tokens, int tok_ld,
                                     const int32_t* __restrict__ row_seq, const int32_t* __restrict__ cu,
                                     const bf16* __restrict__ embed, int vocab, const bf16* __restrict__ g,
                                     bf16* __restrict__ r, bf16* __restrict__ y, int rows, int H, float eps,
                                     unsigned int* err) {
    pdl_launch();
    pdl_wait();
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int seq = row_seq[row];
    int tok = tokens[(long long)seq * tok_ld + (row - cu[seq])];   // the sequence's row-th new token
    if (tok < 0 || tok >= vocab) {
        if (lane == 0) raise_error(err, HRA_DEVERR_TOKEN_RANGE);
        tok = tok < 0 ? 0 : vocab - 1;
    }
    norm_row<NC>(reinterpret_cast<const uint4*>(embed + (long long)tok * H),
                 reinterpret_cast<uint4*>(r + (long long)row * H), lane, g, y + (long long)row * H, H, eps);
}

// g == nullptr: plain gather (copy_out must be set).
template <int NC>
__global__ void rmsnorm_kernel(const bf16* __restrict__ x, const int32_t* __restrict__ idx,
                               const bf16* __restrict__ g, bf16* __restrict__ y, bf16* __restrict__ copy_out,
                               int rows, int H, float eps) {
    pdl_launch();
    pdl_wait();
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const long long src_row = idx ? idx[row] : row;
    norm_row<NC>(reinterpret_cast<const uint4*>(x + src_row * H),
                 copy_out ? reinterpret_cast<uint4*>(copy_out + (long long)row * H) : nullptr, lane, g,
                 y + (long long)row * H, H, eps);
}

// One CTA per (row, group of 8 heads); half a warp per head of the merged QKV row.  The row's
// cos/sin are staged in shared memory once per CTA.  Lane l of a half-warp holds head elements [l*E, l*E + E) (E = hd/16, one 16- or 8-byte
// load); the RoPE partner of element i < hd/2 is i + hd/2, held by lane l ^ 8 of the same half-warp.
template <int HD>
__global__ void qk_rope_kv_kernel(const QkRopeArgs a) {
    pdl_launch();
    pdl_wait();
    constexpr int E = HD / 16;
    constexpr int HALF = HD / 2;
    __shared__ float2 s_cs[HALF];
    const int heads = a.nq + 2 * a.nkv;
    const int row = blockIdx.x;
    const int sub = threadIdx.x & 15;
    const int nhw = blockDim.x >> 4;
    const int hw0 = (threadIdx.x >> 4) + blockIdx.y * nhw;   // this CTA's group of heads
    const int seq = a.row_seq[row], pos = a.row_pos[row];
    const int trow = a.rope_row_is_pos ? pos : row;
    for (int i = threadIdx.x; i < HALF; i += blockDim.x) s_cs[i] = a.rope[(long long)i * a.rope_rows + trow];
    __syncthreads();
    const long long head_stride = (long long)a.n_slots * HD;
    {
        const int hh_raw = hw0;
        const bool valid = hh_raw < heads;       // half-warp uniform
        const int hh = valid ? hh_raw : 0;
        const bf16* src = a.qkv + (long long)row * heads * HD + (long long)hh * HD + sub * E;
        float x[E];
        if (a.part != nullptr) {
            // the projection's split-K partials, summed in split order and rounded once to bf16
            const float* ps = a.part + (long long)row * a.ldp + (long long)hh * HD + sub * E;
#pragma unroll
            for (int e = 0; e < E; ++e) x[e] = 0.f;
            constexpr int kBatch = 8;   // split partials loaded together before they are added
            for (int s0 = 0; s0 < a.splits; s0 += kBatch) {
                float4 v[kBatch][E / 4];
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
#pragma unroll
                    for (int e = 0; e < E / 4; ++e)
                        v[b][e] = s0 + b < a.splits
                                      ? *reinterpret_cast<const float4*>(ps + (s0 + b) * a.split_stride + 4 * e)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    if (s0 + b < a.splits) {
#pragma unroll
                        for (int e = 0; e < E / 4; ++e) {
                            x[4 * e] += v[b][e].x;
                            x[4 * e + 1] += v[b][e].y;
                            x[4 * e + 2] += v[b][e].z;
                            x[4 * e + 3] += v[b][e].w;
                        }
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < E; ++e) x[e] = round_bf(x[e]);
        } else if constexpr (E == 8) {
            unpack8(*reinterpret_cast<const uint4*>(src), x);
        } else {
            const uint2 u = *reinterpret_cast<const uint2*>(src);
            const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
            const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
            x[0] = f0.x; x[1] = f0.y; x[2] = f1.x; x[3] = f1.y;
        }
        const bool is_v = hh >= a.nq + a.nkv;
        const bool is_q = hh < a.nq;
        // compensated sum of squares over the 16 lanes of this half-warp (all lanes take part)
        float ss = 0.f, sc = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) csum_add(ss, sc, __fmul_rn(x[e], x[e]));
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
            const float s2 = __shfl_xor_sync(0xffffffffu, ss, o);
            const float c2 = __shfl_xor_sync(0xffffffffu, sc, o);
            float t, er;
            two_sum(ss, s2, t, er);
            ss = t;
            sc = __fadd_rn(__fadd_rn(sc, c2), er);
        }
        ss = __fadd_rn(ss, sc);
        const float inv = 1.0f / sqrtf(ss / (float)HD + a.eps);
        const bf16* gain = (is_q ? a.q_norm : a.k_norm) + sub * E;
        float xn[E], pn[E];
#pragma unroll
        for (int e = 0; e < E; ++e) xn[e] = is_v ? 0.f : __fmul_rn(__fmul_rn(x[e], inv), bf2f(gain[e]));
#pragma unroll
        for (int e = 0; e < E; ++e) pn[e] = __shfl_xor_sync(0xffffffffu, xn[e], 8);
        if (!valid) return;
        bf16* dst;
        if (is_v) {
            dst = a.kv_layer + ((long long)(seq * 2 + 1) * a.nkv + (hh - a.nq - a.nkv)) * head_stride +
                  (long long)pos * HD + sub * E;
            if (a.part != nullptr) {
                if constexpr (E == 8) {
                    *reinterpret_cast<uint4*>(dst) = pack8(x);
                } else {
                    uint2 u;
                    *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(x[0], x[1]);
                    *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(x[2], x[3]);
                    *reinterpret_cast<uint2*>(dst) = u;
                }
            } else if constexpr (E == 8) {
                *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
            } else {
                *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
            }
            return;
        }
        float out[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float2 c = s_cs[(sub * E + e) % HALF];   // (cos, sin)
            if (sub < 8)   // first half: a*cos - b*sin with a = own, b = partner
                out[e] = __fsub_rn(__fmul_rn(xn[e], c.x), __fmul_rn(pn[e], c.y));
            else           // second half: b*cos + a*sin with b = own, a = partner
                out[e] = __fadd_rn(__fmul_rn(xn[e], c.x), __fmul_rn(pn[e], c.y));
        }
        if (is_q) dst = a.q_out + ((long long)row * a.nq + hh) * HD + sub * E;
        else dst = a.kv_layer + ((long long)(seq * 2) * a.nkv + (hh - a.nq)) * head_stride + (long long)pos * HD + sub * E;
        if constexpr (E == 8) {
            *reinterpret_cast<uint4*>(dst) = pack8(out);
        } else {
            uint2 u;
            *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(out[0], out[1]);
            *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(out[2], out[3]);
            *reinterpret_cast<uint2*>(dst) = u;
        }
    }
}

inline unsigned blocks_for(long long threads, int per_block) {
    return (unsigned)((threads + per_block - 1) / per_block);
}

}  // namespace

cudaError_t launch_build_rowmap(const SeqMeta& meta, int total_rows, int32_t* row_seq, int32_t* row_pos,
                                int32_t* cu, int32_t* last_row, int32_t* seq_start, unsigned int* err,
                                cudaStream_t st, unsigned int* zero_ptr, int zero_words) {
    const int threads = 256;
    const unsigned blocks = meta.mode == 2 ? 1u : blocks_for(total_rows > 0 ? total_rows : 1, threads);
    HRA_LAUNCH(build_rowmap_kernel, dim3(blocks), dim3(threads), 0, st, meta, total_rows, row_seq, row_pos, cu, last_row,
               seq_start, err, zero_ptr, zero_ptr ? zero_words : 0);
    return cudaGetLastError();
}

cudaError_t launch_rope_table(int n_rows, const int32_t* pos_of_row, int head_dim, double theta,
                              float2* table, cudaStream_t st) {
    const long long n = (long long)n_rows * (head_dim / 2);
    HRA_LAUNCH(rope_table_kernel, dim3(blocks_for(n, 256)), dim3(256), 0, st, n_rows, pos_of_row, head_dim, theta, table);
    return cudaGetLastError();
}

cudaError_t launch_embed_rmsnorm(const int32_t* tokens, int tok_ld, const int32_t* row_seq,
                                 const int32_t* cu, const bf16* embed, int vocab, const bf16* g,
                                 bf16* r, bf16* y, int rows, int H, float eps, unsigned int* err,
                                 cudaStream_t st) {
    const dim3 grid(blocks_for((long long)rows * 32, 256));
    switch (H) {
        case 256: HRA_LAUNCH(embed_rmsnorm_kernel<1>, grid, dim3(256), 0, st, tokens, tok_ld, row_seq, cu, embed, vocab, g, r, y, rows, H, eps, err); break;
        case 2560: HRA_LAUNCH(embed_rmsnorm_kernel<10>, grid, dim3(256), 0, st, tokens, tok_ld, row_seq, cu, embed, vocab, g, r, y, rows, H, eps, err); break;
        default: HRA_LAUNCH(embed_rmsnorm_kernel<0>, grid, dim3(256), 0, st, tokens, tok_ld, row_seq, cu, embed, vocab, g, r, y, rows, H, eps, err); break;
    }
    return cudaSuccess;
}

cudaError_t launch_rmsnorm(const bf16* x, const int32_t* idx, const bf16* g, bf16* y, bf16* copy_out,
                           int rows, int H, float eps, cudaStream_t st) {
    const dim3 grid(blocks_for((long long)rows * 32, 256));
    switch (H) {
        case 256: HRA_LAUNCH(rmsnorm_kernel<1>, grid, dim3(256), 0, st, x, idx, g, y, copy_out, rows, H, eps); break;
        case 2560: HRA_LAUNCH(rmsnorm_kernel<10>, grid, dim3(256), 0, st, x, idx, g, y, copy_out, rows, H, eps); break;
        default: HRA_LAUNCH(rmsnorm_kernel<0>, grid, dim3(256), 0, st, x, idx, g, y, copy_out, rows, H, eps); break;
    }
    return cudaSuccess;
}

cudaError_t launch_qk_rope_kv(const QkRopeArgs& a, cudaStream_t st) {
    const int heads = a.nq + 2 * a.nkv;
    constexpr int kHeadsPerCta = 8;
    const dim3 grid(a.rows, (heads + kHeadsPerCta - 1) / kHeadsPerCta);
    if (a.hd == 128) HRA_LAUNCH(qk_rope_kv_kernel<128>, grid, dim3(kHeadsPerCta * 16), 0, st, a);
    else if (a.hd == 64) HRA_LAUNCH(qk_rope_kv_kernel<64>, grid, dim3(kHeadsPerCta * 16), 0, st, a);
    else return cudaErrorInvalidValue;
    return cudaSuccess;
}

}  // namespace hra
