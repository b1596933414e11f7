// decode_pass.cu -- the decoder pass over at most 64 token rows as one persistent kernel.
//
// Source: "Stabilize Higgs Audio termination and prefill" (FlashRT PR #141), Performance (the AR
// decode time per frame: one backbone pass per audio frame), and vLLM-Omni PR #8226, Step-overhead
// reductions (per-frame launch overhead as the limit of the streaming loop).  The arithmetic is the
// one of the layer-by-layer path: every layer computes
//   qkv = y . Wqkv^T; per-head q/k RMSNorm + rotate-half RoPE; K/V to the cache slot of the row
//   att = softmax(q k^T / sqrt(hd)) v over cache slots 0..pos (GQA)
//   r = bf16(r + att . Wo^T); y = RMSNorm(r) * mlp_norm
//   h = bf16(silu(bf16(g)) * bf16(u)), [g; u] = y . Wgu^T
//   r = bf16(r + h . Wdown^T); y = RMSNorm(r) * (next layer's attention norm, or the final norm)
// with every projection summed in fp32 over K splits in split order.
//
// One CTA per SM (launched cooperatively, so all of them are resident) walks the phases of every
// layer, with a grid-wide barrier after each:
//   QKV   projection partials        QK    split sum, q/k norm, RoPE, K/V write (half-warp items)
//   ATTN  attention units            O     output-projection partials
//   ORES  residual + chunk sums      ONORM RMSNorm with the MLP norm
//   GU    gate/up partials           SWIGLU
//   DOWN  down-projection partials   DRES, DNORM (next attention norm, or the final norm)
// Every split sum issues all its loads before the first add, so a phase costs about one L2 round
// trip; the splits are added in split order.
// Projections run on tcgen05 with the weight rows as the N = 256 operand and the (at most 64)
// activation rows as the M = 128 operand: one instruction then consumes 256 weight rows x 16 K.
// The weight stream does not stop at the barriers: when a projection's MMAs have drained the
// shared-memory ring, the producer refills it with the next projection's weight tiles (weights do
// not depend on activations), so each projection starts with its first stages already loaded.
//
// Roles in a projection phase: warp 0 lane 0 TMA producer, warp 1 lane 0 MMA issuer (warp 1 owns
// the TMEM allocation), warps 4, 5, 8, 9 epilogue (TMEM lane quarters 0 and 1 = rows 0..63).
// Every wait is bounded; on a timeout the kernel raises HRA_DEVERR_WAIT_TIMEOUT, lets its own copies
// and MMAs drain (again bounded), frees its TMEM and returns.
#include <string.h>

#include <algorithm>

#include "internal.h"

namespace hra {

bool g_decode_pass_enabled = false;

namespace {

constexpr int kDpThreads = 320;
constexpr int kDpStages = 3;
constexpr int kDpA = 64 * 128;                 // activation box: 64 rows x 64 bf16
constexpr int kDpW = 256 * 128;                // weight box(es): 256 rows x 64 bf16
constexpr int kDpStage = kDpA + kDpW;          // the A descriptor spans 16 KB: rows 64..127 read W
constexpr int kDpAS = 3;                       // K/V stages of an attention group
constexpr int kDpAttn = 16 * 128 * 2 + kDpAS * 2 * 64 * 128 * 2;   // q tile + K/V stages (hd <= 128)
constexpr int kDpMisc = 1024;
constexpr int kDpSmem = 1024 + kDpStages * kDpStage + kDpAttn + kDpMisc;
static_assert(kDpStages * kDpStage >= kDpAttn, "the second attention group works in the ring");
static_assert(kDpSmem <= 232448, "shared memory per CTA");
constexpr int kDpTmemCols = 512;               // two 256-column fp32 accumulators
constexpr int kDpPK = 64;                      // keys per attention tile
constexpr int kDpChunk = 128;                  // columns per residual/norm item (one warp, 4 a lane)
constexpr int kDpSplitBatch = 8;               // split partials loaded together before they are added
constexpr float kDpLog2e = 1.4426950408889634f;
enum DpProj : int { DP_QKV = 0, DP_O = 1, DP_GU = 2, DP_DOWN = 3 };

__device__ __forceinline__ float dp_silu(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int atom_acq_rel_add(unsigned int* p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// Warp-wide compensated sum of (s, c) pairs; every lane gets the combined pair.
__device__ __forceinline__ void csum_warp_pair(float& s, float& c) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const float c2 = __shfl_xor_sync(0xffffffffu, c, o);
        float t, e;
        two_sum(s, s2, t, e);
        s = t;
        c = __fadd_rn(__fadd_rn(c, c2), e);
    }
}

template <int HD>
__device__ __forceinline__ uint32_t dp_swz(int row, int chunk) {
    return (uint32_t)(row * HD * 2 + ((chunk ^ (row & 7)) << 4));
}

// Grid-wide barrier number `n` (1-based) of this launch.  All threads of the CTA take part; each
// warp is reconverged before the CTA barrier.  Thread 0 arrives with a release add (ordering every
// write the CTA made before the CTA barrier) and waits with acquire loads.  Returns false once any
// wait of this CTA has given up.
__device__ bool dp_grid_sync(unsigned int* cnt, unsigned int n, volatile int* abort_flag, unsigned int* err) {
    fence_proxy_async_global();
    __syncwarp();
    __syncthreads();
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0 && !*abort_flag) {
            red_release_add(cnt, 1u);
            const unsigned int target = n * gridDim.x;
            if (ld_acquire_u32(cnt) < target) {
                const uint64_t t0 = global_timer_ns();
                for (uint32_t it = 1;; ++it) {
                    if (ld_acquire_u32(cnt) >= target) break;
                    if ((it & 15u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) {
                        *abort_flag = 1;
                        raise_error(err, HRA_DEVERR_WAIT_TIMEOUT);
                        break;
                    }
                }
            }
        }
        __syncwarp();
    }
    __syncthreads();
    return *abort_flag == 0;
}

struct DpGemm {
    int nt, splits, kbps, n_kb;   // units = nt x splits; unit u: tile u % nt, K split u / nt
    int ldp;                      // floats per partial-plane row
};

struct DpLayer {
    const bf16* q_norm;
    const bf16* k_norm;
    const bf16* mlp_norm;
    const bf16* next_norm;        // next layer's attention norm, or the final norm (last layer)
    bf16* kv;                     // this layer's cache block [cache_batch][2][nkv][n_slots][hd]
};

struct DpParams {
    CUtensorMap wmap[kDecodePassMaxLayers][4];   // weights: QKV, O, gate/up (128-row boxes), down
    CUtensorMap amap[4];                         // activations feeding them: y, att, y, h
    DpLayer layer[kDecodePassMaxLayers];
    DpGemm g[4];
    int L, M, H, nq, nkv, F, Dq, Dqkv, n_slots;
    float eps;
    const float2* rope;           // transposed table: (table row t, pair i) at i * rope_rows + t
    int rope_rows, rope_row_is_pos;
    const int32_t* row_seq;
    const int32_t* row_pos;
    const int32_t* last_row;      // output row b = row last_row[b] (n_out of them); null: row b
    int n_out;
    bf16* r;
    bf16* y;
    bf16* q;
    bf16* att;
    bf16* h;
    bf16* out;
    float* part;
    float* apart;                 // [splits][M][nq][hd + 2]
    int attn_splits;
    unsigned int* sync;           // [0] barrier; [1, 1 + M nkv) attention items
    float2* pairs;                // [M][H / kDpChunk] compensated sums of squares
    unsigned int* err;
};

// ---------------------------------------------------------------- attention unit (128 threads)
// One (row i, kv head j, key split sp) of single-query attention over cache slots 0..pos: the
// method of decode_attn_kernel (attention.cu), run by a group of four warps (named barrier
// bar_id), K/V tiles streaming through kDpAS shared-memory stages.  Writes att directly for one split; otherwise its (o, m, l) partial, and the
// item's last split to finish merges the splits in split order.
template <int HD, int G>
__device__ void dp_attention_unit(const DpParams& p, const DpLayer& ly, int i, int j, int sp, int splits,
                                  uint8_t* smem, int tid, int* s_flag, int bar_id) {
    auto group_sync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(bar_id) : "memory"); };
    constexpr int KS = HD / 16, DN = HD / 8;
    constexpr uint32_t TILE = kDpPK * HD * 2;
    const uint32_t sQ = smem_u32(smem);
    const uint32_t sK0 = sQ + 16 * HD * 2;
    const uint32_t sV0 = sK0 + kDpAS * TILE;
    const int warp = tid >> 5, lane = tid & 31;
    const int seq = p.row_seq[i], pos = p.row_pos[i];
    const int nkeys = pos + 1;
    const int per = (nkeys + splits - 1) / splits;
    const int chunk = (per + kDpPK - 1) / kDpPK * kDpPK;
    const int k0 = sp * chunk, k1 = min(nkeys, k0 + chunk);
    const int n_t = k1 > k0 ? (k1 - k0 + kDpPK - 1) / kDpPK : 0;
    const long long hstride = (long long)p.n_slots * HD;
    const bf16* kbase = ly.kv + ((long long)(seq * 2) * p.nkv + j) * hstride + (long long)k0 * HD;
    const bf16* vbase = ly.kv + ((long long)(seq * 2 + 1) * p.nkv + j) * hstride + (long long)k0 * HD;
    const bf16* qbase = p.q + ((long long)i * p.nq + j * G) * HD;
    auto load_tile = [&](uint32_t sb, const bf16* gb, int rows_valid) {
        for (int idx = tid; idx < kDpPK * (HD / 8); idx += 128) {
            const int r = idx / (HD / 8), c = idx % (HD / 8);
            const bool ok = r < rows_valid;
            cp_async16(sb + dp_swz<HD>(r, c), gb + (ok ? (long long)r * HD + c * 8 : 0), ok ? 16u : 0u);
        }
    };
    auto load_kv = [&](int t) {   // tile t of the split into stage t % kDpAS
        const int rv = min(kDpPK, k1 - k0 - t * kDpPK);
        load_tile(sK0 + (t % kDpAS) * TILE, kbase + (long long)t * kDpPK * HD, rv);
        load_tile(sV0 + (t % kDpAS) * TILE, vbase + (long long)t * kDpPK * HD, rv);
    };
    for (int idx = tid; idx < 16 * (HD / 8); idx += 128) {
        const int r = idx / (HD / 8), c = idx % (HD / 8);
        const bool ok = r < G;
        cp_async16(sQ + dp_swz<HD>(r, c), qbase + (ok ? (long long)r * HD + c * 8 : 0), ok ? 16u : 0u);
    }
#pragma unroll
    for (int t = 0; t < kDpAS - 1; ++t) {
        if (t < n_t) load_kv(t);
        cp_async_commit();
    }

    uint32_t qf[KS][4];
    float o[DN][4];
#pragma unroll
    for (int d = 0; d < DN; ++d) o[d][0] = o[d][1] = o[d][2] = o[d][3] = 0.f;
    float m_a = -INFINITY, l_a = 0.f;
    const int tig = lane & 3;
    const float scale_log2 = (1.0f / sqrtf((float)HD)) * kDpLog2e;

    for (int t = 0; t < n_t; ++t) {
        if (t + kDpAS - 1 < n_t) load_kv(t + kDpAS - 1);   // its stage was freed by tile t - 1
        cp_async_commit();
        cp_async_wait<kDpAS - 1>();
        group_sync();
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) ldmatrix_x4(qf[ks], sQ + dp_swz<HD>(lane & 15, ks * 2 + (lane >> 4)));
        }
        const uint32_t sK = sK0 + (t % kDpAS) * TILE;
        const uint32_t sV = sV0 + (t % kDpAS) * TILE;
        const int kw = k0 + t * kDpPK + warp * 16;
        float s[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t kb[4];
            ldmatrix_x4(kb, sK + dp_swz<HD>(warp * 16 + (lane & 7) + ((lane >> 4) << 3), ks * 2 + ((lane >> 3) & 1)));
            mma_bf16_16816(s[0], qf[ks], kb[0], kb[1]);
            mma_bf16_16816(s[1], qf[ks], kb[2], kb[3]);
        }
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
        const float mref = mn == -INFINITY ? 0.f : mn;
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
        {
            const float a4[4][2] = {{s[0][0], s[0][1]}, {s[0][2], s[0][3]}, {s[1][0], s[1][1]}, {s[1][2], s[1][3]}};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const __nv_bfloat162 hh = __floats2bfloat162_rn(a4[x][0], a4[x][1]);
                const float2 hf = __bfloat1622float2(hh);
                ph[x] = *reinterpret_cast<const uint32_t*>(&hh);
                pl[x] = pack_bf2(a4[x][0] - hf.x, a4[x][1] - hf.y);
            }
        }
#pragma unroll
        for (int dp = 0; dp < DN / 2; ++dp) {
            uint32_t vb[4];
            ldmatrix_x4_trans(vb, sV + dp_swz<HD>(warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), dp * 2 + (lane >> 4)));
            mma_bf16_16816(o[2 * dp], ph, vb[0], vb[1]);
            mma_bf16_16816(o[2 * dp + 1], ph, vb[2], vb[3]);
            mma_bf16_16816(o[2 * dp], pl, vb[0], vb[1]);
            mma_bf16_16816(o[2 * dp + 1], pl, vb[2], vb[3]);
        }
        group_sync();   // the stage is refilled next iteration
    }
    cp_async_wait<0>();
    group_sync();

    float* s_o = reinterpret_cast<float*>(smem + 16 * HD * 2);   // [4][G][HD] over the stages
    float* s_ml = s_o + 4 * G * HD;                               // [4][G][2]
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    const int gq = lane >> 2;
    if (gq < G) {
        float* dst = s_o + (warp * G + gq) * HD + 2 * tig;
#pragma unroll
        for (int d = 0; d < DN; ++d) {
            dst[d * 8] = o[d][0];
            dst[d * 8 + 1] = o[d][1];
        }
        if (tig == 0) {
            s_ml[(warp * G + gq) * 2] = m_a;
            s_ml[(warp * G + gq) * 2 + 1] = l_a;
        }
    }
    group_sync();
    for (int idx = tid; idx < G * HD; idx += 128) {
        const int hg = idx / HD, dc = idx % HD;
        float Mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w)
            if (s_ml[(w * G + hg) * 2 + 1] > 0.f) Mx = fmaxf(Mx, s_ml[(w * G + hg) * 2]);
        float Ls = 0.f, Os = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float lw = s_ml[(w * G + hg) * 2 + 1];
            if (lw > 0.f) {
                const float f = exp2f(s_ml[(w * G + hg) * 2] - Mx);
                Ls += lw * f;
                Os += s_o[(w * G + hg) * HD + dc] * f;
            }
        }
        if (splits == 1) {
            p.att[((long long)i * p.nq + j * G + hg) * HD + dc] = f2bf(Os / Ls);
        } else {
            float* dst = p.apart + (((long long)sp * p.M + i) * p.nq + j * G + hg) * (HD + 2);
            dst[dc] = Os;
            if (dc == 0) {
                dst[HD] = Mx;
                dst[HD + 1] = Ls;
            }
        }
    }
    if (splits == 1) {
        group_sync();   // s_o / s_ml are reused by the next unit
        return;
    }
    // the item's last split to finish merges all splits (in split order): the group's writes are
    // ordered before the counter by the group barrier and the acq_rel add
    group_sync();
    if (tid == 0) {
        unsigned int* c = p.sync + 1 + i * p.nkv + j;
        const unsigned int old = atom_acq_rel_add(c, 1u);
        const bool last = old == (unsigned int)splits - 1u;
        if (last) *c = 0u;
        *s_flag = last ? 1 : 0;
    }
    group_sync();
    if (*s_flag) {
        // every split's (m, l) into shared memory, then each output element sums its splits' o in
        // split order with all of a batch's loads in flight
        float* s_m = reinterpret_cast<float*>(smem + 16 * HD * 2);   // [G][splits]
        float* s_l = s_m + G * splits;
        for (int idx = tid; idx < G * splits; idx += 128) {
            const int hg = idx / splits, s2 = idx % splits;
            const float* pp = p.apart + (((long long)s2 * p.M + i) * p.nq + j * G + hg) * (HD + 2);
            s_m[idx] = __ldcg(pp + HD);
            s_l[idx] = __ldcg(pp + HD + 1);
        }
        group_sync();
        for (int idx = tid; idx < G * HD; idx += 128) {
            const int hg = idx / HD, d = idx % HD;
            const int hq = j * G + hg;
            float Mx = -INFINITY;
            for (int s2 = 0; s2 < splits; ++s2)
                if (s_l[hg * splits + s2] > 0.f) Mx = fmaxf(Mx, s_m[hg * splits + s2]);
            float Ls = 0.f, Os = 0.f;
            for (int s0 = 0; s0 < splits; s0 += kDpSplitBatch) {
                float ov[kDpSplitBatch];
#pragma unroll
                for (int b = 0; b < kDpSplitBatch; ++b)
                    ov[b] = s0 + b < splits
                                ? __ldcg(p.apart + (((long long)(s0 + b) * p.M + i) * p.nq + hq) * (HD + 2) + d)
                                : 0.f;
#pragma unroll
                for (int b = 0; b < kDpSplitBatch; ++b) {
                    if (s0 + b < splits) {
                        const float lw = s_l[hg * splits + s0 + b];
                        if (lw > 0.f) {
                            const float f = exp2f(s_m[hg * splits + s0 + b] - Mx);
                            Ls += lw * f;
                            Os += ov[b] * f;
                        }
                    }
                }
            }
            p.att[((long long)i * p.nq + hq) * HD + d] = f2bf(Os / Ls);
        }
    }
    group_sync();
}

// ---------------------------------------------------------------- q/k norm + RoPE + K/V write
// Half a warp per (row, head) of the merged QKV row, E = HD / 16 elements per lane; the method of
// qk_rope_kv_kernel (elementwise.cu) with the split partials summed in split order.
template <int HD>
__device__ void dp_qk_item(const DpParams& p, const DpLayer& ly, int row, int hh, int sub, bool valid) {
    constexpr int E = HD / 16, HALF = HD / 2;
    const DpGemm& g = p.g[0];
    const long long split_stride = (long long)p.M * g.ldp;
    const float* ps = p.part + (long long)row * g.ldp + (long long)hh * HD + sub * E;
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = 0.f;
    for (int s0 = 0; s0 < g.splits; s0 += kDpSplitBatch) {
        float4 v[kDpSplitBatch][E / 4];   // every load of the batch in flight before the first add
#pragma unroll
        for (int b = 0; b < kDpSplitBatch; ++b)
#pragma unroll
            for (int e = 0; e < E / 4; ++e)
                v[b][e] = s0 + b < g.splits ? ldcg4(ps + (s0 + b) * split_stride + 4 * e) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int b = 0; b < kDpSplitBatch; ++b)
            if (s0 + b < g.splits) {
#pragma unroll
                for (int e = 0; e < E / 4; ++e) {
                    x[4 * e] += v[b][e].x;
                    x[4 * e + 1] += v[b][e].y;
                    x[4 * e + 2] += v[b][e].z;
                    x[4 * e + 3] += v[b][e].w;
                }
            }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = round_bf(x[e]);
    const bool is_v = hh >= p.nq + p.nkv, is_q = hh < p.nq;
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
    const float inv = 1.0f / sqrtf(ss / (float)HD + p.eps);
    const bf16* gain = (is_q ? ly.q_norm : ly.k_norm) + sub * E;
    float xn[E], pn[E];
#pragma unroll
    for (int e = 0; e < E; ++e) xn[e] = is_v ? 0.f : __fmul_rn(__fmul_rn(x[e], inv), bf2f(gain[e]));
#pragma unroll
    for (int e = 0; e < E; ++e) pn[e] = __shfl_xor_sync(0xffffffffu, xn[e], 8);
    if (!valid) return;   // a half-warp without an item only took part in the shuffles
    const int seq = p.row_seq[row], pos = p.row_pos[row];
    const long long head_stride = (long long)p.n_slots * HD;
    bf16* dst;
    float out[E];
    if (is_v) {
        dst = ly.kv + ((long long)(seq * 2 + 1) * p.nkv + (hh - p.nq - p.nkv)) * head_stride + (long long)pos * HD + sub * E;
#pragma unroll
        for (int e = 0; e < E; ++e) out[e] = x[e];
    } else {
        const int trow = p.rope_row_is_pos ? pos : row;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float2 c = p.rope[(long long)((sub * E + e) % HALF) * p.rope_rows + trow];
            if (sub < 8)
                out[e] = __fsub_rn(__fmul_rn(xn[e], c.x), __fmul_rn(pn[e], c.y));
            else
                out[e] = __fadd_rn(__fmul_rn(xn[e], c.x), __fmul_rn(pn[e], c.y));
        }
        if (is_q)
            dst = p.q + ((long long)row * p.nq + hh) * HD + sub * E;
        else
            dst = ly.kv + ((long long)(seq * 2) * p.nkv + (hh - p.nq)) * head_stride + (long long)pos * HD + sub * E;
    }
    if constexpr (E == 8) {
        *reinterpret_cast<uint4*>(dst) = pack8(out);
    } else {
        uint2 u;
        *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(out[0], out[1]);
        *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(out[2], out[3]);
        *reinterpret_cast<uint2*>(dst) = u;
    }
}

// ---------------------------------------------------------------- residual + RMSNorm
// Residual item, one warp per (row m, 128-column chunk c): r = bf16(r + sum of the projection's split
// partials, split order), and the chunk's compensated sum of squares of the rounded r.
__device__ void dp_res_item(const DpParams& p, int gi, int m, int c, int lane) {
    const DpGemm& g = p.g[gi];
    const int nch = p.H / kDpChunk;
    const int col = c * kDpChunk + lane * 4;
    const long long split_stride = (long long)p.M * g.ldp;
    const float* base = p.part + (long long)m * g.ldp + col;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < g.splits; s0 += 2 * kDpSplitBatch) {
        float4 v[2 * kDpSplitBatch];
#pragma unroll
        for (int b = 0; b < 2 * kDpSplitBatch; ++b)
            v[b] = s0 + b < g.splits ? ldcg4(base + (s0 + b) * split_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int b = 0; b < 2 * kDpSplitBatch; ++b)
            if (s0 + b < g.splits) {
                a[0] += v[b].x;
                a[1] += v[b].y;
                a[2] += v[b].z;
                a[3] += v[b].w;
            }
    }
    uint2* rp = reinterpret_cast<uint2*>(p.r + (long long)m * p.H + col);
    const uint2 ru = __ldcg(rp);
    const float2 r01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ru.x));
    const float2 r23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ru.y));
    const __nv_bfloat162 o01 = __floats2bfloat162_rn(r01.x + a[0], r01.y + a[1]);
    const __nv_bfloat162 o23 = __floats2bfloat162_rn(r23.x + a[2], r23.y + a[3]);
    uint2 out;
    out.x = *reinterpret_cast<const uint32_t*>(&o01);
    out.y = *reinterpret_cast<const uint32_t*>(&o23);
    *rp = out;
    const float2 v01 = __bfloat1622float2(o01), v23 = __bfloat1622float2(o23);
    float ss = 0.f, sc = 0.f;
    csum_add(ss, sc, __fmul_rn(v01.x, v01.x));
    csum_add(ss, sc, __fmul_rn(v01.y, v01.y));
    csum_add(ss, sc, __fmul_rn(v23.x, v23.x));
    csum_add(ss, sc, __fmul_rn(v23.y, v23.y));
    csum_warp_pair(ss, sc);
    if (lane == 0) p.pairs[m * nch + c] = make_float2(ss, sc);
}

// Norm item, one warp per (row m, chunk c): the row's chunk sums combined in chunk order, then
// y = bf16((r * inv) * gain) for the chunk -- into y, or for the last layer into the output row.
__device__ void dp_norm_item(const DpParams& p, int m, int c, const bf16* gain, bool final_layer, int lane) {
    const int nch = p.H / kDpChunk;
    bf16* dst_row = nullptr;
    if (!final_layer) {
        dst_row = p.y + (long long)m * p.H;
    } else if (p.last_row == nullptr) {
        dst_row = m < p.n_out ? p.out + (long long)m * p.H : nullptr;
    } else {
        for (int b = 0; b < p.n_out; ++b)
            if (p.last_row[b] == m) dst_row = p.out + (long long)b * p.H;
    }
    if (dst_row == nullptr) return;
    float2 pr[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};   // chunks lane and lane + 32
#pragma unroll
    for (int q = 0; q < 2; ++q)
        if (lane + 32 * q < nch) pr[q] = __ldcg(p.pairs + m * nch + lane + 32 * q);
    float ts = 0.f, tc = 0.f;
    for (int k = 0; k < nch; ++k) {   // chunk order, the same in every lane
        const float2 v = make_float2(__shfl_sync(0xffffffffu, pr[k >> 5].x, k & 31),
                                     __shfl_sync(0xffffffffu, pr[k >> 5].y, k & 31));
        float t, e;
        two_sum(ts, v.x, t, e);
        ts = t;
        tc = __fadd_rn(__fadd_rn(tc, v.y), e);
    }
    const float tot = __fadd_rn(ts, tc);
    const float inv = 1.0f / sqrtf(tot / (float)p.H + p.eps);
    const int col = c * kDpChunk + lane * 4;
    const uint2 ru = __ldcg(reinterpret_cast<const uint2*>(p.r + (long long)m * p.H + col));
    const uint2 gu = *reinterpret_cast<const uint2*>(gain + col);
    const float2 r01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ru.x));
    const float2 r23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ru.y));
    const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gu.x));
    const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gu.y));
    const __nv_bfloat162 o01 = __floats2bfloat162_rn((r01.x * inv) * g01.x, (r01.y * inv) * g01.y);
    const __nv_bfloat162 o23 = __floats2bfloat162_rn((r23.x * inv) * g23.x, (r23.y * inv) * g23.y);
    uint2 out;
    out.x = *reinterpret_cast<const uint32_t*>(&o01);
    out.y = *reinterpret_cast<const uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(dst_row + col) = out;
}

// SwiGLU item, one thread per (row m, 8 columns j0..j0+7): h = bf16(silu(bf16(g)) * bf16(u)) with
// g and u the gate/up split partials summed in split order.
__device__ void dp_swiglu_item(const DpParams& p, int m, int j0) {
    const DpGemm& g = p.g[2];
    const long long split_stride = (long long)p.M * g.ldp;
    const float* base = p.part + (long long)m * g.ldp + j0;
    float ga[8] = {0, 0, 0, 0, 0, 0, 0, 0}, ua[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int s0 = 0; s0 < g.splits; s0 += 4) {
        float4 v[4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float* pp = base + (s0 + b) * split_stride;
            const bool ok = s0 + b < g.splits;
            v[b][0] = ok ? ldcg4(pp) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[b][1] = ok ? ldcg4(pp + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[b][2] = ok ? ldcg4(pp + p.F) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[b][3] = ok ? ldcg4(pp + p.F + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (s0 + b < g.splits) {
                ga[0] += v[b][0].x; ga[1] += v[b][0].y; ga[2] += v[b][0].z; ga[3] += v[b][0].w;
                ga[4] += v[b][1].x; ga[5] += v[b][1].y; ga[6] += v[b][1].z; ga[7] += v[b][1].w;
                ua[0] += v[b][2].x; ua[1] += v[b][2].y; ua[2] += v[b][2].z; ua[3] += v[b][2].w;
                ua[4] += v[b][3].x; ua[5] += v[b][3].y; ua[6] += v[b][3].z; ua[7] += v[b][3].w;
            }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) ga[e] = dp_silu(round_bf(ga[e])) * round_bf(ua[e]);
    *reinterpret_cast<uint4*>(p.h + (long long)m * p.F + j0) = pack8(ga);
}

// ---------------------------------------------------------------- the kernel
template <int HD, int G>
__global__ void __launch_bounds__(kDpThreads, 1) decode_pass_kernel(const __grid_constant__ DpParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* attn_smem = smem + kDpStages * kDpStage;
    uint8_t* misc = attn_smem + kDpAttn;
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);   // full[S], empty[S], tfull[2], tempty[2], drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kDpStages + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* consumed_slot = reinterpret_cast<int*>(tmem_slot + 2); // ring iterations the MMA consumed
    int* s_flag = reinterpret_cast<int*>(tmem_slot + 4);        // attention groups 0 and 1

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bid = blockIdx.x, G_ = gridDim.x;
    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + kDpStages + s); };
    auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * kDpStages + b); };
    auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * kDpStages + 2 + b); };
    const uint32_t drain_bar = smem_u32(bars + 2 * kDpStages + 4);
    auto a_tile = [&](int s) { return smem_u32(smem + s * kDpStage); };
    auto w_tile = [&](int s) { return smem_u32(smem + s * kDpStage + kDpA); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kDpStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *consumed_slot = 0;
        mbar_fence_init();
        for (int a = 0; a < 4; ++a) tma_prefetch_map(&p.amap[a]);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kDpTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // producer state (warp 0 lane 0): ring iterations whose weight load (it_w) and activation load
    // (it_a) have been issued; MMA state (warp 1 lane 0): iterations consumed and units done;
    // epilogue state: units drained.
    int it_w = 0, it_a = 0, it_m = 0, n_unit_m = 0, n_unit_e = 0;
    unsigned int nbar = 0;

    // k-blocks this CTA runs in projection gi (its units u = bid, bid + G_, ...)
    auto cta_iters = [&](int gi) {
        const DpGemm& g = p.g[gi];
        int n = 0;
        for (int u = bid; u < g.nt * g.splits; u += G_) {
            const int sp = u / g.nt;
            n += min(g.n_kb, sp * g.kbps + g.kbps) - sp * g.kbps;
        }
        return n;
    };
    // the (tile, k-block) of this CTA's j-th iteration of projection gi
    auto iter_at = [&](int gi, int j, int& tile, int& kb) {
        const DpGemm& g = p.g[gi];
        for (int u = bid; u < g.nt * g.splits; u += G_) {
            const int sp = u / g.nt;
            const int kb0 = sp * g.kbps, n = min(g.n_kb, kb0 + g.kbps) - kb0;
            if (j < n) {
                tile = u - sp * g.nt;
                kb = kb0 + j;
                return;
            }
            j -= n;
        }
        tile = 0;
        kb = 0;
    };
    auto load_w = [&](int l, int gi, int s, int tile, int kb) {
        const CUtensorMap* m = &p.wmap[l][gi];
        if (gi == DP_GU) {
            tma_load_2d(w_tile(s), m, full_bar(s), kb * 64, tile * 128);
            tma_load_2d(w_tile(s) + kDpW / 2, m, full_bar(s), kb * 64, p.F + tile * 128);
        } else {
            tma_load_2d(w_tile(s), m, full_bar(s), kb * 64, tile * 256);
        }
    };
    // producer: issue the weight loads of the first ring stages of projection (l, gi) -- as many as
    // the ring holds -- without their activation loads (those follow the barrier before the phase)
    auto preissue = [&](int l, int gi) -> bool {
        const int n = min(kDpStages, cta_iters(gi));
        for (int j = 0; j < n; ++j) {
            const int s = it_w % kDpStages;
            const uint32_t ph = (uint32_t)(it_w / kDpStages) & 1u;
            if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) return false;
            int tile, kb;
            iter_at(gi, j, tile, kb);
            mbar_expect_tx(full_bar(s), kDpA + kDpW);
            load_w(l, gi, s, tile, kb);
            ++it_w;
        }
        return true;
    };

    // one projection phase: all roles; returns false on abort
    auto gemm_phase = [&](int l, int gi) -> bool {
        const DpGemm& g = p.g[gi];
        const int units = g.nt * g.splits;
        if (warp == 0) {
            if (lane == 0) {
                const int n = cta_iters(gi);
                fence_proxy_async_global();
                bool ok = true;
                for (int j = 0; j < n && ok; ++j) {
                    const int s = it_a % kDpStages;
                    int tile, kb;
                    iter_at(gi, j, tile, kb);
                    if (it_a == it_w) {   // not pre-issued: weight and activation together
                        const uint32_t ph = (uint32_t)(it_w / kDpStages) & 1u;
                        if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(full_bar(s), kDpA + kDpW);
                        load_w(l, gi, s, tile, kb);
                        ++it_w;
                    }
                    tma_load_2d(a_tile(s), &p.amap[gi], full_bar(s), kb * 64, 0);
                    ++it_a;
                }
                // the next projection's first weight tiles, as the MMAs drain the ring (not before
                // the output projection: the attention between them works in the ring)
                if (ok && gi != DP_QKV) {
                    int nl = l, ng = gi + 1;
                    if (ng == 4) {
                        ng = 0;
                        ++nl;
                    }
                    if (nl < p.L) ok = preissue(nl, ng);
                }
                if (!ok) {
                    *abort_flag = 1;
                    raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                }
            }
        } else if (warp == 1) {
            if (lane == 0) {
                constexpr uint32_t idesc = idesc_bf16_f32(128, 256);
                bool ok = true;
                for (int u = bid; u < units && ok; u += G_, ++n_unit_m) {
                    const int sp = u / g.nt;
                    const int kb0 = sp * g.kbps, kb1 = min(g.n_kb, kb0 + g.kbps);
                    const int buf = n_unit_m & 1;
                    if (!mbar_wait(tempty_bar(buf), ((uint32_t)(n_unit_m >> 1) & 1u) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)(buf * 256);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        const int s = it_m % kDpStages;
                        const uint32_t ph = (uint32_t)(it_m / kDpStages) & 1u;
                        if (!mbar_wait(full_bar(s), ph, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = sdesc_sw128(a_tile(s));
                        const uint64_t bd = sdesc_sw128(w_tile(s));
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma_bf16(d_tmem, ad + 2ull * k, bd + 2ull * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        tc_commit(empty_bar(s));
                        ++it_m;
                        *consumed_slot = it_m;
                    }
                    if (!ok) break;
                    tc_commit(tfull_bar(buf));
                }
                if (!ok) {
                    *abort_flag = 1;
                    raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                }
            }
        } else if (warp == 4 || warp == 5 || warp == 8 || warp == 9) {
            // epilogue: TMEM lane quarter (warp & 3) = rows 32 (warp & 3) .. + 31; warps 4/5 take
            // columns 0..127, warps 8/9 columns 128..255 (gate/up: 64 gate + the matching 64 up)
            const int quad = warp & 3;
            const int half = warp >= 8 ? 1 : 0;
            const int row = quad * 32 + lane;
            const bool row_ok = row < p.M;
            const long long split_stride = (long long)p.M * g.ldp;
            for (int u = bid; u < units; u += G_, ++n_unit_e) {
                const int sp = u / g.nt, tile = u - sp * g.nt;
                const int buf = n_unit_e & 1;
                const bool got = __all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), (uint32_t)(n_unit_e >> 1) & 1u, abort_flag));
                // the four epilogue warps agree (they meet at a named barrier below)
                uint32_t any_fail;
                asm volatile(
                    "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, 3, 128, pi;\n"
                    " selp.u32 %0, 1, 0, po;\n}"
                    : "=r"(any_fail)
                    : "r"((uint32_t)!got)
                    : "memory");
                if (any_fail) {
                    *abort_flag = 1;
                    raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(buf * 256);
                float* prow = p.part + sp * split_stride + (long long)row * g.ldp;
                if (gi != DP_GU) {
                    for (int c = 0; c < 128; c += 32) {
                        float v[32];
                        tmem_ld32(tq + half * 128 + c, v);
                        if (row_ok) {
                            float4* dst = reinterpret_cast<float4*>(prow + tile * 256 + half * 128 + c);
#pragma unroll
                            for (int q4 = 0; q4 < 8; ++q4)
                                dst[q4] = make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
                        }
                    }
                } else {
                    // gate columns tile*128 + half*64 + [0, 64) and the matching up columns
                    const int gcol = tile * 128 + half * 64;
                    for (int c = 0; c < 64; c += 32) {
                        float vg[32], vu[32];
                        tmem_ld32(tq + half * 64 + c, vg);
                        tmem_ld32(tq + 128 + half * 64 + c, vu);
                        if (row_ok) {
                            float4* dg = reinterpret_cast<float4*>(prow + gcol + c);
                            float4* du = reinterpret_cast<float4*>(prow + p.F + gcol + c);
#pragma unroll
                            for (int q4 = 0; q4 < 8; ++q4) {
                                dg[q4] = make_float4(vg[4 * q4], vg[4 * q4 + 1], vg[4 * q4 + 2], vg[4 * q4 + 3]);
                                du[q4] = make_float4(vu[4 * q4], vu[4 * q4 + 1], vu[4 * q4 + 2], vu[4 * q4 + 3]);
                            }
                        }
                    }
                }
                tc_fence_before();
                if (lane == 0) mbar_arrive(tempty_bar(buf));
            }
        }
        return true;
    };

    // ------------------------------------------------------------ layers
    if (threadIdx.x == 0) {
        if (!preissue(0, DP_QKV)) {
            *abort_flag = 1;
            raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
        }
    }
    const int heads = p.nq + 2 * p.nkv;
    const int nch = p.H / kDpChunk;
    for (int l = 0; l < p.L && *abort_flag == 0; ++l) {
        const DpLayer& ly = p.layer[l];
        // QKV projection
        gemm_phase(l, DP_QKV);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        // split sum + q/k norm + RoPE + K/V write: half a warp per (row, head)
        {
            const int hw_per_cta = kDpThreads / 16;
            const int items = p.M * heads;
            // warp-uniform trip count: both halves of a warp take part in every shuffle, a half
            // without an item computes on item 0 and writes nothing
            for (int base = bid * hw_per_cta; base < items; base += G_ * hw_per_cta) {
                const int it = base + (threadIdx.x >> 4);
                const bool valid = it < items;
                const int itv = valid ? it : 0;
                const int row = itv / heads, hh = itv - row * heads;
                if (__any_sync(0xffffffffu, valid)) dp_qk_item<HD>(p, ly, row, hh, threadIdx.x & 15, valid);
            }
        }
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        // attention: two groups of four warps (2-5 in the attention area, 6-9 in the ring, idle
        // between the QKV and output projections), one unit each at a time; once both groups of
        // the CTA are done, the producer starts the output projection's weight tiles into the ring
        if (warp >= 2) {
            const int gidx = (warp - 2) >> 2;
            uint8_t* gsm = gidx == 0 ? attn_smem : smem;
            const int splits = p.attn_splits;
            const int units = p.M * p.nkv * splits;
            for (int u = 2 * bid + gidx; u < units; u += 2 * G_) {
                const int sp = u % splits, ij = u / splits;
                dp_attention_unit<HD, G>(p, ly, ij / p.nkv, ij % p.nkv, sp, splits, gsm, threadIdx.x - 64 - 128 * gidx,
                                         s_flag + gidx, 1 + gidx);
            }
            asm volatile("bar.arrive 5, 288;" ::: "memory");
        } else if (warp == 0) {
            asm volatile("bar.sync 5, 288;" ::: "memory");
            if (lane == 0) {
                fence_proxy_async_smem();   // the attention's use of the ring before the copies into it
                if (!preissue(l, DP_O)) {
                    *abort_flag = 1;
                    raise_error(p.err, HRA_DEVERR_WAIT_TIMEOUT);
                }
            }
            __syncwarp();
        }
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        // output projection; residual; RMSNorm with the MLP norm
        gemm_phase(l, DP_O);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        for (int it = bid * (kDpThreads / 32) + warp; it < p.M * nch; it += G_ * (kDpThreads / 32))
            dp_res_item(p, DP_O, it / nch, it % nch, lane);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        for (int it = bid * (kDpThreads / 32) + warp; it < p.M * nch; it += G_ * (kDpThreads / 32))
            dp_norm_item(p, it / nch, it % nch, ly.mlp_norm, false, lane);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        // gate/up; SwiGLU; down; residual; RMSNorm with the next layer's attention norm (or the final
        // norm into the output rows)
        gemm_phase(l, DP_GU);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        for (int it = bid * kDpThreads + threadIdx.x; it < p.M * (p.F / 8); it += G_ * kDpThreads)
            dp_swiglu_item(p, it / (p.F / 8), (it % (p.F / 8)) * 8);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        gemm_phase(l, DP_DOWN);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        for (int it = bid * (kDpThreads / 32) + warp; it < p.M * nch; it += G_ * (kDpThreads / 32))
            dp_res_item(p, DP_DOWN, it / nch, it % nch, lane);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
        for (int it = bid * (kDpThreads / 32) + warp; it < p.M * nch; it += G_ * (kDpThreads / 32))
            dp_norm_item(p, it / nch, it % nch, ly.next_norm, l == p.L - 1, lane);
        if (!dp_grid_sync(p.sync, ++nbar, abort_flag, p.err)) break;
    }

    // ------------------------------------------------------------ drain and free
    __syncthreads();
    if (*abort_flag) {
        // every issued copy lands and every issued MMA finishes before the shared memory and the
        // TMEM go away: stages whose weight tile went out ahead of the barrier get their
        // activation box now (any valid box: the data is not used), then the producer waits for
        // the unconsumed stages and the MMA thread for its last MMA (both bounded)
        volatile int no_abort = 0;
        if (threadIdx.x == 0) {
            for (int it = it_a; it < it_w; ++it)
                tma_load_2d(a_tile(it % kDpStages), &p.amap[0], full_bar(it % kDpStages), 0, 0);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int it = *consumed_slot; it < it_w; ++it)
                (void)mbar_wait(full_bar(it % kDpStages), (uint32_t)(it / kDpStages) & 1u, &no_abort);
        } else if (warp == 1 && lane == 0) {
            tc_commit(drain_bar);
            (void)mbar_wait(drain_bar, 0u, &no_abort);
        }
        __syncthreads();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kDpTmemCols);
}

// K split plan of one projection: tiles x splits units over the SMs, minimising the k-blocks of the
// busiest SM (plus a small charge per split for its partial plane).
DpGemm dp_plan(int nt, int n_kb, int nsm, int ldp, int max_splits) {
    DpGemm best{nt, 1, n_kb, n_kb, ldp};
    double best_cost = 1e30;
    for (int kbps = 1; kbps <= n_kb; ++kbps) {
        const int splits = (n_kb + kbps - 1) / kbps;
        if (splits > max_splits) continue;
        const long long units = (long long)nt * splits;
        const long long rounds = (units + nsm - 1) / nsm;
        const double cost = (double)rounds * kbps + 0.1 * splits;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = DpGemm{nt, splits, kbps, n_kb, ldp};
        }
    }
    return best;
}

// Shared-memory opt-in of one instantiation (once per device) and whether one CTA of it fits on an
// SM, the condition of the cooperative launch.
template <int HD, int G>
bool dp_configure() {
    static int state[64] = {0};   // 0 unknown, 1 fits, 2 does not
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (state[dev] == 0) {
        int n = 0;
        const bool ok =
            cudaFuncSetAttribute(decode_pass_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDpSmem) ==
                cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_pass_kernel<HD, G>, kDpThreads, kDpSmem) ==
                cudaSuccess &&
            n >= 1;
        state[dev] = ok ? 1 : 2;
    }
    return state[dev] == 1;
}

bool dp_fits(int hd, int g) {
    if (hd == 128) {
        switch (g) {
            case 1: return dp_configure<128, 1>();
            case 2: return dp_configure<128, 2>();
            case 4: return dp_configure<128, 4>();
            case 8: return dp_configure<128, 8>();
        }
    } else if (hd == 64) {
        switch (g) {
            case 1: return dp_configure<64, 1>();
            case 2: return dp_configure<64, 2>();
            case 4: return dp_configure<64, 4>();
            case 8: return dp_configure<64, 8>();
        }
    }
    return false;
}

template <int HD, int G>
cudaError_t launch_dp(const DpParams& prm, int grid, cudaStream_t st) {
    if (!dp_configure<HD, G>()) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDpThreads);
    cfg.dynamicSmemBytes = kDpSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, decode_pass_kernel<HD, G>, prm);
}

template <int HD>
cudaError_t launch_dp_g(const DpParams& prm, int g, int grid, cudaStream_t st) {
    switch (g) {
        case 1: return launch_dp<HD, 1>(prm, grid, st);
        case 2: return launch_dp<HD, 2>(prm, grid, st);
        case 4: return launch_dp<HD, 4>(prm, grid, st);
        case 8: return launch_dp<HD, 8>(prm, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool decode_pass_supported(const DecodePassCall& c) {
    if (c.M < 1 || c.M > 64 || c.L < 1 || c.L > kDecodePassMaxLayers) return false;
    if (c.hd != 64 && c.hd != 128) return false;
    const int g = c.nq / c.nkv;
    if (c.nq % c.nkv != 0 || (g != 1 && g != 2 && g != 4 && g != 8)) return false;
    const int Dq = c.nq * c.hd, Dqkv = (c.nq + 2 * c.nkv) * c.hd;
    if (c.H % 256 != 0 || c.H > 64 * kDpChunk || Dq % 256 != 0 || Dqkv % 256 != 0 || c.F % 128 != 0) return false;
    int sms = 0, coop = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return false;
    sms = device_sm_count();
    return sms >= 16 && decode_pass_scratch_bytes(c.M, c.H, c.nq, c.nkv, c.hd, c.F, sms) <= c.part_bytes &&
           dp_fits(c.hd, g);
}

size_t decode_pass_scratch_bytes(int M, int H, int nq, int nkv, int hd, int F, int nsm) {
    const int Dq = nq * hd, Dqkv = (nq + 2 * nkv) * hd;
    const DpGemm g0 = dp_plan(Dqkv / 256, H / 64, nsm, Dqkv, 32);
    const DpGemm g1 = dp_plan(H / 256, Dq / 64, nsm, H, 32);
    const DpGemm g2 = dp_plan(F / 128, H / 64, nsm, 2 * F, 4);
    const DpGemm g3 = dp_plan(H / 256, F / 64, nsm, H, 32);
    size_t b = 0;
    for (const DpGemm& g : {g0, g1, g2, g3}) b = std::max(b, (size_t)g.splits * M * g.ldp * sizeof(float));
    return b;
}

int decode_pass_counter_words(int M, int nkv) { return 1 + M * nkv; }

size_t decode_pass_sync_bytes(int M, int nkv, int F, int H) {
    (void)F;
    const size_t counters = (size_t)decode_pass_counter_words(M, nkv);
    return ((counters * 4 + 255) / 256) * 256 + (size_t)M * (H / kDpChunk) * sizeof(float2);
}

cudaError_t launch_decode_pass(const DecodePassCall& c, cudaStream_t st) {
    if (!decode_pass_supported(c)) return cudaErrorInvalidValue;
    const int nsm = device_sm_count();
    DpParams prm;
    memset(&prm, 0, sizeof(prm));
    const int Dq = c.nq * c.hd, Dqkv = (c.nq + 2 * c.nkv) * c.hd;
    for (int l = 0; l < c.L; ++l) {
        if (!make_map_2d(&prm.wmap[l][0], c.layers[l].w_qkv, Dqkv, c.H, 256) ||
            !make_map_2d(&prm.wmap[l][1], c.layers[l].w_o, c.H, Dq, 256) ||
            !make_map_2d(&prm.wmap[l][2], c.layers[l].w_gate_up, 2 * c.F, c.H, 128) ||
            !make_map_2d(&prm.wmap[l][3], c.layers[l].w_down, c.H, c.F, 256))
            return cudaErrorInvalidValue;
        prm.layer[l].q_norm = c.layers[l].q_norm;
        prm.layer[l].k_norm = c.layers[l].k_norm;
        prm.layer[l].mlp_norm = c.layers[l].mlp_norm;
        prm.layer[l].next_norm = l + 1 < c.L ? c.layers[l + 1].attn_norm : c.final_norm;
        prm.layer[l].kv = c.layers[l].kv;
    }
    if (!make_map_2d(&prm.amap[0], c.y, c.M, c.H, 64) || !make_map_2d(&prm.amap[1], c.att, c.M, Dq, 64) ||
        !make_map_2d(&prm.amap[2], c.y, c.M, c.H, 64) || !make_map_2d(&prm.amap[3], c.h, c.M, c.F, 64))
        return cudaErrorInvalidValue;
    prm.g[0] = dp_plan(Dqkv / 256, c.H / 64, nsm, Dqkv, 32);
    prm.g[1] = dp_plan(c.H / 256, Dq / 64, nsm, c.H, 32);
    prm.g[2] = dp_plan(c.F / 128, c.H / 64, nsm, 2 * c.F, 4);
    prm.g[3] = dp_plan(c.H / 256, c.F / 64, nsm, c.H, 32);
    prm.L = c.L;
    prm.M = c.M;
    prm.H = c.H;
    prm.nq = c.nq;
    prm.nkv = c.nkv;
    prm.F = c.F;
    prm.Dq = Dq;
    prm.Dqkv = Dqkv;
    prm.n_slots = c.n_slots;
    prm.eps = c.eps;
    prm.rope = c.rope;
    prm.rope_rows = c.rope_rows;
    prm.rope_row_is_pos = c.rope_row_is_pos;
    prm.row_seq = c.row_seq;
    prm.row_pos = c.row_pos;
    prm.last_row = c.last_row;
    prm.n_out = c.n_out;
    prm.r = c.r;
    prm.y = c.y;
    prm.q = c.q;
    prm.att = c.att;
    prm.h = c.h;
    prm.out = c.out;
    prm.part = c.part;
    prm.apart = c.apart;
    // two units per SM at most: (row, kv head) items times key splits of >= 128 keys
    int splits = std::max(1, 2 * nsm / std::max(1, c.M * c.nkv));
    splits = std::min(splits, std::max(1, (c.max_pos + 1) / 128));
    splits = std::min(splits, std::max(1, c.attn_splits_max));
    prm.attn_splits = splits;
    prm.sync = c.sync;
    const size_t counters = (size_t)decode_pass_counter_words(c.M, c.nkv);
    prm.pairs = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(c.sync) + (counters * 4 + 255) / 256 * 256);
    prm.err = c.err;
    // every counter of the kernel starts at zero (the kernel leaves them at zero, the barrier aside)
    if (!c.sync_zeroed) {
        cudaError_t e = cudaMemsetAsync(c.sync, 0, counters * 4, st);
        if (e != cudaSuccess) return e;
    }
    return c.hd == 128 ? launch_dp_g<128>(prm, c.nq / c.nkv, nsm, st) : launch_dp_g<64>(prm, c.nq / c.nkv, nsm, st);
}

}  // namespace hra
