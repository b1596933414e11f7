// api.cu -- the extern "C" entry points declared in include/hra.h.
//
// Host orchestration only: argument validation (before the first launch), the workspace plan,
// and the stream-ordered kernel sequence of each operation.  No allocation, no synchronisation
// (except hra_device_error, which exists to synchronise).
//
// Prefill per layer ("flashrt-structures 0.2.0, prefill_tower/fp8_chain.py" page, its per-layer chain; "Stabilize
// Higgs Audio termination and prefill", Summary):
//   QKV GEMM -> q/k norm + RoPE + KV write -> causal attention -> o GEMM (+residual)
//   -> RMSNorm -> gate/up GEMM (+SwiGLU) -> down GEMM (+residual) -> RMSNorm (next layer / final)
// In the last layer only the rows that feed the last hidden are carried past the KV write
// (attention of the last query, o-projection, MLP and final norm of B rows), unless
// HRA_PREFILL_FULL_LAST_LAYER asks for every row.
#include <stdio.h>
#include <string.h>

#include <cmath>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

using namespace hra;

namespace {

std::atomic<uint64_t> g_launches{0};

// Event probe: brackets launches of one kernel class with CUDA event pairs (see hra.h).
struct Probe {
    std::mutex mu;
    int active = HRA_PROBE_NONE;
    std::vector<cudaEvent_t> pool;                 // 2 events per slot
    std::vector<std::pair<size_t, double>> used;   // (slot, flops)
} g_probe;

template <typename F>
cudaError_t probed(int cls, double flops, cudaStream_t st, F&& launch) {
    if (cls == HRA_PROBE_NONE || g_probe.active != cls) return launch();
    std::lock_guard<std::mutex> lk(g_probe.mu);
    const size_t slot = g_probe.used.size();
    while (g_probe.pool.size() < 2 * (slot + 1)) {
        cudaEvent_t e;
        cudaError_t err = cudaEventCreate(&e);
        if (err != cudaSuccess) return err;
        g_probe.pool.push_back(e);
    }
    cudaError_t err = cudaEventRecord(g_probe.pool[2 * slot], st);
    if (err != cudaSuccess) return err;
    err = launch();
    if (err != cudaSuccess) return err;
    err = cudaEventRecord(g_probe.pool[2 * slot + 1], st);
    if (err != cudaSuccess) return err;
    g_probe.used.emplace_back(slot, flops);
    return cudaSuccess;
}

constexpr size_t kAlign = 256;

inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

inline bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Region {
    size_t off = 0;
    size_t take(size_t bytes) {
        const size_t o = off;
        off += align_up(bytes);
        return o;
    }
};

// Offsets (bytes) of every buffer inside a caller workspace.
struct Layout {
    size_t err, row_seq, row_pos, cu, last_row, start, rope, r, y, qkv, q, att, h, rl, part, apart, x8, xs, sync, asched,
        total;
    size_t part_bytes;
    int attn_splits;
};

bool dims_ok(const hra_dims* d) {
    if (d == nullptr) return false;
    if (d->n_layers < 1 || d->hidden < 64 || d->hidden % 64 != 0) return false;
    if (d->head_dim != 64 && d->head_dim != 128) return false;
    if (d->n_q_heads < 1 || d->n_kv_heads < 1 || d->n_q_heads % d->n_kv_heads != 0) return false;
    const int g = d->n_q_heads / d->n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return false;
    if ((d->n_q_heads * d->head_dim) % 64 != 0 || d->ffn < 64 || d->ffn % 64 != 0) return false;
    if (d->vocab < 1) return false;
    if (!(d->rms_eps >= 0.f) || !(d->rope_theta > 0.f)) return false;
    return true;
}

bool audio_dims_ok(const hra_dims* d) {
    if (d == nullptr || d->hidden < 64 || d->hidden % 64 != 0) return false;
    if (d->n_codebooks < 1 || d->n_codebooks > 16) return false;
    if (d->codebook_size < 2 || (d->n_codebooks * d->codebook_size) % 8 != 0) return false;
    if (d->bos_id < 0 || d->bos_id >= d->codebook_size || d->eoc_id < 0 || d->eoc_id >= d->codebook_size)
        return false;
    return true;
}

// Shared plan of the backbone passes.  `rows` = packed rows that run the full layers, `last_rows`
// = rows of the last-layer tail (batch), `rope_rows` = rows of the RoPE table.
Layout backbone_layout(const hra_dims& d, int batch, int rows, int rope_rows, int max_pos, bool fp8 = false,
                      bool nvfp4 = false) {
    const size_t H = d.hidden, hd = d.head_dim, Dq = (size_t)d.n_q_heads * hd;
    const size_t Dqkv = (size_t)(d.n_q_heads + 2 * d.n_kv_heads) * hd, F = d.ffn;
    const size_t T = (size_t)std::max(rows, batch);
    Region g;
    Layout L;
    L.err = g.take(256);
    L.row_seq = g.take(T * 4);
    L.row_pos = g.take(T * 4);
    L.cu = g.take((size_t)(batch + 1) * 4);
    L.last_row = g.take((size_t)batch * 4);
    L.start = g.take((size_t)batch * 4);
    L.rope = g.take((size_t)rope_rows * (hd / 2) * sizeof(float2));
    L.r = g.take(T * H * 2);
    L.y = g.take(T * H * 2);
    L.qkv = g.take(T * Dqkv * 2);
    L.q = g.take(T * Dq * 2);
    L.att = g.take(T * Dq * 2);
    L.h = g.take(T * F * 2);
    L.rl = g.take((size_t)batch * H * 2);
    const int m_split = std::min(std::max(rows, batch), 128);
    size_t part = 0;
    part = std::max(part, linear_partial_bound(m_split, (int)Dqkv, (int)H, EPI_STORE));
    part = std::max(part, linear_partial_bound(m_split, (int)H, (int)Dq, EPI_RESIDUAL));
    part = std::max(part, linear_partial_bound(m_split, (int)F, (int)H, EPI_SWIGLU));
    part = std::max(part, linear_partial_bound(m_split, (int)H, (int)F, EPI_RESIDUAL));
    if (std::max(rows, batch) > 128) part = std::max(part, linear_tail_bound());
    L.part = g.take(part);
    L.part_bytes = part;
    L.attn_splits = decode_attention_splits(batch, d.n_kv_heads, max_pos);
    L.apart = g.take(decode_attention_scratch_bytes(batch, d.n_q_heads, d.head_dim, L.attn_splits));
    // FP8 variant: the E4M3 copy of the current projection's input (the widest input is the FFN's)
    L.x8 = (fp8 || nvfp4) ? g.take(T * std::max(std::max(H, Dq), F)) : 0;
    // NVFP4 band: the E4M3 block scales of that input (one per 16 elements)
    L.xs = nvfp4 ? g.take(T * std::max(std::max(H, Dq), F) / 16) : 0;
    // counters and per-row sums of the persistent decoder pass (M <= 64 rows), cleared by the
    // call's row-map kernel
    L.sync = g.take(decode_pass_sync_bytes((int)std::min<size_t>(T, 64), d.n_kv_heads, (int)F, (int)H));
    // the prefill attention's work list (built once per call)
    L.asched = g.take(attention_schedule_bytes((int)T, batch));
    L.total = g.off;
    return L;
}

struct Ptrs {
    uint8_t* base;
    template <typename T>
    T* at(size_t off) const { return reinterpret_cast<T*>(base + off); }
};

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return HRA_OK;
    return HRA_ERR_CUDA;
}

#define HRA_TRY(expr)                               \
    do {                                            \
        cudaError_t e_ = (expr);                    \
        if (e_ != cudaSuccess) return cuda_status(e_); \
    } while (0)

// FP8 variant / calibration of one layer's projections: `layers` (the E4M3 weights and scales) makes
// every projection quantize its input into x8 and run the FP8 GEMM; `amax` records max |input| of
// each projection (4 per layer: QKV, output, gate/up, down inputs).
struct QuantCtx {
    const hra_fp8_layer* layers;
    float* amax;
    uint8_t* x8;
    int layer;
    const hra_nvfp4_layer* nv4;   // NVFP4 band: QKV in FP8 from here, the other three in NVFP4
    uint8_t* xs;                  // block scales of the quantized input (NVFP4)
};
enum Proj : int { PROJ_QKV = 0, PROJ_O = 1, PROJ_GATE_UP = 2, PROJ_DOWN = 3 };

// norm_gain / norm_out: for EPI_RESIDUAL, the RMSNorm that follows (fused into a split-K reduction
// when the plan splits; otherwise run as its own kernel here).
cudaError_t linear(const bf16* a, const void* w, void* out, int M, int N, int K, int epi, const Ptrs& P,
                   const Layout& L, cudaStream_t st, int probe_class = HRA_PROBE_NONE,
                   const void* norm_gain = nullptr, bf16* norm_out = nullptr, float eps = 0.f,
                   const int32_t* norm_rows = nullptr, int norm_nrows = 0, const QkRopeArgs* qk = nullptr,
                   bool* qk_done = nullptr, const QuantCtx* qc = nullptr,
                   int proj = PROJ_QKV) {
    LinearCall c{};
    if (qc != nullptr && qc->amax != nullptr) {
        cudaError_t e = launch_absmax(a, (long long)M * K, qc->amax + 4 * qc->layer + proj, st);
        if (e != cudaSuccess) return e;
    }
    if (qc != nullptr && qc->nv4 != nullptr && proj != PROJ_QKV) {
        // NVFP4: the input to E2M1 codes + per-16 E4M3 block scales under its static global scale,
        // then the NVFP4 GEMM; the RMSNorm that follows a residual projection runs on its own
        const hra_nvfp4_layer& f = qc->nv4[qc->layer];
        cudaError_t e = launch_nvfp4_quantize(a, M, K, f.a_scale + proj, qc->x8, qc->xs, st);
        if (e != cudaSuccess) return e;
        Nvfp4Call n{};
        n.a_codes = qc->x8;
        n.a_scales = qc->xs;
        n.w_codes = reinterpret_cast<const uint8_t*>(f.codes[proj]);
        n.w_scales = reinterpret_cast<const uint8_t*>(f.scales[proj]);
        n.g_a = f.a_scale + proj;
        n.g_w = f.w_scale + proj;
        n.out = out;
        n.err = P.at<unsigned int>(L.err);
        n.M = M;
        n.N = N;
        n.K = K;
        n.epi = epi;
        const double n_w = epi == EPI_SWIGLU ? 2.0 * N : (double)N;
        const int cls = probe_class == HRA_PROBE_GATE_UP ? HRA_PROBE_GATE_UP : HRA_PROBE_NONE;
        e = probed(cls, 2.0 * M * (double)K * n_w, st, [&] { return launch_linear_nvfp4(n, st); });
        if (e != cudaSuccess || norm_out == nullptr) return e;
        return launch_rmsnorm(reinterpret_cast<const bf16*>(out), norm_rows, reinterpret_cast<const bf16*>(norm_gain),
                              norm_out, nullptr, norm_rows ? norm_nrows : M, N, eps, st);
    }
    if (qc != nullptr && qc->nv4 != nullptr) {   // the band's QKV: static FP8
        const hra_nvfp4_layer& f = qc->nv4[qc->layer];
        cudaError_t e = launch_fp8_quantize(a, (long long)M * K, f.a_scale, qc->x8, st);
        if (e != cudaSuccess) return e;
        a = reinterpret_cast<const bf16*>(qc->x8);
        w = f.w_qkv;
        c.fp8 = true;
        c.a_scale = f.a_scale;
        c.w_scale = f.w_scale;
    } else if (qc != nullptr && qc->layers != nullptr) {
        const hra_fp8_layer& f = qc->layers[qc->layer];
        const void* w8s[4] = {f.w_qkv, f.w_o, f.w_gate_up, f.w_down};
        cudaError_t e = launch_fp8_quantize(a, (long long)M * K, f.a_scale + proj, qc->x8, st);
        if (e != cudaSuccess) return e;
        a = reinterpret_cast<const bf16*>(qc->x8);   // E4M3 codes from here on
        w = w8s[proj];
        c.fp8 = true;
        c.a_scale = f.a_scale + proj;
        c.w_scale = f.w_scale + proj;
    }
    c.qk = qk;
    c.qk_done = qk_done;
    c.a = a;
    c.w = reinterpret_cast<const bf16*>(w);
    c.out = out;
    c.M = M;
    c.N = N;
    c.K = K;
    c.epi = epi;
    c.split_req = 0;
    c.partial = P.at<float>(L.part);
    c.err = P.at<unsigned int>(L.err);
    bool norm_done = false;
    if (norm_out != nullptr && norm_rows == nullptr) {
        c.norm_gain = reinterpret_cast<const bf16*>(norm_gain);
        c.norm_out = norm_out;
        c.norm_eps = eps;
        c.norm_done = &norm_done;
    }
    const double n_w = epi == EPI_SWIGLU ? 2.0 * N : (double)N;   // weight rows
    const double work = probe_class == HRA_PROBE_DECODE_LINEAR ? 2.0 * K * n_w : 2.0 * M * (double)K * n_w;
    cudaError_t e = probed(probe_class, work, st, [&] { return launch_linear(c, st); });
    if (e != cudaSuccess || norm_out == nullptr || norm_done) return e;
    return launch_rmsnorm(reinterpret_cast<const bf16*>(out), norm_rows, reinterpret_cast<const bf16*>(norm_gain),
                          norm_out, nullptr, norm_rows ? norm_nrows : M, N, eps, st);
}

bool layer_ptrs_ok(const hra_layer_weights& l) {
    return aligned16(l.attn_norm) && aligned16(l.w_qkv) && aligned16(l.q_norm) && aligned16(l.k_norm) &&
           aligned16(l.w_o) && aligned16(l.mlp_norm) && aligned16(l.w_gate_up) && aligned16(l.w_down);
}

// One full layer (attention block + MLP) over `rows` packed rows; leaves the residual in r.
// `attn_last_only` switches the tail to the B-row path (prefill's last layer).
int run_layers(const hra_dims& d, const hra_weights& w, const hra_kv_cache& kv, const Ptrs& P, const Layout& L,
               int rows, int batch, int max_len, bool prefill, bool full_last, bf16* out_hidden,
               const int32_t* seq_lens_host, int max_pos, cudaStream_t st, int rope_rows = 0,
               const int32_t* start_host = nullptr, const hra_fp8_layer* fp8 = nullptr, float* amax = nullptr,
               const hra_nvfp4_layer* nv4 = nullptr) {
    const int H = d.hidden, hd = d.head_dim, nq = d.n_q_heads, nkv = d.n_kv_heads, F = d.ffn;
    const int Dq = nq * hd, Dqkv = (nq + 2 * nkv) * hd;
    const float eps = d.rms_eps;
    bf16* r = P.at<bf16>(L.r);
    bf16* y = P.at<bf16>(L.y);
    bf16* qkv = P.at<bf16>(L.qkv);
    bf16* q = P.at<bf16>(L.q);
    bf16* att = P.at<bf16>(L.att);
    bf16* h = P.at<bf16>(L.h);
    bf16* rl = P.at<bf16>(L.rl);
    const int32_t* row_seq = P.at<int32_t>(L.row_seq);
    const int32_t* row_pos = P.at<int32_t>(L.row_pos);
    const int32_t* last_row = P.at<int32_t>(L.last_row);
    const size_t layer_elems = (size_t)kv.batch * 2 * nkv * (size_t)kv.n_slots * hd;
    // prefill: causal QK^T + PV FLOPs over the used keys, 4 nq hd sum_b (len_b s_b + len_b (len_b + 1) / 2)
    // with s_b the cached positions before the sequence's rows;
    // decode (seq_lens_host = positions): K/V bytes read, 4 nkv hd sum_b (pos_b + 1)
    double attn_work = 0.0;
    for (int b = 0; b < batch && seq_lens_host != nullptr; ++b) {
        const double n = (double)seq_lens_host[b];
        const double s0 = start_host ? (double)start_host[b] : 0.0;
        attn_work += prefill ? 4.0 * nq * hd * (n * s0 + n * (n + 1.0) / 2.0) : 4.0 * nkv * hd * (n + 1.0);
    }
    const int lin_probe = prefill ? 0 : HRA_PROBE_DECODE_LINEAR;

    // At most 64 rows in BF16, when selected (hra_set_decode_pass): the whole pass is one persistent
    // kernel (decode_pass.cu).  Every row runs every layer; the final norm goes to the last row of
    // each sequence (prefill) or to every row (decode).
    if (g_decode_pass_enabled && rows <= 64 && fp8 == nullptr && amax == nullptr && nv4 == nullptr &&
        d.n_layers <= kDecodePassMaxLayers) {
        DecodePassCall c{};
        for (int l = 0; l < d.n_layers; ++l) {
            const hra_layer_weights& lw = w.layers[l];
            DecodePassLayer& dl = c.layers[l];
            dl.w_qkv = reinterpret_cast<const bf16*>(lw.w_qkv);
            dl.w_o = reinterpret_cast<const bf16*>(lw.w_o);
            dl.w_gate_up = reinterpret_cast<const bf16*>(lw.w_gate_up);
            dl.w_down = reinterpret_cast<const bf16*>(lw.w_down);
            dl.attn_norm = reinterpret_cast<const bf16*>(lw.attn_norm);
            dl.q_norm = reinterpret_cast<const bf16*>(lw.q_norm);
            dl.k_norm = reinterpret_cast<const bf16*>(lw.k_norm);
            dl.mlp_norm = reinterpret_cast<const bf16*>(lw.mlp_norm);
            dl.kv = reinterpret_cast<bf16*>(kv.base) + (size_t)l * layer_elems;
        }
        c.final_norm = reinterpret_cast<const bf16*>(w.final_norm);
        c.L = d.n_layers;
        c.M = rows;
        c.H = H;
        c.nq = nq;
        c.nkv = nkv;
        c.hd = hd;
        c.F = F;
        c.n_slots = kv.n_slots;
        c.eps = eps;
        c.rope = P.at<float2>(L.rope);
        c.rope_rows = prefill ? rope_rows : batch;
        c.rope_row_is_pos = prefill ? 1 : 0;
        c.row_seq = row_seq;
        c.row_pos = row_pos;
        c.last_row = prefill ? last_row : nullptr;
        c.n_out = prefill ? batch : rows;
        int mp = 0;
        for (int b = 0; b < batch && seq_lens_host != nullptr; ++b)
            mp = std::max(mp, prefill ? (start_host ? start_host[b] : 0) + seq_lens_host[b] - 1 : seq_lens_host[b]);
        c.max_pos = seq_lens_host != nullptr ? mp : max_pos;
        c.r = r;
        c.y = y;
        c.q = q;
        c.att = att;
        c.h = h;
        c.out = out_hidden;
        c.part = P.at<float>(L.part);
        c.part_bytes = L.part_bytes;
        c.apart = P.at<float>(L.apart);
        // the attention scratch holds L.attn_splits splits of `batch` rows
        c.attn_splits_max = std::max(1, L.attn_splits * batch / std::max(1, rows));
        c.sync = P.at<unsigned int>(L.sync);
        c.sync_zeroed = true;   // cleared by the call's row-map kernel
        c.err = P.at<unsigned int>(L.err);
        if (decode_pass_supported(c)) {
            HRA_TRY(launch_decode_pass(c, st));
            return HRA_OK;
        }
    }

    // the prefill attention's work list: the same sequences for every layer (a single sequence needs
    // none: its query tiles in order)
    if (prefill && batch > 1 && (d.n_layers > 1 || full_last))
        HRA_TRY(launch_attention_schedule(P.at<int32_t>(L.cu), P.at<int32_t>(L.start), batch, max_len, nq, nkv,
                                          P.at<int32_t>(L.asched), st));

    for (int l = 0; l < d.n_layers; ++l) {
        const hra_layer_weights& lw = w.layers[l];
        bf16* kvl = reinterpret_cast<bf16*>(kv.base) + (size_t)l * layer_elems;
        const bool last = l == d.n_layers - 1;
        const QuantCtx qc{fp8, amax, (fp8 || nv4) ? P.at<uint8_t>(L.x8) : nullptr, l, nv4,
                          nv4 ? P.at<uint8_t>(L.xs) : nullptr};
        const QuantCtx* qcp = (fp8 != nullptr || amax != nullptr || nv4 != nullptr) ? &qc : nullptr;
        QkRopeArgs qa{};
        qa.qkv = qkv;
        qa.q_norm = reinterpret_cast<const bf16*>(lw.q_norm);
        qa.k_norm = reinterpret_cast<const bf16*>(lw.k_norm);
        qa.rope = P.at<float2>(L.rope);
        qa.rope_rows = prefill ? rope_rows : batch;
        qa.row_seq = row_seq;
        qa.row_pos = row_pos;
        qa.rope_row_is_pos = prefill ? 1 : 0;
        qa.q_out = q;
        qa.kv_layer = kvl;
        qa.n_slots = kv.n_slots;
        qa.rows = rows;
        qa.nq = nq;
        qa.nkv = nkv;
        qa.hd = hd;
        qa.eps = eps;
        bool qk_done = false;
        HRA_TRY(linear(y, lw.w_qkv, qkv, rows, Dqkv, H, EPI_STORE, P, L, st, prefill ? HRA_PROBE_QKV : lin_probe, nullptr,
                       nullptr, 0.f, nullptr, 0, &qa, &qk_done, qcp, PROJ_QKV));
        if (!qk_done) HRA_TRY(launch_qk_rope_kv(qa, st));

        const bool tail = prefill && last && !full_last;
        if (!tail) {
            if (prefill) {
                PrefillAttnArgs pa{q, kvl, P.at<int32_t>(L.cu), P.at<int32_t>(L.start), att, batch, max_len,
                                   kv.n_slots, nq, nkv, hd, rows, kv.batch, P.at<unsigned int>(L.err),
                                   batch > 1 ? P.at<int32_t>(L.asched) : nullptr};
                HRA_TRY(probed(HRA_PROBE_ATTENTION, attn_work, st, [&] {
                    return launch_prefill_attention_tc(pa, st);
                }));
            } else {
                DecodeAttnArgs da{};
                da.q = q;
                da.kv_layer = kvl;
                da.q_row = nullptr;
                da.seq = row_seq;
                da.pos = row_pos;
                da.out = att;
                da.part = P.at<float>(L.apart);
                da.rows = rows;
                da.max_pos = max_pos;
                da.n_slots = kv.n_slots;
                da.nq = nq;
                da.nkv = nkv;
                da.hd = hd;
                da.splits = std::min(L.attn_splits, decode_attention_splits(rows, nkv, max_pos));
                HRA_TRY(probed(HRA_PROBE_DECODE_ATTENTION, attn_work, st,
                               [&] { return launch_decode_attention(da, st); }));
            }
            HRA_TRY(linear(att, lw.w_o, r, rows, H, Dq, EPI_RESIDUAL, P, L, st,
                           prefill ? HRA_PROBE_O_PROJ : lin_probe, lw.mlp_norm, y, eps, nullptr, 0, nullptr,
                           nullptr, qcp, PROJ_O));
            HRA_TRY(linear(y, lw.w_gate_up, h, rows, F, H, EPI_SWIGLU, P, L, st,
                           prefill ? HRA_PROBE_GATE_UP : lin_probe, nullptr, nullptr, 0.f, nullptr, 0, nullptr,
                           nullptr, qcp, PROJ_GATE_UP));
            if (!last) {
                HRA_TRY(linear(h, lw.w_down, r, rows, H, F, EPI_RESIDUAL, P, L, st,
                               prefill ? HRA_PROBE_DOWN : lin_probe, w.layers[l + 1].attn_norm, y, eps, nullptr, 0,
                               nullptr, nullptr, qcp, PROJ_DOWN));
            } else if (!prefill) {
                HRA_TRY(linear(h, lw.w_down, r, rows, H, F, EPI_RESIDUAL, P, L, st, lin_probe, w.final_norm,
                               out_hidden, eps, nullptr, 0, nullptr, nullptr, qcp, PROJ_DOWN));
            } else {
                HRA_TRY(linear(h, lw.w_down, r, rows, H, F, EPI_RESIDUAL, P, L, st, HRA_PROBE_DOWN,
                               w.final_norm, out_hidden, eps, last_row, batch, nullptr, nullptr, qcp,
                               PROJ_DOWN));
            }
        } else {
            // last prefill layer, rows that feed the last hidden only
            DecodeAttnArgs da{};
            da.q = q;
            da.kv_layer = kvl;
            da.q_row = last_row;
            da.seq = row_seq;
            da.pos = row_pos;
            da.out = att;
            da.part = P.at<float>(L.apart);
            da.rows = batch;
            da.max_pos = max_pos;
            da.n_slots = kv.n_slots;
            da.nq = nq;
            da.nkv = nkv;
            da.hd = hd;
            da.splits = std::min(L.attn_splits, decode_attention_splits(batch, nkv, max_pos));
            HRA_TRY(launch_decode_attention(da, st));
            HRA_TRY(launch_rmsnorm(r, last_row, nullptr, nullptr, rl, batch, H, eps, st));   // gather
            HRA_TRY(linear(att, lw.w_o, rl, batch, H, Dq, EPI_RESIDUAL, P, L, st, 0, lw.mlp_norm, y, eps, nullptr, 0,
                           nullptr, nullptr, qcp, PROJ_O));
            HRA_TRY(linear(y, lw.w_gate_up, h, batch, F, H, EPI_SWIGLU, P, L, st, 0, nullptr, nullptr, 0.f, nullptr, 0,
                           nullptr, nullptr, qcp, PROJ_GATE_UP));
            HRA_TRY(linear(h, lw.w_down, rl, batch, H, F, EPI_RESIDUAL, P, L, st, 0, w.final_norm, out_hidden, eps,
                           nullptr, 0, nullptr, nullptr, qcp, PROJ_DOWN));
        }
    }
    return HRA_OK;
}

bool weights_ok(const hra_dims& d, const hra_weights* w) {
    if (w == nullptr || w->layers == nullptr || !aligned16(w->final_norm)) return false;
    for (int l = 0; l < d.n_layers; ++l)
        if (!layer_ptrs_ok(w->layers[l])) return false;
    return true;
}

bool kv_ok(const hra_kv_cache* kv) {
    return kv != nullptr && aligned16(kv->base) && kv->batch >= 1 && kv->n_slots >= 1;
}

}  // namespace

namespace hra {
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace hra

extern "C" {

uint64_t hra_launch_counter(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t hra_set_decode_pass(int32_t enable) {
    const bool prev = hra::g_decode_pass_enabled;
    hra::g_decode_pass_enabled = enable != 0;
    return prev ? 1 : 0;
}

int32_t hra_set_gemm_pairs(int32_t enable) {
    const bool prev = hra::g_gemm_pairs;
    hra::g_gemm_pairs = enable != 0;
    return prev ? 1 : 0;
}

int hra_probe_select(int kernel_class) {
    std::lock_guard<std::mutex> lk(g_probe.mu);
    g_probe.active = kernel_class;
    return HRA_OK;
}

int hra_probe_collect(double* total_ms, int64_t* launches, double* total_work) {
    std::lock_guard<std::mutex> lk(g_probe.mu);
    double ms = 0.0, fl = 0.0;
    for (const auto& u : g_probe.used) {
        if (cudaEventSynchronize(g_probe.pool[2 * u.first + 1]) != cudaSuccess) return HRA_ERR_CUDA;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, g_probe.pool[2 * u.first], g_probe.pool[2 * u.first + 1]) != cudaSuccess)
            return HRA_ERR_CUDA;
        ms += t;
        fl += u.second;
    }
    if (total_ms) *total_ms = ms;
    if (launches) *launches = (int64_t)g_probe.used.size();
    if (total_work) *total_work = fl;
    g_probe.used.clear();
    return HRA_OK;
}


size_t hra_prefill_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens, int32_t max_len) {
    return hra_prefill_chunk_workspace_size(dims, batch, total_tokens, max_len, max_len);
}

size_t hra_prefill_chunk_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens, int32_t max_len,
                                        int32_t max_end) {
    if (!dims_ok(dims) || batch < 1 || total_tokens < batch || max_len < 1 || max_end < max_len) return 0;
    return backbone_layout(*dims, batch, total_tokens, max_end, max_end - 1).total;
}

namespace {

constexpr int H_ALIGN_FP8(int k) { return k % 128; }

int prefill_impl(const hra_dims* dims, const hra_weights* weights, const int32_t* tokens_dev, const int32_t* seq_lens,
                 const int32_t* start_pos, int32_t batch, int32_t max_len, const hra_kv_cache* kv,
                 void* last_hidden_dev, void* workspace, size_t workspace_bytes, uint32_t flags, void* stream,
                 const hra_fp8_layer* fp8 = nullptr, float* amax = nullptr, bool validate_only = false,
                 const hra_nvfp4_layer* nv4 = nullptr) {
    if (dims == nullptr || weights == nullptr || tokens_dev == nullptr || seq_lens == nullptr || kv == nullptr)
        return HRA_ERR_INVALID_ARG;
    if (!dims_ok(dims)) return HRA_ERR_UNSUPPORTED;
    const hra_dims& d = *dims;
    if (batch < 1 || batch > kMaxBatch || max_len < 1) return HRA_ERR_INVALID_ARG;
    if (!aligned16(weights->embed) || !weights_ok(d, weights) || !kv_ok(kv) || !aligned16(last_hidden_dev) ||
        !aligned16(workspace) || (reinterpret_cast<uintptr_t>(tokens_dev) & 3u) != 0)
        return HRA_ERR_INVALID_ARG;
    if (batch > kv->batch) return HRA_ERR_INVALID_ARG;
    SeqMeta meta{};
    meta.batch = batch;
    meta.mode = 0;
    long long T = 0;
    int max_end = 1;
    for (int b = 0; b < batch; ++b) {
        const int n = seq_lens[b];
        const int s0 = start_pos ? start_pos[b] : 0;
        if (n < 1 || n > max_len || s0 < 0 || (long long)s0 + n > kv->n_slots) return HRA_ERR_RANGE;
        meta.vals[b] = (int32_t)T;
        meta.start[b] = s0;
        T += n;
        max_end = std::max(max_end, s0 + n);
    }
    meta.vals[batch] = (int32_t)T;
    if (T > (1 << 30)) return HRA_ERR_RANGE;
    if (fp8 != nullptr) {
        if ((H_ALIGN_FP8(d.hidden) | H_ALIGN_FP8(d.n_q_heads * d.head_dim) | H_ALIGN_FP8(d.ffn)) != 0)
            return HRA_ERR_UNSUPPORTED;   // FP8 K blocks are 128 elements
        for (int l = 0; l < d.n_layers; ++l) {
            const hra_fp8_layer& f = fp8[l];
            if (!aligned16(f.w_qkv) || !aligned16(f.w_o) || !aligned16(f.w_gate_up) || !aligned16(f.w_down) ||
                f.w_scale == nullptr || f.a_scale == nullptr || (reinterpret_cast<uintptr_t>(f.w_scale) & 3u) ||
                (reinterpret_cast<uintptr_t>(f.a_scale) & 3u))
                return HRA_ERR_INVALID_ARG;
        }
    }
    if (nv4 != nullptr) {
        if (H_ALIGN_FP8(d.hidden) != 0) return HRA_ERR_UNSUPPORTED;   // the band's FP8 QKV: 128-element K blocks
        for (int l = 0; l < d.n_layers; ++l) {
            const hra_nvfp4_layer& f = nv4[l];
            if (!aligned16(f.w_qkv) || f.w_scale == nullptr || f.a_scale == nullptr ||
                (reinterpret_cast<uintptr_t>(f.w_scale) & 3u) || (reinterpret_cast<uintptr_t>(f.a_scale) & 3u))
                return HRA_ERR_INVALID_ARG;
            for (int p = 1; p < 4; ++p)
                if (!aligned16(f.codes[p]) || f.scales[p] == nullptr) return HRA_ERR_INVALID_ARG;
        }
    }
    const Layout L = backbone_layout(d, batch, (int)T, max_end, max_end - 1, fp8 != nullptr, nv4 != nullptr);
    if (workspace_bytes < L.total) return HRA_ERR_WORKSPACE;
    if (validate_only) return HRA_OK;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Ptrs P{reinterpret_cast<uint8_t*>(workspace)};
    HRA_TRY(launch_build_rowmap(meta, (int)T, P.at<int32_t>(L.row_seq), P.at<int32_t>(L.row_pos),
                                P.at<int32_t>(L.cu), P.at<int32_t>(L.last_row), P.at<int32_t>(L.start),
                                P.at<unsigned int>(L.err), st, P.at<unsigned int>(L.sync),
                                decode_pass_counter_words(std::min((int)T, 64), d.n_kv_heads)));
    HRA_TRY(launch_rope_table(max_end, nullptr, d.head_dim, (double)d.rope_theta, P.at<float2>(L.rope), st));
    HRA_TRY(launch_embed_rmsnorm(tokens_dev, max_len, P.at<int32_t>(L.row_seq), P.at<int32_t>(L.cu),
                                 reinterpret_cast<const bf16*>(weights->embed), d.vocab,
                                 reinterpret_cast<const bf16*>(weights->layers[0].attn_norm), P.at<bf16>(L.r),
                                 P.at<bf16>(L.y), (int)T, d.hidden, d.rms_eps, P.at<unsigned int>(L.err), st));
    return run_layers(d, *weights, *kv, P, L, (int)T, batch, max_len, true,
                      (flags & HRA_PREFILL_FULL_LAST_LAYER) != 0, reinterpret_cast<bf16*>(last_hidden_dev), seq_lens,
                      max_end - 1, st, max_end, start_pos, fp8, amax, nv4);
}

}  // namespace

int hra_prefill(const hra_dims* dims, const hra_weights* weights, const int32_t* tokens_dev,
                const int32_t* seq_lens, int32_t batch, int32_t max_len, const hra_kv_cache* kv,
                void* last_hidden_dev, void* workspace, size_t workspace_bytes, uint32_t flags, void* stream) {
    return prefill_impl(dims, weights, tokens_dev, seq_lens, nullptr, batch, max_len, kv, last_hidden_dev, workspace,
                        workspace_bytes, flags, stream);
}

int hra_prefill_chunk(const hra_dims* dims, const hra_weights* weights, const int32_t* tokens_dev,
                      const int32_t* seq_lens, const int32_t* start_pos, int32_t batch, int32_t max_len,
                      const hra_kv_cache* kv, void* last_hidden_dev, void* workspace, size_t workspace_bytes,
                      uint32_t flags, void* stream) {
    if (start_pos == nullptr) return HRA_ERR_INVALID_ARG;
    return prefill_impl(dims, weights, tokens_dev, seq_lens, start_pos, batch, max_len, kv, last_hidden_dev,
                        workspace, workspace_bytes, flags, stream);
}

size_t hra_prefill_fp8_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens, int32_t max_len) {
    if (!dims_ok(dims) || batch < 1 || total_tokens < batch || max_len < 1) return 0;
    return backbone_layout(*dims, batch, total_tokens, max_len, max_len - 1, true).total;
}

int hra_prefill_fp8(const hra_dims* dims, const hra_weights* weights, const hra_fp8_layer* fp8_layers,
                    const int32_t* tokens_dev, const int32_t* seq_lens, int32_t batch, int32_t max_len,
                    const hra_kv_cache* kv, void* last_hidden_dev, void* workspace, size_t workspace_bytes,
                    uint32_t flags, void* stream) {
    if (fp8_layers == nullptr) return HRA_ERR_INVALID_ARG;
    return prefill_impl(dims, weights, tokens_dev, seq_lens, nullptr, batch, max_len, kv, last_hidden_dev, workspace,
                        workspace_bytes, flags, stream, fp8_layers, nullptr);
}

size_t hra_prefill_nvfp4_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens, int32_t max_len) {
    if (!dims_ok(dims) || batch < 1 || total_tokens < batch || max_len < 1) return 0;
    return backbone_layout(*dims, batch, total_tokens, max_len, max_len - 1, false, true).total;
}

int hra_prefill_nvfp4(const hra_dims* dims, const hra_weights* weights, const hra_nvfp4_layer* nvfp4_layers,
                      const int32_t* tokens_dev, const int32_t* seq_lens, int32_t batch, int32_t max_len,
                      const hra_kv_cache* kv, void* last_hidden_dev, void* workspace, size_t workspace_bytes,
                      uint32_t flags, void* stream) {
    if (nvfp4_layers == nullptr) return HRA_ERR_INVALID_ARG;
    return prefill_impl(dims, weights, tokens_dev, seq_lens, nullptr, batch, max_len, kv, last_hidden_dev, workspace,
                        workspace_bytes, flags, stream, nullptr, nullptr, false, nvfp4_layers);
}

int hra_nvfp4_quantize_weight(const void* w_dev, int32_t rows, int32_t K, void* codes_dev, void* scales_dev,
                              float* g_dev, void* stream) {
    if (!aligned16(w_dev) || !aligned16(codes_dev) || scales_dev == nullptr || g_dev == nullptr ||
        (reinterpret_cast<uintptr_t>(g_dev) & 3u) || rows < 1 || K < 16 || K % 16 != 0)
        return HRA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bf16* w = reinterpret_cast<const bf16*>(w_dev);
    HRA_TRY(launch_zero_floats(g_dev, 1, st));
    HRA_TRY(launch_absmax(w, (long long)rows * K, g_dev, st));
    HRA_TRY(launch_amax_div(g_dev, g_dev, 1, 6.0f * 448.0f, st));   // g = max|w| / (6 * 448), 1 if 0
    HRA_TRY(launch_nvfp4_quantize(w, rows, K, g_dev, reinterpret_cast<uint8_t*>(codes_dev),
                                  reinterpret_cast<uint8_t*>(scales_dev), st));
    return HRA_OK;
}

int hra_nvfp4_band_scales(const float* amax_dev, float* scale_dev, int32_t n_layers, void* stream) {
    if (amax_dev == nullptr || scale_dev == nullptr || (reinterpret_cast<uintptr_t>(amax_dev) & 3u) ||
        (reinterpret_cast<uintptr_t>(scale_dev) & 3u) || n_layers < 1)
        return HRA_ERR_INVALID_ARG;
    HRA_TRY(launch_nvfp4_band_scales(amax_dev, scale_dev, n_layers, reinterpret_cast<cudaStream_t>(stream)));
    return HRA_OK;
}

size_t hra_linear_nvfp4_workspace_size(void) { return 256; }

int hra_linear_nvfp4(const void* a_codes_dev, const void* a_scales_dev, const void* w_codes_dev,
                     const void* w_scales_dev, void* out_dev, int32_t M, int32_t N, int32_t K, const float* g_a_dev,
                     const float* g_w_dev, int32_t epilogue, void* workspace, size_t workspace_bytes, void* stream) {
    if (!aligned16(a_codes_dev) || !aligned16(w_codes_dev) || a_scales_dev == nullptr || w_scales_dev == nullptr ||
        !aligned16(out_dev) || !aligned16(workspace) || g_a_dev == nullptr || g_w_dev == nullptr ||
        (reinterpret_cast<uintptr_t>(g_a_dev) & 3u) || (reinterpret_cast<uintptr_t>(g_w_dev) & 3u))
        return HRA_ERR_INVALID_ARG;
    if (M < 1 || N < 8 || N % 8 != 0 || K < 64 || K % 64 != 0) return HRA_ERR_INVALID_ARG;
    if (epilogue < EPI_STORE || epilogue > EPI_F32) return HRA_ERR_INVALID_ARG;
    if (workspace_bytes < hra_linear_nvfp4_workspace_size()) return HRA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    HRA_TRY(cudaMemsetAsync(workspace, 0, 4, st));
    Nvfp4Call n{};
    n.a_codes = reinterpret_cast<const uint8_t*>(a_codes_dev);
    n.a_scales = reinterpret_cast<const uint8_t*>(a_scales_dev);
    n.w_codes = reinterpret_cast<const uint8_t*>(w_codes_dev);
    n.w_scales = reinterpret_cast<const uint8_t*>(w_scales_dev);
    n.g_a = g_a_dev;
    n.g_w = g_w_dev;
    n.out = out_dev;
    n.err = reinterpret_cast<unsigned int*>(workspace);
    n.M = M;
    n.N = N;
    n.K = K;
    n.epi = epilogue;
    HRA_TRY(launch_linear_nvfp4(n, st));
    return HRA_OK;
}

size_t hra_fp8_calibrate_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens, int32_t max_len) {
    const size_t pf = hra_prefill_workspace_size(dims, batch, total_tokens, max_len);
    if (pf == 0) return 0;
    return align_up(pf) + align_up((size_t)batch * dims->hidden * 2);
}

int hra_fp8_calibrate(const hra_dims* dims, const hra_weights* weights, const int32_t* tokens_dev,
                      const int32_t* seq_lens, int32_t batch, int32_t max_len, const hra_kv_cache* kv,
                      float* amax_dev, float* scale_dev, void* workspace, size_t workspace_bytes, void* stream) {
    if (dims == nullptr || seq_lens == nullptr || amax_dev == nullptr || scale_dev == nullptr ||
        (reinterpret_cast<uintptr_t>(amax_dev) & 3u) || (reinterpret_cast<uintptr_t>(scale_dev) & 3u))
        return HRA_ERR_INVALID_ARG;
    if (!dims_ok(dims)) return HRA_ERR_UNSUPPORTED;
    if (batch < 1 || batch > kMaxBatch) return HRA_ERR_INVALID_ARG;
    long long T = 0;
    for (int b = 0; b < batch; ++b) T += seq_lens[b];
    if (T < batch || T > (1 << 30)) return HRA_ERR_RANGE;
    const size_t need = hra_fp8_calibrate_workspace_size(dims, batch, (int32_t)T, max_len);
    if (need == 0) return HRA_ERR_INVALID_ARG;
    if (workspace_bytes < need) return HRA_ERR_WORKSPACE;
    const size_t pf = align_up(hra_prefill_workspace_size(dims, batch, (int32_t)T, max_len));
    void* last = reinterpret_cast<uint8_t*>(workspace) + pf;
    // the bf16 prefill with every row through the last layer, recording max |input| per projection
    int rc = prefill_impl(dims, weights, tokens_dev, seq_lens, nullptr, batch, max_len, kv, last, workspace, pf,
                          HRA_PREFILL_FULL_LAST_LAYER, stream, nullptr, amax_dev, /*validate_only=*/true);
    if (rc != HRA_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int n = 4 * dims->n_layers;
    HRA_TRY(launch_zero_floats(amax_dev, n, st));
    rc = prefill_impl(dims, weights, tokens_dev, seq_lens, nullptr, batch, max_len, kv, last, workspace, pf,
                      HRA_PREFILL_FULL_LAST_LAYER, stream, nullptr, amax_dev);
    if (rc != HRA_OK) return rc;
    HRA_TRY(launch_amax_to_scale(amax_dev, scale_dev, n, st));
    return HRA_OK;
}

int hra_fp8_quantize_weight(const void* w_dev, int64_t n, void* w8_dev, float* scale_dev, void* stream) {
    if (!aligned16(w_dev) || w8_dev == nullptr || (reinterpret_cast<uintptr_t>(w8_dev) & 7u) || scale_dev == nullptr ||
        (reinterpret_cast<uintptr_t>(scale_dev) & 3u) || n < 8 || n % 8 != 0)
        return HRA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    HRA_TRY(launch_zero_floats(scale_dev, 1, st));
    HRA_TRY(launch_absmax(reinterpret_cast<const bf16*>(w_dev), n, scale_dev, st));
    HRA_TRY(launch_amax_to_scale(scale_dev, scale_dev, 1, st));
    HRA_TRY(launch_fp8_quantize(reinterpret_cast<const bf16*>(w_dev), n, scale_dev, reinterpret_cast<uint8_t*>(w8_dev),
                                st));
    return HRA_OK;
}

int hra_nvfp4_quantize(const void* x_dev, int32_t rows, int32_t K, const float* g_dev, void* codes_dev,
                       void* scales_dev, void* stream) {
    if (!aligned16(x_dev) || !aligned16(codes_dev) || scales_dev == nullptr || g_dev == nullptr ||
        (reinterpret_cast<uintptr_t>(g_dev) & 3u) || rows < 1 || K < 16 || K % 16 != 0)
        return HRA_ERR_INVALID_ARG;
    HRA_TRY(launch_nvfp4_quantize(reinterpret_cast<const bf16*>(x_dev), rows, K, g_dev,
                                  reinterpret_cast<uint8_t*>(codes_dev), reinterpret_cast<uint8_t*>(scales_dev),
                                  reinterpret_cast<cudaStream_t>(stream)));
    return HRA_OK;
}

int hra_fp8_quantize(const void* x_dev, int64_t n, const float* scale_dev, void* x8_dev, void* stream) {
    if (!aligned16(x_dev) || x8_dev == nullptr || (reinterpret_cast<uintptr_t>(x8_dev) & 7u) || scale_dev == nullptr ||
        (reinterpret_cast<uintptr_t>(scale_dev) & 3u) || n < 8 || n % 8 != 0)
        return HRA_ERR_INVALID_ARG;
    HRA_TRY(launch_fp8_quantize(reinterpret_cast<const bf16*>(x_dev), n, scale_dev, reinterpret_cast<uint8_t*>(x8_dev),
                                reinterpret_cast<cudaStream_t>(stream)));
    return HRA_OK;
}

size_t hra_decode_workspace_size(const hra_dims* dims, int32_t batch, int32_t n_slots) {
    if (!dims_ok(dims) || batch < 1 || n_slots < 1) return 0;
    return backbone_layout(*dims, batch, batch, batch, n_slots - 1).total;
}

namespace {

// pos_host: host positions (validated here); otherwise pos_dev (device, checked on the device) with
// pos_bound, a host upper bound of every position, for the attention split count.
int decode_impl(const hra_dims* dims, const hra_weights* weights, const void* in_emb_dev, const int32_t* pos_host,
                int32_t* pos_dev, int32_t pos_bound, int advance, int32_t batch, const hra_kv_cache* kv,
                void* hidden_dev, void* workspace, size_t workspace_bytes, void* stream, bool validate_only = false) {
    if (dims == nullptr || weights == nullptr || in_emb_dev == nullptr || kv == nullptr ||
        (pos_host == nullptr && pos_dev == nullptr))
        return HRA_ERR_INVALID_ARG;
    if (!dims_ok(dims)) return HRA_ERR_UNSUPPORTED;
    const hra_dims& d = *dims;
    if (batch < 1 || batch > kMaxBatch) return HRA_ERR_INVALID_ARG;
    if (!weights_ok(d, weights) || !kv_ok(kv) || !aligned16(in_emb_dev) || !aligned16(hidden_dev) ||
        !aligned16(workspace) || (pos_dev != nullptr && (reinterpret_cast<uintptr_t>(pos_dev) & 3u) != 0))
        return HRA_ERR_INVALID_ARG;
    if (batch > kv->batch) return HRA_ERR_INVALID_ARG;
    SeqMeta meta{};
    meta.batch = batch;
    int max_pos = 0;
    if (pos_host != nullptr) {
        meta.mode = 1;
        for (int b = 0; b < batch; ++b) {
            if (pos_host[b] < 0 || pos_host[b] >= kv->n_slots) return HRA_ERR_RANGE;
            meta.vals[b] = pos_host[b];
            max_pos = std::max(max_pos, (int)pos_host[b]);
        }
    } else {
        if (pos_bound < 0 || pos_bound >= kv->n_slots) return HRA_ERR_RANGE;
        meta.mode = 2;
        meta.pos_dev = pos_dev;
        meta.n_slots = kv->n_slots;
        meta.advance = advance ? 1 : 0;
        max_pos = pos_bound;
    }
    const Layout L = backbone_layout(d, batch, batch, batch, kv->n_slots - 1);
    if (workspace_bytes < L.total) return HRA_ERR_WORKSPACE;
    if (validate_only) return HRA_OK;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const Ptrs P{reinterpret_cast<uint8_t*>(workspace)};
    HRA_TRY(launch_build_rowmap(meta, batch, P.at<int32_t>(L.row_seq), P.at<int32_t>(L.row_pos),
                                P.at<int32_t>(L.cu), P.at<int32_t>(L.last_row), nullptr, P.at<unsigned int>(L.err),
                                st, P.at<unsigned int>(L.sync), decode_pass_counter_words(std::min(batch, 64), d.n_kv_heads)));
    HRA_TRY(launch_rope_table(batch, P.at<int32_t>(L.row_pos), d.head_dim, (double)d.rope_theta,
                              P.at<float2>(L.rope), st));
    // r = input embedding, y = RMSNorm(r) with layer 0's attention gain
    HRA_TRY(launch_rmsnorm(reinterpret_cast<const bf16*>(in_emb_dev), nullptr,
                           reinterpret_cast<const bf16*>(weights->layers[0].attn_norm), P.at<bf16>(L.y),
                           P.at<bf16>(L.r), batch, d.hidden, d.rms_eps, st));
    return run_layers(d, *weights, *kv, P, L, batch, batch, 0, false, false, reinterpret_cast<bf16*>(hidden_dev),
                      pos_host, max_pos, st);
}

}  // namespace

int hra_decode(const hra_dims* dims, const hra_weights* weights, const void* in_emb_dev, const int32_t* pos,
               int32_t batch, const hra_kv_cache* kv, void* hidden_dev, void* workspace, size_t workspace_bytes,
               void* stream) {
    if (pos == nullptr) return HRA_ERR_INVALID_ARG;
    return decode_impl(dims, weights, in_emb_dev, pos, nullptr, 0, 0, batch, kv, hidden_dev, workspace,
                       workspace_bytes, stream);
}

int hra_decode_dev(const hra_dims* dims, const hra_weights* weights, const void* in_emb_dev, int32_t* pos_dev,
                   int32_t pos_bound, int32_t advance, int32_t batch, const hra_kv_cache* kv, void* hidden_dev,
                   void* workspace, size_t workspace_bytes, void* stream) {
    if (pos_dev == nullptr) return HRA_ERR_INVALID_ARG;
    return decode_impl(dims, weights, in_emb_dev, nullptr, pos_dev, pos_bound, advance, batch, kv, hidden_dev,
                       workspace, workspace_bytes, stream);
}

// Codebook-step workspace: error word and per-row counters (cleared by the head projection), per-row
// argmax candidates, then the fp32 logit partials [splits][batch][K * Vc].
struct CbLayout {
    size_t counters, cand, part;
};
CbLayout codebook_layout(const hra_dims* dims, int32_t batch) {
    Region g;
    CbLayout L;
    g.take(4 + 4 * (size_t)batch);
    L.counters = 4;
    L.cand = g.take(4 * (size_t)batch * dims->n_codebooks);
    L.part = g.off;
    return L;
}

size_t hra_codebook_workspace_size(const hra_dims* dims, int32_t batch) {
    if (!audio_dims_ok(dims) || batch < 1) return 0;
    const int N = dims->n_codebooks * dims->codebook_size;
    Region g;
    g.off = codebook_layout(dims, batch).part;
    const size_t plane = (size_t)batch * N * sizeof(float);
    size_t part = std::max(plane, linear_partial_bound(std::min(batch, 128), N, dims->hidden, EPI_F32));
    if (batch <= kHeadMaxBatch) part = std::max(part, (size_t)kHeadMaxSplits * plane);
    if (batch > 128) part = std::max(part, linear_tail_bound());
    g.take(part);
    return g.off;
}

namespace {

// The codebook step, greedy (sampling == nullptr) or sampled; validate_only checks the arguments
// and returns without enqueueing anything.
int codebook_impl(const hra_dims* dims, const void* hidden_dev, const void* head_w_dev, const void* code_emb_dev,
                  hra_delay_state* state_dev, const float* eoc_bias_dev, const hra_sampling* sampling,
                  const uint64_t* seeds_dev, int32_t batch, int32_t* codes_dev, void* next_emb_dev, int32_t* done_dev,
                  float* logits_dev, void* workspace, size_t workspace_bytes, void* stream, bool validate_only) {
    if (dims == nullptr || !audio_dims_ok(dims)) return dims == nullptr ? HRA_ERR_INVALID_ARG : HRA_ERR_UNSUPPORTED;
    if (batch < 1 || batch > 1024) return HRA_ERR_INVALID_ARG;
    if (sampling != nullptr) {
        if (!(sampling->temperature > 0.f) || !std::isfinite(sampling->temperature) || sampling->top_k < 0 ||
            !(sampling->top_p > 0.f) || !(sampling->top_p <= 1.f) || seeds_dev == nullptr ||
            (reinterpret_cast<uintptr_t>(seeds_dev) & 7u) != 0)
            return HRA_ERR_INVALID_ARG;
        if (dims->codebook_size > 2048) return HRA_ERR_UNSUPPORTED;
    }
    if (!aligned16(hidden_dev) || !aligned16(head_w_dev) || !aligned16(code_emb_dev) || !aligned16(state_dev) ||
        !aligned16(next_emb_dev) || !aligned16(workspace) || codes_dev == nullptr || done_dev == nullptr ||
        (reinterpret_cast<uintptr_t>(codes_dev) & 3u) || (reinterpret_cast<uintptr_t>(done_dev) & 3u) ||
        (eoc_bias_dev && (reinterpret_cast<uintptr_t>(eoc_bias_dev) & 3u)) ||
        (logits_dev && (reinterpret_cast<uintptr_t>(logits_dev) & 3u)))
        return HRA_ERR_INVALID_ARG;
    if (workspace_bytes < hra_codebook_workspace_size(dims, batch)) return HRA_ERR_WORKSPACE;
    if (validate_only) return HRA_OK;
    const int K = dims->n_codebooks, Vc = dims->codebook_size, H = dims->hidden;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = reinterpret_cast<uint8_t*>(workspace);
    const CbLayout CL = codebook_layout(dims, batch);
    unsigned int* err = reinterpret_cast<unsigned int*>(base);
    float* part = reinterpret_cast<float*>(base + CL.part);
    const double head_flops = 2.0 * batch * (double)K * Vc * H;

    int splits = 1;
    if (batch <= kHeadMaxBatch) {
        // the head as 256-row tiles x K splits; the finalize sums the split planes in order
        HeadCall hc{};
        hc.hidden = reinterpret_cast<const bf16*>(hidden_dev);
        hc.head_w = reinterpret_cast<const bf16*>(head_w_dev);
        hc.partial = part;
        hc.err = err;
        hc.zero_ptr = err;   // error word + per-row counters
        hc.zero_words = 1 + batch;
        hc.splits_used = &splits;
        hc.B = batch;
        hc.N = K * Vc;
        hc.H = H;
        HRA_TRY(probed(HRA_PROBE_AUDIO_HEAD, head_flops, st, [&] { return launch_audio_head(hc, st); }));
    } else {
        LinearCall c{};
        c.a = reinterpret_cast<const bf16*>(hidden_dev);
        c.w = reinterpret_cast<const bf16*>(head_w_dev);
        c.out = part;
        c.M = batch;
        c.N = K * Vc;
        c.K = H;
        c.epi = EPI_F32;
        c.split_req = 0;
        c.partial = part;
        c.err = err;
        c.partial_only = true;
        c.splits_used = &splits;
        c.zero_ptr = err;                 // error word + per-row counters
        c.zero_words = 1 + batch;
        HRA_TRY(probed(HRA_PROBE_AUDIO_HEAD, head_flops, st, [&] { return launch_linear(c, st); }));
    }

    CodebookArgs a{};
    a.partial = part;
    a.counters = reinterpret_cast<int*>(base + CL.counters);
    a.cand = reinterpret_cast<int*>(base + CL.cand);
    a.splits = splits;
    a.eoc_bias = eoc_bias_dev;
    a.code_emb = reinterpret_cast<const bf16*>(code_emb_dev);
    a.state = reinterpret_cast<int4*>(state_dev);
    a.codes = codes_dev;
    a.next_emb = reinterpret_cast<bf16*>(next_emb_dev);
    a.done = done_dev;
    a.logits_out = logits_dev;
    a.err = err;
    a.batch = batch;
    a.K = K;
    a.Vc = Vc;
    a.H = H;
    a.bos = dims->bos_id;
    a.eoc = dims->eoc_id;
    if (sampling != nullptr) {
        a.seeds = seeds_dev;
        a.temperature = sampling->temperature;
        a.top_k = sampling->top_k;
        a.top_p = sampling->top_p;
    }
    HRA_TRY(launch_codebook_finalize(a, st));
    return HRA_OK;
}

}  // namespace

int hra_codebook_step(const hra_dims* dims, const void* hidden_dev, const void* head_w_dev, const void* code_emb_dev,
                      hra_delay_state* state_dev, const float* eoc_bias_dev, int32_t batch, int32_t* codes_dev,
                      void* next_emb_dev, int32_t* done_dev, float* logits_dev, void* workspace,
                      size_t workspace_bytes, void* stream) {
    return codebook_impl(dims, hidden_dev, head_w_dev, code_emb_dev, state_dev, eoc_bias_dev, nullptr, nullptr, batch,
                         codes_dev, next_emb_dev, done_dev, logits_dev, workspace, workspace_bytes, stream, false);
}

int hra_codebook_step_sampled(const hra_dims* dims, const void* hidden_dev, const void* head_w_dev,
                              const void* code_emb_dev, hra_delay_state* state_dev, const float* eoc_bias_dev,
                              const hra_sampling* sampling, const uint64_t* seeds_dev, int32_t batch,
                              int32_t* codes_dev, void* next_emb_dev, int32_t* done_dev, float* logits_dev,
                              void* workspace, size_t workspace_bytes, void* stream) {
    if (sampling == nullptr) return HRA_ERR_INVALID_ARG;
    return codebook_impl(dims, hidden_dev, head_w_dev, code_emb_dev, state_dev, eoc_bias_dev, sampling, seeds_dev,
                         batch, codes_dev, next_emb_dev, done_dev, logits_dev, workspace, workspace_bytes, stream,
                         false);
}

int hra_ar_frame(const hra_dims* dims, const hra_weights* weights, const void* head_w_dev, const void* code_emb_dev,
                 hra_delay_state* state_dev, const float* eoc_bias_dev, const hra_sampling* sampling,
                 const uint64_t* seeds_dev, void* hidden_dev, int32_t* pos_dev, int32_t pos_bound, int32_t batch,
                 const hra_kv_cache* kv, int32_t* codes_dev, void* next_emb_dev, int32_t* done_dev, void* backbone_ws,
                 size_t backbone_ws_bytes, void* codebook_ws, size_t codebook_ws_bytes, void* stream) {
    if (pos_dev == nullptr) return HRA_ERR_INVALID_ARG;
    // both steps' arguments are checked before anything is enqueued
    int rc = decode_impl(dims, weights, next_emb_dev, nullptr, pos_dev, pos_bound, 1, batch, kv, hidden_dev,
                         backbone_ws, backbone_ws_bytes, stream, /*validate_only=*/true);
    if (rc != HRA_OK) return rc;
    rc = codebook_impl(dims, hidden_dev, head_w_dev, code_emb_dev, state_dev, eoc_bias_dev, sampling, seeds_dev, batch,
                       codes_dev, next_emb_dev, done_dev, nullptr, codebook_ws, codebook_ws_bytes, stream, true);
    if (rc != HRA_OK) return rc;
    rc = codebook_impl(dims, hidden_dev, head_w_dev, code_emb_dev, state_dev, eoc_bias_dev, sampling, seeds_dev, batch,
                       codes_dev, next_emb_dev, done_dev, nullptr, codebook_ws, codebook_ws_bytes, stream, false);
    if (rc != HRA_OK) return rc;
    return decode_impl(dims, weights, next_emb_dev, nullptr, pos_dev, pos_bound, 1, batch, kv, hidden_dev,
                       backbone_ws, backbone_ws_bytes, stream);
}

size_t hra_linear_workspace_size(int32_t M, int32_t N, int32_t K, int32_t epilogue, int32_t split_k) {
    if (M < 1 || N < 8 || K < 64) return 0;
    return 256 + align_up(linear_partial_bytes(M, N, K, epilogue, split_k, false));
}

int hra_linear(const void* a_dev, const void* w_dev, void* out_dev, int32_t M, int32_t N, int32_t K,
               int32_t epilogue, int32_t split_k, void* workspace, size_t workspace_bytes, void* stream) {
    if (!aligned16(a_dev) || !aligned16(w_dev) || !aligned16(out_dev) || !aligned16(workspace))
        return HRA_ERR_INVALID_ARG;
    if (M < 1 || N < 8 || N % 8 != 0 || K < 64 || K % 64 != 0 || split_k < 0) return HRA_ERR_INVALID_ARG;
    if (epilogue < EPI_STORE || epilogue > EPI_F32) return HRA_ERR_INVALID_ARG;
    if (workspace_bytes < hra_linear_workspace_size(M, N, K, epilogue, split_k)) return HRA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = reinterpret_cast<uint8_t*>(workspace);
    HRA_TRY(cudaMemsetAsync(base, 0, 4, st));
    LinearCall c{};
    c.a = reinterpret_cast<const bf16*>(a_dev);
    c.w = reinterpret_cast<const bf16*>(w_dev);
    c.out = out_dev;
    c.M = M;
    c.N = N;
    c.K = K;
    c.epi = epilogue;
    c.split_req = split_k;
    c.partial = reinterpret_cast<float*>(base + 256);
    c.err = reinterpret_cast<unsigned int*>(base);
    HRA_TRY(launch_linear(c, st));
    return HRA_OK;
}

size_t hra_linear_fp8_workspace_size(int32_t M, int32_t N, int32_t K, int32_t epilogue) {
    if (M < 1 || N < 8 || K < 128) return 0;
    size_t part = linear_partial_bound(M, N, K, epilogue);
    if (M > 128) part = std::max(part, linear_tail_bound());
    return 256 + align_up(part);
}

int hra_linear_fp8(const void* a8_dev, const void* w8_dev, void* out_dev, int32_t M, int32_t N, int32_t K,
                   const float* a_scale_dev, const float* w_scale_dev, int32_t epilogue, void* workspace,
                   size_t workspace_bytes, void* stream) {
    if (!aligned16(a8_dev) || !aligned16(w8_dev) || !aligned16(out_dev) || !aligned16(workspace) ||
        a_scale_dev == nullptr || w_scale_dev == nullptr || (reinterpret_cast<uintptr_t>(a_scale_dev) & 3u) ||
        (reinterpret_cast<uintptr_t>(w_scale_dev) & 3u))
        return HRA_ERR_INVALID_ARG;
    if (M < 1 || N < 8 || N % 8 != 0 || K < 128 || K % 128 != 0) return HRA_ERR_INVALID_ARG;
    if (epilogue < EPI_STORE || epilogue > EPI_F32) return HRA_ERR_INVALID_ARG;
    if (workspace_bytes < hra_linear_fp8_workspace_size(M, N, K, epilogue)) return HRA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* base = reinterpret_cast<uint8_t*>(workspace);
    HRA_TRY(cudaMemsetAsync(base, 0, 4, st));
    LinearCall c{};
    c.a = reinterpret_cast<const bf16*>(a8_dev);
    c.w = reinterpret_cast<const bf16*>(w8_dev);
    c.out = out_dev;
    c.M = M;
    c.N = N;
    c.K = K;
    c.epi = epilogue;
    c.partial = reinterpret_cast<float*>(base + 256);
    c.err = reinterpret_cast<unsigned int*>(base);
    c.fp8 = true;
    c.a_scale = a_scale_dev;
    c.w_scale = w_scale_dev;
    HRA_TRY(launch_linear(c, st));
    return HRA_OK;
}

int32_t hra_device_error(const void* workspace, void* stream) {
    if (workspace == nullptr) return HRA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return HRA_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, workspace, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return HRA_ERR_CUDA;
    return (int32_t)v;
}

const char* hra_status_string(int status) {
    switch (status) {
        case HRA_OK: return "ok";
        case HRA_ERR_INVALID_ARG: return "invalid argument (null, misaligned or non-positive size)";
        case HRA_ERR_UNSUPPORTED: return "unsupported dims";
        case HRA_ERR_WORKSPACE: return "workspace too small";
        case HRA_ERR_RANGE: return "sequence length or position outside the cache";
        case HRA_ERR_CUDA: return "CUDA launch or driver error";
        default: return "unknown status";
    }
}

}  // extern "C"
