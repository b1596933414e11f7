// internal.h -- host-side declarations shared by the translation units of the hra library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace hra {

// Streaming-multiprocessor count of the current device (cached per device).
int device_sm_count();

// Host-side count of kernel launches issued by the library.
void count_launches(int n);

// Launch with programmatic stream serialization (see pdl_wait / pdl_launch in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launches(1);
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch through launch_pdl and return the error from the enclosing function if it fails.
#define HRA_LAUNCH(...)                                  \
    do {                                                 \
        cudaError_t hra_e_ = ::hra::launch_pdl(__VA_ARGS__); \
        if (hra_e_ != cudaSuccess) return hra_e_;        \
    } while (0)

// Per packed row: q heads and k heads get RMSNorm over head_dim (shared gains) + rotate-half RoPE
// (table row = rope_row_is_pos ? row_pos[row] : row); q goes to q_out [rows, nq, hd]; k and v go to
// cache slot row_pos[row] of cache sequence row_seq[row] of this layer.
struct QkRopeArgs {
    const bf16* qkv;
    const bf16* q_norm;
    const bf16* k_norm;
    const float2* rope;     // transposed table: (row r, pair i) at i * rope_rows + r
    int rope_rows;
    const int32_t* row_seq;
    const int32_t* row_pos;
    int rope_row_is_pos;
    bf16* q_out;
    bf16* kv_layer;     // this layer's cache block: [cache_batch][2][nkv][n_slots][hd]
    int n_slots;
    int rows, nq, nkv, hd;
    float eps;
    // optional: take the merged row as the sum of fp32 split partials (part[s * split_stride +
    // row * ldp + col], s in split order) rounded to bf16, instead of reading qkv
    const float* part;
    int splits;
    long long split_stride;
    int ldp;
};
// ------------------------------------------------------------------ projection GEMM
enum EpiMode : int { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SWIGLU = 2, EPI_F32 = 3 };

// out = epilogue(a [M, K] . w^T); w has N rows (2N for EPI_SWIGLU, gate rows then up rows).
// split_req: 0 = automatic, >= 1 forces that many K splits (only when M <= 128).
struct LinearCall {
    const bf16* a;
    const bf16* w;
    void* out;
    int M, N, K;
    int epi;
    int split_req;
    float* partial;        // fp32 scratch for split partials (>= linear_partial_bytes())
    unsigned int* err;     // sticky device error word
    bool partial_only;     // leave the split partials unreduced (EPI_F32 only; out == partial)
    int* splits_used;      // optional: receives the number of K splits launched
    // EPI_RESIDUAL only: when the plan splits K, the reduction also writes
    // norm_out = RMSNorm(out) * norm_gain (one CTA per row) and sets *norm_done.
    const bf16* norm_gain;
    bf16* norm_out;
    float norm_eps;
    bool* norm_done;
    // CTA 0 clears zero_words words at zero_ptr after earlier kernels finished (0 = none)
    unsigned int* zero_ptr;
    int zero_words;
    // EPI_STORE of the merged QKV projection: when set and the large-M path runs, the epilogue does the
    // per-head q/k norm + RoPE + K/V cache write itself (out is not written) and sets *qk_done.
    const QkRopeArgs* qk;
    bool* qk_done;
    // FP8: a and w hold E4M3 codes (K a multiple of 128); the accumulators are scaled by
    // (*a_scale) * (*w_scale), device scalars.  Always runs the tile kernel (any M).
    bool fp8;
    const float* a_scale;
    const float* w_scale;
};
size_t linear_partial_bytes(int M, int N, int K, int epi, int split_req, bool partial_only);
cudaError_t launch_linear(const LinearCall& c, cudaStream_t st);
// Largest partial buffer any automatic plan with M <= m_max rows and these N, K can ask for.
size_t linear_partial_bound(int m_max, int N, int K, int epi);
// Largest last-round piece buffer any plan with more than one M tile can ask for.
size_t linear_tail_bound();

// ------------------------------------------------------------------ row bookkeeping + norms + RoPE
constexpr int kMaxBatch = 512;

// Host-built batch description passed by value to the row-map kernel.
struct SeqMeta {
    int32_t batch;
    int32_t mode;           // 0: prefill (vals = cu_seqlens[0..batch]); 1: decode (vals = pos[0..batch));
                            // 2: decode with positions read from pos_dev (device)
    int32_t vals[kMaxBatch + 1];
    int32_t start[kMaxBatch];   // prefill: position of each sequence's first new row (0 from scratch)
    int32_t* pos_dev;           // mode 2: [batch] positions; a position outside [0, n_slots) raises
                                // HRA_DEVERR_POS_RANGE and is clamped; when advance != 0 each is
                                // incremented after it is read
    int32_t n_slots;
    int32_t advance;
};

// Writes row_seq[T], row_pos[T] (sequence index and position of each packed row), and for prefill
// cu[batch+1], last_row[batch]; for decode last_row[b] = b.  Also clears the call's error word.
// Prefill also writes seq_start[batch] = meta.start (may be null for decode).  zero_words words at
// zero_ptr are cleared as well (the counters of the persistent decoder pass).
cudaError_t launch_build_rowmap(const SeqMeta& meta, int total_rows, int32_t* row_seq, int32_t* row_pos,
                                int32_t* cu, int32_t* last_row, int32_t* seq_start, unsigned int* err,
                                cudaStream_t st, unsigned int* zero_ptr = nullptr, int zero_words = 0);

// cos/sin table, transposed: entry (row r, pair i) at i * n_rows + r (float2), for position
// pos_of_row[r] (or r when null).
cudaError_t launch_rope_table(int n_rows, const int32_t* pos_of_row, int head_dim, double theta,
                              float2* table, cudaStream_t st);

// r[row] = embed[tokens[row_seq * ld + (row - cu[row_seq])]]; y = RMSNorm(r) * g.
cudaError_t launch_embed_rmsnorm(const int32_t* tokens, int tok_ld, const int32_t* row_seq,
                                 const int32_t* cu, const bf16* embed, int vocab, const bf16* g,
                                 bf16* r, bf16* y, int rows, int H, float eps, unsigned int* err,
                                 cudaStream_t st);

// y[i] = RMSNorm(x[idx ? idx[i] : i]) * g; when copy_out != null also copy_out[i] = x[idx[i]].
cudaError_t launch_rmsnorm(const bf16* x, const int32_t* idx, const bf16* g, bf16* y, bf16* copy_out,
                           int rows, int H, float eps, cudaStream_t st);

cudaError_t launch_qk_rope_kv(const QkRopeArgs& a, cudaStream_t st);

// ------------------------------------------------------------------ attention
// Causal prefill attention over the cache for every packed row.
struct PrefillAttnArgs {
    const bf16* q;          // [T, nq, hd]
    const bf16* kv_layer;   // [cache_batch][2][nkv][n_slots][hd]
    const int32_t* cu;      // [batch + 1] device
    const int32_t* start;   // [batch] device: position of each sequence's first row (cached keys below)
    bf16* out;              // [T, nq * hd]
    int batch, max_len, n_slots, nq, nkv, hd;
    int total_rows;         // T (rows of q)
    int cache_batch;        // sequences the cache holds (kv_layer spans cache_batch * 2 * nkv * n_slots rows)
    unsigned int* err;      // sticky device error word
    const int32_t* sched;   // work list from launch_attention_schedule (same batch, lengths and starts);
                            // may be null for a single sequence
};
// the tcgen05 kernel (attention_tc.cu): head_dim 64 or 128, n_q / n_kv in {1, 2, 4, 8}
cudaError_t launch_prefill_attention_tc(const PrefillAttnArgs& a, cudaStream_t st);
// The prefill attention's work list for one call's sequences (the same for every layer): the
// non-empty (query tile, sequence) pairs sorted by key tiles, heaviest first; sched[0] = count.
size_t attention_schedule_bytes(int rows, int batch);
cudaError_t launch_attention_schedule(const int32_t* cu, const int32_t* start, int batch, int max_len, int nq,
                                      int nkv, int32_t* sched, cudaStream_t st);

// cuTensorMapEncodeTiled (bf16 elements, 128-byte swizzle, zero fill out of bounds) for a tensor of
// `rank` dims (innermost first), strides in bytes of dims 1.. and the box; `map` is a CUtensorMap.
bool encode_tensor_map(void* map, int rank, const void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                       const uint32_t* box);

// Single-query attention: row i (sequence seq[i], query position pos[i]) attends slots 0..pos[i].
struct DecodeAttnArgs {
    const bf16* q;          // q rows [*, nq, hd]
    const bf16* kv_layer;
    const int32_t* q_row;   // [rows] q row of attention row i (null: i)
    const int32_t* seq;     // cache sequence, indexed by q row
    const int32_t* pos;     // query position, indexed by q row
    bf16* out;              // [rows, nq * hd]
    float* part;            // scratch: splits * rows * nq * (hd + 2) floats
    int rows, max_pos, n_slots, nq, nkv, hd;
    int splits;
};
int decode_attention_splits(int rows, int nkv, int max_pos);
size_t decode_attention_scratch_bytes(int rows, int nq, int hd, int splits);
cudaError_t launch_decode_attention(const DecodeAttnArgs& a, cudaStream_t st);

// ------------------------------------------------------------------ persistent decoder pass
// Every layer over M <= 64 token rows in one cooperative launch (decode_pass.cu): the arithmetic of
// the layer-by-layer path, with grid-wide barriers between the phases of a layer.
constexpr int kDecodePassMaxLayers = 40;
struct DecodePassLayer {
    const bf16* w_qkv;
    const bf16* w_o;
    const bf16* w_gate_up;
    const bf16* w_down;
    const bf16* attn_norm;
    const bf16* q_norm;
    const bf16* k_norm;
    const bf16* mlp_norm;
    bf16* kv;                 // this layer's cache block [cache_batch][2][nkv][n_slots][hd]
};
struct DecodePassCall {
    DecodePassLayer layers[kDecodePassMaxLayers];
    const bf16* final_norm;
    int L, M, H, nq, nkv, hd, F, n_slots;
    float eps;
    const float2* rope;       // transposed table (see QkRopeArgs)
    int rope_rows, rope_row_is_pos;
    const int32_t* row_seq;
    const int32_t* row_pos;
    const int32_t* last_row;  // output row b = row last_row[b], b < n_out; null: output row b = row b
    int n_out;
    int max_pos;              // upper bound of every row's position (sizes the attention's key splits)
    bf16* r;                  // residual [M, H] (in: the layer-0 input), y [M, H] (in: its RMSNorm)
    bf16* y;
    bf16* q;                  // [M, nq * hd]
    bf16* att;                // [M, nq * hd]
    bf16* h;                  // [M, F]
    bf16* out;                // [n_out, H] final-norm output
    float* part;              // projection split partials
    size_t part_bytes;
    float* apart;             // attention split partials
    int attn_splits_max;      // splits the attention scratch holds
    unsigned int* sync;       // decode_pass_sync_bytes(M, nkv, F, H) bytes
    bool sync_zeroed;         // the first decode_pass_counter_words(M, nkv) words of sync are zero
    unsigned int* err;
};
int decode_pass_counter_words(int M, int nkv);
bool decode_pass_supported(const DecodePassCall& c);
size_t decode_pass_scratch_bytes(int M, int H, int nq, int nkv, int hd, int F, int nsm);
size_t decode_pass_sync_bytes(int M, int nkv, int F, int H);
cudaError_t launch_decode_pass(const DecodePassCall& c, cudaStream_t st);
// process-wide switch between the persistent pass (opt-in) and the layer-by-layer kernels (default)
extern bool g_decode_pass_enabled;
// process-wide switch: projection GEMMs of at least 512 BF16 rows on 2-CTA clusters (default) or
// on single CTAs
extern bool g_gemm_pairs;

// ------------------------------------------------------------------ codebook step finalize
struct CodebookArgs {
    const float* partial;   // [splits][batch][K * Vc] fp32 logits partials
    int* counters;          // [batch], zero on entry: CTAs of a row that have finished their argmax
    int* cand;              // [batch][K] argmax of each codebook
    int splits;
    const float* eoc_bias;  // [batch, K] or null
    const bf16* code_emb;   // [K][Vc][H]
    int4* state;            // hra_delay_state [batch]
    int32_t* codes;         // [batch, K]
    bf16* next_emb;         // [batch, H]
    int32_t* done;          // [batch]
    float* logits_out;      // [batch, K, Vc] or null
    unsigned int* err;
    int batch, K, Vc, H, bos, eoc;
    // sampled step (seeds != null): temperature, top-k (0 = off), top-p (1 = off), per-row seeds
    const uint64_t* seeds;  // [batch]
    float temperature, top_p;
    int top_k;
};
cudaError_t launch_codebook_finalize(const CodebookArgs& a, cudaStream_t st);

// ------------------------------------------------------------------ audio-head projection, batch <= 128 (head.cu)
constexpr int kHeadMaxBatch = 128;
constexpr int kHeadMaxSplits = 8;

// Work split of the head: nt tiles of 256 weight rows x `splits` K ranges of kbps 64-wide blocks.
struct HeadPlan {
    int nt, splits, kbps;
};
// Tiles of 256 head rows times K splits, at most max_splits (split_req > 0 forces that many), over
// the SMs about once.
HeadPlan head_plan(int N, int H, int max_splits = kHeadMaxSplits, int split_req = 0);

// partial[split][b][n] = sum over the split's K range of hidden[b][k] * head_w[n][k] (fp32).
struct HeadCall {
    const bf16* hidden;         // [B, H]
    const bf16* head_w;         // [N, H]
    float* partial;             // [splits][B][N]
    unsigned int* err;
    unsigned int* zero_ptr;     // cleared by the first CTA once the kernels ahead have finished
    int zero_words;
    int* splits_used;           // optional: receives the number of K splits
    int B, N, H;
    int max_splits;             // 0: kHeadMaxSplits
    int split_req;              // > 0: exactly this many K splits
    bool no_l2_prefetch;        // do not send the CTA's later weight tiles towards L2 ahead of use
};
cudaError_t launch_audio_head(const HeadCall& c, cudaStream_t st);

// ------------------------------------------------------------------ NVFP4 projection (nvfp4.cu)
// out = epilogue((g_a g_w) sum_k e2m1(a) dec(sa) e2m1(w) dec(sw)); codes one per byte [rows][K],
// block scales [rows][K/16] E4M3; w has N rows (2N for EPI_SWIGLU: gate rows, then up rows).
struct Nvfp4Call {
    const uint8_t* a_codes;
    const uint8_t* a_scales;
    const uint8_t* w_codes;
    const uint8_t* w_scales;
    const float* g_a;       // device scalars
    const float* g_w;
    void* out;
    unsigned int* err;
    int M, N, K;            // K a multiple of 64
    int epi;                // EPI_STORE / EPI_RESIDUAL / EPI_SWIGLU / EPI_F32
};
cudaError_t launch_linear_nvfp4(const Nvfp4Call& c, cudaStream_t st);
// NVFP4 band input scales from the calibration amax [n_layers][4] (see hra_nvfp4_band_scales)
cudaError_t launch_nvfp4_band_scales(const float* amax, float* scale, int n_layers, cudaStream_t st);
// out[i] = amax[i] > 0 ? amax[i] / div : 1
cudaError_t launch_amax_div(const float* amax, float* out, int n, float div, cudaStream_t st);

// 2-D uint8 tensor map [rows, cols] (cols innermost), boxes of 64 bytes x box_rows, no swizzle.
bool make_map_u8(CUtensorMap* m, const void* base, int rows, int cols, int box_rows);

// 2-D bf16 tensor map [rows, cols] (cols innermost), 64-element x box_rows boxes, 128-byte
// swizzle; encodings are cached by (base, shape, box).
bool make_map_2d(CUtensorMap* m, const void* base, int rows, int cols, int box_rows);

// ------------------------------------------------------------------ E4M3 quantization (fp8.cu)
// out = e4m3(x / *scale), n a multiple of 8 (x 16-byte, out 8-byte aligned)
cudaError_t launch_fp8_quantize(const bf16* x, long long n, const float* scale, uint8_t* out, cudaStream_t st);
// NVFP4: codes [rows][K] (one E2M1 code per byte), scales [rows][K/16] E4M3; K a multiple of 16
cudaError_t launch_nvfp4_quantize(const bf16* x, int rows, int K, const float* g, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t st);
// *amax = max(*amax, max |x|), n a multiple of 8
cudaError_t launch_absmax(const bf16* x, long long n, float* amax, cudaStream_t st);
cudaError_t launch_zero_floats(float* v, int n, cudaStream_t st);
// scale[i] = amax[i] > 0 ? amax[i] / 448 : 1
cudaError_t launch_amax_to_scale(const float* amax, float* scale, int n, cudaStream_t st);

}  // namespace hra
