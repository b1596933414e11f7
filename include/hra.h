/*
 * hra.h -- C ABI of the GB300 (sm_103a) Higgs-Audio-style hot path.
 *
 * Two operations make up the path:
 *   1. hra_prefill: batched BF16 prefill of a Qwen3-style decoder backbone -- embedding lookup,
 *      RMSNorm, merged QKV projection, per-head q/k RMSNorm + RoPE with the KV-cache write, causal
 *      attention over the used keys of ragged prompts, o-projection, residual + RMSNorm, SwiGLU
 *      gate/up/down MLP -- returning the last position's final hidden and the filled cache.
 *      Source: "Stabilize Higgs Audio termination and prefill" (FlashRT PR #141), Summary (the
 *      BF16 batched prefill is kernelized: embedding lookup, projection GEMMs, q/k norm + RoPE
 *      and the KV writes); the per-layer chain and the used-key rule follow the
 *      "flashrt-structures 0.2.0, prefill_tower/fp8_chain.py" page, its description and its
 *      per-layer chain.
 *   2. hra_codebook_step: per-frame delayed-codebook step -- audio-head projection to K codebook
 *      logit rows, per-codebook argmax under the delay pattern, BOS/EOC handling with stop flags,
 *      and the sum of the K codebook embeddings into the next input.
 *      Source: FlashRT PR #141, Summary (one shared delayed-codebook helper takes the per-frame
 *      argmax, applies the delays and sums the codebook embeddings) and Root cause (delayed EOC).
 * hra_decode is the single-token backbone pass of the autoregressive audio loop (FlashRT PR #141,
 * Performance: the AR decode time per frame); its input is the summed codebook embedding.
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev / device buffers are CUDA device pointers owned by the caller; the
 *     library never allocates, frees or synchronises inside hra_prefill / hra_decode /
 *     hra_codebook_step / hra_linear.  All work is enqueued on `stream` (a cudaStream_t passed as
 *     void*, NULL = legacy default stream) in stream order.
 *   - Device pointers must be 16-byte aligned; bf16 tensors are row-major and contiguous; weight
 *     matrices are [out_features, in_features] (each output row is one weight row).
 *   - Host arrays (seq_lens, pos) are read before the call returns and may be reused afterwards.
 *   - Every argument is validated before the first launch; on a non-zero return nothing was
 *     enqueued.  Device-side faults of the input data (a token id outside [0, vocab)) never trap:
 *     the id is clamped and a sticky bit is set in the workspace's error word, read with
 *     hra_device_error().
 *   - Numerics: bf16 storage, fp32 accumulation, bf16 rounding at each norm output, projection
 *     output, q/k after norm + RoPE, attention output, gate/up/SwiGLU outputs, and the residual
 *     after each add.  Logits are fp32.
 */
#ifndef HRA_H
#define HRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------------------------- */
#define HRA_OK 0
#define HRA_ERR_INVALID_ARG (-1)   /* null or misaligned pointer, non-positive size              */
#define HRA_ERR_UNSUPPORTED (-2)   /* dims outside what the kernels implement                     */
#define HRA_ERR_WORKSPACE (-3)     /* workspace smaller than the matching *_workspace_size()      */
#define HRA_ERR_RANGE (-4)         /* a sequence length or position outside the cache            */
#define HRA_ERR_CUDA (-5)          /* a CUDA launch or driver call failed                        */

/* Sticky device error bits (hra_device_error). */
#define HRA_DEVERR_TOKEN_RANGE 1u  /* a token id was outside [0, vocab); it was clamped          */
#define HRA_DEVERR_WAIT_TIMEOUT 2u /* a pipeline wait inside a kernel gave up (kernel bug guard) */
#define HRA_DEVERR_CODE_RANGE 4u   /* a code index outside [0, codebook_size) was clamped        */
#define HRA_DEVERR_POS_RANGE 8u    /* a device-resident position was outside [0, n_slots); the row
                                       ran at the nearest slot inside the cache                   */

/* ---- model description ---------------------------------------------------------------------- */
/* Backbone and audio-head shape.  Supported: head_dim in {64, 128}; n_q_heads % n_kv_heads == 0;
 * hidden, n_q_heads * head_dim and ffn multiples of 64; 1 <= n_codebooks <= 16;
 * codebook_size >= 2 with bos_id, eoc_id < codebook_size. */
typedef struct hra_dims {
    int32_t n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
    float rope_theta, rms_eps;
    int32_t n_codebooks, codebook_size, bos_id, eoc_id;
} hra_dims;

/* One decoder layer, all bf16 device pointers, [out, in] row-major:
 *   attn_norm [hidden]; w_qkv [(n_q + 2 n_kv) * head_dim, hidden] (q rows, then k rows, then v rows);
 *   q_norm, k_norm [head_dim] (shared by all heads); w_o [hidden, n_q * head_dim]; mlp_norm [hidden];
 *   w_gate_up [2 * ffn, hidden] (gate rows, then up rows); w_down [hidden, ffn]. */
typedef struct hra_layer_weights {
    const void *attn_norm, *w_qkv, *q_norm, *k_norm, *w_o, *mlp_norm, *w_gate_up, *w_down;
} hra_layer_weights;

/* embed [vocab, hidden] bf16 (device); layers: HOST array of n_layers entries; final_norm [hidden]. */
typedef struct hra_weights {
    const void* embed;
    const hra_layer_weights* layers;
    const void* final_norm;
} hra_weights;

/* KV cache, bf16 device memory laid out [n_layers][batch][2][n_kv_heads][n_slots][head_dim]
 * (index 0 = K after norm + RoPE, in rotate-half order; 1 = V).  Slot p of sequence b holds
 * position p of that sequence.  Only slots that a call writes are touched. */
typedef struct hra_kv_cache {
    void* base;
    int32_t batch;
    int32_t n_slots;
} hra_kv_cache;

/* Per-row delay state (device, 16 bytes per row): frame = frames emitted so far; eoc_frame = the
 * stream's end frame in codebook-0 time, -1 while no EOC has been seen; done = 1 once the last
 * codebook has emitted EOC (sticky). */
typedef struct hra_delay_state {
    int32_t frame, eoc_frame, done, reserved;
} hra_delay_state;

/* ---- prefill -------------------------------------------------------------------------------- */
/* Compute the last layer for every row (default: only the rows needed for the last hidden). */
#define HRA_PREFILL_FULL_LAST_LAYER 1u

/* Bytes of workspace hra_prefill needs for this batch shape (total_tokens = sum of seq_lens). */
size_t hra_prefill_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens,
                                  int32_t max_len);

/* Batched prefill of `batch` ragged prompts.
 *   tokens_dev   int32 [batch, max_len] device; prompt b is tokens[b, 0 : seq_lens[b]]; the rest
 *                are pads and are never read.
 *   seq_lens     int32 [batch] HOST; each in [1, min(max_len, kv->n_slots)].  batch <= 512 and
 *                batch <= kv->batch.
 *   kv           cache; slots [0, seq_lens[b]) of sequence b are written in every layer.
 *   last_hidden_dev bf16 [batch, hidden]: final RMSNorm output at position seq_lens[b] - 1.
 *   workspace    device scratch of at least hra_prefill_workspace_size() bytes (16-byte aligned).
 * Returns HRA_OK or a negative status (nothing enqueued). */
int hra_prefill(const hra_dims* dims, const hra_weights* weights, const int32_t* tokens_dev,
                const int32_t* seq_lens, int32_t batch, int32_t max_len, const hra_kv_cache* kv,
                void* last_hidden_dev, void* workspace, size_t workspace_bytes, uint32_t flags,
                void* stream);

/* Prefill of one chunk per sequence after the positions already in its cache: a later piece of a
 * long prompt (chunked prefill), a single token of a running sequence, or a mix of both in one
 * launch -- the mixed prefill batches whose launch bound must come from the real batch
 * (vLLM-Omni PR #8226, Purpose).  Same arguments as hra_prefill, plus:
 *   start_pos    host int32 [batch]: sequence b's seq_lens[b] tokens sit at positions
 *                start_pos[b] .. start_pos[b] + seq_lens[b] - 1; 0 <= start_pos[b] and
 *                start_pos[b] + seq_lens[b] <= kv->n_slots (else HRA_ERR_RANGE).
 *   tokens_dev   int32 [batch, max_len]: row b holds the chunk's tokens (not the whole prompt).
 *   kv           slots [0, start_pos[b]) of sequence b must hold that sequence's earlier keys and
 *                values (from earlier calls); they are read, never written.  Slots
 *                [start_pos[b], start_pos[b] + seq_lens[b]) are written; the rest stay untouched.
 *   last_hidden_dev bf16 [batch, hidden]: final RMSNorm output at position
 *                start_pos[b] + seq_lens[b] - 1.
 *   workspace    at least hra_prefill_chunk_workspace_size() bytes, with max_end the largest
 *                start_pos[b] + seq_lens[b].
 * With every start_pos[b] = 0 this is hra_prefill.  Returns HRA_OK or a negative status (nothing
 * enqueued); start_pos == NULL is HRA_ERR_INVALID_ARG. */
size_t hra_prefill_chunk_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens,
                                        int32_t max_len, int32_t max_end);
int hra_prefill_chunk(const hra_dims* dims, const hra_weights* weights, const int32_t* tokens_dev,
                      const int32_t* seq_lens, const int32_t* start_pos, int32_t batch, int32_t max_len,
                      const hra_kv_cache* kv, void* last_hidden_dev, void* workspace,
                      size_t workspace_bytes, uint32_t flags, void* stream);

/* ---- decode pass ---------------------------------------------------------------------------- */
size_t hra_decode_workspace_size(const hra_dims* dims, int32_t batch, int32_t n_slots);

/* One single-token pass through every layer for `batch` rows (batch <= 512).
 *   in_emb_dev  bf16 [batch, hidden]: the input embedding of each row (e.g. the summed codebook
 *               embedding from hra_codebook_step).
 *   pos         int32 [batch] HOST: the position of each row's token, in [0, kv->n_slots); the pass
 *               writes cache slot pos[b] of row b in every layer and attends slots [0, pos[b]].
 *   hidden_dev  bf16 [batch, hidden]: final RMSNorm output of each row. */
int hra_decode(const hra_dims* dims, const hra_weights* weights, const void* in_emb_dev,
               const int32_t* pos, int32_t batch, const hra_kv_cache* kv, void* hidden_dev,
               void* workspace, size_t workspace_bytes, void* stream);

/* hra_decode with the positions in device memory, for loops captured once and replayed (a CUDA
 * graph of the AR audio loop: host launch overhead was the per-frame limit, "Stabilize Higgs Audio
 * termination and prefill", Performance; vLLM-Omni PR #8226, Step-overhead reductions).
 *   pos_dev      device int32 [batch]: row b runs at position pos_dev[b] (read when the pass
 *                starts).  A position outside [0, kv->n_slots) sets HRA_DEVERR_POS_RANGE and the
 *                row runs at the nearest slot inside the cache (0 or n_slots - 1), overwriting it.
 *   pos_bound    host upper bound of every position of this call, 0 <= pos_bound < kv->n_slots
 *                (else HRA_ERR_RANGE); sizes the attention's key splits.  A captured graph passes
 *                the largest position it will ever see.
 *   advance      non-zero: every pos_dev[b] is incremented once it has been read, so replaying the
 *                pass walks the positions forward with no host work.
 * Other arguments as hra_decode. */
int hra_decode_dev(const hra_dims* dims, const hra_weights* weights, const void* in_emb_dev,
                   int32_t* pos_dev, int32_t pos_bound, int32_t advance, int32_t batch,
                   const hra_kv_cache* kv, void* hidden_dev, void* workspace, size_t workspace_bytes,
                   void* stream);

/* ---- delayed-codebook step ------------------------------------------------------------------ */
size_t hra_codebook_workspace_size(const hra_dims* dims, int32_t batch);

/* One frame for `batch` rows (batch <= 1024).
 *   hidden_dev   bf16 [batch, hidden]
 *   head_w_dev   bf16 [n_codebooks * codebook_size, hidden]: row k*codebook_size + v gives the logit
 *                of code v in codebook k.
 *   code_emb_dev bf16 [n_codebooks, codebook_size, hidden]: codebook embedding tables.
 *   state_dev    hra_delay_state [batch], read and advanced in place.
 *   eoc_bias_dev fp32 [batch, n_codebooks] added to each codebook's EOC logit before the argmax, or
 *                NULL.
 *   codes_dev    int32 [batch, n_codebooks] out; next_emb_dev bf16 [batch, hidden] out =
 *                bf16(sum over k ascending of fp32 code_emb[k][code_k]); done_dev int32 [batch] out.
 *   logits_dev   fp32 [batch, n_codebooks, codebook_size] out (raw logits, bias not added), or NULL.
 * Delay rule per row (t = frame, e = eoc_frame): codebook k is BOS while t < k; EOC when e >= 0 and
 * t - k >= e; otherwise the argmax over all codebook_size logits (lowest index on ties).  If e < 0
 * and an argmaxed codebook k chose EOC, e becomes the smallest such t - k and every codebook with
 * t - k >= e emits EOC in this frame.  done |= (e >= 0 and t >= e + n_codebooks - 1); t += 1. */
int hra_codebook_step(const hra_dims* dims, const void* hidden_dev, const void* head_w_dev,
                      const void* code_emb_dev, hra_delay_state* state_dev,
                      const float* eoc_bias_dev, int32_t batch, int32_t* codes_dev,
                      void* next_emb_dev, int32_t* done_dev, float* logits_dev, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Sampling parameters of hra_codebook_step_sampled (one set for the whole batch). */
typedef struct {
    float temperature; /* > 0: logits are divided by it                                        */
    int32_t top_k;     /* 0 = off; else keep the entries at or above the top_k-th largest       */
    float top_p;       /* in (0, 1]; 1 = off; else keep the shortest prefix (z descending)       */
                       /* whose probability reaches top_p                                        */
} hra_sampling;

/* hra_codebook_step with each non-forced codebook sampled instead of argmaxed (vLLM-Omni PR
 * #8226, Purpose: temperature / top-k / top-p with per-request seeded exponential noise; Test
 * Plan: temperature 1, top-k 50, top-p 0.95).  For row b and codebook k at frame t:
 *   z_v = (logit_v (+ eoc_bias[b][k] on the EOC entry)) / temperature (fp32; NaN counts as -inf);
 *   entries ordered by z descending, ties by ascending index; top-k keeps every entry whose z is
 *   >= the top_k-th largest; top-p keeps an entry while the probability (softmax of z over the
 *   kept entries) of the kept entries before it is < top_p;
 *   the code is the kept entry with the smallest E_v / exp(z_v - z_max) (lowest index on ties),
 *   E_v = -log(u), u = ((w >> 8) + 1) / 2^24 with w = word (v & 3) of Philox4x32-10 at counter
 *   (v >> 2, k, t, 0) under key (seed_b low 32 bits, seed_b high 32 bits).
 * The delay state machine, outputs and workspace are those of hra_codebook_step.
 *   sampling     host parameters (NULL = HRA_ERR_INVALID_ARG); temperature must be finite and
 *                > 0, top_k >= 0, 0 < top_p <= 1 (else HRA_ERR_INVALID_ARG).
 *   seeds_dev    device uint64 [batch] (8-byte aligned): each row's seed, read every step.
 * codebook_size must be <= 2048 (else HRA_ERR_UNSUPPORTED). */
int hra_codebook_step_sampled(const hra_dims* dims, const void* hidden_dev, const void* head_w_dev,
                              const void* code_emb_dev, hra_delay_state* state_dev,
                              const float* eoc_bias_dev, const hra_sampling* sampling,
                              const uint64_t* seeds_dev, int32_t batch, int32_t* codes_dev,
                              void* next_emb_dev, int32_t* done_dev, float* logits_dev,
                              void* workspace, size_t workspace_bytes, void* stream);

/* One frame of the AR audio loop, fully stream-ordered and free of host data dependencies (so a
 * CUDA graph can capture it once and replay it per frame): hra_codebook_step on hidden_dev
 * (codes, next embedding, done, delay state advanced), then hra_decode_dev on the next embedding
 * at the device positions pos_dev (advanced by one), writing the next hidden back to hidden_dev.
 * Sources: the per-frame codebook step and decode pass ("Stabilize Higgs Audio termination and
 * prefill", Summary and Performance: AR decode ms/frame); graph-captured per-frame work
 * (vLLM-Omni PR #8226, Purpose and Step-overhead reductions).
 *   hidden_dev   bf16 [batch, hidden], in: this frame's backbone hidden; out: the next one.
 *   backbone_ws  >= hra_decode_workspace_size(dims, batch, kv->n_slots) bytes;
 *   codebook_ws  >= hra_codebook_workspace_size(dims, batch) bytes (two separate buffers, so
 *                hra_device_error can read either call's error bits).
 *   sampling, seeds_dev  NULL: the greedy step (hra_codebook_step); else the sampled step
 *                (hra_codebook_step_sampled) with these parameters and per-row seeds.
 * Every argument of both steps is checked before anything is enqueued. */
int hra_ar_frame(const hra_dims* dims, const hra_weights* weights, const void* head_w_dev,
                 const void* code_emb_dev, hra_delay_state* state_dev, const float* eoc_bias_dev,
                 const hra_sampling* sampling, const uint64_t* seeds_dev,
                 void* hidden_dev, int32_t* pos_dev, int32_t pos_bound, int32_t batch,
                 const hra_kv_cache* kv, int32_t* codes_dev, void* next_emb_dev, int32_t* done_dev,
                 void* backbone_ws, size_t backbone_ws_bytes, void* codebook_ws,
                 size_t codebook_ws_bytes, void* stream);

/* The same step for callers that cannot allocate device memory -- for instance a streaming-audio
 * callback with a hard per-frame deadline (cudaMalloc may synchronise the device and take
 * milliseconds), or a runtime whose device memory belongs to an allocator that forbids side
 * allocations.  No pages' counterpart: it is an interface convenience, computing exactly what
 * hra_codebook_step computes.  Instead of a caller workspace it uses a fixed 32 MiB scratch array
 * that each GPU loading this library reserves once and holds until the process exits; it calls
 * no cudaMalloc, cudaFree or other allocating routine.
 *   - Limit: accepted while hra_codebook_workspace_size(dims, batch) <= 32 MiB (batch <= 127 for
 *     8 codebooks x 1026 entries at hidden 2560); larger requests return HRA_ERR_WORKSPACE and
 *     enqueue nothing.
 *   - The first call on a device loads the scratch for that device (CUDA loads the module that
 *     holds it on first use, which reserves the 32 MiB then) and looks up its address: make one
 *     warm-up call outside any deadline path and before any stream capture.
 *   - Device error bits (HRA_DEVERR_*) are not reported: they land in the private scratch, which no
 *     caller can pass to hra_device_error.  A caller that needs them uses hra_codebook_step with a
 *     workspace of its own.
 *   - Every call on a device shares the one scratch array, which keeps the last call's contents;
 *     the step clears its error word and overwrites every partial it reads.  Calls that overlap on
 *     the GPU (different streams without ordering) race on the scratch and must be serialised by
 *     the caller.
 * Arguments and results are those of hra_codebook_step without the workspace. */
int hra_codebook_step_noalloc(const hra_dims* dims, const void* hidden_dev, const void* head_w_dev,
                              const void* code_emb_dev, hra_delay_state* state_dev,
                              const float* eoc_bias_dev, int32_t batch, int32_t* codes_dev,
                              void* next_emb_dev, int32_t* done_dev, float* logits_dev, void* stream);

/* ---- projection (diagnostic access to the tensor-core GEMM used by the path) ----------------- */
#define HRA_EPI_STORE 0     /* out bf16 [M, N] = bf16(acc)                                        */
#define HRA_EPI_RESIDUAL 1  /* out bf16 [M, N] = bf16(out + acc)   (in place)                      */
#define HRA_EPI_SWIGLU 2    /* w has 2N rows (gate N, then up N): out bf16 [M, N] =
                               bf16(silu(bf16(gate)) * bf16(up))                                    */
#define HRA_EPI_F32 3       /* out fp32 [M, N] = acc                                                */

size_t hra_linear_workspace_size(int32_t M, int32_t N, int32_t K, int32_t epilogue, int32_t split_k);

/* out = epilogue(a_dev [M, K] x w_dev^T), w_dev [N (or 2N), K], bf16, fp32 accumulation.
 * K must be a multiple of 64 and N of 16; split_k = 0 picks the split automatically; > 1 forces a
 * K split whose fp32 partials go through the workspace. */
int hra_linear(const void* a_dev, const void* w_dev, void* out_dev, int32_t M, int32_t N, int32_t K,
               int32_t epilogue, int32_t split_k, void* workspace, size_t workspace_bytes,
               void* stream);

/* ---- static-FP8 variant of the prefill projections ------------------------------------------ */
/* The FP8 band of the prefill chain ("flashrt-structures 0.2.0, prefill_tower/fp8_chain.py" page, its
 * description: RMSNorm then FP8, merged-QKV,
 * output, gate/up and down FP8 GEMMs with static activation scales; "Stabilize Higgs Audio
 * termination and prefill", Summary: activation scales calibrated on a fixed prompt):
 *   weights      w8 = e4m3(w / s_w) with one per-tensor scale s_w = max|w| / 448;
 *   activations  each projection's input x8 = e4m3(x / s_a) with a static per-layer, per-projection
 *                scale s_a (from hra_fp8_calibrate: max|x| / 448);
 *   GEMM         fp32 sum of the E4M3 products times s_a * s_w, then the bf16 path's epilogue.
 * e4m3() rounds to nearest (ties to even) and saturates finite overflow to +-448 (OCP E4M3, "fn").
 * Every other step (norms, RoPE, attention, SwiGLU, residuals, rounding points) is the bf16
 * prefill's.  Scales are device fp32 scalars so that no call needs a host round trip. */
typedef struct {
    const void* w_qkv;      /* E4M3 [(nq + 2 nkv) hd, H] */
    const void* w_o;        /* E4M3 [H, nq hd]            */
    const void* w_gate_up;  /* E4M3 [2F, H]               */
    const void* w_down;     /* E4M3 [H, F]                */
    const float* w_scale;   /* device float [4]: s_w of qkv, o, gate_up, down */
    const float* a_scale;   /* device float [4]: s_a of the inputs of the same four projections */
} hra_fp8_layer;

/* Weight preparation: w8_dev[i] = e4m3(w[i] / s_w) and *scale_dev = s_w = max|w| / 448 (1 for an
 * all-zero tensor).  w_dev bf16 [n] (16-byte aligned), n a multiple of 8; w8_dev 8-byte aligned. */
int hra_fp8_quantize_weight(const void* w_dev, int64_t n, void* w8_dev, float* scale_dev, void* stream);

/* x8_dev[i] = e4m3(x[i] / *scale_dev) (IEEE division), n a multiple of 8. */
int hra_fp8_quantize(const void* x_dev, int64_t n, const float* scale_dev, void* x8_dev, void* stream);

/* ---- NVFP4 quantization (the FP4 band of the prefill chain) ---------------------------------- */
/* The chain's FP4 band (the fp8_chain page, its precision bands: the FFN pair and the output
 * projection in NVFP4, with block scales computed from the data) in NVIDIA's published NVFP4 format: each block of 16 consecutive
 * elements along K of x_dev bf16 [rows, K] gets the E4M3 scale s = e4m3(amax_block / (6 g)) and
 * the FP4 E2M1 codes e2m1(x / (g * s)) (all 0 when g * s is 0), g = *g_dev the tensor's fp32
 * global scale (e.g. max|x| / (6 * 448)); e2m1() rounds to the nearest of 0, 0.5, 1, 1.5, 2, 3, 4,
 * 6 (ties to the even mantissa) and saturates at +-6; each step is one fp32 rounding.
 *   codes_dev   uint8 [rows, K]: one E2M1 code per byte (sign in bit 3), 16-byte aligned.
 *   scales_dev  uint8 [rows, K / 16]: E4M3 block scales.
 * K a multiple of 16, x_dev 16-byte aligned, g_dev 4-byte aligned (else HRA_ERR_INVALID_ARG).
 * *g_dev must be finite and > 0 (it is device memory, so this is not checked): with any other value
 * the codes and scales are unspecified. */
int hra_nvfp4_quantize(const void* x_dev, int32_t rows, int32_t K, const float* g_dev, void* codes_dev,
                       void* scales_dev, void* stream);

/* NVFP4 weights for the band: w_dev bf16 [rows, K] -> *g_dev = max|w| / (6 * 448) (1 for an all-zero
 * tensor; fp32, on the device) and the codes / block scales of hra_nvfp4_quantize under it.
 * w_dev and codes_dev 16-byte aligned, g_dev 4-byte aligned, K a multiple of 16. */
int hra_nvfp4_quantize_weight(const void* w_dev, int32_t rows, int32_t K, void* codes_dev, void* scales_dev,
                              float* g_dev, void* stream);

/* NVFP4 projection (the band's GEMM): out = epilogue((*g_a) (*g_w) sum_k e2m1(a[m][k]) dec(sa[m][k/16])
 * e2m1(w[n][k]) dec(sw[n][k/16])), fp32 accumulation; a_codes [M, K] and w_codes [N, K] (2N rows
 * for HRA_EPI_SWIGLU: gate rows, then up rows) one E2M1 code per byte, a_scales [M, K/16] and
 * w_scales [N, K/16] E4M3; g_a, g_w device fp32 scalars; epilogues as hra_linear.  K a multiple of
 * 64, N of 8; codes, out and workspace 16-byte aligned.  The product of an E2M1 value and its E4M3
 * block scale is exact in f16, so the tensor cores run on those f16 values and the sum differs
 * from the exact NVFP4 sum only by the order of fp32 additions. */
size_t hra_linear_nvfp4_workspace_size(void);
int hra_linear_nvfp4(const void* a_codes_dev, const void* a_scales_dev, const void* w_codes_dev,
                     const void* w_scales_dev, void* out_dev, int32_t M, int32_t N, int32_t K,
                     const float* g_a_dev, const float* g_w_dev, int32_t epilogue, void* workspace,
                     size_t workspace_bytes, void* stream);

/* The NVFP4 band of the prefill chain (the fp8_chain page, its precision bands): the merged QKV
 * stays in static FP8; the output, gate/up and down projections run in NVFP4 -- E2M1 weights with
 * E4M3 block scales and a global scale, each input quantized per call (block scales from its own
 * data) under a static global scale.
 *   w_qkv        E4M3 [(nq + 2 nkv) hd, H] (hra_fp8_quantize_weight)
 *   codes[p], scales[p], p = 1 (w_o), 2 (w_gate_up), 3 (w_down): hra_nvfp4_quantize_weight output;
 *                entry 0 unused
 *   w_scale      device float [4]: [0] the QKV weight scale, [1..3] the weights' global scales g_w
 *   a_scale      device float [4]: [0] the QKV input's static E4M3 scale (calibration amax / 448),
 *                [1..3] the inputs' static NVFP4 global scales (calibration amax / (6 * 448)) */
typedef struct {
    const void* w_qkv;
    const void* codes[4];
    const void* scales[4];
    const float* w_scale;
    const float* a_scale;
} hra_nvfp4_layer;

/* The band's static input scales from hra_fp8_calibrate's amax_dev [n_layers][4] (device): the
 * QKV input's E4M3 scale amax / 448 and the other three inputs' NVFP4 global scales amax / (6 * 448)
 * (1 where amax is 0), into scale_dev [n_layers][4] (device, the layers' a_scale arrays). */
int hra_nvfp4_band_scales(const float* amax_dev, float* scale_dev, int32_t n_layers, void* stream);

/* hra_prefill with the NVFP4 band in every layer (nvfp4_layers: host array [n_layers]); everything
 * else (embedding, norms, RoPE, attention, SwiGLU, residuals) is the bf16 prefill's.  hidden must
 * be a multiple of 128 (else HRA_ERR_UNSUPPORTED). */
size_t hra_prefill_nvfp4_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens,
                                        int32_t max_len);
int hra_prefill_nvfp4(const hra_dims* dims, const hra_weights* weights, const hra_nvfp4_layer* nvfp4_layers,
                      const int32_t* tokens_dev, const int32_t* seq_lens, int32_t batch, int32_t max_len,
                      const hra_kv_cache* kv, void* last_hidden_dev, void* workspace,
                      size_t workspace_bytes, uint32_t flags, void* stream);

/* FP8 projection: out = epilogue((a8 . w8^T) * (*a_scale) * (*w_scale)), a8 E4M3 [M, K], w8 E4M3
 * [N, K] (2N rows for EPI_SWIGLU), K a multiple of 128; epilogues as hra_linear. */
size_t hra_linear_fp8_workspace_size(int32_t M, int32_t N, int32_t K, int32_t epilogue);
int hra_linear_fp8(const void* a8_dev, const void* w8_dev, void* out_dev, int32_t M, int32_t N, int32_t K,
                   const float* a_scale_dev, const float* w_scale_dev, int32_t epilogue, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Calibration: the bf16 prefill of the calibration batch (every row through the last layer, the
 * cache written as by hra_prefill), recording amax_dev[4 l + p] = max |input| of projection p
 * (0 qkv, 1 o, 2 gate_up, 3 down) of layer l over all rows, and scale_dev[4 l + p] =
 * amax / 448 (1 where amax is 0).  Both device float [4 n_layers].  Arguments as hra_prefill;
 * the workspace holds hra_fp8_calibrate_workspace_size() bytes. */
size_t hra_fp8_calibrate_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens,
                                        int32_t max_len);
int hra_fp8_calibrate(const hra_dims* dims, const hra_weights* weights, const int32_t* tokens_dev,
                      const int32_t* seq_lens, int32_t batch, int32_t max_len, const hra_kv_cache* kv,
                      float* amax_dev, float* scale_dev, void* workspace, size_t workspace_bytes,
                      void* stream);

/* hra_prefill with every projection of every layer in FP8 (fp8_layers: host array [n_layers]).
 * weights still supplies the embedding, the norm gains and the final norm.  hidden, n_q_heads *
 * head_dim and ffn must be multiples of 128 (else HRA_ERR_UNSUPPORTED). */
size_t hra_prefill_fp8_workspace_size(const hra_dims* dims, int32_t batch, int32_t total_tokens,
                                      int32_t max_len);
int hra_prefill_fp8(const hra_dims* dims, const hra_weights* weights, const hra_fp8_layer* fp8_layers,
                    const int32_t* tokens_dev, const int32_t* seq_lens, int32_t batch, int32_t max_len,
                    const hra_kv_cache* kv, void* last_hidden_dev, void* workspace,
                    size_t workspace_bytes, uint32_t flags, void* stream);

/* ---- measurement ---------------------------------------------------------------------------- */
/* Number of kernels the library has launched in this process (host-side count). */
uint64_t hra_launch_counter(void);

/* Kernel classes the event probe can bracket. */
#define HRA_PROBE_NONE 0
#define HRA_PROBE_QKV 1        /* QKV projection of full prefill layers                         */
#define HRA_PROBE_O_PROJ 2     /* o-projection of full prefill layers                           */
#define HRA_PROBE_GATE_UP 3    /* gate/up + SwiGLU projection of full prefill layers            */
#define HRA_PROBE_DOWN 4       /* down projection of full prefill layers                        */
#define HRA_PROBE_ATTENTION 5  /* causal prefill attention of full layers                       */
#define HRA_PROBE_AUDIO_HEAD 6 /* audio-head projection of hra_codebook_step                    */
#define HRA_PROBE_DECODE_ATTENTION 7 /* single-query attention (+ split combine) of hra_decode    */
#define HRA_PROBE_DECODE_LINEAR 8    /* every projection of hra_decode, with its split-K reduction */

/* While a class is selected, every launch of that class is bracketed by a CUDA event pair
 * recorded on the launching stream (events are created on first use; do not select a class while
 * a stream is being captured).  hra_probe_collect synchronises those events, returns the summed
 * elapsed milliseconds, the number of launches and their summed algorithmic work, and clears
 * them.  The work is FLOPs for classes 1-6 and bytes for the HBM-bound classes 7 (K/V bytes read)
 * and 8 (weight bytes read).  Returns HRA_OK or HRA_ERR_CUDA. */
int hra_probe_select(int kernel_class);
int hra_probe_collect(double* total_ms, int64_t* launches, double* total_work);

/* ---- decoder-pass form ---------------------------------------------------------------------- */
/* Selects how a backbone pass over at most 64 token rows in BF16 runs (hra_decode, hra_decode_dev,
 * hra_ar_frame, and hra_prefill / hra_prefill_chunk calls with at most 64 packed rows):
 *   enable != 0: one persistent cooperative kernel walks every layer, with grid-wide barriers
 *     between the phases of a layer, and streams the next projection's weights into shared memory
 *     across those barriers (FlashRT PR #141, Performance: the AR decode time per frame;
 *     vLLM-Omni PR #8226, Step-overhead reductions);
 *   enable == 0 (default): one kernel per step of each layer, chained by programmatic dependent
 *     launch (measured faster on GB300 for the batch sizes of the path).
 * Both compute the same arithmetic (results may differ in the order of fp32 split sums).  In the
 * persistent form every row runs every layer, including a prefill's last layer.  The setting is
 * process-wide; calls already enqueued or captured keep the form they were issued with.  Returns
 * the previous setting (0 or 1). */
int32_t hra_set_decode_pass(int32_t enable);

/* ---- projection GEMM form ------------------------------------------------------------------- */
/* Selects how the BF16 projection GEMMs of at least 512 rows run (the QKV, o, gate/up and down
 * projections of hra_prefill / hra_prefill_chunk and hra_linear; "Stabilize Higgs Audio
 * termination and prefill", Summary: the projection GEMMs):
 *   enable != 0 (default): on clusters of two CTAs, each pair computing 256 x 256 output tiles
 *     with one M = 256 tensor-core MMA per K step (each CTA stages its 128 activation rows and
 *     half of the weight rows);
 *   enable == 0: one CTA per 128 x 256 (or 128 x 128) tile.
 * Both compute the same arithmetic; the K pieces of a last round (and so the fp32 order of their
 * sums) can differ.  Process-wide; calls already enqueued or captured keep their form.  Returns
 * the previous setting (0 or 1). */
int32_t hra_set_gemm_pairs(int32_t enable);

/* ---- errors --------------------------------------------------------------------------------- */
/* Synchronise `stream` and return the sticky HRA_DEVERR_* bits of the last call that used this
 * workspace (each call clears them first), or a negative status. */
int32_t hra_device_error(const void* workspace, void* stream);

/* Human-readable text of a status code. */
const char* hra_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* HRA_H */
