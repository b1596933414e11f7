// noalloc.cu -- the delayed-codebook step for callers that cannot allocate device memory.
//
// hra_codebook_step needs a caller-provided workspace (the audio-head logit partials and an error
// word).  Some callers cannot call cudaMalloc at all: a streaming-audio callback with a hard
// per-frame deadline (cudaMalloc may synchronise the device and take milliseconds), or a host
// runtime whose device memory belongs to an allocator that forbids side allocations.  For them,
// hra_codebook_step_noalloc runs the same step with its scratch in a fixed array that every GPU
// loading this library reserves once, for the life of the process.
#include <mutex>

#include "internal.h"

namespace {

// 32 MiB per device, held until exit.  The module that holds it is loaded lazily by CUDA: on each
// device the first cudaGetSymbolAddress below loads it, and the driver reserves the array then, so
// that first call is the slow one.
constexpr size_t kScratchBytes = 32u << 20;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {nullptr};

// Device address of g_scratch on the current device.  In host code the name g_scratch is only a
// host-side stand-in, never a device pointer, so the address is looked up once per device (with
// that device current) and cached.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HRA_ERR_CUDA;
    if (dev < 0 || dev >= 64) return HRA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return HRA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return HRA_OK;
}

}  // namespace

extern "C" int hra_codebook_step_noalloc(const hra_dims* dims, const void* hidden_dev, const void* head_w_dev,
                                         const void* code_emb_dev, hra_delay_state* state_dev,
                                         const float* eoc_bias_dev, int32_t batch, int32_t* codes_dev,
                                         void* next_emb_dev, int32_t* done_dev, float* logits_dev,
                                         void* stream) {
    if (dims == nullptr || batch < 1) return HRA_ERR_INVALID_ARG;
    const size_t need = hra_codebook_workspace_size(dims, batch);
    if (need == 0) return HRA_ERR_UNSUPPORTED;
    if (need > kScratchBytes) return HRA_ERR_WORKSPACE;   // more than the fixed scratch holds
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != HRA_OK) return rc;
    // The step clears the error word itself and overwrites every partial it later reads.
    return hra_codebook_step(dims, hidden_dev, head_w_dev, code_emb_dev, state_dev, eoc_bias_dev, batch, codes_dev,
                             next_emb_dev, done_dev, logits_dev, scratch, kScratchBytes, stream);
}
