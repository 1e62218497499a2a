// Library-wide entry points of libdllm.so: status strings, ABI checks, the
// per-device error word and cached device facts.

#include <atomic>

#include "common.cuh"

namespace dllm {
namespace {

// First device-side error since the last dllm_get_device_error (one per device).
__device__ int g_error_word;

// Per-device facts, looked up on first use and then read on every launch
// without a lock: a lookup that races with another thread's stores the same
// value, and the atomics publish it.
constexpr int kMaxDevices = 64;
std::atomic<int*> g_err_ptr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];

}  // namespace

thread_local int t_last_cuda_error = 0;
thread_local int t_inject_code = 0;        // status to report instead of a CUDA call
thread_local int t_inject_countdown = 0;   // the call that reports it (1 = the next one)

void note_cuda_error(cudaError_t e) { t_last_cuda_error = static_cast<int>(e); }

cudaError_t injected_cuda_error() {
    if (t_inject_countdown <= 0) return cudaSuccess;
    if (--t_inject_countdown > 0) return cudaSuccess;
    return static_cast<cudaError_t>(t_inject_code);
}

int* error_word_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int* p = g_err_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void* q = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&q, g_error_word);
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return nullptr;
    }
    g_err_ptr[dev].store(static_cast<int*>(q), std::memory_order_release);
    return static_cast<int*>(q);
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    const int n0 = g_sm_count[dev].load(std::memory_order_acquire);
    if (n0 > 0) return n0;
    int n = 0;
    const cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
        note_cuda_error(e);
        return -1;
    }
    g_sm_count[dev].store(n, std::memory_order_release);
    return n;
}

}  // namespace dllm

extern "C" const char* dllm_strerror(int code) {
    switch (code) {
        case DLLM_OK: return "ok";
        case DLLM_ERR_INVAL: return "invalid argument (size, pointer or value out of range)";
        case DLLM_ERR_ALIGN: return "alignment rule broken (logits must be 16-byte aligned, ldv a multiple of 8)";
        case DLLM_ERR_CUDA: return "CUDA runtime call failed";
        case DLLM_ERR_DEVICE: return "device error word set";
        case DLLM_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case DLLM_ERR_UNSUPPORTED: return "shape beyond this build's limits";
        case DLLM_ERR_SCRATCH_LIMIT: return "shape needs more scratch than dllm_step_noalloc's built-in buffer holds";
        default: return "unknown status code";
    }
}

extern "C" int dllm_abi_version(void) { return DLLM_ABI_VERSION; }

extern "C" int dllm_inject_cuda_error(int32_t cuda_error, int32_t countdown) {
    if (countdown < 0 || (countdown > 0 && cuda_error == 0)) return DLLM_ERR_INVAL;
    dllm::t_inject_code = cuda_error;
    dllm::t_inject_countdown = countdown;
    return DLLM_OK;
}

extern "C" int dllm_last_cuda_error(const char** name) {
    const int e = dllm::t_last_cuda_error;
    if (name) *name = cudaGetErrorName(static_cast<cudaError_t>(e));
    return e;
}

extern "C" size_t dllm_struct_size(int which) {
    switch (which) {
        case 0: return sizeof(dllm_step_args);
        case 1: return sizeof(dllm_pack_args);
        case 2: return sizeof(dllm_compact_args);
        case 3: return sizeof(dllm_advance_args);
        case 4: return sizeof(dllm_refill_args);
        case 5: return sizeof(dllm_loop_config);
        case 6: return sizeof(dllm_loop_info_t);
        case 7: return sizeof(dllm_vocab_shard);
        case 8: return sizeof(dllm_loop_control);
        default: return 0;
    }
}

extern "C" int dllm_get_device_error(void* stream, int32_t* code) {
    if (!code) return DLLM_ERR_INVAL;
    int* p = dllm::error_word_ptr();
    if (!p) return DLLM_ERR_CUDA;
    cudaStream_t s = dllm::as_stream(stream);
    int v = 0;
    DLLM_CUDA_TRY(cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s));
    DLLM_CUDA_TRY(cudaStreamSynchronize(s));
    if (v != 0) {
        DLLM_CUDA_TRY(cudaMemsetAsync(p, 0, sizeof(int), s));
        DLLM_CUDA_TRY(cudaStreamSynchronize(s));
    }
    *code = v;
    return DLLM_OK;
}
