// Shared helpers of libdllm.so: inline PTX wrappers for sm_103a, launch
// bookkeeping and the per-device error word.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "dllm.h"

namespace dllm {

// ---------------------------------------------------------------------------
// Host helpers.
// ---------------------------------------------------------------------------
// Remember the failing CUDA status for dllm_last_cuda_error().
void note_cuda_error(cudaError_t e);

// Fault injection (dllm_inject_cuda_error): a CUDA status to report in
// place of one of this thread's coming CUDA calls, or cudaSuccess.
cudaError_t injected_cuda_error();

#define DLLM_CUDA_TRY(expr)                                             \
    do {                                                                \
        cudaError_t _e = ::dllm::injected_cuda_error();                 \
        if (_e == cudaSuccess) _e = (expr);                             \
        if (_e != cudaSuccess) {                                        \
            ::dllm::note_cuda_error(_e);                                \
            return DLLM_ERR_CUDA;                                       \
        }                                                               \
    } while (0)

// Device address of the current device's error word (set up once per device).
int* error_word_ptr();

// SM count of the current device (cached per device).
int sm_count();

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch: a kernel launched with
// launch_dependent() may become resident while the previous kernel in the
// stream still runs; it must call pdl_wait() before touching anything that
// kernel writes (a no-op for an ordinary launch).  pdl_release() lets the
// next such kernel be scheduled early.  Every kernel that a dependent launch
// may follow waits before it finishes, so completion stays transitive.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` so that it may overlap the tail of the previous kernel in
// the stream (it must call pdl_wait() first, see above).
template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// mbarrier (CTA scope) -------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One bounded try: the thread may be suspended until the phase completes
// or about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns = 1000000u) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Non-blocking test of phase `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of a barrier; gives up after `limit_ns` and
// returns false (the caller records DLLM_DEVERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
#if defined(DLLM_WAIT_SLEEP_NS) && DLLM_WAIT_SLEEP_NS > 0
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t ts = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(DLLM_WAIT_SLEEP_NS);
        if (mbar_test_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && globaltimer_ns() - ts > limit_ns) return false;
    }
#else
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
#endif
}

// Bulk (TMA-engine) copy global -> shared, completing on an mbarrier --------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Arithmetic -------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed f32x2 arithmetic (sm_100 and later): a 64-bit register pair holds
// two floats, low word first.
__device__ __forceinline__ unsigned long long f32x2_splat(float x) {
    const unsigned long long u = __float_as_uint(x);
    return (u << 32) | u;
}

// acc += (2^(lo * s + n), 2^(hi * s + n)) for the two bf16 values of `w`
// (lo = the low half, widened exactly by moving it to the top 16 bits; hi =
// the high half with the low 16 bits cleared).  s and n are f32x2 pairs.
// Each half is rounded exactly as fmaf, ex2.approx.ftz and a float add
// would round it.
__device__ __forceinline__ void acc_exp2_bf16x2(unsigned long long& acc, uint32_t w, unsigned long long s,
                                                unsigned long long n) {
    asm("{\n\t.reg .b32 l, h;\n\t.reg .b64 p;\n\t"
        "prmt.b32 l, %1, 0, 0x1044;\n\t"
        "and.b32 h, %1, 0xffff0000;\n\t"
        "mov.b64 p, {l, h};\n\t"
        "fma.rn.f32x2 p, p, %2, %3;\n\t"
        "mov.b64 {l, h}, p;\n\t"
        "ex2.approx.ftz.f32 l, l;\n\t"
        "ex2.approx.ftz.f32 h, h;\n\t"
        "mov.b64 p, {l, h};\n\t"
        "add.rn.f32x2 %0, %0, p;\n\t}"
        : "+l"(acc)
        : "r"(w), "l"(s), "l"(n));
}

// Elementwise max of two packed bf16 pairs.
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Atomic add with acquire-release semantics at GPU scope (orders this
// thread's earlier writes before it and later reads after it).
__device__ __forceinline__ int atom_add_acqrel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Atomic add with release semantics at GPU scope: this thread's earlier
// writes are visible to whoever acquires a later value of the counter.
__device__ __forceinline__ int atom_add_release_gpu(int* p, int v) {
    int old;
    asm volatile("atom.release.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Unsigned division by a divisor fixed at launch (Granlund and Montgomery,
// "Division by Invariant Integers using Multiplication", PLDI 1994, section
// 4): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(m, n) + n) >> l for every 0 <= n < 2^31 (the sum stays
// below 2^32 because umulhi(m, n) < n).
struct FastDiv {
    uint32_t m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const unsigned long long num = (1ull << 32) * ((1ull << l) - d);   // < 2^63: 2^l - d < d <= 2^31
    return FastDiv{static_cast<uint32_t>(num / d + 1), l};
}

__device__ __forceinline__ int fast_div(int n, const FastDiv& f) {
    const uint32_t u = static_cast<uint32_t>(n);
    return static_cast<int>((__umulhi(u, f.m) + u) >> f.l);
}

// Relaxed (but strong, single-copy atomic) accesses at GPU scope: no
// ordering with this thread's other accesses, no fence.
__device__ __forceinline__ int atom_add_relaxed_gpu(int* p, int v) {
    int old;
    asm volatile("atom.relaxed.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed_gpu_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void st_release_cta_shared(int* p, int v) {
    asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_cta_shared(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

}  // namespace dllm
