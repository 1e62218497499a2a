// Read-bandwidth ceiling of the GPU, for the roofline of the step kernel:
// a device buffer read once per launch, with no arithmetic on the data.
//
//   dllm_probe_bulk_read  every warp streams its share of the buffer through
//                         a private ring of `stages` shared-memory slots of
//                         `copy_bytes` (cp.async.bulk completing on an
//                         mbarrier, L2 evict-first) -- the step kernel's own
//                         way of reading logits -- touching one word per copy;
//   dllm_probe_load_read  every thread reads 16-byte vectors, grid-stride.
//
// Measurement support for bench.py only (built as libdllm_probe.so, beside
// libdllm.so); not part of the step's hot path.  Returns 0, -1 for an
// invalid argument, -6 for a shape beyond the device, or -(1000 + the
// cudaError_t) when a CUDA call fails.

#include <stdint.h>

#include "common.cuh"

namespace dllm {
namespace {

__global__ void bulk_read_kernel(const char* src, long long ncopies, int copy_bytes, int stages, unsigned* sink) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, W = blockDim.x >> 5;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)W * stages * copy_bytes);
    if (lane < stages) mbar_init(smem_addr(&bars[warp * stages + lane]), 1);
    __syncwarp();
    if (lane == 0) mbar_fence_init();
    __syncwarp();
    const long long gw = (long long)blockIdx.x * W + warp, nw = (long long)gridDim.x * W;
    const long long c0 = ncopies * gw / nw, c1 = ncopies * (gw + 1) / nw;
    const uint32_t ring = smem_addr(smem + (size_t)warp * stages * copy_bytes), bar0 = smem_addr(&bars[warp * stages]);
    const uint64_t pol = l2_policy_evict_first();
    long long issued = c0;
    for (int s = 0; s < stages && issued < c1; ++s, ++issued)
        if (lane == 0) {
            mbar_arrive_expect_tx(bar0 + s * 8, copy_bytes);
            bulk_g2s(ring + s * copy_bytes, src + issued * copy_bytes, copy_bytes, bar0 + s * 8, pol);
        }
    unsigned acc = 0;
    uint32_t k = 0;
    bool ok = true;
    for (long long consumed = c0; consumed < c1 && ok; ++consumed, ++k) {
        const int slot = (int)(k % (uint32_t)stages);
        ok = mbar_wait_bounded(bar0 + slot * 8, (k / (uint32_t)stages) & 1u, 1000000000ull);
        if (!ok) break;
        acc ^= *reinterpret_cast<const unsigned*>(smem + ((size_t)warp * stages + slot) * copy_bytes + lane * 4);
        __syncwarp();
        if (issued < c1) {
            if (lane == 0) {
                mbar_arrive_expect_tx(bar0 + slot * 8, copy_bytes);
                bulk_g2s(ring + slot * copy_bytes, src + issued * copy_bytes, copy_bytes, bar0 + slot * 8, pol);
            }
            ++issued;
        }
    }
    if (!ok) {   // let copies in flight land before shared memory goes away
        for (; k < (uint32_t)(issued - c0); ++k)
            if (!mbar_wait_bounded(bar0 + (k % (uint32_t)stages) * 8, (k / (uint32_t)stages) & 1u, 100000000ull)) break;
        if (lane == 0) atomicExch(sink + 1, 1u);
    }
    if (acc == 0x9e3779b9u) sink[0] = acc;   // keeps the reads
}

__global__ void load_read_kernel(const uint4* src, long long n, unsigned* sink) {
    unsigned acc = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const uint4 v = __ldcs(src + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (acc == 0x9e3779b9u) sink[0] = acc;
}

}  // namespace
}  // namespace dllm

// buf: device, `bytes` (a multiple of copy_bytes, 16-byte aligned); sink:
// device, 2 words (sink[1] is set if a wait ran out).  One launch on
// `stream` of `blocks` CTAs of `warps` warps.
extern "C" int dllm_probe_bulk_read(const void* buf, size_t bytes, int blocks, int warps, int stages, int copy_bytes,
                                    unsigned* sink, void* stream) {
    if (!buf || !sink || blocks < 1 || warps < 1 || warps > 32 || stages < 1 || stages > 16 || copy_bytes < 16 ||
        copy_bytes % 16 != 0 || bytes % copy_bytes != 0 || (reinterpret_cast<uintptr_t>(buf) & 15u) != 0)
        return DLLM_ERR_INVAL;
    const size_t smem = (size_t)warps * stages * copy_bytes + (size_t)warps * stages * 8;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return -(1000 + (int)e);
    if (smem > (size_t)optin) return DLLM_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(dllm::bulk_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return -(1000 + (int)e);
    dllm::bulk_read_kernel<<<blocks, warps * 32, smem, dllm::as_stream(stream)>>>(
        static_cast<const char*>(buf), (long long)(bytes / copy_bytes), copy_bytes, stages, sink);
    e = cudaGetLastError();
    return e == cudaSuccess ? DLLM_OK : -(1000 + (int)e);
}

extern "C" int dllm_probe_load_read(const void* buf, size_t bytes, int blocks, int threads, unsigned* sink,
                                    void* stream) {
    if (!buf || !sink || blocks < 1 || threads < 32 || threads > 1024 || bytes % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(buf) & 15u) != 0)
        return DLLM_ERR_INVAL;
    dllm::load_read_kernel<<<blocks, threads, 0, dllm::as_stream(stream)>>>(static_cast<const uint4*>(buf),
                                                                           (long long)(bytes / 16), sink);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DLLM_OK : -(1000 + (int)e);
}
