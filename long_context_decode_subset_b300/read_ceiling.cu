// read_ceiling.cu -- the practical read ceiling the score pass is compared with.
//
// The score pass reads the key summary once (Bt * Hkv * N * d_sel * 2 bytes)
// and is timed alone with CUDA events after an L2 flush.  A copy benchmark's
// bandwidth leaves out what any kernel timed that way pays: the launch after
// the flush, the first copies' latency and the drain.  This program reads the
// same number of bytes the same way, with nothing else to do, so that the
// score pass can be placed against it:
//   plain  -- 16-byte non-caching loads, 148 x 4 CTAs of 512 threads, grid-stride,
//             four loads in flight per thread;
//   ring   -- 32 KB cp.async.bulk copies into a six-slot shared-memory ring per
//             CTA (the score pass's ring depth), one CTA per SM, one thread
//             issuing and waiting.
// Each figure is the median of 20 launches, each after a 256 MiB write that
// flushes L2, timed with CUDA events around the launch alone.
//
// Usage: read_ceiling BYTES [BYTES ...]; BYTES a multiple of 32768.  Prints
// one JSON object per size; exits non-zero on a CUDA error or a copy that
// did not land within half a second.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

namespace {

constexpr int kRing = 6;
constexpr uint32_t kChunk = 32768;

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtime()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool landed(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool wait_landed(uint64_t* bar, uint32_t parity)
{
    const uint64_t t0 = gtime();
    while (!landed(bar, parity))
        if (gtime() - t0 > 500000000ull) return false;
    return true;
}

__global__ void __launch_bounds__(512) plain_kernel(const uint4* __restrict__ a, size_t n, unsigned* sink)
{
    uint32_t x = 0;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v[k].x), "=r"(v[k].y), "=r"(v[k].z), "=r"(v[k].w)
                         : "l"(a + i + k * stride));
#pragma unroll
        for (int k = 0; k < 4; ++k) x ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    }
    for (; i < n; i += stride) {
        const uint4 v = a[i];
        x ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (x == 0x9e3779b9u) sink[blockIdx.x] = x;   // keeps the loads
}

__global__ void __launch_bounds__(32, 1) ring_kernel(const unsigned char* __restrict__ a, size_t nchunks,
                                                     unsigned* sink, unsigned* err)
{
    extern __shared__ __align__(1024) unsigned char ring[];
    __shared__ uint64_t bar[kRing];
    if (threadIdx.x != 0) return;
    for (int s = 0; s < kRing; ++s)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&bar[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // this CTA's chunks: [c0, c0 + n)
    const size_t c0 = nchunks * blockIdx.x / gridDim.x;
    const size_t n = nchunks * (blockIdx.x + 1) / gridDim.x - c0;
    auto issue = [&](size_t c) {
        const int s = (int)(c % kRing);
        asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                     ::"r"(saddr(&bar[s])), "r"(kChunk) : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(saddr(ring + (size_t)s * kChunk)), "l"(a + (c0 + c) * kChunk), "r"(kChunk),
                     "r"(saddr(&bar[s]))
                     : "memory");
    };
    for (size_t c = 0; c < n && c < (size_t)kRing; ++c) issue(c);
    uint32_t x = 0;
    for (size_t c = 0; c < n; ++c) {
        const int s = (int)(c % kRing);
        if (!wait_landed(&bar[s], (uint32_t)(c / kRing) & 1u)) {
            atomicOr(err, 1u);
            // the copies still in flight land (or time out) before the CTA leaves
            for (size_t d = c; d < n && d < c + kRing; ++d) wait_landed(&bar[d % kRing], (uint32_t)(d / kRing) & 1u);
            return;
        }
        x ^= *reinterpret_cast<const uint32_t*>(ring + (size_t)s * kChunk);
        if (c + kRing < n) issue(c + kRing);
    }
    if (x == 0x9e3779b9u) sink[blockIdx.x] = x;
}

bool ok(cudaError_t e, const char* what)
{
    if (e == cudaSuccess) return true;
    std::fprintf(stderr, "read_ceiling: %s: %s\n", what, cudaGetErrorString(e));
    return false;
}

}  // namespace

int main(int argc, char** argv)
{
    std::vector<size_t> sizes;
    for (int i = 1; i < argc; ++i) {
        const size_t b = std::strtoull(argv[i], nullptr, 10);
        if (b == 0 || b % kChunk != 0) {
            std::fprintf(stderr, "read_ceiling: %s is not a positive multiple of %u bytes\n", argv[i], kChunk);
            return 2;
        }
        sizes.push_back(b);
    }
    if (sizes.empty()) {
        std::fprintf(stderr, "usage: read_ceiling BYTES [BYTES ...]\n");
        return 2;
    }
    const size_t most = *std::max_element(sizes.begin(), sizes.end());
    const size_t flush_bytes = 256u << 20;
    int sms = 0;
    if (!ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0), "device query")) return 1;
    unsigned char *a = nullptr, *flush = nullptr;
    unsigned *sink = nullptr, *err = nullptr;
    if (!ok(cudaMalloc(&a, most), "cudaMalloc") || !ok(cudaMalloc(&flush, flush_bytes), "cudaMalloc") ||
        !ok(cudaMalloc(&sink, 4 * 4096), "cudaMalloc") || !ok(cudaMalloc(&err, 4), "cudaMalloc"))
        return 1;
    if (!ok(cudaMemset(a, 1, most), "cudaMemset") || !ok(cudaMemset(err, 0, 4), "cudaMemset")) return 1;
    if (!ok(cudaFuncSetAttribute(ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRing * kChunk),
            "cudaFuncSetAttribute"))
        return 1;
    cudaEvent_t e0, e1;
    if (!ok(cudaEventCreate(&e0), "cudaEventCreate") || !ok(cudaEventCreate(&e1), "cudaEventCreate")) return 1;
    for (const size_t bytes : sizes) {
        float med[2];
        for (int mode = 0; mode < 2; ++mode) {
            std::vector<float> t;
            for (int rep = 0; rep < 23; ++rep) {   // the first three are warm-up
                cudaMemsetAsync(flush, rep & 0xff, flush_bytes);
                cudaEventRecord(e0);
                if (mode == 0)
                    plain_kernel<<<sms * 4, 512>>>(reinterpret_cast<const uint4*>(a), bytes / 16, sink);
                else
                    ring_kernel<<<sms, 32, kRing * kChunk>>>(a, bytes / kChunk, sink, err);
                cudaEventRecord(e1);
                if (!ok(cudaEventSynchronize(e1), "launch")) return 1;
                float ms = 0.0f;
                cudaEventElapsedTime(&ms, e0, e1);
                if (rep >= 3) t.push_back(ms * 1e3f);
            }
            std::sort(t.begin(), t.end());
            med[mode] = t[t.size() / 2];
        }
        std::printf("{\"bytes\": %zu, \"plain_loads_us\": %.3f, \"bulk_ring_us\": %.3f}\n", bytes, med[0], med[1]);
    }
    unsigned h = 0;
    if (!ok(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost), "cudaMemcpy")) return 1;
    if (h) {
        std::fprintf(stderr, "read_ceiling: a copy did not land in time\n");
        return 1;
    }
    return ok(cudaGetLastError(), "launch") ? 0 : 1;
}
