// ar_probe.cu -- bandwidth probes that give the roofline denominators, and
// latency probes of the host link that bound the small calls.
//
// Host link: zero-copy kernels that stream to and from mapped pinned host
// memory with 16-byte accesses, alone and both directions at once (the pages'
// peer-copy probe measures both directions at once too: "fix(group): run each
// rank on a non-blocking stream", section "Why").  HBM: a 16-byte copy kernel
// between two device buffers.  Every probe owns its buffers and a private
// non-blocking stream, and times with CUDA events on that stream.
#include <algorithm>
#include <cstring>

#include "ar_internal.h"

namespace {

// Each thread keeps kUnroll independent 16-byte accesses in flight per loop
// trip: over a long-latency link the bandwidth a kernel sees is bytes in
// flight / latency.
constexpr int kUnroll = 8;

__global__ void probe_write_kernel(uint4 *dst, uint64_t nvec) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint4 v = make_uint4(0x3c003c00u, blockIdx.x, threadIdx.x, 0x12345678u);
    uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) dst[i + k * stride] = v;
    }
    for (; i < nvec; i += stride) dst[i] = v;
}

__global__ void probe_read_kernel(const uint4 *src, uint64_t nvec, unsigned int *sink) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    unsigned int x = 0;
    uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) v[k] = src[i + k * stride];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) x ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    }
    for (; i < nvec; i += stride) {
        const uint4 v = src[i];
        x ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (x == 0x9e3779b9u) sink[0] = x;  // keeps the loads alive; practically never taken
}

__global__ void probe_copy_kernel(uint4 *dst, const uint4 *src, uint64_t nvec) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < nvec; i += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) v[k] = src[i + k * stride];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) dst[i + k * stride] = v[k];
    }
    for (; i < nvec; i += stride) dst[i] = src[i];
}

// %globaltimer: one nanosecond clock for every SM.
__device__ __forceinline__ unsigned long long probe_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Both directions at once, as concurrent streams: the first `wblocks` blocks
// store 16-byte vectors to one mapped host buffer, the other blocks load them
// from another, each block a contiguous chunk of kBidirUnroll x blockDim
// vectors per step (wrapping around its buffer), until `dur_ns` have passed
// since the block started.  Each block adds the bytes it moved to counts[0]
// (stored) or counts[1] (loaded).  The loop ends on the time window; every
// index is reduced below nvec.  The stored values vary with the index, as a
// payload does: with one value repeated in every store the writers took the
// link at ~185 GB/s and held the readers to ~58 on a GB300, against ~170 each
// way with varying values.  (A kernel that copies one host buffer to another
// ties each store to a load and reaches only ~138 GB/s each way.)
constexpr int kBidirUnroll = 4;
__global__ void probe_bidir_kernel(uint4 *dst, const uint4 *src, uint64_t nvec, int wblocks, uint64_t dur_ns,
                                   unsigned long long *counts, unsigned int *sink) {
    const bool writer = (int)blockIdx.x < wblocks;
    const uint64_t nb = writer ? (uint64_t)wblocks : (uint64_t)gridDim.x - (uint64_t)wblocks;
    const uint64_t bi = writer ? (uint64_t)blockIdx.x : (uint64_t)blockIdx.x - (uint64_t)wblocks;
    const uint64_t chunk = (uint64_t)kBidirUnroll * blockDim.x;
    const uint64_t step = (nb * chunk) % nvec;
    __shared__ unsigned long long s_t0;
    if (threadIdx.x == 0) s_t0 = probe_timer_ns();
    __syncthreads();
    const unsigned long long t0 = s_t0;
    uint64_t start = (bi * chunk) % nvec;
    unsigned long long moved = 0;
    unsigned int x = 0;
    while (probe_timer_ns() - t0 < dur_ns) {
        uint64_t idx[kBidirUnroll];
#pragma unroll
        for (int k = 0; k < kBidirUnroll; ++k) {
            idx[k] = start + (uint64_t)k * blockDim.x + threadIdx.x;
            if (idx[k] >= nvec) idx[k] %= nvec;
        }
        if (writer) {
#pragma unroll
            for (int k = 0; k < kBidirUnroll; ++k) dst[idx[k]] = make_uint4((unsigned)idx[k], blockIdx.x, threadIdx.x, 0x12345678u);
        } else {
            uint4 v[kBidirUnroll];
#pragma unroll
            for (int k = 0; k < kBidirUnroll; ++k) v[k] = __ldcg(src + idx[k]);
#pragma unroll
            for (int k = 0; k < kBidirUnroll; ++k) x ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
        }
        moved += (unsigned long long)kBidirUnroll * 16ull;
        start += step;
        if (start >= nvec) start -= nvec;
    }
    atomicAdd(&counts[writer ? 0 : 1], moved);
    if (x == 0x9e3779b9u) sink[0] = x;
}

// ---- latencies of the host link (one block or two, so nothing queues)

// n dependent 8-byte loads, each from the line the previous one named: one
// round trip to the memory behind `buf` per load.
__global__ void probe_chase_kernel(const unsigned long long *buf, int n, unsigned long long *out) {
    unsigned long long i = 0;
    const unsigned long long t0 = probe_timer_ns();
    for (int k = 0; k < n; ++k) {
        unsigned long long v;
        asm volatile("ld.relaxed.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(buf + i * 16) : "memory");
        i = v;
    }
    out[0] = probe_timer_ns() - t0;
    out[1] = i;
}

// n rounds of: every thread of one block stores 16 bytes to host memory (4
// KiB with 256 threads), barrier, thread 0 a system-scope (SYS) or GPU-scope
// fence (returns once the stores are ordered for every observer of that
// scope), barrier -- the publish step of a block.
template <int SYS>
__global__ void probe_store_fence_kernel(uint4 *dst, int n, unsigned long long *out) {
    const unsigned long long t0 = probe_timer_ns();
    for (int k = 0; k < n; ++k) {
        dst[(uint64_t)(k & 63) * blockDim.x + threadIdx.x] = make_uint4(k, 1, 2, 3);
        __syncthreads();
        if (threadIdx.x == 0) {
            if (SYS)
                asm volatile("fence.sc.sys;" ::: "memory");
            else
                asm volatile("fence.sc.gpu;" ::: "memory");
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) out[0] = probe_timer_ns() - t0;
}

// Two blocks pass a counter back and forth n times through two flag words
// (release store, acquire polls), system or GPU scope.  Every wait is bounded
// (100 ms); a wait that runs out sets *err and ends the kernel.
template <int SYS>
__global__ void probe_pingpong_kernel(unsigned long long *f, int n, unsigned long long *out, unsigned int *err) {
    if (threadIdx.x != 0) return;
    unsigned long long *mine = f + (blockIdx.x ? 16 : 0), *theirs = f + (blockIdx.x ? 0 : 16);
    const unsigned long long t0 = probe_timer_ns();
    for (int k = 1; k <= n; ++k) {
        const unsigned long long want = (unsigned long long)k;
        if (blockIdx.x == 0) {
            if (SYS) asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(mine), "l"(want) : "memory");
            else asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(mine), "l"(want) : "memory");
        }
        const unsigned long long s = probe_timer_ns();
        for (;;) {
            unsigned long long v;
            if (SYS) asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(theirs) : "memory");
            else asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(theirs) : "memory");
            if (v >= want) break;
            if (*(volatile unsigned int *)err || probe_timer_ns() - s > 100000000ull) {
                atomicExch(err, 1u);
                return;
            }
        }
        if (blockIdx.x == 1) {
            if (SYS) asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(mine), "l"(want) : "memory");
            else asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(mine), "l"(want) : "memory");
        }
    }
    if (blockIdx.x == 0) out[0] = probe_timer_ns() - t0;
}

int grid_for(const void *k, int threads) {
    int dev = 0, sms = 0, occ = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, threads, 0);
    if (occ < 1) occ = 1;
    return sms * occ;
}

struct Timer {
    cudaEvent_t a = nullptr, b = nullptr;
    Timer() {
        cudaEventCreate(&a);
        cudaEventCreate(&b);
    }
    ~Timer() {
        cudaEventDestroy(a);
        cudaEventDestroy(b);
    }
};

}  // namespace

extern "C" {

AR_API int ar_probe_host_link(uint64_t bytes, int reps, double gbs[4]) {
    if (!gbs || reps < 1 || bytes < 16 || bytes % 16) return AR_EINVAL;
    const int threads = 512;
    const uint64_t nvec = bytes / 16;
    void *hw = nullptr, *hr = nullptr;
    uint4 *dw = nullptr, *dr = nullptr;
    unsigned int *sink = nullptr;
    cudaStream_t s1 = nullptr, s2 = nullptr;
    int rc = AR_OK;
    const unsigned fl = cudaHostAllocMapped | cudaHostAllocPortable;
    if (cudaHostAlloc(&hw, bytes, fl) != cudaSuccess || cudaHostAlloc(&hr, bytes, fl) != cudaSuccess ||
        cudaMalloc((void **)&sink, 256) != cudaSuccess) {
        rc = AR_ENOMEM;
    }
    if (rc == AR_OK) {
        std::memset(hw, 0, bytes);
        std::memset(hr, 1, bytes);
        if (cudaHostGetDevicePointer((void **)&dw, hw, 0) != cudaSuccess ||
            cudaHostGetDevicePointer((void **)&dr, hr, 0) != cudaSuccess ||
            cudaStreamCreateWithFlags(&s1, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking) != cudaSuccess)
            rc = AR_ECUDA;
    }
    if (rc == AR_OK) {
        const int gw = grid_for((const void *)probe_write_kernel, threads);
        const int gr = grid_for((const void *)probe_read_kernel, threads);
        Timer t1;
        float ms = 0.f;
        // warm up both directions once
        probe_write_kernel<<<gw, threads, 0, s1>>>(dw, nvec);
        probe_read_kernel<<<gr, threads, 0, s1>>>(dr, nvec, sink);
        cudaStreamSynchronize(s1);
        // write alone
        cudaEventRecord(t1.a, s1);
        for (int i = 0; i < reps; ++i) probe_write_kernel<<<gw, threads, 0, s1>>>(dw, nvec);
        cudaEventRecord(t1.b, s1);
        cudaEventSynchronize(t1.b);
        cudaEventElapsedTime(&ms, t1.a, t1.b);
        gbs[0] = (double)bytes * reps / (ms * 1e-3) / 1e9;
        // read alone
        cudaEventRecord(t1.a, s1);
        for (int i = 0; i < reps; ++i) probe_read_kernel<<<gr, threads, 0, s1>>>(dr, nvec, sink);
        cudaEventRecord(t1.b, s1);
        cudaEventSynchronize(t1.b);
        cudaEventElapsedTime(&ms, t1.a, t1.b);
        gbs[1] = (double)bytes * reps / (ms * 1e-3) / 1e9;
        // both at once: half the blocks store, half load, for a fixed window
        // (at least 1 ms, about `bytes` each way); two blocks per SM, all
        // resident at once, so every block's window overlaps every other's.
        // Rates over the kernel's event time; the best of three windows.
        int dev = 0, sms = 0, occ = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, (const void *)probe_bidir_kernel, threads, 0);
        const int gb = sms * (occ < 2 ? (occ < 1 ? 1 : occ) : 2);
        const uint64_t dur_ns = std::max<uint64_t>(1000000ull, bytes / 150ull);
        unsigned long long *counts = nullptr;
        if (cudaMalloc((void **)&counts, 16) != cudaSuccess) rc = AR_ENOMEM;
        gbs[2] = gbs[3] = 0.0;
        for (int rep = 0; rep < 4 && rc == AR_OK; ++rep) {
            unsigned long long c[2] = {0, 0};
            cudaMemsetAsync(counts, 0, 16, s1);
            cudaEventRecord(t1.a, s1);
            probe_bidir_kernel<<<gb, threads, 0, s1>>>(dw, dr, nvec, gb / 2, dur_ns, counts, sink);
            cudaEventRecord(t1.b, s1);
            if (cudaMemcpyAsync(c, counts, 16, cudaMemcpyDeviceToHost, s1) != cudaSuccess ||
                cudaStreamSynchronize(s1) != cudaSuccess) {
                rc = AR_ECUDA;
                break;
            }
            cudaEventElapsedTime(&ms, t1.a, t1.b);
            const double w = (double)c[0] / (ms * 1e-3) / 1e9, r = (double)c[1] / (ms * 1e-3) / 1e9;
            if (rep > 0 && w + r > gbs[2] + gbs[3]) {  // the first window warms up
                gbs[2] = w;
                gbs[3] = r;
            }
        }
        if (counts) cudaFree(counts);
        if (cudaGetLastError() != cudaSuccess) rc = AR_ECUDA;
    }
    if (s1) cudaStreamDestroy(s1);
    if (s2) cudaStreamDestroy(s2);
    if (hw) cudaFreeHost(hw);
    if (hr) cudaFreeHost(hr);
    if (sink) cudaFree(sink);
    (void)cudaGetLastError();
    return rc;
}

AR_API int ar_probe_host_link_latency(int reps, double ns[5]) {
    if (!ns || reps < 1 || reps > 100000) return AR_EINVAL;
    constexpr int kLines = 4096;                  // chase over 4096 lines of 128 B (512 KiB)
    const uint64_t host_bytes = (uint64_t)kLines * 128;
    void *hb = nullptr, *hf = nullptr;
    unsigned long long *dhb = nullptr, *dhf = nullptr, *dflag = nullptr, *dout = nullptr;
    unsigned int *derr = nullptr;
    cudaStream_t st = nullptr;
    int rc = AR_OK;
    const unsigned fl = cudaHostAllocMapped | cudaHostAllocPortable;
    if (cudaHostAlloc(&hb, host_bytes, fl) != cudaSuccess || cudaHostAlloc(&hf, 4096, fl) != cudaSuccess ||
        cudaMalloc((void **)&dflag, 4096) != cudaSuccess || cudaMalloc((void **)&dout, 64) != cudaSuccess ||
        cudaMalloc((void **)&derr, 64) != cudaSuccess)
        rc = AR_ENOMEM;
    if (rc == AR_OK) {
        unsigned long long *h = static_cast<unsigned long long *>(hb);
        std::memset(hb, 0, host_bytes);
        for (int i = 0; i < kLines; ++i) h[(size_t)i * 16] = (unsigned long long)((i * 1237 + 1) % kLines);
        if (cudaHostGetDevicePointer((void **)&dhb, hb, 0) != cudaSuccess ||
            cudaHostGetDevicePointer((void **)&dhf, hf, 0) != cudaSuccess ||
            cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess ||
            cudaMemsetAsync(derr, 0, 64, st) != cudaSuccess)
            rc = AR_ECUDA;
    }
    unsigned long long hout[2] = {0, 0};
    auto run = [&](auto launch, int per) -> double {
        double best = 1e30;
        for (int rep = 0; rep < 3 && rc == AR_OK; ++rep) {
            launch();
            if (cudaMemcpyAsync(hout, dout, 16, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
                cudaStreamSynchronize(st) != cudaSuccess) {
                rc = AR_ECUDA;
                break;
            }
            unsigned int e = 0;
            if (cudaMemcpy(&e, derr, 4, cudaMemcpyDeviceToHost) != cudaSuccess) rc = AR_ECUDA;
            else if (e) rc = AR_ETIMEOUT;
            const double v = (double)hout[0] / per;
            if (v < best) best = v;
        }
        return best;
    };
    if (rc == AR_OK) ns[0] = run([&] { probe_chase_kernel<<<1, 1, 0, st>>>(dhb, reps, dout); }, reps);
    if (rc == AR_OK)
        ns[1] = run([&] { probe_store_fence_kernel<1><<<1, 256, 0, st>>>(reinterpret_cast<uint4 *>(dhb), reps, dout); },
                    reps);
    if (rc == AR_OK)
        ns[4] = run([&] { probe_store_fence_kernel<0><<<1, 256, 0, st>>>(reinterpret_cast<uint4 *>(dhb), reps, dout); },
                    reps);
    if (rc == AR_OK) {
        std::memset(hf, 0, 4096);
        // a round trip is two one-way trips
        ns[2] = run(
            [&] {
                std::memset(hf, 0, 4096);
                probe_pingpong_kernel<1><<<2, 32, 0, st>>>(dhf, reps, dout, derr);
            },
            2 * reps);
    }
    if (rc == AR_OK)
        ns[3] = run(
            [&] {
                cudaMemsetAsync(dflag, 0, 4096, st);
                probe_pingpong_kernel<0><<<2, 32, 0, st>>>(dflag, reps, dout, derr);
            },
            2 * reps);
    if (rc == AR_OK && cudaGetLastError() != cudaSuccess) rc = AR_ECUDA;
    if (st) {
        cudaStreamSynchronize(st);
        cudaStreamDestroy(st);
    }
    if (hb) cudaFreeHost(hb);
    if (hf) cudaFreeHost(hf);
    if (dflag) cudaFree(dflag);
    if (dout) cudaFree(dout);
    if (derr) cudaFree(derr);
    (void)cudaGetLastError();
    return rc;
}

AR_API int ar_probe_hbm_copy(uint64_t bytes, int reps, double *gbs) {
    if (!gbs || reps < 1 || bytes < 16 || bytes % 16) return AR_EINVAL;
    const int threads = 512;
    uint4 *a = nullptr, *b = nullptr;
    cudaStream_t s = nullptr;
    int rc = AR_OK;
    if (cudaMalloc((void **)&a, bytes) != cudaSuccess || cudaMalloc((void **)&b, bytes) != cudaSuccess)
        rc = AR_ENOMEM;
    if (rc == AR_OK && (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
                        cudaMemsetAsync(a, 1, bytes, s) != cudaSuccess))
        rc = AR_ECUDA;
    if (rc == AR_OK) {
        const int g = grid_for((const void *)probe_copy_kernel, threads);
        Timer t;
        float ms = 0.f;
        probe_copy_kernel<<<g, threads, 0, s>>>(b, a, bytes / 16);
        cudaEventRecord(t.a, s);
        for (int i = 0; i < reps; ++i) probe_copy_kernel<<<g, threads, 0, s>>>(i & 1 ? a : b, i & 1 ? b : a, bytes / 16);
        cudaEventRecord(t.b, s);
        cudaEventSynchronize(t.b);
        cudaEventElapsedTime(&ms, t.a, t.b);
        *gbs = 2.0 * (double)bytes * reps / (ms * 1e-3) / 1e9;
        if (cudaGetLastError() != cudaSuccess) rc = AR_ECUDA;
    }
    if (s) cudaStreamDestroy(s);
    if (a) cudaFree(a);
    if (b) cudaFree(b);
    (void)cudaGetLastError();
    return rc;
}

}  // extern "C"
