// ar_noalloc.cu -- ar_allreduce_noalloc: an all-reduce entry point that
// allocates nothing.
//
// Some callers cannot allocate device memory when they reduce: code that runs
// inside another library's memory pool or arena (which owns every allocation
// on the device), code that must not call cudaMalloc on a latency-critical
// path (it can synchronise the device), and embedded runtimes that set up all
// memory once at start-up.  For them this entry point takes the R ranks'
// inputs and outputs from the caller and keeps its own working memory (the
// exchange slots, the per-block flags and an abort word) in one file-scope
// device array of fixed size, which every GPU that loads this library holds
// until the process exits.
//
// It is a single-launch form of the one-shot exchange-and-add kernel: one
// cooperative grid of B x R blocks, block (b, r) playing block b of rank r, so
// all R ranks are resident together by construction.  Each call first clears
// the flags, the abort word and the error record (cudaMemsetAsync on the
// array), then launches.  Calls on one stream follow each other; calls that
// overlap on the GPU (different streams, no ordering between them) share the
// array and race.
//
// A block whose wait for a peer runs out of time (which needs the GPU to stop
// scheduling part of a resident cooperative grid) leaves without writing its
// outputs and records itself in the array's error record.  The enqueueing call
// has already returned AR_OK by then, so the record is read separately:
// ar_noalloc_status() copies it out once the caller has synchronised with the
// call's stream, and the next call on the device clears it.
#include <atomic>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "ar_allreduce.cuh"
#include "ar_internal.h"
#include "ar_sync.cuh"

namespace tda {
namespace {

constexpr uint64_t kNoAllocMaxBytes = 1ull << 20;   // per rank: 524288 fp16/bf16 elements
constexpr int kNoAllocMaxBlocks = 64;                // per rank
constexpr uint64_t kNoAllocSlotBytes = (uint64_t)kMaxRanks * kNoAllocMaxBytes;                        // 8 MiB
constexpr uint64_t kNoAllocFlagBytes = (uint64_t)kMaxRanks * kNoAllocMaxBlocks * kFlagStrideWords * 8;  // 64 KiB
constexpr uint64_t kNoAllocMiscBytes = 256;          // abort word + an error record
constexpr uint64_t kNoAllocScratchBytes = kNoAllocSlotBytes + kNoAllocFlagBytes + kNoAllocMiscBytes;
constexpr uint64_t kNoAllocAbortOffset = kNoAllocSlotBytes + kNoAllocFlagBytes;
constexpr uint64_t kNoAllocErrOffset = kNoAllocAbortOffset + 64;
static_assert(64 + sizeof(ar_error_info) <= kNoAllocMiscBytes, "error record fits the misc area");

// The scratch: [R][kNoAllocMaxBytes] slots, then the flags, then the abort
// word and an error record.  Device code reaches it through the pointer the
// host passes in; the host gets that pointer from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct RankPtrs {
    const uint16_t *in[kMaxRanks];
    uint16_t *out[kMaxRanks];
};

template <class Ops, int R>
__global__ void __launch_bounds__(kThreads)
    allreduce_noalloc_kernel(RankPtrs ptrs, uint64_t numel, uint8_t *scratch, uint64_t timeout_ns) {
    __shared__ int s_bail;
    const int rank = blockIdx.y;
    const int b = blockIdx.x;
    const int B = gridDim.x;
    const int tid = threadIdx.x;
    const uint16_t *in = ptrs.in[0];
    uint16_t *out = ptrs.out[0];
#pragma unroll
    for (int q = 1; q < R; ++q) {
        if (rank == q) {
            in = ptrs.in[q];
            out = ptrs.out[q];
        }
    }

    DevState d;
    d.slots = scratch;
    d.flags = reinterpret_cast<unsigned long long *>(scratch + kNoAllocSlotBytes);
    d.ctr = nullptr;
    d.abort_word = reinterpret_cast<unsigned int *>(scratch + kNoAllocAbortOffset);
    d.err = reinterpret_cast<ar_error_info *>(scratch + kNoAllocErrOffset);
    d.slot_bytes = kNoAllocMaxBytes;
    d.timeout_ns = timeout_ns;
    d.bmax = kNoAllocMaxBlocks;
    d.cmax = kNoAllocMaxBlocks;
    d.sys_scope = 0;
    d.ll = nullptr;
    d.ll_vecs = 0;

    const uint64_t nvec_full = numel / 8;
    const int tail = (int)(numel % 8);
    const uint64_t nv = nvec_full + (tail ? 1 : 0);
    const uint64_t ntiles = (nv + kThreads - 1) / kThreads;
    const uint64_t nstages = ntiles > (uint64_t)b ? (ntiles - b + B - 1) / B : 0;
    const uint64_t slot_vecs = kNoAllocMaxBytes / 16;
    uint4 *const slot_base = reinterpret_cast<uint4 *>(scratch);
    uint4 *const my_slot = slot_base + (uint64_t)rank * slot_vecs;
    if (tid == 0) s_bail = 0;
    __syncthreads();

    for (uint64_t s = 0; s < nstages; ++s) {
        const uint64_t v = ((uint64_t)b + s * B) * kThreads + tid;
        const uint4 own = load_own(in, v, nvec_full, tail);
        if (v < nv) my_slot[v] = own;
        __syncthreads();
        if (tid == 0) publish_stage(d, rank, b, s + 1);  // flags start at 0 every call
        if (wait_peers(d, R, rank, b, s + 1, &s_bail)) return;
        if (v < nv) {
            uint4 vals[R];
#pragma unroll
            for (int p = 0; p < R; ++p) {
                uint4 x = own;
                if (p != rank) x = ld_cg_v4(slot_base + (uint64_t)p * slot_vecs + v);
                vals[p] = x;
            }
            float acc[8];
            accumulate8<Ops, true>(acc, vals[0]);
#pragma unroll
            for (int p = 1; p < R; ++p) accumulate8<Ops, false>(acc, vals[p]);
            store_out(out, v, nvec_full, tail, narrow8<Ops>(acc));
        }
    }
}

template <class Ops>
const void *noalloc_ptr(int R) {
    switch (R) {
        case 1: return (const void *)allreduce_noalloc_kernel<Ops, 1>;
        case 2: return (const void *)allreduce_noalloc_kernel<Ops, 2>;
        case 3: return (const void *)allreduce_noalloc_kernel<Ops, 3>;
        case 4: return (const void *)allreduce_noalloc_kernel<Ops, 4>;
        case 5: return (const void *)allreduce_noalloc_kernel<Ops, 5>;
        case 6: return (const void *)allreduce_noalloc_kernel<Ops, 6>;
        case 7: return (const void *)allreduce_noalloc_kernel<Ops, 7>;
        case 8: return (const void *)allreduce_noalloc_kernel<Ops, 8>;
        default: return nullptr;
    }
}

// Per-device set-up, done by the first call on each device: the array's
// device address, the SM count and the kernels' occupancy.  Host threads may
// make their first calls at the same time: the set-up runs under a lock, and
// `done` is published with release order after the other fields, so a thread
// that reads it true (acquire) without the lock sees them complete.  A set-up
// that fails leaves `done` false, and the next call tries again.
constexpr int kMaxDevices = 64;
struct DeviceSetup {
    std::atomic<bool> done{false};
    uint8_t *scratch = nullptr;
    int sms = 0;
    int bps = 0;  // smallest occupancy over the 16 kernel variants
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_lock;

int device_setup(int dev, DeviceSetup **out) {
    if (dev < 0 || dev >= kMaxDevices) return AR_EINVAL;
    DeviceSetup &s = g_setup[dev];
    if (s.done.load(std::memory_order_acquire)) {
        *out = &s;
        return AR_OK;
    }
    std::lock_guard<std::mutex> guard(g_setup_lock);
    if (!s.done.load(std::memory_order_relaxed)) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            (void)cudaGetLastError();
            return AR_ECUDA;
        }
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return AR_ECUDA;
        int bps = 1 << 30;
        for (int R = 1; R <= kMaxRanks; ++R) {
            for (const void *k : {noalloc_ptr<F16Ops>(R), noalloc_ptr<BF16Ops>(R)}) {
                int n = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, 0) != cudaSuccess) return AR_ECUDA;
                if (n < bps) bps = n;
            }
        }
        if (bps < 1) return AR_ECUDA;
        s.scratch = static_cast<uint8_t *>(p);
        s.sms = sms;
        s.bps = bps;
        s.done.store(true, std::memory_order_release);
    }
    *out = &s;
    return AR_OK;
}

}  // namespace
}  // namespace tda

extern "C" AR_API int ar_allreduce_noalloc(int R, int dtype, const void *const *ins, void *const *outs,
                                           size_t numel, ar_stream_t stream) {
    using namespace tda;
    if (R < 1 || R > kMaxRanks || (dtype != AR_F16 && dtype != AR_BF16) || !ins || !outs) return AR_EINVAL;
    if (numel > kNoAllocMaxBytes / 2) return AR_ETOOBIG;
    RankPtrs ptrs;
    std::memset(&ptrs, 0, sizeof(ptrs));
    for (int r = 0; r < R; ++r) {
        if (!ins[r] || !outs[r] || ((uintptr_t)ins[r] | (uintptr_t)outs[r]) % 16) return AR_EINVAL;
        ptrs.in[r] = static_cast<const uint16_t *>(ins[r]);
        ptrs.out[r] = static_cast<uint16_t *>(outs[r]);
    }
    if (numel == 0) return AR_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    DeviceSetup *ds = nullptr;
    int rc = device_setup(dev, &ds);
    if (rc != AR_OK) return rc;

    const uint64_t nv = (numel + 7) / 8;
    const uint64_t tiles = (nv + kThreads - 1) / kThreads;
    uint64_t blocks = (uint64_t)ds->sms * ds->bps / R;
    if (blocks > (uint64_t)kNoAllocMaxBlocks) blocks = kNoAllocMaxBlocks;
    if (blocks > tiles) blocks = tiles;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Flags, abort word and error record start at zero on every call (this
    // clears the record a timed-out earlier call left).
    if (cudaMemsetAsync(ds->scratch + kNoAllocSlotBytes, 0, kNoAllocFlagBytes + kNoAllocMiscBytes, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    const void *k = dtype == AR_F16 ? noalloc_ptr<F16Ops>(R) : noalloc_ptr<BF16Ops>(R);
    uint64_t a1 = numel;
    uint8_t *a2 = ds->scratch;
    uint64_t a3 = 1000000000ull;  // 1 s: a wait can only run out if the GPU stops scheduling the grid
    void *args[] = {&ptrs, &a1, &a2, &a3};
    if (cudaLaunchCooperativeKernel(k, dim3((unsigned)blocks, (unsigned)R), dim3(kThreads), args, 0, s) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    return AR_OK;
}

// The device's set-up, then a synchronous copy between the host and the
// array's error record (no allocation: cudaMemcpy between pageable host memory
// and the array stages through the driver's own buffers).
static int noalloc_record_copy(ar_error_info *host, bool to_device) {
    using namespace tda;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    DeviceSetup *ds = nullptr;
    const int rc = device_setup(dev, &ds);
    if (rc != AR_OK) return rc;
    uint8_t *rec = ds->scratch + kNoAllocErrOffset;
    const cudaError_t e = to_device ? cudaMemcpy(rec, host, sizeof(ar_error_info), cudaMemcpyHostToDevice)
                                    : cudaMemcpy(host, rec, sizeof(ar_error_info), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    return AR_OK;
}

extern "C" AR_API int ar_noalloc_status(ar_error_info *info) {
    ar_error_info e;
    std::memset(&e, 0, sizeof(e));
    const int rc = noalloc_record_copy(&e, false);
    if (rc != AR_OK) return rc;
    if (info) *info = e;
    return e.code;
}

extern "C" AR_API int ar_noalloc_debug_record(const ar_error_info *info) {
    if (!info) return AR_EINVAL;
    ar_error_info e = *info;
    return noalloc_record_copy(&e, true);
}
