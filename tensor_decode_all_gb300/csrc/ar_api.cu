// ar_api.cu -- the C ABI declared in include/ar.h: handles, slot allocation,
// argument checks, launch planning and the enqueue calls.
//
// The enqueue calls (ar_allreduce, ar_allgather) do no host synchronisation
// and no CPU work beyond argument checks, so they may be captured in CUDA
// graphs ("[Kernel] Two-rank FP16 all-reduce through pinned host memory for
// GPUs without P2P", section "Purpose").  Every decline happens before any
// CUDA work is enqueued and returns its own code, so a caller can keep its
// fallback path ("[SM120] Add optional FlashInfer PCIe-IPC all-reduce for
// switch-free hosts", section "Modifications").
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <new>

#include "ar_internal.h"

using tda::Ctr;
using tda::DevState;

// Kernel families, for the occupancy table.
// Kernel families, each with its own blocks per SM (the smallest over its
// variants): the allgather's bulk-gather kernel holds a tile of every peer in
// shared memory and fits fewer blocks per SM than the per-thread gather.
enum { kOneShot = 0, kTwoShot = 1, kTagged = 2, kAllgather = 3, kPush = 4, kAllgatherBulk = 5, kFamilies = 6 };

struct ar_handle {
    int R = 0, dtype = 0, kind = 0, device = 0;
    uint64_t max_numel = 0, itemsize = 0, slot_bytes = 0;
    int sm_count = 0;
    // Blocks per SM of each kernel family, for [one rank's launch / all ranks
    // in one launch][untraced / traced kernels][family] (the smallest over
    // the family's variants).
    int bps[2][2][kFamilies] = {};
    int bmax = 0;                              // flag slots per rank
    int cmax = 0;                              // counter slots per rank (>= bmax)
    int algo = AR_ALGO_AUTO;
    int twoshot_sub = 0;                       // tactic: two-shot sub-tile (64/128/256); 0 = size rule
    uint64_t twoshot_min_bytes = ~0ull;        // tactic: AUTO picks two-shot from this size per rank
    int max_blocks = 0;                        // tactic: cap on blocks per rank; 0 = occupancy
    uint64_t tagged_max_bytes = 0;             // tactic: AUTO picks the tagged form up to this size
    uint64_t cluster_twoshot_min_bytes = ~0ull;  // tactic: cluster form is two-shot from this size
    uint64_t cluster_max_bytes = 0;            // tactic: AUTO runs launches of all ranks in the cluster form up to this size
    bool all_fused = true;                     // tactic: ar_allreduce_all launches all ranks at once
    int pace_mbs = 0;                          // tactic: pinned slots, pace of single-stage calls (MB/s); 0 = off
    int pace_multi_mbs = 0;                    // tactic: the same for calls of several stages per block
    uint64_t pace_min_bytes = 0;               // tactic: pace calls from this many bytes per rank
    int clock_khz = 0;                         // peak SM clock, for the pacing delay in cycles
    bool cluster_ok = false;                   // the cluster kernels can be scheduled on this GPU
    int cluster_max = 0;                       // clusters of R blocks of the cluster kernels resident at once
    cudaEvent_t ev_fork[tda::kMaxRanks] = {};  // ar_allreduce_all: stream r > 0 -> stream 0
    cudaEvent_t ev_join = nullptr;             // ar_allreduce_all: stream 0 -> streams r > 0
    void *ll_host = nullptr;                   // pinned kind: host address of the tagged buffers
    ulonglong2 *ll_dev = nullptr;              // [2][R][ll_vecs]
    uint64_t ll_vecs = 0, ll_bytes = 0;
    void *push_host = nullptr;                 // pinned kind: host address of the push areas
    uint8_t *push_dev = nullptr;               // push form: [2][R][R][slot_bytes], allocated on first use
    uint64_t push_bytes = 0;
    void *pflags_host = nullptr;               // pinned kind: host address of the push flags
    unsigned long long *pflags_dev = nullptr;  // push form: [R][R][bmax] flag lines
    uint64_t pflags_bytes = 0;
    ar_trace_record *trace = nullptr;          // caller's trace buffer (ar_set_trace), or null
    uint32_t trace_depth = 0;
    bool pdl = true;                           // launch as programmatic dependents
    void *slots_host = nullptr;            // pinned kind: host address of the slots
    uint8_t *slots_dev = nullptr;          // device address of the slots
    void *flags_host = nullptr;            // pinned kind: host address of the flags
    unsigned long long *flags_dev = nullptr;
    unsigned long long *flags_hbm = nullptr;   // pinned kind: the same flag lines in HBM (gpu_scope)
    bool gpu_scope = true;                 // tactic: pinned kind, the ranks synchronise at GPU scope
    uint64_t flags_bytes = 0;
    Ctr *ctr = nullptr;                    // [R][bmax] then the abort word
    unsigned int *abort_word = nullptr;
    uint64_t ctr_bytes = 0;
    ar_error_info *err_host = nullptr;
    ar_error_info *err_dev = nullptr;
    std::atomic<uint64_t> timeout_ns{1000000000ull};
    // Host-side record of each rank's latest call, to refuse two ranks of one
    // call sequence number on the same stream (that pairing cannot finish).
    std::atomic<uint64_t> host_calls[tda::kMaxRanks];
    std::atomic<uintptr_t> host_stream[tda::kMaxRanks];
    // Whether recent input pointers are mapped host memory (zero-copy calls
    // run unpaced): a cache, so that a caller reusing its buffers pays the
    // runtime query (a few microseconds) once per buffer.  Entries pack the address with the answer in
    // bit 0 (addresses are 16-byte aligned); 0 is empty.  An entry may outlive
    // its buffer; the answer only sets when stores start, never the bits.
    static constexpr int kIoCache = 1024;
    std::atomic<uintptr_t> io_cache[kIoCache];
};

namespace {

thread_local int g_last_error = AR_OK;


uint64_t itemsize_of(int dtype) {
    switch (dtype) {
        case AR_F16: return 2;
        case AR_BF16: return 2;
        case AR_C64: return 8;
        default: return 0;
    }
}

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

bool valid_stream_handle(cudaStream_t s) {
    return s != nullptr && s != cudaStreamLegacy && s != cudaStreamPerThread;
}

// The blocking/non-blocking rule matters for eager launches (a blocking stream
// serialises with the legacy stream).  Under stream capture the call becomes a
// graph node whose ordering comes from the graph's edges, and querying the
// flags of a capturing stream invalidates the capture (cudaStreamGetFlags
// returns success but the capture is dead), so the flags are only read
// outside capture.
int check_stream(cudaStream_t s) {
    if (!valid_stream_handle(s)) return AR_ESTREAM;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ESTREAM;
    }
    if (cs == cudaStreamCaptureStatusActive) return AR_OK;
    if (cs != cudaStreamCaptureStatusNone) return AR_ESTREAM;  // an invalidated capture
    unsigned int flags = 0;
    if (cudaStreamGetFlags(s, &flags) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ESTREAM;
    }
    if (!(flags & cudaStreamNonBlocking)) return AR_ESTREAM;
    return AR_OK;
}

int check_device(const ar_handle *h) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    return dev == h->device ? AR_OK : AR_EINVAL;
}

DevState dev_state(const ar_handle *h) {
    DevState d;
    d.slots = h->slots_dev;
    // Pinned-host slots with the gpu_scope tactic: the flags in HBM, and every
    // flag, tagged word and push flag at GPU scope (every rank is a kernel of
    // this GPU); without it, flags in host memory and system scope throughout.
    // HBM slots: flags in HBM at GPU scope.
    const bool sys = h->kind == AR_SLOT_PINNED_HOST && !h->gpu_scope;
    d.flags = h->kind == AR_SLOT_PINNED_HOST && h->gpu_scope ? h->flags_hbm : h->flags_dev;
    d.ctr = h->ctr;
    d.abort_word = h->abort_word;
    d.err = h->err_dev;
    d.slot_bytes = h->slot_bytes;
    d.timeout_ns = h->timeout_ns.load(std::memory_order_relaxed);
    d.bmax = h->bmax;
    d.cmax = h->cmax;
    d.sys_scope = sys ? 1 : 0;
    d.ll = h->ll_dev;
    d.ll_vecs = h->ll_vecs;
    d.trace = h->trace;
    d.trace_depth = h->trace_depth;
    d.algo = AR_ALGO_ONESHOT;
    d.push = h->push_dev;
    d.push_flags = h->pflags_dev;
    d.pace_cycles = 0;
    return d;
}

void free_all(ar_handle *h) {
    if (h->slots_host) cudaFreeHost(h->slots_host);
    else if (h->slots_dev) cudaFree(h->slots_dev);
    if (h->flags_host) cudaFreeHost(h->flags_host);
    else if (h->flags_dev) cudaFree(h->flags_dev);
    if (h->flags_hbm) cudaFree(h->flags_hbm);
    if (h->ll_host) cudaFreeHost(h->ll_host);
    else if (h->ll_dev) cudaFree(h->ll_dev);
    if (h->push_host) cudaFreeHost(h->push_host);
    else if (h->push_dev) cudaFree(h->push_dev);
    if (h->pflags_host) cudaFreeHost(h->pflags_host);
    else if (h->pflags_dev) cudaFree(h->pflags_dev);
    h->push_host = h->pflags_host = nullptr;
    h->push_dev = nullptr;
    h->pflags_dev = nullptr;
    if (h->ctr) cudaFree(h->ctr);
    if (h->err_host) cudaFreeHost(h->err_host);
    for (auto &e : h->ev_fork)
        if (e) cudaEventDestroy(e);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    (void)cudaGetLastError();
    for (auto &e : h->ev_fork) e = nullptr;
    h->ev_join = nullptr;
    h->slots_host = nullptr;
    h->slots_dev = nullptr;
    h->flags_host = nullptr;
    h->flags_dev = nullptr;
    h->flags_hbm = nullptr;
    h->ll_host = nullptr;
    h->ll_dev = nullptr;
    h->ctr = nullptr;
    h->abort_word = nullptr;
    h->err_host = nullptr;
    h->err_dev = nullptr;
}

// Zero flags, counters, abort word and error record.  Caller has synchronised.
int zero_state(ar_handle *h) {
    if (h->flags_host) std::memset(h->flags_host, 0, h->flags_bytes);
    else if (cudaMemset(h->flags_dev, 0, h->flags_bytes) != cudaSuccess) return AR_ECUDA;
    if (h->flags_hbm && cudaMemset(h->flags_hbm, 0, h->flags_bytes) != cudaSuccess) return AR_ECUDA;
    if (cudaMemset(h->ctr, 0, h->ctr_bytes) != cudaSuccess) return AR_ECUDA;
    // Stale tagged words would carry tags the restarted counters reuse.
    if (h->ll_host) std::memset(h->ll_host, 0, h->ll_bytes);
    else if (h->ll_dev && cudaMemset(h->ll_dev, 0, h->ll_bytes) != cudaSuccess) return AR_ECUDA;
    // push flags are stage counts too
    if (h->pflags_host) std::memset(h->pflags_host, 0, h->pflags_bytes);
    else if (h->pflags_dev && cudaMemset(h->pflags_dev, 0, h->pflags_bytes) != cudaSuccess) return AR_ECUDA;
    std::memset((void *)h->err_host, 0, sizeof(ar_error_info));
    for (int r = 0; r < tda::kMaxRanks; ++r) {
        h->host_calls[r].store(0);
        h->host_stream[r].store(0);
    }
    for (auto &e : h->io_cache) {
        e.store(0);
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return AR_ECUDA;
    return AR_OK;
}

// Occupancy of each kernel family a handle may launch (the smallest over the
// family's variants), so that R * blocks of any launched variant fit on the GPU
// at the same time: the co-residency the spin-waits need.  Also loads each
// variant into the context now (cudaFuncGetAttributes), so that no kernel is
// loaded lazily while its first launch is being captured into a graph.
int kernel_occupancy(const void *k, int *bps, size_t smem = 0) {
    if (!k) return AR_ECUDA;
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, k) != cudaSuccess) return AR_ECUDA;
    // kernels with dynamic shared memory: allow it (static plus dynamic may
    // pass the default 48 KiB)
    if (smem > 0 && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return AR_ECUDA;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, tda::kThreads, smem) != cudaSuccess) return AR_ECUDA;
    if (n < *bps) *bps = n;
    return AR_OK;
}

// Occupancy of every family for one (launch kind, traced) pair.
int family_occupancy(const ar_handle *h, bool fused, bool traced, int *bps) {
    const int kUnset = 1 << 30;
    for (int f = 0; f < kFamilies; ++f) bps[f] = kUnset;
    int rc = AR_OK;
    if (h->dtype == AR_F16 || h->dtype == AR_BF16) {
        for (int u = 1; u <= 2 && rc == AR_OK; ++u)
            for (int a = 0; a < (traced ? 1 : 2) && rc == AR_OK; ++a)
                rc = kernel_occupancy(
                    tda::allreduce_kernel_ptr(h->dtype, h->R, a ? tda::oneshot_ahead_variant(u) : u, fused, traced),
                    &bps[kOneShot]);
        for (int sub = 64; sub <= 256 && rc == AR_OK; sub *= 2)
            for (int m = 0; m < (traced ? 1 : 2) && rc == AR_OK; ++m)
                rc = kernel_occupancy(
                    tda::allreduce_kernel_ptr(h->dtype, h->R, tda::twoshot_variant(sub, m != 0), fused, traced),
                    &bps[kTwoShot]);
        if (rc == AR_OK)
            rc = kernel_occupancy(tda::allreduce_kernel_ptr(h->dtype, h->R, tda::kTaggedVariant, fused, traced),
                                  &bps[kTagged]);
        if (rc == AR_OK)
            rc = kernel_occupancy(tda::allreduce_kernel_ptr(h->dtype, h->R, tda::kPushVariant, fused, traced),
                                  &bps[kPush]);
    }
    for (int u = 1; u <= 2 && rc == AR_OK; ++u)
        for (int vw = 1; vw <= 16 && rc == AR_OK; vw *= 2)
            for (int a = 0; a < (traced || vw < 8 ? 1 : 2) && rc == AR_OK; ++a)
                rc = kernel_occupancy(
                    tda::allgather_kernel_ptr(vw, h->R, a ? tda::oneshot_ahead_variant(u) : u, fused, traced),
                    &bps[kAllgather]);
    // the bulk-gather kernel: slots in HBM, R >= 5, untraced
    if (h->kind == AR_SLOT_HBM && h->R >= 5 && !traced)
        for (int u = 1; u <= 2 && rc == AR_OK; ++u)
            rc = kernel_occupancy(tda::allgather_kernel_ptr(16, h->R, tda::allgather_bulk_variant(u), fused, false),
                                  &bps[kAllgatherBulk], tda::allgather_bulk_smem(h->R, u));
    if (rc != AR_OK) return rc;
    for (int f = 0; f < kFamilies; ++f) {
        if (bps[f] == kUnset) bps[f] = bps[kAllgather];  // complex64 handles launch no all-reduce kernel
        if (bps[f] < 1) return AR_ECUDA;
    }
    return AR_OK;
}

int handle_occupancy(ar_handle *h) {
    int rc = AR_OK;
    for (int fused = 0; fused < 2 && rc == AR_OK; ++fused)
        for (int traced = 0; traced < 2 && rc == AR_OK; ++traced)
            rc = family_occupancy(h, fused != 0, traced != 0, h->bps[fused][traced]);
    return rc;
}

// The cluster form's kernels: load every variant into the context now (no
// lazy loading during a capture), and check that a cluster of R blocks of the
// largest variant can be scheduled at all.  A GPU or build without cluster
// launches leaves the handle on the flag forms (cluster_ok false).
int cluster_setup(ar_handle *h) {
    h->cluster_ok = false;
    if (h->dtype != AR_F16 && h->dtype != AR_BF16) return AR_OK;
    for (int traced = 0; traced < 2; ++traced)
        for (int paced = 0; paced < 2; ++paced)
            for (int sub : {0, 64, 128, 256}) {
                const void *k = tda::allreduce_cluster_kernel_ptr(h->dtype, h->R, sub, traced != 0, paced != 0);
                cudaFuncAttributes attr;
                if (!k || cudaFuncGetAttributes(&attr, k) != cudaSuccess) {
                    (void)cudaGetLastError();
                    return AR_OK;
                }
            }
    int fit = 1 << 30;
    for (int paced = 0; paced < 2; ++paced)
    for (int sub : {0, 64, 128, 256}) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, (unsigned)h->R);
        cfg.blockDim = dim3(tda::kThreads);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)h->R;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tda::allreduce_cluster_kernel_ptr(h->dtype, h->R, sub, false, paced != 0),
                                           &cfg) !=
                cudaSuccess ||
            n < 1) {
            (void)cudaGetLastError();
            return AR_OK;
        }
        fit = n < fit ? n : fit;
    }
    h->cluster_ok = true;
    h->cluster_max = fit;
    return AR_OK;
}

// Measured on a GB300 (one-shot vs two-shot, bf16, 64 KiB..8 MiB per rank):
// in HBM two-shot wins from 512 KiB at R = 8 and from about 2 MiB at R = 4
// (R = 5..7 take R = 4's threshold; R <= 3 stays one-shot).  Over the host
// link, where one-shot reads R(R-1)S bytes against two-shot's (2R-1)S, with
// the ranks synchronising at GPU scope (graphs of 200 calls, one-shot /
// two-shot us/call): from 32 KiB at R = 8 (9.56 vs 11.98; 16 KiB 7.79 vs
// 8.10), from 128 KiB at R = 4 (9.58 vs 10.90; 64 KiB 6.84 vs 7.67) and from
// 512 KiB at R = 3 (18.75 vs 18.89, 1 MiB 34.9 vs 45.3; 256 KiB 10.99 vs
// 11.35).  R = 5..7 take 64 KiB, between R = 4's and R = 8's.
uint64_t twoshot_threshold(int R, int slot_kind) {
    if (slot_kind == AR_SLOT_PINNED_HOST)
        return R <= 2 ? ~0ull : R == 3 ? (512ull << 10) : R == 4 ? (128ull << 10) : R < 8 ? (64ull << 10) : (32ull << 10);
    if (R < 4) return ~0ull;
    return R >= 8 ? (512ull << 10) : (2ull << 20);
}

// Largest call the tagged-word form takes under AR_ALGO_AUTO.  Measured on a
// GB300 (bf16, graphs of 100 calls, tagged vs the flag forms): in HBM it is
// faster up to 512 KiB at R = 2 (2 KiB: 2.7 vs 3.2 us; 256 KiB: 3.5 vs
// 3.7 us), up to 256 KiB at R = 3 (3.7 vs 4.0 us) and up to 64 KiB at R = 4;
// from R = 5 on it is level at best and then slower: every thread polls
// 2(R - 1) tagged vectors where one warp polls R flags.  Over the host link its
// polls re-read words that have not landed yet.  With the flags in host memory
// at system scope it won small calls (up to 16 KiB at R = 2, 8 KiB: 3.5 vs
// 4.0 us; 8 KiB at R = 3); with the ranks synchronising at GPU scope (flags
// in HBM, the default) the one-shot form wins at every size (R = 2 2 KiB
// 3.22 vs 3.52 us, 8 KiB 3.32 vs 3.73; R = 3 2 KiB 3.51 vs 4.37), so AUTO
// never picks it for pinned-host slots.
uint64_t tagged_threshold(int R, int slot_kind) {
    if (slot_kind == AR_SLOT_PINNED_HOST) return 0;
    if (R <= 2) return 512ull << 10;
    if (R == 3) return 256ull << 10;
    return R == 4 ? (64ull << 10) : 0;
}

// Cluster form (launches of all ranks at once): two-shot from this size per
// rank.  Measured on a GB300 (bf16, graphs of 100 calls, one-shot / two-shot
// cluster form, us/call): in HBM one-shot wins at every size the form takes
// up to R = 4 (R = 4 1 MiB 6.4 / 8.5), and two-shot from 512 KiB at R = 8
// (6.8 / 7.4; 256 KiB 4.4 / 5.4); over the host link one-shot wins everywhere
// at R = 2 (256 KiB 7.0 / 9.4), two-shot from 128 KiB at R = 4 (10.3 / 12.1;
// 64 KiB 7.1 / 7.3) and from 32 KiB at R = 8 (8.3 / 12.1).  R = 3 takes
// R = 4's size, R = 5..7 R = 8's.
uint64_t cluster_twoshot_threshold(int R, int slot_kind) {
    if (R < 3) return ~0ull;
    if (slot_kind == AR_SLOT_PINNED_HOST) return R >= 5 ? (32ull << 10) : (128ull << 10);
    return R >= 5 ? (512ull << 10) : ~0ull;
}

// Largest call (bytes per rank) that AUTO runs in the cluster form when all
// ranks launch at once; larger calls take the flag forms, whose grids keep
// more blocks resident than clusters of R blocks can.  Measured on a GB300
// with the final kernels (bf16, graphs of calls of every rank; cluster form /
// flag forms in one launch, us/call): in HBM the cluster form wins up to
// 2 MiB at R = 2 (5.73 / 6.07; 4 MiB 9.54 / 8.02), up to 1 MiB at R = 4 (1 MiB
// 6.34 / 6.33, 512 KiB 3.64 / 4.45; 2 MiB 9.86 / 9.02) and at R = 8 up to the
// decode-sized 768 KiB (6.6 / 8.3; 512 KiB 6.00 / 7.58; 1 MiB 10.66 / 9.49);
// over the host link, where the flag forms' first-stage stores are paced and
// their flags are in HBM (GPU scope), up to 512 KiB at R = 2 (9.59 / 9.71;
// 1 MiB 15.98 / 15.69), 256 KiB at R = 4 (14.48 / 15.15; 512 KiB 31.14 /
// 23.79) and 64 KiB at R = 8 (10.82 / 12.06; 128 KiB 18.55 / 15.90).  R = 3
// takes R = 4's limit, R = 5..7 R = 8's.
uint64_t cluster_limit(int R, int slot_kind) {
    if (slot_kind == AR_SLOT_PINNED_HOST) return R <= 2 ? (512ull << 10) : R <= 4 ? (256ull << 10) : (64ull << 10);
    return R <= 2 ? (2ull << 20) : R <= 4 ? (1ull << 20) : (896ull << 10);
}

// Under stream capture, true if a dependency edge from stream `sr` into the
// next node of stream `s0` would add nothing: every node `sr` depends on is
// already a dependency of `s0`.  In a chain of ar_allreduce_all calls that is
// the case (after a call's join both depend on that call's kernel), and
// skipping the redundant edge leaves the next launch with the single
// programmatic edge from the previous kernel on s0.  Any query failure
// answers false (keep the edge).
bool fork_redundant(cudaStream_t s0, cudaStream_t sr) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaGraphNode_t *d = nullptr;
    const cudaGraphEdgeData *ed = nullptr;
    size_t n0 = 0, nr = 0;
    if (cudaStreamGetCaptureInfo(s0, &st, nullptr, nullptr, &d, &ed, &n0) != cudaSuccess ||
        st != cudaStreamCaptureStatusActive || n0 > 64) {
        (void)cudaGetLastError();
        return false;
    }
    cudaGraphNode_t deps0[64];
    for (size_t i = 0; i < n0; ++i) deps0[i] = d[i];
    if (cudaStreamGetCaptureInfo(sr, &st, nullptr, nullptr, &d, &ed, &nr) != cudaSuccess ||
        st != cudaStreamCaptureStatusActive) {
        (void)cudaGetLastError();
        return false;
    }
    for (size_t i = 0; i < nr; ++i) {
        bool found = false;
        for (size_t j = 0; j < n0 && !found; ++j) found = deps0[j] == d[i];
        if (!found) return false;
    }
    return true;
}

// Pace of a call's slot traffic over the host link (stores and loads
// together, MB/s), for calls of one stage per block and of several, and the
// smallest call paced.  Measured on a GB300 (bf16, per-rank launches, graphs
// of 100 calls; unpaced / 220 / 280 / 356 / 440 GB/s, us per call): R = 2
// 256 KiB 7.97 / 8.26 / 7.39 / 7.15 / 7.22, 1 MiB 23.8 / 23.4 / 20.7 / 19.3 /
// 21.1; R = 8 two-shot 1 MiB 122.5 / 114.4 / 98.4 / 96.0 / 103.1; calls of
// several stages per block: R = 2 4 MiB 77.0 / 63.5 / 69.5 / 72.5 / 74.2,
// R = 8 4 MiB 421 / 355 / 366 / 373 / 384; below 128 KiB level or slower
// (R = 8 32 KiB one-shot 12.8 unpaced, 13.4 at 356).  In the cluster form
// (one wave of clusters) R = 2 256 KiB 6.98 -> 5.84, 1 MiB 20.5 -> 15.9 at 356.
constexpr int kPaceSingleMbs = 356000;
constexpr int kPaceMultiMbs = 220000;
constexpr uint64_t kPaceMinBytes = 128ull << 10;

int choose_algo(int R, uint64_t bytes, int slot_kind) {
    const uint64_t tagged = tagged_threshold(R, slot_kind);
    if (tagged && bytes <= tagged) return AR_ALGO_TAGGED;
    return bytes >= twoshot_threshold(R, slot_kind) ? AR_ALGO_TWOSHOT : AR_ALGO_ONESHOT;
}

// The form a handle's call of `bytes` per rank takes: forced, or its tactic.
int handle_bps(const ar_handle *h, int algo, bool fused);

// The tagged form runs only calls of one stage: every block one 256-vector
// tile, so that each buffer position belongs to a single block index.
bool tagged_fits(const ar_handle *h, uint64_t bytes, bool fused) {
    if (!h->ll_dev) return false;
    const uint64_t tiles = ((bytes + 15) / 16 + tda::kThreads - 1) / tda::kThreads;
    uint64_t blocks = (uint64_t)h->sm_count * (uint64_t)handle_bps(h, AR_ALGO_TAGGED, fused) / (uint64_t)h->R;
    if (blocks > (uint64_t)h->bmax) blocks = (uint64_t)h->bmax;
    if (h->max_blocks > 0 && blocks > (uint64_t)h->max_blocks) blocks = (uint64_t)h->max_blocks;
    return tiles <= blocks;
}

// The form a call of `bytes` per rank takes: forced, or by the handle's
// tactics; the tagged form only where it fits (else one-shot).
int handle_algo(const ar_handle *h, uint64_t bytes, bool fused) {
    if (h->algo == AR_ALGO_TAGGED) return tagged_fits(h, bytes, fused) ? AR_ALGO_TAGGED : AR_ALGO_ONESHOT;
    if (h->algo == AR_ALGO_PUSH) return h->push_dev ? AR_ALGO_PUSH : AR_ALGO_ONESHOT;
    if (fused && h->cluster_ok &&
        (h->algo == AR_ALGO_CLUSTER || (h->algo == AR_ALGO_AUTO && bytes <= h->cluster_max_bytes)))
        return AR_ALGO_CLUSTER;
    if (h->algo != AR_ALGO_AUTO && h->algo != AR_ALGO_CLUSTER) return h->algo;
    if (h->tagged_max_bytes && bytes <= h->tagged_max_bytes && tagged_fits(h, bytes, fused)) return AR_ALGO_TAGGED;
    return bytes >= h->twoshot_min_bytes ? AR_ALGO_TWOSHOT : AR_ALGO_ONESHOT;
}

// Blocks per SM of the kernel family a call of `algo` launches.
int handle_bps(const ar_handle *h, int algo, bool fused) {
    const int f = algo == AR_ALGO_TWOSHOT ? kTwoShot
                  : algo == AR_ALGO_TAGGED ? kTagged
                  : algo == AR_ALGO_PUSH   ? kPush
                                           : kOneShot;
    return h->bps[fused ? 1 : 0][h->trace ? 1 : 0][f];
}

// Blocks per rank a handle launches for a plan: the plan's, within the flag
// slots and the tactic's cap.
int handle_blocks(const ar_handle *h, int plan_blocks) {
    int b = plan_blocks < h->bmax ? plan_blocks : h->bmax;
    if (h->max_blocks > 0 && b > h->max_blocks) b = h->max_blocks;
    return b;
}

// Sub-tile size (vectors) of the two-shot form.  In HBM: 256, unless
// 256-vector sub-tiles would give fewer than half the blocks the GPU can
// hold: then 128, which spreads a mid-sized call over twice the blocks
// (measured on a GB300, bf16: R=8 768 KiB 9.9 -> 9.5 us; from 2 MiB up 256
// is as fast or faster).  Over the host link: 64 while 256-vector sub-tiles
// would make fewer than 8 tiles, else 256 (GPU-scope flags, bf16, per-rank
// launches, 64 / 128 / 256 vectors, us/call: R=8 32 KiB 8.17 / 8.63 / 9.57,
// 64 KiB 11.02 / 11.56 / 11.86, 128 KiB 16.21 / 16.80 / 16.87, 256 KiB (8
// tiles) 26.59 / 26.90 / 26.56; R=4 128 KiB (8 tiles) 9.81 / 9.63 / 9.53,
// 1 MiB 48.9 / 47.3 / 43.1).
int twoshot_sub_for(int R, uint64_t nv, uint64_t bmax, int slot_kind) {
    const uint64_t tiles256 = (nv + 256ull * R - 1) / (256ull * R);
    if (slot_kind != AR_SLOT_HBM) return tiles256 < 8 ? 64 : 256;
    return 2 * tiles256 < bmax ? 128 : 256;
}

int plan_compute_sub(int R, uint64_t bytes, int vec, int algo, int sub, int threads, int sms, int bps, ar_plan *p);

// Cluster form: 0 (one-shot) below the handle's two-shot size, else the
// handle's two-shot sub-tile tactic if set, else the smallest sub-tile whose
// tiles still fit one per cluster (at most `grid` clusters), else 256.
// Measured (R = 8 bf16 768 KiB HBM, one stage per cluster): 64-vector
// sub-tiles 6.7 us (96 clusters), 128: 6.9 (48), 256: 8.0 (24).
int cluster_sub_for(int R, uint64_t bytes, uint64_t twoshot_min, uint64_t grid, int forced_sub) {
    if (bytes < twoshot_min) return 0;
    if (forced_sub) return forced_sub;
    const uint64_t nv = (bytes + 15) / 16;
    for (int sub = 64; sub <= 128; sub *= 2)
        if ((nv + (uint64_t)R * sub - 1) / ((uint64_t)R * sub) <= grid) return sub;
    return 256;
}

// The cluster form's sub-tile for a call of `bytes` per rank on this handle
// (the target is the blocks per rank the handle launches).
int handle_blocks(const ar_handle *h, int plan_blocks);
// The most clusters a call launches: the handle's per-(rank, block) counters
// and the block cap.  Clusters wait on nothing outside themselves, so a grid
// of more clusters than the GPU holds at once (ar_info.cluster_form) simply
// runs in waves -- and small single-stage clusters in waves beat fewer
// clusters that loop over several stages (R = 8 bf16 768 KiB HBM, bf16: 96
// clusters of 64-vector sub-tiles 6.7 us; 36 clusters, one wave, 128-vector
// sub-tiles over two stages: 10.4 us).
int handle_cluster_grid(const ar_handle *h) {
    // a traced call writes one record per (rank, block) into [depth][R][bmax]
    int b = h->trace ? h->bmax : h->cmax;
    if (h->max_blocks > 0 && b > h->max_blocks) b = h->max_blocks;
    return b;
}

int handle_cluster_sub(const ar_handle *h, uint64_t bytes) {
    return cluster_sub_for(h->R, bytes, h->cluster_twoshot_min_bytes, (uint64_t)handle_cluster_grid(h),
                           h->twoshot_sub);
}

// Plan of a cluster-form call: one tile of 256 vectors (one-shot) or R
// sub-tiles (two-shot) per cluster and stage; as many clusters as tiles, up to
// the handle's blocks per rank (the clusters wait on nothing outside
// themselves, so they need not all be resident at once).
void plan_cluster(int R, uint64_t bytes, int sub, int bmax, ar_plan *p) {
    // (bmax here: the most clusters a call launches -- the handle's blocks per
    // rank, within the clusters the GPU holds at once)
    std::memset(p, 0, sizeof(*p));
    const uint64_t nv = (bytes + 15) / 16;
    const uint64_t tile_vecs = sub ? (uint64_t)R * (uint64_t)sub : (uint64_t)tda::kThreads;
    const uint64_t tiles = (nv + tile_vecs - 1) / tile_vecs;
    const uint64_t blocks = tiles < (uint64_t)bmax ? tiles : (uint64_t)bmax;
    p->blocks = (int32_t)blocks;
    p->threads = tda::kThreads;
    p->vec_bytes = 16;
    p->unroll = (int32_t)((tile_vecs + tda::kThreads - 1) / tda::kThreads);
    p->algo = AR_ALGO_CLUSTER;
    p->flag_rounds = sub ? 2 : 1;
    p->subtile_vecs = sub;
    p->tile_bytes = tile_vecs * 16;
    p->tiles = tiles;
    p->max_stages = blocks ? (tiles + blocks - 1) / blocks : 0;
}

int handle_twoshot_sub(const ar_handle *h, uint64_t bytes) {
    if (h->twoshot_sub) return h->twoshot_sub;
    const uint64_t bmax = (uint64_t)h->sm_count * (uint64_t)handle_bps(h, AR_ALGO_TWOSHOT, false) / (uint64_t)h->R;
    return twoshot_sub_for(h->R, (bytes + 15) / 16, bmax, h->kind);
}

int plan_compute(int R, uint64_t bytes, int vec, int algo, int threads, int sms, int bps, ar_plan *p) {
    return plan_compute_sub(R, bytes, vec, algo, 0, threads, sms, bps, p);
}

// sub: two-shot sub-tile in vectors (64, 128, 256), or 0 for 256.
int plan_compute_sub(int R, uint64_t bytes, int vec, int algo, int sub, int threads, int sms, int bps, ar_plan *p) {
    if (!p || R < 1 || R > tda::kMaxRanks || threads < 32 || threads % 32 || sms < 1 || bps < 1)
        return AR_EINVAL;
    if (vec != 16 && vec != 8 && vec != 4 && vec != 2 && vec != 1) return AR_EINVAL;
    if (algo != AR_ALGO_ONESHOT && algo != AR_ALGO_TWOSHOT && algo != AR_ALGO_TAGGED && algo != AR_ALGO_PUSH)
        return AR_EINVAL;
    if (algo != AR_ALGO_ONESHOT && vec != 16) return AR_EINVAL;
    std::memset(p, 0, sizeof(*p));
    const uint64_t bmax = (uint64_t)sms * (uint64_t)bps / (uint64_t)R;
    if (bmax < 1) return AR_EINVAL;
    const uint64_t nv = (bytes + vec - 1) / vec;
    // One-shot: two vectors per thread per stage once every block has at least
    // two stages' worth of single vectors; one otherwise (spreads small
    // payloads over more blocks).  Two-shot: one sub-tile of `threads` vectors
    // per rank, so R vectors per thread per stage.
    if (algo == AR_ALGO_TWOSHOT && sub == 0) sub = 256;
    if (algo == AR_ALGO_TWOSHOT && sub != 64 && sub != 128 && sub != 256) return AR_EINVAL;
    const uint64_t tile_vecs = algo == AR_ALGO_TWOSHOT                            ? (uint64_t)R * (uint64_t)sub
                               : (algo == AR_ALGO_TAGGED || algo == AR_ALGO_PUSH) ? (uint64_t)threads
                                                        : (uint64_t)threads * (nv >= bmax * (uint64_t)threads * 2 ? 2 : 1);
    const int unroll = (int)((tile_vecs + threads - 1) / threads);
    const uint64_t tiles = (nv + tile_vecs - 1) / tile_vecs;
    const uint64_t blocks = tiles < bmax ? tiles : bmax;
    p->blocks = (int32_t)blocks;
    p->algo = algo;
    p->flag_rounds = algo == AR_ALGO_TWOSHOT ? 2 : 1;
    p->subtile_vecs = algo == AR_ALGO_TWOSHOT ? sub : 0;
    p->threads = threads;
    p->vec_bytes = vec;
    p->unroll = unroll;
    p->tile_bytes = tile_vecs * (uint64_t)vec;
    p->tiles = tiles;
    p->max_stages = blocks ? (tiles + blocks - 1) / blocks : 0;
    return AR_OK;
}

// Largest power-of-two vector width (<= 16) dividing the byte count and both
// addresses: the allgather writes shard p at out + p * bytes.
int allgather_vec(uint64_t bytes, const void *in, const void *out) {
    const uintptr_t a = (uintptr_t)in | (uintptr_t)out;
    int vw = 16;
    while (vw > 1 && ((bytes % vw) || (a % vw))) vw >>= 1;
    return vw;
}

int max_blocks_override() {
    const char *e = std::getenv("AR_MAX_BLOCKS");
    if (!e || !*e) return 0;
    const long v = std::strtol(e, nullptr, 10);
    return v > 0 ? (int)v : 0;
}

// True while some rank has issued more calls on the handle than another: a
// call is half issued.  The form, the tactics and the trace setting decide a
// call's kernel and grid, so they change only between calls; changed in
// between, the ranks of one call would run different forms.
bool call_half_issued(const ar_handle *h) {
    const uint64_t c = h->host_calls[0].load(std::memory_order_acquire);
    for (int r = 1; r < h->R; ++r)
        if (h->host_calls[r].load(std::memory_order_acquire) != c) return true;
    return false;
}

// Common checks and bookkeeping of one enqueue call.
int begin_call(ar_handle *h, int rank, const void *in, void *out, size_t numel, cudaStream_t s,
               uint64_t *call_index) {
    if (!h || rank < 0 || rank >= h->R) return AR_EINVAL;
    if (numel > h->max_numel) return AR_ETOOBIG;
    if (numel == 0) return AR_OK;
    if (!in || !out) return AR_EINVAL;
    int rc = check_stream(s);
    if (rc != AR_OK) return rc;
    rc = check_device(h);
    if (rc != AR_OK) return rc;
    if (*reinterpret_cast<volatile int32_t *>(&h->err_host->code) != AR_OK) return AR_ESTATE;
    const uint64_t c = h->host_calls[rank].fetch_add(1, std::memory_order_acq_rel) + 1;
    for (int p = 0; p < h->R; ++p) {
        if (p == rank) continue;
        if (h->host_calls[p].load(std::memory_order_acquire) == c &&
            h->host_stream[p].load(std::memory_order_acquire) == (uintptr_t)s) {
            h->host_calls[rank].fetch_sub(1, std::memory_order_acq_rel);
            return AR_ESTREAM;
        }
    }
    h->host_stream[rank].store((uintptr_t)s, std::memory_order_release);
    *call_index = c;
    return AR_OK;
}

// Checks and bookkeeping of a call that enqueues every rank at once: the same
// declines as a per-rank call, for every rank's pointers, plus one rule of its
// own: every rank must have issued the same number of calls on the handle (a
// per-rank sequence left half-issued would pair with the wrong call).
int begin_fused(ar_handle *h, const void *const *ins, void *const *outs, size_t numel, cudaStream_t s,
                tda::RankIO *io) {
    if (!h || !ins || !outs) return AR_EINVAL;
    if (numel > h->max_numel) return AR_ETOOBIG;
    if (numel == 0) return AR_OK;
    *io = tda::RankIO{};
    for (int r = 0; r < h->R; ++r) {
        if (!ins[r] || !outs[r] || (((uintptr_t)ins[r] | (uintptr_t)outs[r]) % 16)) return AR_EINVAL;
        io->in[r] = const_cast<void *>(ins[r]);
        io->out[r] = outs[r];
    }
    int rc = check_stream(s);
    if (rc != AR_OK) return rc;
    rc = check_device(h);
    if (rc != AR_OK) return rc;
    if (*reinterpret_cast<volatile int32_t *>(&h->err_host->code) != AR_OK) return AR_ESTATE;
    if (call_half_issued(h)) return AR_EINVAL;
    for (int r = 0; r < h->R; ++r) {
        h->host_calls[r].fetch_add(1, std::memory_order_acq_rel);
        h->host_stream[r].store((uintptr_t)s, std::memory_order_release);
    }
    return AR_OK;
}

// Closes the bookkeeping of an accepted call: a call whose launch failed
// enqueued nothing, so it is taken off the host's count for `rank` (every
// rank for rank < 0), which stays equal to the number of kernels issued.
int end_call(ar_handle *h, int rank, int rc) {
    if (rc == AR_OK) return rc;
    for (int r = 0; r < h->R; ++r)
        if (rank < 0 || r == rank) h->host_calls[r].fetch_sub(1, std::memory_order_acq_rel);
    return rc;
}

// Pacing delay between consecutive blocks' first-stage slot stores, in SM
// cycles, for a call of `bytes` per rank planned as `plan` on `blocks` blocks
// per rank.  The handle's pace (one for calls of one stage per block, one for
// calls of several) is the rate at which the call's slot traffic -- stores and
// the peers' loads together -- is to cross the host link; the paced stores,
// the first stage's R S, take their share of it, R S / (W + Rd): 1 / R for
// the one-shot form (W = R S, Rd = R (R - 1) S) and 1 / 3 for the two-shot
// form (W = (R + 1) S, Rd = (2R - 1) S; its second-round stores of reduced
// sub-tiles are not paced).  So one tile of every rank leaves every
// R * tile_bytes / (pace * share), converted at the GPU's peak SM clock.  Only
// for slots in host memory, R >= 2, calls of at least pace_min_bytes per rank
// and a pace set; capped so that no block of the largest grid waits more than
// about 2 ms.
uint32_t pace_cycles(const ar_handle *h, uint64_t bytes, const ar_plan &plan, int blocks) {
    if (h->kind != AR_SLOT_PINNED_HOST || h->R < 2 || h->clock_khz <= 0 || bytes < h->pace_min_bytes) return 0;
    const int pace = plan.tiles > (uint64_t)blocks ? h->pace_multi_mbs : h->pace_mbs;
    if (pace <= 0) return 0;
    const double R = (double)h->R;
    const double share = plan.subtile_vecs ? 1.0 / 3.0 : 1.0 / R;
    const double ns = R * (double)plan.tile_bytes * 1000.0 / ((double)pace * share);
    double cyc = ns * (double)h->clock_khz / 1e6;
    const double cap = 4e6 / (double)(h->bmax > 0 ? h->bmax : 1);
    if (cyc > cap) cyc = cap;
    return (uint32_t)(cyc + 0.5);
}

// True if an input pointer of the call (the rank's own, or all R for a launch
// of every rank) is mapped host memory.  Such zero-copy calls read their
// inputs over the host link before the slot stores, which staggers the stores
// by itself, so they are not paced: measured on a GB300 (R=2 fp16
// 256 KiB, in and out in pinned host memory, graphs of 100 calls, GB/s at
// pace 356 / 300 / 250 / 200 / 150 / none): per-rank launches 31.2 / 30.5 /
// 31.4 / 28.9 / 26.4 / 33.0, one launch of both ranks 31.0 / 30.5 / 29.9 /
// 28.7 / 26.8 / 31.4.  Pointers the runtime does not know (an error from the
// query) count as device memory.
static_assert(ar_handle::kIoCache == 1024, "host_ptr hashes to 10 bits");
bool host_ptr(ar_handle *h, const void *p) {
    const uintptr_t a = (uintptr_t)p;
    const int slot = (int)((a >> 4) * 0x9E3779B97F4A7C15ull >> 54);  // 10 bits: kIoCache slots
    const uintptr_t e = h->io_cache[slot].load(std::memory_order_relaxed);
    if ((e & ~(uintptr_t)1) == a) return (e & 1) != 0;
    cudaPointerAttributes attr;
    bool host = false;
    if (cudaPointerGetAttributes(&attr, p) == cudaSuccess) host = attr.type == cudaMemoryTypeHost;
    else (void)cudaGetLastError();
    h->io_cache[slot].store(a | (host ? 1 : 0), std::memory_order_relaxed);
    return host;
}

bool host_io(ar_handle *h, const tda::RankIO &io, int n) {
    for (int r = 0; r < n; ++r)
        if (io.in[r] && host_ptr(h, io.in[r])) return true;
    return false;
}

// The pace of a call: the handle's, unless the call is zero copy.
uint32_t call_pace(ar_handle *h, uint32_t pace, const tda::RankIO &io, int n) {
    return pace && host_io(h, io, n) ? 0u : pace;
}

// The cluster form's pacing: only when every cluster of the call is resident
// at once (a cluster of a later wave starts when an earlier one ends, already
// behind the others).
uint32_t cluster_pace_cycles(const ar_handle *h, uint64_t bytes, const ar_plan &plan) {
    return plan.blocks <= h->cluster_max ? pace_cycles(h, bytes, plan, plan.blocks) : 0;
}

// The all-reduce launch both entry points share: form, plan and grid from the
// handle, then one launch for `rank` (or, rank < 0, all ranks at once).
int enqueue_allreduce(ar_handle *h, const tda::RankIO &io, size_t numel, int rank, cudaStream_t s) {
    const uint64_t bytes = numel * h->itemsize;
    const bool fused = rank < 0;
    const int algo = handle_algo(h, bytes, fused);
    if (algo == AR_ALGO_CLUSTER) {
        ar_plan plan;
        plan_cluster(h->R, bytes, handle_cluster_sub(h, bytes), handle_cluster_grid(h), &plan);
        const int blocks = plan.blocks;  // within handle_cluster_grid: counters, trace, block cap
        DevState d = dev_state(h);
        d.algo = AR_ALGO_CLUSTER;
        d.pace_cycles = call_pace(h, cluster_pace_cycles(h, bytes, plan), io, fused ? h->R : 1);
        const cudaError_t e =
            tda::launch_allreduce_cluster(h->dtype, h->R, plan.subtile_vecs, blocks, s, io, numel, d, h->pdl);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return AR_ECUDA;
        }
        return AR_OK;
    }
    const int bps = handle_bps(h, algo, fused);
    ar_plan plan;
    int rc = plan_compute_sub(h->R, bytes, 16, algo, handle_twoshot_sub(h, bytes), tda::kThreads, h->sm_count, bps,
                              &plan);
    if (rc != AR_OK) return rc;
    const int blocks = handle_blocks(h, plan.blocks);
    // two-shot: flag rounds merged across tiles for slots in HBM and calls of
    // several tiles per block, untraced (see allreduce_twoshot_kernel)
    const bool merged = h->kind == AR_SLOT_HBM && !h->trace && plan.tiles > (uint64_t)blocks;
    // one-shot: publish one stage ahead for slots in HBM, R <= 4 and calls of
    // several tiles per block, untraced (see allreduce_oneshot).  Measured on a
    // GB300 (bf16, graphs, A/B on one box): HBM R = 4 1 MiB 7.47 -> 6.63 us,
    // R = 2 2-8 MiB 4-6 % faster, 64 MiB level; at R = 8 (forced one-shot,
    // 16 MiB) it lost 123 -> 160 us, and over the host link up to 12 % (R = 2
    // 8 MiB 124.5 -> 141.1 us): those keep the plain form.
    const bool ahead = h->kind == AR_SLOT_HBM && h->R <= 4 && !h->trace && plan.tiles > (uint64_t)blocks;
    const int variant = algo == AR_ALGO_TWOSHOT  ? tda::twoshot_variant(plan.subtile_vecs, merged)
                        : algo == AR_ALGO_TAGGED ? tda::kTaggedVariant
                        : algo == AR_ALGO_PUSH   ? tda::kPushVariant
                        : ahead                  ? tda::oneshot_ahead_variant(plan.unroll)
                                                 : plan.unroll;
    DevState d = dev_state(h);
    d.algo = algo;
    if (algo == AR_ALGO_ONESHOT || algo == AR_ALGO_TWOSHOT)
        d.pace_cycles = call_pace(h, pace_cycles(h, bytes, plan, blocks), io, fused ? h->R : 1);
    const cudaError_t e = tda::launch_allreduce(h->dtype, h->R, variant, blocks, s, io, numel, rank, d, h->pdl);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    return AR_OK;
}

// Slots in HBM, untraced: 16-byte vectors at R >= 5 take the allgather's
// bulk-gather kernel.
bool allgather_takes_bulk(const ar_handle *h, int vw) {
    return h->kind == AR_SLOT_HBM && !h->trace && vw == 16 && h->R >= 5;
}

int enqueue_allgather(ar_handle *h, const tda::RankIO &io, size_t numel, int rank, int vw, cudaStream_t s) {
    const uint64_t bytes = numel * h->itemsize;
    const bool bulk = allgather_takes_bulk(h, vw);
    ar_plan plan;
    int rc = plan_compute(h->R, bytes, vw, AR_ALGO_ONESHOT, tda::kThreads, h->sm_count,
                          h->bps[rank < 0 ? 1 : 0][h->trace ? 1 : 0][bulk ? kAllgatherBulk : kAllgather], &plan);
    if (rc != AR_OK) return rc;
    const int blocks = handle_blocks(h, plan.blocks);
    DevState d = dev_state(h);
    // the one-shot form's link bytes: share 1/R; zero-copy calls not paced
    d.pace_cycles = call_pace(h, pace_cycles(h, bytes, plan, blocks), io, rank < 0 ? h->R : 1);
    // the others publish one stage ahead in HBM for calls of several tiles per
    // block, as the one-shot all-reduce does (16- and 8-byte vectors)
    const bool ahead = h->kind == AR_SLOT_HBM && !h->trace && vw >= 8 && plan.tiles > (uint64_t)blocks;
    const int unroll = bulk    ? tda::allgather_bulk_variant(plan.unroll)
                       : ahead ? tda::oneshot_ahead_variant(plan.unroll)
                               : plan.unroll;
    const cudaError_t e = tda::launch_allgather(vw, h->R, unroll, blocks, s, io, bytes, rank, d, h->pdl);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    return AR_OK;
}

// The push form's receive areas and flags, in the slots' kind of memory:
// 2 * R * R * slot_bytes and R * R * bmax flag lines, zeroed.  Done once, when
// the form is first selected; every later call allocates nothing.  Synchronises
// the device (no call may be running on the handle).
int alloc_push(ar_handle *h) {
    if (cudaDeviceSynchronize() != cudaSuccess) return AR_ECUDA;
    const uint64_t R = (uint64_t)h->R;
    h->push_bytes = 2ull * R * R * h->slot_bytes;
    h->pflags_bytes = R * R * (uint64_t)h->bmax * tda::kFlagStrideWords * 8ull;
    auto undo = [&](int code) {
        if (h->push_host) cudaFreeHost(h->push_host);
        else if (h->push_dev) cudaFree(h->push_dev);
        if (h->pflags_host) cudaFreeHost(h->pflags_host);
        else if (h->pflags_dev) cudaFree(h->pflags_dev);
        (void)cudaGetLastError();
        h->push_host = h->pflags_host = nullptr;
        h->push_dev = nullptr;
        h->pflags_dev = nullptr;
        return code;
    };
    if (h->kind == AR_SLOT_PINNED_HOST) {
        const unsigned fl = cudaHostAllocMapped | cudaHostAllocPortable;
        if (cudaHostAlloc(&h->push_host, h->push_bytes, fl) != cudaSuccess) return undo(AR_ENOMEM);
        if (cudaHostGetDevicePointer((void **)&h->push_dev, h->push_host, 0) != cudaSuccess) return undo(AR_ECUDA);
        if (cudaHostAlloc(&h->pflags_host, h->pflags_bytes, fl) != cudaSuccess) return undo(AR_ENOMEM);
        if (cudaHostGetDevicePointer((void **)&h->pflags_dev, h->pflags_host, 0) != cudaSuccess)
            return undo(AR_ECUDA);
        std::memset(h->push_host, 0, h->push_bytes);
        std::memset(h->pflags_host, 0, h->pflags_bytes);
    } else {
        if (cudaMalloc((void **)&h->push_dev, h->push_bytes) != cudaSuccess) return undo(AR_ENOMEM);
        if (cudaMalloc((void **)&h->pflags_dev, h->pflags_bytes) != cudaSuccess) return undo(AR_ENOMEM);
        if (cudaMemset(h->push_dev, 0, h->push_bytes) != cudaSuccess ||
            cudaMemset(h->pflags_dev, 0, h->pflags_bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            return undo(AR_ECUDA);
    }
    return AR_OK;
}

}  // namespace

extern "C" {

AR_API int ar_last_error(void) { return g_last_error; }

AR_API const char *ar_strerror(int code) {
    switch (code) {
        case AR_OK: return "AR_OK: success";
        case AR_EINVAL: return "AR_EINVAL: invalid argument";
        case AR_ETOOBIG: return "AR_ETOOBIG: numel exceeds the handle's max_numel";
        case AR_ESTREAM: return "AR_ESTREAM: stream is NULL, legacy, per-thread default, blocking, or another rank's";
        case AR_ENOMEM: return "AR_ENOMEM: allocation failed";
        case AR_ECUDA: return "AR_ECUDA: a CUDA runtime call failed";
        case AR_ETIMEOUT: return "AR_ETIMEOUT: a block timed out waiting for a peer's flag";
        case AR_ESTATE: return "AR_ESTATE: a device error is recorded; call ar_reset";
        default: return "unknown ar error code";
    }
}

AR_API ar_handle *ar_create(int R, int dtype, size_t max_numel, int slot_kind) {
    g_last_error = AR_OK;
    const uint64_t isz = itemsize_of(dtype);
    if (R < 1 || R > tda::kMaxRanks || isz == 0 || max_numel < 1 ||
        (slot_kind != AR_SLOT_PINNED_HOST && slot_kind != AR_SLOT_HBM) ||
        max_numel > (uint64_t)1 << 40) {
        g_last_error = AR_EINVAL;
        return nullptr;
    }
    ar_handle *h = new (std::nothrow) ar_handle();
    if (!h) {
        g_last_error = AR_ENOMEM;
        return nullptr;
    }
    auto fail = [&](int code) -> ar_handle * {
        free_all(h);
        delete h;
        g_last_error = code;
        return nullptr;
    };
    h->R = R;
    h->dtype = dtype;
    h->kind = slot_kind;
    h->max_numel = max_numel;
    h->itemsize = isz;
    h->slot_bytes = round_up(max_numel * isz, tda::kSlotAlign);
    if (const char *e = std::getenv("AR_SPIN_TIMEOUT_NS")) {
        const unsigned long long v = std::strtoull(e, nullptr, 10);
        if (v >= 1000ull) h->timeout_ns.store(v);
    }
    if (cudaGetDevice(&h->device) != cudaSuccess) return fail(AR_ECUDA);
    if (cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess)
        return fail(AR_ECUDA);
    if (cudaDeviceGetAttribute(&h->clock_khz, cudaDevAttrClockRate, h->device) != cudaSuccess) return fail(AR_ECUDA);
    if (const char *e = std::getenv("AR_PDL")) h->pdl = e[0] != '0';
    if (const char *e = std::getenv("AR_TWOSHOT_SUB")) {
        const long v = std::strtol(e, nullptr, 10);
        if (v == 64 || v == 128 || v == 256) h->twoshot_sub = (int)v;
    }
    h->twoshot_min_bytes = twoshot_threshold(R, slot_kind);
    h->tagged_max_bytes = (dtype == AR_F16 || dtype == AR_BF16) ? tagged_threshold(R, slot_kind) : 0;
    h->cluster_twoshot_min_bytes = cluster_twoshot_threshold(R, slot_kind);
    h->pace_mbs = slot_kind == AR_SLOT_PINNED_HOST ? kPaceSingleMbs : 0;
    h->pace_multi_mbs = slot_kind == AR_SLOT_PINNED_HOST ? kPaceMultiMbs : 0;
    h->pace_min_bytes = kPaceMinBytes;
    if (const char *e = std::getenv("AR_ALGO")) {
        if (!std::strcmp(e, "oneshot")) h->algo = AR_ALGO_ONESHOT;
        else if (!std::strcmp(e, "twoshot")) h->algo = AR_ALGO_TWOSHOT;
        else if (!std::strcmp(e, "tagged")) h->algo = AR_ALGO_TAGGED;
        else if (!std::strcmp(e, "cluster")) h->algo = AR_ALGO_CLUSTER;
        // ("push" needs its receive areas: ar_set_algo allocates them)
    }
    int rc = handle_occupancy(h);
    if (rc != AR_OK) return fail(rc);
    rc = cluster_setup(h);
    if (rc != AR_OK) return fail(rc);
    h->cluster_max_bytes = h->cluster_ok ? cluster_limit(R, slot_kind) : 0;
    h->all_fused = h->cluster_ok;
    for (int r = 0; r < R; ++r)
        if (cudaEventCreateWithFlags(&h->ev_fork[r], cudaEventDisableTiming) != cudaSuccess) return fail(AR_ECUDA);
    if (cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) return fail(AR_ECUDA);
    // The two-shot kernel fits 6 blocks per SM up to R = 4, which helps in HBM
    // (R=4 bf16 32 MiB: 84 vs 101 us at 4 blocks).
    // Over the host link fewer resident blocks keep the link just as busy with
    // less contention: pinned handles cap the two-shot form at 4 blocks per SM
    // (R=4 bf16 8 MiB: 362 us at 4, 382 at 6) and the allgather at 3 (R=4
    // complex64 4 MB: 267 us at 3, 277 at 5).
    int bps_max = 1;
    for (auto &by_trace : h->bps)
        for (auto &fam : by_trace) {
            if (h->kind == AR_SLOT_PINNED_HOST && fam[kTwoShot] > 4) fam[kTwoShot] = 4;
            if (h->kind == AR_SLOT_PINNED_HOST && fam[kAllgather] > 3) fam[kAllgather] = 3;
            for (int f = 0; f < kFamilies; ++f) bps_max = fam[f] > bps_max ? fam[f] : bps_max;
        }
    h->bmax = h->sm_count * bps_max / R;
    if (const int cap = max_blocks_override()) h->bmax = cap < h->bmax ? cap : h->bmax;
    if (h->bmax < 1) return fail(AR_ECUDA);

    const uint64_t slots_total = 2ull * (uint64_t)R * h->slot_bytes;
    h->flags_bytes = (uint64_t)R * (uint64_t)h->bmax * tda::kFlagStrideWords * 8ull;
    h->cmax = h->bmax > tda::kCounterSlots ? h->bmax : tda::kCounterSlots;
    h->ctr_bytes = round_up((uint64_t)R * (uint64_t)h->cmax * sizeof(Ctr), 256) + 256;

    if (slot_kind == AR_SLOT_PINNED_HOST) {
        const unsigned fl = cudaHostAllocMapped | cudaHostAllocPortable;
        if (cudaHostAlloc(&h->slots_host, slots_total, fl) != cudaSuccess) return fail(AR_ENOMEM);
        if (cudaHostGetDevicePointer((void **)&h->slots_dev, h->slots_host, 0) != cudaSuccess)
            return fail(AR_ECUDA);
        if (cudaHostAlloc(&h->flags_host, h->flags_bytes, fl) != cudaSuccess) return fail(AR_ENOMEM);
        if (cudaHostGetDevicePointer((void **)&h->flags_dev, h->flags_host, 0) != cudaSuccess)
            return fail(AR_ECUDA);
        if (cudaMalloc((void **)&h->flags_hbm, h->flags_bytes) != cudaSuccess) return fail(AR_ENOMEM);
        std::memset(h->slots_host, 0, slots_total);
    } else {
        if (cudaMalloc((void **)&h->slots_dev, slots_total) != cudaSuccess) return fail(AR_ENOMEM);
        if (cudaMalloc((void **)&h->flags_dev, h->flags_bytes) != cudaSuccess) return fail(AR_ENOMEM);
        if (cudaMemset(h->slots_dev, 0, slots_total) != cudaSuccess) return fail(AR_ECUDA);
    }
    // Tagged-word buffers (fp16/bf16 handles): one 256-vector tile per block,
    // at 32 bytes per 16 payload bytes, per rank and parity.
    if (dtype == AR_F16 || dtype == AR_BF16) {
        h->ll_vecs = (uint64_t)h->bmax * tda::kThreads * 2;
        h->ll_bytes = 2ull * (uint64_t)R * h->ll_vecs * 16ull;
        if (slot_kind == AR_SLOT_PINNED_HOST) {
            if (cudaHostAlloc(&h->ll_host, h->ll_bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess)
                return fail(AR_ENOMEM);
            if (cudaHostGetDevicePointer((void **)&h->ll_dev, h->ll_host, 0) != cudaSuccess) return fail(AR_ECUDA);
        } else if (cudaMalloc((void **)&h->ll_dev, h->ll_bytes) != cudaSuccess) {
            return fail(AR_ENOMEM);
        }
    }
    if (cudaMalloc((void **)&h->ctr, h->ctr_bytes) != cudaSuccess) return fail(AR_ENOMEM);
    h->abort_word = reinterpret_cast<unsigned int *>(reinterpret_cast<uint8_t *>(h->ctr) + h->ctr_bytes - 256);
    if (cudaHostAlloc((void **)&h->err_host, sizeof(ar_error_info),
                      cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess)
        return fail(AR_ENOMEM);
    if (cudaHostGetDevicePointer((void **)&h->err_dev, h->err_host, 0) != cudaSuccess)
        return fail(AR_ECUDA);
    rc = zero_state(h);
    if (rc != AR_OK) return fail(rc);
    return h;
}

AR_API int ar_allreduce(ar_handle *h, int rank, const void *in, void *out, size_t numel,
                        ar_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (h && h->dtype != AR_F16 && h->dtype != AR_BF16) return AR_EINVAL;
    if (((uintptr_t)in | (uintptr_t)out) % 16) return AR_EINVAL;
    uint64_t call = 0;
    int rc = begin_call(h, rank, in, out, numel, s, &call);
    if (rc != AR_OK || numel == 0) return rc;
    tda::RankIO io = {};
    io.in[0] = const_cast<void *>(in);
    io.out[0] = out;
    return end_call(h, rank, enqueue_allreduce(h, io, numel, rank, s));
}

AR_API int ar_allgather(ar_handle *h, int rank, const void *in, void *out, size_t numel,
                        ar_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (((uintptr_t)in | (uintptr_t)out) % 16) return AR_EINVAL;
    uint64_t call = 0;
    int rc = begin_call(h, rank, in, out, numel, s, &call);
    if (rc != AR_OK || numel == 0) return rc;
    tda::RankIO io = {};
    io.in[0] = const_cast<void *>(in);
    io.out[0] = out;
    return end_call(h, rank, enqueue_allgather(h, io, numel, rank, allgather_vec(numel * h->itemsize, in, out), s));
}

AR_API int ar_allreduce_fused(ar_handle *h, const void *const *ins, void *const *outs, size_t numel,
                              ar_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (h && h->dtype != AR_F16 && h->dtype != AR_BF16) return AR_EINVAL;
    tda::RankIO io;
    int rc = begin_fused(h, ins, outs, numel, s, &io);
    if (rc != AR_OK || numel == 0) return rc;
    return end_call(h, -1, enqueue_allreduce(h, io, numel, -1, s));
}

AR_API int ar_allgather_fused(ar_handle *h, const void *const *ins, void *const *outs, size_t numel,
                              ar_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    tda::RankIO io;
    int rc = begin_fused(h, ins, outs, numel, s, &io);
    if (rc != AR_OK || numel == 0) return rc;
    const uint64_t bytes = numel * h->itemsize;
    int vw = 16;
    for (int r = 0; r < h->R; ++r) {
        const int v = allgather_vec(bytes, ins[r], outs[r]);
        if (v < vw) vw = v;
    }
    return end_call(h, -1, enqueue_allgather(h, io, numel, -1, vw, s));
}

AR_API int ar_allreduce_all(ar_handle *h, const void *const *ins, void *const *outs, size_t numel,
                            const ar_stream_t *streams) {
    if (!h || !ins || !outs || !streams) return AR_EINVAL;
    if (h->dtype != AR_F16 && h->dtype != AR_BF16) return AR_EINVAL;
    if (numel > h->max_numel) return AR_ETOOBIG;
    if (numel == 0) return AR_OK;
    const int R = h->R;
    cudaStream_t st[tda::kMaxRanks];
    int capturing = -1;
    for (int r = 0; r < R; ++r) {
        if (!ins[r] || !outs[r] || (((uintptr_t)ins[r] | (uintptr_t)outs[r]) % 16)) return AR_EINVAL;
        st[r] = reinterpret_cast<cudaStream_t>(streams[r]);
        const int rc = check_stream(st[r]);
        if (rc != AR_OK) return rc;
        for (int q = 0; q < r; ++q)
            if (st[q] == st[r]) return AR_ESTREAM;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st[r], &cs) != cudaSuccess) {
            (void)cudaGetLastError();
            return AR_ESTREAM;
        }
        const int c = cs == cudaStreamCaptureStatusActive ? 1 : 0;
        if (capturing >= 0 && c != capturing) return AR_ESTREAM;
        capturing = c;
    }
    int rc = check_device(h);
    if (rc != AR_OK) return rc;
    if (*reinterpret_cast<volatile int32_t *>(&h->err_host->code) != AR_OK) return AR_ESTATE;
    if (call_half_issued(h)) return AR_EINVAL;
    if (!h->all_fused) {
        // R per-rank launches, every argument checked above, so no rank is
        // declined after another has been enqueued.
        for (int r = 0; r < R; ++r) {
            rc = ar_allreduce(h, r, ins[r], outs[r], numel, streams[r]);
            if (rc != AR_OK) return rc;
        }
        return AR_OK;
    }
    tda::RankIO io;
    rc = begin_fused(h, ins, outs, numel, st[0], &io);
    if (rc != AR_OK) return rc;
    for (int r = 1; r < R; ++r) {
        if (capturing == 1 && fork_redundant(st[0], st[r])) continue;
        if (cudaEventRecord(h->ev_fork[r], st[r]) != cudaSuccess || cudaStreamWaitEvent(st[0], h->ev_fork[r], 0) != cudaSuccess) {
            (void)cudaGetLastError();
            return end_call(h, -1, AR_ECUDA);
        }
    }
    rc = end_call(h, -1, enqueue_allreduce(h, io, numel, -1, st[0]));
    if (rc != AR_OK) return rc;
    if (capturing == 1 && R > 1) {
        // Join under capture: every other stream now depends on exactly the
        // launched kernel.  (An event wait would add the kernel to what the
        // stream already depended on, and a chain of calls would collect an
        // edge from every earlier call into every later one.)  Nothing is
        // lost: whatever the stream depended on before was already a
        // dependency of the kernel, through the fork or through streams[0].
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        const cudaGraphNode_t *d = nullptr;
        const cudaGraphEdgeData *ed = nullptr;
        size_t nd = 0;
        if (cudaStreamGetCaptureInfo(st[0], &cs, nullptr, nullptr, &d, &ed, &nd) != cudaSuccess ||
            cs != cudaStreamCaptureStatusActive || nd != 1) {
            (void)cudaGetLastError();
            return AR_ECUDA;
        }
        cudaGraphNode_t kernel = d[0];
        for (int r = 1; r < R; ++r) {
            if (cudaStreamUpdateCaptureDependencies(st[r], &kernel, nullptr, 1, cudaStreamSetCaptureDependencies) !=
                cudaSuccess) {
                (void)cudaGetLastError();
                return AR_ECUDA;
            }
        }
        return AR_OK;
    }
    if (R > 1 && cudaEventRecord(h->ev_join, st[0]) != cudaSuccess) {
        (void)cudaGetLastError();
        return AR_ECUDA;
    }
    for (int r = 1; r < R; ++r) {
        if (cudaStreamWaitEvent(st[r], h->ev_join, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            return AR_ECUDA;
        }
    }
    return AR_OK;
}

AR_API int ar_status(ar_handle *h, ar_error_info *info) {
    if (!h) return AR_EINVAL;
    const volatile ar_error_info *v = h->err_host;
    ar_error_info e;
    e.code = v->code;
    e.rank = v->rank;
    e.block = v->block;
    e.peer = v->peer;
    e.want = v->want;
    e.seen = v->seen;
    if (info) *info = e;
    return e.code;
}

AR_API int ar_reset(ar_handle *h) {
    if (!h) return AR_EINVAL;
    if (check_device(h) != AR_OK) return AR_EINVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) return AR_ECUDA;
    return zero_state(h);
}

AR_API int ar_destroy(ar_handle *h) {
    if (!h) return AR_OK;
    int dev = -1;
    cudaGetDevice(&dev);
    if (dev != h->device) cudaSetDevice(h->device);
    const cudaError_t e = cudaDeviceSynchronize();
    free_all(h);
    if (dev >= 0 && dev != h->device) cudaSetDevice(dev);
    delete h;
    return e == cudaSuccess ? AR_OK : AR_ECUDA;
}

AR_API int ar_set_timeout(ar_handle *h, uint64_t timeout_ns) {
    if (!h || timeout_ns < 1000ull) return AR_EINVAL;
    h->timeout_ns.store(timeout_ns);
    return AR_OK;
}

AR_API int ar_query(const ar_handle *h, ar_info *info) {
    if (!h || !info) return AR_EINVAL;
    info->R = h->R;
    info->dtype = h->dtype;
    info->slot_kind = h->kind;
    info->device = h->device;
    info->threads = tda::kThreads;
    info->max_blocks = h->bmax;
    info->sm_count = h->sm_count;
    info->blocks_per_sm = h->bps[0][0][kOneShot];
    info->blocks_per_sm_twoshot = h->bps[0][0][kTwoShot];
    info->blocks_per_sm_allgather = h->bps[0][0][kAllgather];
    info->algo = h->algo;
    info->pdl = h->pdl ? 1 : 0;
    info->max_numel = h->max_numel;
    info->slot_bytes = h->slot_bytes;
    info->total_slot_bytes = 2ull * (uint64_t)h->R * h->slot_bytes;
    info->timeout_ns = h->timeout_ns.load();
    uint64_t tag_blocks = (uint64_t)h->sm_count * (uint64_t)handle_bps(h, AR_ALGO_TAGGED, false) / (uint64_t)h->R;
    if (tag_blocks > (uint64_t)h->bmax) tag_blocks = (uint64_t)h->bmax;
    if (h->max_blocks > 0 && tag_blocks > (uint64_t)h->max_blocks) tag_blocks = (uint64_t)h->max_blocks;
    const uint64_t tag_bytes = tag_blocks * tda::kThreads * 16ull;
    info->tagged_capacity_bytes = !h->ll_dev ? 0 : (tag_bytes < h->slot_bytes ? tag_bytes : h->slot_bytes);
    info->blocks_per_sm_tagged = h->bps[0][0][kTagged];
    info->cluster_form = h->cluster_ok ? h->cluster_max : 0;
    return AR_OK;
}

AR_API int ar_plan_compute(int R, uint64_t bytes, int vec_bytes, int algo, int threads, int sm_count,
                           int blocks_per_sm, ar_plan *plan) {
    return plan_compute(R, bytes, vec_bytes, algo, threads, sm_count, blocks_per_sm, plan);
}

AR_API int ar_choose_algo(int R, uint64_t bytes, int slot_kind) { return choose_algo(R, bytes, slot_kind); }

AR_API int ar_set_pdl(ar_handle *h, int enable) {
    if (!h) return AR_EINVAL;
    h->pdl = enable != 0;
    return AR_OK;
}

AR_API int ar_set_algo(ar_handle *h, int algo) {
    if (!h || (algo != AR_ALGO_AUTO && algo != AR_ALGO_ONESHOT && algo != AR_ALGO_TWOSHOT &&
               algo != AR_ALGO_TAGGED && algo != AR_ALGO_CLUSTER && algo != AR_ALGO_PUSH))
        return AR_EINVAL;
    if ((algo == AR_ALGO_TWOSHOT || algo == AR_ALGO_TAGGED || algo == AR_ALGO_CLUSTER || algo == AR_ALGO_PUSH) &&
        h->dtype == AR_C64)
        return AR_EINVAL;
    if (call_half_issued(h)) return AR_EINVAL;
    if (algo == AR_ALGO_PUSH && !h->push_dev) {
        const int rc = alloc_push(h);
        if (rc != AR_OK) return rc;
    }
    h->algo = algo;
    return AR_OK;
}

AR_API int ar_set_trace(ar_handle *h, void *records, uint64_t capacity) {
    if (!h || call_half_issued(h)) return AR_EINVAL;
    if (!records) {
        h->trace = nullptr;
        h->trace_depth = 0;
        return AR_OK;
    }
    const uint64_t per_call = (uint64_t)h->R * (uint64_t)h->bmax;
    if (capacity < per_call || ((uintptr_t)records % 16)) return AR_EINVAL;
    const uint64_t depth = capacity / per_call;
    h->trace = static_cast<ar_trace_record *>(records);
    h->trace_depth = (uint32_t)(depth > 0xffffffffull ? 0xffffffffull : depth);
    return AR_OK;
}

AR_API int ar_debug_seed_stages(ar_handle *h, uint64_t stages) {
    if (!h) return AR_EINVAL;
    if (check_device(h) != AR_OK) return AR_EINVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) return AR_ECUDA;
    const size_t n = (size_t)h->R * (size_t)h->cmax;
    Ctr *host = new (std::nothrow) Ctr[n];
    if (!host) return AR_ENOMEM;
    int rc = AR_OK;
    if (cudaMemcpy(host, h->ctr, n * sizeof(Ctr), cudaMemcpyDeviceToHost) != cudaSuccess) rc = AR_ECUDA;
    if (rc == AR_OK) {
        for (size_t i = 0; i < n; ++i) host[i].seq = stages;
        if (cudaMemcpy(h->ctr, host, n * sizeof(Ctr), cudaMemcpyHostToDevice) != cudaSuccess) rc = AR_ECUDA;
    }
    delete[] host;
    if (rc != AR_OK) (void)cudaGetLastError();
    return rc;
}

AR_API int ar_get_tactics(const ar_handle *h, ar_tactics *t) {
    if (!h || !t) return AR_EINVAL;
    t->twoshot_min_bytes = h->twoshot_min_bytes;
    t->twoshot_sub = h->twoshot_sub;
    t->max_blocks = h->max_blocks;
    t->tagged_max_bytes = h->tagged_max_bytes;
    t->cluster_twoshot_min_bytes = h->cluster_twoshot_min_bytes;
    t->cluster_max_bytes = h->cluster_max_bytes;
    t->all_fused = h->all_fused ? 1 : 0;
    t->pace_mbs = h->pace_mbs;
    t->pace_min_bytes = h->pace_min_bytes;
    t->pace_multi_mbs = h->pace_multi_mbs;
    t->gpu_scope = h->kind != AR_SLOT_PINNED_HOST || h->gpu_scope ? 1 : 0;
    return AR_OK;
}

AR_API int ar_set_tactics(ar_handle *h, const ar_tactics *t) {
    if (!h || !t) return AR_EINVAL;
    if (t->twoshot_sub != 0 && t->twoshot_sub != 64 && t->twoshot_sub != 128 && t->twoshot_sub != 256)
        return AR_EINVAL;
    if (t->max_blocks < 0 || call_half_issued(h)) return AR_EINVAL;
    if (t->all_fused != 0 && t->all_fused != 1) return AR_EINVAL;
    if ((t->pace_mbs != 0 && t->pace_mbs < 1000) || (t->pace_multi_mbs != 0 && t->pace_multi_mbs < 1000))
        return AR_EINVAL;
    if (t->gpu_scope != 0 && t->gpu_scope != 1) return AR_EINVAL;
    if (h->kind != AR_SLOT_PINNED_HOST && t->gpu_scope != 1) return AR_EINVAL;
    h->twoshot_min_bytes = t->twoshot_min_bytes;
    h->twoshot_sub = t->twoshot_sub;
    h->max_blocks = t->max_blocks;
    h->tagged_max_bytes = t->tagged_max_bytes;
    h->cluster_twoshot_min_bytes = t->cluster_twoshot_min_bytes;
    h->cluster_max_bytes = t->cluster_max_bytes;
    h->all_fused = t->all_fused == 1;
    h->pace_mbs = t->pace_mbs;
    h->pace_min_bytes = t->pace_min_bytes;
    h->pace_multi_mbs = t->pace_multi_mbs;
    h->gpu_scope = t->gpu_scope == 1;
    return AR_OK;
}

AR_API int ar_supports(const ar_handle *h, int op, size_t numel, const void *in, const void *out) {
    if (!h || (op != 0 && op != 1)) return AR_EINVAL;
    if (op == 0 && h->dtype != AR_F16 && h->dtype != AR_BF16) return AR_EINVAL;
    if (((uintptr_t)in | (uintptr_t)out) % 16) return AR_EINVAL;
    if (numel > h->max_numel) return AR_ETOOBIG;
    if (numel > 0 && (!in || !out)) return AR_EINVAL;
    return AR_OK;
}

AR_API int ar_plan_for(const ar_handle *h, int op, size_t numel, ar_plan *plan) {
    if (!h || !plan || op < 0 || op > 2) return AR_EINVAL;
    if (numel > h->max_numel) return AR_ETOOBIG;
    const uint64_t bytes = numel * h->itemsize;
    if (op == 2) {
        // all ranks in one launch (ar_allreduce_fused; ar_allreduce_all when it fuses)
        if (h->dtype != AR_F16 && h->dtype != AR_BF16) return AR_EINVAL;
        const int algo = handle_algo(h, bytes, true);
        if (algo == AR_ALGO_CLUSTER) {
            plan_cluster(h->R, bytes, handle_cluster_sub(h, bytes), handle_cluster_grid(h), plan);
            plan->pace_cycles = (int32_t)cluster_pace_cycles(h, bytes, *plan);
            return AR_OK;
        }
        const int rc = plan_compute_sub(h->R, bytes, 16, algo, handle_twoshot_sub(h, bytes), tda::kThreads,
                                        h->sm_count, handle_bps(h, algo, true), plan);
        if (rc != AR_OK) return rc;
        if (plan->blocks > 0) {
            plan->blocks = handle_blocks(h, plan->blocks);
            plan->max_stages = (plan->tiles + plan->blocks - 1) / plan->blocks;
            if (algo == AR_ALGO_ONESHOT || algo == AR_ALGO_TWOSHOT)
                plan->pace_cycles = (int32_t)pace_cycles(h, bytes, *plan, plan->blocks);
        }
        return AR_OK;
    }
    const int vec = op == 0 ? 16 : allgather_vec(bytes, nullptr, nullptr);
    int algo = AR_ALGO_ONESHOT,
        bps = h->bps[0][h->trace ? 1 : 0][allgather_takes_bulk(h, vec) ? kAllgatherBulk : kAllgather];
    if (op == 0) {
        algo = handle_algo(h, bytes, false);
        bps = handle_bps(h, algo, false);
    }
    int rc = plan_compute_sub(h->R, bytes, vec, algo, op == 0 ? handle_twoshot_sub(h, bytes) : 0, tda::kThreads,
                              h->sm_count, bps, plan);
    if (rc == AR_OK && plan->blocks > 0) {
        plan->blocks = handle_blocks(h, plan->blocks);
        plan->max_stages = (plan->tiles + plan->blocks - 1) / plan->blocks;
        if (op == 1 || algo == AR_ALGO_ONESHOT || algo == AR_ALGO_TWOSHOT)
            plan->pace_cycles = (int32_t)pace_cycles(h, bytes, *plan, plan->blocks);
    }
    return rc;
}

}  // extern "C"

namespace tda {

const void *allreduce_kernel_ptr(int dtype, int R, int unroll, bool fused, bool traced) {
    if (unroll < 0) {
        if (dtype == AR_F16) return allreduce_twoshot_kernel_ptr_f16(R, unroll, fused, traced);
        if (dtype == AR_BF16) return allreduce_twoshot_kernel_ptr_bf16(R, unroll, fused, traced);
        return nullptr;
    }
    if (dtype == AR_F16) return allreduce_kernel_ptr_f16(R, unroll, fused, traced);
    if (dtype == AR_BF16) return allreduce_kernel_ptr_bf16(R, unroll, fused, traced);
    return nullptr;
}

cudaError_t launch_allreduce(int dtype, int R, int unroll, int blocks, cudaStream_t s,
                             const RankIO &io, uint64_t numel, int rank, const DevState &d, bool pdl) {
    const void *k = allreduce_kernel_ptr(dtype, R, unroll, rank < 0, d.trace != nullptr);
    if (!k) return cudaErrorInvalidValue;
    const uint16_t *a0 = static_cast<const uint16_t *>(io.in[0]);
    uint16_t *a1 = static_cast<uint16_t *>(io.out[0]);
    uint64_t a2 = numel;
    int a3 = rank;
    DevState a4 = d;
    RankIO a5 = io;
    void *args[] = {&a0, &a1, &a2, &a3, &a4, &a5};
    return launch(k, blocks, rank < 0 ? R : 1, rank < 0, s, args, pdl);
}

const void *allreduce_cluster_kernel_ptr(int dtype, int R, int sub, bool traced, bool paced) {
    if (dtype == AR_F16) return allreduce_cluster_kernel_ptr_f16(R, sub, traced, paced);
    if (dtype == AR_BF16) return allreduce_cluster_kernel_ptr_bf16(R, sub, traced, paced);
    return nullptr;
}

cudaError_t launch_allreduce_cluster(int dtype, int R, int sub, int blocks, cudaStream_t s, const RankIO &io,
                                     uint64_t numel, const DevState &d, bool pdl) {
    // The kernel with the pacing code for paced calls, and also for two-shot
    // calls: compiled with the clock read at its start it measured faster in
    // that variant (R = 8 bf16 768 KiB HBM, 64-vector sub-tiles: 6.60 against
    // 7.88 us; 512 KiB 6.03 against 6.75 us), a code-generation effect, while
    // unpaced one-shot calls are faster without it (R = 8 2 KiB: 2.87 against
    // 3.2 us; over the host link 4.2 against 5.3 us).
    const void *k = allreduce_cluster_kernel_ptr(dtype, R, sub, d.trace != nullptr, d.pace_cycles != 0 || sub != 0);
    if (!k || blocks < 1) return cudaErrorInvalidValue;
    const uint16_t *a0 = static_cast<const uint16_t *>(io.in[0]);
    uint16_t *a1 = static_cast<uint16_t *>(io.out[0]);
    uint64_t a2 = numel;
    int a3 = -1;
    DevState a4 = d;
    RankIO a5 = io;
    void *args[] = {&a0, &a1, &a2, &a3, &a4, &a5};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, (unsigned)R);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = (unsigned)R;
    attr[n].val.clusterDim.z = 1;
    ++n;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelExC(&cfg, k, args);
}

cudaError_t launch(const void *k, int blocks, int ranks, bool cooperative, cudaStream_t s, void **args,
                   bool pdl, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, (unsigned)ranks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace tda
