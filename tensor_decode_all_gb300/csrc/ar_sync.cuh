// ar_sync.cuh -- the per-block flag protocol of the exchange kernels.
//
// Publish: after every thread of the block has stored its part of the stage
// into the rank's slot, the block passes a barrier and thread 0 stores the new
// stage count into the block's flag with release semantics.  Wait: lanes of
// warp 0 poll their peer's flag for the same block index with acquire
// semantics until it reaches the stage count this rank needs, then the block
// passes a barrier.  The release -> acquire pair plus the two barriers order
// the peer's slot stores before this block's slot loads (the data-then-flag
// order of "[Kernel] Two-rank FP16 all-reduce through pinned host memory for
// GPUs without P2P", section "Purpose").
//
// Scope: flags in mapped host memory use .sys (the pages' case: two GPUs
// reach the host buffer); flags in HBM use .gpu, whether the slots are in HBM
// or in host memory (the gpu_scope tactic picks for host-memory slots).  The scope of a release/acquire pair is the set of
// threads it orders, not a place in memory: when every rank is a kernel of
// this GPU, a GPU-scope release orders the block's earlier slot stores to host
// memory before the flag for every reader that acquires it.
//
// Every wait is bounded by %globaltimer.  A block that runs out of time sets
// the sticky abort word, records itself in the handle's error record (the
// first one only) and leaves the kernel without writing its output; later
// waits on the same handle see the abort word and leave at once.  No wait is
// unbounded, so no call can hang the GPU.
#pragma once

#include <cstdint>

#include "ar_internal.h"

namespace tda {

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p, int sys) {
    unsigned long long v;
    if (sys)
        asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    else
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v, int sys) {
    if (sys)
        asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
    else
        asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Loads that bypass L1 (cache at L2 only): peer slot data is read once per
// call and must never come from a line an earlier call left in L1.  These are
// plain data loads; their ordering after a peer's release comes from the
// acquire on the flag and the barrier that follows it.
__device__ __forceinline__ uint4 ld_cg_v4(const void *p) { return __ldcg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ uint2 ld_cg_v2(const void *p) { return __ldcg(reinterpret_cast<const uint2 *>(p)); }
__device__ __forceinline__ unsigned int ld_cg_u32(const void *p) {
    return __ldcg(reinterpret_cast<const unsigned int *>(p));
}
__device__ __forceinline__ unsigned short ld_cg_u16(const void *p) {
    return __ldcg(reinterpret_cast<const unsigned short *>(p));
}
__device__ __forceinline__ unsigned char ld_cg_u8(const void *p) {
    return __ldcg(reinterpret_cast<const unsigned char *>(p));
}

// Tagged-word exchange: 16-byte accesses of two 64-bit words, each word's
// high half a tag.  Each 64-bit word is read and written whole (single-copy
// atomic for an aligned 64-bit relaxed access), so a reader that sees the
// tag it expects also sees the data stored with it; no fence is needed.
__device__ __forceinline__ ulonglong2 ld_tagged(const ulonglong2 *p, int sys) {
    ulonglong2 v;
    if (sys)
        asm volatile("ld.relaxed.sys.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    else
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_tagged(ulonglong2 *p, ulonglong2 v, int sys) {
    if (sys)
        asm volatile("st.relaxed.sys.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(v.x), "l"(v.y) : "memory");
    else
        asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(v.x), "l"(v.y) : "memory");
}

// Trace of one block in one call, kept in shared memory by thread 0 (no
// registers held across the kernel).
struct TraceMarks {
    unsigned long long t0;
    long long c0;
    uint32_t pub, peers;
};

// T: the kernel is built with tracing (its launches come from a handle with
// a trace buffer); without it, none of this is compiled in.
template <bool T>
__device__ __forceinline__ void trace_start(const DevState &d, TraceMarks &m) {
    if constexpr (T) {
        m.t0 = global_timer_ns();
        m.c0 = clock64();
        m.pub = 0;
        m.peers = 0;
    }
}
template <bool T>
__device__ __forceinline__ void trace_published(const DevState &d, TraceMarks &m) {
    if constexpr (T) {
        if (m.pub == 0) m.pub = (uint32_t)(clock64() - m.c0) | 1u;
    }
}
template <bool T>
__device__ __forceinline__ void trace_peers(const DevState &d, TraceMarks &m) {
    if constexpr (T) {
        if (m.peers == 0) m.peers = (uint32_t)(clock64() - m.c0) | 1u;
    }
}
template <bool T>
__device__ __forceinline__ void trace_finish(const DevState &d, const TraceMarks &m, int R, int rank, int block,
                                             unsigned long long calls, unsigned long long stages) {
    if constexpr (T) {
        const uint64_t i = ((calls % d.trace_depth) * (uint64_t)R + (uint64_t)rank) * (uint64_t)d.bmax + block;
        ar_trace_record rec;
        rec.rank = rank;
        rec.block = block;
        rec.call = (uint32_t)calls;
        rec.stages = (uint32_t)stages;
        rec.t_start_ns = m.t0;
        rec.t_end_ns = global_timer_ns();
        rec.cyc_published = m.pub;
        rec.cyc_peers = m.peers;
        rec.cyc_end = (uint32_t)(clock64() - m.c0);
        rec.algo = (uint32_t)d.algo;
        d.trace[i] = rec;
    }
}

// The tag of a block's stage count x in the high half of a tagged word: a
// value in 1 .. 2^32 - 1, never 0, so a word still holding the buffer's initial
// zeros never passes for data however long the counts run (x mod (2^32 - 1),
// plus one: consecutive counts give consecutive tags, wrapping from 2^32 - 1
// to 1).
__device__ __forceinline__ unsigned long long stage_tag(unsigned long long x) {
    return (unsigned long long)((uint32_t)(x % 0xffffffffull) + 1u) << 32;
}

// Programmatic dependent launch.  When a rank's next call is launched with the
// programmatic-serialization attribute, its blocks may become resident before
// this call ends.  Each kernel therefore waits (griddepcontrol.wait: the
// preceding kernel has completed and its memory is visible) before it touches
// any memory.  A block lets its dependents be scheduled once it has seen its
// peers' last flags: by then every block of every rank of this call is
// resident, so the next call's early blocks cannot keep a peer block of this
// call from being scheduled (which would leave this call waiting for it).  Both
// instructions do nothing when the launch has no programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Pacing of the first stage's slot stores (slots in host memory).  Block b
// of every rank starts them b * pace SM cycles after its own start, so the
// call's stores reach the host link about as fast as it drains them instead
// of all at once.  A block's release then waits for its own stores rather
// than for the whole call's, its flag comes up early, and the peers' reads of
// the early blocks' tiles overlap the later blocks' stores (both directions
// of the link busy at once).  The host bounds b * pace (a few ms at most);
// pace = 0 stores at once.
__device__ __forceinline__ void pace_first_stage(long long c0, int b, uint32_t pace) {
    if (pace == 0) return;
    const long long until = c0 + (long long)b * (long long)pace;
    while (clock64() < until) {
    }
}

// Block 0 of a rank, once it knows its call count: set the call count of this
// rank's blocks that the call does not launch (gridDim.x <= b < cmax) to the
// count every launched block will have after the call.  Every block of a rank
// then counts the same calls, so the slot parity -- a block's call count & 1 --
// is the same for all blocks of a call.  Without it, a call on a smaller grid
// leaves the counts of the unused blocks behind, and a later call whose tiles
// map a slot region to another block index could write that region in the
// same parity half a peer is still reading from the call before.  No block of
// this call touches those counters, and the next call's blocks read them only
// after this grid has completed (griddepcontrol.wait).  Stores only, issued
// early, so they overlap the call's work.
__device__ __forceinline__ void advance_idle_blocks(const DevState &d, int rank, unsigned long long calls_after) {
    if (blockIdx.x != 0) return;
    for (int b = (int)gridDim.x + (int)threadIdx.x; b < d.cmax; b += (int)blockDim.x)
        d.ctr[(size_t)rank * d.cmax + b].calls = calls_after;
}

// The rank a block plays, and its input and output.  A kernel built for one
// rank's launch (F = false) takes the rank argument and its own in/out
// arguments, unchanged.  A kernel built for a launch of all ranks at once
// (F = true) takes the block's row of the grid and that rank's pointers from
// io (selects over the R entries: an index into the parameter array would
// copy it to local memory).
template <bool F>
__device__ __forceinline__ int block_rank(int rank_arg) { return F ? (int)blockIdx.y : rank_arg; }

template <int R, bool F, class T>
__device__ __forceinline__ T *rank_ptr(T *own, void *const (&table)[kMaxRanks], int rank) {
    if (!F) return own;
    T *p = static_cast<T *>(table[0]);
#pragma unroll
    for (int q = 1; q < R; ++q)
        if (rank == q) p = static_cast<T *>(table[q]);
    return p;
}

__device__ __forceinline__ unsigned long long *flag_ptr(const DevState &d, int rank, int block) {
    return d.flags + ((size_t)rank * d.bmax + block) * kFlagStrideWords;
}

// Thread 0, after a barrier that follows the block's slot stores: publish.
__device__ __forceinline__ void publish_stage(const DevState &d, int rank, int block,
                                              unsigned long long value) {
    st_release_u64(flag_ptr(d, rank, block), value, d.sys_scope);
}

// Record the first device-side error of the handle (lane that gave up).
static __device__ __noinline__ void record_timeout(const DevState &d, int rank, int block, int peer,
                                            unsigned long long want, unsigned long long seen) {
    if (atomicCAS(d.abort_word, 0u, 1u) == 0u) {
        volatile ar_error_info *e = d.err;
        e->rank = rank;
        e->block = block;
        e->peer = peer;
        e->want = want;
        e->seen = seen;
        __threadfence_system();
        e->code = AR_ETIMEOUT;
        __threadfence_system();
    }
}

// The warp that polls peers' flags.  It is not warp 0, whose thread 0 raises
// this block's own flag just before: a release stalls its warp until the
// block's slot stores are acknowledged (over the host link that is the whole
// write), and the peers' flags can be watched meanwhile.  A block may read its
// peers' data before its own release completes: nothing it reads depends on it.
constexpr int kPollWarp = 1;

// Called by all threads of the block.  Warp kPollWarp waits until every peer
// p != rank has published at least `target` stages for block `block`.  Returns
// true if the block must leave (timeout here or abort elsewhere).  Ends with a
// barrier.
__device__ __forceinline__ bool wait_peers(const DevState &d, int R, int rank, int block,
                                           unsigned long long target, int *s_bail) {
    if ((threadIdx.x >> 5) == kPollWarp) {
        const int lane = threadIdx.x & 31;
        const bool mine = lane < R && lane != rank;
        const unsigned long long *f = mine ? flag_ptr(d, lane, block) : nullptr;
        unsigned long long seen = 0;
        bool ok = true;
        if (mine) {
            seen = ld_acquire_u64(f, d.sys_scope);
            ok = seen >= target;
        }
        if (!__all_sync(0xffffffffu, ok)) {
            const unsigned long long t0 = global_timer_ns();
            unsigned int iter = 0;
            for (;;) {
                if (!ok) {
                    seen = ld_acquire_u64(f, d.sys_scope);
                    ok = seen >= target;
                }
                if (__all_sync(0xffffffffu, ok)) break;
                // The abort word and the clock every 8th poll only: read each
                // time, the abort word's round trip would follow every flag
                // poll's and halve how often the flag is looked at.
                if ((++iter & 7u) != 0u) {
                    if (iter > 64u) __nanosleep(64);
                    continue;
                }
                int stop = 0;
                if (lane == 0) {
                    if (ld_relaxed_u32(d.abort_word) != 0u)
                        stop = 1;
                    else if (global_timer_ns() - t0 > d.timeout_ns)
                        stop = 2;
                }
                stop = __shfl_sync(0xffffffffu, stop, 0);
                if (stop) {
                    if (stop == 2) {
                        const unsigned int late = __ballot_sync(0xffffffffu, !ok);
                        const int peer = __ffs(late) - 1;
                        const unsigned long long peer_seen = __shfl_sync(0xffffffffu, seen, peer);
                        if (lane == 0) record_timeout(d, rank, block, peer, target, peer_seen);
                    }
                    if (lane == 0) *s_bail = 1;
                    break;
                }
                if (iter > 64u) __nanosleep(64);
            }
        }
    }
    __syncthreads();
    return *s_bail != 0;
}

}  // namespace tda
