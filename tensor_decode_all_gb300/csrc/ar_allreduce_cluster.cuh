// ar_allreduce_cluster.cuh -- the exchange-and-add with every rank of a call in
// one launch, each rank's block b in one thread-block cluster.
//
// A launch of all R ranks at once (ar_allreduce_fused, ar_allreduce_all) is a
// grid of B x R blocks, block (b, r) playing block b of rank r.  Launched with
// clusters of 1 x R blocks, the R blocks that pair with each other -- block b of
// every rank -- form one cluster, which the hardware schedules together on one
// GPU processing cluster.  The per-block flag of the flag protocol ("[Kernel]
// Two-rank FP16 all-reduce through pinned host memory for GPUs without P2P",
// section "Purpose": publish the data, make it visible, raise a flag, wait for
// the peers' flags) then has a hardware counterpart: each block arrives on the
// cluster barrier with release semantics after its slot stores, and waits on
// it with acquire semantics before it reads its peers' slots.  The data still
// moves through the same double-buffered slots (HBM or mapped host memory);
// only the flag round trip through memory is replaced.  A cluster waits for
// nothing outside itself, so the grid needs no co-residency and no cooperative
// launch, and it can hold more clusters than the GPU holds at once.
//
// Release and acquire at cluster scope order the slot stores before the
// peers' loads for any memory the blocks share, host memory included: every
// block of a cluster runs on this GPU.  The form therefore exists only for
// logical ranks on one GPU, where all ranks of a call are launched together;
// separate per-rank launches keep the flag protocol.
//
// Two variants, the same arithmetic and bits as the others (rank-order fp32
// sum, one rounding):
//   one-shot (SUB = 0): per stage, tile = 256 vectors; store into the slot,
//     barrier, add all R tiles in rank order, store out;
//   two-shot (SUB = 64, 128, 256): tile = R sub-tiles of SUB vectors; store the
//     tile, barrier, rank r reduces sub-tile r from all R slots and writes the
//     result over it in its own slot, barrier, every rank copies the R results.
//
// Handle state: each block reads its (rank, block) call count, whose parity
// picks the slot half, and advances it, as the other forms do (block 0 of a
// rank also advances the counts of the blocks the call does not launch).
// Both stores are made at the start, where they overlap the call's work.  The
// stage counts and flags are left as they are: no flag is raised, so the flag
// forms' next waits still expect the values they would have without this call.
#pragma once

#include "ar_allreduce.cuh"

namespace tda {

// Cluster barrier: arrive with release semantics (this block's prior stores,
// as observed by its threads after the block-wide arrival, are ordered before
// the peers' loads that follow their wait), then wait with acquire semantics.
// Every thread of the block executes both, convergently.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Resident blocks per SM the kernel is built for: 6 (40 registers a thread).
// More resident clusters run a call in fewer waves, which outweighs the few
// bytes some variants then spill to local memory (R = 8 bf16 768 KiB HBM,
// 64-vector sub-tiles: 8.2 us at 40 registers and 110 resident clusters with
// 64 bytes of spill, 10.3 us at 64 registers and 74 clusters without).  The
// 256-vector sub-tiles from R = 4 hold R * 8 vectors of a tile per thread and
// get no bound (at 64 registers they would spill up to 200 bytes).
template <int R, int SUB>
constexpr int cluster_min_blocks() {
    return (SUB == 256 && R >= 4) ? 1 : 6;
}

// P: the kernel with the pacing code, for calls whose first-stage slot stores
// are paced (slots in host memory, a pace set, one wave of clusters) and, as
// measured faster, for two-shot calls.  Unpaced one-shot calls take the kernel
// without it: at R = 8, held to 40 registers, its presence cost small calls
// 0.3-1 us even with no pace.
template <class Ops, int R, int SUB, bool T, bool P>
__global__ void __launch_bounds__(kThreads, cluster_min_blocks<R, SUB>())
    allreduce_cluster_kernel(const uint16_t *in_arg, uint16_t *out_arg, uint64_t numel, int rank_arg, DevState d,
                             RankIO io) {
    static_assert(SUB == 0 || SUB == 64 || SUB == 128 || SUB == 256, "one-shot or a two-shot sub-tile");
    __shared__ unsigned long long s_calls;
    __shared__ TraceMarks s_tr;

    const int rank = (int)blockIdx.y;
    const uint16_t *in = rank_ptr<R, true>(in_arg, io.in, rank);
    uint16_t *out = rank_ptr<R, true>(out_arg, io.out, rank);
    const int b = blockIdx.x;
    const int B = gridDim.x;
    const int tid = threadIdx.x;
    const uint64_t nvec_full = numel / 8;
    const int tail = (int)(numel % 8);
    const uint64_t nv = nvec_full + (tail ? 1 : 0);
    constexpr uint64_t kTileVecs = SUB == 0 ? (uint64_t)kThreads : (uint64_t)SUB * R;
    constexpr int kPer = (int)((kTileVecs + kThreads - 1) / kThreads);
    const uint64_t ntiles = (nv + kTileVecs - 1) / kTileVecs;
    const uint64_t nstages = ntiles > (uint64_t)b ? (ntiles - b + B - 1) / B : 0;

    pdl_wait();
    long long c0 = 0;
    if constexpr (P) c0 = clock64();
    // stage 0's tile of this rank's input, loaded while thread 0 fetches the
    // call count (the slot half it goes to)
    uint4 own[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const uint64_t li = (uint64_t)u * kThreads + tid;
        own[u] = li < kTileVecs ? load_own(in, (uint64_t)b * kTileVecs + li, nvec_full, tail)
                                : make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid == 0) {
        trace_start<T>(d, s_tr);
        s_calls = d.ctr[(size_t)rank * d.cmax + b].calls;
    }
    __syncthreads();
    const unsigned long long calls = s_calls;
    // The count after this call, stored now so that the store overlaps the
    // call's work: no block of this call reads it again, and the next call
    // reads it only after this grid has completed (griddepcontrol.wait).
    if (tid == 0) d.ctr[(size_t)rank * d.cmax + b].calls = calls + 1ull;
    const int parity = (int)(calls & 1ull);
    advance_idle_blocks(d, rank, calls + 1ull);
    const uint64_t slot_vecs = d.slot_bytes / 16;
    uint4 *const slot_base = reinterpret_cast<uint4 *>(d.slots) + (uint64_t)parity * R * slot_vecs;
    uint4 *const my_slot = slot_base + (uint64_t)rank * slot_vecs;

    for (uint64_t s = 0; s < nstages; ++s) {
        const uint64_t tbase = ((uint64_t)b + s * B) * kTileVecs;

        // publish this rank's tile
        if (s > 0) {
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const uint64_t li = (uint64_t)u * kThreads + tid;
                own[u] = li < kTileVecs ? load_own(in, tbase + li, nvec_full, tail) : make_uint4(0u, 0u, 0u, 0u);
            }
        } else if constexpr (P) {
            pace_first_stage(c0, b, d.pace_cycles);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const uint64_t li = (uint64_t)u * kThreads + tid;
            if (li < kTileVecs && tbase + li < nv) my_slot[tbase + li] = own[u];
        }
        cluster_arrive_release();
        cluster_wait_acquire();
        if (tid == 0) {
            trace_published<T>(d, s_tr);
            trace_peers<T>(d, s_tr);
        }

        if constexpr (SUB == 0) {
            // every rank adds all R tiles in rank order (its own from registers)
            if (s + 1 == nstages) pdl_trigger();
            const uint64_t v = tbase + tid;
            if (v < nv) {
                // each contribution added as it arrives, in rank order (fewer
                // live registers than holding all R first; the same adds)
                float acc[8];
                accumulate8<Ops, true>(acc, rank == 0 ? own[0] : ld_cg_v4(slot_base + v));
#pragma unroll
                for (int p = 1; p < R; ++p)
                    accumulate8<Ops, false>(acc, p == rank ? own[0] : ld_cg_v4(slot_base + (uint64_t)p * slot_vecs + v));
                store_out(out, v, nvec_full, tail, narrow8<Ops>(acc));
            }
        } else {
            // rank r reduces sub-tile r in rank order and writes the result over it
            const uint64_t vr = tbase + (uint64_t)rank * SUB + tid;
            if (tid < SUB && vr < nv) {
                float acc[8];
                accumulate8<Ops, true>(acc, ld_cg_v4(slot_base + vr));
#pragma unroll
                for (int p = 1; p < R; ++p) accumulate8<Ops, false>(acc, ld_cg_v4(slot_base + (uint64_t)p * slot_vecs + vr));
                my_slot[vr] = narrow8<Ops>(acc);
            }
            cluster_arrive_release();
            cluster_wait_acquire();
            if (s + 1 == nstages) pdl_trigger();
            // every rank copies the R rounded sub-tiles
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const uint64_t li = (uint64_t)u * kThreads + tid;
                const uint64_t v = tbase + li;
                if (li < kTileVecs && v < nv)
                    store_out(out, v, nvec_full, tail, ld_cg_v4(slot_base + (li / SUB) * slot_vecs + v));
            }
        }
    }

    if (tid == 0) trace_finish<T>(d, s_tr, R, rank, b, calls, nstages);
}

template <class Ops, int SUB, bool T, bool P>
const void *allreduce_cluster_ptr_r(int R) {
    switch (R) {
        case 1: return (const void *)allreduce_cluster_kernel<Ops, 1, SUB, T, P>;
        case 2: return (const void *)allreduce_cluster_kernel<Ops, 2, SUB, T, P>;
        case 3: return (const void *)allreduce_cluster_kernel<Ops, 3, SUB, T, P>;
        case 4: return (const void *)allreduce_cluster_kernel<Ops, 4, SUB, T, P>;
        case 5: return (const void *)allreduce_cluster_kernel<Ops, 5, SUB, T, P>;
        case 6: return (const void *)allreduce_cluster_kernel<Ops, 6, SUB, T, P>;
        case 7: return (const void *)allreduce_cluster_kernel<Ops, 7, SUB, T, P>;
        case 8: return (const void *)allreduce_cluster_kernel<Ops, 8, SUB, T, P>;
        default: return nullptr;
    }
}

template <class Ops, bool T, bool P>
const void *allreduce_cluster_ptr_tp(int R, int sub) {
    switch (sub) {
        case 0: return allreduce_cluster_ptr_r<Ops, 0, T, P>(R);
        case 64: return allreduce_cluster_ptr_r<Ops, 64, T, P>(R);
        case 128: return allreduce_cluster_ptr_r<Ops, 128, T, P>(R);
        case 256: return allreduce_cluster_ptr_r<Ops, 256, T, P>(R);
        default: return nullptr;
    }
}

// sub = 0: one-shot; 64, 128, 256: two-shot with sub-tiles of that many
// vectors.  paced: the kernel with the pacing code (see P above).
template <class Ops>
const void *allreduce_cluster_ptr(int R, int sub, bool traced, bool paced) {
    if (traced)
        return paced ? allreduce_cluster_ptr_tp<Ops, true, true>(R, sub) : allreduce_cluster_ptr_tp<Ops, true, false>(R, sub);
    return paced ? allreduce_cluster_ptr_tp<Ops, false, true>(R, sub) : allreduce_cluster_ptr_tp<Ops, false, false>(R, sub);
}

}  // namespace tda
