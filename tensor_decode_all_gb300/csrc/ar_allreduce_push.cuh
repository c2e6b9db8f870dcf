// ar_allreduce_push.cuh -- the push form of the exchange-and-add.
//
// In the pull form every rank publishes its tile once, in its own slot, and
// every reader fetches its peers' tiles from their slots.  In the push form
// ("[SM120] Add optional FlashInfer PCIe-IPC all-reduce for switch-free
// hosts", section "Motivation": writers store straight into the readers'
// receive areas, staged so that each rank keeps one outbound and one inbound
// stream) a writer stores its tile into a receive area of every peer, and a
// reader finds all its peers' tiles in its own area.  Across GPUs that turns
// remote reads into remote writes; on one GPU every area lives in the same
// memory, so the form moves R - 1 times the pull form's slot writes and the
// same reads, and exists to measure that trade here.
//
// Layout: recv[parity][reader q][writer p][slot bytes]; flags
// pflag[reader q][writer p][block], one 128-byte line each.  Per stage s,
// block b of rank r:
//   1. loads its tile of in_r (256 vectors);
//   2. stores it into recv[parity][q][r] for q = r + 1, r + 2, ... (mod R), one
//      peer after another, so that at each step every rank writes to one peer
//      and receives from one;
//   3. barrier; thread 0 makes the stores visible (one fence at the slots'
//      scope) and raises pflag[q][r][b] to the new stage count for every q;
//   4. waits until pflag[r][p][b] reaches it for every peer p;
//   5. adds all R tiles in rank order (its own from registers), rounds once,
//      stores out_r -- the same arithmetic, so the same bits.
// Parity and stage counts come from the same per-(rank, block) counters as
// the other forms, so the forms interleave on one handle.
#pragma once

#include "ar_allreduce.cuh"

namespace tda {

__device__ __forceinline__ unsigned long long *push_flag_ptr(const DevState &d, int reader, int writer, int block,
                                                           int R) {
    return d.push_flags + (((size_t)reader * R + writer) * d.bmax + block) * kFlagStrideWords;
}

__device__ __forceinline__ void fence_release_scope(int sys) {
    if (sys)
        asm volatile("fence.acq_rel.sys;" ::: "memory");
    else
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v, int sys) {
    if (sys)
        asm volatile("st.relaxed.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
    else
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Warp kPollWarp waits until every writer p != rank has pushed `target` stages
// of block `block` to this rank.  Bounded like wait_peers; ends with a barrier.
__device__ __forceinline__ bool wait_pushes(const DevState &d, int R, int rank, int block,
                                            unsigned long long target, int *s_bail) {
    if ((threadIdx.x >> 5) == kPollWarp) {
        const int lane = threadIdx.x & 31;
        const bool mine = lane < R && lane != rank;
        const unsigned long long *f = mine ? push_flag_ptr(d, rank, lane, block, R) : nullptr;
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

template <class Ops, int R, bool F, bool T>
__device__ __forceinline__ void allreduce_push_body(const uint16_t *in_arg, uint16_t *out_arg, uint64_t numel,
                                                    int rank_arg, const DevState &d, const RankIO &io) {
    __shared__ unsigned long long s_seq;
    __shared__ unsigned long long s_calls;
    __shared__ int s_bail;
    __shared__ TraceMarks s_tr;

    const int rank = block_rank<F>(rank_arg);
    const uint16_t *in = rank_ptr<R, F>(in_arg, io.in, rank);
    uint16_t *out = rank_ptr<R, F>(out_arg, io.out, rank);
    const int b = blockIdx.x;
    const int B = gridDim.x;
    const int tid = threadIdx.x;
    const uint64_t nvec_full = numel / 8;
    const int tail = (int)(numel % 8);
    const uint64_t nv = nvec_full + (tail ? 1 : 0);
    const uint64_t ntiles = (nv + kThreads - 1) / kThreads;
    const uint64_t nstages = ntiles > (uint64_t)b ? (ntiles - b + B - 1) / B : 0;

    pdl_wait();
    if (tid == 0) {
        trace_start<T>(d, s_tr);
        const Ctr c = d.ctr[(size_t)rank * d.cmax + b];
        s_seq = c.seq;
        s_calls = c.calls;
        s_bail = 0;
    }
    uint4 own = load_own(in, (uint64_t)b * kThreads + tid, nvec_full, tail);
    __syncthreads();
    const unsigned long long seq = s_seq;
    const int parity = (int)(s_calls & 1ull);
    advance_idle_blocks(d, rank, s_calls + 1ull);
    const uint64_t slot_vecs = d.slot_bytes / 16;
    // recv[parity][reader][writer]
    uint4 *const area = reinterpret_cast<uint4 *>(d.push) + (uint64_t)parity * R * R * slot_vecs;

    for (uint64_t s = 0; s < nstages; ++s) {
        const uint64_t v = ((uint64_t)b + s * B) * kThreads + tid;
        // 2. push to the peers, one after another
        if (v < nv) {
#pragma unroll
            for (int k = 1; k < R; ++k) {
                const int q = (rank + k) % R;
                area[((uint64_t)q * R + rank) * slot_vecs + v] = own;
            }
        }
        __syncthreads();
        // 3. one fence, then every peer's flag
        if (tid == 0) {
            fence_release_scope(d.sys_scope);
#pragma unroll
            for (int k = 1; k < R; ++k) {
                const int q = (rank + k) % R;
                st_relaxed_u64(push_flag_ptr(d, q, rank, b, R), seq + s + 1, d.sys_scope);
            }
            trace_published<T>(d, s_tr);
        }
        uint4 nxt = make_uint4(0u, 0u, 0u, 0u);
        if (s + 1 < nstages) nxt = load_own(in, v + (uint64_t)B * kThreads, nvec_full, tail);
        // 4. every peer's push to this rank
        if (wait_pushes(d, R, rank, b, seq + s + 1, &s_bail)) return;
        if (tid == 0) trace_peers<T>(d, s_tr);
        if (s + 1 == nstages) pdl_trigger();
        // 5. add in rank order, round once, store
        if (v < nv) {
            float acc[8];
            accumulate8<Ops, true>(acc, rank == 0 ? own : ld_cg_v4(area + ((uint64_t)rank * R + 0) * slot_vecs + v));
#pragma unroll
            for (int p = 1; p < R; ++p)
                accumulate8<Ops, false>(acc, p == rank ? own : ld_cg_v4(area + ((uint64_t)rank * R + p) * slot_vecs + v));
            store_out(out, v, nvec_full, tail, narrow8<Ops>(acc));
        }
        own = nxt;
    }

    if (tid == 0) {
        Ctr c;
        c.seq = seq + nstages;
        c.calls = s_calls + 1;
        d.ctr[(size_t)rank * d.cmax + b] = c;
        trace_finish<T>(d, s_tr, R, rank, b, s_calls, nstages);
    }
}

template <class Ops, int R, bool T>
__global__ void __launch_bounds__(kThreads)
    allreduce_push_rank(const uint16_t *in, uint16_t *out, uint64_t numel, int rank, DevState d, RankIO io) {
    allreduce_push_body<Ops, R, false, T>(in, out, numel, rank, d, io);
}

template <class Ops, int R, bool T>
__global__ void __launch_bounds__(kThreads, R <= 3 ? 5 : 4)
    allreduce_push_all(const uint16_t *in, uint16_t *out, uint64_t numel, int rank, DevState d, RankIO io) {
    allreduce_push_body<Ops, R, true, T>(in, out, numel, rank, d, io);
}

template <class Ops, bool F, bool T>
const void *allreduce_push_ptr(int R) {
    switch (R) {
        case 1: return F ? (const void *)allreduce_push_all<Ops, 1, T> : (const void *)allreduce_push_rank<Ops, 1, T>;
        case 2: return F ? (const void *)allreduce_push_all<Ops, 2, T> : (const void *)allreduce_push_rank<Ops, 2, T>;
        case 3: return F ? (const void *)allreduce_push_all<Ops, 3, T> : (const void *)allreduce_push_rank<Ops, 3, T>;
        case 4: return F ? (const void *)allreduce_push_all<Ops, 4, T> : (const void *)allreduce_push_rank<Ops, 4, T>;
        case 5: return F ? (const void *)allreduce_push_all<Ops, 5, T> : (const void *)allreduce_push_rank<Ops, 5, T>;
        case 6: return F ? (const void *)allreduce_push_all<Ops, 6, T> : (const void *)allreduce_push_rank<Ops, 6, T>;
        case 7: return F ? (const void *)allreduce_push_all<Ops, 7, T> : (const void *)allreduce_push_rank<Ops, 7, T>;
        case 8: return F ? (const void *)allreduce_push_all<Ops, 8, T> : (const void *)allreduce_push_rank<Ops, 8, T>;
        default: return nullptr;
    }
}

}  // namespace tda
