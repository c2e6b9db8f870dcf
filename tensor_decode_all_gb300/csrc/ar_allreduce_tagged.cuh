// ar_allreduce_tagged.cuh -- the tagged-word form of the exchange-and-add, for
// latency-bound (small) calls.
//
// The flag protocol pays, per stage, for a release that waits until the
// block's slot stores are acknowledged, then for the peer's poll of the flag,
// then for the peer's read of the data: three trips across the slot memory's
// link.  Here every 8-byte word of the exchange buffer carries 4 bytes of
// payload in its low half and a 4-byte tag in its high half, derived from the
// block's stage count (the value the flag would have been raised to).
// A writer stores its tagged words with plain relaxed stores and no fence; a
// reader loads its peers' words until every tag matches, which proves the
// payload beside it is this stage's.  One trip, at twice the bytes: worth it
// where the call is bound by latency rather than bandwidth.
//
// Per stage s, thread t of block b of rank r (payload vector v = tile * 256 +
// t, buffer position w = (s * bmax + b) * 256 + t):
//   1. loads vector v of in_r (8 elements, 16 bytes) and stores it as two
//      tagged 16-byte vectors into ll[parity][r] at 2w, 2w + 1;
//   2. loads the peers' two tagged vectors at 2w, 2w + 1 until their four tags
//      equal the stage's tag (bounded by the timeout, abandoned on abort);
//   3. adds the R contributions in fp32 in rank order, rounds once, stores
//      out_r -- the same arithmetic, so the same bits, as the other forms.
// Threads do not wait for each other: no barrier inside a stage.  A buffer
// position belongs to one block index, whose tags never repeat within 2^32 - 1
// stages and are never 0 (the buffer's initial contents), and parity
// double-buffering keeps a rank one call ahead from overwriting words a peer
// still reads.
#pragma once

#include "ar_internal.h"
#include "ar_sync.cuh"

namespace tda {

template <class Ops, int R, bool F, bool T>
__device__ __forceinline__ void allreduce_tagged_body(const uint16_t *in_arg, uint16_t *out_arg, uint64_t numel,
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
    ulonglong2 *const base = d.ll + (uint64_t)parity * R * d.ll_vecs;
    ulonglong2 *const mine = base + (uint64_t)rank * d.ll_vecs;
    const int sys = d.sys_scope;
    bool bail = false;

    for (uint64_t s = 0; s < nstages; ++s) {
        const uint64_t v = ((uint64_t)b + s * B) * kThreads + tid;
        const unsigned long long tag = stage_tag(seq + s + 1);
        // The buffer is indexed by (stage, block, thread), not by payload
        // vector: a word is only ever written by block b of its rank, whose
        // tags only grow, so a stale word can never carry the tag a reader
        // expects (indexed by vector, a word could be left by another block
        // index of an earlier call with another grid size, whose own count
        // may have passed through the same value).  The host takes this form
        // only for calls that fit (one stage per block).
        const uint64_t w = ((uint64_t)s * d.bmax + b) * kThreads + tid;
        const bool live = v < nv && !bail && 2 * w + 1 < d.ll_vecs;

        // 1. publish this vector as two tagged vectors
        if (live) {
            st_tagged(mine + 2 * w, make_ulonglong2(tag | own.x, tag | own.y), sys);
            st_tagged(mine + 2 * w + 1, make_ulonglong2(tag | own.z, tag | own.w), sys);
        }
        if (tid == 0) trace_published<T>(d, s_tr);
        // the next stage's input, overlapping the wait
        uint4 nxt = make_uint4(0u, 0u, 0u, 0u);
        if (s + 1 < nstages && !bail) nxt = load_own(in, v + (uint64_t)B * kThreads, nvec_full, tail);

        // 2. the peers' words of this stage
        uint4 got[R];
        if (live) {
            unsigned int pending = ((1u << R) - 1u) & ~(1u << rank);
            unsigned long long t0 = 0;
            unsigned int iter = 0;
            while (pending) {
#pragma unroll
                for (int p = 0; p < R; ++p) {
                    if (pending & (1u << p)) {
                        const ulonglong2 *src = base + (uint64_t)p * d.ll_vecs + 2 * w;
                        const ulonglong2 lo = ld_tagged(src, sys);
                        const ulonglong2 hi = ld_tagged(src + 1, sys);
                        if (((lo.x & lo.y & hi.x & hi.y) >> 32) == (tag >> 32) &&
                            ((lo.x | lo.y | hi.x | hi.y) >> 32) == (tag >> 32)) {
                            got[p] = make_uint4((uint32_t)lo.x, (uint32_t)lo.y, (uint32_t)hi.x, (uint32_t)hi.y);
                            pending &= ~(1u << p);
                        }
                    }
                }
                if (!pending) break;
                ++iter;
                if (iter == 1) {
                    t0 = global_timer_ns();
                } else if ((iter & 15u) == 0u) {
                    if (ld_relaxed_u32(d.abort_word) != 0u) {
                        bail = true;
                    } else if (global_timer_ns() - t0 > d.timeout_ns) {
                        const int peer = __ffs(pending) - 1;
                        record_timeout(d, rank, b, peer, seq + s + 1, 0ull);
                        bail = true;
                    }
                    if (bail) {
                        s_bail = 1;
                        break;
                    }
                }
                if (iter > 32u) __nanosleep(32);
            }
        }
        if (tid == 0) trace_peers<T>(d, s_tr);
        // Every peer block of this call has now published its last stage, so
        // all of them are resident: this rank's next call may be scheduled.
        if (s + 1 == nstages) {
            __syncthreads();
            pdl_trigger();
        }

        // 3. add in rank order, round once, store.  Where v < nv the peers'
        // words were read: the host sends this form only calls of one stage
        // per block, so w = b * 256 + tid stays inside the buffer and `live`
        // differs from this test only by `bail`, checked here again.
        if (v < nv && !bail) {
            uint4 vals[R];
#pragma unroll
            for (int p = 0; p < R; ++p) {
                uint4 x = own;
                if (p != rank) x = got[p];
                vals[p] = x;
            }
            float acc[8];
            accumulate8<Ops, true>(acc, vals[0]);
#pragma unroll
            for (int p = 1; p < R; ++p) accumulate8<Ops, false>(acc, vals[p]);
            store_out(out, v, nvec_full, tail, narrow8<Ops>(acc));
        }
        own = nxt;
    }

    __syncthreads();
    if (s_bail) return;
    if (tid == 0) {
        Ctr c;
        c.seq = seq + nstages;
        c.calls = s_calls + 1;
        d.ctr[(size_t)rank * d.cmax + b] = c;
        trace_finish<T>(d, s_tr, R, rank, b, s_calls, nstages);
    }
}

// Both entries are held to 64 registers (4 blocks per SM), so that a call
// spreads over as many blocks as the one-shot form's.
template <class Ops, int R, bool T>
__global__ void __launch_bounds__(kThreads, 4)
    allreduce_tagged_rank(const uint16_t *in, uint16_t *out, uint64_t numel, int rank, DevState d, RankIO io) {
    allreduce_tagged_body<Ops, R, false, T>(in, out, numel, rank, d, io);
}

template <class Ops, int R, bool T>
__global__ void __launch_bounds__(kThreads, 4)
    allreduce_tagged_all(const uint16_t *in, uint16_t *out, uint64_t numel, int rank, DevState d, RankIO io) {
    allreduce_tagged_body<Ops, R, true, T>(in, out, numel, rank, d, io);
}

}  // namespace tda
