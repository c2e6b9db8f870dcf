// ar_allreduce.cuh -- the exchange-and-add kernel of one logical rank.
//
// One launch per rank per call; all R launches of a call run at the same time
// on their own streams.  (Or one cooperative launch of a B x R grid for all
// ranks of a call, block (b, r) playing block b of rank r: the same code, with
// co-residency guaranteed by the launch.)  Block b of every rank handles the
// same tiles (tile t belongs to block t % B, in stage t / B), so block b pairs
// only with block b of its peers, through one flag per (rank, block).
//
// Per stage, each block of rank r ("[Kernel] Two-rank FP16 all-reduce through
// pinned host memory for GPUs without P2P", section "Purpose"):
//   1. loads its tile of in_r (16 B per thread per vector, coalesced);
//   2. stores it into slot[parity][r] (parity = the block's call count & 1, so a
//      rank one call ahead never overwrites a slot a peer still reads);
//   3. barrier; thread 0 raises flag[r][b] to the new stage count (release);
//   4. warp 0 waits until flag[p][b] reaches the same count for every p != r
//      (acquire, bounded by the timeout); barrier;
//   5. loads the peers' tiles from their slots (its own stays in registers),
//      adds all R contributions in fp32 in rank order 0..R-1 with
//      round-to-nearest adds (no fused multiply-add), rounds once to the
//      16-bit type and stores out_r.
// The next stage's input is loaded before the wait, so the load overlaps the
// flag round trip.  After the last stage thread 0 advances the block's
// counters.  Every rank computes the same bits: the order of the adds is the
// rank order everywhere ("[SM120] Add optional FlashInfer PCIe-IPC all-reduce
// for switch-free hosts", section "Accuracy": at eight ranks the order decides
// the last bf16 bit).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ar_internal.h"
#include "ar_sync.cuh"

namespace tda {

struct F16Ops {
    static __device__ __forceinline__ float2 widen2(uint32_t w) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
    static __device__ __forceinline__ uint32_t narrow2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
};

struct BF16Ops {
    static __device__ __forceinline__ float2 widen2(uint32_t w) {
        // bfloat16 is the upper half of a binary32: widening is a shift.
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ uint32_t narrow2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
};

// acc[0..7] (+)= the 8 elements of v.
template <class Ops, bool kFirst>
__device__ __forceinline__ void accumulate8(float (&acc)[8], const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = Ops::widen2(w[j]);
        if (kFirst) {
            acc[2 * j] = f.x;
            acc[2 * j + 1] = f.y;
        } else {
            acc[2 * j] = __fadd_rn(acc[2 * j], f.x);
            acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], f.y);
        }
    }
}

template <class Ops>
__device__ __forceinline__ uint4 narrow8(const float (&acc)[8]) {
    uint4 r;
    r.x = Ops::narrow2(acc[0], acc[1]);
    r.y = Ops::narrow2(acc[2], acc[3]);
    r.z = Ops::narrow2(acc[4], acc[5]);
    r.w = Ops::narrow2(acc[6], acc[7]);
    return r;
}

// Load vector v of the caller's input: a full 16-byte vector, or the partial
// last vector (tail elements, zero-filled), or nothing past the end.
// (Element j of a vector lives in 32-bit word j / 2; the tail paths pick the
// word with selects rather than an indexed array, which would need local memory.)
__device__ __forceinline__ uint4 load_own(const uint16_t *in, uint64_t v, uint64_t nvec_full,
                                          int tail) {
    if (v < nvec_full) return *reinterpret_cast<const uint4 *>(in + v * 8);
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (v == nvec_full && tail) {
#pragma unroll
        for (int j = 0; j < 7; ++j) {
            if (j < tail) {
                const uint32_t e = (uint32_t)in[v * 8 + j] << ((j & 1) * 16);
                if (j < 2) r.x |= e;
                else if (j < 4) r.y |= e;
                else if (j < 6) r.z |= e;
                else r.w |= e;
            }
        }
    }
    return r;
}

__device__ __forceinline__ void store_out(uint16_t *out, uint64_t v, uint64_t nvec_full, int tail,
                                          const uint4 r) {
    if (v < nvec_full) {
        *reinterpret_cast<uint4 *>(out + v * 8) = r;
    } else if (v == nvec_full && tail) {
#pragma unroll
        for (int j = 0; j < 7; ++j) {
            if (j < tail) {
                const uint32_t w = j < 2 ? r.x : (j < 4 ? r.y : (j < 6 ? r.z : r.w));
                out[v * 8 + j] = (uint16_t)(w >> ((j & 1) * 16));
            }
        }
    }
}

// A (publish ahead): with several stages per block, a block publishes stage
// s + 1 (loads its input, stores it into the slot, raises the flag) before it
// waits for and reads its peers' stage s, so one stage's flag round overlaps
// the next stage's publish.  Stage s + 1 uses its own slot region, so nothing
// a peer still reads is touched; the flag counts published stages as before.
template <class Ops, int R, int U, bool F, bool T, bool A>
__device__ __forceinline__ void allreduce_oneshot(const uint16_t *in_arg, uint16_t *out_arg, uint64_t numel,
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
    constexpr uint64_t kTileVecs = (uint64_t)kThreads * U;
    const uint64_t ntiles = (nv + kTileVecs - 1) / kTileVecs;
    const uint64_t nstages = ntiles > (uint64_t)b ? (ntiles - b + B - 1) / B : 0;

    pdl_wait();
    const long long c0 = clock64();
    if (tid == 0) {
        trace_start<T>(d, s_tr);
        const Ctr c = d.ctr[(size_t)rank * d.cmax + b];
        s_seq = c.seq;
        s_calls = c.calls;
        s_bail = 0;
    }

    // Stage 0's own input, loaded while thread 0 fetches the counters.
    uint4 own[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint64_t v = (uint64_t)b * kTileVecs + (uint64_t)u * kThreads + tid;
        own[u] = load_own(in, v, nvec_full, tail);
    }
    __syncthreads();
    const unsigned long long seq = s_seq;
    const int parity = (int)(s_calls & 1ull);
    advance_idle_blocks(d, rank, s_calls + 1ull);
    const uint64_t slot_vecs = d.slot_bytes / 16;
    uint4 *const slot_base = reinterpret_cast<uint4 *>(d.slots) + (uint64_t)parity * R * slot_vecs;
    uint4 *const my_slot = slot_base + (uint64_t)rank * slot_vecs;
    if (nstages) pace_first_stage(c0, b, d.pace_cycles);
    if (A && nstages) {
        // stage 0 published before the loop; the loop publishes one ahead
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = (uint64_t)b * kTileVecs + (uint64_t)u * kThreads + tid;
            if (v < nv) my_slot[v] = own[u];
        }
        __syncthreads();
        if (tid == 0) {
            publish_stage(d, rank, b, seq + 1);
            trace_published<T>(d, s_tr);
        }
    }

    for (uint64_t s = 0; s < nstages; ++s) {
        const uint64_t tile = (uint64_t)b + s * B;
        const uint64_t v0 = tile * kTileVecs + tid;

        uint4 nxt[U];
        if constexpr (A) {
            // 2-3. publish stage s + 1 (its input, its slot stores, its flag)
            if (s + 1 < nstages) {
                const uint64_t vn = (tile + B) * kTileVecs + tid;
#pragma unroll
                for (int u = 0; u < U; ++u) nxt[u] = load_own(in, vn + (uint64_t)u * kThreads, nvec_full, tail);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint64_t v = vn + (uint64_t)u * kThreads;
                    if (v < nv) my_slot[v] = nxt[u];
                }
                __syncthreads();
                if (tid == 0) publish_stage(d, rank, b, seq + s + 2);
            }
        } else {
            // 2. publish this stage's data
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint64_t v = v0 + (uint64_t)u * kThreads;
                if (v < nv) my_slot[v] = own[u];
            }
            __syncthreads();
            // 3. raise the flag
            if (tid == 0) {
                publish_stage(d, rank, b, seq + s + 1);
                trace_published<T>(d, s_tr);
            }

            // next stage's input, overlapping the wait
            if (s + 1 < nstages) {
                const uint64_t vn = (tile + B) * kTileVecs + tid;
#pragma unroll
                for (int u = 0; u < U; ++u) nxt[u] = load_own(in, vn + (uint64_t)u * kThreads, nvec_full, tail);
            }
        }

        // 4. wait for the peers
        if (wait_peers(d, R, rank, b, seq + s + 1, &s_bail)) return;
        if (tid == 0) trace_peers<T>(d, s_tr);
        // Every peer block of this call has now published its last stage, so
        // all of them are resident: this rank's next call may be scheduled.
        if (s + 1 == nstages) pdl_trigger();

        // 5. gather, add in rank order, round once, store
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = v0 + (uint64_t)u * kThreads;
            if (v < nv) {
                // (A per-p select of the value, not a store into vals[p] under
                // "p == rank": the compiler turns the latter into a store to
                // vals[rank], a runtime index that needs local memory.)
                uint4 vals[R];
#pragma unroll
                for (int p = 0; p < R; ++p) {
                    uint4 peer = own[u];
                    if (p != rank) peer = ld_cg_v4(slot_base + (uint64_t)p * slot_vecs + v);
                    vals[p] = peer;
                }
                float acc[8];
                accumulate8<Ops, true>(acc, vals[0]);
#pragma unroll
                for (int p = 1; p < R; ++p) accumulate8<Ops, false>(acc, vals[p]);
                store_out(out, v, nvec_full, tail, narrow8<Ops>(acc));
            }
        }
        if (s + 1 < nstages) {
#pragma unroll
            for (int u = 0; u < U; ++u) own[u] = nxt[u];
        }
    }

    if (tid == 0) {
        Ctr c;
        c.seq = seq + nstages;
        c.calls = s_calls + 1;
        d.ctr[(size_t)rank * d.cmax + b] = c;
        trace_finish<T>(d, s_tr, R, rank, b, s_calls, nstages);
    }
}

// One rank's launch.
template <class Ops, int R, int U, bool T, bool A = false>
__global__ void __launch_bounds__(kThreads)
    allreduce_kernel_rank(const uint16_t *in, uint16_t *out, uint64_t numel, int rank, DevState d, RankIO io) {
    allreduce_oneshot<Ops, R, U, false, T, A>(in, out, numel, rank, d, io);
}

// A launch of all ranks, held to the blocks per SM the one-rank kernel gets
// unasked (5 up to R = 3, else 4): with fewer resident blocks a decode-sized
// call would need a second stage, and a large one would move less at once.
template <class Ops, int R, int U, bool T, bool A = false>
__global__ void __launch_bounds__(kThreads, R <= 3 ? 5 : 4)
    allreduce_kernel_all(const uint16_t *in, uint16_t *out, uint64_t numel, int rank, DevState d, RankIO io) {
    allreduce_oneshot<Ops, R, U, true, T, A>(in, out, numel, rank, d, io);
}

// Two-shot variant, for large payloads at R >= 4, where the one-shot form's
// R * (R - 1) * S bytes of peer-slot reads per call saturate L2.  A tile is R
// sub-tiles of SUB vectors (SUB = 256, 128 or 64: smaller sub-tiles spread a
// mid-sized payload over more blocks).  For one tile, each block of rank r:
//   1. copies the whole tile of in_r into slot[parity][r]; barrier; raises its
//      flag (release);
//   2. waits for every peer's flag; reduces sub-tile r: reads it from all R
//      slots, adds in fp32 in rank order 0..R-1, rounds once;
//   3. writes the result over sub-tile r of its own slot (only rank r ever
//      reads sub-tile r of any slot as input); barrier; raises its flag;
//   4. waits for every peer's flag; copies sub-tile p of slot p (rank p's
//      rounded result) into out_r for every p.
// With several tiles per block, step 3 of tile k shares its flag round with
// step 1 of tile k + 1 (one round per tile, plus one), and the next tile's
// input is copied into shared memory while a round's flags are awaited.
// Each element is reduced once, by one rank, in rank order, so every rank
// receives the same bits as the one-shot form and the oracle.  Per call, slot
// reads fall from R * (R - 1) * S to about 2 * R * S bytes.
//
// Blocks per SM: the form is bound by the latency of its flag rounds, so more
// resident blocks keep more tiles in flight.  Up to R = 4 the
// kernel fits in 40 registers without spilling and runs 6 blocks per SM; above
// that the sub-tile accumulators need more, and it keeps 4.
template <int R>
constexpr int twoshot_min_blocks() { return R <= 4 ? 6 : 4; }

// 16-byte asynchronous copy from global to shared memory (no register
// staging), and the waits that make a thread's own copies visible to it.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned int a = (unsigned int)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(a), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

template <class Ops, int R, int SUB, bool F, bool T, bool M>
__global__ void __launch_bounds__(kThreads, twoshot_min_blocks<R>())
    allreduce_twoshot_kernel(const uint16_t *in_arg, uint16_t *out_arg, uint64_t numel, int rank_arg, DevState d, RankIO io) {
    static_assert(SUB == 64 || SUB == 128 || SUB == 256, "sub-tile of 64, 128 or 256 vectors");
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
    constexpr uint64_t kTileVecs = (uint64_t)SUB * R;
    // vectors each thread moves in phases 1 and 3
    constexpr int kPer = (int)((kTileVecs + kThreads - 1) / kThreads);
    const uint64_t ntiles = (nv + kTileVecs - 1) / kTileVecs;
    const uint64_t nstages = ntiles > (uint64_t)b ? (ntiles - b + B - 1) / B : 0;
    // The next stage's tile of in_r, copied asynchronously while this stage's
    // two flag rounds run.  Each thread copies, and later reads back, only its
    // own vectors of the tile, so its own wait is the only ordering needed.
    __shared__ uint4 s_next[kTileVecs];

    pdl_wait();
    const long long c0 = clock64();
    if (tid == 0) {
        trace_start<T>(d, s_tr);
        const Ctr c = d.ctr[(size_t)rank * d.cmax + b];
        s_seq = c.seq;
        s_calls = c.calls;
        s_bail = 0;
    }
    __syncthreads();
    const unsigned long long seq = s_seq;
    const int parity = (int)(s_calls & 1ull);
    advance_idle_blocks(d, rank, s_calls + 1ull);
    const uint64_t slot_vecs = d.slot_bytes / 16;
    uint4 *const slot_base = reinterpret_cast<uint4 *>(d.slots) + (uint64_t)parity * R * slot_vecs;
    uint4 *const my_slot = slot_base + (uint64_t)rank * slot_vecs;

    // M = false: two flag rounds per tile.  M = true: each reduced sub-tile
    // rides on the next tile's flag round (below); the host picks it for slots
    // in HBM and calls of several tiles per block.  Measured on a GB300 (bf16,
    // graphs): merged rounds take R = 8 16 MiB from 92.1 to 82.3 us and 64 MiB
    // from 340 to 297 us, but cost 2-5 % on single-stage calls of 256-vector
    // sub-tiles and 3-4 % on multi-stage calls over the host link, which keep
    // the two rounds.
    const uint64_t rounds = M ? (nstages ? nstages + 1 : 0) : 2 * nstages;
    if constexpr (!M) {
        for (uint64_t s = 0; s < nstages; ++s) {
            const uint64_t tbase = ((uint64_t)b + s * B) * kTileVecs;

            // 1. publish the whole tile (tile-local vector u * kThreads + tid):
            // full vectors of a later stage from the prefetched copy, the rest
            // (stage 0, a partial last vector) loaded here
            if (s > 0) cp_async_wait_all();
            uint4 pub[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const uint64_t li = (uint64_t)u * kThreads + tid;
                if (s > 0 && li < kTileVecs && tbase + li < nvec_full)
                    pub[u] = s_next[li];
                else
                    pub[u] = li < kTileVecs ? load_own(in, tbase + li, nvec_full, tail) : make_uint4(0u, 0u, 0u, 0u);
            }
            if (s == 0) pace_first_stage(c0, b, d.pace_cycles);
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const uint64_t li = (uint64_t)u * kThreads + tid;
                if (li < kTileVecs && tbase + li < nv) my_slot[tbase + li] = pub[u];
            }
            __syncthreads();
            if (tid == 0) {
                publish_stage(d, rank, b, seq + 2 * s + 1);
                trace_published<T>(d, s_tr);
            }
            if (s + 1 < nstages) {
                const uint64_t tn = tbase + (uint64_t)B * kTileVecs;
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const uint64_t li = (uint64_t)u * kThreads + tid;
                    if (li < kTileVecs && tn + li < nvec_full) cp_async16(&s_next[li], in + (tn + li) * 8);
                }
                cp_async_commit();
            }
            if (wait_peers(d, R, rank, b, seq + 2 * s + 1, &s_bail)) {
                cp_async_wait_all();
                return;
            }
            if (tid == 0) trace_peers<T>(d, s_tr);

            // 2. reduce sub-tile `rank` in rank order; the result replaces it in my slot
            const uint64_t vr = tbase + (uint64_t)rank * SUB + tid;
            uint4 res = make_uint4(0u, 0u, 0u, 0u);
            if (tid < SUB && vr < nv) {
                uint4 vals[R];
#pragma unroll
                for (int p = 0; p < R; ++p) vals[p] = ld_cg_v4(slot_base + (uint64_t)p * slot_vecs + vr);
                float acc[8];
                accumulate8<Ops, true>(acc, vals[0]);
#pragma unroll
                for (int p = 1; p < R; ++p) accumulate8<Ops, false>(acc, vals[p]);
                res = narrow8<Ops>(acc);
                my_slot[vr] = res;
            }
            __syncthreads();
            if (tid == 0) publish_stage(d, rank, b, seq + 2 * s + 2);
            if (wait_peers(d, R, rank, b, seq + 2 * s + 2, &s_bail)) {
                cp_async_wait_all();
                return;
            }
            // Every peer block of this call has now published its last stage, so
            // all of them are resident: this rank's next call may be scheduled.
            if (s + 1 == nstages) pdl_trigger();

            // 3. gather the R rounded sub-tiles
            uint4 got[kPer];
            if constexpr (SUB == kThreads) {
                // tile-local vector u * kThreads + tid lies in sub-tile u; this
                // thread reduced vector tid of sub-tile `rank` itself
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const uint64_t v = tbase + (uint64_t)u * kThreads + tid;
                    got[u] = res;
                    if (u != rank && v < nv) got[u] = ld_cg_v4(slot_base + (uint64_t)u * slot_vecs + v);
                }
            } else {
                // a sub-tile is narrower than the block: read every result, this
                // rank's included, from the slots (the barrier above orders them)
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const uint64_t li = (uint64_t)u * kThreads + tid;
                    const uint64_t v = tbase + li;
                    got[u] = make_uint4(0u, 0u, 0u, 0u);
                    if (li < kTileVecs && v < nv) got[u] = ld_cg_v4(slot_base + (li / SUB) * slot_vecs + v);
                }
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const uint64_t li = (uint64_t)u * kThreads + tid;
                if (li < kTileVecs && tbase + li < nv) store_out(out, tbase + li, nvec_full, tail, got[u]);
            }
        }
    }

    // Merged rounds, round k = 0 .. nstages:
    //   publish input tile k (k < nstages) and this rank's reduced sub-tile of
    //   tile k - 1 (k > 0) into the slot; barrier; raise the flag to seq + k + 1;
    //   wait for every peer's flag to reach it; copy the R reduced sub-tiles of
    //   tile k - 1 into out_r (k > 0); reduce sub-tile `rank` of tile k in rank
    //   order (k < nstages), kept in registers until the next round publishes it.
    // Each reduced sub-tile rides on the next tile's flag round, so a block
    // of n stages waits n + 1 times rather than 2n.  The reduced sub-tile r of
    // tile k - 1 overwrites this rank's own input sub-tile r of that tile, which
    // only this rank ever reads (it reduced it in the round before); peers read
    // it only after this round's flag.
    if constexpr (M) {
        uint4 res = make_uint4(0u, 0u, 0u, 0u);
        for (uint64_t k = 0; k < rounds; ++k) {
            const uint64_t tbase = ((uint64_t)b + k * B) * kTileVecs;    // tile k (k < nstages)
            const uint64_t pbase = tbase - (uint64_t)B * kTileVecs;       // tile k - 1 (k > 0)

            // 1. publish tile k (tile-local vector u * kThreads + tid): full
            // vectors of a later stage from the prefetched copy, the rest (stage 0,
            // a partial last vector) loaded here; and tile k - 1's reduced vector
            if (k < nstages) {
                if (k > 0) cp_async_wait_all();
                uint4 pub[kPer];
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const uint64_t li = (uint64_t)u * kThreads + tid;
                    if (k > 0 && li < kTileVecs && tbase + li < nvec_full)
                        pub[u] = s_next[li];
                    else
                        pub[u] = li < kTileVecs ? load_own(in, tbase + li, nvec_full, tail) : make_uint4(0u, 0u, 0u, 0u);
                }
                if (k == 0) pace_first_stage(c0, b, d.pace_cycles);
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const uint64_t li = (uint64_t)u * kThreads + tid;
                    if (li < kTileVecs && tbase + li < nv) my_slot[tbase + li] = pub[u];
                }
            }
            if (k > 0) {
                const uint64_t vr = pbase + (uint64_t)rank * SUB + tid;
                if (tid < SUB && vr < nv) my_slot[vr] = res;
            }
            __syncthreads();
            if (tid == 0) {
                publish_stage(d, rank, b, seq + k + 1);
                trace_published<T>(d, s_tr);
            }
            if (k + 1 < nstages) {
                const uint64_t tn = tbase + (uint64_t)B * kTileVecs;
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const uint64_t li = (uint64_t)u * kThreads + tid;
                    if (li < kTileVecs && tn + li < nvec_full) cp_async16(&s_next[li], in + (tn + li) * 8);
                }
                cp_async_commit();
            }
            if (wait_peers(d, R, rank, b, seq + k + 1, &s_bail)) {
                cp_async_wait_all();
                return;
            }
            if (tid == 0) trace_peers<T>(d, s_tr);
            // Every peer block of this call has now published its last round, so
            // all of them are resident: this rank's next call may be scheduled.
            if (k + 1 == rounds) pdl_trigger();

            // 2. copy the R rounded sub-tiles of tile k - 1 to out_r
            if (k > 0) {
                uint4 got[kPer];
                if constexpr (SUB == kThreads) {
                    // tile-local vector u * kThreads + tid lies in sub-tile u; this
                    // thread reduced vector tid of sub-tile `rank` itself
#pragma unroll
                    for (int u = 0; u < kPer; ++u) {
                        const uint64_t v = pbase + (uint64_t)u * kThreads + tid;
                        got[u] = res;
                        if (u != rank && v < nv) got[u] = ld_cg_v4(slot_base + (uint64_t)u * slot_vecs + v);
                    }
                } else {
                    // a sub-tile is narrower than the block: read every result, this
                    // rank's included, from the slots (the barrier above orders them)
#pragma unroll
                    for (int u = 0; u < kPer; ++u) {
                        const uint64_t li = (uint64_t)u * kThreads + tid;
                        const uint64_t v = pbase + li;
                        got[u] = make_uint4(0u, 0u, 0u, 0u);
                        if (li < kTileVecs && v < nv) got[u] = ld_cg_v4(slot_base + (li / SUB) * slot_vecs + v);
                    }
                }
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const uint64_t li = (uint64_t)u * kThreads + tid;
                    if (li < kTileVecs && pbase + li < nv) store_out(out, pbase + li, nvec_full, tail, got[u]);
                }
            }

            // 3. reduce sub-tile `rank` of tile k in rank order (published next round)
            if (k < nstages) {
                const uint64_t vr = tbase + (uint64_t)rank * SUB + tid;
                if (tid < SUB && vr < nv) {
                    uint4 vals[R];
#pragma unroll
                    for (int p = 0; p < R; ++p) vals[p] = ld_cg_v4(slot_base + (uint64_t)p * slot_vecs + vr);
                    float acc[8];
                    accumulate8<Ops, true>(acc, vals[0]);
#pragma unroll
                    for (int p = 1; p < R; ++p) accumulate8<Ops, false>(acc, vals[p]);
                    res = narrow8<Ops>(acc);
                }
            }
        }

    }

    if (tid == 0) {
        Ctr c;
        c.seq = seq + rounds;
        c.calls = s_calls + 1;
        d.ctr[(size_t)rank * d.cmax + b] = c;
        trace_finish<T>(d, s_tr, R, rank, b, s_calls, nstages);
    }
}

}  // namespace tda

#include "ar_allreduce_tagged.cuh"
#include "ar_allreduce_push.cuh"

namespace tda {

template <class Ops, bool F, bool T>
const void *allreduce_tagged_ptr(int R) {
    switch (R) {
        case 1: return F ? (const void *)allreduce_tagged_all<Ops, 1, T> : (const void *)allreduce_tagged_rank<Ops, 1, T>;
        case 2: return F ? (const void *)allreduce_tagged_all<Ops, 2, T> : (const void *)allreduce_tagged_rank<Ops, 2, T>;
        case 3: return F ? (const void *)allreduce_tagged_all<Ops, 3, T> : (const void *)allreduce_tagged_rank<Ops, 3, T>;
        case 4: return F ? (const void *)allreduce_tagged_all<Ops, 4, T> : (const void *)allreduce_tagged_rank<Ops, 4, T>;
        case 5: return F ? (const void *)allreduce_tagged_all<Ops, 5, T> : (const void *)allreduce_tagged_rank<Ops, 5, T>;
        case 6: return F ? (const void *)allreduce_tagged_all<Ops, 6, T> : (const void *)allreduce_tagged_rank<Ops, 6, T>;
        case 7: return F ? (const void *)allreduce_tagged_all<Ops, 7, T> : (const void *)allreduce_tagged_rank<Ops, 7, T>;
        case 8: return F ? (const void *)allreduce_tagged_all<Ops, 8, T> : (const void *)allreduce_tagged_rank<Ops, 8, T>;
        default: return nullptr;
    }
}

// Kernel entry for (element ops, R, unroll, one rank or all ranks, traced or
// not), as an untyped address for cudaLaunchKernelExC and the occupancy
// calculator.
template <class Ops, int R, int U, bool F, bool T, bool A>
constexpr const void *oneshot_entry() {
    return F ? (const void *)allreduce_kernel_all<Ops, R, U, T, A> : (const void *)allreduce_kernel_rank<Ops, R, U, T, A>;
}

template <class Ops, int U, bool F, bool T, bool A>
const void *allreduce_ptr_ru(int R) {
    switch (R) {
        case 1: return oneshot_entry<Ops, 1, U, F, T, A>();
        case 2: return oneshot_entry<Ops, 2, U, F, T, A>();
        case 3: return oneshot_entry<Ops, 3, U, F, T, A>();
        case 4: return oneshot_entry<Ops, 4, U, F, T, A>();
        case 5: return oneshot_entry<Ops, 5, U, F, T, A>();
        case 6: return oneshot_entry<Ops, 6, U, F, T, A>();
        case 7: return oneshot_entry<Ops, 7, U, F, T, A>();
        case 8: return oneshot_entry<Ops, 8, U, F, T, A>();
        default: return nullptr;
    }
}

template <class Ops, int SUB, bool F, bool T, bool M>
const void *allreduce_twoshot_ptr_r(int R) {
    switch (R) {
        case 1: return (const void *)allreduce_twoshot_kernel<Ops, 1, SUB, F, T, M>;
        case 2: return (const void *)allreduce_twoshot_kernel<Ops, 2, SUB, F, T, M>;
        case 3: return (const void *)allreduce_twoshot_kernel<Ops, 3, SUB, F, T, M>;
        case 4: return (const void *)allreduce_twoshot_kernel<Ops, 4, SUB, F, T, M>;
        case 5: return (const void *)allreduce_twoshot_kernel<Ops, 5, SUB, F, T, M>;
        case 6: return (const void *)allreduce_twoshot_kernel<Ops, 6, SUB, F, T, M>;
        case 7: return (const void *)allreduce_twoshot_kernel<Ops, 7, SUB, F, T, M>;
        case 8: return (const void *)allreduce_twoshot_kernel<Ops, 8, SUB, F, T, M>;
        default: return nullptr;
    }
}

template <class Ops, bool F, bool T, bool M>
const void *allreduce_twoshot_ptr(int R, int sub) {
    switch (sub) {
        case 256: return allreduce_twoshot_ptr_r<Ops, 256, F, T, M>(R);
        case 128: return allreduce_twoshot_ptr_r<Ops, 128, F, T, M>(R);
        case 64: return allreduce_twoshot_ptr_r<Ops, 64, F, T, M>(R);
        default: return nullptr;
    }
}

// U = 1 or 2: one-shot with that many vectors per thread per stage;
// U = oneshot_ahead_variant(1 or 2): the same, publishing one stage ahead
// (untraced only: a traced launch takes the plain one-shot kernel);
// U = twoshot_variant(sub): the two-shot form with sub-tiles of `sub` vectors;
// U = kTaggedVariant: the tagged-word form; U = kPushVariant: the push form.
// fused: the kernel for one launch of all ranks (grid blocks x R); traced:
// the kernel that writes trace records.
template <class Ops, bool F, bool T>
const void *allreduce_ptr_ft(int R, int U) {
    if (U == kTaggedVariant) return allreduce_tagged_ptr<Ops, F, T>(R);
    if (U == kPushVariant) return allreduce_push_ptr<Ops, F, T>(R);
    if (U < 0) return nullptr;  // two-shot: allreduce_twoshot_ptr_any, in its own translation unit
    const int u = oneshot_unroll(U);
    if (!T && oneshot_ahead(U))
        return u == 1 ? allreduce_ptr_ru<Ops, 1, F, false, true>(R) : allreduce_ptr_ru<Ops, 2, F, false, true>(R);
    return u == 1 ? allreduce_ptr_ru<Ops, 1, F, T, false>(R) : allreduce_ptr_ru<Ops, 2, F, T, false>(R);
}

// One-shot, tagged-word and push kernels (U >= 0).
template <class Ops>
const void *allreduce_ptr(int R, int U, bool fused, bool traced) {
    if (traced) return fused ? allreduce_ptr_ft<Ops, true, true>(R, U) : allreduce_ptr_ft<Ops, false, true>(R, U);
    return fused ? allreduce_ptr_ft<Ops, true, false>(R, U) : allreduce_ptr_ft<Ops, false, false>(R, U);
}

// Two-shot kernels (U < 0).  Instantiated by their own translation units, so
// that a dtype's kernels compile in parallel.
// Traced launches always take the kernel of two rounds per tile (no merged
// traced kernel is built).
template <class Ops>
const void *allreduce_twoshot_ptr_any(int R, int U, bool fused, bool traced) {
    const int sub = twoshot_sub(U);
    if (traced)
        return fused ? allreduce_twoshot_ptr<Ops, true, true, false>(R, sub)
                     : allreduce_twoshot_ptr<Ops, false, true, false>(R, sub);
    if (twoshot_merged(U))
        return fused ? allreduce_twoshot_ptr<Ops, true, false, true>(R, sub)
                     : allreduce_twoshot_ptr<Ops, false, false, true>(R, sub);
    return fused ? allreduce_twoshot_ptr<Ops, true, false, false>(R, sub)
                 : allreduce_twoshot_ptr<Ops, false, false, false>(R, sub);
}

}  // namespace tda
