// ar_allgather.cu -- the allgather kernel of one logical rank.
//
// Every rank ends with out = shard_0 || shard_1 || ... || shard_{R-1}, the
// rank-major concatenation used for the complex64 S_j and core uploads in
// "fix(group): run each rank on a non-blocking stream", sections "What" and
// "Why".  It uses the same slot and
// flag protocol as the all-reduce (slots in host memory: with the first
// stage's slot stores paced as the one-shot form's, the link bytes being the
// same): per stage, a block copies its tile of the
// shard into slot[parity][r] and into its own place in out, raises its flag,
// waits for its peers' flags for the same block index, then copies the peers'
// tiles from their slots into their places in out.  Pure copies: the result
// is bit-exact, NaN payloads included.
#include "ar_internal.h"
#include "ar_sync.cuh"

namespace tda {
namespace {

template <int VW>
struct Vec;
template <>
struct Vec<16> {
    using T = uint4;
    static __device__ __forceinline__ T ldcg(const void *p) { return ld_cg_v4(p); }
};
template <>
struct Vec<8> {
    using T = uint2;
    static __device__ __forceinline__ T ldcg(const void *p) { return ld_cg_v2(p); }
};
template <>
struct Vec<4> {
    using T = unsigned int;
    static __device__ __forceinline__ T ldcg(const void *p) { return ld_cg_u32(p); }
};
template <>
struct Vec<2> {
    using T = unsigned short;
    static __device__ __forceinline__ T ldcg(const void *p) { return ld_cg_u16(p); }
};
template <>
struct Vec<1> {
    using T = unsigned char;
    static __device__ __forceinline__ T ldcg(const void *p) { return ld_cg_u8(p); }
};

// Blocks per SM: 5 up to R = 4, 4 above (where the 16-byte two-vector
// variant holds R - 1 peer vectors per thread and would spill at 5).  Measured
// on a GB300, complex64 1000 x 500 shards in HBM: R=4 21.8 -> 20.3 us (against
// the unbounded build's 3 blocks per SM), R=8 64.9 -> 64.3 us, R=8 500 KB
// 12.0 -> 11.4 us.
// A (publish ahead, slots in HBM, several stages per block): a block
// publishes stage s + 1 -- loads its input, stores it into the slot and into
// its own place in out, raises the flag -- before it waits for and copies its
// peers' stage s, so each flag round overlaps the next stage's publish.  Stage
// s + 1 has its own slot region, so nothing a peer still reads is touched.
template <int VW, int R, int U, bool F, bool T, bool A>
__global__ void __launch_bounds__(kThreads, R <= 4 ? 5 : 4)
    allgather_kernel(const uint8_t *in_arg, uint8_t *out_arg, uint64_t bytes, int rank_arg, DevState d, RankIO io) {
    using V = typename Vec<VW>::T;
    __shared__ unsigned long long s_seq;
    __shared__ unsigned long long s_calls;
    __shared__ int s_bail;
    __shared__ TraceMarks s_tr;

    const int rank = block_rank<F>(rank_arg);
    const uint8_t *in = rank_ptr<R, F>(in_arg, io.in, rank);
    uint8_t *out = rank_ptr<R, F>(out_arg, io.out, rank);

    const int b = blockIdx.x;
    const int B = gridDim.x;
    const int tid = threadIdx.x;
    const uint64_t nv = bytes / VW;
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
    const V *src = reinterpret_cast<const V *>(in);
    V *dst = reinterpret_cast<V *>(out);

    V own[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint64_t v = (uint64_t)b * kTileVecs + (uint64_t)u * kThreads + tid;
        if (v < nv) own[u] = src[v];
    }
    __syncthreads();
    const unsigned long long seq = s_seq;
    const int parity = (int)(s_calls & 1ull);
    advance_idle_blocks(d, rank, s_calls + 1ull);
    const uint64_t slot_vecs = d.slot_bytes / VW;
    V *const slot_base = reinterpret_cast<V *>(d.slots) + (uint64_t)parity * R * slot_vecs;
    V *const my_slot = slot_base + (uint64_t)rank * slot_vecs;
    if (nstages) pace_first_stage(c0, b, d.pace_cycles);
    if (A && nstages) {
        // stage 0 published before the loop; the loop publishes one ahead
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = (uint64_t)b * kTileVecs + (uint64_t)u * kThreads + tid;
            if (v < nv) {
                my_slot[v] = own[u];
                dst[(uint64_t)rank * nv + v] = own[u];
            }
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
        V nxt[U];
        if constexpr (A) {
            // publish stage s + 1
            if (s + 1 < nstages) {
                const uint64_t vn = (tile + B) * kTileVecs + tid;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint64_t v = vn + (uint64_t)u * kThreads;
                    if (v < nv) nxt[u] = src[v];
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint64_t v = vn + (uint64_t)u * kThreads;
                    if (v < nv) {
                        my_slot[v] = nxt[u];
                        dst[(uint64_t)rank * nv + v] = nxt[u];
                    }
                }
                __syncthreads();
                if (tid == 0) publish_stage(d, rank, b, seq + s + 2);
            }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint64_t v = v0 + (uint64_t)u * kThreads;
                if (v < nv) {
                    my_slot[v] = own[u];
                    dst[(uint64_t)rank * nv + v] = own[u];
                }
            }
            __syncthreads();
            if (tid == 0) {
                publish_stage(d, rank, b, seq + s + 1);
                trace_published<T>(d, s_tr);
            }

            if (s + 1 < nstages) {
                const uint64_t vn = (tile + B) * kTileVecs + tid;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint64_t v = vn + (uint64_t)u * kThreads;
                    if (v < nv) nxt[u] = src[v];
                }
            }
        }

        if (wait_peers(d, R, rank, b, seq + s + 1, &s_bail)) return;
        if (tid == 0) trace_peers<T>(d, s_tr);
        // Every peer block of this call has now published its last stage, so
        // all of them are resident: this rank's next call may be scheduled.
        if (s + 1 == nstages) pdl_trigger();

#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = v0 + (uint64_t)u * kThreads;
            if (v < nv) {
                // peers in groups of 4: 4 loads in flight, a bounded register set
                constexpr int kChunk = 4;
#pragma unroll
                for (int p0 = 0; p0 < R; p0 += kChunk) {
                    V vals[kChunk];
#pragma unroll
                    for (int q = 0; q < kChunk; ++q) {
                        const int p = p0 + q;
                        if (p < R && p != rank) vals[q] = Vec<VW>::ldcg(slot_base + (uint64_t)p * slot_vecs + v);
                    }
#pragma unroll
                    for (int q = 0; q < kChunk; ++q) {
                        const int p = p0 + q;
                        if (p < R && p != rank) dst[(uint64_t)p * nv + v] = vals[q];
                    }
                }
            }
        }
        if (!A && s + 1 < nstages) {
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

// Bulk gather (slots in HBM, 16-byte vectors, untraced): the same protocol
// and the same publish (ordinary stores into the slot and into the rank's own
// place in out, one stage ahead, then the flag), but once the peers' flags of
// a stage are up thread 0 moves their tiles with bulk asynchronous copies:
// one cp.async.bulk per peer from its slot into shared memory, completing on
// an mbarrier, then one bulk store per peer from shared memory into its place
// in out.  The copies hold no registers, so a block has (R - 1) whole tiles in
// flight where its threads held four 16-byte vectors each.  Used from R = 5
// (measured on a GB300, complex64 1000 x 500 shards, graphs, us/call, bulk /
// per-thread gather: R = 8 55.8-55.9 / 58.0, in one launch of every rank
// 55.3 / 58.2; R = 4 18.2 / 18.1).  Storing each stage's tiles one stage
// later, so that the loads complete during the next flag round, measured R = 8
// 58.9 / 57.6 and R = 4 17.9 / 18.1 (one buffer: the next loads wait for the
// stores to have read it).
//  - The peers' slot stores are ordinary (generic-proxy) stores ordered by
//    their release and this block's acquire; thread 0 puts a proxy fence
//    between that acquire and its bulk (async-proxy) reads.
//  - Before a stage's bulk loads reuse the shared buffer, the previous stage's
//    bulk stores have finished reading it (wait_group.read).
//  - The mbarrier wait is bounded like the flag waits; thread 0 records a
//    wait that runs out (peer = its own rank: its own copies) and sets the
//    block's bail word, which the next flag wait returns to every thread, so
//    the whole block leaves together, after its bulk stores have completed.
//  - Before the block ends, all its bulk stores have completed (wait_group 0).
// Dynamic shared memory: (R - 1) * kThreads * U * 16 bytes.
__device__ __forceinline__ unsigned smem_addr(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }

template <int R, int U, bool F>
__global__ void __launch_bounds__(kThreads, R <= 4 ? 5 : 4)
    allgather_bulk_kernel(const uint8_t *in_arg, uint8_t *out_arg, uint64_t bytes, int rank_arg, DevState d,
                          RankIO io) {
    using V = uint4;
    extern __shared__ __align__(128) uint4 s_tiles[];  // [R - 1][kTileVecs]
    __shared__ __align__(8) unsigned long long s_mbar;
    __shared__ unsigned long long s_seq;
    __shared__ unsigned long long s_calls;
    __shared__ int s_bail;

    const int rank = block_rank<F>(rank_arg);
    const uint8_t *in = rank_ptr<R, F>(in_arg, io.in, rank);
    uint8_t *out = rank_ptr<R, F>(out_arg, io.out, rank);

    const int b = blockIdx.x;
    const int B = gridDim.x;
    const int tid = threadIdx.x;
    const uint64_t nv = bytes / 16;
    constexpr uint64_t kTileVecs = (uint64_t)kThreads * U;
    const uint64_t ntiles = (nv + kTileVecs - 1) / kTileVecs;
    const uint64_t nstages = ntiles > (uint64_t)b ? (ntiles - b + B - 1) / B : 0;
    const unsigned mbar = smem_addr(&s_mbar);

    pdl_wait();
    if (tid == 0) {
        const Ctr c = d.ctr[(size_t)rank * d.cmax + b];
        s_seq = c.seq;
        s_calls = c.calls;
        s_bail = 0;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const V *src = reinterpret_cast<const V *>(in);
    V *dst = reinterpret_cast<V *>(out);
    V nxt[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint64_t v = (uint64_t)b * kTileVecs + (uint64_t)u * kThreads + tid;
        if (v < nv) nxt[u] = src[v];
    }
    __syncthreads();
    const unsigned long long seq = s_seq;
    const int parity = (int)(s_calls & 1ull);
    advance_idle_blocks(d, rank, s_calls + 1ull);
    const uint64_t slot_vecs = d.slot_bytes / 16;
    V *const slot_base = reinterpret_cast<V *>(d.slots) + (uint64_t)parity * R * slot_vecs;
    V *const my_slot = slot_base + (uint64_t)rank * slot_vecs;

    // publish stage s (tile b + s * B) from nxt; the flag goes to seq + s + 1
    auto publish = [&](uint64_t s) {
        const uint64_t v0 = ((uint64_t)b + s * B) * kTileVecs + tid;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = v0 + (uint64_t)u * kThreads;
            if (v < nv) {
                my_slot[v] = nxt[u];
                dst[(uint64_t)rank * nv + v] = nxt[u];
            }
        }
        __syncthreads();
        if (tid == 0) publish_stage(d, rank, b, seq + s + 1);
    };
    if (nstages) publish(0);

    for (uint64_t s = 0; s < nstages; ++s) {
        const uint64_t tile = (uint64_t)b + s * B;
        const uint64_t v0 = tile * kTileVecs;
        if (s + 1 < nstages) {
            const uint64_t vn = (tile + B) * kTileVecs + tid;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint64_t v = vn + (uint64_t)u * kThreads;
                if (v < nv) nxt[u] = src[v];
            }
            publish(s + 1);
        }
        if (wait_peers(d, R, rank, b, seq + s + 1, &s_bail)) break;
        if (s + 1 == nstages) pdl_trigger();
        if (tid == 0) {
            const uint64_t nvec = nv - v0 < kTileVecs ? nv - v0 : kTileVecs;
            const unsigned nbytes = (unsigned)(nvec * 16);
            // the previous stage's bulk stores have read the buffer
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            // the peers' slot stores, acquired through their flags, before the bulk reads
            asm volatile("fence.proxy.async.global;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar),
                         "r"(nbytes * (unsigned)(R - 1))
                         : "memory");
            int j = 0;
#pragma unroll
            for (int p = 0; p < R; ++p) {
                if (p == rank) continue;
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_addr(s_tiles + (uint64_t)j * kTileVecs)),
                    "l"(slot_base + (uint64_t)p * slot_vecs + v0), "r"(nbytes), "r"(mbar)
                    : "memory");
                ++j;
            }
            // wait for this stage's phase (bounded by the handle's timeout)
            const unsigned ph = (unsigned)(s & 1ull);
            const unsigned long long t0 = global_timer_ns();
            unsigned done = 0;
            for (unsigned it = 0; !done; ++it) {
                asm volatile(
                    "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                    : "=r"(done)
                    : "r"(mbar), "r"(ph)
                    : "memory");
                if (!done && (it & 255u) == 255u && global_timer_ns() - t0 > d.timeout_ns) break;
            }
            if (!done) {
                record_timeout(d, rank, b, rank, seq + s + 1, 0);
                s_bail = 1;
            } else {
                j = 0;
#pragma unroll
                for (int p = 0; p < R; ++p) {
                    if (p == rank) continue;
                    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                                     dst + (uint64_t)p * nv + v0),
                                 "r"(smem_addr(s_tiles + (uint64_t)j * kTileVecs)), "r"(nbytes)
                                 : "memory");
                    ++j;
                }
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        }
    }

    if (tid == 0) {
        // every bulk store of this block has completed before it ends
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        if (!s_bail) {
            Ctr c;
            c.seq = seq + nstages;
            c.calls = s_calls + 1;
            d.ctr[(size_t)rank * d.cmax + b] = c;
        }
    }
}

template <int VW, int U, bool F, bool T, bool A>
const void *allgather_ptr_ru(int R) {
    switch (R) {
        case 1: return (const void *)allgather_kernel<VW, 1, U, F, T, A>;
        case 2: return (const void *)allgather_kernel<VW, 2, U, F, T, A>;
        case 3: return (const void *)allgather_kernel<VW, 3, U, F, T, A>;
        case 4: return (const void *)allgather_kernel<VW, 4, U, F, T, A>;
        case 5: return (const void *)allgather_kernel<VW, 5, U, F, T, A>;
        case 6: return (const void *)allgather_kernel<VW, 6, U, F, T, A>;
        case 7: return (const void *)allgather_kernel<VW, 7, U, F, T, A>;
        case 8: return (const void *)allgather_kernel<VW, 8, U, F, T, A>;
        default: return nullptr;
    }
}

// The publish-ahead kernels exist for 16- and 8-byte vectors, untraced; any
// other request for them takes the plain kernel.
template <int VW, bool F, bool T>
const void *allgather_ptr_rft(int R, int U) {
    const int u = oneshot_unroll(U);
    if constexpr (!T && VW >= 8) {
        if (oneshot_ahead(U))
            return u == 1 ? allgather_ptr_ru<VW, 1, F, false, true>(R) : allgather_ptr_ru<VW, 2, F, false, true>(R);
    }
    return u == 1 ? allgather_ptr_ru<VW, 1, F, T, false>(R) : allgather_ptr_ru<VW, 2, F, T, false>(R);
}

template <int VW>
const void *allgather_ptr_r(int R, int U, bool fused, bool traced) {
    if (traced) return fused ? allgather_ptr_rft<VW, true, true>(R, U) : allgather_ptr_rft<VW, false, true>(R, U);
    return fused ? allgather_ptr_rft<VW, true, false>(R, U) : allgather_ptr_rft<VW, false, false>(R, U);
}

template <int U, bool F>
const void *allgather_bulk_ptr(int R) {
    switch (R) {
        case 1: return (const void *)allgather_bulk_kernel<1, U, F>;
        case 2: return (const void *)allgather_bulk_kernel<2, U, F>;
        case 3: return (const void *)allgather_bulk_kernel<3, U, F>;
        case 4: return (const void *)allgather_bulk_kernel<4, U, F>;
        case 5: return (const void *)allgather_bulk_kernel<5, U, F>;
        case 6: return (const void *)allgather_bulk_kernel<6, U, F>;
        case 7: return (const void *)allgather_bulk_kernel<7, U, F>;
        case 8: return (const void *)allgather_bulk_kernel<8, U, F>;
        default: return nullptr;
    }
}

}  // namespace

const void *allgather_kernel_ptr(int vec_bytes, int R, int unroll, bool fused, bool traced) {
    if (allgather_bulk(unroll)) {
        // 16-byte vectors, untraced only
        if (vec_bytes != 16 || traced) return nullptr;
        const int u = allgather_bulk_unroll(unroll);
        if (u == 1) return fused ? allgather_bulk_ptr<1, true>(R) : allgather_bulk_ptr<1, false>(R);
        if (u == 2) return fused ? allgather_bulk_ptr<2, true>(R) : allgather_bulk_ptr<2, false>(R);
        return nullptr;
    }
    switch (vec_bytes) {
        case 16: return allgather_ptr_r<16>(R, unroll, fused, traced);
        case 8: return allgather_ptr_r<8>(R, unroll, fused, traced);
        case 4: return allgather_ptr_r<4>(R, unroll, fused, traced);
        case 2: return allgather_ptr_r<2>(R, unroll, fused, traced);
        case 1: return allgather_ptr_r<1>(R, unroll, fused, traced);
        default: return nullptr;
    }
}

cudaError_t launch_allgather(int vec_bytes, int R, int unroll, int blocks, cudaStream_t s,
                             const RankIO &io, uint64_t bytes, int rank, const DevState &d, bool pdl) {
    const void *k = allgather_kernel_ptr(vec_bytes, R, unroll, rank < 0, d.trace != nullptr);
    if (!k) return cudaErrorInvalidValue;
    const size_t smem = allgather_bulk(unroll) ? (size_t)allgather_bulk_smem(R, allgather_bulk_unroll(unroll)) : 0;
    const uint8_t *a0 = static_cast<const uint8_t *>(io.in[0]);
    uint8_t *a1 = static_cast<uint8_t *>(io.out[0]);
    uint64_t a2 = bytes;
    int a3 = rank;
    DevState a4 = d;
    RankIO a5 = io;
    void *args[] = {&a0, &a1, &a2, &a3, &a4, &a5};
    return launch(k, blocks, rank < 0 ? R : 1, rank < 0, s, args, pdl, smem);
}

}  // namespace tda
