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

}  // namespace

const void *allgather_kernel_ptr(int vec_bytes, int R, int unroll, bool fused, bool traced) {
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
    const uint8_t *a0 = static_cast<const uint8_t *>(io.in[0]);
    uint8_t *a1 = static_cast<uint8_t *>(io.out[0]);
    uint64_t a2 = bytes;
    int a3 = rank;
    DevState a4 = d;
    RankIO a5 = io;
    void *args[] = {&a0, &a1, &a2, &a3, &a4, &a5};
    return launch(k, blocks, rank < 0 ? R : 1, rank < 0, s, args, pdl);
}

}  // namespace tda
