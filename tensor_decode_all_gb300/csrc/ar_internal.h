// ar_internal.h -- declarations shared by the library's translation units.
//
// Memory layout of one handle (all addresses as seen by the GPU):
//   slots : [2 parities][R ranks][slot_bytes]        pinned host or HBM
//   flags : [R ranks][bmax blocks] x 128 B lines     HBM; for pinned-host slots also a
//           copy in mapped host memory, and the gpu_scope tactic picks which one
//           a call uses; word 0 of each line is the flag, a 64-bit count of
//           published stages
//   ctr   : [R ranks][cmax blocks] x {seq, calls}    HBM; private to one block (cmax >= bmax)
//   abort : one 32-bit word in HBM, non-zero once any block has given up
//   err   : one ar_error_info in mapped pinned host memory
//   ll    : [2 parities][R ranks][ll_vecs] x 16 B   same memory as the slots; the
//           tagged-word form's exchange buffers (8 payload bytes per 16 B)
//   push  : [2 parities][R readers][R writers][slot_bytes]  same memory as the
//           slots; the push form's receive areas, allocated when the form is
//           first selected, with flags [R][R][bmax] x 128 B lines
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ar.h"

namespace tda {

constexpr int kMaxRanks = 8;
constexpr int kThreads = 256;           // threads per block of the exchange kernels (>= 64: see kPollWarp)
constexpr int kFlagStrideWords = 16;    // 16 x 8 B = one 128-byte line per flag
constexpr uint64_t kSlotAlign = 256;
// Counter slots per rank: at least this many, so a cluster-form call can run
// up to this many single-stage clusters (in waves) whatever the flag grids are.
constexpr int kCounterSlots = 512;
// Kernel variant codes for the two-shot form: a negative "unroll" whose
// magnitude is the sub-tile size in vectors (256, 128 or 64), plus one for the
// kernel that merges each reduced sub-tile into the next tile's flag round.
constexpr int twoshot_variant(int sub, bool merged = false) { return -(sub + (merged ? 1 : 0)); }
constexpr int twoshot_sub(int variant) { return (-variant) & ~1; }
constexpr bool twoshot_merged(int variant) { return ((-variant) & 1) != 0; }
// Kernel variant codes of the one-shot form: its vectors per thread per stage
// (1 or 2), plus 4 for the kernel that publishes one stage ahead.
constexpr int oneshot_ahead_variant(int unroll) { return 4 + unroll; }
constexpr int oneshot_unroll(int variant) { return variant > 4 ? variant - 4 : variant; }
constexpr bool oneshot_ahead(int variant) { return variant > 4; }
// Kernel variant codes of the allgather's bulk-gather kernel (slots in HBM,
// 16-byte vectors, untraced): its vectors per thread per stage, plus 8.
constexpr int allgather_bulk_variant(int unroll) { return 8 + unroll; }
constexpr bool allgather_bulk(int variant) { return variant > 8; }
constexpr int allgather_bulk_unroll(int variant) { return variant - 8; }
// Its dynamic shared memory: one tile of every peer.
constexpr uint64_t allgather_bulk_smem(int R, int unroll) {
    return (uint64_t)(R > 1 ? R - 1 : 0) * (uint64_t)kThreads * (uint64_t)unroll * 16ull;
}
// Kernel variant code of the tagged-word form.
constexpr int kTaggedVariant = 0;
// Kernel variant code of the push form.
constexpr int kPushVariant = 3;

// Per-(rank, block) counters.  `seq` counts the stages this block has
// published over all calls (its flag's value at the end of the last call);
// `calls` counts the calls it took part in, whose parity picks the slot buffer.
struct Ctr {
    unsigned long long seq;
    unsigned long long calls;
};

// Everything a rank's kernel needs besides its own in/out pointers.  Passed
// by value as a kernel argument (captured graphs keep a copy).
struct DevState {
    uint8_t *slots;            // [2][R][slot_bytes]
    unsigned long long *flags; // [R][bmax][kFlagStrideWords]
    Ctr *ctr;                  // [R][bmax]
    unsigned int *abort_word;  // sticky, HBM
    ar_error_info *err;        // device alias of mapped host memory
    uint64_t slot_bytes;
    uint64_t timeout_ns;
    int bmax;                  // flag slots per rank (the largest grid of a flag-protocol launch)
    int sys_scope;             // 1: the ranks synchronise at system scope (flags in host memory, the pages'
                               // two-GPU case); 0: at GPU scope (flags in HBM; slots in either memory)
    ulonglong2 *ll;            // [2][R][ll_vecs] tagged-word buffers (same memory as the slots)
    uint64_t ll_vecs;          // 16-byte tagged vectors per rank and parity: 2 per 16 payload bytes
    ar_trace_record *trace;    // [depth][R][bmax] or null (tracing off)
    uint32_t trace_depth;
    int32_t algo;              // AR_ALGO_* of this launch, for the trace
    int cmax;                  // counter slots per rank (>= bmax; cluster-form grids may use them all)
    uint8_t *push;             // push form: [2][R reader][R writer][slot_bytes] receive areas, or null
    unsigned long long *push_flags;  // push form: [R reader][R writer][bmax][kFlagStrideWords]
    uint32_t pace_cycles;      // block b starts its first stage's slot stores b * pace_cycles SM cycles
                               // after its start (0: at once); see the pacing tactic
};

// The input and output pointers of every rank, passed by value to a launch
// of all R ranks at once (grid blocks x R; block (b, r) plays block b of rank
// r with in[r] / out[r]).  A launch for one rank passes its own pointers as
// separate arguments, and its kernel ignores this.
struct RankIO {
    void *in[kMaxRanks];   // read only
    void *out[kMaxRanks];
};

// Launch kernel k on s with kThreads threads a block and a grid of `blocks`
// (one rank) or blocks x ranks (all ranks, ranks > 1 or a negative rank
// argument): the latter as a cooperative launch, so that the runtime either
// makes every block resident at once or refuses the launch.  With pdl, as a
// programmatic dependent of the preceding work on s.
cudaError_t launch(const void *k, int blocks, int ranks, bool cooperative, cudaStream_t s, void **args,
                   bool pdl, size_t smem = 0);

// Launchers (one per kernel family).  rank >= 0: that rank's kernel, `blocks`
// blocks; rank < 0: all R ranks in one cooperative grid of blocks x R.
// Return cudaSuccess or the launch error.
cudaError_t launch_allreduce(int dtype, int R, int unroll, int blocks, cudaStream_t s,
                             const RankIO &io, uint64_t numel, int rank, const DevState &d, bool pdl);
cudaError_t launch_allgather(int vec_bytes, int R, int unroll, int blocks, cudaStream_t s,
                             const RankIO &io, uint64_t bytes, int rank, const DevState &d, bool pdl);

// Kernel entry addresses, for launches and occupancy queries.  fused: the
// kernel built for one launch of all ranks (grid blocks x R) rather than one
// rank's launch; traced: the kernel that writes trace records.
const void *allreduce_kernel_ptr(int dtype, int R, int unroll, bool fused, bool traced);
const void *allreduce_kernel_ptr_f16(int R, int unroll, bool fused, bool traced);   // ar_allreduce_f16.cu
const void *allreduce_kernel_ptr_bf16(int R, int unroll, bool fused, bool traced);  // ar_allreduce_bf16.cu
const void *allreduce_twoshot_kernel_ptr_f16(int R, int unroll, bool fused, bool traced);   // ..._f16_twoshot.cu
const void *allreduce_twoshot_kernel_ptr_bf16(int R, int unroll, bool fused, bool traced);  // ..._bf16_twoshot.cu
const void *allgather_kernel_ptr(int vec_bytes, int R, int unroll, bool fused, bool traced);
// Cluster-barrier form (all ranks in one launch, clusters of 1 x R blocks):
// sub = 0 one-shot, 64/128/256 two-shot sub-tile.
// paced: the kernel with the code that paces the first stage's slot stores.
const void *allreduce_cluster_kernel_ptr(int dtype, int R, int sub, bool traced, bool paced = false);
const void *allreduce_cluster_kernel_ptr_f16(int R, int sub, bool traced, bool paced);   // ar_allreduce_f16_cluster.cu
const void *allreduce_cluster_kernel_ptr_bf16(int R, int sub, bool traced, bool paced);  // ar_allreduce_bf16_cluster.cu
// Launch the cluster form: grid blocks x R, clusters of 1 x R, not cooperative
// (a cluster waits only on itself).
cudaError_t launch_allreduce_cluster(int dtype, int R, int sub, int blocks, cudaStream_t s, const RankIO &io,
                                     uint64_t numel, const DevState &d, bool pdl);

}  // namespace tda
