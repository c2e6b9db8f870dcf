/*
 * ar.h -- C ABI of the logical-rank all-reduce / allgather library (libtda_ar.so).
 *
 * R "logical ranks" share one GPU.  Each rank is a kernel launched on its own
 * non-blocking stream; the R kernels of one call run at the same time and meet
 * through a shared, double-buffered slot and per-block flags.  The operation
 * is the flag-synchronised exchange-and-add of "[Kernel] Two-rank FP16
 * all-reduce through pinned host memory for GPUs without P2P", section
 * "Purpose": a block publishes its share of the data in a shared
 * slot, makes it visible before it sets its own flag, and sums once it has seen
 * the flags of the matching blocks of the other ranks, rounding a single time;
 * consecutive calls use the two halves of the slot in turn; the host only
 * enqueues kernels and never waits, so the calls can be captured in CUDA graphs.
 * That page is about two ranks; this library takes 1 <= R <= 8 and sums in
 * rank order 0..R-1 on every rank (the order matters from three ranks on:
 * "[SM120] Add optional FlashInfer PCIe-IPC all-reduce for switch-free hosts",
 * section "Accuracy").
 *
 * Conventions for every entry point:
 *   - Pointers named in/out are device-accessible addresses (cudaMalloc'd or
 *     mapped pinned host memory) owned by the caller, 16-byte aligned.
 *   - `stream` is a cudaStream_t created with cudaStreamNonBlocking, owned by
 *     the caller.  The legacy default stream, the per-thread default stream and
 *     blocking streams are refused (AR_ESTREAM): a stream that serialises with
 *     the legacy stream can hold back a peer rank's kernel while this rank's
 *     kernel waits for it ("fix(group): run each rank on a non-blocking
 *     stream", sections "What" and "Why").
 *   - Return value: AR_OK (0) or an ar_code below.  An enqueue call that
 *     returns AR_ECUDA because its launch failed is not counted as a call of
 *     its rank (the other ranks' kernels of that call, if they were enqueued,
 *     time out: reset the handle).  A call that returns an
 *     error other than AR_ECUDA has enqueued nothing, so the caller can keep
 *     its own fallback path ("[SM120] Add optional FlashInfer PCIe-IPC
 *     all-reduce for switch-free hosts", section "Modifications": a shape the
 *     backend cannot take is reported and the caller keeps NCCL).
 *   - Errors found on the device (a peer that never arrives) cannot be
 *     returned by the enqueueing call; they are recorded in the handle and read
 *     with ar_status() after the caller has synchronised.
 *   - Host threads: the enqueue calls of different ranks may come from
 *     different threads at the same time (one thread per rank, each on its own
 *     stream).  The calls that change a handle's settings (ar_set_algo,
 *     ar_set_tactics, ar_set_trace, ar_set_pdl, ar_set_timeout), ar_reset and
 *     ar_destroy must not run concurrently with any other call on the handle.
 */
#ifndef TDA_AR_H
#define TDA_AR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define AR_API __attribute__((visibility("default")))
#else
#define AR_API
#endif

/* A CUDA stream handle (identical to cudaStream_t), spelled without CUDA headers. */
typedef struct CUstream_st *ar_stream_t;

typedef struct ar_handle ar_handle;

/* Element types.  AR_F16 = IEEE binary16, AR_BF16 = bfloat16 (all-reduce and
 * allgather); AR_C64 = complex64, two binary32 (allgather only: the pages
 * gather complex64 tensors and never reduce them). */
enum ar_dtype { AR_F16 = 1, AR_BF16 = 2, AR_C64 = 3 };

/* Where the shared slots live.
 * AR_SLOT_PINNED_HOST: page-locked host memory mapped into the GPU
 *   (cudaHostAlloc mapped|portable), as on the pages, where two GPUs without
 *   peer access both map it ("[Kernel] Two-rank FP16 all-reduce through pinned
 *   host memory for GPUs without P2P", section "Purpose").  The per-block
 *   flags are in HBM with GPU-scope release/acquire by default, or in mapped
 *   host memory with system-scope release/acquire (ar_tactics.gpu_scope = 0).
 * AR_SLOT_HBM: device memory of this GPU; flags in HBM, GPU-scope
 *   release/acquire. */
enum ar_slot_kind { AR_SLOT_PINNED_HOST = 0, AR_SLOT_HBM = 1 };

enum ar_code {
    AR_OK = 0,
    AR_EINVAL = 1,    /* bad handle, rank, R, dtype, slot kind, NULL or misaligned pointer,
                         wrong current device, or an operation the handle's dtype lacks */
    AR_ETOOBIG = 2,   /* numel > max_numel: declined, nothing enqueued; the workspace
                         cannot grow after ar_create ("[SM120] Add optional FlashInfer
                         PCIe-IPC all-reduce for switch-free hosts", section "Modifications") */
    AR_ESTREAM = 3,   /* NULL, legacy, per-thread-default or blocking stream, or the same
                         stream as another rank's pending call of the same sequence number */
    AR_ENOMEM = 4,    /* slot, flag or counter allocation failed in ar_create */
    AR_ECUDA = 5,     /* a CUDA runtime call failed (launch error, no device, ...) */
    AR_ETIMEOUT = 6,  /* recorded on the device: a block waited longer than the timeout for
                         a peer's flag (or tagged words).  Outputs of that call and of every
                         later call are undefined until ar_reset(). */
    AR_ESTATE = 7     /* the handle needs ar_reset() (a device error is recorded) */
};

/* How an all-reduce call moves its data (all give the same bits).
 * AR_ALGO_ONESHOT: one flag round per tile; every rank reads every peer's tile
 *   (the pages' exchange-and-add).  Per call, peer-slot reads are R*(R-1)*S.
 * AR_ALGO_TWOSHOT: two flag rounds per tile; rank r reduces the r-th sub-tile
 *   for everyone, then every rank copies the R reduced sub-tiles.  Per call,
 *   slot reads are about 2*R*S; for large payloads at R >= 4.
 * AR_ALGO_TAGGED: no flags and no fences; every 8-byte word of a separate
 *   exchange buffer holds 4 payload bytes and a 4-byte tag naming the stage,
 *   and a reader polls its peers' words until the tags match.  One trip over
 *   the slot memory instead of three, at twice the bytes: for latency-bound
 *   calls of one tile (4 KiB) per block, up to ar_info.tagged_capacity_bytes
 *   per rank (larger calls take the one-shot form).  Not part of the pages'
 *   design.
 * AR_ALGO_CLUSTER: for calls that launch every rank at once (ar_allreduce_fused,
 *   ar_allreduce_all) only: block b of every rank forms one thread-block cluster
 *   and the hardware cluster barrier (arrive with release, wait with acquire)
 *   takes the place of the per-block flags; the data moves through the same
 *   slots, one-shot or two-shot by size (ar_tactics.cluster_twoshot_min_bytes).
 *   Valid because the ranks are logical ranks on one GPU; per-rank calls on a
 *   handle set to it take the AR_ALGO_AUTO rule.  Not part of the pages' design.
 * AR_ALGO_PUSH: writers store their tile into a receive area of every peer, one
 *   peer after another, and each reader sums its own area; one flag per
 *   (reader, writer, block) ("[SM120] Add optional FlashInfer PCIe-IPC all-reduce
 *   for switch-free hosts", section "Motivation").  On one GPU every area is in
 *   the same memory, so it writes R - 1 times the pull form's slot bytes; kept
 *   for measurement, never chosen by AUTO.  Its receive areas (2 * R * R *
 *   slot_bytes, in the slots' kind of memory) are allocated when ar_set_algo
 *   first selects it.
 * AR_ALGO_AUTO: chosen per call from the handle's tactics (ar_tactics). */
enum ar_algo {
    AR_ALGO_AUTO = -1,
    AR_ALGO_ONESHOT = 0,
    AR_ALGO_TWOSHOT = 1,
    AR_ALGO_TAGGED = 2,
    AR_ALGO_CLUSTER = 3,
    AR_ALGO_PUSH = 4
};

/* Details of the first device-side error recorded in a handle. */
typedef struct ar_error_info {
    int32_t code;       /* AR_OK or AR_ETIMEOUT */
    int32_t rank;       /* rank whose block gave up waiting */
    int32_t block;      /* that block's index */
    int32_t peer;       /* the first peer whose flag (or tagged word) had not arrived */
    uint64_t want;      /* flag value (stage count) the block waited for */
    uint64_t seen;      /* flag value it last saw (0 for tagged words) */
} ar_error_info;

/* One trace record: one block of one rank in one call (see ar_set_trace).
 * Times from %globaltimer (ns, the same clock on every SM) at the start and
 * end of the block's work; phase marks in SM clock cycles after the start. */
typedef struct ar_trace_record {
    int32_t rank;
    int32_t block;
    uint32_t call;          /* the rank's call count before this call (the same for every block) */
    uint32_t stages;        /* stages the block ran in this call */
    uint64_t t_start_ns;    /* after the wait for the preceding work on the stream */
    uint64_t t_end_ns;      /* after the block's last output store; 0: record not written */
    uint32_t cyc_published; /* first stage: this block's data published (flag raised) */
    uint32_t cyc_peers;     /* first stage: every peer's data of that stage seen */
    uint32_t cyc_end;       /* last output store */
    uint32_t algo;          /* AR_ALGO_* of the call (allgather: AR_ALGO_ONESHOT) */
} ar_trace_record;

/* Static facts about a handle, for tests and tools. */
typedef struct ar_info {
    int32_t R, dtype, slot_kind, device;
    int32_t threads;        /* threads per block of the exchange kernels */
    int32_t max_blocks;     /* flag/counter slots per rank: an upper bound on blocks per rank */
    int32_t sm_count;
    int32_t blocks_per_sm;  /* occupancy of the one-shot all-reduce kernels */
    int32_t blocks_per_sm_twoshot;   /* ... of the two-shot all-reduce kernels */
    int32_t blocks_per_sm_allgather; /* ... of the allgather kernels */
    int32_t algo;           /* AR_ALGO_AUTO unless forced with ar_set_algo */
    int32_t pdl;            /* 1 if calls launch as programmatic dependents (ar_set_pdl) */
    uint64_t max_numel;
    uint64_t slot_bytes;    /* bytes of one (parity, rank) slot, a multiple of 256 */
    uint64_t total_slot_bytes; /* 2 * R * slot_bytes: the allocation that cannot grow */
    uint64_t timeout_ns;
    uint64_t tagged_capacity_bytes;  /* largest per-rank call the tagged form takes (one 4 KiB tile per
                                        block of one rank's launch, within the slot; 0: complex64) */
    int32_t blocks_per_sm_tagged;    /* occupancy of the tagged-form kernels */
    int32_t cluster_form;            /* clusters of R blocks of the cluster form (AR_ALGO_CLUSTER) the GPU
                                        holds at once (a call launches at most that many); 0: the form
                                        cannot run here */
} ar_info;

/* Launch plan of one call, computed on the host (no GPU needed). */
typedef struct ar_plan {
    int32_t blocks;         /* grid size per rank (same on every rank); R * blocks fit on the GPU */
    int32_t threads;        /* threads per block */
    int32_t vec_bytes;      /* bytes per vector access: 16 for all-reduce */
    int32_t unroll;         /* vectors per thread per tile (two-shot: R * subtile_vecs / threads, rounded up) */
    int32_t algo;           /* AR_ALGO_ONESHOT, _TWOSHOT or _TAGGED (allgather: one-shot) */
    int32_t flag_rounds;    /* flag rounds of a block with one tile: 1 or 2 (a two-shot block with n tiles
                               waits n + 1 times: each reduced sub-tile rides on the next tile's round) */
    int32_t subtile_vecs;   /* two-shot: vectors per sub-tile (64, 128 or 256; a tile is R sub-tiles); else 0 */
    int32_t pace_cycles;    /* SM cycles between the first-stage slot stores of consecutive blocks (the
                               pace_mbs tactics, slots in host memory); 0: all at once.  ar_plan_for
                               only, for inputs in device memory (zero-copy calls run unpaced); ar_plan_compute leaves it 0 */
    uint64_t tile_bytes;    /* bytes a block handles per stage (threads * unroll * vec_bytes) */
    uint64_t tiles;         /* ceil(bytes / tile_bytes); tile t goes to block t % blocks, stage t / blocks */
    uint64_t max_stages;    /* stages of block 0 = ceil(tiles / blocks) */
} ar_plan;

/* Per-handle tactics: which all-reduce form AR_ALGO_AUTO picks by size, and the
 * launch shape.  ar_create fills them from the built-in table (ar_choose_algo;
 * tagged_max_bytes 0 for complex64 handles);
 * ar_set_tactics replaces them, for instance with values measured on this GPU
 * and stored by the caller (the Python package's tune module does both). */
typedef struct ar_tactics {
    uint64_t twoshot_min_bytes; /* AUTO picks two-shot from this many bytes per rank; UINT64_MAX: never */
    int32_t twoshot_sub;        /* two-shot sub-tile in vectors (both two-shot forms): 64, 128 or 256;
                                   0 = the size rule */
    int32_t max_blocks;         /* cap on blocks per rank (>= 1); 0 = as many as fit (occupancy) */
    uint64_t tagged_max_bytes;  /* AUTO picks the tagged form up to this many bytes per rank; 0: never */
    uint64_t cluster_twoshot_min_bytes; /* cluster form: two-shot from this many bytes per rank; UINT64_MAX:
                                           never (one-shot) */
    uint64_t cluster_max_bytes; /* under AUTO, a launch of every rank at once takes the cluster form up to
                                   this many bytes per rank, the flag forms above it; 0: never */
    int32_t all_fused;          /* ar_allreduce_all: 1 = one launch of every rank; 0 = one launch per rank */
    int32_t pace_mbs;           /* slots in host memory: the rate (MB/s) at which a call's slot traffic,
                                   stores and the peers' loads together, is to cross the host link, for
                                   calls of one stage per block.  The first stage's slot stores of block
                                   b of every rank start b * R * tile_bytes / (pace * share) after the
                                   block starts, share = the paced stores' part of the traffic (1/R one-
                                   shot, 1/3 two-shot, 1/R allgather), so the stores reach the link about
                                   as fast as it drains them rather than all at once.  One-shot, two-shot
                                   and cluster all-reduce forms (the cluster form only when all its
                                   clusters are resident at once) and the allgather.  0 = all at once; otherwise >= 1000.  Default 356000 for
                                   pinned-host handles; ignored for HBM.  Calls whose inputs are in
                                   mapped host memory (zero copy) run unpaced: their input loads cross
                                   the link first and stagger the stores already.  Timing only:
                                   the results do not change */
    uint64_t pace_min_bytes;    /* pace only calls of at least this many bytes per rank (default 128 KiB) */
    int32_t pace_multi_mbs;     /* as pace_mbs, for calls of several stages per block (default 220000) */
    int32_t gpu_scope;          /* slots in host memory: the scope at which the ranks synchronise.  1 = GPU
                                   scope: the per-block flags in HBM, raised and read with GPU-scope
                                   release/acquire, and the tagged words and push flags (in host memory)
                                   read and written at GPU scope -- the R ranks are kernels of one GPU, so
                                   GPU scope holds every thread that observes them.  0 = system scope,
                                   flags in mapped host memory, as two GPUs that share only the host
                                   buffer need ("[Kernel] Two-rank FP16 all-reduce through pinned host
                                   memory for GPUs without P2P", section "Purpose").  The slot data stays
                                   in host memory either way, so every payload byte still crosses the
                                   host link; results are the same.  Default 1.  Always 1 for HBM handles
                                   (0 refused there) */
} ar_tactics;

/*
 * ar_create -- allocate a handle for R logical ranks.
 *
 * R in [1, 8]; dtype an ar_dtype; max_numel >= 1 elements per rank; slot_kind an
 * ar_slot_kind.  Allocates, owned by the library until ar_destroy():
 *   slots   [2 parities][R ranks][slot_bytes], slot_bytes = round_up(max_numel *
 *           itemsize, 256), in pinned host or HBM memory per slot_kind.  The size
 *           is fixed here and cannot grow: the cost law is 2 * R * max_numel *
 *           itemsize, as for the workspace in "[SM120] Add optional FlashInfer
 *           PCIe-IPC all-reduce for switch-free hosts", section "Modifications";
 *   flags   one 64-bit flag per (rank, block), each on its own 128-byte line, in
 *           HBM, and for pinned-host slots a second set in mapped host memory
 *           (used when ar_tactics.gpu_scope is 0);
 *   counters one 64-bit stage counter and one 64-bit call counter per (rank,
 *           block), in device memory: the call parity that picks the slot buffer
 *           comes from them, never from the host, so captured graphs replay
 *           correctly.
 * All of it starts at zero.  Uses the current CUDA device, which every later
 * call must also have current.  Returns NULL on failure; ar_last_error() then
 * gives the code (AR_EINVAL, AR_ENOMEM or AR_ECUDA).
 * The wait timeout starts at 1 s, or at the value of the environment variable
 * AR_SPIN_TIMEOUT_NS if set (bounded device spin: "fix(qwen3): re-enable CUDA
 * Graph under TP via startup decode-graph pre-capture",
 * section "Description": without one, a wedged rank waits forever).
 */
AR_API ar_handle *ar_create(int R, int dtype, size_t max_numel, int slot_kind);

/* Code of the last failed ar_create() on this thread (AR_OK if none). */
AR_API int ar_last_error(void);

/*
 * ar_allreduce -- enqueue rank `rank`'s part of one all-reduce on `stream`.
 *
 * in:  numel elements of the handle's dtype (AR_F16 or AR_BF16), contiguous,
 *      16-byte aligned, device-accessible, owned by the caller.
 * out: numel elements, same rules; out == in is allowed (in place), any other
 *      overlap is not.
 * After all R ranks have enqueued their call with the same numel and their
 * streams have run it, every out_r[i] holds
 *     RNE( f32(x_0[i]) + f32(x_1[i]) + ... + f32(x_{R-1}[i]) )
 * with binary32 additions left to right in rank order and one rounding to the
 * dtype: the same bits on every rank.
 * Contract between ranks: every rank 0..R-1 issues the same sequence of calls on
 * this handle with the same numel, each rank on its own non-blocking stream,
 * and the R kernels of a call must be able to run at the same time (they wait
 * for each other on the device).  No host synchronisation and no CPU work is
 * done: the call may be captured into a CUDA graph (all R ranks' calls in the
 * same graph, or graphs launched together).
 * numel == 0 enqueues nothing and returns AR_OK.
 * Errors: AR_EINVAL, AR_ETOOBIG, AR_ESTREAM, AR_ESTATE (a device error is
 * recorded: call ar_reset first), AR_ECUDA (launch failed).
 */
AR_API int ar_allreduce(ar_handle *h, int rank, const void *in, void *out, size_t numel,
                        ar_stream_t stream);

/*
 * ar_allgather -- enqueue rank `rank`'s part of one allgather on `stream`.
 *
 * in:  numel elements of the handle's dtype (any dtype; AR_C64 is the pages'
 *      case, the complex64 S_j and core uploads of "fix(group): run each rank
 *      on a non-blocking stream", section "Why"), 16-byte aligned.
 * out: R * numel elements: after the call every rank's out holds shard 0, then
 *      shard 1, ..., then shard R-1 (rank-major concatenation), bit for bit.
 *      out must not overlap in.
 * Same contract between ranks, errors and graph rules as ar_allreduce.
 */
AR_API int ar_allgather(ar_handle *h, int rank, const void *in, void *out, size_t numel,
                        ar_stream_t stream);

/*
 * ar_allreduce_fused / ar_allgather_fused -- one call of every rank at once,
 * as a single launch on one stream.  Same operation, same bits and same
 * handle state as R per-rank calls: ins[r] and outs[r] (host arrays of R
 * device pointers, owned by the caller, each following the per-rank call's
 * rules) are rank r's in and out.  The launch is cooperative, a grid of
 * B x R blocks in which block (b, r) plays block b of rank r: the runtime
 * either makes all R ranks' blocks resident together or refuses the launch
 * (AR_ECUDA), so the ranks' waits for each other never depend on separate
 * launches being scheduled side by side.  The pages run one rank per GPU and
 * have no such form; on one GPU it is the co-resident way to run the ranks.
 * Per-rank and fused calls may alternate on one handle, in order: a fused
 * call counts as one call of every rank, and needs every rank to have issued
 * the same number of calls before it (else AR_EINVAL, nothing enqueued).
 * stream: non-blocking, as for the per-rank calls.  Capturable.
 * Errors: as ar_allreduce / ar_allgather.
 */
AR_API int ar_allreduce_fused(ar_handle *h, const void *const *ins, void *const *outs, size_t numel,
                              ar_stream_t stream);
AR_API int ar_allgather_fused(ar_handle *h, const void *const *ins, void *const *outs, size_t numel,
                              ar_stream_t stream);

/*
 * ar_allreduce_all -- enqueue one all-reduce call of every rank, rank r's on
 * streams[r] (a host array of R non-blocking streams, owned by the caller),
 * for a caller that drives all R logical ranks from one place.  ins[r] /
 * outs[r] as for ar_allreduce_fused.  The handle's tactic (ar_tactics.all_fused)
 * decides how: either R per-rank launches, exactly as R ar_allreduce calls, or
 * one launch of every rank on streams[0], ordered after the work already on
 * every streams[r] and before the work enqueued on them afterwards (streams[0]
 * waits for an event recorded on each other stream; each other stream waits
 * for an event recorded after the launch; the events belong to the handle).
 * Either way each rank's output is ready on its own stream, with the same
 * bits.  Graph capture: all R streams in the same capture (forked from it);
 * a stream whose captured work is already all ahead of streams[0] (nothing
 * new on it since the previous call's join) adds no edge, so back-to-back
 * calls keep the programmatic edge between their kernels.
 * One launch pays a graph's per-kernel launch cost once instead of R times,
 * which is what a graph replaying one all-reduce is made of.  Errors: as
 * ar_allreduce_fused; AR_ESTREAM if some of the streams are being captured
 * and others are not, or two ranks share a stream.
 */
AR_API int ar_allreduce_all(ar_handle *h, const void *const *ins, void *const *outs, size_t numel,
                            const ar_stream_t *streams);

/*
 * ar_status -- the first device-side error recorded in the handle (AR_OK or
 * AR_ETIMEOUT), copied into *info if info is not NULL.  Reads mapped host
 * memory only (no CUDA call); the answer covers the kernels the caller has
 * already synchronised with.  This is the library's watchdog report: a rank
 * that never arrives ends its peers' bounded waits with a recorded code
 * instead of a hang ("fix(qwen3): re-enable CUDA Graph under TP via startup
 * decode-graph pre-capture", section "Description": NCCL has no device-side
 * timeout, so a wedged rank would otherwise wait forever).
 */
AR_API int ar_status(ar_handle *h, ar_error_info *info);

/*
 * ar_reset -- synchronise the device, then zero every flag, counter and the
 * error record.  Required after AR_ETIMEOUT; afterwards the handle behaves as
 * if just created.  No graph that uses the handle may be running.  The
 * recovery half of the watchdog of "fix(qwen3): re-enable CUDA Graph under TP
 * via startup decode-graph pre-capture", section "Description": after a
 * timeout the caller resets the exchange state rather than the process.
 */
AR_API int ar_reset(ar_handle *h);

/*
 * ar_destroy -- synchronise the device and free everything ar_create
 * allocated.  Every CUDA graph that captured calls on this handle must be
 * destroyed first (captured kernels hold the handle's addresses; teardown
 * order as in "[SM120] Add optional FlashInfer PCIe-IPC all-reduce for
 * switch-free hosts", review of destroy(): release the workspace before what
 * it depends on, and "fix(qwen3): re-enable CUDA Graph under TP ...", section
 * "Description": graphs go before the communicator).  NULL is a no-op.
 */
AR_API int ar_destroy(ar_handle *h);

/* Set the device wait timeout in nanoseconds (>= 1000).  Applies to calls
 * enqueued afterwards; a captured graph keeps the value in force at capture. */
AR_API int ar_set_timeout(ar_handle *h, uint64_t timeout_ns);

/*
 * ar_set_trace -- record when each block of each rank ran.  records: device
 * memory (owned by the caller, zeroed by the caller) holding `capacity`
 * ar_trace_record entries; NULL stops tracing.  Thread 0 of every block of
 * every later call (enqueued or captured after this) writes one record, at
 * index ((call % depth) * R + rank) * max_blocks + block, depth = capacity /
 * (R * max_blocks) (ar_info.max_blocks), so the last `depth` calls of each
 * block are kept.  capacity < R * max_blocks, a buffer not 16-byte aligned,
 * or a call that is half issued (traced calls may launch another grid)
 * returns AR_EINVAL.  Traced calls run kernels built with the trace code (a
 * few stores per block and call); untraced calls run kernels built without
 * it, so tracing off costs nothing.  A captured graph keeps the setting in
 * force at capture (and writes to that buffer while it lives).
 * The pages measure with serving metrics and a probe; this shows, without an
 * external profiler, that the R rank kernels of a call run at the same time
 * and where a call's time goes.
 */
AR_API int ar_set_trace(ar_handle *h, void *records, uint64_t capacity);

/*
 * ar_debug_seed_stages -- test hook: synchronise the device, then set the
 * stage count of every (rank, block) of the handle to `stages` (call counts
 * unchanged), as if that many stages had run.  Lets a test cross the point
 * where the tagged-word form's 32-bit tags wrap (near 2^32 - 1 stages)
 * without running billions of calls.  Use on an idle handle only: every rank
 * must have completed the same calls.  Errors: AR_EINVAL (NULL handle),
 * AR_ECUDA.
 */
AR_API int ar_debug_seed_stages(ar_handle *h, uint64_t stages);

/* Static facts about the handle. */
AR_API int ar_query(const ar_handle *h, ar_info *info);

/*
 * ar_plan_for -- the launch plan ar_allreduce (op 0), ar_allgather (op 1) or a
 * launch of every rank's all-reduce at once (op 2: ar_allreduce_fused, and
 * ar_allreduce_all when it fuses) would use for numel elements on this
 * handle.  For the cluster form, blocks is the number of clusters (each of R
 * blocks) and flag_rounds the cluster barriers per tile.  Pure host
 * arithmetic.
 */
AR_API int ar_plan_for(const ar_handle *h, int op, size_t numel, ar_plan *plan);

/*
 * ar_plan_compute -- the same plan from explicit machine facts, so the host
 * logic can be checked without a GPU: R ranks, `bytes` per rank, vector size
 * vec_bytes (16, 8, 4, 2 or 1), algo AR_ALGO_ONESHOT or AR_ALGO_TWOSHOT,
 * `threads` per block, and a GPU that holds sm_count * blocks_per_sm blocks of
 * the kernel at once.  Two-shot plans here use 256-vector sub-tiles; a handle
 * with HBM slots uses 128 when that leaves more than half its blocks idle, one
 * with pinned-host slots 64 while 256 would make fewer than 8 tiles
 * (ar_plan_for shows its choice).
 */
AR_API int ar_plan_compute(int R, uint64_t bytes, int vec_bytes, int algo, int threads, int sm_count,
                           int blocks_per_sm, ar_plan *plan);

/* The all-reduce form a new handle's AR_ALGO_AUTO picks for R ranks, `bytes`
 * per rank and a slot kind (a tactic table measured on a GB300 with the
 * default tactics, the ranks synchronising at GPU scope; a handle's own
 * tactics may differ, see ar_tactics).  HBM slots: tagged-word form up to
 * 512 KiB (R <= 2), 256 KiB (R = 3) or 64 KiB (R = 4) (within
 * ar_info.tagged_capacity_bytes); otherwise one-shot for R <= 3, two-shot
 * from 512 KiB (R >= 8) or 2 MiB (R = 4..7).  Pinned-host slots: never the
 * tagged form; one-shot for R <= 2, two-shot from 512 KiB (R = 3), 128 KiB
 * (R = 4), 64 KiB (R = 5..7) or 32 KiB (R >= 8), where one-shot reads
 * R(R-1)S bytes over the host link against two-shot's (2R-1)S.  Pure host
 * arithmetic. */
AR_API int ar_choose_algo(int R, uint64_t bytes, int slot_kind);

/* Launch this handle's kernels as programmatic dependents of the preceding
 * work on their stream (CUDA programmatic dependent launch), so that a rank's
 * next kernel is scheduled while its current one finishes.  Each kernel still
 * waits for the preceding kernel to complete, and for its writes to be
 * visible, before it reads or writes any memory, and lets its dependents be
 * scheduled only once all blocks of the call's ranks are resident (after its
 * last wait for its peers' flags); the bits do not change.  On by default; the
 * environment variable AR_PDL=0 turns it off at ar_create.  Applies to calls
 * enqueued (or captured) afterwards. */
AR_API int ar_set_pdl(ar_handle *h, int enable);

/* Force the all-reduce form of a handle (AR_ALGO_AUTO restores the rule):
 * AR_ALGO_ONESHOT, AR_ALGO_TWOSHOT, AR_ALGO_TAGGED (only for calls of one tile
 * per block; larger calls take the one-shot form), AR_ALGO_CLUSTER (only for
 * launches of every rank at once; per-rank calls take the AUTO rule) or
 * AR_ALGO_PUSH (allocates its receive areas on first selection, synchronising
 * the device; AR_ENOMEM if they do not fit).  The environment variable
 * AR_ALGO=oneshot|twoshot|tagged|cluster sets it at ar_create.
 * Every rank of a call must see the same setting; set it before enqueuing.
 * AR_EINVAL for an unknown form, a two-shot / tagged form on a complex64
 * handle, or a call that is half issued (some rank has enqueued more calls on
 * the handle than another; the setting is unchanged). */
AR_API int ar_set_algo(ar_handle *h, int algo);

/* Read or replace a handle's tactics (see ar_tactics).  Every rank shares the
 * handle, so all ranks see the same values; change them only between calls.
 * Errors: AR_EINVAL for a NULL argument, a sub-tile other than 0/64/128/256,
 * a negative block cap, or a call that is half issued (some rank has enqueued
 * more calls than another; the tactics are unchanged). */
AR_API int ar_get_tactics(const ar_handle *h, ar_tactics *t);
AR_API int ar_set_tactics(ar_handle *h, const ar_tactics *t);

/*
 * ar_supports -- would ar_allreduce (op 0) or ar_allgather (op 1) accept this
 * call?  Makes the argument checks the enqueue calls make before any CUDA
 * work, except the stream's (no CUDA call here): AR_OK, or the code the call
 * would return -- AR_EINVAL (NULL handle, unknown op, all-reduce on a
 * complex64 handle, NULL or non-16-byte-aligned in/out when numel > 0) or
 * AR_ETOOBIG (numel > max_numel).  Lets a caller route a tensor to its
 * fallback before it enqueues anything ("[SM120] Add optional FlashInfer
 * PCIe-IPC all-reduce for switch-free hosts", section "Modifications").
 */
AR_API int ar_supports(const ar_handle *h, int op, size_t numel, const void *in, const void *out);

/*
 * ar_allreduce_noalloc -- an all-reduce that allocates nothing.  None of the
 * cited sources has a counterpart: this entry point is for callers that cannot allocate device
 * memory where they reduce -- code running inside another library's memory
 * pool or arena, which owns every allocation on the device; code on a
 * latency-critical path where cudaMalloc, which can synchronise the device,
 * is not allowed; runtimes that reserve all memory once at start-up.
 *
 * One call reduces all R ranks (1 <= R <= 8) at once: ins[r] and outs[r]
 * (host arrays of R device pointers, each 16-byte aligned, owned by the
 * caller) hold rank r's numel elements of dtype (AR_F16 or AR_BF16); every
 * outs[r] receives the same bits as ar_allreduce: the rank-order fp32 sum with
 * one rounding.  outs[r] == ins[r] is allowed.
 * Working memory: the exchange slots (R ranks x at most 1 MiB), per-block flags
 * and an abort word live in one file-scope device array of 8 MiB + 64 KiB +
 * 256 B, which every GPU that loads this library holds until the process
 * exits.  The call allocates nothing.  numel > 524288 (more than 1 MiB per
 * rank) returns AR_ETOOBIG and enqueues nothing.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and the kernels' occupancy; make that first call
 * before any stream capture.  Each call clears the flags (cudaMemsetAsync on
 * `stream`) and then launches one cooperative grid of blocks x R on `stream`,
 * so all R ranks' blocks are resident together.  Every call shares the array
 * and it keeps the last call's contents: calls that overlap on the GPU (on
 * streams with no ordering between them) race and give undefined results.
 * A wait for a peer is bounded (1 s).  A block whose wait runs out leaves
 * without writing its part of the outputs and records itself in an error
 * record inside the same array; the call itself has already returned AR_OK.
 * Read that record with ar_noalloc_status() after synchronising with
 * `stream` and before the next call on the device, which clears it.
 * Errors: AR_EINVAL, AR_ETOOBIG, AR_ECUDA.
 */
AR_API int ar_allreduce_noalloc(int R, int dtype, const void *const *ins, void *const *outs, size_t numel,
                                ar_stream_t stream);

/*
 * ar_noalloc_status -- the error record of ar_allreduce_noalloc's array on
 * the current device: AR_OK, or AR_ETIMEOUT with the rank, block and peer of
 * the first block whose wait ran out (copied into *info if info is not NULL).
 * It covers the calls the caller has synchronised with since the last call
 * that started on the device (each call clears the record before it
 * launches).  A synchronous copy out of the array; allocates nothing.  Does
 * the device's first-call set-up if no call has run on it yet.
 * Returns the recorded code, or AR_ECUDA if the record could not be read.
 */
AR_API int ar_noalloc_status(ar_error_info *info);

/*
 * ar_noalloc_debug_record -- test hook: write *info into the error record of
 * ar_allreduce_noalloc's array on the current device, as a block that timed
 * out would, so the status plumbing can be checked without making a wait run
 * out.  The next ar_allreduce_noalloc call on the device clears it.  Use while
 * no call is running on the device.  Errors: AR_EINVAL (NULL), AR_ECUDA.
 */
AR_API int ar_noalloc_debug_record(const ar_error_info *info);

/* Human-readable name of an ar_code.  Never NULL. */
AR_API const char *ar_strerror(int code);

/*
 * Bandwidth probes: the denominators of the roofline.  Each allocates its own
 * buffers, runs its copy kernels `reps` times on a private non-blocking stream,
 * times them with CUDA events and frees everything.
 *
 * ar_probe_host_link: GPU kernels stream `bytes` to mapped pinned host memory
 *   (write), from it (read), and both at once: half the blocks store to one
 *   mapped host buffer while the other half load from another, for a fixed
 *   window (at least 1 ms), about as many bytes each way.
 *   gbs[0] = write GB/s, gbs[1] = read GB/s, gbs[2] = write GB/s while reading,
 *   gbs[3] = read GB/s while writing.  (1 GB = 1e9 bytes.)
 * ar_probe_hbm_copy: a device-to-device copy kernel over `bytes`; *gbs counts
 *   read + write bytes.
 */
AR_API int ar_probe_host_link(uint64_t bytes, int reps, double gbs[4]);

/*
 * ar_probe_host_link_latency: the latencies that bound the protocol at small
 *   sizes, each the best of three runs of `reps` (1..100000) repetitions, in ns:
 *   ns[0] = one dependent 8-byte load from mapped pinned host memory (a round
 *           trip over the host link);
 *   ns[1] = one block stores 4 KiB to mapped host memory, then a system-scope
 *           fence returns (the block's stores acknowledged: its publish step);
 *   ns[2] = a flag's one-way trip through mapped host memory at system scope
 *           (release store by one block seen by another block's acquire polls:
 *           half a ping-pong round trip) -- the flag step of a pinned call;
 *   ns[3] = the same through HBM at GPU scope -- the flag step of an HBM call,
 *           and of a pinned call whose ranks synchronise at GPU scope (the
 *           gpu_scope tactic, the default);
 *   ns[4] = as ns[1] with a GPU-scope fence -- the publish step of a pinned
 *           call at GPU scope.
 * Two blocks of one kernel play the ping-pong (always resident together); each
 * of their waits is bounded (100 ms): AR_ETIMEOUT if one runs out.  Allocates
 * and frees its own buffers and stream.  Errors: AR_EINVAL, AR_ENOMEM,
 * AR_ECUDA, AR_ETIMEOUT.
 */
AR_API int ar_probe_host_link_latency(int reps, double ns[5]);
AR_API int ar_probe_hbm_copy(uint64_t bytes, int reps, double *gbs);

#ifdef __cplusplus
}
#endif

#endif /* TDA_AR_H */
