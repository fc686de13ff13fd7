/*
 * ra.h — C ABI of the GB300 ring all-reduce library (libra.so).
 *
 * N "virtual ranks" live in one GPU's memory; each rank r owns a send buffer
 * and a receive buffer (device pointers). The calls follow the shape of
 * ncclAllReduce(sendbuff, recvbuff, count, datatype, op, comm, stream) as the
 * arjunsriva.com page "AllReduce, All the Way Down" (section "The Contract:
 * What AllReduce Means") states it, with the communicator replaced by
 * `nranks` and one host array of N device pointers per side.
 *
 * What is computed (tirogla.com "Ring all-reduce", section "How it works"):
 * the buffer of `count` elements is cut into N chunks, chunk c covering
 * elements [c*count/N, (c+1)*count/N) with floor division (section "Code"), so
 * chunks may differ by one element and may be empty. Element i of chunk c is
 * reduced in ring order, left to right,
 *
 *     x_c (+) x_{c+1} (+) ... (+) x_{c+N-1}      (rank indices mod N)
 *
 * which is the order in which the reduce-scatter phase of the ring visits
 * chunk c (it starts at rank c and ends at rank c-1, which then owns it).
 * Every hop is rounded to the buffer dtype: fp32 hops are fp32 operations;
 * fp16/bf16 hops compute in fp32 and round to nearest even once; int32 sum and
 * prod wrap modulo 2^32. RA_AVG is the ring sum followed by one multiply by
 * 1.0f/N (fp32) rounded to the dtype (int32: wrapped sum / N, truncated).
 * RA_MIN / RA_MAX follow IEEE 754-2019 minimum / maximum (NaN propagates,
 * -0 < +0). Results are bit-identical on every rank (same page,
 * "Implementation notes").
 *
 * Common rules for the three collectives:
 *  - count is the FULL per-rank vector length L in every call (also for
 *    reduce-scatter and all-gather, whose compact side holds one chunk).
 *  - sendbufs / recvbufs are host arrays of `nranks` device pointers. The
 *    arrays are read during the call only; the device buffers belong to the
 *    caller and must stay alive until the work on `stream` has completed.
 *  - The library allocates no device memory and keeps no state between
 *    calls; calls are reentrant. Work is enqueued on `stream` (a
 *    cudaStream_t; NULL = the legacy default stream) and the call returns
 *    without waiting. The collective kernels are programmatic dependent
 *    launches: their CTAs may be placed on the GPU while the previous kernel
 *    on `stream` is finishing, but no thread reads or writes memory before
 *    that kernel has completed, so the stream's order holds as for any
 *    launch (a graph captured from the stream records programmatic edges).
 *  - Arguments are checked on the host before any launch; on any error
 *    nothing is enqueued. Every pointer must be aligned to the element size;
 *    a pointer to a zero-length buffer may be NULL. Any other alignment is
 *    accepted: the vector path is used when the buffers share their address
 *    modulo ra_vector_bytes(), a per-element path otherwise.
 *  - Buffers may be device memory or host memory the device can address
 *    (pinned host memory under unified addressing, or any host memory on
 *    systems whose GPU accesses system memory coherently): the kernels then
 *    read and write host memory directly over the host link, which replaces
 *    explicit copies for callers whose data lives on the host. Such calls
 *    launch one resident wave (it streams the host link faster than a CTA per
 *    trip) and the all-gather takes plain stores; the TMA-staged bulk engine
 *    and the tree / Rabenseifner orders take device memory only and return
 *    RA_ERR_UNSUPPORTED for a host buffer, before enqueuing anything.
 *  - Buffers must not overlap, except in the exact in-place layout named for
 *    each call (each element is then read and written by the same thread).
 *    Send buffers may overlap each other (they are only read).
 *  - count == 0 returns RA_SUCCESS and launches nothing. nranks == 1 copies.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RA_MAX_RANKS 64
/* largest accepted count: keeps c*count (c <= 64) inside 63 bits */
#define RA_MAX_COUNT ((((uint64_t)1) << 57) - 1)

typedef enum {
  RA_SUCCESS = 0,
  RA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, nranks outside [1, 64], bad enum, count too big */
  RA_ERR_UNSUPPORTED = 2, /* a dtype/op/option combination the library does not provide */
  RA_ERR_ALIAS = 3,       /* buffers overlap other than in the allowed in-place layout */
  RA_ERR_CUDA = 4,        /* the CUDA launch failed; see ra_last_cuda_error() */
  RA_ERR_SCRATCH_LIMIT = 5 /* ra_allreduce_bulk_noalloc: nranks above RA_NOALLOC_STATUS_WORDS */
} ra_status_t;

typedef enum { RA_FLOAT32 = 0, RA_FLOAT16 = 1, RA_BFLOAT16 = 2, RA_INT32 = 3 } ra_dtype_t;

/* bitfern.com "AllReduce Explained", section "What Is AllReduce?": sum,
 * average, minimum, maximum and product reductions. */
typedef enum { RA_SUM = 0, RA_AVG = 1, RA_MIN = 2, RA_MAX = 3, RA_PROD = 4 } ra_op_t;

/*
 * All-reduce (tirogla.com "Ring all-reduce", "How it works": reduce-scatter
 * then all-gather). sendbufs[r]: count elements of rank r. recvbufs[r]: count
 * elements; on completion every recvbufs[r] holds the reduction of all ranks.
 * In place: recvbufs[r] == sendbufs[r].
 * HBM traffic: reads N*count*e bytes, writes N*count*e bytes, in one launch.
 */
ra_status_t ra_allreduce(const void* const* sendbufs, void* const* recvbufs, size_t count,
                         ra_dtype_t dtype, ra_op_t op, int nranks, void* stream);

/*
 * Reduce-scatter (infra-guide "Collective communication primitives", section
 * 3.5: rank i keeps reduced shard i). sendbufs[r]: count elements.
 * recvbufs[r]: chunk r only, (end_r - begin_r) elements, compact. The shard
 * is reduced in the same ring order as ra_allreduce, so the all-gather of
 * these shards equals ra_allreduce bit for bit (same page, section 3.8).
 * In place: recvbufs[r] == sendbufs[r] + begin_r elements.
 * HBM traffic: reads N*count*e, writes count*e.
 */
ra_status_t ra_reduce_scatter(const void* const* sendbufs, void* const* recvbufs, size_t count,
                              ra_dtype_t dtype, ra_op_t op, int nranks, void* stream);

/*
 * All-gather (ramchalamkr.github.io "NCCL Primitives Deep Dive", section 1;
 * infra-guide section 3.6). sendbufs[r]: chunk r, (end_r - begin_r) elements,
 * compact. recvbufs[r]: count elements; on completion each holds every chunk
 * at its place. `op` is ignored (no reduction happens).
 * In place: sendbufs[r] == recvbufs[r] + begin_r elements.
 * HBM traffic: reads count*e, writes N*count*e.
 */
ra_status_t ra_allgather(const void* const* sendbufs, void* const* recvbufs, size_t count,
                         ra_dtype_t dtype, ra_op_t op, int nranks, void* stream);

/* Reduction order (the algorithm whose association the result reproduces). */
typedef enum {
  RA_ORDER_RING = 0,         /* tirogla.com "Ring all-reduce", "How it works" (the default) */
  RA_ORDER_TREE = 1,         /* double binary tree (same page, cost model): in-order trees over ranks
                                0..N-1 (first N/2 chunks) and N-1..0 (the rest) */
  RA_ORDER_RABENSEIFNER = 2  /* recursive halving / doubling, power-of-two nranks (same page) */
} ra_order_t;

/* Precision of the partials travelling between ranks. */
typedef enum {
  RA_ACCUM_DTYPE = 0, /* every hop rounded to the buffer dtype (the default) */
  RA_ACCUM_FP32 = 1   /* fp16/bf16: partials kept in fp32, rounded once at the end (after the
                         avg multiply); tirogla.com "Ring all-reduce", "Implementation notes".
                         No effect on fp32 and int32 buffers. */
} ra_accum_t;

/* How the fused all-reduce moves its loads. */
typedef enum {
  RA_ENGINE_REGISTERS = 0, /* every thread keeps its loads in flight in registers (the default) */
  RA_ENGINE_BULK = 1       /* a producer thread per CTA streams tiles of all ranks into shared memory
                              with bulk copies (the Tensor Memory Accelerator) and the other warps fold
                              from there: several times the bytes in flight per SM, for runs confined
                              to a few SMs by max_sms. All-reduce with the ring order and dtype
                              accumulation, nranks <= 16; needs `status` */
} ra_engine_t;

/* Options of the extended calls; NULL means all defaults. */
typedef struct {
  ra_order_t order;   /* RA_ORDER_RING by default */
  ra_accum_t accum;   /* RA_ACCUM_DTYPE by default */
  int max_sms;        /* 0: the launch may fill every SM; k > 0: at most k SMs' worth of CTAs, leaving the
                         rest to work running beside the collective (arjunsriva.com "AllReduce, All the
                         Way Down": communication kernels compete with compute for SMs). The hardware
                         places the CTAs: the budget bounds the collective's share of CTA slots, not
                         which SMs it runs on, and a launch shape with several CTAs per SM may spread
                         over more than k SMs (the bulk engine runs one CTA per SM); a hard partition
                         of the SMs needs green contexts */
  ra_engine_t engine; /* RA_ENGINE_REGISTERS by default */
  int* status;        /* RA_ENGINE_BULK only: one int of device memory, owned by the caller, that the
                         kernel sets to a nonzero code if one of its bounded waits gives up (1: a
                         bulk copy did not land within 1 s; 2: a stage was not released within 1 s)
                         instead of hanging; it is never cleared by the library */
} ra_options_t;

/*
 * All-reduce / reduce-scatter with options: ra_allreduce(...) is
 * ra_allreduce_ex(..., NULL, stream). Same buffers, in-place rules and errors
 * as the plain calls, plus RA_ERR_UNSUPPORTED for RA_ORDER_RABENSEIFNER with a
 * nranks that is not a power of two, for RA_ACCUM_FP32 with an order other
 * than the ring, and for RA_ENGINE_BULK outside its range (reduce-scatter,
 * another order or accumulation, nranks > 16, buffers without a common
 * address phase), and RA_ERR_INVALID_ARG for an unknown order/accum/engine,
 * a negative max_sms or RA_ENGINE_BULK without a status word.
 */
ra_status_t ra_allreduce_ex(const void* const* sendbufs, void* const* recvbufs, size_t count, ra_dtype_t dtype,
                            ra_op_t op, int nranks, const ra_options_t* options, void* stream);
ra_status_t ra_reduce_scatter_ex(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                 ra_dtype_t dtype, ra_op_t op, int nranks, const ra_options_t* options,
                                 void* stream);

/*
 * Gradient buckets (bitfern.com "AllReduce Explained", "PyTorch DDP and
 * Gradient Synchronization"; tirogla.com "Ring all-reduce", "Implementation
 * notes": DDP's default bucket is 25 MB). Host only, touches no GPU.
 * param_counts[nparams]: element counts of the parameters, laid out
 * contiguously in this order in the flat gradient buffer. Parameters are
 * visited in reverse (the order backward produces their gradients) and packed
 * into buckets of at most bucket_bytes (a parameter larger than that gets its
 * own bucket). Writes up to max_buckets contiguous element ranges
 * [bucket_begin[b], bucket_begin[b] + bucket_count[b]) in the order they
 * become ready, and the number of buckets to *nbuckets (also when max_buckets
 * is too small, which returns RA_ERR_INVALID_ARG; NULL arrays with
 * max_buckets 0 query the count).
 */
ra_status_t ra_bucket_plan(const size_t* param_counts, int nparams, size_t bucket_bytes, int elem_size,
                           size_t* bucket_begin, size_t* bucket_count, int max_buckets, int* nbuckets);

/*
 * Bucketed all-reduce: bucket b (an element range of every rank's buffer,
 * listed in ascending or descending order, disjoint) is all-reduced as an
 * all-reduce of its own (its own chunk bounds), after `stream` waits for
 * ready_events[b] (a cudaEvent_t the producer recorded when the bucket's
 * gradients were complete; NULL entries or a NULL array wait for nothing).
 * The waits and launches are enqueued on `stream` in bucket order, so buckets
 * overlap with work on other streams as soon as they are ready. A run of
 * buckets with no ready event of their own (NULL entries, or a NULL array)
 * goes out as one grouped launch of up to 64 buckets when the options are the
 * default engine and ring order; each bucket's result bits are still those of
 * an all-reduce of its own. Buffers, in-place rule and options as
 * ra_allreduce_ex.
 */
ra_status_t ra_allreduce_buckets(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                 ra_dtype_t dtype, ra_op_t op, int nranks, int nbuckets, const size_t* bucket_begin,
                                 const size_t* bucket_count, void* const* ready_events,
                                 const ra_options_t* options, void* stream);

/*
 * The literal ring schedule, one kernel launch per ring step (tirogla.com
 * "Ring all-reduce", "How it works"): reduce-scatter step s = 0..N-2 has rank
 * r combine chunk (r-s-1) mod N arriving from rank r-1 with its own copy;
 * all-gather step s has rank r copy chunk (r-s) mod N from rank r-1. Every
 * message is a read of rank r-1's buffer in HBM. Same arguments, rounding,
 * in-place rule and final result (bit for bit) as ra_allreduce; it moves
 * about 5(N-1)*S bytes instead of 2N*S, which is what the fused kernel saves.
 * nsteps: run only the first nsteps of the 2(N-1) steps (negative = all);
 * after a partial run each rank's buffer holds the schedule's state for the
 * chunks the steps have touched and is undefined elsewhere.
 */
ra_status_t ra_allreduce_ringsteps(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                   ra_dtype_t dtype, ra_op_t op, int nranks, int nsteps, void* stream);

/*
 * Chunk bounds (tirogla.com "Ring all-reduce", section "Code"):
 * *begin = c*count/nranks, *end = (c+1)*count/nranks, floor division, exact
 * for every count <= RA_MAX_COUNT. Host only; touches no GPU.
 */
ra_status_t ra_chunk_range(size_t count, int nranks, int c, size_t* begin, size_t* end);

/*
 * Planner introspection (host only, no GPU): how chunk c is split between the
 * vector path and the per-element path for buffers of `elem_size`-byte
 * elements that share their address phase `phase_bytes` modulo `align_bytes`
 * (a power of two from ra_vector_bytes() to 512; the library uses the largest
 * such alignment the buffers share). Writes [vec_begin, vec_end) (elements
 * moved as whole vectors, starting on the alignment grid; empty if vec_begin
 * == vec_end) inside [begin, end); the rest of the chunk takes the
 * per-element path.
 */
ra_status_t ra_plan_chunk(size_t count, int nranks, int c, int elem_size, int align_bytes, int phase_bytes,
                          size_t* begin, size_t* end, size_t* vec_begin, size_t* vec_end);

/* A static, human-readable name for a status code. */
const char* ra_status_string(ra_status_t status);

/* The cudaError_t of the last RA_ERR_CUDA returned on the calling thread (0 if none). */
int ra_last_cuda_error(void);

/*
 * Self-test of the bulk engine's bounded waits (host-visible failure
 * reporting without a GPU fault): runs the RA_ENGINE_BULK all-reduce with the
 * first tile of CTA (0, withhold_chunk) never copied in, so that CTA's
 * consumers wait for it in vain and give up after 1 s; the CTA records a
 * nonzero code (1 or 2, as for ra_options_t.status), waits (bounded) for its
 * other copies in flight and winds down. The launch completes and the context
 * stays usable. The receive buffers' contents are unspecified afterwards.
 * status: caller-owned device ints, 0 before the call. status_per_chunk 0:
 * every chunk reports into status[0] (one int); 1: chunk c reports into
 * status[c] (nranks ints), as ra_allreduce_bulk_noalloc's words do.
 * withhold_chunk in [0, nranks); count must give that chunk at least one
 * whole tile for the self-test to fire. Same other arguments as ra_allreduce.
 */
ra_status_t ra_selftest_bulk_timeout(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                     ra_dtype_t dtype, ra_op_t op, int nranks, int withhold_chunk, int* status,
                                     int status_per_chunk, void* stream);

/* Bytes per vector access of the library's compiled kernels (16 or 32): the address
 * phase (address mod this) the buffers must share for the vector path. */
int ra_vector_bytes(void);

/* Status words held by the library for ra_allreduce_bulk_noalloc: one per chunk. */
#define RA_NOALLOC_STATUS_WORDS 16

/*
 * The RA_ENGINE_BULK all-reduce for a caller that cannot allocate device
 * memory. The web pages have no counterpart: this is an interface of this
 * library only. Result bits, buffers, in-place rules and other errors are
 * those of ra_allreduce_ex with RA_ENGINE_BULK; the difference is where the
 * status words live. ra_allreduce_ex wants a device int from the caller;
 * here the library keeps RA_NOALLOC_STATUS_WORDS ints of its own, a fixed
 * array inside libra.so's device image, and the call allocates nothing.
 *
 * Who needs this: a caller whose device memory is all held by another
 * allocator (a framework's caching pool), which has no device allocation
 * call of its own to use and would only fragment that pool with a stray
 * cudaMalloc; a caller between the kernels of a training step, where
 * cudaFree would make the host wait for the whole device, including the
 * compute that the bulk engine is meant to run beside; and a caller that
 * wants the per-chunk codes in pinned host memory (chunk_status may be host
 * memory). The buffers themselves must be device memory (RA_ERR_UNSUPPORTED
 * otherwise): a program whose buffers are pinned host memory calls
 * ra_allreduce, which reads and writes them over the host link.
 *
 * Set-up: every call looks up the array's device address in the current
 * context (cudaGetSymbolAddress) and keeps nothing between calls, so a call
 * after a context switch or a device reset uses that context's copy. A failed
 * lookup returns RA_ERR_CUDA. The first lookup in a context can load the
 * library's kernels into it, so make the first call there before any stream
 * capture begins.
 *
 * Each call enqueues on `stream`: a clear of words [0, nranks) of the array;
 * the kernel, whose CTAs for chunk c record in word c the code of a bounded
 * wait that gave up (1: a bulk copy did not land within 1 s; 2: a stage was
 * not released within 1 s); and, if chunk_status is not NULL, a copy of
 * those nranks words to chunk_status (device memory or host memory, nranks
 * ints, caller-owned; pageable host memory makes the call wait until the
 * kernel has finished). Read chunk_status once the stream has passed the
 * call: 0 everywhere means every chunk finished. max_sms as in ra_options_t.
 * count == 0 enqueues nothing and leaves chunk_status untouched.
 *
 * Limit: nranks must be at most RA_NOALLOC_STATUS_WORDS (16, the bulk
 * engine's own limit); a larger nranks (up to RA_MAX_RANKS) returns
 * RA_ERR_SCRATCH_LIMIT before anything is enqueued.
 *
 * Errors: every check, the plan and the kernel's shared-memory set-up come
 * before the first enqueue, so an error returned from them enqueues nothing.
 * Only a failure of one of the three enqueues itself (RA_ERR_CUDA) can leave
 * the earlier ones queued; they touch nothing but the library's words and,
 * for the copy, chunk_status.
 *
 * Concurrency: each context has one copy of the array (on the usual primary
 * context: one per device), shared by all calls there. Two calls in flight at
 * once in one context (on different streams, or from different threads) race
 * on it: one call's clear can erase the other's codes, and a copy can return
 * the other's codes. The reduced buffers are not affected. Calls on one
 * stream run one after the other and do not race.
 */
ra_status_t ra_allreduce_bulk_noalloc(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                      ra_dtype_t dtype, ra_op_t op, int nranks, int max_sms, int* chunk_status,
                                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
