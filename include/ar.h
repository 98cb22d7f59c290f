/*
 * ar.h -- simulated AllReduce on one GB300 (sm_103a).
 *
 * C ABI of the library libar_gb300.so.  N "ranks" are N equal-length buffers
 * resident in one GPU's HBM; a collective combines them element by element
 * with SUM, MAX or AVG (SUM, then divide by N) and leaves the result in every
 * buffer, exactly as the data-parallel gradient AllReduce leaves the same
 * reduced gradient on every process.
 *
 * Sources for the operations (page title, section):
 *   [concept]  "AllReduce" (concept page), §3 技术原理 and §4 关键参数
 *   [tutorial] "Allreduce：大模型分布式训练的核心通信算法与优化实践", §2.2, §3.1-3.2,
 *              §4.1, §4.4
 *   [chapter]  "AllReduce算法详解：Ring AllReduce原理，Tree AllReduce原理，性能对比与
 *              选择", §4.2-4.3
 *   [notes]    "AllReduce 集合通信", §语义, §两阶段流程, §通信量推导, §DDP 梯度同步中的地位
 *   [primer]   "【AI Infra小白入门⑩】集合通信基础：AllReduce、Ring算法与NCCL全解析",
 *              §二, §三, §四 4.1
 *
 * Common conventions
 *   - Every function returns AR_OK (0) or a negative ar_status; none throws,
 *     none keeps a pointer after it returns, none allocates caller-visible
 *     memory.  Work is enqueued on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and the call returns once it is enqueued; the
 *     results are valid when the stream reaches that point.
 *   - Buffers are device pointers of the current CUDA device, one per rank,
 *     each holding `count` elements of `dtype`, pairwise distinct and
 *     non-overlapping (checked; AR_ERR_INVALID_ARG otherwise).  They must be
 *     aligned to the element size.  When all of them sit at the same address
 *     modulo 16 (16-byte aligned or not) the kernels move 16-byte vectors,
 *     cut at that offset.  Buffers at different offsets modulo 16 still move
 *     in aligned 16-byte words in the fused kernels (each rank's words staged
 *     in shared memory, folded there in the first buffer's frame and written
 *     back at each rank's own offset) for every order and rank count, and
 *     for AllGather and Broadcast; the step-wise and copy kernels then take
 *     a slower one-element-per-thread path.  (For a bucketed call this holds per
 *     tensor: each tensor's N buffers.)
 *   - 1 <= nranks <= AR_MAX_RANKS; 0 <= count <= AR_MAX_COUNT (else
 *     AR_ERR_INVALID_ARG, as for a buffer whose end would pass the top of the
 *     address space); count == 0 and nranks == 1 do
 *     nothing (a single rank already holds the reduction; AVG divides by 1).
 *     With count == 0 the buffer pointers are not examined (NULL is fine,
 *     as an empty tensor's is); the host array itself must not be NULL.
 *   - Chunks: each rank buffer is split into N contiguous chunks,
 *     chunk c = [floor(c*count/N), floor((c+1)*count/N)); rank c owns chunk c
 *     after ReduceScatter.  [concept §3], [tutorial §2.2], [notes §两阶段流程].
 *   - Element step: f32 is IEEE binary32 addition (round to nearest even,
 *     subnormals kept); bf16 and f16 (IEEE binary16, the FP16 of [tutorial
 *     §4.2]) are exact widening to binary32, addition, and rounding to nearest
 *     even back to the storage type after every step; i32 adds with
 *     two's-complement wrap-around; MAX is IEEE 754-2019 maximum (NaN
 *     propagates, +0 > -0).  AVG is SUM followed by one IEEE binary32 division
 *     by N of each reduced element (for bf16 and f16 the quotient is rounded
 *     to the storage type); AVG on i32 is AR_ERR_UNSUPPORTED.  NaN results
 *     carry no payload guarantee.
 *   - Orders (bit-exact with a step-wise execution of the same schedule):
 *       AR_RING / AR_RING_STEPWISE: chunk c is folded in ring order
 *         x[c+1], x[c+2], ..., x[c+N-1], x[c] (indices mod N), one rounding per
 *         step -- the order in which ReduceScatter carries chunk c around the
 *         ring.  [tutorial §2.2], [notes §两阶段流程], [primer §三 3.1].
 *       AR_TREE / AR_TREE_STEPWISE: balanced pairwise tree over rank indices,
 *         (x0 (+) x1), (x2 (+) x3), ... then pairs of pairs, lower ranks first;
 *         N must be a power of two (AR_ERR_UNSUPPORTED otherwise).
 *         [primer §四 4.1], [chapter §4.3].
 *       AR_NAIVE (AllReduce and Reduce only): index order x[0], x[1], ...,
 *         x[N-1], the order in which a central root folds the buffers it
 *         gathers ("AllReduce 集合通信" §朴素实现与主节点瓶颈, tutorial §2.1).
 *       AR_BINOMIAL_STEPWISE (AllReduce only): the tree that reduces to a
 *         root and then broadcasts ([chapter §4.3]), executed literally:
 *         reduce step k = 0 .. log2(N)-1 (distance h = 2^k, nearest ranks
 *         first as in [primer §四 4.1]) has every rank r = h (mod 2h) send
 *         its whole buffer to rank r-h, which folds it in (lower rank first);
 *         rank 0 then holds the result (and divides it by N for AVG);
 *         broadcast step k = log2(N)-1 .. 0 has every rank r = 0 (mod 2h)
 *         send it to rank r+h.  2 log2(N) steps, each moving whole buffers
 *         (the root sends and receives D elements per level: 2 D log2(N) at
 *         the root, [chapter §4.3]).  Every element is folded in the
 *         balanced pairwise order of AR_TREE, so the values equal AR_TREE's.
 *         N must be a power of two.
 *       AR_DBTREE (AllReduce only): double binary tree -- two binary trees
 *         run at once, each reducing half of the data ([concept §3]; the
 *         pages give no shape).  Positions 1..N form an in-order binary tree
 *         (the root of a range is its position with the most trailing zero
 *         bits); tree A holds rank p-1 at position p and reduces elements
 *         [0, floor(D/2)); tree B holds rank p mod N and reduces the rest.  A
 *         node folds ((left subtree) (+) own) (+) (right subtree).
 *     The fused algorithms make one pass over HBM (each element of each rank
 *     read once and written once); the step-wise ones execute the literal
 *     schedule, one grid-wide phase per communication step, in a single
 *     persistent cooperative kernel.  A small plain (one-buffer-per-rank)
 *     step-wise call -- at most 3072 element updates in a phase, N buffers
 *     within 160 KiB -- runs the same schedule in one thread block, the
 *     buffers staged in its shared memory and a block barrier between
 *     phases: same results, no grid barrier.  A somewhat larger one runs it
 *     in one thread-block cluster (up to 16 blocks, each holding some ranks'
 *     buffers in at most 160 KiB of shared memory), senders read through
 *     distributed shared memory and a cluster barrier between phases, while
 *     no block folds more than 1024 elements in a phase: same results.
 */
#ifndef AR_GB300_H
#define AR_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st* ar_stream_t;

#define AR_MAX_RANKS 64
/* Largest element count a call accepts (per buffer; for bucketed calls also
 * per tensor and for the sum over tensors).  2^56 elements is far beyond any
 * device allocation; the limit keeps every byte offset and buffer end
 * representable, so the range checks cannot be defeated by wrap-around. */
#define AR_MAX_COUNT (1LL << 56)
#define AR_DEFAULT_BUCKET_CAP_BYTES (25LL << 20) /* DDP's 25 MB bucket [tutorial §4.1] */

typedef enum { AR_F32 = 0, AR_BF16 = 1, AR_I32 = 2, AR_F16 = 3 } ar_dtype;
typedef enum { AR_SUM = 0, AR_MAX = 1, AR_AVG = 2 } ar_op;
typedef enum {
  AR_RING = 0,
  AR_RING_STEPWISE = 1,
  AR_TREE = 2,
  AR_TREE_STEPWISE = 3,
  AR_NAIVE = 4,
  AR_DBTREE = 5,
  AR_BINOMIAL_STEPWISE = 6
} ar_algo;

typedef enum {
  AR_OK = 0,
  AR_ERR_INVALID_ARG = -1, /* null/duplicate/overlapping/misaligned pointer, bad size or enum */
  AR_ERR_UNSUPPORTED = -2, /* AVG on i32, tree order with N not a power of two, ... */
  AR_ERR_CUDA = -3,        /* a CUDA call failed; ar_last_cuda_error() holds the cause */
  AR_ERR_TIMEOUT = -4,     /* asynchronous: a step-wise grid barrier gave up (see ar_device_status) */
  AR_ERR_NO_DEVICE = -5,   /* no usable CUDA device */
  AR_ERR_TOO_LARGE = -6,   /* the call needs more descriptor space than one launch holds */
  AR_ERR_HOST = -7         /* host-side failure (out of host memory) */
} ar_status;

/*
 * AllReduce: afterwards every bufs[r] holds the reduction of all N inputs.
 * [concept §3]: every process ends with the same (+)_i D_i; [notes §语义]:
 * AllReduce = Reduce + Broadcast.
 *   bufs    host array of nranks device pointers (read and overwritten in place)
 *   count   elements per rank
 *   dtype, op, algo   see above
 *   stream  CUDA stream to enqueue on
 * Errors: AR_ERR_INVALID_ARG, AR_ERR_UNSUPPORTED, AR_ERR_CUDA, AR_ERR_NO_DEVICE.
 * The step-wise algorithms also use a small per-device synchronisation block
 * that the library allocates on first use (so the first step-wise call on a
 * device must not be made during stream capture) and report barrier timeouts
 * asynchronously through ar_device_status.  Step-wise calls on one device
 * must not overlap in time (they share that block).
 */
int ar_allreduce(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_op op, ar_algo algo,
                 ar_stream_t stream);

/*
 * ReduceScatter: afterwards chunk r of bufs[r] holds the reduced chunk r (in
 * the order of `algo`, AVG already divided); the other chunks of each buffer
 * are left unspecified.  [tutorial §4.4], [concept §3] (each process ends with
 * exactly 1/N of the global result).
 * Arguments and errors as ar_allreduce.
 */
int ar_reduce_scatter(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_op op, ar_algo algo,
                      ar_stream_t stream);

/*
 * AllGather: on entry chunk r of bufs[r] holds shard r; afterwards every
 * buffer holds all N shards, copied bit for bit (no arithmetic).
 * [concept §3], [tutorial §2.2 第二阶段], [notes §两阶段流程].
 *   algo    AR_RING / AR_TREE: one fused copy pass; AR_RING_STEPWISE /
 *           AR_TREE_STEPWISE: the literal forwarding schedule.
 * Arguments and errors as ar_allreduce.
 */
int ar_all_gather(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_algo algo, ar_stream_t stream);

/*
 * Reduce: afterwards bufs[root] holds the reduction of all N inputs (the
 * order of `algo`: AR_RING, AR_TREE or AR_NAIVE); the other buffers are left
 * unchanged.  [notes §语义] (Reduce: the result lands at the root only),
 * [primer §二].  One pass: N reads and one write per element.
 *   root   0 <= root < nranks (AR_ERR_INVALID_ARG otherwise)
 * The step-wise orders are AR_ERR_UNSUPPORTED here.  Other arguments and
 * errors as ar_allreduce.
 */
int ar_reduce(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_op op, ar_algo algo, int root,
              ar_stream_t stream);

/*
 * Broadcast: afterwards every buffer holds bufs[root], copied bit for bit.
 * [notes §语义] (Broadcast: the root's data goes to every process),
 * [primer §二].  One pass: one read and N-1 writes per element.
 * Arguments and errors as ar_all_gather, plus root as in ar_reduce.
 */
int ar_broadcast(void* const* bufs, int nranks, int64_t count, ar_dtype dtype, int root, ar_stream_t stream);

/*
 * AllReduce of rank buffers held in host memory, through the GPU (an addition
 * with no counterpart on the pages, which keep gradients on the devices: the
 * end-to-end call for data that starts and ends on the host).  Either way the
 * result is the one ar_allreduce gives with this algo, bit for bit.
 *   dev_bufs == NULL (zero-copy): the host buffers must be page-locked memory
 *     mapped for the current device at the same address (cudaHostAlloc, or
 *     cudaHostRegister with mapping, under unified addressing; checked, else
 *     AR_ERR_INVALID_ARG).  One fused launch on `stream` reads every rank's
 *     elements across the CPU-GPU link and writes the result back across it.
 *     piece_elems is ignored.
 *   dev_bufs != NULL (staged): the buffers are cut into pieces of
 *     `piece_elems` elements.  Each piece is copied into the device buffers,
 *     AllReduced there by the fused kernel, and copied back.  The upload of
 *     the next piece, the reduction of this one and the download of the
 *     previous one run at the same time: the copies on two streams the
 *     library keeps per device, the reductions on `stream`, ordered by events.
 *     Page-locked host memory lets the copies overlap; pageable memory gives
 *     the same result, but the CUDA runtime stages and mostly serialises its
 *     copies.
 *   host_bufs   host array of nranks host pointers, `count` elements each;
 *               overwritten with the result
 *   dev_bufs    NULL, or a host array of nranks device pointers of the current
 *               device, `count` elements each: working space, overwritten
 *   piece_elems elements per staged piece, rounded up to a multiple of 64;
 *               0 = count / 8 clamped to 1-16 MiB per rank, with the first
 *               and last three pieces 1/8, 1/4 and 1/2 of that
 *   algo        AR_RING, AR_TREE, AR_NAIVE or AR_DBTREE (the step-wise
 *               orders: AR_ERR_UNSUPPORTED)
 * The call returns once everything is enqueued; the host buffers hold the
 * result once `stream` reaches that point (e.g. after
 * cudaStreamSynchronize(stream)) and must not be touched before.  The work
 * starts after the work already on `stream`.  Staged calls on one device are
 * serialised on the host and share its two copy streams; they are not for
 * stream capture.
 * Errors as ar_allreduce; all 2N ranges must be pairwise disjoint.  A CUDA
 * failure part-way returns AR_ERR_CUDA with some pieces already enqueued:
 * synchronise the device before reusing the buffers.
 */
int ar_allreduce_host(void* const* host_bufs, void* const* dev_bufs, int nranks, int64_t count, ar_dtype dtype,
                      ar_op op, ar_algo algo, int64_t piece_elems, ar_stream_t stream);

/*
 * 8-bit quantised AllReduce with error feedback ([tutorial §4.2]: gradients
 * travel as 8-bit integers that the receiver dequantises; error feedback
 * carries the compression error into the next round).  The pages give no
 * scheme; this one (binary32 throughout, round to nearest):
 *   every rank r: y = grads[r] + residuals[r]; per block of 128 elements
 *   from the start of the buffer s = max|y| / 127; q = round-half-even(y / s)
 *   clamped to [-127, 127] (0 when s = 0); residuals[r] = y - q * s;
 *   chunk c's owner folds q * s of all ranks in ring order x[c+1], ..., x[c]
 *   (AVG: divides by N once), requantises with the same rule per block cut at
 *   the chunk's ends, and every rank's grads receive that requantised value.
 * On a network this moves 2(N-1)/N * D one-byte codes per rank (plus one
 * scale per block) instead of 2(N-1)/N * D floats.
 *   grads, residuals  host arrays of nranks device pointers to count floats
 *               each (all 2N ranges disjoint); both updated in place.  Start
 *               training with zeroed residuals.
 *   op          AR_SUM or AR_AVG (AR_MAX: AR_ERR_UNSUPPORTED)
 * Inputs must be finite.  Errors as ar_allreduce.  All 2N buffers 16-byte
 * aligned: 16-byte accesses; otherwise each lane's four elements are loaded
 * one by one (same results).
 */
int ar_allreduce_int8_ef(void* const* grads, void* const* residuals, int nranks, int64_t count, ar_op op,
                         ar_stream_t stream);

/*
 * DDP bucket plan [tutorial §4.1], [notes §DDP 梯度同步中的地位]: walk the
 * tensors in reverse registration order; add each to the current bucket while
 * the bucket's bytes stay <= cap_bytes; a tensor that does not fit opens the
 * next bucket (so a tensor larger than the cap sits alone).  Inside a bucket
 * tensors lie in the order they were added.  Bucket 0 holds the
 * last-registered tensors.
 *   counts            [ntensors] element counts, registration order
 *   bucket_of_tensor  [ntensors] out: bucket id of each tensor
 *   offset_in_bucket  [ntensors] out: element offset of each tensor in its bucket
 *   bucket_count      [ntensors] out (capacity ntensors): elements per bucket
 *   nbuckets          out: number of buckets
 * Host-only; errors: AR_ERR_INVALID_ARG (also for a negative count, or
 * counts whose sum exceeds AR_MAX_COUNT).
 */
int ar_bucket_plan(const int64_t* counts, int ntensors, ar_dtype dtype, int64_t cap_bytes, int32_t* bucket_of_tensor,
                   int64_t* offset_in_bucket, int64_t* bucket_count, int32_t* nbuckets);

/*
 * Bucketed gradient AllReduce, DDP style: the ntensors gradients of each rank
 * are grouped into buckets by ar_bucket_plan, every bucket is AllReduced as
 * one flat buffer (chunks and order follow the bucket, as if the bucket had
 * been packed), and the result is written back into every rank's tensors.
 * With op == AR_AVG the 1/N scale is applied inside the reduction.
 *   grads       host array [nranks * ntensors] of device pointers, row-major by
 *               rank: grads[r * ntensors + t] is rank r's tensor t
 *   counts      [ntensors] element counts
 *   bucket_cap_bytes  cap per bucket (AR_DEFAULT_BUCKET_CAP_BYTES for DDP)
 *   workspace   NULL: fused path, one pass that reads every gradient element
 *               of every rank once and writes it once (no packing);
 *               otherwise host array [nranks] of device buffers of
 *               workspace_bytes each: the literal path packs into them,
 *               AllReduces, and unpacks.  workspace_bytes >= total bytes of
 *               all buckets packs everything at once; >= the largest bucket
 *               runs bucket by bucket; less is AR_ERR_INVALID_ARG.
 *   algo        any ar_algo but AR_NAIVE; the step-wise ones run their
 *               schedule on every bucket at once.
 * Both paths give bit-identical results.  Errors as ar_allreduce, plus
 * AR_ERR_TOO_LARGE if one tensor row (nranks pointers) cannot be described.
 */
int ar_bucketed_allreduce(void* const* grads, const int64_t* counts, int ntensors, int nranks, ar_dtype dtype,
                          ar_op op, ar_algo algo, int64_t bucket_cap_bytes, void* const* workspace,
                          int64_t workspace_bytes, ar_stream_t stream);

/*
 * Allocation-free bucketed AllReduce.  The pages have no counterpart: this is
 * an addition for callers that are not allowed to allocate -- a process whose
 * device memory is handed out by another allocator or a fixed pool that must
 * account for every byte, an engine that bans allocation on its hot path
 * because cudaMalloc can synchronise the device and stall every stream, or a
 * runtime that must not fail for lack of memory once it has started.
 *
 * Same result, bit for bit, as ar_bucketed_allreduce with the same arguments:
 * the literal path (pack each bucket, AllReduce it, unpack), with the pack
 * buffers taken from an array of AR_NOALLOC_SCRATCH_BYTES compiled into the
 * library instead of a caller workspace.  Each rank gets a slice of
 * AR_NOALLOC_SCRATCH_BYTES / nranks bytes (rounded down to 256); a bucket
 * larger than that slice, or more than AR_NOALLOC_MAX_TENSORS tensors, is
 * rejected with AR_ERR_TOO_LARGE before any work is queued.  The call makes
 * no cudaMalloc/cudaFree and no other allocating call, on the device or the
 * host heap.
 *   algo   AR_RING or AR_TREE; the step-wise orders need a barrier block the
 *          library would allocate, so they return AR_ERR_UNSUPPORTED here, as
 *          do AR_NAIVE and AR_DBTREE (which ar_bucketed_allreduce does not
 *          take either); a value outside ar_algo is AR_ERR_INVALID_ARG.
 * Other arguments and errors as ar_bucketed_allreduce (without workspace).
 * The array is shared by all calls and keeps the last call's contents (every
 * byte this call reads from it, it has written first, so nothing needs
 * clearing).  Calls that overlap on the GPU -- on different streams, or from
 * different host threads onto different streams -- race on it and corrupt
 * each other's results; keep them ordered, e.g. on one stream.  Host-side
 * calls are serialised by a lock.  The array occupies device memory on every
 * GPU where the library's device code is loaded, until the process exits
 * (with CUDA's default lazy module loading, from the first call on that GPU).
 * The first call on each device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress, no allocation).  The address
 * is remembered together with the context it belongs to: after the device's
 * context has been torn down and replaced (cudaDeviceReset), the next call
 * looks it up again.
 */
#define AR_NOALLOC_SCRATCH_BYTES (32 << 20)
#define AR_NOALLOC_MAX_TENSORS 1024
int ar_bucketed_allreduce_noalloc(void* const* grads, const int64_t* counts, int ntensors, int nranks, ar_dtype dtype,
                                  ar_op op, ar_algo algo, int64_t bucket_cap_bytes, ar_stream_t stream);

/*
 * Overlapped bucket reduction, the way DDP's reducer runs it: a bucket's
 * AllReduce starts as soon as all of its gradients are ready, while the rest
 * of the backward pass is still computing, and buckets start in bucket order.
 * [tutorial §4.1 通信与计算重叠], [notes §DDP 梯度同步中的地位].
 *
 *   ar_reducer_create   plans the buckets of `grads` (as ar_bucketed_allreduce,
 *                       fused path) and builds their launch tables once.
 *                       comm_stream carries every bucket reduction.
 *                       Arguments as ar_bucketed_allreduce (no workspace;
 *                       AR_NAIVE is AR_ERR_UNSUPPORTED).  *out receives the
 *                       handle; it allocates host memory and CUDA events only.
 *   ar_reducer_mark_ready  tensor t's gradients (on every rank) have been
 *                       produced by the work enqueued so far on
 *                       compute_stream.  When this completes a bucket, an
 *                       event is recorded on compute_stream; every bucket
 *                       whose predecessors have all started is then enqueued
 *                       on comm_stream behind that event.  Marking a tensor
 *                       twice in one iteration is AR_ERR_INVALID_ARG.
 *   ar_reducer_finish   makes compute_stream wait for the iteration's
 *                       reductions and resets for the next iteration.
 *                       AR_ERR_INVALID_ARG if some tensor was never marked.
 *   ar_reducer_destroy  releases the handle (after the streams are idle).
 * Results are bit-identical to ar_bucketed_allreduce with the same arguments.
 * A handle is used from one host thread at a time.
 */
typedef struct ar_reducer ar_reducer;
int ar_reducer_create(void* const* grads, const int64_t* counts, int ntensors, int nranks, ar_dtype dtype, ar_op op,
                      ar_algo algo, int64_t bucket_cap_bytes, ar_stream_t comm_stream, ar_reducer** out);
int ar_reducer_mark_ready(ar_reducer* red, int tensor, ar_stream_t compute_stream);
int ar_reducer_finish(ar_reducer* red, ar_stream_t compute_stream);
int ar_reducer_destroy(ar_reducer* red);
/* Number of buckets of a reducer (or AR_ERR_INVALID_ARG for NULL). */
int ar_reducer_buckets(const ar_reducer* red);
/* Caps the thread blocks of each bucket reduction (fused orders; 0 = no cap,
 * one block per tile).  On one GPU the reductions share SMs and HBM with the
 * compute they overlap; a few blocks striding over the tiles leave the rest
 * of the GPU to that compute, the way a collective library confines itself
 * to a few channels.  Results do not depend on it. */
int ar_reducer_set_max_blocks(ar_reducer* red, int max_blocks);

/*
 * Prepared collectives.  A training loop reduces the same buffers every
 * step; a plan checks the arguments and builds the launch tables once, and
 * each run only enqueues the kernels (same results as the direct call).
 *   kind    AR_PLAN_ALLREDUCE, AR_PLAN_REDUCE_SCATTER, AR_PLAN_ALL_GATHER
 *           (op ignored) or AR_PLAN_REDUCE (root used; others ignore it)
 *   other arguments as the corresponding direct call; *out receives the plan
 * The buffers must stay allocated while the plan is used: a run does not
 * check them again.  A plan may be run from any thread, on any stream, any
 * number of times, and captured into a CUDA graph (the first step-wise call
 * on a device, plan or direct, must be made outside capture).  Each launch
 * copies the plan's tables into its kernel parameters, so a plan may be
 * destroyed as soon as its last run has returned, with kernels still pending.
 * Step-wise runs on one device must not overlap in time (the shared barrier
 * block, as for the direct calls).
 * Errors: as the direct calls, at create; a run returns AR_ERR_CUDA on a
 * launch failure and AR_ERR_INVALID_ARG for a NULL plan.
 */
typedef struct ar_plan ar_plan;
enum { AR_PLAN_ALLREDUCE = 0, AR_PLAN_REDUCE_SCATTER = 1, AR_PLAN_ALL_GATHER = 2, AR_PLAN_REDUCE = 3 };
int ar_plan_create(int kind, void* const* bufs, int nranks, int64_t count, ar_dtype dtype, ar_op op, ar_algo algo,
                   int root, ar_plan** out);
int ar_plan_run(const ar_plan* plan, ar_stream_t stream);
int ar_plan_destroy(ar_plan* plan);

/* Chunk c of a rank buffer of `count` elements split N ways: [*lo, *hi).
 * Host-only; errors: AR_ERR_INVALID_ARG. */
int ar_chunk_range(int64_t count, int nranks, int c, int64_t* lo, int64_t* hi);

/*
 * Synchronises `stream`, then reads and clears the current device's
 * asynchronous status word: *status = AR_OK, or AR_ERR_TIMEOUT when a
 * step-wise barrier gave up waiting since the last read (the kernel then
 * stopped early and its buffers hold partial results).
 * Errors: AR_ERR_INVALID_ARG (status NULL), AR_ERR_CUDA.
 */
int ar_device_status(ar_stream_t stream, int* status);

/* Time limit of one step-wise barrier wait, in nanoseconds (default 1e9).
 * Values <= 0 restore the default. */
int ar_set_barrier_timeout_ns(int64_t ns);

/* Test hook for failure detection: in the next step-wise launch, block 0
 * does not arrive at barrier `barrier` (0-based), so every wait on it runs out
 * and the kernel reports AR_ERR_TIMEOUT through ar_device_status.  -1 clears
 * the hook.  Nothing faults or hangs: every wait is bounded. */
int ar_debug_skip_barrier(int barrier);

/* The cudaError_t value behind the calling thread's most recent
 * AR_ERR_CUDA / AR_ERR_NO_DEVICE return (0 if none). */
int ar_last_cuda_error(void);

/* Human-readable name of an ar_status value. */
const char* ar_strerror(int status);

/* Number of kernels this library has enqueued since it was loaded, on all
 * devices and streams (for accounting launches inside a timed region). */
int64_t ar_kernel_launches(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int ar_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AR_GB300_H */
