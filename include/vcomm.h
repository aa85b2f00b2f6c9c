/*
 * vcomm.h -- collectives among N virtual ranks that all live in one GPU's memory.
 *
 * A communicator (vcomm_t) stands for N ranks whose send and receive buffers are
 * ordinary device allocations on the current GPU.  Each call moves or reduces data
 * between those buffers entirely on that GPU; no other GPU, process or network is
 * involved and no NCCL call is made.
 *
 * The interface follows the NCCL calls described in the NCCL book (aireadcode.com),
 * section 2.1 (communicator, async error) and chapter 6 (ncclAllReduce(sendbuff,
 * recvbuff, count, datatype, op, comm, stream) -> ncclInfo -> ncclEnqueueCheck), with
 * one change that the virtual ranks force: every rank's buffer is named at once, so
 * sendbuffs / recvbuffs are host arrays of N device pointers, rank r at index r.
 * The collectives' meaning is the collective table of "AI Systems Performance
 * Engineering (3)" (all-reduce, reduce-scatter, all-gather, broadcast, all-to-all).
 *
 * Stream contract ("NCCL Expert Course 29: ProcessGroupNCCL, Stream, Event and
 * Work"): every collective is enqueued on the caller's stream and returns as soon as
 * it is enqueued.  The caller keeps the device buffers alive and unmodified until the
 * stream work completes.  The host pointer arrays and tables are copied before the
 * call returns and may be freed right after it (as ncclInfo copies the user's config,
 * NCCL book chapter 6).
 *
 * Errors: a call returns vInvalidArgument for bad arguments and launches nothing.
 * Failures found on the device (a staged transfer that waits past its deadline, an
 * abort, a bad all-to-all table) are recorded in the communicator's sticky async
 * error (NCCL book section 2.1, asyncResult / ncclCommGetAsyncError); every later
 * call on that communicator returns that error without launching, and the
 * communicator must be destroyed.
 *
 * Threading: a communicator is used by one host thread at a time.  Staged ring transfers
 * on one communicator share its FIFOs, so they must not overlap on the GPU: issue them on
 * one stream or order the streams (NCCL orders a communicator's operations the same way).
 *
 * CUDA graphs: collectives may be captured into a graph.  A ring transfer can be
 * captured only after an eager ring call of at least the same size on the same
 * communicator (its FIFOs are allocated then; capturing it earlier returns
 * vInvalidUsage); the captured transfer clears its control words (and, for LL and LL128,
 * its FIFOs, whose lines carry the flags) before every replay.  Graph
 * replays are ordered by the caller: vcommDestroy waits only for eager launches.
 *
 * Launch: the one-pass kernels are launched with programmatic stream serialization
 * (programmatic dependent launch): a kernel may become resident while the previous
 * kernel on the stream finishes, and waits for that kernel's completion (and its memory)
 * before touching any buffer, so stream order is kept.  VCOMM_PDL=0 launches them
 * plainly.
 */
#ifndef VCOMM_H
#define VCOMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle, declared the same way cuda_runtime_api.h does. */
typedef struct CUstream_st* cudaStream_t;

#define VCOMM_MAX_RANKS 64
#define VCOMM_MAX_CHANNELS 64

typedef struct vcomm* vcomm_t;

/* Result codes.  vInvalidUsage = 5 matches NCCL's ncclInvalidUsage ("NCCL Expert
 * Course 17", duplicate-device probe, "code=5"). */
typedef enum {
    vSuccess = 0,
    vUnhandledCudaError = 1, /* a CUDA runtime call failed (no device, launch error, ...) */
    vSystemError = 2,        /* host allocation failed */
    vInternalError = 3,
    vInvalidArgument = 4,    /* bad pointer, size, type, op, root or communicator */
    vInvalidUsage = 5,       /* valid arguments the communicator cannot serve, e.g. a staged
                                protocol whose CTAs cannot all be resident at once */
    vTimeout = 6,            /* a staged transfer waited past its deadline (async) */
    vInProgress = 7,
    vAborted = 8             /* vcommAbort stopped a running staged transfer (async) */
} vResult_t;

typedef enum { vFloat32 = 0, vFloat16 = 1, vBFloat16 = 2, vInt32 = 3 } vDataType_t;

/* Reductions.  sum and prod on fp16/bf16 widen both operands to fp32, apply one fp32
 * operation (round to nearest even) and round back to the storage type; int32 sum and
 * prod wrap modulo 2^32; min/max keep the running partial unless the next element
 * compares strictly below/above it. */
typedef enum { vSum = 0, vProd = 1, vMin = 2, vMax = 3 } vRedOp_t;

/* Staging protocols of the ring path (NCCL book section 2.4, "protocol"):
 * Simple moves raw data through FIFO slots guarded by head/tail counters; LL packs
 * 4 bytes of data with a 4-byte flag in every 8-byte word (half the bandwidth); LL128
 * carries 120 bytes of data and an 8-byte flag in every 128-byte line.
 * vProtoAuto lets the planner choose the protocol its cost model predicts fastest for the
 * collective, size and channel count (a ring cost model in the form of the NCCL book's
 * ring.cc, latency + bytes / bandwidth per protocol and channel count, fitted to staged-ring
 * times measured on GB300 for every collective, protocol and size from 1 KiB to 1 GiB per
 * rank: 2.2 % median error, and a pick within 15 % of the fastest protocol measured). */
typedef enum { vProtoSimple = 0, vProtoLL = 1, vProtoLL128 = 2, vProtoAuto = 3 } vProto_t;

/* Algorithms.  vAlgoOnePass: one kernel reads every rank's buffer once and writes
 * every output once (the virtual-rank counterpart of NCCL's symmetric-memory kernels,
 * NCCL book chapter 5 section 5).  vAlgoRing: the literal ring of the NCCL book
 * section 2.3, N-1 reduce-scatter steps then N-1 all-gather steps, each hop staged
 * through a device FIFO with the communicator's protocol.  Both give identical bits.
 * vAlgoAuto picks the smaller predicted time (on GB300 the one-pass kernels are faster
 * at every size: about 2 us of latency against 8-55 us for the ring's steps).
 * vAlgoTree (all-reduce only; other collectives run one-pass): the double binary tree of
 * the NCCL book chapter 4 (ncclGetBtree / ncclGetDtree).  The first half of the buffer,
 * up to alignUp(ceil(count / 2), 16 / elemSize) elements, is reduced up tree 0, the rest
 * up tree 1; a tree node combines its own element, then child 0's partial, then child
 * 1's; every rank receives the root's result.  Its bits generally differ from the ring
 * order's (a different reduction order). */
typedef enum { vAlgoAuto = 0, vAlgoOnePass = 1, vAlgoRing = 2, vAlgoTree = 3 } vAlgo_t;

typedef enum {
    vCollAllReduce = 0, vCollReduceScatter = 1, vCollAllGather = 2,
    vCollBroadcast = 3, vCollAllToAll = 4, vCollAllToAllv = 5,
    vCollReduce = 6, vCollGather = 7, vCollScatter = 8
} vColl_t;

/* ------------------------------------------------------------------------------- */
/* Communicator lifecycle                                                           */
/* ------------------------------------------------------------------------------- */

/* Create a communicator of nRanks virtual ranks on the current CUDA device.
 * nRanks in [1, VCOMM_MAX_RANKS]; nChannels in [1, VCOMM_MAX_CHANNELS] is the number
 * of channels (independent CTA groups, each owning a contiguous sub-range of every
 * rank's block: NCCL book section 2.2, "each channel handles count/nChannels
 * elements"); protocol is the ring path's staging.  Out-of-range values give
 * vInvalidArgument and *comm is left NULL (as ncclCommInitRankDev rejects nranks < 1
 * with ncclInvalidArgument, "NCCL Expert Course 17").  No usable device gives
 * vUnhandledCudaError.  The communicator owns a small status block in pinned host
 * memory and, once a ring transfer is planned, its staging FIFOs in device memory.
 * Environment (read once here): VCOMM_ALGO=auto|onepass|ring|tree, VCOMM_CHUNK_BYTES,
 * VCOMM_TIMEOUT_MS, VCOMM_COPY_TMA=0|1 (0, the default: every thread loads and stores; 1:
 * all-gather, gather and broadcast stage tiles in shared memory with TMA bulk copies when
 * blocks are 16-byte aligned), VCOMM_GRID=flat|persistent (flat, the default: the
 * one-pass kernels launch one CTA per slice of work; persistent: about one resident wave
 * of CTAs striding over it), VCOMM_PDL=0|1 (1, the default: programmatic dependent
 * launch of the one-pass kernels), VCOMM_DEBUG=INFO (prints every plan to stderr). */
vResult_t vcommInit(vcomm_t* comm, int nRanks, int nChannels, vProto_t protocol);

/* Wait for the last enqueued work that uses the communicator's device memory (staged
 * ring transfers, variable all-to-all, bulk-copy fan-out), then free everything it owns.
 * The other collectives touch only the caller's buffers and need not have finished.
 * A NULL or already destroyed communicator gives vInvalidArgument. */
vResult_t vcommDestroy(vcomm_t comm);

/* Store the communicator's rank count N in *nRanks: the length that every sendbuffs and
 * recvbuffs array of a call on it must have (the communicator's nRanks field, NCCL book
 * section 2.1).  Host only.  A NULL pointer or a bad communicator gives vInvalidArgument. */
vResult_t vcommCount(vcomm_t comm, int* nRanks);

/* Store the sticky asynchronous error (vSuccess if none) in *asyncError.  Reads host
 * memory that the kernels write; it does not synchronize any stream.  A vTimeout is
 * fatal for the stream it happened on: the outputs of that call are undefined, and after
 * a timed-out bulk-copy fan-out (VCOMM_COPY_TMA=1) a load that had still not landed when
 * its CTA gave up may write into shared memory that a later kernel on the GPU uses, so
 * no later result is to be trusted either. */
vResult_t vcommGetAsyncError(vcomm_t comm, vResult_t* asyncError);

/* Ask running and future ring transfers of this communicator to stop: their waits
 * return and the sticky error becomes vAborted. */
vResult_t vcommAbort(vcomm_t comm);

const char* vcommGetErrorString(vResult_t result);

/* Group batching (NCCL book chapter 6 ncclPrepareTasks and chapter 7 ncclGroupStart /
 * ncclGroupEnd).  Between vcommGroupStart and vcommGroupEnd every collective call on
 * this communicator is recorded (its pointer arrays copied) and nothing is enqueued.  An
 * all-reduce is checked at the call, so its argument errors are returned there; the other
 * collectives return vSuccess and are checked when vcommGroupEnd enqueues them.
 * vcommGroupEnd enqueues the recorded calls: one-pass all-reduces of the same type, op,
 * stream and vector width are fused into one kernel launch (each keeping its own block
 * order, so the bits equal separate calls); a launch holds as many as its 32 KiB
 * parameter block fits, 32,496 / (40 + 16 N) of them (193 at N = 8), and a larger batch
 * takes several launches.  Every other call is enqueued as its own launch,
 * in call order.  Calls in one group must not depend on each other's results.  Groups
 * nest; only the outermost end enqueues.  vcommGroupEnd returns the first error of the
 * recorded calls, or vInvalidUsage without a matching start.  The work table travels in
 * the launch's parameters: no device memory, no upload, and on a stream being captured
 * into a CUDA graph the fused launch is captured like any other. */
vResult_t vcommGroupStart(vcomm_t comm);
vResult_t vcommGroupEnd(vcomm_t comm);

/* Tuning knobs (host only, take effect for later calls).  chunkBytes is the ring
 * path's data bytes per rank per chunk (one chunk = 4 FIFO slots, one slice = 2 slots;
 * NCCL book chapter 6, ALLREDUCE_CHUNKSTEPS / ALLREDUCE_SLICESTEPS); a slot holds
 * chunkBytes / 4 data bytes in chunkBytes / 4 FIFO bytes (Simple), twice that (LL) or
 * 128-byte lines of 120 data bytes (LL128).  It must be a power of two in [4 KiB,
 * 64 MiB], or 0 for the planner's default: the largest power of two <= 1 MiB that keeps
 * all of the communicator's FIFOs (8 slots per channel and rank) within 1 GiB.
 * timeoutMs bounds every device-side wait (>= 1). */
vResult_t vcommSetAlgo(vcomm_t comm, vAlgo_t algo);
vResult_t vcommSetProtocol(vcomm_t comm, vProto_t protocol);
vResult_t vcommSetChunkBytes(vcomm_t comm, size_t chunkBytes);
vResult_t vcommSetTimeoutMs(vcomm_t comm, int timeoutMs);

/* ------------------------------------------------------------------------------- */
/* Collectives.  sendbuffs / recvbuffs: host arrays of nRanks pointers to memory the */
/* device can access (device allocations, pinned or managed host memory: the kernels */
/* read and write it directly, so host buffers need no staging copies).              */
/* Any element-aligned pointer is accepted; when every pointer and the sizes allow   */
/* 16-byte (or 32-byte) vectors the vector path runs, otherwise an element path (for */
/* 2-byte types, 16-byte vectors realigned to the outputs where the offsets allow);  */
/* the output bits are the same.  The element paths read no byte outside the 16-byte */
/* aligned blocks that hold a buffer's own elements.  count == 0 returns vSuccess    */
/* and launches nothing (NCCL book chapter 6, taskAppend).  With nRanks == 1 every   */
/* collective is a copy.                                                             */
/* ------------------------------------------------------------------------------- */

/* All-reduce ("AI Systems Performance Engineering (3)", collective table, all-reduce row;
 * NCCL book section 2.3, the ring as reduce-scatter then all-gather):
 * recvbuffs[r][e] = the reduction over all ranks of sendbuffs[.][e], e < count, for
 * every rank r.  Element e belongs to block b = e / B with
 * B = alignUp(ceil(count / nRanks), 16 / elemSize) (the tail-chunk rule of
 * RingARAlgorithm::getNextSendAddr, NCCL book section 2.3), and block b is reduced in
 * ring order: ranks b+1, b+2, ..., b (mod nRanks), each partial rounded to the data
 * type.  In place (sendbuffs[r] == recvbuffs[r]) is allowed; other overlap is not. */
vResult_t vAllReduce(const void* const* sendbuffs, void* const* recvbuffs, size_t count,
                     vDataType_t datatype, vRedOp_t op, vcomm_t comm, cudaStream_t stream);

/* Reduce-scatter ("AI Systems Performance Engineering (3)", collective table,
 * reduce-scatter row: rank r ends with the reduction of block r; the reduce-scatter half
 * of the ring in the NCCL book section 2.3).
 * sendbuffs[r] holds nRanks * recvcount elements; recvbuffs[r][t] = the reduction of
 * sendbuffs[.][r * recvcount + t] in ring order ranks r+1, ..., r.  In place means
 * recvbuffs[r] == sendbuffs[r] + r * recvcount. */
vResult_t vReduceScatter(const void* const* sendbuffs, void* const* recvbuffs, size_t recvcount,
                         vDataType_t datatype, vRedOp_t op, vcomm_t comm, cudaStream_t stream);

/* vReduceScatter with a fused epilogue: recvbuffs[r][t] = (float)acc * scale computed
 * in fp32 (round to nearest even) and stored as outType, which is vFloat32 or the
 * input type.  datatype must be a floating type.  For gradient averaging scale is
 * 1/nRanks ("AI Systems Performance Engineering (3)", p.grad /= world_size). */
vResult_t vReduceScatterScaleCast(const void* const* sendbuffs, void* const* recvbuffs,
                                  size_t recvcount, vDataType_t datatype, vRedOp_t op,
                                  vDataType_t outType, float scale, vcomm_t comm,
                                  cudaStream_t stream);

/* All-gather ("AI Systems Performance Engineering (3)", collective table, all-gather row:
 * every rank ends with every rank's piece, in rank order; the ring all-gather of "NCCL
 * Expert Course 17" and NCCL book section 2.3 when staged):
 * recvbuffs[r][s * sendcount + t] = sendbuffs[s][t] for every r.  op is ignored (the
 * data is moved as bytes).  In place means sendbuffs[r] == recvbuffs[r] + r * sendcount. */
vResult_t vAllGather(const void* const* sendbuffs, void* const* recvbuffs, size_t sendcount,
                     vDataType_t datatype, vRedOp_t op, vcomm_t comm, cudaStream_t stream);

/* Broadcast ("AI Systems Performance Engineering (3)", collective table, broadcast row:
 * the root's buffer copied to every rank):
 * recvbuffs[r][0..count) = sendbuffs[root][0..count) for every r; root in [0, nRanks).
 * Only sendbuffs[root] is read; the other entries may be NULL.  op is ignored. */
vResult_t vBroadcast(const void* const* sendbuffs, void* const* recvbuffs, size_t count,
                     vDataType_t datatype, vRedOp_t op, int root, vcomm_t comm,
                     cudaStream_t stream);

/* Uniform all-to-all ("AI Systems Performance Engineering (3)", collective table,
 * all-to-all row: rank i's block j goes to rank j as its block i): count elements per
 * block, nRanks blocks per buffer;
 * recvbuffs[j][i * count + t] = sendbuffs[i][j * count + t].  op is ignored.
 * Send and receive buffers must not overlap. */
vResult_t vAllToAll(const void* const* sendbuffs, void* const* recvbuffs, size_t count,
                    vDataType_t datatype, vRedOp_t op, vcomm_t comm, cudaStream_t stream);

/* Variable all-to-all.  counts, sdispls and rdispls are DEVICE arrays of nRanks *
 * nRanks int32 values, in elements: counts[i * nRanks + j] elements go from
 * sendbuffs[i] + sdispls[i * nRanks + j] to recvbuffs[j] + rdispls[j * nRanks + i].
 * The caller guarantees that every block lies inside its buffers.  A rank that sends
 * (receives) nothing may pass a NULL send (receive) buffer, as an empty tensor has.  A
 * negative entry, or a positive count whose source or destination buffer is NULL, makes
 * the kernel skip that block and sets the sticky error vInvalidArgument.  Send and
 * receive buffers must not overlap.
 * Each call hands out its tiles from a pair of counters that the communicator owns.
 * Eager calls rotate through 64 pairs; a call captured into a CUDA graph keeps the pair
 * it was captured with, taken from a second set of 64 that eager calls never use.  So an
 * eager call may run on the GPU at the same time as a replay of a captured call, and up
 * to 64 eager calls may be in flight together; beyond that, vAllToAllv kernels on one
 * communicator must not overlap on the GPU (two replays of one graph, or of calls
 * captured 64 captured calls apart, share a pair). */
vResult_t vAllToAllv(const void* const* sendbuffs, void* const* recvbuffs, const int32_t* counts,
                     const int32_t* sdispls, const int32_t* rdispls, vDataType_t datatype,
                     vcomm_t comm, cudaStream_t stream);

/* Rooted collectives ("AI Systems Performance Engineering (3)", collective table:
 * reduce, gather and scatter rows).  root in [0, nRanks); recvbuffs / sendbuffs entries
 * that the call does not use may be NULL.
 *
 * vReduce: recvbuffs[root][e] = the reduction of sendbuffs[.][e] for e < count, every
 * element in the order of a ring chain that ends at the root: ranks root+1, ..., root
 * (the order block `root` of vAllReduce uses).  In place: recvbuffs[root] ==
 * sendbuffs[root].
 * vGather: recvbuffs[root][s * sendcount + t] = sendbuffs[s][t].  In place:
 * sendbuffs[root] == recvbuffs[root] + root * sendcount.
 * vScatter: recvbuffs[r][t] = sendbuffs[root][r * recvcount + t].  In place:
 * recvbuffs[root] == sendbuffs[root] + root * recvcount. */
vResult_t vReduce(const void* const* sendbuffs, void* const* recvbuffs, size_t count,
                  vDataType_t datatype, vRedOp_t op, int root, vcomm_t comm, cudaStream_t stream);
vResult_t vGather(const void* const* sendbuffs, void* const* recvbuffs, size_t sendcount,
                  vDataType_t datatype, int root, vcomm_t comm, cudaStream_t stream);
vResult_t vScatter(const void* const* sendbuffs, void* const* recvbuffs, size_t recvcount,
                   vDataType_t datatype, int root, vcomm_t comm, cudaStream_t stream);

/* Ring all-reduce for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call; it exists for code that must not call cudaMalloc (allocator
 * or memory-pool callbacks, which must not re-enter the allocator; runtimes that own all
 * device memory and hand it out themselves).  No communicator is needed and nothing is
 * allocated: the staging FIFOs and control words live in one fixed device array inside
 * this library (64 KiB + 8 MiB, held on every GPU that loads the library until the
 * process exits).
 * The result is bit-identical to vAllReduce.  The caller passes the buffers as for
 * vAllReduce plus nRanks (2..64), nChannels and protocol (Simple, LL or LL128); the
 * ring uses chunks of 64 KiB of data (32 KiB for LL and LL128, whose slots take more FIFO
 * bytes than they carry), so nRanks * nChannels may be at most 64 -- larger rings
 * return vInvalidArgument (as do the usual argument errors), and a ring whose CTAs
 * cannot all be resident returns vInvalidUsage.  The first call on a device looks up
 * the array's address (cudaGetSymbolAddress), so make it before any stream capture;
 * every call checks the kept address (cudaPointerGetAttributes) and looks it up again
 * after a cudaDeviceReset.
 * Every call clears and reuses the same array: calls whose kernels overlap on the GPU
 * (another stream, another thread) race and must be serialized by the caller.  Waits
 * inside the kernel still end after 2 s without progress, but such a failure is not
 * reported (there is no communicator to hold an error) and the output is then
 * undefined. */
vResult_t vAllReduceNoAlloc(const void* const* sendbuffs, void* const* recvbuffs, size_t count,
                            vDataType_t datatype, vRedOp_t op, int nRanks, int nChannels,
                            vProto_t protocol, cudaStream_t stream);

/* ------------------------------------------------------------------------------- */
/* Planner (host only; needs no GPU)                                                */
/* ------------------------------------------------------------------------------- */

typedef struct {
    int nRanks, nChannels;
    int proto;                 /* vProto_t requested */
    int algo;                  /* vAlgo_t requested */
    int coll;                  /* vColl_t */
    int datatype;              /* vDataType_t */
    size_t count;              /* elements: AR/BC/Reduce count, RS/Scatter recvcount,
                                  AG/Gather sendcount, A2A block */
    size_t chunkBytes;         /* ring chunk bytes per rank (0 = default) */
    int aligned16;             /* 1 if every buffer pointer is 16-byte aligned */
    int smCount;               /* streaming multiprocessors of the device */
    size_t l2Bytes;            /* L2 cache size of the device (kept for callers; the current
                                  plans do not depend on it) */
    int aligned32;             /* 1 if every buffer pointer is 32-byte aligned */
    int noBulkCopy;            /* 1: never use TMA bulk copies (a communicator sets it unless
                                  VCOMM_COPY_TMA=1) */
    int persistentGrid;        /* 1: one-pass grids of about one resident wave whose CTAs
                                  stride over their work (VCOMM_GRID=persistent); 0 (the
                                  default): one CTA per slice of work, dispatched in order */
} vPlanRequest_t;

typedef struct {
    int algo;                  /* vAlgo_t chosen: vAlgoOnePass or vAlgoRing */
    int proto;                 /* vProto_t used by the ring path */
    int nChannels;
    int ctasPerChannel;        /* one-pass: CTAs in each channel's group */
    int gridCtas;              /* CTAs launched */
    int threadsPerCta;
    int vectorized;            /* 1 when the 16-byte vector path runs */
    int launches;              /* kernel launches of the call */
    size_t blockElems;         /* B: elements of one rank block (AR rule, or RS/AG block) */
    size_t channelElems;       /* elements of each block that one channel owns */
    size_t chunkElems;         /* ring: elements per block per chunk */
    size_t slotPayloadElems;   /* ring: data elements carried by one FIFO slot */
    size_t slotBytes;          /* ring: bytes of one FIFO slot (payload + flags) */
    size_t fifoBytes;          /* ring: bytes of one (channel, rank) FIFO, 8 slots */
    double minBytes;           /* algorithmic minimum HBM bytes read + written */
    double busFactor;          /* busBW = algBW * busFactor (nSteps / nRanks) */
    int vecBytes;              /* bytes per vector access of the one-pass kernels: 0, 16, 32 */
    int bulkCopy;              /* 1: all-gather / gather / broadcast through TMA bulk copies */
    double predictedUs;        /* the planner's cost model for this plan (GB300 fit) */
    size_t tileBytes;          /* copies (load/store path): bytes each CTA moves per tile */
    int tmaStages;             /* bulk-copy fan-out: shared-memory tile stages per CTA */
} vPlanInfo_t;

/* Compute the plan a collective with these parameters would run.  Pure host
 * arithmetic; returns vInvalidArgument for out-of-range requests. */
vResult_t vPlanCompute(const vPlanRequest_t* request, vPlanInfo_t* plan);

/* The element range [*lo, *hi) of block `block` owned by `channel` under `plan`
 * (empty when *lo == *hi).  count is the request's total element count per rank
 * (AR count; nRanks * recvcount for RS).  Host only. */
vResult_t vPlanChannelRange(const vPlanInfo_t* plan, size_t count, int channel, int block,
                            size_t* lo, size_t* hi);

/* Test hook for failure detection: rank `rank` of every later ring transfer never
 * starts (its CTAs return at once), so its neighbours' bounded waits run out and the
 * transfer ends with the sticky error vTimeout.  -1 turns the hook off. */
vResult_t vcommTestSetStallRank(vcomm_t comm, int rank);

/* Test hook for the LL128 line check: in every later LL128 ring transfer rank `rank`
 * expects wrong line flags (as if its predecessor had stored wrong ones; the per-warp
 * release flags it polls stay right), so it finds a line whose flag does not match after
 * the release flag did and ends the transfer with the sticky error vInternalError.  -1
 * turns the hook off. */
vResult_t vcommTestSetBadFlagRank(vcomm_t comm, int rank);

/* Test hook: staged ring transfers sleep for pseudo-random times of up to maxNs
 * nanoseconds (0 = off, at most 1,000,000) where a producer publishes a slot and where a
 * consumer observes one, so that tests exercise orderings of stores and flag reads that
 * rarely occur on their own.  Results must not change. */
vResult_t vcommTestSetJitterNs(vcomm_t comm, unsigned int maxNs);

/* Links of `rank` in tree `tree` (0 or 1) of the double binary tree over nRanks ranks
 * (NCCL book chapter 4, ncclGetBtree / ncclGetDtree): tree 0 hangs from rank 0, a
 * rank's lowest set bit fixes its level; tree 1 mirrors it (rank r -> nRanks-1-r) for an
 * even rank count and shifts it (r -> r+1) for an odd one.  -1 marks a missing link. */
vResult_t vPlanTreeLinks(int nRanks, int rank, int tree, int* parent, int* child0, int* child1);

/* vPlanCompute for this communicator's device and settings.  `aligned` is the largest
 * power-of-two alignment (in bytes, up to 32) shared by every buffer pointer. */
vResult_t vcommQueryPlan(vcomm_t comm, vColl_t coll, size_t count, vDataType_t datatype,
                         int aligned, vPlanInfo_t* plan);

#ifdef __cplusplus
}
#endif
#endif /* VCOMM_H */
