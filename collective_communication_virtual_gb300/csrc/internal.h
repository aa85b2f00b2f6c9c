// internal.h -- argument blocks and launchers shared by the host side of libvcomm and
// its kernels.  Not part of the public ABI (that is include/vcomm.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "vcomm.h"

namespace vc {

constexpr int kFifoSlots = 8;        // NCCL_STEPS: slots per (channel, rank) FIFO
constexpr int kChunkSlots = 4;       // ALLREDUCE_CHUNKSTEPS = NCCL_STEPS / 2
constexpr int kSliceSlots = 2;       // ALLREDUCE_SLICESTEPS = NCCL_STEPS / 4
constexpr int kOnePassThreads = 512;
constexpr int kRingThreads = 512;
constexpr int kCtrlStride = 32;      // u64 words per (channel, rank) control block (256 B)

// First-error-wins status word.  The device copy decides the winner; a mirror in
// pinned, device-mapped host memory lets the host read it without synchronizing.
struct Status {
    unsigned int code;               // vResult_t, 0 = no error
    unsigned int channel;
    unsigned int rank;
    unsigned int step;               // ring: slot sequence number that gave up
};

// One-pass kernels: all-reduce, reduce-scatter, all-gather, broadcast, all-to-all.
struct OnePassArgs {
    const void* send[VCOMM_MAX_RANKS];
    void* recv[VCOMM_MAX_RANKS];
    int nRanks;
    int ctasPerChannel;
    int root;                        // broadcast, scatter
    int orderRoot;                   // >= 0: every element reduced in the order of block
                                     // orderRoot (reduce to root); -1: per block
    int outRoot;                     // >= 0: only recv[outRoot] is written (reduce, gather)
    int hasScale;                    // reduce-scatter epilogue
    float scale;
    size_t count;                    // AR: count; RS: N*recvcount; AG: sendcount; BC: count; A2A: block
    size_t blockElems;               // B
    size_t chanElems;                // elements of each block owned by one channel
    size_t tileBytes;                // copy kernels: bytes of one CTA's tile
};

struct A2AvArgs {
    const void* send[VCOMM_MAX_RANKS];
    void* recv[VCOMM_MAX_RANKS];
    const int32_t* counts;           // [sender * N + receiver]
    const int32_t* sdispls;          // [sender * N + receiver]
    const int32_t* rdispls;          // [receiver * N + sender]
    int nRanks;
    int elemSize;
    size_t tileBytes;
    unsigned int* tileCounter;       // {next tile, CTAs done}: zero at launch, reset by the
                                     // last CTA to finish
    Status* status;                  // device copy
    volatile Status* statusHost;     // pinned mirror
};
// Tile-counter pairs of a communicator.  Eager variable all-to-alls rotate through the
// first kTileCounterSlots pairs, so that calls in flight at the same time (on different
// streams) use different counters; a call captured into a CUDA graph keeps its pair for
// every replay, so captured calls take theirs, one per captured call, from the next
// kCapturedCounterSlots pairs, which eager calls never use.
constexpr int kTileCounterSlots = 64;
constexpr int kCapturedCounterSlots = 64;
constexpr int kAllCounterSlots = kTileCounterSlots + kCapturedCounterSlots;

// Staged ring kernels: one CTA per (channel, rank).
struct RingArgs {
    const void* send[VCOMM_MAX_RANKS];
    void* recv[VCOMM_MAX_RANKS];
    int nRanks;
    int nChannels;
    int coll;                        // vColl_t: AR, RS, AG or BC
    int op;                          // vRedOp_t
    int root;
    int aligned;                     // user buffers allow 16-byte vectors
    int hasScale;
    float scale;
    size_t count;                    // as OnePassArgs
    size_t blockElems;
    size_t chanElems;
    size_t chunkElems;               // elements per block per chunk (4 slots)
    size_t slotElems;                // payload elements per slot
    size_t slotBytes;                // physical bytes per slot
    char* fifo;                      // (channel, rank) FIFO at fifo + (ch * N + r) * 8 * slotBytes
    unsigned long long* ctrl;        // (channel, rank) block: [0] = head, [16] = tail
    unsigned long long epochHi;      // launch epoch << 32 (Simple counters, LL128 flags)
    unsigned int llEpoch;            // (epoch & 0xFF) << 24 (LL flags)
    unsigned long long timeoutNs;
    volatile unsigned int* abortHost;   // host-set abort (pinned, mapped)
    unsigned int* abortDev;          // set by any CTA that gives up
    Status* status;                  // device copy
    volatile Status* statusHost;     // pinned mirror
    int testStallRank;               // test hook: this rank never posts data (-1 = off)
    unsigned int testJitterNs;       // test hook: random sleeps up to this long where the
                                     // protocols publish or observe a slot (0 = off)
    int testBadFlagRank;             // test hook: this rank expects wrong LL128 line flags
                                     // (its release flags are right; -1 = off)
};

// Double-binary-tree all-reduce.  prog[t] lists tree t's ranks in post-order (children
// before parents, child 0's subtree before child 1's); nchild[t][i] is the number of
// children of prog[t][i].
struct TreeArgs {
    const void* send[VCOMM_MAX_RANKS];
    void* recv[VCOMM_MAX_RANKS];
    signed char prog[2][VCOMM_MAX_RANKS];
    signed char nchild[2][VCOMM_MAX_RANKS];
    int nRanks;
    size_t count;
    size_t split;                    // elements [0, split) use tree 0
};
constexpr int kTreeMaxStack = 16;
// Elements a thread reduces at once on the element paths (buffers that 16-byte vectors
// cannot cover); the planner and the group batcher size their work units by it.
constexpr int kElemsPerThread = 8;

cudaError_t launch_allreduce_tree(const TreeArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                  int threads, cudaStream_t s);

// A batch of all-reduces of one type and op run by one launch (group batching).  The work
// table travels inside the kernel's parameter block (which may hold up to 32,764 bytes), so
// a batch needs no upload, no device memory and no host staging, and a launch captured
// into a CUDA graph carries its own copy.  table: items[0..nItems) (item i describes
// all-reduce i), then at byte ptrByteOff the rank pointers: item i's 2*N pointers are
// ptrs[items[i].ptrOff .. + 2N) (send pointers, then receive pointers).
// Programmatic dependent launch of the one-pass kernels for the calling thread's next
// launches (set from the communicator of the call: on unless it was created with
// VCOMM_PDL=0).
bool& pdl_enabled();

// Largest grid the flat one-pass launches use; kernels stride over anything beyond.
constexpr int kMaxGridCtas = 1 << 30;
constexpr int kGroupTableBytes = 32 * 1024 - 256;
struct GroupItem {
    unsigned long long unitStart;    // first flat work unit of this item
    unsigned long long count;        // elements per rank
    unsigned long long blockElems;   // B of this all-reduce
    unsigned long long unitsPerBlock;
    int ptrOff;
    int pad;
};
struct GroupArgs {
    int nItems;
    int nRanks;
    unsigned long long totalUnits;
    int ptrByteOff;                  // multiple of 16
    int pad;
    alignas(16) unsigned char table[kGroupTableBytes];
};
// Items one launch can hold for nRanks ranks, and the most for any rank count.
constexpr int group_capacity(int nRanks) {
    return (int)((kGroupTableBytes - 16) / (sizeof(GroupItem) + 2 * (size_t)nRanks * sizeof(void*)));
}
constexpr int kMaxGroupItems = group_capacity(1);
static_assert(sizeof(GroupArgs) <= 32764, "kernel parameters are limited to 32,764 bytes");

// Launchers (defined in the kernel translation units).  Each returns the launch status.
// vb: bytes per vector of the one-pass reductions, 0 (element path), 16 or 32.
cudaError_t launch_allreduce_onepass(const OnePassArgs& a, vDataType_t dt, vRedOp_t op, int vb,
                                     int grid, int threads, cudaStream_t s);
cudaError_t launch_reduce_scatter_onepass(const OnePassArgs& a, vDataType_t dt, vRedOp_t op,
                                          vDataType_t outType, int vb, int grid, int threads,
                                          cudaStream_t s);
cudaError_t launch_allreduce_group(const GroupArgs& a, vDataType_t dt, vRedOp_t op, int vb, int grid,
                                   int threads, cudaStream_t s);
cudaError_t launch_allgather_onepass(const OnePassArgs& a, int elemSize, int vb, int grid,
                                     int threads, cudaStream_t s);
cudaError_t launch_broadcast_onepass(const OnePassArgs& a, int elemSize, int vb, int grid,
                                     int threads, cudaStream_t s);
cudaError_t launch_alltoall_onepass(const OnePassArgs& a, int elemSize, int vb, int grid,
                                    int threads, cudaStream_t s);
// Bulk-copy (TMA) all-gather / gather / broadcast: blocks must be 16-byte aligned and a
// multiple of 16 bytes.  Grid: up to 3 single-warp CTAs per SM (64 KiB of stages each).
constexpr int kTmaCtasPerSm = 3;
cudaError_t launch_fanout_tma(const OnePassArgs& a, int elemSize, bool broadcast, int grid, int stages,
                              Status* st, volatile Status* stHost, cudaStream_t s);
cudaError_t launch_scatter_onepass(const OnePassArgs& a, int elemSize, int vb, int grid,
                                   int threads, cudaStream_t s);
cudaError_t launch_alltoallv(const A2AvArgs& a, int grid, int threads, cudaStream_t s);

// Cooperative launch of the staged ring (all CTAs co-resident or the launch fails).
cudaError_t launch_ring(const RingArgs& a, vDataType_t dt, vRedOp_t op, vDataType_t outType,
                        vProto_t proto, int grid, int threads, cudaStream_t s);
// Largest co-resident grid for the ring kernel of this type/op/protocol.
cudaError_t ring_max_coresident(vDataType_t dt, vRedOp_t op, vDataType_t outType, vProto_t proto,
                                int threads, int smCount, int* maxCtas);

}  // namespace vc
